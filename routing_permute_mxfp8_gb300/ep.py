"""Expert-parallel MegaMoE forward (epWorldSize > 1) over torch.distributed.

MegaMoE README, A8W8-FP scenario, with W = ep_world_size ranks, rank r holding
the experts [r*E/W, (r+1)*E/W):
  stage 1  each rank MX-quantises its tokens and sends every (token, choice)
           row to the rank that holds the chosen expert (mm_moe_ep_dispatch,
           then an all-to-all of the per-rank counts and of the rows, their
           E8M0 scales and their local expert ids);
  stage 2-3 each rank runs its experts' GEMM1 + activation + GEMM2 on the rows
           it received (mm_moe_expert_ffn: the received FP8 rows and scales
           passed through, each row's result written at its own position, the
           order in which the rows go back);
  stage 4  the O rows go back to their source ranks in the order they came
           (the reverse all-to-all; with combineQuantMode 3 / 4 as MXFP8
           E5M2 / E4M3 codes and E8M0 scales), where mm_moe_combine forms
           Y[i] = sum_k W[i,k] O[pi(i,k)] in fp32 and rounds once to bf16.
Shared experts take part in no exchange: each rank runs them on its own
tokens (quantised in the shared experts' input type, through the expert-side
entry point with one local expert) and the combine adds their rows after the
K routed terms, as the single-GPU step does.
Every step on the data runs in the library's kernels; this module only
allocates buffers and calls the collectives.  With the NCCL backend the
exchanges run on device memory; with gloo (which exchanges host memory) the
buffers are staged through the host.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

import routing_permute_mxfp8_gb300 as _mm


def _a2a_rows(send, send_counts, recv_counts, group):
    """All-to-all of the rows of a 2-D tensor with per-rank row counts
    (python lists); rows travel as bytes.  Returns the received rows."""
    row_bytes = send.shape[1] * send.element_size()
    sb = send.contiguous().view(torch.uint8).reshape(send.shape[0], row_bytes)
    staged = dist.get_backend(group) == "gloo" and sb.is_cuda
    src = sb.cpu() if staged else sb
    out = torch.empty((sum(recv_counts), row_bytes), dtype=torch.uint8, device=src.device)
    dist.all_to_all_single(out, src, output_split_sizes=list(recv_counts), input_split_sizes=list(send_counts),
                           group=group)
    if staged:
        out = out.to(send.device)
    return out.view(send.dtype).reshape(out.shape[0], send.shape[1])


def mega_moe_ep(x, topk_ids, topk_weights, weight1, weight2, weight_scales1, weight_scales2, moe_expert_num: int, *,
                group=None, weight_dtype: int = _mm.DT_FP8_E4M3FN, weight_scale_layout: int = _mm.WSCALE_ROWS,
                dispatch_quant_out_dtype: int = _mm.DT_FP8_E4M3FN, activation: str = "swiglu",
                activation_params=(), dev_err=None, shared_weight1=None, shared_weight2=None,
                shared_weight_scales1=None, shared_weight_scales2=None, shared_weight_dtype=None,
                shared_expert_quant_out_dtype=None, combine_quant_mode: int = 0):
    """MegaMoE forward of this rank's tokens with expert parallelism.

    x [N, H] bf16, topk_ids [N, K] int32 (global expert ids), topk_weights [N, K]
    fp32 / bf16 of this rank; weight1 / weight2 / their scales hold this rank's
    E/W local experts in the layouts of mm_mega_moe; shared_weight* hold the
    shared experts (every rank holds all of them, [S, ...] as in mm_mega_moe).
    Collective: every rank of `group` calls it.  Returns y [N, H] bf16.
    """
    world = dist.get_world_size(group)
    if moe_expert_num % world != 0:
        raise _mm.MMError("moe_expert_num must be a multiple of the EP world size")
    e_local = moe_expert_num // world
    if weight1.shape[0] != e_local:
        raise _mm.MMError(f"weight1 holds {weight1.shape[0]} experts, {e_local} expected on each rank")
    n, h = x.shape
    # stage 1: quantise and order the rows by destination rank
    send_x, send_s, send_e, counts, exp_idx = _mm.mm_moe_ep_dispatch(
        x, topk_ids, moe_expert_num, world, dispatch_quant_out_dtype, dev_err=dev_err)
    send_counts = [int(c) for c in counts.cpu().tolist()]
    # exchange the counts, then the rows, scales and local expert ids
    cnt = counts.view(torch.uint8).reshape(world, 8)
    recv_cnt = _a2a_rows(cnt, [1] * world, [1] * world, group)
    recv_counts = [int(c) for c in recv_cnt.reshape(world, 8).view(torch.int64).reshape(-1).cpu().tolist()]
    recv_x = _a2a_rows(send_x, send_counts, recv_counts, group)
    recv_s = _a2a_rows(send_s, send_counts, recv_counts, group)
    recv_e = _a2a_rows(send_e.view(-1, 1), send_counts, recv_counts, group)
    m = recv_x.shape[0]
    # stages 2-3 on this rank's experts: one choice per received row, weight 1,
    # the received FP8 rows and scales passed through
    if m > 0:
        o_rows = _mm.mm_moe_expert_ffn(recv_x, recv_s, recv_e.reshape(m).contiguous(), weight1, weight2,
                                       weight_scales1, weight_scales2, e_local, x_dtype=dispatch_quant_out_dtype,
                                       weight_dtype=weight_dtype, weight_scale_layout=weight_scale_layout,
                                       activation=activation, activation_params=activation_params,
                                       dev_err=dev_err)[0]
    else:
        o_rows = torch.empty((0, h), dtype=torch.bfloat16, device=x.device)
    # stage 4: rows back to their source ranks in send order (MXFP8 codes and
    # scales under combine quantisation), then the weighted sum
    if combine_quant_mode not in (0, 3, 4):
        raise _mm.MMError("combine_quant_mode must be 0, 3 or 4")
    cfmt = {3: _mm.DT_FP8_E5M2, 4: _mm.DT_FP8_E4M3FN}.get(combine_quant_mode)
    back_s = None
    if cfmt is None:
        back = _a2a_rows(o_rows, recv_counts, send_counts, group)
    else:
        if m > 0:
            oq, os_ = _mm.mm_mx_quantize(o_rows, cfmt, scale_cols=h // 32)
        else:
            oq = torch.empty((0, h), dtype=torch.uint8, device=x.device)
            os_ = torch.empty((0, h // 32), dtype=torch.uint8, device=x.device)
        back = _a2a_rows(oq, recv_counts, send_counts, group)
        back_s = _a2a_rows(os_, recv_counts, send_counts, group)
    if n == 0:
        return torch.empty((0, h), dtype=torch.bfloat16, device=x.device)
    shared = None
    if shared_weight1 is not None and shared_weight1.shape[0] > 0:
        shared = _shared_rows(x, shared_weight1, shared_weight2, shared_weight_scales1, shared_weight_scales2,
                              weight_dtype if shared_weight_dtype is None else shared_weight_dtype,
                              dispatch_quant_out_dtype if shared_expert_quant_out_dtype is None
                              else shared_expert_quant_out_dtype,
                              weight_scale_layout, activation, activation_params, dev_err)
    return _mm.mm_moe_combine(back, exp_idx, topk_weights, shared_rows=shared, expert_scales=back_s,
                              expert_rows_dtype=cfmt)


def _shared_rows(x, w1, w2, s1, s2, w_dtype, x_dtype, layout, activation, activation_params, dev_err):
    """[S, N, H] bf16: every shared expert's output for this rank's tokens (the
    tokens MX-quantised in the shared experts' input type, then the expert side
    with one local expert)."""
    n, h = x.shape
    xq, xs = _mm.mm_mx_quantize(x, x_dtype, scale_cols=h // 32)
    ids = torch.zeros(n, dtype=torch.int32, device=x.device)
    out = torch.empty((w1.shape[0], n, h), dtype=torch.bfloat16, device=x.device)
    S = w1.shape[0]
    # one expert's scales: a [1, ...] slice of the pages' layout, or one
    # expert's equal share of a prepared buffer
    one = (lambda t, s: t[s:s + 1]) if layout == _mm.WSCALE_ROWS else (lambda t, s: t.reshape(S, -1)[s])
    for s in range(S):
        _mm.mm_moe_expert_ffn(xq, xs, ids, w1[s:s + 1], w2[s:s + 1], one(s1, s), one(s2, s), 1, x_dtype=x_dtype,
                              weight_dtype=w_dtype, weight_scale_layout=layout, activation=activation,
                              activation_params=activation_params, out=out[s], dev_err=dev_err)
    return out
