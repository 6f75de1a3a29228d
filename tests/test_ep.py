"""Expert parallelism (MegaMoE README, A8W8-FP stages 1-4 with epWorldSize > 1):
the exchange plan of routing_permute_mxfp8_gb300.ep with two ranks.

CPU (gloo, two processes): the three kernel entry points the EP path calls
are replaced, inside the test only, by CPU versions built from the oracle, so
the collectives, split sizes, row orders and the combine indices are checked
on the host: the two-rank result must equal, bit for bit, the same fakes run
on one rank without any exchange, and the oracle's MegaMoE within tolerance.

GPU (two processes on the one GPU, gloo with the buffers staged through host
memory): the library's kernels on each rank; Y must equal the single-process
mm_mega_moe bit for bit (each row's GEMMs, its bf16 O and the k-ordered
combine are the same arithmetic), and the oracle within tolerance.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
W = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cfg(a4w4=False, shared=0):
    import synth
    # 2 ranks x 4 experts; Zipf routing so the two ranks receive unequal row counts
    cfg = synth.CONFIGS["tiny"].scaled(n=96, e=8, k=3, routing="zipf", dispatch_fmt=23, gate_dtype="bf16",
                                       shared=shared)
    # A4W4-FP: MXFP4 rows exchanged (packed, H/2 bytes a row), FP4 weights
    return cfg.scaled(weight_fmt=296, dispatch_fmt=296) if a4w4 else cfg


def _pack_fp4(c):
    """One FP4 code per byte -> the library's packed bytes (element 2i in bits 0-3)."""
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def _problem(a4w4=False, shared=0):
    import oracle
    import synth
    cfg = _cfg(a4w4, shared)
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    gate = synth.topk_weights(cfg)
    w1, s1 = oracle.quantized_weights(cfg, 1)
    w2, s2 = oracle.quantized_weights(cfg, 2)
    return cfg, x, ids, gate, (w1, s1, w2, s2)


def _shared(cfg):
    import oracle
    if not cfg.shared:
        return None
    sw1, ss1 = oracle.quantized_weights(cfg, 1, shared=True)
    sw2, ss2 = oracle.quantized_weights(cfg, 2, shared=True)
    return sw1, ss1, sw2, ss2


def _oracle_fakes(mm, cfg):
    """CPU stand-ins for mm_moe_ep_dispatch / mm_mega_moe / mm_moe_expert_ffn / mm_moe_combine,
    computed by the oracle (test infrastructure only)."""
    import oracle

    def dispatch(x, ids, moe_expert_num, world, fmt, workspace=None, dev_err=None):
        e_local = moe_expert_num // world
        idn = ids.numpy()
        n, k = idn.shape
        h = x.shape[1]
        srt, exp, cnt, bad = oracle.route((idn // e_local).astype(np.int32), world)
        assert bad == 0
        q, sc = oracle.permute(x.view(torch.int16).numpy().view(np.uint16), oracle.DT_BF16, k, srt, n * k, fmt)
        send_e = (idn.reshape(-1)[srt] % e_local).astype(np.int32)
        return (torch.from_numpy(q), torch.from_numpy(np.ascontiguousarray(sc[:, :h // 32])), torch.from_numpy(send_e),
                torch.from_numpy(cnt.astype(np.int64)), torch.from_numpy(exp.astype(np.int32)))

    def mega(xq, ids, gate, w1, w2, s1, s2, e, *, x_scales=None, dispatch_quant_out_dtype=None, **kw):
        assert kw.get("dispatch_quant_mode") == 0
        _, yb = oracle.mega_moe_tokens(None, ids.numpy(), gate.numpy(), w1.numpy(), s1.numpy(), w2.numpy(), s2.numpy(),
                                       dispatch_quant_out_dtype, cfg.weight_fmt,
                                       x_prequant=(xq.numpy(), x_scales.numpy()))
        return (torch.from_numpy(yb.view(np.int16)).view(torch.bfloat16),)

    def expert_ffn(xq, xs, eids, w1, w2, s1, s2, e, *, x_dtype=None, out=None, **kw):
        m = xq.shape[0]
        y = mega(xq, eids.view(m, 1), torch.ones((m, 1)), w1, w2, s1, s2, e, x_scales=xs,
                 dispatch_quant_out_dtype=x_dtype, dispatch_quant_mode=0)[0]
        if out is not None:
            out.copy_(y)
        return y, None

    def mx_quantize(src, out_dtype, scale_cols=None):
        q, sc = oracle.mx_quantize(src.view(torch.int16).numpy().view(np.uint16), oracle.DT_BF16, out_dtype,
                                   s_cols=scale_cols)
        return torch.from_numpy(q), torch.from_numpy(np.ascontiguousarray(sc))

    def combine(rows, idx, gate, out=None, shared_rows=None, expert_scales=None, expert_rows_dtype=None):
        if expert_scales is not None:   # combine quantisation: DQ_MX of the MXFP8 rows
            tab = np.array([oracle.fp8_value(c, expert_rows_dtype) for c in range(256)])
            sc = np.repeat(expert_scales.numpy().astype(np.float64) - 127.0, 32, axis=1)
            r = (tab[rows.numpy()] * np.exp2(sc)).astype(np.float32)
        else:
            r = rows.float().numpy()
        g = gate.float().numpy()
        n, k = g.shape
        acc = np.zeros((n, rows.shape[1]), np.float32)
        ix = idx.numpy().reshape(n, k)
        for kk in range(k):
            ok = ix[:, kk] >= 0
            acc[ok] += g[ok, kk:kk + 1] * r[ix[ok, kk]]
        if shared_rows is not None:
            for s in range(shared_rows.shape[0]):
                acc += shared_rows[s].float().numpy()
        return torch.from_numpy(acc).to(torch.bfloat16)

    mm.mm_moe_ep_dispatch = dispatch
    mm.mm_mega_moe = mega
    mm.mm_moe_expert_ffn = expert_ffn
    mm.mm_mx_quantize = mx_quantize
    mm.mm_moe_combine = combine


def _slices(cfg, rank):
    per = cfg.n // W
    return slice(rank * per, (rank + 1) * per)


def _cpu_rank(rank, port, out, shared, cq):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import routing_permute_mxfp8_gb300 as mm
    from routing_permute_mxfp8_gb300 import ep
    cfg, x, ids, gate, (w1, s1, w2, s2) = _problem(shared=shared)
    sh = _shared(cfg)
    _oracle_fakes(mm, cfg)
    dist.init_process_group("gloo", rank=rank, world_size=W)
    sl = _slices(cfg, rank)
    el = cfg.e // W
    mine = slice(rank * el, (rank + 1) * el)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    xt = t(x[sl].view(np.int16)).view(torch.bfloat16)
    gt = t(gate[sl].view(np.int16)).view(torch.bfloat16)
    skw = {} if sh is None else dict(shared_weight1=t(sh[0]), shared_weight_scales1=t(sh[1]),
                                     shared_weight2=t(sh[2]), shared_weight_scales2=t(sh[3]))
    y = ep.mega_moe_ep(xt, t(ids[sl]), gt, t(w1[mine]), t(w2[mine]), t(s1[mine]), t(s2[mine]), cfg.e,
                       weight_dtype=cfg.weight_fmt, dispatch_quant_out_dtype=cfg.dispatch_fmt,
                       combine_quant_mode=cq, **skw)
    # the same fakes on one rank, no exchange: every expert local
    sx, ss, se, cnt, ei = mm.mm_moe_ep_dispatch(xt, t(ids[sl]), cfg.e, 1, cfg.dispatch_fmt)
    o = mm.mm_mega_moe(sx, se.view(-1, 1), torch.ones((sx.shape[0], 1)), t(w1), t(w2), t(s1), t(s2), cfg.e,
                       x_scales=ss, dispatch_quant_mode=0, dispatch_quant_out_dtype=cfg.dispatch_fmt)[0]
    shr = None if sh is None else ep._shared_rows(xt, t(sh[0]), t(sh[2]), t(sh[1]), t(sh[3]), cfg.weight_fmt,
                                                 cfg.dispatch_fmt, mm.WSCALE_ROWS, "swiglu", (), None)
    if cq:
        cfmt = {3: 23, 4: 24}[cq]
        oq, os_ = mm.mm_mx_quantize(o, cfmt, scale_cols=cfg.h // 32)
        y1 = mm.mm_moe_combine(oq, ei, gt, shared_rows=shr, expert_scales=os_, expert_rows_dtype=cfmt)
    else:
        y1 = mm.mm_moe_combine(o, ei, gt, shared_rows=shr)
    out[rank] = (y.view(torch.int16).numpy().copy(), y1.view(torch.int16).numpy().copy())
    dist.barrier()
    dist.destroy_process_group()


def _check_against_oracle(cfg, x, ids, gate, w, y_bits, cq=0):
    import oracle
    import synth
    w1, s1, w2, s2 = w
    y_ref, _ = oracle.mega_moe_tokens(x, ids, gate, w1, s1, w2, s2, cfg.dispatch_fmt, cfg.weight_fmt,
                                      shared=_shared(cfg), combine_fmt={0: None, 3: 23, 4: 24}[cq])
    yg = synth.bf16_bits_to_f32(y_bits.view(np.uint16)).astype(np.float64)
    rel = np.linalg.norm(yg - y_ref) / np.linalg.norm(y_ref)
    mx = np.abs(yg - y_ref).max() / np.abs(y_ref).max()
    assert rel <= 5e-3 and mx <= 2e-2, (rel, mx)


@pytest.mark.parametrize("shared,cq", [(0, 0), (1, 0), (1, 4)], ids=["plain", "shared", "shared_combine_e4m3"])
def test_ep_exchange_two_gloo_ranks_cpu(shared, cq):
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork after CUDA is initialised
    mp.spawn(_cpu_rank, args=(port, out, shared, cq), nprocs=W, join=True)
    cfg, x, ids, gate, w = _problem(shared=shared)
    ys = []
    for r in range(W):
        y, y1 = out[r]
        assert np.array_equal(y, y1), r          # exchange changes nothing in the result
        ys.append(y)
    _check_against_oracle(cfg, x, ids, gate, w, np.concatenate(ys), cq)


def _gpu_rank(rank, port, out, a4w4, shared):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import routing_permute_mxfp8_gb300 as mm
    from routing_permute_mxfp8_gb300 import ep
    torch.cuda.set_device(0)
    cfg, x, ids, gate, (w1, s1, w2, s2) = _problem(a4w4, shared)
    sh = _shared(cfg)
    if cfg.weight_fmt == 296:
        w1, w2 = _pack_fp4(w1), _pack_fp4(w2)
        if sh is not None:
            sh = (_pack_fp4(sh[0]), sh[1], _pack_fp4(sh[2]), sh[3])
    dist.init_process_group("gloo", rank=rank, world_size=W)
    sl = _slices(cfg, rank)
    el = cfg.e // W
    mine = slice(rank * el, (rank + 1) * el)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    xt = t(x[sl].view(np.int16)).view(torch.bfloat16)
    gt = t(gate[sl].view(np.int16)).view(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    skw = {} if sh is None else dict(shared_weight1=t(sh[0]), shared_weight_scales1=t(sh[1]),
                                     shared_weight2=t(sh[2]), shared_weight_scales2=t(sh[3]))
    y = ep.mega_moe_ep(xt, t(ids[sl]), gt, t(w1[mine]), t(w2[mine]), t(s1[mine]), t(s2[mine]), cfg.e,
                       weight_dtype=cfg.weight_fmt, dispatch_quant_out_dtype=cfg.dispatch_fmt, dev_err=err, **skw)
    # single process, all experts on this GPU (ep_world_size = 1)
    y1 = mm.mm_mega_moe(xt, t(ids[sl]), gt, t(w1), t(w2), t(s1), t(s2), cfg.e, weight_dtype=cfg.weight_fmt,
                        dispatch_quant_out_dtype=cfg.dispatch_fmt, **skw)[0]
    torch.cuda.synchronize()
    out[rank] = (y.view(torch.int16).cpu().numpy(), y1.view(torch.int16).cpu().numpy(), int(err.item()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.gpu
@pytest.mark.parametrize("a4w4,shared", [(False, 0), (True, 0), (False, 2), (True, 1)],
                         ids=["a8w8", "a4w4", "a8w8_shared2", "a4w4_shared1"])
def test_ep_two_ranks_on_one_gpu_matches_single_process(a4w4, shared):
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork after CUDA is initialised
    mp.spawn(_gpu_rank, args=(port, out, a4w4, shared), nprocs=W, join=True)
    cfg, x, ids, gate, w = _problem(a4w4, shared)
    ys = []
    for r in range(W):
        y, y1, err = out[r]
        assert err == 0
        assert np.array_equal(y, y1), r
        ys.append(y)
    _check_against_oracle(cfg, x, ids, gate, w, np.concatenate(ys))


def _gpu_rank_combine_quant(rank, port, out, cq):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import routing_permute_mxfp8_gb300 as mm
    from routing_permute_mxfp8_gb300 import ep
    torch.cuda.set_device(0)
    cfg, x, ids, gate, (w1, s1, w2, s2) = _problem(shared=1)
    sh = _shared(cfg)
    dist.init_process_group("gloo", rank=rank, world_size=W)
    sl = _slices(cfg, rank)
    el = cfg.e // W
    mine = slice(rank * el, (rank + 1) * el)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    xt = t(x[sl].view(np.int16)).view(torch.bfloat16)
    gt = t(gate[sl].view(np.int16)).view(torch.bfloat16)
    skw = dict(shared_weight1=t(sh[0]), shared_weight_scales1=t(sh[1]), shared_weight2=t(sh[2]),
               shared_weight_scales2=t(sh[3]))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = ep.mega_moe_ep(xt, t(ids[sl]), gt, t(w1[mine]), t(w2[mine]), t(s1[mine]), t(s2[mine]), cfg.e,
                       weight_dtype=cfg.weight_fmt, dispatch_quant_out_dtype=cfg.dispatch_fmt, dev_err=err,
                       combine_quant_mode=cq, **skw)
    # the same kernels on this rank alone, no exchange: every expert local
    cfmt = {3: 23, 4: 24}[cq]
    sx, ss, se, cnt, ei = mm.mm_moe_ep_dispatch(xt, t(ids[sl]), cfg.e, 1, cfg.dispatch_fmt)
    o = mm.mm_moe_expert_ffn(sx, ss, se, t(w1), t(w2), t(s1), t(s2), cfg.e, x_dtype=cfg.dispatch_fmt,
                             weight_dtype=cfg.weight_fmt)[0]
    oq, os_ = mm.mm_mx_quantize(o, cfmt, scale_cols=cfg.h // 32)
    shr = ep._shared_rows(xt, t(sh[0]), t(sh[2]), t(sh[1]), t(sh[3]), cfg.weight_fmt, cfg.dispatch_fmt,
                          mm.WSCALE_ROWS, "swiglu", (), None)
    y1 = mm.mm_moe_combine(oq, ei, gt, shared_rows=shr, expert_scales=os_, expert_rows_dtype=cfmt)
    torch.cuda.synchronize()
    out[rank] = (y.view(torch.int16).cpu().numpy(), y1.view(torch.int16).cpu().numpy(), int(err.item()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.gpu
@pytest.mark.parametrize("cq", [3, 4])
def test_ep_combine_quantisation_two_ranks_on_one_gpu(cq):
    """combineQuantMode 3 / 4: the returned rows travel as MXFP8 codes and
    scales; two ranks give the bits of the same kernels on one rank without
    the exchange, and the oracle's combine-quantised Y within tolerance."""
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork after CUDA is initialised
    mp.spawn(_gpu_rank_combine_quant, args=(port, out, cq), nprocs=W, join=True)
    cfg, x, ids, gate, w = _problem(shared=1)
    ys = []
    for r in range(W):
        y, y1, err = out[r]
        assert err == 0
        assert np.array_equal(y, y1), r
        ys.append(y)
    _check_against_oracle(cfg, x, ids, gate, w, np.concatenate(ys), cq)
