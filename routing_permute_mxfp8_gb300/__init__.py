"""GB300 (sm_103a) MoE routing, token permute with MX quantisation and the
MXFP8 expert FFN (MegaMoE at ep_world_size = 1).

This module only marshals arguments: it allocates outputs and workspaces as
torch tensors and calls the C ABI of ``libmm_moe.so`` (declared in
``include/mm_moe.h``) on the current CUDA stream.  Every step runs in the
library's CUDA kernels; there is no other implementation to fall back on,
and every entry point raises if the library is not built or a call fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MMError", "lib_path", "load", "mm_version", "mm_moe_init_routing", "mm_moe_token_permute",
    "mm_mega_moe", "mm_mega_moe_workspace_size", "mm_prepare_weight_scales", "mm_mx_quantize",
    "DT_FP8_E5M2", "DT_FP8_E4M3FN", "QUANT_NONE", "QUANT_MXFP8_E5M2", "QUANT_MXFP8_E4M3FN",
    "mm_moe_ep_dispatch", "mm_moe_combine", "mm_moe_expert_ffn",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATHS = {False: os.path.join(_HERE, "libmm_moe.so"), True: os.path.join(_HERE, "libmm_moe_check.so")}
_libs = {}
# the checked build (device index checks, MM_DEVERR_BOUNDS) instead of the
# normal one: use_checked_library(True), or MM_MOE_CHECKED=1 in the environment
_checked = os.environ.get("MM_MOE_CHECKED", "0") == "1"

DT_F32, DT_F16, DT_I32, DT_I64, DT_BF16 = 0, 1, 3, 9, 27
DT_FP8_E5M2, DT_FP8_E4M3FN = 23, 24
DT_FP4_E2M1 = 296   # packed two codes per byte, element 2i in bits 0-3
QUANT_NONE, QUANT_MXFP8_E5M2, QUANT_MXFP8_E4M3FN = -1, 2, 3
QUANT_MXFP4_E2M1 = 9   # moe_token_permute: packed [M, H/2] codes, scales [M, CeilDiv(H, 64), 2]
WSCALE_ROWS, WSCALE_PREPARED = 0, 1

_TORCH_DT = {torch.float32: DT_F32, torch.float16: DT_F16, torch.bfloat16: DT_BF16,
             torch.int32: DT_I32, torch.int64: DT_I64,
             torch.float8_e5m2: DT_FP8_E5M2, torch.float8_e4m3fn: DT_FP8_E4M3FN}
_FP8_TORCH = {DT_FP8_E5M2: torch.float8_e5m2, DT_FP8_E4M3FN: torch.float8_e4m3fn}
_QUANT_FMT = {QUANT_MXFP8_E5M2: DT_FP8_E5M2, QUANT_MXFP8_E4M3FN: DT_FP8_E4M3FN}


class MMError(RuntimeError):
    pass


def lib_path() -> str:
    return _LIB_PATHS[_checked]


def use_checked_library(on: bool = True):
    """Route the following calls to libmm_moe_check.so (the checked build,
    whose kernels report MM_DEVERR_BOUNDS for an index outside its buffer)
    or back to libmm_moe.so.  Each library keeps its own host-side state
    (timing, routing path, no-allocation scratch)."""
    global _checked
    _checked = bool(on)


def load():
    """Load the selected library (libmm_moe.so, or libmm_moe_check.so after
    use_checked_library(True)); raises if it has not been built."""
    path = _LIB_PATHS[_checked]
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise MMError(f"{path} is missing: build it with `python -m routing_permute_mxfp8_gb300.build`")
    L = ctypes.CDLL(path)
    p, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    psz = ctypes.POINTER(ctypes.c_size_t)
    L.mm_status_string.argtypes, L.mm_status_string.restype = [i32], ctypes.c_char_p
    L.mm_version.restype = i32
    L.mm_moe_init_routing_workspace_size.argtypes = [i64, i64, i64, psz]
    L.mm_moe_init_routing.argtypes = [p, i32, p, i64, i64, i64, i64, i32, i32, p, p, p, p, p, p, sz, p, p]
    L.mm_moe_init_routing_v3_workspace_size.argtypes = [i64, i64, i64, psz]
    L.mm_moe_init_routing_v3.argtypes = [p, i32, p, i64, i64, i64, i64, i64, i64, i32, i32, p, p, p, p, p, p, sz,
                                         p, p]
    L.mm_moe_token_permute_out_rows.argtypes, L.mm_moe_token_permute_out_rows.restype = [i64, i64], i64
    L.mm_moe_token_permute_workspace_size.argtypes = [i64, i64, psz]
    L.mm_moe_token_permute.argtypes = [p, i32, p, i32, i64, i64, i64, i64, i64, i32, i32, p, p, p, p, sz, p, p]
    L.mm_mega_moe_workspace_size.argtypes = [i64, i64, i64, i64, i64, i64, i32, psz]
    L.mm_mega_moe.argtypes = ([p, p, p, p, i32, p, p, p, p, i32, i32, p, p, p, p, i32, i64, i64, i64, i64, i64, i64,
                               i64, i64, i64, i64, i64, i64, ctypes.c_char_p, p, i64, p, p, p, p, p, p, p, p, sz, p,
                               p])
    L.mm_prepared_weight_scales_size.argtypes = [i32, i64, i64, i64, psz]
    L.mm_prepare_weight_scales.argtypes = [p, i32, i64, i64, i64, p, p]
    L.mm_mx_quantize.argtypes = [p, i32, i64, i64, i32, p, p, i64, p]
    L.mm_selftest_wait_timeout.argtypes = [i64, p, p]
    L.mm_moe_ep_dispatch_workspace_size.argtypes = [i64, i64, i64, psz]
    L.mm_moe_expert_ffn_workspace_size.argtypes = [i64, i64, i64, i64, i32, psz]
    L.mm_moe_expert_ffn.argtypes = [p, p, i32, p, i64, i64, p, p, p, p, i32, i32, i64, i64, ctypes.c_char_p, p, i64,
                                    p, p, p, sz, p, p]
    L.mm_moe_ep_dispatch.argtypes = [p, i32, p, i64, i64, i64, i64, i64, i64, p, p, p, p, p, p, sz, p, p]
    L.mm_moe_combine.argtypes = [p, i32, p, p, p, i32, i64, i64, i64, p, i64, p, p]
    for name in ("mm_moe_init_routing_workspace_size", "mm_moe_init_routing", "mm_moe_token_permute_workspace_size",
                 "mm_moe_token_permute", "mm_mega_moe_workspace_size", "mm_mega_moe",
                 "mm_prepared_weight_scales_size", "mm_prepare_weight_scales", "mm_mx_quantize",
                 "mm_selftest_wait_timeout", "mm_moe_ep_dispatch_workspace_size", "mm_moe_ep_dispatch",
                 "mm_moe_combine", "mm_moe_expert_ffn_workspace_size", "mm_moe_expert_ffn"):
        getattr(L, name).restype = i32
    _libs[path] = L
    return L


def mm_version() -> int:
    return int(load().mm_version())


def _check(status: int, what: str):
    if status != 0:
        msg = load().mm_status_string(status).decode()
        raise MMError(f"{what}: {msg} (status {status})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dt(t) -> int:
    if t.dtype not in _TORCH_DT:
        raise MMError(f"unsupported dtype {t.dtype}")
    return _TORCH_DT[t.dtype]


def _scale_cols(h: int) -> int:
    return ((h + 31) // 32 + 1) // 2 * 2


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise MMError("inputs must be contiguous CUDA tensors")


_SRC_DTYPES = (torch.bfloat16, torch.float16, torch.float32)
_BYTE_DTYPES = (torch.uint8, torch.float8_e4m3fn, torch.float8_e5m2)


def _need_dtype(t, allowed, what):
    """The C ABI reads raw memory: a tensor of another dtype would be
    reinterpreted silently (an int64 index tensor read as pairs of int32
    words), so it is refused here."""
    if t is not None and t.dtype not in allowed:
        names = " or ".join(str(d).replace("torch.", "") for d in allowed)
        raise MMError(f"{what} must be {names}, got {str(t.dtype).replace('torch.', '')}")


def _need(cond, msg):
    """Shapes the C ABI cannot see: it takes sizes and raw pointers, so a
    tensor smaller than the sizes it is passed with would be read or written
    past its end on the GPU.  Mismatches are refused here."""
    if not cond:
        raise MMError(msg)


def _need_rows_of(idx, n, what, of):
    _need(idx.dim() in (1, 2) and idx.shape[0] == n, f"{what} must be [N] or [N, K] with N = {of}.shape[0] = {n}")


def _need_out(out, shape, what="out"):
    if out is not None:
        _need(out.dtype == torch.bfloat16 and tuple(out.shape) == tuple(shape),
              f"{what} must be a bfloat16 tensor of shape {list(shape)}")


def _need_weights(w1, w2, s1, s2, e, h, aw, fp4, what=""):
    """Expert weights [E, 2I, H] and [E, H, A] (A = I, or 2I under gelu; packed
    FP4 halves the last dimension), and E8M0 scales holding at least one byte
    per 32 reduction elements of every output row (the pages' layout or a
    prepared buffer)."""
    pk = 2 if fp4 else 1
    _need(w1.dim() == 3 and w1.shape[0] == e and w1.shape[2] * pk == h,
          f"{what}weight1 must be [{e}, 2I, {h // pk}], got {list(w1.shape)}")
    _need(w2.dim() == 3 and w2.shape[0] == e and w2.shape[1] == h and w2.shape[2] * pk == aw,
          f"{what}weight2 must be [{e}, {h}, {aw // pk}], got {list(w2.shape)}")
    _need(s1.numel() >= e * w1.shape[1] * (h // 32),
          f"{what}weight_scales1 holds {s1.numel()} bytes, {e * w1.shape[1] * (h // 32)} needed")
    _need(s2.numel() >= e * h * (aw // 32), f"{what}weight_scales2 holds {s2.numel()} bytes, {e * h * (aw // 32)} needed")


def _workspace(nbytes: int, device, workspace):
    if workspace is not None:
        if workspace.numel() < nbytes:
            raise MMError(f"workspace holds {workspace.numel()} bytes, {nbytes} needed")
        return workspace
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


def _dev_err(dev_err):
    return None if dev_err is None else _ptr(dev_err)


# --------------------------------------------------------------------------- routing / permute
def mm_moe_init_routing(x, expert_idx, expert_num: int, quant_mode: int = QUANT_NONE,
                        expert_tokens_num_type: int = 1, *, active_expert_range=None, workspace=None,
                        dev_err=None):
    """MoeInitRoutingV3 (Dropless).

    Returns (expanded_x [N*K, H], expanded_row_idx [N*K] int32 (scatter),
    expert_tokens (count or cumsum [E'] int64, or key_value [E, 2] int64 with
    expert_tokens_num_type 2), expanded_scale [N*K, AlignUp(H/32, 2)] uint8 E8M0
    (empty without quantisation), sorted_row_idx [N*K] int32 (gather)).
    active_expert_range = (start, end): only ids in [start, end) are routed
    (E' = end - start; the first availableIdxNum rows of the outputs are valid);
    None: the full range (mm_moe_init_routing), else mm_moe_init_routing_v3.
    """
    _need_dtype(x, _SRC_DTYPES, "x")
    _need_dtype(expert_idx, (torch.int32,), "expert_idx")
    _need(x.dim() == 2, "x must be [N, H]")
    _need_rows_of(expert_idx, x.shape[0], "expert_idx", "x")
    _need_cuda(x, expert_idx)
    L = load()
    n, h = x.shape
    k = expert_idx.shape[1] if expert_idx.dim() == 2 else 1
    rows = n * k
    dev = x.device
    out_dt = x.dtype if quant_mode == QUANT_NONE else _FP8_TORCH.get(_QUANT_FMT.get(quant_mode), torch.uint8)
    expanded_x = torch.empty((rows, h // 2 if quant_mode == QUANT_MXFP4_E2M1 else h), dtype=out_dt, device=dev)
    scale = (torch.empty((rows, _scale_cols(h)), dtype=torch.uint8, device=dev) if quant_mode != QUANT_NONE
             else torch.empty((0,), dtype=torch.uint8, device=dev))
    exp_idx = torch.empty(rows, dtype=torch.int32, device=dev)
    srt_idx = torch.empty(rows, dtype=torch.int32, device=dev)
    v3 = active_expert_range is not None or expert_tokens_num_type == 2
    start, end = (0, expert_num) if active_expert_range is None else (int(active_expert_range[0]),
                                                                      int(active_expert_range[1]))
    tokens = (torch.empty((expert_num, 2), dtype=torch.int64, device=dev) if expert_tokens_num_type == 2
              else torch.empty(max(end - start, 0), dtype=torch.int64, device=dev))
    need = ctypes.c_size_t(0)
    if v3:
        _check(L.mm_moe_init_routing_v3_workspace_size(n, k, expert_num, ctypes.byref(need)), "mm_moe_init_routing_v3")
    else:
        _check(L.mm_moe_init_routing_workspace_size(n, k, expert_num, ctypes.byref(need)), "mm_moe_init_routing")
    ws = _workspace(need.value, dev, workspace)
    sc = _ptr(scale) if scale.numel() else None
    if v3:
        _check(L.mm_moe_init_routing_v3(_ptr(x), _dt(x), _ptr(expert_idx), n, h, k, expert_num, start, end,
                                        quant_mode, expert_tokens_num_type, _ptr(expanded_x), sc, _ptr(exp_idx),
                                        _ptr(srt_idx), _ptr(tokens), _ptr(ws), ws.numel(), _dev_err(dev_err),
                                        _stream(dev)), "mm_moe_init_routing_v3")
    else:
        _check(L.mm_moe_init_routing(_ptr(x), _dt(x), _ptr(expert_idx), n, h, k, expert_num, quant_mode,
                                     expert_tokens_num_type, _ptr(expanded_x), sc, _ptr(exp_idx), _ptr(srt_idx),
                                     _ptr(tokens), _ptr(ws), ws.numel(), _dev_err(dev_err), _stream(dev)),
               "mm_moe_init_routing")
    return expanded_x, exp_idx, tokens, scale, srt_idx


def mm_moe_token_permute(tokens, indices, num_experts: int, num_out_tokens=None, padded_mode: bool = False,
                         quant_mode: int = QUANT_NONE, *, workspace=None, dev_err=None):
    """moe_token_permute: returns (permuted_tokens [M, H], sorted_indices [F] int32,
    expanded_scale [M, AlignUp(H/32, 2)] uint8 E8M0 or an empty tensor).  With
    QUANT_MXFP4_E2M1: permuted_tokens [M, H/2] packed uint8, expanded_scale
    [M, CeilDiv(H, 64), 2]."""
    _need_dtype(tokens, _SRC_DTYPES, "tokens")
    _need_dtype(indices, (torch.int32, torch.int64), "indices")
    _need(tokens.dim() == 2, "tokens must be [N, H]")
    _need_rows_of(indices, tokens.shape[0], "indices", "tokens")
    _need_cuda(tokens, indices)
    L = load()
    n, h = tokens.shape
    topk = indices.shape[1] if indices.dim() == 2 else 1
    f = indices.numel()
    nout = 0 if num_out_tokens is None else int(num_out_tokens)
    m = int(L.mm_moe_token_permute_out_rows(f, nout))
    dev = tokens.device
    out_dt = tokens.dtype if quant_mode == QUANT_NONE else _FP8_TORCH.get(_QUANT_FMT.get(quant_mode), torch.uint8)
    permuted = torch.empty((m, h // 2 if quant_mode == QUANT_MXFP4_E2M1 else h), dtype=out_dt, device=dev)
    scale = (torch.empty((m, _scale_cols(h)), dtype=torch.uint8, device=dev) if quant_mode != QUANT_NONE
             else torch.empty((0,), dtype=torch.float32, device=dev))
    if quant_mode == QUANT_MXFP4_E2M1:
        scale = scale.view(m, (h + 63) // 64, 2)
    sorted_indices = torch.empty(f, dtype=torch.int32, device=dev)
    need = ctypes.c_size_t(0)
    _check(L.mm_moe_token_permute_workspace_size(f, num_experts, ctypes.byref(need)), "mm_moe_token_permute")
    ws = _workspace(need.value, dev, workspace)
    _check(L.mm_moe_token_permute(_ptr(tokens), _dt(tokens), _ptr(indices), _dt(indices), n, topk, h, num_experts,
                                  nout, int(bool(padded_mode)), quant_mode,
                                  _ptr(permuted) if m else None,
                                  _ptr(scale) if (quant_mode != QUANT_NONE and m) else None,
                                  _ptr(sorted_indices), _ptr(ws), ws.numel(), _dev_err(dev_err), _stream(dev)),
           "mm_moe_token_permute")
    return permuted, sorted_indices, scale


# --------------------------------------------------------------------------- MegaMoE
def mm_mega_moe_workspace_size(bs, h, k, moe_expert_num, intermediate, shared_expert_num=0,
                               weight_scale_layout=WSCALE_ROWS) -> int:
    need = ctypes.c_size_t(0)
    _check(load().mm_mega_moe_workspace_size(bs, h, k, moe_expert_num, intermediate, shared_expert_num,
                                             weight_scale_layout, ctypes.byref(need)), "mm_mega_moe_workspace_size")
    return need.value


def _fp8_code(t, default):
    if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return _TORCH_DT[t.dtype]
    return default


def mm_mega_moe(x, topk_ids, topk_weights, weight1, weight2, weight_scales1, weight_scales2, moe_expert_num: int, *,
                weight_dtype: int = DT_FP8_E4M3FN, weight_scale_layout: int = WSCALE_ROWS,
                shared_weight1=None, shared_weight2=None, shared_weight_scales1=None, shared_weight_scales2=None,
                shared_weight_dtype: int | None = None, ep_world_size: int = 1, max_recv_token_num: int = 0,
                dispatch_quant_mode: int = 4, dispatch_quant_out_dtype: int = DT_FP8_E4M3FN,
                shared_expert_quant_out_dtype: int | None = None,
                combine_quant_mode: int = 0, activation: str = "swiglu", activation_params=(),
                x_scales=None, out=None, workspace=None, dev_err=None, want_expanded_row_idx=False,
                want_act=False, want_dispatch=False):
    """MegaMoE forward, A8W8-FP, A8W4-FP or A4W4-FP, ep_world_size = 1.

    x [BS, H] bf16; topk_ids [BS, K] int32; topk_weights [BS, K] fp32 / bf16;
    weight1 [E, 2I, H] and weight2 [E, H, I] FP8 (torch float8 or uint8 with
    weight_dtype), or with weight_dtype=DT_FP4_E2M1 packed FP4 bytes
    [E, 2I, H/2] and [E, H, I/2]; weight_scales1 / 2 uint8 E8M0 in the pages' layout
    (weight_scale_layout=0) or prepared by mm_prepare_weight_scales (1).  Under
    activation="gelu", weight2 is [E, H, 2I] and A_hat 2I wide.
    Returns (y [BS, H] bf16, expert_token_nums [E] int32) and, on request,
    expanded_row_idx [BS*K] int32, A_hat codes / scales and the dispatched
    X_hat codes [BS*K, H] / scales [BS*K, H/32], in sorted order.
    With dispatch_quant_mode=0, x holds FP8 codes (uint8 [BS, H]) and x_scales their
    E8M0 scales [BS, H/32] (pre-quantised pass-through).
    A4W4-FP: dispatch_quant_out_dtype=DT_FP4_E2M1 with FP4 weights; the dispatched
    X_hat is packed FP4 ([BS*K, H/2] when returned; x [BS, H/2] in pass-through) and
    A_hat is MXFP8 E4M3.  shared_expert_quant_out_dtype: the shared experts' own input
    type (sharedExpertQuantOutDtype; None: the dispatch type).
    """
    _need_dtype(x, (torch.bfloat16,) if dispatch_quant_mode != 0 else _BYTE_DTYPES, "x")
    _need_dtype(topk_ids, (torch.int32,), "topk_ids")
    _need_dtype(topk_weights, (torch.float32, torch.bfloat16), "topk_weights")
    for name, t in (("weight1", weight1), ("weight2", weight2), ("shared_weight1", shared_weight1),
                    ("shared_weight2", shared_weight2)):
        _need_dtype(t, _BYTE_DTYPES, name)
    for name, t in (("weight_scales1", weight_scales1), ("weight_scales2", weight_scales2), ("x_scales", x_scales),
                    ("shared_weight_scales1", shared_weight_scales1),
                    ("shared_weight_scales2", shared_weight_scales2)):
        _need_dtype(t, (torch.uint8,), name)
    if topk_ids.dim() != 2 or tuple(topk_weights.shape) != tuple(topk_ids.shape) or topk_ids.shape[0] != x.shape[0]:
        raise MMError("topk_ids and topk_weights must both be [BS, K] with BS = x.shape[0]")
    _need(x.dim() == 2, "x must be [BS, H]")
    fp4_x = dispatch_quant_out_dtype == DT_FP4_E2M1
    bs = x.shape[0]
    h = x.shape[1] * 2 if fp4_x and dispatch_quant_mode == 0 else x.shape[1]   # packed FP4 pass-through
    k = topk_ids.shape[1]
    wdt = _fp8_code(weight1, weight_dtype)
    _need(weight1.dim() == 3, "weight1 must be [E, 2I, H]")
    inter = weight1.shape[1] // 2
    aw = 2 * inter if activation == "gelu" else inter   # width of A_hat
    _need_weights(weight1, weight2, weight_scales1, weight_scales2, moe_expert_num, h, aw, wdt == DT_FP4_E2M1)
    shared = (shared_weight1, shared_weight2, shared_weight_scales1, shared_weight_scales2)
    s_num = 0 if shared_weight1 is None else shared_weight1.shape[0]
    swdt = wdt if shared_weight1 is None else _fp8_code(shared_weight1, wdt if shared_weight_dtype is None
                                                         else shared_weight_dtype)
    if s_num > 0:
        _need(all(t is not None for t in shared), "shared experts need all four of shared_weight1 / 2 and their scales")
        _need(shared_weight1.dim() == 3 and shared_weight1.shape[1] == weight1.shape[1],
              "shared_weight1 must be [S, 2I, H] with the routed experts' 2I")
        _need_weights(*shared, s_num, h, aw, swdt == DT_FP4_E2M1, what="shared_")
    if x_scales is not None:
        _need(x_scales.numel() >= bs * (h // 32), f"x_scales must be [BS, H/32] = [{bs}, {h // 32}]")
    _need_out(out, (bs, h))
    _need_cuda(x, topk_ids, topk_weights, weight1, weight2, weight_scales1, weight_scales2)
    L = load()
    dev = x.device
    y = out if out is not None else torch.empty((bs, h), dtype=torch.bfloat16, device=dev)
    counts = torch.empty(moe_expert_num, dtype=torch.int32, device=dev)
    exp_idx = torch.empty(bs * k, dtype=torch.int32, device=dev) if want_expanded_row_idx else None
    act_q = torch.empty((bs * k, aw), dtype=torch.uint8, device=dev) if want_act else None
    act_s = torch.empty((bs * k, aw // 32), dtype=torch.uint8, device=dev) if want_act else None
    dsp_q = torch.empty((bs * k, h // 2 if fp4_x else h), dtype=torch.uint8, device=dev) if want_dispatch else None
    dsp_s = torch.empty((bs * k, h // 32), dtype=torch.uint8, device=dev) if want_dispatch else None
    need = mm_mega_moe_workspace_size(bs, h, k, moe_expert_num, inter, s_num, weight_scale_layout)
    ws = _workspace(need, dev, workspace)
    params = list(activation_params)
    parr = (ctypes.c_float * max(len(params), 1))(*params) if params else None
    gdt = _dt(topk_weights)
    _check(L.mm_mega_moe(
        _ptr(x), _ptr(x_scales), _ptr(topk_ids), _ptr(topk_weights), gdt, _ptr(weight1), _ptr(weight2), _ptr(weight_scales1),
        _ptr(weight_scales2), wdt, weight_scale_layout, _ptr(shared_weight1), _ptr(shared_weight2),
        _ptr(shared_weight_scales1), _ptr(shared_weight_scales2), swdt, s_num, bs, h, k, moe_expert_num,
        ep_world_size, inter, max_recv_token_num, dispatch_quant_mode, dispatch_quant_out_dtype,
        shared_expert_quant_out_dtype or 0, combine_quant_mode, activation.encode() if activation else None, parr,
        len(params), _ptr(y), _ptr(counts),
        _ptr(exp_idx), _ptr(act_q), _ptr(act_s), _ptr(dsp_q), _ptr(dsp_s), _ptr(ws), ws.numel(), _dev_err(dev_err),
        _stream(dev)),
        "mm_mega_moe")
    res = [y, counts]
    if want_expanded_row_idx:
        res.append(exp_idx)
    if want_act:
        res += [act_q, act_s]
    if want_dispatch:
        res += [dsp_q, dsp_s]
    return tuple(res)


def mm_prepare_weight_scales(scales, k_red: int, which: int):
    """Rearrange E8M0 weight scales [E, N_out, CeilDiv(K_red, 64), 2] (or [E, N_out, K_red/32])
    into the tile layout of the grouped GEMMs (weight_scale_layout = 1).
    which = 1 for weight_scales1, 2 for weight_scales2."""
    _need_dtype(scales, (torch.uint8,), "scales")
    _need_cuda(scales)
    L = load()
    e, n_out = scales.shape[0], scales.shape[1]
    need = ctypes.c_size_t(0)
    _check(L.mm_prepared_weight_scales_size(which, e, n_out, k_red, ctypes.byref(need)), "mm_prepare_weight_scales")
    dst = torch.empty(need.value, dtype=torch.uint8, device=scales.device)
    _check(L.mm_prepare_weight_scales(_ptr(scales), which, e, n_out, k_red, _ptr(dst), _stream(scales.device)),
           "mm_prepare_weight_scales")
    return dst


def mm_selftest_wait_timeout(limit_ns: int, dev_err):
    """One CTA waits, with a limit of limit_ns, on an mbarrier that nothing
    completes (the kernels' bounded-wait failure path): MM_DEVERR_TIMEOUT is
    OR-ed into dev_err (a device int32 tensor) and the context stays usable."""
    _need_cuda(dev_err)
    _check(load().mm_selftest_wait_timeout(int(limit_ns), _ptr(dev_err), _stream(dev_err.device)),
           "mm_selftest_wait_timeout")


def mm_mx_quantize(src, out_dtype: int = DT_FP8_E4M3FN, scale_cols: int | None = None):
    """Q_MX along the last dimension of a 2-D fp32 / bf16 / fp16 tensor.
    Returns (codes [rows, cols] uint8 -- [rows, cols / 2] packed for DT_FP4_E2M1 --,
    scales [rows, scale_cols] uint8 E8M0)."""
    _need_dtype(src, _SRC_DTYPES, "src")
    _need_cuda(src)
    L = load()
    rows, cols = src.shape
    sc = _scale_cols(cols) if scale_cols is None else scale_cols
    q = torch.empty((rows, cols // 2 if out_dtype == DT_FP4_E2M1 else cols), dtype=torch.uint8, device=src.device)
    s = torch.empty((rows, sc), dtype=torch.uint8, device=src.device)
    _check(L.mm_mx_quantize(_ptr(src), _dt(src), rows, cols, out_dtype, _ptr(q), _ptr(s), sc,
                            _stream(src.device)), "mm_mx_quantize")
    return q, s


# --------------------------------------------------------------------------- expert parallelism
def mm_moe_ep_dispatch(x, topk_ids, moe_expert_num: int, ep_world_size: int,
                       dispatch_quant_out_dtype: int = DT_FP8_E4M3FN, *, workspace=None, dev_err=None):
    """Source side of the expert-parallel dispatch (MegaMoE stage 1 with
    epWorldSize > 1): rows j = i*K + k sorted stably by destination rank
    id // (E / W), each token MX-quantised once.  Returns (send_x [N*K, H] uint8
    FP8 codes ([N*K, H/2] packed for DT_FP4_E2M1), send_scales [N*K, H/32] uint8 E8M0,
    send_expert [N*K] int32 local
    expert on the destination rank, rank_counts [W] int64, expanded_row_idx
    [N*K] int32 position of row j in the send order)."""
    _need_dtype(x, (torch.bfloat16, torch.float16), "x")
    _need_dtype(topk_ids, (torch.int32,), "topk_ids")
    _need(x.dim() == 2 and topk_ids.dim() == 2 and topk_ids.shape[0] == x.shape[0],
          "x must be [N, H] and topk_ids [N, K]")
    _need_cuda(x, topk_ids)
    L = load()
    n, h = x.shape
    k = topk_ids.shape[1]
    rows = n * k
    dev = x.device
    send_x = torch.empty((rows, h // 2 if dispatch_quant_out_dtype == DT_FP4_E2M1 else h), dtype=torch.uint8,
                         device=dev)
    send_s = torch.empty((rows, h // 32), dtype=torch.uint8, device=dev)
    send_e = torch.empty(rows, dtype=torch.int32, device=dev)
    counts = torch.empty(ep_world_size, dtype=torch.int64, device=dev)
    exp_idx = torch.empty(rows, dtype=torch.int32, device=dev)
    need = ctypes.c_size_t(0)
    _check(L.mm_moe_ep_dispatch_workspace_size(n, k, ep_world_size, ctypes.byref(need)), "mm_moe_ep_dispatch")
    ws = _workspace(need.value, dev, workspace)
    _check(L.mm_moe_ep_dispatch(_ptr(x), _dt(x), _ptr(topk_ids), n, h, k, moe_expert_num, ep_world_size,
                                dispatch_quant_out_dtype, _ptr(send_x), _ptr(send_s), _ptr(send_e), _ptr(counts),
                                _ptr(exp_idx), _ptr(ws), ws.numel(), _dev_err(dev_err), _stream(dev)),
           "mm_moe_ep_dispatch")
    return send_x, send_s, send_e, counts, exp_idx


def mm_moe_combine(expert_rows, row_idx, topk_weights, out=None, shared_rows=None, expert_scales=None,
                   expert_rows_dtype=None):
    """Y[i] = sum_k W[i,k] * expert_rows[row_idx[i*K + k]] + sum_s shared_rows[s, i] in
    fp32, k in order then s, one bf16 rounding (MegaMoE stage 4); row_idx < 0 leaves
    a term out.  expert_rows [*, H] bf16, or MXFP8 codes (uint8 / torch float8, type
    expert_rows_dtype) with expert_scales [*, H/32] E8M0 (combineQuantMode 3 / 4);
    row_idx [N*K] int32, topk_weights [N, K] fp32 / bf16, shared_rows [S, N, H] bf16
    or None."""
    quant = expert_scales is not None
    _need_dtype(expert_rows, _BYTE_DTYPES if quant else (torch.bfloat16,), "expert_rows")
    if quant:
        _need_dtype(expert_scales, (torch.uint8,), "expert_scales")
    rdt = _fp8_code(expert_rows, expert_rows_dtype) if quant else DT_BF16
    _need_dtype(row_idx, (torch.int32,), "row_idx")
    _need_dtype(topk_weights, (torch.float32, torch.bfloat16), "topk_weights")
    _need(expert_rows.dim() == 2 and topk_weights.dim() == 2, "expert_rows must be [*, H] and topk_weights [N, K]")
    n, k = topk_weights.shape
    h = expert_rows.shape[1]
    if row_idx.numel() != n * k:
        raise MMError("row_idx must hold N*K entries")
    if quant:
        _need(tuple(expert_scales.shape) == (expert_rows.shape[0], h // 32),
              f"expert_scales must be [{expert_rows.shape[0]}, {h // 32}] (one E8M0 byte per 32 codes of each row)")
    _need_out(out, (n, h))
    s_num = 0
    if shared_rows is not None:
        _need_dtype(shared_rows, (torch.bfloat16,), "shared_rows")
        if shared_rows.dim() != 3 or tuple(shared_rows.shape[1:]) != (n, h):
            raise MMError("shared_rows must be [S, N, H]")
        s_num = shared_rows.shape[0]
    _need_cuda(expert_rows, row_idx, topk_weights, expert_scales, out, shared_rows)
    y = out if out is not None else torch.empty((n, h), dtype=torch.bfloat16, device=expert_rows.device)
    _check(load().mm_moe_combine(_ptr(expert_rows), rdt, _ptr(expert_scales), _ptr(row_idx), _ptr(topk_weights),
                                 _dt(topk_weights), n, h, k, _ptr(shared_rows), s_num, _ptr(y),
                                 _stream(expert_rows.device)), "mm_moe_combine")
    return y


def mm_moe_expert_ffn(x, x_scales, expert_ids, weight1, weight2, weight_scales1, weight_scales2, local_experts: int, *,
                      x_dtype: int = DT_FP8_E4M3FN, weight_dtype: int = DT_FP8_E4M3FN,
                      weight_scale_layout: int = WSCALE_ROWS, activation: str = "swiglu", activation_params=(),
                      out=None, workspace=None, dev_err=None):
    """The expert side of expert parallelism (MegaMoE stages 2-3 on the rows a
    rank receives): out[r] = the FFN of local expert expert_ids[r] on row r.
    x [M, H] FP8 codes (uint8 or torch float8, type x_dtype; [M, H/2] packed for
    DT_FP4_E2M1), x_scales [M, H/32] uint8 E8M0, expert_ids [M] int32; weights as
    for mm_mega_moe with E =
    local_experts.  Returns (out [M, H] bf16, expert_token_nums [local_experts]
    int32)."""
    _need_dtype(x, _BYTE_DTYPES, "x")
    _need_dtype(x_scales, (torch.uint8,), "x_scales")
    _need_dtype(expert_ids, (torch.int32,), "expert_ids")
    for name, t in (("weight1", weight1), ("weight2", weight2)):
        _need_dtype(t, _BYTE_DTYPES, name)
    for name, t in (("weight_scales1", weight_scales1), ("weight_scales2", weight_scales2)):
        _need_dtype(t, (torch.uint8,), name)
    _need(x.dim() == 2 and weight1.dim() == 3, "x must be [M, H] and weight1 [E, 2I, H]")
    m = x.shape[0]
    h = x.shape[1] * 2 if x_dtype == DT_FP4_E2M1 else x.shape[1]
    if expert_ids.numel() != m or x_scales.shape[0] != m:
        raise MMError("expert_ids and x_scales must hold one entry / row per row of x")
    _need(x_scales.numel() >= m * (h // 32), f"x_scales must be [M, H/32] = [{m}, {h // 32}]")
    inter = weight1.shape[1] // 2
    aw = 2 * inter if activation == "gelu" else inter
    _need_weights(weight1, weight2, weight_scales1, weight_scales2, local_experts, h, aw,
                  _fp8_code(weight1, weight_dtype) == DT_FP4_E2M1)
    _need_out(out, (m, h))
    _need_cuda(x, x_scales, expert_ids, weight1, weight2, weight_scales1, weight_scales2)
    L = load()
    dev = x.device
    y = out if out is not None else torch.empty((m, h), dtype=torch.bfloat16, device=dev)
    counts = torch.empty(local_experts, dtype=torch.int32, device=dev)
    need = ctypes.c_size_t(0)
    _check(L.mm_moe_expert_ffn_workspace_size(m, h, local_experts, inter, weight_scale_layout, ctypes.byref(need)),
           "mm_moe_expert_ffn_workspace_size")
    ws = _workspace(need.value, dev, workspace)
    params = list(activation_params)
    parr = (ctypes.c_float * max(len(params), 1))(*params) if params else None
    _check(L.mm_moe_expert_ffn(_ptr(x), _ptr(x_scales), _fp8_code(x, x_dtype), _ptr(expert_ids), m, h, _ptr(weight1),
                               _ptr(weight2), _ptr(weight_scales1), _ptr(weight_scales2),
                               _fp8_code(weight1, weight_dtype), weight_scale_layout, local_experts, inter,
                               activation.encode(), parr, len(params), _ptr(y), _ptr(counts), _ptr(ws), ws.numel(),
                               _dev_err(dev_err), _stream(dev)), "mm_moe_expert_ffn")
    return y, counts


# --------------------------------------------------------------------------- diagnostics
STAGES = ("wscale", "route", "dispatch", "gemm1", "gemm2", "combine", "diag")


def timing_enable(on: bool = True):
    """Record CUDA events around every stage of the following calls (mm_timing_enable)."""
    L = load()
    L.mm_timing_enable.argtypes, L.mm_timing_enable.restype = [ctypes.c_int], ctypes.c_int
    _check(L.mm_timing_enable(1 if on else 0), "mm_timing_enable")


def timing_select(stages=None):
    """Record events only around the named stages (all when None) while timing is on (mm_timing_select)."""
    L = load()
    mask = (1 << len(STAGES)) - 1 if stages is None else sum(1 << STAGES.index(s) for s in stages)
    L.mm_timing_select.argtypes, L.mm_timing_select.restype = [ctypes.c_uint32], ctypes.c_int
    _check(L.mm_timing_select(mask), "mm_timing_select")


def timing_read():
    """{stage: (device ms summed over recorded calls, kernel launches)} since the last read."""
    L = load()
    n = len(STAGES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    L.mm_timing_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    L.mm_timing_read.restype = ctypes.c_int
    _check(L.mm_timing_read(ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(cnt, ctypes.c_void_p), n), "mm_timing_read")
    return {s: (ms[i], int(cnt[i])) for i, s in enumerate(STAGES)}


ROUTE_AUTO, ROUTE_CLUSTER, ROUTE_GRID, ROUTE_KERNELS = 0, 1, 2, 3


def set_routing_path(path: int):
    """Routing implementation for the following calls, process-wide (mm_set_routing_path):
    ROUTE_AUTO, ROUTE_CLUSTER, ROUTE_GRID or ROUTE_KERNELS.  All give identical results."""
    L = load()
    L.mm_set_routing_path.argtypes, L.mm_set_routing_path.restype = [ctypes.c_int], ctypes.c_int
    _check(L.mm_set_routing_path(int(path)), "mm_set_routing_path")


# --------------------------------------------------------------------------- no-allocation variant
NOALLOC_SCRATCH_BYTES = 4 << 20


def mm_moe_init_routing_noalloc(x, expert_idx, expert_num: int, quant_mode: int = QUANT_NONE,
                                expert_tokens_num_type: int = 1, *, dev_err=None):
    """mm_moe_init_routing without a workspace: the library's fixed 4 MiB device
    scratch array is used instead (for callers that cannot provide scratch
    memory).  Same outputs as mm_moe_init_routing.  Calls that may overlap on
    the GPU race on the shared array; keep them on one stream."""
    _need_dtype(x, _SRC_DTYPES, "x")
    _need_dtype(expert_idx, (torch.int32,), "expert_idx")
    _need(x.dim() == 2, "x must be [N, H]")
    _need_rows_of(expert_idx, x.shape[0], "expert_idx", "x")
    _need_cuda(x, expert_idx)
    L = load()
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.mm_moe_init_routing_noalloc.argtypes = [p, i32, p, i64, i64, i64, i64, i32, i32, p, p, p, p, p, p, p]
    L.mm_moe_init_routing_noalloc.restype = i32
    n, h = x.shape
    k = expert_idx.shape[1] if expert_idx.dim() == 2 else 1
    rows = n * k
    dev = x.device
    out_dt = x.dtype if quant_mode == QUANT_NONE else _FP8_TORCH.get(_QUANT_FMT.get(quant_mode), torch.uint8)
    expanded_x = torch.empty((rows, h // 2 if quant_mode == QUANT_MXFP4_E2M1 else h), dtype=out_dt, device=dev)
    scale = (torch.empty((rows, _scale_cols(h)), dtype=torch.uint8, device=dev) if quant_mode != QUANT_NONE
             else torch.empty((0,), dtype=torch.uint8, device=dev))
    exp_idx = torch.empty(rows, dtype=torch.int32, device=dev)
    srt_idx = torch.empty(rows, dtype=torch.int32, device=dev)
    tokens = torch.empty(expert_num, dtype=torch.int64, device=dev)
    _check(L.mm_moe_init_routing_noalloc(_ptr(x), _dt(x), _ptr(expert_idx), n, h, k, expert_num, quant_mode,
                                         expert_tokens_num_type, _ptr(expanded_x),
                                         _ptr(scale) if scale.numel() else None, _ptr(exp_idx), _ptr(srt_idx),
                                         _ptr(tokens), _dev_err(dev_err), _stream(dev)),
           "mm_moe_init_routing_noalloc")
    return expanded_x, exp_idx, tokens, scale, srt_idx
