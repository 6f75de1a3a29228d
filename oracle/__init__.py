"""CPU oracle for the MoE routing / permute / MXFP8 expert-FFN path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product
library (``routing_permute_mxfp8_gb300``) never does, and shares no code
with it.

The arithmetic lives in ``oracle.c`` (plain C, double precision, OpenMP
over independent rows); this module builds it with gcc and wraps it for
numpy arrays.  Each wrapper names the page passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lib = None

E5M2 = 23
E4M3 = 24
E2M1 = 296   # FLOAT4_E2M1; the oracle keeps one 4-bit code per byte (bits 0-3)
DT_F32, DT_F16, DT_BF16 = 0, 1, 27


def build() -> str:
    """Compile oracle.c (gcc -O2, OpenMP) into oracle/_oracle.so."""
    tmp = _LIB_PATH + ".tmp"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"],
                   check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        build()
    L = ctypes.CDLL(_LIB_PATH)
    p, i64, i32, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    u8, u16 = ctypes.c_uint8, ctypes.c_uint16
    L.orc_num_threads.restype = i32
    L.orc_fp8_value.argtypes, L.orc_fp8_value.restype = [u8, i32], d
    L.orc_fp8_round.argtypes, L.orc_fp8_round.restype = [d, i32], u8
    L.orc_fp8_round_array.argtypes, L.orc_fp8_round_array.restype = [p, i64, i32, p], None
    L.orc_bf16_round.argtypes, L.orc_bf16_round.restype = [d], u16
    L.orc_mx_block.argtypes, L.orc_mx_block.restype = [p, i64, i32, p, p], None
    L.orc_mx_quantize_rows.argtypes, L.orc_mx_quantize_rows.restype = [p, i64, i64, i32, p, p, i64], None
    L.orc_mx_quantize_src.argtypes, L.orc_mx_quantize_src.restype = [p, i32, i64, i64, i32, p, p, i64], None
    L.orc_route.argtypes, L.orc_route.restype = [p, i32, i64, i64, i64, p, p, p], i64
    L.orc_route_range.argtypes, L.orc_route_range.restype = [p, i32, i64, i64, i64, i64, i64, p, p, p], i64
    L.orc_permute.argtypes, L.orc_permute.restype = [p, i32, i64, i64, p, i64, i32, p, p, i64], None
    L.orc_expert_row.argtypes = [p, p, i32, p, p, p, p, i32, i64, i64, i32, i32, p, p, p, p]
    L.orc_expert_row.restype = None
    L.orc_mega_moe_tokens.argtypes = [p, p, p, i32, p, p, p, p, p, p, p, p, i64, i64, i64, i64, i64,
                                      i32, i32, i32, p, i64, p, p, p, p, p, p, i32, p, i32, i32]
    L.orc_mega_moe_tokens.restype = None
    L.orc_act_code.argtypes, L.orc_act_code.restype = [i32], i32
    _lib = L
    return L


def _ptr(a):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return int(_load().orc_num_threads())


def fp8_value(code: int, fmt: int) -> float:
    """Value of one FP8 code (format definition of FLOAT8_E4M3FN / FLOAT8_E5M2), or of
    one FLOAT4_E2M1 code (bits 0-3)."""
    return float(_load().orc_fp8_value(code, fmt))


def fp8_round(t: float, fmt: int) -> int:
    """FP8 code of t: saturate, nearest, ties to even, sign kept."""
    return int(_load().orc_fp8_round(float(t), fmt))


def fp8_round_array(t, fmt: int) -> np.ndarray:
    t = np.ascontiguousarray(t, dtype=np.float64)
    out = np.zeros(t.shape, dtype=np.uint8)
    _load().orc_fp8_round_array(_ptr(t), t.size, fmt, _ptr(out))
    return out


def bf16_round(t: float) -> int:
    return int(_load().orc_bf16_round(float(t)))


def mx_block(v, fmt: int):
    """Q_MX of one group (MegaMoE A8W8-FP stage 1): returns (codes uint8[n], scale code)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    q = np.zeros(v.size, dtype=np.uint8)
    s = np.zeros(1, dtype=np.uint8)
    _load().orc_mx_block(_ptr(v), v.size, fmt, _ptr(q), _ptr(s))
    return q, int(s[0])


def mx_quantize_f64(x: np.ndarray, fmt: int, s_cols: int | None = None):
    """Q_MX along the last axis of a 2-D double matrix; scales [rows, s_cols]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    rows, cols = x.shape
    s_cols = (cols + 31) // 32 if s_cols is None else s_cols
    q = np.zeros((rows, cols), dtype=np.uint8)
    s = np.zeros((rows, s_cols), dtype=np.uint8)
    _load().orc_mx_quantize_rows(_ptr(x), rows, cols, fmt, _ptr(q), _ptr(s), s_cols)
    return q, s


def mx_quantize(x: np.ndarray, dtype: int, fmt: int, s_cols: int | None = None):
    """Q_MX along the last axis of a 2-D matrix given as fp32 (float32 array)
    or as bf16 / fp16 bit patterns (uint16 array, dtype DT_BF16 / DT_F16)."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    s_cols = (cols + 31) // 32 if s_cols is None else s_cols
    q = np.zeros((rows, cols), dtype=np.uint8)
    s = np.zeros((rows, s_cols), dtype=np.uint8)
    _load().orc_mx_quantize_src(_ptr(x), dtype, rows, cols, fmt, _ptr(q), _ptr(s), s_cols)
    return q, s


def route(ids: np.ndarray, num_experts: int):
    """keyValueSort + inverse map + histogram (MoeInitRoutingV3 steps 1-3).

    Returns (sorted_row_idx int32[R], expanded_row_idx int32[R], counts int64[E], n_invalid).
    """
    ids = np.ascontiguousarray(ids)
    is64 = 1 if ids.dtype == np.int64 else 0
    if not is64:
        ids = ids.astype(np.int32, copy=False)
    n = ids.shape[0]
    k = ids.shape[1] if ids.ndim == 2 else 1
    rows = n * k
    srt = np.empty(rows, dtype=np.int32)
    exp = np.empty(rows, dtype=np.int32)
    cnt = np.empty(num_experts, dtype=np.int64)
    bad = _load().orc_route(_ptr(ids), is64, n, k, num_experts, _ptr(srt), _ptr(exp), _ptr(cnt))
    return srt, exp, cnt, int(bad)


def route_range(ids: np.ndarray, num_experts: int, start: int, end: int):
    """route() with MoeInitRoutingV3's active expert range [start, end)
    (activeExpertRangeOptional): only ids in the range are sorted (step 6:
    availableIdxNum of them); counts int64[end - start]; the fourth value is the
    number of ids outside [0, num_experts) (ids outside the range are no error)."""
    ids = np.ascontiguousarray(ids)
    is64 = 1 if ids.dtype == np.int64 else 0
    if not is64:
        ids = ids.astype(np.int32, copy=False)
    n = ids.shape[0]
    k = ids.shape[1] if ids.ndim == 2 else 1
    rows = n * k
    srt = np.empty(rows, dtype=np.int32)
    exp = np.empty(rows, dtype=np.int32)
    cnt = np.empty(max(end - start, 0), dtype=np.int64)
    bad = _load().orc_route_range(_ptr(ids), is64, n, k, num_experts, start, end, _ptr(srt), _ptr(exp), _ptr(cnt))
    return srt, exp, cnt, int(bad)


def key_value_counts(counts: np.ndarray, start: int, num_experts: int) -> np.ndarray:
    """MoeInitRoutingV3 expertTokensNumType 2 (key_value): [num_experts, 2] int64
    holding (expert id, token count) for each expert of the active range with a
    non-zero count, in ascending expert order; the rows after them are 0."""
    out = np.zeros((num_experts, 2), dtype=np.int64)
    m = 0
    for e, c in enumerate(counts):
        if c != 0:
            out[m] = (start + e, c)
            m += 1
    return out


def permute(x: np.ndarray, dtype: int, k: int, sorted_row_idx: np.ndarray, m_out: int, fmt: int = -1):
    """Gather (+ optional Q_MX) of token rows in sorted order (MoeInitRoutingV3
    step 5 / moe_token_permute).  fmt = -1 copies; 23 / 24 quantise with
    scales [m_out, AlignUp(CeilDiv(H, 32), 2)]."""
    x = np.ascontiguousarray(x)
    h = x.shape[1]
    srt = np.ascontiguousarray(sorted_row_idx, dtype=np.int32)
    s_cols = ((h + 31) // 32 + 1) // 2 * 2
    if fmt < 0:
        out = np.zeros((m_out, h), dtype=x.dtype)
        sc = np.zeros((0,), dtype=np.uint8)
        _load().orc_permute(_ptr(x), dtype, h, k, _ptr(srt), m_out, -1, _ptr(out), None, 0)
    else:
        out = np.zeros((m_out, h), dtype=np.uint8)
        sc = np.zeros((m_out, s_cols), dtype=np.uint8)
        _load().orc_permute(_ptr(x), dtype, h, k, _ptr(srt), m_out, fmt, _ptr(out), _ptr(sc), s_cols)
    return out, sc


# Activations of the MegaMoE README ("Activation function formulas") and the
# defaults its activation_params description gives.
ACTIVATIONS = {"swiglu": 0, "swiglustep": 1, "swigluoai": 2, "situglu": 3, "gelu": 4}


def activation_spec(name="swiglu", params=()):
    """(kind, [c, alpha, beta, beta_lin]) for an activation name and its
    activation_params list: clamp c (absent or 0: not enabled, +inf) for
    swiglu / swiglustep / swigluoai; swigluoai alpha 1.702 and beta 1.0 by
    default; situglu [beta] or [beta, beta_lin] (beta 1.0 when the list is
    empty; beta_lin 0 = not configured); gelu takes a placeholder only."""
    kind = ACTIVATIONS[name]
    params = [float(v) for v in params]
    c, alpha, beta, beta_lin = np.inf, 1.702, 1.0, 0.0
    if kind in (0, 1, 2) and params:
        c = params[0] if params[0] != 0.0 else np.inf
        if kind == 2 and len(params) == 3:
            alpha, beta = params[1], params[2]
    if kind == 3:
        beta = params[0] if params else 1.0
        beta_lin = params[1] if len(params) > 1 else 0.0
    return kind, np.array([c, alpha, beta, beta_lin], dtype=np.float64)


def expert_row(xq, xs, x_fmt, w1, s1, w2, s2, w_fmt, a_fmt, activation="swiglu", act_params=()):
    """One expanded row through one expert (A8W8-FP / A8W4-FP stages 2-3).

    xq uint8[H], xs uint8[H/32]; w1 [2I, H], s1 [2I, 2*ceil(H/64)];
    w2 [H, W], s2 [H, 2*ceil(W/64)] with W = I (gated) or 2I (gelu).
    Returns (aq uint8[W], as uint8[W/32], o float64[H]).
    """
    kind, p = activation_spec(activation, act_params)
    h = xq.size
    inter = w1.shape[0] // 2
    aw = w2.shape[1]
    aq = np.zeros(aw, dtype=np.uint8)
    a_s = np.zeros((aw + 31) // 32, dtype=np.uint8)
    o = np.zeros(h, dtype=np.float64)
    arrs = [np.ascontiguousarray(a) for a in (xq, xs, w1, s1, w2, s2)]
    _load().orc_expert_row(_ptr(arrs[0]), _ptr(arrs[1]), x_fmt, _ptr(arrs[2]), _ptr(arrs[3]),
                           _ptr(arrs[4]), _ptr(arrs[5]), w_fmt, h, inter, a_fmt, kind, _ptr(p), _ptr(aq),
                           _ptr(a_s), _ptr(o))
    return aq, a_s, o


def act_format(x_fmt: int) -> int:
    """Format of A_hat for dispatch format x_fmt: x_fmt itself (A8W8-FP, A8W4-FP),
    MXFP8 E4M3 under an FP4 E2M1 dispatch (A4W4-FP stage 2, so that GEMM2 is A8W4)."""
    return int(_load().orc_act_code(int(x_fmt)))


def mega_moe_tokens(x_bf16, ids, gate, w1, s1, w2, s2, x_fmt, w_fmt, tokens=None,
                    shared=None, shared_w_fmt=None, want_act=False, activation="swiglu", act_params=(),
                    x_prequant=None, shared_x_fmt=None, combine_fmt=None):
    """MegaMoE forward at ep_world_size = 1 for selected tokens (A8W8-FP / A8W4-FP /
    A4W4-FP stages 1-4; x_fmt 296 dispatches MXFP4 E2M1 codes, one per byte).  x_prequant = (codes uint8[N, H], scales uint8[N, ceil(H/32)]):
    pre-quantised pass-through (dispatchQuantMode = 0): X_hat and S_X are the given
    ones and x_bf16 is not read.

    x_bf16 uint16[N, H]; ids int32[N, K]; gate float32[N, K] or bf16 bits uint16[N, K];
    w1 uint8[E, 2I, H], s1 uint8[E, 2I, 2*ceil(H/64)], w2 uint8[E, H, I],
    s2 uint8[E, H, 2*ceil(I/64)]; shared = (sw1, ss1, sw2, ss2) with a leading
    shared-expert dimension, or None; shared_x_fmt: the shared experts' own input
    quantisation type (the parameter table's sharedExpertQuantOutDtype; None: x_fmt);
    combine_fmt: 23 / 24 for combineQuantMode 3 / 4 (routed rows enter the sum as
    DQ_MX(Q_MX(bf16(O)))), None: no combine quantisation.
    Returns (y float64[T, H], y_bf16 uint16[T, H]) and, with want_act, the
    activation codes uint8[T, K, I] (format act_format(x_fmt)) and scales uint8[T, K, I/32].
    """
    kind, p = activation_spec(activation, act_params)
    n, h = x_bf16.shape if x_prequant is None else x_prequant[0].shape
    k = ids.shape[1]
    e, two_i, _ = w1.shape
    inter = two_i // 2
    aw = two_i if kind == ACTIVATIONS["gelu"] else inter
    tokens = np.arange(n, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    t = tokens.size
    y = np.zeros((t, h), dtype=np.float64)
    yb = np.zeros((t, h), dtype=np.uint16)
    gate = np.ascontiguousarray(gate)
    gate_is_bf16 = 1 if gate.dtype == np.uint16 else 0
    if shared is None:
        sw = [None] * 4
        n_sh = 0
        shared_w_fmt = w_fmt
    else:
        sw = [np.ascontiguousarray(a) for a in shared]
        n_sh = sw[0].shape[0]
        shared_w_fmt = w_fmt if shared_w_fmt is None else shared_w_fmt
    aq = np.zeros((t, k, aw), dtype=np.uint8) if want_act else None
    a_s = np.zeros((t, k, (aw + 31) // 32), dtype=np.uint8) if want_act else None
    xq = xs = None
    if x_prequant is not None and shared_x_fmt is not None and shared_x_fmt != x_fmt:
        raise ValueError("pass-through: the shared experts take the dispatch type")
    if x_prequant is not None:
        xq, xs = (np.ascontiguousarray(a, dtype=np.uint8) for a in x_prequant)
        x_bf16 = None
    arrs = [None if a is None else np.ascontiguousarray(a)
            for a in (x_bf16, ids.astype(np.int32, copy=False), w1, s1, w2, s2)]
    _load().orc_mega_moe_tokens(
        _ptr(arrs[0]), _ptr(arrs[1]), _ptr(gate), gate_is_bf16, _ptr(arrs[2]), _ptr(arrs[3]),
        _ptr(arrs[4]), _ptr(arrs[5]), _ptr(sw[0]), _ptr(sw[1]), _ptr(sw[2]), _ptr(sw[3]), n_sh, h, k,
        e, inter, x_fmt, w_fmt, shared_w_fmt, _ptr(tokens), t, _ptr(y), _ptr(yb), _ptr(aq), _ptr(a_s),
        _ptr(xq), _ptr(xs), kind, _ptr(p), -1 if shared_x_fmt is None else int(shared_x_fmt),
        -1 if combine_fmt is None else int(combine_fmt))
    if want_act:
        return y, yb, aq, a_s
    return y, yb


def quantized_weights(cfg, which: int, shared: bool = False, fmt: int | None = None):
    """fp32 N(0, 0.02) source weights of every expert (seeded generator) MX-quantised
    by the oracle along the reduction dimension.  Returns (codes [E, N_out, K_red],
    scales [E, N_out, 2*ceil(K_red/64)]) in the MegaMoE weight / weightScales layouts."""
    import synth
    fmt = cfg.weight_fmt if fmt is None else fmt
    n_exp = cfg.shared if shared else cfg.e
    if which == 1:
        n_out, k_red = 2 * cfg.inter, cfg.h
    else:
        n_out, k_red = cfg.h, cfg.act_width
    s_cols = 2 * ((k_red + 63) // 64)
    q = np.empty((n_exp, n_out, k_red), dtype=np.uint8)
    s = np.empty((n_exp, n_out, s_cols), dtype=np.uint8)
    for ex in range(n_exp):
        w = synth.weight_f32(cfg, which, ex, shared=shared)
        q[ex], s[ex] = mx_quantize(w, DT_F32, fmt, s_cols)
    return q, s
