"""Pins of the CPU oracle against what the pages and the mathematics fix.

No test here compares the oracle with itself or with the CUDA path: FP8
values come from torch's float8 decode, rounding from an exhaustive code
search, sorts from numpy's stable argsort, GEMMs from numpy matmul, the
worked example and the hand-computed MX blocks from tests/golden/.
"""
import json
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
import synth
from tests import _pins as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMTS = [P.E4M3, P.E5M2]
FMTS_ALL = FMTS + [P.E2M1]   # with FLOAT4_E2M1 (A8W4-FP weights)


# ---------------------------------------------------------------- FP8 codes
@pytest.mark.parametrize("fmt", FMTS)
def test_fp8_decode_matches_torch(fmt):
    tab = P.fp8_table(fmt)
    for c in range(256):
        v = oracle.fp8_value(c, fmt)
        if np.isnan(tab[c]):
            assert np.isnan(v), c
        else:
            assert v == tab[c], (c, v, tab[c])


def test_fp4_decode_matches_spec_list():
    """FLOAT4_E2M1: the 16 codes against the OCP MX v1.0 value list."""
    tab = P.fp8_table(P.E2M1)
    for c in range(16):
        v = oracle.fp8_value(c, P.E2M1)
        assert v == tab[c] and np.signbit(v) == (c >= 8), (c, v)
    # largest finite value, the subnormal, one
    assert oracle.fp8_value(0x7, P.E2M1) == 6.0
    assert oracle.fp8_value(0x1, P.E2M1) == 0.5
    assert oracle.fp8_value(0x2, P.E2M1) == 1.0


def test_fp8_closed_forms():
    # largest finite values, smallest subnormals, one, infinities / NaN
    assert oracle.fp8_value(0x7E, P.E4M3) == 448.0
    assert oracle.fp8_value(0x01, P.E4M3) == 2.0 ** -9
    assert oracle.fp8_value(0x08, P.E4M3) == 2.0 ** -6
    assert oracle.fp8_value(0x38, P.E4M3) == 1.0
    assert np.isnan(oracle.fp8_value(0x7F, P.E4M3))
    assert oracle.fp8_value(0x7B, P.E5M2) == 57344.0
    assert oracle.fp8_value(0x01, P.E5M2) == 2.0 ** -16
    assert oracle.fp8_value(0x3C, P.E5M2) == 1.0
    assert oracle.fp8_value(0x7C, P.E5M2) == np.inf


def _hard_values(fmt, n, seed):
    rng = np.random.default_rng(seed)
    tab = P.fp8_table(fmt)
    fin = np.sort(np.unique(np.abs(tab[np.isfinite(tab)])))
    mids = (fin[1:] + fin[:-1]) / 2                      # exact ties
    near = np.concatenate([mids * (1 + 1e-12), mids * (1 - 1e-12)])
    mag = np.exp2(rng.uniform(-24, np.log2(P.MAXV[fmt]) + 1, n))
    rnd = mag * rng.choice([-1.0, 1.0], n)
    special = np.array([0.0, -0.0, P.MAXV[fmt], -P.MAXV[fmt], P.MAXV[fmt] * 1.07, 1e30, -1e30,
                        2.0 ** -30, -(2.0 ** -30)])
    grid = np.concatenate([fin, -fin])
    allv = np.concatenate([rnd, mids, -mids, near, -near, grid, special])
    return allv


@pytest.mark.parametrize("fmt", FMTS_ALL)
def test_fp8_round_brute_force(fmt):
    t = _hard_values(fmt, 1_000_000, 1 + fmt)
    got = oracle.fp8_round_array(t, fmt)
    want = P.brute_round(t, fmt)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(t[i], got[i], want[i]) for i in bad[:10]]


@pytest.mark.parametrize("fmt", FMTS)
def test_fp8_round_matches_torch_in_range(fmt):
    rng = np.random.default_rng(7)
    t = rng.uniform(-P.MAXV[fmt], P.MAXV[fmt], 200_000).astype(np.float32)
    t = np.concatenate([t, (t / 1e3).astype(np.float32), (t / 1e6).astype(np.float32)])
    want = torch.from_numpy(t).to(P._TORCH[fmt]).view(torch.uint8).numpy()
    got = oracle.fp8_round_array(t.astype(np.float64), fmt)
    assert np.array_equal(got, want)


# ------------------------------------------------------------ MX quantiser
def _golden_blocks():
    rows = []
    for line in open(os.path.join(GOLDEN, "mx_blocks.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        fmt, sc, vals, codes = [f.strip() for f in line.split("|")]
        rows.append((int(fmt), int(sc), [float(v) for v in vals.split()],
                     [int(c, 16) for c in codes.split()]))
    return rows


@pytest.mark.parametrize("block", _golden_blocks())
def test_mx_hand_blocks(block):
    fmt, sc, vals, codes = block
    v = np.zeros(32)
    v[: len(vals)] = vals
    q, s = oracle.mx_block(v, fmt)
    assert s == sc
    assert list(q[: len(codes)]) == codes


@pytest.mark.parametrize("fmt", FMTS_ALL)
def test_mx_scale_puts_amax_in_top_binade(fmt):
    """With s = code - 127, amax * 2^-s lies in [2^emax, 2^(emax+1)) unless the
    scale is clamped: the group's largest element uses the format's top binade."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4000, 32)) * np.exp2(rng.integers(-40, 40, (4000, 1)))
    for r in range(x.shape[0]):
        _, s = oracle.mx_block(x[r], fmt)
        t = np.abs(x[r]).max() * 2.0 ** -(s - 127)
        top = {P.E4M3: 256.0, P.E5M2: 32768.0, P.E2M1: 4.0}[fmt]
        assert top <= t < 2 * top


@pytest.mark.parametrize("fmt", FMTS_ALL)
def test_mx_roundtrip_bound(fmt):
    """|DQ(Q(v)) - v| <= half the local FP8 spacing times 2^s for unsaturated
    elements; saturated ones decode to the largest finite value."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((2000, 32)) * np.exp2(rng.integers(-10, 10, (2000, 1)))
    tab = P.fp8_table(fmt)
    fin = np.sort(np.unique(np.abs(tab[np.isfinite(tab)])))
    for r in range(x.shape[0]):
        q, s = oracle.mx_block(x[r], fmt)
        sc = 2.0 ** (s - 127)
        t = np.abs(x[r]) / sc
        back = np.abs(tab[q])
        for ti, bi in zip(t, back):
            if ti >= P.MAXV[fmt]:
                assert bi == P.MAXV[fmt]
                continue
            i = np.searchsorted(fin, ti)
            lo = fin[max(i - 1, 0)]
            hi = fin[min(i, fin.size - 1)]
            assert abs(bi - ti) <= (hi - lo) / 2 + 1e-300


@pytest.mark.parametrize("fmt", FMTS_ALL)
def test_mx_rows_match_brute_force(fmt):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-6, 6, (64, 1)))
    x[3, 32:64] = 0.0
    x[4, :32] = -0.0
    q, s = oracle.mx_quantize_f64(x, fmt)
    qb, sb = P.brute_mx_rows(x, fmt)
    assert np.array_equal(s, sb)
    assert np.array_equal(q, qb)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    t = (rng.standard_normal(100_000) * np.exp2(rng.integers(-60, 60, 100_000))).astype(np.float32)
    want = torch.from_numpy(t).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in t[:20000]], dtype=np.uint16)
    assert np.array_equal(got, want[:20000])


# ------------------------------------------------------------------ routing
def test_route_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "permute_example.json")))
    ids = np.array(g["indices"], dtype=np.int32)
    srt, exp, cnt, bad = oracle.route(ids, 2)
    assert bad == 0
    assert srt.tolist() == g["sorted_indices_first"]
    assert exp.tolist() == g["sorted_indices"]
    assert cnt.tolist() == g["counts"]
    assert (srt // ids.shape[1]).tolist() == g["source_tokens"]
    # shapes printed by the page
    x = np.arange(4 * g["hidden"], dtype=np.uint16).reshape(4, g["hidden"])
    out, sc = oracle.permute(x, oracle.DT_F16, 2, srt, g["num_out_tokens"])
    assert list(out.shape) == g["shape_permuted_truncated"]
    assert list(exp.shape) == g["shape_sorted_indices"]
    assert list(sc.shape) == g["shape_scale_unquantized"]
    out, sc = oracle.permute(x, oracle.DT_F16, 2, srt, 8, fmt=P.E5M2)
    assert list(out.shape) == g["shape_permuted_mxfp8"]
    assert list(sc.shape) == g["shape_scale_mxfp8"]


@pytest.mark.parametrize("n,k,e,distinct", [(1000, 8, 64, True), (777, 4, 5, False), (1, 1, 1, True),
                                            (4096, 8, 256, True)])
def test_route_matches_numpy_stable_argsort(n, k, e, distinct):
    rng = np.random.default_rng(n + k + e)
    if distinct:
        ids = np.argsort(rng.random((n, e)), axis=1)[:, :k].astype(np.int32)
    else:
        ids = rng.integers(0, e, (n, k)).astype(np.int32)
    srt, exp, cnt, bad = oracle.route(ids, e)
    flat = ids.reshape(-1)
    want = np.argsort(flat, kind="stable")
    assert bad == 0
    assert np.array_equal(srt, want)
    inv = np.empty_like(want)
    inv[want] = np.arange(want.size)
    assert np.array_equal(exp, inv)
    assert np.array_equal(cnt, np.bincount(flat, minlength=e))
    # invariants: permutation, sorted keys, stability, totals
    assert np.array_equal(np.sort(srt), np.arange(n * k))
    keys = flat[srt]
    assert np.all(np.diff(keys) >= 0)
    same = np.diff(keys) == 0
    assert np.all(np.diff(srt)[same] > 0)
    assert cnt.sum() == n * k


def test_route_int64_and_invalid_ids():
    ids = np.array([[0, 5], [2, -1], [1, 0]], dtype=np.int64)
    srt, exp, cnt, bad = oracle.route(ids, 3)
    assert bad == 2
    assert srt.tolist() == [0, 5, 4, 2, -1, -1]
    assert exp.tolist() == [0, -1, 3, -1, 2, 1]
    assert cnt.tolist() == [2, 1, 1]


@pytest.mark.parametrize("n,k,e,start,end", [(300, 4, 16, 0, 16), (300, 4, 16, 4, 12), (257, 8, 64, 63, 64),
                                             (64, 2, 8, 3, 3), (500, 6, 40, 0, 7)])
def test_route_active_range_matches_numpy(n, k, e, start, end):
    """MoeInitRoutingV3 with activeExpertRangeOptional = [start, end): the ids of
    the range sorted stably (numpy argsort), availableIdxNum = their number
    (step 6), counts of the range's experts; other ids (and out-of-range
    ones, counted as errors) get no row."""
    rng = np.random.default_rng(7 * n + start)
    ids = rng.integers(-1, e + 1, (n, k)).astype(np.int32)
    srt, exp, cnt, bad = oracle.route_range(ids, e, start, end)
    flat = ids.reshape(-1)
    act = (flat >= start) & (flat < end)
    order = np.nonzero(act)[0][np.argsort(flat[act], kind="stable")]
    avail = int(act.sum())
    assert avail == len(order)
    assert np.array_equal(srt[:avail], order)
    assert np.all(srt[avail:] == -1)
    want_exp = np.full(flat.size, -1, np.int32)
    want_exp[order] = np.arange(avail)
    assert np.array_equal(exp, want_exp)
    assert np.array_equal(cnt, np.bincount(flat[act] - start, minlength=end - start)[: end - start])
    assert bad == int(((flat < 0) | (flat >= e)).sum())
    if start == 0 and end == e:   # the full range is route()
        r = oracle.route(ids, e)
        assert all(np.array_equal(a, b) for a, b in zip(r[:3], (srt, exp, cnt))) and r[3] == bad


def test_key_value_counts_hand_example():
    """expertTokensNumType 2: (expert, count) of the range's non-zero experts in
    ascending order, [expertNum, 2]; rows after them 0."""
    kv = oracle.key_value_counts(np.array([0, 3, 0, 2]), 4, 6)
    assert kv.tolist() == [[5, 3], [7, 2], [0, 0], [0, 0], [0, 0], [0, 0]]


# ------------------------------------------------------------------ permute
@pytest.mark.parametrize("fmt", [-1, P.E4M3, P.E5M2, P.E2M1])
def test_permute_matches_gather(fmt):
    cfg = synth.CONFIGS["tiny"].scaled(n=96, h=160)
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    srt, exp, cnt, _ = oracle.route(ids, cfg.e)
    m = cfg.rows - 7
    out, sc = oracle.permute(x, oracle.DT_BF16, cfg.k, srt, m, fmt=fmt)
    src = x[srt[:m] // cfg.k]
    if fmt < 0:
        assert np.array_equal(out, src)
        return
    qb, sb = P.brute_mx_rows(P.bf16_bits_to_f64(src), fmt)
    assert np.array_equal(out, qb)
    g = (cfg.h + 31) // 32
    assert sc.shape == (m, (g + 1) // 2 * 2)
    assert np.array_equal(sc[:, :g], sb)
    assert np.all(sc[:, g:] == 0)


# ---------------------------------------------------------------- expert FFN
def _numpy_grouped_moe(cfg, x, ids, gate, w, shared=None, shared_fmt=None, shared_xfmt=None, combine_fmt=None):
    """Grouped-by-expert FFN with numpy matmuls on dequantised operands, from
    the MegaMoE A8W8-FP stage formulas; sort by numpy stable argsort.  The
    activation is re-quantised in the dispatch type, except in the A4W4-FP
    scenario (FP4 E2M1 dispatch), whose stage 2 re-quantises it to MXFP8 E4M3.
    Shared experts quantise their input in shared_xfmt when given (the
    parameter table's sharedExpertQuantOutDtype), with the same rule for
    their activation."""
    (w1, s1, w2, s2) = w
    fx = cfg.dispatch_fmt
    xq, xs = P.brute_mx_rows(P.bf16_bits_to_f64(x), fx)
    n, h = x.shape
    k = ids.shape[1]
    inter = cfg.inter
    order = np.argsort(ids.reshape(-1), kind="stable")
    pos = np.empty_like(order)
    pos[order] = np.arange(order.size)
    rows = order // k
    o_all = np.zeros((order.size, h))
    aq_all = np.zeros((order.size, inter), dtype=np.uint8)

    def ffn(rows_q, rows_s, W1, S1, W2, S2, wfmt, fx=fx):
        fa = P.E4M3 if fx == P.E2M1 else fx
        xd = P.dequant_rows(rows_q, rows_s, fx)
        w1d = P.dequant_rows(W1, S1, wfmt)
        hv = xd @ w1d.T
        g, u = hv[:, :inter], hv[:, inter:]
        a = (g * expit(g) * u).astype(np.float32).astype(np.float64)
        aq, a_s = P.brute_mx_rows(a, fa)
        o = P.dequant_rows(aq, a_s, fa) @ P.dequant_rows(W2, S2, wfmt).T
        return aq, o

    flat = ids.reshape(-1)[order]
    for e in range(cfg.e):
        sel = np.nonzero(flat == e)[0]
        if sel.size == 0:
            continue
        aq, o = ffn(xq[rows[sel]], xs[rows[sel]], w1[e], s1[e], w2[e], s2[e], cfg.weight_fmt)
        if combine_fmt is not None:   # combineQuantMode: the bf16 row as MX codes on the wire
            ob = torch.from_numpy(o).to(torch.bfloat16).double().numpy()
            oq, os_ = P.brute_mx_rows(ob, combine_fmt)
            o = P.dequant_rows(oq, os_, combine_fmt)
        o_all[sel] = o
        aq_all[sel] = aq
    gw = P.bf16_bits_to_f64(gate) if gate.dtype == np.uint16 else gate.astype(np.float64)
    y = np.zeros((n, h))
    for kk in range(k):
        y += gw[:, kk:kk + 1] * o_all[pos.reshape(n, k)[:, kk]]
    if shared is not None:
        sfx = fx if shared_xfmt is None else shared_xfmt
        sq, ss = (xq, xs) if sfx == fx else P.brute_mx_rows(P.bf16_bits_to_f64(x), sfx)
        for s in range(shared[0].shape[0]):
            _, o = ffn(sq, ss, shared[0][s], shared[1][s], shared[2][s], shared[3][s],
                       cfg.weight_fmt if shared_fmt is None else shared_fmt, fx=sfx)
            y += o
    return y, aq_all[pos.reshape(n, k)]


def _weights(cfg, shared=False):
    w1, s1 = oracle.quantized_weights(cfg, 1, shared=shared)
    w2, s2 = oracle.quantized_weights(cfg, 2, shared=shared)
    return w1, s1, w2, s2


@pytest.mark.parametrize("name,kw", [
    ("tiny", {}),
    ("tiny", dict(dispatch_fmt=P.E5M2, gate_dtype="bf16", routing="zipf")),
    ("tiny", dict(n=16, shared=1)),
    ("tiny", dict(n=24, e=1, k=1)),     # K = 1, one expert: a dense two-layer FFN
    # A8W4-FP: FLOAT4_E2M1 weights, MXFP8 E4M3 activations
    ("tiny", dict(weight_fmt=P.E2M1, dispatch_fmt=P.E4M3)),
    ("tiny", dict(weight_fmt=P.E2M1, dispatch_fmt=P.E4M3, n=16, shared=1, routing="zipf")),
    # A4W4-FP: MXFP4 E2M1 tokens and weights, the activation re-quantised to MXFP8 E4M3
    ("tiny", dict(weight_fmt=P.E2M1, dispatch_fmt=P.E2M1)),
    ("tiny", dict(weight_fmt=P.E2M1, dispatch_fmt=P.E2M1, n=16, shared=1, routing="zipf", gate_dtype="bf16")),
])
def test_mega_moe_matches_numpy_grouped(name, kw):
    cfg = synth.CONFIGS[name].scaled(**kw)
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    gate = synth.topk_weights(cfg)
    if cfg.e == 1:
        gate = np.ones_like(gate, dtype=np.float32)
    w = _weights(cfg)
    sh = _weights(cfg, shared=True) if cfg.shared else None
    y, yb, aq, _ = oracle.mega_moe_tokens(x, ids, gate, *w, cfg.dispatch_fmt, cfg.weight_fmt,
                                          shared=sh, want_act=True)
    y_ref, aq_ref = _numpy_grouped_moe(cfg, x, ids, gate, w, shared=sh)
    assert np.array_equal(aq, aq_ref)
    scale = np.abs(y_ref).max()
    assert np.max(np.abs(y - y_ref)) <= 1e-11 * scale
    want_b = torch.from_numpy(y_ref.astype(np.float32)).to(torch.bfloat16).float().numpy()
    got_b = P.bf16_bits_to_f64(yb)
    assert np.max(np.abs(got_b - want_b)) <= 2.0 ** -8 * np.abs(want_b).max()


@pytest.mark.parametrize("routed,shared_fmt,dispatch", [(P.E2M1, P.E4M3, P.E4M3), (P.E4M3, P.E2M1, P.E4M3),
                                                       (P.E5M2, P.E4M3, P.E4M3), (P.E2M1, P.E4M3, P.E2M1)])
def test_mega_moe_shared_weight_type_matches_numpy(routed, shared_fmt, dispatch):
    """Shared experts whose weight type differs from the routed experts' (the
    last case: FP4 tokens through FP8 shared weights under A4W4-FP)."""
    cfg = synth.CONFIGS["tiny"].scaled(n=16, shared=2, weight_fmt=routed, dispatch_fmt=dispatch)
    x, ids, gate = synth.tokens_bf16(cfg), synth.topk_ids(cfg), synth.topk_weights(cfg)
    w = _weights(cfg)
    sh = _weights(cfg.scaled(weight_fmt=shared_fmt), shared=True)
    y, _ = oracle.mega_moe_tokens(x, ids, gate, *w, cfg.dispatch_fmt, cfg.weight_fmt, shared=sh,
                                  shared_w_fmt=shared_fmt)
    y_ref, _ = _numpy_grouped_moe(cfg, x, ids, gate, w, shared=sh, shared_fmt=shared_fmt)
    assert np.max(np.abs(y - y_ref)) <= 1e-11 * np.abs(y_ref).max()


def test_mega_moe_metamorphic():
    cfg = synth.CONFIGS["tiny"].scaled(n=32)
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    gate = synth.topk_weights(cfg)
    w = _weights(cfg)
    y, _ = oracle.mega_moe_tokens(x, ids, gate, *w, cfg.dispatch_fmt, cfg.weight_fmt)
    perm = np.random.default_rng(0).permutation(cfg.n)
    yp, _ = oracle.mega_moe_tokens(x[perm], ids[perm], gate[perm], *w, cfg.dispatch_fmt, cfg.weight_fmt)
    assert np.array_equal(yp, y[perm])
    y2, _ = oracle.mega_moe_tokens(x, ids, gate * 2, *w, cfg.dispatch_fmt, cfg.weight_fmt)
    assert np.array_equal(y2, 2 * y)
    sub = np.array([5, 0, 31])
    ys, _ = oracle.mega_moe_tokens(x, ids, gate, *w, cfg.dispatch_fmt, cfg.weight_fmt, tokens=sub)
    assert np.array_equal(ys, y[sub])


def test_swiglu_special_values():
    """Row with G = 0 gives A = 0; the silu reading is z / (1 + e^-z)."""
    cfg = synth.CONFIGS["tiny"].scaled(e=1, k=1, n=1)
    h, inter = cfg.h, cfg.inter
    s_cols1, s_cols2 = 2 * ((h + 63) // 64), 2 * ((inter + 63) // 64)
    xq = np.full(h, 0x38, dtype=np.uint8)          # 1.0
    xs = np.full(h // 32, 127, dtype=np.uint8)
    w1 = np.zeros((2 * inter, h), dtype=np.uint8)
    w1[inter:, 0] = 0x38                             # up row = x[0] = 1, gate = 0
    w1[0, 0] = 0x40                                  # gate[0] = 2
    s1 = np.full((2 * inter, s_cols1), 127, dtype=np.uint8)
    w2 = np.zeros((h, inter), dtype=np.uint8)
    w2[:, 0] = 0x38
    s2 = np.full((h, s_cols2), 127, dtype=np.uint8)
    aq, a_s, o = oracle.expert_row(xq, xs, P.E4M3, w1, s1, w2, s2, P.E4M3, P.E4M3)
    a0 = np.float32(2.0 * expit(2.0))
    assert np.all(P.fp8_table(P.E4M3)[aq[1:32]] == 0)
    deq = P.fp8_table(P.E4M3)[aq[0]] * 2.0 ** (int(a_s[0]) - 127)
    assert abs(deq - a0) <= a0 * 2 ** -3
    assert np.allclose(o, deq)


# ------------------------------------------------- activations, pass-through
def _one_expert(cfg):
    """Quantised x row of token 0 and expert 0's quantised weights."""
    x = synth.tokens_bf16(cfg)
    xq, xs = oracle.mx_quantize(x[:1], oracle.DT_BF16, cfg.dispatch_fmt)
    w1, s1 = oracle.quantized_weights(cfg, 1)
    w2, s2 = oracle.quantized_weights(cfg, 2)
    return xq[0], xs[0], w1[0], s1[0], w2[0], s2[0]


def _row(cfg, act, params=()):
    xq, xs, w1, s1, w2, s2 = _one_expert(cfg)
    return oracle.expert_row(xq, xs, cfg.dispatch_fmt, w1, s1, w2, s2, cfg.weight_fmt, cfg.dispatch_fmt,
                             activation=act, act_params=params)


def test_activation_special_cases_reduce_to_swiglu():
    """MegaMoE "Activation function formulas": with the clamp disabled
    (absent, 0 or FLT_MAX) every gated form below is SwiGLU exactly or in
    the limit: swiglustep with c = inf; swigluoai with alpha = 1, beta = 0;
    situglu with beta -> inf (beta tanh(G/beta) -> G) and linear_beta -> inf."""
    cfg = synth.CONFIGS["tiny"]
    aq0, as0, o0 = _row(cfg, "swiglu")
    for act, params in (("swiglu", (0.0,)), ("swiglu", (np.finfo(np.float32).max,)), ("swiglustep", ()),
                        ("swigluoai", (0.0, 1.0, 0.0))):
        aq, a_s, o = _row(cfg, act, params)
        assert np.array_equal(aq, aq0) and np.array_equal(a_s, as0), act
        assert np.array_equal(o, o0), act
    aq, a_s, o = _row(cfg, "situglu", (1e7, 1e7))
    assert np.array_equal(a_s, as0)
    assert np.abs(_code_steps(aq, aq0, cfg.dispatch_fmt)).max() <= 1
    assert np.abs(o - o0).max() <= 1e-3 * np.abs(o0).max()


def _code_steps(a, b, fmt):
    """Signed code distance of two FP8 code arrays (codes ordered by value)."""
    def ordv(c):
        c = c.astype(np.int64)
        return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)
    return ordv(a) - ordv(b)


def test_activation_clamp_cases():
    """Clamp c: G_c = min(G, c), U_c = clip(U, -c, c).  For a c below every |G|
    and |U| the gated products reduce to constants times the signs of U:
    swiglu A = SiLU(c) * c * sign(U) where G > c; swiglustep A = min(SiLU(G), c)
    U_c; a clamp far above the data changes nothing."""
    cfg = synth.CONFIGS["tiny"].scaled(n=1)
    aq0, _, o0 = _row(cfg, "swiglu")
    aq1, _, o1 = _row(cfg, "swiglu", (1e30,))
    assert np.array_equal(aq0, aq1) and np.array_equal(o0, o1)
    # pin through the A8W8 formulas written with a tiny clamp: A = SiLU(min(G, c)) clip(U)
    c = 1e-3
    xq, xs, w1, s1, w2, s2 = _one_expert(cfg)
    xd = P.dequant_rows(xq[None], xs[None], cfg.dispatch_fmt)[0]
    hv = P.dequant_rows(w1, s1, cfg.weight_fmt) @ xd
    g, u = hv[:cfg.inter], hv[cfg.inter:]
    assert np.mean(np.abs(u) > c) > 0.9             # nearly every U clips to +-c
    gc = np.minimum(g, c)
    want = (gc * expit(gc) * np.clip(u, -c, c)).astype(np.float32).astype(np.float64)
    wq, ws = P.brute_mx_rows(want[None], cfg.dispatch_fmt)
    aq, a_s, _ = _row(cfg, "swiglu", (c,))
    assert np.array_equal(aq, wq[0]) and np.array_equal(a_s, ws[0])


def test_gelu_matches_tanh_form():
    """gelu: the README prints GELU(Z) = Z/2 (1 + tanh(sqrt(2/pi) (Z + 0.044715 Z^3)))
    = Z sigma(sqrt(8/pi) (...)).  The oracle evaluates the sigma form; the tanh
    form (numpy) must give the same quantised activation of the full 2I-wide
    Linear1 output, and GELU_tanh(1) = 0.84119199 (the approximation's value)."""
    cfg = synth.CONFIGS["tiny"].scaled(activation="gelu", act_params=(float(np.finfo(np.float32).max),))
    xq, xs, w1, s1, w2, s2 = _one_expert(cfg)
    assert w2.shape[1] == 2 * cfg.inter
    xd = P.dequant_rows(xq[None], xs[None], cfg.dispatch_fmt)[0]
    z = P.dequant_rows(w1, s1, cfg.weight_fmt) @ xd
    tanh_form = 0.5 * z * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (z + 0.044715 * z ** 3)))
    want = tanh_form.astype(np.float32).astype(np.float64)
    wq, ws = P.brute_mx_rows(want[None], cfg.dispatch_fmt)
    aq, a_s, o = oracle.expert_row(xq, xs, cfg.dispatch_fmt, w1, s1, w2, s2, cfg.weight_fmt, cfg.dispatch_fmt,
                                   activation="gelu", act_params=cfg.act_params)
    assert np.array_equal(a_s, ws[0])
    assert np.abs(_code_steps(aq, wq[0], cfg.dispatch_fmt)).max() <= 1
    assert abs(0.5 * (1 + np.tanh(np.sqrt(2 / np.pi) * 1.044715)) - 0.8411919906) < 1e-9


@pytest.mark.parametrize("routed,dispatch,shared_w,shared_x", [
    (P.E2M1, P.E2M1, P.E4M3, P.E4M3),    # A4W4-FP routed experts, A8W8-FP shared experts
    (P.E4M3, P.E4M3, P.E2M1, P.E2M1),    # A8W8-FP routed, A4W4-FP shared
    (P.E5M2, P.E5M2, P.E4M3, P.E4M3),    # E5M2 routed, E4M3 shared (activations differ too)
    (P.E2M1, P.E4M3, P.E2M1, P.E2M1),    # A8W4-FP routed, A4W4-FP shared
])
def test_mega_moe_shared_quant_type_matches_numpy(routed, dispatch, shared_w, shared_x):
    """Shared experts with their own input quantisation type (the MegaMoE
    parameter table's sharedExpertQuantOutDtype) and weight type."""
    cfg = synth.CONFIGS["tiny"].scaled(n=16, shared=2, weight_fmt=routed, dispatch_fmt=dispatch)
    x, ids, gate = synth.tokens_bf16(cfg), synth.topk_ids(cfg), synth.topk_weights(cfg)
    w = _weights(cfg)
    sh = _weights(cfg.scaled(weight_fmt=shared_w), shared=True)
    y, _ = oracle.mega_moe_tokens(x, ids, gate, *w, cfg.dispatch_fmt, cfg.weight_fmt, shared=sh,
                                  shared_w_fmt=shared_w, shared_x_fmt=shared_x)
    y_ref, _ = _numpy_grouped_moe(cfg, x, ids, gate, w, shared=sh, shared_fmt=shared_w, shared_xfmt=shared_x)
    assert np.max(np.abs(y - y_ref)) <= 1e-11 * np.abs(y_ref).max()
    # the shared experts' type matters: the routed type instead gives another Y
    y_same, _ = oracle.mega_moe_tokens(x, ids, gate, *w, cfg.dispatch_fmt, cfg.weight_fmt, shared=sh,
                                       shared_w_fmt=shared_w)
    assert np.max(np.abs(y_same - y_ref)) > 1e-6 * np.abs(y_ref).max()


@pytest.mark.parametrize("cfmt,kw", [(P.E5M2, {}), (P.E4M3, dict(shared=1, routing="zipf")),
                                     (P.E4M3, dict(weight_fmt=P.E2M1, dispatch_fmt=P.E2M1))])
def test_combine_quantisation_matches_numpy(cfmt, kw):
    """combineQuantMode 3 / 4: each routed row enters the combine as
    DQ_MX(Q_MX(bf16(O))) in that FP8 type; shared-expert rows stay local."""
    cfg = synth.CONFIGS["tiny"].scaled(n=16, **kw)
    x, ids, gate = synth.tokens_bf16(cfg), synth.topk_ids(cfg), synth.topk_weights(cfg)
    w = _weights(cfg)
    sh = _weights(cfg, shared=True) if cfg.shared else None
    y, _ = oracle.mega_moe_tokens(x, ids, gate, *w, cfg.dispatch_fmt, cfg.weight_fmt, shared=sh, combine_fmt=cfmt)
    y_ref, _ = _numpy_grouped_moe(cfg, x, ids, gate, w, shared=sh, combine_fmt=cfmt)
    assert np.max(np.abs(y - y_ref)) <= 1e-11 * np.abs(y_ref).max()
    y0, _ = oracle.mega_moe_tokens(x, ids, gate, *w, cfg.dispatch_fmt, cfg.weight_fmt, shared=sh)
    assert np.max(np.abs(y0 - y)) > 1e-4 * np.abs(y0).max()   # the quantisation shows


@pytest.mark.parametrize("kw", [{}, dict(weight_fmt=P.E2M1, dispatch_fmt=P.E2M1)])
def test_prequant_passthrough_equals_internal_quantisation(kw):
    """dispatchQuantMode = 0: X_hat, S_X given by the caller.  Passing the
    oracle's own Q_MX(x) must reproduce the internal-quantisation result."""
    cfg = synth.CONFIGS["tiny"].scaled(n=16, shared=1, **kw)
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    gate = synth.topk_weights(cfg)
    w = _weights(cfg)
    sh = _weights(cfg, shared=True)
    y0, _ = oracle.mega_moe_tokens(x, ids, gate, *w, cfg.dispatch_fmt, cfg.weight_fmt, shared=sh)
    xq, xs = oracle.mx_quantize(x, oracle.DT_BF16, cfg.dispatch_fmt)
    y1, _ = oracle.mega_moe_tokens(None, ids, gate, *w, cfg.dispatch_fmt, cfg.weight_fmt, shared=sh,
                                   x_prequant=(xq, xs))
    assert np.array_equal(y0, y1)


# ------------------------------------------- gated activations, every branch
def _gated_reference(g, u, act, params):
    """The MegaMoE README's "Activation function formulas", written out in
    numpy from the page (not from the oracle): sigma(z) = 1 / (1 + e^-z),
    SiLU(z) = z sigma(z), G_c = min(G, c), U_c = clip(U, -c, c), the clamp c
    +inf when not configured or 0; defaults from the activation_params row of
    the parameter table: alpha 1.702 and beta 1.0 for swigluoai, beta 1.0 for
    situglu, linear_beta not enabled."""
    p = list(params)
    c = np.inf
    if act in ("swiglu", "swiglustep", "swigluoai") and p and p[0] != 0.0:
        c = p[0]
    gc, uc = np.minimum(g, c), np.clip(u, -c, c)
    if act == "swiglu":
        return gc * expit(gc) * uc
    if act == "swiglustep":
        return np.minimum(g * expit(g), c) * uc
    if act == "swigluoai":
        alpha, beta = (p[1], p[2]) if len(p) == 3 else (1.702, 1.0)
        return gc * expit(alpha * gc) * (uc + beta)
    assert act == "situglu"
    beta = p[0] if p else 1.0
    lin = u if len(p) < 2 else p[1] * np.tanh(u / p[1])
    return beta * np.tanh(g / beta) * expit(g) * lin


# parameter sets chosen so that each branch's terms matter at the data's
# scale (|G|, |U| about 0.3 at scale shift 0 and about 2.5 at shift 3): the
# clamp cuts inside the data, alpha and beta are away from 1 and 0 (and
# negative), the situglu betas are small enough that tanh bends
GATED_PIN_CASES = [
    ("swiglustep", (0.3,)), ("swiglustep", (1.5,)), ("swiglustep", ()),
    ("swigluoai", ()), ("swigluoai", (0.0, 0.5, -0.5)), ("swigluoai", (0.4, 1.702, 1.0)),
    ("swigluoai", (2.0, 3.0, -0.5)), ("swigluoai", (0.0, 1.702, 1.0)),
    ("situglu", ()), ("situglu", (0.5,)), ("situglu", (2.0,)), ("situglu", (0.5, 0.3)), ("situglu", (2.0, 4.0)),
    ("swiglu", (0.3,)),
]


@pytest.mark.parametrize("shift", [0, 3])
@pytest.mark.parametrize("act,params", GATED_PIN_CASES)
def test_gated_activation_branches_match_the_formulas(act, params, shift):
    """Every gated branch of the oracle against the page's formula evaluated
    independently in numpy on the dequantised Linear1 output, for several
    tokens of one expert: A rounded to fp32, then MX-quantised by the
    brute-force quantiser; codes and scales must be identical.  The token
    scales are raised by 2^shift (exact: E8M0 codes + shift) so both the small
    and the saturating regimes of tanh, sigma and the clamp are reached."""
    cfg = synth.CONFIGS["tiny"].scaled(n=6)
    x = synth.tokens_bf16(cfg)
    xq, xs = oracle.mx_quantize(x, oracle.DT_BF16, cfg.dispatch_fmt)
    xs = (xs.astype(np.int32) + shift).astype(np.uint8)
    w1, s1 = oracle.quantized_weights(cfg, 1)
    w2, s2 = oracle.quantized_weights(cfg, 2)
    w1d = P.dequant_rows(w1[0], s1[0], cfg.weight_fmt)
    mism = 0
    for t in range(cfg.n):
        xd = P.dequant_rows(xq[t][None], xs[t][None], cfg.dispatch_fmt)[0]
        hv = w1d @ xd
        g, u = hv[:cfg.inter], hv[cfg.inter:]
        want = _gated_reference(g, u, act, params).astype(np.float32).astype(np.float64)
        wq, ws = P.brute_mx_rows(want[None], cfg.dispatch_fmt)
        aq, a_s, _ = oracle.expert_row(xq[t], xs[t], cfg.dispatch_fmt, w1[0], s1[0], w2[0], s2[0],
                                       cfg.weight_fmt, cfg.dispatch_fmt, activation=act, act_params=params)
        assert np.array_equal(a_s, ws[0]), (act, params, t)
        mism += int(np.count_nonzero(aq != wq[0]))
    assert mism == 0, (act, params, mism)


def test_gated_activation_defaults_are_the_parameter_table_values():
    """activation_params = [] means: no clamp, swigluoai alpha 1.702 and beta
    1.0, situglu beta 1.0 without linear_beta (parameter table).  The empty
    list must equal the explicit list of those values."""
    cfg = synth.CONFIGS["tiny"].scaled(n=1)
    fmax = float(np.finfo(np.float32).max)
    for act, explicit in (("swigluoai", (fmax, 1.702, 1.0)), ("situglu", (1.0,)), ("swiglustep", (fmax,))):
        aq0, as0, o0 = _row(cfg, act, ())
        aq1, as1, o1 = _row(cfg, act, explicit)
        assert np.array_equal(aq0, aq1) and np.array_equal(as0, as1) and np.array_equal(o0, o1), act
