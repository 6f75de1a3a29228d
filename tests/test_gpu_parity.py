"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Integer, index, FP8 and E8M0 outputs of routing / permute / quantisation
must be bit-exact.  MegaMoE's Y must satisfy the stated tolerance
(relative Frobenius error <= 5e-3, max abs error <= 2e-2 * max|Y|), and the
activation codes that follow GEMM1 may differ by one code step in at most
0.1 % of elements (the GEMM sums in fp32 on the tensor cores, the oracle in
double).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import routing_permute_mxfp8_gb300 as mm

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
Y_REL_FROB = 5e-3
Y_MAX_ABS = 2e-2
ACT_FRAC = 1e-3


def t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bf16(bits):
    return t(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def host(x):
    torch.cuda.synchronize()
    if x.dtype in (torch.bfloat16, torch.float16):
        return x.view(torch.int16).cpu().numpy().view(np.uint16)
    if x.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return x.view(torch.uint8).cpu().numpy()
    return x.cpu().numpy()


def zeros_err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


# ------------------------------------------------------------- routing + permute
ROUTE_CASES = [
    # n, h, e, k, quant, ids kind
    (1000, 512, 64, 8, -1, "distinct"),
    (1000, 512, 64, 8, 2, "distinct"),
    (1000, 512, 64, 8, 3, "distinct"),
    (1, 16, 1, 1, 3, "distinct"),
    (333, 160, 300, 7, 3, "distinct"),           # ragged H (5 groups), E not a power of two
    (2048, 48, 5, 3, 2, "any"),                  # repeated experts in a token, odd group count
    (4096, 1024, 2048, 4, 3, "distinct"),        # many experts
    (16384, 7168, 256, 8, -1, "distinct"),       # full routing workload, bf16 copy
    (16384, 7168, 256, 8, 3, "distinct"),        # full routing workload, MXFP8 E4M3
    (8388607, 16, 256, 2, 3, "any"),             # N*K = 16777214, the largest the sort limit allows
    # the automatic choice's boundaries: 131072 ids (one 16-CTA cluster) and
    # 131080 (the cooperative grid); 4096 keys (cluster, 8 warps per CTA)
    # and 4097 (grid)
    (16384, 32, 256, 8, 2, "any"),
    (16385, 32, 256, 8, 2, "any"),
    (300, 32, 4096, 12, -1, "distinct"),
    (300, 32, 4097, 12, 3, "distinct"),
    (16384, 7168, 256, 8, 9, "distinct"),        # full routing workload, MXFP4 E2M1 (V3 quantMode 9)
    (333, 160, 300, 7, 9, "any"),                # MXFP4, ragged H
]


def _ids(n, e, k, kind, seed):
    rng = np.random.default_rng(seed)
    if kind == "distinct":
        return np.argsort(rng.random((n, e)), axis=1)[:, :k].astype(np.int32)
    return rng.integers(0, e, (n, k)).astype(np.int32)


def _random_route_case(seed):
    rng = np.random.default_rng(2000 + seed)
    e = int(rng.integers(1, 600))
    return (int(rng.integers(1, 5000)), 16 * int(rng.integers(1, 80)), e, int(rng.integers(1, min(e, 16) + 1)),
            int(rng.choice([-1, 2, 3, 9])), str(rng.choice(["distinct", "any"])))


@pytest.mark.parametrize("seed", range(6))
def test_init_routing_random_shapes(seed):
    test_init_routing_bit_exact(*_random_route_case(seed))


@pytest.mark.parametrize("n,h,e,k,quant,kind", ROUTE_CASES)
def test_init_routing_bit_exact(n, h, e, k, quant, kind):
    cfg = synth.CONFIGS["routing"].scaled(n=n, h=h, e=e, k=k)
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg) if kind == "distinct" and (n, h) == (16384, 7168) else _ids(n, e, k, kind, n + e)
    err = zeros_err()
    for ttype in (0, 1):
        ex, exp_idx, tok, sc, srt = mm.mm_moe_init_routing(bf16(x), t(ids), e, quant, ttype, dev_err=err)
        r_srt, r_exp, r_cnt, bad = oracle.route(ids, e)
        assert bad == 0 and host(err)[0] == 0
        assert np.array_equal(host(srt), r_srt)
        assert np.array_equal(host(exp_idx), r_exp)
        assert np.array_equal(host(tok), np.cumsum(r_cnt) if ttype == 0 else r_cnt)
    fmt = {-1: -1, 2: 23, 3: 24, 9: 296}[quant]
    r_out, r_sc = oracle.permute(x, oracle.DT_BF16, k, r_srt, n * k, fmt=fmt)
    assert np.array_equal(host(ex), pack_fp4(r_out) if fmt == 296 else r_out)
    if quant != -1:
        assert np.array_equal(host(sc), r_sc)


ROUTE_PATHS = {"cluster": mm.ROUTE_CLUSTER, "grid": mm.ROUTE_GRID, "kernels": mm.ROUTE_KERNELS}

# MoeInitRoutingV3 with activeExpertRangeOptional: (n, h, e, k, start, end, quant, bad ids)
RANGE_CASES = [
    (300, 256, 16, 4, 4, 12, 3, False),
    (1000, 512, 64, 8, 63, 64, -1, False),      # one expert at the end of the ids
    (4096, 256, 256, 8, 32, 64, 2, True),       # an eighth of the experts; ids -1 and E mixed in
    (70000, 128, 512, 2, 0, 300, 3, False),     # above the cluster kernel's range
    (513, 384, 8, 8, 0, 8, -1, True),           # the full range through the v3 entry point
    (700, 256, 32, 4, 8, 24, 9, True),          # MXFP4 rows
]


@pytest.mark.parametrize("n,h,e,k,start,end,quant,bad", RANGE_CASES)
def test_init_routing_active_range(n, h, e, k, start, end, quant, bad):
    """Only ids in [start, end) are routed (computation step 6: availableIdxNum of
    them, in the first rows); counts / cumsum of the range's experts and the
    key_value form; ids outside [0, E) flagged, other ids left out silently."""
    cfg = synth.CONFIGS["routing"].scaled(n=n, h=h, e=e, k=k)
    x = synth.tokens_bf16(cfg)
    ids = _ids(n, e, k, "any", n + e + start)
    if bad:
        ids[1, 0], ids[n // 2, k - 1] = -1, e
    r_srt, r_exp, r_cnt, r_bad = oracle.route_range(ids, e, start, end)
    avail = int(((ids >= start) & (ids < end)).sum())
    fmt = {-1: -1, 2: 23, 3: 24, 9: 296}[quant]
    r_out, r_sc = oracle.permute(x, oracle.DT_BF16, k, r_srt, avail, fmt=fmt)
    if fmt == 296:
        r_out = pack_fp4(r_out)
    for ttype in (0, 1, 2):
        err = zeros_err()
        ex, exp_idx, tok, sc, srt = mm.mm_moe_init_routing(bf16(x), t(ids), e, quant, ttype,
                                                           active_expert_range=(start, end), dev_err=err)
        assert (host(err)[0] & 1) == (1 if r_bad else 0)
        assert np.array_equal(host(srt), r_srt)
        assert np.array_equal(host(exp_idx), r_exp)
        want = {0: np.cumsum(r_cnt), 1: r_cnt, 2: oracle.key_value_counts(r_cnt, start, e)}[ttype]
        assert np.array_equal(host(tok), want), ttype
        assert np.array_equal(host(ex)[:avail], r_out)
        if quant != -1:
            assert np.array_equal(host(sc)[:avail], r_sc)


@pytest.mark.parametrize("route_path", list(ROUTE_PATHS), indirect=True)
@pytest.mark.parametrize("case", [RANGE_CASES[i] for i in (0, 2, 4)])
def test_init_routing_active_range_every_path(route_path, case):
    test_init_routing_active_range(*case)


@pytest.fixture
def route_path(request):
    """Runs the test with one routing implementation forced, then restores the automatic choice."""
    mm.set_routing_path(ROUTE_PATHS[request.param])
    yield request.param
    mm.set_routing_path(mm.ROUTE_AUTO)


@pytest.mark.parametrize("route_path", list(ROUTE_PATHS), indirect=True)
@pytest.mark.parametrize("case", [ROUTE_CASES[i] for i in (1, 3, 4, 5, 6, 8, 10, 12, 15)])
def test_init_routing_every_path(route_path, case):
    """The cluster kernel, the cooperative grid launch and the four kernels
    give the oracle's bits (E up to 2048, ragged chunks, repeated ids)."""
    test_init_routing_bit_exact(*case)


@pytest.mark.parametrize("route_path", list(ROUTE_PATHS), indirect=True)
def test_routing_paths_out_of_range_and_empty(route_path):
    test_out_of_range_ids_are_left_out_and_flagged()
    test_empty_batch_writes_zero_counts(0)
    test_empty_batch_writes_zero_counts(1)


@pytest.mark.parametrize("route_path", list(ROUTE_PATHS), indirect=True)
@pytest.mark.parametrize("case", ["zipf_shared_e5m2_h512", "max_experts", "topk32_shared4"])
def test_mega_moe_every_routing_path(route_path, case):
    run_mega(synth.CONFIGS["tiny"].scaled(**MEGA_CASES[case]))


@pytest.mark.parametrize("dtype,idx64,num_out,quant,one_d", [
    (torch.bfloat16, False, 6, -1, False),
    (torch.float16, True, 0, 2, False),
    (torch.float16, False, -5, 3, False),
    (torch.float32, False, 100000, -1, False),
    (torch.bfloat16, True, None, 3, True),
    (torch.bfloat16, False, 0, 9, False),      # MXFP4 E2M1 (the article's quant_mode 9)
    (torch.float16, True, -7, 9, False),
])
def test_token_permute_bit_exact(dtype, idx64, num_out, quant, one_d, shape=None):
    n, h, e, k = shape if shape else (700, 256, 16, 1 if one_d else 4)
    rng = np.random.default_rng(9)
    xf = rng.standard_normal((n, h)).astype(np.float32)
    xt = torch.from_numpy(xf).to(dtype)
    ids = _ids(n, e, k, "distinct", 4)
    ids_t = t(ids.reshape(-1) if one_d else ids)
    if idx64:
        ids_t = ids_t.long()
    perm, sidx, sc = mm.mm_moe_token_permute(xt.to(DEV), ids_t, e, num_out_tokens=num_out, quant_mode=quant)
    r_srt, r_exp, _, _ = oracle.route(ids, e)
    m = n * k if not num_out else (min(num_out, n * k) if num_out > 0 else max(n * k + num_out, 0))
    assert perm.shape[0] == m and sidx.shape[0] == n * k
    assert np.array_equal(host(sidx), r_exp)
    src_dt = {torch.bfloat16: oracle.DT_BF16, torch.float16: oracle.DT_F16, torch.float32: oracle.DT_F32}[dtype]
    src = xt.view(torch.int16).numpy().view(np.uint16) if dtype != torch.float32 else xf
    fmt = {-1: -1, 2: 23, 3: 24, 9: 296}[quant]
    r_out, r_sc = oracle.permute(src, src_dt, k, r_srt, m, fmt=fmt)
    got = host(perm)
    if fmt == 296:
        assert got.shape == (m, h // 2) and tuple(sc.shape) == (m, (h + 63) // 64, 2)
        r_out = pack_fp4(r_out)
    assert np.array_equal(got.view(r_out.dtype) if fmt < 0 else got, r_out)
    if quant != -1:
        assert np.array_equal(host(sc).reshape(m, -1), r_sc)


@pytest.mark.parametrize("seed", range(6))
def test_token_permute_random_shapes(seed):
    rng = np.random.default_rng(3000 + seed)
    one_d = bool(rng.integers(0, 2))
    e = int(rng.integers(1, 300))
    k = 1 if one_d else int(rng.integers(1, min(e, 12) + 1))
    n = int(rng.integers(1, 3000))
    quant = int(rng.choice([-1, 2, 3, 9]))
    dtype = [torch.bfloat16, torch.float16, torch.float32][int(rng.integers(0, 2 if quant != -1 else 3))]
    h = 32 * int(rng.integers(1, 40)) if quant == 9 else 16 * int(rng.integers(1, 80))
    num_out = [None, 0, int(rng.integers(1, 2 * n * k)), -int(rng.integers(0, n * k + 5))][int(rng.integers(0, 4))]
    test_token_permute_bit_exact(dtype, bool(rng.integers(0, 2)), num_out, quant, one_d, shape=(n, h, e, k))


def test_out_of_range_ids_are_left_out_and_flagged():
    ids = np.array([[0, 5], [2, -1], [1, 0]], dtype=np.int32)
    x = synth.f32_to_bf16_bits(np.arange(3 * 32, dtype=np.float32).reshape(3, 32))
    err = zeros_err()
    ex, exp_idx, tok, _, srt = mm.mm_moe_init_routing(bf16(x), t(ids), 3, -1, 1, dev_err=err)
    r_srt, r_exp, r_cnt, bad = oracle.route(ids, 3)
    assert bad == 2
    assert host(err)[0] & 1
    assert np.array_equal(host(srt), r_srt)
    assert np.array_equal(host(exp_idx), r_exp)
    assert np.array_equal(host(tok), r_cnt)
    r_out, _ = oracle.permute(x, oracle.DT_BF16, 2, r_srt, 4)
    assert np.array_equal(host(ex)[:4], r_out)


@pytest.mark.parametrize("ttype", [0, 1])
def test_empty_batch_writes_zero_counts(ttype):
    """No rows (num_rows = 0, bs = 0): every expert's count, and the cumsum,
    is 0 (the histogram of an empty id list), so the count outputs are
    written even though nothing else is.  Called through the C ABI on
    buffers that hold junk beforehand."""
    L = mm.load()
    e = 16
    vp = lambda a: ctypes.c_void_p(a.data_ptr())
    dummy = torch.zeros(64, dtype=torch.uint8, device=DEV)
    tok = torch.full((e,), -7, dtype=torch.int64, device=DEV)
    st = L.mm_moe_init_routing(vp(dummy), 27, vp(dummy), 0, 64, 4, e, 3, ttype, vp(dummy), vp(dummy), vp(dummy),
                               vp(dummy), vp(tok), vp(dummy), 64, None, None)
    assert st == 0
    assert np.array_equal(host(tok), np.zeros(e, np.int64))
    cnt = torch.full((e,), -7, dtype=torch.int32, device=DEV)
    st = L.mm_mega_moe(vp(dummy), None, vp(dummy), vp(dummy), 0, vp(dummy), vp(dummy), vp(dummy), vp(dummy), 24, 0,
                       None, None, None, None, 24, 0, 0, 256, 2, e, 1, 128, 0, 4, 24, 0, 0, b"swiglu", None, 0,
                       vp(dummy), vp(cnt), None, None, None, None, None, vp(dummy), 64, None, None)
    assert st == 0
    assert np.array_equal(host(cnt), np.zeros(e, np.int32))


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """A wait that nothing completes ends after its limit with
    MM_DEVERR_TIMEOUT set, without a fault; the next MegaMoE call is exact."""
    err = zeros_err()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    mm.mm_selftest_wait_timeout(20_000_000, err)  # 20 ms
    e1.record()
    torch.cuda.synchronize()
    assert host(err)[0] & 4
    assert 19.0 <= e0.elapsed_time(e1) < 1000.0
    run_mega(synth.CONFIGS["tiny"])


# ---------------------------------------------------------------- MX quantiser
def pack_fp4(codes):
    """Oracle FP4 codes (one per byte) -> the library's packed bytes (element
    2i in bits 0-3, 2i+1 in bits 4-7)."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def gpu_codes(codes, fmt):
    return t(pack_fp4(codes) if fmt == 296 else codes)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("fmt", [23, 24, 296])
def test_mx_quantize_bit_exact(dtype, fmt):
    rng = np.random.default_rng(fmt)
    rows, cols = 513, 320
    x = rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-20, 12, (rows, 1)))
    x[0, :32] = 0.0
    x[1, :32] = -0.0
    x[2, 5] = 1e30 if dtype == torch.float32 else 3e4
    x[3, :] = 1e-41 if dtype == torch.float32 else 1e-7     # fp32 subnormals / tiny values
    x[4, 7] = -448.0 * 1.0001
    xt = torch.from_numpy(x.astype(np.float32)).to(dtype)
    q, s = mm.mm_mx_quantize(xt.to(DEV), fmt)
    src_dt = {torch.bfloat16: oracle.DT_BF16, torch.float16: oracle.DT_F16, torch.float32: oracle.DT_F32}[dtype]
    src = xt.view(torch.int16).numpy().view(np.uint16) if dtype != torch.float32 else xt.numpy()
    rq, rs = oracle.mx_quantize(src, src_dt, fmt, s_cols=s.shape[1])
    assert np.array_equal(host(s), rs)
    assert np.array_equal(host(q), pack_fp4(rq) if fmt == 296 else rq)


# -------------------------------------------------------------------- MegaMoE
def _weights(cfg, shared=False):
    w1, s1 = oracle.quantized_weights(cfg, 1, shared=shared)
    w2, s2 = oracle.quantized_weights(cfg, 2, shared=shared)
    return w1, s1, w2, s2


def _code_ord(c):
    c = c.astype(np.int32)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def check_act(aq_gpu, as_gpu, exp_idx, aq_ref, as_ref, tokens, k):
    """Activation codes of sampled tokens: scales equal and codes within one
    step, except in at most ACT_FRAC of the elements."""
    rows = exp_idx.reshape(-1, k)[tokens]                      # [T, K] sorted rows
    g = aq_gpu[rows]                                           # [T, K, I]
    gs = as_gpu[rows]                                          # [T, K, I/32]
    same_scale = np.repeat(gs == as_ref, 32, axis=-1)
    step = np.abs(_code_ord(g) - _code_ord(aq_ref))
    bad = (~same_scale) | (step > 1)
    diff = (step != 0) | (~same_scale)
    assert bad.mean() <= ACT_FRAC, (bad.mean(), diff.mean())
    assert diff.mean() <= ACT_FRAC, diff.mean()


def check_dispatch(xq_gpu, xs_gpu, x, cfg, r_srt, tokens=None):
    """Dispatched rows of a MegaMoE call (expert-sorted order) against
    oracle.permute with the dispatch format: codes and E8M0 scales identical.
    With sampled tokens only the rows of those tokens are compared (the
    oracle quantises every row; that part is cheap)."""
    q_ref, s_ref = oracle.permute(x, oracle.DT_BF16, cfg.k, r_srt, r_srt.size, cfg.dispatch_fmt)
    if cfg.dispatch_fmt == 296:   # A4W4-FP: the library's X_hat is packed FP4
        q_ref = pack_fp4(q_ref)
    rows = np.arange(r_srt.size) if tokens is None else np.nonzero(np.isin(r_srt // cfg.k, tokens))[0]
    assert np.array_equal(xq_gpu[rows], q_ref[rows])
    assert np.array_equal(xs_gpu[rows], s_ref[rows, :xs_gpu.shape[1]])


def check_y(y_gpu, y_ref):
    yg = y_gpu.astype(np.float64)
    rel = np.linalg.norm(yg - y_ref) / np.linalg.norm(y_ref)
    mx = np.abs(yg - y_ref).max() / np.abs(y_ref).max()
    assert rel <= Y_REL_FROB, rel
    assert mx <= Y_MAX_ABS, mx
    return rel, mx


def _sparse_weights(cfg, experts, shared=False):
    """Oracle-quantised weights of the listed experts; every other expert is
    all-zero (codes 0, scale code 127), which keeps full-size runs cheap to
    build while every checked token sees its real weights."""
    n_exp = cfg.shared if shared else cfg.e
    s1c, s2c = 2 * ((cfg.h + 63) // 64), 2 * ((cfg.act_width + 63) // 64)
    w1 = np.zeros((n_exp, 2 * cfg.inter, cfg.h), np.uint8)
    s1 = np.full((n_exp, 2 * cfg.inter, s1c), 127, np.uint8)
    w2 = np.zeros((n_exp, cfg.h, cfg.act_width), np.uint8)
    s2 = np.full((n_exp, cfg.h, s2c), 127, np.uint8)
    for e in experts:
        w1[e], s1[e] = oracle.mx_quantize(synth.weight_f32(cfg, 1, int(e), shared=shared), oracle.DT_F32,
                                          cfg.weight_fmt, s1c)
        w2[e], s2[e] = oracle.mx_quantize(synth.weight_f32(cfg, 2, int(e), shared=shared), oracle.DT_F32,
                                          cfg.weight_fmt, s2c)
    return w1, s1, w2, s2


def run_mega(cfg, tokens=None, layout=0, check_acts=True, sparse=False):
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    gate = synth.topk_weights(cfg)
    if sparse:
        needed = np.unique(ids[np.asarray(tokens)].reshape(-1))
        w1, s1, w2, s2 = _sparse_weights(cfg, needed)
        sh = _sparse_weights(cfg, range(cfg.shared), shared=True) if cfg.shared else None
    else:
        w1, s1, w2, s2 = _weights(cfg)
        sh = _weights(cfg, shared=True) if cfg.shared else None
    gt = bf16(gate) if gate.dtype == np.uint16 else t(gate)
    ws1, ws2 = t(s1), t(s2)
    if layout == 1:
        ws1 = mm.mm_prepare_weight_scales(ws1, cfg.h, 1)
        ws2 = mm.mm_prepare_weight_scales(ws2, cfg.act_width, 2)
    kw = {}
    if sh is not None:
        sw1, ss1, sw2, ss2 = gpu_codes(sh[0], cfg.weight_fmt), t(sh[1]), gpu_codes(sh[2], cfg.weight_fmt), t(sh[3])
        if layout == 1:
            ss1 = mm.mm_prepare_weight_scales(ss1, cfg.h, 1)
            ss2 = mm.mm_prepare_weight_scales(ss2, cfg.act_width, 2)
        kw = dict(shared_weight1=sw1, shared_weight2=sw2, shared_weight_scales1=ss1, shared_weight_scales2=ss2)
    err = zeros_err()
    y, counts, exp_idx, aq, a_s, xq, xs = mm.mm_mega_moe(
        bf16(x), t(ids), gt, gpu_codes(w1, cfg.weight_fmt), gpu_codes(w2, cfg.weight_fmt), ws1, ws2, cfg.e,
        weight_dtype=cfg.weight_fmt, weight_scale_layout=layout, activation=cfg.activation,
        activation_params=cfg.act_params, dispatch_quant_out_dtype=cfg.dispatch_fmt, dev_err=err,
        want_expanded_row_idx=True, want_act=True, want_dispatch=True, **kw)
    assert host(err)[0] == 0
    r_srt, r_exp, r_cnt, _ = oracle.route(ids, cfg.e)
    assert np.array_equal(host(counts), r_cnt.astype(np.int32))
    assert np.array_equal(host(exp_idx), r_exp)
    # stage 1 (dispatch): the X_hat rows and scales inside the step, bit-exact
    # against the oracle's permute + Q_MX in the dispatch format
    check_dispatch(host(xq), host(xs), x, cfg, r_srt, tokens)
    tok = np.arange(cfg.n) if tokens is None else np.asarray(tokens)
    y_ref, _, aq_ref, as_ref = oracle.mega_moe_tokens(x, ids, gate, w1, s1, w2, s2, cfg.dispatch_fmt,
                                                      cfg.weight_fmt, tokens=tok, shared=sh, want_act=True,
                                                      activation=cfg.activation, act_params=cfg.act_params)
    yg = host(y).view(np.uint16)
    yg = synth.bf16_bits_to_f32(yg)[tok]
    if check_acts:
        check_act(host(aq), host(a_s), r_exp, aq_ref, as_ref, tok, cfg.k)
    return check_y(yg, y_ref), host(y)


MEGA_CASES = {
    "tiny": dict(),
    "tiny_e5m2_zipf_bf16gate": dict(dispatch_fmt=23, routing="zipf", gate_dtype="bf16"),
    "tiny_e5m2_weights": dict(weight_fmt=23),
    "tiny_shared": dict(shared=1),
    "tiny_ragged": dict(n=37, e=5, k=3),
    "tiny_k1_e1": dict(n=200, e=1, k=1),
    "wide": dict(n=300, h=1024, inter=384, e=16, k=4),
    "h896_ragged_n": dict(n=256, h=896, inter=256, e=8, k=4, shared=1),   # last GEMM2 n tile half empty
    "zipf_shared_e5m2_h512": dict(n=300, h=512, inter=256, e=8, k=4, shared=1, routing="zipf", dispatch_fmt=23),
    "many_mtiles": dict(n=640, h=512, inter=512, e=4, k=2),
    # Zipf routing over 32 experts: one-tile experts beside experts with
    # several m tiles, so the tile order interleaves the two kinds
    "zipf_mixed_sizes": dict(n=1024, h=512, inter=256, e=32, k=4, routing="zipf"),
    # A8W4-FP: MXFP4 E2M1 weights (packed), MXFP8 E4M3 activations
    "a8w4_tiny": dict(weight_fmt=296, dispatch_fmt=24),
    "a8w4_shared_zipf": dict(n=300, h=512, inter=256, e=8, k=4, shared=1, routing="zipf", weight_fmt=296,
                             dispatch_fmt=24),
    "a8w4_e5m2_tokens": dict(n=256, h=896, inter=384, e=8, k=4, weight_fmt=296, dispatch_fmt=23),
    # A4W4-FP: MXFP4 E2M1 tokens and weights, A_hat MXFP8 E4M3 (GEMM2 A8W4)
    "a4w4_tiny": dict(weight_fmt=296, dispatch_fmt=296),
    "a4w4_shared_zipf_bf16gate": dict(n=300, h=512, inter=256, e=8, k=4, shared=1, routing="zipf", weight_fmt=296,
                                      dispatch_fmt=296, gate_dtype="bf16"),
    "a4w4_h896_ragged": dict(n=257, h=896, inter=384, e=8, k=4, weight_fmt=296, dispatch_fmt=296),
    "a4w4_gelu": dict(n=200, h=512, inter=256, e=8, k=4, activation="gelu", weight_fmt=296, dispatch_fmt=296,
                      act_params=(float(np.finfo(np.float32).max),)),
    "a4w4_swigluoai": dict(n=128, e=8, k=4, activation="swigluoai", act_params=(0.05, 1.5, 0.25), weight_fmt=296,
                           dispatch_fmt=296),
    "a4w4_small_seg_zipf": dict(n=300, h=256, inter=384, e=32, k=2, routing="zipf", weight_fmt=296, dispatch_fmt=296),
    # the README's other activations ("Activation function formulas") and clamps
    "swiglu_clamp": dict(n=128, e=8, k=4, act_params=(0.05,)),
    "swiglustep_clamp": dict(n=128, e=8, k=4, activation="swiglustep", act_params=(0.002,)),
    "swigluoai_default": dict(n=128, e=8, k=4, activation="swigluoai"),
    "swigluoai_params": dict(n=128, e=8, k=4, shared=1, activation="swigluoai", act_params=(0.05, 1.5, 0.25)),
    "situglu_beta": dict(n=128, e=8, k=4, activation="situglu", act_params=(0.5,)),
    "situglu_linear": dict(n=128, e=8, k=4, activation="situglu", act_params=(0.5, 0.3)),
    "gelu": dict(n=128, e=8, k=4, shared=1, activation="gelu", act_params=(float(np.finfo(np.float32).max),)),
    "gelu_a8w4": dict(n=200, h=512, inter=256, e=8, k=4, activation="gelu", weight_fmt=296,
                      act_params=(float(np.finfo(np.float32).max),)),
    # 1024 routed + 1 shared segments: the segment table leaves no shared
    # memory for GEMM2's output staging, so O rows are stored directly
    "many_experts": dict(n=256, h=256, inter=128, e=1024, k=8, shared=1),
    # the limits: top-K 32 with 4 shared experts (36 destinations and combine
    # terms per token), and 2048 routed experts + 4 shared segments
    "topk32_shared4": dict(n=96, h=256, inter=128, e=64, k=32, shared=4),
    "max_experts": dict(n=256, h=256, inter=128, e=2048, k=8, shared=4),
    # segments of 1 to 128 rows (one padded m tile) next to segments of two and
    # more tiles: every row count up to 128 and the step to two m tiles, FP8 and
    # FP4 weights, shared experts, gelu, both dispatch formats
    "small_seg_zipf_mixed": dict(n=400, h=512, inter=256, e=48, k=3, routing="zipf"),
    "small_seg_single_rows": dict(n=5, h=256, inter=128, e=8, k=1),
    "small_seg_128_rows": dict(n=128, h=384, inter=128, e=1, k=1, shared=1),
    "small_seg_129_rows": dict(n=129, h=384, inter=128, e=1, k=1, shared=1),
    "small_seg_112_rows_e5m2": dict(n=112, h=256, inter=256, e=1, k=1, dispatch_fmt=23),
    "small_seg_fp4_shared": dict(n=100, h=512, inter=256, e=16, k=4, shared=1, weight_fmt=296, dispatch_fmt=24),
    "small_seg_fp4_e5m2_zipf": dict(n=300, h=256, inter=384, e=32, k=2, routing="zipf", weight_fmt=296, dispatch_fmt=23),
    "small_seg_gelu_shared": dict(n=90, h=512, inter=256, e=8, k=3, shared=1, activation="gelu",
                             act_params=(float(np.finfo(np.float32).max),)),
    "small_seg_gelu_fp4_zipf": dict(n=200, h=256, inter=128, e=16, k=4, routing="zipf", weight_fmt=296, dispatch_fmt=24,
                               activation="gelu", act_params=(float(np.finfo(np.float32).max),)),
    "small_seg_swigluoai_h896": dict(n=70, h=896, inter=256, e=4, k=2, shared=2, activation="swigluoai",
                                act_params=(0.4, 1.702, 1.0)),
}


def _random_mega_cfg(seed):
    """A seeded random MegaMoE problem: shapes, routing, formats, shared
    experts and activation drawn independently (sizes small enough for the
    oracle to finish in seconds, large enough for several tiles)."""
    rng = np.random.default_rng(1000 + seed)
    e = int(rng.choice([1, 3, 8, 17, 40, 64]))
    k = int(rng.integers(1, min(e, 8) + 1))
    act = str(rng.choice(["swiglu", "swiglu", "swigluoai", "situglu", "swiglustep", "gelu"]))
    params = {"swiglu": (), "swigluoai": (), "situglu": (0.7,), "swiglustep": (0.5,),
              "gelu": (float(np.finfo(np.float32).max),)}[act]
    return synth.CONFIGS["tiny"].scaled(
        n=int(rng.integers(1, 400)), h=128 * int(rng.integers(1, 9)), inter=128 * int(rng.integers(1, 5)), e=e, k=k,
        routing=str(rng.choice(["uniform", "zipf"])), dispatch_fmt=int(rng.choice([23, 24])),
        weight_fmt=int(rng.choice([23, 24, 296])), gate_dtype=str(rng.choice(["fp32", "bf16"])),
        shared=int(rng.integers(0, 3)), activation=act, act_params=params, seed=seed)


@pytest.mark.parametrize("seed", range(10))
def test_mega_moe_random_shapes(seed):
    cfg = _random_mega_cfg(seed)
    if cfg.weight_fmt == 296:   # FP4 weights: A8W4-FP with either FP8 dispatch, or A4W4-FP
        cfg = cfg.scaled(dispatch_fmt=(23, 24, 296)[seed % 3])
    run_mega(cfg, layout=seed % 2)  # odd seeds: weight scales prepared once (mm_prepare_weight_scales)


@pytest.mark.parametrize("case", list(MEGA_CASES))
def test_mega_moe_small(case):
    cfg = synth.CONFIGS["tiny"].scaled(**MEGA_CASES[case])
    run_mega(cfg)


@pytest.mark.parametrize("fmts", [(24, 24), (296, 296)], ids=["a8w8", "a4w4"])
def test_mega_moe_prequant_passthrough(fmts):
    """dispatch_quant_mode 0: the caller's FP8 (or packed FP4) codes and E8M0
    scales are used as X_hat, S_X.  Feeding Q_MX(x) (oracle) gives the
    internal-quantisation result bit for bit, and matches the oracle's
    pass-through run."""
    wf, df = fmts
    cfg = synth.CONFIGS["tiny"].scaled(n=96, shared=1, routing="zipf", weight_fmt=wf, dispatch_fmt=df)
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    gate = synth.topk_weights(cfg)
    w1, s1, w2, s2 = _weights(cfg)
    sh = _weights(cfg, shared=True)
    xq, xs = oracle.mx_quantize(x, oracle.DT_BF16, cfg.dispatch_fmt)
    kw = dict(shared_weight1=gpu_codes(sh[0], wf), shared_weight_scales1=t(sh[1]),
              shared_weight2=gpu_codes(sh[2], wf), shared_weight_scales2=t(sh[3]),
              dispatch_quant_out_dtype=cfg.dispatch_fmt, weight_dtype=wf)
    err = zeros_err()
    g1, g2 = gpu_codes(w1, wf), gpu_codes(w2, wf)
    y0 = mm.mm_mega_moe(bf16(x), t(ids), t(gate), g1, g2, t(s1), t(s2), cfg.e, dev_err=err, **kw)[0]
    y1 = mm.mm_mega_moe(gpu_codes(xq, df), t(ids), t(gate), g1, g2, t(s1), t(s2), cfg.e, dev_err=err,
                        dispatch_quant_mode=0, x_scales=t(xs), **kw)[0]
    assert host(err)[0] == 0
    assert np.array_equal(host(y0).view(np.uint16), host(y1).view(np.uint16))
    y_ref, _ = oracle.mega_moe_tokens(None, ids, gate, w1, s1, w2, s2, cfg.dispatch_fmt, cfg.weight_fmt,
                                      shared=sh, x_prequant=(xq, xs))
    check_y(synth.bf16_bits_to_f32(host(y1).view(np.uint16)), y_ref)


@pytest.mark.parametrize("routed_fmt,shared_fmt,dispatch", [(296, 24, 24), (24, 296, 24), (23, 24, 24),
                                                            (296, 24, 296)])
def test_mega_moe_shared_weight_type_differs(routed_fmt, shared_fmt, dispatch):
    """Routed and shared experts with different weight types (the shared
    expert's own MMA format), e.g. FP4 routed experts beside an FP8 shared one;
    the last case dispatches FP4 tokens (A4W4-FP) into FP8 shared weights."""
    cfg = synth.CONFIGS["tiny"].scaled(n=128, e=8, k=4, shared=2, weight_fmt=routed_fmt, dispatch_fmt=dispatch)
    cfg_sh = cfg.scaled(weight_fmt=shared_fmt)
    x, ids, gate = synth.tokens_bf16(cfg), synth.topk_ids(cfg), synth.topk_weights(cfg)
    w1, s1, w2, s2 = _weights(cfg)
    sh = _weights(cfg_sh, shared=True)
    err = zeros_err()
    y, counts = mm.mm_mega_moe(
        bf16(x), t(ids), t(gate), gpu_codes(w1, routed_fmt), gpu_codes(w2, routed_fmt), t(s1), t(s2), cfg.e,
        weight_dtype=routed_fmt, dispatch_quant_out_dtype=cfg.dispatch_fmt, dev_err=err,
        shared_weight1=gpu_codes(sh[0], shared_fmt), shared_weight_scales1=t(sh[1]),
        shared_weight2=gpu_codes(sh[2], shared_fmt), shared_weight_scales2=t(sh[3]), shared_weight_dtype=shared_fmt)
    assert host(err)[0] == 0
    y_ref, _ = oracle.mega_moe_tokens(x, ids, gate, w1, s1, w2, s2, cfg.dispatch_fmt, routed_fmt, shared=sh,
                                      shared_w_fmt=shared_fmt)
    check_y(synth.bf16_bits_to_f32(host(y).view(np.uint16)), y_ref)


@pytest.mark.parametrize("routed,dispatch,shared_w,shared_x,act", [
    (296, 296, 24, 24, "swiglu"),     # A4W4-FP routed experts, A8W8-FP E4M3 shared experts
    (24, 24, 296, 296, "swiglu"),     # A8W8-FP routed, A4W4-FP shared
    (23, 23, 24, 24, "swiglu"),       # E5M2 routed, E4M3 shared: A_hat types differ too
    (24, 24, 24, 23, "gelu"),         # E4M3 routed, E5M2 shared, gelu
    (296, 24, 296, 296, "swigluoai"),  # A8W4-FP routed, A4W4-FP shared
])
def test_mega_moe_shared_quant_type(routed, dispatch, shared_w, shared_x, act):
    """Shared experts with their own input quantisation type (the MegaMoE
    parameter table's sharedExpertQuantOutDtype): the routed rows' X_hat
    bit-exact, routed A_hat codes within one step, Y against the oracle."""
    params = (float(np.finfo(np.float32).max),) if act == "gelu" else ()
    cfg = synth.CONFIGS["tiny"].scaled(n=160, h=512, inter=256, e=8, k=3, shared=2, routing="zipf",
                                       weight_fmt=routed, dispatch_fmt=dispatch, activation=act, act_params=params)
    x, ids, gate = synth.tokens_bf16(cfg), synth.topk_ids(cfg), synth.topk_weights(cfg)
    w1, s1, w2, s2 = _weights(cfg)
    sh = _weights(cfg.scaled(weight_fmt=shared_w), shared=True)
    err = zeros_err()
    y, counts, exp_idx, aq, a_s, xq, xs = mm.mm_mega_moe(
        bf16(x), t(ids), t(gate), gpu_codes(w1, routed), gpu_codes(w2, routed), t(s1), t(s2), cfg.e,
        weight_dtype=routed, dispatch_quant_out_dtype=dispatch, shared_expert_quant_out_dtype=shared_x,
        shared_weight1=gpu_codes(sh[0], shared_w), shared_weight_scales1=t(sh[1]),
        shared_weight2=gpu_codes(sh[2], shared_w), shared_weight_scales2=t(sh[3]), shared_weight_dtype=shared_w,
        activation=act, activation_params=params, dev_err=err, want_expanded_row_idx=True, want_act=True,
        want_dispatch=True)
    assert host(err)[0] == 0
    r_srt, r_exp, r_cnt, _ = oracle.route(ids, cfg.e)
    assert np.array_equal(host(counts), r_cnt.astype(np.int32))
    check_dispatch(host(xq), host(xs), x, cfg, r_srt)
    y_ref, _, aq_ref, as_ref = oracle.mega_moe_tokens(x, ids, gate, w1, s1, w2, s2, dispatch, routed, shared=sh,
                                                      shared_w_fmt=shared_w, shared_x_fmt=shared_x, want_act=True,
                                                      activation=act, act_params=params)
    check_act(host(aq), host(a_s), r_exp, aq_ref, as_ref, np.arange(cfg.n), cfg.k)
    check_y(synth.bf16_bits_to_f32(host(y).view(np.uint16)), y_ref)


@pytest.mark.parametrize("kw", [
    dict(shared=1, n=96),
    # gelu reads W1's scale tiles block by block; with I / 128 odd, one GEMM1
    # tile's two blocks straddle the last gate pair and the first up pair
    dict(shared=1, n=96, inter=384, activation="gelu", act_params=(float(np.finfo(np.float32).max),)),
    dict(n=128, inter=384, activation="gelu", act_params=(float(np.finfo(np.float32).max),), weight_fmt=296,
         dispatch_fmt=24),
], ids=["swiglu", "gelu_odd_pairs", "gelu_a8w4_odd_pairs"])
def test_mega_moe_prepared_scales_identical(kw):
    cfg = synth.CONFIGS["tiny"].scaled(**kw)
    _, y0 = run_mega(cfg, layout=0)
    _, y1 = run_mega(cfg, layout=1)
    assert np.array_equal(y0, y1)


def test_mega_moe_qwen3_shape_sampled():
    cfg = synth.CONFIGS["qwen3"].scaled(n=512)
    run_mega(cfg, tokens=np.arange(0, 512, 7))


# Full-size workloads in the launch configuration the benchmark times: the
# routing outputs are checked in full, Y and the activation codes on a token
# sample the oracle evaluates one token at a time.
@pytest.mark.slow
def test_mega_moe_qwen3_full_size():
    cfg = synth.CONFIGS["qwen3"]
    run_mega(cfg, tokens=np.linspace(0, cfg.n - 1, 40).astype(np.int64), layout=1)


@pytest.mark.slow
def test_mega_moe_dsv3_prefill_full_size():
    cfg = synth.CONFIGS["dsv3_prefill"]
    run_mega(cfg, tokens=np.array([0, 1, 777, 2048, 4095, 5000, 6001, 7333, 8000, 8191]), layout=1, sparse=True)


@pytest.mark.slow
def test_mega_moe_dsv3_decode_full_size():
    cfg = synth.CONFIGS["dsv3_decode"]
    run_mega(cfg, tokens=np.array([0, 5, 17, 63, 64, 100, 126, 127]), layout=1, sparse=True)


@pytest.mark.slow
def test_mega_moe_dsv3_prefill_a8w4_full_size():
    """A8W4-FP (MXFP4 weights, MXFP8 E4M3 activations) at the DeepSeek-V3 prefill shape."""
    cfg = synth.CONFIGS["dsv3_prefill"].scaled(weight_fmt=296, dispatch_fmt=24)
    run_mega(cfg, tokens=np.array([0, 3, 1500, 4096, 7000, 8191]), layout=1, sparse=True)


@pytest.mark.slow
def test_mega_moe_dsv3_prefill_a4w4_full_size():
    """A4W4-FP (MXFP4 tokens and weights, MXFP8 E4M3 activation) at the DeepSeek-V3 prefill shape."""
    cfg = synth.CONFIGS["dsv3_prefill"].scaled(weight_fmt=296, dispatch_fmt=296)
    run_mega(cfg, tokens=np.array([0, 2, 1501, 4097, 7001, 8191]), layout=1, sparse=True)


@pytest.mark.slow
def test_mega_moe_dsv3_decode_a4w4_full_size():
    """A4W4-FP at the decode shape, with its shared expert."""
    cfg = synth.CONFIGS["dsv3_decode"].scaled(weight_fmt=296, dispatch_fmt=296)
    run_mega(cfg, tokens=np.array([0, 9, 64, 127]), layout=1, sparse=True)


@pytest.mark.slow
def test_mega_moe_dsv3_decode_gelu_full_size():
    """gelu (whole 2I-wide Linear1 output) with a shared expert at the decode shape."""
    cfg = synth.CONFIGS["dsv3_decode"].scaled(activation="gelu", act_params=(float(np.finfo(np.float32).max),))
    run_mega(cfg, tokens=np.array([0, 31, 64, 127]), layout=1, sparse=True)


def test_mega_moe_back_to_back_calls_share_a_workspace():
    """Calls enqueued back to back on one stream, one workspace, no host
    synchronisation between them: each kernel starts early (programmatic
    dependent launch) but reads an earlier kernel's output only after that
    kernel has finished, so every call gives the bits it gives alone."""
    cfgs = [synth.CONFIGS["tiny"].scaled(**MEGA_CASES[c]) for c in ("zipf_shared_e5m2_h512", "wide", "tiny_shared")]
    h, inter = 1024, 512
    cfgs = [c.scaled(h=h, inter=inter, dispatch_fmt=24, weight_fmt=24) for c in cfgs]
    inputs = []
    for c in cfgs:
        x, ids, gate = bf16(synth.tokens_bf16(c)), t(synth.topk_ids(c)), t(synth.topk_weights(c))
        w = [t(a) for a in _weights(c)]
        sh = [t(a) for a in _weights(c, shared=True)] if c.shared else None
        kw = dict(shared_weight1=sh[0], shared_weight_scales1=sh[1], shared_weight2=sh[2],
                  shared_weight_scales2=sh[3]) if sh else {}
        inputs.append((c, x, ids, gate, w, kw))
    need = max(mm.mm_mega_moe_workspace_size(c.n, c.h, c.k, c.e, c.inter, c.shared, 0) for c in cfgs)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    alone = []
    for c, x, ids, gate, w, kw in inputs:
        alone.append(host(mm.mm_mega_moe(x, ids, gate, w[0], w[2], w[1], w[3], c.e, workspace=ws, **kw)[0]).copy())
    ys = [torch.empty((c.n, c.h), dtype=torch.bfloat16, device=DEV) for c in cfgs]
    for rep in range(3):
        for (c, x, ids, gate, w, kw), y in zip(inputs, ys):
            mm.mm_mega_moe(x, ids, gate, w[0], w[2], w[1], w[3], c.e, workspace=ws, out=y, **kw)
    torch.cuda.synchronize()
    for y, a in zip(ys, alone):
        assert np.array_equal(host(y), a)


@pytest.mark.slow
def test_mega_moe_full_size_repeatable_back_to_back():
    """The DeepSeek-V3-shaped prefill step (Zipf routing, E5M2 dispatch) run
    24 times back to back on one stream and one workspace, into three
    rotating outputs, without host synchronisation: every run gives the same
    bits (deterministic kernels, no race between a kernel's early launch and
    its predecessor's writes)."""
    cfg = synth.CONFIGS["dsv3_prefill"]
    gen = torch.Generator(device=DEV)
    gen.manual_seed(3)
    w = []
    for n_out, k_red in ((2 * cfg.inter, cfg.h), (cfg.h, cfg.inter)):
        q, sc = mm.mm_mx_quantize(torch.randn((cfg.e * n_out, k_red), generator=gen, device=DEV) * 0.02, 24,
                                  scale_cols=k_red // 32)
        w += [q.view(cfg.e, n_out, k_red), mm.mm_prepare_weight_scales(sc.view(cfg.e, n_out, k_red // 32), k_red,
                                                                       1 if n_out == 2 * cfg.inter else 2)]
    x, ids = bf16(synth.tokens_bf16(cfg)), t(synth.topk_ids(cfg))
    gate = bf16(synth.topk_weights(cfg))
    ws = torch.empty(mm.mm_mega_moe_workspace_size(cfg.n, cfg.h, cfg.k, cfg.e, cfg.inter, 0, mm.WSCALE_PREPARED),
                     dtype=torch.uint8, device=DEV)
    ys = [torch.empty((cfg.n, cfg.h), dtype=torch.bfloat16, device=DEV) for _ in range(3)]
    err = zeros_err()
    ref = None
    for rnd in range(8):
        for y in ys:
            mm.mm_mega_moe(x, ids, gate, w[0], w[2], w[1], w[3], cfg.e, weight_scale_layout=mm.WSCALE_PREPARED,
                           dispatch_quant_out_dtype=23, workspace=ws, out=y, dev_err=err)
        torch.cuda.synchronize()
        for y in ys:
            h = host(y)
            if ref is None:
                ref = h.copy()
            assert np.array_equal(h, ref), rnd
    assert host(err)[0] == 0


@pytest.mark.parametrize("route_path", ["cluster", "kernels"], indirect=True)
def test_mega_moe_in_cuda_graph(route_path):
    """The whole call captured in a CUDA graph (caller's workspace and
    output; routing as one cluster launch, or as its four ordinary kernels)
    replays to the same Y bits as a direct call."""
    cfg = synth.CONFIGS["tiny"].scaled(n=96, shared=1)
    x, ids, gate = bf16(synth.tokens_bf16(cfg)), t(synth.topk_ids(cfg)), t(synth.topk_weights(cfg))
    w1, s1, w2, s2 = (t(a) for a in _weights(cfg))
    sh = [t(a) for a in _weights(cfg, shared=True)]
    kw = dict(shared_weight1=sh[0], shared_weight_scales1=sh[1], shared_weight2=sh[2], shared_weight_scales2=sh[3])
    ws = torch.empty(mm.mm_mega_moe_workspace_size(cfg.n, cfg.h, cfg.k, cfg.e, cfg.inter, cfg.shared, 0),
                     dtype=torch.uint8, device=DEV)
    y = torch.empty((cfg.n, cfg.h), dtype=torch.bfloat16, device=DEV)
    y0 = mm.mm_mega_moe(x, ids, gate, w1, w2, s1, s2, cfg.e, workspace=ws, **kw)[0].clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        mm.mm_mega_moe(x, ids, gate, w1, w2, s1, s2, cfg.e, workspace=ws, out=y, **kw)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    y.zero_()
    with torch.cuda.graph(graph):
        mm.mm_mega_moe(x, ids, gate, w1, w2, s1, s2, cfg.e, workspace=ws, out=y, **kw)
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(host(y), host(y0))


def test_mega_moe_out_of_range_ids_left_out():
    """An id outside [0, E) is flagged and its term leaves Y: the reference
    gives that term weight 0 (on a valid, unused expert) in the oracle."""
    cfg = synth.CONFIGS["tiny"].scaled(n=96, shared=1)
    x, gate = synth.tokens_bf16(cfg), synth.topk_weights(cfg)
    ids = synth.topk_ids(cfg)
    bad = [(5, 1, cfg.e), (7, 0, -1), (40, 1, 1 << 20)]
    ids_ref, gate_ref = ids.copy(), gate.copy()
    for i, kk, v in bad:
        ids[i, kk] = v
        ids_ref[i, kk] = next(e for e in range(cfg.e) if e not in ids_ref[i])
        gate_ref[i, kk] = 0.0
    w1, s1, w2, s2 = _weights(cfg)
    sh = _weights(cfg, shared=True)
    err = zeros_err()
    y, counts = mm.mm_mega_moe(bf16(x), t(ids), t(gate), t(w1), t(w2), t(s1), t(s2), cfg.e, dev_err=err,
                               shared_weight1=t(sh[0]), shared_weight_scales1=t(sh[1]), shared_weight2=t(sh[2]),
                               shared_weight_scales2=t(sh[3]))
    assert host(err)[0] & 1
    _, _, r_cnt, n_bad = oracle.route(ids, cfg.e)
    assert n_bad == len(bad)
    assert np.array_equal(host(counts), r_cnt.astype(np.int32))
    y_ref, _ = oracle.mega_moe_tokens(x, ids_ref, gate_ref, w1, s1, w2, s2, cfg.dispatch_fmt, cfg.weight_fmt,
                                      shared=sh)
    check_y(synth.bf16_bits_to_f32(host(y).view(np.uint16)), y_ref)


def test_mega_moe_duplicate_ids_flagged():
    cfg = synth.CONFIGS["tiny"]
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    ids[3, 1] = ids[3, 0]
    gate = synth.topk_weights(cfg)
    w1, s1, w2, s2 = _weights(cfg)
    err = zeros_err()
    mm.mm_mega_moe(bf16(x), t(ids), t(gate), t(w1), t(w2), t(s1), t(s2), cfg.e, dev_err=err)
    assert host(err)[0] & 2


# ------------------------------------------------------- expert parallelism
@pytest.mark.parametrize("route_path", list(ROUTE_PATHS), indirect=True)
def test_ep_dispatch_every_routing_path(route_path):
    test_ep_dispatch_bit_exact(4, 24)


@pytest.mark.parametrize("w,fmt", [(1, 24), (2, 23), (4, 24), (16, 23), (4, 296)])
def test_ep_dispatch_bit_exact(w, fmt):
    """mm_moe_ep_dispatch against the oracle: the stable sort by destination
    rank id // (E/W) (the routing of MoeInitRoutingV3 on rank keys), Q_MX of
    every token in the send order, the local expert ids, the per-rank counts
    and the scatter index."""
    cfg = synth.CONFIGS["tiny"].scaled(n=300, h=512, e=16, k=4, routing="zipf")
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    el = cfg.e // w
    err = zeros_err()
    sx, ss, se, cnt, ei = mm.mm_moe_ep_dispatch(bf16(x), t(ids), cfg.e, w, fmt, dev_err=err)
    assert host(err)[0] == 0
    srt, exp, ocnt, bad = oracle.route((ids // el).astype(np.int32), w)
    q, sc = oracle.permute(x, oracle.DT_BF16, cfg.k, srt, srt.size, fmt)
    assert np.array_equal(host(cnt), ocnt)
    assert np.array_equal(host(ei), exp)
    assert np.array_equal(host(se), ids.reshape(-1)[srt] % el)
    assert np.array_equal(host(sx), pack_fp4(q) if fmt == 296 else q)
    assert np.array_equal(host(ss), sc[:, :cfg.h // 32])


@pytest.mark.slow
@pytest.mark.parametrize("fmt", [23, 296])
def test_ep_dispatch_full_size(fmt):
    """mm_moe_ep_dispatch at the DeepSeek-V3 prefill batch of one source rank
    (8192 tokens, hidden 7168, 256 experts, top-K 8, Zipf routing) over 8
    ranks, with E5M2 rows and with packed FP4 rows (A4W4-FP): counts, scatter
    index, local expert ids, codes and scales of all 65536 rows bit-exact
    against the oracle's routing on rank keys and its Q_MX."""
    cfg = synth.CONFIGS["dsv3_prefill"].scaled(dispatch_fmt=fmt)
    w = 8
    el = cfg.e // w
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    err = zeros_err()
    sx, ss, se, cnt, ei = mm.mm_moe_ep_dispatch(bf16(x), t(ids), cfg.e, w, fmt, dev_err=err)
    assert host(err)[0] == 0
    srt, exp, ocnt, bad = oracle.route((ids // el).astype(np.int32), w)
    assert bad == 0
    assert np.array_equal(host(cnt), ocnt)
    assert np.array_equal(host(ei), exp)
    assert np.array_equal(host(se), ids.reshape(-1)[srt] % el)
    q, sc = oracle.permute(x, oracle.DT_BF16, cfg.k, srt, srt.size, fmt)
    assert np.array_equal(host(ss), sc[:, :cfg.h // 32])
    assert np.array_equal(host(sx), pack_fp4(q) if fmt == 296 else q)


@pytest.mark.slow
@pytest.mark.parametrize("row_fmt", [27, 24])
def test_ep_combine_full_size(row_fmt):
    """mm_moe_combine at the DeepSeek-V3 prefill batch (8192 tokens, top-K 8,
    hidden 7168, bf16 gates, one block per token as in the step), with the
    returned rows as bf16 or as MXFP8 E4M3 codes and E8M0 scales from the
    oracle's Q_MX (combineQuantMode 4), picked by a scatter index that leaves
    some terms out (-1).  Sampled tokens against the fp64 sum of the oracle's
    row values, within half a bf16 step of the result plus the fp32
    accumulation bound (the fp32 order itself is checked bit for bit at small
    sizes)."""
    cfg = synth.CONFIGS["dsv3_prefill"]
    n, k, h = cfg.n, cfg.k, cfg.h
    nrows = 6000
    rng = np.random.default_rng(31)
    rows = (rng.standard_normal((nrows, h), dtype=np.float32) *
            np.exp2(rng.integers(-6, 6, (nrows, 1))).astype(np.float32))
    idx = rng.integers(-1, nrows, size=n * k).astype(np.int32)
    gate = synth.topk_weights(cfg)
    gw = synth.bf16_bits_to_f32(gate).reshape(n, k).astype(np.float64)
    if row_fmt == 27:
        rb = torch.from_numpy(rows).to(torch.bfloat16)
        vals = rb.float().numpy().astype(np.float64)
        y = mm.mm_moe_combine(rb.to(DEV), t(idx), bf16(gate))
    else:
        q, sc = oracle.mx_quantize(rows, oracle.DT_F32, row_fmt, s_cols=h // 32)
        tab = np.array([oracle.fp8_value(c, row_fmt) for c in range(256)])
        vals = tab[q] * np.exp2(np.repeat(sc.astype(np.float64) - 127.0, 32, axis=1))
        y = mm.mm_moe_combine(t(q), t(idx), bf16(gate), expert_scales=t(sc), expert_rows_dtype=row_fmt)
    yv = synth.bf16_bits_to_f32(host(y).view(np.uint16)).astype(np.float64)
    ix = idx.reshape(n, k)
    for i in (0, 1, 777, 2048, 4095, 5000, 7333, 8191):
        ok = ix[i] >= 0
        terms = gw[i, ok, None] * vals[ix[i, ok]]
        ref = terms.sum(axis=0)
        bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -20 * np.abs(terms).sum(axis=0)
        assert np.all(np.abs(yv[i] - ref) <= bound), i


@pytest.mark.parametrize("case", [
    dict(n=700, h=512, inter=256, e=8, k=1, routing="zipf"),
    dict(n=300, h=896, inter=384, e=5, k=1, weight_fmt=296, dispatch_fmt=23),
    dict(n=200, h=512, inter=256, e=16, k=1, activation="gelu", act_params=(float(np.finfo(np.float32).max),)),
    dict(n=300, h=512, inter=256, e=8, k=1, routing="zipf", weight_fmt=296, dispatch_fmt=296),   # A4W4-FP rows
])
def test_expert_ffn_equals_mega_moe_top1(case):
    """mm_moe_expert_ffn (the expert side of expert parallelism: GEMM2 writes
    each received row's result at the row's own position, no combine pass)
    gives mm_mega_moe's bits for the same rows at top-K 1 with weight 1 and
    pass-through quantisation, and the oracle's Y within tolerance."""
    cfg = synth.CONFIGS["tiny"].scaled(**case)
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    w1, s1, w2, s2 = _weights(cfg)
    fmt = cfg.dispatch_fmt
    xq, xs = oracle.mx_quantize(x, oracle.DT_BF16, fmt)   # the received rows: FP8 (FP4) codes + E8M0 scales
    xq, xs = gpu_codes(xq, fmt), t(xs)
    ids1 = t(ids.reshape(cfg.n))
    err = zeros_err()
    out, cnt = mm.mm_moe_expert_ffn(xq, xs, ids1, gpu_codes(w1, cfg.weight_fmt), gpu_codes(w2, cfg.weight_fmt), t(s1),
                                    t(s2), cfg.e, x_dtype=fmt, weight_dtype=cfg.weight_fmt,
                                    activation=cfg.activation, activation_params=cfg.act_params, dev_err=err)
    ones = torch.ones((cfg.n, 1), dtype=torch.float32, device=DEV)
    y, cnt2 = mm.mm_mega_moe(xq, ids1.view(cfg.n, 1), ones, gpu_codes(w1, cfg.weight_fmt), gpu_codes(w2, cfg.weight_fmt),
                             t(s1), t(s2), cfg.e, weight_dtype=cfg.weight_fmt, dispatch_quant_mode=0,
                             dispatch_quant_out_dtype=fmt, x_scales=xs, activation=cfg.activation,
                             activation_params=cfg.act_params)
    assert host(err)[0] == 0
    assert np.array_equal(host(out), host(y))
    assert np.array_equal(host(cnt), host(cnt2))
    assert np.array_equal(host(cnt), np.bincount(ids.reshape(-1), minlength=cfg.e))
    y_ref, _ = oracle.mega_moe_tokens(x, ids, np.ones((cfg.n, 1), np.float32), w1, s1, w2, s2, fmt, cfg.weight_fmt,
                                      activation=cfg.activation, act_params=cfg.act_params)
    check_y(synth.bf16_bits_to_f32(host(out).view(np.uint16)), y_ref)


@pytest.mark.slow
def test_expert_ffn_full_size_equals_mega_moe_top1():
    """The expert side of expert parallelism at the size one rank of an
    8-way DeepSeek-V3 prefill receives (16384 rows, hidden 7168,
    intermediate 2048, 32 local experts with Zipf-skewed loads, E5M2 rows,
    prepared weight scales): bit-identical to mm_mega_moe at top-K 1.
    Weights are drawn on the GPU (any values serve for bit-identity; the
    oracle comparison runs at the small sizes above)."""
    m, h, inter, e = 16384, 7168, 2048, 32
    gen = torch.Generator(device=DEV)
    gen.manual_seed(5)
    w = []
    for n_out, k_red in ((2 * inter, h), (h, inter)):
        q, sc = mm.mm_mx_quantize(torch.randn((e * n_out, k_red), generator=gen, device=DEV) * 0.02, 24,
                                  scale_cols=k_red // 32)
        w += [q.view(e, n_out, k_red), sc.view(e, n_out, k_red // 32)]
    p1 = mm.mm_prepare_weight_scales(w[1], h, 1)
    p2 = mm.mm_prepare_weight_scales(w[3], inter, 2)
    xq, xs = mm.mm_mx_quantize(torch.randn((m, h), generator=gen, device=DEV), 23, scale_cols=h // 32)
    rng = np.random.default_rng(11)
    pz = 1.0 / np.arange(1, e + 1)
    ids = t(rng.permutation(e)[rng.choice(e, m, p=pz / pz.sum())].astype(np.int32))
    err = zeros_err()
    out, cnt = mm.mm_moe_expert_ffn(xq, xs, ids, w[0], w[2], p1, p2, e, x_dtype=23,
                                    weight_scale_layout=mm.WSCALE_PREPARED, dev_err=err)
    ones = torch.ones((m, 1), dtype=torch.float32, device=DEV)
    y, cnt2 = mm.mm_mega_moe(xq, ids.view(m, 1), ones, w[0], w[2], p1, p2, e, weight_scale_layout=mm.WSCALE_PREPARED,
                             dispatch_quant_mode=0, dispatch_quant_out_dtype=23, x_scales=xs)
    assert host(err)[0] == 0
    assert np.array_equal(host(cnt), host(cnt2))
    assert np.array_equal(host(out), host(y))


@pytest.mark.parametrize("fmt,n_shared", [(23, 0), (24, 2)])
def test_moe_combine_mxfp8_rows(fmt, n_shared):
    """mm_moe_combine on rows sent as MXFP8 (combineQuantMode 3 / 4): each
    routed term is DQ_MX of its row (codes and E8M0 scales of the oracle's
    Q_MX), then the fp32 sum in k order and the shared rows, one bf16 rounding."""
    rng = np.random.default_rng(11 + fmt)
    n, k, h, nrows = 150, 5, 512, 600
    rows = (rng.standard_normal((nrows, h)) * np.exp2(rng.integers(-8, 6, (nrows, 1)))).astype(np.float32)
    q, sc = oracle.mx_quantize(rows, oracle.DT_F32, fmt, s_cols=h // 32)
    idx = rng.integers(-1, nrows, size=n * k).astype(np.int32)
    g = rng.random((n, k)).astype(np.float32)
    sh_b = torch.from_numpy(rng.standard_normal((n_shared, n, h)).astype(np.float32)).to(torch.bfloat16)
    y = mm.mm_moe_combine(t(q), t(idx), t(g), expert_scales=t(sc), expert_rows_dtype=fmt,
                          shared_rows=sh_b.to(DEV) if n_shared else None)
    tab = np.array([oracle.fp8_value(c, fmt) for c in range(256)])
    dq = (tab[q] * np.exp2(np.repeat(sc.astype(np.float64) - 127.0, 32, axis=1))).astype(np.float32)
    acc = np.zeros((n, h), np.float32)
    ix = idx.reshape(n, k)
    for kk in range(k):
        ok = ix[:, kk] >= 0
        acc[ok] = (g[ok, kk:kk + 1].astype(np.float64) * dq[ix[ok, kk]] + acc[ok]).astype(np.float32)
    for s_ in range(n_shared):
        acc = (acc.astype(np.float64) + sh_b[s_].float().numpy()).astype(np.float32)
    assert torch.equal(y.cpu(), torch.from_numpy(acc).to(torch.bfloat16))


@pytest.mark.parametrize("gate_bf16,n_shared", [(False, 0), (True, 0), (False, 2), (True, 4)])
def test_moe_combine_rows(gate_bf16, n_shared):
    """mm_moe_combine: fp32 sum in k order of weighted rows chosen by an index
    (negative: left out), then the shared experts' rows, one bf16 rounding --
    MegaMoE stage 4."""
    rng = np.random.default_rng(5 + n_shared)
    n, k, h, nrows = 200, 6, 384, 900
    rows = rng.standard_normal((nrows, h)).astype(np.float32)
    rows_b = torch.from_numpy(rows).to(torch.bfloat16)
    idx = rng.integers(-1, nrows, size=n * k).astype(np.int32)
    g = rng.random((n, k)).astype(np.float32)
    gt = torch.from_numpy(g)
    if gate_bf16:
        gt = gt.to(torch.bfloat16)
    sh_b = torch.from_numpy(rng.standard_normal((n_shared, n, h)).astype(np.float32)).to(torch.bfloat16)
    y = mm.mm_moe_combine(rows_b.to(DEV), torch.from_numpy(idx).to(DEV), gt.to(DEV),
                          shared_rows=sh_b.to(DEV) if n_shared else None)
    r = rows_b.float().numpy()
    gw = gt.float().numpy()
    acc = np.zeros((n, h), np.float32)
    ix = idx.reshape(n, k)
    for kk in range(k):
        ok = ix[:, kk] >= 0
        # a fused multiply-add: the fp32 product is exact in float64, one rounding to fp32
        acc[ok] = (gw[ok, kk:kk + 1].astype(np.float64) * r[ix[ok, kk]] + acc[ok]).astype(np.float32)
    for s in range(n_shared):   # weight 1: a plain fp32 addition
        acc = (acc.astype(np.float64) + sh_b[s].float().numpy()).astype(np.float32)
    want = torch.from_numpy(acc).to(torch.bfloat16)
    assert torch.equal(y.cpu(), want)
