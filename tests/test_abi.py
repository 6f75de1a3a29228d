"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import routing_permute_mxfp8_gb300 as mm
from routing_permute_mxfp8_gb300 import build as mmbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mm_moe.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(mm.lib_path()):
        mmbuild.build()
    return mm.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for want in ("mm_moe_init_routing", "mm_moe_token_permute", "mm_mega_moe", "mm_mx_quantize",
                 "mm_prepare_weight_scales", "mm_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_checked_build_exports_the_same_symbols(lib):
    """libmm_moe_check.so (MM_CHECK: device index checks) has the same ABI
    and says which build it is."""
    checked = ctypes.CDLL(os.path.join(os.path.dirname(mm.lib_path()), "libmm_moe_check.so"))
    missing = [n for n in declared_functions() if not hasattr(checked, n)]
    assert not missing, missing
    assert checked.mm_checked_build() == 1
    assert lib.mm_checked_build() == 0
    mm.use_checked_library(True)
    try:
        assert mm.lib_path().endswith("libmm_moe_check.so") and mm.load().mm_checked_build() == 1
    finally:
        mm.use_checked_library(False)
    assert mm.load().mm_checked_build() == 0


def test_status_strings(lib):
    assert lib.mm_status_string(0) == b"ok"
    assert lib.mm_status_string(3) == b"workspace too small"
    assert mm.mm_version() >= 100


def _ws(lib, fn, *args):
    n = ctypes.c_size_t(0)
    st = getattr(lib, fn)(*args, ctypes.byref(n))
    return st, n.value


def test_workspace_queries(lib):
    st, n = _ws(lib, "mm_moe_init_routing_workspace_size", 16384, 8, 256)
    assert st == 0 and n >= 16384 * 8 * 4
    assert _ws(lib, "mm_moe_init_routing_workspace_size", 16384, 8, 0)[0] == 1
    assert _ws(lib, "mm_moe_init_routing_workspace_size", 1 << 22, 4, 8)[0] == 1   # F >= 16777215
    assert _ws(lib, "mm_moe_init_routing_workspace_size", 16777215, 1, 8)[0] == 1  # F = the sort limit
    assert _ws(lib, "mm_moe_init_routing_workspace_size", 16777214, 1, 8)[0] == 0  # largest F allowed
    st, n = _ws(lib, "mm_mega_moe_workspace_size", 8192, 7168, 8, 256, 2048, 0, 0)
    assert st == 0 and n > 8192 * 8 * 7168 * 3
    assert _ws(lib, "mm_mega_moe_workspace_size", 64, 200, 2, 8, 128, 0, 0)[0] == 2   # H % 128
    assert _ws(lib, "mm_mega_moe_workspace_size", 64, 256, 2, 8, 100, 0, 0)[0] == 2   # I % 128
    assert _ws(lib, "mm_mega_moe_workspace_size", 64, 256, 33, 64, 128, 0, 0)[0] == 1  # topK > 32
    assert _ws(lib, "mm_mega_moe_workspace_size", 64, 256, 2, 8, 128, 5, 0)[0] == 1   # shared > 4
    assert lib.mm_moe_token_permute_out_rows(8, 6) == 6
    assert lib.mm_moe_token_permute_out_rows(8, 0) == 8
    assert lib.mm_moe_token_permute_out_rows(8, 20) == 8
    assert lib.mm_moe_token_permute_out_rows(8, -3) == 5
    assert lib.mm_moe_token_permute_out_rows(8, -30) == 0


def _mega(lib, **kw):
    a = dict(x=1, xs=None, ids=1, w=1, gdt=0, w1=1, w2=1, s1=1, s2=1, wdt=24, layout=0, sw1=None, sw2=None, ss1=None,
             ss2=None, swdt=24, s=0, bs=64, h=256, k=2, e=8, ep=1, inter=128, maxrecv=0, dqm=4, dqd=24, sqd=0, cqm=0,
             act=b"swiglu", params=None, nparams=0, y=1, counts=None, exp=None, aq=None, asc=None, dq=None, dsc=None,
             ws=None,
             wsb=0, err=None, stream=None)
    a.update(kw)
    vp = lambda v: None if v is None else ctypes.c_void_p(16 * v)
    return lib.mm_mega_moe(vp(a["x"]), vp(a["xs"]), vp(a["ids"]), vp(a["w"]), a["gdt"], vp(a["w1"]), vp(a["w2"]), vp(a["s1"]),
                           vp(a["s2"]), a["wdt"], a["layout"], vp(a["sw1"]), vp(a["sw2"]), vp(a["ss1"]),
                           vp(a["ss2"]), a["swdt"], a["s"], a["bs"], a["h"], a["k"], a["e"], a["ep"], a["inter"],
                           a["maxrecv"], a["dqm"], a["dqd"], a["sqd"], a["cqm"], a["act"], a["params"], a["nparams"],
                           vp(a["y"]), vp(a["counts"]), vp(a["exp"]), vp(a["aq"]), vp(a["asc"]), vp(a["dq"]),
                           vp(a["dsc"]), vp(a["ws"]),
                           a["wsb"], vp(a["err"]), a["stream"])


def test_selftest_wait_timeout_host_validation(lib):
    assert lib.mm_selftest_wait_timeout(0, ctypes.c_void_p(16), None) == 1             # limit must be > 0
    assert lib.mm_selftest_wait_timeout(20_000_000_000, ctypes.c_void_p(16), None) == 1  # at most 10 s
    assert lib.mm_selftest_wait_timeout(1_000_000, None, None) == 1                    # dev_err required


def test_timing_stage_selector(lib):
    lib.mm_timing_select.argtypes = [ctypes.c_uint32]
    assert lib.mm_timing_select(1 << 3) == 0        # GEMM1 only
    assert lib.mm_timing_select(1 << 7) == 1        # no such stage
    assert lib.mm_timing_select((1 << 7) - 1) == 0  # every stage (the default)


def test_routing_path_selector(lib):
    for path in (1, 2, 3, 0):
        assert lib.mm_set_routing_path(path) == 0
    assert lib.mm_set_routing_path(-1) == 1
    assert lib.mm_set_routing_path(4) == 1


def test_mega_moe_host_rejections(lib):
    assert _mega(lib, ep=2) == 2                     # ep_world_size != 1
    assert _mega(lib, cqm=3) == 2                    # combine quantisation
    assert _mega(lib, dqm=0) == 1                    # pass-through without x_scales
    assert _mega(lib, xs=1) == 1                     # x_scales with internal quantisation
    assert _mega(lib, dqm=3) == 2                    # other dispatch quant modes
    assert _mega(lib, act=b"relu") == 2              # unknown activation
    assert _mega(lib, act=b"gelu") == 1              # gelu needs its [FLT_MAX] placeholder
    assert _mega(lib, dqd=296) == 2                  # FP4 dispatch (A4W4-FP) needs FP4 routed weights
    assert _mega(lib, dqd=296, wdt=296) == 3         # A4W4-FP passes the checks (stops at the workspace)
    assert _mega(lib, dqd=296, wdt=296, s=1, sw1=1, sw2=1, ss1=1, ss2=1, swdt=24) == 3  # FP8 shared experts
    assert _mega(lib, dqd=1) == 2                    # INT8 dispatch (not an MX scenario)
    sh = dict(s=1, sw1=1, sw2=1, ss1=1, ss2=1)
    assert _mega(lib, sqd=23, **sh) == 3             # shared experts in their own type: accepted
    assert _mega(lib, sqd=296, swdt=24, **sh) == 3   # FP4 shared input, FP8 shared weights
    assert _mega(lib, sqd=296, swdt=296, **sh) == 3
    assert _mega(lib, sqd=1, **sh) == 2              # INT8
    assert _mega(lib, sqd=23, dqm=0, xs=1, **sh) == 1  # pass-through: the shared experts take the dispatch type
    assert _mega(lib, gdt=27 + 1) == 1               # gating weight dtype
    assert _mega(lib, maxrecv=100) == 1              # below bs*k rows
    assert _mega(lib, ws=None, wsb=0) == 3           # workspace missing
    assert _mega(lib, bs=0) == 0                     # empty batch: nothing to do
    assert _mega(lib, dq=1) == 1                     # dispatch diagnostic codes without their scales
    assert _mega(lib, aq=1) == 1                     # activation diagnostic codes without their scales
    f = lambda *v: (ctypes.c_float * len(v))(*v)
    for act, params in ((b"swiglu", (2.0, 1.0)), (b"swiglu", (-1.0,)), (b"swiglu", (float("nan"),)),
                        (b"swigluoai", (1.0,)), (b"swigluoai", (0.0, float("inf"), 1.0)), (b"situglu", (0.0,)),
                        (b"situglu", (1.0, -2.0)), (b"situglu", (1.0, 2.0, 3.0)), (b"gelu", (1.0,))):
        assert _mega(lib, act=act, params=f(*params), nparams=len(params)) == 1, (act, params)
    # valid lists pass the activation check (and stop at the missing workspace)
    fmax = 3.4028234663852886e38
    for act, params in ((b"swiglu", (0.0,)), (b"swiglustep", (7.0,)), (b"swigluoai", ()),
                        (b"swigluoai", (7.0, 1.702, 1.0)), (b"situglu", ()), (b"situglu", (2.0, 3.0)),
                        (b"gelu", (fmax,))):
        assert _mega(lib, act=act, params=f(*params) if params else None, nparams=len(params)) == 3, act


def test_init_routing_v3_host_rejections(lib):
    """Active expert range and count-type checks, before anything is enqueued."""
    vp = lambda v: None if v is None else ctypes.c_void_p(16 * v)

    def call(start, end, ttype=1, e=8, ws=None, wsb=0):
        return lib.mm_moe_init_routing_v3(vp(1), 27, vp(1), 64, 256, 2, e, start, end, -1, ttype, vp(1), None, vp(1),
                                          None, vp(1), vp(ws), wsb, None, None)
    assert call(0, 8) == 3           # valid: stops at the missing workspace
    assert call(3, 4) == 3
    assert call(-1, 4) == 1          # start < 0
    assert call(4, 4) == 1           # empty range
    assert call(5, 4) == 1
    assert call(0, 9) == 1           # end > expert_num
    assert call(0, 8, ttype=2) == 3  # key_value counts
    assert call(0, 8, ttype=3) == 2
    assert call(0, 6000, ttype=2, e=6000) == 1   # key_value: expert_num <= 5120
    n_v3, n_base = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.mm_moe_init_routing_v3_workspace_size(64, 2, 8, ctypes.byref(n_v3)) == 0
    assert lib.mm_moe_init_routing_workspace_size(64, 2, 8, ctypes.byref(n_base)) == 0
    assert n_v3.value >= n_base.value + 8 * 8
    # mm_moe_init_routing itself keeps types 0 / 1
    assert lib.mm_moe_init_routing(vp(1), 27, vp(1), 64, 256, 2, 8, -1, 2, vp(1), None, vp(1), None, vp(1), None, 0,
                                   None, None) == 2


def test_permute_host_rejections(lib):
    vp = lambda v: ctypes.c_void_p(16 * v)
    call = lambda **kw: lib.mm_moe_token_permute(
        vp(1), kw.get("dt", 27), vp(1), kw.get("idt", 3), 4, 2, kw.get("h", 128), kw.get("e", 2), 0,
        kw.get("pad", 0), kw.get("q", -1), vp(1), vp(1), vp(1), None, 0, None, None)
    assert call(pad=1) == 2          # padded_mode is not supported (as in the article)
    assert call(q=4) == 2            # not a quant mode of the article
    assert call(q=9, dt=0) == 2      # MXFP4 takes fp16 / bf16 tokens
    assert call(q=9) == 3            # MXFP4 accepted (stops at the missing workspace)
    assert call(idt=0) == 1          # indices dtype
    assert call(q=2, h=24) == 2      # H % 16 for MXFP8
    assert call() == 3               # workspace missing


def test_binding_fails_loudly_without_its_library(monkeypatch, tmp_path):
    """No fallback path: with the CUDA library absent the binding raises."""
    absent = str(tmp_path / "absent" / "libmm_moe.so")
    monkeypatch.setattr(mm, "_LIB_PATHS", {False: absent, True: absent})
    monkeypatch.setattr(mm, "_libs", {})
    with pytest.raises(mm.MMError):
        mm.load()


def test_binding_refuses_host_tensors():
    """The operations run only in the CUDA kernels: host (CPU) tensors are
    rejected, never computed on the CPU."""
    import torch
    x = torch.zeros((4, 256), dtype=torch.bfloat16)
    ids = torch.zeros((4, 2), dtype=torch.int32)
    with pytest.raises(mm.MMError):
        mm.mm_moe_init_routing(x, ids, 8)
    with pytest.raises(mm.MMError):
        mm.mm_moe_token_permute(x, ids, 8)


def test_binding_refuses_index_and_data_types_the_abi_would_misread():
    """The C entry points read expert ids as int32 (MoeInitRoutingV3 parameter
    table: expertIdx INT32) and x / weights as the stated codes.  Tensors of
    another dtype (torch's default int64 for ids, most of all) are refused with
    MMError before any pointer reaches the library, on any device."""
    import torch
    x = torch.zeros((4, 256), dtype=torch.bfloat16)
    ids64 = torch.zeros((4, 2), dtype=torch.int64)
    ids32 = ids64.to(torch.int32)
    for call in (lambda: mm.mm_moe_init_routing(x, ids64, 8),
                 lambda: mm.mm_moe_init_routing_noalloc(x, ids64, 8)):
        with pytest.raises(mm.MMError, match="expert_idx must be int32"):
            call()
    with pytest.raises(mm.MMError, match="x must be"):
        mm.mm_moe_init_routing(x.to(torch.int16), ids32, 8)
    with pytest.raises(mm.MMError, match="indices must be"):
        mm.mm_moe_token_permute(x, ids32.to(torch.int16), 8)
    w1 = torch.zeros((8, 256, 256), dtype=torch.uint8)
    w2 = torch.zeros((8, 256, 128), dtype=torch.uint8)
    s1 = torch.zeros((8, 256, 8), dtype=torch.uint8)
    s2 = torch.zeros((8, 256, 4), dtype=torch.uint8)
    gate = torch.zeros((4, 2), dtype=torch.float32)
    with pytest.raises(mm.MMError, match="topk_ids must be int32"):
        mm.mm_mega_moe(x, ids64, gate, w1, w2, s1, s2, 8)
    with pytest.raises(mm.MMError, match="topk_weights must be"):
        mm.mm_mega_moe(x, ids32, gate.to(torch.float16), w1, w2, s1, s2, 8)
    with pytest.raises(mm.MMError, match="x must be bfloat16"):
        mm.mm_mega_moe(x.float(), ids32, gate, w1, w2, s1, s2, 8)
    with pytest.raises(mm.MMError, match="weight1 must be"):
        mm.mm_mega_moe(x, ids32, gate, w1.to(torch.int8), w2, s1, s2, 8)
    with pytest.raises(mm.MMError, match="weight_scales2 must be uint8"):
        mm.mm_mega_moe(x, ids32, gate, w1, w2, s1, s2.to(torch.int32), 8)
    with pytest.raises(mm.MMError, match="BS = x.shape"):
        mm.mm_mega_moe(x, ids32[:3], gate[:3], w1, w2, s1, s2, 8)


def test_expert_parallel_host_rejections(lib):
    """mm_moe_ep_dispatch, mm_moe_combine and mm_moe_expert_ffn refuse bad
    arguments with a status before anything is enqueued (MegaMoE README,
    parameter table: epWorldSize, moeExpertNum, dispatchQuantOutDtype,
    combineQuantMode; the constraints' "reports an error" rule)."""
    vp = lambda v: None if v is None else ctypes.c_void_p(16 * v)

    def dispatch(n=64, h=256, k=2, e=8, w=2, xdt=27, qdt=24, ptr=1, ws=None, wsb=0, counts=1):
        return lib.mm_moe_ep_dispatch(vp(ptr), xdt, vp(ptr), n, h, k, e, w, qdt, vp(ptr), vp(ptr), vp(ptr),
                                      vp(counts), vp(ptr), vp(ws), wsb, None, None)
    assert dispatch() == 3                 # valid: stops at the missing workspace
    assert dispatch(qdt=296) == 3          # packed FP4 rows (A4W4-FP)
    assert dispatch(w=0) == 1              # ep_world_size
    assert dispatch(w=3) == 1              # E not a multiple of W
    assert dispatch(k=9) == 1              # top-K above E
    assert dispatch(k=33, e=64) == 1       # top-K above 32
    assert dispatch(n=1 << 22, k=4) == 1   # N*K at the sort limit
    assert dispatch(xdt=0) == 1            # fp32 tokens
    assert dispatch(qdt=1) == 2            # INT8 is not an MX type
    assert dispatch(h=192) == 2            # H % 128
    assert dispatch(ptr=None) == 1         # missing buffers
    assert lib.mm_moe_ep_dispatch(ctypes.c_void_p(8), 27, vp(1), 64, 256, 2, 8, 2, 24, vp(1), vp(1), vp(1), vp(1),
                                  vp(1), None, 0, None, None) == 1  # x not 16-byte aligned
    assert dispatch(n=0, counts=None) == 0  # no rows, nothing to zero
    n_ws = ctypes.c_size_t(0)
    assert lib.mm_moe_ep_dispatch_workspace_size(64, 2, 2, ctypes.byref(n_ws)) == 0 and n_ws.value > 0
    assert lib.mm_moe_ep_dispatch_workspace_size(64, 2, 0, ctypes.byref(n_ws)) == 1

    def combine(rdt=27, sc=None, n=64, h=256, k=2, gdt=0, sh=None, ns=0, y=1, rows=1):
        return lib.mm_moe_combine(vp(rows), rdt, vp(sc), vp(1), vp(1), gdt, n, h, k, vp(sh), ns, vp(y), None)
    assert combine(n=0) == 0               # no tokens: nothing to do
    assert combine(ns=5, sh=1) == 1        # at most 4 shared experts
    assert combine(k=33, ns=4, sh=1) == 1  # k + n_shared <= 36
    assert combine(n=1 << 22, k=4) == 1    # N*K at the dispatch's row limit
    assert combine(gdt=1) == 1             # gating weights fp32 or bf16
    assert combine(rdt=296, sc=1) == 2     # MXFP4 rows are not a combine quantisation
    assert combine(h=100) == 2             # H % 8
    assert combine(rdt=23, sc=1, h=48) == 2  # MXFP8 rows: H % 32
    assert combine(rdt=24) == 1            # MXFP8 rows without their scales
    assert combine(ns=1) == 1              # shared experts without their rows
    assert combine(y=None) == 1
    assert combine(rows=None) == 1
    assert lib.mm_moe_combine(vp(1), 27, None, vp(1), vp(1), 0, 64, 256, 2, None, 0, ctypes.c_void_p(24),
                              None) == 1   # y not 16-byte aligned

    def ffn(rows=64, h=256, xdt=24, wdt=24, e=4, inter=128, xs=1, act=b"swiglu", ws=None, wsb=0, counts=1):
        return lib.mm_moe_expert_ffn(vp(1), vp(xs), xdt, vp(1), rows, h, vp(1), vp(1), vp(1), vp(1), wdt, 0, e, inter,
                                     act, None, 0, vp(1), vp(counts), vp(ws), wsb, None, None)
    assert ffn() == 3                      # valid: stops at the missing workspace
    assert ffn(xdt=296, wdt=296) == 3      # A4W4-FP rows
    assert ffn(xdt=296) == 2               # FP4 rows need FP4 weights
    assert ffn(xdt=1) == 2                 # not an MX type
    assert ffn(xs=None) == 1               # the received rows' scales are required
    assert ffn(h=200) == 2                 # H % 128
    assert ffn(inter=100) == 2             # I % 128
    assert ffn(e=0) == 1
    assert ffn(act=b"relu") == 2
    assert ffn(rows=0, counts=None) == 0   # no rows received
    n_ws = ctypes.c_size_t(0)
    assert lib.mm_moe_expert_ffn_workspace_size(64, 256, 4, 128, 0, ctypes.byref(n_ws)) == 0 and n_ws.value > 0


def test_quantize_and_scale_preparation_host_rejections(lib):
    """mm_mx_quantize and the weight-scale preparation check sizes, types and
    alignment on the host; the prepared layout's size is the pages' scale
    bytes, with 256-row pairs of GEMM2's output rows padded."""
    vp = lambda v: None if v is None else ctypes.c_void_p(16 * v)

    def quant(src_dt=27, rows=8, cols=256, out_dt=24, sc_cols=8, ptr=1):
        return lib.mm_mx_quantize(vp(ptr), src_dt, rows, cols, out_dt, vp(ptr), vp(ptr), sc_cols, None)
    assert quant(rows=0) == 0              # nothing to do
    assert quant(rows=-1) == 1
    assert quant(cols=0) == 1
    assert quant(src_dt=3) == 1            # int32 source
    assert quant(out_dt=1) == 1            # INT8 is not an MX type
    assert quant(cols=40) == 2             # cols % 16
    assert quant(sc_cols=7) == 1           # fewer scale columns than groups
    assert quant(ptr=None) == 1
    size = lambda which, e, n, k: _ws(lib, "mm_prepared_weight_scales_size", which, e, n, k)
    assert size(1, 2, 512, 256) == (0, 2 * 512 * 256 // 32)
    assert size(2, 2, 384, 256) == (0, 2 * 2 * 2 * (256 // 128) * 512)   # 384 rows padded to two pairs
    assert size(3, 2, 512, 256)[0] == 1    # GEMM 1 or 2
    assert size(1, 2, 512, 200)[0] == 1    # K % 128
    assert size(1, 2, 384, 256)[0] == 1    # GEMM1 output rows come in gate / up pairs of 128
    assert lib.mm_prepare_weight_scales(ctypes.c_void_p(2), 1, 2, 512, 256, vp(1), None) == 1  # misaligned
    assert lib.mm_prepare_weight_scales(None, 1, 2, 512, 256, vp(1), None) == 1


def test_binding_refuses_mismatched_shapes():
    """The C ABI takes sizes and raw pointers, so the binding checks that the
    tensors agree with the sizes it passes (a smaller tensor would be read past
    its end on the GPU).  Consistent arguments pass every shape check and stop
    at the device check, for FP8 and packed FP4 weights, gelu, shared experts,
    prepared scales and pass-through inputs."""
    import torch
    u8 = lambda *s: torch.zeros(s, dtype=torch.uint8)
    bf = lambda *s: torch.zeros(s, dtype=torch.bfloat16)
    i32 = lambda *s: torch.zeros(s, dtype=torch.int32)
    f32 = lambda *s: torch.zeros(s, dtype=torch.float32)
    device = "inputs must be contiguous CUDA tensors"

    def refused(fn, match):
        with pytest.raises(mm.MMError, match=match):
            fn()

    # routing, permute, no-allocation routing, expert-parallel dispatch: ids agree with x
    x, ids = bf(6, 256), i32(6, 2)
    refused(lambda: mm.mm_moe_init_routing(x, i32(5, 2), 8), "expert_idx must be")
    refused(lambda: mm.mm_moe_init_routing_noalloc(x, i32(7, 2), 8), "expert_idx must be")
    refused(lambda: mm.mm_moe_token_permute(x, i32(5), 8), "indices must be")
    refused(lambda: mm.mm_moe_ep_dispatch(x, i32(5, 2), 8, 2), "topk_ids")
    refused(lambda: mm.mm_moe_init_routing(x, ids, 8), device)
    refused(lambda: mm.mm_moe_token_permute(x, i32(6), 8), device)
    refused(lambda: mm.mm_moe_ep_dispatch(x, ids, 8, 2), device)

    # MegaMoE: E = 8, H = 256, I = 128
    e, h, i = 8, 256, 128
    gate = f32(6, 2)
    w = dict(weight1=u8(e, 2 * i, h), weight2=u8(e, h, i), weight_scales1=u8(e, 2 * i, h // 32),
             weight_scales2=u8(e, h, i // 32))
    mega = lambda **kw: mm.mm_mega_moe(kw.pop("x", x), ids, gate, kw.pop("weight1", w["weight1"]),
                                       kw.pop("weight2", w["weight2"]), kw.pop("weight_scales1", w["weight_scales1"]),
                                       kw.pop("weight_scales2", w["weight_scales2"]), kw.pop("e", e), **kw)
    refused(lambda: mega(), device)
    refused(lambda: mega(e=16), r"weight1 must be \[16")                      # E disagrees with the weights
    refused(lambda: mega(weight1=u8(e, 2 * i, 512)), "weight1 must be")       # H disagrees with x
    refused(lambda: mega(weight2=u8(e, h, 2 * i)), "weight2 must be")         # A_hat width
    refused(lambda: mega(weight_scales2=u8(e, h, 2)), "weight_scales2 holds")
    refused(lambda: mega(out=bf(6, 128)), "out must be")
    refused(lambda: mega(weight2=u8(e, h, 2 * i), weight_scales2=u8(e, h, 2 * i // 32), activation="gelu",
                         activation_params=(3.4e38,)), device)
    refused(lambda: mega(weight1=u8(e, 2 * i, h // 2), weight2=u8(e, h, i // 2), weight_dtype=296), device)  # FP4
    refused(lambda: mega(weight1=u8(e, 2 * i, h // 2), weight_dtype=296), "weight2 must be")
    # prepared buffers of mm_prepared_weight_scales_size bytes (GEMM2's 256 output rows = one pair)
    prepared = dict(weight_scales1=u8(e * 2 * i * h // 32), weight_scales2=u8(e * 2 * 1 * (i // 128) * 512))
    refused(lambda: mega(weight_scale_layout=1, **prepared), device)
    sh = dict(shared_weight1=u8(1, 2 * i, h), shared_weight2=u8(1, h, i), shared_weight_scales1=u8(1, 2 * i, h // 32),
              shared_weight_scales2=u8(1, h, i // 32))
    refused(lambda: mega(**sh), device)
    refused(lambda: mega(**dict(sh, shared_weight_scales2=None)), "shared experts need all four")
    refused(lambda: mega(**dict(sh, shared_weight2=u8(1, h, 2 * i))), "shared_weight2 must be")
    refused(lambda: mega(**dict(sh, shared_weight1=u8(1, 2 * i, h // 2), shared_weight2=u8(1, h, i // 2)),
                         shared_weight_dtype=296), device)
    xq = u8(6, h)
    refused(lambda: mega(x=xq, dispatch_quant_mode=0, x_scales=u8(6, h // 32)), device)   # pass-through
    refused(lambda: mega(x=xq, dispatch_quant_mode=0, x_scales=u8(6, 4)), "x_scales must be")

    # expert side: M = 10 received rows, 4 local experts
    ffn = lambda **kw: mm.mm_moe_expert_ffn(kw.pop("x", u8(10, h)), kw.pop("x_scales", u8(10, h // 32)), i32(10),
                                            kw.pop("weight1", u8(4, 2 * i, h)), kw.pop("weight2", u8(4, h, i)),
                                            u8(4, 2 * i, h // 32), u8(4, h, i // 32), kw.pop("e", 4), **kw)
    refused(lambda: ffn(), device)
    refused(lambda: ffn(e=8), "weight1 must be")
    refused(lambda: ffn(x_scales=u8(10, 2)), "x_scales must be")
    refused(lambda: ffn(out=bf(10, 128)), "out must be")
    refused(lambda: ffn(x=u8(10, h // 2), weight1=u8(4, 2 * i, h // 2), weight2=u8(4, h, i // 2), x_dtype=296,
                        weight_dtype=296), device)

    # combine: 6 tokens, top-K 2, 20 expert rows
    comb = lambda **kw: mm.mm_moe_combine(kw.pop("rows", bf(20, h)), i32(12), gate, **kw)
    refused(lambda: comb(), device)
    refused(lambda: comb(out=bf(6, 128)), "out must be")
    refused(lambda: comb(rows=u8(20, h), expert_scales=u8(19, h // 32), expert_rows_dtype=24), "expert_scales must be")
    refused(lambda: comb(rows=u8(20, h), expert_scales=u8(20, h // 32), expert_rows_dtype=24), device)
    refused(lambda: comb(shared_rows=bf(1, 6, 128)), "shared_rows must be")
