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
