"""mm_moe_init_routing_noalloc against mm_moe_init_routing.

The no-allocation entry point is for callers that cannot give the library
device scratch memory (a host program or plug-in with no device allocator of
its own, or one that must not call cudaMalloc / cudaFree while serving); its
scratch is a fixed array inside the library.  It must produce exactly what
the workspace-based entry point produces.  Two different problems are run
back to back, so scratch left in the shared array by the first call cannot
hide a fault in the second.  The entry point is called through the C ABI
(ctypes), not through any Python re-implementation.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import routing_permute_mxfp8_gb300 as mm

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _abi():
    lib = mm.load()
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f = lib.mm_moe_init_routing_noalloc
    f.argtypes = [p, i32, p, i64, i64, i64, i64, i32, i32, p, p, p, p, p, p, p]
    f.restype = i32
    return f


def _noalloc(f, x, ids, e, quant, ttype):
    n, h = x.shape
    k = ids.shape[1]
    rows = n * k
    if quant == mm.QUANT_NONE:
        ex = torch.empty((rows, h), dtype=x.dtype, device=DEV)
        sc = None
    else:
        ex = torch.empty((rows, h), dtype=torch.uint8, device=DEV)
        sc = torch.empty((rows, ((h + 31) // 32 + 1) // 2 * 2), dtype=torch.uint8, device=DEV)
    exp_idx = torch.empty(rows, dtype=torch.int32, device=DEV)
    srt = torch.empty(rows, dtype=torch.int32, device=DEV)
    tok = torch.empty(e, dtype=torch.int64, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = f(vp(x), 27, vp(ids), n, h, k, e, quant, ttype, vp(ex), vp(sc), vp(exp_idx), vp(srt), vp(tok), vp(err),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    torch.cuda.synchronize()
    return ex, exp_idx, tok, sc, srt, err


def _same(a, b):
    if a is None or b is None or b.numel() == 0:
        return a is None or a.numel() == 0 or b.numel() == 0
    return torch.equal(a.view(torch.uint8).flatten().cpu(), b.contiguous().view(torch.uint8).flatten().cpu())


@pytest.mark.parametrize("order", ["quant_first", "copy_first"])
def test_noalloc_matches_workspace_entry_point_twice(order):
    f = _abi()
    cases = [dict(n=2048, h=1024, e=64, k=8, quant=mm.QUANT_MXFP8_E4M3FN, ttype=1),
             dict(n=700, h=256, e=300, k=4, quant=mm.QUANT_NONE, ttype=0)]
    if order == "copy_first":
        cases = cases[::-1]
    for c in cases:
        cfg = synth.CONFIGS["routing"].scaled(n=c["n"], h=c["h"], e=c["e"], k=c["k"])
        x = torch.from_numpy(synth.tokens_bf16(cfg).view(np.int16)).to(DEV).view(torch.bfloat16)
        ids = torch.from_numpy(synth.topk_ids(cfg)).to(DEV)
        ref = mm.mm_moe_init_routing(x, ids, c["e"], c["quant"], c["ttype"])
        ex, exp_idx, tok, sc, srt, err = _noalloc(f, x, ids, c["e"], c["quant"], c["ttype"])
        assert int(err.item()) == 0
        assert _same(ex, ref[0])
        assert torch.equal(exp_idx.cpu(), ref[1].cpu())
        assert torch.equal(tok.cpu(), ref[2].cpu())
        assert _same(sc, ref[3])
        assert torch.equal(srt.cpu(), ref[4].cpu())


def test_noalloc_rejects_a_problem_larger_than_its_scratch():
    f = _abi()
    # 2^20 expanded rows need > 4 MiB of scratch; rejected before any launch
    st = f(ctypes.c_void_p(16), 27, ctypes.c_void_p(16), 1 << 17, 128, 8, 256, -1, 1, ctypes.c_void_p(16), None,
           None, None, None, None, None)
    assert st == 3


@pytest.mark.parametrize("ttype", [0, 1])
def test_noalloc_empty_batch_writes_zero_counts(ttype):
    """num_rows = 0: the counts (or cumsum) output is all zeros, as from the
    workspace-based entry point; nothing else is written."""
    f = _abi()
    e = 32
    tok = torch.full((e,), -7, dtype=torch.int64, device=DEV)
    dummy = torch.zeros(64, dtype=torch.uint8, device=DEV)
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    st = f(vp(dummy), 27, vp(dummy), 0, 64, 4, e, 3, ttype, vp(dummy), vp(dummy), vp(dummy), vp(dummy), vp(tok),
           None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(tok.cpu(), torch.zeros(e, dtype=torch.int64))
