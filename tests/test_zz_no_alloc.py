"""mm_moe_init_routing_noalloc against mm_moe_init_routing and the oracle.

The no-allocation entry point is for callers that cannot give the library
device scratch memory (a host program or plug-in with no device allocator of
its own, or one that must not call cudaMalloc / cudaFree while serving); its
scratch is a fixed array inside the library.  It must produce exactly what
the workspace-based entry point produces, and what the CPU oracle computes
from the operator pages.  Different problems are run back to back, so
scratch left in the shared array by one call cannot hide a fault in the
next; the scatter index is taken both from the caller and from the array.
The entry point is called through the C ABI (ctypes), not through any
Python re-implementation.
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


def _abi():
    lib = mm.load()
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f = lib.mm_moe_init_routing_noalloc
    f.argtypes = [p, i32, p, i64, i64, i64, i64, i32, i32, p, p, p, p, p, p, p]
    f.restype = i32
    return f


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(f, x, ids, e, quant, ttype, with_idx=True):
    n, h = x.shape
    k = ids.shape[1]
    rows = n * k
    if quant == mm.QUANT_NONE:
        ex = torch.empty((rows, h), dtype=x.dtype, device=DEV)
        sc = None
    else:
        ex = torch.empty((rows, h), dtype=torch.uint8, device=DEV)
        sc = torch.empty((rows, ((h + 31) // 32 + 1) // 2 * 2), dtype=torch.uint8, device=DEV)
    exp_idx = torch.empty(rows, dtype=torch.int32, device=DEV) if with_idx else None
    srt = torch.empty(rows, dtype=torch.int32, device=DEV)
    tok = torch.empty(e, dtype=torch.int64, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = f(_vp(x), 27, _vp(ids), n, h, k, e, quant, ttype, _vp(ex), _vp(sc), _vp(exp_idx), _vp(srt), _vp(tok),
           _vp(err), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    torch.cuda.synchronize()
    return ex, exp_idx, tok, sc, srt, err


def _same(a, b):
    if a is None or b is None or b.numel() == 0:
        return a is None or a.numel() == 0 or b.numel() == 0
    return torch.equal(a.view(torch.uint8).flatten().cpu(), b.contiguous().view(torch.uint8).flatten().cpu())


CASES = [dict(n=2048, h=1024, e=64, k=8, quant=mm.QUANT_MXFP8_E4M3FN, ttype=1),
         dict(n=700, h=256, e=300, k=4, quant=mm.QUANT_NONE, ttype=0),
         dict(n=513, h=512, e=16, k=3, quant=mm.QUANT_MXFP8_E5M2, ttype=0)]


def _inputs(c):
    cfg = synth.CONFIGS["routing"].scaled(n=c["n"], h=c["h"], e=c["e"], k=c["k"])
    xb = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    x = torch.from_numpy(xb.view(np.int16)).to(DEV).view(torch.bfloat16)
    return xb, ids, x, torch.from_numpy(ids).to(DEV)


def _check_against_oracle(c, xb, ids, ex, tok, sc, srt):
    """Indices, counts, expanded rows and scales bit-exact against the oracle
    (MoeInitRoutingV3 steps 1-3 and 5)."""
    o_srt, _, o_cnt, bad = oracle.route(ids, c["e"])
    assert bad == 0
    want_tok = np.cumsum(o_cnt) if c["ttype"] == 0 else o_cnt
    assert np.array_equal(tok.cpu().numpy(), want_tok)
    assert np.array_equal(srt.cpu().numpy(), o_srt)
    fmt = {mm.QUANT_NONE: -1, mm.QUANT_MXFP8_E4M3FN: 24, mm.QUANT_MXFP8_E5M2: 23}[c["quant"]]
    o_x, o_sc = oracle.permute(xb, oracle.DT_BF16, c["k"], o_srt, o_srt.size, fmt)
    assert np.array_equal(ex.contiguous().view(torch.uint8).cpu().numpy().reshape(-1),
                          o_x.view(np.uint8).reshape(-1))
    if fmt >= 0:
        assert np.array_equal(sc.cpu().numpy(), o_sc)


@pytest.mark.parametrize("order", [0, 1, 2])
def test_noalloc_matches_workspace_entry_point_and_oracle(order):
    """Three different problems in a rotated order, each twice: with the
    caller's expanded_row_idx and with the scatter index kept in the shared
    array (expanded_row_idx = NULL, after another problem has left stale
    data there).  Every output equals the workspace entry point's and the
    oracle's, bit for bit, in copy and both MXFP8 modes."""
    f = _abi()
    cases = CASES[order:] + CASES[:order]
    for c in cases:
        xb, ids_np, x, ids = _inputs(c)
        ref = mm.mm_moe_init_routing(x, ids, c["e"], c["quant"], c["ttype"])
        for with_idx in (True, False):
            ex, exp_idx, tok, sc, srt, err = _noalloc(f, x, ids, c["e"], c["quant"], c["ttype"], with_idx)
            assert int(err.item()) == 0
            assert _same(ex, ref[0])
            if with_idx:
                assert torch.equal(exp_idx.cpu(), ref[1].cpu())
            assert torch.equal(tok.cpu(), ref[2].cpu())
            assert _same(sc, ref[3])
            assert torch.equal(srt.cpu(), ref[4].cpu())
            _check_against_oracle(c, xb, ids_np, ex, tok, sc, srt)


def test_noalloc_rejects_a_problem_larger_than_its_scratch():
    """10240 experts and 131072 ids need 20 MiB of histograms, more than the
    4 MiB array: MM_ERR_WORKSPACE before anything is enqueued.  Every pointer
    is a real device buffer of the full size, so only the scratch check
    decides the result (a regression would compute, not fault)."""
    f = _abi()
    n, k, e, h = 16384, 8, 10240, 16
    x = torch.zeros((n, h), dtype=torch.bfloat16, device=DEV)
    ids = (torch.arange(n * k, dtype=torch.int32, device=DEV) % e).view(n, k)
    ex = torch.empty((n * k, h), dtype=torch.bfloat16, device=DEV)
    exp_idx = torch.empty(n * k, dtype=torch.int32, device=DEV)
    srt = torch.empty(n * k, dtype=torch.int32, device=DEV)
    tok = torch.zeros(e, dtype=torch.int64, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = f(_vp(x), 27, _vp(ids), n, h, k, e, -1, 1, _vp(ex), None, _vp(exp_idx), _vp(srt), _vp(tok), _vp(err),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 3
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(tok.abs().sum().item()) == 0


@pytest.mark.parametrize("ttype", [0, 1])
def test_noalloc_empty_batch_writes_zero_counts(ttype):
    """num_rows = 0: the counts (or cumsum) output is all zeros, as from the
    workspace-based entry point; nothing else is written."""
    f = _abi()
    e = 32
    tok = torch.full((e,), -7, dtype=torch.int64, device=DEV)
    dummy = torch.zeros(64, dtype=torch.uint8, device=DEV)
    st = f(_vp(dummy), 27, _vp(dummy), 0, 64, 4, e, 3, ttype, _vp(dummy), _vp(dummy), _vp(dummy), _vp(dummy),
           _vp(tok), None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(tok.cpu(), torch.zeros(e, dtype=torch.int64))
