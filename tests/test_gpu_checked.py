"""The checked build of the library (libmm_moe_check.so: the same sources
compiled with MM_CHECK, whose kernels test every index they compute on the
GPU against the buffer it addresses) on the parity cases of every stage.

Each case must give the oracle's results exactly as the normal build does
and raise no MM_DEVERR_BOUNDS (the parity helpers assert that the device
error word stays 0), and a MegaMoE step must be bit-identical between the
two builds.  Nothing here plants a bad index: the checks guard against an
inconsistency inside the library, and this shows the indices stay in
bounds on routing (every path), dispatch, both GEMMs, combine and the
expert-parallel calls.
"""
import numpy as np
import pytest
import torch

import synth
import routing_permute_mxfp8_gb300 as mm
from tests import test_gpu_parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def checked_library():
    mm.use_checked_library(True)
    assert mm.load().mm_checked_build() == 1
    yield
    mm.set_routing_path(mm.ROUTE_AUTO)
    mm.use_checked_library(False)


@pytest.mark.parametrize("path", [mm.ROUTE_CLUSTER, mm.ROUTE_GRID, mm.ROUTE_KERNELS])
@pytest.mark.parametrize("case", [P.ROUTE_CASES[i] for i in (1, 4, 5, 6)])
def test_routing_checked(path, case):
    mm.set_routing_path(path)
    P.test_init_routing_bit_exact(*case)


@pytest.mark.parametrize("case", ["tiny_shared", "zipf_mixed_sizes", "a8w4_shared_zipf", "a4w4_shared_zipf_bf16gate",
                                  "gelu", "max_experts", "topk32_shared4", "small_seg_zipf_mixed", "h896_ragged_n",
                                  "many_experts"])
def test_mega_moe_checked(case):
    P.run_mega(synth.CONFIGS["tiny"].scaled(**P.MEGA_CASES[case]))


@pytest.mark.parametrize("path", [mm.ROUTE_CLUSTER, mm.ROUTE_KERNELS])
def test_mega_moe_checked_equals_normal_build(path):
    cfg = synth.CONFIGS["tiny"].scaled(**P.MEGA_CASES["zipf_shared_e5m2_h512"])
    mm.set_routing_path(path)
    _, y_checked = P.run_mega(cfg)
    mm.use_checked_library(False)
    mm.set_routing_path(path)
    _, y_normal = P.run_mega(cfg)
    assert np.array_equal(y_checked, y_normal)


def test_permute_expert_parallel_and_combine_checked():
    P.test_token_permute_bit_exact(torch.bfloat16, False, 6, -1, False)
    P.test_token_permute_bit_exact(torch.float16, True, -7, 9, False)
    P.test_ep_dispatch_bit_exact(4, 24)
    P.test_ep_dispatch_bit_exact(4, 296)
    P.test_moe_combine_rows(True, 2)
    P.test_out_of_range_ids_are_left_out_and_flagged()
    P.test_expert_ffn_equals_mega_moe_top1(dict(n=700, h=512, inter=256, e=8, k=1, routing="zipf"))


def test_shared_quant_type_and_active_range_checked():
    P.test_mega_moe_shared_quant_type(296, 296, 24, 24, "swiglu")
    P.test_mega_moe_shared_quant_type(23, 23, 24, 24, "swiglu")
    P.test_init_routing_active_range(*P.RANGE_CASES[2])
