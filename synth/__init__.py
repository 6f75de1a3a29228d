"""Seeded synthetic inputs for the MoE routing / permute / expert-FFN path.

This module holds none of the method's arithmetic: it draws token
activations, expert choices, gating weights and fp32 source weights from a
counter-based generator (``synth.c``), and converts fp32 to bf16 bit
patterns.  Both the CPU oracle (through the tests) and the CUDA path
(through the tests and ``bench.py``) take their inputs from here.

Workloads (all seeded, seed 0 by default):

* ``tiny``          N=64, H=256, I=128, E=8, K=2, uniform routing, E4M3
* ``routing``       N=16384, H=7168, E=256, K=8, uniform routing (no FFN)
* ``qwen3``         N=4096, H=2048, I=768, E=128, K=8, uniform routing, E4M3
* ``dsv3_prefill``  N=8192, H=7168, I=2048, E=256, K=8, Zipf(s=1) routing,
                    E5M2 dispatch, E4M3 weights, bf16 gating weights
* ``dsv3_decode``   N=128, same dimensions, uniform routing, 1 shared expert

Recipe: x is bf16(N(0,1)); expert ids per token are K distinct draws, either
uniform (the first K of a random permutation of the E experts) or Zipf
(Plackett-Luce sampling without replacement with p_r proportional to 1/r^s
over a seeded permutation of the experts, done with the Gumbel-top-k
trick); gating weights are the softmax over K of N(0,1) logits, kept in
fp32 or rounded to bf16; source weights are fp32 N(0, 0.02) in the storage
layout [E, N_out, K_red] (reduction dimension contiguous).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_synth.so")
_lib = None

# dtype codes shared with the C interface of the library (FP8 codes follow
# the MegaMoE parameter table: 23 = FLOAT8_E5M2, 24 = FLOAT8_E4M3FN).
FP8_E5M2 = 23
FP8_E4M3 = 24

# generator streams
S_X, S_ROUTE, S_LOGITS, S_PERM = 1, 2, 3, 4
S_W1, S_W2, S_SW1, S_SW2 = 1 << 20, 2 << 20, 3 << 20, 4 << 20


def build() -> str:
    """Compile the generator (host C, OpenMP) next to this file."""
    tmp = _LIB_PATH + ".tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        build()
    lib = ctypes.CDLL(_LIB_PATH)
    u64, i64, f64 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
    p = ctypes.c_void_p
    lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, f64, p]
    lib.synth_normal_f64.argtypes = [u64, u64, u64, i64, p]
    lib.synth_uniform_f64.argtypes = [u64, u64, u64, i64, p]
    for f in (lib.synth_normal_f32, lib.synth_normal_f64, lib.synth_uniform_f64):
        f.restype = None
    _lib = lib
    return lib


def normal_f32(seed: int, stream: int, shape, scale: float = 1.0, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().synth_normal_f32(seed, stream, offset, out.size, scale, out.ctypes.data)
    return out


def normal_f64(seed: int, stream: int, shape, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float64)
    _load().synth_normal_f64(seed, stream, offset, out.size, out.ctypes.data)
    return out


def uniform_f64(seed: int, stream: int, shape, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float64)
    _load().synth_uniform_f64(seed, stream, offset, out.size, out.ctypes.data)
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class MoeConfig:
    name: str
    n: int            # tokens
    h: int            # hidden
    inter: int        # intermediate (0: routing / permute only)
    e: int            # routed experts
    k: int            # top-K
    routing: str      # "uniform" or "zipf"
    dispatch_fmt: int = FP8_E4M3
    weight_fmt: int = FP8_E4M3
    gate_dtype: str = "fp32"   # topk_weights dtype: "fp32" or "bf16"
    shared: int = 0            # shared experts
    seed: int = 0
    zipf_s: float = 1.0
    activation: str = "swiglu"  # MegaMoE activation; "gelu" keeps the whole 2I-wide Linear1 output
    act_params: tuple = ()

    @property
    def rows(self) -> int:
        return self.n * self.k

    @property
    def act_width(self) -> int:
        """Width of the activation output = reduction length of weight2."""
        return 2 * self.inter if self.activation == "gelu" else self.inter

    def scaled(self, **kw) -> "MoeConfig":
        d = dict(self.__dict__)
        d.update(kw)
        return MoeConfig(**d)


CONFIGS = {
    "tiny": MoeConfig("tiny", 64, 256, 128, 8, 2, "uniform"),
    "routing": MoeConfig("routing", 16384, 7168, 0, 256, 8, "uniform"),
    "qwen3": MoeConfig("qwen3", 4096, 2048, 768, 128, 8, "uniform"),
    "dsv3_prefill": MoeConfig("dsv3_prefill", 8192, 7168, 2048, 256, 8, "zipf",
                              dispatch_fmt=FP8_E5M2, weight_fmt=FP8_E4M3, gate_dtype="bf16"),
    "dsv3_decode": MoeConfig("dsv3_decode", 128, 7168, 2048, 256, 8, "uniform", shared=1),
}


def tokens_bf16(cfg: MoeConfig) -> np.ndarray:
    """x: [N, H] bf16 bit patterns of N(0,1) draws."""
    return f32_to_bf16_bits(normal_f32(cfg.seed, S_X, (cfg.n, cfg.h)))


def topk_ids(cfg: MoeConfig) -> np.ndarray:
    """[N, K] int32 distinct expert ids per token."""
    u = uniform_f64(cfg.seed, S_ROUTE, (cfg.n, cfg.e))
    if cfg.routing == "uniform":
        # the first K entries of a uniformly random permutation of the experts
        return np.argsort(u, axis=1, kind="stable")[:, : cfg.k].astype(np.int32)
    if cfg.routing == "zipf":
        perm = np.argsort(uniform_f64(cfg.seed, S_PERM, (cfg.e,)), kind="stable")
        ranks = np.arange(1, cfg.e + 1, dtype=np.float64)
        logp = -cfg.zipf_s * np.log(ranks)
        score = logp[None, :] - np.log(-np.log(u))      # Gumbel-top-k
        top = np.argsort(-score, axis=1, kind="stable")[:, : cfg.k]
        return perm[top].astype(np.int32)
    raise ValueError(cfg.routing)


def topk_weights(cfg: MoeConfig) -> np.ndarray:
    """[N, K] gating weights: softmax over K of N(0,1) logits.

    Returned as float32, or as bf16 bit patterns (uint16) when the workload
    asks for bf16 gating weights.
    """
    z = normal_f64(cfg.seed, S_LOGITS, (cfg.n, cfg.k))
    z = np.exp(z - z.max(axis=1, keepdims=True))
    w = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return f32_to_bf16_bits(w) if cfg.gate_dtype == "bf16" else w


def weight_f32(cfg: MoeConfig, which: int, expert: int, shared: bool = False) -> np.ndarray:
    """fp32 N(0, 0.02) source weights of one expert, storage layout [N_out, K_red].

    which = 1: weight1, [2I, H] (rows [0, I) gate, [I, 2I) up);
    which = 2: weight2, [H, I] ([H, 2I] under gelu).
    """
    if which == 1:
        shape, stream = (2 * cfg.inter, cfg.h), (S_SW1 if shared else S_W1)
    else:
        shape, stream = (cfg.h, cfg.act_width), (S_SW2 if shared else S_W2)
    return normal_f32(cfg.seed, stream | expert, shape, scale=0.02)
