"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds no attention arithmetic: it only draws random numbers,
rounds them to bfloat16 and lays them out as ``[B, H, L, d]``.  Both the
float64 oracle and the CUDA path consume exactly the same bf16 bit patterns.

Workloads (GPT-2-small-like activations stand in for the trained model; the
pages' datasets are not used):

* ``tiny``   B=1 H=1  L=128   d=64,  LSSAR p=3 (small enough for the oracle)
* ``gpt2``   B=8 H=12 L=1024  d=64,  LSSAR p=3, also the softmax mode
* ``extrap`` B=1 H=12 L=8192  d=64,  LSSAR p=15
* ``needle`` B=1 H=12 L=16384 d=64,  LSSAR p=15, needle-structured queries
* ``wide``   B=4 H=16 L=4096  d=128, LSSA and LSSAR p in {1, 3, 15}

iid inputs: ``numpy.random.default_rng(seed)`` draws q, then k, then v as
float32 N(0, 1) and rounds each to bf16 (round to nearest even).

odd_key inputs (near-uniform rows): the generator draws q (float32 N(0,1),
rounded to bf16), then one key k0 per head and v, then per head a component
c uniform on 0..d-1.  Every key of the head is k0 except key 2 (1-based),
whose component c is moved away from zero by ``odd_ulps`` bf16 steps (its bit
pattern plus odd_ulps).  Each row then holds i-1 equal keys and one slightly
different one, so its LSSA row is uniform up to a small controlled spread.

needle inputs: the same generator draws k, then v (float32 N(0,1), rounded
to bf16), then j(i) uniform on the integers 1..i for every row i (1-based),
then noise ~ N(0, I/d) as float32.  Query i is
``0.9 * k_j / ||k_j|| + 0.44 * noise_i`` (k_j the bf16-rounded key, arithmetic
in float64), rounded to bf16.
"""

from dataclasses import dataclass

import numpy as np

MODE_SOFTMAX = 0
MODE_LSSA = 1
MODE_LSSAR = 2
MODE_SOFTMAX_RW = 3     # ablation: re-weighting on a softmax normaliser
MODE_SIGMOID_RW = 4     # ablation: sigmoid + L1 + re-weighting


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    d: int
    structure: str            # "iid" or "needle"
    runs: tuple               # ((mode, p), ...) exercised on this shape

    @property
    def shape(self):
        return (self.B, self.H, self.L, self.d)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 128, 64, "iid",
                     ((MODE_LSSAR, 3), (MODE_LSSA, 1), (MODE_SOFTMAX, 1))),
    "gpt2": Workload("gpt2", 8, 12, 1024, 64, "iid",
                     ((MODE_LSSAR, 3), (MODE_SOFTMAX, 1))),
    "extrap": Workload("extrap", 1, 12, 8192, 64, "iid", ((MODE_LSSAR, 15),)),
    "needle": Workload("needle", 1, 12, 16384, 64, "needle", ((MODE_LSSAR, 15),)),
    "wide": Workload("wide", 4, 16, 4096, 128, "iid",
                     ((MODE_LSSA, 1), (MODE_LSSAR, 1), (MODE_LSSAR, 3), (MODE_LSSAR, 15))),
}


def f32_to_bf16_bits(x):
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    r = np.where(nan, (u >> 16) | 0x40, r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b):
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(b):
    """Exact widening of bfloat16 bit patterns to float64."""
    return bf16_bits_to_f32(b).astype(np.float64)


def make_qkv(B, H, L, d, seed=0, structure="iid", odd_ulps=1):
    """Seeded q, k, v as uint16 bf16 bit arrays of shape [B, H, L, d]."""
    rng = np.random.default_rng(seed)
    shape = (B, H, L, d)
    if structure == "odd_key":
        q = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        k0 = f32_to_bf16_bits(rng.standard_normal((B, H, d), dtype=np.float32))
        v = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        c = rng.integers(0, d, size=(B, H))
        k = np.repeat(k0[:, :, None, :], L, axis=2).copy()
        if L >= 2:
            bi, hi = np.meshgrid(np.arange(B), np.arange(H), indexing="ij")
            k[bi, hi, 1, c] = (k0[bi, hi, c].astype(np.int64) + int(odd_ulps)).astype(np.uint16)
        return q, k, v
    if structure == "iid":
        q = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        k = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        v = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        return q, k, v
    if structure == "needle":
        k = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        v = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        hi = np.broadcast_to(np.arange(1, L + 1, dtype=np.int64)[None, None, :], (B, H, L))
        j = rng.integers(1, hi + 1)                      # uniform on 1..i (1-based)
        noise = rng.standard_normal(shape, dtype=np.float32).astype(np.float64) / np.sqrt(d)
        kf = bf16_bits_to_f64(k)
        kn = kf / np.maximum(np.sqrt(np.sum(kf * kf, axis=-1, keepdims=True)), 1e-30)
        picked = np.take_along_axis(kn, (j - 1)[..., None].repeat(d, axis=-1), axis=2)
        q = f32_to_bf16_bits((0.9 * picked + 0.44 * noise).astype(np.float32))
        return q, k, v
    raise ValueError(f"unknown structure {structure!r}")


def make_dout(B, H, L, d, seed=0):
    """Seeded upstream gradient of the output for the backward pass: float32
    N(0, 1) rounded to bf16 (uint16 bits, [B, H, L, d]), drawn from its own
    stream (seed, 1) so it never repeats q, k or v."""
    rng = np.random.default_rng([seed, 1])
    return f32_to_bf16_bits(rng.standard_normal((B, H, L, d), dtype=np.float32))


def make_workload(name, seed=0):
    """q, k, v bf16 bit arrays for a named workload."""
    w = WORKLOADS[name]
    return make_qkv(w.B, w.H, w.L, w.d, seed=seed, structure=w.structure)


def needle_targets(B, H, L, d, seed=0):
    """The j(i) (1-based) drawn by :func:`make_qkv` for the needle structure."""
    rng = np.random.default_rng(seed)
    shape = (B, H, L, d)
    rng.standard_normal(shape, dtype=np.float32)
    rng.standard_normal(shape, dtype=np.float32)
    hi = np.broadcast_to(np.arange(1, L + 1, dtype=np.int64)[None, None, :], (B, H, L))
    return rng.integers(1, hi + 1)
