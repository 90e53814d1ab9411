"""Seeded synthetic inputs shared bit-for-bit by the CUDA path and the oracle.

This module holds no attention arithmetic: it only draws numbers.  It is the
single input source for the tests, the benchmark and the smoke check, so both
sides of every parity comparison see identical bits.

Generator (each piece implemented from its published definition):
  * SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014): state advances by the golden-ratio increment
    0x9E3779B97F4A7C15 and each output is the state passed through the
    variant-13 finaliser (shifts 30, 27, 31; multipliers 0xBF58476D1CE4E5B9,
    0x94D049BB133111EB).  The k-th output depends only on (seed, k), so the
    stream is generated counter-style, vectorised, in chunks.
  * A uniform in (0, 1) from the top 53 bits: (x >> 11 + 0.5) * 2^-53.
  * Box-Muller (1958): outputs 2m and 2m+1 give u1, u2 and the normal pair
    r cos(2 pi u2), r sin(2 pi u2) with r = sqrt(-2 ln u1).
  * Round-to-nearest-even from double straight to IEEE binary16 or bfloat16.

Workloads: the shapes, dtypes, scales, masks and value distributions of the
pages' examples (an N=128 / N=4096 single head with d=64, as in the
tiny-flash-attention walkthrough and the HBM-traffic example of "CUDA 算子工程"
ch. 14), widened to multi-head batches.  Seeds are 1000*k + {0, 1, 2} for
Q, K, V of workload k.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

FP16 = 0
BF16 = 1
DTYPE_NAMES = {FP16: "fp16", BF16: "bf16"}

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 (0-based) of SplitMix64 seeded with `seed`."""
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + k * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def normals(seed: int, n: int) -> np.ndarray:
    """n iid standard normals (float64) from SplitMix64 + Box-Muller."""
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, 2 * _CHUNK):
        hi = min(n, lo + 2 * _CHUNK)
        out[lo:hi] = normals_range(seed, lo, hi)
    return out


def round_to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float64 values to nearest-even binary16 / bfloat16; return uint16 bits."""
    x = np.asarray(x, dtype=np.float64)
    # significant bits and smallest subnormal exponent of the target format
    prec, emin_sub = (11, -24) if dtype == FP16 else (8, -133)
    _, e = np.frexp(x)
    qexp = np.maximum(e - prec, emin_sub)
    quantum = np.ldexp(1.0, qexp)
    y = np.rint(x / quantum) * quantum                 # np.rint rounds half to even
    if dtype == FP16:
        with np.errstate(over="ignore"):
            return y.astype(np.float16).view(np.uint16)
    return (y.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bits_to_float(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact float32 view of 16-bit patterns (for host-side checks and plots)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == FP16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def tensor_bits(seed: int, shape, dtype: int, mult: float = 1.0) -> np.ndarray:
    """A tensor of iid N(0, mult^2) values, rounded to `dtype`, as uint16 bits.

    Element e is output e of the stream whatever the chunking, so the chunks
    are drawn on several threads (numpy releases the GIL in its array loops)
    with the same bits as one pass."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)

    def chunk(s0):                              # chunk starts stay even: pairs stay whole
        s1 = min(n, s0 + 2 * _CHUNK)
        out[s0:s1] = round_to_bits(normals_range(seed, s0, s1) * mult, dtype)

    starts = range(0, n, 2 * _CHUNK)
    if len(starts) > 1:
        workers = min(len(starts), os.cpu_count() or 1, 16)
        with ThreadPoolExecutor(workers) as pool:
            list(pool.map(chunk, starts))
    else:
        for s0 in starts:
            chunk(s0)
    return out.reshape(shape)


def normals_range(seed: int, lo: int, hi: int) -> np.ndarray:
    """Elements lo .. hi-1 (lo even) of the normal stream of `seed`."""
    assert lo % 2 == 0
    npairs = (hi - lo + 1) // 2
    raw = splitmix64(seed, lo, 2 * npairs)
    u = ((raw >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    pair = np.empty((npairs, 2), dtype=np.float64)
    pair[:, 0] = r * np.cos(t)
    pair[:, 1] = r * np.sin(t)
    return pair.reshape(-1)[: hi - lo]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: int
    scale: float
    causal: bool
    seed_base: int
    qk_mult: float = 1.0
    v_mult: float = 1.0
    note: str = ""

    @property
    def shape(self):
        return (self.B, self.H, self.N, self.d)

    @property
    def flops(self) -> float:
        """4*B*H*N^2*d, halved for the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def compulsory_bytes(self) -> int:
        """Q, K, V read once and O written once (16-bit) plus the fp32 LSE."""
        n = self.B * self.H * self.N * self.d
        return 4 * 2 * n + 4 * self.B * self.H * self.N

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "N": self.N, "d": self.d,
                "dtype": DTYPE_NAMES[self.dtype], "scale": self.scale,
                "causal": self.causal, "qk_std": self.qk_mult, "seed_base": self.seed_base}


WORKLOADS = {
    w.name: w for w in [
        Workload("C1_b1h1n128d64_fp16", 1, 1, 128, 64, FP16, 1 / 8, False, 1000,
                 note="walkthrough shape: L=128, D=64, BlockM=BlockN=64"),
        Workload("C2_b1h1n4096d64_fp16", 1, 1, 4096, 64, FP16, 1 / 8, False, 2000,
                 note="the HBM-traffic example shape, one head"),
        Workload("C2x16_b1h16n4096d64_fp16", 1, 16, 4096, 64, FP16, 1 / 8, False, 2100,
                 note="the traffic example shape, 16 heads: S and P (512 MiB each) exceed L2"),
        Workload("C3_b4h16n4096d64_fp16_causal", 4, 16, 4096, 64, FP16, 1 / 8, True, 3000),
        Workload("C4_b2h32n8192d128_bf16", 2, 32, 8192, 128, BF16, 1 / math.sqrt(128), False,
                 4000, qk_mult=2.0, note="Q, K drawn with std 2 to widen the score range"),
        Workload("C5_b1h8n16384d128_bf16_causal", 1, 8, 16384, 128, BF16, 1 / math.sqrt(128),
                 True, 5000),
        Workload("C5r_b1h8n4000d128_bf16_causal", 1, 8, 4000, 128, BF16, 1 / math.sqrt(128),
                 True, 5000, note="ragged: N not a multiple of the 128-row tile"),
        Workload("T_b2h32n4096d128_bf16", 2, 32, 4096, 128, BF16, 1 / math.sqrt(128), False,
                 6000, note="N=4096, d=128 non-causal throughput point"),
        Workload("T_b2h32n4096d128_fp16", 2, 32, 4096, 128, FP16, 1 / math.sqrt(128), False,
                 7000),
        Workload("D256_b2h16n4096d256_bf16", 2, 16, 4096, 256, BF16, 1 / 16, False, 8000,
                 note="wide head: same FLOPs per launch as T, d=256"),
        Workload("D256c_b2h16n4096d256_bf16_causal", 2, 16, 4096, 256, BF16, 1 / 16, True, 8100),
        Workload("D192_b2h16n4096d192_bf16", 2, 16, 4096, 192, BF16, 1 / math.sqrt(192), False,
                 8200),
        Workload("D96_b2h32n4096d96_bf16", 2, 32, 4096, 96, BF16, 1 / math.sqrt(96), False, 8300,
                 note="d=96 served by the 128-wide kernel with zero-filled columns"),
    ]
}


def workload(name: str) -> Workload:
    for key, w in WORKLOADS.items():
        if key == name or key.split("_")[0] == name:
            return w
    raise KeyError(name)


def make_inputs(w: Workload, shape=None, seed_base: int | None = None):
    """(q, k, v) uint16 bit tensors [B, H, N, d] for workload `w`."""
    shape = shape or w.shape
    sb = w.seed_base if seed_base is None else seed_base
    q = tensor_bits(sb + 0, shape, w.dtype, w.qk_mult)
    k = tensor_bits(sb + 1, shape, w.dtype, w.qk_mult)
    v = tensor_bits(sb + 2, shape, w.dtype, w.v_mult)
    return q, k, v


def sample_rows(BH: int, N: int, count: int, seed: int, include_edges: bool = True) -> np.ndarray:
    """Flat row indices bh*N + i to check at full size: a seeded spread plus edges."""
    raw = splitmix64(seed, 0, max(count, 1))
    picks = (raw % np.uint64(BH * N)).astype(np.int64)
    rows = [picks]
    if include_edges:
        edge_i = sorted({0, 1, N // 2, N - 2, N - 1} & set(range(N)))
        for bh in sorted({0, BH - 1}):
            rows.append(np.array([bh * N + i for i in edge_i], dtype=np.int64))
    return np.unique(np.concatenate(rows))
