"""Seeded synthetic inputs for the MX hot path (tests and benchmark).

This module only draws input tensors: bf16/f16 bit patterns (uint16 numpy
arrays) with the shapes and value distributions of the workloads below.  It
holds none of the quantizer's or the matmul's arithmetic, and imports neither
the oracle nor the CUDA binding; both sides receive the same arrays from here.

Workloads (seed 0 unless a caller says otherwise; tensor i of a workload uses
seed + i):

* ``pipeline_operands``  -- A[M,K], Bt[N,K] = N(0,1) * 2^U(-20,20), one factor
  per 32 consecutive elements along K (the MX-FP8 pipeline at 256^3).
* ``sweep_input``        -- [R,C] = N(0,1) * 2^U(-30,30), one factor per
  8-row x 4-column block, plus four injected block kinds on 1% of blocks
  each (disjoint): all-zero (with -0), subnormal-only, at-max, exact ties.
* ``gemm_operands``      -- A[M,K], Bt[N,K] = N(0,1) * 2^U(-8,8) per row.
* ``fused_operands``     -- X[M,K] = N(0,1), each element x100 with prob 1e-3;
  the weight W[K,N] = N(0, 0.02) is drawn directly in its K-contiguous
  transposed layout Wt[N,K] (i.i.d. entries, so the layout does not change
  the distribution).
* ``fp4_input``          -- [R,C] = N(0,1) * 2^U(-20,20) per 8x4 block, with 2%
  of blocks made of exact e2m1 grid-midpoint ties around an anchor.
* ``special_values``     -- small tensors of +-0, subnormals, format maxima,
  Inf and NaN for edge-case tests.

The tie and at-max constructions use only the published definitions of the
target element formats (e4m3fn: 3 fraction bits, normal exponents -6..8,
max 448; e5m2: 2 fraction bits, normal exponents -14..15, max 57344; e2m1:
grid {0, .5, 1, 1.5, 2, 3, 4, 6}).
"""
from __future__ import annotations

import numpy as np

BF16_MAX_BITS = 0x7F7F  # largest finite bf16
F16_MAX_BITS = 0x7BFF   # 65504

_FMT_MAX = {"e4m3fn": 448.0, "e5m2": 57344.0, "e2m1": 6.0}


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(seed))


def to_bits(x: np.ndarray, in_dtype: str) -> np.ndarray:
    """Round binary32 values to bf16 / f16 (nearest-even) and return the bit
    patterns as uint16.  Uses torch's / numpy's own conversions."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if in_dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if in_dtype == "bf16":
        import torch
        return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    raise ValueError(in_dtype)


def from_bits(h: np.ndarray, in_dtype: str) -> np.ndarray:
    """bf16/f16 bit patterns -> binary32 values (library conversions)."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    if in_dtype == "f16":
        return h.view(np.float16).astype(np.float32)
    return (h.astype(np.uint32) << 16).view(np.float32)


def _normal(rng, n) -> np.ndarray:
    return rng.standard_normal(n, dtype=np.float32)


# ------------------------------------------------------------- config 1 / 3

def pipeline_operands(M: int = 256, N: int = 256, K: int = 256, seed: int = 0):
    """A[M,K], Bt[N,K] bf16 bits: N(0,1) * 2^U(-20,20) per 32-block along K."""
    out = []
    for i, rows in enumerate((M, N)):
        rng = _rng(seed + i)
        x = _normal(rng, rows * K).reshape(rows, K // 32, 32)
        e = rng.integers(-20, 21, size=(rows, K // 32, 1)).astype(np.float32)
        out.append(to_bits((x * np.exp2(e)).reshape(rows, K), "bf16"))
    return out[0], out[1]


def gemm_operands(M: int = 8192, N: int = 8192, K: int = 8192, seed: int = 0):
    """A[M,K], Bt[N,K] bf16 bits: N(0,1) * 2^U(-8,8), one factor per row."""
    out = []
    for i, rows in enumerate((M, N)):
        rng = _rng(seed + i)
        x = _normal(rng, rows * K).reshape(rows, K)
        e = rng.integers(-8, 9, size=(rows, 1)).astype(np.float32)
        x *= np.exp2(e)
        out.append(to_bits(x, "bf16"))
    return out[0], out[1]


# --------------------------------------------------------------- config 2

def _tie_values(out_fmt: str) -> np.ndarray:
    """Exact midpoints between adjacent codes of the target format (magnitudes),
    normal and subnormal range, every midpoint below the format maximum."""
    if out_fmt == "e4m3fn":
        mbits, emin, emax_, maxv = 3, -6, 8, 448.0
    elif out_fmt == "e5m2":
        mbits, emin, emax_, maxv = 2, -14, 15, 57344.0
    else:
        raise ValueError(out_fmt)
    vals = []
    q = 2.0 ** (emin - mbits)  # subnormal quantum
    for j in range(2 ** mbits):
        vals.append((2 * j + 1) * q / 2)
    for e in range(emin, emax_ + 1):
        for f in range(2 ** mbits):
            v = (1 + (2 * f + 1) / 2 ** (mbits + 1)) * 2.0 ** e
            if v + 2.0 ** (e - mbits - 1) <= maxv:  # both neighbours representable
                vals.append(v)
    return np.array(vals, np.float64)


def sweep_input(rows: int = 8192, cols: int = 8192, in_dtype: str = "bf16",
                out_fmt: str = "e4m3fn", seed: int = 0, inject: bool = True) -> np.ndarray:
    """QuantizeMX sweep input (8-row x 4-column blocks), uint16 bits [rows, cols].

    Per block: N(0,1) * 2^u, u ~ U(-30,30) (clamped to <= 11 for f16 so that no
    element overflows; blocks that underflow become subnormal or zero).
    Injected on disjoint random 1% subsets of blocks:
      (i)   all-zero blocks, each element +0 or -0;
      (ii)  subnormal-only blocks: random non-zero subnormal patterns of the
            input format with random signs;
      (iii) at-max blocks: half hold +-(largest finite input value) in one
            element, half have a block maximum of exactly fmt_max * 2^k
            (fmt_max the target format's largest finite value);
      (iv)  exact-tie blocks: one anchor +-fmt_max * 2^k fixes the scale, the
            other 31 elements are exact midpoints between adjacent target codes
            times 2^k, drawn over the normal and subnormal ranges.
    """
    assert rows % 8 == 0 and cols % 4 == 0
    rng = _rng(seed)
    gr, gc = rows // 8, cols // 4
    nblk = gr * gc
    x = _normal(rng, rows * cols).reshape(gr, 8, gc, 4)
    hi = 11 if in_dtype == "f16" else 30
    u = np.minimum(rng.integers(-30, 31, size=(gr, 1, gc, 1)), hi).astype(np.float32)
    x *= np.exp2(u)
    bits = to_bits(x.reshape(rows, cols), in_dtype).reshape(gr, 8, gc, 4)
    if not inject or nblk < 8:
        return bits.reshape(rows, cols)

    # block-major view: [nblk, 32] with block id = g * gc + c
    blk = bits.transpose(0, 2, 1, 3).reshape(nblk, 32)
    n1 = max(1, nblk // 100)
    chosen = rng.choice(nblk, size=4 * n1, replace=False)
    zero_ids, sub_ids, max_ids, tie_ids = np.split(chosen, 4)
    sign = lambda n: (rng.integers(0, 2, size=n).astype(np.uint16) << 15)

    # (i) all-zero with signed zeros
    blk[zero_ids] = sign(zero_ids.size * 32).reshape(-1, 32)
    # (ii) subnormal-only
    mant_max = 0x7F if in_dtype == "bf16" else 0x3FF
    mant = rng.integers(1, mant_max + 1, size=(sub_ids.size, 32)).astype(np.uint16)
    blk[sub_ids] = mant | sign(sub_ids.size * 32).reshape(-1, 32)
    # (iii) at-max
    fmt_max = _FMT_MAX[out_fmt]
    half = max_ids.size // 2
    pos = rng.integers(0, 32, size=max_ids.size)
    in_max = BF16_MAX_BITS if in_dtype == "bf16" else F16_MAX_BITS
    blk[max_ids[:half], pos[:half]] = np.uint16(in_max) | sign(half)
    if in_dtype == "bf16":
        klo, khi = -60, 60
    else:  # keep fmt_max * 2^k finite and the block's other values in range
        klo, khi = (-4, 7) if out_fmt == "e4m3fn" else (-10, 0)
    nb = max_ids.size - half
    top = fmt_max * np.exp2(rng.integers(klo, khi + 1, size=(nb, 1)).astype(np.float64))
    vals = np.clip(rng.standard_normal((nb, 32)) * (top / 8), -top, top)
    vals[np.arange(nb), pos[half:]] = top[:, 0] * np.where(rng.integers(0, 2, nb) == 1, -1.0, 1.0)
    blk[max_ids[half:]] = to_bits(vals.astype(np.float32), in_dtype)
    # (iv) exact ties
    ties = _tie_values(out_fmt)
    if in_dtype == "bf16":
        klo, khi = -30, 30
    else:
        klo, khi = (-10, 5) if out_fmt == "e4m3fn" else (-7, 0)
    nt = tie_ids.size
    scale = np.exp2(rng.integers(klo, khi + 1, size=(nt, 1)).astype(np.float64))
    vals = rng.choice(ties, size=(nt, 32)) * scale * np.where(rng.integers(0, 2, (nt, 32)) == 1, -1.0, 1.0)
    vals[np.arange(nt), rng.integers(0, 32, size=nt)] = (
        fmt_max * scale[:, 0] * np.where(rng.integers(0, 2, nt) == 1, -1.0, 1.0))
    blk[tie_ids] = to_bits(vals.astype(np.float32), in_dtype)

    bits = blk.reshape(gr, gc, 8, 4).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(bits).reshape(rows, cols)


# --------------------------------------------------------------- config 4

def fused_operands(M: int = 16384, N: int = 28672, K: int = 8192, seed: int = 0):
    """X[M,K] bf16 bits: N(0,1), each element x100 with probability 1e-3.
    Wt[N,K] bf16 bits: N(0, 0.02) (the weight W[K,N], stored transposed)."""
    rng = _rng(seed)
    x = _normal(rng, M * K)
    out = rng.random(M * K, dtype=np.float32) < 1e-3
    x[out] *= 100.0
    xb = to_bits(x.reshape(M, K), "bf16")
    rng = _rng(seed + 1)
    w = _normal(rng, N * K) * np.float32(0.02)
    return xb, to_bits(w.reshape(N, K), "bf16")


# --------------------------------------------------------------- config 5

_E2M1_TIES = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def fp4_input(rows: int = 16384, cols: int = 16384, seed: int = 0,
              tie_fraction: float = 0.02) -> np.ndarray:
    """FP4 sweep input (8x4 blocks), bf16 bits [rows, cols].

    Per block N(0,1) * 2^u, u ~ U(-20,20).  A ``tie_fraction`` share of blocks
    hold one anchor +-4 * 2^u (it fixes the block's scale at 127 + u) and 31
    exact e2m1 grid midpoints {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5} * 2^u with
    random signs.
    """
    assert rows % 8 == 0 and cols % 4 == 0
    rng = _rng(seed)
    gr, gc = rows // 8, cols // 4
    x = _normal(rng, rows * cols).reshape(gr, 8, gc, 4)
    u = rng.integers(-20, 21, size=(gr, 1, gc, 1))
    x *= np.exp2(u.astype(np.float32))
    bits = to_bits(x.reshape(rows, cols), "bf16").reshape(gr, 8, gc, 4)
    nblk = gr * gc
    nt = int(round(nblk * tie_fraction))
    if nt == 0:
        return bits.reshape(rows, cols)
    blk = bits.transpose(0, 2, 1, 3).reshape(nblk, 32)
    ids = rng.choice(nblk, size=nt, replace=False)
    uu = u.reshape(nblk)[ids].astype(np.float64)
    vals = rng.choice(_E2M1_TIES, size=(nt, 32)) * np.where(rng.integers(0, 2, (nt, 32)) == 1, -1.0, 1.0)
    anchor = rng.integers(0, 32, size=nt)
    vals[np.arange(nt), anchor] = 4.0 * np.where(rng.integers(0, 2, nt) == 1, -1.0, 1.0)
    vals *= np.exp2(uu)[:, None]
    blk[ids] = to_bits(vals.astype(np.float32), "bf16")
    bits = blk.reshape(gr, gc, 8, 4).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(bits).reshape(rows, cols)


# ------------------------------------------------------------- edge cases

def special_values(in_dtype: str = "bf16") -> np.ndarray:
    """A pool of edge-case bit patterns for the input format: signed zeros,
    the smallest and largest subnormals, the smallest normal, +-1, the
    largest finite value, +-Inf and NaNs of both signs (quiet, and with other
    payloads)."""
    if in_dtype == "bf16":
        pats = [0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x0080, 0x3F80, 0xBF80,
                0x7F7F, 0xFF7F, 0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x7F81, 0xFFA4, 0x4000, 0x3F00]
    else:
        pats = [0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x0400, 0x3C00, 0xBC00,
                0x7BFF, 0xFBFF, 0x7C00, 0xFC00, 0x7E00, 0xFE00, 0x7C01, 0xFD55, 0x4000, 0x3800]
    return np.array(pats, np.uint16)


def random_bits(rows: int, cols: int, in_dtype: str = "bf16", seed: int = 0,
                special_fraction: float = 0.0, block_exp: tuple[int, int] | None = None,
                block: tuple[int, int] = (8, 4)) -> np.ndarray:
    """General small-test input: N(0,1) with an optional per-block 2^U(lo,hi)
    factor over blocks of ``block`` (rows, cols), and a fraction of elements
    replaced by ``special_values`` patterns."""
    rng = _rng(seed)
    x = _normal(rng, rows * cols).reshape(rows, cols)
    if block_exp is not None:
        br, bc = block
        lo, hi = block_exp
        u = rng.integers(lo, hi + 1, size=(rows // br, 1, cols // bc, 1)).astype(np.float32)
        x = (x.reshape(rows // br, br, cols // bc, bc) * np.exp2(u)).reshape(rows, cols)
    bits = to_bits(x, in_dtype)
    if special_fraction > 0:
        m = rng.random((rows, cols)) < special_fraction
        pool = special_values(in_dtype)
        bits[m] = rng.choice(pool, size=int(m.sum()))
    return bits
