"""Shared helpers for the libmx tests (host-side marshalling and checks)."""
from __future__ import annotations

import re

import numpy as np

from conftest import ROOT


def header_functions() -> list[str]:
    """Names of every function declared in include/mx.h."""
    src = open(f"{ROOT}/include/mx.h").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mx_\w+)\s*\(", src)))


def to_device_bits(bits: np.ndarray, in_dtype: str):
    """uint16 bit patterns -> CUDA tensor of bf16 / f16 with those bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    t = t.view(torch.bfloat16 if in_dtype == "bf16" else torch.float16)
    return t.cuda()


def to_device_u8(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def sf_pack(plain: np.ndarray) -> np.ndarray:
    """Test-side packing of plain E8M0 scales [mn, kb] into the tensor-core
    scale-factor layout documented in include/mx.h: 512-byte tiles of 128 rows
    x 4 scale columns, tile (tm, tk) at (tm * ceil(kb/4) + tk) * 512, scale
    (r, c) at (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4 inside its tile,
    padding 0."""
    mn, kb = plain.shape
    ntm, ntk = -(-mn // 128), -(-kb // 4)
    padded = np.zeros((ntm * 128, ntk * 4), np.uint8)
    padded[:mn, :kb] = plain
    # [tm, q(=r//32 within tile), r32, tk, c]
    t = padded.reshape(ntm, 4, 32, ntk, 4)
    t = t.transpose(0, 3, 2, 1, 4)  # [tm, tk, r32, q, c]
    return np.ascontiguousarray(t).reshape(-1)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """One bf16 unit in the last place at |x| (x as float64)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126.0)
    return np.where(ax > 0, np.exp2(e - 7), np.exp2(-133.0))


def check_gemm(c_gpu: np.ndarray, c_ref: np.ndarray, s_ref: np.ndarray, out_dtype: str,
               rel: float = 1e-4) -> float:
    """|C - C_ref| <= rel * sum_k |a_k b_k| (+ 1 bf16 ulp of C_ref for bf16
    output), element-wise.  Returns the largest error / allowance."""
    c = c_gpu.astype(np.float64)
    tol = rel * s_ref
    if out_dtype == "bf16":
        tol = tol + bf16_ulp(c_ref)
    err = np.abs(c - c_ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        details = [(tuple(i), float(c[tuple(i)]), float(c_ref[tuple(i)]), float(tol[tuple(i)])) for i in idx]
        raise AssertionError(f"{int(bad.sum())} elements out of tolerance, e.g. {details}")
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(tol > 0, err / tol, 0.0)
    return float(ratio.max()) if ratio.size else 0.0
