"""CPU oracle for the OCP-MX microscaling hot path (QuantizeMX + ScaledMatmul).

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the library and its Python binding
never do.  The oracle shares no code with the CUDA path: the arithmetic lives in
``mx_oracle.c`` (plain C, compiled here with gcc), and this module only
marshals numpy arrays into it.

Each function names the step of the page "MX Microscaling: Quantize,
Block-Scaling and E8M0" (or, for the matmul, the ScaledMatmul contract of the
page "MX-FP8 Microscaling Legalization", sections 3-4) that it follows.

Parity unpinned: the FP8 handling of NaN inputs (no page value fixes it; the
reading is NaN -> 0x7F | sign), and which FP4 lane stride / nibble parity the
silicon uses (both are parameters; the default reading is stride 2, parity 0).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmx_oracle.so")

IN_DTYPES = {"bf16": 0, "f16": 1}
FORMATS = {"e4m3fn": 0, "e5m2": 1, "e2m1": 2}
GEOMETRIES = {"8x4": 0, "1x32": 1}
LAYOUTS = {"plain": 0, "interleave": 1}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # MX_ORACLE_LIB points the tests at a deliberately broken build of the
        # oracle (see tests/test_oracle_mutants.py); unset in normal use.
        lib = ctypes.CDLL(os.environ.get("MX_ORACLE_LIB") or build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        sigs = {
            "mxo_widen_bf16": (ctypes.c_float, [ctypes.c_uint16]),
            "mxo_widen_f16": (ctypes.c_float, [ctypes.c_uint16]),
            "mxo_emax": (I, [I]),
            "mxo_emax_bias": (I, [I, I]),
            "mxo_exponent_byte": (ctypes.c_uint8, [ctypes.c_float]),
            "mxo_e8m0_from_max_exponent": (ctypes.c_uint8, [ctypes.c_uint8, I]),
            "mxo_prescale": (ctypes.c_float, [ctypes.c_float, ctypes.c_uint8]),
            "mxo_narrow": (ctypes.c_uint8, [I, ctypes.c_float]),
            "mxo_decode": (ctypes.c_double, [I, ctypes.c_uint8]),
            "mxo_decode_e2m1": (ctypes.c_float, [ctypes.c_uint8]),
            "mxo_decode_e8m0": (ctypes.c_double, [ctypes.c_uint8]),
            "mxo_lane_remap": (I64, [I64, I64]),
            "mxo_scale_row_slot": (I64, [I64, I]),
            "mxo_quantize": (I, [P, I, I64, I64, I64, I, I, I, I, I, I64, I, P, P]),
            "mxo_dequantize": (I, [P, P, I64, I64, I, I, I, I, I64, I, P]),
            "mxo_scaled_matmul_entries": (None, [P, P, P, P, I, I, I64, P, P, I64, P, P]),
            "mxo_dequantize_rows": (None, [P, P, I, I64, P, I64, P]),
            "mxo_narrow_array": (None, [I, P, I64, P]),
            "mxo_prescale_array": (None, [P, P, I64, P]),
            "mxo_widen_array": (None, [I, P, I64, P]),
            "mxo_exponent_byte_array": (None, [P, I64, P]),
            "mxo_decode_array": (None, [I, P, I64, P]),
            "mxo_pack_nibbles": (None, [P, I64, I64, I, P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ------------------------------------------------------------------ geometry

def block_extents(geometry: str, dim: int) -> tuple[int, int]:
    """(rows, cols) spanned by one 32-element block.

    8x4: 8 along the partition axis named by ``dim`` and 4 along the other
    (page 2, "Block geometry": 8 partitions x 4 free-dim columns).  1x32: 32
    consecutive elements along ``dim`` (the OCP block_size along the HLO dim).
    """
    if dim not in (-1, -2):
        raise ValueError("dim must be -1 or -2")
    if geometry == "8x4":
        return (8, 4) if dim == -2 else (4, 8)
    if geometry == "1x32":
        return (32, 1) if dim == -2 else (1, 32)
    raise ValueError(geometry)


def scale_shape(rows: int, cols: int, geometry: str, dim: int) -> tuple[int, int]:
    br, bc = block_extents(geometry, dim)
    return rows // br, cols // bc


def scale_buffer_rows(scale_rows: int, layout: str) -> int:
    """Rows of the scale buffer: plain = scale rows; interleaved = room for
    slot (i & 3) + 32 * (i >> 2) of every scale row, whole 32-row groups."""
    if layout == "plain":
        return scale_rows
    return 32 * ((scale_rows + 3) // 4)


def data_bytes(rows: int, cols: int, fmt: str) -> int:
    return rows * cols // 2 if fmt == "e2m1" else rows * cols


# ------------------------------------------------------------------ scalars

def widen_bf16(h: int) -> float:
    return _load().mxo_widen_bf16(h)


def widen_f16(h: int) -> float:
    return _load().mxo_widen_f16(h)


def emax(fmt: str) -> int:
    return _load().mxo_emax(FORMATS[fmt])


def emax_bias(fmt: str, emax_alt: bool = False) -> int:
    return _load().mxo_emax_bias(FORMATS[fmt], int(emax_alt))


def exponent_byte(x: float) -> int:
    return _load().mxo_exponent_byte(x)


def e8m0_from_max_exponent(max_exp: int, bias: int) -> int:
    return _load().mxo_e8m0_from_max_exponent(max_exp, bias)


def prescale(x: float, e8m0: int) -> float:
    return _load().mxo_prescale(x, e8m0)


def narrow(fmt: str, y: float) -> int:
    return _load().mxo_narrow(FORMATS[fmt], y)


def decode(fmt: str, code: int) -> float:
    return _load().mxo_decode(FORMATS[fmt], code)


def decode_e2m1_bits(nib: int) -> float:
    """The page's e2m1 decoder (binary32 bit construction)."""
    return _load().mxo_decode_e2m1(nib)


def decode_e8m0(e: int) -> float:
    return _load().mxo_decode_e8m0(e)


def lane_remap(index: int, stride: int) -> int:
    return _load().mxo_lane_remap(index, stride)


def scale_row_slot(i: int, layout: str) -> int:
    return _load().mxo_scale_row_slot(i, LAYOUTS[layout])


# ------------------------------------------------------------------- arrays

def narrow_array(fmt: str, y: np.ndarray) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.shape, np.uint8)
    _load().mxo_narrow_array(FORMATS[fmt], _ptr(y), y.size, _ptr(out))
    return out


def prescale_array(x: np.ndarray, e8m0: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    e = np.ascontiguousarray(np.broadcast_to(e8m0, x.shape), dtype=np.uint8)
    out = np.empty(x.shape, np.float32)
    _load().mxo_prescale_array(_ptr(x), _ptr(e), x.size, _ptr(out))
    return out


def widen_array(in_dtype: str, h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    _load().mxo_widen_array(IN_DTYPES[in_dtype], _ptr(h), h.size, _ptr(out))
    return out


def exponent_byte_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().mxo_exponent_byte_array(_ptr(x), x.size, _ptr(out))
    return out


def pack_nibbles(nibs, lane_stride: int = 2, nibble_parity: int = 0) -> np.ndarray:
    """The page's pack_nibble applied to element k = 0..n-1 in order."""
    n = np.ascontiguousarray(nibs, dtype=np.uint8)
    out = np.zeros(n.size // 2, np.uint8)
    _load().mxo_pack_nibbles(_ptr(n), n.size, lane_stride, nibble_parity, _ptr(out))
    return out


def decode_array(fmt: str, codes: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().mxo_decode_array(FORMATS[fmt], _ptr(c), c.size, _ptr(out))
    return out


# ----------------------------------------------------------------- quantize

class OracleError(RuntimeError):
    pass


def quantize(x: np.ndarray, in_dtype: str, out_fmt: str, *, geometry: str = "8x4",
             dim: int = -2, scale_layout: str = "plain", emax_alt: bool = False,
             lane_stride: int = 2, nibble_parity: int = 0, cols: int | None = None,
             scale_fill: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """QuantizeMX of a 2-D array of bf16/f16 bit patterns (uint16).

    ``x`` is [rows, ld]; ``cols`` (default ld) is the logical width.  Returns
    (data, scale): data is dense [rows, cols] bytes (FP8) or [rows, cols/2]
    packed nibbles (e2m1); scale is the scale buffer, [buffer rows, scale cols],
    pre-filled with ``scale_fill`` where the layout leaves rows unwritten.
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if x.ndim != 2:
        raise ValueError("2-D input expected")
    rows, ld = x.shape
    cols = ld if cols is None else cols
    srows, scols = scale_shape(rows, cols, geometry, dim) if rows and cols else (0, 0)
    data = np.zeros((rows, cols // 2 if out_fmt == "e2m1" else cols), np.uint8)
    scale = np.full((scale_buffer_rows(srows, scale_layout), scols), scale_fill, np.uint8)
    rc = _load().mxo_quantize(_ptr(x), IN_DTYPES[in_dtype], rows, cols, ld,
                              FORMATS[out_fmt], GEOMETRIES[geometry], dim,
                              LAYOUTS[scale_layout], int(emax_alt), lane_stride,
                              nibble_parity, _ptr(data), _ptr(scale))
    if rc != 0:
        raise OracleError(f"mxo_quantize failed with code {rc}")
    return data, scale


def dequantize(data: np.ndarray, scale: np.ndarray, rows: int, cols: int, fmt: str, *,
               geometry: str = "8x4", dim: int = -2, scale_layout: str = "plain",
               lane_stride: int = 2, nibble_parity: int = 0) -> np.ndarray:
    """Element values decode(code) * 2^(E8M0 - 127) in binary64, [rows, cols]."""
    data = np.ascontiguousarray(data, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.uint8)
    out = np.empty((rows, cols), np.float64)
    rc = _load().mxo_dequantize(_ptr(data), _ptr(scale), rows, cols, FORMATS[fmt],
                                GEOMETRIES[geometry], dim, LAYOUTS[scale_layout],
                                lane_stride, nibble_parity, _ptr(out))
    if rc != 0:
        raise OracleError(f"mxo_dequantize failed with code {rc}")
    return out


# ------------------------------------------------------------ scaled matmul

def scaled_matmul_entries(a, bt, sa, sb, fmt_a: str, fmt_b: str, ms, ns):
    """C[m, n] and S[m, n] = sum_k |a_k b_k| for each listed (m, n), straight
    from the definition in binary64 (k-ordered sum).  a [M,K], bt [N,K] FP8
    codes; sa [M,K/32], sb [N,K/32] plain E8M0."""
    a = np.ascontiguousarray(a, np.uint8)
    bt = np.ascontiguousarray(bt, np.uint8)
    sa = np.ascontiguousarray(sa, np.uint8)
    sb = np.ascontiguousarray(sb, np.uint8)
    ms = np.ascontiguousarray(ms, np.int64)
    ns = np.ascontiguousarray(ns, np.int64)
    c = np.empty(ms.shape, np.float64)
    s = np.empty(ms.shape, np.float64)
    _load().mxo_scaled_matmul_entries(_ptr(a), _ptr(bt), _ptr(sa), _ptr(sb),
                                      FORMATS[fmt_a], FORMATS[fmt_b], a.shape[1],
                                      _ptr(ms), _ptr(ns), ms.size, _ptr(c), _ptr(s))
    return c, s


def dequantize_rows(q, s, fmt: str, rows=None) -> np.ndarray:
    """Rows of a K-contiguous FP8 operand as binary64 values (plain scales)."""
    q = np.ascontiguousarray(q, np.uint8)
    s = np.ascontiguousarray(s, np.uint8)
    idx = np.arange(q.shape[0], dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    out = np.empty((idx.size, q.shape[1]), np.float64)
    _load().mxo_dequantize_rows(_ptr(q), _ptr(s), FORMATS[fmt], q.shape[1], _ptr(idx),
                                idx.size, _ptr(out))
    return out


def scaled_matmul(a, bt, sa, sb, fmt_a: str, fmt_b: str | None = None, rows=None, cols=None):
    """Dequantise-then-matmul in binary64 over a block of rows x cols.

    The matmul step is numpy's binary64 matmul (a library routine); products
    of dequantised values are exact in binary64, only the summation order
    differs from ``scaled_matmul_entries``.  Returns (C, S) for the selected
    rows (default all) and columns (default all).
    """
    fmt_b = fmt_a if fmt_b is None else fmt_b
    da = dequantize_rows(a, sa, fmt_a, rows)
    db = dequantize_rows(bt, sb, fmt_b, cols)
    return da @ db.T, np.abs(da) @ np.abs(db).T


# ---------------------------------------------------- general block-scaled dot

class DotDimsError(ValueError):
    """A dot-dimension-number check of the ScaledMatmul contract failed."""


def check_dot_dims(lhs_shape, rhs_shape, lhs_batch, rhs_batch, lhs_contract, rhs_contract):
    """The ScaledMatmul contract's checks (page "MX-FP8 Microscaling
    Legalization", section 4.2 and the ScaledMatmul verifier list): ranks >= 2;
    as many batch dimensions on each side, in bounds, of equal extents;
    contracting dimensions in bounds, of equal size and not overlapping the
    batch dimensions.  Reading: exactly one contracting dimension per side
    (MX blocks run along one axis), its extent a multiple of 32.  Negative
    indices count from the end."""
    lr, rr = len(lhs_shape), len(rhs_shape)
    if lr < 2 or rr < 2:
        raise DotDimsError("operands must have rank >= 2")
    if len(lhs_batch) != len(rhs_batch):
        raise DotDimsError("batch dimension counts differ")
    if len(lhs_contract) != 1 or len(rhs_contract) != 1:
        raise DotDimsError("exactly one contracting dimension per operand")

    def norm(d, r):
        d = int(d)
        if not -r <= d < r:
            raise DotDimsError(f"dimension {d} out of bounds for tensor of rank {r}")
        return d % r

    lb = [norm(d, lr) for d in lhs_batch]
    rb = [norm(d, rr) for d in rhs_batch]
    lc, rc = norm(lhs_contract[0], lr), norm(rhs_contract[0], rr)
    if len(set(lb)) != len(lb) or len(set(rb)) != len(rb):
        raise DotDimsError("repeated batch dimension")
    if lc in lb or rc in rb:
        raise DotDimsError("contracting dimension overlaps a batch dimension")
    for a, b in zip(lb, rb):
        if lhs_shape[a] != rhs_shape[b]:
            raise DotDimsError("batch extents differ")
    if lhs_shape[lc] != rhs_shape[rc]:
        raise DotDimsError("contracting extents differ")
    if lhs_shape[lc] % 32 != 0:
        raise DotDimsError("contracting extent not a multiple of the 32-element block")
    return lb, rb, lc, rc


def block_values(codes, scale, fmt: str, axis: int) -> np.ndarray:
    """decode(code) * 2^(E8M0 - 127) in binary64 for an N-d FP8 operand whose
    scale tensor is the operand's shape with `axis` divided by 32 (one E8M0 per
    32 consecutive elements along `axis`)."""
    codes = np.asarray(codes, np.uint8)
    scale = np.asarray(scale, np.uint8)
    e8m0 = np.array([decode_e8m0(e) for e in range(256)], np.float64)
    return decode_array(fmt, codes) * np.repeat(e8m0[scale], 32, axis=axis)


def block_scaled_dot(lhs, rhs, lhs_scale, rhs_scale, fmt: str, *, lhs_batch=(), rhs_batch=(),
                     lhs_contract=(-1,), rhs_contract=(-1,), fmt_rhs: str | None = None):
    """block_scaled_dot(lhs, rhs, lhs_scale, rhs_scale) with dot dimension
    numbers (page "MX-FP8 Microscaling Legalization", sections 3.2 and 4.2):

      out[b..., i..., j...] = sum_k  lhs_val[.., k, ..] * rhs_val[.., k, ..]

    over the contracting axis k, with the batch axes b paired in the listed
    order, i the remaining lhs axes and j the remaining rhs axes in their own
    order (the dot-general result order: batch, lhs free, rhs free).  Values
    are decode(code) * 2^(E8M0 - 127) (block_values).  The contraction is
    numpy's binary64 einsum (a library routine; every product is exact in
    binary64).  Returns (C, S), S the same sum over |products|.
    """
    lhs = np.asarray(lhs, np.uint8)
    rhs = np.asarray(rhs, np.uint8)
    lb, rb, lc, rc = check_dot_dims(lhs.shape, rhs.shape, lhs_batch, rhs_batch, lhs_contract, rhs_contract)
    vl = block_values(lhs, lhs_scale, fmt, lc)
    vr = block_values(rhs, rhs_scale, fmt if fmt_rhs is None else fmt_rhs, rc)
    letters = iter("abcdefghijklmnopqrstuvwxyz")
    ls, rs = [None] * lhs.ndim, [None] * rhs.ndim
    batch = []
    for a, b in zip(lb, rb):
        ls[a] = rs[b] = next(letters)
        batch.append(ls[a])
    ls[lc] = rs[rc] = next(letters)
    lfree = [i for i in range(lhs.ndim) if ls[i] is None]
    rfree = [i for i in range(rhs.ndim) if rs[i] is None]
    for i in lfree:
        ls[i] = next(letters)
    for i in rfree:
        rs[i] = next(letters)
    out = "".join(batch) + "".join(ls[i] for i in lfree) + "".join(rs[i] for i in rfree)
    sub = f"{''.join(ls)},{''.join(rs)}->{out}"
    return np.einsum(sub, vl, vr), np.einsum(sub, np.abs(vl), np.abs(vr))
