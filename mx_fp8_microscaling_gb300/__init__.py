"""Python binding of libmx (OCP-MX microscaling on sm_103a).

Argument marshalling only: every computation runs in the CUDA kernels of
``libmx.so`` (built in-tree by ``build.py``).  Tensors are PyTorch CUDA
tensors; PyTorch supplies device memory and the current stream.  Importing
this package raises if the library has not been built: there is no fallback.

The functions carry the C-ABI names of ``include/mx.h``:

    mx_quantize(x, out_dtype, ...)            -> (data, scale)
    mx_quantize_sizes(...)                    -> (data_bytes, scale_rows, scale_cols)
    mx_repack_scales(plain, k)                -> sf
    mx_sf_layout_bytes(mn, k)                 -> int
    mx_scaled_matmul(a, bt, a_scale, b_scale, ...) -> c
    mx_fused_quantize_matmul(x, wt, w_scale_sf, ...) -> c
    mx_get_device_status()                    -> int
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmx.so")

# enum values of include/mx.h
MX_OK = 0
MX_ERR_INVALID_ARG = 1
MX_ERR_TIMEOUT = 9
DTYPES = {"bf16": 1, "f16": 2, "f32": 3, "e4m3fn": 4, "e5m2": 5, "e2m1": 6, "e8m0": 7}
GEOMETRIES = {"8x4": 0, "1x32": 1}
LAYOUTS = {"plain": 0, "interleave": 1, "sf": 2}
STATUS_NAMES = {0: "MX_OK", 1: "MX_ERR_INVALID_ARG", 2: "MX_ERR_UNSUPPORTED_DTYPE", 3: "MX_ERR_BLOCK_SIZE",
                4: "MX_ERR_DIM", 5: "MX_ERR_SHAPE", 6: "MX_ERR_ALIGNMENT", 7: "MX_ERR_WORKSPACE",
                8: "MX_ERR_CUDA", 9: "MX_ERR_TIMEOUT", 10: "MX_ERR_DEVICE", 11: "MX_ERR_SCALE_METHOD"}


class MxError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


MAX_RANK = 8


class DotDims(ctypes.Structure):
    _fields_ = [("lhs_n_batch", ctypes.c_int32), ("rhs_n_batch", ctypes.c_int32),
                ("lhs_batch", ctypes.c_int64 * MAX_RANK), ("rhs_batch", ctypes.c_int64 * MAX_RANK),
                ("lhs_n_contract", ctypes.c_int32), ("rhs_n_contract", ctypes.c_int32),
                ("lhs_contract", ctypes.c_int64 * MAX_RANK), ("rhs_contract", ctypes.c_int64 * MAX_RANK)]


class QuantCfg(ctypes.Structure):
    _fields_ = [("geometry", ctypes.c_int32), ("scale_layout", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("dim", ctypes.c_int32),
                ("scale_method", ctypes.c_int32), ("fp4_lane_stride", ctypes.c_int32),
                ("fp4_nibble_parity", ctypes.c_int32), ("emax_alt", ctypes.c_int32)]


class HostJob(ctypes.Structure):
    _fields_ = [("in_host", ctypes.c_void_p), ("in_dtype", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("ld_in", ctypes.c_int64), ("out_dtype", ctypes.c_int32),
                ("cfg", QuantCfg), ("out_data_host", ctypes.c_void_p), ("out_scale_host", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmx is not built ({LIB_PATH} missing); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    PS = ctypes.POINTER(SZ)
    PI64 = ctypes.POINTER(I64)
    sigs = {
        "mx_quant_cfg_default": [ctypes.POINTER(QuantCfg)],
        "mx_quantize_sizes": [I, I, I64, I64, ctypes.POINTER(QuantCfg), PS, PI64, PI64, PS],
        "mx_quantize": [P, I, I64, I64, I64, I, ctypes.POINTER(QuantCfg), P, P, P],
        "mx_dequantize": [P, P, I, I64, I64, ctypes.POINTER(QuantCfg), I, P, I64, P],
        "mx_quantize_host_workspace": [I, I64, I64, I, ctypes.POINTER(QuantCfg), I64, PS],
        "mx_quantize_host": [P, I, I64, I64, I64, I, ctypes.POINTER(QuantCfg), P, P, I64, P, SZ, P],
        "mx_quantize_host_batch_workspace": [ctypes.POINTER(HostJob), I, I64, PS],
        "mx_quantize_host_batch": [ctypes.POINTER(HostJob), I, I64, P, SZ, P],
        "mx_sf_layout_bytes": [I64, I64, PS],
        "mx_repack_scales": [P, I64, I64, I64, P, P],
        "mx_scaled_matmul_workspace": [I64, I64, I64, I, PS],
        "mx_scaled_matmul": [P, P, P, P, I, I, I64, I64, I64, I, P, I64, P, SZ, P],
        "mx_scaled_matmul_noalloc": [P, P, P, P, I, I64, I64, I64, I, P, I64, P],
        "mx_fused_quantize_matmul_workspace": [I64, I64, I64, PS],
        "mx_fused_quantize_matmul": [P, I, I64, P, P, I, I64, I64, I64, I, P, I64, P, SZ, P],
        "mx_block_scaled_dot_shape": [PI64, I, PI64, I, ctypes.POINTER(DotDims), PI64, ctypes.POINTER(I)],
        "mx_block_scaled_dot_workspace": [PI64, I, PI64, I, ctypes.POINTER(DotDims), PS],
        "mx_block_scaled_dot": [P, PI64, I, P, P, PI64, I, P, ctypes.POINTER(DotDims), I, I, P, P, SZ, P],
        "mx_get_device_status": [ctypes.POINTER(I)],
        "mx_status_string": [I],
        "mx_version": [],
        "mx_debug_gemm_fault_injection": [I, ctypes.c_uint64],
        "mx_debug_set_gemm_variant": [I],
        "mx_debug_last_gemm_launch": [P, P],
        "mx_debug_last_gemm_operands": [P, P],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "mx_status_string" else I
    return lib


_lib = _load()


def _check(status: int, what: str):
    if status != MX_OK:
        raise MxError(status, what)


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev_ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmx takes CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _in_dtype(t: torch.Tensor) -> str:
    if t.dtype == torch.bfloat16:
        return "bf16"
    if t.dtype == torch.float16:
        return "f16"
    raise ValueError(f"QuantizeMX input must be bf16 or f16, got {t.dtype}")


def make_cfg(geometry="8x4", dim=-2, scale_layout="plain", fp4_lane_stride=2, fp4_nibble_parity=0,
             emax_alt=False, block_size=32, scale_method=0) -> QuantCfg:
    cfg = QuantCfg()
    _lib.mx_quant_cfg_default(ctypes.byref(cfg))
    cfg.geometry = GEOMETRIES[geometry] if isinstance(geometry, str) else geometry
    cfg.scale_layout = LAYOUTS[scale_layout] if isinstance(scale_layout, str) else scale_layout
    cfg.block_size = block_size
    cfg.dim = dim
    cfg.scale_method = scale_method
    cfg.fp4_lane_stride = fp4_lane_stride
    cfg.fp4_nibble_parity = fp4_nibble_parity
    cfg.emax_alt = int(emax_alt)
    return cfg


def _view2d(x: torch.Tensor, dim: int) -> tuple[int, int, int]:
    """Rows, cols and row pitch of the 2-D view of x: leading dimensions fold
    into rows (the last dimension must be contiguous)."""
    if x.dim() < 2:
        raise ValueError("QuantizeMX needs rank >= 2")
    if x.stride(-1) != 1:
        raise ValueError("the last dimension must be contiguous")
    cols = x.shape[-1]
    rows = 1
    for s in x.shape[:-1]:
        rows *= s
    ld = x.stride(-2) if x.dim() >= 2 else cols
    # leading dims must be dense over rows for the folded view
    expect = ld * x.shape[-2]
    for i in range(x.dim() - 3, -1, -1):
        if x.shape[i] > 1 and x.stride(i) != expect:
            raise ValueError("leading dimensions must fold into rows with a single pitch")
        expect *= x.shape[i]
    return rows, cols, ld


def mx_quantize_sizes(rows: int, cols: int, in_dtype="bf16", out_dtype="e4m3fn", cfg: QuantCfg | None = None):
    db, sr, sc, sbytes = ctypes.c_size_t(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_size_t()
    _check(_lib.mx_quantize_sizes(DTYPES[in_dtype], DTYPES[out_dtype], rows, cols,
                                  ctypes.byref(cfg) if cfg is not None else None, ctypes.byref(db),
                                  ctypes.byref(sr), ctypes.byref(sc), ctypes.byref(sbytes)),
           "mx_quantize_sizes")
    return db.value, sr.value, sc.value


def mx_quantize(x: torch.Tensor, out_dtype: str = "e4m3fn", *, geometry="8x4", dim=-2, scale_layout="plain",
                fp4_lane_stride=2, fp4_nibble_parity=0, emax_alt=False, block_size=32, scale_method=0,
                out_data: torch.Tensor | None = None, out_scale: torch.Tensor | None = None, stream=None):
    """QuantizeMX of x (bf16/f16, CUDA).  Returns (data, scale) uint8 tensors:
    data [rows, cols] (FP8) or [rows, cols/2] (e2m1) over the folded 2-D view,
    scale [buffer rows, scale cols].  Pre-allocated outputs may be passed."""
    in_dtype = _in_dtype(x)
    rows, cols, ld = _view2d(x, dim)
    cfg = make_cfg(geometry, dim, scale_layout, fp4_lane_stride, fp4_nibble_parity, emax_alt, block_size,
                   scale_method)
    data_bytes, srows, scols = mx_quantize_sizes(rows, cols, in_dtype, out_dtype, cfg)
    if out_data is None:
        out_data = torch.empty((rows, cols // 2 if out_dtype == "e2m1" else cols), dtype=torch.uint8,
                               device=x.device)
    if out_scale is None:
        out_scale = torch.empty((srows, scols), dtype=torch.uint8, device=x.device)
    if out_data.numel() < data_bytes or out_scale.numel() < srows * scols:
        raise ValueError("output buffer too small")
    _check(_lib.mx_quantize(_dev_ptr(x), DTYPES[in_dtype], rows, cols, ld, DTYPES[out_dtype],
                            ctypes.byref(cfg), _dev_ptr(out_data), _dev_ptr(out_scale), _stream(stream)),
           "mx_quantize")
    return out_data, out_scale


def mx_quantize_host_workspace(rows: int, cols: int, in_dtype: str = "bf16", out_dtype: str = "e4m3fn",
                               cfg: QuantCfg | None = None, chunk_rows: int = 0) -> int:
    n = ctypes.c_size_t()
    _check(_lib.mx_quantize_host_workspace(DTYPES[in_dtype], rows, cols, DTYPES[out_dtype],
                                           ctypes.byref(cfg) if cfg is not None else None, chunk_rows,
                                           ctypes.byref(n)), "mx_quantize_host_workspace")
    return n.value


def mx_quantize_host(x: torch.Tensor, out_dtype: str = "e4m3fn", *, out_data: torch.Tensor,
                     out_scale: torch.Tensor, geometry="8x4", dim=-2, scale_layout="plain", fp4_lane_stride=2,
                     fp4_nibble_parity=0, emax_alt=False, chunk_rows: int = 0,
                     workspace: torch.Tensor | None = None, stream=None) -> None:
    """QuantizeMX of a HOST tensor x (bf16/f16, 2-D, rows may be strided)
    into HOST tensors out_data / out_scale (sizes of mx_quantize_sizes),
    pipelined through device slots.  Pinned host tensors overlap the copies.
    Asynchronous on `stream`."""
    if x.is_cuda or out_data.is_cuda or out_scale.is_cuda:
        raise ValueError("mx_quantize_host takes host tensors")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("mx_quantize_host takes a 2-D tensor with unit column stride")
    rows, cols = x.shape
    cfg = make_cfg(geometry, dim, scale_layout, fp4_lane_stride, fp4_nibble_parity, emax_alt)
    in_dtype = _in_dtype(x)
    need = mx_quantize_host_workspace(rows, cols, in_dtype, out_dtype, cfg, chunk_rows)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    _check(_lib.mx_quantize_host(ctypes.c_void_p(x.data_ptr()), DTYPES[in_dtype], rows, cols, x.stride(0),
                                 DTYPES[out_dtype], ctypes.byref(cfg), ctypes.c_void_p(out_data.data_ptr()),
                                 ctypes.c_void_p(out_scale.data_ptr()), chunk_rows, _dev_ptr(workspace),
                                 workspace.numel(), _stream(stream)),
           "mx_quantize_host")


def make_host_jobs(specs) -> ctypes.Array:
    """specs: sequence of dicts with x (host bf16/f16 2-D tensor), out_dtype,
    out_data, out_scale (host uint8 tensors) and the mx_quantize keyword
    arguments geometry / dim / scale_layout / fp4_lane_stride /
    fp4_nibble_parity / emax_alt.  The tensors must stay alive while the
    jobs run."""
    jobs = (HostJob * max(1, len(specs)))()
    for j, sp in zip(jobs, specs):
        x = sp["x"]
        if x.is_cuda or x.dim() != 2 or x.stride(1) != 1:
            raise ValueError("host jobs take 2-D host tensors with unit column stride")
        j.in_host = x.data_ptr()
        j.in_dtype = DTYPES[_in_dtype(x)]
        j.rows, j.cols = x.shape
        j.ld_in = x.stride(0)
        j.out_dtype = DTYPES[sp.get("out_dtype", "e4m3fn")]
        j.cfg = make_cfg(sp.get("geometry", "8x4"), sp.get("dim", -2), sp.get("scale_layout", "plain"),
                         sp.get("fp4_lane_stride", 2), sp.get("fp4_nibble_parity", 0), sp.get("emax_alt", False))
        j.out_data_host = sp["out_data"].data_ptr()
        j.out_scale_host = sp["out_scale"].data_ptr()
    return jobs


def mx_quantize_host_batch_workspace(jobs, njobs: int, chunk_rows: int = 0) -> int:
    n = ctypes.c_size_t()
    _check(_lib.mx_quantize_host_batch_workspace(jobs, njobs, chunk_rows, ctypes.byref(n)),
           "mx_quantize_host_batch_workspace")
    return n.value


def mx_quantize_host_batch(specs, *, chunk_rows: int = 0, workspace: torch.Tensor | None = None, stream=None):
    """Several host-to-host QuantizeMX jobs (see make_host_jobs) in one
    pipelined call.  Asynchronous on `stream`."""
    jobs = make_host_jobs(specs)
    if workspace is None:
        workspace = torch.empty(mx_quantize_host_batch_workspace(jobs, len(specs), chunk_rows), dtype=torch.uint8,
                                device="cuda")
    _check(_lib.mx_quantize_host_batch(jobs, len(specs), chunk_rows, _dev_ptr(workspace), workspace.numel(),
                                       _stream(stream)), "mx_quantize_host_batch")


def mx_dequantize(data: torch.Tensor, scale: torch.Tensor, rows: int, cols: int, in_dtype: str = "e4m3fn",
                  out_dtype: str = "f32", *, geometry="8x4", dim=-2, scale_layout="plain", fp4_lane_stride=2,
                  fp4_nibble_parity=0, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """decode(code) * 2^(E - 127) for an MX tensor as mx_quantize wrote it."""
    cfg = make_cfg(geometry, dim, scale_layout, fp4_lane_stride, fp4_nibble_parity)
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float32 if out_dtype == "f32" else torch.bfloat16,
                          device=data.device)
    _check(_lib.mx_dequantize(_dev_ptr(data), _dev_ptr(scale), DTYPES[in_dtype], rows, cols, ctypes.byref(cfg),
                              DTYPES[out_dtype], _dev_ptr(out), out.stride(0), _stream(stream)),
           "mx_dequantize")
    return out


def mx_sf_layout_bytes(mn: int, k: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.mx_sf_layout_bytes(mn, k, ctypes.byref(n)), "mx_sf_layout_bytes")
    return n.value


def mx_repack_scales(plain: torch.Tensor, k: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Plain E8M0 scales [mn, k/32] -> tensor-core SF layout (uint8, flat)."""
    mn = plain.shape[0]
    if out is None:
        out = torch.empty(mx_sf_layout_bytes(mn, k), dtype=torch.uint8, device=plain.device)
    _check(_lib.mx_repack_scales(_dev_ptr(plain), mn, k, plain.stride(0), _dev_ptr(out), _stream(stream)),
           "mx_repack_scales")
    return out


def mx_scaled_matmul_workspace(M: int, N: int, K: int, scales_are_sf_layout: bool = False) -> int:
    n = ctypes.c_size_t()
    _check(_lib.mx_scaled_matmul_workspace(M, N, K, int(scales_are_sf_layout), ctypes.byref(n)),
           "mx_scaled_matmul_workspace")
    return n.value


def mx_scaled_matmul(a: torch.Tensor, bt: torch.Tensor, a_scale: torch.Tensor, b_scale: torch.Tensor,
                     elem_dtype: str = "e4m3fn", out_dtype: str = "f32", *, scales_are_sf_layout: bool = False,
                     out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                     K: int | None = None, stream=None) -> torch.Tensor:
    """C = ScaledMatmul(A [M,K], Bt [N,K]) with E8M0 scales, f32 or bf16 out.
    e2m1 operands are packed two a byte ([M, K/2] bytes)."""
    M, Kb = a.shape
    N = bt.shape[0]
    K = (2 * Kb if elem_dtype == "e2m1" else Kb) if K is None else K
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32 if out_dtype == "f32" else torch.bfloat16, device=a.device)
    ws_bytes = mx_scaled_matmul_workspace(M, N, K, scales_are_sf_layout)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=a.device)
    _check(_lib.mx_scaled_matmul(_dev_ptr(a), _dev_ptr(bt), _dev_ptr(a_scale), _dev_ptr(b_scale),
                                 int(scales_are_sf_layout), DTYPES[elem_dtype], M, N, K, DTYPES[out_dtype],
                                 _dev_ptr(out), out.stride(0), _dev_ptr(workspace),
                                 workspace.numel() if workspace is not None else 0, _stream(stream)),
           "mx_scaled_matmul")
    return out


def mx_scaled_matmul_noalloc(a: torch.Tensor, bt: torch.Tensor, a_scale: torch.Tensor, b_scale: torch.Tensor,
                             elem_dtype: str = "e4m3fn", out_dtype: str = "f32", *,
                             out: torch.Tensor | None = None, K: int | None = None, stream=None) -> torch.Tensor:
    """ScaledMatmul with plain scales whose scratch lives in the library's
    fixed device array (for callers that cannot allocate a workspace; see
    include/mx.h).  The output tensor is still the caller's."""
    M, Kb = a.shape
    N = bt.shape[0]
    K = (2 * Kb if elem_dtype == "e2m1" else Kb) if K is None else K
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32 if out_dtype == "f32" else torch.bfloat16, device=a.device)
    _check(_lib.mx_scaled_matmul_noalloc(_dev_ptr(a), _dev_ptr(bt), _dev_ptr(a_scale), _dev_ptr(b_scale),
                                         DTYPES[elem_dtype], M, N, K, DTYPES[out_dtype], _dev_ptr(out),
                                         out.stride(0), _stream(stream)),
           "mx_scaled_matmul_noalloc")
    return out


def make_dot_dims(lhs_batch=(), rhs_batch=(), lhs_contract=(-1,), rhs_contract=(-1,)) -> DotDims:
    d = DotDims()
    d.lhs_n_batch, d.rhs_n_batch = len(lhs_batch), len(rhs_batch)
    d.lhs_n_contract, d.rhs_n_contract = len(lhs_contract), len(rhs_contract)
    for dst, src in ((d.lhs_batch, lhs_batch), (d.rhs_batch, rhs_batch), (d.lhs_contract, lhs_contract),
                     (d.rhs_contract, rhs_contract)):
        if len(src) > MAX_RANK:
            raise ValueError("more dimensions than MX_MAX_RANK")
        for i, v in enumerate(src):
            dst[i] = int(v)
    return d


def _dims_array(shape):
    return (ctypes.c_int64 * max(1, len(shape)))(*[int(v) for v in shape])


def mx_block_scaled_dot_shape(lhs_shape, rhs_shape, dims: DotDims) -> tuple:
    out = (ctypes.c_int64 * MAX_RANK)()
    rank = ctypes.c_int()
    _check(_lib.mx_block_scaled_dot_shape(_dims_array(lhs_shape), len(lhs_shape), _dims_array(rhs_shape),
                                          len(rhs_shape), ctypes.byref(dims), out, ctypes.byref(rank)),
           "mx_block_scaled_dot_shape")
    return tuple(out[i] for i in range(rank.value))


def mx_block_scaled_dot_workspace(lhs_shape, rhs_shape, dims: DotDims) -> int:
    n = ctypes.c_size_t()
    _check(_lib.mx_block_scaled_dot_workspace(_dims_array(lhs_shape), len(lhs_shape), _dims_array(rhs_shape),
                                              len(rhs_shape), ctypes.byref(dims), ctypes.byref(n)),
           "mx_block_scaled_dot_workspace")
    return n.value


def mx_block_scaled_dot(lhs: torch.Tensor, rhs: torch.Tensor, lhs_scale: torch.Tensor, rhs_scale: torch.Tensor,
                        elem_dtype: str = "e4m3fn", out_dtype: str = "f32", *, lhs_batch=(), rhs_batch=(),
                        lhs_contract=(-1,), rhs_contract=(-1,), out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """block_scaled_dot with dot dimension numbers; operands are dense uint8
    code tensors, scales their shape with the contracting extent / 32.  e2m1
    operands are packed two a byte along their last (contracting) axis."""
    for t in (lhs, rhs, lhs_scale, rhs_scale):
        if not t.is_contiguous():
            raise ValueError("mx_block_scaled_dot takes dense (contiguous) tensors")
    dims = make_dot_dims(lhs_batch, rhs_batch, lhs_contract, rhs_contract)
    lshape, rshape = tuple(lhs.shape), tuple(rhs.shape)
    if elem_dtype == "e2m1":  # logical extents: two elements a byte along the last axis
        lshape, rshape = lshape[:-1] + (2 * lshape[-1],), rshape[:-1] + (2 * rshape[-1],)
    shape = mx_block_scaled_dot_shape(lshape, rshape, dims)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32 if out_dtype == "f32" else torch.bfloat16, device=lhs.device)
    ws_bytes = mx_block_scaled_dot_workspace(lshape, rshape, dims)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=lhs.device)
    _check(_lib.mx_block_scaled_dot(_dev_ptr(lhs), _dims_array(lshape), lhs.dim(), _dev_ptr(lhs_scale),
                                    _dev_ptr(rhs), _dims_array(rshape), rhs.dim(), _dev_ptr(rhs_scale),
                                    ctypes.byref(dims), DTYPES[elem_dtype], DTYPES[out_dtype], _dev_ptr(out),
                                    _dev_ptr(workspace), workspace.numel() if workspace is not None else 0,
                                    _stream(stream)),
           "mx_block_scaled_dot")
    return out


def mx_fused_quantize_matmul_workspace(M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.mx_fused_quantize_matmul_workspace(M, N, K, ctypes.byref(n)), "mx_fused_quantize_matmul_workspace")
    return n.value


def mx_fused_quantize_matmul(x: torch.Tensor, wt: torch.Tensor, w_scale_sf: torch.Tensor,
                             elem_dtype: str = "e4m3fn", out_dtype: str = "bf16", *,
                             out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """QuantizeMX(x along K) fused with ScaledMatmul against Wt [N,K]."""
    M, K = x.shape
    N = wt.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32 if out_dtype == "f32" else torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(mx_fused_quantize_matmul_workspace(M, N, K), dtype=torch.uint8, device=x.device)
    _check(_lib.mx_fused_quantize_matmul(_dev_ptr(x), DTYPES[_in_dtype(x)], x.stride(0), _dev_ptr(wt),
                                         _dev_ptr(w_scale_sf), DTYPES[elem_dtype], M, N, K, DTYPES[out_dtype],
                                         _dev_ptr(out), out.stride(0), _dev_ptr(workspace), workspace.numel(),
                                         _stream(stream)),
           "mx_fused_quantize_matmul")
    return out


def mx_get_device_status() -> int:
    s = ctypes.c_int()
    _check(_lib.mx_get_device_status(ctypes.byref(s)), "mx_get_device_status")
    return s.value


def mx_status_string(status: int) -> str:
    return _lib.mx_status_string(status).decode()


def mx_version() -> int:
    return _lib.mx_version()


def mx_debug_gemm_fault_injection(skip_producer: int, timeout_ns: int = 0):
    """Bit 0: the GEMMs issue no loads; bit 1: the fused single launch never
    publishes its quantize items.  Either makes the kernels' bounded waits run
    out after ``timeout_ns`` (0 restores the 2 s default)."""
    _check(_lib.mx_debug_gemm_fault_injection(int(skip_producer), timeout_ns), "mx_debug_gemm_fault_injection")


def mx_debug_set_gemm_variant(variant: int):
    """0 automatic, 1 force the 1-SM ScaledMatmul kernel, 2 force the 2-SM pair
    kernel (the fused call then runs as one launch whenever its input allows),
    3 force the 1-SM kernel without split-K, 4 automatic with the fused call
    as two launches (QuantizeMX, then ScaledMatmul)."""
    _check(_lib.mx_debug_set_gemm_variant(int(variant)), "mx_debug_set_gemm_variant")


def mx_debug_last_gemm_launch():
    """(kernel, split_k) of the last ScaledMatmul launch: kernel 1 = 1-SM,
    2 = pair, 3 = pair with the fused activation quantize (one launch for
    the whole fused call), 0 = none yet; split_k = CTAs per tile along K."""
    kernel, split = ctypes.c_int(0), ctypes.c_int(0)
    _check(_lib.mx_debug_last_gemm_launch(ctypes.byref(kernel), ctypes.byref(split)), "mx_debug_last_gemm_launch")
    return kernel.value, split.value


def mx_debug_last_gemm_operands():
    """(a_mn_major, b_mn_major) of the last ScaledMatmul launch: 1 where the
    operand was read in place as MN-major tiles (a dot operand stored
    [batch..., K, rows...]), 0 for K-major rows."""
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    _check(_lib.mx_debug_last_gemm_operands(ctypes.byref(a), ctypes.byref(b)), "mx_debug_last_gemm_operands")
    return a.value, b.value


def raw_library() -> ctypes.CDLL:
    """The loaded ctypes handle (for callers that want the C-ABI directly)."""
    return _lib
