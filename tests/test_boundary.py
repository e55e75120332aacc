"""The C-ABI boundary without a GPU: the library loads, exports every
function include/mx.h declares, and rejects bad arguments with the documented
status codes before touching the device."""
import ctypes

import pytest

from helpers import header_functions


@pytest.fixture(scope="module")
def mx():
    import mx_fp8_microscaling_gb300 as mx
    return mx


@pytest.fixture(scope="module")
def lib(mx):
    return mx.raw_library()


FAKE = ctypes.c_void_p(0x10000)          # never dereferenced: every call below fails validation first
FAKE_MISALIGNED = ctypes.c_void_p(0x10004)
FAKE_ODD = ctypes.c_void_p(0x10001)


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert "mx_quantize" in names and "mx_scaled_matmul" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(mx):
    assert mx.mx_version() >= 100
    for code, name in mx.STATUS_NAMES.items():
        assert mx.mx_status_string(code).startswith(name)


def test_default_cfg(mx):
    cfg = mx.QuantCfg()
    assert mx.raw_library().mx_quant_cfg_default(ctypes.byref(cfg)) == 0
    assert (cfg.geometry, cfg.scale_layout, cfg.block_size, cfg.dim, cfg.scale_method,
            cfg.fp4_lane_stride, cfg.fp4_nibble_parity, cfg.emax_alt) == (0, 0, 32, -2, 0, 2, 0, 0)


@pytest.mark.parametrize("rows,cols,kw,expect", [
    (64, 64, dict(geometry="8x4", dim=-2), (64 * 64, 8, 16)),
    (64, 64, dict(geometry="8x4", dim=-1), (64 * 64, 16, 8)),
    (64, 64, dict(geometry="1x32", dim=-1), (64 * 64, 64, 2)),
    (64, 64, dict(geometry="1x32", dim=-2), (64 * 64, 2, 64)),
    (8192, 8192, dict(geometry="8x4", dim=-2, scale_layout="interleave"), (8192 * 8192, 8192, 2048)),
    (40, 64, dict(geometry="8x4", dim=-2, scale_layout="interleave"), (40 * 64, 64, 16)),
    (200, 96, dict(geometry="1x32", dim=-1, scale_layout="sf"), (200 * 96, 256, 4)),
])
def test_quantize_sizes(mx, rows, cols, kw, expect):
    cfg = mx.make_cfg(**kw)
    assert mx.mx_quantize_sizes(rows, cols, "bf16", "e4m3fn", cfg) == expect


def test_quantize_sizes_fp4(mx):
    cfg = mx.make_cfg(geometry="8x4", dim=-2, scale_layout="interleave")
    assert mx.mx_quantize_sizes(16384, 16384, "bf16", "e2m1", cfg) == (16384 * 16384 // 2, 16384, 4096)


def _quantize_status(lib, mx, in_dtype=1, out_dtype=4, rows=64, cols=64, ld=64, cfg=None,
                     src=FAKE, data=FAKE, scale=FAKE):
    cfg = cfg if cfg is not None else mx.make_cfg()
    return lib.mx_quantize(src, in_dtype, rows, cols, ld, out_dtype, ctypes.byref(cfg), data, scale, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(in_dtype=3), 2),                       # f32 input: only bf16/f16
    (dict(out_dtype=7), 2),                      # e8m0 data
    (dict(out_dtype=3), 2),
    (dict(rows=-8), 1),
    (dict(ld=32), 1),                            # pitch < width
    (dict(cols=66, ld=72), 5),                   # x4 container
    (dict(rows=12), 5),                          # 8x4 needs rows % 8
    (dict(src=None), 1),
    (dict(scale=None), 1),
    (dict(src=FAKE_ODD), 6),                     # bf16 input needs 2-byte alignment
    (dict(data=FAKE_ODD), 6),
])
def test_quantize_argument_errors(lib, mx, kwargs, status):
    assert _quantize_status(lib, mx, **kwargs) == status


@pytest.mark.parametrize("cfg_kw,status", [
    (dict(block_size=16), 3),
    (dict(block_size=64), 3),
    (dict(dim=-3), 4),
    (dict(dim=2), 4),
    (dict(scale_method=1), 11),
    (dict(geometry=2), 1),
    (dict(scale_layout=3), 1),
    (dict(scale_layout="sf"), 1),                # SF layout needs 1x32 along dim=-1
    (dict(fp4_lane_stride=3), 1),
    (dict(fp4_nibble_parity=2), 1),
    (dict(emax_alt=2), 1),
])
def test_quantize_cfg_errors(lib, mx, cfg_kw, status):
    cfg = mx.make_cfg(**{k: v for k, v in cfg_kw.items() if k != "emax_alt"})
    if "emax_alt" in cfg_kw:
        cfg.emax_alt = cfg_kw["emax_alt"]
    assert _quantize_status(lib, mx, cfg=cfg) == status


def test_fp4_stride_needs_window_divisibility(lib, mx):
    cfg = mx.make_cfg(geometry="8x4", dim=-2, fp4_lane_stride=4)
    assert _quantize_status(lib, mx, out_dtype=6, rows=8, cols=36, ld=40, cfg=cfg) == 5


def test_empty_quantize_is_a_no_op(lib, mx):
    assert _quantize_status(lib, mx, rows=0, src=None, data=None, scale=None) == 0


def _matmul_status(lib, elem=4, M=128, N=128, K=128, out=3, ldc=128, a=FAKE, bt=FAKE, sa=FAKE, sb=FAKE,
                   c=FAKE, sf=1, ws=None, ws_bytes=0):
    return lib.mx_scaled_matmul(a, bt, sa, sb, sf, elem, M, N, K, out, c, ldc, ws, ws_bytes, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(elem=7), 2),          # e8m0 is a scale type, not an operand type
    (dict(elem=1), 2),
    (dict(out=4), 2),           # output only f32 / bf16
    (dict(K=48), 5),
    (dict(K=0), 5),
    (dict(M=-1), 1),
    (dict(ldc=64), 1),
    (dict(a=None), 1),
    (dict(a=FAKE_MISALIGNED), 6),  # TMA needs 16-byte aligned operands
    (dict(c=FAKE_ODD), 6),         # f32 output needs 4-byte alignment
    (dict(sf=0), 7),            # plain scales need workspace
    (dict(sf=0, ws=FAKE, ws_bytes=16), 7),
])
def test_matmul_argument_errors(lib, kwargs, status):
    assert _matmul_status(lib, **kwargs) == status


def test_matmul_workspace_sizes(mx):
    # two SF buffers, each ceil(mn/128) * ceil(k/128) * 512 bytes
    assert mx.mx_scaled_matmul_workspace(8192, 8192, 8192) == 2 * 64 * 64 * 512
    assert mx.mx_scaled_matmul_workspace(8192, 8192, 8192, True) == 0
    assert mx.mx_sf_layout_bytes(200, 96) == 2 * 1 * 512
    # fused: codes, SF scales, then one 8-byte ready word per 128 x 256 item
    # and a done word (2 + 1 words: 24 bytes, rounded up to 32)
    assert mx.mx_fused_quantize_matmul_workspace(256, 512, 256) == 256 * 256 + 2 * 2 * 512 + 32
    # 300 * 1056 codes, 3 x 9 scale tiles, 3 x 5 + 1 words (128 bytes)
    assert mx.mx_fused_quantize_matmul_workspace(300, 512, 1056) == 300 * 1056 + 3 * 9 * 512 + 128


def test_fused_argument_errors(lib):
    st = lib.mx_fused_quantize_matmul(FAKE, 3, 128, FAKE, FAKE, 4, 128, 128, 128, 1, FAKE, 128, FAKE, 1 << 20, None)
    assert st == 2  # x must be bf16/f16
    st = lib.mx_fused_quantize_matmul(FAKE, 1, 128, FAKE, FAKE, 4, 128, 128, 128, 1, FAKE, 128, FAKE, 16, None)
    assert st == 7  # workspace too small


def test_folded_view_rules(mx):
    import torch
    x = torch.zeros(2, 3, 8, 32, dtype=torch.bfloat16)
    assert mx._view2d(x, -1) == (48, 32, 32)
    y = torch.zeros(16, 64, dtype=torch.bfloat16)[:, :32]
    assert mx._view2d(y, -1) == (16, 32, 64)
    with pytest.raises(ValueError):
        mx._view2d(torch.zeros(8, 32, dtype=torch.bfloat16).t(), -1)


# ---- general block-scaled dot: the contract's dimension checks

@pytest.mark.parametrize("lshape,rshape,lb,rb,lc,rc,status", [
    ((4,), (4, 32), (), (), (0,), (1,), 5),                   # rank < 2
    ((2, 32), (2, 32), (0,), (), (1,), (1,), 4),              # batch counts differ
    ((2, 32), (2, 32), (2,), (0,), (1,), (1,), 4),            # batch index out of bounds
    ((2, 32), (3, 32), (0,), (0,), (1,), (1,), 5),            # batch extents differ
    ((2, 32), (2, 64), (), (), (1,), (1,), 5),                # contracting sizes differ
    ((2, 32), (2, 32), (1,), (1,), (1,), (1,), 4),            # contracting overlaps batch
    ((2, 32, 32), (2, 32), (), (), (1, 2), (1,), 4),          # two contracting dims
    ((2, 48), (2, 48), (), (), (1,), (1,), 5),                # K not a multiple of 32
    ((2, 2, 32), (2, 2, 32), (0, 0), (0, 1), (2,), (2,), 4),  # repeated batch dim
    ((2, 32), (2, 32), (), (), (5,), (1,), 4),                # contracting index out of bounds
    ((2, 32), (2, 32), (), (), (-3,), (1,), 4),               # negative index past the rank
])
def test_dot_dimension_errors(mx, lshape, rshape, lb, rb, lc, rc, status):
    dims = mx.make_dot_dims(lb, rb, lc, rc)
    with pytest.raises(mx.MxError) as e:
        mx.mx_block_scaled_dot_shape(lshape, rshape, dims)
    assert e.value.status == status
    with pytest.raises(mx.MxError) as e:
        mx.mx_block_scaled_dot_workspace(lshape, rshape, dims)
    assert e.value.status == status


@pytest.mark.parametrize("lshape,rshape,lb,rb,lc,rc,shape", [
    ((3, 64), (5, 64), (), (), (1,), (1,), (3, 5)),
    ((3, 64), (64, 5), (), (), (1,), (0,), (3, 5)),
    ((2, 3, 4, 32), (32, 3, 2, 5), (0, 1), (2, 1), (3,), (0,), (2, 3, 4, 5)),
    ((2, 32, 3, 2), (3, 32, 2), (0,), (2,), (1,), (1,), (2, 3, 2, 3)),
    ((130, 2, 64), (2, 72, 64), (-2,), (0,), (-1,), (-1,), (2, 130, 72)),
])
def test_dot_result_shape(mx, lshape, rshape, lb, rb, lc, rc, shape):
    assert mx.mx_block_scaled_dot_shape(lshape, rshape, mx.make_dot_dims(lb, rb, lc, rc)) == shape


def test_dot_workspace_counts_only_needed_copies(mx):
    sf = lambda mn, k: -(-mn // 128) * -(-k // 128) * 512  # noqa: E731
    r256 = lambda n: -(-n // 256) * 256  # noqa: E731
    d = mx.make_dot_dims((0,), (0,), (2,), (2,))
    # both operands already [batch, rows, K]: only the SF scales
    assert mx.mx_block_scaled_dot_workspace((4, 200, 256), (4, 300, 256), d) == r256(4 * sf(200, 256)) + \
        r256(4 * sf(300, 256))
    # rhs stored [batch, K, N]: a canonical copy of it and of its scales too
    d = mx.make_dot_dims((0,), (0,), (2,), (1,))
    assert mx.mx_block_scaled_dot_workspace((4, 200, 256), (4, 256, 300), d) == r256(4 * 300 * 256) + \
        r256(4 * 300 * 8) + r256(4 * sf(200, 256)) + r256(4 * sf(300, 256))


def test_dot_argument_errors(lib, mx):
    import ctypes as ct
    dims = mx.make_dot_dims((0,), (0,), (2,), (2,))
    shape = (ct.c_int64 * 3)(2, 128, 128)
    call = lambda **kw: lib.mx_block_scaled_dot(  # noqa: E731
        kw.get("lhs", FAKE), shape, 3, FAKE, kw.get("rhs", FAKE), shape, 3, FAKE, ct.byref(dims),
        kw.get("elem", 4), kw.get("out_dtype", 3), kw.get("out", FAKE), kw.get("ws", FAKE),
        kw.get("ws_bytes", 1 << 30), None)
    assert call(elem=7) == 2
    assert call(out_dtype=4) == 2
    assert call(lhs=None) == 1
    assert call(lhs=FAKE_MISALIGNED) == 6   # read in place by TMA
    assert call(out=FAKE_ODD) == 6
    assert call(ws_bytes=16) == 7
    assert call(ws=None) == 7
    assert lib.mx_block_scaled_dot(FAKE, shape, 3, FAKE, FAKE, shape, 3, FAKE, None, 4, 3, FAKE, FAKE, 1 << 30,
                                   None) == 1


def test_fp4_dot_needs_contracting_axis_innermost(lib, mx):
    import ctypes as ct
    # rhs [B, K, N]: packed e2m1 pairs would run along N, not K
    dims = mx.make_dot_dims((0,), (0,), (2,), (1,))
    ls = (ct.c_int64 * 3)(2, 128, 128)
    rs = (ct.c_int64 * 3)(2, 128, 64)
    st = lib.mx_block_scaled_dot(FAKE, ls, 3, FAKE, FAKE, rs, 3, FAKE, ct.byref(dims), 6, 3, FAKE, FAKE, 1 << 30,
                                 None)
    assert st == 2


def test_host_quantize_workspace_and_errors(mx, lib):
    import ctypes as ct
    cfg = mx.make_cfg("1x32", -1, "plain")
    # three slots of (input chunk + codes + scales), each 256-byte rounded
    slot = 128 * 512 * 2 + 128 * 512 + 128 * 16
    assert mx.mx_quantize_host_workspace(1000, 512, "bf16", "e4m3fn", cfg, 128) == 3 * slot
    cfg_sf = mx.make_cfg("1x32", -1, "sf")
    with pytest.raises(mx.MxError) as e:
        mx.mx_quantize_host_workspace(1000, 512, "bf16", "e4m3fn", cfg_sf, 100)   # SF: multiples of 128 rows
    assert e.value.status == 5
    cfg84 = mx.make_cfg("8x4", -2, "interleave")
    with pytest.raises(mx.MxError) as e:
        mx.mx_quantize_host_workspace(1024, 512, "bf16", "e4m3fn", cfg84, 24)  # 4 scale rows of 8x4 = 32
    assert e.value.status == 5
    assert mx.mx_quantize_host_workspace(1024, 512, "bf16", "e4m3fn", cfg84, 32) > 0
    st = lib.mx_quantize_host(FAKE, 1, 256, 512, 512, 4, ct.byref(cfg), FAKE, FAKE, 128, FAKE, 16, None)
    assert st == 7
    st = lib.mx_quantize_host(FAKE, 1, 256, 512, 512, 4, ct.byref(cfg), FAKE, FAKE, 128, FAKE_MISALIGNED,
                              1 << 30, None)
    assert st == 6


def test_host_quantize_batch_workspace_and_checks(mx, lib):
    import ctypes as ct
    import torch
    small = torch.zeros(256, 512, dtype=torch.bfloat16)
    big = torch.zeros(2048, 512, dtype=torch.bfloat16)
    d = torch.empty(2048 * 512, dtype=torch.uint8)
    s = torch.empty(2048 * 16, dtype=torch.uint8)
    spec = lambda x: dict(x=x, out_data=d, out_scale=s, geometry="1x32", dim=-1)  # noqa: E731
    jobs = mx.make_host_jobs([spec(small), spec(big)])
    # the slot is the larger job's (chunks of 1024 rows here)
    one_big = mx.make_host_jobs([spec(big)])
    assert mx.mx_quantize_host_batch_workspace(jobs, 2, 1024) == mx.mx_quantize_host_batch_workspace(one_big, 1, 1024)
    assert mx.mx_quantize_host_batch_workspace(jobs, 2, 1024) > mx.mx_quantize_host_batch_workspace(
        mx.make_host_jobs([spec(small)]), 1, 1024)
    # a bad job anywhere fails the whole call before anything runs
    bad = mx.make_host_jobs([spec(small), spec(big)])
    bad[1].cols = 500   # not a multiple of 32 along the block
    assert lib.mx_quantize_host_batch(bad, 2, 0, FAKE, 1 << 30, None) == 5
    assert lib.mx_quantize_host_batch(jobs, 2, 0, FAKE, 16, None) == 7


def test_debug_hooks_check_arguments(mx, lib):
    # the kernel-choice hook takes 0..4; the last-launch query wants both pointers
    assert lib.mx_debug_set_gemm_variant(5) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_debug_set_gemm_variant(-1) == mx.MX_ERR_INVALID_ARG
    for v in (4, 3, 0):
        assert lib.mx_debug_set_gemm_variant(v) == mx.MX_OK
    one = ctypes.c_int()
    assert lib.mx_debug_last_gemm_launch(None, ctypes.byref(one)) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_debug_last_gemm_launch(ctypes.byref(one), None) == mx.MX_ERR_INVALID_ARG
    kernel, split = mx.mx_debug_last_gemm_launch()
    assert kernel in (0, 1, 2, 3) and split >= (1 if kernel else 0)
    assert lib.mx_debug_last_gemm_operands(None, ctypes.byref(one)) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_debug_last_gemm_operands(ctypes.byref(one), None) == mx.MX_ERR_INVALID_ARG
    a_mn, b_mn = mx.mx_debug_last_gemm_operands()
    assert a_mn in (0, 1) and b_mn in (0, 1)
