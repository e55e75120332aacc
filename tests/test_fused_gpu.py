"""Activation quantize fused with ScaledMatmul (page "MX-FP8 Microscaling
Legalization", section 4.3: QuantizeMX feeds ScaledMatmul by dataflow) as
ONE kernel launch: the pair GEMM's epilogue warps quantize X into the
workspace while the tensor cores run, and the operand loads wait for each
item's ready word.

Every case checks, against the CPU oracle:
  - the quantized X the launch left in the workspace, bit for bit (codes,
    and the SF-layout scales of every row < M, zero past K in the last
    scale tile), against QuantizeMX of X along K (1x32 blocks, EMAX);
  - C within |C - C_ref| <= 1e-4 * sum_k |a_k b_k| (+ 1 bf16 ulp for bf16);
  - that the call really ran as the single fused launch.
"""
import numpy as np
import pytest

import mx_synth as syn
import oracle as orc
from helpers import check_gemm, sf_pack, to_device_bits, to_device_u8

pytestmark = pytest.mark.gpu

TOL = 1e-4
FUSED_KERNEL = 3  # mx_debug_last_gemm_launch: pair kernel with the fused quantize


@pytest.fixture(scope="module")
def mx():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mx_fp8_microscaling_gb300 as mx
    return mx


@pytest.fixture
def force_pair(mx):
    mx.mx_debug_set_gemm_variant(2)
    yield
    mx.mx_debug_set_gemm_variant(0)


def _r16(x):
    return (x + 15) // 16 * 16


def _unpack_tc(packed, K):
    """Tensor-core nibble order (element 2i low, 2i+1 high) -> codes."""
    out = np.empty((packed.shape[0], K), np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def _weight(w_bits, fmt):
    """Pre-quantized weight: device codes, device SF scales, oracle codes and
    plain scales (codes unpacked for e2m1)."""
    if fmt == "e2m1":
        q, s = orc.quantize(w_bits, "bf16", "e2m1", geometry="1x32", dim=-1, lane_stride=1, nibble_parity=1)
        return to_device_u8(q), to_device_u8(sf_pack(s)), _unpack_tc(q, w_bits.shape[1]), s
    q, s = orc.quantize(w_bits, "bf16", fmt, geometry="1x32", dim=-1)
    return to_device_u8(q), to_device_u8(sf_pack(s)), q, s


def _x_ref(x_bits, in_dtype, fmt, K):
    """QuantizeMX(X) along K: (packed codes as the launch stores them, codes
    for the GEMM oracle, plain scales)."""
    if fmt == "e2m1":
        q, s = orc.quantize(x_bits, in_dtype, "e2m1", geometry="1x32", dim=-1, lane_stride=1, nibble_parity=1,
                            cols=K)
        return q, _unpack_tc(q, K), s
    q, s = orc.quantize(x_bits, in_dtype, fmt, geometry="1x32", dim=-1, cols=K)
    return q, q, s


def _run(mx, x_dev, wq, wsf, fmt, out_dtype, M, N, K, workspace=None):
    import torch
    if workspace is None:
        workspace = torch.empty(mx.mx_fused_quantize_matmul_workspace(M, N, K), dtype=torch.uint8, device="cuda")
    c = mx.mx_fused_quantize_matmul(x_dev, wq, wsf, fmt, out_dtype, workspace=workspace)
    torch.cuda.synchronize()
    return c, workspace, mx.mx_debug_last_gemm_launch()[0]


def _check_workspace_x(ws, xq_ref, xs_ref, M, K, fmt):
    """The quantized X the launch left in the workspace, bit for bit."""
    nbytes = M * K // 2 if fmt == "e2m1" else M * K
    xq = ws[:nbytes].cpu().numpy().reshape(M, -1)
    bad = np.argwhere(xq != xq_ref)
    assert bad.size == 0, f"{len(bad)} code bytes differ, first at {bad[:3].tolist()}"
    ntk = -(-K // 128)
    sf_bytes = -(-M // 128) * ntk * 512
    sf = ws[_r16(M * K):_r16(M * K) + sf_bytes].cpu().numpy()
    want = sf_pack(np.pad(xs_ref, ((0, 0), (0, 4 * ntk - xs_ref.shape[1]))))
    live = sf_pack(np.ones((M, 4 * ntk), np.uint8)) == 1  # rows < M, every column of a touched tile
    assert np.array_equal(sf[live], want[live]), "SF-layout scales differ"


def _check_c(c, xg, xs, wg, ws_plain, fmt, out_dtype, rows=None):
    c_ref, s_ref = orc.scaled_matmul(xg, wg, xs, ws_plain, fmt, rows=rows)
    got = c.float().cpu().numpy() if rows is None else c[rows].float().cpu().numpy()
    check_gemm(got, c_ref, s_ref, out_dtype, TOL)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("M,N,K", [(384, 512, 512),     # several tiles and items
                                   (256, 256, 160),     # K ends inside an item and a scale tile
                                   (300, 520, 1056),    # ragged M and N, K tail
                                   (512, 768, 2304)])   # several scale groups along K
def test_fused_single_launch_matches_oracle(mx, force_pair, fmt, out_dtype, M, N, K):
    x_bits, w_bits = syn.fused_operands(M, N, K, seed=M + N + K)
    wq, wsf, wg, ws_plain = _weight(w_bits, fmt)
    xq_ref, xg, xs = _x_ref(x_bits, "bf16", fmt, K)
    c, ws, kernel = _run(mx, to_device_bits(x_bits, "bf16"), wq, wsf, fmt, out_dtype, M, N, K)
    assert kernel == FUSED_KERNEL
    _check_workspace_x(ws, xq_ref, xs, M, K, fmt)
    _check_c(c, xg, xs, wg, ws_plain, fmt, out_dtype)
    assert mx.mx_get_device_status() == 0


def test_fused_single_launch_fp4(mx, force_pair):
    """MXFP4: X quantized to e2m1 in the tensor cores' nibble order."""
    M, N, K = 384, 512, 768
    x_bits, w_bits = syn.fused_operands(M, N, K, seed=4)
    wq, wsf, wg, ws_plain = _weight(w_bits, "e2m1")
    xq_ref, xg, xs = _x_ref(x_bits, "bf16", "e2m1", K)
    c, ws, kernel = _run(mx, to_device_bits(x_bits, "bf16"), wq, wsf, "e2m1", "bf16", M, N, K)
    assert kernel == FUSED_KERNEL
    _check_workspace_x(ws, xq_ref, xs, M, K, "e2m1")
    _check_c(c, xg, xs, wg, ws_plain, "e2m1", "bf16")


def test_fused_f16_input_and_row_pitch(mx, force_pair):
    """f16 activations (f16 subnormals widen to normals) read through a row
    pitch wider than K."""
    import torch
    M, N, K, ld = 256, 256, 512, 640
    rng = np.random.default_rng(3)
    vals = (rng.standard_normal((M, ld)) * np.exp2(rng.integers(-20, 12, (M, 1)))).astype(np.float32)
    vals[:8, :32] = np.float32(2.0 ** -24) * rng.integers(1, 1024, (8, 32))  # subnormal-only blocks
    x_bits = vals.astype(np.float16).view(np.uint16)
    _, w_bits = syn.fused_operands(1, N, K, seed=5)
    wq, wsf, wg, ws_plain = _weight(w_bits, "e4m3fn")
    xq_ref, xg, xs = _x_ref(x_bits, "f16", "e4m3fn", K)
    x_dev = to_device_bits(x_bits, "f16")[:, :K]
    assert x_dev.stride(0) == ld
    c, ws, kernel = _run(mx, x_dev, wq, wsf, "e4m3fn", "bf16", M, N, K)
    assert kernel == FUSED_KERNEL
    _check_workspace_x(ws, xq_ref, xs, M, K, "e4m3fn")
    _check_c(c, xg, xs, wg, ws_plain, "e4m3fn", "bf16")
    torch.cuda.synchronize()


def test_fused_special_values(mx, force_pair):
    """Random 16-bit patterns (Inf, NaN, subnormals, both zeros): the
    quantized X must match bit for bit; C is compared on rows free of Inf/NaN
    (the others hold NaN codes)."""
    M, N, K = 256, 256, 256
    rng = np.random.default_rng(6)
    x_bits = rng.integers(0, 1 << 16, size=(M, K), dtype=np.uint16)
    clean = np.arange(M) % 4 != 0
    # finite, moderate values on three rows in four
    x_bits[clean] = syn.fused_operands(int(clean.sum()), 1, K, seed=7)[0]
    _, w_bits = syn.fused_operands(1, N, K, seed=8)
    wq, wsf, wg, ws_plain = _weight(w_bits, "e4m3fn")
    xq_ref, xg, xs = _x_ref(x_bits, "bf16", "e4m3fn", K)
    c, ws, kernel = _run(mx, to_device_bits(x_bits, "bf16"), wq, wsf, "e4m3fn", "f32", M, N, K)
    assert kernel == FUSED_KERNEL
    _check_workspace_x(ws, xq_ref, xs, M, K, "e4m3fn")
    rows = np.nonzero(clean)[0]
    _check_c(c, xg, xs, wg, ws_plain, "e4m3fn", "f32", rows=rows)


def test_fused_more_than_one_tile_group(mx, force_pair):
    """36 panels of 128 rows: two tile groups, so items run ahead of the
    tiles by the look-ahead rule and the last group is partial."""
    M, N, K = 4608, 512, 512
    x_bits, w_bits = syn.fused_operands(M, N, K, seed=9)
    wq, wsf, wg, ws_plain = _weight(w_bits, "e4m3fn")
    xq_ref, xg, xs = _x_ref(x_bits, "bf16", "e4m3fn", K)
    c, ws, kernel = _run(mx, to_device_bits(x_bits, "bf16"), wq, wsf, "e4m3fn", "bf16", M, N, K)
    assert kernel == FUSED_KERNEL
    _check_workspace_x(ws, xq_ref, xs, M, K, "e4m3fn")
    _check_c(c, xg, xs, wg, ws_plain, "e4m3fn", "bf16")


def test_fused_reused_workspace_takes_no_stale_item(mx, force_pair):
    """Two calls in a row on one workspace with different X: the second
    launch's loads must wait for its own items, not take the first call's
    (its ready words still hold the first launch's value)."""
    M, N, K = 512, 512, 1024
    _, w_bits = syn.fused_operands(1, N, K, seed=10)
    wq, wsf, wg, ws_plain = _weight(w_bits, "e4m3fn")
    ws = None
    for seed in (11, 12):
        x_bits = syn.fused_operands(M, 1, K, seed=seed)[0]
        xq_ref, xg, xs = _x_ref(x_bits, "bf16", "e4m3fn", K)
        c, ws, kernel = _run(mx, to_device_bits(x_bits, "bf16"), wq, wsf, "e4m3fn", "f32", M, N, K, workspace=ws)
        assert kernel == FUSED_KERNEL
        _check_workspace_x(ws, xq_ref, xs, M, K, "e4m3fn")
        _check_c(c, xg, xs, wg, ws_plain, "e4m3fn", "f32")


def test_fused_automatic_choice(mx):
    """Without forcing: a long product (at least 32 pair tiles per cluster)
    runs as one launch; a shorter pair-kernel product as QuantizeMX + the
    pair GEMM; a small-M one as QuantizeMX + the 1-SM GEMM; all against the
    oracle (sampled rows)."""
    for (M, N, K), want in (((16384, 12800, 256), FUSED_KERNEL), ((2048, 2048, 512), 2), ((64, 512, 512), 1)):
        x_bits, w_bits = syn.fused_operands(M, N, K, seed=13)
        wq, wsf, wg, ws_plain = _weight(w_bits, "e4m3fn")
        xq_ref, xg, xs = _x_ref(x_bits, "bf16", "e4m3fn", K)
        c, ws, kernel = _run(mx, to_device_bits(x_bits, "bf16"), wq, wsf, "e4m3fn", "bf16", M, N, K)
        assert kernel == want, (M, N, K, kernel)
        _check_workspace_x(ws, xq_ref, xs, M, K, "e4m3fn")
        rows = np.unique(np.concatenate([np.arange(0, M, 97), [M - 1]]))
        _check_c(c, xg, xs, wg, ws_plain, "e4m3fn", "bf16", rows=rows)


def test_fused_two_launch_ablation_agrees(mx):
    """The two-launch path (variant 4) and the single launch give the same
    quantized X and the same C bits (same tiles, same accumulation order)."""
    import torch
    M, N, K = 1024, 2048, 1024
    x_bits, w_bits = syn.fused_operands(M, N, K, seed=14)
    wq, wsf, _, _ = _weight(w_bits, "e4m3fn")
    x_dev = to_device_bits(x_bits, "bf16")
    mx.mx_debug_set_gemm_variant(2)
    try:
        c1, ws1, k1 = _run(mx, x_dev, wq, wsf, "e4m3fn", "bf16", M, N, K)
        mx.mx_debug_set_gemm_variant(4)
        c2, ws2, k2 = _run(mx, x_dev, wq, wsf, "e4m3fn", "bf16", M, N, K)
    finally:
        mx.mx_debug_set_gemm_variant(0)
    assert k1 == FUSED_KERNEL and k2 == 2
    assert torch.equal(ws1[:M * K], ws2[:M * K])
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


def test_fused_ready_wait_times_out_without_fault(mx, force_pair):
    """With the items never published, the operand loads' waits run out
    after 50 ms: MX_ERR_TIMEOUT in the status word, no fault, no hang, and
    the context still computes correctly afterwards."""
    M, N, K = 256, 256, 256
    x_bits, w_bits = syn.fused_operands(M, N, K, seed=15)
    wq, wsf, wg, ws_plain = _weight(w_bits, "e4m3fn")
    x_dev = to_device_bits(x_bits, "bf16")
    assert mx.mx_get_device_status() == 0
    mx.mx_debug_gemm_fault_injection(2, 50_000_000)
    try:
        _run(mx, x_dev, wq, wsf, "e4m3fn", "f32", M, N, K)
    finally:
        mx.mx_debug_gemm_fault_injection(0, 0)
    assert mx.mx_get_device_status() == mx.MX_ERR_TIMEOUT
    assert mx.mx_get_device_status() == 0
    xq_ref, xg, xs = _x_ref(x_bits, "bf16", "e4m3fn", K)
    c, ws, kernel = _run(mx, x_dev, wq, wsf, "e4m3fn", "f32", M, N, K)
    assert kernel == FUSED_KERNEL
    _check_c(c, xg, xs, wg, ws_plain, "e4m3fn", "f32")


def test_fused_graph_replay_with_new_input(mx, force_pair):
    """A captured fused call replayed after new activations are copied into
    its input buffer: each replay must wait for its own quantize items (the
    launch parameters, tag included, are the same on every replay)."""
    import torch
    M, N, K = 512, 1024, 1024
    _, w_bits = syn.fused_operands(1, N, K, seed=16)
    wq, wsf, wg, ws_plain = _weight(w_bits, "e4m3fn")
    xs_bits = [syn.fused_operands(M, 1, K, seed=s)[0] for s in (17, 18, 19)]
    x_dev = to_device_bits(xs_bits[0], "bf16")
    ws = torch.empty(mx.mx_fused_quantize_matmul_workspace(M, N, K), dtype=torch.uint8, device="cuda")
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    mx.mx_fused_quantize_matmul(x_dev, wq, wsf, "e4m3fn", "f32", out=out, workspace=ws, stream=stream)  # warm-up
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        mx.mx_fused_quantize_matmul(x_dev, wq, wsf, "e4m3fn", "f32", out=out, workspace=ws,
                                    stream=torch.cuda.current_stream())
    for bits in xs_bits[1:] + xs_bits[:1]:
        x_dev.copy_(to_device_bits(bits, "bf16"))
        graph.replay()
        torch.cuda.synchronize()
        xq_ref, xg, xs = _x_ref(bits, "bf16", "e4m3fn", K)
        _check_workspace_x(ws, xq_ref, xs, M, K, "e4m3fn")
        _check_c(out, xg, xs, wg, ws_plain, "e4m3fn", "f32")
    assert mx.mx_get_device_status() == 0
