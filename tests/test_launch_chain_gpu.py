"""Back-to-back dependent launches on one stream with no host synchronisation
in between.  Every kernel is launched with programmatic stream serialization
allowed and may start while the previous one finishes; each must still read
only what the previous kernels wrote.  Chains of QuantizeMX -> dequantize and
QuantizeMX -> repack -> ScaledMatmul over several tensors, checked against the
oracle once at the end."""
import numpy as np
import pytest

import mx_synth as syn
import oracle as orc
from helpers import check_gemm, to_device_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mx_fp8_microscaling_gb300 as mx
    return mx


def test_quantize_dequantize_chain(mx):
    import torch
    rows, cols, n = 1024, 4096, 6
    bits = [syn.random_bits(rows, cols, "bf16", seed=100 + i) for i in range(n)]
    xs = [to_device_bits(b, "bf16") for b in bits]
    outs = []
    for x in xs:   # quantize i, then dequantize i (reads what quantize i wrote), no sync
        q, s = mx.mx_quantize(x, "e4m3fn", geometry="8x4", dim=-2)
        outs.append((q, s, mx.mx_dequantize(q, s, rows, cols, "e4m3fn", "f32", geometry="8x4", dim=-2)))
    torch.cuda.synchronize()
    for b, (q, s, d) in zip(bits, outs):
        want_q, want_s = orc.quantize(b, "bf16", "e4m3fn", geometry="8x4", dim=-2)
        assert np.array_equal(q.cpu().numpy(), want_q)
        assert np.array_equal(s.cpu().numpy(), want_s)
        want = orc.dequantize(want_q, want_s, rows, cols, "e4m3fn", geometry="8x4", dim=-2).astype(np.float32)
        got = d.cpu().numpy()
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_quantize_repack_matmul_chain(mx):
    # each step's operands are quantized, their scales repacked and the GEMM
    # run, all enqueued back to back; the output buffer is reused by every
    # step, so a GEMM that started writing before the previous one finished
    # reading or writing would show
    import torch
    M, N, K, steps = 384, 512, 1024, 5
    ops = [syn.gemm_operands(M, N, K, seed=200 + i) for i in range(steps)]
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    results = []
    for a_bits, b_bits in ops:
        qa, sa = mx.mx_quantize(to_device_bits(a_bits, "bf16"), "e4m3fn", geometry="1x32", dim=-1)
        qb, sb = mx.mx_quantize(to_device_bits(b_bits, "bf16"), "e4m3fn", geometry="1x32", dim=-1)
        mx.mx_scaled_matmul(qa, qb, sa, sb, "e4m3fn", "f32", out=c)
        results.append(c.clone())   # a torch copy kernel in the chain as well
    torch.cuda.synchronize()
    for (a_bits, b_bits), got in zip(ops, results):
        oa, osa = orc.quantize(a_bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
        ob, osb = orc.quantize(b_bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
        c_ref, s_ref = orc.scaled_matmul(oa, ob, osa, osb, "e4m3fn")
        check_gemm(got.cpu().numpy(), c_ref, s_ref, "f32")
