"""QuantizeMX from host to host (the pipelined chunk runtime): bit-identical
to mx_quantize on the device and to the oracle, for every scale layout,
multi-chunk inputs with a short last chunk, strided host rows, pinned and
pageable host memory; rows the interleaved layout never addresses stay
untouched."""
import numpy as np
import pytest

import mx_synth as syn
import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mx_fp8_microscaling_gb300 as mx
    return mx


BLOCK_ROWS = {("8x4", -2): 8, ("8x4", -1): 4, ("1x32", -1): 1, ("1x32", -2): 32}

CASES = [  # geometry, dim, layout, fmt, rows, cols, chunk_rows
    ("8x4", -2, "plain", "e4m3fn", 2560, 256, 1024),
    ("8x4", -2, "plain", "e4m3fn", 1000, 256, 8),          # one scale row per chunk
    ("8x4", -2, "interleave", "e4m3fn", 1000, 256, 96),    # 3 interleave groups per chunk, short last
    ("1x32", -1, "plain", "e5m2", 301, 128, 0),             # default chunk size
    ("8x4", -2, "interleave", "e5m2", 2560 + 8, 192, 1024),
    ("1x32", -1, "plain", "e4m3fn", 300, 512, 128),
    ("1x32", -1, "sf", "e4m3fn", 300, 384, 128),
    ("1x32", -1, "interleave", "e2m1", 520, 256, 256),
    ("8x4", -1, "plain", "e2m1", 1040, 128, 512),
    ("1x32", -2, "plain", "e5m2", 4096 + 64, 64, 4096),
]


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_host_quantize_matches_device_and_oracle(mx, case, pinned):
    import torch
    geometry, dim, layout, fmt, rows, cols, chunk = CASES[case]
    pad = 8
    bits = syn.random_bits(rows, cols + pad, "bf16", seed=case, block_exp=(-20, 20), block=(1, 4))
    host = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    host_x = host[:, :cols]                      # strided rows: ld = cols + pad
    db, sr, sc = mx.mx_quantize_sizes(rows, cols, "bf16", fmt, mx.make_cfg(geometry, dim, layout))
    out_d = torch.full((db,), 0xAB, dtype=torch.uint8)
    out_s = torch.full((sr * sc,), 0xCD, dtype=torch.uint8)
    if pinned:
        host_x = host.pin_memory()[:, :cols]
        out_d, out_s = out_d.pin_memory(), out_s.pin_memory()
    mx.mx_quantize_host(host_x, fmt, out_data=out_d, out_scale=out_s, geometry=geometry, dim=dim,
                        scale_layout=layout, chunk_rows=chunk)
    torch.cuda.synchronize()
    dev_d, dev_s = mx.mx_quantize(host_x.cuda(), fmt, geometry=geometry, dim=dim, scale_layout=layout)
    torch.cuda.synchronize()
    got_s = out_s.numpy().reshape(sr, sc)
    if layout == "interleave":
        live = np.zeros(sr, bool)
        live[[(i & 3) + 32 * (i >> 2) for i in range(rows // BLOCK_ROWS[(geometry, dim)])]] = True
        assert np.all(got_s[~live] == 0xCD)
        assert np.array_equal(got_s[live], dev_s.cpu().numpy().reshape(sr, sc)[live])
    else:
        assert np.array_equal(got_s, dev_s.cpu().numpy().reshape(sr, sc))
    assert np.array_equal(out_d.numpy(), dev_d.cpu().numpy().reshape(-1))
    if layout != "sf":
        want_d, want_s = orc.quantize(bits[:, :cols], "bf16", fmt, geometry=geometry, dim=dim,
                                      scale_layout=layout, scale_fill=0xCD)
        assert np.array_equal(out_d.numpy(), want_d.reshape(-1))
        assert np.array_equal(got_s, want_s)


def test_host_quantize_repeated_calls_share_the_pipeline(mx):
    # back-to-back calls on one stream reuse the copy streams and slots
    import torch
    rows, cols = 1024, 256
    outs = []
    for seed in range(3):
        bits = syn.random_bits(rows, cols, "bf16", seed=10 + seed, block_exp=(-8, 8))
        x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        d = torch.empty(rows * cols, dtype=torch.uint8).pin_memory()
        s = torch.empty(rows * cols // 32, dtype=torch.uint8).pin_memory()
        mx.mx_quantize_host(x, "e4m3fn", out_data=d, out_scale=s, geometry="1x32", dim=-1, chunk_rows=128)
        outs.append((bits, d, s))
    torch.cuda.synchronize()
    for bits, d, s in outs:
        want_d, want_s = orc.quantize(bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
        assert np.array_equal(d.numpy(), want_d.reshape(-1))
        assert np.array_equal(s.numpy(), want_s.reshape(-1))


def test_host_quantize_batch_equals_separate_calls(mx):
    # mixed geometries, layouts, formats and input types in one pipeline,
    # including an empty job; each result equals the device quantizer's
    import torch
    specs, want = [], []
    shapes = [("8x4", -2, "interleave", "e4m3fn", "bf16", 1000, 256), ("1x32", -1, "sf", "e5m2", "f16", 300, 384),
              ("8x4", -2, "plain", "e2m1", "bf16", 0, 64), ("1x32", -1, "plain", "e2m1", "bf16", 520, 128),
              ("8x4", -1, "plain", "e4m3fn", "f16", 1040, 192)]
    for i, (geometry, dim, layout, fmt, in_dtype, rows, cols) in enumerate(shapes):
        bits = syn.random_bits(max(rows, 1), cols, in_dtype, seed=50 + i, block_exp=(-12, 12), block=(1, 4))[:rows]
        x = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16 if in_dtype == "bf16" else torch.float16).pin_memory()
        db, sr, sc = mx.mx_quantize_sizes(rows, cols, in_dtype, fmt, mx.make_cfg(geometry, dim, layout))
        d = torch.full((max(db, 1),), 0x5A, dtype=torch.uint8).pin_memory()
        s = torch.full((max(sr * sc, 1),), 0x5A, dtype=torch.uint8).pin_memory()
        specs.append(dict(x=x, out_dtype=fmt, out_data=d, out_scale=s, geometry=geometry, dim=dim,
                          scale_layout=layout))
        if rows:
            dd, ds = mx.mx_quantize(x.cuda(), fmt, geometry=geometry, dim=dim, scale_layout=layout)
            want.append((dd, ds, layout, sr, sc, rows // BLOCK_ROWS[(geometry, dim)]))
        else:
            want.append(None)
    mx.mx_quantize_host_batch(specs, chunk_rows=0)
    torch.cuda.synchronize()
    for sp, w in zip(specs, want):
        if w is None:
            assert torch.all(sp["out_data"] == 0x5A)   # an empty job writes nothing
            continue
        dd, ds, layout, sr, sc, nscale = w
        assert np.array_equal(sp["out_data"].numpy()[:dd.numel()], dd.cpu().numpy().reshape(-1))
        got = sp["out_scale"].numpy()[:sr * sc].reshape(sr, sc)
        ref = ds.cpu().numpy().reshape(sr, sc)
        if layout == "interleave":
            live = np.zeros(sr, bool)
            live[[(i & 3) + 32 * (i >> 2) for i in range(nscale)]] = True
            assert np.all(got[~live] == 0x5A)
            got, ref = got[live], ref[live]
        assert np.array_equal(got, ref)
