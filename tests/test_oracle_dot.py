"""Pins of the oracle's general block-scaled dot (dot dimension numbers).

The ScaledMatmul contract of the page "MX-FP8 Microscaling Legalization"
(sections 3.2 and 4.2) carries lhs/rhs batch and contracting dimension lists;
the result follows the dot-general order batch, lhs free, rhs free.  These
pins check the oracle against things other than itself: a pure-Python loop
over the index space with torch's float8 decoding, integer matmuls, exact
power-of-two scale shifts, the already-pinned 2-D GEMM oracle, and the
contract's dimension checks.  Two planted mistakes (a scale index shifted
along a neighbouring axis, swapped free-axis order) must be caught.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle as orc

TORCH_FP8 = {"e4m3fn": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}

# (lhs shape, rhs shape, lhs_batch, rhs_batch, lhs_contract, rhs_contract)
CASES = [
    ((3, 64), (5, 64), (), (), (1,), (1,)),             # A [M,K] x Bt [N,K]
    ((3, 64), (64, 5), (), (), (1,), (0,)),             # A [M,K] x B [K,N]
    ((64, 3), (64, 5), (), (), (0,), (0,)),             # both K-major on axis 0
    ((2, 3, 32), (2, 32, 4), (0,), (0,), (2,), (1,)),   # batched [B,M,K] x [B,K,N]
    ((3, 2, 64), (4, 2, 64), (1,), (1,), (2,), (2,)),   # batch in the middle
    ((2, 3, 4, 32), (32, 3, 2, 5), (0, 1), (2, 1), (3,), (0,)),  # two batch dims, reordered
    ((2, 32, 3, 2), (3, 32, 2), (0,), (2,), (1,), (1,)),  # two lhs free dims around K
]


def torch_decode(fmt, codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(TORCH_FP8[fmt])
    return t.to(torch.float64).numpy()


def random_operand(rng, shape, axis, lo=0x30, hi=0x60):
    # finite positive/negative codes and scales in a narrow range, so every
    # sum of products below is exact in binary64 and results compare with ==
    codes = rng.integers(lo, hi, size=shape).astype(np.uint8) | (rng.integers(0, 2, size=shape) << 7).astype(np.uint8)
    sshape = list(shape)
    sshape[axis] //= 32
    scale = rng.integers(124, 131, size=sshape).astype(np.uint8)
    return codes, scale


def brute_force(lhs, rhs, ls, rs, fmt, lb, rb, lc, rc):
    """Each output entry as a Python sum over k, indices mapped by hand."""
    lhs_v, rhs_v = torch_decode(fmt, lhs), torch_decode(fmt, rhs)
    lfree = [i for i in range(lhs.ndim) if i not in lb and i != lc]
    rfree = [i for i in range(rhs.ndim) if i not in rb and i != rc]
    out_shape = [lhs.shape[i] for i in lb] + [lhs.shape[i] for i in lfree] + [rhs.shape[i] for i in rfree]
    out = np.zeros(out_shape, np.float64)
    K = lhs.shape[lc]
    for idx in itertools.product(*[range(n) for n in out_shape]):
        b, rest = idx[:len(lb)], idx[len(lb):]
        i, j = rest[:len(lfree)], rest[len(lfree):]
        li, ri = [0] * lhs.ndim, [0] * rhs.ndim
        for axis_l, axis_r, v in zip(lb, rb, b):
            li[axis_l] = ri[axis_r] = v
        for axis, v in zip(lfree, i):
            li[axis] = v
        for axis, v in zip(rfree, j):
            ri[axis] = v
        total = 0.0
        for k in range(K):
            li[lc] = ri[rc] = k
            ls_i, rs_i = list(li), list(ri)
            ls_i[lc] //= 32
            rs_i[rc] //= 32
            a = lhs_v[tuple(li)] * 2.0 ** (int(ls[tuple(ls_i)]) - 127)
            w = rhs_v[tuple(ri)] * 2.0 ** (int(rs[tuple(rs_i)]) - 127)
            total += a * w
        out[idx] = total
    return out


def run_case(dot, case, fmt, seed):
    lshape, rshape, lb, rb, lc, rc = case
    rng = np.random.default_rng(seed)
    lhs, ls = random_operand(rng, lshape, lc[0])
    rhs, rs = random_operand(rng, rshape, rc[0])
    got, _ = dot(lhs, rhs, ls, rs, fmt, lhs_batch=lb, rhs_batch=rb, lhs_contract=lc, rhs_contract=rc)
    want = brute_force(lhs, rhs, ls, rs, fmt, list(lb), list(rb), lc[0], rc[0])
    return got.shape == want.shape and np.array_equal(got, want)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_dot_matches_index_loop(case, fmt):
    assert run_case(orc.block_scaled_dot, CASES[case], fmt, seed=100 + case)


def test_dot_rank2_equals_pinned_gemm_oracle():
    rng = np.random.default_rng(7)
    a, sa = random_operand(rng, (6, 96), 1, lo=0, hi=0x7E)
    bt, sb = random_operand(rng, (9, 96), 1, lo=0, hi=0x7E)
    C, S = orc.block_scaled_dot(a, bt, sa, sb, "e4m3fn", lhs_contract=(1,), rhs_contract=(1,))
    ms, ns = [v.reshape(-1) for v in np.meshgrid(np.arange(6), np.arange(9), indexing="ij")]
    c, s = orc.scaled_matmul_entries(a, bt, sa, sb, "e4m3fn", "e4m3fn", ms, ns)
    assert np.allclose(C.reshape(-1), c, rtol=0, atol=1e-13 * s.max())
    assert np.allclose(S.reshape(-1), s, rtol=1e-13)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_dot_unit_scales_batched_integer_matmul(fmt):
    # scales 127 and small-integer codes: [B,M,K] x [B,K,N] is a batched
    # integer matmul (torch, float64)
    rng = np.random.default_rng(11)
    B, M, N, K = 3, 4, 5, 64
    a_int = rng.integers(-8, 9, size=(B, M, K))
    b_int = rng.integers(-8, 9, size=(B, K, N))
    a = np.array([orc.narrow(fmt, float(v)) for v in a_int.reshape(-1)], np.uint8).reshape(a_int.shape)
    b = np.array([orc.narrow(fmt, float(v)) for v in b_int.reshape(-1)], np.uint8).reshape(b_int.shape)
    sa = np.full((B, M, K // 32), 127, np.uint8)
    sb = np.full((B, K // 32, N), 127, np.uint8)
    C, S = orc.block_scaled_dot(a, b, sa, sb, fmt, lhs_batch=(0,), rhs_batch=(0,), lhs_contract=(2,),
                                rhs_contract=(1,))
    ref = torch.matmul(torch.tensor(a_int, dtype=torch.float64), torch.tensor(b_int, dtype=torch.float64))
    assert np.array_equal(C, ref.numpy())
    assert np.array_equal(S, np.abs(a_int) @ np.abs(b_int))


def test_dot_scale_block_shift_is_exact():
    # raising one lhs scale block by d multiplies exactly the products of
    # that block's 32 elements by 2^d: C changes by (2^d - 1) * that block's part
    rng = np.random.default_rng(13)
    lhs, ls = random_operand(rng, (2, 3, 64), 2)
    rhs, rs = random_operand(rng, (2, 64, 4), 1)
    kw = dict(lhs_batch=(0,), rhs_batch=(0,), lhs_contract=(2,), rhs_contract=(1,))
    C0, _ = orc.block_scaled_dot(lhs, rhs, ls, rs, "e4m3fn", **kw)
    ls2 = ls.copy()
    ls2[1, 2, 1] += 3
    C1, _ = orc.block_scaled_dot(lhs, rhs, ls2, rs, "e4m3fn", **kw)
    mask_l = np.zeros_like(lhs)
    mask_l[1, 2, 32:] = lhs[1, 2, 32:]
    part, _ = orc.block_scaled_dot(mask_l, rhs, ls, rs, "e4m3fn", **kw)
    assert np.array_equal(C1 - C0, 7.0 * part)
    assert np.array_equal(np.delete(C1, 2, axis=1)[0], np.delete(C0, 2, axis=1)[0])


@pytest.mark.parametrize("lshape,rshape,lb,rb,lc,rc", [
    ((4,), (4, 32), (), (), (0,), (1,)),                  # rank < 2
    ((2, 32), (2, 32), (0,), (), (1,), (1,)),             # batch counts differ
    ((2, 32), (2, 32), (2,), (0,), (1,), (1,)),           # batch out of bounds
    ((2, 32), (3, 32), (0,), (0,), (1,), (1,)),           # batch extents differ
    ((2, 32), (2, 64), (), (), (1,), (1,)),               # contracting sizes differ
    ((2, 32), (2, 32), (1,), (1,), (1,), (1,)),           # contracting overlaps batch
    ((2, 32, 32), (2, 32), (), (), (1, 2), (1,)),         # two contracting dims
    ((2, 48), (2, 48), (), (), (1,), (1,)),               # K not a multiple of 32
    ((2, 2, 32), (2, 2, 32), (0, 0), (0, 1), (2,), (2,)),  # repeated batch dim
])
def test_dot_dimension_checks(lshape, rshape, lb, rb, lc, rc):
    with pytest.raises(orc.DotDimsError):
        orc.check_dot_dims(lshape, rshape, lb, rb, lc, rc)


def test_negative_indices_count_from_the_end():
    assert orc.check_dot_dims((2, 3, 32), (2, 32, 4), (0,), (-3,), (-1,), (-2,)) == ([0], [0], 2, 1)


# ---- planted mistakes: the loop pin must reject each

def _mutant_scale_axis(lhs, rhs, ls, rs, fmt, **kw):
    real = orc.block_values

    def wrong(codes, scale, f, axis):
        # scale index shifted by one along a neighbouring axis
        codes = np.asarray(codes, np.uint8)
        e = np.exp2(np.asarray(scale, np.float64) - 127)
        return orc.decode_array(f, codes) * np.roll(np.repeat(e, 32, axis=axis), 1, axis=(axis + 1) % codes.ndim)

    orc.block_values = wrong
    try:
        return orc.block_scaled_dot(lhs, rhs, ls, rs, fmt, **kw)
    finally:
        orc.block_values = real


def _mutant_free_order(lhs, rhs, ls, rs, fmt, **kw):
    C, S = orc.block_scaled_dot(lhs, rhs, ls, rs, fmt, **kw)
    nb = len(kw.get("lhs_batch", ()))
    n_lfree = lhs.ndim - nb - 1
    perm = list(range(nb)) + list(range(nb + n_lfree, C.ndim)) + list(range(nb, nb + n_lfree))
    return np.transpose(C, perm), np.transpose(S, perm)


@pytest.mark.parametrize("mutant", [_mutant_scale_axis, _mutant_free_order])
def test_loop_pin_catches_planted_mistakes(mutant):
    caught = [not run_case(mutant, CASES[i], "e4m3fn", seed=100 + i) for i in (1, 3, 5, 6)]
    assert any(caught) and caught.count(True) >= 3
