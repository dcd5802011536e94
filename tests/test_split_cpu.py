"""CPU check of the arithmetic behind the tensor-core selection scores.

The training-time selection forms q_bar . K_bar on the tensor cores from a
three-term bf16 split of each fp32 operand (x = x1 + x2 + x3, each term the bf16
rounding of what the previous ones leave) and keeps the six products a_i b_j with
i + j <= 4 (1-based), accumulated in fp32. The claim the selection relies on is
that the result is as accurate as an fp32 dot product: these tests model the
split and the product sum in numpy (bf16 rounding to nearest even written out
here) and compare them with fp64 dot products.
"""
import numpy as np
import pytest


def bf16_rn(x):
    """fp32 -> bf16 (the upper 16 bits), round to nearest, ties to even."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (r & 0xFFFF).astype(np.uint32)


def bf16_to_f32(h):
    return (np.asarray(h, dtype=np.uint32) << 16).view(np.float32)


def split3(x):
    x = np.asarray(x, dtype=np.float32)
    t1 = bf16_to_f32(bf16_rn(x))
    with np.errstate(invalid="ignore"):
        r1 = np.where(np.isfinite(x), x - t1, np.float32(0)).astype(np.float32)
    t2 = bf16_to_f32(bf16_rn(r1))
    r2 = (r1 - t2).astype(np.float32)
    t3 = bf16_to_f32(bf16_rn(r2))
    return t1, t2, t3


PAIRS = [(0, 0), (0, 1), (1, 0), (0, 2), (1, 1), (2, 0)]


def six_term_dot(a, b):
    """The six kept products accumulated in fp32, one element product at a time
    (each product of two bf16 values is exact in fp32), in the order of the
    kernel's MMAs: per 16-dim step, the six products."""
    sa, sb = split3(a), split3(b)
    acc = np.float32(0)
    for k0 in range(0, len(a), 16):
        for i, j in PAIRS:
            for k in range(k0, k0 + 16):
                acc = np.float32(np.float64(acc) + np.float64(sa[i][k]) * np.float64(sb[j][k]))
    return acc


def test_split_terms_are_bf16_and_shrink():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(10000).astype(np.float32) * np.float32(3.0)
    t1, t2, t3 = split3(x)
    for t in (t1, t2, t3):  # every term is a bf16 value
        assert np.array_equal(bf16_to_f32(bf16_rn(t)), t)
    ax = np.abs(x).astype(np.float64)
    assert np.all(np.abs(t2) <= ax * 2.0 ** -8 + 1e-30)
    assert np.all(np.abs(t3) <= ax * 2.0 ** -16 + 1e-30)
    # what the three terms leave is below 2^-24 |x| (plus rounding of the last)
    rest = x.astype(np.float64) - (t1.astype(np.float64) + t2 + t3)
    assert np.all(np.abs(rest) <= ax * 2.0 ** -24)


def test_split_of_bf16_values_is_exact():
    h = bf16_to_f32(bf16_rn(np.linspace(-5, 5, 1001).astype(np.float32)))
    t1, t2, t3 = split3(h)
    assert np.array_equal(t1, h) and not t2.any() and not t3.any()


def test_non_finite_values_keep_zero_tails():
    x = np.array([np.inf, -np.inf, np.nan, 1.5], dtype=np.float32)
    t1, t2, t3 = split3(x)
    assert np.isinf(t1[0]) and np.isinf(t1[1]) and np.isnan(t1[2])
    assert not t2[:3].any() and not t3[:3].any()


@pytest.mark.parametrize("d", [64, 128])
def test_six_term_dot_matches_fp32_accuracy(d):
    # pooled keys and head-mean queries of the workloads: per-block centres plus
    # noise, AR(1)-like queries; compare against fp64 dot products
    rng = np.random.default_rng(d)
    worst_six, worst_f32 = 0.0, 0.0
    for _ in range(400):
        a = (rng.standard_normal(d) * rng.uniform(0.1, 4.0)).astype(np.float32)
        b = (rng.standard_normal(d) + rng.standard_normal(d) * 0.5).astype(np.float32)
        exact = float(np.dot(a.astype(np.float64), b.astype(np.float64)))
        scale = float(np.dot(np.abs(a).astype(np.float64), np.abs(b).astype(np.float64)))
        f32 = np.float32(0)
        for x, y in zip(a, b):  # a plain fp32 FMA chain
            f32 = np.float32(np.float64(x) * np.float64(y) + np.float64(f32))
        worst_six = max(worst_six, abs(float(six_term_dot(a, b)) - exact) / scale)
        worst_f32 = max(worst_f32, abs(float(f32) - exact) / scale)
    # as accurate as the fp32 chain (within a small factor) and far inside the
    # near-tie band of 1e-5 of the largest score
    assert worst_six <= max(4 * worst_f32, 2.0 ** -22)
    assert worst_six < 1e-6
