"""Pins of the seeded input generator (CPU)."""
import numpy as np
import pytest

import synth


def test_splitmix64_known_answers():
    # First four outputs of the splitmix64 generator seeded with 0, as printed by
    # Vigna's public-domain reference splitmix64.c (state += golden gamma, then mix).
    g = np.uint64(0x9E3779B97F4A7C15)
    with np.errstate(over="ignore"):
        got = [int(synth.splitmix64(np.uint64(i) * g)) for i in range(4)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F,
                   0xF88BB8A8724C81EC]


def test_normals_exact_grid_and_moments():
    x = synth.normals(0, synth.STREAM_VALUE, 3, 5, np.arange(4000)[:, None], np.arange(64)[None, :])
    assert np.all(x * 65536 == np.round(x * 65536))          # multiples of 2**-16
    assert np.all(np.abs(x) < 6)
    assert np.all(x.astype(np.float32).astype(np.float64) == x)  # exact in fp32
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1.0) < 0.02
    # Irwin-Hall(12): fourth moment 3 - 1.2/12 = 2.9
    assert abs((x ** 4).mean() - 2.9) < 0.08


def test_streams_and_fields_independent():
    a = synth.normals(0, synth.STREAM_VALUE, 0, 0, np.arange(1000), 0)
    for other in [synth.normals(0, synth.STREAM_EVICT, 0, 0, np.arange(1000), 0),
                  synth.normals(0, synth.STREAM_VALUE, 1, 0, np.arange(1000), 0),
                  synth.normals(0, synth.STREAM_VALUE, 0, 1, np.arange(1000), 0),
                  synth.normals(1, synth.STREAM_VALUE, 0, 0, np.arange(1000), 0)]:
        assert abs(np.corrcoef(a, other)[0, 1]) < 0.12


def test_bf16_rounding_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5 - 2 ** -9, 1.0 + 2 ** -8 + 2 ** -20])
    bits = synth.to_storage(x, "bf16")
    back = synth.bf16_bits_to_f64(bits)
    # ties go to the even mantissa; above the tie rounds up
    assert list(back) == [1.0, 1.0, 1.0 + 4 * 2 ** -8, -2.5, 1.0 + 2 ** -7]


def test_keys_share_block_centre():
    w = synth.WORKLOADS["tiny-f32"]
    k = synth.keys(w, 0, 0, 0, 128).astype(np.float64)
    # tokens of one block scatter around one centre (noise sd 0.5), the two blocks differ
    c0, c1 = k[:64].mean(0), k[64:].mean(0)
    assert (k[:64] - c0).std() == pytest.approx(0.5, rel=0.1)
    assert np.abs(c0 - c1).mean() > 0.5


def test_queries_ar1():
    w = synth.WORKLOADS["tiny-f32"].with_(head_dim=64)
    q = synth.queries(w, 0, range(4), 400).astype(np.float64)
    eps0 = synth.normals(0, synth.STREAM_QINNOV, 0, np.arange(4)[:, None], 0, np.arange(64)[None, :])
    a = 1.0 / np.sqrt(1.0 - 0.95 ** 2)  # stationary start: Var q_0 = 1 / (1 - rho^2)
    assert np.array_equal(q[0], (a * eps0).astype(np.float32))
    lag1 = np.mean([np.corrcoef(q[:-1, 0, j], q[1:, 0, j])[0, 1] for j in range(64)])
    assert lag1 == pytest.approx(0.95, abs=0.05)
    # one more step by hand, from the definition
    eps5 = synth.normals(0, synth.STREAM_QINNOV, 0, np.arange(4)[:, None], 5, np.arange(64)[None, :])
    qq = a * eps0
    for s in range(1, 6):
        qq = 0.95 * qq + synth.normals(0, synth.STREAM_QINNOV, 0, np.arange(4)[:, None], s,
                                       np.arange(64)[None, :])
    assert np.array_equal(q[5], qq.astype(np.float32))
    assert eps5.shape == (4, 64)


def test_queries_stationary_from_the_first_step():
    # the variance of q_s is 1 / (1 - rho^2) at every step, so early steps look
    # like late ones; the unnormalised start grows from 1 instead
    w = synth.WORKLOADS["1b-bf16"].with_(dtype="f32")
    q = synth.queries(w, 0, range(w.n_q_heads), 200).astype(np.float64)
    var = (q ** 2).mean(axis=(1, 2))
    target = 1.0 / (1.0 - w.rho ** 2)
    assert var[:5].mean() == pytest.approx(target, rel=0.15)
    assert var[150:].mean() == pytest.approx(target, rel=0.15)
    q0 = synth.queries(w.with_(q_stationary=False), 0, range(w.n_q_heads), 3).astype(np.float64)
    assert (q0[0] ** 2).mean() == pytest.approx(1.0, rel=0.15)


def test_request_base_offsets_the_request_field():
    w = synth.WORKLOADS["1b-bf16"]
    ws = w.with_(request_base=8)
    # request b of a rank whose requests start at 8 is request 8 + b of the job
    assert np.array_equal(synth.keys(ws, 0, 3, 50, 9), synth.keys(w, 8, 3, 50, 9))
    assert np.array_equal(synth.evict(ws, 2, 1, 7, 5), synth.evict(w, 10, 1, 7, 5))
    assert np.array_equal(synth.queries(ws, 1, [0, 2], 4), synth.queries(w, 9, [0, 2], 4))
    with pytest.raises(ValueError):
        synth.keys(w.with_(request_base=synth.MAX_REQUESTS - 1), 1, 0, 0, 1)
