"""Pins of the fp64 oracle against closed forms, brute force, invariants and a
library routine (torch SDPA, fp64, CPU). None of these re-types the oracle's own
formula: each checks it through a different route, chosen so that a dropped
term, a wrong sign, index or divisor, or a transposed operand fails one of them.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import synth
from oracle import nosa_oracle as O


# --------------------------------------------------------------------------
# Two-stage pooling: closed forms
# --------------------------------------------------------------------------
def test_pool_constant_block():
    c = np.arange(8) * 0.375 - 1.25          # dyadic: sums are exact
    kb, eb, se = O.pool_block(np.tile(c, (64, 1)), np.full(64, 0.25), 16)
    assert kb.shape == (4, 8) and np.array_equal(kb, np.tile(c, (4, 1)))
    assert np.array_equal(eb, np.full(4, 0.25)) and se == 0.25


def test_pool_linear_ramp_closed_form():
    a, b = np.array([1.0, -2.0, 0.5]), np.array([0.25, 1.0, -0.125])
    j = np.arange(64, dtype=np.float64)
    kb, eb, se = O.pool_block(a[None, :] + j[:, None] * b[None, :], j.copy(), 16)
    # mean index of sub-block s is 16 s + 7.5
    for s in range(4):
        assert np.allclose(kb[s], a + (16 * s + 7.5) * b, atol=0, rtol=0)
        assert eb[s] == 16 * s + 7.5
    assert se == 55.5                           # max over sub-blocks, the last one
    _, eb2, se2 = O.pool_block(np.zeros((64, 3)), -j, 16)
    assert se2 == -7.5 and eb2[0] == -7.5       # decreasing ramp: the first one


def test_pool_sub_block_permutation_invariance():
    rng = np.random.default_rng(1)
    k, e = rng.normal(size=(64, 5)), rng.normal(size=64)
    kb, eb, se = O.pool_block(k, e, 16)
    perm = np.concatenate([rng.permutation(16) + 16 * s for s in range(4)])
    kb2, eb2, se2 = O.pool_block(k[perm], e[perm], 16)
    assert np.allclose(kb, kb2) and np.allclose(eb, eb2) and np.isclose(se, se2)
    swap = np.concatenate([np.arange(16, 32), np.arange(0, 16), np.arange(32, 64)])
    kb3, _, _ = O.pool_block(k[swap], e[swap], 16)
    assert np.allclose(kb3[0], kb[1]) and np.allclose(kb3[1], kb[0])


# --------------------------------------------------------------------------
# Block scores: closed forms and identities
# --------------------------------------------------------------------------
def test_score_basis_query_closed_form():
    rng = np.random.default_rng(2)
    kbar = rng.normal(size=(6, 4, 16))
    for j in (0, 7, 15):
        q = np.zeros(16)
        q[j] = 3.0
        assert np.allclose(O.block_scores(q, kbar), 3.0 * kbar[:, :, j].max(axis=1) / 4.0)


def test_score_equals_max_over_subblocks_of_mean_token_logits():
    # linearity: q.mean(k) = mean(q.k); the block score is the max of the
    # sub-blocks' mean per-token logits (a different route from pooled keys).
    rng = np.random.default_rng(3)
    d, n_blk = 32, 5
    k = rng.normal(size=(n_blk * 64, d))
    q = rng.normal(size=d)
    kbar = np.stack([O.pool_block(k[i * 64:(i + 1) * 64], np.zeros(64), 16)[0]
                     for i in range(n_blk)])
    tok_logit = (k @ q) / math.sqrt(d)
    want = tok_logit.reshape(n_blk, 4, 16).mean(axis=2).max(axis=1)
    assert np.allclose(O.block_scores(q, kbar), want, rtol=1e-12, atol=1e-12)


def test_group_query_is_mean_of_heads_scores():
    rng = np.random.default_rng(4)
    qg, kbar = rng.normal(size=(3, 16)), rng.normal(size=(4, 4, 16))
    per_head = np.stack([kbar @ qg[g] for g in range(3)]).mean(axis=0)     # [N][P]
    assert np.allclose(O.block_scores(O.group_query(qg), kbar), per_head.max(axis=1) / 4.0)


# --------------------------------------------------------------------------
# Top-k with ties: brute force over all subsets
# --------------------------------------------------------------------------
def _brute_top(scores, cand, m):
    """Max-sum subset; among equal sums the lexicographically smallest index tuple."""
    best = None
    for sub in itertools.combinations(sorted(cand), m):
        key = (-sum(int(scores[i]) for i in sub), sub)
        if best is None or key < best:
            best = key
    return list(best[1]) if best else []


@pytest.mark.parametrize("seed", range(40))
def test_top_m_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 12))
    scores = rng.integers(-3, 4, size=n).astype(np.float64)   # small ints: many exact ties
    cand = np.sort(rng.choice(n, size=int(rng.integers(0, n + 1)), replace=False))
    m = int(rng.integers(0, 6))
    got = list(O.top_m(scores, cand, m))
    assert got == _brute_top(scores, cand, min(m, len(cand)))


@pytest.mark.parametrize("seed", range(40))
def test_dual_select_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(0, 12))
    k = int(rng.integers(1, 6))
    k_e = int(rng.integers(0, k + 1))
    sq = rng.integers(-4, 5, size=n).astype(np.float64)
    se = rng.integers(-4, 5, size=n).astype(np.float64)
    elig = rng.random(n) < 0.6
    g_e, g_q, new_elig = O.dual_select(sq, se, elig, n, k, k_e)
    eligible = [i for i in range(n) if elig[i]]
    want_e = _brute_top(se, eligible, min(k_e, len(eligible)))
    rest = [i for i in range(n) if i not in want_e]
    want_q = _brute_top(sq, rest, min(k - len(want_e), len(rest)))
    assert list(g_e) == want_e and list(g_q) == want_q
    assert len(g_e) + len(g_q) == min(k, n)                    # R12
    assert set(g_e).isdisjoint(g_q)
    assert set(np.flatnonzero(new_elig)) == set(want_e)        # R5


def test_select_decides_in_fp32():
    # two scores that differ in fp64 but round to the same fp32: a tie, lower index wins
    s = np.array([1.0, 1.0 + 2.0 ** -40, 0.5])
    assert list(O.top_m(s, np.arange(3), 1)) == [0]
    assert list(O.top_m(np.array([-0.0, 0.0]), np.arange(2), 1)) == [0]


# --------------------------------------------------------------------------
# Set-difference: invariants against Python sets
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(30))
def test_set_difference_invariants(seed):
    rng = np.random.default_rng(200 + seed)
    k = int(rng.integers(1, 9))
    n = int(rng.integers(k, 20))
    slot = -np.ones(k, dtype=np.int64)
    held = rng.choice(n, size=int(rng.integers(0, k + 1)), replace=False)
    slot[rng.choice(k, size=len(held), replace=False)] = held
    gamma = sorted(rng.choice(n, size=int(rng.integers(0, k + 1)), replace=False).tolist())
    jc = int(rng.integers(-1, n))
    loads, free, new = O.set_difference(gamma, slot, jc)
    res = set(int(b) for b in slot if b >= 0)
    assert set(int(b) for b in new if b >= 0) == set(gamma)
    assert [l[0] for l in loads] == sorted(set(gamma) - res)
    assert all(l[0] not in res for l in loads)
    assert [l[1] for l in loads] == free[:len(loads)] and free == sorted(free)
    assert all(l[2] == (O.TAIL if l[0] == jc else O.HOST) for l in loads)
    for s in range(k):                      # slots kept by selected blocks are untouched
        if slot[s] >= 0 and slot[s] in gamma:
            assert new[s] == slot[s]


# --------------------------------------------------------------------------
# Attention with the additive eviction logit: torch SDPA (fp64, CPU) and closed forms
# --------------------------------------------------------------------------
@pytest.mark.parametrize("zero_e", [True, False])
def test_attend_matches_torch_sdpa(zero_e):
    rng = np.random.default_rng(5)
    G, n, d = 4, 150, 64
    q, k, v = rng.normal(size=(G, d)), rng.normal(size=(n, d)), rng.normal(size=(n, d))
    e = np.zeros(n) if zero_e else rng.normal(size=n) * 2
    out, lse = O.attend(q, k, v, e)
    tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    mask = torch.from_numpy(e)[None, None, None, :].expand(1, 1, G, n)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)[0, 0]
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    ref_lse = torch.logsumexp(tq[0, 0] @ tk[0, 0].T / math.sqrt(d) + mask[0, 0], dim=-1)
    assert np.allclose(lse, ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_attend_two_token_closed_form():
    q = np.array([[2.0, 0.0, 0.0, 0.0]])
    k = np.array([[1.0, 0, 0, 0], [0.0, 0, 0, 0]])
    v = np.array([[1.0, 2, 3, 4], [-1.0, 0, 1, 0]])
    e = np.array([0.0, 0.5])
    # logits: 2*1/2 + 0 = 1.0 and 0 + 0.5 = 0.5
    w0 = 1.0 / (1.0 + math.exp(-0.5))
    out, lse = O.attend(q, k, v, e)
    assert np.allclose(out[0], w0 * v[0] + (1 - w0) * v[1], rtol=1e-14)
    assert math.isclose(lse[0], math.log(math.exp(1.0) + math.exp(0.5)), rel_tol=1e-14)


def test_attend_identical_keys_is_eviction_softmax():
    rng = np.random.default_rng(6)
    k = np.tile(rng.normal(size=8), (10, 1))
    v, e = rng.normal(size=(10, 8)), rng.normal(size=10)
    out, _ = O.attend(rng.normal(size=(1, 8)), k, v, e)
    w = np.exp(e - e.max())
    assert np.allclose(out[0], (w / w.sum()) @ v, rtol=1e-12)


# --------------------------------------------------------------------------
# Payload byte layout: offsets worked out by hand
# --------------------------------------------------------------------------
def test_payload_layout_offsets():
    B, d = 64, 128
    k = np.arange(B * d, dtype=np.uint16).reshape(B, d)
    v = (np.arange(B * d, dtype=np.uint32) + 7).astype(np.uint16).reshape(B, d)
    e = np.arange(B, dtype=np.float32) * 0.5
    p = O.encode_payload(k, v, e, "bf16")
    assert p.size == 33024 == O.payload_bytes(64, 128, "bf16")
    u16 = lambda off: int(p[off]) | (int(p[off + 1]) << 8)
    # K(t=3, dim=17): chunk 2, element 1 -> ((2*64 + 3) * 16) + 2 = 2098
    assert u16(2098) == 3 * d + 17
    # K(t=63, dim=127): chunk 15, element 7 -> (15*64 + 63) * 16 + 14 = 16382
    assert u16(16382) == 63 * d + 127
    # V(t=5, dim=9) at 16384 + (5*128 + 9) * 2 = 17682
    assert u16(17682) == 5 * d + 9 + 7
    # e[10] at 32768 + 40
    assert np.frombuffer(p[32808:32812].tobytes(), np.float32)[0] == 5.0
    pf = O.encode_payload(np.arange(64 * 64, dtype=np.float32).reshape(64, 64),
                          np.zeros((64, 64), np.float32), np.zeros(64, np.float32), "f32")
    # f32, d=64: K(t=1, dim=6): chunk 1, element 2 -> (64 + 1) * 16 + 8 = 1048
    assert pf.size == 33024 and np.frombuffer(pf[1048:1052].tobytes(), np.float32)[0] == 70.0
    assert O.payload_bytes(64, 64, "bf16") == 16640


# --------------------------------------------------------------------------
# The unit state machine
# --------------------------------------------------------------------------
def _make_unit(w, b=0, h=0, k=None, k_e=None):
    u = O.UnitOracle(w.head_dim, w.dtype, k or w.k, w.k_e if k_e is None else k_e,
                     w.max_context, w.block, w.sub_block)
    u.append(synth.keys(w, b, h, 0, w.prompt), synth.values(w, b, h, 0, w.prompt),
             synth.evict(w, b, h, 0, w.prompt))
    return u


def _step_inputs(w, b, h, s):
    t = w.prompt + s
    return (synth.keys(w, b, h, t, 1)[0], synth.values(w, b, h, t, 1)[0],
            synth.evict(w, b, h, t, 1)[0])


def test_incremental_pool_equals_from_scratch():
    w = synth.WORKLOADS["tiny-f32"].with_(prompt=700, steps=80)
    u = _make_unit(w)
    for s in range(w.steps):
        u.begin_step(*_step_inputs(w, 0, 0, s))
    n = u.n_cand
    k, _, e = u.tokens_f64(0, n * 64)
    assert np.array_equal(u.k_bar[:n], k.reshape(n, 4, 16, 64).mean(axis=2))
    assert np.array_equal(u.se[:n], e.reshape(n, 4, 16).mean(axis=2).max(axis=1))
    assert u.L == 780 and n == 12 and u.elig[:n].all()


def test_dense_equivalence_when_k_covers_all_blocks():
    # k >= #candidates: every block is selected, so the step equals dense
    # attention over all L tokens with the eviction bias (torch SDPA, fp64).
    w = synth.WORKLOADS["tiny-f32"].with_(prompt=400, steps=3)
    u = _make_unit(w, k=16, k_e=6)
    q = synth.queries(w, 0, range(4), 3)
    for s in range(3):
        info = u.decode_step(q[s], *_step_inputs(w, 0, 0, s))
        assert len(info["gamma"]) == u.n_cand
        k, v, e = u.tokens_f64(0, u.L)
        tq = torch.from_numpy(q[s].astype(np.float64))[None, None]
        mask = torch.from_numpy(e)[None, None, None, :].expand(1, 1, 4, u.L)
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, torch.from_numpy(k)[None, None], torch.from_numpy(v)[None, None], attn_mask=mask)
        assert np.allclose(info["out"], ref[0, 0].numpy(), rtol=1e-11, atol=1e-12)


def test_bf16_unit_dense_equivalence():
    w = synth.WORKLOADS["1b-bf16"].with_(batch=1, prompt=300, steps=2)
    u = _make_unit(w, b=0, h=3, k=8, k_e=2)
    q = synth.queries(w, 0, range(6, 8), 2)      # q-heads 6, 7 belong to KV head 3 (G = 2)
    for s in range(2):
        info = u.decode_step(q[s], *_step_inputs(w, 0, 3, s))
        k, v, e = u.tokens_f64(0, u.L)
        qf = synth.storage_to_f64(q[s], "bf16")
        out, _ = O.attend(qf, k, v, e)
        assert np.allclose(info["out"], out, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("name,steps", [("tiny-f32", 200), ("1b-bf16", 160)])
def test_locality_eviction_and_slot_invariants(name, steps):
    w = synth.WORKLOADS[name]
    w = w.with_(prompt=min(w.prompt, 64 * (w.k + 6) + 17), steps=steps)
    u = _make_unit(w, b=0, h=0)
    G = w.group
    q = synth.queries(w, 0, range(G), steps)
    ever_out = set()
    prev_ge = None
    for s in range(steps):
        info = u.decode_step(q[s], *_step_inputs(w, 0, 0, s))
        ge, gq = set(info["g_e"].tolist()), set(info["g_q"].tolist())
        n = u.n_cand
        assert len(ge) == min(w.k_e, n) and len(ge) + len(gq) == min(w.k, n)
        assert n not in ge | gq                                   # tail never a candidate
        assert not (ge & ever_out)                                 # strict eviction
        if prev_ge is not None:
            ever_out |= prev_ge - ge
            newcomers = ge - prev_ge
            assert newcomers <= {u.just_completed}                 # only the new block enters
        prev_ge = ge
        assert set(int(b) for b in u.slot2blk if b >= 0) == ge | gq
        if s >= 1 and n >= w.k:
            assert info["gamma_locality"] >= w.k_e / w.k - 1e-12   # gamma(t) >= k_e / k
            assert info["n_host"] <= w.k - w.k_e
        assert info["n_host"] + sum(1 for l in info["loads"] if l[2] == O.TAIL) == len(info["loads"])


def test_cold_step_loads_everything_from_host():
    w = synth.WORKLOADS["tiny-f32"].with_(prompt=64 * 12, steps=1)
    u = _make_unit(w)
    info = u.decode_step(synth.queries(w, 0, range(4), 1)[0], *_step_inputs(w, 0, 0, 0))
    # prompt of exactly 12 blocks: block 11 was the tail and opens as a candidate now
    assert u.n_cand == 12 and u.just_completed == 11
    assert len(info["loads"]) == 8
    srcs = {l[0]: l[2] for l in info["loads"]}
    assert all(v == (O.TAIL if b == 11 else O.HOST) for b, v in srcs.items())


# --------------------------------------------------------------------------
# bf16 pooled-key variant: rounding and fp32 token-order summation
# --------------------------------------------------------------------------
def test_round_bf16_ties_to_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, -3.0],
                 dtype=np.float32)
    assert list(O.round_bf16(x)) == [1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -3.0]


def test_pooled_bf16_exact_means_unchanged():
    c = np.arange(8) * 0.25 - 1.0                      # bf16-exact values
    kb = O.pooled_keys_bf16(np.tile(c, (64, 1)), 16)
    assert np.array_equal(kb, np.tile(c, (4, 1)))


def test_pooled_bf16_follows_fp32_token_order():
    # 2**24 + 1 is not an fp32 value: summed in token order the ones vanish, so the
    # sub-block mean is 0, not the exact 14/16.
    k = np.zeros((64, 2))
    k[:16, 0] = [2.0 ** 24] + [1.0] * 14 + [-(2.0 ** 24)]
    k[:16, 1] = [1.0] * 14 + [2.0 ** 24, -(2.0 ** 24)]  # other order: exact 14/16
    kb = O.pooled_keys_bf16(k, 16)
    assert kb[0, 0] == 0.0 and kb[0, 1] == 0.875
    assert O.pool_block(k, np.zeros(64), 16)[0][0, 0] == 0.875


def test_stored_means_f32_token_order_and_exact_cases():
    # The same 2**24 construction in fp32 storage: token order decides the mean.
    k = np.zeros((64, 2))
    k[:16, 0] = [2.0 ** 24] + [1.0] * 14 + [-(2.0 ** 24)]
    k[:16, 1] = [1.0] * 14 + [2.0 ** 24, -(2.0 ** 24)]
    m = O.stored_means_f32(k, 16)
    assert m.shape == (4, 2) and m[0, 0] == 0.0 and m[0, 1] == 0.875
    # values whose every partial sum is exact in fp32: the model is the exact mean
    r = np.random.default_rng(5)
    ints = r.integers(-2000, 2000, size=(64, 8)) * 2.0 ** -7
    assert np.array_equal(O.stored_means_f32(ints, 16), O.pool_block(ints, np.zeros(64), 16)[0])
    # 1-D input (eviction logits) pools the same way as one key column
    assert np.array_equal(O.stored_means_f32(ints[:, 3], 16), O.stored_means_f32(ints, 16)[:, 3])


def test_stored_means_f32_within_the_fp32_summation_bound():
    # |fl32 token-order mean - exact mean| <= 15 u sum|x| / 16 (15 additions, u = 2^-24;
    # the product by 1/16 is exact), on values with many significant bits
    r = np.random.default_rng(6)
    x = r.standard_normal((64, 32)).astype(np.float32).astype(np.float64) * 2.0 ** r.integers(-6, 6, (64, 32))
    m32 = O.stored_means_f32(x, 16)
    exact = O.pool_block(x, np.zeros(64), 16)[0]
    bound = 15 * 2.0 ** -24 * np.abs(x).reshape(4, 16, 32).sum(axis=1) / 16
    assert np.all(np.abs(m32 - exact) <= bound)
    assert np.any(m32 != exact)  # the rounding is really there


# --------------------------------------------------------------------------
# Fused front-end: the packed projection and its split (R21, R22)
# --------------------------------------------------------------------------
def test_project_split_layout_one_hot():
    # W[r] picks hidden element r % D: each output names the row it came from.
    Hq, Hkv, d, D = 4, 2, 4, 64
    F = O.frontend_rows(Hq, Hkv, d)
    assert F == (4 + 4) * 4 + 2
    W = np.zeros((F, D))
    W[np.arange(F), np.arange(F) % D] = 1.0
    x = np.stack([np.arange(D) + 1000.0 * b for b in range(3)])
    q, k, v, e = O.project(x, W, Hq, Hkv, d)
    for b in range(3):
        for g in range(Hq):
            for dim in range(d):
                assert q[b, g, dim] == x[b, (g * d + dim) % D]
        for h in range(Hkv):
            for dim in range(d):
                assert k[b, h, dim] == x[b, (Hq * d + h * d + dim) % D]
                assert v[b, h, dim] == x[b, ((Hq + Hkv) * d + h * d + dim) % D]
            assert e[b, h] == x[b, ((Hq + 2 * Hkv) * d + h) % D]


def test_project_matches_integer_arithmetic():
    # The generator's hidden states and weights are small integers times powers
    # of two: the exact result is an integer dot product.
    w = synth.WORKLOADS["1b-bf16"]
    D = synth.hidden_width(w)
    rows = np.arange(0, O.frontend_rows(w.n_q_heads, w.n_kv_heads, w.head_dim), 37)
    xi = synth.small_ints(w.seed, synth.STREAM_HIDDEN, 3, 0, np.array([[70000]]),
                          np.arange(D)[None, :])[0]
    Wi = synth.small_ints(w.seed, synth.STREAM_WEIGHT, 0, 0, rows[:, None], np.arange(D)[None, :])
    exact = [sum(int(a) * int(c) for a, c in zip(xi, Wi[j])) * 2.0 ** -11 for j in range(len(rows))]
    x = synth.hidden(w, 3, 70000, 1, D)
    Wf = np.zeros((O.frontend_rows(w.n_q_heads, w.n_kv_heads, w.head_dim), D))
    Wf[rows] = synth.proj_weights(w, D, rows)
    q, k, v, e = O.project(x, Wf, w.n_q_heads, w.n_kv_heads, w.head_dim)
    y = np.concatenate([q.reshape(-1), k.reshape(-1), v.reshape(-1), e.reshape(-1)])
    assert list(y[rows]) == exact
    # Any fp32 summation order gives the same bits (every partial sum is exact).
    rng = np.random.default_rng(0)
    prod = (x[0][None, :] * Wf[rows]).astype(np.float32)
    for _ in range(3):
        perm = rng.permutation(D)
        acc = np.zeros(len(rows), dtype=np.float32)
        for i in perm:
            acc = np.add(acc, prod[:, i], dtype=np.float32)
        assert list(acc.astype(np.float64)) == exact


def test_frontend_storage_rounds_to_nearest_even():
    # ties to even; a value above the tie rounds up; and R22's fp32 step first:
    # 2**-30 does not survive fp64 -> fp32, so that value is a tie in bf16.
    q = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -8 + 2 ** -20,
                  1.0 + 2 ** -8 + 2 ** -30])
    qs, ks, vs, es = O.frontend_storage(q, q, q, q, "bf16")
    vals = (qs.astype(np.uint32) << np.uint32(16)).view(np.float32)
    assert list(vals) == [1.0, 1.0 + 2 ** -6, -2.5, 1.0 + 2 ** -7, 1.0]
    assert es.dtype == np.float32 and es[0] == np.float32(1.0 + 2 ** -8)


# --------------------------------------------------------------------------
# Training-time forward (R23)
# --------------------------------------------------------------------------
def _prefill_inputs(L, d, G, seed, e_scale=1.0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((L, d)).astype(np.float32)
    v = rng.standard_normal((L, d)).astype(np.float32)
    e = (e_scale * rng.standard_normal(L)).astype(np.float32)
    q = rng.standard_normal((L, G, d)).astype(np.float32)
    return k, v, e, q


def test_prefill_dense_equals_causal_sdpa():
    # k larger than the number of blocks: every position attends to every earlier
    # token, i.e. causal attention with the eviction logit as an additive bias.
    L, d, G = 300, 16, 2
    k, v, e, q = _prefill_inputs(L, d, G, 1)
    res = O.prefill_unit(k, v, e, q, "f32", k=8, k_e=3)
    kt = torch.tensor(k, dtype=torch.float64)
    vt = torch.tensor(v, dtype=torch.float64)
    qt = torch.tensor(q, dtype=torch.float64).permute(1, 0, 2)      # [G][L][d]
    bias = torch.tensor(e, dtype=torch.float64)[None, :].expand(L, L).clone()
    bias = bias.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool), 1), float("-inf"))
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, kt[None].expand(G, L, d), vt[None].expand(G, L, d), attn_mask=bias)
    for t in (0, 1, 63, 64, 65, 127, 128, 200, 299):
        assert np.allclose(res[t][2], ref[:, t].numpy(), atol=1e-12, rtol=0)


def test_prefill_first_block_attends_causally():
    L, d, G = 64, 8, 3
    k, v, e, q = _prefill_inputs(L, d, G, 2)
    res = O.prefill_unit(k, v, e, q, "f32", k=4, k_e=2)
    for t in (0, 5, 63):
        g_e, g_q, out, _ = res[t]
        assert len(g_e) == 0 and len(g_q) == 0
        ref, _ = O.attend(q[t].astype(np.float64), k[:t + 1].astype(np.float64),
                          v[:t + 1].astype(np.float64), e[:t + 1].astype(np.float64))
        assert np.allclose(out, ref, atol=1e-13, rtol=0)


def test_prefill_eviction_sets_follow_the_block_recurrence():
    # Distinct integer block eviction scores: Gamma_e at every position of block b
    # is E_b with E_0 = {} and E_b = the k_e best of E_{b-1} + {b-1}, computed here
    # by brute force on Python sets.
    B, nblk, d, G, k_e = 64, 12, 8, 1, 4
    rng = np.random.default_rng(3)
    scores = rng.permutation(nblk).astype(np.float32)
    e = np.repeat(scores, B)
    L = nblk * B
    k, v, _, q = _prefill_inputs(L, d, G, 4)
    res = O.prefill_unit(k, v, e, q, "f32", k=6, k_e=k_e, positions=set())
    E = set()
    for b in range(nblk):
        if b >= 1:
            cand = sorted(E | {b - 1}, key=lambda j: (-scores[j], j))
            E = set(cand[:k_e])
        for t in range(b * B, (b + 1) * B):
            assert set(int(x) for x in res[t][0]) == E, (b, t)


def test_prefill_strict_eviction_and_budget():
    L, d, G, kk, k_e = 64 * 14 + 9, 8, 2, 5, 3
    k, v, e, q = _prefill_inputs(L, d, G, 5)
    res = O.prefill_unit(k, v, e, q, "f32", k=kk, k_e=k_e, positions=set())
    left = set()
    prev = set()
    for t in range(L):
        g_e, g_q = set(int(x) for x in res[t][0]), set(int(x) for x in res[t][1])
        n_cand = t // 64
        assert not (g_e & g_q)
        assert len(g_e | g_q) == min(kk, n_cand)
        assert not (g_e & left)                     # once left out, never again
        left |= prev - g_e
        prev = g_e
