"""nosa_sparse_attention_noalloc: the block-sparse decode attention for callers
that cannot allocate device memory (a serving engine or framework that owns all
device memory in its own pool, or a loop that must not call cudaMalloc / cudaFree
because they can synchronise the device). It keeps its split-K scratch in a
static array of the library instead of a caller workspace; its output must match
nosa_sparse_attention's on the same inputs, call after call.

This file is collected last on purpose, and passes both alone in a fresh process
and after the other tests.
"""
import numpy as np
import pytest
import torch

import synth
import trainable_sparse_attention_decode_gb300 as nosa
from oracle import nosa_oracle as O

pytestmark = pytest.mark.gpu


def _case(dtype, d, hq, hkv, batch, n_blocks, seed):
    rng = np.random.default_rng(seed)
    U = batch * hkv
    pool = U * n_blocks + 1
    units = np.zeros((pool + U, O.payload_bytes(64, d, dtype)), np.uint8)
    for i in range(pool + U):
        units[i] = O.encode_payload(synth.to_storage(rng.normal(size=(64, d)), dtype),
                                    synth.to_storage(rng.normal(size=(64, d)), dtype),
                                    rng.normal(size=64).astype(np.float32), dtype)
    tab = rng.integers(-1, pool, size=(U, n_blocks)).astype(np.int32)
    q = synth.to_storage(rng.normal(size=(batch, hq, d)) * 2, dtype)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    qt = torch.from_numpy(q.view(np.int16) if dtype == "bf16" else q).cuda().view(dt)
    return (torch.from_numpy(units[:pool].reshape(-1)).cuda(),
            torch.from_numpy(units[pool:].reshape(-1)).cuda(),
            torch.from_numpy(tab).cuda(), qt, dt)


def _close(a, b, dtype):
    """The tolerance of the attention parity tests: 1e-5 absolute (fp32); for bf16
    relative RMS error <= 1e-2 and elementwise <= 1e-2 RMS + half a bf16 ulp."""
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    if dtype == "f32":
        return float(np.max(np.abs(a - b))) <= 1e-5
    rms = np.sqrt(np.mean(b ** 2, axis=-1, keepdims=True))
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(b), 1e-30))) - 8)
    return bool(np.all(np.sqrt(np.mean((a - b) ** 2, axis=-1)) <= 1e-2 * rms[..., 0])
                and np.all(np.abs(a - b) <= 1e-2 * rms + half_ulp))


@pytest.mark.parametrize("dtype,d,hq,hkv,batch,n_blocks,tail_len", [
    ("bf16", 128, 32, 8, 4, 24, 41), ("f32", 64, 4, 1, 2, 9, 64), ("bf16", 64, 16, 8, 2, 12, 1)])
def test_noalloc_matches_workspace_entry_point_twice(dtype, d, hq, hkv, batch, n_blocks, tail_len):
    units, tail, tab, q, dt = _case(dtype, d, hq, hkv, batch, n_blocks, seed=11)
    cfg = nosa.nosa_config(batch, hq, hkv, d, dtype, 8, 4, 4096)
    ws = torch.empty(nosa.nosa_attention_workspace_bytes(cfg, n_blocks), dtype=torch.uint8,
                     device="cuda")
    ref = torch.empty((batch, hq, d), dtype=dt, device="cuda")
    ref_lse = torch.empty((batch, hq), dtype=torch.float32, device="cuda")
    nosa.nosa_sparse_attention(cfg, units, tab, tail, tail_len, q, ref, ref_lse, ws)
    for _ in range(2):  # two calls in a row share (and reuse) the static scratch
        out = torch.full((batch, hq, d), float("nan"), dtype=dt, device="cuda")
        lse = torch.full((batch, hq), float("nan"), dtype=torch.float32, device="cuda")
        nosa.nosa_sparse_attention_noalloc(cfg, units, tab, tail, tail_len, q, out, lse)
        torch.cuda.synchronize()
        assert _close(out, ref, dtype)
        assert torch.allclose(lse, ref_lse, rtol=0, atol=1e-5)


@pytest.mark.parametrize("dtype,d,hq,hkv,batch,n_blocks,tail_len", [
    ("bf16", 128, 32, 8, 4, 24, 41), ("f32", 64, 4, 1, 2, 9, 64)])
def test_noalloc_matches_oracle(dtype, d, hq, hkv, batch, n_blocks, tail_len):
    # the oracle's attend() over each unit's blocks and tail, element by element,
    # with some table entries empty and one unit without any block
    from nosa_harness import attn_close, to_f64
    rng = np.random.default_rng(5)
    U, G = batch * hkv, hq // hkv
    pool = U * n_blocks + 1
    units = np.zeros((pool + U, O.payload_bytes(64, d, dtype)), np.uint8)
    toks = []
    for i in range(pool + U):
        k = synth.to_storage(rng.normal(size=(64, d)), dtype)
        v = synth.to_storage(rng.normal(size=(64, d)), dtype)
        e = rng.normal(size=64).astype(np.float32)
        units[i] = O.encode_payload(k, v, e, dtype)
        toks.append((synth.storage_to_f64(k, dtype), synth.storage_to_f64(v, dtype),
                     e.astype(np.float64)))
    tab = rng.integers(0, pool, size=(U, n_blocks)).astype(np.int32)
    tab[rng.random(size=(U, n_blocks)) < 0.15] = -1
    tab[1] = -1
    q = synth.to_storage(rng.normal(size=(batch, hq, d)) * 2, dtype)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    qt = torch.from_numpy(q.view(np.int16) if dtype == "bf16" else q).cuda().view(dt)
    cfg = nosa.nosa_config(batch, hq, hkv, d, dtype, 8, 4, 4096)
    out = torch.full((batch, hq, d), float("nan"), dtype=dt, device="cuda")
    lse = torch.full((batch, hq), float("nan"), dtype=torch.float32, device="cuda")
    nosa.nosa_sparse_attention_noalloc(cfg, torch.from_numpy(units[:pool].reshape(-1)).cuda(),
                                       torch.from_numpy(tab).cuda(),
                                       torch.from_numpy(units[pool:].reshape(-1)).cuda(),
                                       tail_len, qt, out, lse)
    torch.cuda.synchronize()
    out_np, lse_np = to_f64(out), lse.cpu().numpy()
    q64 = synth.storage_to_f64(q, dtype)
    for u in range(U):
        b, h = divmod(u, hkv)
        kt, vt, et = toks[pool + u]
        parts = [toks[i] for i in tab[u] if i >= 0] + [(kt[:tail_len], vt[:tail_len], et[:tail_len])]
        rows = slice(h * G, (h + 1) * G)
        o_ref, lse_ref = O.attend(q64[b, rows], np.concatenate([p_[0] for p_ in parts]),
                                  np.concatenate([p_[1] for p_ in parts]),
                                  np.concatenate([p_[2] for p_ in parts]))
        assert attn_close(out_np[b, rows], o_ref, dtype) <= 1.0, f"unit {u}"
        assert np.max(np.abs(lse_np[b, rows] - lse_ref)) < 1e-4, f"unit {u}"


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    # 8192 units x 8 heads x 128 dims of fp32 partials is 32 MiB per split: more
    # than the 16 MiB array whatever the split count.
    cfg = nosa.nosa_config(1024, 64, 8, 128, "bf16", 8, 4, 1 << 20)
    need = nosa.nosa_attention_workspace_bytes(cfg, 1024)
    assert need > 16 << 20
    units = torch.zeros(33024, dtype=torch.uint8, device="cuda")
    tab = torch.full((1024 * 8, 1024), -1, dtype=torch.int32, device="cuda")
    q = torch.zeros((1024, 64, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(nosa.NosaError) as ei:
        nosa.nosa_sparse_attention_noalloc(cfg, units, tab, None, 0, q, out, None)
    assert ei.value.status == 4 and "static array" in str(ei.value)
