"""The standalone block-sparse attention entry point against the oracle's attend()."""
import numpy as np
import pytest
import torch

import synth
import trainable_sparse_attention_decode_gb300 as nosa
from nosa_harness import attn_close, to_f64
from oracle import nosa_oracle as O

pytestmark = pytest.mark.gpu


def _units(w, n_units_total, rng):
    """Random tokens encoded as block units, with their stored values."""
    d = w.head_dim
    raw_t = np.float32 if w.dtype == "f32" else np.uint16
    toks = []
    buf = np.zeros((n_units_total, O.payload_bytes(64, d, w.dtype)), np.uint8)
    for i in range(n_units_total):
        k = synth.to_storage(rng.normal(size=(64, d)), w.dtype)
        v = synth.to_storage(rng.normal(size=(64, d)), w.dtype)
        e = rng.normal(size=64).astype(np.float32)
        buf[i] = O.encode_payload(k, v, e, w.dtype)
        toks.append((synth.storage_to_f64(k, w.dtype), synth.storage_to_f64(v, w.dtype),
                     e.astype(np.float64)))
    return buf, toks


@pytest.mark.parametrize("dtype,d,hq,hkv,n_blocks,tail_len", [
    ("f32", 64, 4, 1, 9, 37), ("bf16", 128, 32, 8, 20, 64), ("bf16", 64, 6, 2, 3, 1),
    ("f32", 128, 8, 1, 5, 0), ("bf16", 128, 24, 8, 0, 12), ("bf16", 64, 8, 8, 70, 50)])
def test_sparse_attention_matches_oracle(dtype, d, hq, hkv, n_blocks, tail_len):
    rng = np.random.default_rng(7)
    batch = 2
    w = synth.Workload("a", batch, hq, hkv, d, dtype, 0, 0, 8, 4)
    U, G = batch * hkv, hq // hkv
    pool = U * n_blocks + 3
    buf, toks = _units(w, pool + U, rng)
    tab = np.full((U, n_blocks), -1, np.int32)
    for u in range(U):
        for j in range(n_blocks):
            if rng.random() < 0.85:
                tab[u, j] = int(rng.integers(0, pool))
    qf = rng.normal(size=(batch, hq, d)) * 2
    q_store = synth.to_storage(qf, dtype)
    cfg = nosa.nosa_config(batch, hq, hkv, d, dtype, 8, 4, 4096)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    units = torch.from_numpy(buf[:pool].reshape(-1)).cuda()
    tail = torch.from_numpy(buf[pool:].reshape(-1)).cuda() if tail_len > 0 else None
    qt = torch.from_numpy(q_store.view(np.int16) if dtype == "bf16" else q_store).cuda()
    qt = qt.view(dt)
    out = torch.empty((batch, hq, d), dtype=dt, device="cuda")
    lse = torch.empty((batch, hq), dtype=torch.float32, device="cuda")
    ws = torch.empty(nosa.nosa_attention_workspace_bytes(cfg, n_blocks), dtype=torch.uint8, device="cuda")
    nosa.nosa_sparse_attention(cfg, units, torch.from_numpy(tab).cuda(), tail, tail_len, qt, out,
                               lse, ws)
    torch.cuda.synchronize()
    out_np, lse_np = to_f64(out), lse.cpu().numpy()
    q64 = synth.storage_to_f64(q_store, dtype)
    for u in range(U):
        b, h = divmod(u, hkv)
        parts = [toks[i] for i in tab[u] if i >= 0]
        if tail_len > 0:
            kt, vt, et = toks[pool + u]
            parts.append((kt[:tail_len], vt[:tail_len], et[:tail_len]))
        rows = slice(h * G, (h + 1) * G)
        if not parts:
            assert np.all(out_np[b, rows] == 0) and np.all(np.isneginf(lse_np[b, rows]))
            continue
        K = np.concatenate([p[0] for p in parts])
        V = np.concatenate([p[1] for p in parts])
        E = np.concatenate([p[2] for p in parts])
        o_ref, lse_ref = O.attend(q64[b, rows], K, V, E)
        assert attn_close(out_np[b, rows], o_ref, dtype) <= 1.0
        assert np.max(np.abs(lse_np[b, rows] - lse_ref)) < 1e-4


@pytest.mark.parametrize("dtype,d,hq,hkv,batch,n_blocks,tail_len", [
    ("bf16", 128, 32, 8, 32, 64, 33),   # the decode shape: 256 units x 65 items
    ("f32", 64, 4, 1, 256, 9, 37),      # fp32, short units
    ("bf16", 64, 8, 8, 40, 3, 0),       # no tail: every unit spread over CTAs
    ("bf16", 128, 16, 2, 128, 12, 64),  # full tail block
])
@pytest.mark.parametrize("streamk", ["1", "0"])
def test_single_launch_splits_match_oracle(dtype, d, hq, hkv, batch, n_blocks, tail_len, streamk,
                                           monkeypatch):
    """Large single launches: the stream-K split (one wave of CTAs sharing the
    concatenated item lists; units cut across CTAs, partials merged by the last)
    and the classic split, each against the oracle; some units have no block."""
    monkeypatch.setenv("NOSA_ATTN_STREAMK", streamk)
    rng = np.random.default_rng(11)
    w = synth.Workload("a", batch, hq, hkv, d, dtype, 0, 0, 8, 4)
    U, G = batch * hkv, hq // hkv
    pool = 300
    buf, toks = _units(w, pool + U, rng)
    tab = rng.integers(0, pool, size=(U, n_blocks)).astype(np.int32)
    tab[rng.random(size=(U, n_blocks)) < 0.1] = -1
    tab[3] = -1                        # units without a block
    tab[U // 2] = -1
    qf = rng.normal(size=(batch, hq, d)) * 2
    q_store = synth.to_storage(qf, dtype)
    cfg = nosa.nosa_config(batch, hq, hkv, d, dtype, 8, 4, 4096)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    units = torch.from_numpy(buf[:pool].reshape(-1)).cuda()
    tail = torch.from_numpy(buf[pool:].reshape(-1)).cuda() if tail_len > 0 else None
    qt = torch.from_numpy(q_store.view(np.int16) if dtype == "bf16" else q_store).cuda().view(dt)
    out = torch.full((batch, hq, d), float("nan"), dtype=dt, device="cuda")
    lse = torch.full((batch, hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(nosa.nosa_attention_workspace_bytes(cfg, n_blocks), dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the merge counters reset themselves: a second call is the same
        nosa.nosa_sparse_attention(cfg, units, torch.from_numpy(tab).cuda(), tail, tail_len, qt, out,
                                   lse, ws)
    torch.cuda.synchronize()
    out_np, lse_np = to_f64(out), lse.cpu().numpy()
    q64 = synth.storage_to_f64(q_store, dtype)
    for u in range(U):
        b, h = divmod(u, hkv)
        parts = [toks[i] for i in tab[u] if i >= 0]
        if tail_len > 0:
            kt, vt, et = toks[pool + u]
            parts.append((kt[:tail_len], vt[:tail_len], et[:tail_len]))
        rows = slice(h * G, (h + 1) * G)
        if not parts:
            assert np.all(out_np[b, rows] == 0) and np.all(np.isneginf(lse_np[b, rows]))
            continue
        K = np.concatenate([p[0] for p in parts])
        V = np.concatenate([p[1] for p in parts])
        E = np.concatenate([p[2] for p in parts])
        o_ref, lse_ref = O.attend(q64[b, rows], K, V, E)
        assert attn_close(out_np[b, rows], o_ref, dtype) <= 1.0, f"unit {u}"
        assert np.max(np.abs(lse_np[b, rows] - lse_ref)) < 1e-4, f"unit {u}"
