"""Parity of the training-time forward with the oracle, through the C ABI.

Every position's selection (Gamma_e then Gamma_q) is compared with the oracle's
(exact, except at near ties, where the oracle adopts the GPU's equivalent choice
and carries on: the eviction sets carry over to later positions); the attention
output within the decode path's tolerances on the checked positions.
"""
import os

import numpy as np
import pytest
import torch

import synth
import synth.gpu
import trainable_sparse_attention_decode_gb300 as nosa
from nosa_harness import near_tie_equivalent, attn_close, to_f64
from oracle import nosa_oracle as O

pytestmark = pytest.mark.gpu


def _forward(cfg, L, q, k, v, e, out, lse, sel, tiled, select_tc=True, env=None):
    """One forward with the tiled tensor-core attention and the tensor-core
    selection on or off (the switches are read at every call; env adds more);
    checks the device error word."""
    switches = {"NOSA_PREFILL_TILED": "1" if tiled else "0",
                "NOSA_PREFILL_SELECT_TC": "1" if select_tc else "0", **(env or {})}
    old = {name: os.environ.get(name) for name in switches}
    os.environ.update(switches)
    try:
        ws = nosa.nosa_prefill_forward(cfg, q, k, v, e, out, lse, sel)
        assert nosa.nosa_prefill_device_error(cfg, L, ws) == 0
    finally:
        for name, value in old.items():
            if value is None:
                del os.environ[name]
            else:
                os.environ[name] = value
    torch.cuda.synchronize()


def _prefill(w, L, units=None, attn_every=1, tiled=True, select_tc=True, env=None):
    cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e,
                           max(L, 1))
    k, v, e = synth.gpu.kv(w, 0, L)
    q = synth.gpu.queries(w, L).permute(1, 0, 2, 3).contiguous()   # [batch][L][Hq][d]
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.batch, L, w.n_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    sel = torch.empty((w.batch, L, w.n_kv_heads, w.k), dtype=torch.int32, device="cuda")
    _forward(cfg, L, q, k, v, e, out, lse, sel, tiled, select_tc, env)
    assert not torch.isnan(out.float()).any(), "an output row was not written"
    assert not torch.isnan(lse).any(), "an lse entry was not written"
    sel_h = sel.cpu().numpy()
    out_h, lse_h = to_f64(out), lse.cpu().numpy().astype(np.float64)
    G = w.group
    units = range(w.units) if units is None else units
    worst, worst_lse, ties = 0.0, 0.0, 0
    for u in units:
        b, h = divmod(u, w.n_kv_heads)
        k_raw = synth.keys(w, b, h, 0, L)
        v_raw = synth.values(w, b, h, 0, L)
        e_raw = synth.evict(w, b, h, 0, L)
        q_raw = synth.queries(w, b, range(h * G, (h + 1) * G), L)
        tie_count = [0]

        def choose(t, sq, se, elig, g_e, g_q):
            row = sel_h[b, t, h]
            ne, nq = len(g_e), len(g_q)
            gpu_e, gpu_q = row[:ne], row[ne:ne + nq]
            assert (row[ne + nq:] == -1).all(), f"unit {u} t {t}: selection longer than the oracle's"
            n = len(sq)
            eligible = [i for i in range(n) if elig[i]]
            ok, tie = near_tie_equivalent(se, eligible, g_e, gpu_e)
            assert ok, f"unit {u} t {t}: Gamma_e {sorted(gpu_e)} != oracle {sorted(g_e)}"
            tie_count[0] += tie
            ge = np.array(sorted(int(x) for x in gpu_e), dtype=np.int64)
            rest = np.setdiff1d(np.arange(n), ge)
            g_q_o = O.top_m(sq, rest, min(w.k - len(ge), len(rest)))
            ok, tie = near_tie_equivalent(sq, rest, g_q_o, gpu_q)
            assert ok, f"unit {u} t {t}: Gamma_q {sorted(gpu_q)} != oracle {sorted(g_q_o)}"
            tie_count[0] += tie
            assert list(gpu_e) == sorted(gpu_e) and list(gpu_q) == sorted(gpu_q)
            return ge, np.array(sorted(int(x) for x in gpu_q), dtype=np.int64)

        positions = set(range(0, L, attn_every)) | {L - 1}
        res = O.prefill_unit(k_raw, v_raw, e_raw, q_raw, w.dtype, w.k, w.k_e,
                             positions=positions, choose=choose)
        ties += tie_count[0]
        for t in sorted(positions):
            o_ref, lse_ref = res[t][2], res[t][3]
            rows = slice(h * G, (h + 1) * G)
            worst = max(worst, attn_close(out_h[b, t, rows], o_ref, w.dtype))
            worst_lse = max(worst_lse, float(np.max(np.abs(lse_h[b, t, rows] - lse_ref))))
    assert worst <= 1.0, f"attention error / tolerance = {worst}"
    assert worst_lse <= (1e-4 if w.dtype == "f32" else 1e-3)
    return ties


def test_tiny_f32_every_position():
    w = synth.WORKLOADS["tiny-f32"]
    _prefill(w, 2048 + 37)


@pytest.mark.parametrize("L", [1, 37, 64, 65, 64 * 9])
def test_short_sequences(L):
    _prefill(synth.WORKLOADS["tiny-f32"], L)


@pytest.mark.parametrize("select_tc", [True, False])
@pytest.mark.parametrize("k_e", [0, 8])
def test_query_only_and_eviction_only(k_e, select_tc):
    w = synth.WORKLOADS["tiny-f32"].with_(k_e=k_e)
    _prefill(w, 64 * 30 + 11, select_tc=select_tc)


@pytest.mark.parametrize("k,k_e,select_tc", [(40, 16, True), (40, 16, False), (48, 8, True)])
def test_selection_widths(k, k_e, select_tc):
    # Gamma_q of up to 24 blocks (32-entry lists: the tensor-core selection's per
    # position, the CUDA-core selection's per lane) and of up to 37 (beyond 32:
    # the CUDA-core selection's warp arg-max rounds, whatever the switch says)
    w = synth.WORKLOADS["tiny-f32"].with_(k=k, k_e=k_e)
    _prefill(w, 64 * 45 + 7, select_tc=select_tc)


def test_8b_shape_cuda_core_selection():
    # the CUDA-core selection (NOSA_PREFILL_SELECT_TC=0) at the 8B shape
    w = synth.WORKLOADS["8b-offload-bf16"].with_(batch=1)
    _prefill(w, 4096 + 128 + 5, units=[0, 5], attn_every=11, select_tc=False)


@pytest.mark.parametrize("tiled", [True, False])
def test_1b_shape_sampled_units(tiled):
    # G = 2, d = 64: one 128-row tile per query block
    w = synth.WORKLOADS["1b-bf16"].with_(batch=2)
    _prefill(w, 8192 + 100, units=[0, 13], attn_every=7, tiled=tiled)


@pytest.mark.parametrize("tiled", [True, False])
def test_8b_shape_sampled_units(tiled):
    # G = 4, d = 128: two 128-row tiles per query block
    w = synth.WORKLOADS["8b-offload-bf16"].with_(batch=1)
    _prefill(w, 4096 + 128 + 5, units=[0, 5], attn_every=11, tiled=tiled)


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (12, 2, 64), (8, 2, 64), (4, 4, 64)])
def test_group_variants(hq, hkv, d):
    # G = 1 (half of the 128-row tile empty), G = 6 (split-K path), G = 4 with d = 64
    w = synth.WORKLOADS["1b-bf16"].with_(batch=1, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                                         k=16, k_e=12)
    _prefill(w, 64 * 20 + 3, units=[0, hkv - 1], attn_every=3)


_TILE_W = synth.WORKLOADS["8b-offload-bf16"].with_(batch=2, n_q_heads=8, n_kv_heads=2, k=8, k_e=6)


@pytest.mark.parametrize("L", [1, 37, 64, 65, 64 * 9 + 5])
def test_tiled_short_and_ragged(L):
    # a single partial block, exact block ends, a ragged last query block
    _prefill(_TILE_W, L)


@pytest.mark.parametrize("k_e", [0, 8])
def test_tiled_query_only_and_eviction_only(k_e):
    _prefill(_TILE_W.with_(k_e=k_e), 64 * 30 + 11, attn_every=2)


def test_tiled_matches_split_path():
    # both attention paths on the same inputs: same selections, outputs within
    # the bf16 tolerance of each other
    w = synth.WORKLOADS["8b-offload-bf16"].with_(batch=1, n_kv_heads=4, n_q_heads=16)
    L = 64 * 40 + 17
    cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e, L)
    k, v, e = synth.gpu.kv(w, 0, L)
    q = synth.gpu.queries(w, L).permute(1, 0, 2, 3).contiguous()
    res = []
    for tiled in (True, False):
        out = torch.empty_like(q)
        lse = torch.empty((1, L, w.n_q_heads), dtype=torch.float32, device="cuda")
        sel = torch.empty((1, L, w.n_kv_heads, w.k), dtype=torch.int32, device="cuda")
        _forward(cfg, L, q, k, v, e, out, lse, sel, tiled)
        res.append((out.float(), lse, sel))
    assert torch.equal(res[0][2], res[1][2])
    d = (res[0][0] - res[1][0]).float()
    rms = res[1][0].float().pow(2).mean().sqrt()
    assert float(d.pow(2).mean().sqrt() / rms) <= 1e-2
    assert float((res[0][1] - res[1][1]).abs().max()) <= 1e-3


def test_workspace_and_argument_errors():
    cfg = nosa.nosa_config(1, 4, 1, 64, "f32", 8, 6, 1000)
    assert nosa.nosa_prefill_workspace_bytes(cfg, 1001) == 0
    assert nosa.nosa_prefill_workspace_bytes(cfg, 0) == 0
    n = nosa.nosa_prefill_workspace_bytes(cfg, 500)
    assert n > 0
    ws = torch.empty(n - 256, dtype=torch.uint8, device="cuda")
    q = torch.zeros((1, 500, 4, 64), device="cuda")
    kv = torch.zeros((1, 500, 1, 64), device="cuda")
    e = torch.zeros((1, 500, 1), device="cuda")
    with pytest.raises(nosa.NosaError) as ei:
        nosa.nosa_prefill_forward(cfg, q, kv, kv, e, torch.empty_like(q), workspace=ws)
    assert ei.value.status == 1


@pytest.mark.parametrize("tiled", [True, False])
def test_phase_timing(tiled):
    # NOSA_FLAG_TIMING in the config: the call records events around its phases
    w = _TILE_W
    L = 64 * 12 + 5
    cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e, L,
                           flags=nosa.NOSA_FLAG_TIMING)
    k, v, e = synth.gpu.kv(w, 0, L)
    q = synth.gpu.queries(w, L).permute(1, 0, 2, 3).contiguous()
    out = torch.empty_like(q)
    _forward(cfg, L, q, k, v, e, out, None, None, tiled)
    f_ms, a_ms = nosa.nosa_prefill_timing()
    assert 0.0 < f_ms < 1000.0 and 0.0 < a_ms < 1000.0


@pytest.mark.slow
@pytest.mark.parametrize("k,select_tc", [(16, True), (16, False), (40, True)])
def test_long_sequence_fallback_paths(k, select_tc):
    # 700 blocks, up to 695 candidates outside E_b: 22 chunks of the tensor-core
    # selection; on the CUDA-core selection the score scratch of 8 positions per
    # warp no longer fits (4 per pooled-key pass); with k = 40, Gamma_q of up to 36
    # blocks beyond 512 candidates (the CUDA-core arg-max rounds over keys in
    # shared memory); the tiled attention with 700-block unions
    w = synth.WORKLOADS["1b-bf16"].with_(batch=1, n_q_heads=4, n_kv_heads=1, head_dim=64, k=k, k_e=4)
    _prefill(w, 64 * 700 + 13, attn_every=97, select_tc=select_tc)


@pytest.mark.parametrize("pb", [1, 2])
@pytest.mark.parametrize("name", ["tiny-f32", "1b-bf16"])
def test_cuda_core_selection_narrow_passes(pb, name):
    # The CUDA-core selection scores 8, 4, 2 or 1 positions per warp in one pass
    # over the pooled keys, the most whose score scratch fits in shared memory;
    # widths 2 and 1 take over only beyond about 1 200 and 2 400 blocks.
    # NOSA_PREFILL_SELECT_PB caps the width, so a short sequence runs them.
    w = synth.WORKLOADS[name].with_(batch=1, k=24, k_e=8)
    _prefill(w, 64 * 45 + 7, units=[0, w.n_kv_heads - 1] if w.n_kv_heads > 1 else None,
             attn_every=5, select_tc=False, env={"NOSA_PREFILL_SELECT_PB": str(pb)})


@pytest.mark.slow
def test_cuda_core_selection_two_position_pass_natural():
    # 1 216 blocks at d = 64: the score scratch of 4 positions per warp no longer
    # fits, so the CUDA-core selection takes its 2-position passes on its own;
    # every position's selection is checked, the attention on sampled positions
    w = synth.WORKLOADS["1b-bf16"].with_(batch=1, n_q_heads=4, n_kv_heads=1, head_dim=64, k=16, k_e=8)
    _prefill(w, 64 * 1215 + 9, attn_every=1999, select_tc=False)
