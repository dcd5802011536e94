"""Parity of the CUDA decode path with the fp64 oracle, through the C ABI.

Every step: selections (lock-step near-tie rule), load lists, slot tables and
gathered bytes exact; the device state (pooled keys, eviction scores,
eligibility, query scores, host-store bytes) against the oracle as the harness
describes; attention within 1e-5 absolute (fp32) or 1e-2 x row RMS (bf16). The
five workloads run at their full shapes and over their full step counts; the
large ones are checked on sampled units (units are independent, so a sampled
unit is checked exactly).
"""
import numpy as np
import pytest
import torch

import synth
import synth.gpu
import trainable_sparse_attention_decode_gb300 as nosa
from nosa_harness import GpuRun

pytestmark = pytest.mark.gpu


def _run(w, units=None, steps=None, check_every=1, attn_every=1, pieces=None, check_bytes=True,
         flags=0, state_every=1):
    steps = w.steps if steps is None else steps
    run = GpuRun(w, units=units, flags=flags, prompt_pieces=pieces, check_bytes=check_bytes,
                 oracle_attention_every=attn_every, state_every=state_every)
    q = synth.gpu.queries(w, steps)
    worst, worst_lse = 0.0, 0.0
    try:
        for s in range(steps):
            _, _, res = run.step(q[s], check=(s % check_every == 0))
            if res:
                worst = max(worst, res["worst_attn"])
                worst_lse = max(worst_lse, res["worst_lse"])
        st = run.stats()
    finally:
        run.close()
    assert st["device_error"] == 0
    assert worst <= 1.0, f"attention error / tolerance = {worst}"
    assert worst_lse <= (1e-5 if w.dtype == "f32" else 1e-4) * 10
    return st, run


def test_tiny_f32_full():
    st, run = _run(synth.WORKLOADS["tiny-f32"])
    assert st["steps"] == 32 and st["cold_host_loads"] in (7, 8)
    assert run.stats_checked  # every unit at every step: load statistics equal the oracle's


def test_1b_bf16_sampled_units():
    w = synth.WORKLOADS["1b-bf16"]
    st, _ = _run(w, units=[0, 9, 37, 63])
    k, ke = w.k, w.k_e
    assert st["gamma_min"] >= ke / k - 1e-12          # locality bound on every unit
    assert st["max_host_loads_unit"] <= k - ke


def test_3b_bf16_sampled_units():
    # all 256 decode steps of the workload
    w = synth.WORKLOADS["3b-bf16"]
    st, run = _run(w, units=[5, 127])
    assert st["steps"] == 256
    assert st["gamma_min"] >= w.k_e / w.k - 1e-12
    assert st["max_host_loads_unit"] <= w.k - w.k_e
    assert run.state_checks == 2 * (256 + 1)


def test_8b_offload_sampled_units():
    # all 64 decode steps of the workload, prompt appended in the bench's 4096-token pieces
    w = synth.WORKLOADS["8b-offload-bf16"]
    st, run = _run(w, units=[0, 255], pieces=[4096] * 16, check_bytes=True)
    assert st["steps"] == 64
    assert st["gamma_min"] >= w.k_e / w.k - 1e-12
    assert st["max_host_loads_unit"] <= w.k - w.k_e
    assert run.state_checks == 2 * (64 + 1)


@pytest.mark.parametrize("case", [
    dict(prompt=37, steps=70, k=4, k_e=2),            # starts with no candidate block
    dict(prompt=64 * 3, steps=70, k=8, k_e=3),        # fewer candidates than k for a while
    dict(prompt=64 * 10 + 5, steps=80, k=4, k_e=0),   # no query-agnostic part
    dict(prompt=64 * 10 + 63, steps=80, k=4, k_e=4),  # no query-aware part
    dict(prompt=1, steps=70, k=4, k_e=2),             # a one-token context (none: STATE error)
    dict(prompt=64 * 300 + 7, steps=40, k=256, k_e=128),  # the largest k the kernels take
])
def test_edge_cases_f32(case):
    w = synth.WORKLOADS["tiny-f32"].with_(**case)
    _run(w)


@pytest.mark.parametrize("hq,hkv,d,dtype", [(8, 8, 128, "bf16"), (12, 2, 64, "bf16"),
                                           (16, 2, 128, "f32"), (12, 4, 64, "f32"),
                                           (48, 8, 64, "bf16")])
def test_group_and_dtype_variants(hq, hkv, d, dtype):
    w = synth.Workload("var", 2, hq, hkv, d, dtype, 64 * 40 + 17, 40, 16, 10)
    _run(w)


@pytest.mark.parametrize("name,units,steps", [("tiny-f32", None, 32), ("1b-bf16", [2, 50], 64),
                                              ("8b-offload-bf16", [7, 200], 16)])
def test_pooled_bf16_variant(name, units, steps):
    # bf16 pooled keys: the oracle models the fp32 token-order sum and bf16 rounding
    w = synth.WORKLOADS[name]
    pieces = [4096] * 16 if name == "8b-offload-bf16" else None
    st, _ = _run(w, units=units, steps=steps, pieces=pieces, flags=nosa.NOSA_FLAG_POOLED_BF16)
    if w.prompt >= 64 * w.k:
        assert st["gamma_min"] >= w.k_e / w.k - 1e-12


def test_prompt_in_ragged_pieces():
    w = synth.WORKLOADS["tiny-f32"].with_(prompt=64 * 20 + 9, steps=20)
    _run(w, pieces=[1, 63, 64, 100, 28, 64 * 10, 64 * 5 + 9, 64])


def test_capacity_and_state_errors():
    w = synth.WORKLOADS["tiny-f32"].with_(prompt=128, steps=1)
    cfg = nosa.nosa_config(1, 4, 1, 64, "f32", 4, 2, 129)
    h = nosa.nosa_create(cfg)
    try:
        q = torch.zeros((1, 4, 64), device="cuda")
        kv = torch.zeros((1, 1, 64), device="cuda")
        e = torch.zeros((1, 1), device="cuda")
        out = torch.empty_like(q)
        with pytest.raises(nosa.NosaError) as ei:
            nosa.nosa_decode_step(h, q, kv, kv, e, out)
        assert ei.value.status == 6
        k, v, ee = synth.gpu.kv(w, 0, 128)
        nosa.nosa_append_kv(h, k, v, ee)
        nosa.nosa_decode_step(h, q, kv, kv, e, out)
        with pytest.raises(nosa.NosaError) as ei:
            nosa.nosa_decode_step(h, q, kv, kv, e, out)
        assert ei.value.status == 4
        with pytest.raises(nosa.NosaError) as ei:
            nosa.nosa_append_kv(h, k[:, :1], v[:, :1], ee[:, :1])
        assert ei.value.status == 4
        torch.cuda.synchronize()
        assert nosa.nosa_stats(h)["device_error"] == 0
    finally:
        nosa.nosa_destroy(h)


@pytest.mark.slow
def test_8b_longgen_sampled_units_long_horizon():
    # 16384 decode steps: selection, loads and slots checked every step on two
    # units, attention and the device state every 16th step, the host-store bytes
    # of every block that completes.
    w = synth.WORKLOADS["8b-longgen-bf16"]
    st, run = _run(w, units=[3, 100], attn_every=16, check_bytes=False, state_every=16)
    assert st["gamma_min"] >= w.k_e / w.k - 1e-12
    assert st["max_host_loads_unit"] <= w.k - w.k_e


def test_gather_numbers_entries_across_unit_tiles(monkeypatch):
    # one chunk of 2 112 units: the gather numbers a chunk's load-list entries
    # 2 048 units at a time in shared memory, so units on both sides of that
    # boundary are checked (slot bytes included)
    monkeypatch.setenv("NOSA_CHUNK_SIZES", "1")
    w = synth.WORKLOADS["1b-bf16"].with_(batch=264, prompt=64 * 12 + 9, steps=12, k=8, k_e=6)
    st, _ = _run(w, units=[0, 2047, 2048, 2049, 2111])
    assert st["host_loads"] > 0


@pytest.mark.parametrize("env", [{"NOSA_FUSED_SELECT": "0"}, {"NOSA_GATHER_STREAMS": "1"},
                                 {"NOSA_SELECT_HINT": "0"}, {"NOSA_GATHER_VEC": "32"},
                                 {"NOSA_PDL": "0"}, {"NOSA_ATTN_SPLITS": "2"}])
def test_step_switches_every_unit(env, monkeypatch):
    # The documented switches of the step (read at nosa_create) change launch
    # shapes and schedules, never the result: a selection kernel of its own, one
    # gather stream, the radix cut at every step, 32-byte gather loads, ordinary
    # instead of programmatic graph edges, a forced split count; three chunks so
    # the stream switches matter, every unit checked.
    for key, val in env.items():
        monkeypatch.setenv(key, val)
    monkeypatch.setenv("NOSA_CHUNK_SIZES", "1,2,1")
    w = synth.WORKLOADS["1b-bf16"].with_(batch=2, prompt=64 * 40 + 9, steps=40)
    _run(w)


@pytest.mark.parametrize("sizes", ["1,2,3,4,1", "3,1,1,2", "0.5,1,2,3,3,1", "0.5,1,2,3,2.5,1.5"])
def test_unequal_chunks_every_unit(sizes, monkeypatch):
    # The step's unit chunks run concurrently and differ in split counts; every
    # unit (not a sample) is checked, so a partial buffer shared across chunks
    # would show on some unit.
    monkeypatch.setenv("NOSA_CHUNK_SIZES", sizes)
    w = synth.WORKLOADS["1b-bf16"].with_(batch=2, prompt=64 * 40 + 9, steps=40)
    _run(w)
