"""Warm decode steps replay a captured graph; with NOSA_GRAPHS=0 every kernel of
every step is launched from the host. Both run the same kernels in the same
order on the same data, and the split-K merge sums the partials in a fixed
order, so the two must produce identical bytes: outputs, lse, selections, slot
tables and the pooled state. The schedules below force graph rebuilds (the
candidate count leaves a graph's score-grid window) and bulk appends between
decode steps.
"""
import os

import numpy as np
import pytest
import torch

import synth
import synth.gpu
import trainable_sparse_attention_decode_gb300 as nosa

pytestmark = pytest.mark.gpu


def _drive(w, schedule, graphs, flags=0):
    """schedule: list of ("step", n) and ("append", n) items after the prompt."""
    old = os.environ.get("NOSA_GRAPHS")
    os.environ["NOSA_GRAPHS"] = "1" if graphs else "0"
    try:
        cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k,
                               w.k_e, w.max_context, flags=flags)
        h = nosa.nosa_create(cfg)
    finally:
        if old is None:
            del os.environ["NOSA_GRAPHS"]
        else:
            os.environ["NOSA_GRAPHS"] = old
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    n_steps = sum(n for kind, n in schedule if kind == "step")
    q = synth.gpu.queries(w, n_steps)
    outs, lses = [], []
    try:
        k, v, e = synth.gpu.kv(w, 0, w.prompt)
        nosa.nosa_append_kv(h, k, v, e)
        t, s = w.prompt, 0
        for kind, n in schedule:
            if kind == "append":
                k, v, e = synth.gpu.kv(w, t, n)
                nosa.nosa_append_kv(h, k, v, e)
                t += n
                continue
            for _ in range(n):
                k, v, e = synth.gpu.kv(w, t, 1, step_major=True)
                out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=dt, device="cuda")
                lse = torch.empty((w.batch, w.n_q_heads), dtype=torch.float32, device="cuda")
                nosa.nosa_decode_step(h, q[s], k[0], v[0], e[0], out, lse)
                outs.append(out)
                lses.append(lse)
                t += 1
                s += 1
        torch.cuda.synchronize()
        state = {what: nosa.nosa_debug_read(h, what).tobytes()
                 for what in ("SEL", "NSEL", "ELIG", "SLOTS", "POOLED", "SE", "SLOTPOOL")}
        st = nosa.nosa_stats(h)
    finally:
        nosa.nosa_destroy(h)
    return torch.stack(outs).cpu(), torch.stack(lses).cpu(), state, st


def _same(a, b):
    out_a, lse_a, state_a, st_a = a
    out_b, lse_b, state_b, st_b = b
    assert torch.equal(out_a.view(torch.uint8) if out_a.dtype == torch.bfloat16 else out_a,
                       out_b.view(torch.uint8) if out_b.dtype == torch.bfloat16 else out_b)
    assert torch.equal(lse_a, lse_b)
    for what in state_a:
        assert state_a[what] == state_b[what], f"{what} differs"
    for key in ("host_loads", "tail_loads", "sum_hits", "hit_samples", "launches", "steps"):
        assert st_a[key] == st_b[key], key
    assert st_a["device_error"] == 0 and st_b["device_error"] == 0


@pytest.mark.parametrize("flags", [0, 1])
def test_graph_replay_matches_host_launches_f32(flags):
    # prompt 2024 tokens: 31 candidates, so the first graph's window ends at 32
    # and the 24th step forces a rebuild; the bulk append jumps 40 blocks ahead.
    w = synth.WORKLOADS["tiny-f32"].with_(prompt=2024, steps=200 + 64 * 40 + 17)
    schedule = [("step", 60), ("append", 64 * 40 + 17), ("step", 140)]
    a = _drive(w, schedule, graphs=True, flags=flags)
    b = _drive(w, schedule, graphs=False, flags=flags)
    _same(a, b)
    if flags:
        assert a[3]["t_count"] == 200 and b[3]["t_count"] == 200


def test_graph_replay_matches_host_launches_bf16_units():
    w = synth.WORKLOADS["1b-bf16"].with_(prompt=64 * 95 + 50, steps=90)
    a = _drive(w, [("step", 90)], graphs=True)
    b = _drive(w, [("step", 90)], graphs=False)
    _same(a, b)


def test_timing_switch():
    w = synth.WORKLOADS["tiny-f32"].with_(steps=40)
    cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e,
                           w.max_context)
    h = nosa.nosa_create(cfg)
    try:
        k, v, e = synth.gpu.kv(w, 0, w.prompt)
        nosa.nosa_append_kv(h, k, v, e)
        q = synth.gpu.queries(w, 40)
        out = torch.empty((w.batch, w.n_q_heads, w.head_dim), device="cuda")
        for s in range(40):
            if s == 10:
                nosa.nosa_set_timing(h, True)
            if s == 30:
                nosa.nosa_set_timing(h, False)
            k, v, e = synth.gpu.kv(w, w.prompt + s, 1, step_major=True)
            nosa.nosa_decode_step(h, q[s], k[0], v[0], e[0], out)
        st = nosa.nosa_stats(h)
        assert st["t_count"] == 20 and st["steps"] == 40
        assert all(t >= 0.0 for t in st["t_us"]) and st["t_us"][7] > 0.0
    finally:
        nosa.nosa_destroy(h)
