"""Parity of the fused front-end path with the oracle, through the C ABI.

A step starts from hidden states: the projection (query, key and value heads and
the eviction head) runs on the tensor cores in the kernel that also appends and
pools the new token; the rest of the step is the plain one. The generator's
hidden states and weights are small integers times powers of two, so every fp32
partial sum of the projection is exact whatever the order of the additions: the
projected queries are compared bit for bit, the projected keys, values and
eviction logits through every downstream check (pooling, selections, loads,
slot tables, gathered bytes, attention) exactly as in the plain parity tests.
"""
import numpy as np
import pytest
import torch

import synth
import synth.gpu
import trainable_sparse_attention_decode_gb300 as nosa
from nosa_harness import FrontRun

pytestmark = pytest.mark.gpu


def _run(w, units=None, steps=None, plain_first=0, check_bytes=True, real=False):
    steps = w.steps if steps is None else steps
    run = FrontRun(w, units=units, real=real, **({} if real else {"check_bytes": check_bytes}))
    q = synth.gpu.queries(w, plain_first) if plain_first else None
    worst, worst_lse = 0.0, 0.0
    try:
        for s in range(steps):
            if s < plain_first:
                _, _, res = run.step(q[s])
            else:
                _, _, res = run.step_hidden()
            worst = max(worst, res["worst_attn"])
            worst_lse = max(worst_lse, res["worst_lse"])
        st = run.stats()
    finally:
        run.close()
    assert st["device_error"] == 0
    assert worst <= 1.0, f"attention error / tolerance = {worst}"
    assert worst_lse <= 1e-3
    if real:
        assert run.proj_checked == (steps - plain_first) * len(run.units)
    return st


def test_tiny_bf16_all_units():
    # one request, one KV head, d = 64, hidden 256: 4 row tiles x 4 splits
    w = synth.WORKLOADS["tiny-f32"].with_(name="tiny-bf16", dtype="bf16", steps=70)
    st = _run(w)
    assert st["steps"] == 70


def test_1b_shape_sampled_units():
    # prompt ends on a block boundary: the first step promotes a block; 48 steps
    # cross three sub-block ends
    w = synth.WORKLOADS["1b-bf16"].with_(steps=48)
    _run(w, units=[2, 50, 63])


def test_8b_offload_shape_sampled_units():
    # hidden 4096, 6152 packed rows: 49 row tiles x 2 splits, the bench's shape
    w = synth.WORKLOADS["8b-offload-bf16"].with_(steps=20)
    _run(w, units=[7, 200], check_bytes=False)


def test_padded_batch_and_ragged_prompt():
    # batch 40 pads the MMA's N to 48 (three 16-column loads), a prompt that ends
    # mid sub-block
    w = synth.WORKLOADS["1b-bf16"].with_(batch=40, prompt=4096 + 17, steps=40)
    _run(w, units=[0, 161, 319])


def test_max_batch():
    # batch 256, the largest the front-end takes: N = 256 per MMA (256
    # tensor-memory columns), the epilogue in eight chunks of 32 requests
    w = synth.WORKLOADS["tiny-f32"].with_(name="tiny-bf16", dtype="bf16", batch=256,
                                          prompt=300, steps=20)
    _run(w, units=[0, 77, 255])


def test_plain_steps_then_hidden_steps():
    # the handle switches from the plain step to the front-end (a new step graph)
    w = synth.WORKLOADS["tiny-f32"].with_(name="tiny-bf16", dtype="bf16", steps=40)
    _run(w, plain_first=12)


def test_real_valued_inputs_tiny():
    # hidden states and weights are bf16 normals: the projection's fp32 sums are
    # inexact, so q, k, v and e are checked elementwise against the oracle's fp64
    # projection within the accumulation bound plus one rounding of the stored type
    w = synth.WORKLOADS["tiny-f32"].with_(name="tiny-bf16", dtype="bf16", steps=40)
    _run(w, real=True)


def test_real_valued_inputs_8b_shape():
    # hidden 4096 (the bench's shape): 49 row tiles, split-K over the hidden width
    w = synth.WORKLOADS["8b-offload-bf16"].with_(batch=4, prompt=4096 + 50, steps=24)
    _run(w, units=[0, 13, 31], real=True)


def test_pack_layout():
    # the packed tile layout read back against its definition
    w = synth.WORKLOADS["1b-bf16"]
    cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, "bf16", w.k, w.k_e,
                           w.max_context)
    D = synth.hidden_width(w)
    W = synth.gpu.proj_weights(w, D)
    P = nosa.nosa_frontend_pack(cfg, W).cpu().numpy()
    Wn = W.view(torch.int16).cpu().numpy().view(np.uint16)
    F, kblocks = Wn.shape[0], D // 64
    tiles = (F + 127) // 128
    assert P.size == tiles * kblocks * 16384
    for t, kb, r, c in [(0, 0, 0, 0), (0, 3, 9, 5), (tiles - 1, kblocks - 1, 127, 7),
                        (tiles - 1, 0, (F - 1) % 128, 2), (5, 7, 100, 1)]:
        off = (t * kblocks + kb) * 16384 + r * 128 + ((c ^ (r % 8)) * 16)
        got = P[off:off + 16].view(np.uint16)
        row = t * 128 + r
        want = Wn[row, kb * 64 + c * 8:kb * 64 + c * 8 + 8] if row < F else np.zeros(8, np.uint16)
        assert np.array_equal(got, want)
    # rows past F are zero
    r = F % 128
    if r:
        off = ((tiles - 1) * kblocks) * 16384 + r * 128
        assert not P[off:off + 128].any()


def test_frontend_argument_errors():
    w = synth.WORKLOADS["tiny-f32"].with_(prompt=128, steps=1)
    cfg32 = nosa.nosa_config(1, 4, 1, 64, "f32", 4, 2, 256)
    h = nosa.nosa_create(cfg32)
    try:
        k, v, e = synth.gpu.kv(w, 0, 128)
        nosa.nosa_append_kv(h, k, v, e)
        x = torch.zeros((1, 256), dtype=torch.bfloat16, device="cuda")
        W = torch.zeros(nosa.nosa_frontend_packed_bytes(cfg32, 256), dtype=torch.uint8, device="cuda")
        out = torch.empty((1, 4, 64), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(nosa.NosaError) as ei:
            nosa.nosa_decode_step_hidden(h, x, W, out)
        assert ei.value.status == 7  # UNSUPPORTED: fp32 handle
    finally:
        nosa.nosa_destroy(h)
    wb = w.with_(dtype="bf16")
    cfg = nosa.nosa_config(1, 4, 1, 64, "bf16", 4, 2, 256)
    h = nosa.nosa_create(cfg)
    try:
        k, v, e = synth.gpu.kv(wb, 0, 128)
        nosa.nosa_append_kv(h, k, v, e)
        x = torch.zeros((1, 96), dtype=torch.bfloat16, device="cuda")
        W = torch.zeros(4096, dtype=torch.uint8, device="cuda")
        out = torch.empty((1, 4, 64), dtype=torch.bfloat16, device="cuda")
        # straight through the C ABI (the binding's own size check would stop it first)
        st = nosa.lib.nosa_decode_step_hidden(h, x.data_ptr(), 96, W.data_ptr(), None,
                                              out.data_ptr(), None, None)
        assert st == 1  # INVALID_ARG: hidden not a multiple of 64
        assert nosa.nosa_stats(h)["steps"] == 0
    finally:
        nosa.nosa_destroy(h)
