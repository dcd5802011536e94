"""Failure detection without a GPU fault: every wait in the kernels is bounded.
A wait that nothing completes must give up after its limit, report a timeout to
the host, and leave the context usable."""
import pytest
import torch

import synth
import synth.gpu
import trainable_sparse_attention_decode_gb300 as nosa

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports():
    timed_out, waited_ms = nosa.nosa_selftest_bounded_wait(0, 200_000_000)
    assert timed_out
    assert 150 <= waited_ms <= 2000
    # the context still runs work afterwards
    w = synth.WORKLOADS["tiny-f32"].with_(prompt=200, steps=1, k=2, k_e=1)
    cfg = nosa.nosa_config(1, 4, 1, 64, "f32", 2, 1, 256)
    h = nosa.nosa_create(cfg)
    try:
        k, v, e = synth.gpu.kv(w, 0, 200)
        nosa.nosa_append_kv(h, k, v, e)
        q = synth.gpu.queries(w, 1)[0]
        kn, vn, en = synth.gpu.kv(w, 200, 1, step_major=True)
        out = torch.empty((1, 4, 64), device="cuda")
        nosa.nosa_decode_step(h, q, kn[0], vn[0], en[0], out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert nosa.nosa_stats(h)["device_error"] == 0
    finally:
        nosa.nosa_destroy(h)


def test_bounded_wait_rejects_bad_limits():
    with pytest.raises(nosa.NosaError):
        nosa.nosa_selftest_bounded_wait(0, 0)
