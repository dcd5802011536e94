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


# --------------------------------------------------------------------------
# Allocation failures injected on the host (NOSA_INJECT_FAIL, read at every
# nosa_create): the allocation reports exhaustion without being attempted, so
# no GPU fault is involved. The create must return the right status, leave its
# output handle NULL, release everything it had allocated, and the next create
# must succeed.
# --------------------------------------------------------------------------
import ctypes as C


def _create_raw(cfg):
    h = C.c_void_p(12345)  # a non-NULL sentinel: the call must overwrite it
    st = nosa.lib.nosa_create(C.byref(cfg), C.byref(h))
    return st, h


def _last_device_allocation(cfg, monkeypatch):
    # the index of nosa_create's last device allocation: the largest N whose
    # injected failure still fails the create
    n = 0
    while True:
        monkeypatch.setenv("NOSA_INJECT_FAIL", f"dev:{n + 1}")
        st, h = _create_raw(cfg)
        if st == 0:
            nosa.lib.nosa_destroy(h)
            monkeypatch.delenv("NOSA_INJECT_FAIL")
            return n
        n += 1
        assert n < 200


@pytest.mark.parametrize("spec,status", [("host", 3), ("dev:0", 2), ("dev:1", 2), ("dev:9", 2),
                                         ("dev:last", 2)])
def test_injected_allocation_failure(spec, status, monkeypatch):
    # about 140 MB of device state (the slot pool and the pooled keys are 67 MB
    # each) and 1.1 GB of pinned host store; a leaked device allocation would show
    w = synth.WORKLOADS["8b-offload-bf16"].with_(batch=4)
    cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e,
                           w.max_context)
    if spec == "dev:last":
        spec = f"dev:{_last_device_allocation(cfg, monkeypatch)}"
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    monkeypatch.setenv("NOSA_INJECT_FAIL", spec)
    for _ in range(3):  # repeated failures do not accumulate anything either
        st, h = _create_raw(cfg)
        assert st == status, nosa.nosa_last_error(None)
        assert h.value is None
        assert nosa.nosa_last_error(None)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free0 - free1) < 64 << 20, f"device memory not released: {free0 - free1} bytes"
    monkeypatch.delenv("NOSA_INJECT_FAIL")
    h = nosa.nosa_create(cfg)  # the next create succeeds and the handle works
    try:
        k, v, e = synth.gpu.kv(w, 0, 256)
        nosa.nosa_append_kv(h, k, v, e)
        q = synth.gpu.queries(w, 1)[0]
        kn, vn, en = synth.gpu.kv(w, 256, 1, step_major=True)
        out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
        nosa.nosa_decode_step(h, q, kn[0], vn[0], en[0], out)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert nosa.nosa_stats(h)["device_error"] == 0
    finally:
        nosa.nosa_destroy(h)
    torch.cuda.synchronize()
    free2, _ = torch.cuda.mem_get_info()
    assert abs(free0 - free2) < 64 << 20


def test_injection_spec_without_match_changes_nothing(monkeypatch):
    monkeypatch.setenv("NOSA_INJECT_FAIL", "dev:999")  # beyond the create's allocations
    cfg = nosa.nosa_config(1, 4, 1, 64, "f32", 2, 1, 256)
    h = nosa.nosa_create(cfg)
    nosa.nosa_destroy(h)
