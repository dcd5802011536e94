"""The pinned host store's layout (csrc/host_store.cu). On a host with one memory
node, a store of 1 GiB or more is laid out in transparent huge pages on which the
process holds long-term pins (the kernel may neither move nor split pages that
the GPU reads); NOSA_HOST_HUGEPAGE=0 keeps a plain cudaHostAlloc, and so does a
host that refuses the pin (injected on the host with NOSA_INJECT_FAIL=pin). The
store is only memory: every layout must give bit-identical decode results."""

import pytest
import torch

import synth
import synth.gpu
import trainable_sparse_attention_decode_gb300 as nosa

pytestmark = pytest.mark.gpu

# 8 units x 4 096 blocks of 64 tokens: a host store of about 1.1 GB
W = synth.WORKLOADS["8b-offload-bf16"].with_(batch=1, prompt=4096, steps=4, k=16, k_e=12)
MAX_CONTEXT = 262144


def _cfg():
    return nosa.nosa_config(W.batch, W.n_q_heads, W.n_kv_heads, W.head_dim, W.dtype, W.k,
                            W.k_e, MAX_CONTEXT)


def _status_kb(field):
    with open("/proc/self/status") as f:
        for line in f:
            if line.startswith(field + ":"):
                return int(line.split()[1])
    return 0


def _huge_pages_possible():
    try:
        with open("/sys/kernel/mm/transparent_hugepage/enabled") as f:
            if "[never]" in f.read():
                return False
        with open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size") as f:
            int(f.read())
    except (OSError, ValueError):
        return False
    try:
        with open("/proc/sys/kernel/io_uring_disabled") as f:
            return f.read().strip() == "0"
    except OSError:
        return True  # a kernel without the switch


def _decode(h):
    k, v, e = synth.gpu.kv(W, 0, W.prompt)
    nosa.nosa_append_kv(h, k, v, e)
    q = synth.gpu.queries(W, W.steps)
    kn, vn, en = synth.gpu.kv(W, W.prompt, W.steps, step_major=True)
    outs = []
    for s in range(W.steps):
        out = torch.empty((W.batch, W.n_q_heads, W.head_dim), dtype=torch.bfloat16, device="cuda")
        nosa.nosa_decode_step(h, q[s], kn[s], vn[s], en[s], out)
        outs.append(out)
    torch.cuda.synchronize()
    return torch.stack(outs), nosa.nosa_stats(h)


def test_store_layout_and_pins(monkeypatch):
    monkeypatch.delenv("NOSA_HOST_HUGEPAGE", raising=False)
    pin0 = _status_kb("VmPin")
    h = nosa.nosa_create(_cfg())
    try:
        st = nosa.nosa_stats(h)
        store = nosa.nosa_debug_size(h, "HOST")
        assert store >= 1 << 30
        if st["host_numa_node"] >= 0:
            assert st["host_store_kind"] == 1
        elif _huge_pages_possible():
            assert st["host_store_kind"] == 2
            assert st["host_store_pinned"] == 1
            assert (_status_kb("VmPin") - pin0) * 1024 >= store
        else:
            assert st["host_store_kind"] == 0
    finally:
        nosa.nosa_destroy(h)
    assert _status_kb("VmPin") == pin0  # the pins go with the store


def test_plain_store_switch(monkeypatch):
    monkeypatch.setenv("NOSA_HOST_HUGEPAGE", "0")
    h = nosa.nosa_create(_cfg())
    try:
        st = nosa.nosa_stats(h)
        if st["host_numa_node"] < 0:
            assert st["host_store_kind"] == 0
            assert st["host_store_pinned"] == 0
    finally:
        nosa.nosa_destroy(h)


def test_refused_pin_falls_back(monkeypatch):
    monkeypatch.delenv("NOSA_HOST_HUGEPAGE", raising=False)
    monkeypatch.setenv("NOSA_INJECT_FAIL", "pin")
    pin0 = _status_kb("VmPin")
    h = nosa.nosa_create(_cfg())
    try:
        st = nosa.nosa_stats(h)
        assert st["host_store_pinned"] == 0
        assert _status_kb("VmPin") == pin0
        # unpinned huge pages are never kept: a plain store, or a bound one in base pages
        assert st["host_store_kind"] == (1 if st["host_numa_node"] >= 0 else 0)
    finally:
        nosa.nosa_destroy(h)


def test_layouts_decode_identically(monkeypatch):
    res = {}
    for mode, inject in (("1", None), ("0", None), ("1", "pin")):
        monkeypatch.setenv("NOSA_HOST_HUGEPAGE", mode)
        if inject:
            monkeypatch.setenv("NOSA_INJECT_FAIL", inject)
        else:
            monkeypatch.delenv("NOSA_INJECT_FAIL", raising=False)
        h = nosa.nosa_create(_cfg())
        try:
            res[(mode, inject)] = _decode(h)
        finally:
            nosa.nosa_destroy(h)
    a, sa = res[("1", None)]
    assert sa["host_loads"] > sa["cold_host_loads"] > 0  # warm steps recalled from the host
    for key in (("0", None), ("1", "pin")):
        b, sb = res[key]
        assert sa["host_loads"] == sb["host_loads"]
        assert torch.equal(a, b)
    assert torch.isfinite(a.float()).all()
