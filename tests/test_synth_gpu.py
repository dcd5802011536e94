"""The CUDA twin of the input generator writes exactly what the numpy generator defines."""
import numpy as np
import pytest
import torch

import synth
import synth.gpu

pytestmark = pytest.mark.gpu


def _np(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny-f32", "1b-bf16", "8b-offload-bf16"])
def test_kv_matches_numpy(name):
    w = synth.WORKLOADS[name]
    t0, n = 2000, 150
    k, v, e = synth.gpu.kv(w, t0, n)
    ks, vs, es = synth.gpu.kv(w, t0, n, step_major=True)
    for b, h in [(0, 0), (w.batch - 1, w.n_kv_heads - 1), (w.batch // 2, 0)]:
        assert np.array_equal(_np(k[b, :, h]), synth.keys(w, b, h, t0, n))
        assert np.array_equal(_np(v[b, :, h]), synth.values(w, b, h, t0, n))
        assert np.array_equal(_np(e[b, :, h]), synth.evict(w, b, h, t0, n))
        assert np.array_equal(_np(ks[:, b, h]), synth.keys(w, b, h, t0, n))
        assert np.array_equal(_np(es[:, b, h]), synth.evict(w, b, h, t0, n))


@pytest.mark.parametrize("name", ["tiny-f32", "8b-longgen-bf16"])
def test_queries_match_numpy(name):
    w = synth.WORKLOADS[name]
    q = synth.gpu.queries(w, 300)
    for b, heads in [(0, [0, 1]), (w.batch - 1, [w.n_q_heads - 1])]:
        assert np.array_equal(_np(q[:, b, heads]), synth.queries(w, b, heads, 300))


@pytest.mark.parametrize("name", ["1b-bf16", "8b-offload-bf16"])
def test_frontend_inputs_match_numpy(name):
    w = synth.WORKLOADS[name]
    D = synth.hidden_width(w)
    x = synth.gpu.hidden(w, 65530, 3)
    W = synth.gpu.proj_weights(w)
    for b in (0, w.batch - 1):
        ref = synth.to_storage(synth.hidden(w, b, 65530, 3, D), "bf16")
        assert np.array_equal(_np(x[:, b]), ref)
    rows = np.array([0, 1, 777, W.shape[0] - 1])
    assert np.array_equal(_np(W[rows]), synth.to_storage(synth.proj_weights(w, D, rows), "bf16"))


@pytest.mark.parametrize("base", [32, 992])
def test_request_base_shards_the_job(base):
    # a rank's requests start at request_base: both generators agree there, and
    # the values differ from those of the job's first requests
    w = synth.WORKLOADS["8b-offload-bf16"].with_(request_base=base)
    w0 = synth.WORKLOADS["8b-offload-bf16"]
    k, v, e = synth.gpu.kv(w, 100, 70)
    q = synth.gpu.queries(w, 5)
    x = synth.gpu.hidden(w, 100, 2)
    for b, h in [(0, 0), (w.batch - 1, w.n_kv_heads - 1)]:
        assert np.array_equal(_np(k[b, :, h]), synth.keys(w, b, h, 100, 70))
        assert np.array_equal(_np(v[b, :, h]), synth.values(w, b, h, 100, 70))
        assert np.array_equal(_np(e[b, :, h]), synth.evict(w, b, h, 100, 70))
        assert np.array_equal(_np(q[:, b, [0, 5]]), synth.queries(w, b, [0, 5], 5))
        assert np.array_equal(_np(x[:, b]), synth.to_storage(synth.hidden(w, b, 100, 2), "bf16"))
        assert not np.array_equal(synth.keys(w, b, h, 100, 70), synth.keys(w0, b, h, 100, 70))
