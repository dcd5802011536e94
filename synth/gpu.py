"""Device-side generation of the synthetic inputs (CUDA twin of ``synth``).

Builds ``synth/_lib/libsynth.so`` from ``synth/gen.cu`` and fills torch CUDA
tensors with exactly the values ``synth`` defines (checked bit for bit by the
tests). Shared by the tests and the bench.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

from . import Workload, q_start_scale

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.cu")
_LIB = os.path.join(_HERE, "_lib", "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    nvcc = os.environ.get("NVCC") or "nvcc"
    tmp = _LIB + ".tmp"
    cmd = [nvcc, "-shared", "-o", tmp, _SRC, "-gencode", "arch=compute_103a,code=sm_103a",
           "-O3", "-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {_SRC}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        L.synth_kv.restype = C.c_int
        L.synth_kv.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                               C.c_longlong, C.c_int, C.c_int, C.c_ulonglong, C.c_int, C.c_int,
                               C.c_int, C.c_void_p]
        L.synth_hidden.restype = C.c_int
        L.synth_hidden.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_longlong, C.c_int,
                                   C.c_ulonglong, C.c_int, C.c_void_p]
        L.synth_proj_weights.restype = C.c_int
        L.synth_proj_weights.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_ulonglong, C.c_void_p]
        L.synth_queries.restype = C.c_int
        L.synth_queries.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_double,
                                    C.c_double,
                                    C.c_ulonglong, C.c_int, C.c_int, C.c_void_p]
        _lib = L
    return _lib


def _torch_dtype(w: Workload):
    import torch
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def kv(w: Workload, t0: int, n: int, device="cuda", step_major=False):
    """Keys, values [batch][n][Hkv][d] and eviction logits [batch][n][Hkv] of tokens t0..t0+n-1.

    With step_major the layouts are [n][batch][Hkv][d] and [n][batch][Hkv], so that
    token s of every request is one contiguous decode-step input.
    """
    import torch
    dt = _torch_dtype(w)
    if step_major:
        shp = (n, w.batch, w.n_kv_heads, w.head_dim)
    else:
        shp = (w.batch, n, w.n_kv_heads, w.head_dim)
    k = torch.empty(shp, dtype=dt, device=device)
    v = torch.empty(shp, dtype=dt, device=device)
    e = torch.empty(shp[:3], dtype=torch.float32, device=device)
    err = _get().synth_kv(k.data_ptr(), v.data_ptr(), e.data_ptr(), w.batch, w.n_kv_heads,
                          w.head_dim, t0, n, w.block, w.seed, 0 if w.dtype == "f32" else 1,
                          1 if step_major else 0, w.request_base,
                          torch.cuda.current_stream().cuda_stream)
    if err:
        raise RuntimeError(f"synth_kv: CUDA error {err}")
    return k, v, e


def queries(w: Workload, steps: int, device="cuda"):
    """AR(1) queries of every request and query head: [steps][batch][Hq][d]."""
    import torch
    q = torch.empty((steps, w.batch, w.n_q_heads, w.head_dim), dtype=_torch_dtype(w), device=device)
    err = _get().synth_queries(q.data_ptr(), w.batch, w.n_q_heads, w.head_dim, steps, w.rho,
                               q_start_scale(w),
                               w.seed, 0 if w.dtype == "f32" else 1, w.request_base,
                               torch.cuda.current_stream().cuda_stream)
    if err:
        raise RuntimeError(f"synth_queries: CUDA error {err}")
    return q


def hidden(w: Workload, t0: int, n: int, D: int | None = None, device="cuda"):
    """Front-end hidden states of tokens t0..t0+n-1: [n][batch][D] bf16 (token-major)."""
    import torch
    from . import hidden_width
    D = hidden_width(w) if D is None else D
    x = torch.empty((n, w.batch, D), dtype=torch.bfloat16, device=device)
    err = _get().synth_hidden(x.data_ptr(), w.batch, D, t0, n, w.seed, w.request_base,
                              torch.cuda.current_stream().cuda_stream)
    if err:
        raise RuntimeError(f"synth_hidden: CUDA error {err}")
    return x


def proj_weights(w: Workload, D: int | None = None, device="cuda"):
    """Packed front-end weights [F][D] bf16 (query, key, value heads, eviction rows)."""
    import torch
    from . import hidden_width
    D = hidden_width(w) if D is None else D
    F = (w.n_q_heads + 2 * w.n_kv_heads) * w.head_dim + w.n_kv_heads
    W = torch.empty((F, D), dtype=torch.bfloat16, device=device)
    err = _get().synth_proj_weights(W.data_ptr(), F, D, w.seed,
                                    torch.cuda.current_stream().cuda_stream)
    if err:
        raise RuntimeError(f"synth_proj_weights: CUDA error {err}")
    return W
