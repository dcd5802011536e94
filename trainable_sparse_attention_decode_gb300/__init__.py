"""Python binding of libnosa (the NOSA decode-step hot path on one GB300).

Thin ctypes marshalling over the C ABI declared in ``include/nosa.h``: every
function here has the C function's name, checks tensor shapes, dtypes, devices
and alignment, passes raw pointers and the current CUDA stream, and raises
``NosaError`` on a non-OK status. All arithmetic runs in the CUDA kernels of
``_lib/libnosa.so``; there is no CPU path. If the library has not been built the
import fails loudly (build it with ``__graft_entry__.build()`` or
``python -m trainable_sparse_attention_decode_gb300._build``).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

__all__ = [
    "NosaError", "NosaConfig", "NosaStats", "lib", "lib_path",
    "NOSA_F32", "NOSA_BF16", "NOSA_FLAG_TIMING", "NOSA_FLAG_POOLED_BF16", "DBG",
    "nosa_config", "nosa_config_validate", "nosa_payload_bytes", "nosa_create",
    "nosa_append_kv", "nosa_decode_step", "nosa_stats", "nosa_stats_reset", "nosa_set_timing",
    "nosa_debug_read", "nosa_debug_size", "nosa_destroy", "nosa_last_error",
    "nosa_attention_workspace_bytes", "nosa_sparse_attention", "nosa_sparse_attention_noalloc",
    "nosa_selftest_bounded_wait", "nosa_frontend_rows", "nosa_decode_step_hidden",
    "nosa_frontend_packed_bytes", "nosa_frontend_pack", "nosa_prefill_workspace_bytes",
    "nosa_prefill_forward", "nosa_prefill_device_error", "nosa_prefill_timing",
    "nosa_numa_choose",
]

NOSA_F32, NOSA_BF16 = 0, 1
NOSA_FLAG_TIMING = 1
NOSA_FLAG_POOLED_BF16 = 2
STATUS = {0: "OK", 1: "INVALID_ARG", 2: "OOM", 3: "HOST_OOM", 4: "CAPACITY", 5: "CUDA",
          6: "STATE", 7: "UNSUPPORTED"}
DBG = {name: i for i, name in enumerate(
    ["SEL", "NSEL", "ELIG", "SLOTS", "LOADS", "NLOAD", "POOLED", "SE", "SQ", "SLOTPOOL",
     "HOST", "TAIL", "TRACE"])}

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "_lib", "libnosa.so")


class NosaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class NosaConfig(C.Structure):
    _fields_ = [("batch", C.c_int32), ("n_q_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("dtype", C.c_int32), ("block", C.c_int32),
                ("sub_block", C.c_int32), ("k", C.c_int32), ("k_e", C.c_int32),
                ("max_context", C.c_int32), ("device", C.c_int32), ("flags", C.c_uint32)]


class NosaStats(C.Structure):
    _fields_ = [("steps", C.c_int64), ("context", C.c_int64), ("host_loads", C.c_int64),
                ("tail_loads", C.c_int64), ("host_bytes", C.c_int64),
                ("cold_host_loads", C.c_int64), ("max_host_loads_unit", C.c_int32),
                ("min_hits", C.c_int32), ("sum_hits", C.c_int64), ("hit_samples", C.c_int64),
                ("gamma_min", C.c_double), ("gamma_mean", C.c_double),
                ("near_ties", C.c_int64), ("device_error", C.c_int32),
                ("host_numa_node", C.c_int32),
                ("t_us", C.c_double * 8), ("t_count", C.c_int64), ("launches", C.c_int64),
                ("host_store_kind", C.c_int32), ("host_store_pinned", C.c_int32)]


def _load():
    if not os.path.exists(lib_path):
        raise ImportError(f"{lib_path} is missing: the CUDA library has not been built "
                          "(run __graft_entry__.build())")
    L = C.CDLL(lib_path)
    P, I32, SZ, VP = C.POINTER, C.c_int32, C.c_size_t, C.c_void_p
    sigs = {
        "nosa_payload_bytes": (SZ, [P(NosaConfig)]),
        "nosa_config_validate": (C.c_int, [P(NosaConfig), C.c_char_p, SZ]),
        "nosa_create": (C.c_int, [P(NosaConfig), P(VP)]),
        "nosa_append_kv": (C.c_int, [VP, I32, VP, VP, VP, VP]),
        "nosa_decode_step": (C.c_int, [VP, VP, VP, VP, VP, VP, VP, VP]),
        "nosa_stats": (C.c_int, [VP, P(NosaStats)]),
        "nosa_stats_reset": (C.c_int, [VP]),
        "nosa_set_timing": (C.c_int, [VP, C.c_int32]),
        "nosa_debug_read": (C.c_int, [VP, I32, SZ, VP, SZ]),
        "nosa_debug_size": (SZ, [VP, I32]),
        "nosa_destroy": (None, [VP]),
        "nosa_last_error": (C.c_char_p, [VP]),
        "nosa_attention_workspace_bytes": (SZ, [P(NosaConfig), I32]),
        "nosa_sparse_attention": (C.c_int, [P(NosaConfig), VP, C.c_int64, VP, I32, VP, I32, VP,
                                            VP, VP, VP, SZ, VP]),
        "nosa_sparse_attention_noalloc": (C.c_int, [P(NosaConfig), VP, C.c_int64, VP, I32, VP,
                                                    I32, VP, VP, VP, VP]),
        "nosa_selftest_bounded_wait": (C.c_int, [I32, C.c_int64, P(I32), P(I32)]),
        "nosa_frontend_rows": (SZ, [P(NosaConfig)]),
        "nosa_decode_step_hidden": (C.c_int, [VP, VP, I32, VP, VP, VP, VP, VP]),
        "nosa_frontend_packed_bytes": (SZ, [P(NosaConfig), I32]),
        "nosa_frontend_pack": (C.c_int, [P(NosaConfig), I32, VP, VP, VP]),
        "nosa_prefill_workspace_bytes": (SZ, [P(NosaConfig), I32]),
        "nosa_prefill_forward": (C.c_int, [P(NosaConfig), I32, VP, VP, VP, VP, VP, VP, VP, VP,
                                           SZ, VP]),
        "nosa_prefill_device_error": (C.c_int, [P(NosaConfig), I32, VP, P(I32)]),
        "nosa_prefill_timing": (C.c_int, [P(C.c_float), P(C.c_float)]),
        "nosa_numa_choose": (I32, [I32, P(I32), I32, P(I32), I32]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _dtype_of(cfg: NosaConfig):
    torch = _torch()
    return torch.float32 if cfg.dtype == NOSA_F32 else torch.bfloat16


def _ptr(t, shape=None, dtype=None, what="tensor", align=16, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{what} is required")
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    p = t.data_ptr()
    if p % align:
        raise ValueError(f"{what} must be {align}-byte aligned")
    return p


def _stream(stream):
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, handle=None):
    if status != 0:
        raise NosaError(status, nosa_last_error(handle))


# ---------------------------------------------------------------------------
# the C ABI, one wrapper per entry point
# ---------------------------------------------------------------------------
def nosa_config(batch, n_q_heads, n_kv_heads, head_dim, dtype, k, k_e, max_context,
                block=64, sub_block=16, device=0, flags=0) -> NosaConfig:
    if isinstance(dtype, str):
        dtype = NOSA_F32 if dtype == "f32" else NOSA_BF16
    return NosaConfig(batch, n_q_heads, n_kv_heads, head_dim, dtype, block, sub_block, k, k_e,
                      max_context, device, flags)


def nosa_config_validate(cfg: NosaConfig):
    buf = C.create_string_buffer(256)
    st = lib.nosa_config_validate(C.byref(cfg), buf, 256)
    return st, buf.value.decode()


def nosa_payload_bytes(cfg: NosaConfig) -> int:
    return int(lib.nosa_payload_bytes(C.byref(cfg)))


def nosa_numa_choose(gpu_node: int, mem_nodes, allowed) -> int:
    """The host-store placement rule (see include/nosa.h): the node to bind, or -1."""
    m = (C.c_int32 * max(1, len(mem_nodes)))(*mem_nodes)
    a = (C.c_int32 * max(1, len(allowed)))(*allowed)
    return lib.nosa_numa_choose(gpu_node, m, len(mem_nodes), a, len(allowed))


def nosa_last_error(handle=None) -> str:
    r = lib.nosa_last_error(handle)
    return r.decode() if r else ""


def nosa_create(cfg: NosaConfig):
    h = C.c_void_p()
    _check(lib.nosa_create(C.byref(cfg), C.byref(h)))
    h.cfg = cfg
    return h


def nosa_append_kv(h, k, v, e, stream=None):
    cfg = h.cfg
    dt = _dtype_of(cfg)
    torch = _torch()
    n = k.shape[1] if not isinstance(k, int) else None
    if n is None:
        raise ValueError("pass tensors to nosa_append_kv")
    shp = (cfg.batch, n, cfg.n_kv_heads, cfg.head_dim)
    _check(lib.nosa_append_kv(h, n, _ptr(k, shp, dt, "k"), _ptr(v, shp, dt, "v"),
                              _ptr(e, shp[:3], torch.float32, "e", 4), _stream(stream)), h)


def nosa_decode_step(h, q, k_new, v_new, e_new, out, lse=None, stream=None):
    cfg = h.cfg
    dt = _dtype_of(cfg)
    torch = _torch()
    qs = (cfg.batch, cfg.n_q_heads, cfg.head_dim)
    ks = (cfg.batch, cfg.n_kv_heads, cfg.head_dim)
    _check(lib.nosa_decode_step(
        h, _ptr(q, qs, dt, "q"), _ptr(k_new, ks, dt, "k_new"), _ptr(v_new, ks, dt, "v_new"),
        _ptr(e_new, ks[:2], torch.float32, "e_new", 4), _ptr(out, qs, dt, "out"),
        _ptr(lse, qs[:2], torch.float32, "lse", 4, allow_none=True), _stream(stream)), h)


def nosa_frontend_rows(cfg: NosaConfig) -> int:
    """Rows of the packed front-end projection: (Hq + 2 Hkv) d + Hkv."""
    return int(lib.nosa_frontend_rows(C.byref(cfg)))


def nosa_frontend_packed_bytes(cfg: NosaConfig, hidden: int) -> int:
    return int(lib.nosa_frontend_packed_bytes(C.byref(cfg), hidden))


def nosa_frontend_pack(cfg: NosaConfig, w, stream=None):
    """Packs the front-end weights w [F][D] bf16 (row-major); returns the packed uint8 tensor."""
    torch = _torch()
    F, D = nosa_frontend_rows(cfg), w.shape[-1]
    packed = torch.empty(nosa_frontend_packed_bytes(cfg, D), dtype=torch.uint8, device=w.device)
    st = lib.nosa_frontend_pack(C.byref(cfg), D, _ptr(w, (F, D), torch.bfloat16, "w"),
                                _ptr(packed, None, torch.uint8, "w_packed"), _stream(stream))
    _check(st)
    return packed


def nosa_decode_step_hidden(h, x, w_packed, out, lse=None, q_out=None, stream=None):
    """One decode step from hidden states x [batch][D] (bf16) and packed weights."""
    cfg = h.cfg
    torch = _torch()
    if isinstance(x, int) or isinstance(w_packed, int):
        raise ValueError("pass tensors to nosa_decode_step_hidden")
    D = x.shape[-1]
    if w_packed.numel() != nosa_frontend_packed_bytes(cfg, D):
        raise ValueError("w_packed is not the packed form for this configuration and width")
    qs = (cfg.batch, cfg.n_q_heads, cfg.head_dim)
    _check(lib.nosa_decode_step_hidden(
        h, _ptr(x, (cfg.batch, D), torch.bfloat16, "x"), D,
        _ptr(w_packed, None, torch.uint8, "w_packed"),
        _ptr(q_out, qs, torch.bfloat16, "q_out", allow_none=True),
        _ptr(out, qs, torch.bfloat16, "out"),
        _ptr(lse, qs[:2], torch.float32, "lse", 4, allow_none=True), _stream(stream)), h)


def nosa_prefill_workspace_bytes(cfg: NosaConfig, seq_len: int) -> int:
    return int(lib.nosa_prefill_workspace_bytes(C.byref(cfg), seq_len))


def nosa_prefill_forward(cfg: NosaConfig, q, k, v, e, out, lse=None, sel=None, workspace=None,
                         stream=None):
    """Training-time forward over whole sequences: q [batch][L][Hq][d], k, v
    [batch][L][Hkv][d], e [batch][L][Hkv] fp32; writes out (and lse, sel if given).
    Returns the workspace (allocated here when not passed)."""
    torch = _torch()
    dt = _dtype_of(cfg)
    L = q.shape[1]
    qs = (cfg.batch, L, cfg.n_q_heads, cfg.head_dim)
    ks = (cfg.batch, L, cfg.n_kv_heads, cfg.head_dim)
    need = nosa_prefill_workspace_bytes(cfg, L)
    if need == 0:
        raise NosaError(1, nosa_last_error() or "invalid configuration or length")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.nosa_prefill_forward(
        C.byref(cfg), L, _ptr(q, qs, dt, "q"), _ptr(k, ks, dt, "k"), _ptr(v, ks, dt, "v"),
        _ptr(e, ks[:3], torch.float32, "e", 4), _ptr(out, qs, dt, "out"),
        _ptr(lse, qs[:3], torch.float32, "lse", 4, allow_none=True),
        _ptr(sel, ks[:3] + (cfg.k,), torch.int32, "sel", 4, allow_none=True),
        _ptr(workspace, None, torch.uint8, "workspace", 256), workspace.numel(), _stream(stream)))
    return workspace


def nosa_prefill_device_error(cfg: NosaConfig, seq_len: int, workspace) -> int:
    """The device error word of the last training-time forward run in workspace
    (0 none, 1 a bounded wait gave up, 2 a table entry out of range); waits for
    the device."""
    out = C.c_int32(0)
    _check(lib.nosa_prefill_device_error(C.byref(cfg), seq_len,
                                         _ptr(workspace, None, _torch().uint8, "workspace", 256),
                                         C.byref(out)))
    return out.value


def nosa_prefill_timing() -> tuple:
    """(front_ms, attention_ms) of the last training-time forward run on this
    thread with NOSA_FLAG_TIMING in its config's flags; waits for it."""
    f, a = C.c_float(0.0), C.c_float(0.0)
    _check(lib.nosa_prefill_timing(C.byref(f), C.byref(a)))
    return f.value, a.value


def nosa_stats(h) -> dict:
    s = NosaStats()
    _check(lib.nosa_stats(h, C.byref(s)), h)
    d = {f: getattr(s, f) for f, _ in NosaStats._fields_ if f not in ("t_us", "pad_")}
    d["t_us"] = list(s.t_us)
    return d


def nosa_stats_reset(h):
    _check(lib.nosa_stats_reset(h), h)


def nosa_set_timing(h, on: bool):
    """Per-phase event timing of the following decode steps on or off."""
    _check(lib.nosa_set_timing(h, 1 if on else 0), h)


def nosa_debug_size(h, what) -> int:
    return int(lib.nosa_debug_size(h, DBG[what] if isinstance(what, str) else what))


def nosa_debug_read(h, what, offset=0, nbytes=None) -> np.ndarray:
    """Synchronous read-back of a debug array (or a byte range of it) as uint8."""
    w = DBG[what] if isinstance(what, str) else what
    if nbytes is None:
        nbytes = nosa_debug_size(h, w) - offset
    out = np.empty(nbytes, dtype=np.uint8)
    _check(lib.nosa_debug_read(h, w, offset, out.ctypes.data, nbytes), h)
    return out


def nosa_destroy(h):
    if h is not None and h.value:
        lib.nosa_destroy(h)
        h.value = None


def nosa_selftest_bounded_wait(device=0, limit_ns=200_000_000):
    """(timed_out, waited_ms) of a bounded device wait that nothing completes."""
    t, m = C.c_int32(), C.c_int32()
    _check(lib.nosa_selftest_bounded_wait(device, limit_ns, C.byref(t), C.byref(m)))
    return bool(t.value), int(m.value)


def nosa_attention_workspace_bytes(cfg: NosaConfig, n_blocks: int) -> int:
    return int(lib.nosa_attention_workspace_bytes(C.byref(cfg), n_blocks))


def nosa_sparse_attention(cfg: NosaConfig, units, block_tab, tail, tail_len, q, out, lse,
                          workspace, stream=None):
    torch = _torch()
    dt = _dtype_of(cfg)
    U = cfg.batch * cfg.n_kv_heads
    n_blocks = block_tab.shape[1]
    qs = (cfg.batch, cfg.n_q_heads, cfg.head_dim)
    _check(lib.nosa_sparse_attention(
        C.byref(cfg), _ptr(units, None, torch.uint8, "units"),
        units.numel() // nosa_payload_bytes(cfg),
        _ptr(block_tab, (U, n_blocks), torch.int32, "block_tab", 4), n_blocks,
        _ptr(tail, None, torch.uint8, "tail", allow_none=True), int(tail_len),
        _ptr(q, qs, dt, "q"), _ptr(out, qs, dt, "out"),
        _ptr(lse, qs[:2], torch.float32, "lse", 4, allow_none=True),
        _ptr(workspace, None, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def nosa_sparse_attention_noalloc(cfg: NosaConfig, units, block_tab, tail, tail_len, q, out,
                                  lse, stream=None):
    """nosa_sparse_attention with the library's static device scratch instead of a
    caller workspace: nothing is allocated, for callers that cannot allocate device
    memory (see include/nosa.h). Calls that overlap on the GPU share that scratch."""
    torch = _torch()
    dt = _dtype_of(cfg)
    U = cfg.batch * cfg.n_kv_heads
    n_blocks = block_tab.shape[1]
    qs = (cfg.batch, cfg.n_q_heads, cfg.head_dim)
    _check(lib.nosa_sparse_attention_noalloc(
        C.byref(cfg), _ptr(units, None, torch.uint8, "units"),
        units.numel() // nosa_payload_bytes(cfg),
        _ptr(block_tab, (U, n_blocks), torch.int32, "block_tab", 4), n_blocks,
        _ptr(tail, None, torch.uint8, "tail", allow_none=True), int(tail_len),
        _ptr(q, qs, dt, "q"), _ptr(out, qs, dt, "out"),
        _ptr(lse, qs[:2], torch.float32, "lse", 4, allow_none=True), _stream(stream)))
