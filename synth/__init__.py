"""Seeded synthetic inputs for the NOSA decode path.

This module is data plumbing shared by the fp64 oracle (tests) and the GPU side
(tests, bench). It holds none of the method's arithmetic: it only defines how the
keys, values, eviction logits and queries of the five workloads are drawn.

Definition (the CUDA generator in ``synth/gen.cu`` implements the same one and is
checked against this file bit for bit):

* ``splitmix64`` is the published 64-bit finaliser of Steele, Lea and Flood
  (golden-gamma increment, then two xor-shift-multiply rounds).
* A draw is addressed by a counter with fields
  ``stream:3 | a:10 | h:7 | t:26 | i:18`` (high to low bits); ``a`` is the request,
  ``h`` the head, ``t`` the token (or block, or decode step) and ``i = 4*dim + j``.
  The word for ``j`` is ``splitmix64(counter ^ splitmix64(seed))``.
* A standard-normal stand-in is the centred Irwin-Hall sum of twelve 16-bit
  uniforms (the four 16-bit lanes of the words ``j = 0, 1, 2``):
  ``(sum - 393210) / 65536``. Mean 0, variance 1 - 2**-32, support (-6, 6).
  Every value is a multiple of 2**-16 below 2**3, so it is exact in fp32 and
  fp64 on any machine; no transcendental function is involved.
* The request field is the request's index in the job: a workload's request b is
  ``request_base + b`` (ranks of a multi-GPU job run disjoint requests).
* Keys: ``k = c[b, h, block(t)] + 0.5 * n[b, h, t]``, one centre ``c`` per
  (request, KV head, 64-token block) and i.i.d. noise ``n``; exact in fp32.
* Values ``v ~ N(0, 1)``; eviction logits ``e ~ N(0, 1)`` (fp32, fixed at write).
* Queries: AR(1) per (request, query head, dim), started in its stationary
  distribution: ``q_0 = a * eps_0`` with ``a = 1 / sqrt(1 - rho**2)`` (fp64; the
  process then has the same variance and lag-1 correlation rho at every step),
  ``q_s = rho * q_{s-1} + eps_s`` in fp64 (a product, then a sum: no fused
  multiply-add), stored as fp64 -> fp32 (RNE) -> dtype. ``q_stationary=False``
  starts from ``q_0 = eps_0`` instead (variance 1 growing to ``a**2`` over the
  first steps).
* bf16 storage rounds fp32 to nearest even.
* Real-valued front-end inputs (``hidden_real``, ``proj_weights_real``):
  normals of the hidden-state and weight streams with head field 1 (the integer
  inputs use 0), the weights scaled by ``2**-6``, both rounded to bf16; their
  projections are not exact in fp32, so the order of the additions shows.
* Front-end inputs (hidden states and the packed projection weights): small
  integers ``(word % 17) - 8`` from word ``j = 0`` of the counter, scaled by
  ``2**-3`` (hidden states, counter ``(5, b, 0, t, 4*i)``) and ``2**-8`` (weights,
  counter ``(6, 0, 0, row, 4*col)``). Every product is an integer multiple of
  ``2**-11`` below ``2**-5`` in magnitude, so every partial sum of a projection
  with fewer than ``2**18`` terms is exact in fp32, whatever the order of the
  additions: the projected values are then the same bits on any correct path.

The GPU kernels never see this module's code; they get the arrays it (or its
CUDA twin) writes.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
import math
import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "splitmix64", "normals", "keys", "values", "evict",
    "queries", "to_storage", "storage_to_f64", "bf16_bits_to_f64",
    "STREAM_CENTER", "STREAM_KNOISE", "STREAM_VALUE", "STREAM_EVICT", "STREAM_QINNOV",
    "STREAM_HIDDEN", "STREAM_WEIGHT", "small_ints", "hidden", "proj_weights", "hidden_width",
    "hidden_real", "proj_weights_real", "MAX_REQUESTS",
]

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

STREAM_CENTER = 0
STREAM_KNOISE = 1
STREAM_VALUE = 2
STREAM_EVICT = 3
STREAM_QINNOV = 4
STREAM_HIDDEN = 5
STREAM_WEIGHT = 6
HIDDEN_SCALE = 2.0 ** -3
WEIGHT_SCALE = 2.0 ** -8

IH_MEAN = 393210          # 12 * 65535 / 2
IH_SCALE = 1.0 / 65536.0  # exact power of two


@dataclass(frozen=True)
class Workload:
    """Shape of one synthetic decode workload (one layer)."""
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str            # "f32" or "bf16"
    prompt: int           # tokens appended before the first decode step
    steps: int            # decode steps, one token appended per step
    k: int
    k_e: int
    rho: float = 0.95
    block: int = 64
    sub_block: int = 16
    seed: int = 0
    request_base: int = 0  # index of request 0 in the job (ranks of a multi-GPU job shard requests)
    q_stationary: bool = True  # AR(1) queries start in their stationary distribution

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def units(self) -> int:
        return self.batch * self.n_kv_heads

    @property
    def max_context(self) -> int:
        return self.prompt + self.steps

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads: one tiny fp32 case and four bf16 cases shaped like the
# 1B / 3B / 8B models of the NOSA paper's decode experiments.
WORKLOADS = {
    "tiny-f32": Workload("tiny-f32", 1, 4, 1, 64, "f32", 2048, 32, 8, 6),
    "1b-bf16": Workload("1b-bf16", 8, 16, 8, 64, "bf16", 16384, 128, 64, 48),
    "3b-bf16": Workload("3b-bf16", 16, 24, 8, 128, "bf16", 32768, 256, 64, 48),
    "8b-longgen-bf16": Workload("8b-longgen-bf16", 16, 32, 8, 128, "bf16", 8192, 16384,
                                128, 96, rho=0.9),
    "8b-offload-bf16": Workload("8b-offload-bf16", 32, 32, 8, 128, "bf16", 65536, 64, 64, 48),
}


def splitmix64(x):
    """splitmix64 finaliser on a uint64 array (wrapping arithmetic)."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
    return z ^ (z >> np.uint64(31))


def _counter(stream, a, h, t, i):
    u = np.uint64
    a = np.asarray(a, dtype=np.uint64)
    h = np.asarray(h, dtype=np.uint64)
    t = np.asarray(t, dtype=np.uint64)
    i = np.asarray(i, dtype=np.uint64)
    return ((u(stream) << u(61)) | (a << u(51)) | (h << u(44)) | (t << u(18)) | i)


def normals(seed: int, stream: int, a, h, t, dim) -> np.ndarray:
    """Exact Irwin-Hall(12) normal stand-ins, broadcast over a, h, t, dim (fp64)."""
    smix = splitmix64(np.uint64(seed))
    dim4 = np.asarray(dim, dtype=np.uint64) * np.uint64(4)
    acc = None
    for j in range(3):
        w = splitmix64(_counter(stream, a, h, t, dim4 + np.uint64(j)) ^ smix)
        s = ((w & np.uint64(0xFFFF)) + ((w >> np.uint64(16)) & np.uint64(0xFFFF))
             + ((w >> np.uint64(32)) & np.uint64(0xFFFF)) + (w >> np.uint64(48)))
        acc = s if acc is None else acc + s
    return (acc.astype(np.int64) - IH_MEAN).astype(np.float64) * IH_SCALE


def _f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    b = x32.astype(np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def to_storage(x64: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 -> fp32 (RNE) -> storage dtype; bf16 is returned as uint16 bit patterns."""
    x32 = np.asarray(x64, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return x32
    if dtype == "bf16":
        return _f32_to_bf16_bits(x32)
    raise ValueError(dtype)


def storage_to_f64(s: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(s, dtype=np.float32).astype(np.float64)
    return bf16_bits_to_f64(np.asarray(s, dtype=np.uint16))


MAX_REQUESTS = 1 << 10  # the counter's request field


def _req(w: Workload, b) -> int:
    """Request index in the job of the workload's request b (the counter field)."""
    a = w.request_base + int(b)
    if not 0 <= a < MAX_REQUESTS:
        raise ValueError(f"request {a} outside the generator's {MAX_REQUESTS} requests")
    return a


def keys(w: Workload, b: int, h: int, t0: int, n: int) -> np.ndarray:
    """Stored keys of tokens [t0, t0+n) of (request b, KV head h): [n][d] storage dtype."""
    t = np.arange(t0, t0 + n, dtype=np.int64)[:, None]
    dim = np.arange(w.head_dim, dtype=np.int64)[None, :]
    b = _req(w, b)
    c = normals(w.seed, STREAM_CENTER, b, h, t // w.block, dim)
    noise = normals(w.seed, STREAM_KNOISE, b, h, t, dim)
    return to_storage(c + 0.5 * noise, w.dtype)


def values(w: Workload, b: int, h: int, t0: int, n: int) -> np.ndarray:
    t = np.arange(t0, t0 + n, dtype=np.int64)[:, None]
    dim = np.arange(w.head_dim, dtype=np.int64)[None, :]
    return to_storage(normals(w.seed, STREAM_VALUE, _req(w, b), h, t, dim), w.dtype)


def evict(w: Workload, b: int, h: int, t0: int, n: int) -> np.ndarray:
    """Per-token eviction logits of (b, KV head h): [n] fp32."""
    t = np.arange(t0, t0 + n, dtype=np.int64)
    return normals(w.seed, STREAM_EVICT, _req(w, b), h, t, 0).astype(np.float32)


def q_start_scale(w: Workload) -> float:
    """Factor a on the first innovation of the AR(1) queries: 1 / sqrt(1 - rho^2)
    (stationary start, fp64), or 1."""
    return 1.0 / math.sqrt(1.0 - w.rho * w.rho) if w.q_stationary else 1.0


def queries(w: Workload, b: int, heads, steps: int) -> np.ndarray:
    """AR(1) queries of request b for the given query heads: [steps][len(heads)][d] storage."""
    heads = np.asarray(list(heads), dtype=np.int64)
    dim = np.arange(w.head_dim, dtype=np.int64)[None, :]
    out = np.empty((steps, len(heads), w.head_dim),
                   dtype=np.float32 if w.dtype == "f32" else np.uint16)
    q = None
    a = _req(w, b)
    for s in range(steps):
        eps = normals(w.seed, STREAM_QINNOV, a, heads[:, None], s, dim)
        if q is None:
            q = np.float64(q_start_scale(w)) * eps
        else:
            q = np.float64(w.rho) * q
            q = q + eps
        out[s] = to_storage(q, w.dtype)
    return out


def small_ints(seed: int, stream: int, a, h, t, col) -> np.ndarray:
    """Integers in [-8, 8]: (word % 17) - 8 of word j = 0 of the counter (int64)."""
    smix = splitmix64(np.uint64(seed))
    c = _counter(stream, a, h, t, np.asarray(col, dtype=np.uint64) * np.uint64(4))
    w = splitmix64(c ^ smix)
    return (w % np.uint64(17)).astype(np.int64) - 8


def hidden_width(w: Workload) -> int:
    """Width D of the hidden states fed to the front-end: n_q_heads * head_dim."""
    return w.n_q_heads * w.head_dim


def hidden(w: Workload, b: int, t0: int, n: int, D: int | None = None) -> np.ndarray:
    """Hidden states of request b for tokens [t0, t0+n): [n][D] fp64 (exact in bf16)."""
    D = hidden_width(w) if D is None else D
    t = np.arange(t0, t0 + n, dtype=np.int64)[:, None]
    col = np.arange(D, dtype=np.int64)[None, :]
    return small_ints(w.seed, STREAM_HIDDEN, _req(w, b), 0, t, col).astype(np.float64) * HIDDEN_SCALE


def proj_weights(w: Workload, D: int | None = None, rows=None) -> np.ndarray:
    """Packed front-end weights [F][D] fp64 (exact in bf16), or the given rows of it.

    F = (n_q_heads + 2 n_kv_heads) head_dim + n_kv_heads: query heads, key heads,
    value heads, then one eviction-head row per KV head.
    """
    D = hidden_width(w) if D is None else D
    F = (w.n_q_heads + 2 * w.n_kv_heads) * w.head_dim + w.n_kv_heads
    r = np.arange(F, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    col = np.arange(D, dtype=np.int64)[None, :]
    return small_ints(w.seed, STREAM_WEIGHT, 0, 0, r[:, None], col).astype(np.float64) * WEIGHT_SCALE


def hidden_real(w: Workload, b: int, t0: int, n: int, D: int | None = None) -> np.ndarray:
    """Real-valued hidden states of request b, tokens [t0, t0+n): [n][D] fp64, bf16-exact."""
    D = hidden_width(w) if D is None else D
    t = np.arange(t0, t0 + n, dtype=np.int64)[:, None]
    col = np.arange(D, dtype=np.int64)[None, :]
    return bf16_bits_to_f64(to_storage(normals(w.seed, STREAM_HIDDEN, _req(w, b), 1, t, col), "bf16"))


def proj_weights_real(w: Workload, D: int | None = None) -> np.ndarray:
    """Real-valued packed front-end weights [F][D] fp64, bf16-exact (normals x 2**-6)."""
    D = hidden_width(w) if D is None else D
    F = (w.n_q_heads + 2 * w.n_kv_heads) * w.head_dim + w.n_kv_heads
    r = np.arange(F, dtype=np.int64)[:, None]
    col = np.arange(D, dtype=np.int64)[None, :]
    x = normals(w.seed, STREAM_WEIGHT, 0, 1, r, col) * 2.0 ** -6
    return bf16_bits_to_f64(to_storage(x, "bf16"))
