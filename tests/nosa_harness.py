"""Lock-step parity harness: runs the CUDA path through the C ABI and the fp64
oracle on the same seeded inputs, unit by unit, step by step.

Comparison rules (the tolerances the spec states):
* selections, load lists, slot tables and gathered bytes: exact, except that a
  top-k cut may differ from the oracle's where the oracle's k-th and (k+1)-th
  fp32 scores differ by less than 1e-5 * max |score| over the cut's candidates;
  then the oracle adopts the GPU's choice and the event is counted (lock-step);
* attention output: <= 1e-5 absolute (fp32), <= 1e-2 * RMS of the oracle's
  output row (bf16).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import synth
import synth.gpu
import trainable_sparse_attention_decode_gb300 as nosa
from oracle import nosa_oracle as O

TIE_REL = 1e-5


def near_tie_equivalent(scores, cand, oracle_set, gpu_set, rel=TIE_REL):
    """(accepted, was_tie): whether gpu_set may replace oracle_set at a top-k cut."""
    o, g = set(int(x) for x in oracle_set), set(int(x) for x in gpu_set)
    if o == g:
        return True, False
    cand = [int(c) for c in cand]
    if len(o) != len(g) or not g <= set(cand):
        return False, False
    s = O.decision_values(np.asarray(scores)).astype(np.float64)
    tol = rel * max(abs(s[c]) for c in cand)
    kth = min(s[i] for i in o)
    rest = [s[c] for c in cand if c not in o]
    if not rest:
        return False, False
    nxt = max(rest)
    if kth - nxt >= tol:
        return False, False
    return all(nxt - tol <= s[i] <= kth + tol for i in (o ^ g)), True


def bf16_half_ulp(x):
    """Half a bf16 ulp at |x|: the largest error of storing x in bf16 (8-bit significand)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 8)


def attn_close(out, ref, dtype):
    """Per-row check; returns the worst ratio of error to tolerance (<= 1 passes).

    fp32: max |o - o*| <= 1e-5. bf16: the 1e-2 x RMS(o*) bound is read as a
    relative RMS error, RMS(o - o*) <= 1e-2 RMS(o*), and elementwise
    |o - o*| <= 1e-2 RMS(o*) + half a bf16 ulp of o* (the rounding of the stored
    bf16 output alone exceeds 1e-2 RMS for elements above ~2.5 RMS).
    """
    worst = 0.0
    for g in range(ref.shape[0]):
        diff = np.abs(out[g] - ref[g])
        if dtype == "f32":
            worst = max(worst, float(np.max(diff)) / 1e-5)
            continue
        rms = float(np.sqrt(np.mean(ref[g] ** 2)))
        worst = max(worst, float(np.sqrt(np.mean(diff ** 2))) / (1e-2 * rms),
                    float(np.max(diff / (1e-2 * rms + bf16_half_ulp(ref[g])))))
    return worst


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class GpuRun:
    """One handle on cuda:0 fed by the device generator, plus oracle twins of sampled units."""

    def __init__(self, w: synth.Workload, units=None, flags=0, prompt_pieces=None,
                 check_bytes=True, oracle_attention_every=1):
        self.w = w
        self.cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype,
                                    w.k, w.k_e, w.max_context, flags=flags)
        self.h = nosa.nosa_create(self.cfg)
        self.U, self.k, self.G, self.d = w.units, w.k, w.group, w.head_dim
        self.maxblk = (w.max_context + w.block - 1) // w.block
        self.W = (self.maxblk + 31) // 32
        self.payload = nosa.nosa_payload_bytes(self.cfg)
        self.units = list(range(self.U)) if units is None else list(units)
        self.check_bytes = check_bytes
        self.attn_every = oracle_attention_every
        self.ties = 0
        self.step_idx = 0
        self.dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        pieces = prompt_pieces or self._default_pieces(w.prompt)
        assert sum(pieces) == w.prompt
        t = 0
        for n in pieces:
            k, v, e = synth.gpu.kv(w, t, n)
            nosa.nosa_append_kv(self.h, k, v, e)
            t += n
        torch.cuda.synchronize()
        self.oracles = {}
        for u in self.units:
            b, hh = divmod(u, w.n_kv_heads)
            uo = O.UnitOracle(w.head_dim, w.dtype, w.k, w.k_e, w.max_context, w.block, w.sub_block,
                              pooled="bf16" if flags & nosa.NOSA_FLAG_POOLED_BF16 else "f32")
            uo.append(synth.keys(w, b, hh, 0, w.prompt), synth.values(w, b, hh, 0, w.prompt),
                      synth.evict(w, b, hh, 0, w.prompt))
            self.oracles[u] = uo
        self.q_all = None

    @staticmethod
    def _default_pieces(n, chunk=8192):
        out = []
        while n > 0:
            out.append(min(chunk, n))
            n -= out[-1]
        return out

    # ---- debug readers ----
    def _i32(self, what, u, count):
        return np.frombuffer(nosa.nosa_debug_read(self.h, what, u * count * 4, count * 4).tobytes(),
                             np.int32)

    def _f32(self, what, offset_elems, count):
        return np.frombuffer(nosa.nosa_debug_read(self.h, what, offset_elems * 4, count * 4).tobytes(),
                             np.float32)

    def pooled(self, u, n):
        P, d = 4, self.d
        return self._f32("POOLED", u * self.maxblk * P * d, n * P * d).reshape(n, P, d)

    def se(self, u, n):
        return self._f32("SE", u * self.maxblk, n)

    def sq(self, u, n):
        return self._f32("SQ", u * self.maxblk, n)

    def slot_bytes(self, u, slot):
        return nosa.nosa_debug_read(self.h, "SLOTPOOL", (u * self.k + slot) * self.payload, self.payload)

    def host_bytes(self, u, blk):
        return nosa.nosa_debug_read(self.h, "HOST", (u * self.maxblk + blk) * self.payload, self.payload)

    # ---- one step ----
    def step(self, q_step, check=True):
        """Runs one decode step on the GPU and, if check, compares every sampled unit."""
        w, s = self.w, self.step_idx
        k, v, e = synth.gpu.kv(w, w.prompt + s, 1, step_major=True)
        out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=self.dt, device="cuda")
        lse = torch.empty((w.batch, w.n_q_heads), dtype=torch.float32, device="cuda")
        nosa.nosa_decode_step(self.h, q_step, k[0], v[0], e[0], out, lse)
        torch.cuda.synchronize()
        self.step_idx += 1
        if not check:
            return out, lse, {}
        t = w.prompt + s

        def tokens(b, hh):
            return (synth.keys(w, b, hh, t, 1)[0], synth.values(w, b, hh, t, 1)[0],
                    synth.evict(w, b, hh, t, 1)[0])

        return out, lse, self.check_units(s, out, lse, tokens, lambda b, hh: self.q_oracle(b, hh, s))

    def check_units(self, s, out, lse, tokens, q_group):
        """Advances every sampled unit's oracle by one step and compares it with the GPU.

        tokens(b, hh) -> the step's stored (k, v, e) of unit (b, hh);
        q_group(b, hh) -> the stored queries of its G query heads.
        """
        w = self.w
        res = {"worst_attn": 0.0, "worst_lse": 0.0}
        do_attn = (s % self.attn_every == 0)
        out_np, lse_np = (to_f64(out), lse.cpu().numpy().astype(np.float64)) if do_attn else (None, None)
        nsel_all = np.frombuffer(nosa.nosa_debug_read(self.h, "NSEL").tobytes(), np.int32).reshape(-1, 2)
        for u in self.units:
            b, hh = divmod(u, w.n_kv_heads)
            uo = self.oracles[u]
            uo.begin_step(*tokens(b, hh))
            qg = q_group(b, hh)
            sq64, se64 = uo.scores(qg)
            n = uo.n_cand
            ne, nq = nsel_all[u]
            sel = self._i32("SEL", u, self.k)
            g_e_gpu, g_q_gpu = sel[:ne], sel[ne:ne + nq]
            g_e_o, g_q_o, _ = uo.select(sq64, se64)
            eligible = [i for i in range(n) if uo.elig[i]]
            ok, tie = near_tie_equivalent(se64, eligible, g_e_o, g_e_gpu)
            assert ok, f"unit {u} step {s}: Gamma_e {sorted(g_e_gpu)} != oracle {sorted(g_e_o)}"
            self.ties += tie
            g_e = np.array(sorted(int(x) for x in g_e_gpu), dtype=np.int64)
            rest = np.setdiff1d(np.arange(n), g_e)
            g_q_o = O.top_m(sq64, rest, min(self.k - len(g_e), len(rest)))
            ok, tie = near_tie_equivalent(sq64, rest, g_q_o, g_q_gpu)
            assert ok, f"unit {u} step {s}: Gamma_q {sorted(g_q_gpu)} != oracle {sorted(g_q_o)}"
            self.ties += tie
            assert list(g_e_gpu) == sorted(g_e_gpu) and list(g_q_gpu) == sorted(g_q_gpu)
            info = uo.commit(g_e, np.array(sorted(int(x) for x in g_q_gpu), dtype=np.int64))
            nload = int(self._i32("NLOAD", u, 1)[0])
            loads = self._i32("LOADS", u, self.k * 3).reshape(self.k, 3)[:nload]
            assert [tuple(map(int, l)) for l in loads] == [tuple(l) for l in info["loads"]], (
                f"unit {u} step {s}: loads differ")
            slots = self._i32("SLOTS", u, self.k)
            assert np.array_equal(slots, uo.slot2blk), f"unit {u} step {s}: slot table differs"
            if self.check_bytes:
                for blk, slot, _src in info["loads"]:
                    assert np.array_equal(self.slot_bytes(u, slot), uo.block_payload(blk)), (
                        f"unit {u} step {s}: slot {slot} bytes differ from block {blk}")
            if do_attn:
                o_ref, lse_ref = uo.attention(qg)
                rows = slice(hh * self.G, (hh + 1) * self.G)
                res["worst_attn"] = max(res["worst_attn"], attn_close(out_np[b, rows], o_ref, w.dtype))
                res["worst_lse"] = max(res["worst_lse"], float(np.max(np.abs(lse_np[b, rows] - lse_ref))))
        return res

    def q_oracle(self, b, hh, s):
        key = (b, hh)
        if self.q_all is None:
            self.q_all = {}
        if key not in self.q_all:
            steps = self.w.steps
            self.q_all[key] = synth.queries(self.w, b, range(hh * self.G, (hh + 1) * self.G), steps)
        return self.q_all[key][s]

    def stats(self):
        return nosa.nosa_stats(self.h)

    def close(self):
        nosa.nosa_destroy(self.h)


class FrontRun(GpuRun):
    """GpuRun whose decode steps start from hidden states (the fused front-end).

    The prompt is appended as in GpuRun; every decode step projects the
    generator's hidden states with the packed weights. The oracle projects the
    same inputs itself (fp64, then the stored forms) and the GPU's queries are
    compared bit for bit with it before the unit checks.
    """

    def __init__(self, w, units=None, D=None, **kw):
        super().__init__(w, units=units, **kw)
        self.D = synth.hidden_width(w) if D is None else D
        self.W_dev = nosa.nosa_frontend_pack(self.cfg, synth.gpu.proj_weights(w, self.D))
        self.W64 = synth.proj_weights(w, self.D)
        self.requests = sorted({u // w.n_kv_heads for u in self.units})

    def step_hidden(self, check=True):
        w, s = self.w, self.step_idx
        t = w.prompt + s
        x = synth.gpu.hidden(w, t, 1, self.D)[0]
        out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.batch, w.n_q_heads), dtype=torch.float32, device="cuda")
        q_out = torch.empty_like(out)
        nosa.nosa_decode_step_hidden(self.h, x, self.W_dev, out, lse, q_out=q_out)
        torch.cuda.synchronize()
        self.step_idx += 1
        if not check:
            return out, lse, {}
        proj = {}
        q_gpu = q_out.view(torch.int16).cpu().numpy().view(np.uint16)
        for b in self.requests:
            x64 = synth.hidden(w, b, t, 1, self.D)
            q, k, v, e = O.project(x64, self.W64, w.n_q_heads, w.n_kv_heads, w.head_dim)
            qs, ks, vs, es = O.frontend_storage(q, k, v, e, "bf16")
            assert np.array_equal(q_gpu[b], qs[0]), f"step {s}: projected queries of request {b} differ"
            proj[b] = (qs[0], ks[0], vs[0], es[0])

        def tokens(b, hh):
            _, ks, vs, es = proj[b]
            return ks[hh], vs[hh], es[hh]

        def q_group(b, hh):
            return proj[b][0][hh * self.G:(hh + 1) * self.G]

        return out, lse, self.check_units(s, out, lse, tokens, q_group)
