"""Lock-step parity harness: runs the CUDA path through the C ABI and the fp64
oracle on the same seeded inputs, unit by unit, step by step.

Comparison rules (the tolerances the spec states, plus the device state):
* selections, load lists, slot tables and gathered bytes: exact, except that a
  top-k cut may differ from the oracle's where the oracle's k-th and (k+1)-th
  fp32 scores differ by less than 1e-5 * max |score| over the cut's candidates;
  then the oracle adopts the GPU's choice and the event is counted (lock-step);
* attention output: <= 1e-5 absolute (fp32), <= 1e-2 * RMS of the oracle's
  output row (bf16);
* device state of every checked unit after every checked step: the sub-block
  mean keys and the block eviction scores of every candidate and of the open
  block's completed sub-blocks bit for bit against the oracle's model of their
  stored precision (``stored_means_f32``: fp32 token-order sums times 1/16;
  ``pooled_keys_bf16`` for bf16 pooled keys); the eligibility bitmask bit for
  bit; the query-aware scores of every candidate within the error bound of an
  fp32 dot product, (d + G + 8) * 2^-24 * sum_i |q_bar_i K_bar_i| / sqrt(d), of
  the scores formed in fp64 from the same stored pooled keys; and the host-store
  bytes of every block, checked once when it becomes a candidate.
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


def near_tie_equivalent(scores, cand, oracle_set, gpu_set, rel=TIE_REL, extra=0.0):
    """(accepted, was_tie): whether gpu_set may replace oracle_set at a top-k cut.

    extra widens the window by an absolute amount: the bound on how far the GPU's
    scores may sit from the oracle's when their inputs differ by a stated rounding
    (the real-valued front-end case); 0 elsewhere."""
    o, g = set(int(x) for x in oracle_set), set(int(x) for x in gpu_set)
    if o == g:
        return True, False
    cand = [int(c) for c in cand]
    if len(o) != len(g) or not g <= set(cand):
        return False, False
    s = O.decision_values(np.asarray(scores)).astype(np.float64)
    tol = rel * max(abs(s[c]) for c in cand) + extra
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
                 check_bytes=True, oracle_attention_every=1, check_state=True, state_every=1):
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
        self.check_state = check_state
        self.state_every = state_every
        self.pkb = bool(flags & nosa.NOSA_FLAG_POOLED_BF16)
        self.attn_every = oracle_attention_every
        self.ties = 0
        self.step_idx = 0
        self.expected = {"host_loads": 0, "tail_loads": 0, "cold_host_loads": 0, "sum_hits": 0,
                         "hit_samples": 0, "min_hits": 0, "max_host_loads_unit": 0,
                         "unit_steps": 0}
        self.stats_checked = False
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
        self.model = {u: {"pk": [], "se": []} for u in self.units}
        self.state_checks = 0
        if check_state:
            for u in self.units:
                uo = self.oracles[u]
                n = uo.n_cand
                for blk in range(n):
                    assert np.array_equal(self.host_bytes(u, blk), uo.block_payload(blk)), (
                        f"unit {u}: host store bytes of prompt block {blk} differ")
                self.check_unit_state(u, uo, None, "after the prompt")

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

    def pooled_stored(self, u, n):
        """Stored sub-block mean keys of blocks [0, n) of unit u, as fp64."""
        P, d = 4, self.d
        if not self.pkb:
            return self.pooled(u, n).astype(np.float64)
        raw = nosa.nosa_debug_read(self.h, "POOLED", u * self.maxblk * P * d * 2, n * P * d * 2)
        bits = np.frombuffer(raw.tobytes(), np.uint16).reshape(n, P, d)
        return synth.bf16_bits_to_f64(bits)

    def elig_words(self, u):
        return np.frombuffer(nosa.nosa_debug_read(self.h, "ELIG", u * self.W * 4, self.W * 4).tobytes(),
                             np.uint32)

    def _model(self, u, uo, upto):
        """The oracle's stored-precision pooled keys and eviction scores of unit u's
        blocks [0, upto) (complete blocks), extended as blocks complete."""
        m = self.model[u]
        B, S = self.w.block, self.w.sub_block
        for blk in range(len(m["pk"]), upto):
            k64, _, e64 = uo.tokens_f64(blk * B, (blk + 1) * B)
            m["pk"].append(O.pooled_keys_bf16(k64, S) if self.pkb else O.stored_means_f32(k64, S))
            m["se"].append(float(O.stored_means_f32(e64, S).max()))
        return m

    def check_unit_state(self, u, uo, qg, when):
        """Pooled keys, eviction scores, eligibility and (with qg) the query-aware
        scores of unit u against the oracle (rules in the module docstring)."""
        B, S, d = self.w.block, self.w.sub_block, self.d
        n = uo.n_cand
        m = self._model(u, uo, n)
        ncs = (uo.L - n * B) // S          # completed sub-blocks of the open block
        nrows = n + (1 if ncs > 0 else 0)
        if nrows:
            pk = self.pooled_stored(u, nrows)
            se = self.se(u, nrows).astype(np.float64)
            if n:
                want = np.stack(m["pk"][:n])
                bad = np.argwhere(pk[:n] != want)
                assert bad.size == 0, (f"unit {u} {when}: pooled key [blk, sub, dim] {bad[0].tolist()} "
                                       f"{pk[:n][tuple(bad[0])]} != {want[tuple(bad[0])]}")
                assert np.array_equal(se[:n], np.array(m["se"][:n])), f"unit {u} {when}: eviction scores differ"
            if ncs > 0:
                k64, _, e64 = uo.tokens_f64(n * B, n * B + ncs * S)
                pk_open = O.pooled_keys_bf16(k64, S) if self.pkb else O.stored_means_f32(k64, S)
                assert np.array_equal(pk[n, :ncs], pk_open), f"unit {u} {when}: open block's pooled keys differ"
                assert se[n] == O.stored_means_f32(e64, S).max(), f"unit {u} {when}: open block's eviction score differs"
        words = self.elig_words(u)
        bits = ((words[np.arange(self.W * 32) // 32] >> (np.arange(self.W * 32) % 32).astype(np.uint32)) & 1)
        want_bits = np.zeros(self.W * 32, dtype=np.uint32)
        want_bits[:n] = uo.elig[:n]
        bad = np.flatnonzero(bits != want_bits)
        assert bad.size == 0, f"unit {u} {when}: eligibility bit of block {bad[0]} differs"
        if qg is not None and n:
            q64 = synth.storage_to_f64(qg, self.w.dtype)
            qbar = O.group_query(q64)
            K = np.stack(m["pk"][:n])                         # [n][P][d] stored values
            ref = (K @ qbar).max(axis=1) / math.sqrt(d)
            bound = ((d + self.G + 8) * 2.0 ** -24 * (np.abs(K) @ np.abs(qbar)).max(axis=1)
                     / math.sqrt(d))
            got = self.sq(u, n).astype(np.float64)
            err = np.abs(got - ref)
            i = int(np.argmax(err - bound))
            assert np.all(err <= bound), (f"unit {u} {when}: query score of block {i} {got[i]} vs {ref[i]} "
                                          f"(bound {bound[i]:.3g})")
        self.state_checks += 1

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
            extra_e, extra_q = self.tie_extra(u, uo, qg)
            ok, tie = near_tie_equivalent(se64, eligible, g_e_o, g_e_gpu, extra=extra_e)
            assert ok, f"unit {u} step {s}: Gamma_e {sorted(g_e_gpu)} != oracle {sorted(g_e_o)}"
            self.ties += tie
            g_e = np.array(sorted(int(x) for x in g_e_gpu), dtype=np.int64)
            rest = np.setdiff1d(np.arange(n), g_e)
            g_q_o = O.top_m(sq64, rest, min(self.k - len(g_e), len(rest)))
            ok, tie = near_tie_equivalent(sq64, rest, g_q_o, g_q_gpu, extra=extra_q)
            assert ok, f"unit {u} step {s}: Gamma_q {sorted(g_q_gpu)} != oracle {sorted(g_q_o)}"
            self.ties += tie
            assert list(g_e_gpu) == sorted(g_e_gpu) and list(g_q_gpu) == sorted(g_q_gpu)
            info = uo.commit(g_e, np.array(sorted(int(x) for x in g_q_gpu), dtype=np.int64))
            self._count(s, n, len(g_e) + len(g_q_gpu), info["loads"])
            nload = int(self._i32("NLOAD", u, 1)[0])
            loads = self._i32("LOADS", u, self.k * 3).reshape(self.k, 3)[:nload]
            assert [tuple(map(int, l)) for l in loads] == [tuple(l) for l in info["loads"]], (
                f"unit {u} step {s}: loads differ")
            slots = self._i32("SLOTS", u, self.k)
            assert np.array_equal(slots, uo.slot2blk), f"unit {u} step {s}: slot table differs"
            if self.check_state:
                if s % self.state_every == 0:
                    self.check_unit_state(u, uo, qg, f"step {s}")
                if uo.just_completed >= 0:
                    jc = uo.just_completed
                    assert np.array_equal(self.host_bytes(u, jc), uo.block_payload(jc)), (
                        f"unit {u} step {s}: host store bytes of block {jc} differ")
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

    def tie_extra(self, u, uo, qg):
        """Extra near-tie window (eviction cut, query cut); the plain path feeds the
        oracle and the GPU the same stored inputs, so none."""
        return 0.0, 0.0

    def q_oracle(self, b, hh, s):
        key = (b, hh)
        if self.q_all is None:
            self.q_all = {}
        if key not in self.q_all:
            steps = self.w.steps
            self.q_all[key] = synth.queries(self.w, b, range(hh * self.G, (hh + 1) * self.G), steps)
        return self.q_all[key][s]

    def _count(self, s, n, gamma, loads):
        """The library's load statistics, rebuilt from the oracle's load lists: every
        load is a host or a tail load; the handle's first decode step counts its host
        loads as cold; any later step of a unit with at least k candidates is a hit
        sample, hits = |Gamma| - host loads."""
        e = self.expected
        n_host = sum(1 for ld in loads if ld[2] == 0)
        e["host_loads"] += n_host
        e["tail_loads"] += len(loads) - n_host
        if s == 0:
            e["cold_host_loads"] += n_host
        elif n >= self.k:
            hits = gamma - n_host
            e["min_hits"] = hits if e["hit_samples"] == 0 else min(e["min_hits"], hits)
            e["sum_hits"] += hits
            e["hit_samples"] += 1
            e["max_host_loads_unit"] = max(e["max_host_loads_unit"], n_host)
        e["unit_steps"] += 1

    def stats(self):
        """nosa_stats; when every unit was checked at every step, its load statistics
        must equal the ones rebuilt from the oracle."""
        st = nosa.nosa_stats(self.h)
        e = self.expected
        if e["unit_steps"] == self.U * self.step_idx and self.step_idx > 0:
            for key in ("host_loads", "tail_loads", "cold_host_loads", "sum_hits", "hit_samples",
                        "min_hits", "max_host_loads_unit"):
                assert st[key] == e[key], f"stats {key}: library {st[key]} != oracle {e[key]}"
            self.stats_checked = True
        return st

    def close(self):
        nosa.nosa_destroy(self.h)


def _bf16_tensor(x64):
    """bf16-exact fp64 values -> a CUDA bf16 tensor with the same values."""
    bits = synth.to_storage(x64, "bf16").view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(bits)).cuda().view(torch.bfloat16)


def _bf16_ulp(x):
    """bf16 ulp at |x| (8-bit significand)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


class FrontRun(GpuRun):
    """GpuRun whose decode steps start from hidden states (the fused front-end).

    The prompt is appended as in GpuRun; every decode step projects the
    generator's hidden states with the packed weights. The oracle projects the
    same inputs itself (fp64, then the stored forms).

    Integer inputs (default): every fp32 partial sum of the projection is exact,
    so the GPU's queries are compared bit for bit and its keys, values and
    eviction logits through every downstream check.

    Real-valued inputs (real=True): the projection's fp32 sums depend on the
    order of the additions, so the GPU's q, k, v (bf16) and e (fp32) of every
    checked unit are compared with the oracle's fp64 projection y elementwise:
    |x_gpu - y| <= (2 D + 16) 2^-24 sum_j |W_ij x_j| (fp32 accumulation, the
    tensor cores' included) + one rounding step of the stored type. Downstream,
    the oracle keeps its own rounding of y, so the device state and the bytes are
    not compared; selections use the near-tie rule with the window widened by the
    bound on the score change those roundings can cause, and the attention keeps
    its tolerance.
    """

    def __init__(self, w, units=None, D=None, real=False, **kw):
        if real:
            kw.setdefault("check_state", False)
            kw.setdefault("check_bytes", False)
        super().__init__(w, units=units, **kw)
        self.real = real
        self.D = synth.hidden_width(w) if D is None else D
        if real:
            self.W64 = synth.proj_weights_real(w, self.D)
            self.W_dev = nosa.nosa_frontend_pack(self.cfg, _bf16_tensor(self.W64))
        else:
            self.W_dev = nosa.nosa_frontend_pack(self.cfg, synth.gpu.proj_weights(w, self.D))
            self.W64 = synth.proj_weights(w, self.D)
        self.absW = np.abs(self.W64)
        self.requests = sorted({u // w.n_kv_heads for u in self.units})
        self.acc_k = {u: 0.0 for u in self.units}   # largest key perturbation bound so far
        self.acc_e = {u: 0.0 for u in self.units}   # largest eviction-logit perturbation bound
        self.proj_checked = 0

    def tie_extra(self, u, uo, qg):
        if not self.real or u not in self.dq:
            return 0.0, 0.0
        n = uo.n_cand
        d = self.d
        # scores: q_bar and (for blocks holding projected tokens) K_bar may each move
        # by their element bounds; eviction scores by the logits' bound
        K = uo.k_bar[:n]
        qbar = np.abs(O.group_query(synth.storage_to_f64(qg, self.w.dtype)))
        dq = self.dq[u]
        dk = self.acc_k[u]
        extra_q = 0.0
        if n:
            extra_q = float(((np.abs(K) @ dq).max() + (qbar.sum() + dq.sum()) * dk) / math.sqrt(d))
        return 2.0 * self.acc_e[u], 2.0 * extra_q

    def _check_projection(self, b, t, y_q, y_k, y_v, y_e, x64, q_gpu):
        """Real-valued inputs: the GPU's projected values of request b against the
        oracle's fp64 projection within the accumulation bound plus one rounding."""
        w, D, d, G = self.w, self.D, self.d, self.G
        acc = (2 * D + 16) * 2.0 ** -24 * (self.absW @ np.abs(x64[0]))   # [F]
        fq, fk = w.n_q_heads * d, w.n_kv_heads * d
        aq, ak, av, ae = acc[:fq], acc[fq:fq + fk], acc[fq + fk:fq + 2 * fk], acc[fq + 2 * fk:]
        qg = synth.bf16_bits_to_f64(q_gpu).reshape(-1)
        yq = y_q.reshape(-1)
        bad = np.abs(qg - yq) > aq + _bf16_ulp(np.maximum(np.abs(yq), np.abs(qg)))
        assert not bad.any(), f"request {b} token {t}: projected query {np.flatnonzero(bad)[0]} off"
        for hh in range(w.n_kv_heads):
            u = b * w.n_kv_heads + hh
            if u not in self.oracles:
                continue
            kg, vg, eg = self.tail_token(u, t)
            ky, vy, ey = y_k[hh], y_v[hh], y_e[hh]
            a_k, a_v = ak[hh * d:(hh + 1) * d], av[hh * d:(hh + 1) * d]
            assert np.all(np.abs(kg - ky) <= a_k + _bf16_ulp(np.maximum(np.abs(ky), np.abs(kg)))), (
                f"unit {u} token {t}: projected key off")
            assert np.all(np.abs(vg - vy) <= a_v + _bf16_ulp(np.maximum(np.abs(vy), np.abs(vg)))), (
                f"unit {u} token {t}: projected value off")
            e_bound = ae[hh] + 2.0 ** -23 * max(abs(ey), abs(eg))
            assert abs(eg - ey) <= e_bound, f"unit {u} token {t}: eviction logit {eg} vs {ey}"
            self.acc_k[u] = max(self.acc_k[u], float((a_k + _bf16_ulp(np.abs(ky)) * 2).max()))
            self.acc_e[u] = max(self.acc_e[u], e_bound)
            qrows = slice(hh * G * d, (hh + 1) * G * d)
            self.dq[u] = (aq[qrows] + 2 * _bf16_ulp(np.abs(yq[qrows]))).reshape(G, d).mean(axis=0)
            self.proj_checked += 1

    def tail_token(self, u, t):
        """The GPU's stored key, value (fp64 of the bf16 values) and eviction logit of
        token t of unit u, read from its tail buffer (block unit layout)."""
        B, d = self.w.block, self.d
        blk, pos = divmod(t, B)
        raw = np.frombuffer(nosa.nosa_debug_read(self.h, "TAIL", (u * 2 + blk % 2) * self.payload,
                                                 self.payload).tobytes(), np.uint8)
        kc = raw[:B * d * 2].view(np.uint16).reshape(d // 8, B, 8)      # 16-byte chunk-major
        k = synth.bf16_bits_to_f64(kc[:, pos, :].reshape(d))
        v = synth.bf16_bits_to_f64(raw[B * d * 2:2 * B * d * 2].view(np.uint16).reshape(B, d)[pos])
        e = float(raw[2 * B * d * 2:2 * B * d * 2 + 4 * B].view(np.float32)[pos])
        return k, v, e

    def step_hidden(self, check=True):
        w, s = self.w, self.step_idx
        t = w.prompt + s
        if self.real:
            x_np = np.concatenate([synth.hidden_real(w, b, t, 1, self.D) for b in range(w.batch)])
            x = _bf16_tensor(x_np)
        else:
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
        self.dq = {}
        for b in self.requests:
            x64 = synth.hidden_real(w, b, t, 1, self.D) if self.real else synth.hidden(w, b, t, 1, self.D)
            q, k, v, e = O.project(x64, self.W64, w.n_q_heads, w.n_kv_heads, w.head_dim)
            qs, ks, vs, es = O.frontend_storage(q, k, v, e, "bf16")
            if self.real:
                self._check_projection(b, t, q[0], k[0], v[0], e[0], x64, q_gpu[b])
            else:
                assert np.array_equal(q_gpu[b], qs[0]), f"step {s}: projected queries of request {b} differ"
            proj[b] = (qs[0], ks[0], vs[0], es[0])

        def tokens(b, hh):
            _, ks, vs, es = proj[b]
            return ks[hh], vs[hh], es[hh]

        def q_group(b, hh):
            return proj[b][0][hh * self.G:(hh + 1) * self.G]

        return out, lse, self.check_units(s, out, lse, tokens, q_group)
