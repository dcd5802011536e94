"""fp64 CPU oracle of the NOSA decode step.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module. The library never calls it
and shares no code, header, table or helper with it: it is the plain, slow
definition the CUDA path is checked against.

Source: "Technical Summary: NOSA: Native and Offloadable Sparse Attention"
(gist.science/paper/2510.13602), section Methodology, part 1 "Algorithm: NOSA"
(dual selection, locality guarantee, block-wise two-stage pooling, ED-DMA) and
part 2 "System: NOSI" (block-sized KV units, set-difference, UVA transfer).
The page states the method in prose only; where it is silent this file takes
the plainest reading and says so at the spot (readings R1..R20):

* R1  The block-level max pools sub-block *scores*: each sub-block's mean key is
      dotted with the query, then the block score is the max over its sub-blocks.
* R2  Selection is per KV head; the group of G query heads that share it is
      represented by the mean query q_bar (equal to averaging the heads' scores
      before the max).
* R3  Scores are scaled by 1/sqrt(d) like attention logits (order-neutral).
* R4  The eviction score of a block is pooled the same way as keys: mean of the
      per-token eviction logits inside each sub-block, max over sub-blocks.
* R5  Eviction eligibility is kept only by blocks in Gamma_e(t); a block that
      Gamma_e did not pick (even one Gamma_q picked) is never eligible again.
* R6  Gamma_q may pick any candidate outside Gamma_e, evicted or not.
* R7  The block holding the newest token is always attended and never a
      candidate; it becomes a candidate (and eligible) when the next token opens
      a new block.
* R9  ED-DMA: the pre-exp eviction logit is added to the scaled q.k logit before
      the softmax (natural-log domain); selection uses the pre-exp block score.
* R10 Ties: the lower block index wins.
* R11 After the prompt every candidate block is eligible and no block is
      resident; no eviction happens during the prompt.
* R12 With too few candidates, take all of them; Gamma_q fills the budget to k.
* R13 Loads are ordered by block index, free slots by slot index, paired by rank.
      A load of the block that was the tail one step earlier is sourced from the
      old tail buffer (TAIL), every other load from the host store (HOST).
* R14 Decisions that turn floating point into indices (the top-k cuts) are taken
      in fp32, the kernels' precision: the fp64 score is rounded to fp32 first.
* R21 Fused front-end: the eviction head is a linear map of the layer's hidden
      state, one pre-exp logit per KV head; its rows are packed after the query,
      key and value rows of the layer's projection, W [F][D] with
      F = (Hq + 2 Hkv) d + Hkv (query heads, key heads, value heads, eviction).
* R22 The projected q, k, v are stored in the handle's dtype (fp64 -> fp32 ->
      bf16, nearest even) and e in fp32, like the inputs of the plain step.
* R23 Training-time forward: every query position t of a sequence is a decode
      step with token t appended (causal): the dual selection with the
      candidates and eligibility of that moment, then attention over the tokens
      of Gamma(t)'s blocks plus those of t's own block up to t. Position 0 starts
      from an empty context.

Every other quantity is fp64.
"""
from __future__ import annotations

import math
import numpy as np

HOST = 0
TAIL = 1

__all__ = [
    "HOST", "TAIL", "pool_block", "group_query", "block_scores", "decision_values",
    "top_m", "dual_select", "set_difference", "attend", "encode_payload",
    "payload_bytes", "UnitOracle", "pooled_keys_bf16", "round_bf16", "stored_means_f32",
    "frontend_rows", "project", "frontend_storage", "prefill_unit",
]


# ----------------------------------------------------------------------------
# Methodology §1, Block-Wise Implementation: two-stage pooling.
# ----------------------------------------------------------------------------
def pool_block(k_blk: np.ndarray, e_blk: np.ndarray, sub_block: int):
    """First pooling stage of one complete block.

    k_blk [B][d] and e_blk [B] are fp64. Returns the sub-block mean keys
    K_bar [B/S][d], the sub-block mean eviction logits e_bar [B/S] and the block's
    eviction score se = max over sub-blocks of e_bar (R4).
    """
    B, d = k_blk.shape
    P = B // sub_block
    k_sub = k_blk.reshape(P, sub_block, d)
    e_sub = e_blk.reshape(P, sub_block)
    k_bar = k_sub.sum(axis=1) / sub_block
    e_bar = e_sub.sum(axis=1) / sub_block
    return k_bar, e_bar, float(e_bar.max())


def round_bf16(x32: np.ndarray) -> np.ndarray:
    """fp32 values rounded to nearest even in bf16, returned as fp64."""
    b = np.asarray(x32, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32).astype(np.float64)


def stored_means_f32(x_blk: np.ndarray, sub_block: int) -> np.ndarray:
    """Sub-block means in the precision the pooled state is kept in (R14).

    The values of each sub-block are summed in fp32, in token order, starting
    from 0, and the sum is multiplied by the fp32 value of 1/S. x_blk is [B][d]
    (keys) or [B] (eviction logits) of stored values, exact in fp32. Returns the
    fp32 means as fp64, [B/S][d] or [B/S]. The exact means of pool_block differ
    from these by at most the rounding of a 16-term fp32 sum.
    """
    x = np.asarray(x_blk, dtype=np.float64)
    B = x.shape[0]
    P = B // sub_block
    x32 = x.astype(np.float32).reshape((P, sub_block) + x.shape[1:])
    acc = np.zeros((P,) + x.shape[1:], dtype=np.float32)
    for j in range(sub_block):
        acc = np.add(acc, x32[:, j], dtype=np.float32)
    return np.multiply(acc, np.float32(1.0 / sub_block), dtype=np.float32).astype(np.float64)


def pooled_keys_bf16(k_blk: np.ndarray, sub_block: int) -> np.ndarray:
    """Sub-block mean keys of the bf16 pooled-key variant (R14 with bf16 storage).

    The fp32 means of stored_means_f32 (token-order fp32 sum times fl32(1/S)),
    rounded to nearest even in bf16. k_blk [B][d] holds the stored keys (exact in
    fp32). Returns [B/S][d] fp64.
    """
    return round_bf16(stored_means_f32(k_blk, sub_block))


def group_query(q_group: np.ndarray) -> np.ndarray:
    """R2: the mean of the G query heads that share one KV head, [G][d] -> [d]."""
    return q_group.sum(axis=0) / q_group.shape[0]


def block_scores(q_bar: np.ndarray, k_bar: np.ndarray) -> np.ndarray:
    """Second pooling stage and query-aware score (R1, R3).

    k_bar [N][P][d]: sq(i) = max_s (q_bar . K_bar[i, s]) / sqrt(d).
    """
    d = k_bar.shape[-1]
    if k_bar.shape[0] == 0:
        return np.zeros(0)
    return (k_bar @ q_bar).max(axis=1) / math.sqrt(d)


# ----------------------------------------------------------------------------
# Methodology §1, Dual-Selection Mechanism.
# ----------------------------------------------------------------------------
def decision_values(scores: np.ndarray) -> np.ndarray:
    """R14: the fp32 value a top-k cut compares (-0 is the same key as +0)."""
    return np.asarray(scores, dtype=np.float64).astype(np.float32) + np.float32(0.0)


def top_m(scores: np.ndarray, cand: np.ndarray, m: int) -> np.ndarray:
    """The m best candidates by score (descending), lower index first on ties (R10).

    ``scores`` is indexed by block; ``cand`` lists candidate block indices.
    Returns the chosen block indices in ascending order.
    """
    cand = np.asarray(cand, dtype=np.int64)
    m = max(0, min(int(m), len(cand)))
    if m == len(cand):
        return np.sort(cand)
    s = decision_values(np.asarray(scores)[cand]).astype(np.float64)
    order = np.lexsort((cand, -s))
    return np.sort(cand[order[:m]])


def dual_select(sq: np.ndarray, se: np.ndarray, elig: np.ndarray, n_cand: int,
                k: int, k_e: int):
    """Gamma = Gamma_e U Gamma_q over the n_cand candidate blocks.

    Gamma_e: top-k_e of the eviction scores se among eligible blocks (query-agnostic,
    strict eviction). Gamma_q: top-(k - |Gamma_e|) of the query-aware scores sq among
    the other candidates (R6, R12). The new eligibility is membership of Gamma_e (R5).
    """
    cands = np.arange(n_cand, dtype=np.int64)
    eligible = cands[np.asarray(elig[:n_cand], dtype=bool)]
    g_e = top_m(se, eligible, min(k_e, len(eligible)))
    rest = np.setdiff1d(cands, g_e, assume_unique=True)
    g_q = top_m(sq, rest, min(k - len(g_e), len(rest)))
    new_elig = np.zeros(n_cand, dtype=bool)
    new_elig[g_e] = True
    return g_e, g_q, new_elig


# ----------------------------------------------------------------------------
# Methodology §2, Optimized Memory Layout: set-difference for block swapping.
# ----------------------------------------------------------------------------
def set_difference(gamma, slot2blk: np.ndarray, just_completed: int):
    """Loads, free slots and the new slot table for the selected set ``gamma`` (R13).

    slot2blk[s] is the block held by slot s (-1: empty). Returns
    (loads [(blk, slot, src)], free_slots, new_slot2blk).
    """
    gamma = set(int(b) for b in gamma)
    resident = set(int(b) for b in slot2blk if b >= 0)
    load_blocks = sorted(gamma - resident)
    free = [s for s in range(len(slot2blk))
            if slot2blk[s] < 0 or int(slot2blk[s]) not in gamma]
    assert len(free) >= len(load_blocks)
    new = np.array(slot2blk, dtype=np.int64).copy()
    loads = []
    for blk, slot in zip(load_blocks, free):
        loads.append((blk, slot, TAIL if blk == just_completed else HOST))
        new[slot] = blk
    for slot in free[len(load_blocks):]:
        new[slot] = -1
    return loads, free, new


# ----------------------------------------------------------------------------
# Methodology §1, ED-DMA: attention with the eviction logit added before the exp.
# ----------------------------------------------------------------------------
def attend(q_group: np.ndarray, k_tok: np.ndarray, v_tok: np.ndarray, e_tok: np.ndarray):
    """Softmax attention of G query rows over n tokens with an additive eviction logit.

    l_j = q . k_j / sqrt(d) + e_j (R9); out = sum_j softmax(l)_j v_j; lse = log sum_j exp(l_j).
    """
    d = q_group.shape[1]
    logits = q_group @ k_tok.T / math.sqrt(d) + e_tok[None, :]
    m = logits.max(axis=1, keepdims=True)
    w = np.exp(logits - m)
    l = w.sum(axis=1)
    out = (w @ v_tok) / l[:, None]
    lse = m[:, 0] + np.log(l)
    return out, lse


# ----------------------------------------------------------------------------
# The block payload bytes (the library's documented block unit layout).
# ----------------------------------------------------------------------------
def payload_bytes(block: int, head_dim: int, dtype: str) -> int:
    elt = 4 if dtype == "f32" else 2
    raw = 2 * block * head_dim * elt + 4 * block
    return (raw + 255) // 256 * 256


def encode_payload(k_raw: np.ndarray, v_raw: np.ndarray, e: np.ndarray, dtype: str) -> np.ndarray:
    """Bytes of one block unit: K in 16-byte chunk-major order, V token-major, e fp32, zero pad.

    K: element (t, dim) sits at byte ((dim // c) * B + t) * 16 + (dim % c) * elt with
    c = 16 // elt; V: element (t, dim) at B*d*elt + (t*d + dim) * elt; e[t] at
    2*B*d*elt + 4*t.
    """
    B, d = k_raw.shape
    elt = 4 if dtype == "f32" else 2
    c = 16 // elt
    kc = np.ascontiguousarray(k_raw.reshape(B, d // c, c).transpose(1, 0, 2))
    out = np.zeros(payload_bytes(B, d, dtype), dtype=np.uint8)
    kb = kc.view(np.uint8).reshape(-1)
    vb = np.ascontiguousarray(v_raw).view(np.uint8).reshape(-1)
    eb = np.ascontiguousarray(e, dtype=np.float32).view(np.uint8).reshape(-1)
    out[:kb.size] = kb
    out[kb.size:kb.size + vb.size] = vb
    out[kb.size + vb.size:kb.size + vb.size + eb.size] = eb
    return out


# ----------------------------------------------------------------------------
# Methodology §1 Dual-Selection (the eviction head scores tokens independently
# of the query) and §2 Kernel Fusion (eviction head, QKV split and pooling in
# one kernel): the front-end that produces a decode step's q, k, v and e from
# the layer's hidden states (R21, R22). The pooling that follows is the unit
# state machine below, unchanged.
# ----------------------------------------------------------------------------
def frontend_rows(n_q_heads: int, n_kv_heads: int, head_dim: int) -> int:
    """Rows F of the packed projection: query, key and value heads, then eviction rows."""
    return (n_q_heads + 2 * n_kv_heads) * head_dim + n_kv_heads


def project(x: np.ndarray, W: np.ndarray, n_q_heads: int, n_kv_heads: int, head_dim: int):
    """y = W x for every request, split into the step's inputs (R21).

    x [batch][D] and W [F][D] (fp64). Returns q [batch][Hq][d], k and v
    [batch][Hkv][d], e [batch][Hkv], all fp64 and unrounded: rows [0, Hq d) are
    query head g = row // d, dim = row % d; the next Hkv d rows are the key heads,
    the next Hkv d the value heads; the last Hkv rows the eviction logits.
    """
    x = np.asarray(x, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    assert W.shape == (frontend_rows(n_q_heads, n_kv_heads, head_dim), x.shape[1])
    y = x @ W.T
    nb, d = x.shape[0], head_dim
    fq = n_q_heads * d
    fk = fq + n_kv_heads * d
    fv = fk + n_kv_heads * d
    q = y[:, :fq].reshape(nb, n_q_heads, d)
    k = y[:, fq:fk].reshape(nb, n_kv_heads, d)
    v = y[:, fk:fv].reshape(nb, n_kv_heads, d)
    e = y[:, fv:]
    return q, k, v, e


def _bf16_bits(x64: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (nearest even) -> bf16 (nearest even), as uint16 bit patterns."""
    b = np.asarray(x64, dtype=np.float64).astype(np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def frontend_storage(q, k, v, e, dtype: str):
    """Stored forms of the projected inputs (R22): q, k, v in dtype (bf16 as
    uint16 bit patterns), e in fp32."""
    if dtype == "f32":
        conv = lambda a: np.asarray(a, dtype=np.float64).astype(np.float32)
    else:
        conv = _bf16_bits
    return conv(q), conv(k), conv(v), np.asarray(e, dtype=np.float64).astype(np.float32)


# ----------------------------------------------------------------------------
# One (request, KV head) unit over time.
# ----------------------------------------------------------------------------
def _to_f64(raw: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(raw, dtype=np.float32).astype(np.float64)
    return (np.asarray(raw, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32).astype(np.float64)


class UnitOracle:
    """State of one unit: every token, pooled candidates, eligibility and the slot table.

    Tokens are kept in their stored form (fp32 or bf16 bit patterns) and widened
    to fp64 where used.
    """

    def __init__(self, head_dim: int, dtype: str, k: int, k_e: int, capacity: int,
                 block: int = 64, sub_block: int = 16, pooled: str = "f32"):
        if block % sub_block or k_e > k:
            raise ValueError("bad configuration")
        self.d, self.dtype, self.k, self.k_e = head_dim, dtype, k, k_e
        self.pooled = pooled  # "f32": exact means (R14); "bf16": the bf16 pooled-key variant
        self.B, self.S = block, sub_block
        self.P = block // sub_block
        self.cap = capacity
        raw_t = np.float32 if dtype == "f32" else np.uint16
        self.k_raw = np.zeros((capacity, head_dim), raw_t)
        self.v_raw = np.zeros((capacity, head_dim), raw_t)
        self.e = np.zeros(capacity, np.float32)
        nblk = (capacity + block - 1) // block
        self.k_bar = np.zeros((nblk, self.P, head_dim))
        self.e_bar = np.zeros((nblk, self.P))
        self.se = np.zeros(nblk)
        self.elig = np.zeros(nblk, dtype=bool)
        self.slot2blk = -np.ones(k, dtype=np.int64)
        self.L = 0
        self.steps = 0
        self.just_completed = -1
        self.n_cand_prev = 0

    # -- R7: appending a token; a block becomes a candidate when the next opens --
    @property
    def n_cand(self) -> int:
        return (self.L - 1) // self.B if self.L > 0 else 0

    def _push(self, k_raw, v_raw, e) -> int:
        if self.L >= self.cap:
            raise ValueError("context capacity exceeded")
        t = self.L
        self.k_raw[t], self.v_raw[t], self.e[t] = k_raw, v_raw, e
        self.L += 1
        opened = -1
        if t % self.B == 0 and t > 0:
            blk = t // self.B - 1
            lo, hi = blk * self.B, (blk + 1) * self.B
            k_blk = _to_f64(self.k_raw[lo:hi], self.dtype)
            kb, eb, sb = pool_block(k_blk, self.e[lo:hi].astype(np.float64), self.S)
            if self.pooled == "bf16":
                kb = pooled_keys_bf16(k_blk, self.S)
            self.k_bar[blk], self.e_bar[blk], self.se[blk] = kb, eb, sb
            self.elig[blk] = True
            opened = blk
        return opened

    def append(self, k_raw: np.ndarray, v_raw: np.ndarray, e: np.ndarray) -> None:
        """Prompt append of n tokens: no selection, no eviction (R11)."""
        for i in range(len(e)):
            self._push(k_raw[i], v_raw[i], e[i])
        self.just_completed = -1

    def tokens_f64(self, lo: int, hi: int):
        return (_to_f64(self.k_raw[lo:hi], self.dtype), _to_f64(self.v_raw[lo:hi], self.dtype),
                self.e[lo:hi].astype(np.float64))

    # -- one decode step, in phases so a harness can compare each one --
    def begin_step(self, k_raw, v_raw, e) -> None:
        """Append the step's token; remember the block that just became a candidate."""
        self.just_completed = self._push(k_raw, v_raw, e)

    def scores(self, q_group_raw: np.ndarray):
        """Query-aware and eviction scores of the current candidates, fp64."""
        q = _to_f64(q_group_raw, self.dtype)
        n = self.n_cand
        sq = block_scores(group_query(q), self.k_bar[:n])
        return sq, self.se[:n].copy()

    def select(self, sq: np.ndarray, se: np.ndarray):
        return dual_select(sq, se, self.elig, self.n_cand, self.k, self.k_e)

    def commit(self, g_e: np.ndarray, g_q: np.ndarray) -> dict:
        """Apply a selection: eligibility update (R5), set-difference (R13), locality."""
        n = self.n_cand
        new_elig = np.zeros(n, dtype=bool)
        new_elig[np.asarray(g_e, dtype=np.int64)] = True
        self.elig[:n] = new_elig
        gamma = sorted(set(int(x) for x in g_e) | set(int(x) for x in g_q))
        resident_prev = set(int(b) for b in self.slot2blk if b >= 0)
        if self.just_completed >= 0:
            resident_prev.add(self.just_completed)
        loads, free, new = set_difference(gamma, self.slot2blk, self.just_completed)
        self.slot2blk = new
        self.steps += 1
        hits = len(set(gamma) & resident_prev)
        return {"loads": loads, "free": free, "gamma": gamma, "hits": hits,
                "n_host": sum(1 for l in loads if l[2] == HOST),
                "gamma_locality": hits / self.k}

    def attention(self, q_group_raw: np.ndarray):
        """Attention over the resident selected blocks plus the tail tokens (R7, R9)."""
        q = _to_f64(q_group_raw, self.dtype)
        parts = [np.arange(b * self.B, (b + 1) * self.B) for b in sorted(self.slot2blk) if b >= 0]
        parts.append(np.arange(self.n_cand * self.B, self.L))
        idx = np.concatenate(parts)
        k, v, e = (_to_f64(self.k_raw[idx], self.dtype), _to_f64(self.v_raw[idx], self.dtype),
                   self.e[idx].astype(np.float64))
        return attend(q, k, v, e)

    def decode_step(self, q_group_raw, k_raw, v_raw, e) -> dict:
        """A whole step with the oracle's own selection."""
        self.begin_step(k_raw, v_raw, e)
        sq, se = self.scores(q_group_raw)
        g_e, g_q, _ = self.select(sq, se)
        info = self.commit(g_e, g_q)
        out, lse = self.attention(q_group_raw)
        info.update({"g_e": g_e, "g_q": g_q, "sq": sq, "se": se, "out": out, "lse": lse})
        return info

    def block_payload(self, blk: int) -> np.ndarray:
        lo, hi = blk * self.B, (blk + 1) * self.B
        return encode_payload(self.k_raw[lo:hi], self.v_raw[lo:hi], self.e[lo:hi], self.dtype)


# ----------------------------------------------------------------------------
# Methodology §1: the locality constraint is imposed during training, so the
# training-time forward applies the same dual selection causally at every query
# position (R23).
# ----------------------------------------------------------------------------
def prefill_unit(k_raw: np.ndarray, v_raw: np.ndarray, e: np.ndarray, q_raw: np.ndarray,
                 dtype: str, k: int, k_e: int, block: int = 64, sub_block: int = 16,
                 positions=None, choose=None) -> dict:
    """Training-time forward of one (request, KV head) unit over a sequence (R23).

    k_raw, v_raw [L][d] and e [L] are the stored tokens, q_raw [L][G][d] the
    stored queries. Positions are taken in order: token t is appended (R7), the
    dual selection (R5, R6, R10, R12) runs on the candidates and eligibility of
    that moment, eligibility becomes Gamma_e(t), and the attention (R9) covers the
    blocks of Gamma(t) plus t's own block up to t. Returns {t: (g_e, g_q, out, lse)}
    with out [G][d] and lse [G] for the positions in `positions` (every position by
    default; the others carry None). choose(t, sq, se, elig, g_e, g_q) may return
    a replacement (g_e, g_q): a harness adopting an equivalent choice at a near tie.
    """
    L, d = np.asarray(k_raw).shape
    uo = UnitOracle(d, dtype, k, k_e, L, block, sub_block)
    res = {}
    for t in range(L):
        if t == 0:
            uo.append(k_raw[:1], v_raw[:1], e[:1])
        else:
            uo.begin_step(k_raw[t], v_raw[t], e[t])
        sq, se = uo.scores(q_raw[t])
        g_e, g_q, _ = uo.select(sq, se)
        if choose is not None:
            alt = choose(t, sq, se, uo.elig[:uo.n_cand].copy(), g_e, g_q)
            if alt is not None:
                g_e, g_q = alt
        uo.commit(g_e, g_q)
        if positions is None or t in positions:
            out, lse = uo.attention(q_raw[t])
            res[t] = (np.asarray(g_e), np.asarray(g_q), out, lse)
        else:
            res[t] = (np.asarray(g_e), np.asarray(g_q), None, None)
    return res
