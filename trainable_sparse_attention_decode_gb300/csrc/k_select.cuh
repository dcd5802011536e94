// Dual selection and set-difference (device code shared by the selection
// kernel and the fused scoring + selection kernel).
//
// NOSA technical summary, Methodology §1 "Dual-Selection Mechanism": the k
// selected blocks of a unit are Gamma = Gamma_e U Gamma_q.
//   Gamma_e : the k_e eligible blocks with the highest eviction score se
//             (query-agnostic). Eligibility is strict: a candidate left out of
//             Gamma_e at step t is never eligible again; new candidates enter
//             eligible.
//   Gamma_q : the k - |Gamma_e| other candidates with the highest query-aware
//             score sq.
// Ties go to the lower block index. The cut is exact: a radix select over the
// order-preserving 32-bit image of the fp32 score finds the threshold key and
// how many keys equal to it are taken, then those are the lowest-indexed ones.
//
// Methodology §2 "Optimized Memory Layout": the set-difference of Gamma against
// the blocks held by the unit's k slots gives the load list (missing blocks,
// ascending) and the free slots (slots whose block left Gamma, ascending), paired
// by rank. A load of the block that was the tail one step earlier is sourced
// from the old tail buffer, every other from the host store.
#pragma once

#include "nosa_internal.cuh"

namespace nosa {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

// Exclusive prefix (in thread order) of one int per thread; *total gets the sum.
template <int NWARPS>
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  int off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NWARPS; ++w) {
    const int t = warp_tot[w];
    off += (w < warp) ? t : 0;
    tot += t;
  }
  __syncthreads();
  *total = tot;
  return off + x - v;
}

constexpr int kSmallCut = 256;  // candidates ranked directly (one per thread)

// Rank (1-based) of the key kept as the next step's Gamma_q threshold hint for a
// cut of `need`: far enough below the cut that the next step's scores rarely
// drift past it (4 need), while the candidates at or above it stay within the
// directly ranked kSmallCut.
__device__ __forceinline__ int hint_rank(int need) {
  return min(4 * need, max(2 * need, kSmallCut / 2));
}

struct SelShared {
  uint32_t hist[256];
  int warp_tot[kSelWarps];
  int bcast[3];
  uint32_t red[3];
  int list[kSmallCut];              // compacted candidates of a small cut
  unsigned long long comp[kSmallCut];  // their (key, lower-index-first) composites
};

// Candidate i takes part in a cut when (flag[i] & tmask) == tval.
// Finds the key threshold `thr` and the number `take_eq` of keys equal to it
// (lowest indices first) such that exactly `need` candidates are chosen.
// Requires 1 <= need < number of candidates.
__device__ void radix_threshold(const uint32_t* key, const uint8_t* flag, uint8_t tmask,
                                uint8_t tval, int n, int need, SelShared& sh, uint32_t* thr,
                                int* take_eq, int* count_eq) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t prefix = 0, pmask = 0;
  int remaining = need;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += kSelThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += kSelThreads) {
      const int i = base + threadIdx.x;
      uint32_t dig = 256;
      if (i < n && (flag[i] & tmask) == tval && (key[i] & pmask) == prefix)
        dig = (key[i] >> shift) & 255u;
      const unsigned grp = __match_any_sync(0xffffffffu, dig);
      if (dig != 256 && lane == __ffs(grp) - 1) atomicAdd(&sh.hist[dig], (uint32_t)__popc(grp));
    }
    __syncthreads();
    if (warp == 0) {
      int cnt[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = (int)sh.hist[255 - 8 * lane - j];
        sum += cnt[j];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - sum;
      if (excl < remaining && remaining <= incl) {
        int cum = excl;
        for (int j = 0; j < 8; ++j) {
          if (cum + cnt[j] >= remaining) {
            sh.bcast[0] = 255 - 8 * lane - j;
            sh.bcast[1] = remaining - cum;
            sh.bcast[2] = cnt[j];
            break;
          }
          cum += cnt[j];
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sh.bcast[0] << shift;
    pmask |= 0xFFu << shift;
    remaining = sh.bcast[1];
  }
  *thr = prefix;
  *take_eq = remaining;
  *count_eq = sh.bcast[2];  // after the last pass: candidates whose key equals thr
}

// Marks (flag |= setbit) the `need` best candidates of a cut, ties to lower index.
__device__ void mark_top(const uint32_t* key, uint8_t* flag, uint8_t tmask, uint8_t tval,
                         uint8_t setbit, int n, int need, int count, SelShared& sh) {
  if (need <= 0) return;
  if (need >= count) {
    for (int i = threadIdx.x; i < n; i += kSelThreads)
      if ((flag[i] & tmask) == tval) flag[i] |= setbit;
    __syncthreads();
    return;
  }
  uint32_t thr;
  int take_eq, count_eq;
  radix_threshold(key, flag, tmask, tval, n, need, sh, &thr, &take_eq, &count_eq);
  if (take_eq == count_eq) {  // no tie at the cut to break: one pass
    for (int i = threadIdx.x; i < n; i += kSelThreads)
      if ((flag[i] & tmask) == tval && key[i] >= thr) flag[i] |= setbit;
    __syncthreads();
    return;
  }
  int run = 0;
  for (int base = 0; base < n; base += kSelThreads) {
    const int i = base + threadIdx.x;
    const bool v = i < n && (flag[i] & tmask) == tval;
    const bool eq = v && key[i] == thr;
    int tot;
    const int ex = block_excl_scan<kSelWarps>(eq ? 1 : 0, sh.warp_tot, &tot);
    if (v && (key[i] > thr || (eq && run + ex < take_eq))) flag[i] |= setbit;
    run += tot;
  }
  __syncthreads();
}

// Gamma_e when few blocks are eligible (the steady state: the previous Gamma_e
// plus at most one new block): compact the eligible blocks in index order from
// the bitmask words, give each one thread, and rank it against the others by
// (key, lower index first); the `need` best are chosen. Also counts a near-tie
// at the cut. Requires 1 <= need < count <= kSmallCut.
__device__ void mark_top_small_eligible(const uint32_t* key, uint8_t* flag, const uint32_t* elig,
                                        int n, int need, int count, SelShared& sh,
                                        unsigned long long* near_ties) {
  const int nw = (n + 31) >> 5;
  int base = 0;
  for (int w0 = 0; w0 < nw; w0 += kSelThreads) {
    const int w = w0 + threadIdx.x;
    uint32_t bits = 0;
    if (w < nw) {
      bits = elig[w];
      if (w == nw - 1 && (n & 31)) bits &= (1u << (n & 31)) - 1u;
    }
    int tot;
    int pos = base + block_excl_scan<kSelWarps>(__popc(bits), sh.warp_tot, &tot);
    while (bits) {
      const int b = __ffs(bits) - 1;
      const int i = w * 32 + b;
      sh.list[pos] = i;
      sh.comp[pos] = ((unsigned long long)key[i] << 32) | (0xFFFFFFFFu - (uint32_t)i);
      ++pos;
      bits &= bits - 1;
    }
    base += tot;
  }
  if (threadIdx.x == 0) {
    sh.red[0] = 0xFFFFFFFFu;
    sh.red[1] = 0u;
    sh.red[2] = 0u;
  }
  __syncthreads();
  if (threadIdx.x < count) {
    const unsigned long long mine = sh.comp[threadIdx.x];
    int rank = 0;
    for (int j = 0; j < count; ++j) rank += (sh.comp[j] > mine) ? 1 : 0;
    const int i = sh.list[threadIdx.x];
    const uint32_t kk = key[i];
    if (rank < need) flag[i] |= 2;
    if (rank == need - 1) sh.red[0] = kk;  // weakest chosen
    if (rank == need) sh.red[1] = kk;      // strongest left out
    atomicMax(&sh.red[2], __float_as_uint(fabsf(key_to_float(kk))));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const float gap = key_to_float(sh.red[0]) - key_to_float(sh.red[1]);
    if (gap < 1e-5f * __uint_as_float(sh.red[2])) atomicAdd(near_ties, 1ull);
  }
}

// Counts a near-tie at a cut: the weakest chosen and the strongest left-out fp32
// scores differ by less than 1e-5 * max |score| over the cut's candidates.
__device__ void near_tie_stat(const uint32_t* key, const uint8_t* flag, uint8_t tmask,
                              uint8_t tval, uint8_t setbit, int n, SelShared& sh,
                              unsigned long long* counter) {
  if (threadIdx.x == 0) {
    sh.red[0] = 0xFFFFFFFFu;
    sh.red[1] = 0u;
    sh.red[2] = 0u;
  }
  __syncthreads();
  uint32_t mn = 0xFFFFFFFFu, mx = 0u, ab = 0u;
  for (int i = threadIdx.x; i < n; i += kSelThreads) {
    if ((flag[i] & tmask) != tval) continue;
    const uint32_t kk = key[i];
    if (flag[i] & setbit) mn = min(mn, kk);
    else mx = max(mx, kk);
    ab = max(ab, __float_as_uint(fabsf(key_to_float(kk))));
  }
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, o));
  }
  if ((threadIdx.x & 31) == 0) {
    atomicMin(&sh.red[0], mn);
    atomicMax(&sh.red[1], mx);
    atomicMax(&sh.red[2], ab);
  }
  __syncthreads();
  if (threadIdx.x == 0 && sh.red[0] != 0xFFFFFFFFu && sh.red[1] != 0u) {
    const float gap = key_to_float(sh.red[0]) - key_to_float(sh.red[1]);
    if (gap < 1e-5f * __uint_as_float(sh.red[2])) atomicAdd(counter, 1ull);
  }
  __syncthreads();
}

// Gamma_q from a threshold hint (the key that admitted about four times the cut's
// size at the unit's previous step): when at least `need` and at most kSmallCut
// candidates have a key >= hint, the cut lies among them (every other key is
// smaller), so they are compacted in index order and ranked against each other
// by (key, lower index first); the `need` best get setbit. Exact whenever it
// answers; returns false (nothing marked) otherwise, and the caller runs the
// radix cut. Also counts a near-tie at the cut (as near_tie_stat) and leaves in
// *hint_out the key of rank min(count, hint_rank(need)) for the next step.
// Candidates: (flag & tmask) == tval. Requires 1 <= need < number of candidates.
__device__ bool mark_top_hint(const uint32_t* key, uint8_t* flag, uint8_t tmask, uint8_t tval,
                              uint8_t setbit, int n, int need, uint32_t hint, SelShared& sh,
                              unsigned long long* near_ties, uint32_t* hint_out) {
  // one pass: candidates at or above the hint, the largest key below it, max |score|
  int mine = 0;
  uint32_t below = 0u, ab = 0u;
  for (int i = threadIdx.x; i < n; i += kSelThreads) {
    if ((flag[i] & tmask) != tval) continue;
    const uint32_t kk = key[i];
    if (kk >= hint) ++mine;
    else below = max(below, kk);
    ab = max(ab, __float_as_uint(fabsf(key_to_float(kk))));
  }
  for (int o = 16; o > 0; o >>= 1) {
    below = max(below, __shfl_xor_sync(0xffffffffu, below, o));
    ab = max(ab, __shfl_xor_sync(0xffffffffu, ab, o));
  }
  if (threadIdx.x == 0) {
    sh.red[0] = 0u;
    sh.red[1] = 0u;
    sh.red[2] = 0u;
  }
  int count;
  block_excl_scan<kSelWarps>(mine, sh.warp_tot, &count);  // (its barriers order the red[] init)
  if ((threadIdx.x & 31) == 0) {
    atomicMax(&sh.red[1], below);
    atomicMax(&sh.red[2], ab);
  }
  if (count < need || count > kSmallCut) return false;  // (count is CTA-uniform)
  // compact the candidates >= hint in index order
  int base = 0;
  for (int b0 = 0; b0 < n; b0 += kSelThreads) {
    const int i = b0 + threadIdx.x;
    const bool on = i < n && (flag[i] & tmask) == tval && key[i] >= hint;
    int tot;
    const int at = base + block_excl_scan<kSelWarps>(on ? 1 : 0, sh.warp_tot, &tot);
    if (on) {
      sh.list[at] = i;
      sh.comp[at] = ((unsigned long long)key[i] << 32) | (0xFFFFFFFFu - (uint32_t)i);
    }
    base += tot;
  }
  __syncthreads();
  const int r_hint = min(count, hint_rank(need)) - 1;
  if (threadIdx.x < count) {
    const unsigned long long c = sh.comp[threadIdx.x];
    int rank = 0;
    for (int j = 0; j < count; ++j) rank += (sh.comp[j] > c) ? 1 : 0;
    const uint32_t kk = (uint32_t)(c >> 32);
    if (rank < need) flag[sh.list[threadIdx.x]] |= setbit;
    if (rank == need - 1) sh.red[0] = kk;                 // weakest chosen
    if (rank == need) atomicMax(&sh.red[1], kk);           // strongest left out (>= any below)
    if (rank == r_hint) *hint_out = kk;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const float gap = key_to_float(sh.red[0]) - key_to_float(sh.red[1]);
    if (gap < 1e-5f * __uint_as_float(sh.red[2])) atomicAdd(near_ties, 1ull);
  }
  return true;
}

// The set-difference of unit u against its slots, by warp 0 alone (the CTA's
// other warps return). Writes the load list (ascending block, paired by rank with
// the ascending free slots) and its length, the new slot table and residency
// mask, and the two attention block tables (slots kept from the previous step;
// slots filled by this step's loads). With at most a few hundred mask words and
// k <= 256 slots, lane-strided words, shuffles and ballots do it without a
// block-wide barrier, which costs a microsecond or more while the scoring kernels
// fill the SMs.
// selm: the unit's selection mask words (this CTA's shared copy); s2b_s: a shared
// copy of its slot table, kept up to date here; res_s: a shared copy of its
// residency words, valid when nw <= NT (else they are read from the state).
template <int NT>
__device__ void setdiff_phase(const Shape& s, const State& st, int u, int n, int just_completed,
                              int cold, int gamma, const uint32_t* selm, int* s2b_s,
                              const uint32_t* res_s) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const unsigned below = (1u << lane) - 1u;
  __shared__ int load_blk[kMaxK];
  __shared__ int free_list[kMaxK];
  __shared__ uint32_t fresh[kMaxK / 32];  // slots this step's loads fill
  uint32_t* resm = st.resmask + (long long)u * s.W;
  int32_t* s2b = st.slot2blk + (long long)u * s.k;
  const int nw = (n + 31) >> 5;

  // Loads: selected and not held by a slot, ascending block index.
  int nload = 0;
  for (int w0 = 0; w0 < nw; w0 += 32) {
    const int w = w0 + lane;
    uint32_t lw = 0u;
    if (w < nw) lw = selm[w] & ~((nw <= NT) ? res_s[w] : resm[w]);
    const int c = __popc(lw);
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    int pos = nload + x - c;
    while (lw) {
      load_blk[pos++] = w * 32 + __ffs(lw) - 1;
      lw &= lw - 1;
    }
    nload += __shfl_sync(0xffffffffu, x, 31);
  }
  // Free slots: empty, or holding a block outside Gamma; ascending slot index.
  // (|Gamma| <= k, so there are at least nload of them.)
  int nfree = 0;
  for (int s0 = 0; s0 < s.k; s0 += 32) {
    const int sl = s0 + lane;
    bool f = false;
    if (sl < s.k) {
      const int b = s2b_s[sl];
      f = (b < 0) || !((selm[b >> 5] >> (b & 31)) & 1u);
    }
    const unsigned m = __ballot_sync(0xffffffffu, f);
    if (f) free_list[nfree + __popc(m & below)] = sl;
    nfree += __popc(m);
  }
  if (lane < kMaxK / 32) fresh[lane] = 0u;
  __syncwarp();

  int32_t* loads = st.loads + (long long)u * s.k * 3;
  bool tail_loaded = false;
  for (int j = lane; j < nload; j += 32) {
    const int blk = load_blk[j], slot = free_list[j];
    const int src = (blk == just_completed) ? 1 : 0;
    loads[3 * j] = blk;
    loads[3 * j + 1] = slot;
    loads[3 * j + 2] = src;
    s2b[slot] = blk;
    s2b_s[slot] = blk;
    atomicOr(&fresh[slot >> 5], 1u << (slot & 31));
    tail_loaded |= (src != 0);
  }
  for (int j = nload + lane; j < nfree; j += 32) {
    s2b[free_list[j]] = -1;
    s2b_s[free_list[j]] = -1;
  }
  for (int w = lane; w < s.W; w += 32) resm[w] = (w < nw) ? selm[w] : 0u;
  if (lane == 0) st.nload[u] = nload;  // the gather numbers the chunk's entries from these
  __syncwarp();
  // Attention tables: slots kept from the previous step (usable while the gather
  // runs) and slots that this step's loads fill.
  int32_t* tres = st.block_tab + (long long)u * s.k;
  int32_t* tnew = st.tab_new + (long long)u * s.k;
  for (int sl = lane; sl < s.k; sl += 32) {
    const bool filled = (fresh[sl >> 5] >> (sl & 31)) & 1u;
    tres[sl] = (!filled && s2b_s[sl] >= 0) ? u * s.k + sl : -1;
    tnew[sl] = (sl < nload) ? u * s.k + free_list[sl] : -1;
  }
  const int n_tail = __any_sync(0xffffffffu, tail_loaded) ? 1 : 0;

  if (lane == 0) {
    const int n_host = nload - n_tail;
    DevStats* ds = st.stats;
    atomicAdd(&ds->host_loads, (unsigned long long)n_host);
    atomicAdd(&ds->tail_loads, (unsigned long long)n_tail);
    if (cold) {
      atomicAdd(&ds->cold_host_loads, (unsigned long long)n_host);
    } else if (n >= s.k) {
      const int hits = gamma - n_host;
      atomicMin(&ds->min_hits, hits);
      atomicAdd(&ds->sum_hits, (unsigned long long)hits);
      atomicAdd(&ds->hit_samples, 1ull);
      atomicMax(&ds->max_host_loads_unit, n_host);
    }
  }
}

// Dual selection and set-difference of unit u by the whole CTA (kSelThreads
// threads). dyn: shared memory of key [maxBlk] u32 + flag [maxBlk] u8.
// flag bits: 1 = eligible, 2 = in Gamma_e, 4 = in Gamma_q. The set-difference
// against the unit's slots runs once Gamma is known.
__device__ __forceinline__ void select_setdiff_unit(const Shape& s, const State& st, int u, int cold,
                                                 int chunk, uint8_t* dyn) {
  const int n = st.io->n_cand;
  const int just_completed = st.io->just_completed;
  __shared__ SelShared sh;
  uint32_t* key = reinterpret_cast<uint32_t*>(dyn);
  uint8_t* flag = dyn + (size_t)s.maxBlk * 4;
  const float* se = st.se + (long long)u * s.maxBlk;
  const float* sq = st.sq + (long long)u * s.maxBlk;  // read through L2 (other CTAs wrote it)
  uint32_t* elig = st.elig + (long long)u * s.W;
  // Loaded now for the set-difference at the end, so that their latency overlaps
  // the selection: the slot table (shared copy) and this thread's residency word.
  __shared__ int s2b_s[kMaxK];
  for (int sl = threadIdx.x; sl < s.k; sl += kSelThreads) s2b_s[sl] = st.slot2blk[(long long)u * s.k + sl];
  const uint32_t res0 =
      ((int)threadIdx.x < ((n + 31) >> 5)) ? st.resmask[(long long)u * s.W + threadIdx.x] : 0u;
  __shared__ uint32_t res_s[kSelThreads];
  // The query-aware scores of the first kSqPre * kSelThreads candidates and the
  // threshold hint, loaded with the eviction scores below (one round trip).
  constexpr int kSqPre = 4;
  float sqv[kSqPre];
#pragma unroll
  for (int r = 0; r < kSqPre; ++r) {
    const int i = threadIdx.x + r * kSelThreads;
    sqv[r] = (i < n) ? __ldcg(sq + i) : 0.f;
  }
  const uint32_t qhint0 = (st.qhint != nullptr) ? st.qhint[u] : 0u;

  int my_elig = 0;
  for (int i = threadIdx.x; i < n; i += kSelThreads) {
    const uint8_t el = (elig[i >> 5] >> (i & 31)) & 1u;
    flag[i] = el;
    key[i] = ordered_key(se[i]);
    my_elig += el;
  }
  int cnt_e;
  block_excl_scan<kSelWarps>(my_elig, sh.warp_tot, &cnt_e);  // also orders the writes above
  const int need_e = min(s.ke, cnt_e);
  if (need_e > 0 && need_e < cnt_e && cnt_e <= kSmallCut) {
    mark_top_small_eligible(key, flag, elig, n, need_e, cnt_e, sh, &st.stats->near_ties);
  } else {
    mark_top(key, flag, 1, 1, 2, n, need_e, cnt_e, sh);
    if (need_e > 0 && need_e < cnt_e)
      near_tie_stat(key, flag, 1, 1, 2, n, sh, &st.stats->near_ties);
  }

  if (threadIdx.x == 0 && chunk == 0) trace_mark(st.trace, kTrSel0E);
#pragma unroll
  for (int r = 0; r < kSqPre; ++r) {
    const int i = threadIdx.x + r * kSelThreads;
    if (i < n) key[i] = ordered_key(sqv[r]);
  }
  for (int i = threadIdx.x + kSqPre * kSelThreads; i < n; i += kSelThreads)
    key[i] = ordered_key(__ldcg(sq + i));
  __syncthreads();
  const int cnt_q = n - need_e;
  const int need_q = min(s.k - need_e, cnt_q);
  // Gamma_q: from the previous step's threshold hint when it brackets the cut,
  // else the radix cut (then the hint for the next step is the key of rank
  // hint_rank(need))
  bool cut = false;
  if (need_q > 0 && need_q < cnt_q && st.qhint != nullptr)
    cut = mark_top_hint(key, flag, 2, 0, 4, n, need_q, qhint0, sh, &st.stats->near_ties,
                        st.qhint + u);
  if (!cut) {
    mark_top(key, flag, 2, 0, 4, n, need_q, cnt_q, sh);
    if (need_q > 0 && need_q < cnt_q) {
      near_tie_stat(key, flag, 2, 0, 4, n, sh, &st.stats->near_ties);
      if (st.qhint != nullptr) {
        const int need2 = min(hint_rank(need_q), cnt_q);
        uint32_t thr2 = 0u;
        if (need2 < cnt_q) {
          int take_eq, count_eq;
          radix_threshold(key, flag, 2, 0, n, need2, sh, &thr2, &take_eq, &count_eq);
        }
        if (threadIdx.x == 0) st.qhint[u] = thr2;
      }
    }
  }

  if (threadIdx.x == 0 && chunk == 0) trace_mark(st.trace, kTrSel0Q);
  // Eligibility and selection masks, one ballot per 32-candidate word. After the
  // step the eligibility words are Gamma_e (strict eviction) and the selection
  // words Gamma_e + Gamma_q, so Gamma_e = sel & elig and Gamma_q = sel & ~elig; the
  // ascending index lists are derived from them where they are read (the debug
  // read), not written here.
  __syncthreads();  // the cuts are done reading key[]
  for (int base = 0; base < n; base += kSelThreads) {
    const int i = base + threadIdx.x;
    const uint8_t f = (i < n) ? flag[i] : 0;
    const unsigned be = __ballot_sync(0xffffffffu, (f & 2) != 0);
    const unsigned bs = __ballot_sync(0xffffffffu, (f & 6) != 0);
    if ((threadIdx.x & 31) == 0 && base + (threadIdx.x & ~31) < n) {
      const int w = (base + (threadIdx.x & ~31)) >> 5;
      elig[w] = be;
      st.selmask[(long long)u * s.W + w] = bs;
      key[w] = bs;  // shared copy for the set-difference
    }
  }
  if (threadIdx.x == 0) {
    st.nsel[2 * u] = need_e;
    st.nsel[2 * u + 1] = need_q;
  }
  if ((int)threadIdx.x < ((n + 31) >> 5)) res_s[threadIdx.x] = res0;
  __syncthreads();  // the selection mask copy, nsel and res_s are visible to the whole CTA
  if (threadIdx.x == 0 && chunk == 0) trace_mark(st.trace, kTrSel0Emit);
  setdiff_phase<kSelThreads>(s, st, u, n, just_completed, cold, need_e + need_q, key, s2b_s, res_s);
}

}  // namespace
}  // namespace nosa
