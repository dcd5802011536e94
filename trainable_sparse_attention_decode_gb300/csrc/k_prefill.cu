// Training-time forward of NOSA (every query position of a sequence is a step).
//
// NOSA technical summary, Methodology §1: the locality constraint is imposed
// during training, so the dual selection runs causally at every query position t
// with token t appended: Gamma_e(t) = top-k_e of the eligible candidates by
// eviction score (strict eviction: eligibility <- Gamma_e(t)), Gamma_q(t) = the
// best k - |Gamma_e(t)| other candidates by the two-stage pooled query score; the
// attention covers the blocks of Gamma(t) plus t's own block up to t.
//
// Candidates change only when a block completes, and Gamma_e does not depend on
// the query, so Gamma_e is the same E_b for all 64 positions of block b and
// follows a short recurrence over blocks: E_0 = {}, E_b = top-k_e(E_{b-1} + {b-1}).
// The path:
//   prefill_pack_kernel    block units (the decode layout), pooled keys and block
//                          eviction scores of every block            (unit, block)
//   prefill_evict_kernel   the eviction sets E_b, one warp per block
//   prefill_select_kernel  per position: pooled query scores of the candidates
//                          outside E_b in fp32 on the CUDA cores, top-(k - |E_b|)
//                          by sorted per-lane lists (or warp arg-max rounds beyond
//                          32); writes the position's block table and tail
//                          (unit, block). Where k - k_e <= 32 and d is 64 or 128
//                          the selection runs on the tensor cores instead
//                          (k_prefill_sel_tc.cu) unless NOSA_PREFILL_SELECT_TC=0.
//   prefill_tile_kernel    (bf16, G <= 4, d in {64, 128}; k_prefill_tc.cu) the
//                          attention of a whole query block on the tensor cores,
//                          over the union of its positions' blocks;
//   attn_split_kernel      otherwise the split-K attention of the decode path, one
//                          virtual unit per (request, position, KV head), with
//                          per-unit tails (the causal partial block).
#include "nosa_internal.cuh"

#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>

namespace nosa {
namespace {

constexpr int kPackThreads = 256;
constexpr int kSelWarps = 8;
constexpr int kSelRegSlots = 16;  // top-m keys per lane held in registers
constexpr int kSelCC = 64;        // candidates per pooled-key chunk (two per lane)
constexpr int kSelDS = 16;        // dims of a chunk per shared-memory slice
constexpr int kSelNS = 3;         // slices in the cp.async ring
constexpr int kSelCStr = 4 * kSelDS + 4;  // floats per candidate in a slice (272 bytes)

__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Block units of the tiled tensor-core attention (bf16 inputs; k_prefill_tc.cu)
// hold their operands in the canonical K-major layout with the 128-byte swizzle
// (rows of 128 bytes = 64 elements along the MMA's K, 16-byte chunk c of row r
// stored at chunk c ^ (r % 8), 8-row groups 1024 bytes apart), so the MMAs read
// a unit where its bulk copy puts it (at a 1024-byte aligned stage):
//   K   bf16, rows = tokens, K = head dim: 64-dim blocks of 64 x 128 bytes
//       (dims 8c .. 8c + 7 of token t at (c / 8) 8192 + 128 t + 16 ((c % 8) ^ (t % 8)));
//   V^T fp16, rows = head dim, K = tokens: d x 128 bytes, each value times 2^vs
//       (vs from the largest |v| of the call, so every value converts exactly
//       unless it is 2^29 below that maximum); tokens 8g .. 8g + 7 of dim r at
//       128 d + 128 r + 16 (g ^ (r % 8));
//   e   fp32 x log2(e), as in the decode layout.

// Largest |v| of the call (as fp32 bits; nonnegative floats order like their
// bits) into *absmax, which starts at 0.
__global__ void __launch_bounds__(256) prefill_vmax_kernel(const __nv_bfloat16* __restrict__ v,
                                                           long long n, uint32_t* __restrict__ absmax) {
  uint32_t best = 0;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    best = max(best, __float_as_uint(fabsf(__bfloat162float(v[i]))));
  for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  if ((threadIdx.x & 31) == 0) atomicMax(absmax, best);
}

// Block unit of (unit u, block blk) from k, v [batch][L][Hkv][d], e [batch][L][Hkv];
// tokens past L are zeros. Complete blocks are pooled: sub-block mean keys (fp32
// token-order sums x 1/16) and the block's eviction score (max of the sub-block
// means of e). grid = (nblk, U).
template <typename T>
__global__ void __launch_bounds__(kPackThreads) prefill_pack_kernel(
    Shape s, const T* __restrict__ k, const T* __restrict__ v, const float* __restrict__ e, int L,
    int nblk, uint8_t* __restrict__ units, float* __restrict__ pk, float* __restrict__ se) {
  const int blk = blockIdx.x, u = blockIdx.y, b = u / s.Hkv, h = u % s.Hkv;
  uint8_t* unit = units + ((long long)u * nblk + blk) * s.payload;
  const int t0 = blk * s.B;
  const int nt = min(s.B, L - t0);
  for (int i = threadIdx.x; i < s.B * s.d; i += blockDim.x) {
    const int t = i / s.d, dim = i % s.d;
    T kv = from_f32<T>(0.f), vv = from_f32<T>(0.f);
    if (t < nt) {
      const long long src = (((long long)b * L + t0 + t) * s.Hkv + h) * s.d + dim;
      kv = k[src];
      vv = v[src];
    }
    *reinterpret_cast<T*>(unit + k_off(t, dim, s.B, s.elt)) = kv;
    *reinterpret_cast<T*>(unit + v_off(t, dim, s.B, s.d, s.elt)) = vv;
  }
  for (int t = threadIdx.x; t < s.B; t += blockDim.x)
    *reinterpret_cast<float*>(unit + e_off(t, s.B, s.d, s.elt)) =
        (t < nt) ? e[((long long)b * L + t0 + t) * s.Hkv + h] : 0.f;
  for (long long i = 2LL * s.B * s.d * s.elt + 4LL * s.B + threadIdx.x; i < s.payload; i += blockDim.x)
    unit[i] = 0;
  if (nt < s.B) return;  // an incomplete block is never a candidate
  for (int i = threadIdx.x; i < s.P * s.d; i += blockDim.x) {
    const int sb = i / s.d, dim = i % s.d;
    float acc = 0.f;
    for (int j = 0; j < s.S; ++j) {
      const long long src = (((long long)b * L + t0 + sb * s.S + j) * s.Hkv + h) * s.d + dim;
      acc += to_f32(k[src]);
    }
    pk[(((long long)u * nblk + blk) * s.P + sb) * s.d + dim] = acc * (1.0f / s.S);
  }
  if (threadIdx.x == 0) {
    float best = 0.f;
    for (int sb = 0; sb < s.P; ++sb) {
      float acc = 0.f;
      for (int j = 0; j < s.S; ++j) acc += e[((long long)b * L + t0 + sb * s.S + j) * s.Hkv + h];
      const float m = acc * (1.0f / s.S);
      best = (sb == 0) ? m : fmaxf(best, m);
    }
    se[(long long)u * nblk + blk] = best;
  }
}

// The packing for the tiled tensor-core attention (bf16, the layout above), block
// by block through shared memory: K and V staged with 16-byte loads; K written as
// whole swizzled 16-byte chunks; V^T as 16-byte chunks of 8 tokens of one head
// dim (consecutive threads take consecutive dims, so the gather from the staged V
// is free of bank conflicts), scaled by 2^vs into fp16; e x log2(e); pooled keys
// from the staged K in token order (the same fp32 sums as prefill_pack_kernel).
template <int D>
__global__ void __launch_bounds__(kPackThreads) prefill_pack_tc_kernel(
    Shape s, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    const float* __restrict__ e, int L, int nblk, uint8_t* __restrict__ units, float* __restrict__ pk,
    float* __restrict__ se, const uint32_t* __restrict__ vmax) {
  constexpr int RS = D + 8;  // padded row of the staged tiles (bf16 elements; 16-byte multiple)
  __shared__ __align__(16) __nv_bfloat16 k_s[64 * RS], v_s[64 * RS];
  const int blk = blockIdx.x, u = blockIdx.y, b = u / s.Hkv, h = u % s.Hkv;
  uint8_t* unit = units + ((long long)u * nblk + blk) * s.payload;
  const int t0 = blk * 64, nt = min(64, L - t0);
  const float vmul = ldexpf(1.0f, v_scale_exp(*vmax));
  for (int i = threadIdx.x; i < 64 * (D / 8); i += blockDim.x) {
    const int t = i / (D / 8), c = i % (D / 8);
    uint4 kx = make_uint4(0u, 0u, 0u, 0u), vx = kx;
    if (t < nt) {
      const long long src = (((long long)b * L + t0 + t) * s.Hkv + h) * D + c * 8;
      kx = *reinterpret_cast<const uint4*>(k + src);
      vx = *reinterpret_cast<const uint4*>(v + src);
    }
    *reinterpret_cast<uint4*>(k_s + t * RS + c * 8) = kx;
    *reinterpret_cast<uint4*>(v_s + t * RS + c * 8) = vx;
    // K chunk c of token t (dims 8c .. 8c + 7 are one chunk of the swizzled row)
    *reinterpret_cast<uint4*>(unit + (c >> 3) * 8192 + t * 128 + (((c & 7) ^ (t & 7)) << 4)) = kx;
  }
  __syncthreads();
  // V^T: row dim holds tokens 0..63 (8 chunks of 8); thread (dim, chunk tg)
  for (int i = threadIdx.x; i < D * 8; i += blockDim.x) {
    const int dim = i % D, tg = i / D;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float a0 = __bfloat162float(v_s[(8 * tg + 2 * q) * RS + dim]) * vmul;
      const float a1 = __bfloat162float(v_s[(8 * tg + 2 * q + 1) * RS + dim]) * vmul;
      const __half2 hh = __floats2half2_rn(a0, a1);
      w[q] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    *reinterpret_cast<uint4*>(unit + 64 * D * 2 + dim * 128 + ((tg ^ (dim & 7)) << 4)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (threadIdx.x < 64) {  // e x log2(e) (the tiled attention works in base 2)
    const int t = threadIdx.x;
    reinterpret_cast<float*>(unit + 2 * 64 * D * 2)[t] =
        (t < nt) ? e[((long long)b * L + t0 + t) * s.Hkv + h] * 1.4426950408889634f : 0.f;
  }
  if (nt < 64) return;  // an incomplete block is never a candidate
  for (int i = threadIdx.x; i < 4 * D; i += blockDim.x) {
    const int sb = i / D, dim = i % D;
    float acc = 0.f;
    for (int j = 0; j < 16; ++j) acc += __bfloat162float(k_s[(sb * 16 + j) * RS + dim]);
    pk[(((long long)u * nblk + blk) * 4 + sb) * D + dim] = acc * (1.0f / 16);
  }
  if (threadIdx.x == 0) {
    float best = 0.f;
    for (int sb = 0; sb < 4; ++sb) {
      float acc = 0.f;
      for (int j = 0; j < 16; ++j) acc += e[((long long)b * L + t0 + sb * 16 + j) * s.Hkv + h];
      const float m = acc * (1.0f / 16);
      best = (sb == 0) ? m : fmaxf(best, m);
    }
    se[(long long)u * nblk + blk] = best;
  }
}

// The eviction sets: for every block b with positions, E_b (ascending block ids)
// into Eb[u][b][k_e] and its size into Ecnt[u][b]. The recurrence E_b =
// top-k_e(E_{b-1} + {b-1}) (ties: the lower id stays) never brings an evicted block
// back, and the smallest member only grows, so E_b is the top-k_e of the whole
// prefix {0 .. b-1} in the order (score descending, id ascending): every block is
// computed on its own. One warp per block b: the k_e-th largest order-preserving
// score key by a bitwise threshold search over the prefix, then the members in
// ascending id order (keys above the threshold, and keys equal to it by ascending
// id until k_e). A NaN score ranks highest (the recurrence never removes one).
// grid = (ceil(nblk / 8), U), 8 warps; the unit's keys staged in shared memory.
__global__ void __launch_bounds__(256) prefill_evict_kernel(Shape s, const float* __restrict__ se,
                                                            int nblk, int32_t* __restrict__ Eb,
                                                            int32_t* __restrict__ Ecnt) {
  extern __shared__ uint32_t ekeys[];  // [min(nblk, b0 + 8)]
  const int u = blockIdx.y, b0 = blockIdx.x * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = min(nblk, b0 + 8);
  for (int i = threadIdx.x; i < nk; i += blockDim.x) {
    const float x = se[(long long)u * nblk + i];
    ekeys[i] = (x != x) ? 0xffffffffu : ordered_key(x);
  }
  __syncthreads();
  const int b = b0 + warp;
  if (b >= nblk) return;
  const int n = b;  // candidates 0 .. b-1
  int32_t* out = Eb + ((long long)u * nblk + b) * s.ke;
  if (n <= s.ke) {
    for (int i = lane; i < n; i += 32) out[i] = i;
    if (lane == 0) Ecnt[(long long)u * nblk + b] = n;
    return;
  }
  uint32_t thr = 0u;  // the largest key with at least k_e keys at or above it
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = thr | (1u << bit);
    int c = 0;
    for (int j = lane; j < n; j += 32) c += ekeys[j] >= cand ? 1 : 0;
    if ((int)__reduce_add_sync(0xffffffffu, (uint32_t)c) >= s.ke) thr = cand;
  }
  int gt = 0;
  for (int j = lane; j < n; j += 32) gt += ekeys[j] > thr ? 1 : 0;
  const int need_eq = s.ke - (int)__reduce_add_sync(0xffffffffu, (uint32_t)gt);
  int run = 0, eq_seen = 0;
  for (int base = 0; base < n; base += 32) {
    const int j = base + lane;
    const uint32_t kj = j < n ? ekeys[j] : 0u;
    const bool eqj = j < n && kj == thr;
    const unsigned beq = __ballot_sync(0xffffffffu, eqj);
    const bool on = (j < n && kj > thr) || (eqj && eq_seen + __popc(beq & ((1u << lane) - 1u)) < need_eq);
    const unsigned bal = __ballot_sync(0xffffffffu, on);
    if (on) out[run + __popc(bal & ((1u << lane) - 1u))] = j;
    run += __popc(bal);
    eq_seen += __popc(beq);
  }
  if (lane == 0) Ecnt[(long long)u * nblk + b] = run;
}

// Loads 4 consecutive elements of q as fp32.
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
  const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
  return make_float4(a.x, a.y, c.x, c.y);
}

// Top-m of one position's scores by sorted per-lane lists: the NP = 32 / PB lanes
// of position i (lane = i * NP + part) each keep the best MM entries of a
// contiguous part of the candidate list, in the selection order (order-preserving
// key descending, then list index ascending: lower block id first at equal
// scores), then the position's m winners are drawn from the heads of its NP lists
// by a shuffle tournament and marked in tk (one bit per block id). A NaN score is
// never selected. Requires m <= MM.
template <int MM, int PB>
__device__ __forceinline__ void select_topm_lists(const float* sqw, int nblk, int ncl, int m,
                                                  const int32_t* cl, uint32_t* taken, int W, int lane) {
  constexpr int NP = 32 / PB;
  const int i = lane / NP, part = lane % NP;
  const int per = (ncl + NP - 1) / NP;
  const int lo = min(ncl, part * per), hi = min(ncl, lo + per);
  const float* sp = sqw + (size_t)i * nblk;
  uint32_t key[MM];
  int idx[MM];
#pragma unroll
  for (int r = 0; r < MM; ++r) {
    key[r] = 0u;
    idx[r] = 0x7fffffff;
  }
  for (int ci = lo; ci < hi; ++ci) {
    const float x = sp[ci];
    const uint32_t kx = x == x ? ordered_key(x) : 0u;
    if (kx > key[MM - 1]) {
      // insert at the first entry it beats (ci is above every index held, so
      // an equal key stays behind); the entries below shift down by one
      bool g[MM];
#pragma unroll
      for (int r = 0; r < MM; ++r) g[r] = kx > key[r];
#pragma unroll
      for (int r = MM - 1; r > 0; --r) {
        key[r] = g[r] ? (g[r - 1] ? key[r - 1] : kx) : key[r];
        idx[r] = g[r] ? (g[r - 1] ? idx[r - 1] : ci) : idx[r];
      }
      key[0] = g[0] ? kx : key[0];
      idx[0] = g[0] ? ci : idx[0];
    }
  }
  uint32_t* tk = taken + (size_t)i * W;
  for (int round = 0; round < m; ++round) {
    uint32_t bk = key[0];
    int bi = idx[0];
#pragma unroll
    for (int o = 1; o < NP; o <<= 1) {
      const uint32_t ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ok > bk || (ok == bk && oi < bi)) {
        bk = ok;
        bi = oi;
      }
    }
    if (bk != 0u && idx[0] == bi) {  // the winning part pops its head and marks the block
      // (bk == 0: nothing valid left; the rounds still run, as the shuffles span the warp)
      const int j = cl[bi];
      atomicOr(&tk[j >> 5], 1u << (j & 31));
#pragma unroll
      for (int r = 0; r < MM - 1; ++r) {
        key[r] = key[r + 1];
        idx[r] = idx[r + 1];
      }
      key[MM - 1] = 0u;
      idx[MM - 1] = 0x7fffffff;
    }
  }
}

// Per position t of block b (CTA (u, b); warp w takes positions 64 b + w, + 8, ...,
// PB of them at a time): q_bar = mean of the G query heads, sq(j) = max over
// sub-blocks of q_bar . K_bar[j][s] / sqrt(d) for candidates j < b outside E_b,
// then the top-(k - |E_b|) (ties: lower block id). Writes the position's
// selection (E_b ascending, then Gamma_q ascending, -1 pad) into sel, its
// attention block table (unit indices) and tail.
// Scoring: lane c of every warp owns candidates c and c + 32 of a chunk of 64 and
// computes their 8 sub-block dot products with each of the warp's PB positions
// (8 x PB accumulators, each a pair of fp32 partial sums over alternate dims,
// paired FMAs): per 4 dims a lane reads 8 key rows and PB q_bar rows from shared
// memory for 32 PB FMAs, which keeps the shared-memory reads under the FMA time.
// The CTA streams each chunk through shared memory 16 dims at a time (cp.async
// ring of kSelNS slices; a candidate's 4 x 16 floats at a 272-byte stride, so the
// 8 lanes of a quarter warp read 8 different banks). Selection: sorted per-lane
// lists (select_topm_lists) for all PB positions at once when m <= 32, else m
// rounds of warp arg-max per position. Blocks run heaviest first (blockIdx.y
// counts down from the last block): the scoring work of block b grows with b.
template <typename T, int D, int PB>
__global__ void __launch_bounds__(kSelWarps * 32, PB >= 4 ? 1 : 2) prefill_select_kernel(
    Shape s, const T* __restrict__ q, int L, int nblk, const float* __restrict__ pk,
    const int32_t* __restrict__ Eb, const int32_t* __restrict__ Ecnt, int32_t* __restrict__ sel,
    int32_t* __restrict__ block_tab, int32_t* __restrict__ tail_tab, int32_t* __restrict__ tail_len,
    float inv_sqrt_d) {
  constexpr int NDS = D / kSelDS;  // dim slices of a chunk
  extern __shared__ __align__(16) uint8_t sm[];
  const int u = blockIdx.x, b = nblk - 1 - (int)blockIdx.y, req = u / s.Hkv, h = u % s.Hkv;
  const int W = (nblk + 31) / 32;
  float* stg = reinterpret_cast<float*>(sm);                                  // [kSelNS][64][kSelCStr]
  float* qb_s = stg + kSelNS * kSelCC * kSelCStr;                              // [kSelWarps][PB][D]
  float* sq_s = qb_s + kSelWarps * PB * D;                                     // [kSelWarps][PB][nblk]
  uint32_t* emask = reinterpret_cast<uint32_t*>(sq_s + (size_t)kSelWarps * PB * nblk);  // [W] E_b membership
  uint32_t* taken_s = emask + ((W + 3) & ~3);                                  // [kSelWarps][PB][W]
  int32_t* cl = reinterpret_cast<int32_t*>(taken_s + kSelWarps * PB * W);     // [nblk] candidates outside E_b
  int32_t* eb_s = cl + nblk;                                                   // [k_e] E_b ascending
  __shared__ int s_ncl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ecnt = Ecnt[(long long)u * nblk + b];
  const int32_t* eb = Eb + ((long long)u * nblk + b) * s.ke;
  for (int i = threadIdx.x; i < W; i += blockDim.x) emask[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < ecnt; i += blockDim.x) {
    const int j = eb[i];
    eb_s[i] = j;
    atomicOr(&emask[j >> 5], 1u << (j & 31));
  }
  __syncthreads();
  const int n_cand = b;  // blocks before the positions' own block
  const int m = min(s.k - ecnt, n_cand - ecnt);
  if (warp == 0) {  // the candidates outside E_b, ascending (scores are kept in this order)
    int run = 0;
    for (int base = 0; base < n_cand; base += 32) {
      const int j = base + lane;
      const bool on = j < n_cand && !((emask[j >> 5] >> (j & 31)) & 1u);
      const unsigned bal = __ballot_sync(0xffffffffu, on);
      if (on) cl[run + __popc(bal & ((1u << lane) - 1u))] = j;
      run += __popc(bal);
    }
    if (lane == 0) s_ncl = run;
  }
  __syncthreads();
  const int ncl = s_ncl;
  const int npos = min(s.B, L - b * s.B);
  float* sqw = sq_s + (size_t)warp * PB * nblk;
  float* qw = qb_s + warp * PB * D;
  uint32_t* tkw = taken_s + (size_t)warp * PB * W;
  const float inv_g = 1.0f / (float)s.G;
  const long long ubase = (long long)u * nblk;
  for (int g0 = 0; g0 < s.B / kSelWarps; g0 += PB) {
    if (kSelWarps * g0 >= npos) break;  // (CTA-uniform: the slice loop below syncs the CTA)
    // q_bar of the batch's positions (fp32 sum over the heads in order, x 1/G)
    if (lane < D / 4) {
      float4 a[PB];
#pragma unroll
      for (int i = 0; i < PB; ++i) a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      const T* qg = q + (((long long)req * L + (long long)b * s.B + warp + kSelWarps * g0) * s.Hq +
                         (long long)h * s.G) * D + 4 * lane;
      for (int g = 0; g < s.G; ++g)
#pragma unroll
        for (int i = 0; i < PB; ++i)
          if (warp + kSelWarps * (g0 + i) < npos) {
            const float4 x = load4(qg + ((long long)kSelWarps * i * s.Hq + g) * D);
            a[i].x += x.x;
            a[i].y += x.y;
            a[i].z += x.z;
            a[i].w += x.w;
          }
#pragma unroll
      for (int i = 0; i < PB; ++i)
        *reinterpret_cast<float4*>(qw + i * D + 4 * lane) =
            make_float4(a[i].x * inv_g, a[i].y * inv_g, a[i].z * inv_g, a[i].w * inv_g);
    }
    __syncwarp();
    if (m > 0) {
      const int nsl = (ncl + kSelCC - 1) / kSelCC * NDS;  // slices of this batch
      auto load_slice = [&](int sl) {
        if (sl < nsl) {
          float* dst = stg + (sl % kSelNS) * kSelCC * kSelCStr;
          const int ch = sl / NDS, ds = sl - ch * NDS;
          for (int i = threadIdx.x; i < kSelCC * 4 * (kSelDS / 4); i += blockDim.x) {  // 16-byte pieces
            const int c4 = i % (kSelDS / 4), r = (i / (kSelDS / 4)) & 3, cc = i / (kSelDS / 4) / 4;
            const int ci = ch * kSelCC + cc;
            if (ci < ncl)
              cp_async16(dst + cc * kSelCStr + r * kSelDS + 4 * c4,
                         pk + ((ubase + cl[ci]) * 4 + r) * D + ds * kSelDS + 4 * c4);
          }
        }
        cp_async_commit();  // (empty groups keep the wait count below meaning "slice sl landed")
      };
#pragma unroll
      for (int sl = 0; sl < kSelNS - 1; ++sl) load_slice(sl);
      float2 acc[8][PB];  // [candidate half * 4 + sub-block][position]
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int i = 0; i < PB; ++i) acc[r][i] = make_float2(0.f, 0.f);
      for (int sl = 0; sl < nsl; ++sl) {
        cp_async_wait<kSelNS - 2>();
        __syncthreads();  // slice sl visible to all; slice sl - 1's buffer is free
        load_slice(sl + kSelNS - 1);
        const int ch = sl / NDS, ds = sl - ch * NDS;
        const float* kr = stg + (sl % kSelNS) * kSelCC * kSelCStr + lane * kSelCStr;
        const float* qr = qw + ds * kSelDS;
#pragma unroll
        for (int d4 = 0; d4 < kSelDS / 4; ++d4) {
          float4 kx[8];
#pragma unroll
          for (int r = 0; r < 8; ++r)
            kx[r] = *reinterpret_cast<const float4*>(kr + (r >> 2) * 32 * kSelCStr + (r & 3) * kSelDS + 4 * d4);
#pragma unroll
          for (int i = 0; i < PB; ++i) {
            const float4 qx = *reinterpret_cast<const float4*>(qr + i * D + 4 * d4);
#pragma unroll
            for (int r = 0; r < 8; ++r)  // (dims x, y of all 8 rows, then z, w: no back-to-back dependences)
              acc[r][i] = __ffma2_rn(make_float2(kx[r].x, kx[r].y), make_float2(qx.x, qx.y), acc[r][i]);
#pragma unroll
            for (int r = 0; r < 8; ++r)
              acc[r][i] = __ffma2_rn(make_float2(kx[r].z, kx[r].w), make_float2(qx.z, qx.w), acc[r][i]);
          }
        }
        if (ds == NDS - 1) {  // chunk done: the lane's two candidates' scores for the PB positions
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const int ci = ch * kSelCC + 32 * c2 + lane;
#pragma unroll
            for (int i = 0; i < PB; ++i) {
              const float sc = fmaxf(fmaxf(acc[4 * c2][i].x + acc[4 * c2][i].y,
                                           acc[4 * c2 + 1][i].x + acc[4 * c2 + 1][i].y),
                                     fmaxf(acc[4 * c2 + 2][i].x + acc[4 * c2 + 2][i].y,
                                           acc[4 * c2 + 3][i].x + acc[4 * c2 + 3][i].y));
              if (ci < ncl) sqw[(size_t)i * nblk + ci] = sc * inv_sqrt_d;
            }
          }
#pragma unroll
          for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int i = 0; i < PB; ++i) acc[r][i] = make_float2(0.f, 0.f);
        }
      }
      __syncthreads();  // the ring is refilled by the next batch
    }
    // top-m of every position of the batch
    for (int w = lane; w < PB * W; w += 32) tkw[w] = 0u;
    __syncwarp();
    if (m > 0 && m <= 16) {
      select_topm_lists<16, PB>(sqw, nblk, ncl, m, cl, tkw, W, lane);
    } else if (m > 16 && m <= 32) {
      select_topm_lists<32, PB>(sqw, nblk, ncl, m, cl, tkw, W, lane);
    } else if (m > 0) {
      for (int i = 0; i < PB; ++i) {
        if (warp + kSelWarps * (g0 + i) >= npos) break;
        const float* sqp = sqw + (size_t)i * nblk;
        uint32_t* tk = tkw + (size_t)i * W;
        // m rounds of warp arg-max over the candidates outside E_b (scores in
        // list order, so a lower list index is a lower block id). Lane l owns
        // list entries l + 32 s as order-preserving keys (0: taken, or a NaN
        // score, never a candidate); a round takes the largest key, at equal
        // keys the lowest index, and only the winning lane looks for its next
        // best. Up to 512 entries the keys live in registers, beyond in shared
        // memory.
        if (ncl <= 32 * kSelRegSlots) {
          uint32_t kr[kSelRegSlots];
#pragma unroll
          for (int sl = 0; sl < kSelRegSlots; ++sl) {
            const int ci = lane + 32 * sl;
            const float x = ci < ncl ? sqp[ci] : 0.f;
            kr[sl] = (ci < ncl && x == x) ? ordered_key(x) : 0u;
          }
          auto best_of = [&](uint32_t& key, int& slot) {
            key = 0u;
            slot = 0;
#pragma unroll
            for (int sl = 0; sl < kSelRegSlots; ++sl)
              if (kr[sl] > key) {
                key = kr[sl];
                slot = sl;
              }
          };
          uint32_t lkey;
          int lslot;
          best_of(lkey, lslot);
          for (int round = 0; round < m; ++round) {
            const uint32_t kmax = __reduce_max_sync(0xffffffffu, lkey);
            if (kmax == 0u) break;  // none left (NaN scores)
            const uint32_t win =
                __reduce_min_sync(0xffffffffu, lkey == kmax ? (uint32_t)(lane + 32 * lslot) : 0xffffffffu);
            if ((int)(win & 31) == lane) {
              const int j = cl[win];
              atomicOr(&tk[j >> 5], 1u << (j & 31));  // (winners of other rounds share words)
#pragma unroll
              for (int sl = 0; sl < kSelRegSlots; ++sl)
                if (sl == lslot) kr[sl] = 0u;
              best_of(lkey, lslot);
            }
          }
        } else {
          auto lane_best = [&](uint32_t& key, int& idx) {
            key = 0u;
            idx = 0x7fffffff;
            for (int ci = lane; ci < ncl; ci += 32) {
              const int j = cl[ci];
              if ((tk[j >> 5] >> (j & 31)) & 1u) continue;
              const float x = sqp[ci];
              if (x != x) continue;
              const uint32_t kx = ordered_key(x);
              if (kx > key) {  // ascending index: the first of equal keys stays
                key = kx;
                idx = ci;
              }
            }
          };
          uint32_t lkey;
          int lidx;
          lane_best(lkey, lidx);
          for (int round = 0; round < m; ++round) {
            const uint32_t kmax = __reduce_max_sync(0xffffffffu, lkey);
            if (kmax == 0u) break;
            const int win = (int)__reduce_min_sync(0xffffffffu, lkey == kmax ? (uint32_t)lidx : 0xffffffffu);
            if ((win & 31) == lane) {
              const int j = cl[win];
              tk[j >> 5] |= 1u << (j & 31);
              lane_best(lkey, lidx);
            }
            __syncwarp();
          }
        }
        __syncwarp();
      }
    }
    __syncwarp();
    // outputs: E_b ascending, then Gamma_q ascending (ballot scan over the mask)
    for (int i = 0; i < PB; ++i) {
      const int p = warp + kSelWarps * (g0 + i);
      if (p >= npos) break;
      const int t = b * s.B + p;
      const long long vu = ((long long)req * L + t) * s.Hkv + h;  // virtual unit of the position
      const uint32_t* tk = tkw + (size_t)i * W;
      int32_t* selp = sel ? sel + vu * s.k : nullptr;
      int32_t* tab = block_tab + vu * s.k;
      for (int e = lane; e < ecnt; e += 32) {
        if (selp) selp[e] = eb_s[e];
        tab[e] = (int32_t)(ubase + eb_s[e]);
      }
      int run = ecnt;
      if (m > 0)
        for (int base = 0; base < n_cand; base += 32) {
          const int j = base + lane;
          const bool on = (j < n_cand) && ((tk[j >> 5] >> (j & 31)) & 1u);
          const unsigned bal = __ballot_sync(0xffffffffu, on);
          if (on) {
            const int at = run + __popc(bal & ((1u << lane) - 1u));
            if (selp) selp[at] = j;
            tab[at] = (int32_t)(ubase + j);
          }
          run += __popc(bal);
        }
      for (int e = run + lane; e < s.k; e += 32) {
        if (selp) selp[e] = -1;
        tab[e] = -1;
      }
      if (lane == 0) {
        tail_tab[vu] = (int32_t)(ubase + b);
        tail_len[vu] = p + 1;
      }
    }
    __syncwarp();
  }
}

// Dynamic shared memory of the selection: slice ring, q_bar, score scratch and
// taken masks of 8 warps x PB positions, E_b mask, candidate list, E_b.
size_t select_smem_bytes(int d, int ke, int nblk, int pb) {
  const int W = (nblk + 31) / 32;
  return (size_t)kSelNS * kSelCC * kSelCStr * 4 + (size_t)kSelWarps * pb * d * 4 +
         (size_t)kSelWarps * pb * nblk * 4 + (size_t)((W + 3) & ~3) * 4 + (size_t)kSelWarps * pb * W * 4 +
         (size_t)nblk * 4 + (size_t)std::max(ke, 1) * 4;
}

// Positions per warp scored in one pass over the candidates: the most (<= 8,
// all of a warp's positions) whose score scratch fits in 220 KB. The widths 2
// and 1 take over beyond about 1 200 and 2 400 blocks; NOSA_PREFILL_SELECT_PB
// (1, 2, 4 or 8, read at every call) caps the width, which changes how often
// the pooled keys are streamed, never the result.
int select_pb(int d, int ke, int nblk) {
  int pb = 8;
  if (const char* g = std::getenv("NOSA_PREFILL_SELECT_PB")) {
    const int v = std::atoi(g);
    if (v == 1 || v == 2 || v == 4) pb = v;
  }
  while (pb > 1 && select_smem_bytes(d, ke, nblk, pb) > 220 * 1024) pb >>= 1;
  return pb;
}

template <typename T, int D, int PB>
cudaError_t launch_select_pb(const Shape& s, dim3 grid, size_t smem, const T* q, int L, int nblk,
                             const float* pk, const int32_t* Eb, const int32_t* Ecnt, int32_t* sel,
                             int32_t* tab, int32_t* ttab, int32_t* tlen, float isd, cudaStream_t stream) {
  static std::atomic<int> lim[64];
  cudaError_t err = raise_smem_limit((const void*)prefill_select_kernel<T, D, PB>, smem, lim);
  if (err != cudaSuccess) return err;
  prefill_select_kernel<T, D, PB><<<grid, kSelWarps * 32, smem, stream>>>(s, q, L, nblk, pk, Eb, Ecnt, sel,
                                                                           tab, ttab, tlen, isd);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_select_d(const Shape& s, dim3 grid, size_t smem, int pb, const T* q, int L, int nblk,
                            const float* pk, const int32_t* Eb, const int32_t* Ecnt, int32_t* sel,
                            int32_t* tab, int32_t* ttab, int32_t* tlen, float isd, cudaStream_t stream) {
  switch (pb) {
    case 8: return launch_select_pb<T, D, 8>(s, grid, smem, q, L, nblk, pk, Eb, Ecnt, sel, tab, ttab, tlen, isd, stream);
    case 4: return launch_select_pb<T, D, 4>(s, grid, smem, q, L, nblk, pk, Eb, Ecnt, sel, tab, ttab, tlen, isd, stream);
    case 2: return launch_select_pb<T, D, 2>(s, grid, smem, q, L, nblk, pk, Eb, Ecnt, sel, tab, ttab, tlen, isd, stream);
    default: return launch_select_pb<T, D, 1>(s, grid, smem, q, L, nblk, pk, Eb, Ecnt, sel, tab, ttab, tlen, isd, stream);
  }
}

template <typename T>
cudaError_t launch_select(const Shape& s, dim3 grid, size_t smem, int pb, const T* q, int L, int nblk,
                          const float* pk, const int32_t* Eb, const int32_t* Ecnt, int32_t* sel,
                          int32_t* tab, int32_t* ttab, int32_t* tlen, float isd, cudaStream_t stream) {
  if (s.d == 64)
    return launch_select_d<T, 64>(s, grid, smem, pb, q, L, nblk, pk, Eb, Ecnt, sel, tab, ttab, tlen, isd, stream);
  return launch_select_d<T, 128>(s, grid, smem, pb, q, L, nblk, pk, Eb, Ecnt, sel, tab, ttab, tlen, isd, stream);
}

}  // namespace

// Byte offsets of the training-time forward's workspace (each 256-byte aligned).
PrefillLayout prefill_layout(const Shape& s, int L, int nsplit) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  PrefillLayout w;
  const int nblk = (L + s.B - 1) / s.B;
  const size_t U = s.U, V = (size_t)s.U * L;  // units, virtual units (request, position, head)
  size_t off = 0;
  w.units = off;     off += up(U * nblk * (size_t)s.payload);
  w.pk = off;        off += up(U * nblk * s.P * s.d * 4);
  w.pk3 = off;       off += up(prefill_keysplit_bytes(s, nblk));
  w.se = off;        off += up(U * nblk * 4);
  w.eb = off;        off += up(U * nblk * (size_t)std::max(s.ke, 1) * 4);
  w.ecnt = off;      off += up(U * nblk * 4);
  w.tab = off;       off += up(V * s.k * 4);
  w.tail_tab = off;  off += up(V * 4);
  w.tail_len = off;  off += up(V * 4);
  w.part_acc = off;  off += nsplit > 1 ? up(V * nsplit * s.G * s.d * 4) : 0;
  w.part_ml = off;   off += nsplit > 1 ? up(V * nsplit * s.G * 2 * 4) : 0;
  w.counters = off;  off += up(V * 4);
  w.vmax = off;      off += 256;
  w.err = off;       off += 256;
  w.total = off;
  return w;
}

size_t prefill_select_smem(const Shape& s, int nblk) {
  return select_smem_bytes(s.d, s.ke, nblk, select_pb(s.d, s.ke, nblk));
}

cudaError_t launch_prefill_front(const Shape& s, int L, const void* q, const void* k,
                                 const void* v, const float* e, int32_t* sel, uint8_t* ws,
                                 const PrefillLayout& w, bool tc, cudaStream_t stream) {
  const int nblk = (L + s.B - 1) / s.B;
  uint8_t* units = ws + w.units;
  float* pk = reinterpret_cast<float*>(ws + w.pk);
  float* se = reinterpret_cast<float*>(ws + w.se);
  int32_t* Eb = reinterpret_cast<int32_t*>(ws + w.eb);
  int32_t* Ecnt = reinterpret_cast<int32_t*>(ws + w.ecnt);
  dim3 grid(nblk, s.U);
  uint32_t* vmax = reinterpret_cast<uint32_t*>(ws + w.vmax);  // zeroed by the caller
  if (s.dtype == 0) {
    prefill_pack_kernel<float><<<grid, kPackThreads, 0, stream>>>(
        s, (const float*)k, (const float*)v, e, L, nblk, units, pk, se);
  } else if (tc) {
    const long long n = (long long)s.batch * L * s.Hkv * s.d;
    const int blocks = (int)std::min<long long>((n + 255) / 256, 4 * 152);
    prefill_vmax_kernel<<<blocks, 256, 0, stream>>>((const __nv_bfloat16*)v, n, vmax);
    if (s.d == 64)
      prefill_pack_tc_kernel<64><<<grid, kPackThreads, 0, stream>>>(
          s, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, e, L, nblk, units, pk, se, vmax);
    else
      prefill_pack_tc_kernel<128><<<grid, kPackThreads, 0, stream>>>(
          s, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, e, L, nblk, units, pk, se, vmax);
  } else {
    prefill_pack_kernel<__nv_bfloat16><<<grid, kPackThreads, 0, stream>>>(
        s, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, e, L, nblk, units, pk, se);
  }
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  prefill_evict_kernel<<<dim3((nblk + 7) / 8, s.U), 256, (size_t)nblk * 4, stream>>>(s, se, nblk, Eb, Ecnt);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  int32_t* tab = reinterpret_cast<int32_t*>(ws + w.tab);
  int32_t* ttab = reinterpret_cast<int32_t*>(ws + w.tail_tab);
  int32_t* tlen = reinterpret_cast<int32_t*>(ws + w.tail_len);
  if (prefill_select_tc_ok(s, L))
    return launch_prefill_select_tc(s, L, q, pk, ws + w.pk3, Eb, Ecnt, sel, tab, ttab, tlen,
                                    reinterpret_cast<int*>(ws + w.err), stream);
  const size_t smem = prefill_select_smem(s, nblk);
  const int pb = select_pb(s.d, s.ke, nblk);
  const dim3 sgrid(s.U, nblk);  // (unit, block counted down from the last)
  const float isd = (float)(1.0 / sqrt((double)s.d));
  if (s.dtype == 0)
    return launch_select<float>(s, sgrid, smem, pb, (const float*)q, L, nblk, pk, Eb, Ecnt, sel, tab, ttab,
                                tlen, isd, stream);
  return launch_select<__nv_bfloat16>(s, sgrid, smem, pb, (const __nv_bfloat16*)q, L, nblk, pk, Eb, Ecnt,
                                      sel, tab, ttab, tlen, isd, stream);
}

}  // namespace nosa
