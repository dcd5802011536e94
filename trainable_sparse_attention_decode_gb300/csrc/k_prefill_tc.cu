// Training-time forward: block-sparse attention tiled by query block, on the
// tensor cores.
//
// NOSA technical summary, Methodology §1 (the dual selection at every query
// position during training) and §2 (ED-DMA: the eviction logit enters the
// attention logits before the exponential). The positions of a query block share
// Gamma_e (E_b) and their own block (the causal tail), and neighbouring positions
// pick mostly the same query-aware blocks, so one CTA per (unit, query block,
// M-tile) streams the union of its positions' blocks once and lets every position
// that selected a block use it:
//   rows      128 rows of (position x G heads) (row = position x G + head): the
//             positions 128 m / G .. of the query block for M-tile m;
//   union     built from the positions' block tables: per block a 64-bit mask of
//             the positions that selected it (the own block: every position);
//   pairs     the union's blocks two at a time: S = Q K^T on the tensor cores
//             (tcgen05.mma kind::f16, bf16 in, fp32 accumulator in tensor memory,
//             M = 128, N = 128 tokens, K = d, double-buffered); each row: logits
//             = S log2(e)/sqrt(d) + e_j log2(e), -inf where the row's position did
//             not select the block (in the own block also past the position);
//             P = exp2(logit - m) in fp16 written over the first half of the S
//             columns it came from; O += P V on the tensor cores with P read from
//             tensor memory (fp16 in: V converted exactly with one power-of-two
//             scale of the call; N = d, K = 128).
// Online softmax with a lazy reference: a row keeps its running max m until a
// pair raises it by more than 8 (base 2), so P <= 2^8; only then is the row's O
// rescaled in tensor memory. Four warps share a row quarter (tensor-memory lanes
// 32 q ..), each owning 32 tokens of one block of a pair: they exchange the row
// max through shared memory (a bounded mbarrier meet per quarter), keep their own
// part of the row sum l (fp32 probabilities, so the log-sum-exp is exact to fp32
// rounding) and rescale a quarter of O each; a warp writes its P over the first 16
// of its 32 S columns. Warp roles: warps 0-15 rows, warp 16 issues the MMAs,
// warp 17 the bulk copies (two stages of a pair's K, two of its V^T and e; K rows
// are interleaved at copy time, block a's 64 rows then block b's, per 64-wide
// head-dim block, so that S is one N = 128 product; the K of pair j + 2 loads as
// soon as S of pair j is done). Everything after the set-up is ordered by
// mbarriers:
//   kfull / vfull[st]   a pair's K / V^T and e landed
//   kempty / vempty[st] S / P V of that pair completed (the stage may be refilled)
//   s_full[sb] S of a pair is in          p_full     the rows wrote P (and rescaled O)
//   pv_done    P V of a pair completed
// S of pair j + 2 reuses the buffer of pair j only after P V of pair j, which
// reads P there, completed. Shared-memory operands are K-major with the 128-byte
// swizzle (rows of 128 bytes, 16-byte chunk c of row r at chunk c ^ (r % 8), 8-row
// groups 1024 bytes apart): K and V^T as the pack kernel lays out the units (pair
// stages 1024-byte aligned), Q written in that form here. Every wait is bounded;
// one that gives up sets the error word and the CTA stops, waits (bounded) for its
// copies and MMAs in flight and frees its tensor memory.
#include "nosa_internal.cuh"
#include "tcgen05.cuh"

#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>

namespace nosa {
namespace {
using namespace tc;

constexpr int kRowWarps = 16;                        // 4 per tensor-memory lane quarter
constexpr int kTileThreads = 32 * (kRowWarps + 2);    // + the MMA warp and the copy warp
constexpr int kPairStages = 2;
constexpr float kLn2F = 0.6931471805599453f;
constexpr float kRescale = 8.0f;                     // lazy-rescale threshold (base 2)

// A pair's K stage: [d/64][128 rows x 128 B] (block a rows 0-63, block b 64-127);
// its V stage: per block V^T (64 x d bf16 = K bytes) and e (256 B), 1024-aligned.
__host__ __device__ inline size_t pair_kbytes(int d) { return (size_t)64 * d * 2; }
__host__ __device__ inline size_t pair_vslot(int d) { return pair_kbytes(d) + 1024; }
__host__ __device__ inline size_t pair_kstage(int d) { return 2 * pair_kbytes(d); }
__host__ __device__ inline size_t pair_vstage(int d) { return 2 * pair_vslot(d); }

// Shared-memory carve-up of one CTA (offsets from a 1024-byte aligned base).
struct TileSmem {
  int d, nblk;
  __host__ __device__ size_t qt() const { return 0; }                                 // [d/64][128 x 128 B] bf16
  __host__ __device__ size_t kst() const { return (size_t)256 * d; }                  // [kPairStages][pair_kstage]
  __host__ __device__ size_t vst() const { return kst() + kPairStages * pair_kstage(d); }  // [kPairStages][pair_vstage]
  __host__ __device__ size_t mx() const { return vst() + kPairStages * pair_vstage(d); }   // [2][4][128] + [4][128] f32
  __host__ __device__ size_t mask() const { return mx() + 6144; }                     // [nblk][2] u32
  __host__ __device__ size_t list() const { return mask() + 8 * (size_t)nblk; }       // [nblk] i32
  __host__ __device__ size_t total() const { return list() + 4 * (size_t)nblk + 1024; }
};

__device__ __forceinline__ float ex2(float x) {  // the SFU's base-2 exponential (ex2(-inf) = 0)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 x = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&x);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 x = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&x);
}
// The four warps of a row quarter meet at `bar` (count 4, one arrival per warp
// after its shared-memory writes); false if one did not come in time.
__device__ __forceinline__ bool quarter_meet(uint64_t* bar, uint32_t parity, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
}

template <int D>
__global__ void __launch_bounds__(kTileThreads, 1)
    prefill_tile_kernel(Shape s, PrefillTileArgs a) {
  static_assert(kRowWarps == 16, "4 row warps per lane quarter");
  constexpr uint32_t KB = 64 * D * 2;  // bytes of a block's K (= of its V^T)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int G = s.G;
  const TileSmem L{D, a.nblk};
  uint8_t* Qt = sm + L.qt();
  uint8_t* kstage = sm + L.kst();
  uint8_t* vstage = sm + L.vst();
  float* mx_s = reinterpret_cast<float*>(sm + L.mx());
  uint32_t* mask_s = reinterpret_cast<uint32_t*>(sm + L.mask());
  int32_t* list_s = reinterpret_cast<int32_t*>(sm + L.list());
  __shared__ __align__(8) uint64_t kfull[kPairStages], kempty[kPairStages], vfull[kPairStages],
      vempty[kPairStages], s_full[2], p_full, pv_done;
  __shared__ __align__(8) uint64_t xch[4][3];  // per row quarter: the max of even / odd pairs, the row sum
  __shared__ uint32_t tmem_base;
  __shared__ int s_cnt;
  __shared__ volatile int s_bad;

  const int b = blockIdx.x, u = a.unit_base + blockIdx.y, tile = blockIdx.z;
  const int req = u / s.Hkv, h = u % s.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npos = min(s.B, a.L - b * s.B);
  const int p_lo = tile * 128 / G, p_hi = min(npos, p_lo + 128 / G);  // this tile's positions
  const long long ublk0 = (long long)u * a.nblk;  // unit index of this unit's block 0
  const long long payload = s.payload;
  const size_t kstride = pair_kstage(D), vstride = pair_vstage(D);
  const uint8_t* usrc = a.units + ublk0 * payload;
  const int mma_warp = kRowWarps, copy_warp = kRowWarps + 1;

  if (tid == 0) {
    for (int i = 0; i < kPairStages; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&p_full, kRowWarps);
    mbar_init(&pv_done, 1);
    for (int q = 0; q < 4; ++q)
      for (int k = 0; k < 3; ++k) mbar_init(&xch[q][k], 4);
    fence_mbar_init();
    s_bad = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_base, a.tmem_cols);
  for (int i = tid; i < 2 * (b + 1); i += kTileThreads) mask_s[i] = 0u;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  // ---- union of this tile's positions' selections --------------------------
  const int np = max(p_hi - p_lo, 0);
  for (int i = tid; i < np * s.k; i += kTileThreads) {
    const int p = p_lo + i / s.k, j = i % s.k;
    const long long vu = ((long long)req * a.L + (long long)b * s.B + p) * s.Hkv + h;
    const int32_t id = a.tab[vu * s.k + j];
    if (id < 0) continue;
    const long long blk = id - ublk0;
    if (blk < 0 || blk >= b) {
      atomicExch(a.err, kDevErrBadIndex);
      continue;
    }
    atomicOr(&mask_s[2 * blk + (p >> 5)], 1u << (p & 31));
  }
  if (tid < 2) {  // the own block holds every position of the tile
    uint32_t w = 0u;
    for (int p = 32 * tid; p < 32 * tid + 32; ++p)
      if (p >= p_lo && p < p_hi) w |= 1u << (p & 31);
    mask_s[2 * b + tid] = w;
  }
  __syncthreads();
  if (warp == 0) {  // blocks with a nonzero mask, ascending
    int run = 0;
    for (int base = 0; base <= b; base += 32) {
      const int j = base + lane;
      const bool on = (j <= b) && ((mask_s[2 * j] | mask_s[2 * j + 1]) != 0u);
      const unsigned bal = __ballot_sync(0xffffffffu, on);
      if (on) list_s[run + __popc(bal & ((1u << lane) - 1u))] = j;
      run += __popc(bal);
    }
    if (lane == 0) s_cnt = run;
  }
  __syncthreads();
  const int cnt = s_cnt;             // (0 only for a tile without positions)
  const int npair = (cnt + 1) >> 1;  // pair j: list entries 2j and 2j + 1 (if any)

  // ---- Q tile: row rr = position (p_lo + rr / G) x head (rr % G); rows past the block are 0
  if (warp < kRowWarps) {
    for (int i = tid; i < 128 * (D / 8); i += 32 * kRowWarps) {
      const int rr = i % 128, c = i / 128;
      const int p = p_lo + rr / G, g = rr % G;
      int4 v = make_int4(0, 0, 0, 0);
      if (p < p_hi) {
        const long long t = (long long)b * s.B + p;
        v = *reinterpret_cast<const int4*>(
            reinterpret_cast<const __nv_bfloat16*>(a.q) +
            (((long long)req * a.L + t) * s.Hq + (long long)h * G + g) * D + c * 8);
      }
      *reinterpret_cast<int4*>(Qt + (size_t)(c >> 3) * 16384 + rr * 128 + (((c & 7) ^ (rr & 7)) << 4)) = v;
    }
    fence_proxy_async();
  }
  __syncthreads();

  const uint32_t o_col = 256;  // O after the two S buffers (128 columns each)

  if (warp == copy_warp) {
    // ======================= bulk copies (one thread) ===========================
    // K of pair j once S of pair j - 2 is done, V^T and e once its P V is done
    if (lane == 0) {
      bool ok = true;
      int kissued = 0, vissued = 0;
      for (int j = 0; j < npair && ok; ++j) {
        const int st = j % kPairStages;
        const uint32_t par = (uint32_t)(((j - kPairStages) / kPairStages) & 1);
        const int nb = min(2, cnt - 2 * j);
        if (j >= kPairStages && !(ok = mbar_wait_bounded(&kempty[st], par))) break;
        uint8_t* kd = kstage + (size_t)st * kstride;
        mbar_arrive_expect_tx(&kfull[st], (uint32_t)(nb * KB));
        for (int hb = 0; hb < nb; ++hb) {
          const uint8_t* src = usrc + (long long)list_s[2 * j + hb] * payload;
#pragma unroll
          for (int kb = 0; kb < D / 64; ++kb) bulk_g2s(kd + kb * 16384 + hb * 8192, src + kb * 8192, 8192u, &kfull[st]);
        }
        ++kissued;
        if (j >= kPairStages && !(ok = mbar_wait_bounded(&vempty[st], par))) break;
        uint8_t* vd = vstage + (size_t)st * vstride;
        mbar_arrive_expect_tx(&vfull[st], (uint32_t)(nb * (KB + 256)));
        for (int hb = 0; hb < nb; ++hb) {  // V^T and e are contiguous in the unit: one copy
          const uint8_t* src = usrc + (long long)list_s[2 * j + hb] * payload;
          bulk_g2s(vd + hb * pair_vslot(D), src + KB, KB + 256u, &vfull[st]);
        }
        ++vissued;
      }
      if (!ok) {
        s_bad = 1;
        atomicExch(a.err, kDevErrWaitTimeout);
        // the copies in flight land before the CTA ends
        for (int j = max(kissued - kPairStages, 0); j < kissued; ++j)
          mbar_wait_bounded(&kfull[j % kPairStages], (uint32_t)((j / kPairStages) & 1));
        for (int j = max(vissued - kPairStages, 0); j < vissued; ++j)
          mbar_wait_bounded(&vfull[j % kPairStages], (uint32_t)((j / kPairStages) & 1));
      }
    }
  } else if (warp == mma_warp) {
    // ======================= MMA issue (one thread) =============================
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_f16(128, D);
      const uint64_t dq = sw128_desc(smem_u32(Qt));
      const uint64_t dkst = sw128_desc(smem_u32(kstage));
      const uint64_t dvst = sw128_desc(smem_u32(vstage));
      const uint32_t kstride16 = (uint32_t)(kstride >> 4), vstride16 = (uint32_t)(vstride >> 4);
      bool ok = true;
      int s_issued = 0, pv_issued = 0;
      auto issue_s = [&](int j) {  // S(j) = Q K_pair(j)^T into S buffer j & 1
        const int st = j % kPairStages;
        if (!mbar_wait_bounded(&kfull[st], (uint32_t)((j / kPairStages) & 1))) return false;
        tc_fence_after();
        const int nb = min(2, cnt - 2 * j);
        const uint32_t idesc_s = idesc_bf16(128, 64 * nb);
        const uint64_t dk = dkst + (uint64_t)(st * kstride16);
        const uint32_t t_d = tmem + (uint32_t)((j & 1) * 128);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)  // K16 step kk: 64-wide block kk / 4, +32 bytes each
          mma_bf16(t_d, dq + (kk >> 2) * 16384 / 16 + 2 * (kk & 3), dk + (kk >> 2) * 16384 / 16 + 2 * (kk & 3),
                   idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(&s_full[j & 1]);
        mma_commit(&kempty[st]);  // the pair's K stage may be refilled once S is done
        ++s_issued;
        return true;
      };
      if (npair > 0) ok = issue_s(0);
      if (ok && npair > 1) ok = issue_s(1);
      for (int j = 0; j < npair && ok; ++j) {
        // the rows wrote P(j) (and are done with S buffer j & 1); V^T of the pair landed
        if (!(ok = mbar_wait_bounded(&p_full, (uint32_t)(j & 1)))) break;
        if (!(ok = mbar_wait_bounded(&vfull[j % kPairStages], (uint32_t)((j / kPairStages) & 1)))) break;
        tc_fence_after();
        const int nb = min(2, cnt - 2 * j);
        const uint64_t dv = dvst + (uint64_t)((j % kPairStages) * vstride16);
        const uint32_t t_p = tmem + (uint32_t)((j & 1) * 128);
        for (int kk = 0; kk < 4 * nb; ++kk)  // 16 tokens: block kk / 4, half (kk / 2) % 2 of it
          mma_tmem_a(tmem + o_col, t_p + (kk >> 2) * 64 + ((kk >> 1) & 1) * 32 + (kk & 1) * 8,
                     dv + (uint64_t)((kk >> 2) * (pair_vslot(D) / 16)) + 2 * (kk & 3), idesc_pv,
                     (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&pv_done);
        mma_commit(&vempty[j % kPairStages]);  // the pair's V stage may be refilled
        ++pv_issued;
        // P V(j) done: its P columns may take S(j + 2)
        if (!(ok = mbar_wait_bounded(&pv_done, (uint32_t)(j & 1)))) break;
        if (j + 2 < npair && !(ok = issue_s(j + 2))) break;
      }
      if (!ok) {
        s_bad = 1;
        atomicExch(a.err, kDevErrWaitTimeout);
        // let the MMAs in flight finish before the memory goes away
        if (s_issued > 0) mbar_wait_bounded(&s_full[(s_issued - 1) & 1], (uint32_t)(((s_issued - 1) >> 1) & 1));
        if (pv_issued > 0) mbar_wait_bounded(&pv_done, (uint32_t)((pv_issued - 1) & 1));
      }
    }
  } else {
    // ======================= rows: softmax, P, O rescale ========================
    // warp (q4, hb, hh): lane quarter q4, block hb of the pair, its token half hh
    const int q4 = warp & 3, hb = (warp >> 2) & 1, hh = warp >> 3, wq = warp >> 2;  // wq: warp in the quarter
    const int rr = 32 * q4 + lane;
    const int p_loc = p_lo + rr / G;
    const bool row_valid = p_loc < p_hi;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const uint32_t t_o = tmem + lane_off + o_col + (uint32_t)(wq * (D / 4));  // this warp's quarter of O
    const float qs = 1.4426950408889634f * a.inv_sqrt_d;
    float m_run = -1e30f, l_run = 0.f;  // l: this warp's tokens only
    bool ok = true;
    for (int j = 0; j < npair; ++j) {
      const int st = j % kPairStages;
      const uint8_t* pvs = vstage + (size_t)st * vstride;
      ok = mbar_wait_bounded(&vfull[st], (uint32_t)((j / kPairStages) & 1)) &&
           mbar_wait_bounded(&s_full[j & 1], (uint32_t)((j >> 1) & 1));
      if (__any_sync(0xffffffffu, !ok || s_bad)) {  // warp-uniform
        ok = false;
        break;
      }
      tc_fence_after();
      const int nb = min(2, cnt - 2 * j);
      const bool mine = hb < nb;  // (warp-uniform)
      // this warp's 32 S columns (tokens 32 hh .. of block hb)
      const uint32_t t_s = tmem + lane_off + (uint32_t)((j & 1) * 128 + hb * 64 + hh * 32);
      float x[32];
      float mx = -INFINITY;
      if (mine) {
        const int jb = list_s[2 * j + hb];
        const uint32_t mb = row_valid ? mask_s[2 * jb + (p_loc >> 5)] : 0u;
        // positions of the half this row attends: t < lim (token index inside the half)
        const int lim = ((mb >> (p_loc & 31)) & 1u) ? ((jb == b) ? p_loc - 32 * hh : s.B) : -1;
        uint32_t sr[32];
        tmem_ld16_nowait(t_s, sr);
        tmem_ld16_nowait(t_s + 16, sr + 16);
        tmem_wait_ld();
        const float4* ev4 = reinterpret_cast<const float4*>(pvs + hb * pair_vslot(D) + KB) + 8 * hh;
        if (__all_sync(0xffffffffu, lim >= 32)) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 e4 = ev4[c];
            x[4 * c + 0] = fmaf(__uint_as_float(sr[4 * c + 0]), qs, e4.x);
            x[4 * c + 1] = fmaf(__uint_as_float(sr[4 * c + 1]), qs, e4.y);
            x[4 * c + 2] = fmaf(__uint_as_float(sr[4 * c + 2]), qs, e4.z);
            x[4 * c + 3] = fmaf(__uint_as_float(sr[4 * c + 3]), qs, e4.w);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 e4 = ev4[c];
            x[4 * c + 0] = 4 * c + 0 <= lim ? fmaf(__uint_as_float(sr[4 * c + 0]), qs, e4.x) : -INFINITY;
            x[4 * c + 1] = 4 * c + 1 <= lim ? fmaf(__uint_as_float(sr[4 * c + 1]), qs, e4.y) : -INFINITY;
            x[4 * c + 2] = 4 * c + 2 <= lim ? fmaf(__uint_as_float(sr[4 * c + 2]), qs, e4.z) : -INFINITY;
            x[4 * c + 3] = 4 * c + 3 <= lim ? fmaf(__uint_as_float(sr[4 * c + 3]), qs, e4.w) : -INFINITY;
          }
        }
        float mx4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
        for (int t = 4; t < 32; t += 4) {
          mx4[0] = fmaxf(mx4[0], x[t]);
          mx4[1] = fmaxf(mx4[1], x[t + 1]);
          mx4[2] = fmaxf(mx4[2], x[t + 2]);
          mx4[3] = fmaxf(mx4[3], x[t + 3]);
        }
        mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      }
      // the row's max over the pair: exchange among the 4 warps of the quarter
      float* mxb = mx_s + (size_t)(j & 1) * 512;
      mxb[wq * 128 + rr] = mx;
      if (!quarter_meet(&xch[q4][j & 1], (uint32_t)((j >> 1) & 1), lane)) {
        ok = false;
        break;
      }
      const float mxp = fmaxf(fmaxf(mxb[rr], mxb[128 + rr]), fmaxf(mxb[256 + rr], mxb[384 + rr]));
      // lazy reference: move it (every row of the warp) only when a row's max
      // rises by more than kRescale; the 4 warps of the quarter decide alike
      const bool grow = __any_sync(0xffffffffu, mxp > m_run + kRescale);
      const float m_use = grow ? fmaxf(m_run, mxp) : m_run;
      const float alpha = ex2(m_run - m_use);
      if (mine) {
        float sum4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pw[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          const float p0 = ex2(x[t] - m_use), p1 = ex2(x[t + 1] - m_use);
          sum4[(t >> 1) & 3] += p0 + p1;
          pw[t >> 1] = pack_f16(p0, p1);
        }
        l_run = l_run * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
        // P over the first 16 of this warp's S columns (already in registers)
        tmem_st16(t_s, reinterpret_cast<const float*>(pw));
      } else {
        l_run *= alpha;
      }
      m_run = m_use;
      // P V of the previous pair done: O is settled. Every row warp observes every
      // phase of pv_done in order (a parity wait cannot tell a phase from the one
      // two later). A new reference scales O by alpha before P V of this pair adds
      // to it (grow is warp-uniform; each warp of the quarter takes a quarter of O).
      if (j > 0) {
        ok = mbar_wait_bounded(&pv_done, (uint32_t)((j - 1) & 1));
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (grow) {
#pragma unroll 1
          for (int c0 = 0; c0 < D / 4; c0 += 16) {
            float v[16];
            tmem_ld16(t_o + c0, v);
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] *= alpha;
            tmem_st16(t_o + c0, v);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full);
    }
    if (!ok) {
      if (lane == 0) {
        s_bad = 1;
        atomicExch(a.err, kDevErrWaitTimeout);
      }
    }
    // the row sum: the 4 warps' parts (same reference)
    float* lsb = mx_s + 1024;
    lsb[wq * 128 + rr] = l_run;
    if (ok && !quarter_meet(&xch[q4][2], 0u, lane)) ok = false;
    const float l_tot = (lsb[rr] + lsb[128 + rr]) + (lsb[256 + rr] + lsb[384 + rr]);
    if (ok && npair > 0 &&
        __all_sync(0xffffffffu, mbar_wait_bounded(&pv_done, (uint32_t)((npair - 1) & 1)))) {
      tc_fence_after();
      const int g = rr % G;
      const long long t = (long long)b * s.B + p_loc;
      const long long row = ((long long)req * a.L + t) * s.Hq + (long long)h * G + g;
      // O carries V's scale 2^vs
      const float inv = l_tot > 0.f ? ldexpf(1.f, -v_scale_exp(*a.vmax)) / l_tot : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + row * D + wq * (D / 4));
#pragma unroll
      for (int c0 = 0; c0 < D / 4; c0 += 16) {
        float v[16];
        tmem_ld16(t_o + c0, v);
        if (row_valid) {
          dst[c0 / 8] = make_uint4(pack_bf16(v[0] * inv, v[1] * inv), pack_bf16(v[2] * inv, v[3] * inv),
                                   pack_bf16(v[4] * inv, v[5] * inv), pack_bf16(v[6] * inv, v[7] * inv));
          dst[c0 / 8 + 1] =
              make_uint4(pack_bf16(v[8] * inv, v[9] * inv), pack_bf16(v[10] * inv, v[11] * inv),
                         pack_bf16(v[12] * inv, v[13] * inv), pack_bf16(v[14] * inv, v[15] * inv));
        }
      }
      if (row_valid && wq == 0 && a.lse) a.lse[row] = l_tot > 0.f ? (m_run + log2f(l_tot)) * kLn2F : -INFINITY;
    } else if (ok && npair > 0 && lane == 0) {
      s_bad = 1;
      atomicExch(a.err, kDevErrWaitTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, a.tmem_cols);
  }
}

int tile_mt(const Shape& s) { return (s.B * s.G + 127) / 128; }
int tile_tmem_cols(const Shape& s) {
  const int need = 256 + s.d;  // two S buffers of a pair (128 columns each) and O
  int c = 32;
  while (c < need) c <<= 1;
  return c;
}
size_t tile_smem(const Shape& s, int nblk) { return TileSmem{s.d, nblk}.total(); }

}  // namespace

bool prefill_tiled_ok(const Shape& s, int L) {
  const char* env = std::getenv("NOSA_PREFILL_TILED");
  if (env && std::strcmp(env, "0") == 0) return false;
  if (s.dtype != 1 || s.B != 64 || (s.d != 64 && s.d != 128)) return false;
  if (s.G != 1 && s.G != 2 && s.G != 4) return false;
  const int nblk = (L + s.B - 1) / s.B;
  return tile_smem(s, nblk) <= 227 * 1024 - 1024;  // below the opt-in limit minus static
}

cudaError_t launch_prefill_tile(const Shape& s, int L, const uint8_t* units, const int32_t* tab,
                                const uint32_t* vmax, const void* q, void* out, float* lse,
                                int* err, cudaStream_t stream) {
  PrefillTileArgs a;
  a.units = units;
  a.tab = tab;
  a.vmax = vmax;
  a.q = q;
  a.out = out;
  a.lse = lse;
  a.err = err;
  a.L = L;
  a.nblk = (L + s.B - 1) / s.B;
  a.mt = tile_mt(s);
  a.tmem_cols = tile_tmem_cols(s);
  a.inv_sqrt_d = (float)(1.0 / std::sqrt((double)s.d));
  const void* fn = s.d == 64 ? (const void*)prefill_tile_kernel<64> : (const void*)prefill_tile_kernel<128>;
  static std::atomic<int> lim[2][64];
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  const size_t cap = (size_t)optin - fa.sharedSizeBytes;  // dynamic shared memory a CTA may have
  size_t smem = tile_smem(s, a.nblk);
  if (smem > cap) return cudaErrorInvalidConfiguration;
  e = raise_smem_limit(fn, cap, lim[s.d == 64 ? 0 : 1]);
  if (e != cudaSuccess) return e;
  // CTAs resident on an SM must not ask for more than its 512 tensor-memory
  // columns together (an allocation would wait for another CTA's release):
  // extra shared memory keeps their number down where needed.
  const int max_ctas = 512 / a.tmem_cols;
  for (int guard = 0; guard < 64; ++guard) {
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kTileThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ <= max_ctas || smem + 4096 > cap) break;
    smem += 4096;
  }
  for (int base = 0; base < s.U; base += 65535) {
    a.unit_base = base;
    const dim3 grid(a.nblk, std::min(65535, s.U - base), a.mt);  // (query block, unit, M-tile)
    if (s.d == 64)
      prefill_tile_kernel<64><<<grid, kTileThreads, smem, stream>>>(s, a);
    else
      prefill_tile_kernel<128><<<grid, kTileThreads, smem, stream>>>(s, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace nosa
