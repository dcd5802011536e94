// Training-time forward: block-sparse attention tiled by query block, on the
// tensor cores.
//
// NOSA technical summary, Methodology §1 (the dual selection at every query
// position during training) and §2 (ED-DMA: the eviction logit enters the
// attention logits before the exponential). The 64 positions of a query block
// share Gamma_e (E_b) and their own block (the causal tail), and neighbouring
// positions pick mostly the same query-aware blocks, so one CTA per (unit, query
// block) streams the union of its positions' blocks once and lets every position
// that selected a block use it:
//   rows      the block's 64 positions x G query heads (row = position x G +
//             head), in M-tiles of 128 rows (G <= 4: one or two tiles);
//   union     built from the positions' block tables: per block a 64-bit mask of
//             the positions that selected it (the own block: every position);
//   per block S = Q K^T on the tensor cores (tcgen05.mma kind::f16, bf16 in, fp32
//             accumulator in tensor memory, M = 128, N = 64, K = d); each row:
//             logits = S log2(e)/sqrt(d) + e_j log2(e), -inf where the row's
//             position did not select the block (in the own block also past the
//             position); P = exp2(logit - m) in fp16 written over the S columns it
//             came from; O += P V on the tensor cores with P read from tensor
//             memory (fp16 in: V converted exactly with one power-of-two scale of
//             the call; M = 128, N = d, K = 64), O in tensor memory.
// Online softmax with a lazy reference: a row keeps its running max m until a
// block raises it by more than 8 (base 2), so P <= 2^8; only then is the row's O
// rescaled in tensor memory (and its sum l in fp32). The sum l adds the fp32
// probabilities, so the log-sum-exp is exact to fp32 rounding.
// Warp roles: warps 0 .. 4 mt - 1 own one row each per thread (warp w reads
// tensor-memory lanes 32 (w % 4) ..), the last warp issues the MMAs and the bulk
// copies. S (then P) is double-buffered in tensor memory and the block units take
// three shared-memory stages, so S of block i + 1 and P V of block i - 1 run on
// the tensor cores while the rows work on block i; S of block i + 2 goes into
// block i's buffer only once P V of block i, which reads P from it, completed.
// Everything after the set-up is ordered by mbarriers:
//   full[st]   a block unit landed (bulk copy)       s_full[sb] S of a block is in
//   p_full     the rows wrote P (and rescaled O)      pv_done    P V completed
// Shared-memory operands are K-major with the 128-byte swizzle (rows of 128 bytes,
// 16-byte chunk c of row r at chunk c ^ (r % 8), 8-row groups 1024 bytes apart): K
// and V^T as the pack kernel lays out the units (stages 1024-byte aligned, so the
// MMAs read a unit where its bulk copy put it), Q written in that form here. Every wait is
// bounded; one that gives up sets the error word and the CTA stops, waits
// (bounded) for its copies and MMAs in flight and frees its tensor memory.
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

constexpr int kRowWarps = 8;                       // at most: 4 per M-tile
constexpr int kTileThreads = 32 * (kRowWarps + 1);  // + the MMA / copy warp
constexpr int kStages = 3;
constexpr float kLn2F = 0.6931471805599453f;
constexpr float kRescale = 8.0f;                   // lazy-rescale threshold (base 2)

// Shared-memory carve-up of one CTA (offsets from a 1024-byte aligned base).
struct TileSmem {
  int mt, d, nblk;
  long long payload;
  __host__ __device__ size_t sstride() const { return ((size_t)payload + 1023) & ~(size_t)1023; }
  __host__ __device__ size_t qt() const { return 0; }                                     // [mt][d/64][128 x 128 B] bf16
  __host__ __device__ size_t stage() const { return (size_t)mt * 256 * d; }               // [kStages][sstride]
  __host__ __device__ size_t mask() const { return stage() + kStages * sstride(); }       // [nblk][2] u32
  __host__ __device__ size_t list() const { return mask() + 8 * (size_t)nblk; }           // [nblk] i32
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

template <int D, int MT>
__global__ void __launch_bounds__(kTileThreads, 1)
    prefill_tile_kernel(Shape s, PrefillTileArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  constexpr int mt = MT;
  const int G = s.G;
  const TileSmem L{mt, D, a.nblk, s.payload};
  uint8_t* Qt = sm + L.qt();
  uint8_t* stage = sm + L.stage();
  uint32_t* mask_s = reinterpret_cast<uint32_t*>(sm + L.mask());
  int32_t* list_s = reinterpret_cast<int32_t*>(sm + L.list());
  __shared__ __align__(8) uint64_t full[kStages], s_full[2], p_full, pv_done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_cnt;
  __shared__ volatile int s_bad;

  const int b = blockIdx.x, u = a.unit_base + blockIdx.y;
  const int req = u / s.Hkv, h = u % s.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npos = min(s.B, a.L - b * s.B);
  const long long ublk0 = (long long)u * a.nblk;  // unit index of this unit's block 0
  const long long payload = s.payload;
  const size_t sstride = L.sstride();
  const uint8_t* usrc = a.units + ublk0 * payload;
  const int row_warps = 4 * mt;
  const int mma_warp = kRowWarps;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&p_full, row_warps);
    mbar_init(&pv_done, 1);
    fence_mbar_init();
    s_bad = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_base, a.tmem_cols);
  for (int i = tid; i < 2 * (b + 1); i += kTileThreads) mask_s[i] = 0u;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  // ---- union of the positions' selections --------------------------------
  for (int i = tid; i < npos * s.k; i += kTileThreads) {
    const int p = i / s.k, j = i - p * s.k;
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
  if (tid < 2) {  // the own block holds every valid position
    const int n = tid == 0 ? min(npos, 32) : max(npos - 32, 0);
    mask_s[2 * b + tid] = n >= 32 ? 0xffffffffu : ((1u << n) - 1u);
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
  const int cnt = s_cnt;  // >= 1 (the own block)

  int issued = 0;  // copies issued (MMA warp, lane 0)
  if (warp == mma_warp && lane == 0) {
    for (; issued < kStages && issued < cnt; ++issued) {
      mbar_arrive_expect_tx(&full[issued], (uint32_t)payload);
      bulk_g2s(stage + (size_t)issued * sstride, usrc + (long long)list_s[issued] * payload,
               (uint32_t)payload, &full[issued]);
    }
  }
  // ---- Q tiles: row r = position (r / G) x head (r % G); rows past the block are 0
  if (warp < mma_warp) {
    for (int i = tid; i < mt * 128 * (D / 8); i += 32 * kRowWarps) {
      const int r = i % (mt * 128), c = i / (mt * 128);
      const int p = r / G, g = r - p * G;
      int4 v = make_int4(0, 0, 0, 0);
      if (p < npos) {
        const long long t = (long long)b * s.B + p;
        v = *reinterpret_cast<const int4*>(
            reinterpret_cast<const __nv_bfloat16*>(a.q) +
            (((long long)req * a.L + t) * s.Hq + (long long)h * G + g) * D + c * 8);
      }
      const int rr = r & 127;
      *reinterpret_cast<int4*>(Qt + (size_t)(r >> 7) * 256 * D + (size_t)(c >> 3) * 16384 + rr * 128 +
                               (((c & 7) ^ (rr & 7)) << 4)) = v;
    }
    fence_proxy_async();
  }
  __syncthreads();

  constexpr uint32_t kbytes = (uint32_t)(64 * D * 2);
  const uint32_t o_col = (uint32_t)(2 * mt * 64);  // O tiles after the two S buffers

  if (warp == mma_warp) {
    // ======================= MMA and copy issue (one thread) ====================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 64);
      constexpr uint32_t idesc_pv = idesc_f16(128, D);
      // descriptor bases; a descriptor's start field counts 16-byte units and
      // stays below 2^14 for any shared-memory address, so offsets add directly
      const uint64_t dq = sw128_desc(smem_u32(Qt));
      const uint64_t dstage = sw128_desc(smem_u32(stage));
      const uint32_t sstride16 = (uint32_t)(sstride >> 4);
      bool ok = true;
      int s_issued = 0, pv_issued = 0;
      auto issue_s = [&](int j) {  // S_j = Q K_j^T into S buffer j & 1
        const int st = j % kStages;
        if (!mbar_wait_bounded(&full[st], (uint32_t)((j / kStages) & 1))) return false;
        tc_fence_after();
        const uint64_t dk = dstage + (uint64_t)(st * sstride16);
        const uint32_t t_d = tmem + (uint32_t)((j & 1) * mt * 64);
#pragma unroll
        for (int mm = 0; mm < mt; ++mm)
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)  // K16 step kk: 64-wide block kk / 4, +32 bytes each
            mma_bf16(t_d + mm * 64, dq + (mm * 256 * D + (kk >> 2) * 16384) / 16 + 2 * (kk & 3),
                     dk + (kk >> 2) * 8192 / 16 + 2 * (kk & 3), idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(&s_full[j & 1]);
        ++s_issued;
        return true;
      };
      ok = issue_s(0);
      if (ok && cnt > 1) ok = issue_s(1);
      for (int i = 0; i < cnt && ok; ++i) {
        // the rows wrote P_i (and are done with S buffer i & 1)
        if (!(ok = mbar_wait_bounded(&p_full, (uint32_t)(i & 1)))) break;
        tc_fence_after();
        // K steps outermost: the M-tiles' accumulations alternate (the tensor pipe
        // runs two independent accumulators back to back faster than one chain).
        // A = P of tile mm in S buffer i & 1 (8 columns per 16 tokens).
        const uint64_t dv = dstage + (uint64_t)((i % kStages) * sstride16) + kbytes / 16;
        const uint32_t t_p = tmem + (uint32_t)((i & 1) * mt * 64);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
          for (int mm = 0; mm < mt; ++mm)
            mma_tmem_a(tmem + o_col + mm * D, t_p + mm * 64 + kk * 8, dv + 2 * kk, idesc_pv,
                       (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&pv_done);
        ++pv_issued;
        // P V_i done: its stage is free and its P columns may take S_{i+2}
        if (!(ok = mbar_wait_bounded(&pv_done, (uint32_t)(i & 1)))) break;
        if (i + 2 < cnt && !(ok = issue_s(i + 2))) break;
        if (issued < cnt) {  // block i + kStages into block i's stage
          const int st = issued % kStages;
          mbar_arrive_expect_tx(&full[st], (uint32_t)payload);
          bulk_g2s(stage + (size_t)st * sstride, usrc + (long long)list_s[issued] * payload,
                   (uint32_t)payload, &full[st]);
          ++issued;
        }
      }
      if (!ok) {
        s_bad = 1;
        atomicExch(a.err, kDevErrWaitTimeout);
        // let the copies and MMAs in flight finish before the memory goes away
        for (int j = max(issued - kStages, 0); j < issued; ++j)
          mbar_wait_bounded(&full[j % kStages], (uint32_t)((j / kStages) & 1));
        if (s_issued > 0) mbar_wait_bounded(&s_full[(s_issued - 1) & 1], (uint32_t)(((s_issued - 1) >> 1) & 1));
        if (pv_issued > 0) mbar_wait_bounded(&pv_done, (uint32_t)((pv_issued - 1) & 1));
      }
    }
  } else if (warp < row_warps) {
    // ======================= rows: softmax, P, O rescale =======================
    const int m = warp >> 2, rr = 32 * (warp & 3) + lane, r = m * 128 + rr;
    const int p_loc = r / G;
    const bool row_valid = p_loc < npos;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t t_o = tmem + lane_off + o_col + (uint32_t)(m * D);
    const float qs = 1.4426950408889634f * a.inv_sqrt_d;
    float m_run = -1e30f, l_run = 0.f;
    bool ok = true;
    for (int i = 0; i < cnt; ++i) {
      const int sb = i & 1;
      const uint8_t* unit = stage + (size_t)(i % kStages) * sstride;
      ok = mbar_wait_bounded(&full[i % kStages], (uint32_t)((i / kStages) & 1)) &&
           mbar_wait_bounded(&s_full[sb], (uint32_t)((i >> 1) & 1));
      if (__any_sync(0xffffffffu, !ok || s_bad)) {  // warp-uniform
        ok = false;
        break;
      }
      tc_fence_after();
      const int jb = list_s[i];
      const uint32_t mb = row_valid ? mask_s[2 * jb + (p_loc >> 5)] : 0u;
      // positions of the block this row attends: t <= lim (-1: none)
      const int lim = ((mb >> (p_loc & 31)) & 1u) ? ((jb == b) ? p_loc : s.B - 1) : -1;
      uint32_t sr[64];
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16)
        tmem_ld16_nowait(tmem + lane_off + (uint32_t)(sb * mt * 64 + m * 64 + c0), sr + c0);
      tmem_wait_ld();
      const float4* ev4 = reinterpret_cast<const float4*>(unit + 2 * (size_t)kbytes);
      float x[64];
      if (__all_sync(0xffffffffu, lim == s.B - 1)) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 e4 = ev4[c];
          x[4 * c + 0] = fmaf(__uint_as_float(sr[4 * c + 0]), qs, e4.x);
          x[4 * c + 1] = fmaf(__uint_as_float(sr[4 * c + 1]), qs, e4.y);
          x[4 * c + 2] = fmaf(__uint_as_float(sr[4 * c + 2]), qs, e4.z);
          x[4 * c + 3] = fmaf(__uint_as_float(sr[4 * c + 3]), qs, e4.w);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 e4 = ev4[c];
          x[4 * c + 0] = 4 * c + 0 <= lim ? fmaf(__uint_as_float(sr[4 * c + 0]), qs, e4.x) : -INFINITY;
          x[4 * c + 1] = 4 * c + 1 <= lim ? fmaf(__uint_as_float(sr[4 * c + 1]), qs, e4.y) : -INFINITY;
          x[4 * c + 2] = 4 * c + 2 <= lim ? fmaf(__uint_as_float(sr[4 * c + 2]), qs, e4.z) : -INFINITY;
          x[4 * c + 3] = 4 * c + 3 <= lim ? fmaf(__uint_as_float(sr[4 * c + 3]), qs, e4.w) : -INFINITY;
        }
      }
      float mx4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
      for (int t = 4; t < 64; t += 4) {
        mx4[0] = fmaxf(mx4[0], x[t]);
        mx4[1] = fmaxf(mx4[1], x[t + 1]);
        mx4[2] = fmaxf(mx4[2], x[t + 2]);
        mx4[3] = fmaxf(mx4[3], x[t + 3]);
      }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      // lazy reference: move it (every row of the warp) only when a row's max
      // rises by more than kRescale
      const bool grow = __any_sync(0xffffffffu, mx > m_run + kRescale);
      const float m_use = grow ? fmaxf(m_run, mx) : m_run;
      const float alpha = ex2(m_run - m_use);
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pw[32];
#pragma unroll
      for (int t = 0; t < 64; t += 2) {
        const float p0 = ex2(x[t] - m_use), p1 = ex2(x[t + 1] - m_use);
        sum4[(t >> 1) & 3] += p0 + p1;
        pw[t >> 1] = pack_f16(p0, p1);
      }
      l_run = l_run * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
      m_run = m_use;
      // P V of the previous block done: O is settled. Every row warp observes
      // every phase of pv_done in order (a parity wait cannot tell a phase from
      // the one two later). A new reference scales O by alpha before P V of this
      // block adds to it (grow is warp-uniform).
      if (i > 0) {
        ok = mbar_wait_bounded(&pv_done, (uint32_t)((i - 1) & 1));
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (grow && i > 0) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
          float v[16];
          tmem_ld16(t_o + c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] *= alpha;
          tmem_st16(t_o + c0, v);
        }
      }
      // P over the first 32 columns of this row's S (already in registers)
      tmem_st32(tmem + lane_off + (uint32_t)(sb * mt * 64 + m * 64), pw);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full);
    }
    if (!ok) {
      if (lane == 0) {
        s_bad = 1;
        atomicExch(a.err, kDevErrWaitTimeout);
      }
    } else if (__all_sync(0xffffffffu, mbar_wait_bounded(&pv_done, (uint32_t)((cnt - 1) & 1)))) {
      tc_fence_after();
      const int g = r - p_loc * G;
      const long long t = (long long)b * s.B + p_loc;
      const long long row = ((long long)req * a.L + t) * s.Hq + (long long)h * G + g;
      // O carries V's scale 2^vs
      const float inv = l_run > 0.f ? ldexpf(1.f, -v_scale_exp(*a.vmax)) / l_run : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + row * D);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 16) {
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
      if (row_valid && a.lse) a.lse[row] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2F : -INFINITY;
    } else if (lane == 0) {
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
  const int need = tile_mt(s) * (2 * 64 + s.d);  // two S buffers and O
  int c = 32;
  while (c < need) c <<= 1;
  return c;
}
size_t tile_smem(const Shape& s, int nblk) {
  return TileSmem{tile_mt(s), s.d, nblk, s.payload}.total();
}

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
  const void* fn = s.d == 64 ? (a.mt == 1 ? (const void*)prefill_tile_kernel<64, 1> : (const void*)prefill_tile_kernel<64, 2>)
                              : (a.mt == 1 ? (const void*)prefill_tile_kernel<128, 1> : (const void*)prefill_tile_kernel<128, 2>);
  static std::atomic<int> lim[4][64];
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  const size_t cap = (size_t)optin - fa.sharedSizeBytes;  // dynamic shared memory a CTA may have
  size_t smem = tile_smem(s, a.nblk);
  if (smem > cap) return cudaErrorInvalidConfiguration;
  e = raise_smem_limit(fn, cap, lim[(s.d == 64 ? 0 : 2) + (a.mt - 1)]);
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
    const dim3 grid(a.nblk, std::min(65535, s.U - base));
    if (s.d == 64 && a.mt == 1)
      prefill_tile_kernel<64, 1><<<grid, kTileThreads, smem, stream>>>(s, a);
    else if (s.d == 64)
      prefill_tile_kernel<64, 2><<<grid, kTileThreads, smem, stream>>>(s, a);
    else if (a.mt == 1)
      prefill_tile_kernel<128, 1><<<grid, kTileThreads, smem, stream>>>(s, a);
    else
      prefill_tile_kernel<128, 2><<<grid, kTileThreads, smem, stream>>>(s, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace nosa
