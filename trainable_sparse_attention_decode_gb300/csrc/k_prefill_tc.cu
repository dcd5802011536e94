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
//   per block S = Q K^T on the tensor cores (tcgen05.mma kind::f16, bf16 in,
//             fp32 accumulator in tensor memory, M = 128, N = 64, K = d); each
//             row: logits = S log2(e)/sqrt(d) + e_j log2(e), -inf where the row's
//             position did not select the block (in the own block also past the
//             position), online softmax in fp32 (the row's sum l and so the
//             log-sum-exp in fp32), P rounded to bf16 into shared memory as the
//             operand of P V on the tensor cores (M = 128,
//             N = d, K = 64) into tensor memory; every row folds it into its
//             fp32 output in registers: O = O alpha + P V.
// Operands are K-major without swizzle (8-row x 16-byte core matrices): K as the
// decode layout stores it, V transposed by the pack kernel, Q and P written in
// that form here; a block unit arrives by one bulk copy (two in flight) and the
// MMAs read it where it lands. Every mbarrier wait is bounded; a wait that gives
// up sets the error word and the CTA drains its copies and frees its tensor
// memory before it exits.
#include "nosa_internal.cuh"
#include "tcgen05.cuh"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>

namespace nosa {
namespace {
using namespace tc;

constexpr int kTileThreads = 256;
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;

// Shared-memory carve-up of one CTA (offsets from a 128-byte aligned base).
struct TileSmem {
  int mt, d, nblk;
  long long payload;
  __host__ __device__ size_t qt() const { return 0; }                               // [mt][128 x d] bf16
  __host__ __device__ size_t pt() const { return (size_t)mt * 256 * d; }            // [mt][128 x 64] bf16
  __host__ __device__ size_t stage() const { return pt() + (size_t)mt * 16384; }    // [2][payload]
  __host__ __device__ size_t mask() const { return stage() + 2 * (size_t)payload; } // [nblk][2] u32
  __host__ __device__ size_t list() const { return mask() + 8 * (size_t)nblk; }     // [nblk] i32
  __host__ __device__ size_t total() const { return list() + 4 * (size_t)nblk + 128; }
};

template <int D>
__global__ void __launch_bounds__(kTileThreads, D == 64 ? 2 : 1)
    prefill_tile_kernel(Shape s, PrefillTileArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                           ~uintptr_t(127));
  const int mt = a.mt, G = s.G;
  const TileSmem L{mt, D, a.nblk, s.payload};
  uint8_t* Qt = sm + L.qt();
  uint8_t* Pt = sm + L.pt();
  uint8_t* stage = sm + L.stage();
  uint32_t* mask_s = reinterpret_cast<uint32_t*>(sm + L.mask());
  int32_t* list_s = reinterpret_cast<int32_t*>(sm + L.list());
  __shared__ __align__(8) uint64_t full[2], mma_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int s_cnt;
  __shared__ volatile int s_bad;

  const int b = blockIdx.x, u = a.unit_base + blockIdx.y;
  const int req = u / s.Hkv, h = u % s.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npos = min(s.B, a.L - b * s.B);
  const long long ublk0 = (long long)u * a.nblk;  // unit index of this unit's block 0
  const long long payload = s.payload;
  const uint8_t* usrc = a.units + ublk0 * payload;

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&mma_bar, 1);
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
  const int cnt = s_cnt;

  int issued = 0;  // copies issued (thread 0)
  if (tid == 0) {
    for (; issued < 2 && issued < cnt; ++issued) {
      mbar_arrive_expect_tx(&full[issued], (uint32_t)payload);
      bulk_g2s(stage + (size_t)issued * payload, usrc + (long long)list_s[issued] * payload,
               (uint32_t)payload, &full[issued]);
    }
  }
  // ---- Q tiles: row r = position (r / G) x head (r % G); rows past the block are 0
  for (int i = tid; i < mt * 128 * (D / 8); i += kTileThreads) {
    const int r = i % (mt * 128), c = i / (mt * 128);
    const int p = r / G, g = r - p * G;
    int4 v = make_int4(0, 0, 0, 0);
    if (p < npos) {
      const long long t = (long long)b * s.B + p;
      v = *reinterpret_cast<const int4*>(
          reinterpret_cast<const __nv_bfloat16*>(a.q) +
          (((long long)req * a.L + t) * s.Hq + (long long)h * G + g) * D + c * 8);
    }
    *reinterpret_cast<int4*>(Qt + (size_t)(r >> 7) * 256 * D + (size_t)c * 2048 + (r & 127) * 16) = v;
  }
  fence_proxy_async();

  // this thread's row (warps 0 .. 4 mt - 1; warp w reads tensor-memory lanes 32 (w % 4) ..)
  const bool has_row = warp < 4 * mt;
  const int m = warp >> 2, rr = 32 * (warp & 3) + lane, r = m * 128 + rr;
  const int p_loc = r / G;
  const bool row_valid = p_loc < npos;
  float m_run = -1e30f, l_run = 0.f;
  float o[D];
#pragma unroll
  for (int i = 0; i < D; ++i) o[i] = 0.f;
  const float qs = kLog2eF * a.inv_sqrt_d;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  const uint32_t t_s = tmem + lane_off + (uint32_t)(m * 64);
  const uint32_t t_pv = tmem + lane_off + (uint32_t)(mt * 64 + m * D);
  constexpr uint32_t idesc_s = idesc_bf16(128, 64);
  constexpr uint32_t idesc_pv = idesc_bf16(128, D);
  const uint32_t kbytes = (uint32_t)(s.B * D * 2);
  __syncthreads();

  for (int i = 0; i < cnt; ++i) {
    const int st = i & 1;
    uint8_t* unit = stage + (size_t)st * payload;
    if (!mbar_wait_bounded(&full[st], (uint32_t)((i >> 1) & 1)) && lane == 0) {
      s_bad = 1;
      atomicExch(a.err, kDevErrWaitTimeout);
    }
    __syncthreads();
    if (s_bad) break;
    const int jb = list_s[i];
    // S = Q K^T (K: token groups 128 bytes apart, dim chunks B * 16 bytes apart)
    if (tid == 0) {
      tc_fence_after();
      for (int mm = 0; mm < mt; ++mm)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t da = kmajor_desc(smem_u32(Qt + (size_t)mm * 256 * D + kk * 4096), 2048, 128);
          const uint64_t db = kmajor_desc(smem_u32(unit + kk * 2 * s.B * 16), s.B * 16, 128);
          mma_bf16(tmem + (uint32_t)(mm * 64), da, db, idesc_s, kk > 0 ? 1u : 0u);
        }
      mma_commit(&mma_bar);
    }
    if (!mbar_wait_bounded(&mma_bar, 0u) && lane == 0) {
      s_bad = 1;
      atomicExch(a.err, kDevErrWaitTimeout);
    }
    tc_fence_after();
    float alpha = 1.f;
    if (has_row) {
      const float* ev = reinterpret_cast<const float*>(unit + 2 * (size_t)kbytes);
      const uint32_t mb = row_valid ? mask_s[2 * jb + (p_loc >> 5)] : 0u;
      const bool row_on = (mb >> (p_loc & 31)) & 1u;
      const int tmax = (jb == b) ? p_loc : s.B - 1;  // own block: causal
      float mx = -INFINITY;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16) {
        float v[16];
        tmem_ld16(t_s + c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = c0 + j;
          const float x = (row_on && t <= tmax) ? fmaf(v[j], qs, ev[t] * kLog2eF) : -INFINITY;
          mx = fmaxf(mx, x);
        }
      }
      const float mn = fmaxf(m_run, mx);
      alpha = exp2f(m_run - mn);
      float sum = 0.f;
      uint8_t* prow = Pt + (size_t)m * 16384 + rr * 16;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16) {
        float v[16];
        tmem_ld16(t_s + c0, v);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const int t = c0 + j;
          const float x0 = (row_on && t <= tmax) ? fmaf(v[j], qs, ev[t] * kLog2eF) : -INFINITY;
          const float x1 = (row_on && t + 1 <= tmax) ? fmaf(v[j + 1], qs, ev[t + 1] * kLog2eF) : -INFINITY;
          const float p0 = exp2f(x0 - mn), p1 = exp2f(x1 - mn);
          sum += p0 + p1;
          const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
          w[j >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
        }
        *reinterpret_cast<uint4*>(prow + (c0 / 8) * 2048) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(prow + (c0 / 8 + 1) * 2048) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      l_run = l_run * alpha + sum;
      m_run = mn;
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (s_bad) break;
    // P V (V^T: dim groups 128 bytes apart, token chunks d * 16 bytes apart)
    if (tid == 0) {
      tc_fence_after();
      for (int mm = 0; mm < mt; ++mm)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t da = kmajor_desc(smem_u32(Pt + (size_t)mm * 16384 + kk * 4096), 2048, 128);
          const uint64_t db = kmajor_desc(smem_u32(unit + kbytes + kk * 2 * D * 16), D * 16, 128);
          mma_bf16(tmem + (uint32_t)(mt * 64 + mm * D), da, db, idesc_pv, kk > 0 ? 1u : 0u);
        }
      mma_commit(&mma_bar);
    }
    const bool ok_pv = mbar_wait_bounded(&mma_bar, 1u);
    if (!ok_pv && lane == 0) {
      s_bad = 1;
      atomicExch(a.err, kDevErrWaitTimeout);
    }
    tc_fence_after();
    // the stage is free again: the block two ahead goes into it
    if (tid == 0 && ok_pv && issued < cnt) {
      mbar_arrive_expect_tx(&full[st], (uint32_t)payload);
      bulk_g2s(unit, usrc + (long long)list_s[issued] * payload, (uint32_t)payload, &full[st]);
      ++issued;
    }
    if (has_row) {
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 16) {
        float pv[16];
        tmem_ld16(t_pv + c0, pv);
#pragma unroll
        for (int j = 0; j < 16; ++j) o[c0 + j] = fmaf(o[c0 + j], alpha, pv[j]);
      }
    }
    // every thread has seen both phases of mma_bar before the next commit
    tc_fence_before();
    __syncthreads();
    if (s_bad) break;
  }

  if (has_row && row_valid && !s_bad) {
    const int g = r - p_loc * G;
    const long long t = (long long)b * s.B + p_loc;
    const long long row = ((long long)req * a.L + t) * s.Hq + (long long)h * G + g;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + row * D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 x = __floats2bfloat162_rn(o[c * 8 + 2 * e] * inv, o[c * 8 + 2 * e + 1] * inv);
        w[e] = *reinterpret_cast<const uint32_t*>(&x);
      }
      dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (a.lse) a.lse[row] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2F : -INFINITY;
  }
  __syncthreads();
  if (s_bad && tid == 0) {  // drain the copies still in flight (bounded)
    for (int j = max(issued - 2, 0); j < issued; ++j)
      mbar_wait_bounded(&full[j & 1], (uint32_t)((j >> 1) & 1));
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
  const int need = tile_mt(s) * (64 + s.d);
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
                                const void* q, void* out, float* lse, int* err,
                                cudaStream_t stream) {
  PrefillTileArgs a;
  a.units = units;
  a.tab = tab;
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
  static std::atomic<int> lim64[64], lim128[64];
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  const size_t cap = (size_t)optin - fa.sharedSizeBytes;  // dynamic shared memory a CTA may have
  size_t smem = tile_smem(s, a.nblk);
  if (smem > cap) return cudaErrorInvalidConfiguration;
  e = raise_smem_limit(fn, cap, s.d == 64 ? lim64 : lim128);
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
