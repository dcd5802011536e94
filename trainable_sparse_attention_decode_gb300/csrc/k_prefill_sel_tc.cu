// Training-time forward: the per-position selection with the pooled query scores
// on the tensor cores.
//
// NOSA technical summary, Methodology §1: at every query position t the query-aware
// part of the selection is the top-(k - |Gamma_e|) of the candidates outside
// Gamma_e by the two-stage pooled score sq(j) = max over sub-blocks s of
// q_bar(t) . K_bar[j][s] / sqrt(d). For the 64 positions of block b (which share
// E_b and the candidate list) the scores are one product Q_bar K_bar^T: 64
// positions x (4 sub-block rows per candidate) x d.
//
// The cut is decided in fp32 and the scores must keep fp32 accuracy, so each fp32
// operand x is split into three bf16 terms x1 + x2 + x3 (x1 = bf16(x), x2 =
// bf16(x - x1), x3 = bf16(x - x1 - x2): 24 significant bits, the split error at
// most about 2^-24 |x|) and the product is the six-term sum
//   a1 b1 + a1 b2 + a2 b1 + a1 b3 + a2 b2 + a3 b1
// (the three terms left out are below 2^-24 |a b|), accumulated in fp32 in tensor
// memory: the error of a score is that of an fp32 dot product. Non-finite inputs
// keep x1 = x and zero tails.
//
// prefill_keysplit_kernel  the three bf16 planes of the pooled keys of every
//                          chunk of 32 consecutive blocks, per 64-dim atom, laid
//                          out as the selection's shared-memory stage (128 rows:
//                          block 32 c + i, sub-block s at row 4 i + s, 128-byte
//                          swizzle), so one bulk copy per plane fills a stage
// prefill_select_tc_kernel one CTA per (unit, block), heaviest blocks first:
//   A     q_bar of the 64 positions, split in 3 planes, 128-byte-swizzled K-major
//         tiles of 64 rows (M = 128: rows 64-127 of a tile read the next tile or a
//         zero pad; their results are never read);
//   B     chunks of 32 consecutive blocks j < b (N = 128 rows), 64 dims per stage,
//         a ring of 3 stages filled by bulk copies (copy warp); the blocks of E_b
//         are scored too and left out in the epilogue;
//   MMA   per stage 4 K16 steps x 6 terms (tcgen05.mma kind::f16, bf16 in, fp32
//         accumulator), a chunk into one of two 128-column tensor-memory buffers;
//   rows  4 epilogue warps, two per lane quarter (position = tensor-memory lane),
//         one pair on the even chunks (buffer 0), one on the odd (buffer 1): the
//         max over each candidate's 4 columns times 1/sqrt(d) goes into the
//         thread's sorted register list of the best m (key descending, block id
//         ascending: the lower id first at equal scores; a NaN score and a block
//         of E_b never enter); at the end the even-chunk thread of a position
//         merges the two lists, sorts the winners by id and writes the position's
//         selection.
// Barriers: full / empty [stage] (copies landed / MMAs read the stage), mma_done
// [buffer] (a chunk's scores are in), tmem_free [buffer] (the epilogue warps read
// them). Every wait is bounded; one that gives up sets the error word, and the CTA
// waits (bounded) for its copies and MMAs in flight, writes nothing and frees its
// tensor memory.
#include "nosa_internal.cuh"
#include "tcgen05.cuh"

#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>

namespace nosa {
namespace {
using namespace tc;

constexpr int kStThreads = 256;                      // 8 warps
constexpr int kStCC = 32;                            // candidates per chunk (N = 128)
constexpr int kStStages = 3;                         // ring of 64-dim stages
constexpr uint32_t kStPlane = 16384;                 // one plane of a stage: 128 rows x 128 B
constexpr uint32_t kStStage = 3 * kStPlane;          // the three planes
constexpr int kStTmemCols = 256;                     // two 128-column score buffers
constexpr int kMmaWarp = 2, kCopyWarp = 3;           // epilogue: warps 0, 1 (even chunks), 4, 5 (odd)
// the six (A plane, B plane) products kept
__constant__ int kTermA[6] = {0, 0, 1, 0, 1, 2};
__constant__ int kTermB[6] = {0, 1, 0, 2, 1, 0};

// bytes of the split keys of one chunk of 32 blocks (all atoms)
__host__ __device__ constexpr uint32_t chunk_bytes(int d) { return (uint32_t)(d / 64) * kStStage; }

__device__ __forceinline__ void split3(float x, uint16_t& h1, uint16_t& h2, uint16_t& h3) {
  const __nv_bfloat16 b1 = __float2bfloat16_rn(x);
  const bool fin = isfinite(x);
  const float r1 = fin ? x - __bfloat162float(b1) : 0.f;  // exact in fp32
  const __nv_bfloat16 b2 = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(b2);              // exact in fp32
  const __nv_bfloat16 b3 = __float2bfloat16_rn(r2);
  h1 = __bfloat16_as_ushort(b1);
  h2 = __bfloat16_as_ushort(b2);
  h3 = __bfloat16_as_ushort(b3);
}

// 8 consecutive fp32 values -> their three bf16 planes (16 bytes each).
__device__ __forceinline__ void split8(const float* x, uint4* v) {
  uint16_t h[3][8];
#pragma unroll
  for (int i = 0; i < 8; ++i) split3(x[i], h[0][i], h[1][i], h[2][i]);
#pragma unroll
  for (int p = 0; p < 3; ++p)
    v[p] = make_uint4((uint32_t)h[p][0] | ((uint32_t)h[p][1] << 16), (uint32_t)h[p][2] | ((uint32_t)h[p][3] << 16),
                      (uint32_t)h[p][4] | ((uint32_t)h[p][5] << 16), (uint32_t)h[p][6] | ((uint32_t)h[p][7] << 16));
}

__device__ __forceinline__ void load8(const float* p, float* x) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* x) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Split keys of chunk C of unit u: [atom][plane][128 rows x 128 B], block 32 C + i,
// sub-block s at row r = 4 i + s (8-row groups 1024 bytes apart, 16-byte chunk c of
// a row at chunk c ^ (r % 8)); blocks past the sequence are zeros. grid (32 x
// chunks, U), 4 d / 8 threads.
template <int D>
__global__ void __launch_bounds__(4 * D / 8) prefill_keysplit_kernel(const float* __restrict__ pk, int nblk,
                                                                     uint8_t* __restrict__ pk3) {
  const int j = blockIdx.x, u = blockIdx.y, nch = gridDim.x / 32;
  const int s = threadIdx.x / (D / 8), cg = threadIdx.x % (D / 8), a = cg / 8, c = cg % 8;
  float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (j < nblk) load8(pk + (((long long)u * nblk + j) * 4 + s) * D + 8 * cg, x);
  uint4 v[3];
  split8(x, v);
  const int r = 4 * (j % 32) + s;
  uint8_t* dst = pk3 + ((long long)u * nch + j / 32) * chunk_bytes(D) + (size_t)a * kStStage +
                 (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
#pragma unroll
  for (int p = 0; p < 3; ++p) *reinterpret_cast<uint4*>(dst + p * kStPlane) = v[p];
}

// Sorts v ascending (bitonic network; N a power of two).
template <int N>
__device__ __forceinline__ void sort_asc(int (&v)[N]) {
#pragma unroll
  for (int k = 2; k <= N; k <<= 1)
#pragma unroll
    for (int jj = k >> 1; jj > 0; jj >>= 1)
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int l = i ^ jj;
        if (l > i) {
          const int x = v[i], y = v[l];
          const bool up = (i & k) == 0;
          v[i] = up ? min(x, y) : max(x, y);
          v[l] = up ? max(x, y) : min(x, y);
        }
      }
}

// Inserts (kx, ix) into a list sorted by (key descending, index ascending) when it
// ranks above the last entry; entries below the insertion point move down one.
template <int MM>
__device__ __forceinline__ void list_insert(uint32_t (&key)[MM], int (&idx)[MM], uint32_t kx, int ix) {
  bool g[MM];
#pragma unroll
  for (int r = 0; r < MM; ++r) g[r] = kx > key[r] || (kx == key[r] && ix < idx[r]);
#pragma unroll
  for (int r = MM - 1; r > 0; --r) {
    key[r] = g[r] ? (g[r - 1] ? key[r - 1] : kx) : key[r];
    idx[r] = g[r] ? (g[r - 1] ? idx[r - 1] : ix) : idx[r];
  }
  key[0] = g[0] ? kx : key[0];
  idx[0] = g[0] ? ix : idx[0];
}

// Shared-memory carve-up (offsets from a 1024-byte aligned base).
struct SelTcSmem {
  int d, nblk, ke;
  __host__ __device__ size_t a() const { return 0; }                                   // [3][d/64] 8 KB tiles + 8 KB zeros
  __host__ __device__ size_t stg() const { return (size_t)(3 * (d / 64) + 1) * 8192; }  // [kStStages][kStStage]
  __host__ __device__ size_t emask() const { return stg() + (size_t)kStStages * kStStage; }
  __host__ __device__ size_t eb() const { return emask() + 4 * (size_t)(((nblk + 31) / 32 + 3) & ~3); }
  __host__ __device__ size_t total() const { return eb() + 4 * (size_t)std::max(ke, 1) + 1024; }
};

template <typename T, int D, int MM>
__global__ void __launch_bounds__(kStThreads, 1) prefill_select_tc_kernel(
    Shape s, const T* __restrict__ q, int L, int nblk, const uint8_t* __restrict__ pk3,
    const int32_t* __restrict__ Eb, const int32_t* __restrict__ Ecnt, int32_t* __restrict__ sel,
    int32_t* __restrict__ block_tab, int32_t* __restrict__ tail_tab, int32_t* __restrict__ tail_len,
    int* __restrict__ err, float inv_sqrt_d) {
  constexpr int NA = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SelTcSmem Lay{D, nblk, s.ke};
  uint8_t* At = sm + Lay.a();
  uint8_t* stg = sm + Lay.stg();
  uint32_t* emask = reinterpret_cast<uint32_t*>(sm + Lay.emask());
  int32_t* eb_s = reinterpret_cast<int32_t*>(sm + Lay.eb());
  // after the scoring the ring holds the odd-chunk lists
  uint32_t* lk = reinterpret_cast<uint32_t*>(stg);              // [64][MM] keys
  int32_t* li = reinterpret_cast<int32_t*>(stg + 64 * MM * 4);  // [64][MM] block ids
  __shared__ __align__(8) uint64_t full[kStStages], empty[kStStages], mma_done[2], tmem_free[2];
  __shared__ uint32_t tmem_base;
  __shared__ volatile int s_bad;

  const int u = blockIdx.x, b = nblk - 1 - (int)blockIdx.y, req = u / s.Hkv, h = u % s.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int W = (nblk + 31) / 32;  // mask words = chunks of 32 blocks
  const int nch_all = W;
  const long long ubase = (long long)u * nblk;

  if (tid == 0) {
    for (int i = 0; i < kStStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&mma_done[i], 1);
      mbar_init(&tmem_free[i], 2);  // the two warps of the buffer's chunk parity
    }
    fence_mbar_init();
    s_bad = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_base, kStTmemCols);
  for (int i = tid; i < W; i += kStThreads) emask[i] = 0u;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  const int ecnt = Ecnt[ubase + b];
  const int32_t* eb = Eb + (ubase + b) * s.ke;
  for (int i = tid; i < ecnt; i += kStThreads) {
    const int j = eb[i];
    eb_s[i] = j;
    atomicOr(&emask[j >> 5], 1u << (j & 31));
  }
  const int n_cand = b;  // blocks before the positions' own block
  int m = min(s.k - ecnt, n_cand - ecnt);
  if (m > MM) {  // (|E_b| = min(k_e, b) and k - k_e <= MM: cannot happen)
    if (tid == 0) atomicExch(err, kDevErrBadIndex);
    m = MM;
  }
  const int npos = min(s.B, L - b * s.B);
  if (m > 0) {
    // A: q_bar of the 64 positions (fp32 sum over the heads in order, x 1/G),
    // split in 3 planes; positions past the sequence and the pad are zeros
    const float inv_g = 1.0f / (float)s.G;
    for (int i = tid; i < 512; i += kStThreads)
      reinterpret_cast<uint4*>(At + 3 * NA * 8192)[i] = make_uint4(0u, 0u, 0u, 0u);
    constexpr int kItems = 64 * (D / 8) / kStThreads;  // 8-dim pieces per thread
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int i = tid + it * kStThreads;
      const int p = i / (D / 8), cg = i % (D / 8), a = cg / 8, c = cg % 8;
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (p < npos) {
        const T* qg = q + (((long long)req * L + (long long)b * s.B + p) * s.Hq + (long long)h * s.G) * D + 8 * cg;
        for (int g = 0; g < s.G; ++g) {
          float y[8];
          load8(qg + (long long)g * D, y);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] += y[e];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= inv_g;
      }
      uint4 v[3];
      split8(x, v);
#pragma unroll
      for (int pl = 0; pl < 3; ++pl)
        *reinterpret_cast<uint4*>(At + (pl * NA + a) * 8192 + (p >> 3) * 1024 + (p & 7) * 128 +
                                  ((c ^ (p & 7)) << 4)) = v[pl];
    }
    fence_proxy_async();
  }
  __syncthreads();

  uint32_t key[MM];
  int idx[MM];
#pragma unroll
  for (int r = 0; r < MM; ++r) {
    key[r] = 0u;
    idx[r] = 0x7fffffff;
  }
  if (m > 0) {
    const int nch = (n_cand + kStCC - 1) / kStCC, nst = nch * NA;
    if (warp == kCopyWarp) {
      // ---- bulk copies: stage i = (chunk i / NA, 64-dim atom i % NA) --------
      if (lane == 0) {
        bool ok = true;
        int issued = 0;
        for (int i = 0; i < nst; ++i) {
          const int slot = i % kStStages;
          if (i >= kStStages && !(ok = mbar_wait_bounded(&empty[slot], (uint32_t)(((i - kStStages) / kStStages) & 1))))
            break;
          if (s_bad) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[slot], kStStage);
          const uint8_t* src = pk3 + ((long long)u * nch_all + i / NA) * chunk_bytes(D) + (size_t)(i % NA) * kStStage;
          uint8_t* dst = stg + (size_t)slot * kStStage;
#pragma unroll
          for (int p = 0; p < 3; ++p) bulk_g2s(dst + p * kStPlane, src + p * kStPlane, kStPlane, &full[slot]);
          ++issued;
        }
        if (!ok) {
          s_bad = 1;
          atomicExch(err, kDevErrWaitTimeout);
          for (int i = max(issued - kStStages, 0); i < issued; ++i)  // the copies in flight land first
            mbar_wait_bounded(&full[i % kStStages], (uint32_t)((i / kStStages) & 1));
        }
      }
    } else if (warp == kMmaWarp) {
      // ---- MMA issue (one thread) -------------------------------------------
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_bf16(128, 128);
        const uint32_t a_base = smem_u32(At), s_base = smem_u32(stg);
        bool ok = true;
        int last = -1;  // last stage whose MMAs were committed
        for (int c = 0; c < nch && ok; ++c) {
          const uint32_t t_d = tmem + (uint32_t)((c & 1) * 128);
          if (c >= 2 && !(ok = mbar_wait_bounded(&tmem_free[c & 1], (uint32_t)(((c - 2) >> 1) & 1)))) break;
          tc_fence_after();
          for (int a = 0; a < NA; ++a) {
            const int i = c * NA + a, slot = i % kStStages;
            if (!(ok = mbar_wait_bounded(&full[slot], (uint32_t)((i / kStStages) & 1))) || s_bad) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
              for (int t = 0; t < 6; ++t) {
                const uint64_t da = sw128_desc(a_base + (uint32_t)((kTermA[t] * NA + a) * 8192)) + 2 * kk;
                const uint64_t db = sw128_desc(s_base + (uint32_t)(slot * kStStage + kTermB[t] * kStPlane)) + 2 * kk;
                mma_bf16(t_d, da, db, idesc, (a | kk | t) ? 1u : 0u);
              }
            mma_commit(&empty[slot]);  // the stage may be refilled once these MMAs read it
            last = i;
          }
          if (ok) mma_commit(&mma_done[c & 1]);
        }
        if (!ok) {
          s_bad = 1;
          atomicExch(err, kDevErrWaitTimeout);
          if (last >= 0) mbar_wait_bounded(&empty[last % kStStages], (uint32_t)((last / kStStages) & 1));
        }
      }
    } else if (warp == 0 || warp == 1 || warp == 4 || warp == 5) {
      // ---- rows: a chunk's scores into the position's list -------------------
      const int gp = warp >> 2;                                 // chunk parity (= score buffer)
      const uint32_t t_lane = (uint32_t)(32 * (warp & 1)) << 16;  // positions 32 (warp & 1) + lane
      for (int c = gp; c < nch; c += 2) {
        const bool ok = mbar_wait_bounded(&mma_done[c & 1], (uint32_t)((c >> 1) & 1));
        if (!__all_sync(0xffffffffu, ok) || s_bad) {
          if (lane == 0) {
            s_bad = 1;
            atomicExch(err, kDevErrWaitTimeout);
          }
          break;
        }
        tc_fence_after();
        // candidates of the chunk: blocks 32 c + i before b and outside E_b
        const uint32_t live = ~emask[c] & (32 * c + 32 <= n_cand ? 0xffffffffu : ((1u << (n_cand - 32 * c)) - 1u));
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r[64];
          const uint32_t t_s = tmem + t_lane + (uint32_t)((c & 1) * 128 + 64 * half);
          tmem_ld16_nowait(t_s, r);
          tmem_ld16_nowait(t_s + 16, r + 16);
          tmem_ld16_nowait(t_s + 32, r + 32);
          tmem_ld16_nowait(t_s + 48, r + 48);
          tmem_wait_ld();
          if (half == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tmem_free[c & 1]);
          }
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) {
            const int i = 16 * half + cc;
            if (!((live >> i) & 1u)) continue;  // (warp-uniform)
            const float sc = fmaxf(fmaxf(__uint_as_float(r[4 * cc]), __uint_as_float(r[4 * cc + 1])),
                                   fmaxf(__uint_as_float(r[4 * cc + 2]), __uint_as_float(r[4 * cc + 3]))) *
                             inv_sqrt_d;
            const uint32_t kx = sc == sc ? ordered_key(sc) : 0u;
            if (kx > key[MM - 1]) list_insert<MM>(key, idx, kx, 32 * c + i);  // (ascending ids: '>' keeps ties)
          }
        }
      }
    }
  }
  __syncthreads();
  if (s_bad) {  // a wait gave up: nothing is written (the error word is set)
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(tmem, kStTmemCols);
    }
    return;
  }
  if (warp == 4 || warp == 5) {  // the odd-chunk lists (the ring is free now)
    const int p = 32 * (warp & 1) + lane;
#pragma unroll
    for (int r = 0; r < MM; ++r) {
      lk[p * MM + r] = key[r];
      li[p * MM + r] = idx[r];
    }
  }
  __syncthreads();
  // outputs, one thread per position: E_b ascending, then Gamma_q ascending, -1 pad
  if (warp < 2) {
    const int p = 32 * warp + lane;
    if (p < npos) {
      // the best m of the two lists (both sorted; ids distinct), then by id
      int ids[MM];
      int jb = 0;
      uint32_t bk = lk[p * MM];
      int bi = li[p * MM];
#pragma unroll
      for (int r = 0; r < MM; ++r) {
        int id = 0x7fffffff;
        if (r < m) {
          const bool own = key[0] > bk || (key[0] == bk && idx[0] < bi);
          if ((own ? key[0] : bk) != 0u) {
            if (own) {
              id = idx[0];
#pragma unroll
              for (int t = 0; t < MM - 1; ++t) {
                key[t] = key[t + 1];
                idx[t] = idx[t + 1];
              }
              key[MM - 1] = 0u;
              idx[MM - 1] = 0x7fffffff;
            } else {
              id = bi;
              ++jb;
              bk = jb < MM ? lk[p * MM + jb] : 0u;
              bi = jb < MM ? li[p * MM + jb] : 0x7fffffff;
            }
          }
        }
        ids[r] = id;
      }
      sort_asc<MM>(ids);
      const int t = b * s.B + p;
      const long long vu = ((long long)req * L + t) * s.Hkv + h;  // virtual unit of the position
      int32_t* selp = sel ? sel + vu * s.k : nullptr;
      int32_t* tab = block_tab + vu * s.k;
      for (int e = 0; e < ecnt; ++e) {
        const int j = eb_s[e];
        if (selp) selp[e] = j;
        tab[e] = (int32_t)(ubase + j);
      }
      int run = ecnt;
#pragma unroll
      for (int r = 0; r < MM; ++r)
        if (ids[r] != 0x7fffffff) {
          if (selp) selp[run] = ids[r];
          tab[run] = (int32_t)(ubase + ids[r]);
          ++run;
        }
      for (int e = run; e < s.k; ++e) {
        if (selp) selp[e] = -1;
        tab[e] = -1;
      }
      tail_tab[vu] = (int32_t)(ubase + b);
      tail_len[vu] = p + 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kStTmemCols);
  }
}

template <typename T, int D, int MM>
cudaError_t launch_select_tc_t(const Shape& s, int L, int nblk, const void* q, const uint8_t* pk3,
                               const int32_t* Eb, const int32_t* Ecnt, int32_t* sel, int32_t* tab,
                               int32_t* ttab, int32_t* tlen, int* err, cudaStream_t stream) {
  const void* fn = (const void*)prefill_select_tc_kernel<T, D, MM>;
  static std::atomic<int> lim[64];
  const size_t smem = SelTcSmem{D, nblk, s.ke}.total();
  cudaError_t e = raise_smem_limit(fn, smem, lim);
  if (e != cudaSuccess) return e;
  const float isd = (float)(1.0 / std::sqrt((double)D));
  prefill_select_tc_kernel<T, D, MM><<<dim3(s.U, nblk), kStThreads, smem, stream>>>(
      s, (const T*)q, L, nblk, pk3, Eb, Ecnt, sel, tab, ttab, tlen, err, isd);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_select_tc_d(const Shape& s, int L, int nblk, const void* q, const uint8_t* pk3,
                               const int32_t* Eb, const int32_t* Ecnt, int32_t* sel, int32_t* tab,
                               int32_t* ttab, int32_t* tlen, int* err, cudaStream_t stream) {
  if (s.k - s.ke <= 16)
    return launch_select_tc_t<T, D, 16>(s, L, nblk, q, pk3, Eb, Ecnt, sel, tab, ttab, tlen, err, stream);
  return launch_select_tc_t<T, D, 32>(s, L, nblk, q, pk3, Eb, Ecnt, sel, tab, ttab, tlen, err, stream);
}

}  // namespace

bool prefill_select_tc_shape(const Shape& s) {
  return (s.d == 64 || s.d == 128) && s.P == 4 && s.k - s.ke <= 32 && s.B == 64;
}

bool prefill_select_tc_ok(const Shape& s, int L) {
  const char* env = std::getenv("NOSA_PREFILL_SELECT_TC");
  if (env && std::strcmp(env, "0") == 0) return false;
  if (!prefill_select_tc_shape(s)) return false;
  const int nblk = (L + s.B - 1) / s.B;
  return SelTcSmem{s.d, nblk, s.ke}.total() <= 227 * 1024 - 1024;
}

size_t prefill_keysplit_bytes(const Shape& s, int nblk) {
  return prefill_select_tc_shape(s) ? (size_t)s.U * ((nblk + 31) / 32) * chunk_bytes(s.d) : 0;
}

cudaError_t launch_prefill_select_tc(const Shape& s, int L, const void* q, const float* pk, uint8_t* pk3,
                                     const int32_t* Eb, const int32_t* Ecnt, int32_t* sel, int32_t* tab,
                                     int32_t* ttab, int32_t* tlen, int* err, cudaStream_t stream) {
  const int nblk = (L + s.B - 1) / s.B;
  if (nblk > 65535) return cudaErrorInvalidConfiguration;
  const dim3 kgrid((nblk + 31) / 32 * 32, s.U);
  if (s.d == 64)
    prefill_keysplit_kernel<64><<<kgrid, 4 * 64 / 8, 0, stream>>>(pk, nblk, pk3);
  else
    prefill_keysplit_kernel<128><<<kgrid, 4 * 128 / 8, 0, stream>>>(pk, nblk, pk3);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (s.dtype == 0)
    return s.d == 64 ? launch_select_tc_d<float, 64>(s, L, nblk, q, pk3, Eb, Ecnt, sel, tab, ttab, tlen, err, stream)
                     : launch_select_tc_d<float, 128>(s, L, nblk, q, pk3, Eb, Ecnt, sel, tab, ttab, tlen, err, stream);
  return s.d == 64
             ? launch_select_tc_d<__nv_bfloat16, 64>(s, L, nblk, q, pk3, Eb, Ecnt, sel, tab, ttab, tlen, err, stream)
             : launch_select_tc_d<__nv_bfloat16, 128>(s, L, nblk, q, pk3, Eb, Ecnt, sel, tab, ttab, tlen, err, stream);
}

}  // namespace nosa
