// Fused front-end of a decode step: the projection of the hidden states (query,
// key and value heads and the eviction head) on the tensor cores, the QKV split,
// and the append of the new token with incremental pooling.
//
// NOSA technical summary, Methodology §2 "Kernel Fusion" (eviction-head
// computation, QKV splitting and pooling in one kernel) and §1 "Dual-Selection
// Mechanism" (the eviction head scores tokens independently of the query; its
// pre-exp logit is pooled for the query-agnostic selection and added to the
// attention logits by ED-DMA).
//
// Y[f][b] = sum_i W[f][i] x[b][i] over the F = (Hq + 2 Hkv) d + Hkv packed rows
// of W (query heads, key heads, value heads, one eviction row per KV head). A
// decode step has few tokens (the batch) against many rows, so the rows are the
// MMA's M side: CTA (tile, split) computes a 128-row x N tile (N = the batch
// padded to a multiple of 16) over its share of the hidden width with
// tcgen05.mma (kind::f16: bf16 operands, fp32 accumulator in tensor memory).
// The weights are packed once (frontend_pack_kernel) so that every 128-row x
// 64-column tile is one contiguous 16 KB run already in the 128-byte-swizzled
// K-major order the MMA reads, tiles of a row block consecutive along the hidden
// width: a CTA streams one contiguous range with bulk copies (full DRAM pages),
// and TMA brings the matching N x 64 hidden-state tiles (same swizzle) into a
// ring of shared-memory stages.
// The splits of a row tile form one thread-block cluster: each CTA leaves its
// fp32 partial tile in shared memory and, after a cluster barrier, sums a share
// of the tile's entries over all ranks (rank order, deterministic) through
// distributed shared memory, then runs the epilogue for that share:
//   query rows    -> q [batch][Hq][d], bf16 (nearest even);
//   key rows      -> the unit's tail block (chunk-major K), value rows -> V
//                    (token-major), both bf16; eviction rows -> e (fp32);
//   at a sub-block end the 16 keys and eviction logits are averaged (fp32 sum in
//   token order, x 1/16) into the pooled keys, the sub-block eviction means and
//   the block's eviction score (running max), as the plain append does.
// While the tensor cores run, the other warps promote the previous block to the
// host store (when this token opens a new block) and publish the step record.
//
// Warp roles (192 threads): warp 0 issues the TMA copies, warp 1 owns the tensor
// memory and issues the MMAs, warps 2-5 do the side work and then the epilogue
// (warp w reads tensor-memory lanes 32 (w % 4) .. 32 (w % 4) + 31). Every
// mbarrier wait is bounded (~2 s): one that gives up sets the error word; the
// copies already issued are drained (bounded) and the tensor memory is freed
// before the CTA exits.
#include "nosa_internal.cuh"
#include "tcgen05.cuh"

#include <atomic>

namespace nosa {
namespace {
using namespace tc;

constexpr int kFrontThreads = 192;
constexpr int kTileM = 128;                   // rows of W per CTA (MMA M)
constexpr int kTileK = 64;                    // hidden elements per stage: 128 bytes of bf16
constexpr int kMaxStages = 10;
constexpr int kABytes = kTileM * kTileK * 2;  // 16 KB weight tile per stage

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Writes rows f0 .. f0 + 7 of the projection for request n (values v8, fp32).
// 8 rows of one kind never straddle a boundary (the boundaries are multiples of
// 64), so a query, key or value item is one aligned 16-byte store (8 bf16: one K
// chunk, or 8 consecutive V or q elements) and its key running sums are two
// float4. The sums run in token order from 0; the sub-block's last token turns
// them into means. Eviction rows (one fp32 pre-exp logit per KV head) are
// written one by one.
// pre: the item's running sums, loaded earlier (NULL: load them here).
__device__ __forceinline__ void store_item(const Shape& s, const State& st, const FrontParams& p,
                                           int n, int f0, const float* v8, const float* pre,
                                           int blk, int pos) {
  const int Fq = s.Hq * s.d, Fk = Fq + s.Hkv * s.d, Fv = Fk + s.Hkv * s.d;
  const bool first = (pos % s.S) == 0, last = (pos % s.S) == s.S - 1;
  const int sb = pos / s.S;
  const long long tail_sel = (long long)(blk & 1) * s.payload;
  if (f0 < Fv) {
    __align__(16) __nv_bfloat16 b8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) b8[e] = __float2bfloat16_rn(v8[e]);
    const int4 packed = *reinterpret_cast<const int4*>(b8);
    if (f0 < Fq) {
      *reinterpret_cast<int4*>(reinterpret_cast<__nv_bfloat16*>(p.q) + (long long)n * Fq + f0) = packed;
      return;
    }
    const bool is_k = f0 < Fk;
    const int r = is_k ? f0 - Fq : f0 - Fk;
    const int h = r / s.d, dim0 = r % s.d;
    const int u = n * s.Hkv + h;
    uint8_t* cur = st.tail + (long long)u * 2 * s.payload + tail_sel;
    if (!is_k) {
      *reinterpret_cast<int4*>(cur + v_off(pos, dim0, s.B, s.d, 2)) = packed;
      return;
    }
    *reinterpret_cast<int4*>(cur + k_off(pos, dim0, s.B, 2)) = packed;
    float4* ks = reinterpret_cast<float4*>(st.ksum + (long long)u * s.d + dim0);
    float rs[8];
    if (first) {
#pragma unroll
      for (int e = 0; e < 8; ++e) rs[e] = 0.f;
    } else if (pre) {
#pragma unroll
      for (int e = 0; e < 8; ++e) rs[e] = pre[e];
    } else {
      const float4 a = ks[0], b = ks[1];
      rs[0] = a.x; rs[1] = a.y; rs[2] = a.z; rs[3] = a.w;
      rs[4] = b.x; rs[5] = b.y; rs[6] = b.z; rs[7] = b.w;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) rs[e] += __bfloat162float(b8[e]);
    if (last) {
      const long long pk0 = (((long long)u * s.maxBlk + blk) * s.P + sb) * s.d + dim0;
#pragma unroll
      for (int e = 0; e < 8; ++e) store_pooled(s, st.pk, pk0 + e, rs[e] * (1.0f / s.S));
    } else {
      ks[0] = make_float4(rs[0], rs[1], rs[2], rs[3]);
      ks[1] = make_float4(rs[4], rs[5], rs[6], rs[7]);
    }
    return;
  }
  const int ne = min(8, p.F - f0);
  float run[8];
#pragma unroll
  for (int e = 0; e < 8; ++e)  // every load before the first store
    run[e] = (e < ne && !first) ? (pre ? pre[e] : st.esum[n * s.Hkv + (f0 + e - Fv)]) : 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (e >= ne) break;
    const int u = n * s.Hkv + (f0 + e - Fv);
    uint8_t* cur = st.tail + (long long)u * 2 * s.payload + tail_sel;
    *reinterpret_cast<float*>(cur + e_off(pos, s.B, s.d, 2)) = v8[e];
    const float rsum = run[e] + v8[e];
    if (last) {
      const float eb = rsum * (1.0f / s.S);
      const long long bi = (long long)u * s.maxBlk + blk;
      st.sube[bi * s.P + sb] = eb;
      st.se[bi] = (sb == 0) ? eb : fmaxf(st.se[bi], eb);
    } else {
      st.esum[u] = rsum;
    }
  }
}

// Loads the running sums that store_item will need for rows f0 .. f0 + 7 of
// request n (key rows: 8 from ksum; eviction rows: up to 8 from esum).
__device__ __forceinline__ void prefetch_sums(const Shape& s, const State& st,
                                              const FrontParams& p, int n, int f0, float* pre) {
  const int Fq = s.Hq * s.d, Fk = Fq + s.Hkv * s.d, Fv = Fk + s.Hkv * s.d;
  if (f0 >= Fq && f0 < Fk) {
    const int r = f0 - Fq;
    const float4* ks = reinterpret_cast<const float4*>(
        st.ksum + (long long)(n * s.Hkv + r / s.d) * s.d + r % s.d);
    const float4 a = ks[0], b = ks[1];
    pre[0] = a.x; pre[1] = a.y; pre[2] = a.z; pre[3] = a.w;
    pre[4] = b.x; pre[5] = b.y; pre[6] = b.z; pre[7] = b.w;
  } else if (f0 >= Fv) {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      pre[e] = (f0 + e < p.F) ? st.esum[n * s.Hkv + (f0 + e - Fv)] : 0.f;
  }
}

// Distributed shared memory of the CTA cluster that shares a row tile.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(const void* local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
  return a;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Every thread of every CTA of the cluster; orders shared-memory writes before
// the peers' reads (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(kFrontThreads, 1)
    frontend_kernel(const __grid_constant__ CUtensorMap tx, Shape s, State st, FrontParams p) {
  TraceScope trace_scope(st.trace, kTrAppend);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int b_bytes = p.npad * 128;
  const int kStages = p.stages;
  uint8_t* sa = smem;                    // [stages][128 rows][128 B]
  uint8_t* sb = smem + kStages * kABytes;  // [stages][npad rows][128 B]
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], accum;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int s_bad;
  __shared__ int s_issued, s_last;

  const int tile = blockIdx.x, split = blockIdx.y;
  const int kb0 = (int)((long long)split * p.kblocks / p.ksplit);
  const int kb1 = (int)((long long)(split + 1) * p.kblocks / p.ksplit);
  const int nk = kb1 - kb0;  // >= 1 (the host keeps ksplit <= kblocks)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = p.L_old / s.B, pos = p.L_old % s.B;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&accum, 1);
    fence_mbar_init();
    s_bad = 0;
    s_issued = 0;
    s_last = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base)),
                 "r"(p.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  // Items of the first chunk of requests handled by this thread in the epilogue
  // (see below); their running sums are loaded while the tensor cores run.
  constexpr int kItemsMax = 4;  // 512 items / (128 threads x ksplit >= 1)
  const uint32_t rank = cluster_rank();
  const int tid2 = threadIdx.x - 64;
  float pre[kItemsMax][8];

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      int i = 0;
      for (; i < nk; ++i) {
        const int stg = i % kStages;
        if (i >= kStages &&
            !mbar_wait_bounded(&empty[stg], (uint32_t)(((i / kStages) - 1) & 1))) {
          s_bad = 1;
          atomicExch(p.err, kDevErrWaitTimeout);
          break;
        }
        if (s_bad) break;
        mbar_arrive_expect_tx(&full[stg], (uint32_t)(kABytes + b_bytes));
        bulk_g2s(sa + stg * kABytes,
                 p.w_packed + ((long long)tile * p.kblocks + kb0 + i) * kABytes, (uint32_t)kABytes,
                 &full[stg]);
        tma_load_2d(smem_u32(sb + stg * b_bytes), &tx, (kb0 + i) * kTileK, 0, smem_u32(&full[stg]));
      }
      s_issued = i;
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      // kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, both
      // K-major, N = npad, M = 128.
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) |
                             ((uint32_t)(p.npad >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);
      for (int i = 0; i < nk; ++i) {
        const int stg = i % kStages;
        if (!mbar_wait_bounded(&full[stg], (uint32_t)((i / kStages) & 1))) {
          s_bad = 1;
          atomicExch(p.err, kDevErrWaitTimeout);
          break;
        }
        tc_fence_after();
        const uint64_t da = sw128_desc(smem_u32(sa + stg * kABytes));
        const uint64_t db = sw128_desc(smem_u32(sb + stg * b_bytes));
#pragma unroll
        for (int kk = 0; kk < kTileK / 16; ++kk)  // 16 bf16 = 32 bytes per MMA step
          mma_bf16(tmem, da + 2 * kk, db + 2 * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&empty[stg]);
      }
      mma_commit(&accum);
    }
  } else {
    // Side work while the tensor cores run.
    const int cta = blockIdx.y * gridDim.x + blockIdx.x, ncta = gridDim.x * gridDim.y;
    if (cta == 0 && tid2 == 0) {
      StepIO io;
      io.q = p.q;
      io.out = p.out;
      io.lse = p.lse;
      io.L_old = p.L_old;
      io.n_cand = blk;
      io.tail_len = pos + 1;
      io.just_completed = (pos == 0 && blk > 0) ? blk - 1 : -1;
      io.tail_off = (long long)(blk & 1) * s.payload;
      *st.io = io;
    }
    if (pos == 0 && blk > 0) {  // the previous block becomes a candidate
      const int cb = blk - 1;
      const int nvec = (int)(s.payload / 16);
      for (int u = cta; u < s.U; u += ncta) {
        const int4* src = reinterpret_cast<const int4*>(st.tail + ((long long)u * 2 + (cb & 1)) * s.payload);
        int4* dst = reinterpret_cast<int4*>(st.host + ((long long)u * s.maxBlk + cb) * s.payload);
        for (int i = tid2; i < nvec; i += 128) dst[i] = src[i];
        if (tid2 == 0) atomicOr(&st.elig[(long long)u * s.W + cb / 32], 1u << (cb % 32));
      }
      __threadfence_system();
    }

    if ((pos % s.S) != 0) {
#pragma unroll
      for (int q = 0; q < kItemsMax; ++q) {
        const int it = (int)rank * 128 + tid2 + q * 128 * p.ksplit;
        const int n = it >> 4, f0 = tile * kTileM + (it & 15) * 8;
        if (it < 32 * 16 && n < p.batch && f0 < p.F) prefetch_sums(s, st, p, n, f0, pre[q]);
      }
    }

    // Wait for the accumulator.
    const bool okw = __all_sync(0xffffffffu, mbar_wait_bounded(&accum, 0));
    if (!okw && lane == 0) {
      s_bad = 1;
      atomicExch(p.err, kDevErrWaitTimeout);
    }
    epi_barrier();
    tc_fence_after();
    if (tid2 == 0) trace_mark(st.trace, kTrFrontMain);
  }

  // Epilogue, per chunk of 32 requests. Each CTA of the cluster (the splits of
  // one row tile) leaves its fp32 partial of the chunk in its shared memory (the
  // stages are idle by now); after a cluster barrier every CTA takes a share of
  // the (request, 8-row group) items, sums the partials of all ranks in rank
  // order (deterministic) through distributed shared memory, and stores them.
  // A second barrier keeps every partial alive until the peers have read it.
  {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
    float* P = reinterpret_cast<float*>(sa);  // [32][128] fp32
    const bool ok = (s_bad == 0);
    for (int c0 = 0; c0 < p.batch; c0 += 32) {
      if (warp >= 2 && ok) {
        float v[16];
        for (int cc = 0; cc < 32; cc += 16) {
          if (c0 + cc >= p.batch) break;
          tmem_ld16(taddr + c0 + cc, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) P[(cc + j) * kTileM + row] = v[j];
        }
      }
      cluster_sync();
      if (warp >= 2 && ok) {
#pragma unroll
        for (int q = 0; q < kItemsMax; ++q) {
          const int it = (int)rank * 128 + tid2 + q * 128 * p.ksplit;
          const int j = it >> 4, g = it & 15;
          const int n = c0 + j, f0 = tile * kTileM + g * 8;
          if (it >= 32 * 16 || n >= p.batch || f0 >= p.F) continue;
          const void* local = P + j * kTileM + g * 8;
          float v8[8];
          for (int r = 0; r < p.ksplit; ++r) {
            const uint32_t a = map_to_rank(local, (uint32_t)r);
            const float4 x0 = ld_cluster_f4(a), x1 = ld_cluster_f4(a + 16);
            const float t8[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) v8[e] = (r == 0) ? t8[e] : v8[e] + t8[e];
          }
          store_item(s, st, p, n, f0, v8, c0 == 0 ? pre[q] : nullptr, blk, pos);
        }
      }
      cluster_sync();
    }
    if (threadIdx.x == 64) trace_mark(st.trace, kTrFrontEpi);
    tc_fence_before();
  }

  __syncthreads();
  if (threadIdx.x == 0 && s_bad) {
    // Drain: wait (bounded) for the last copy issued into each stage.
    for (int stg = 0; stg < kStages; ++stg) {
      int last = -1;
      for (int i = stg; i < s_issued; i += kStages) last = i;
      if (last >= 0) mbar_wait_bounded(&full[stg], (uint32_t)((last / kStages) & 1));
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(p.tmem_cols)
                 : "memory");
  }
}

// Packed weights: tile (t, kb) = rows [128 t, 128 t + 128) x columns [64 kb, 64 kb + 64)
// of W is 16 KB at ((t * kblocks + kb) * 16384); inside it row r's 16-byte chunk c
// (columns 8c .. 8c + 7) sits at r * 128 + (c ^ (r % 8)) * 16, the 128-byte swizzle.
// Rows past F are zeros. grid = (kblocks, tiles), 128 threads; thread r copies row r.
__global__ void __launch_bounds__(128) frontend_pack_kernel(const __nv_bfloat16* __restrict__ w,
                                                            uint8_t* __restrict__ packed, int F,
                                                            int D) {
  const int kb = blockIdx.x, t = blockIdx.y, r = threadIdx.x;
  const int kblocks = gridDim.x;
  const int row = t * kTileM + r;
  uint8_t* dst = packed + ((long long)t * kblocks + kb) * kABytes + r * 128;
  const int4* src = reinterpret_cast<const int4*>(w + (long long)row * D + kb * kTileK);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int4 v = (row < F) ? src[c] : make_int4(0, 0, 0, 0);
    *reinterpret_cast<int4*>(dst + ((c ^ (r & 7)) * 16)) = v;
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return (EncodeTiledFn) nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// 2-D bf16 row-major [rows][cols] map with a {64, box_rows} box, 128-byte swizzle;
// rows outside the tensor read as zeros.
bool encode_rows(CUtensorMap* map, const void* base, long long rows, long long cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool frontend_available() { return encode_fn() != nullptr; }

int frontend_stages(int npad) {
  const int per = kABytes + npad * 128;
  int st = (205 * 1024) / per;
  return st < 2 ? 2 : (st > kMaxStages ? kMaxStages : st);
}

size_t frontend_smem_bytes(int npad, int stages) {
  return 1024 + (size_t)stages * (kABytes + npad * 128);
}

bool frontend_encode(FrontArgs& fa, const void* x, int batch, int D) {
  return encode_rows(&fa.tx, x, batch, D, fa.p.npad);
}

size_t frontend_packed_bytes(int F, int D) {
  return (size_t)((F + kTileM - 1) / kTileM) * (D / kTileK) * kABytes;
}

cudaError_t launch_frontend_pack(const void* w, void* packed, int F, int D, cudaStream_t stream) {
  dim3 grid(D / kTileK, (F + kTileM - 1) / kTileM);
  frontend_pack_kernel<<<grid, kTileM, 0, stream>>>(static_cast<const __nv_bfloat16*>(w),
                                                    static_cast<uint8_t*>(packed), F, D);
  return cudaGetLastError();
}

const void* frontend_kernel_ptr() { return reinterpret_cast<const void*>(frontend_kernel); }

namespace {
cudaLaunchConfig_t front_config(const FrontParams& p, cudaStream_t stream,
                                cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t c = {};
  c.gridDim = dim3(p.tiles, p.ksplit, 1);
  c.blockDim = dim3(kFrontThreads, 1, 1);
  c.dynamicSmemBytes = frontend_smem_bytes(p.npad, p.stages);
  c.stream = stream;
  attr->id = cudaLaunchAttributeClusterDimension;
  attr->val.clusterDim.x = 1;
  attr->val.clusterDim.y = (unsigned)p.ksplit;  // the splits of a row tile
  attr->val.clusterDim.z = 1;
  c.attrs = attr;
  c.numAttrs = 1;
  return c;
}
std::atomic<int> g_front_smem_lim[64];
}  // namespace

int frontend_max_clusters(const FrontParams& p) {
  if (raise_smem_limit((const void*)frontend_kernel, frontend_smem_bytes(p.npad, p.stages),
                       g_front_smem_lim) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t c = front_config(p, nullptr, &attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (const void*)frontend_kernel, &c) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_frontend(const Shape& s, const State& st, const FrontArgs& fa,
                            cudaStream_t stream) {
  cudaError_t err = raise_smem_limit((const void*)frontend_kernel,
                                     frontend_smem_bytes(fa.p.npad, fa.p.stages), g_front_smem_lim);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t c = front_config(fa.p, stream, &attr);
  return cudaLaunchKernelEx(&c, frontend_kernel, fa.tx, s, st, fa.p);
}

}  // namespace nosa
