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
// TMA streams 128 x 64 weight tiles and N x 64 hidden-state tiles into a ring of
// 128-byte-swizzled shared-memory stages (the K-major layout the MMA reads).
// With several splits, each CTA stores its fp32 partial tile; the CTA that
// finishes a tile last sums the partials in split order (deterministic) and runs
// the epilogue:
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

#include <atomic>

namespace nosa {
namespace {

constexpr int kFrontThreads = 192;
constexpr int kTileM = 128;                   // rows of W per CTA (MMA M)
constexpr int kTileK = 64;                    // hidden elements per stage: 128 bytes of bf16
constexpr int kStages = 4;
constexpr int kABytes = kTileM * kTileK * 2;  // 16 KB weight tile per stage

// Shared-memory matrix descriptor of a K-major operand tile in the canonical
// 128-byte-swizzled layout (rows of 128 bytes, groups of 8 rows 1024 bytes apart).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address / 16
  d |= (uint64_t)1 << 16;                           // leading-dimension offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;                 // stride between 8-row groups / 16
  d |= (uint64_t)1 << 46;                           // descriptor version of tcgen05
  d |= (uint64_t)2 << 61;                           // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every MMA this thread issued before it has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Writes row f of the projection for request n (value y, fp32) where it belongs.
__device__ __forceinline__ void emit(const Shape& s, const State& st, const FrontParams& p, int f,
                                     int n, float y, int blk, int pos) {
  const int Fq = s.Hq * s.d, Fk = Fq + s.Hkv * s.d, Fv = Fk + s.Hkv * s.d;
  const bool sub_end = (pos % s.S) == s.S - 1;
  const int p0 = pos - (s.S - 1);  // first token of the completed sub-block
  if (f < Fq) {
    reinterpret_cast<__nv_bfloat16*>(p.q)[(long long)n * Fq + f] = __float2bfloat16_rn(y);
    return;
  }
  if (f < Fv) {
    const bool is_k = f < Fk;
    const int r = is_k ? f - Fq : f - Fk;
    const int h = r / s.d, dim = r % s.d;
    const int u = n * s.Hkv + h;
    uint8_t* cur = st.tail + ((long long)u * 2 + (blk & 1)) * s.payload;
    const __nv_bfloat16 yb = __float2bfloat16_rn(y);
    if (!is_k) {
      *reinterpret_cast<__nv_bfloat16*>(cur + v_off(pos, dim, s.B, s.d, 2)) = yb;
      return;
    }
    *reinterpret_cast<__nv_bfloat16*>(cur + k_off(pos, dim, s.B, 2)) = yb;
    if (sub_end) {
      float acc = 0.f;
      for (int j = 0; j < s.S - 1; ++j)
        acc += __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(cur + k_off(p0 + j, dim, s.B, 2)));
      acc += __bfloat162float(yb);
      const int sb = pos / s.S;
      store_pooled(s, st.pk, (((long long)u * s.maxBlk + blk) * s.P + sb) * s.d + dim,
                   acc * (1.0f / s.S));
    }
    return;
  }
  const int h = f - Fv;  // eviction row of KV head h
  const int u = n * s.Hkv + h;
  uint8_t* cur = st.tail + ((long long)u * 2 + (blk & 1)) * s.payload;
  *reinterpret_cast<float*>(cur + e_off(pos, s.B, s.d, 2)) = y;
  if (sub_end) {
    float ea = 0.f;
    for (int j = 0; j < s.S - 1; ++j)
      ea += *reinterpret_cast<const float*>(cur + e_off(p0 + j, s.B, s.d, 2));
    ea += y;
    const float eb = ea * (1.0f / s.S);
    const int sb = pos / s.S;
    const long long bi = (long long)u * s.maxBlk + blk;
    st.sube[bi * s.P + sb] = eb;
    st.se[bi] = (sb == 0) ? eb : fmaxf(st.se[bi], eb);
  }
}

__global__ void __launch_bounds__(kFrontThreads, 1)
    frontend_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx,
                    Shape s, State st, FrontParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int b_bytes = p.npad * 128;
  uint8_t* sa = smem;                    // [kStages][128 rows][128 B]
  uint8_t* sb = smem + kStages * kABytes;  // [kStages][npad rows][128 B]
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], accum;
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
        tma_load_2d(smem_u32(sa + stg * kABytes), &tw, (kb0 + i) * kTileK, tile * kTileM,
                    smem_u32(&full[stg]));
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
    const int tid2 = threadIdx.x - 64;
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
    if (cta == 0 && tid2 < kMaxChunks) st.work_count[tid2] = 0;
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

    // Epilogue.
    const int quarter = warp & 3;
    const int f = tile * kTileM + quarter * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&accum, 0));
    ok = ok && !__any_sync(0xffffffffu, s_bad != 0);
    if (!ok) {
      if (lane == 0) {
        s_bad = 1;
        atomicExch(p.err, kDevErrWaitTimeout);
      }
    } else {
      tc_fence_after();
      float v[16];
      if (p.ksplit == 1) {
        for (int c0 = 0; c0 < p.npad; c0 += 16) {
          __syncwarp();  // the load below is warp-collective; the stores above diverge
          tmem_ld16(taddr + c0, v);
          for (int j = 0; j < 16; ++j) {
            const int n = c0 + j;
            if (n < p.batch && f < p.F) emit(s, st, p, f, n, v[j], blk, pos);
          }
        }
      } else {
        float* part = p.part + (long long)split * p.npad * p.Fpad;
        for (int c0 = 0; c0 < p.npad; c0 += 16) {
          __syncwarp();
          tmem_ld16(taddr + c0, v);
          for (int j = 0; j < 16; ++j) {
            const int n = c0 + j;
            if (n < p.batch) part[(long long)n * p.Fpad + f] = v[j];
          }
        }
      }
    }
    tc_fence_before();
    if (p.ksplit > 1) {
      // The CTA that publishes a tile's last partial sums them all in split order.
      __threadfence();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      // A CTA whose tile failed does not count itself: the tile is then never
      // completed and the error word tells the host.
      if (tid2 == 0) s_last = (s_bad == 0) && (atomicAdd(&p.counters[tile], 1) == p.ksplit - 1);
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (s_last) {
        __threadfence();
        for (int n = 0; n < p.batch; ++n) {
          float y = 0.f;
          for (int sp = 0; sp < p.ksplit; ++sp)
            y += __ldcg(p.part + ((long long)sp * p.npad + n) * p.Fpad + f);
          if (f < p.F) emit(s, st, p, f, n, y, blk, pos);
        }
        if (tid2 == 0) p.counters[tile] = 0;
      }
    }
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

size_t frontend_smem_bytes(int npad) { return 1024 + (size_t)kStages * (kABytes + npad * 128); }

bool frontend_encode(FrontArgs& fa, const void* x, const void* w, int batch, int D, int F) {
  return encode_rows(&fa.tx, x, batch, D, fa.p.npad) && encode_rows(&fa.tw, w, F, D, kTileM);
}

const void* frontend_kernel_ptr() { return reinterpret_cast<const void*>(frontend_kernel); }

cudaError_t launch_frontend(const Shape& s, const State& st, const FrontArgs& fa,
                            cudaStream_t stream) {
  const size_t smem = frontend_smem_bytes(fa.p.npad);
  static std::atomic<int> lim[64];
  cudaError_t err = raise_smem_limit((const void*)frontend_kernel, smem, lim);
  if (err != cudaSuccess) return err;
  dim3 grid(fa.p.tiles, fa.p.ksplit);
  frontend_kernel<<<grid, kFrontThreads, smem, stream>>>(fa.tw, fa.tx, s, st, fa.p);
  return cudaGetLastError();
}

}  // namespace nosa
