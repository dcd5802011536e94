// Query-aware block scores: second pooling stage.
//
// NOSA technical summary, Methodology §1 "Block-Wise Implementation" (two-stage
// pooling: mean inside sub-blocks, max at block level) and "Dual-Selection
// Mechanism" (the query-aware part Gamma_q). For unit (b, h) with query group
// q_g (g < G), q_bar = (1/G) sum_g q_g and
//     sq(i) = max_{s < 4} (q_bar . K_bar[i, s]) / sqrt(d)       for every candidate i.
// This streams all pooled keys of every unit once per step (HBM-bound).
//
// Mapping: 8 warps per CTA, 4 blocks per warp. A block's 4 pooled rows are read
// by the warp as lanes (row r = lane / 8, column group c = lane % 8); each lane
// holds q_bar for its columns in registers, reduces over the 8 lanes of a row and
// then takes the max over the 4 rows.
//
// Fused forms: the scoring CTAs of a unit count themselves out (a fence, then
// an add on the unit's counter); the last one, which then sees every score of
// the unit, runs the unit's dual selection and set-difference (k_select.cuh) at
// once. A unit's selection thus starts as soon as its own scores exist,
// overlapping the scoring of later units, and no separate selection launch sits
// between the scoring and the gather.
#include "k_select.cuh"

#include <algorithm>

namespace nosa {
namespace {

constexpr int kScoreWarps = 8;
constexpr int kScoreBPW = 4;  // blocks per warp
constexpr int kScoreBPC = kScoreWarps * kScoreBPW;

// Pooled keys are fp32 (PT = float) or bf16 (PT = __nv_bfloat16): each lane
// loads 16-byte chunks of its row (4 fp32 or 8 bf16 values) and widens them.
template <typename PT> __device__ __forceinline__ void widen16(const uint4 r, float* f);
template <> __device__ __forceinline__ void widen16<float>(const uint4 r, float* f) {
  f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
  f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}
template <> __device__ __forceinline__ void widen16<__nv_bfloat16>(const uint4 r, float* f) {
  f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x); f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
  f[4] = bf16_lo(r.z); f[5] = bf16_hi(r.z); f[6] = bf16_lo(r.w); f[7] = bf16_hi(r.w);
}

// MODE 0: scores only; 1: + the unit's selection and set-difference in its last
// scoring CTA.
template <typename T, typename PT, int D, int MODE>
__global__ void __launch_bounds__(256) score_kernel(Shape s, State st, float inv_sqrt_d,
                                                    int ubase, int cold, int chunk) {
  constexpr bool FUSED = MODE >= 1;
  griddep_wait();               // the append (programmatic edge in the step graph)
  griddep_launch_dependents();  // the chunk's gather may become resident (it waits)
  TraceScope trace_scope(st.trace, chunk >= 0 && chunk < 8 ? kTrScore + chunk : -1);
  constexpr int EPC = 16 / (int)sizeof(PT);  // pooled values per 16-byte chunk
  constexpr int M = D / EPC / 8;             // chunks per lane per pooled row
  static_assert(M >= 1, "row too short for 8 lanes");
  static_assert(kSelThreads == 256, "the selection runs on the scoring CTA's threads");
  extern __shared__ __align__(16) uint8_t sel_dyn[];  // fused: the selection's key / flag arrays
  __shared__ __align__(16) float qbar[D];
  __shared__ int s_last;
  const int n_cand = st.io->n_cand;
  // scoring CTAs of a unit (at least one, which then selects an empty candidate set)
  const int nct = max(1, (n_cand + kScoreBPC - 1) / kScoreBPC);
  if ((int)blockIdx.x >= nct) return;  // grid sized for a larger count
  const T* __restrict__ q = static_cast<const T*>(st.io->q);
  const int u = ubase + blockIdx.y, b = u / s.Hkv, h = u % s.Hkv;
  const T* qg = q + ((long long)b * s.Hq + (long long)h * s.G) * D;
  const float inv_g = 1.0f / (float)s.G;
  for (int dim = threadIdx.x; dim < D; dim += blockDim.x) {
    float acc = 0.f;
    for (int g = 0; g < s.G; ++g) acc += to_f32(qg[g * D + dim]);
    qbar[dim] = acc * inv_g;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 3, c = lane & 7;
  float qr[M][EPC];
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int e = 0; e < EPC; ++e) qr[m][e] = qbar[(c + 8 * m) * EPC + e];

  const int base = blockIdx.x * kScoreBPC + warp * kScoreBPW;
  const PT* pk = reinterpret_cast<const PT*>(st.pk);
  uint4 x[kScoreBPW][M];
#pragma unroll
  for (int j = 0; j < kScoreBPW; ++j) {
    const int i = base + j;
    const uint4* row = reinterpret_cast<const uint4*>(
        pk + (((long long)u * s.maxBlk + (i < n_cand ? i : 0)) * 4 + r) * D);
#pragma unroll
    for (int m = 0; m < M; ++m)
      x[j][m] = (i < n_cand) ? __ldg(row + c + 8 * m) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int j = 0; j < kScoreBPW; ++j) {
    float p = 0.f;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float f[EPC];
      widen16<PT>(x[j][m], f);
#pragma unroll
      for (int e = 0; e < EPC; ++e) p = fmaf(f[e], qr[m][e], p);
    }
    p += __shfl_xor_sync(0xffffffffu, p, 1);
    p += __shfl_xor_sync(0xffffffffu, p, 2);
    p += __shfl_xor_sync(0xffffffffu, p, 4);
    p = fmaxf(p, __shfl_xor_sync(0xffffffffu, p, 8));
    p = fmaxf(p, __shfl_xor_sync(0xffffffffu, p, 16));
    const int i = base + j;
    if (lane == 0 && i < n_cand) st.sq[(long long)u * s.maxBlk + i] = p * inv_sqrt_d;
  }
  if constexpr (FUSED) {
    // Count this CTA out; the CTA that completes the count selects. The barrier
    // orders the CTA's score writes before thread 0's fence and add; the last
    // CTA fences again before it reads the other CTAs' scores (through L2).
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int prev = atomicAdd(st.sel_cnt + u, 1);
      s_last = (prev == nct - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0) st.sel_cnt[u] = 0;  // ready for the next step
    if (threadIdx.x == 0 && chunk == 0) trace_mark(st.trace, kTrSel0Begin);
    select_setdiff_unit(s, st, u, cold, chunk, sel_dyn);
    if (threadIdx.x == 0 && chunk == 0) trace_mark(st.trace, kTrSel0End);
  }
}

}  // namespace

template <typename T, typename PT, int MODE>
cudaError_t launch_score_t(const Shape& s, const State& st, int ubase, dim3 grid, float isd,
                           int cold, int chunk, cudaStream_t stream, int occ) {
  const size_t smem = MODE >= 1 ? std::max((size_t)s.maxBlk * 5, smem_for_occupancy(occ)) : 0;
  if (s.d == 64) {
    if (MODE >= 1) {
      static std::atomic<int> lim[64];
      const cudaError_t e = raise_smem_limit((const void*)score_kernel<T, PT, 64, MODE>, smem, lim);
      if (e != cudaSuccess) return e;
    }
    score_kernel<T, PT, 64, MODE><<<grid, 256, smem, stream>>>(s, st, isd, ubase, cold, chunk);
  } else {
    if (MODE >= 1) {
      static std::atomic<int> lim[64];
      const cudaError_t e = raise_smem_limit((const void*)score_kernel<T, PT, 128, MODE>, smem, lim);
      if (e != cudaSuccess) return e;
    }
    score_kernel<T, PT, 128, MODE><<<grid, 256, smem, stream>>>(s, st, isd, ubase, cold, chunk);
  }
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_score_any(const Shape& s, const State& st, int n_cap, int ubase, int ucount,
                             int cold, int chunk, cudaStream_t stream, int occ = 0) {
  if (ucount <= 0) return cudaSuccess;
  if (MODE == 0 && n_cap <= 0) return cudaSuccess;
  // the fused kernel always has a CTA per unit: it selects even an empty candidate set
  dim3 grid(std::max(1, (n_cap + kScoreBPC - 1) / kScoreBPC), ucount);
  const float isd = (float)(1.0 / sqrt((double)s.d));
  if (s.dtype == 0)
    return s.pkb ? launch_score_t<float, __nv_bfloat16, MODE>(s, st, ubase, grid, isd, cold, chunk, stream, occ)
                 : launch_score_t<float, float, MODE>(s, st, ubase, grid, isd, cold, chunk, stream, occ);
  return s.pkb ? launch_score_t<__nv_bfloat16, __nv_bfloat16, MODE>(s, st, ubase, grid, isd, cold, chunk, stream, occ)
               : launch_score_t<__nv_bfloat16, float, MODE>(s, st, ubase, grid, isd, cold, chunk, stream, occ);
}

cudaError_t launch_score(const Shape& s, const State& st, int n_cap, int ubase, int ucount,
                         cudaStream_t stream) {
  return launch_score_any<0>(s, st, n_cap, ubase, ucount, 0, 0, stream);
}

bool score_select_fused_ok(const Shape& s) { return (size_t)s.maxBlk * 5 <= 40960; }

cudaError_t launch_score_select(const Shape& s, const State& st, int n_cap, int ubase, int ucount,
                                int cold, int chunk, cudaStream_t stream, int max_ctas_per_sm) {
  return launch_score_any<1>(s, st, n_cap, ubase, ucount, cold, chunk, stream, max_ctas_per_sm);
}

}  // namespace nosa
