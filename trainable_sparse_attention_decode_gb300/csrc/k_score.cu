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
#include "nosa_internal.cuh"

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

template <typename T, typename PT, int D>
__global__ void __launch_bounds__(256) score_kernel(Shape s, State st, float inv_sqrt_d,
                                                    int ubase) {
  constexpr int EPC = 16 / (int)sizeof(PT);  // pooled values per 16-byte chunk
  constexpr int M = D / EPC / 8;             // chunks per lane per pooled row
  static_assert(M >= 1, "row too short for 8 lanes");
  __shared__ __align__(16) float qbar[D];
  const int n_cand = st.io->n_cand;
  if (blockIdx.x * kScoreBPC >= n_cand) return;  // grid sized for a larger count
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
}

}  // namespace

template <typename T, typename PT>
cudaError_t launch_score_t(const Shape& s, const State& st, int ubase, dim3 grid, float isd,
                           cudaStream_t stream) {
  if (s.d == 64)
    score_kernel<T, PT, 64><<<grid, 256, 0, stream>>>(s, st, isd, ubase);
  else
    score_kernel<T, PT, 128><<<grid, 256, 0, stream>>>(s, st, isd, ubase);
  return cudaGetLastError();
}

cudaError_t launch_score(const Shape& s, const State& st, int n_cap, int ubase, int ucount,
                         cudaStream_t stream) {
  if (n_cap <= 0 || ucount <= 0) return cudaSuccess;
  dim3 grid((n_cap + kScoreBPC - 1) / kScoreBPC, ucount);
  const float isd = (float)(1.0 / sqrt((double)s.d));
  if (s.dtype == 0)
    return s.pkb ? launch_score_t<float, __nv_bfloat16>(s, st, ubase, grid, isd, stream)
                 : launch_score_t<float, float>(s, st, ubase, grid, isd, stream);
  return s.pkb ? launch_score_t<__nv_bfloat16, __nv_bfloat16>(s, st, ubase, grid, isd, stream)
               : launch_score_t<__nv_bfloat16, float>(s, st, ubase, grid, isd, stream);
}

}  // namespace nosa
