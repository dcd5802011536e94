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

template <typename T, int D>
__global__ void __launch_bounds__(256) score_kernel(Shape s, State st, const T* __restrict__ q,
                                                    int n_cand, float inv_sqrt_d, int ubase) {
  constexpr int M = D / 32;  // float4 per lane per pooled row
  __shared__ __align__(16) float qbar[D];
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
  float4 qr[M];
#pragma unroll
  for (int m = 0; m < M; ++m) qr[m] = *reinterpret_cast<const float4*>(&qbar[c * 4 + 32 * m]);

  const int base = blockIdx.x * kScoreBPC + warp * kScoreBPW;
  float4 x[kScoreBPW][M];
#pragma unroll
  for (int j = 0; j < kScoreBPW; ++j) {
    const int i = base + j;
    const float4* row = reinterpret_cast<const float4*>(
        st.pk + (((long long)u * s.maxBlk + (i < n_cand ? i : 0)) * 4 + r) * D);
#pragma unroll
    for (int m = 0; m < M; ++m)
      x[j][m] = (i < n_cand) ? __ldg(row + c + 8 * m) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int j = 0; j < kScoreBPW; ++j) {
    float p = 0.f;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      p = fmaf(x[j][m].x, qr[m].x, p);
      p = fmaf(x[j][m].y, qr[m].y, p);
      p = fmaf(x[j][m].z, qr[m].z, p);
      p = fmaf(x[j][m].w, qr[m].w, p);
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

cudaError_t launch_score(const Shape& s, const State& st, const void* q, int n_cand, int ubase,
                         int ucount, cudaStream_t stream) {
  if (n_cand <= 0 || ucount <= 0) return cudaSuccess;
  dim3 grid((n_cand + kScoreBPC - 1) / kScoreBPC, ucount);
  const float isd = (float)(1.0 / sqrt((double)s.d));
  if (s.dtype == 0) {
    if (s.d == 64) score_kernel<float, 64><<<grid, 256, 0, stream>>>(s, st, (const float*)q, n_cand, isd, ubase);
    else score_kernel<float, 128><<<grid, 256, 0, stream>>>(s, st, (const float*)q, n_cand, isd, ubase);
  } else {
    if (s.d == 64)
      score_kernel<__nv_bfloat16, 64><<<grid, 256, 0, stream>>>(s, st, (const __nv_bfloat16*)q, n_cand, isd, ubase);
    else
      score_kernel<__nv_bfloat16, 128><<<grid, 256, 0, stream>>>(s, st, (const __nv_bfloat16*)q, n_cand, isd, ubase);
  }
  return cudaGetLastError();
}

}  // namespace nosa
