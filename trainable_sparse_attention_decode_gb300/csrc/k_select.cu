// Dual selection and set-difference as a kernel of their own: one CTA per unit
// of a chunk, after the scoring kernel (the device code is in k_select.cuh; the
// fused scoring kernel in k_score.cu runs the same code in the last scoring CTA
// of each unit instead).
#include "k_select.cuh"

namespace nosa {
namespace {

// grid = units of the chunk, block = kSelThreads. Dynamic shared memory:
// key [maxBlk] u32 + flag [maxBlk] u8.
__global__ void __launch_bounds__(kSelThreads) select_setdiff_kernel(Shape s, State st, int cold,
                                                                     int ubase, int chunk) {
  extern __shared__ __align__(16) uint8_t dyn[];
  TraceScope trace_scope(st.trace, chunk < 8 ? kTrSelect + chunk : -1);
  select_setdiff_unit(s, st, ubase + blockIdx.x, cold, chunk, dyn);
}

}  // namespace

cudaError_t launch_select_setdiff(const Shape& s, const State& st, int cold, int ubase,
                                  int ucount, int chunk, cudaStream_t stream) {
  const size_t smem = (size_t)s.maxBlk * 5;
  static std::atomic<int> lim[64];
  cudaError_t err = raise_smem_limit((const void*)select_setdiff_kernel, smem, lim);
  if (err != cudaSuccess) return err;
  select_setdiff_kernel<<<ucount, kSelThreads, smem, stream>>>(s, st, cold, ubase, chunk);
  return cudaGetLastError();
}

}  // namespace nosa
