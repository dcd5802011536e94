// UVA gather of missing blocks into freed slots.
//
// NOSA technical summary, Methodology §2 "High-Bandwidth Communication": the
// host-to-device recall is done by custom kernels that read pinned host memory
// through unified virtual addressing, instead of many small copy calls. Here
// every load-list entry (block, slot, src) of every unit is one work item in a
// flat list built by the set-difference kernel; a grid of CTAs strides over the
// items, and each CTA copies one block unit at a time with all its threads
// issuing up to 9 independent 16-byte loads each before storing, so that many
// host-link transactions are in flight per SM.
#include "nosa_internal.cuh"

namespace nosa {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherVPT = 9;  // 16-byte vectors per thread per pass

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(Shape s, State st, int ubase,
                                                                int chunk) {
  const int n = st.work_count[chunk];
  const int32_t* work = st.work + (long long)ubase * s.k;  // this chunk's list
  const int vpp = (int)(s.payload / 16);
  for (int w = blockIdx.x; w < n; w += gridDim.x) {
    const int entry = work[w];
    const int u = entry / s.k;
    const int blk = st.loads[3 * entry], slot = st.loads[3 * entry + 1];
    const int src = st.loads[3 * entry + 2];
    const int4* sp = reinterpret_cast<const int4*>(
        src ? st.tail + ((long long)u * 2 + (blk & 1)) * s.payload
            : st.host + ((long long)u * s.maxBlk + blk) * s.payload);
    int4* dp = reinterpret_cast<int4*>(st.slots + ((long long)u * s.k + slot) * s.payload);
    for (int base = 0; base < vpp; base += kGatherThreads * kGatherVPT) {
      int4 r[kGatherVPT];
#pragma unroll
      for (int i = 0; i < kGatherVPT; ++i) {
        const int idx = base + i * kGatherThreads + threadIdx.x;
        if (idx < vpp) r[i] = __ldcs(sp + idx);
      }
#pragma unroll
      for (int i = 0; i < kGatherVPT; ++i) {
        const int idx = base + i * kGatherThreads + threadIdx.x;
        if (idx < vpp) dp[idx] = r[i];
      }
    }
  }
}

}  // namespace

cudaError_t launch_gather(const Shape& s, const State& st, int grid, int ubase, int chunk,
                          cudaStream_t stream) {
  gather_kernel<<<grid, kGatherThreads, 0, stream>>>(s, st, ubase, chunk);
  return cudaGetLastError();
}

}  // namespace nosa
