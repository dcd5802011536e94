// UVA gather of missing blocks into freed slots.
//
// NOSA technical summary, Methodology §2 "High-Bandwidth Communication": the
// host-to-device recall is done by custom kernels that read pinned host memory
// through unified virtual addressing, instead of many small copy calls. Here
// every load-list entry (block, slot, src) of a chunk of units is one work item:
// the set-difference leaves each unit's list and count, every CTA numbers the
// chunk's entries itself (an exclusive prefix of the units' counts in shared
// memory, a binary search per entry), a small grid of CTAs takes the entries in
// turn, and each CTA copies one block unit at a time, every thread issuing
// all its loads before storing, so that enough host-link transactions are in
// flight without flooding the memory system (the gather runs next to HBM-bound
// kernels, whose traffic queues behind slow host reads).
//
// Two load widths: 16-byte vectors (9 per thread per pass), or 32-byte vectors
// (ld.global.nc.v8.b32 with a 256-byte L2 fetch hint, 5 per thread per pass),
// which halve the number of host read requests per byte.
#include "nosa_internal.cuh"

#include <cstdlib>

namespace nosa {
namespace {

constexpr int kGatherThreads = 256;

struct alignas(32) V32 {
  uint32_t r[8];
};

__device__ __forceinline__ V32 load_host32(const V32* p) {
  V32 v;
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::256B.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(v.r[0]), "=r"(v.r[1]), "=r"(v.r[2]), "=r"(v.r[3]), "=r"(v.r[4]), "=r"(v.r[5]),
        "=r"(v.r[6]), "=r"(v.r[7])
      : "l"(p));
  return v;
}

__device__ __forceinline__ void store32(V32* p, const V32& v) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.r[0]),
               "r"(v.r[1]), "r"(v.r[2]), "r"(v.r[3]), "r"(v.r[4]), "r"(v.r[5]), "r"(v.r[6]),
               "r"(v.r[7])
               : "memory");
}

template <typename V> struct Mover;
template <> struct Mover<int4> {
  static constexpr int kPer = 9;
  static __device__ __forceinline__ int4 load(const int4* p) { return __ldcs(p); }
  static __device__ __forceinline__ void store(int4* p, const int4& v) { *p = v; }
};
template <> struct Mover<V32> {
  static constexpr int kPer = 5;
  static __device__ __forceinline__ V32 load(const V32* p) { return load_host32(p); }
  static __device__ __forceinline__ void store(V32* p, const V32& v) { store32(p, v); }
};

constexpr int kGatherTile = 2048;                     // units numbered per pass
constexpr int kGatherSer = kGatherTile / kGatherThreads;  // consecutive units per thread

// grid = the chunk's CTAs (any count), block = kGatherThreads. Units
// [ubase, ubase + ucount); entry g of the chunk (units in order, each unit's
// loads in list order) goes to CTA g % gridDim.x.
template <typename V>
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(Shape s, State st, int ubase,
                                                                int ucount, int chunk) {
  constexpr int kPer = Mover<V>::kPer;
  griddep_wait();  // the chunk's selection (programmatic edge in the step graph)
  TraceScope trace_scope(st.trace, chunk < 8 ? kTrGather + chunk : -1);
  __shared__ int pre[kGatherTile + 1];  // exclusive prefix of the tile's load counts
  __shared__ int warp_tot[kGatherThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int vpp = (int)(s.payload / sizeof(V));  // payload is a multiple of 256 B
  long long done = 0;                            // entries of the earlier tiles
  for (int t0 = 0; t0 < ucount; t0 += kGatherTile) {
    const int nt = min(kGatherTile, ucount - t0);
    int v[kGatherSer];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kGatherSer; ++i) {
      const int idx = threadIdx.x * kGatherSer + i;
      v[i] = idx < nt ? st.nload[ubase + t0 + idx] : 0;
      sum += v[i];
    }
    int x = sum;  // inclusive warp scan, then the warps' totals
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int ex = x - sum, tot = 0;
#pragma unroll
    for (int w = 0; w < kGatherThreads / 32; ++w) {
      ex += (w < warp) ? warp_tot[w] : 0;
      tot += warp_tot[w];
    }
#pragma unroll
    for (int i = 0; i < kGatherSer; ++i) {
      pre[threadIdx.x * kGatherSer + i] = ex;
      ex += v[i];
    }
    if (threadIdx.x == 0) pre[kGatherTile] = tot;
    __syncthreads();
    // pre[i] for i >= nt is tot (those units count 0), so pre[nt] = tot.
    const int first = (int)(((long long)blockIdx.x - done % gridDim.x + gridDim.x) % gridDim.x);
    for (int w = first; w < tot; w += gridDim.x) {
      int lo = 0, hi = nt;  // pre[lo] <= w < pre[hi]: the unit holding entry w
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= w) lo = mid; else hi = mid;
      }
      const int u = ubase + t0 + lo;
      const int entry = u * s.k + (w - pre[lo]);
      const int blk = st.loads[3 * entry], slot = st.loads[3 * entry + 1];
      const int src = st.loads[3 * entry + 2];
      const V* sp = reinterpret_cast<const V*>(
          src ? st.tail + ((long long)u * 2 + (blk & 1)) * s.payload
              : st.host + ((long long)u * s.maxBlk + blk) * s.payload);
      V* dp = reinterpret_cast<V*>(st.slots + ((long long)u * s.k + slot) * s.payload);
      for (int base = 0; base < vpp; base += kGatherThreads * kPer) {
        V r[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int idx = base + i * kGatherThreads + threadIdx.x;
          if (idx < vpp) r[i] = Mover<V>::load(sp + idx);
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int idx = base + i * kGatherThreads + threadIdx.x;
          if (idx < vpp) Mover<V>::store(dp + idx, r[i]);
        }
      }
    }
    done += tot;
    __syncthreads();  // pre and warp_tot are rewritten by the next tile
  }
  // only now: the filled-slot attention's CTAs would otherwise hold SMs while waiting
  griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_gather(const Shape& s, const State& st, int grid, int ubase, int ucount,
                          int chunk, bool wide, cudaStream_t stream) {
  if (wide)
    gather_kernel<V32><<<grid, kGatherThreads, 0, stream>>>(s, st, ubase, ucount, chunk);
  else
    gather_kernel<int4><<<grid, kGatherThreads, 0, stream>>>(s, st, ubase, ucount, chunk);
  return cudaGetLastError();
}

}  // namespace nosa

// ---------------------------------------------------------------------------
// Self-test of the bounded waits: one thread arms an mbarrier that nothing will
// ever complete and waits on it with the same bounded wait the attention kernel
// uses; the wait must give up after limit_ns and report it.
// ---------------------------------------------------------------------------
namespace nosa {
namespace {
__global__ void bounded_wait_probe_kernel(unsigned long long limit_ns, int* result) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    const uint64_t t0 = global_ns();
    const bool done = mbar_wait_bounded(&bar, 0, limit_ns);
    result[0] = done ? kDevErrNone : kDevErrWaitTimeout;
    result[1] = (int)((global_ns() - t0) / 1000000ull);  // elapsed ms
    mbar_arrive(&bar);  // complete the phase so the barrier is left quiescent
  }
}
}  // namespace

namespace {
__global__ void trace_reset_kernel(unsigned long long* trace) {
  const int i = threadIdx.x;
  if (i < kTraceSlots) trace[2 * i] = ~0ull;  // starts: min-reduced; ends stay 0
}
}  // namespace

cudaError_t launch_trace_reset(unsigned long long* trace, cudaStream_t stream) {
  trace_reset_kernel<<<1, 64, 0, stream>>>(trace);
  return cudaGetLastError();
}

cudaError_t launch_bounded_wait_probe(unsigned long long limit_ns, int* result,
                                      cudaStream_t stream) {
  bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(limit_ns, result);
  return cudaGetLastError();
}
}  // namespace nosa
