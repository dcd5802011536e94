// Block-sparse decode attention for callers that cannot allocate device memory.
//
// nosa_sparse_attention keeps its split-K partials (and the per-unit counters
// and error word of its merge) in a workspace the caller allocates. Some
// callers have no way to get one: a serving engine or framework that reserves
// all device memory up front in its own pool (a cudaMalloc from inside this
// library can then fail even though the pool holds free memory, and memory the
// pool does not know about upsets its accounting), or a latency-critical loop
// that must not call cudaMalloc / cudaFree because they can synchronise the
// device. nosa_sparse_attention_noalloc serves them: the same kernel, with its
// scratch in one fixed array of this library's device memory.
//
// The array is a file-scope static __device__ object of kNoAllocScratchBytes
// (16 MiB): every GPU that loads the library holds it until the process exits.
// In host code its name is only a host-side stand-in, never a device address,
// so the first call on each device (with that device current) asks the runtime
// for the array's device address once and caches it with the device's current
// context; make that first call before any stream capture. A call that finds
// another context current (after cudaDeviceReset the module loads again and
// the array may move) looks the address up again, so that call too must come
// before any stream capture. All calls share the array and it keeps the last call's
// contents: the merge counters and the error word are cleared by each call
// (cudaMemsetAsync on the caller's stream), and calls that overlap on the GPU
// (different streams, or different host threads without ordering) race on it.
#include "nosa.h"
#include "nosa_internal.cuh"

#include <mutex>
#include <string>

namespace nosa {
void set_thread_error(const std::string& msg);  // defined with the other entry points
}

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];
CUcontext g_scratch_ctx[kMaxDevices];

// The calling thread's current driver context (nullptr if the driver offers no
// query); fetched through the runtime's entry-point lookup, so the library needs
// no link to the driver library.
CUcontext current_context() {
  using CtxGetCurrent = CUresult (*)(CUcontext*);
  static CtxGetCurrent fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return (CtxGetCurrent) nullptr;
    }
    return reinterpret_cast<CtxGetCurrent>(ptr);
  }();
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of the scratch array on device `dev` (current): looked up on
// the first call and again whenever the device's current context has changed.
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const CUcontext ctx = current_context();
  if (g_scratch_addr[dev] == nullptr || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = current_context();  // (the lookup makes the context current)
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" nosa_status nosa_sparse_attention_noalloc(const nosa_config* cfg, const void* units,
                                                     int64_t n_units, const int32_t* block_tab,
                                                     int32_t n_blocks, const void* tail,
                                                     int32_t tail_len, const void* q, void* out,
                                                     float* lse, void* stream) {
  char why[256];
  const nosa_status vs = nosa_config_validate(cfg, why, sizeof(why));
  if (vs != NOSA_OK) {
    nosa::set_thread_error(why);
    return vs;
  }
  if (cfg->device >= kMaxDevices || n_blocks < 0) {
    nosa::set_thread_error("device ordinal or n_blocks out of range");
    return NOSA_ERR_INVALID_ARG;
  }
  const size_t need = nosa_attention_workspace_bytes(cfg, n_blocks);
  if (need == 0 || need > kNoAllocScratchBytes) {
    nosa::set_thread_error("nosa_sparse_attention_noalloc: this shape needs " +
                           std::to_string(need) + " bytes of split-K scratch, more than the " +
                           std::to_string(kNoAllocScratchBytes) +
                           "-byte static array; use nosa_sparse_attention with a workspace");
    return NOSA_ERR_CAPACITY;
  }
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != cfg->device) cudaSetDevice(cfg->device);
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(cfg->device, &scratch);
  if (prev >= 0 && prev != cfg->device) cudaSetDevice(prev);
  if (e != cudaSuccess) {
    nosa::set_thread_error(std::string("cudaGetSymbolAddress of the scratch array failed: ") +
                           cudaGetErrorString(e));
    return NOSA_ERR_CUDA;
  }
  return nosa_sparse_attention(cfg, units, n_units, block_tab, n_blocks, tail, tail_len, q, out,
                               lse, scratch, kNoAllocScratchBytes, stream);
}
