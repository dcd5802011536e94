// CUDA twin of synth/__init__.py: writes the same seeded synthetic inputs on the
// device, bit for bit (integer hashing, exact fp64 arithmetic, then the same
// RNE roundings). Shared by the tests and the bench; holds none of the method's
// arithmetic.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

// Irwin-Hall(12) normal stand-in addressed by (stream, a, h, t, dim); exact.
__device__ __forceinline__ double ih_normal(uint64_t smix, uint64_t stream, uint64_t a, uint64_t h,
                                            uint64_t t, uint64_t dim) {
  const uint64_t base = (stream << 61) | (a << 51) | (h << 44) | (t << 18) | (dim * 4);
  long long s = 0;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const uint64_t w = splitmix64((base + (uint64_t)j) ^ smix);
    s += (long long)((w & 0xFFFF) + ((w >> 16) & 0xFFFF) + ((w >> 32) & 0xFFFF) + (w >> 48));
  }
  return (double)(s - 393210) * (1.0 / 65536.0);
}

template <typename T> __device__ __forceinline__ T store_as(double x);
template <> __device__ __forceinline__ float store_as<float>(double x) { return __double2float_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 store_as<__nv_bfloat16>(double x) {
  return __float2bfloat16_rn(__double2float_rn(x));
}

// k, v: [batch][n][Hkv][d]; e: [batch][n][Hkv] for tokens t0 .. t0+n-1
// (token-major [n][batch][Hkv][d] and [n][batch][Hkv] when step_major).
template <typename T>
__global__ void kv_kernel(T* k, T* v, float* e, int batch, int hkv, int d, long long t0, int n,
                          int block, uint64_t smix, int step_major, int b0) {
  const long long total = (long long)batch * n * hkv * d;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int dim = (int)(i % d);
    long long r = i / d;
    const int h = (int)(r % hkv);
    r /= hkv;
    long long t;
    int b;
    if (step_major) {
      b = (int)(r % batch);
      t = t0 + r / batch;
    } else {
      t = t0 + r % n;
      b = (int)(r / n);
    }
    b += b0;  // request index in the job (a rank's requests start at b0)
    const double c = ih_normal(smix, 0, b, h, t / block, dim);
    const double nz = ih_normal(smix, 1, b, h, t, dim);
    k[i] = store_as<T>(c + 0.5 * nz);
    if (v) v[i] = store_as<T>(ih_normal(smix, 2, b, h, t, dim));
    if (e && dim == 0) e[i / d] = (float)ih_normal(smix, 3, b, h, t, 0);
  }
}

// q: [steps][batch][hq][d], AR(1) over steps, fp64 state (no fused multiply-add);
// the first innovation is scaled by a0 (1 / sqrt(1 - rho^2) for a stationary start).
template <typename T>
__global__ void q_kernel(T* q, int batch, int hq, int d, int steps, double rho, double a0,
                         uint64_t smix, int b0) {
  const int total = batch * hq * d;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int dim = i % d, g = (i / d) % hq, b = b0 + i / (d * hq);
  double x = 0.0;
  for (int s = 0; s < steps; ++s) {
    const double eps = ih_normal(smix, 4, b, g, s, dim);
    x = (s == 0) ? __dmul_rn(a0, eps) : __dadd_rn(__dmul_rn(rho, x), eps);
    q[(long long)s * total + i] = store_as<T>(x);
  }
}

// Integer in [-8, 8] from word j = 0 of the counter (front-end inputs).
__device__ __forceinline__ int small_int(uint64_t smix, uint64_t stream, uint64_t a, uint64_t h,
                                         uint64_t t, uint64_t col) {
  const uint64_t base = (stream << 61) | (a << 51) | (h << 44) | (t << 18) | (col * 4);
  return (int)(splitmix64(base ^ smix) % 17ull) - 8;
}

// x: [n][batch][D] bf16 hidden states of tokens t0 .. t0+n-1 (integers x 2^-3).
__global__ void hidden_kernel(__nv_bfloat16* x, int batch, int D, long long t0, int n,
                              uint64_t smix, int b0) {
  const long long total = (long long)n * batch * D;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int col = (int)(i % D);
    const long long r = i / D;
    const int b = b0 + (int)(r % batch);
    const long long t = t0 + r / batch;
    x[i] = __float2bfloat16_rn((float)small_int(smix, 5, b, 0, t, col) * 0.125f);
  }
}

// W: [F][D] bf16 packed front-end weights (integers x 2^-8).
__global__ void weight_kernel(__nv_bfloat16* W, int F, int D, uint64_t smix) {
  const long long total = (long long)F * D;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int col = (int)(i % D);
    const long long row = i / D;
    W[i] = __float2bfloat16_rn((float)small_int(smix, 6, 0, 0, row, col) * 0.00390625f);
  }
}

uint64_t seed_mix(uint64_t seed) {
  uint64_t x = seed + 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

}  // namespace

extern "C" {

// dtype 0 = fp32, 1 = bf16. Returns a cudaError_t.
// b0: index of the first request (requests b0 .. b0 + batch - 1 of the job).
int synth_kv(void* k, void* v, float* e, int batch, int hkv, int d, long long t0, int n,
             int block, unsigned long long seed, int dtype, int step_major, int b0, void* stream) {
  const uint64_t smix = seed_mix(seed);
  const long long total = (long long)batch * n * hkv * d;
  const int threads = 256;
  const long long want = (total + threads - 1) / threads;
  const int grid = (int)(want < 65536 ? want : 65536);
  cudaStream_t s = (cudaStream_t)stream;
  if (total == 0) return 0;
  if (dtype == 0)
    kv_kernel<float><<<grid, threads, 0, s>>>((float*)k, (float*)v, e, batch, hkv, d, t0, n,
                                               block, smix, step_major, b0);
  else
    kv_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>((__nv_bfloat16*)k, (__nv_bfloat16*)v, e,
                                                       batch, hkv, d, t0, n, block, smix, step_major,
                                                       b0);
  return (int)cudaGetLastError();
}

int synth_queries(void* q, int batch, int hq, int d, int steps, double rho, double a0,
                  unsigned long long seed, int dtype, int b0, void* stream) {
  const uint64_t smix = seed_mix(seed);
  const int total = batch * hq * d;
  cudaStream_t s = (cudaStream_t)stream;
  if (total == 0 || steps == 0) return 0;
  if (dtype == 0)
    q_kernel<float><<<(total + 127) / 128, 128, 0, s>>>((float*)q, batch, hq, d, steps, rho, a0,
                                                         smix, b0);
  else
    q_kernel<__nv_bfloat16><<<(total + 127) / 128, 128, 0, s>>>((__nv_bfloat16*)q, batch, hq, d,
                                                                 steps, rho, a0, smix, b0);
  return (int)cudaGetLastError();
}

int synth_hidden(void* x, int batch, int D, long long t0, int n, unsigned long long seed,
                 int b0, void* stream) {
  const long long total = (long long)n * batch * D;
  if (total == 0) return 0;
  const long long want = (total + 255) / 256;
  hidden_kernel<<<(int)(want < 65536 ? want : 65536), 256, 0, (cudaStream_t)stream>>>(
      (__nv_bfloat16*)x, batch, D, t0, n, seed_mix(seed), b0);
  return (int)cudaGetLastError();
}

int synth_proj_weights(void* W, int F, int D, unsigned long long seed, void* stream) {
  const long long total = (long long)F * D;
  if (total == 0) return 0;
  const long long want = (total + 255) / 256;
  weight_kernel<<<(int)(want < 65536 ? want : 65536), 256, 0, (cudaStream_t)stream>>>(
      (__nv_bfloat16*)W, F, D, seed_mix(seed));
  return (int)cudaGetLastError();
}

}  // extern "C"
