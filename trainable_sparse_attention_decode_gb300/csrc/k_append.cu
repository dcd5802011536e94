// Append + incremental two-stage pooling (first stage).
//
// NOSA technical summary, Methodology §1 "Block-Wise Implementation": keys and
// eviction logits are mean-pooled inside 16-token sub-blocks; the block's
// eviction score is the max over its sub-block means. Both are produced here,
// incrementally: a sub-block is averaged the moment its 16th token arrives (fp32
// sum in token order, then x 1/16), and the block's eviction score is the
// running max of its completed sub-block means. The query-dependent max over
// sub-blocks happens in the score kernel.
//
// Block lifecycle (the newest block is the "tail"): tokens go into the tail
// buffer (block b uses buffer b % 2). When a token opens a new block, the block
// before it becomes a candidate: it is marked eligible for the query-agnostic
// selection and written back to the pinned host store (Methodology §2: the KV
// cache lives in host memory in block-sized units).
#include "nosa_internal.cuh"

namespace nosa {
namespace {

// Copies one block unit (16-byte vectors) with the whole CTA.
__device__ __forceinline__ void copy_unit(uint8_t* dst, const uint8_t* src, long long payload) {
  const int nvec = (int)(payload / 16);
  const int4* s4 = reinterpret_cast<const int4*>(src);
  int4* d4 = reinterpret_cast<int4*>(dst);
  for (int i = threadIdx.x; i < nvec; i += blockDim.x) d4[i] = s4[i];
}

// One decode-step token per unit. grid = U, block = 128 threads (d <= 128).
// CTA 0 also publishes the step's arguments (StepIO) for the kernels after it.
template <typename T>
__global__ void __launch_bounds__(128) append_step_kernel(Shape s, State st, StepArgs a) {
  griddep_launch_dependents();  // the chunks' scoring may become resident (it waits)
  TraceScope trace_scope(st.trace, kTrAppend);
  const T* __restrict__ k_new = static_cast<const T*>(a.k_new);
  const T* __restrict__ v_new = static_cast<const T*>(a.v_new);
  const float* __restrict__ e_new = a.e_new;
  const int u = blockIdx.x;
  const int t = a.L_old;
  const int blk = t / s.B, pos = t % s.B;
  uint8_t* cur = st.tail + ((long long)u * 2 + (blk & 1)) * s.payload;
  if (u == 0 && threadIdx.x == 0) {
    StepIO io;
    io.q = a.q;
    io.out = a.out;
    io.lse = a.lse;
    io.L_old = a.L_old;
    io.n_cand = blk;  // (L_old + 1 - 1) / B complete blocks precede the tail
    io.tail_len = pos + 1;
    io.just_completed = (pos == 0 && blk > 0) ? blk - 1 : -1;
    io.tail_off = (long long)(blk & 1) * s.payload;
    *st.io = io;
  }

  // The block before a newly opened one becomes a candidate.
  if (pos == 0 && blk > 0) {
    const int cb = blk - 1;
    const uint8_t* old = st.tail + ((long long)u * 2 + (cb & 1)) * s.payload;
    copy_unit(st.host + ((long long)u * s.maxBlk + cb) * s.payload, old, s.payload);
    if (threadIdx.x == 0) atomicOr(&st.elig[(long long)u * s.W + cb / 32], 1u << (cb % 32));
    __threadfence_system();
  }

  // Write the token into the tail unit.
  const long long in_row = (long long)u * s.d;  // [b][Hkv][d] row of unit u = b*Hkv + h
  for (int dim = threadIdx.x; dim < s.d; dim += blockDim.x) {
    *reinterpret_cast<T*>(cur + k_off(pos, dim, s.B, s.elt)) = k_new[in_row + dim];
    *reinterpret_cast<T*>(cur + v_off(pos, dim, s.B, s.d, s.elt)) = v_new[in_row + dim];
  }
  const float e_tok = e_new[u];
  if (threadIdx.x == 0) *reinterpret_cast<float*>(cur + e_off(pos, s.B, s.d, s.elt)) = e_tok;

  // Running fp32 sums of the open sub-block (0 + k_0 + k_1 + ..., token order);
  // when the sub-block completes: mean key, mean eviction logit, running block max.
  const bool first = (pos % s.S) == 0, last = (pos % s.S) == s.S - 1;
  const int sb = pos / s.S;
  for (int dim = threadIdx.x; dim < s.d; dim += blockDim.x) {
    const float r = (first ? 0.f : st.ksum[in_row + dim]) + to_f32(k_new[in_row + dim]);
    if (last)
      store_pooled(s, st.pk, (((long long)u * s.maxBlk + blk) * s.P + sb) * s.d + dim,
                   r * (1.0f / s.S));
    else
      st.ksum[in_row + dim] = r;
  }
  if (threadIdx.x == 0) {
    const float r = (first ? 0.f : st.esum[u]) + e_tok;
    if (last) {
      const float eb = r * (1.0f / s.S);
      const long long bi = (long long)u * s.maxBlk + blk;
      st.sube[bi * s.P + sb] = eb;
      st.se[bi] = (sb == 0) ? eb : fmaxf(st.se[bi], eb);
    } else {
      st.esum[u] = r;
    }
  }
}

// The tail block `blk` (full) becomes a candidate before a bulk append opens
// the next block. grid = U.
__global__ void __launch_bounds__(256) promote_tail_kernel(Shape s, State st, int blk) {
  const int u = blockIdx.x;
  const uint8_t* src = st.tail + ((long long)u * 2 + (blk & 1)) * s.payload;
  copy_unit(st.host + ((long long)u * s.maxBlk + blk) * s.payload, src, s.payload);
  if (threadIdx.x == 0) atomicOr(&st.elig[(long long)u * s.W + blk / 32], 1u << (blk % 32));
  __threadfence_system();
}

// Bulk append of n tokens per request. grid = (blocks touched, U), one block
// unit assembled in shared memory per CTA. Inputs k, v [batch][n][Hkv][d],
// e [batch][n][Hkv].
template <typename T>
__global__ void __launch_bounds__(256) append_bulk_kernel(Shape s, State st,
                                                          const T* __restrict__ k,
                                                          const T* __restrict__ v,
                                                          const float* __restrict__ e,
                                                          int L_old, int n) {
  extern __shared__ __align__(16) uint8_t unit_s[];
  __shared__ float ebar_s[8];
  const int u = blockIdx.y, b = u / s.Hkv, h = u % s.Hkv;
  const int first_blk = L_old / s.B;
  const int blk = first_blk + blockIdx.x;
  const int L_new = L_old + n;
  const int last_blk = (L_new - 1) / s.B;
  const int t_lo = max(L_old, blk * s.B), t_hi = min(L_new, (blk + 1) * s.B);
  const bool resume = (blk == first_blk) && (L_old % s.B != 0);
  uint8_t* tail_buf = st.tail + ((long long)u * 2 + (blk & 1)) * s.payload;
  const int nvec = (int)(s.payload / 16);

  // Tokens already in the tail unit, else zeros.
  for (int i = threadIdx.x; i < nvec; i += blockDim.x)
    reinterpret_cast<int4*>(unit_s)[i] =
        resume ? reinterpret_cast<const int4*>(tail_buf)[i] : make_int4(0, 0, 0, 0);
  __syncthreads();

  const int nt = t_hi - t_lo;
  for (int idx = threadIdx.x; idx < nt * s.d; idx += blockDim.x) {
    const int i = idx / s.d, dim = idx % s.d;
    const int t = t_lo + i, pos = t - blk * s.B;
    const long long src = (((long long)b * n + (t - L_old)) * s.Hkv + h) * s.d + dim;
    *reinterpret_cast<T*>(unit_s + k_off(pos, dim, s.B, s.elt)) = k[src];
    *reinterpret_cast<T*>(unit_s + v_off(pos, dim, s.B, s.d, s.elt)) = v[src];
  }
  for (int i = threadIdx.x; i < nt; i += blockDim.x) {
    const int t = t_lo + i, pos = t - blk * s.B;
    *reinterpret_cast<float*>(unit_s + e_off(pos, s.B, s.d, s.elt)) =
        e[((long long)b * n + (t - L_old)) * s.Hkv + h];
  }
  __syncthreads();

  // Sub-blocks completed by this call.
  const int pos_lo = t_lo - blk * s.B, pos_hi = t_hi - blk * s.B;
  const long long bi = (long long)u * s.maxBlk + blk;
  for (int sb = 0; sb < s.P; ++sb) {
    const int end = (sb + 1) * s.S;
    if (end > pos_hi || end <= pos_lo) continue;
    for (int dim = threadIdx.x; dim < s.d; dim += blockDim.x) {
      float acc = 0.f;
      for (int j = 0; j < s.S; ++j)
        acc += to_f32(*reinterpret_cast<const T*>(unit_s + k_off(sb * s.S + j, dim, s.B, s.elt)));
      store_pooled(s, st.pk, (bi * s.P + sb) * s.d + dim, acc * (1.0f / s.S));
    }
  }
  // A call that ends inside a sub-block leaves that sub-block's running sums
  // (token order, from 0) for the decode steps that complete it.
  if (blk == last_blk && pos_hi % s.S != 0) {
    const int o0 = (pos_hi / s.S) * s.S;
    for (int dim = threadIdx.x; dim < s.d; dim += blockDim.x) {
      float r = 0.f;
      for (int j = o0; j < pos_hi; ++j)
        r += to_f32(*reinterpret_cast<const T*>(unit_s + k_off(j, dim, s.B, s.elt)));
      st.ksum[(long long)u * s.d + dim] = r;
    }
    if (threadIdx.x == 0) {
      float r = 0.f;
      for (int j = o0; j < pos_hi; ++j)
        r += *reinterpret_cast<const float*>(unit_s + e_off(j, s.B, s.d, s.elt));
      st.esum[u] = r;
    }
  }
  if (threadIdx.x == 0) {
    float se_run = 0.f;
    int ncomplete = 0;
    for (int sb = 0; sb < s.P; ++sb) {
      const int end = (sb + 1) * s.S;
      if (end > pos_hi) break;
      float eb;
      if (end <= pos_lo) {
        eb = st.sube[bi * s.P + sb];  // completed by an earlier call
      } else {
        float ea = 0.f;
        for (int j = 0; j < s.S; ++j)
          ea += *reinterpret_cast<const float*>(unit_s + e_off(sb * s.S + j, s.B, s.d, s.elt));
        eb = ea * (1.0f / s.S);
        st.sube[bi * s.P + sb] = eb;
      }
      se_run = (sb == 0) ? eb : fmaxf(se_run, eb);
      ++ncomplete;
    }
    if (ncomplete > 0) st.se[bi] = se_run;
    ebar_s[0] = se_run;
  }
  __syncthreads();

  if (blk < last_blk) {
    // Complete, and a candidate once this call returns: host store + eligibility.
    copy_unit(st.host + bi * s.payload, unit_s, s.payload);
    if (threadIdx.x == 0) atomicOr(&st.elig[(long long)u * s.W + blk / 32], 1u << (blk % 32));
    __threadfence_system();
  } else {
    copy_unit(tail_buf, unit_s, s.payload);
  }
}

}  // namespace

cudaError_t launch_append_step(const Shape& s, const State& st, const StepArgs& a,
                               cudaStream_t stream) {
  if (s.dtype == 0)
    append_step_kernel<float><<<s.U, 128, 0, stream>>>(s, st, a);
  else
    append_step_kernel<__nv_bfloat16><<<s.U, 128, 0, stream>>>(s, st, a);
  return cudaGetLastError();
}

cudaError_t launch_promote_tail(const Shape& s, const State& st, int blk, cudaStream_t stream) {
  promote_tail_kernel<<<s.U, 256, 0, stream>>>(s, st, blk);
  return cudaGetLastError();
}

cudaError_t launch_append_bulk(const Shape& s, const State& st, const void* k, const void* v,
                               const float* e, int L_old, int n, cudaStream_t stream) {
  const int first_blk = L_old / s.B, last_blk = (L_old + n - 1) / s.B;
  dim3 grid(last_blk - first_blk + 1, s.U);
  const size_t smem = (size_t)s.payload;
  cudaError_t err;
  if (s.dtype == 0) {
    err = cudaFuncSetAttribute(append_bulk_kernel<float>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    append_bulk_kernel<float><<<grid, 256, smem, stream>>>(s, st, (const float*)k,
                                                           (const float*)v, e, L_old, n);
  } else {
    err = cudaFuncSetAttribute(append_bulk_kernel<__nv_bfloat16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    append_bulk_kernel<__nv_bfloat16><<<grid, 256, smem, stream>>>(
        s, st, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, e, L_old, n);
  }
  return cudaGetLastError();
}

}  // namespace nosa
