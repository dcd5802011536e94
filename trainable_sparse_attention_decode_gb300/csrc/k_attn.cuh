// Block-sparse flash-decoding attention with the exp-delayed eviction logit.
//
// NOSA technical summary, Methodology §1 "ED-DMA (Exp-Delayed DMA)": selection
// works on pre-exp eviction scores and the exponential is applied in the
// attention stage. For a query head g of unit (b, h) and every attended token j
// (the tokens of the unit's selected blocks and of its tail block):
//     l_j = q_g . k_j / sqrt(d) + e_j,   out_g = sum_j softmax(l)_j v_j,
//     lse_g = log sum_j exp(l_j).
// The kernel works in the log2 domain (q is pre-scaled by log2(e)/sqrt(d) and
// e_j by log2(e)), an identity.
//
// Split-K: grid = (splits, units). A CTA (4 warps) walks its share of the unit's
// block list; one thread streams whole block units (K | V | e, 16.6 or 33 KB)
// into a ring of shared-memory stages with bulk asynchronous copies completing
// on mbarriers (no tensor map: the units are contiguous). Each warp owns 16 of
// the 64 tokens of every block and keeps its own running max / sum / accumulator;
// the 4 warps merge at the end and the CTA writes one partial per query head.
// Several launches may contribute partials to the same units (the decode step
// runs one over the slots it already held while the gather fills the others,
// then one over the freshly filled slots); the CTA that publishes a unit's last
// partial merges them all into the output (a fence-and-count pattern, no spin).
//
// Token work inside a warp:
//   logits : lane (t = lane % 16, half = lane / 16) dots token t with one half of
//            the head dimension (K is 16-byte-chunk-major in the unit, so the 16
//            lanes of a half read 16 consecutive chunks: no bank conflicts), the
//            halves are added with one shuffle;
//   p . V  : lane (chunk c = lane % NCH, token group) accumulates one 16-byte
//            chunk of the head dimension over its tokens (V is token-major).
// Every spin on an mbarrier gives up after ~2 s, sets an error word and drains
// the copies already issued before the CTA exits.
#pragma once

#include "nosa_internal.cuh"

namespace nosa {

struct AttnKParams {
  const uint8_t* units;
  long long n_units;
  const int32_t* block_tab;
  int n_blocks;
  const uint8_t* tail;
  long long tail_stride;
  int tail_len;
  const void* q;
  float* part_acc;
  float* part_ml;
  int nsplit, bps, stages;
  int split_base, nsplit_total;
  int part_stride;  // partial slots per unit in part_acc / part_ml (>= nsplit_total)
  int unit_base;
  int* counters;
  void* out;
  float* lse;
  long long payload;
  int Hq, Hkv;
  float qscale;  // log2(e) / sqrt(d)
  int* err;
  const StepIO* dyn;  // decode step: q, out, lse, tail_len and the tail offset live here
  const int32_t* tail_tab;   // per-unit tail unit index (or null)
  const int32_t* tail_lens;  // per-unit tail length
  // stream-K partition (attn_streamk_kernel): CTA c of sk_ctas takes items
  // [c T / C, (c + 1) T / C) of the units' concatenated item lists (T = unit
  // count x nv; nv = n_blocks + tail); a unit has up to seg_cap partials.
  int sk_ctas, nv, seg_cap;
  long long sk_items;
  unsigned long long* trace;  // step trace (or null) and this launch's slot
  int trace_slot;
};

template <typename T> struct Unpack16;
template <> struct Unpack16<__nv_bfloat16> {
  static __device__ __forceinline__ void run(const uint4 r, float* f) {
    f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x);
    f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    f[4] = bf16_lo(r.z); f[5] = bf16_hi(r.z);
    f[6] = bf16_lo(r.w); f[7] = bf16_hi(r.w);
  }
};
template <> struct Unpack16<float> {
  static __device__ __forceinline__ void run(const uint4 r, float* f) {
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
  }
};

template <typename T, int D, int G, int W>
struct AttnGeom {
  static constexpr int B = 64;
  static constexpr int NT = 32 * W;       // threads per CTA
  static constexpr int TPW = B / W;       // tokens of each block per warp
  static constexpr int PARTS = 32 / TPW;  // head-dim parts of the logit lanes
  static constexpr int ELT = (int)sizeof(T);
  static constexpr int CE = 16 / ELT;     // elements per 16-byte chunk
  static constexpr int NCH = D / CE;      // chunks per token row
  static constexpr int NCHP = NCH / PARTS;  // chunks per part (logit lanes)
  static constexpr int TG = 32 / NCH;     // token groups of the p.V lanes
  static constexpr int TPL = TPW / TG;    // tokens per p.V lane per block
  static constexpr int GP = (G + 3) / 4 * 4;
  static constexpr int QP = D / PARTS + 4;  // padded floats per query part row
  static_assert(NCH >= 2 && NCH <= 32, "token row must be 32..512 bytes");
  static_assert(NCHP >= 1 && TPL >= 1, "warp split does not fit the row");
  static size_t smem_bytes(int stages, long long payload, int bps) {
    size_t off = (size_t)stages * payload;
    off += (size_t)G * PARTS * QP * 4 + (size_t)B * GP * 4 + (size_t)(bps + 1) * 4;
    off = (off + 7) & ~(size_t)7;
    off += (size_t)2 * stages * 8;
    return off;
  }
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Building blocks of the split-K attention.
// ---------------------------------------------------------------------------

// Online-softmax state of one warp over its TPW tokens of every block it sees.
template <typename T, int D, int G, int W>
struct AttnWarpState {
  static constexpr int CE = AttnGeom<T, D, G, W>::CE;
  float m_run[G], l_run[G];
  float2 acc[G][CE / 2];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -1e30f;
      l_run[g] = 0.f;
#pragma unroll
      for (int e = 0; e < CE / 2; ++e) acc[g][e] = make_float2(0.f, 0.f);
    }
  }
};

// The G queries of unit (b, h) into q_s (scaled by log2(e) / sqrt(d), split into
// head-dim parts for the logit lanes).
template <typename T, int D, int G, int W>
__device__ __forceinline__ void attn_stage_q(float* q_s, const void* q_in, int b, int h, int Hq,
                                             float qscale, int tid) {
  using Gm = AttnGeom<T, D, G, W>;
  constexpr int PARTS = Gm::PARTS, QP = Gm::QP;
  const T* qg = reinterpret_cast<const T*>(q_in) + ((long long)b * Hq + (long long)h * G) * D;
  for (int i = tid; i < G * D; i += Gm::NT) {
    const int g = i / D, dim = i % D;
    q_s[(g * PARTS + dim / (D / PARTS)) * QP + (dim % (D / PARTS))] = to_f32(qg[i]) * qscale;
  }
}

// One block unit in shared memory: the warp's TPW tokens enter its online softmax.
// valid: whether this lane's logit token counts (false: a tail position past the end).
template <typename T, int D, int G, int W>
__device__ __forceinline__ void attn_block(const uint8_t* buf, const float* q_s, float* p_s,
                                           bool valid, AttnWarpState<T, D, G, W>& st, int warp,
                                           int lane) {
  using Gm = AttnGeom<T, D, G, W>;
  constexpr int B = Gm::B, ELT = Gm::ELT, CE = Gm::CE, NCH = Gm::NCH, NCHP = Gm::NCHP;
  constexpr int TG = Gm::TG, TPL = Gm::TPL, GP = Gm::GP, QP = Gm::QP;
  constexpr int TPW = Gm::TPW, PARTS = Gm::PARTS;
  const int t = lane % TPW, hh = lane / TPW;  // logit lane: token, head-dim part
  const int tok = warp * TPW + t;
  const int c = lane % NCH, tg = lane / NCH;

  // ---- logits of this warp's TPW tokens ----
  float2 d2[G];
#pragma unroll
  for (int g = 0; g < G; ++g) d2[g] = make_float2(0.f, 0.f);
  const uint4* kp = reinterpret_cast<const uint4*>(buf) + (hh * NCHP) * B + tok;
#pragma unroll
  for (int cc = 0; cc < NCHP; ++cc) {
    float kf[CE];
    Unpack16<T>::run(kp[cc * B], kf);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float4* qp = reinterpret_cast<const float4*>(q_s + (g * PARTS + hh) * QP + cc * CE);
#pragma unroll
      for (int e4 = 0; e4 < CE / 4; ++e4) {
        const float4 qv = qp[e4];
        d2[g] = __ffma2_rn(make_float2(qv.x, qv.y), make_float2(kf[4 * e4], kf[4 * e4 + 1]), d2[g]);
        d2[g] = __ffma2_rn(make_float2(qv.z, qv.w), make_float2(kf[4 * e4 + 2], kf[4 * e4 + 3]), d2[g]);
      }
    }
  }
  const float ev = reinterpret_cast<const float*>(buf + 2 * B * D * ELT)[tok] * kLog2e;
  float pg[G], alpha[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float dot = d2[g].x + d2[g].y;
#pragma unroll
    for (int o = TPW; o < 32; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    const float lg = valid ? dot + ev : -INFINITY;
    float mx = lg;
#pragma unroll
    for (int o = 1; o < TPW; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float mn = fmaxf(st.m_run[g], mx);
    alpha[g] = exp2f(st.m_run[g] - mn);
    pg[g] = exp2f(lg - mn);
    st.l_run[g] = st.l_run[g] * alpha[g] + pg[g];
    st.m_run[g] = mn;
  }
  if (hh == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) p_s[tok * GP + g] = pg[g];
  }
  __syncwarp();

  // ---- acc = acc * alpha + sum_t p_t v_t ----
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float2 a2 = make_float2(alpha[g], alpha[g]);
#pragma unroll
    for (int e = 0; e < CE / 2; ++e) st.acc[g][e] = __fmul2_rn(st.acc[g][e], a2);
  }
  const uint8_t* vbase = buf + (size_t)B * D * ELT;
#pragma unroll
  for (int i = 0; i < TPL; ++i) {
    const int tk = warp * TPW + tg + i * TG;
    float vf[CE];
    Unpack16<T>::run(*reinterpret_cast<const uint4*>(vbase + ((size_t)tk * D + c * CE) * ELT), vf);
    float pv[GP];
#pragma unroll
    for (int g4 = 0; g4 < GP / 4; ++g4) {
      const float4 x = *reinterpret_cast<const float4*>(p_s + tk * GP + 4 * g4);
      pv[4 * g4] = x.x;
      pv[4 * g4 + 1] = x.y;
      pv[4 * g4 + 2] = x.z;
      pv[4 * g4 + 3] = x.w;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float2 p2 = make_float2(pv[g], pv[g]);
#pragma unroll
      for (int e = 0; e < CE / 2; ++e)
        st.acc[g][e] = __ffma2_rn(p2, make_float2(vf[2 * e], vf[2 * e + 1]), st.acc[g][e]);
    }
  }
  __syncwarp();
}

// Combines the W warps' states into the CTA's (M, A, L) per (query head, dim) and
// writes them as partial `pidx` of the unit ([unit][nst][G][D] accumulators and
// [unit][nst][G][2] (max, sum)), or, when pidx < 0, as the output itself (same
// arithmetic as a merge of one partial). red: shared memory of [W][G][D] + 2 [W][G]
// floats. The caller brackets it with __syncthreads (red may alias idle stages).
template <typename T, int D, int G, int W>
__device__ __forceinline__ void attn_reduce(AttnWarpState<T, D, G, W>& st, float* red, int tid,
                                            int warp, int lane, float* part_acc, float* part_ml,
                                            long long pbase, void* out, float* lse,
                                            long long row0) {
  using Gm = AttnGeom<T, D, G, W>;
  constexpr int CE = Gm::CE, NCH = Gm::NCH, TPW = Gm::TPW, NT = Gm::NT;
  const int c = lane % NCH, tg = lane / NCH;
  // Warp totals: each token's p sits in every head-dim part of the warp; sum
  // over the tokens of one part.
  float lw[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float x = st.l_run[g];
#pragma unroll
    for (int o = 1; o < TPW; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    lw[g] = x;
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < CE / 2; ++e)
#pragma unroll
      for (int o = NCH; o < 32; o <<= 1) {
        st.acc[g][e].x += __shfl_xor_sync(0xffffffffu, st.acc[g][e].x, o);
        st.acc[g][e].y += __shfl_xor_sync(0xffffffffu, st.acc[g][e].y, o);
      }
  float* red_acc = red;                // [W][G][D]
  float* red_m = red_acc + W * G * D;  // [W][G]
  float* red_l = red_m + W * G;        // [W][G]
  if (tg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < CE / 2; ++e) {
        red_acc[(warp * G + g) * D + c * CE + 2 * e] = st.acc[g][e].x;
        red_acc[(warp * G + g) * D + c * CE + 2 * e + 1] = st.acc[g][e].y;
      }
  }
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      red_m[warp * G + g] = st.m_run[g];
      red_l[warp * G + g] = lw[g];
    }
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += NT) {
    const int g = i / D, dim = i % D;
    float M = red_m[g];
#pragma unroll
    for (int w = 1; w < W; ++w) M = fmaxf(M, red_m[w * G + g]);
    float A = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float sc = exp2f(red_m[w * G + g] - M);
      A += red_acc[(w * G + g) * D + dim] * sc;
      L += red_l[w * G + g] * sc;
    }
    if (pbase < 0) {  // a single partial: it is the output
      const float inv = L > 0.f ? 1.f / L : 0.f;
      reinterpret_cast<T*>(out)[(row0 + g) * D + dim] = from_f32<T>(A * inv);
      if (dim == 0 && lse != nullptr) lse[row0 + g] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    } else {
      part_acc[(pbase + g) * D + dim] = A;
      if (dim == 0) {
        part_ml[(pbase + g) * 2] = M;
        part_ml[(pbase + g) * 2 + 1] = L;
      }
    }
  }
}

// The unit's nst partials merged into out / lse (by the CTA that published the
// last one): per-partial weights exp2(m_j - M) / L staged in shared memory, then
// the accumulators summed in partial order with independent loads.
// scratch: 3 * nst * G floats of shared memory.
template <typename T, int D, int G, int W>
__device__ __forceinline__ void attn_merge(const float* part_acc, const float* part_ml,
                                           long long ubase, int nst, float* scratch, void* out,
                                           float* lse, long long row0, int tid) {
  constexpr int NT = AttnGeom<T, D, G, W>::NT;
  float* ml_s = scratch;           // [nst][G][2]
  float* w_s = ml_s + 2 * nst * G;  // [nst][G]
  __shared__ float s_M[8], s_L[8];
  for (int i = tid; i < 2 * nst * G; i += NT) ml_s[i] = __ldcg(part_ml + ubase * 2 + i);
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int j = 0; j < nst; ++j) M = fmaxf(M, ml_s[(j * G + tid) * 2]);
    float L = 0.f;
    for (int j = 0; j < nst; ++j) {
      const float sc = exp2f(ml_s[(j * G + tid) * 2] - M);
      w_s[j * G + tid] = sc;
      L += ml_s[(j * G + tid) * 2 + 1] * sc;
    }
    s_M[tid] = M;
    s_L[tid] = L;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int j = 0; j < nst; ++j) w_s[j * G + tid] *= inv;
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += NT) {
    const int g = i / D, dim = i % D;
    const float* ac = part_acc + (ubase + g) * D + dim;
    float A = 0.f;
#pragma unroll 8
    for (int j = 0; j < nst; ++j) A += __ldcg(ac + (long long)j * G * D) * w_s[j * G + g];
    reinterpret_cast<T*>(out)[(row0 + g) * D + dim] = from_f32<T>(A);
    if (dim == 0 && lse != nullptr)
      lse[row0 + g] = s_L[g] > 0.f ? (s_M[g] + log2f(s_L[g])) * kLn2 : -INFINITY;
  }
}

template <typename T, int D, int G, int W>
__global__ void __launch_bounds__(32 * W) attn_split_kernel(AttnKParams p) {
  griddep_wait();  // the chunk's gather (programmatic edge in the step graph)
  TraceScope trace_scope(p.trace, p.trace_slot);
  using Gm = AttnGeom<T, D, G, W>;
  constexpr int B = Gm::B, GP = Gm::GP, QP = Gm::QP, NT = Gm::NT, PARTS = Gm::PARTS;
  constexpr int TPW = Gm::TPW;

  extern __shared__ __align__(128) uint8_t smem[];
  const long long payload = p.payload;
  uint8_t* stage_buf = smem;
  float* q_s = reinterpret_cast<float*>(smem + (size_t)p.stages * payload);
  float* p_s = q_s + G * PARTS * QP;
  int* list = reinterpret_cast<int*>(p_s + B * GP);
  uint64_t* full =
      reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(list + p.bps + 1) + 7) & ~uintptr_t(7));
  uint64_t* empty = full + p.stages;
  __shared__ int s_nl;
  __shared__ volatile int s_bad;

  const int u = p.unit_base + blockIdx.y, sp = blockIdx.x;
  const int b = u / p.Hkv, h = u % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const void* q_in = p.q;
  void* out = p.out;
  float* lse = p.lse;
  int tail_len = p.tail_len;
  const uint8_t* tail = p.tail;
  if (p.dyn != nullptr) {
    q_in = p.dyn->q;
    out = p.dyn->out;
    lse = p.dyn->lse;
    tail_len = p.dyn->tail_len;
    if (tail != nullptr) tail += p.dyn->tail_off;
  }
  if (p.tail_tab != nullptr) {  // per-unit tail (p.tail_stride is 0)
    tail = p.units + (long long)p.tail_tab[p.unit_base + blockIdx.y] * p.payload;
    tail_len = p.tail_lens[p.unit_base + blockIdx.y];
  }
  // Virtual item list: the n_blocks table entries, then the tail (if any),
  // dealt to the splits in turn (split sp takes items sp, sp + nsplit, ...), so
  // that a table whose valid entries sit at its front (the slots a gather just
  // filled) still spreads them over every split.
  const int ns = p.nsplit;
  const bool has_tail = (tail != nullptr) && (p.n_blocks % ns == sp);

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W);
    }
    fence_mbar_init();
    s_bad = 0;
  }
  if (warp == 0) {  // compact the valid blocks of this split, in order
    int cnt = 0;
    for (int base = sp; base < p.n_blocks; base += 32 * ns) {
      const int j = base + lane * ns;
      int idx = (j < p.n_blocks) ? p.block_tab[(long long)u * p.n_blocks + j] : -1;
      if (idx >= 0 && (long long)idx >= p.n_units) {  // bad index: skip it, flag it
        atomicExch(p.err, kDevErrBadIndex);
        idx = -1;
      }
      const unsigned m = __ballot_sync(0xffffffffu, idx >= 0);
      if (idx >= 0) list[cnt + __popc(m & ((1u << lane) - 1u))] = idx;
      cnt += __popc(m);
    }
    if (lane == 0) {
      if (has_tail) list[cnt] = -2;
      s_nl = cnt + (has_tail ? 1 : 0);
    }
    __syncwarp();
  }
  // Thread 0 (which initialised the barriers and, with warp 0, built the list)
  // starts the first copies before the queries are staged, so the pipeline fill
  // overlaps the query load.
  int issued = 0;  // meaningful in thread 0 only
  if (tid == 0) {
    const int pre = min(p.stages, s_nl);
    for (int s = 0; s < pre; ++s) {
      const int idx = list[s];
      const uint8_t* src = idx >= 0 ? p.units + (long long)idx * payload
                                    : tail + (long long)u * p.tail_stride;
      mbar_arrive_expect_tx(&full[s], (uint32_t)payload);
      bulk_g2s(stage_buf + (size_t)s * payload, src, (uint32_t)payload, &full[s]);
    }
    issued = pre;
  }
  attn_stage_q<T, D, G, W>(q_s, q_in, b, h, p.Hq, p.qscale, tid);
  __syncthreads();
  const int nl = s_nl;

  AttnWarpState<T, D, G, W> st;
  st.init();
  const int tok = warp * TPW + lane % TPW;

  for (int it = 0; it < nl; ++it) {
    if (__any_sync(0xffffffffu, s_bad != 0)) break;
    const int si = it % p.stages;
    const uint32_t par = (uint32_t)((it / p.stages) & 1);
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[si], par));
    if (!ok) {
      if (lane == 0) {
        s_bad = 1;
        atomicExch(p.err, kDevErrWaitTimeout);
      }
      break;
    }
    const uint8_t* buf = stage_buf + (size_t)si * payload;
    attn_block<T, D, G, W>(buf, q_s, p_s, (list[it] >= 0) || (tok < tail_len), st, warp, lane);
    if (lane == 0) mbar_arrive(&empty[si]);

    // ---- refill this stage with the block `stages` items ahead ----
    if (tid == 0 && issued < nl && s_bad == 0) {
      if (!mbar_wait_bounded(&empty[si], par)) {
        s_bad = 1;
        atomicExch(p.err, kDevErrWaitTimeout);
      } else {
        const int idx = list[issued];
        const uint8_t* src = idx >= 0 ? p.units + (long long)idx * payload
                                      : tail + (long long)u * p.tail_stride;
        mbar_arrive_expect_tx(&full[si], (uint32_t)payload);
        bulk_g2s(stage_buf + (size_t)si * payload, src, (uint32_t)payload, &full[si]);
        ++issued;
      }
    }
  }

  __syncthreads();
  if (s_bad != 0 && tid == 0) {
    // Drain: wait (bounded) for the last copy issued into each stage.
    for (int s = 0; s < p.stages; ++s) {
      int last = -1;
      for (int li = s; li < issued; li += p.stages) last = li;
      if (last >= 0) mbar_wait_bounded(&full[s], (uint32_t)((last / p.stages) & 1));
    }
  }
  __syncthreads();

  const int nst = p.nsplit_total;
  const long long row0 = (long long)b * p.Hq + (long long)h * G;
  float* red = reinterpret_cast<float*>(stage_buf);  // the stages are idle now
  attn_reduce<T, D, G, W>(st, red, tid, warp, lane, p.part_acc, p.part_ml,
                          nst == 1 ? -1 : ((long long)u * p.part_stride + p.split_base + sp) * G,
                          out, lse, row0);
  if (nst == 1) return;

  // The CTA that writes the unit's last partial merges all of them (no waiting:
  // every other CTA has already published its partial before counting itself).
  // The barrier orders the CTA's partial writes before thread 0's release add,
  // and the release makes them visible at GPU scope with the count.
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) {
    int prev;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(p.counters + u)
                 : "memory");
    s_last = (prev == nst - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  attn_merge<T, D, G, W>(p.part_acc, p.part_ml, (long long)u * p.part_stride * G, nst,
                         reinterpret_cast<float*>(stage_buf), out, lse, row0, tid);
  if (tid == 0) p.counters[u] = 0;
}

// attn_reduce for a CTA without a [W][G][D] buffer: the warps' states are
// combined one query head at a time through a [W][D] buffer (same arithmetic).
// red: W * D + 2 * W * G floats. Starts and ends with a __syncthreads.
template <typename T, int D, int G, int W>
__device__ __forceinline__ void attn_reduce_by_head(AttnWarpState<T, D, G, W>& st, float* red, int tid,
                                                    int warp, int lane, float* part_acc,
                                                    float* part_ml, long long pbase, void* out,
                                                    float* lse, long long row0) {
  using Gm = AttnGeom<T, D, G, W>;
  constexpr int CE = Gm::CE, NCH = Gm::NCH, TPW = Gm::TPW, NT = Gm::NT;
  const int c = lane % NCH, tg = lane / NCH;
  float lw[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float x = st.l_run[g];
#pragma unroll
    for (int o = 1; o < TPW; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    lw[g] = x;
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < CE / 2; ++e)
#pragma unroll
      for (int o = NCH; o < 32; o <<= 1) {
        st.acc[g][e].x += __shfl_xor_sync(0xffffffffu, st.acc[g][e].x, o);
        st.acc[g][e].y += __shfl_xor_sync(0xffffffffu, st.acc[g][e].y, o);
      }
  float* red_acc = red;                // [W][D]
  float* red_m = red_acc + W * D;      // [W][G]
  float* red_l = red_m + W * G;        // [W][G]
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      red_m[warp * G + g] = st.m_run[g];
      red_l[warp * G + g] = lw[g];
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (tg == 0) {
#pragma unroll
      for (int e = 0; e < CE / 2; ++e) {
        red_acc[warp * D + c * CE + 2 * e] = st.acc[g][e].x;
        red_acc[warp * D + c * CE + 2 * e + 1] = st.acc[g][e].y;
      }
    }
    __syncthreads();
    for (int dim = tid; dim < D; dim += NT) {
      float M = red_m[g];
#pragma unroll
      for (int w = 1; w < W; ++w) M = fmaxf(M, red_m[w * G + g]);
      float A = 0.f, L = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float sc = exp2f(red_m[w * G + g] - M);
        A += red_acc[w * D + dim] * sc;
        L += red_l[w * G + g] * sc;
      }
      if (pbase < 0) {
        const float inv = L > 0.f ? 1.f / L : 0.f;
        reinterpret_cast<T*>(out)[(row0 + g) * D + dim] = from_f32<T>(A * inv);
        if (dim == 0 && lse != nullptr) lse[row0 + g] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
      } else {
        part_acc[(pbase + g) * D + dim] = A;
        if (dim == 0) {
          part_ml[(pbase + g) * 2] = M;
          part_ml[(pbase + g) * 2 + 1] = L;
        }
      }
    }
    __syncthreads();
  }
}

// Tail block unit of unit u (decode-step buffer, per-unit table, or standalone stride).
__device__ __forceinline__ const uint8_t* attn_tail_src(const AttnKParams& p, const uint8_t* tail, int u) {
  if (p.tail_tab != nullptr) return p.units + (long long)p.tail_tab[u] * p.payload;
  return tail + (long long)u * p.tail_stride;
}

// CTA of the stream-K partition that holds item x.
__device__ __forceinline__ int sk_cta_of(long long x, long long T, int C) {
  return (int)(((x + 1) * C - 1) / T);
}

// Stream-K split of the same attention: one wave of CTAs, each streaming an equal
// share of the concatenated item lists (a share crosses unit boundaries), so no
// SM idles while a last partial wave runs. At a unit boundary the CTA folds its
// state into the unit's partial (one partial per CTA that touches the unit; the
// direct output when one CTA holds the whole unit) and restages the queries; the
// copy ring keeps running across the boundary. The unit's last partial to land
// triggers the merge, as in attn_split_kernel.
template <typename T, int D, int G, int W>
__global__ void __launch_bounds__(32 * W) attn_streamk_kernel(AttnKParams p) {
  using Gm = AttnGeom<T, D, G, W>;
  constexpr int B = Gm::B, GP = Gm::GP, QP = Gm::QP, PARTS = Gm::PARTS, TPW = Gm::TPW;

  extern __shared__ __align__(128) uint8_t smem[];
  const long long payload = p.payload;
  uint8_t* stage_buf = smem;
  float* q_s = reinterpret_cast<float*>(smem + (size_t)p.stages * payload);
  float* p_s = q_s + G * PARTS * QP;
  float* red = p_s + B * GP;                                        // [W][D] + 2 [W][G]
  int* list = reinterpret_cast<int*>(red + W * D + 2 * W * G);      // [bps + 1] block or -2 (tail)
  int* lunit = list + p.bps + 1;                                    // [bps + 1] unit - u_first
  uint64_t* full = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(lunit + p.bps + 1) + 7) & ~uintptr_t(7));
  uint64_t* empty = full + p.stages;
  __shared__ int s_nl, s_last;
  __shared__ volatile int s_bad;

  const int cta = blockIdx.x, C = p.sk_ctas, nv = p.nv;
  const long long NI = p.sk_items;
  const long long g0 = (long long)cta * NI / C, g1 = (long long)(cta + 1) * NI / C;
  if (g0 >= g1) return;  // (whole CTA: no item, no unit touched)
  const int u_first = p.unit_base + (int)(g0 / nv), u_last = p.unit_base + (int)((g1 - 1) / nv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const void* q_in = p.q;
  void* out = p.out;
  float* lse = p.lse;
  int tail_len0 = p.tail_len;
  const uint8_t* tail = p.tail;
  if (p.dyn != nullptr) {
    q_in = p.dyn->q;
    out = p.dyn->out;
    lse = p.dyn->lse;
    tail_len0 = p.dyn->tail_len;
    if (tail != nullptr) tail += p.dyn->tail_off;
  }
  const bool with_tail = (tail != nullptr) || (p.tail_tab != nullptr);

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W);
    }
    fence_mbar_init();
    s_bad = 0;
  }
  if (warp == 0) {  // the CTA's items in order: valid blocks and tails, tagged by unit
    int cnt = 0;
    for (long long base = g0; base < g1; base += 32) {
      const long long x = base + lane;
      int idx = -1, lu = 0;
      if (x < g1) {
        const int uu = p.unit_base + (int)(x / nv), j = (int)(x % nv);
        lu = uu - u_first;
        if (j < p.n_blocks) {
          idx = p.block_tab[(long long)uu * p.n_blocks + j];
          if (idx >= 0 && (long long)idx >= p.n_units) {
            atomicExch(p.err, kDevErrBadIndex);
            idx = -1;
          }
        } else if (with_tail) {
          idx = -2;
        }
      }
      const bool on = idx >= 0 || idx == -2;
      const unsigned m = __ballot_sync(0xffffffffu, on);
      if (on) {
        const int at = cnt + __popc(m & ((1u << lane) - 1u));
        list[at] = idx;
        lunit[at] = lu;
      }
      cnt += __popc(m);
    }
    if (lane == 0) s_nl = cnt;
    __syncwarp();
  }
  __syncthreads();
  const int nl = s_nl;
  int issued = 0;  // meaningful in thread 0 only
  auto src_of = [&](int i) -> const uint8_t* {
    const int idx = list[i];
    return idx >= 0 ? p.units + (long long)idx * payload : attn_tail_src(p, tail, u_first + lunit[i]);
  };
  if (tid == 0) {
    const int pre = min(p.stages, nl);
    for (int s = 0; s < pre; ++s) {
      mbar_arrive_expect_tx(&full[s], (uint32_t)payload);
      bulk_g2s(stage_buf + (size_t)s * payload, src_of(s), (uint32_t)payload, &full[s]);
    }
    issued = pre;
  }

  const int tok = warp * TPW + lane % TPW;
  int it = 0;
  for (int uu = u_first; uu <= u_last; ++uu) {
    const int b = uu / p.Hkv, h = uu % p.Hkv;
    const int tail_len = p.tail_lens != nullptr ? p.tail_lens[uu] : tail_len0;
    __syncthreads();  // q_s, p_s and red are free
    attn_stage_q<T, D, G, W>(q_s, q_in, b, h, p.Hq, p.qscale, tid);
    __syncthreads();
    AttnWarpState<T, D, G, W> st;
    st.init();
    for (; it < nl && lunit[it] == uu - u_first; ++it) {
      if (__any_sync(0xffffffffu, s_bad != 0)) break;
      const int si = it % p.stages;
      const uint32_t par = (uint32_t)((it / p.stages) & 1);
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[si], par));
      if (!ok) {
        if (lane == 0) {
          s_bad = 1;
          atomicExch(p.err, kDevErrWaitTimeout);
        }
        break;
      }
      attn_block<T, D, G, W>(stage_buf + (size_t)si * payload, q_s, p_s, (list[it] >= 0) || (tok < tail_len),
                             st, warp, lane);
      if (lane == 0) mbar_arrive(&empty[si]);
      if (tid == 0 && issued < nl && s_bad == 0) {
        if (!mbar_wait_bounded(&empty[si], par)) {
          s_bad = 1;
          atomicExch(p.err, kDevErrWaitTimeout);
        } else {
          mbar_arrive_expect_tx(&full[si], (uint32_t)payload);
          bulk_g2s(stage_buf + (size_t)si * payload, src_of(issued), (uint32_t)payload, &full[si]);
          ++issued;
        }
      }
    }
    __syncthreads();
    if (s_bad != 0) break;
    // this CTA's share of unit uu: the output itself or one of its partials
    const long long ib = (long long)(uu - p.unit_base) * nv;
    const int c_first = sk_cta_of(ib, NI, C), c_last = sk_cta_of(ib + nv - 1, NI, C);
    const int nseg = c_last - c_first + 1;
    const long long row0 = (long long)b * p.Hq + (long long)h * G;
    attn_reduce_by_head<T, D, G, W>(st, red, tid, warp, lane, p.part_acc, p.part_ml,
                                    nseg == 1 ? -1 : ((long long)uu * p.seg_cap + (cta - c_first)) * G,
                                    out, lse, row0);
    if (nseg == 1) continue;
    if (tid == 0) {
      int prev;
      asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                   : "=r"(prev)
                   : "l"(p.counters + uu)
                   : "memory");
      s_last = (prev == nseg - 1);
    }
    __syncthreads();
    if (!s_last) continue;
    __threadfence();
    attn_merge<T, D, G, W>(p.part_acc, p.part_ml, (long long)uu * p.seg_cap * G, nseg, red, out, lse,
                           row0, tid);
    if (tid == 0) p.counters[uu] = 0;
  }
  __syncthreads();
  if (s_bad != 0 && tid == 0) {  // drain: the last copy issued into each stage
    for (int s = 0; s < p.stages; ++s) {
      int last = -1;
      for (int li = s; li < issued; li += p.stages) last = li;
      if (last >= 0) mbar_wait_bounded(&full[s], (uint32_t)((last / p.stages) & 1));
    }
  }
}

template <typename T, int D, int G, int W>
size_t attn_streamk_smem(int stages, long long payload, int bps) {
  using Gm = AttnGeom<T, D, G, W>;
  size_t off = (size_t)stages * payload;
  off += (size_t)G * Gm::PARTS * Gm::QP * 4 + (size_t)Gm::B * Gm::GP * 4;
  off += (size_t)(W * D + 2 * W * G) * 4;
  off += (size_t)2 * (bps + 1) * 4;
  off = (off + 7) & ~(size_t)7;
  off += (size_t)2 * stages * 8;
  return off;
}

template <typename T, int D, int G, int W>
cudaError_t launch_attn_variant(const Shape& s, const AttnArgs& a, int stages, int bps,
                                cudaStream_t stream) {
  AttnKParams p;
  p.units = a.units;
  p.n_units = a.n_units;
  p.block_tab = a.block_tab;
  p.n_blocks = a.n_blocks;
  p.tail = a.tail;
  p.tail_stride = a.tail_stride;
  p.tail_len = a.tail_len;
  p.q = a.q;
  p.part_acc = a.part_acc;
  p.part_ml = a.part_ml;
  p.nsplit = a.nsplit;
  p.split_base = a.split_base;
  p.nsplit_total = a.nsplit_total;
  p.part_stride = a.part_stride > 0 ? a.part_stride : a.nsplit_total;
  p.unit_base = a.unit_base;
  p.counters = a.counters;
  p.out = a.out;
  p.lse = a.lse;
  p.bps = bps;
  p.stages = stages;
  p.payload = s.payload;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.qscale = (float)(1.4426950408889634 / sqrt((double)D));
  p.err = a.err;
  p.dyn = a.dyn;
  p.tail_tab = a.tail_tab;
  p.tail_lens = a.tail_lens;
  p.sk_ctas = a.sk_ctas;
  p.nv = a.n_blocks + ((a.tail != nullptr || a.tail_tab != nullptr) ? 1 : 0);
  p.seg_cap = a.seg_cap;
  p.sk_items = (long long)a.unit_count * p.nv;
  p.trace = a.trace;
  p.trace_slot = a.trace_slot;
  if (a.sk_ctas > 0) {
    const size_t smem = attn_streamk_smem<T, D, G, W>(stages, s.payload, bps);
    static std::atomic<int> lim_sk[64];
    cudaError_t err = raise_smem_limit((const void*)attn_streamk_kernel<T, D, G, W>, smem, lim_sk);
    if (err != cudaSuccess) return err;
    attn_streamk_kernel<T, D, G, W><<<a.sk_ctas, 32 * W, smem, stream>>>(p);
    return cudaGetLastError();
  }
  const size_t smem = std::max(AttnGeom<T, D, G, W>::smem_bytes(stages, s.payload, bps),
                               smem_for_occupancy(a.max_ctas_per_sm));
  static std::atomic<int> lim[64];
  cudaError_t err = raise_smem_limit((const void*)attn_split_kernel<T, D, G, W>, smem, lim);
  if (err != cudaSuccess) return err;
  dim3 grid(a.nsplit, a.unit_count);
  attn_split_kernel<T, D, G, W><<<grid, 32 * W, smem, stream>>>(p);
  return cudaGetLastError();
}

// CTAs per SM of one variant at the given pipeline depth (0 if it cannot run).
template <typename T, int D, int G, int W>
int attn_occupancy_variant(const Shape& s, int stages, int bps) {
  const size_t smem = AttnGeom<T, D, G, W>::smem_bytes(stages, s.payload, bps);
  static std::atomic<int> lim[64];
  if (raise_smem_limit((const void*)attn_split_kernel<T, D, G, W>, smem, lim) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_split_kernel<T, D, G, W>, 32 * W, smem) !=
      cudaSuccess)
    return 0;
  return n;
}

// CTAs per SM of the stream-K kernel (0 if it cannot run).
template <typename T, int D, int G, int W>
int attn_streamk_occupancy_variant(const Shape& s, int stages, int bps) {
  const size_t smem = attn_streamk_smem<T, D, G, W>(stages, s.payload, bps);
  static std::atomic<int> lim[64];
  if (raise_smem_limit((const void*)attn_streamk_kernel<T, D, G, W>, smem, lim) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_streamk_kernel<T, D, G, W>, 32 * W, smem) !=
      cudaSuccess)
    return 0;
  return n;
}

template <typename T, int D, int W>
int attn_streamk_occupancy_dispatch_g(const Shape& s, int stages, int bps) {
  switch (s.G) {
    case 1: return attn_streamk_occupancy_variant<T, D, 1, W>(s, stages, bps);
    case 2: return attn_streamk_occupancy_variant<T, D, 2, W>(s, stages, bps);
    case 3: return attn_streamk_occupancy_variant<T, D, 3, W>(s, stages, bps);
    case 4: return attn_streamk_occupancy_variant<T, D, 4, W>(s, stages, bps);
    case 6: return attn_streamk_occupancy_variant<T, D, 6, W>(s, stages, bps);
    case 8: return attn_streamk_occupancy_variant<T, D, 8, W>(s, stages, bps);
    default: return 0;
  }
}

template <typename T, int D, int W>
int attn_occupancy_dispatch_g(const Shape& s, int stages, int bps) {
  switch (s.G) {
    case 1: return attn_occupancy_variant<T, D, 1, W>(s, stages, bps);
    case 2: return attn_occupancy_variant<T, D, 2, W>(s, stages, bps);
    case 3: return attn_occupancy_variant<T, D, 3, W>(s, stages, bps);
    case 4: return attn_occupancy_variant<T, D, 4, W>(s, stages, bps);
    case 6: return attn_occupancy_variant<T, D, 6, W>(s, stages, bps);
    case 8: return attn_occupancy_variant<T, D, 8, W>(s, stages, bps);
    default: return 0;
  }
}

template <typename T, int D>
int attn_occupancy_dispatch_w(const Shape& s, int stages, int bps, int warps) {
  return warps == 8 ? attn_occupancy_dispatch_g<T, D, 8>(s, stages, bps)
                    : attn_occupancy_dispatch_g<T, D, 4>(s, stages, bps);
}
template <typename T, int D>
int attn_streamk_occupancy_dispatch_w(const Shape& s, int stages, int bps, int warps) {
  return warps == 8 ? attn_streamk_occupancy_dispatch_g<T, D, 8>(s, stages, bps)
                    : attn_streamk_occupancy_dispatch_g<T, D, 4>(s, stages, bps);
}

template <typename T, int D, int W>
cudaError_t launch_attn_dispatch_g(const Shape& s, const AttnArgs& a, int stages, int bps,
                                   cudaStream_t stream) {
  switch (s.G) {
    case 1: return launch_attn_variant<T, D, 1, W>(s, a, stages, bps, stream);
    case 2: return launch_attn_variant<T, D, 2, W>(s, a, stages, bps, stream);
    case 3: return launch_attn_variant<T, D, 3, W>(s, a, stages, bps, stream);
    case 4: return launch_attn_variant<T, D, 4, W>(s, a, stages, bps, stream);
    case 6: return launch_attn_variant<T, D, 6, W>(s, a, stages, bps, stream);
    case 8: return launch_attn_variant<T, D, 8, W>(s, a, stages, bps, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int D>
cudaError_t launch_attn_dispatch_w(const Shape& s, const AttnArgs& a, int stages, int bps,
                                   int warps, cudaStream_t stream) {
  return warps == 8 ? launch_attn_dispatch_g<T, D, 8>(s, a, stages, bps, stream)
                    : launch_attn_dispatch_g<T, D, 4>(s, a, stages, bps, stream);
}

cudaError_t launch_attention_f32(const Shape& s, const AttnArgs& a, int stages, int bps,
                                 int warps, cudaStream_t stream);

cudaError_t launch_attention_bf16(const Shape& s, const AttnArgs& a, int stages, int bps,
                                  int warps, cudaStream_t stream);
int attention_occupancy_f32(const Shape& s, int stages, int bps, int warps);
int attention_occupancy_bf16(const Shape& s, int stages, int bps, int warps);
int attention_streamk_occupancy_f32(const Shape& s, int stages, int bps, int warps);
int attention_streamk_occupancy_bf16(const Shape& s, int stages, int bps, int warps);

}  // namespace nosa
