// Internal declarations shared by the NOSA kernels and the C ABI.
//
// Device state of one handle (U units = batch * n_kv_heads, maxBlk blocks of
// capacity per unit, W = ceil(maxBlk / 32) bitmask words per unit). Every array
// is unit-major so that one CTA (or one warp) per unit touches a contiguous
// range.
#pragma once

#include <cuda.h>  // CUtensorMap (the driver itself is reached through the runtime's entry-point query)
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include <atomic>

namespace nosa {

constexpr int kMaxK = 256;         // selected blocks per unit
constexpr int kMaxChunks = 16;     // unit chunks of a pipelined decode step
constexpr int kMaxBlocks = 65535;  // capacity in blocks per unit

// Shape of a handle (all host-derived, passed by value to kernels).
struct Shape {
  int U, batch, Hq, Hkv, G, d, B, S, P, k, ke, maxBlk, W;
  int dtype;  // 0 fp32, 1 bf16
  int pkb;    // pooled keys stored in bf16 (else fp32)
  int elt;    // bytes per element of q, k, v, out
  int kbytes; // B * d * elt  (K part of a block unit, = V part)
  long long payload;  // bytes per block unit
};

// Device-side error codes (written to DevStats::error by a kernel that gives up).
enum : int { kDevErrNone = 0, kDevErrWaitTimeout = 1, kDevErrBadIndex = 2 };

// Device-side counters (updated with atomics by the set-difference and select kernels).
struct DevStats {
  unsigned long long host_loads, tail_loads, cold_host_loads, sum_hits, hit_samples, near_ties;
  int max_host_loads_unit;
  int min_hits;
  int error;
  int pad_;
};

// Arguments of one decode step. The append kernel (the step's first kernel)
// receives them by value and publishes StepIO for every kernel after it, so a
// captured step graph needs new arguments on its first node only.
struct StepArgs {
  const void* k_new;   // [batch][Hkv][d]
  const void* v_new;   // [batch][Hkv][d]
  const float* e_new;  // [batch][Hkv]
  const void* q;       // [batch][Hq][d]
  void* out;           // [batch][Hq][d]
  float* lse;          // [batch][Hq] or null
  int L_old;           // context before this step's token
};

// Per-step values derived from StepArgs (device-resident, written by the append kernel).
struct StepIO {
  const void* q;
  void* out;
  float* lse;
  int L_old;
  int n_cand;          // candidate blocks after the append: L_old / B
  int tail_len;        // tokens in the tail block after the append (1..B)
  int just_completed;  // block that just became a candidate, else -1
  long long tail_off;  // byte offset of the tail block's buffer: (n_cand % 2) * payload
};

// Fused front-end (projection of the hidden states + QKV split + append and
// pooling), launched instead of the append kernel. Grid = (tiles, ksplit).
struct FrontParams {
  int F, Fpad;      // packed rows of W ((Hq + 2 Hkv) d + Hkv) and rows padded to the tile
  int D;            // hidden width (multiple of 64)
  int kblocks;      // D / 64
  int ksplit;       // splits of the hidden width (<= min(kblocks, 8)): one cluster per row tile
  int tiles;        // Fpad / 128
  int npad;         // batch padded to a multiple of 16 (the MMA's N)
  int tmem_cols;    // tensor-memory columns allocated (power of two >= max(32, npad))
  int stages;       // TMA ring depth (frontend_stages)
  int batch;
  int L_old;        // context before this step's token
  void* q;          // [batch][Hq][d] bf16, written (the step's queries)
  void* out;        // published in StepIO
  float* lse;
  int* err;         // device error word
  const uint8_t* w_packed;  // weights in the packed tile layout (frontend_pack)
};
struct FrontArgs {
  CUtensorMap tx;   // x [batch][D] bf16, box 64 x npad, 128-byte swizzle
  FrontParams p;
};
bool frontend_available();
int frontend_stages(int npad);
size_t frontend_smem_bytes(int npad, int stages);
// Encodes fa.tx (fa.p.npad must be set). False if the driver's tensor-map encoder
// is unavailable or rejects the arguments.
bool frontend_encode(FrontArgs& fa, const void* x, int batch, int D);
size_t frontend_packed_bytes(int F, int D);
cudaError_t launch_frontend_pack(const void* w, void* packed, int F, int D, cudaStream_t stream);
const void* frontend_kernel_ptr();
// Clusters of the front-end that can be resident at once for these parameters (0 on error).
int frontend_max_clusters(const FrontParams& p);

// Training-time forward (k_prefill.cu): byte offsets into the caller's workspace.
struct PrefillLayout {
  size_t units, pk, pk3, se, eb, ecnt, tab, tail_tab, tail_len, part_acc, part_ml, counters, vmax, err,
      total;
};
// s describes the real units (batch * Hkv); L is the sequence length.
PrefillLayout prefill_layout(const Shape& s, int L, int nsplit);
size_t prefill_select_smem(const Shape& s, int nblk);
// Packs, pools, runs the eviction-set recurrence and the per-position selection;
// sel (optional) receives the selections [batch][L][Hkv][k].
// tc: block units in the tensor-core layout of the tiled attention (K and V^T
// 128-byte swizzled, V^T in fp16 scaled by 2^vs from the largest |v|).
cudaError_t launch_prefill_front(const Shape& s, int L, const void* q, const void* k,
                                 const void* v, const float* e, int32_t* sel, uint8_t* ws,
                                 const PrefillLayout& w, bool tc, cudaStream_t stream);
// Selection with the pooled query scores on the tensor cores (k_prefill_sel_tc.cu):
// shapes with d in {64, 128}, 64-token blocks of 4 sub-blocks and k - k_e <= 32.
bool prefill_select_tc_shape(const Shape& s);
// ... and NOSA_PREFILL_SELECT_TC is not 0 and the shared memory fits.
bool prefill_select_tc_ok(const Shape& s, int L);
// Bytes of the split pooled-key images (0 for shapes the path does not cover).
size_t prefill_keysplit_bytes(const Shape& s, int nblk);
cudaError_t launch_prefill_select_tc(const Shape& s, int L, const void* q, const float* pk, uint8_t* pk3,
                                     const int32_t* Eb, const int32_t* Ecnt, int32_t* sel, int32_t* tab,
                                     int32_t* ttab, int32_t* tlen, int* err, cudaStream_t stream);
// Tiled tensor-core attention of the training-time forward (k_prefill_tc.cu):
// one CTA per (unit, query block), grid (nblk, unit_count).
struct PrefillTileArgs {
  const uint8_t* units;  // [U][nblk] block units (V transposed)
  const int32_t* tab;    // [batch][L][Hkv][k] per-position block tables (unit index, -1 pad)
  const uint32_t* vmax;  // largest |v| of the call (fp32 bits): the V scale 2^vs
  const void* q;         // [batch][L][Hq][d] bf16
  void* out;             // [batch][L][Hq][d] bf16
  float* lse;            // [batch][L][Hq] or null
  int* err;              // device error word
  int L, nblk;
  int unit_base;         // first unit of this launch
  int mt;                // 128-row M tiles: ceil(64 G / 128)
  int tmem_cols;         // tensor-memory columns per CTA
  float inv_sqrt_d;
};
// True when the tiled path covers this shape (bf16, G in {1, 2, 4}, d in {64, 128},
// shared memory within the limit) and NOSA_PREFILL_TILED is not 0.
bool prefill_tiled_ok(const Shape& s, int L);
cudaError_t launch_prefill_tile(const Shape& s, int L, const uint8_t* units, const int32_t* tab,
                                const uint32_t* vmax, const void* q, void* out, float* lse,
                                int* err, cudaStream_t stream);

struct State {
  uint8_t* slots;      // [U][k] block units (device)
  uint8_t* tail;       // [U][2] block units (device); block b lives in buffer b % 2
  uint8_t* host;       // [U][maxBlk] block units (pinned, mapped host memory; device view)
  float* pk;           // [U][maxBlk][P][d] sub-block mean keys (fp32, or bf16 when Shape::pkb)
  float* sube;         // [U][maxBlk][P]    sub-block mean eviction logits
  float* se;           // [U][maxBlk]       block eviction score (max of sube)
  float* sq;           // [U][maxBlk]       query-aware block score of the current step
  uint32_t* elig;      // [U][W]            eviction eligibility bitmask
  uint32_t* selmask;   // [U][W]            Gamma of the current step
  uint32_t* resmask;   // [U][W]            blocks held by slots
  int32_t* nsel;       // [U][2]
  int32_t* slot2blk;   // [U][k]
  int32_t* loads;      // [U][k][3]         (block, slot, src)
  int32_t* nload;      // [U]               entries of the unit's load list
  int32_t* block_tab;  // [U][k]            slots kept from the previous step (slot pool index), -1 none
  int32_t* tab_new;    // [U][k]            slots filled by this step's loads, -1 none
  int32_t* att_cnt;    // [U]               split CTAs finished (the last one merges; self-resetting)
  int32_t* sel_cnt;    // [U]               scoring CTAs finished (the last one selects; self-resetting)
  uint32_t* qhint;     // [U]               Gamma_q threshold hint (ordered key) for the next step, or null
  float* part_acc;     // split-K partial accumulators
  float* part_ml;      // split-K partial (max, sum)
  DevStats* stats;
  StepIO* io;          // the current decode step's arguments
  float* ksum;         // [U][d] fp32 running key sum of the open sub-block (token order)
  float* esum;         // [U]    fp32 running eviction-logit sum of the open sub-block
  // Step trace (NOSA_TRACE=1 at create, else null): per traced launch of a step,
  // the first CTA's start and the last CTA's end on the global timer (ns).
  unsigned long long* trace;  // [kTraceSlots][2]
};

// Trace slots of a decode step's launches (chunk c < 8).
constexpr int kTraceSlots = 48;
enum : int {
  kTrAppend = 0, kTrScore = 1, kTrSelect = 9, kTrGather = 17, kTrAttnKept = 25, kTrAttnNew = 33,
  // phases of the fused front-end (earliest and latest CTA at each point):
  kTrFrontMain = 41,  // the main loop's accumulator complete
  kTrFrontEpi = 42,   // epilogue done
  // the first chunk's fused selection, per unit (earliest and latest unit):
  kTrSel0Begin = 43,  // the unit's scores complete, its selecting CTA starts
  kTrSel0E = 45,      // ... Gamma_e marked
  kTrSel0Q = 46,      // ... Gamma_q marked
  kTrSel0Emit = 47,   // ... selection lists and masks written
  kTrSel0End = 44     // its selection and set-difference done
};

// Pinned host store placement (host_store.cu): the node to bind the store of a
// device to (-1: none), and allocation / release of the store.
int host_store_node(int device);
// kind: 0 cudaHostAlloc, 1 a registered mapping bound to `node`, 2 a registered,
// pinned mapping in transparent huge pages (unbound). *pin_fd: a descriptor that holds
// long-term pins on the store's pages until host_store_free closes it (-1: none).
// try_pin = false: the pin is not attempted (as if the host refused it).
cudaError_t host_store_alloc(size_t bytes, int node, void** out, int* kind, size_t* mapped,
                             int* pin_fd, bool try_pin);
void host_store_free(void* p, size_t mapped, int kind, int pin_fd);

// ---------------------------------------------------------------------------
// Host-side launchers (each returns the launch error, if any).
// ---------------------------------------------------------------------------
cudaError_t launch_append_step(const Shape& s, const State& st, const StepArgs& a,
                               cudaStream_t stream);
cudaError_t launch_promote_tail(const Shape& s, const State& st, int blk, cudaStream_t stream);
cudaError_t launch_frontend(const Shape& s, const State& st, const FrontArgs& fa,
                            cudaStream_t stream);
cudaError_t launch_append_bulk(const Shape& s, const State& st, const void* k, const void* v,
                               const float* e, int L_old, int n, cudaStream_t stream);
// The per-unit kernels below handle units [ubase, ubase + ucount) of one chunk
// and read the step's query, candidate count and tail from State::io. The score
// grid covers n_cap >= n_cand candidates (surplus CTAs return at once).
cudaError_t launch_score(const Shape& s, const State& st, int n_cap, int ubase, int ucount,
                         cudaStream_t stream);
cudaError_t launch_select_setdiff(const Shape& s, const State& st, int cold, int ubase,
                                  int ucount, int chunk, cudaStream_t stream);
// Scoring with the selection and set-difference fused into the last scoring CTA
// of each unit (one launch instead of launch_score + launch_select_setdiff), for
// shapes whose selection arrays fit the CTA's shared memory.
bool score_select_fused_ok(const Shape& s);
cudaError_t launch_score_select(const Shape& s, const State& st, int n_cap, int ubase, int ucount,
                                int cold, int chunk, cudaStream_t stream, int max_ctas_per_sm = 0);
// Copies the load-list entries of units [ubase, ubase + ucount) (grid: CTAs;
// wide: 32-byte loads with a 256-byte L2 fetch hint instead of 16-byte loads).
cudaError_t launch_gather(const Shape& s, const State& st, int grid, int ubase, int ucount,
                          int chunk, bool wide, cudaStream_t stream);
// Sets every trace slot's start to the maximum (the ends are zeroed by the caller).
cudaError_t launch_trace_reset(unsigned long long* trace, cudaStream_t stream);
// result[0] = error code of a bounded wait that nothing completes, result[1] = ms waited.
cudaError_t launch_bounded_wait_probe(unsigned long long limit_ns, int* result,
                                      cudaStream_t stream);

// Split-K attention over block units. block_tab [U][n_blocks] holds unit indices
// into `units` (-1 skip). The tail unit of unit u is at tail + u * tail_stride.
// One launch writes partials [split_base, split_base + nsplit) of each unit; the
// CTA that finishes last among all nsplit_total partials of a unit (counted in
// counters[u], which it resets to 0) merges them into out / lse.
struct AttnArgs {
  const uint8_t* units;
  long long n_units;        // valid unit indices are [0, n_units)
  const int32_t* block_tab;
  int n_blocks;
  const uint8_t* tail;      // may be null
  long long tail_stride;    // bytes
  int tail_len;
  const void* q;
  void* out;
  float* lse;
  float* part_acc;          // [U][nsplit][G][d]
  float* part_ml;           // [U][nsplit][G][2]
  int nsplit;
  int split_base;
  int nsplit_total;
  // Partial slots per unit in part_acc / part_ml (0: nsplit_total). The decode
  // step's chunks have different split counts and run concurrently, so there
  // every unit owns a fixed range of slots.
  int part_stride = 0;
  int unit_base;            // this launch covers units [unit_base, unit_base + unit_count)
  int unit_count;
  int* counters;            // [U]
  int* err;                 // device error word
  // Decode step: q, out, lse and tail_len come from *dyn, and the tail pointer
  // (when not null) is offset by dyn->tail_off. Null for the standalone call.
  const StepIO* dyn = nullptr;
  // Per-unit tails (training-time forward): unit u's tail is units[tail_tab[u]]
  // with tail_lens[u] tokens (tail must be non-null; tail_stride is then 0).
  const int32_t* tail_tab = nullptr;
  const int32_t* tail_lens = nullptr;
  // Stream-K (single launch over all items): sk_ctas > 0 CTAs share the items
  // equally; seg_cap partial slots per unit (then also nsplit = nsplit_total).
  int sk_ctas = 0;
  int seg_cap = 0;
  // Cap on resident CTAs per SM (0: none), reached by asking for more shared
  // memory than the kernel uses: fewer copies in flight leave more of the
  // memory system to a concurrent host-link gather. Launch shape only.
  int max_ctas_per_sm = 0;
  // Step trace (see State::trace): the array and this launch's slot (-1: none).
  unsigned long long* trace = nullptr;
  int trace_slot = -1;
};
// Dynamic shared memory that caps a kernel at `ctas` resident CTAs per SM
// (0 when ctas <= 0): the SM's 228 KB split `ctas` ways, less the per-CTA
// reservation and a margin for static shared memory.
inline size_t smem_for_occupancy(int ctas) {
  return ctas > 0 ? (size_t)(233472 / ctas) - 8192 : 0;
}
// How a single attention launch over n_blocks table entries (+ tail) per unit is
// split: stream-K with sk_ctas CTAs (0: the classic split into nsplit per unit);
// slots = partial slots per unit the workspace must hold.
struct AttnPlan {
  int nsplit, sk_ctas, seg_cap, slots;
};
AttnPlan attention_plan_single(const Shape& s, int n_blocks);
size_t attention_workspace_bytes(const Shape& s, int nsplit);
int attention_pick_nsplit(const Shape& s, int n_blocks, int has_tail);
cudaError_t launch_attention(const Shape& s, const AttnArgs& a, cudaStream_t stream);
bool attention_supported(int dtype, int d, int G);

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device, calling the driver only when the limit must grow (the caller
// passes one cache array of 64 per kernel).
inline cudaError_t raise_smem_limit(const void* func, size_t bytes, std::atomic<int>* cache) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && cache[dev].load(std::memory_order_relaxed) >= (int)bytes) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && dev < 64) cache[dev].store((int)bytes, std::memory_order_relaxed);
  return e;
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Stores a sub-block mean key in the handle's pooled-key precision.
__device__ __forceinline__ void store_pooled(const Shape& s, float* pk, long long idx, float v) {
  if (s.pkb)
    reinterpret_cast<__nv_bfloat16*>(pk)[idx] = __float2bfloat16_rn(v);
  else
    pk[idx] = v;
}

// Byte offsets inside a block unit (layout documented in include/nosa.h).
__device__ __forceinline__ long long k_off(int t, int dim, int B, int elt) {
  const int c = 16 / elt;
  return ((long long)(dim / c) * B + t) * 16 + (long long)(dim % c) * elt;
}
__device__ __forceinline__ long long v_off(int t, int dim, int B, int d, int elt) {
  return (long long)B * d * elt + ((long long)t * d + dim) * elt;
}
__device__ __forceinline__ long long e_off(int t, int B, int d, int elt) {
  return 2LL * B * d * elt + 4LL * t;
}

// Power-of-two exponent vs applied to V for the fp16 P V product of the tiled
// training-time attention: the largest |v| times 2^vs lies in [2^14, 2^15).
__device__ __forceinline__ int v_scale_exp(uint32_t absmax_bits) {
  const float m = __uint_as_float(absmax_bits);
  if (!(m > 0.f) || !(m < INFINITY)) return 0;
  int e;
  frexpf(m, &e);  // m = f 2^e, f in [0.5, 1)
  return 15 - e;
}

// Monotone map of fp32 scores to uint32 (larger float -> larger key); -0 == +0.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Records a CTA's start on entry and its end when the scope closes (any return)
// in a trace slot: the slot keeps the earliest start and the latest end. No-op
// without a trace array or slot.
// One point in time of one CTA (thread 0 of the calling group): the slot keeps
// the earliest and the latest over the CTAs.
__device__ __forceinline__ void trace_mark(unsigned long long* trace, int id) {
  if (trace == nullptr) return;
  const unsigned long long t = global_ns();
  atomicMin(trace + 2 * id, t);
  atomicMax(trace + 2 * id + 1, t);
}

// Programmatic dependent launch inside the step graph: a kernel whose incoming
// edge is programmatic may become resident before its producer has finished and
// waits here until the producer grids have completed and their memory is
// visible; with ordinary edges (and outside graphs) both are no-ops. A producer
// lets its programmatic dependents be scheduled once all of its CTAs have called
// griddep_launch_dependents or exited.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

struct TraceScope {
  unsigned long long* slot;
  __device__ __forceinline__ TraceScope(unsigned long long* trace, int id)
      : slot((trace != nullptr && id >= 0 && threadIdx.x == 0) ? trace + 2 * id : nullptr) {
    if (slot) atomicMin(slot, (unsigned long long)global_ns());
  }
  __device__ __forceinline__ ~TraceScope() {
    if (slot) atomicMax(slot + 1, (unsigned long long)global_ns());
  }
};

// ---- mbarrier and bulk-copy primitives (inline PTX, sm_90+ forms) ----------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                   smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete; gives up after
// `limit_ns` nanoseconds and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}
// One bulk (non-tensor) global -> shared copy completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

#endif  // __CUDACC__

}  // namespace nosa
