// C ABI of the NOSA decode-step hot path: handle lifecycle, argument checks and
// the per-step launch sequence. The kernels live in k_*.cu; this file owns the
// device memory (slot pool, tail buffers, pooled metadata, bitmasks, scratch)
// and the pinned, mapped host store of block units.
#include "nosa.h"
#include "nosa_internal.cuh"
#include "k_attn.cuh"

#include <algorithm>
#include <array>
#include <climits>
#include <map>
#include <mutex>
#include <cstdlib>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

using namespace nosa;

namespace {

constexpr int kMaxSplits = 64;
constexpr int kRing = 64;     // timing event sets in flight (eager steps)
constexpr int kNumEv = 8;
constexpr int kGraphRing = 16; // step graphs in flight when timing (each owns an event set)
constexpr int kScoreCap = 32; // a step graph's score grid covers this many more candidates

thread_local std::string g_thread_err;

struct DeviceGuard {
  int prev = -1;
  int want;
  explicit DeviceGuard(int dev) : want(dev) {
    cudaGetDevice(&prev);
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    if (prev >= 0 && prev != want) cudaSetDevice(prev);
  }
};

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Host-only validation. Returns NOSA_OK, NOSA_ERR_INVALID_ARG or NOSA_ERR_UNSUPPORTED.
nosa_status validate(const nosa_config* c, std::string& why) {
  if (!c) { why = "config is NULL"; return NOSA_ERR_INVALID_ARG; }
  if (c->batch < 1 || c->n_q_heads < 1 || c->n_kv_heads < 1) {
    why = "batch and head counts must be >= 1"; return NOSA_ERR_INVALID_ARG;
  }
  if (c->n_q_heads % c->n_kv_heads != 0) {
    why = "n_q_heads must be a multiple of n_kv_heads"; return NOSA_ERR_INVALID_ARG;
  }
  if (c->dtype != NOSA_F32 && c->dtype != NOSA_BF16) { why = "unknown dtype"; return NOSA_ERR_INVALID_ARG; }
  if (c->block < 1 || c->sub_block < 1 || c->block % c->sub_block != 0) {
    why = "block must be a positive multiple of sub_block"; return NOSA_ERR_INVALID_ARG;
  }
  if (c->k < 1 || c->k_e < 0 || c->k_e > c->k) { why = "need 0 <= k_e <= k and k >= 1"; return NOSA_ERR_INVALID_ARG; }
  if (c->max_context < 1) { why = "max_context must be >= 1"; return NOSA_ERR_INVALID_ARG; }
  if (c->device < 0) { why = "device must be >= 0"; return NOSA_ERR_INVALID_ARG; }
  if (c->flags & ~(NOSA_FLAG_TIMING | NOSA_FLAG_POOLED_BF16)) {
    why = "unknown flag bits"; return NOSA_ERR_INVALID_ARG;
  }
  if (c->head_dim < 1) { why = "head_dim must be >= 1"; return NOSA_ERR_INVALID_ARG; }
  if (c->block != 64 || c->sub_block != 16) {
    why = "compiled for block = 64, sub_block = 16"; return NOSA_ERR_UNSUPPORTED;
  }
  if (c->head_dim != 64 && c->head_dim != 128) { why = "head_dim must be 64 or 128"; return NOSA_ERR_UNSUPPORTED; }
  const int G = c->n_q_heads / c->n_kv_heads;
  if (!(G == 1 || G == 2 || G == 3 || G == 4 || G == 6 || G == 8)) {
    why = "n_q_heads / n_kv_heads must be 1, 2, 3, 4, 6 or 8"; return NOSA_ERR_UNSUPPORTED;
  }
  if (c->k > kMaxK) { why = "k must be <= 256"; return NOSA_ERR_UNSUPPORTED; }
  const long long maxblk = (c->max_context + (long long)c->block - 1) / c->block;
  if (maxblk > 32768) { why = "max_context must be <= 32768 blocks"; return NOSA_ERR_UNSUPPORTED; }
  if ((long long)c->batch * c->n_kv_heads > 65535) {
    why = "batch * n_kv_heads must be <= 65535"; return NOSA_ERR_UNSUPPORTED;
  }
  return NOSA_OK;
}

long long payload_of(int block, int d, int dtype) {
  const int elt = dtype == NOSA_F32 ? 4 : 2;
  const long long raw = 2LL * block * d * elt + 4LL * block;
  return (raw + 255) / 256 * 256;
}

Shape shape_of(const nosa_config& c) {
  Shape s;
  s.batch = c.batch;
  s.Hq = c.n_q_heads;
  s.Hkv = c.n_kv_heads;
  s.U = c.batch * c.n_kv_heads;
  s.G = c.n_q_heads / c.n_kv_heads;
  s.d = c.head_dim;
  s.B = c.block;
  s.S = c.sub_block;
  s.P = c.block / c.sub_block;
  s.k = c.k;
  s.ke = c.k_e;
  s.maxBlk = (c.max_context + c.block - 1) / c.block;
  s.W = (s.maxBlk + 31) / 32;
  s.dtype = c.dtype;
  s.elt = c.dtype == NOSA_F32 ? 4 : 2;
  s.kbytes = c.block * c.head_dim * s.elt;
  s.payload = payload_of(c.block, c.head_dim, c.dtype);
  s.pkb = (c.flags & NOSA_FLAG_POOLED_BF16) ? 1 : 0;
  return s;
}

// Pipeline stages of the attention CTA (NOSA_ATTN_STAGES overrides, read once).
int attn_stages(long long payload) {
  static const int forced = [] {
    const char* g = std::getenv("NOSA_ATTN_STAGES");
    const int v = g ? std::atoi(g) : 0;
    return (v >= 2 && v <= 6) ? v : 0;
  }();
  if (forced) return (int)std::min<long long>(forced, 200000 / payload);
  // Measured on GB300: three resident CTAs with a 2-stage ring beat two CTAs
  // with 3 stages (71.9% vs 63.5% of HBM peak at d = 128 bf16), so the ring is
  // sized to leave room for three CTAs per SM.
  return (int)std::max<long long>(2, std::min<long long>(4, 70000 / payload));
}

// Warps per attention CTA (4 or 8; NOSA_ATTN_WARPS overrides, read once).
int attn_warps() {
  static const int w = [] {
    const char* g = std::getenv("NOSA_ATTN_WARPS");
    return (g && std::atoi(g) == 8) ? 8 : 4;
  }();
  return w;
}

int sm_count_current() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

// ---------------------------------------------------------------------------
// Attention helpers shared by nosa_decode_step and nosa_sparse_attention.
// ---------------------------------------------------------------------------
namespace nosa {

bool attention_supported(int dtype, int d, int G) {
  return (dtype == 0 || dtype == 1) && (d == 64 || d == 128) &&
         (G == 1 || G == 2 || G == 3 || G == 4 || G == 6 || G == 8);
}

// Standalone-attention workspace: partial accumulators, partial (max, sum),
// per-unit split counters, then a 16-byte tail whose first int is the error word.
size_t attention_workspace_bytes(const Shape& s, int nsplit) {
  size_t acc = (size_t)s.U * nsplit * s.G * s.d * 4;
  size_t ml = (size_t)s.U * nsplit * s.G * 2 * 4;
  size_t cnt = (size_t)s.U * 4;
  return ((acc + 15) & ~(size_t)15) + ((ml + 15) & ~(size_t)15) + ((cnt + 15) & ~(size_t)15) + 16;
}

// Splits per unit: about 20 blocks per split, at least half a CTA per resident
// slot, one split when the units alone fill the slots twice (and >= 2 blocks per
// split); NOSA_ATTN_SPLITS overrides.
int attention_pick_nsplit_uncached(const Shape& s, int n_blocks);

// The pick depends only on the shape and the device; it is cached (the
// occupancy query behind it costs a driver call).
int attention_pick_nsplit(const Shape& s, int n_blocks, int /*has_tail*/) {
  static std::mutex mu;
  static std::map<std::array<long long, 7>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const std::array<long long, 7> key = {dev, s.dtype, s.d, s.G, s.U, n_blocks, attn_warps()};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const int ns = attention_pick_nsplit_uncached(s, n_blocks);
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = ns;
  return ns;
}

int attention_pick_nsplit_uncached(const Shape& s, int n_blocks) {
  const int nv = n_blocks + 1;
  // CTAs are scheduled as others finish, not in lockstep waves: long CTAs (about
  // 20 blocks) amortise each CTA's start-up and merge; small launches still get
  // half a CTA per resident slot (in the decode step the attention shares the GPU
  // with scoring and the gather). Measured on GB300 at the 8B-offload shape: 3
  // splits (22 blocks each) 106 us alone against 113 us for 7; in the step 3
  // splits per unit chunk beat 6 (101.6 k against 84 k tokens/s).
  const int stages = attn_stages(s.payload);
  const int bps_est = std::min(nv, 64);
  int occ = s.dtype == 0 ? attention_occupancy_f32(s, stages, bps_est, attn_warps())
                         : attention_occupancy_bf16(s, stages, bps_est, attn_warps());
  if (occ < 1) occ = 1;
  // The occupancy query above also raises the kernel's shared-memory limit, here at
  // create; the tuning override comes after it so that it leaves the kernel in the
  // same state (a limit first raised while a cold step is being enqueued held that
  // step's gathers to a fifth of the link on GB300).
  if (const char* g = std::getenv("NOSA_ATTN_SPLITS")) {
    const int v = std::atoi(g);
    if (v >= 1) return std::min(std::min(v, kMaxSplits), std::max(1, nv));
  }
  const double slots = (double)sm_count_current() * occ;
  if (s.U >= 2 * slots) return 1;  // enough CTAs already, and one split needs no merge
  const int by_blocks = std::max(1, nv / 20);
  const int by_fill = (int)std::ceil(0.5 * slots / std::max(s.U, 1));
  const int max_ns = std::max(1, std::min(kMaxSplits, nv / 2));
  const int best = std::max(1, std::min(max_ns, std::max(by_blocks, by_fill)));
  return best;
}

// Single-launch plan: stream-K over one wave of resident CTAs when each CTA's
// share fits its item list (<= 256) and a unit spans at most 16 CTAs; otherwise
// the classic split. NOSA_ATTN_STREAMK=0 forces the classic split. The partial
// slots cover both a launch with a tail and one without.
AttnPlan attention_plan_single_uncached(const Shape& s, int n_blocks) {
  AttnPlan pl;
  pl.nsplit = attention_pick_nsplit(s, n_blocks, 1);
  pl.sk_ctas = 0;
  pl.seg_cap = 0;
  pl.slots = pl.nsplit;
  const char* g = std::getenv("NOSA_ATTN_STREAMK");
  if ((g && std::strcmp(g, "0") == 0) || n_blocks < 1) return pl;
  const int stages = attn_stages(s.payload);
  const int occ = s.dtype == 0 ? attention_streamk_occupancy_f32(s, stages, 256, attn_warps())
                               : attention_streamk_occupancy_bf16(s, stages, 256, attn_warps());
  if (occ < 1) return pl;
  const long long C = (long long)sm_count_current() * occ;
  int cap = 0;
  for (int nv = n_blocks; nv <= n_blocks + 1; ++nv) {
    const long long T = (long long)s.U * nv;
    const long long minlen = T / C;  // items of the shortest share
    if (minlen < 2 || (T + C - 1) / C > 256) return pl;
    cap = std::max<int>(cap, (int)((nv + minlen - 1) / minlen + 1));
  }
  // the merge's scratch (3 x partials x G floats) lives in the CTA's reduce
  // buffer (W x d + 2 W x G floats)
  const int W = attn_warps();
  if (cap > 16 || 3 * cap * s.G > W * s.d + 2 * W * s.G) return pl;
  pl.sk_ctas = (int)C;
  pl.seg_cap = cap;
  pl.slots = std::max(cap, pl.nsplit);  // (a launch without items takes the classic split)
  return pl;
}

AttnPlan attention_plan_single(const Shape& s, int n_blocks) {
  static std::mutex mu;
  static std::map<std::array<long long, 8>, AttnPlan> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const char* g = std::getenv("NOSA_ATTN_STREAMK");
  const long long sk_off = (g && std::strcmp(g, "0") == 0) ? 1 : 0;
  const std::array<long long, 8> key = {dev, s.dtype, s.d, s.G, s.U, n_blocks, attn_warps(), sk_off};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const AttnPlan pl = attention_plan_single_uncached(s, n_blocks);
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = pl;
  return pl;
}

// Message returned by nosa_last_error(NULL) on this thread.
void set_thread_error(const std::string& msg) { g_thread_err = msg; }

cudaError_t launch_attention(const Shape& s, const AttnArgs& a, cudaStream_t stream) {
  const int stages = attn_stages(s.payload);
  const int nv = a.n_blocks + ((a.tail || a.tail_tab) ? 1 : 0);
  int bps = std::max(1, (nv + a.nsplit - 1) / a.nsplit);
  if (a.sk_ctas > 0) {  // items of the longest stream-K share
    const long long T = (long long)a.unit_count * nv;
    bps = (int)std::max<long long>(1, (T + a.sk_ctas - 1) / a.sk_ctas);
  }
  return s.dtype == 0 ? launch_attention_f32(s, a, stages, bps, attn_warps(), stream)
                      : launch_attention_bf16(s, a, stages, bps, attn_warps(), stream);
}

}  // namespace nosa

// ---------------------------------------------------------------------------
// The handle
// ---------------------------------------------------------------------------
// A captured warm decode step. Every per-step value reaches the kernels through
// the append node's arguments (the append kernel publishes StepIO), so between
// rebuilds a step costs one node update and one graph launch. The score grids
// cover candidates [0, n_cap); the graph is rebuilt when the count leaves
// [n_cap - kScoreCap, n_cap).
struct StepGraph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraphNode_t append_node = nullptr;
  cudaKernelNodeParams append_params{};
  int n_cap = 0;
  bool front = false;          // first node is the fused front-end (else the append)
  int front_gen = 0;           // ... set up for this front-end configuration
  bool pending = false;        // timing events of the last launch not yet read
  cudaEvent_t done = nullptr;  // recorded after each launch: a rebuild waits for it
};

struct InjectFailFlags {
  bool host = false;
  bool pin = false;
  int dev_index = -1;
};

struct nosa_handle {
  nosa_config cfg;
  InjectFailFlags inject;  // failure injection of nosa_create (NOSA_INJECT_FAIL)
  Shape s;
  State st;
  std::vector<void*> dev_allocs;
  uint8_t* host_store = nullptr;
  size_t host_bytes = 0;
  int host_kind = 0;           // how the store was made (host_store_alloc)
  int host_pin_fd = -1;          // holds long-term pins on the store (-1: none)
  size_t host_map_bytes = 0;   // ... its mapped length
  int host_node = -1;            // NUMA node the store is bound to (-1: not bound)
  long long L = 0;
  long long steps = 0;
  int nsplit_new = 4;   // attention splits over the slots the gather filled (warm steps)
  int gather_grid = 1;
  bool pdl = true;               // programmatic edges in the step graph (NOSA_PDL=0: off)
  bool broken = false;
  std::string err;
  cudaStream_t last_stream = nullptr;
  // Internal streams of the pipelined step: selection chain (medium priority),
  // gather (highest), attention over kept slots (lowest), attention over filled
  // slots (medium); events order them per unit chunk.
  cudaStream_t s_sco = nullptr, s_sel = nullptr, s_gat = nullptr, s_att = nullptr, s_new = nullptr;
  cudaStream_t s_gat2 = nullptr;  // gathers of odd chunks (fused step)
  cudaEvent_t ev_jgat2 = nullptr;
  int gather_streams = 2;
  bool gather_wide = false;  // 32-byte gather loads (NOSA_GATHER_VEC=32)
  cudaEvent_t ev_in = nullptr, ev_att = nullptr, ev_new = nullptr;
  cudaEvent_t ev_app = nullptr;  // the step's append is done
  // Fused step: chunk c is scored and selected on its own stream (priority
  // falling with c) and attended over its kept slots on its own lowest-priority
  // stream, and over its filled slots on its own stream as well; ev_jch / ev_jka
  // / ev_jfa join them into the origin stream.
  cudaStream_t s_chunk[kMaxChunks] = {}, s_katt[kMaxChunks] = {}, s_fatt[kMaxChunks] = {};
  cudaEvent_t ev_jch[kMaxChunks] = {}, ev_jka[kMaxChunks] = {}, ev_jfa[kMaxChunks] = {};
  cudaEvent_t ev_jsco = nullptr, ev_jsel = nullptr, ev_jgat = nullptr;  // joins of a captured step
  cudaStream_t s_cap = nullptr;                       // origin stream of captures
  bool use_graphs = true;
  bool fused_select = true;  // selection in the last scoring CTA of each unit
  int score_occ = 0;         // resident scoring CTAs per SM cap (0: none)
  int attn_occ = 0;          // resident attention CTAs per SM cap in the step (0: none)
  StepGraph plain;               // step graph without timing events
  StepGraph graphs[kGraphRing];  // step graphs with timing events (ring)
  cudaEvent_t gev[kGraphRing][kNumEv];
  int graph_pos = 0;
  long long graph_builds = 0;
  cudaEvent_t ev_sco[kMaxChunks] = {}, ev_sel[kMaxChunks] = {}, ev_gat[kMaxChunks] = {};
  int nchunks = 1;
  int cu_base[kMaxChunks] = {}, cu_count[kMaxChunks] = {}, nsplit_c[kMaxChunks] = {};
  bool timing = false;    // timing events recorded for the next steps
  bool ev_made = false;   // the event sets below exist
  cudaEvent_t ev[kRing][kNumEv];
  bool pending[kRing];
  int ring_pos = 0;
  double t_us[8];
  long long t_count = 0;
  long long launches = 0;  // kernels launched by decode steps
  // Fused front-end (set up on the first nosa_decode_step_hidden of a width).
  void* q_buf = nullptr;     // [batch][Hq][d] bf16 step queries
  int fe_hidden = 0, fe_ksplit = 0, fe_stages = 0;
  int fe_gen = 0;               // bumped when the front-end's launch shape changes

  nosa_status fail(nosa_status code, const std::string& msg) {
    err = msg;
    if (code == NOSA_ERR_CUDA) broken = true;
    return code;
  }
  nosa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(NOSA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  }
};

namespace {

// Failure injection on the host (no GPU fault involved): NOSA_INJECT_FAIL, read
// at every nosa_create, makes one of its allocations report exhaustion without
// being attempted. "host": the pinned host store; "pin": the long-term pin of the
// host store (the store then falls back as it does where pinning is refused);
// "dev:N": the N-th device allocation (from 0). Anything else: no injection.
InjectFailFlags inject_fail_from_env() {
  InjectFailFlags f;
  const char* g = std::getenv("NOSA_INJECT_FAIL");
  if (g == nullptr) return f;
  if (std::strcmp(g, "host") == 0) f.host = true;
  else if (std::strcmp(g, "pin") == 0) f.pin = true;
  else if (std::strncmp(g, "dev:", 4) == 0 && g[4] >= '0' && g[4] <= '9') f.dev_index = std::atoi(g + 4);
  return f;
}

template <typename T>
cudaError_t dev_alloc(nosa_handle* h, T** p, size_t bytes) {
  if (h->inject.dev_index == (int)h->dev_allocs.size()) return cudaErrorMemoryAllocation;
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, std::max<size_t>(bytes, 16));
  if (e != cudaSuccess) return e;
  h->dev_allocs.push_back(q);
  *p = static_cast<T*>(q);
  return cudaSuccess;
}

void free_all(nosa_handle* h) {
  if (h->q_buf) cudaFree(h->q_buf);
  h->q_buf = nullptr;
  for (void* p : h->dev_allocs) cudaFree(p);
  h->dev_allocs.clear();
  host_store_free(h->host_store, h->host_map_bytes, h->host_kind, h->host_pin_fd);
  h->host_store = nullptr;
  for (StepGraph* gp : {&h->plain}) {
    if (gp->exec) cudaGraphExecDestroy(gp->exec);
    if (gp->graph) cudaGraphDestroy(gp->graph);
    if (gp->done) cudaEventDestroy(gp->done);
    *gp = StepGraph();
  }
  for (StepGraph& g : h->graphs) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (g.graph) cudaGraphDestroy(g.graph);
    if (g.done) cudaEventDestroy(g.done);
    g = StepGraph();
  }
  if (h->ev_made) {
    for (int r = 0; r < kRing; ++r)
      for (int i = 0; i < kNumEv; ++i) cudaEventDestroy(h->ev[r][i]);
    for (int r = 0; r < kGraphRing; ++r)
      for (int i = 0; i < kNumEv; ++i) cudaEventDestroy(h->gev[r][i]);
    h->ev_made = false;
    h->timing = false;
  }
  for (cudaEvent_t* e : {&h->ev_in, &h->ev_att, &h->ev_new, &h->ev_jsco, &h->ev_jsel, &h->ev_jgat,
                         &h->ev_app})
    if (*e) cudaEventDestroy(*e), *e = nullptr;
  for (int c = 0; c < kMaxChunks; ++c) {
    if (h->ev_jch[c]) cudaEventDestroy(h->ev_jch[c]), h->ev_jch[c] = nullptr;
    if (h->ev_jka[c]) cudaEventDestroy(h->ev_jka[c]), h->ev_jka[c] = nullptr;
    if (h->ev_jfa[c]) cudaEventDestroy(h->ev_jfa[c]), h->ev_jfa[c] = nullptr;
    if (h->s_fatt[c]) cudaStreamDestroy(h->s_fatt[c]), h->s_fatt[c] = nullptr;
    if (h->s_chunk[c]) cudaStreamDestroy(h->s_chunk[c]), h->s_chunk[c] = nullptr;
    if (h->s_katt[c]) cudaStreamDestroy(h->s_katt[c]), h->s_katt[c] = nullptr;
  }
  for (int c = 0; c < kMaxChunks; ++c) {
    if (h->ev_sco[c]) cudaEventDestroy(h->ev_sco[c]), h->ev_sco[c] = nullptr;
    if (h->ev_sel[c]) cudaEventDestroy(h->ev_sel[c]), h->ev_sel[c] = nullptr;
    if (h->ev_gat[c]) cudaEventDestroy(h->ev_gat[c]), h->ev_gat[c] = nullptr;
  }
  for (cudaStream_t* t : {&h->s_sco, &h->s_sel, &h->s_gat, &h->s_att, &h->s_new, &h->s_cap,
                          &h->s_gat2})
    if (*t) cudaStreamDestroy(*t), *t = nullptr;
  if (h->ev_jgat2) cudaEventDestroy(h->ev_jgat2), h->ev_jgat2 = nullptr;
}

// Events of one step: e0 start (caller's stream); e1 after the append (scoring
// stream); e2 after the last chunk's select + set-difference (selection stream); e4 before
// the first and e5 after the last chunk's gather (gather stream); e3 before the
// first and e6 after the last attention over kept slots (attention stream); e7
// after the join (caller's stream).
void harvest_set(nosa_handle* h, cudaEvent_t* e, bool* pending) {
  if (!*pending) return;
  if (cudaEventSynchronize(e[7]) != cudaSuccess) return;
  const int pairs[6][3] = {{0, 0, 1}, {1, 1, 2}, {3, 3, 6}, {4, 4, 5}, {5, 6, 7}, {7, 0, 7}};
  for (const auto& pr : pairs) {
    float ms;
    if (cudaEventElapsedTime(&ms, e[pr[1]], e[pr[2]]) == cudaSuccess) h->t_us[pr[0]] += ms * 1000.0;
  }
  h->t_count += 1;
  *pending = false;
}

void harvest(nosa_handle* h, int r) { harvest_set(h, h->ev[r], &h->pending[r]); }

void harvest_all(nosa_handle* h) {
  if (!h->ev_made) return;
  for (int r = 0; r < kRing; ++r) harvest(h, r);
  for (int r = 0; r < kGraphRing; ++r) harvest_set(h, h->gev[r], &h->graphs[r].pending);
}

cudaError_t make_timing_events(nosa_handle* h) {
  if (h->ev_made) return cudaSuccess;
  std::vector<cudaEvent_t*> slots;
  for (int r = 0; r < kRing; ++r)
    for (int i = 0; i < kNumEv; ++i) slots.push_back(&h->ev[r][i]);
  for (int r = 0; r < kGraphRing; ++r)
    for (int i = 0; i < kNumEv; ++i) slots.push_back(&h->gev[r][i]);
  for (size_t j = 0; j < slots.size(); ++j) {
    const cudaError_t e = cudaEventCreate(slots[j]);
    if (e != cudaSuccess) {
      for (size_t m = 0; m < j; ++m) cudaEventDestroy(*slots[m]);
      return e;
    }
  }
  std::memset(h->pending, 0, sizeof(h->pending));
  h->ev_made = true;
  return cudaSuccess;
}

DevStats fresh_stats() {
  DevStats d;
  std::memset(&d, 0, sizeof(d));
  d.min_hits = INT_MAX;
  return d;
}

}  // namespace

extern "C" {

size_t nosa_payload_bytes(const nosa_config* cfg) {
  std::string why;
  if (validate(cfg, why) != NOSA_OK) return 0;
  return (size_t)payload_of(cfg->block, cfg->head_dim, cfg->dtype);
}

nosa_status nosa_config_validate(const nosa_config* cfg, char* msg, size_t msg_len) {
  std::string why;
  nosa_status st = validate(cfg, why);
  if (msg && msg_len > 0) {
    std::snprintf(msg, msg_len, "%s", why.c_str());
  }
  return st;
}

const char* nosa_last_error(const nosa_handle* h) {
  return h ? h->err.c_str() : g_thread_err.c_str();
}

nosa_status nosa_create(const nosa_config* cfg, nosa_handle** out) {
  if (!out) { g_thread_err = "out is NULL"; return NOSA_ERR_INVALID_ARG; }
  *out = nullptr;
  std::string why;
  nosa_status vs = validate(cfg, why);
  if (vs != NOSA_OK) { g_thread_err = why; return vs; }
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || cfg->device >= ndev) {
    g_thread_err = "no such CUDA device";
    cudaGetLastError();
    return NOSA_ERR_CUDA;
  }
  DeviceGuard guard(cfg->device);
  nosa_handle* h = new nosa_handle();
  h->cfg = *cfg;
  h->inject = inject_fail_from_env();
  h->s = shape_of(*cfg);
  std::memset(&h->st, 0, sizeof(h->st));
  std::memset(h->pending, 0, sizeof(h->pending));
  std::memset(h->t_us, 0, sizeof(h->t_us));
  const Shape& s = h->s;
  State& st = h->st;
  const size_t U = s.U, k = s.k, mb = s.maxBlk, W = s.W;
  cudaError_t e = cudaSuccess;
  auto A = [&](auto** p, size_t bytes) {
    if (e == cudaSuccess) e = dev_alloc(h, p, bytes);
  };
  A(&st.slots, U * k * s.payload);
  A(&st.tail, U * 2 * s.payload);
  const size_t pk_elt = s.pkb ? 2 : 4;
  A(&st.pk, U * mb * s.P * s.d * pk_elt);
  A(&st.sube, U * mb * s.P * 4);
  A(&st.se, U * mb * 4);
  A(&st.sq, U * mb * 4);
  A(&st.elig, U * W * 4);
  A(&st.selmask, U * W * 4);
  A(&st.resmask, U * W * 4);
  A(&st.nsel, U * 2 * 4);
  A(&st.slot2blk, U * k * 4);
  A(&st.loads, U * k * 3 * 4);
  A(&st.nload, U * 4);
  A(&st.block_tab, U * k * 4);
  A(&st.tab_new, U * k * 4);
  A(&st.att_cnt, U * 4);
  A(&st.sel_cnt, U * 4);
  A(&st.qhint, U * 4);
  A(&st.part_acc, U * 2 * kMaxSplits * s.G * s.d * 4);
  A(&st.part_ml, U * 2 * kMaxSplits * s.G * 2 * 4);
  A(&st.stats, sizeof(DevStats));
  A(&st.io, sizeof(StepIO));
  A(&st.ksum, U * s.d * 4);
  A(&st.esum, U * 4);
  st.trace = nullptr;
  if (const char* g = std::getenv("NOSA_TRACE"))  // step trace (diagnostics)
    if (std::atoi(g) != 0) A(&st.trace, kTraceSlots * 2 * 8);
  if (e != cudaSuccess) {
    g_thread_err = std::string("device allocation failed: ") + cudaGetErrorString(e);
    cudaGetLastError();
    free_all(h);
    delete h;
    return NOSA_ERR_OOM;
  }
  // Zeroed state: empty slots (-1), nothing eligible or resident.
  if (e == cudaSuccess) e = cudaMemset(st.slots, 0, U * k * s.payload);
  if (e == cudaSuccess) e = cudaMemset(st.tail, 0, U * 2 * s.payload);
  if (e == cudaSuccess) e = cudaMemset(st.pk, 0, U * mb * s.P * s.d * pk_elt);
  if (e == cudaSuccess) e = cudaMemset(st.sube, 0, U * mb * s.P * 4);
  if (e == cudaSuccess) e = cudaMemset(st.se, 0, U * mb * 4);
  if (e == cudaSuccess) e = cudaMemset(st.sq, 0, U * mb * 4);
  if (e == cudaSuccess) e = cudaMemset(st.elig, 0, U * W * 4);
  if (e == cudaSuccess) e = cudaMemset(st.selmask, 0, U * W * 4);
  if (e == cudaSuccess) e = cudaMemset(st.resmask, 0, U * W * 4);
  if (e == cudaSuccess) e = cudaMemset(st.nsel, 0, U * 2 * 4);
  if (e == cudaSuccess) e = cudaMemset(st.slot2blk, 0xFF, U * k * 4);
  if (e == cudaSuccess) e = cudaMemset(st.loads, 0, U * k * 3 * 4);
  if (e == cudaSuccess) e = cudaMemset(st.nload, 0, U * 4);
  if (e == cudaSuccess) e = cudaMemset(st.block_tab, 0xFF, U * k * 4);
  if (e == cudaSuccess) e = cudaMemset(st.tab_new, 0xFF, U * k * 4);
  if (e == cudaSuccess) e = cudaMemset(st.att_cnt, 0, U * 4);
  if (e == cudaSuccess) e = cudaMemset(st.sel_cnt, 0, U * 4);
  if (e == cudaSuccess) e = cudaMemset(st.qhint, 0, U * 4);
  if (e == cudaSuccess) e = cudaMemset(st.ksum, 0, U * s.d * 4);
  if (e == cudaSuccess) e = cudaMemset(st.esum, 0, U * 4);
  DevStats ds = fresh_stats();
  if (e == cudaSuccess) e = cudaMemcpy(st.stats, &ds, sizeof(ds), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    g_thread_err = std::string("device initialisation failed: ") + cudaGetErrorString(e);
    free_all(h);
    delete h;
    return NOSA_ERR_CUDA;
  }
  h->host_bytes = U * mb * (size_t)s.payload;
  void* hp = nullptr;
  // On the GPU's NUMA node when the host has several (host_store.cu).
  h->host_node = host_store_node(cfg->device);
  e = h->inject.host ? cudaErrorMemoryAllocation
                     : host_store_alloc(h->host_bytes, h->host_node, &hp, &h->host_kind,
                                        &h->host_map_bytes, &h->host_pin_fd, !h->inject.pin);
  if (h->host_kind != 1) h->host_node = -1;  // only kind 1 is bound to a node
  if (e != cudaSuccess) {
    g_thread_err = std::string("pinned host allocation failed: ") + cudaGetErrorString(e);
    cudaGetLastError();
    free_all(h);
    delete h;
    return NOSA_ERR_HOST_OOM;
  }
  h->host_store = static_cast<uint8_t*>(hp);
  void* dp = nullptr;
  e = cudaHostGetDevicePointer(&dp, hp, 0);
  if (e != cudaSuccess) {
    g_thread_err = std::string("no device view of the host store: ") + cudaGetErrorString(e);
    free_all(h);
    delete h;
    return NOSA_ERR_CUDA;
  }
  st.host = static_cast<uint8_t*>(dp);
  if (const char* g = std::getenv("NOSA_LOADED_SPLITS")) {
    const int v = std::atoi(g);
    if (v > 0 && v <= kMaxSplits) h->nsplit_new = v;
  }
  // Unit chunks of the pipelined step, by relative size: NOSA_CHUNK_SIZES (a
  // comma-separated list of weights, up to 16), else NOSA_UNIT_CHUNKS chunks
  // growing by NOSA_CHUNK_GROWTH, else by the unit count. Measured on GB300:
  // every chunk adds a selection tail and four launches, which pay off only when
  // the units are many (64 units: one chunk, 55 us against 71 us with five; 128
  // units: two; 256 units: 0.5,1,2,3,2.5,1.5, small first chunks so that the first
  // gather starts early and smaller last ones so that little attention is left
  // after the last gather: 262.5 us against 263.5 for 0.5,1,2,3,3,1 with the same
  // splits, 263.7 for 0.5,1,1.5,2.5,2.5,2 and 266.5 for 0.5,1,2,3,2,2).
  std::vector<double> weights = s.U <= 96 ? std::vector<double>{1}
                                : s.U <= 192 ? std::vector<double>{1, 1}
                                             : std::vector<double>{0.5, 1, 2, 3, 2.5, 1.5};
  if (const char* g = std::getenv("NOSA_UNIT_CHUNKS")) {
    const int v = std::atoi(g);
    if (v > 0) {
      double growth = 1.0;
      if (const char* gr = std::getenv("NOSA_CHUNK_GROWTH")) {
        const double x = std::atof(gr);
        if (x >= 0.25 && x <= 16.0) growth = x;
      }
      weights.clear();
      double w = 1.0;
      for (int c = 0; c < std::min(v, kMaxChunks); ++c, w *= growth) weights.push_back(w);
    }
  }
  if (const char* g = std::getenv("NOSA_CHUNK_SIZES")) {
    std::vector<double> ws;
    for (const char* p = g; *p && (int)ws.size() < kMaxChunks;) {
      char* end = nullptr;
      const double x = std::strtod(p, &end);
      if (end == p) break;
      if (x > 0) ws.push_back(x);
      p = (*end == ',') ? end + 1 : end;
    }
    if (!ws.empty()) weights = ws;
  }
  const int nchunks = std::max(1, std::min((int)weights.size(), s.U));
  h->nchunks = nchunks;
  {
    double total = 0.0;
    for (int c = 0; c < nchunks; ++c) total += weights[c];
    double acc = 0.0;
    int prev = 0;
    for (int c = 0; c < nchunks; ++c) {
      acc += weights[c];
      int end = (c == nchunks - 1) ? s.U : (int)std::llround(s.U * acc / total);
      end = std::max(end, prev + 1);                    // every chunk holds a unit
      end = std::min(end, s.U - (nchunks - 1 - c));     // and leaves one for each later chunk
      h->cu_base[c] = prev;
      h->cu_count[c] = end - prev;
      prev = end;
    }
  }
  // Splits of the step's attention launches (one per chunk, over its kept slots).
  // With one or two chunks, each chunk's own plan (about 20 blocks per split, half
  // a CTA per resident slot). With more, the chunks' launches overlap one another,
  // the scoring and the gathers: the fill rule then counts the whole step's units,
  // not the chunk's (a 12-unit chunk alone would take 19 splits), and a split
  // takes about 16 blocks. GB300, 8B-offload (six chunks): 4 splits per chunk
  // 262.5 us per step, 3 266.6, 5 263.9, the chunk-wise plans 266.1; 8B-longgen
  // (two chunks, k = 128): its chunk-wise 6 splits 136.2 us, 8 splits 143.3.
  // NOSA_ATTN_SPLITS forces the count.
  for (int c = 0; c < nchunks; ++c) {
    Shape sc = s;
    sc.U = h->cu_count[c];
    h->nsplit_c[c] = attention_pick_nsplit(sc, s.k, 1);
  }
  // The gather shares the GPU with scoring and attention, and the fused step runs
  // two gathers at once: 24 CTAs each keep enough host reads in flight for the
  // link (one CTA moves about 28 GB/s) and leave the SMs to the scoring and the
  // attention (GB300, 300-step medians: 8B-offload 262.5-263 us per step with 20
  // or 24 CTAs, 263.5 with 28 or 32, 282 with 64 at an earlier chunking; 3B and
  // 8B-longgen the same with 24 as with 32); NOSA_GATHER_CTAS overrides the grid.
  h->gather_grid = 24;
  if (const char* g = std::getenv("NOSA_PDL")) h->pdl = std::atoi(g) != 0;
  if (const char* g = std::getenv("NOSA_GATHER_CTAS")) {
    const int v = std::atoi(g);
    if (v > 0) h->gather_grid = v;
  }
  if (nchunks > 2 && std::getenv("NOSA_ATTN_SPLITS") == nullptr) {
    const int nv = s.k + 1;
    const int by_len = std::max(1, (nv + 8) / 16);
    const int ns = std::min(std::max(attention_pick_nsplit(s, s.k, 1), by_len),
                            std::max(1, std::min(kMaxSplits, nv / 2)));
    for (int c = 0; c < nchunks; ++c) h->nsplit_c[c] = ns;
  }
  // The selection runs in the scoring kernel where its arrays fit shared memory
  // (NOSA_FUSED_SELECT=0: a selection kernel of its own after each chunk's scoring).
  h->fused_select = score_select_fused_ok(s);
  if (const char* g = std::getenv("NOSA_FUSED_SELECT"))
    if (std::atoi(g) == 0) h->fused_select = false;
  int prio_lo = 0, prio_hi = 0;
  cudaDeviceGetStreamPriorityRange(&prio_lo, &prio_hi);
  const int prio_mid = (prio_lo + prio_hi) / 2;
  // Priorities (prio_hi is the most urgent): the gather (keeps the host link
  // busy); the chunks' scoring and selection, chunk 0 first, so that they finish
  // in chunk order without a gap between them; the attention over filled slots
  // (it ends the step); the attention over kept slots last (the bulk of the HBM
  // work, with the most slack). The unfused step keeps one scoring stream and a
  // selection stream.
  const int prio_sel = (prio_hi < prio_mid) ? prio_hi + 1 : prio_hi;
  e = cudaStreamCreateWithPriority(&h->s_gat, cudaStreamNonBlocking, prio_hi);
  // A second gather stream (fused step; NOSA_GATHER_STREAMS=1: one): the chunks'
  // gathers alternate between the two, so chunk c + 1's starts as soon as its
  // selection exists instead of after chunk c's gather kernel ends (GB300,
  // 8B-offload: 280 us against 292 us per step).
  if (const char* g = std::getenv("NOSA_GATHER_STREAMS"))
    if (std::atoi(g) == 1) h->gather_streams = 1;
  if (!h->fused_select) h->gather_streams = 1;
  if (const char* g = std::getenv("NOSA_GATHER_VEC")) h->gather_wide = std::atoi(g) == 32;
  if (e == cudaSuccess && h->gather_streams == 2) {
    e = cudaStreamCreateWithPriority(&h->s_gat2, cudaStreamNonBlocking, prio_hi);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_jgat2, cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&h->s_sel, cudaStreamNonBlocking, prio_sel);
  if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&h->s_sco, cudaStreamNonBlocking, prio_mid);
  // (the filled-slot attention of a fused step stays below every chunk's scoring:
  // a chunk whose scoring is starved delays its gather)
  const int prio_new = h->fused_select && prio_hi < prio_lo ? prio_lo - 1 : prio_sel;
  // the kept-slot attention of a fused step: the lowest level (NOSA_KEPT_PRIO=1:
  // one level up, with the filled-slot attention)
  int prio_katt = prio_lo;
  if (const char* g = std::getenv("NOSA_KEPT_PRIO"))
    if (std::atoi(g) == 1 && prio_hi < prio_lo) prio_katt = prio_lo - 1;
  if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&h->s_new, cudaStreamNonBlocking, prio_new);
  if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&h->s_att, cudaStreamNonBlocking, prio_lo);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->s_cap, cudaStreamNonBlocking);
  for (int c = 0; c < h->nchunks && e == cudaSuccess; ++c) {
    // chunk c's scoring: one level below the previous chunk's, above the kept-slot attention
    const int pc = prio_hi < prio_lo ? std::min(prio_hi + 1 + c, prio_lo - 1) : prio_hi;
    e = cudaStreamCreateWithPriority(&h->s_chunk[c], cudaStreamNonBlocking, pc);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&h->s_katt[c], cudaStreamNonBlocking, prio_katt);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_jch[c], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_jka[c], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&h->s_fatt[c], cudaStreamNonBlocking, prio_new);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_jfa[c], cudaEventDisableTiming);
  }
  for (cudaEvent_t* ep : {&h->ev_in, &h->ev_att, &h->ev_new, &h->ev_jsco, &h->ev_jsel, &h->ev_jgat,
                          &h->ev_app})
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ep, cudaEventDisableTiming);
  for (int c = 0; c < kMaxChunks && e == cudaSuccess; ++c) {
    e = cudaEventCreateWithFlags(&h->ev_sel[c], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_sco[c], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_gat[c], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    g_thread_err = std::string("stream/event creation failed: ") + cudaGetErrorString(e);
    free_all(h);
    delete h;
    return NOSA_ERR_CUDA;
  }
  if (cfg->flags & NOSA_FLAG_TIMING) {
    e = make_timing_events(h);
    if (e != cudaSuccess) {
      g_thread_err = std::string("event creation failed: ") + cudaGetErrorString(e);
      free_all(h);
      delete h;
      return NOSA_ERR_CUDA;
    }
    h->timing = true;
  }
  // Warm decode steps replay a captured graph (NOSA_GRAPHS=0 launches every
  // kernel from the host instead).
  if (const char* g = std::getenv("NOSA_GRAPHS")) h->use_graphs = std::atoi(g) != 0;

  // Caps on resident CTAs per SM of the step's scoring and attention kernels
  // (NOSA_SCORE_OCC, NOSA_ATTN_OCC; launch shapes only).
  if (const char* g = std::getenv("NOSA_SCORE_OCC")) h->score_occ = std::max(0, std::atoi(g));
  if (const char* g = std::getenv("NOSA_ATTN_OCC")) h->attn_occ = std::max(0, std::atoi(g));
  // Gamma_q from the previous step's threshold hint (NOSA_SELECT_HINT=0: the
  // radix cut at every step; the result is the same).
  if (const char* g = std::getenv("NOSA_SELECT_HINT"))
    if (std::atoi(g) == 0) st.qhint = nullptr;
  *out = h;
  return NOSA_OK;
}

nosa_status nosa_append_kv(nosa_handle* h, int32_t n_tokens, const void* k, const void* v,
                           const float* e, void* stream) {
  if (!h) return NOSA_ERR_INVALID_ARG;
  if (h->broken) return h->fail(NOSA_ERR_STATE, "handle unusable after an earlier CUDA error");
  if (n_tokens < 0) return h->fail(NOSA_ERR_INVALID_ARG, "n_tokens < 0");
  if (n_tokens == 0) return NOSA_OK;
  if (!k || !v || !e) return h->fail(NOSA_ERR_INVALID_ARG, "NULL input");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(e, 4))
    return h->fail(NOSA_ERR_INVALID_ARG, "k, v need 16-byte and e 4-byte alignment");
  if (h->L + n_tokens > h->cfg.max_context)
    return h->fail(NOSA_ERR_CAPACITY, "context would exceed max_context");
  DeviceGuard guard(h->cfg.device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaSuccess;
  const int L = (int)h->L;
  if (L > 0 && L % h->s.B == 0) err = launch_promote_tail(h->s, h->st, L / h->s.B - 1, s);
  if (err == cudaSuccess) err = launch_append_bulk(h->s, h->st, k, v, e, L, n_tokens, s);
  if (err != cudaSuccess) return h->cuda_fail(err, "append launch");
  h->L += n_tokens;
  h->last_stream = s;
  return NOSA_OK;
}

}  // extern "C"

namespace {

// Kernel nodes of a captured step whose edges can become programmatic.
struct CapNodes {
  cudaGraphNode_t append = nullptr;
  cudaGraphNode_t score[kMaxChunks] = {};
  cudaGraphNode_t gather[kMaxChunks] = {};
  cudaGraphNode_t attn_new[kMaxChunks] = {};
};

// Turns the step graph's edges on the critical path into programmatic ones (the
// dependent kernel becomes resident while its producer runs and waits in
// griddep_wait for the producer's completion and memory): append -> each chunk's
// fused scoring + selection, a chunk's selection -> its gather, its gather -> the
// attention over the slots it filled. An edge that capture did not produce
// directly (timing event nodes between the two) is left as it is.
cudaError_t make_programmatic_edges(cudaGraph_t graph, const CapNodes& n, int nchunks) {
  cudaGraphEdgeData pe;
  std::memset(&pe, 0, sizeof(pe));
  pe.from_port = cudaGraphKernelNodePortProgrammatic;
  pe.type = cudaGraphDependencyTypeProgrammatic;
  auto convert = [&](cudaGraphNode_t from, cudaGraphNode_t to) -> cudaError_t {
    if (from == nullptr || to == nullptr) return cudaSuccess;
    if (cudaGraphRemoveDependencies(graph, &from, &to, nullptr, 1) != cudaSuccess) {
      cudaGetLastError();  // no direct edge: nothing to convert
      return cudaSuccess;
    }
    cudaError_t e = cudaGraphAddDependencies(graph, &from, &to, &pe, 1);
    if (e != cudaSuccess) {  // put the ordinary edge back
      cudaGetLastError();
      e = cudaGraphAddDependencies(graph, &from, &to, nullptr, 1);
    }
    return e;
  };
  cudaError_t e = cudaSuccess;
  for (int c = 0; c < nchunks && c < kMaxChunks && e == cudaSuccess; ++c) {
    e = convert(n.append, n.score[c]);
    if (e == cudaSuccess) e = convert(n.score[c], n.gather[c]);
    if (e == cudaSuccess) e = convert(n.gather[c], n.attn_new[c]);
  }
  return e;
}

// Enqueues one decode step on `origin`: the units are processed in chunks that
// form a pipeline over five internal streams. Scoring of chunk c+1 (HBM) runs
// while chunk c is selected, gathered (host link) and attended over its kept
// slots (HBM); attention over the filled slots of chunk c follows its gather. `origin` forks at the start and joins at the end. Under stream
// capture (`capture`), timing events become graph nodes and the append node is
// returned in *append_node.
cudaError_t enqueue_step(nosa_handle* h, cudaStream_t origin, const StepArgs& args,
                         const FrontArgs* front, int n_cap, bool cold, cudaEvent_t* ev,
                         bool capture, CapNodes* nodes) {
  const Shape& sh = h->s;
  State& st = h->st;
  auto mark = [&](cudaEvent_t e, cudaStream_t t) {
    if (capture) cudaEventRecordWithFlags(e, t, cudaEventRecordExternal);
    else cudaEventRecord(e, t);
  };
  // Under capture: the node just captured on stream t (the kernel launched last).
  auto last_node = [&](cudaStream_t t) -> cudaGraphNode_t {
    cudaStreamCaptureStatus cs;
    const cudaGraphNode_t* deps = nullptr;
    size_t nd = 0;
    if (cudaStreamGetCaptureInfo(t, &cs, nullptr, nullptr, &deps, nullptr, &nd) != cudaSuccess ||
        nd != 1 || cs != cudaStreamCaptureStatusActive)
      return nullptr;
    return deps[0];
  };
  if (ev) mark(ev[0], origin);
  cudaError_t err = cudaSuccess;
  if (st.trace != nullptr) {  // fresh trace: starts at the maximum, ends at 0
    err = cudaMemsetAsync(st.trace, 0, kTraceSlots * 2 * 8, origin);
    if (err == cudaSuccess) err = launch_trace_reset(st.trace, origin);
  }
  if (err == cudaSuccess) err = cudaEventRecord(h->ev_in, origin);
  if (err == cudaSuccess) err = cudaStreamWaitEvent(h->s_sco, h->ev_in, 0);
  if (err == cudaSuccess)
    err = front ? launch_frontend(sh, st, *front, h->s_sco) : launch_append_step(sh, st, args, h->s_sco);
  if (err == cudaSuccess && capture && nodes) {
    nodes->append = last_node(h->s_sco);
    if (nodes->append == nullptr) err = cudaErrorStreamCaptureInvalidated;
  }
  if (ev) mark(ev[1], h->s_sco);
  // Fused step: every chunk's scoring + selection on its own stream, all started
  // together after the append, chunk 0 at the highest priority, so that the
  // chunks complete in order with no idle gap between them (each chunk's
  // selection tail overlaps the next chunk's scoring). Unfused: scoring of every
  // chunk back to back on one stream, each chunk's selection on another.
  const bool fused = h->fused_select;
  if (fused) {
    if (err == cudaSuccess) err = cudaEventRecord(h->ev_app, h->s_sco);
    for (int c = 0; c < h->nchunks && err == cudaSuccess; ++c) {
      err = cudaStreamWaitEvent(h->s_chunk[c], h->ev_app, 0);
      if (err == cudaSuccess)
        err = launch_score_select(sh, st, n_cap, h->cu_base[c], h->cu_count[c], cold ? 1 : 0, c,
                                  h->s_chunk[c], h->score_occ);
      if (err == cudaSuccess && capture && nodes && c < kMaxChunks)
        nodes->score[c] = last_node(h->s_chunk[c]);
      if (err == cudaSuccess) err = cudaEventRecord(h->ev_sel[c], h->s_chunk[c]);
    }
  }
  for (int c = 0; c < h->nchunks && err == cudaSuccess && !fused; ++c) {
    err = launch_score(sh, st, n_cap, h->cu_base[c], h->cu_count[c], h->s_sco);
    if (err == cudaSuccess) err = cudaEventRecord(h->ev_sco[c], h->s_sco);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(h->s_sel, h->ev_sco[c], 0);
    if (err == cudaSuccess)
      err = launch_select_setdiff(sh, st, cold ? 1 : 0, h->cu_base[c], h->cu_count[c], c, h->s_sel);
    if (err == cudaSuccess) err = cudaEventRecord(h->ev_sel[c], h->s_sel);
  }
  if (ev) mark(ev[2], fused ? h->s_chunk[h->nchunks - 1] : h->s_sel);
  AttnArgs a;
  a.units = st.slots;
  a.n_units = (long long)sh.U * sh.k;
  a.n_blocks = sh.k;
  a.tail_stride = 2 * sh.payload;
  a.tail_len = 0;  // from StepIO
  a.q = nullptr;
  a.out = nullptr;
  a.lse = nullptr;
  a.dyn = st.io;
  a.part_acc = st.part_acc;
  a.part_ml = st.part_ml;
  a.counters = st.att_cnt;
  a.err = &st.stats->error;
  a.max_ctas_per_sm = h->attn_occ;
  a.part_stride = 2 * kMaxSplits;  // every unit's own range of the partial buffers
  for (int c = 0; c < h->nchunks && err == cudaSuccess; ++c) {
    const int ns_kept = h->nsplit_c[c];
    const int ns_new = cold ? ns_kept : h->nsplit_new;
    a.nsplit_total = ns_kept + ns_new;
    a.unit_base = h->cu_base[c];
    a.unit_count = h->cu_count[c];
    // gather of chunk c (host link)
    cudaStream_t tg = (h->gather_streams == 2 && (c & 1)) ? h->s_gat2 : h->s_gat;
    err = cudaStreamWaitEvent(tg, h->ev_sel[c], 0);
    if (ev && c == 0) mark(ev[4], tg);
    if (err == cudaSuccess) err = launch_gather(sh, st, h->gather_grid, h->cu_base[c], h->cu_count[c], c,
                                                  h->gather_wide, tg);
    if (err == cudaSuccess && capture && nodes && c < kMaxChunks) nodes->gather[c] = last_node(tg);
    if (err == cudaSuccess) err = cudaEventRecord(h->ev_gat[c], tg);
    if (ev && c == h->nchunks - 1) mark(ev[5], tg);
    // attention over the slots kept from the previous step, plus the tail (fused
    // step: on the chunk's own stream, so chunks do not wait for one another)
    cudaStream_t ta = fused ? h->s_katt[c] : h->s_att;
    if (err == cudaSuccess) err = cudaStreamWaitEvent(ta, h->ev_sel[c], 0);
    if (ev && c == 0) mark(ev[3], ta);
    if (err == cudaSuccess) {
      a.block_tab = st.block_tab;
      a.tail = st.tail;  // + StepIO::tail_off
      a.nsplit = ns_kept;
      a.split_base = 0;
      a.trace = st.trace;
      a.trace_slot = c < 8 ? kTrAttnKept + c : -1;
      err = launch_attention(sh, a, ta);
    }
    // attention over the slots this chunk's gather filled (fused step: on the
    // chunk's own stream, so a chunk's launch does not wait for the previous one's)
    cudaStream_t tf = fused ? h->s_fatt[c] : h->s_new;
    if (err == cudaSuccess) err = cudaStreamWaitEvent(tf, h->ev_gat[c], 0);
    if (err == cudaSuccess) {
      a.block_tab = st.tab_new;
      a.tail = nullptr;
      a.nsplit = ns_new;
      a.split_base = ns_kept;
      a.trace_slot = c < 8 ? kTrAttnNew + c : -1;
      err = launch_attention(sh, a, tf);
      if (err == cudaSuccess && capture && nodes && c < kMaxChunks) nodes->attn_new[c] = last_node(tf);
    }
    if (fused && err == cudaSuccess) err = cudaEventRecord(h->ev_jfa[c], tf);
  }
  if (ev) mark(ev[6], fused ? h->s_katt[h->nchunks - 1] : h->s_att);
  if (fused) {  // join every chunk's attention streams (after the timing mark)
    for (int c = 0; c < h->nchunks && err == cudaSuccess; ++c) {
      err = cudaEventRecord(h->ev_jka[c], h->s_katt[c]);
      if (err == cudaSuccess) err = cudaStreamWaitEvent(origin, h->ev_jka[c], 0);
      if (err == cudaSuccess) err = cudaStreamWaitEvent(origin, h->ev_jfa[c], 0);
    }
  } else {
    if (err == cudaSuccess) err = cudaEventRecord(h->ev_att, h->s_att);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(origin, h->ev_att, 0);
    if (err == cudaSuccess) err = cudaEventRecord(h->ev_new, h->s_new);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(origin, h->ev_new, 0);
  }
  if (capture) {
    // A capture must join every stream it forked, including their last nodes.
    if (err == cudaSuccess) err = cudaEventRecord(h->ev_jsco, h->s_sco);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(origin, h->ev_jsco, 0);
    if (!h->fused_select) {  // (the fused step never forks the selection stream)
      if (err == cudaSuccess) err = cudaEventRecord(h->ev_jsel, h->s_sel);
      if (err == cudaSuccess) err = cudaStreamWaitEvent(origin, h->ev_jsel, 0);
    }
    for (int c = 0; c < h->nchunks && fused; ++c) {  // the chunks' scoring streams
      if (err == cudaSuccess) err = cudaEventRecord(h->ev_jch[c], h->s_chunk[c]);
      if (err == cudaSuccess) err = cudaStreamWaitEvent(origin, h->ev_jch[c], 0);
    }
    if (err == cudaSuccess) err = cudaEventRecord(h->ev_jgat, h->s_gat);
    if (h->gather_streams == 2 && h->nchunks >= 2) {  // the second gather stream
      if (err == cudaSuccess) err = cudaEventRecord(h->ev_jgat2, h->s_gat2);
      if (err == cudaSuccess) err = cudaStreamWaitEvent(origin, h->ev_jgat2, 0);
    }
    if (err == cudaSuccess) err = cudaStreamWaitEvent(origin, h->ev_jgat, 0);
  }
  if (ev) mark(ev[7], origin);
  return err;
}

// Captures a warm step into g (replacing what it held) with these arguments.
cudaError_t build_step_graph(nosa_handle* h, StepGraph& g, const StepArgs& args,
                             const FrontArgs* front, int N, cudaEvent_t* ev) {
  if (g.done == nullptr) {
    const cudaError_t e = cudaEventCreateWithFlags(&g.done, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
  } else if (g.exec != nullptr) {
    const cudaError_t e = cudaEventSynchronize(g.done);  // its last launch has finished
    if (e != cudaSuccess) return e;
  }
  if (g.exec) cudaGraphExecDestroy(g.exec);
  if (g.graph) cudaGraphDestroy(g.graph);
  g.exec = nullptr;
  g.graph = nullptr;
  const int n_cap = (N / kScoreCap + 1) * kScoreCap;
  cudaError_t err = cudaStreamBeginCapture(h->s_cap, cudaStreamCaptureModeRelaxed);
  if (err != cudaSuccess) return err;
  CapNodes nodes;
  const cudaError_t e_enq = enqueue_step(h, h->s_cap, args, front, n_cap, false, ev, true, &nodes);
  const cudaGraphNode_t node = nodes.append;
  cudaGraph_t graph = nullptr;
  err = cudaStreamEndCapture(h->s_cap, &graph);
  if (e_enq != cudaSuccess) err = e_enq;
  if (err == cudaSuccess && h->pdl && h->fused_select)
    err = make_programmatic_edges(graph, nodes, h->nchunks);
  if (err == cudaSuccess)
    err = cudaGraphInstantiateWithFlags(&g.exec, graph, cudaGraphInstantiateFlagUseNodePriority);
  if (err == cudaSuccess) err = cudaGraphKernelNodeGetParams(node, &g.append_params);
  if (err != cudaSuccess) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (graph) cudaGraphDestroy(graph);
    g.exec = nullptr;
    return err;
  }
  g.graph = graph;
  g.append_node = node;
  g.n_cap = n_cap;
  g.front = front != nullptr;
  g.front_gen = h->fe_gen;
  h->graph_builds += 1;
  return cudaSuccess;
}

// Runs one decode step whose first kernel is the append (front == NULL) or the
// fused front-end; the checks of the public entry points come first.
nosa_status run_step(nosa_handle* h, const StepArgs& args, const FrontArgs* front,
                     cudaStream_t s) {
  const Shape& sh = h->s;
  const int N = args.L_old / sh.B;  // candidates after the append
  const bool cold = (h->steps == 0);
  cudaError_t err = cudaSuccess;
  if (h->use_graphs && !cold && N > 0) {
    const int r = h->timing ? h->graph_pos : 0;
    StepGraph& g = h->timing ? h->graphs[r] : h->plain;
    cudaEvent_t* ev = h->timing ? h->gev[r] : nullptr;
    if (h->timing) harvest_set(h, ev, &g.pending);
    if (g.exec == nullptr || g.front != (front != nullptr) ||
        (front != nullptr && g.front_gen != h->fe_gen) || N >= g.n_cap ||
        N < g.n_cap - kScoreCap) {
      err = build_step_graph(h, g, args, front, N, ev);
    } else {
      cudaKernelNodeParams kp = g.append_params;
      StepArgs a = args;
      FrontArgs fa;
      void* kargs_append[3] = {const_cast<Shape*>(&h->s), &h->st, &a};
      void* kargs_front[4] = {&fa.tx, const_cast<Shape*>(&h->s), &h->st, &fa.p};
      if (front) {
        fa = *front;
        kp.kernelParams = kargs_front;
      } else {
        kp.kernelParams = kargs_append;
      }
      kp.extra = nullptr;
      err = cudaGraphExecKernelNodeSetParams(g.exec, g.append_node, &kp);
    }
    if (err == cudaSuccess) err = cudaGraphLaunch(g.exec, s);
    if (err == cudaSuccess) err = cudaEventRecord(g.done, s);
    if (err == cudaSuccess && h->timing) {
      g.pending = true;
      h->graph_pos = (r + 1) % kGraphRing;
    }
  } else {
    cudaEvent_t* ev = nullptr;
    if (h->timing) {
      const int r = h->ring_pos;
      harvest(h, r);
      ev = h->ev[r];
      h->pending[r] = true;
      h->ring_pos = (r + 1) % kRing;
    }
    err = enqueue_step(h, s, args, front, N, cold, ev, false, nullptr);
  }
  if (err != cudaSuccess) return h->cuda_fail(err, "decode step launch");
  // first kernel; per chunk: scoring and selection (fused: one launch), gather,
  // attention over kept and over filled slots
  h->launches += 1 + h->nchunks * (h->fused_select ? 4 : ((N > 0 ? 1 : 0) + 4));
  h->L += 1;
  h->steps += 1;
  h->last_stream = s;
  return NOSA_OK;
}

nosa_status step_checks(nosa_handle* h, const void* out, const float* lse) {
  if (h->broken) return h->fail(NOSA_ERR_STATE, "handle unusable after an earlier CUDA error");
  if (h->L < 1) return h->fail(NOSA_ERR_STATE, "decode step before any context was appended");
  if (h->L + 1 > h->cfg.max_context) return h->fail(NOSA_ERR_CAPACITY, "context is full");
  if (!out) return h->fail(NOSA_ERR_INVALID_ARG, "NULL output");
  if (!aligned(out, 16) || (lse && !aligned(lse, 4)))
    return h->fail(NOSA_ERR_INVALID_ARG, "out needs 16-byte and lse 4-byte alignment");
  return NOSA_OK;
}

}  // namespace

extern "C" {

nosa_status nosa_decode_step(nosa_handle* h, const void* q, const void* k_new, const void* v_new,
                             const float* e_new, void* out, float* lse, void* stream) {
  if (!h) return NOSA_ERR_INVALID_ARG;
  const nosa_status cs = step_checks(h, out, lse);
  if (cs != NOSA_OK) return cs;
  if (!q || !k_new || !v_new || !e_new) return h->fail(NOSA_ERR_INVALID_ARG, "NULL input");
  if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(e_new, 4))
    return h->fail(NOSA_ERR_INVALID_ARG, "q, k_new, v_new need 16-byte alignment");
  DeviceGuard guard(h->cfg.device);
  StepArgs args;
  args.k_new = k_new;
  args.v_new = v_new;
  args.e_new = e_new;
  args.q = q;
  args.out = out;
  args.lse = lse;
  args.L_old = (int)h->L;
  return run_step(h, args, nullptr, static_cast<cudaStream_t>(stream));
}

size_t nosa_frontend_rows(const nosa_config* cfg) {
  std::string why;
  if (validate(cfg, why) != NOSA_OK) return 0;
  return (size_t)(cfg->n_q_heads + 2 * cfg->n_kv_heads) * cfg->head_dim + cfg->n_kv_heads;
}

size_t nosa_frontend_packed_bytes(const nosa_config* cfg, int32_t hidden) {
  const size_t F = nosa_frontend_rows(cfg);
  if (F == 0 || hidden < 64 || hidden > 65536 || hidden % 64 != 0) return 0;
  return frontend_packed_bytes((int)F, hidden);
}

nosa_status nosa_frontend_pack(const nosa_config* cfg, int32_t hidden, const void* w,
                               void* w_packed, void* stream) {
  const size_t F = nosa_frontend_rows(cfg);
  if (F == 0) { g_thread_err = "invalid configuration"; return NOSA_ERR_INVALID_ARG; }
  if (hidden < 64 || hidden > 65536 || hidden % 64 != 0) {
    g_thread_err = "hidden must be a multiple of 64 in [64, 65536]";
    return NOSA_ERR_INVALID_ARG;
  }
  if (!w || !w_packed || !aligned(w, 16) || !aligned(w_packed, 16)) {
    g_thread_err = "w and w_packed must be non-NULL and 16-byte aligned";
    return NOSA_ERR_INVALID_ARG;
  }
  DeviceGuard guard(cfg->device);
  const cudaError_t e = launch_frontend_pack(w, w_packed, (int)F, hidden,
                                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    g_thread_err = std::string("pack launch: ") + cudaGetErrorString(e);
    return NOSA_ERR_CUDA;
  }
  return NOSA_OK;
}

nosa_status nosa_decode_step_hidden(nosa_handle* h, const void* x, int32_t hidden,
                                    const void* w_packed, void* q_out, void* out, float* lse,
                                    void* stream) {
  const void* w = w_packed;
  if (!h) return NOSA_ERR_INVALID_ARG;
  const nosa_status cs = step_checks(h, out, lse);
  if (cs != NOSA_OK) return cs;
  const Shape& sh = h->s;
  if (sh.dtype != NOSA_BF16) return h->fail(NOSA_ERR_UNSUPPORTED, "the fused front-end needs bf16");
  if (sh.batch > 256) return h->fail(NOSA_ERR_UNSUPPORTED, "the fused front-end needs batch <= 256");
  if (!x || !w) return h->fail(NOSA_ERR_INVALID_ARG, "NULL input");
  if (hidden < 64 || hidden > 65536 || hidden % 64 != 0)
    return h->fail(NOSA_ERR_INVALID_ARG, "hidden must be a multiple of 64 in [64, 65536]");
  if (!aligned(x, 16) || !aligned(w, 16) || (q_out && !aligned(q_out, 16)))
    return h->fail(NOSA_ERR_INVALID_ARG, "x, w_packed, q_out need 16-byte alignment");
  DeviceGuard guard(h->cfg.device);
  if (!frontend_available())
    return h->fail(NOSA_ERR_UNSUPPORTED, "the driver offers no tensor-map encoder");
  const int F = (sh.Hq + 2 * sh.Hkv) * sh.d + sh.Hkv;
  const int tiles = (F + 127) / 128;
  const int kblocks = hidden / 64;
  const int npad = sh.batch <= 16 ? 16 : (sh.batch + 15) / 16 * 16;
  if (h->fe_hidden != hidden) {
    // Splits per row tile (the cluster size): about one CTA per SM, at most 8,
    // and every cluster resident at once (checked with the occupancy query).
    // A shorter stage ring lets two CTAs share an SM, which raises the number
    // of clusters that fit; the split count comes first, then the ring depth.
    FrontParams q;
    std::memset(&q, 0, sizeof(q));
    q.tiles = tiles;
    q.npad = npad;
    const int max_stages = frontend_stages(npad);
    int ksplit = std::max(1, std::min(std::min(kblocks, 8), sm_count_current() / tiles));
    if (const char* g = std::getenv("NOSA_FRONT_KSPLIT")) {  // tuning override
      const int v = std::atoi(g);
      if (v >= 1) ksplit = std::min(std::min(kblocks, 8), v);
    }
    auto fits = [&](int ks, int st) {
      q.ksplit = ks;
      q.stages = st;
      return ks == 1 || frontend_max_clusters(q) >= tiles;
    };
    int stages = max_stages;
    for (; ksplit > 1; --ksplit) {
      for (stages = max_stages; stages >= 3 && !fits(ksplit, stages); --stages) {
      }
      if (stages >= 3) break;
    }
    if (ksplit == 1) stages = max_stages;
    q.stages = stages;
    if (!h->q_buf) {
      const cudaError_t e = cudaMalloc(&h->q_buf, (size_t)sh.batch * sh.Hq * sh.d * 2);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return h->fail(NOSA_ERR_OOM, "front-end query buffer");
      }
    }
    h->fe_hidden = hidden;
    h->fe_ksplit = ksplit;
    h->fe_stages = q.stages;
    h->fe_gen += 1;
  }
  const int ksplit = h->fe_ksplit;
  FrontArgs fa;
  std::memset(&fa, 0, sizeof(fa));
  FrontParams& p = fa.p;
  p.F = F;
  p.Fpad = tiles * 128;
  p.D = hidden;
  p.kblocks = kblocks;
  p.ksplit = ksplit;
  p.tiles = tiles;
  p.npad = npad;
  p.tmem_cols = 32;
  while (p.tmem_cols < npad) p.tmem_cols *= 2;
  p.stages = h->fe_stages;
  p.batch = sh.batch;
  p.L_old = (int)h->L;
  p.q = q_out ? q_out : h->q_buf;
  p.out = out;
  p.lse = lse;
  p.err = &h->st.stats->error;
  p.w_packed = static_cast<const uint8_t*>(w);
  if (!frontend_encode(fa, x, sh.batch, hidden))
    return h->fail(NOSA_ERR_INVALID_ARG, "tensor-map encoding of x failed");
  StepArgs args;
  std::memset(&args, 0, sizeof(args));
  args.q = p.q;
  args.out = out;
  args.lse = lse;
  args.L_old = p.L_old;
  return run_step(h, args, &fa, static_cast<cudaStream_t>(stream));
}

nosa_status nosa_stats(nosa_handle* h, nosa_stats_t* out) {
  if (!h || !out) return NOSA_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return h->cuda_fail(e, "synchronise");
  harvest_all(h);
  DevStats ds;
  e = cudaMemcpy(&ds, h->st.stats, sizeof(ds), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return h->cuda_fail(e, "stats read");
  std::memset(out, 0, sizeof(*out));
  out->steps = h->steps;
  out->context = h->L;
  out->host_loads = (int64_t)ds.host_loads;
  out->tail_loads = (int64_t)ds.tail_loads;
  out->host_bytes = (int64_t)ds.host_loads * h->s.payload;
  out->cold_host_loads = (int64_t)ds.cold_host_loads;
  out->max_host_loads_unit = ds.max_host_loads_unit;
  out->min_hits = ds.hit_samples ? ds.min_hits : 0;
  out->sum_hits = (int64_t)ds.sum_hits;
  out->hit_samples = (int64_t)ds.hit_samples;
  out->gamma_min = ds.hit_samples ? (double)ds.min_hits / h->s.k : 0.0;
  out->gamma_mean = ds.hit_samples ? (double)ds.sum_hits / ((double)h->s.k * ds.hit_samples) : 0.0;
  out->near_ties = (int64_t)ds.near_ties;
  out->device_error = ds.error;
  out->host_numa_node = h->host_node;
  out->host_store_kind = h->host_kind;
  out->host_store_pinned = h->host_pin_fd >= 0 ? 1 : 0;
  for (int i = 0; i < 8; ++i) out->t_us[i] = h->t_us[i];
  out->t_count = h->t_count;
  out->launches = h->launches;
  return NOSA_OK;
}

nosa_status nosa_stats_reset(nosa_handle* h) {
  if (!h) return NOSA_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return h->cuda_fail(e, "synchronise");
  harvest_all(h);
  DevStats old;
  e = cudaMemcpy(&old, h->st.stats, sizeof(old), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return h->cuda_fail(e, "stats read");
  DevStats ds = fresh_stats();
  ds.error = old.error;  // a device error is not a counter
  e = cudaMemcpy(h->st.stats, &ds, sizeof(ds), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return h->cuda_fail(e, "stats reset");
  std::memset(h->t_us, 0, sizeof(h->t_us));
  h->t_count = 0;
  h->launches = 0;
  return NOSA_OK;
}

nosa_status nosa_set_timing(nosa_handle* h, int32_t on) {
  if (!h) return NOSA_ERR_INVALID_ARG;
  if (!on) {
    h->timing = false;
    return NOSA_OK;
  }
  DeviceGuard guard(h->cfg.device);
  const cudaError_t e = make_timing_events(h);
  if (e != cudaSuccess) return h->cuda_fail(e, "event creation");
  h->timing = true;
  return NOSA_OK;
}

size_t nosa_debug_size(const nosa_handle* h, int32_t what) {
  if (!h) return 0;
  const Shape& s = h->s;
  const size_t U = s.U, k = s.k, mb = s.maxBlk, W = s.W;
  switch (what) {
    case NOSA_DBG_SEL: return U * k * 4;
    case NOSA_DBG_NSEL: return U * 2 * 4;
    case NOSA_DBG_ELIG: return U * W * 4;
    case NOSA_DBG_SLOTS: return U * k * 4;
    case NOSA_DBG_LOADS: return U * k * 3 * 4;
    case NOSA_DBG_NLOAD: return U * 4;
    case NOSA_DBG_POOLED: return U * mb * s.P * s.d * (s.pkb ? 2 : 4);
    case NOSA_DBG_SE: return U * mb * 4;
    case NOSA_DBG_SQ: return U * mb * 4;
    case NOSA_DBG_SLOTPOOL: return U * k * (size_t)s.payload;
    case NOSA_DBG_HOST: return h->host_bytes;
    case NOSA_DBG_TAIL: return U * 2 * (size_t)s.payload;
    case NOSA_DBG_TRACE: return h->st.trace ? (size_t)kTraceSlots * 2 * 8 : 0;
    default: return 0;
  }
}

nosa_status nosa_debug_read(nosa_handle* h, int32_t what, size_t offset, void* dst, size_t bytes) {
  if (!h || !dst) return NOSA_ERR_INVALID_ARG;
  const size_t size = nosa_debug_size(h, what);
  if (size == 0) return h->fail(NOSA_ERR_INVALID_ARG, "unknown debug array");
  if (offset > size || bytes > size - offset) return h->fail(NOSA_ERR_INVALID_ARG, "range outside the array");
  DeviceGuard guard(h->cfg.device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return h->cuda_fail(e, "synchronise");
  const State& st = h->st;
  if (what == NOSA_DBG_SEL) {
    if (bytes == 0) return NOSA_OK;
    // The lists are not kept on the device: between steps the eligibility words are
    // the last step's Gamma_e (strict eviction; blocks completed since are in no
    // list) and the selection words its Gamma, so Gamma_e = sel & elig ascending,
    // then Gamma_q = sel & ~elig ascending, -1 padded to k.
    const size_t k = (size_t)h->s.k, W = (size_t)h->s.W, row = k * 4;
    const size_t u0 = offset / row, u1 = (offset + bytes + row - 1) / row;
    std::vector<uint32_t> sm((u1 - u0) * W), el((u1 - u0) * W);
    e = cudaMemcpy(sm.data(), st.selmask + u0 * W, sm.size() * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess)
      e = cudaMemcpy(el.data(), st.elig + u0 * W, el.size() * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return h->cuda_fail(e, "debug read");
    std::vector<int32_t> lists((u1 - u0) * k, -1);
    for (size_t u = 0; u < u1 - u0; ++u) {
      size_t j = 0;
      for (int pass = 0; pass < 2; ++pass)
        for (size_t w = 0; w < W; ++w) {
          uint32_t bits = sm[u * W + w] & (pass == 0 ? el[u * W + w] : ~el[u * W + w]);
          for (; bits != 0u && j < k; bits &= bits - 1)
            lists[u * k + j++] = (int32_t)(w * 32 + __builtin_ctz(bits));
        }
    }
    std::memcpy(dst, reinterpret_cast<const uint8_t*>(lists.data()) + (offset - u0 * row), bytes);
    return NOSA_OK;
  }
  const void* base = nullptr;
  switch (what) {
    case NOSA_DBG_NSEL: base = st.nsel; break;
    case NOSA_DBG_ELIG: base = st.elig; break;
    case NOSA_DBG_SLOTS: base = st.slot2blk; break;
    case NOSA_DBG_LOADS: base = st.loads; break;
    case NOSA_DBG_NLOAD: base = st.nload; break;
    case NOSA_DBG_POOLED: base = st.pk; break;
    case NOSA_DBG_SE: base = st.se; break;
    case NOSA_DBG_SQ: base = st.sq; break;
    case NOSA_DBG_SLOTPOOL: base = st.slots; break;
    case NOSA_DBG_TAIL: base = st.tail; break;
    case NOSA_DBG_TRACE: base = st.trace; break;
    case NOSA_DBG_HOST:
      e = cudaMemcpy(dst, st.host + offset, bytes, cudaMemcpyDefault);
      if (e != cudaSuccess) return h->cuda_fail(e, "debug read");
      return NOSA_OK;
  }
  e = cudaMemcpy(dst, static_cast<const uint8_t*>(base) + offset, bytes, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return h->cuda_fail(e, "debug read");
  return NOSA_OK;
}

void nosa_destroy(nosa_handle* h) {
  if (!h) return;
  {
    DeviceGuard guard(h->cfg.device);
    cudaDeviceSynchronize();
    free_all(h);
  }
  delete h;
}

size_t nosa_attention_workspace_bytes(const nosa_config* cfg, int32_t n_blocks) {
  std::string why;
  if (validate(cfg, why) != NOSA_OK || n_blocks < 0) return 0;
  DeviceGuard guard(cfg->device);
  const Shape s = shape_of(*cfg);
  return attention_workspace_bytes(s, attention_plan_single(s, n_blocks).slots);
}

nosa_status nosa_sparse_attention(const nosa_config* cfg, const void* units, int64_t n_units,
                                  const int32_t* block_tab, int32_t n_blocks, const void* tail,
                                  int32_t tail_len, const void* q, void* out, float* lse,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  std::string why;
  nosa_status vs = validate(cfg, why);
  if (vs != NOSA_OK) { g_thread_err = why; return vs; }
  if (n_blocks < 0 || n_units < 0 || (n_blocks > 0 && (!units || !block_tab)) || !q || !out ||
      !workspace) {
    g_thread_err = "NULL or negative argument"; return NOSA_ERR_INVALID_ARG;
  }
  if (tail && (tail_len < 0 || tail_len > cfg->block)) {
    g_thread_err = "tail_len must be in [0, block]"; return NOSA_ERR_INVALID_ARG;
  }
  if (!aligned(units, 16) || !aligned(tail, 16) || !aligned(q, 16) || !aligned(out, 16) ||
      !aligned(workspace, 16) || !aligned(block_tab, 4) || (lse && !aligned(lse, 4))) {
    g_thread_err = "misaligned pointer"; return NOSA_ERR_INVALID_ARG;
  }
  DeviceGuard guard(cfg->device);
  const Shape s = shape_of(*cfg);
  const AttnPlan plan = attention_plan_single(s, n_blocks);
  const bool streamk = plan.sk_ctas > 0 && (n_blocks + (tail ? 1 : 0)) > 0;
  const int nsplit = streamk ? plan.seg_cap : plan.nsplit;
  const size_t need = attention_workspace_bytes(s, plan.slots);
  if (workspace_bytes < need) {
    g_thread_err = "workspace too small (see nosa_attention_workspace_bytes)";
    return NOSA_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t acc_bytes = ((size_t)s.U * nsplit * s.G * s.d * 4 + 15) & ~(size_t)15;
  const size_t ml_bytes = ((size_t)s.U * nsplit * s.G * 2 * 4 + 15) & ~(size_t)15;
  AttnArgs a;
  a.units = static_cast<const uint8_t*>(units);
  a.n_units = units ? n_units : 0;
  a.block_tab = block_tab;
  a.n_blocks = n_blocks;
  a.tail = static_cast<const uint8_t*>(tail);
  a.tail_stride = s.payload;
  a.tail_len = tail_len;
  a.q = q;
  a.out = out;
  a.lse = lse;
  const size_t cnt_bytes = ((size_t)s.U * 4 + 15) & ~(size_t)15;
  a.part_acc = reinterpret_cast<float*>(ws);
  a.part_ml = reinterpret_cast<float*>(ws + acc_bytes);
  a.nsplit = nsplit;
  a.split_base = 0;
  a.nsplit_total = nsplit;
  a.unit_base = 0;
  a.unit_count = s.U;
  a.counters = reinterpret_cast<int*>(ws + acc_bytes + ml_bytes);
  a.err = reinterpret_cast<int*>(ws + acc_bytes + ml_bytes + cnt_bytes);
  if (streamk) {
    a.sk_ctas = plan.sk_ctas;
    a.seg_cap = plan.seg_cap;
  }
  // counters and error word start at zero (one memset over both)
  cudaError_t e = cudaMemsetAsync(a.counters, 0, cnt_bytes + sizeof(int), st);
  if (e == cudaSuccess) e = launch_attention(s, a, st);
  if (e != cudaSuccess) {
    g_thread_err = std::string("attention launch: ") + cudaGetErrorString(e);
    return NOSA_ERR_CUDA;
  }
  return NOSA_OK;
}

namespace {
// Events of the last timed training-time forward of this thread.
struct PrefillTimer {
  int dev = -1;
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  bool pending = false;
  cudaError_t ensure(int device) {
    if (dev == device && ev[0]) return cudaSuccess;
    for (auto& e : ev)
      if (e) cudaEventDestroy(e), e = nullptr;
    for (auto& e : ev) {
      const cudaError_t r = cudaEventCreate(&e);
      if (r != cudaSuccess) return r;
    }
    dev = device;
    return cudaSuccess;
  }
};
thread_local PrefillTimer g_prefill_timer;

Shape prefill_virtual_shape(const Shape& s, int L) {
  Shape sv = s;  // one virtual unit per (request, position, KV head)
  sv.batch = s.batch * L;
  sv.U = s.batch * L * s.Hkv;
  return sv;
}
nosa_status prefill_checks(const nosa_config* cfg, int32_t seq_len) {
  std::string why;
  const nosa_status vs = validate(cfg, why);
  if (vs != NOSA_OK) {
    g_thread_err = why;
    return vs;
  }
  if (seq_len < 1 || seq_len > cfg->max_context) {
    g_thread_err = "seq_len must be in [1, max_context]";
    return NOSA_ERR_INVALID_ARG;
  }
  if (seq_len > 131072 || (long long)cfg->batch * seq_len * cfg->n_kv_heads > (1LL << 30)) {
    g_thread_err = "seq_len must be <= 131072 and batch * seq_len * n_kv_heads <= 2^30";
    return NOSA_ERR_UNSUPPORTED;
  }
  return NOSA_OK;
}
}  // namespace

size_t nosa_prefill_workspace_bytes(const nosa_config* cfg, int32_t seq_len) {
  if (prefill_checks(cfg, seq_len) != NOSA_OK) return 0;
  DeviceGuard guard(cfg->device);
  const Shape s = shape_of(*cfg);
  const int nsplit = prefill_tiled_ok(s, seq_len)
                         ? 1
                         : attention_pick_nsplit(prefill_virtual_shape(s, seq_len), s.k, 1);
  return prefill_layout(s, seq_len, nsplit).total;
}

nosa_status nosa_prefill_forward(const nosa_config* cfg, int32_t seq_len, const void* q,
                                 const void* k, const void* v, const float* e, void* out,
                                 float* lse, int32_t* sel, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  const nosa_status cs = prefill_checks(cfg, seq_len);
  if (cs != NOSA_OK) return cs;
  if (!q || !k || !v || !e || !out || !workspace) {
    g_thread_err = "NULL argument";
    return NOSA_ERR_INVALID_ARG;
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(e, 4) || (lse && !aligned(lse, 4)) || (sel && !aligned(sel, 4)) ||
      !aligned(workspace, 256)) {
    g_thread_err = "misaligned pointer (q, k, v, out 16 bytes; workspace 256 bytes)";
    return NOSA_ERR_INVALID_ARG;
  }
  DeviceGuard guard(cfg->device);
  const Shape s = shape_of(*cfg);
  const Shape sv = prefill_virtual_shape(s, seq_len);
  const bool tiled = prefill_tiled_ok(s, seq_len);
  const int nsplit = tiled ? 1 : attention_pick_nsplit(sv, s.k, 1);
  const PrefillLayout w = prefill_layout(s, seq_len, nsplit);
  if (workspace_bytes < w.total) {
    g_thread_err = "workspace too small (see nosa_prefill_workspace_bytes)";
    return NOSA_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int nblk = (seq_len + s.B - 1) / s.B;
  const bool timing = (cfg->flags & NOSA_FLAG_TIMING) != 0;
  PrefillTimer& tm = g_prefill_timer;
  cudaError_t err = cudaSuccess;
  if (timing) {
    tm.pending = false;
    err = tm.ensure(cfg->device);
    if (err == cudaSuccess) err = cudaEventRecord(tm.ev[0], st);
  }
  if (err == cudaSuccess) err = cudaMemsetAsync(ws + w.counters, 0, w.err + 256 - w.counters, st);
  if (err == cudaSuccess) err = launch_prefill_front(s, seq_len, q, k, v, e, sel, ws, w, tiled, st);
  if (timing && err == cudaSuccess) err = cudaEventRecord(tm.ev[1], st);
  auto finish = [&]() {
    if (timing && err == cudaSuccess) {
      err = cudaEventRecord(tm.ev[2], st);
      tm.pending = err == cudaSuccess;
    }
  };
  if (tiled) {
    if (err == cudaSuccess)
      err = launch_prefill_tile(s, seq_len, ws + w.units, reinterpret_cast<const int32_t*>(ws + w.tab),
                                reinterpret_cast<const uint32_t*>(ws + w.vmax), q, out, lse,
                                reinterpret_cast<int*>(ws + w.err), st);
    finish();
    if (err != cudaSuccess) {
      g_thread_err = std::string("training-time forward launch: ") + cudaGetErrorString(err);
      return NOSA_ERR_CUDA;
    }
    return NOSA_OK;
  }
  AttnArgs a;
  a.units = ws + w.units;
  a.n_units = (long long)s.U * nblk;
  a.block_tab = reinterpret_cast<const int32_t*>(ws + w.tab);
  a.n_blocks = s.k;
  a.tail = ws + w.units;
  a.tail_stride = 0;
  a.tail_len = 0;
  a.q = q;
  a.out = out;
  a.lse = lse;
  a.part_acc = reinterpret_cast<float*>(ws + w.part_acc);
  a.part_ml = reinterpret_cast<float*>(ws + w.part_ml);
  a.nsplit = nsplit;
  a.split_base = 0;
  a.nsplit_total = nsplit;
  a.counters = reinterpret_cast<int*>(ws + w.counters);
  a.err = reinterpret_cast<int*>(ws + w.err);
  a.tail_tab = reinterpret_cast<const int32_t*>(ws + w.tail_tab);
  a.tail_lens = reinterpret_cast<const int32_t*>(ws + w.tail_len);
  for (long long base = 0; base < sv.U && err == cudaSuccess; base += 65535) {
    a.unit_base = (int)base;
    a.unit_count = (int)std::min<long long>(65535, sv.U - base);
    err = launch_attention(sv, a, st);
  }
  finish();
  if (err != cudaSuccess) {
    g_thread_err = std::string("training-time forward launch: ") + cudaGetErrorString(err);
    return NOSA_ERR_CUDA;
  }
  return NOSA_OK;
}

nosa_status nosa_prefill_timing(float* front_ms, float* attention_ms) {
  PrefillTimer& tm = g_prefill_timer;
  if (!tm.pending) {
    g_thread_err = "no timed training-time forward on this thread";
    return NOSA_ERR_STATE;
  }
  DeviceGuard guard(tm.dev);
  float f = 0.f, a = 0.f;
  cudaError_t e = cudaEventSynchronize(tm.ev[2]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&f, tm.ev[0], tm.ev[1]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&a, tm.ev[1], tm.ev[2]);
  if (e != cudaSuccess) {
    g_thread_err = std::string("prefill timing events: ") + cudaGetErrorString(e);
    return NOSA_ERR_CUDA;
  }
  if (front_ms) *front_ms = f;
  if (attention_ms) *attention_ms = a;
  return NOSA_OK;
}

nosa_status nosa_prefill_device_error(const nosa_config* cfg, int32_t seq_len,
                                      const void* workspace, int32_t* err) {
  const nosa_status cs = prefill_checks(cfg, seq_len);
  if (cs != NOSA_OK) return cs;
  if (!workspace || !err) {
    g_thread_err = "NULL argument";
    return NOSA_ERR_INVALID_ARG;
  }
  DeviceGuard guard(cfg->device);
  const Shape s = shape_of(*cfg);
  const int nsplit = prefill_tiled_ok(s, seq_len)
                         ? 1
                         : attention_pick_nsplit(prefill_virtual_shape(s, seq_len), s.k, 1);
  const PrefillLayout w = prefill_layout(s, seq_len, nsplit);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(err, static_cast<const uint8_t*>(workspace) + w.err, sizeof(int32_t),
                   cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    g_thread_err = std::string("reading the device error word: ") + cudaGetErrorString(e);
    return NOSA_ERR_CUDA;
  }
  return NOSA_OK;
}

}  // extern "C"

extern "C" nosa_status nosa_selftest_bounded_wait(int32_t device, int64_t limit_ns,
                                                  int32_t* timed_out, int32_t* waited_ms) {
  if (!timed_out || !waited_ms || limit_ns <= 0 || limit_ns > 10000000000LL) {
    g_thread_err = "bad argument";
    return NOSA_ERR_INVALID_ARG;
  }
  DeviceGuard guard(device);
  int* d = nullptr;
  cudaError_t e = cudaMalloc(&d, 2 * sizeof(int));
  if (e != cudaSuccess) {
    g_thread_err = std::string("cudaMalloc: ") + cudaGetErrorString(e);
    return NOSA_ERR_OOM;
  }
  int h[2] = {-1, -1};
  e = launch_bounded_wait_probe((unsigned long long)limit_ns, d, nullptr);
  if (e == cudaSuccess) e = cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) {
    g_thread_err = std::string("bounded-wait probe: ") + cudaGetErrorString(e);
    return NOSA_ERR_CUDA;
  }
  *timed_out = (h[0] == kDevErrWaitTimeout) ? 1 : 0;
  *waited_ms = h[1];
  return NOSA_OK;
}
