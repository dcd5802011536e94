/*
 * nosa.h -- C ABI of the NOSA decode-step hot path on one GB300 (sm_103a).
 *
 * NOSA ("Native and Offloadable Sparse Attention", technical summary at
 * gist.science/paper/2510.13602) keeps the KV cache of long contexts in host
 * memory in block-sized units and, at every decode step, attends only to k
 * selected blocks per (request, KV head) that are cached on the GPU:
 *
 *   1. two-stage pooled block scoring (Methodology §1, "Block-Wise
 *      Implementation": mean pooling inside 16-token sub-blocks, max pooling
 *      over the sub-blocks of a 64-token block);
 *   2. dual selection Gamma = Gamma_e U Gamma_q (Methodology §1, "Dual-Selection
 *      Mechanism"): a query-agnostic top-k_e over eviction scores under the
 *      strict rule that a block left out of Gamma_e is never eligible again,
 *      plus a query-aware top-(k - |Gamma_e|) over q . pooled-key scores;
 *   3. the set-difference of Gamma against the GPU-resident block slots
 *      (Methodology §2, "Optimized Memory Layout");
 *   4. a UVA gather of the missing blocks from pinned host memory into the
 *      freed slots (Methodology §2, "High-Bandwidth Communication");
 *   5. block-sparse flash-decoding attention over the selected blocks and the
 *      newest (tail) block, with each token's eviction logit added to its
 *      scaled q.k logit before the softmax (Methodology §1, "ED-DMA").
 *
 * A "unit" is one (request b, KV head h); units are independent. Query head g
 * of a request belongs to KV head g / G with G = n_q_heads / n_kv_heads.
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device (or managed) addresses and stay valid
 *     until the stream has reached the call. q, k, v, out and block units must
 *     be 16-byte aligned; e, lse and index tables 4-byte aligned
 *     (NOSA_ERR_INVALID_ARG otherwise).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls marked "async" only enqueue work on it.
 *   - Every call returns a nosa_status; nosa_last_error(h) gives a message.
 *     After a CUDA error the handle enters NOSA_ERR_STATE and refuses further
 *     steps (destroy it).
 *   - A handle is not thread-safe; use one host thread per handle.
 */
#ifndef NOSA_H
#define NOSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NOSA_OK = 0,
  NOSA_ERR_INVALID_ARG = 1, /* bad configuration, pointer, size or alignment     */
  NOSA_ERR_OOM = 2,         /* device allocation failed                          */
  NOSA_ERR_HOST_OOM = 3,    /* pinned host allocation failed                     */
  NOSA_ERR_CAPACITY = 4,    /* the context would exceed max_context              */
  NOSA_ERR_CUDA = 5,        /* a CUDA call or kernel failed                      */
  NOSA_ERR_STATE = 6,       /* handle unusable after an earlier CUDA error       */
  NOSA_ERR_UNSUPPORTED = 7  /* shape outside the compiled kernel variants        */
} nosa_status;

typedef enum { NOSA_F32 = 0, NOSA_BF16 = 1 } nosa_dtype;

/* Flags of nosa_config.flags. */
#define NOSA_FLAG_TIMING 1u /* record CUDA events around each phase (stats.t_us) */
/* Store the pooled (sub-block mean) keys in bf16 instead of fp32: each mean is the
 * fp32 sum of the sub-block's keys in token order times 1/16, rounded to nearest
 * even in bf16. Halves the scoring traffic (the largest HBM stream of a step at
 * long context); selections then follow the rounded pooled keys. */
#define NOSA_FLAG_POOLED_BF16 2u

/*
 * Configuration, fixed at nosa_create.
 *   batch, n_q_heads, n_kv_heads : requests and heads; n_q_heads % n_kv_heads == 0,
 *                                  G = n_q_heads / n_kv_heads in {1,2,3,4,6,8}.
 *   head_dim                     : d, 64 or 128.
 *   dtype                        : nosa_dtype of q, k, v and out.
 *   block, sub_block             : B and S tokens; B = 64, S = 16 (P = 4 sub-blocks).
 *   k, k_e                       : selected blocks per unit and the query-agnostic
 *                                  share; 0 <= k_e <= k, 1 <= k <= 256.
 *   max_context                  : capacity in tokens per request (sizes the host store);
 *                                  ceil(max_context / B) <= 32768,
 *                                  batch * n_kv_heads <= 65535.
 *   device                       : CUDA device ordinal.
 *   flags                        : NOSA_FLAG_* bits.
 */
typedef struct {
  int32_t batch, n_q_heads, n_kv_heads, head_dim;
  int32_t dtype;
  int32_t block, sub_block, k, k_e;
  int32_t max_context;
  int32_t device;
  uint32_t flags;
} nosa_config;

/*
 * Block unit ("minimal block-sized unit", Methodology §2). One unit holds the
 * B tokens of one (request, KV head, block) and is the byte image copied
 * between the host store, the tail buffers and the slot pool:
 *   K : bytes [0, B*d*elt)        16-byte chunk-major: element (t, dim) at
 *                                 ((dim / c) * B + t) * 16 + (dim % c) * elt, c = 16 / elt
 *   V : bytes [B*d*elt, 2*B*d*elt) token-major: element (t, dim) at + (t*d + dim) * elt
 *   e : fp32 eviction logits, e[t] at 2*B*d*elt + 4*t
 *   zero padding to a multiple of 256 bytes.
 * elt = 4 (NOSA_F32) or 2 (NOSA_BF16). Returns the unit size in bytes
 * (33024 for B=64, d=128 bf16 or d=64 fp32; 16640 for d=64 bf16), 0 if invalid.
 */
size_t nosa_payload_bytes(const nosa_config* cfg);

/*
 * Checks a configuration without touching any GPU. Writes a reason into msg
 * (if non-NULL, NUL-terminated, at most msg_len bytes) when it is rejected.
 */
nosa_status nosa_config_validate(const nosa_config* cfg, char* msg, size_t msg_len);

typedef struct nosa_handle nosa_handle;

/*
 * Creates a handle: allocates, on cfg->device, the slot pool [U][k] units, the
 * double-buffered tail [U][2] units, pooled keys [U][maxBlk][P][d] fp32,
 * eviction scores, eligibility bitmasks, slot tables and scratch; and the host
 * store [U][maxBlk] units in pinned, mapped host memory (U = batch *
 * n_kv_heads, maxBlk = ceil(max_context / B)). The handle owns all of it.
 * A host store of 1 GiB or more is laid out in transparent huge pages, faulted
 * in at once and held by long-term page pins (an io_uring buffer registration,
 * close-on-exec, excluded from fork) so that the host kernel cannot split or
 * move its pages while the GPU reads them; the pins count against the process's
 * locked-memory limit unless it holds CAP_IPC_LOCK, and where they are refused
 * the store is a plain cudaHostAlloc (environment NOSA_HOST_HUGEPAGE=0 asks
 * for that directly). nosa_stats reports which (host_store_kind,
 * host_store_pinned); nosa_destroy drops the pins.
 * Errors: INVALID_ARG, UNSUPPORTED, OOM, HOST_OOM, CUDA. *out is NULL on error.
 */
nosa_status nosa_create(const nosa_config* cfg, nosa_handle** out);

/*
 * Appends n_tokens tokens to every request (the prompt, or more context).
 * Async. k, v : device [batch][n_tokens][n_kv_heads][d] of cfg dtype;
 * e : device fp32 [batch][n_tokens][n_kv_heads]. Blocks that become candidates
 * (every block but the newest) are pooled, marked eligible and written to the
 * host store; no selection or eviction happens here (the cold start: the next
 * decode step loads min(k, N) blocks). CAPACITY if the context would exceed
 * max_context (nothing is enqueued). n_tokens = 0 is a no-op.
 */
nosa_status nosa_append_kv(nosa_handle* h, int32_t n_tokens, const void* k, const void* v,
                           const float* e, void* stream);

/*
 * One decode step for every request. Async.
 *   q     : device [batch][n_q_heads][d] cfg dtype (the step's queries)
 *   k_new : device [batch][n_kv_heads][d] cfg dtype (the step's new key)
 *   v_new : device [batch][n_kv_heads][d] cfg dtype
 *   e_new : device fp32 [batch][n_kv_heads] (the new token's eviction logit)
 *   out   : device [batch][n_q_heads][d] cfg dtype (written)
 *   lse   : device fp32 [batch][n_q_heads] natural-log sum-exp of the logits, or NULL
 * Order: append the token (incremental pooling: a completed 16-token sub-block
 * is averaged, the block's eviction score is the max of its sub-block means;
 * the block before a newly opened one becomes a candidate, eligible, and is
 * written back to the host store) -> score -> dual select -> set-difference ->
 * gather -> split-K attention -> combine. The context must be >= 1 token
 * before the call (STATE otherwise). CAPACITY when the context is full.
 * Every step after the first replays a CUDA graph of the whole step captured
 * by the handle (rebuilt when the candidate count leaves a 32-block window), so
 * its host cost is one graph-node update and one graph launch; the environment
 * variable NOSA_GRAPHS=0 at create time launches every kernel instead.
 */
nosa_status nosa_decode_step(nosa_handle* h, const void* q, const void* k_new, const void* v_new,
                             const float* e_new, void* out, float* lse, void* stream);

/*
 * Fused front-end (NOSA technical summary, Methodology §2 "Kernel Fusion": the
 * eviction head, the QKV split and the pooling in one kernel; §1 "Dual-Selection
 * Mechanism": the eviction head scores tokens independently of the query).
 *
 * Rows of the packed projection for this configuration:
 * F = (n_q_heads + 2 * n_kv_heads) * head_dim + n_kv_heads (0 if cfg is invalid).
 */
size_t nosa_frontend_rows(const nosa_config* cfg);

/*
 * Bytes of the packed form of the front-end weights for this configuration and
 * hidden width: ceil(F / 128) * (hidden / 64) * 16384 (0 if invalid).
 */
size_t nosa_frontend_packed_bytes(const nosa_config* cfg, int32_t hidden);

/*
 * Packs the front-end weights once (they are static) into the layout the fused
 * front-end streams: every 128-row x 64-column tile of W becomes one contiguous
 * 16 KB run, rows stored in the 128-byte-swizzled order the tensor cores read
 * (row r's 16-byte chunk c at r * 128 + (c XOR (r mod 8)) * 16), the tiles of a
 * row block consecutive along the hidden width; rows past F are zeros. Async.
 *   w        : device bf16 [F][hidden], row-major (F = nosa_frontend_rows)
 *   w_packed : device, nosa_frontend_packed_bytes(cfg, hidden) bytes, written
 * Both 16-byte aligned. Errors: INVALID_ARG, CUDA.
 */
nosa_status nosa_frontend_pack(const nosa_config* cfg, int32_t hidden, const void* w,
                               void* w_packed, void* stream);

/*
 * One decode step whose inputs are projected from the layer's hidden states by
 * the library: y = W x for every request, split into the query heads (rows
 * [0, Hq d): head g = row / d), the key heads (next Hkv d rows), the value
 * heads (next Hkv d rows) and the eviction logits (last Hkv rows, one pre-exp
 * logit per KV head); q, k, v are rounded to bf16 (nearest even), e stays fp32.
 * The projection runs on the tensor cores (fp32 accumulation; the order of the
 * additions is unspecified) in the same kernel as the append and the pooling;
 * the rest of the step is nosa_decode_step's.
 *   x      : device bf16 [batch][hidden], row-major (the step's hidden states)
 *   hidden : width D, a multiple of 64 in [64, 65536]
 *   w_packed : the weights W [F][hidden] packed by nosa_frontend_pack, read only
 *   q_out  : device bf16 [batch][n_q_heads][head_dim] receiving the step's
 *            queries, or NULL (then they stay in an internal buffer)
 *   out, lse, stream: as for nosa_decode_step.
 * x, w_packed, q_out and out need 16-byte alignment. UNSUPPORTED unless cfg->dtype is
 * NOSA_BF16 and batch <= 256 (or when the driver offers no tensor-map encoder);
 * OOM if the front-end's query buffer cannot be allocated on the first call.
 * Other errors as nosa_decode_step. The projection splits the hidden width over
 * the CTAs of a thread-block cluster per 128-row tile of W (all clusters
 * resident at once) and sums the splits through distributed shared memory in
 * rank order.
 */
nosa_status nosa_decode_step_hidden(nosa_handle* h, const void* x, int32_t hidden,
                                    const void* w_packed, void* q_out, void* out, float* lse,
                                    void* stream);

/*
 * Training-time forward (NOSA technical summary, Methodology §1: the locality
 * constraint is imposed during training, so the dual selection applies at every
 * query position). For every position t of a sequence of seq_len tokens, with
 * token t appended (causal): Gamma_e(t) = the k_e best eligible candidates by
 * block eviction score, eligibility becoming Gamma_e(t) (strict eviction), and
 * Gamma_q(t) = the k - |Gamma_e(t)| best other candidates by the two-stage pooled
 * query score; the attention covers the blocks of Gamma(t) plus t's own block up
 * to t, with the eviction logit added before the softmax. Position 0 starts from
 * an empty context. Everything stays on the device; nothing is offloaded.
 *   q    : device [batch][seq_len][n_q_heads][head_dim] cfg dtype
 *   k, v : device [batch][seq_len][n_kv_heads][head_dim] cfg dtype
 *   e    : device fp32 [batch][seq_len][n_kv_heads]
 *   out  : device [batch][seq_len][n_q_heads][head_dim] cfg dtype (written)
 *   lse  : device fp32 [batch][seq_len][n_q_heads] or NULL
 *   sel  : device int32 [batch][seq_len][n_kv_heads][k] or NULL: the selection of
 *          each position (Gamma_e ascending, then Gamma_q ascending, -1 pad)
 *   workspace : device, nosa_prefill_workspace_bytes(cfg, seq_len) bytes,
 *          256-byte aligned, owned by the caller (contents are scratch)
 * seq_len in [1, cfg->max_context] and <= 131072. Async on stream. Errors:
 * INVALID_ARG (sizes, NULL, alignment, workspace too small), UNSUPPORTED, CUDA.
 * In bf16 with n_q_heads / n_kv_heads in {1, 2, 4} and head_dim in {64, 128} the
 * attention runs per query block on the tensor cores (environment variable
 * NOSA_PREFILL_TILED=0: the split-K decode attention per position instead).
 * With head_dim in {64, 128} and k - k_e <= 32 the selection's pooled query
 * scores run on the tensor cores from a three-term bf16 split of the fp32
 * operands (fp32-accurate; NOSA_PREFILL_SELECT_TC=0: fp32 on the CUDA cores).
 */
size_t nosa_prefill_workspace_bytes(const nosa_config* cfg, int32_t seq_len);
nosa_status nosa_prefill_forward(const nosa_config* cfg, int32_t seq_len, const void* q,
                                 const void* k, const void* v, const float* e, void* out,
                                 float* lse, int32_t* sel, void* workspace,
                                 size_t workspace_bytes, void* stream);
/*
 * The device error word of the last nosa_prefill_forward run in `workspace` with
 * the same cfg and seq_len: 0 none, 1 a bounded wait in a kernel gave up (the
 * selections or outputs of the affected query blocks are not written), 2 a block
 * table entry out of range (skipped) or a selection wider than the tensor-core
 * selection's lists (clamped; not reachable with |Gamma_e| = min(k_e, blocks)). Waits for the device (cudaDeviceSynchronize) and then
 * copies the 4-byte word to *err (host). INVALID_ARG on NULL or sizes outside the
 * forward's limits; CUDA on a failed copy.
 */
nosa_status nosa_prefill_device_error(const nosa_config* cfg, int32_t seq_len,
                                      const void* workspace, int32_t* err);
/*
 * Device time of the last nosa_prefill_forward called on this thread with
 * NOSA_FLAG_TIMING in cfg->flags (which then records CUDA events on its stream
 * around its two phases): *front_ms = packing, eviction sets and per-position
 * selection; *attention_ms = the attention. Waits for the second phase's end
 * event. Either pointer may be NULL. STATE if no timed forward ran on this
 * thread; CUDA on an event error.
 */
nosa_status nosa_prefill_timing(float* front_ms, float* attention_ms);

/* Counters, host-readable. gamma_* covers steps after the first decode step
 * with at least k candidates; gamma(t) = |Gamma(t) ∩ R(t-1)| / k where R(t-1)
 * is the resident blocks plus the block that was the tail at t-1. */
typedef struct {
  int64_t steps;                 /* decode steps run                               */
  int64_t context;               /* tokens per request after the last call         */
  int64_t host_loads;            /* blocks gathered from the host store            */
  int64_t tail_loads;            /* blocks copied from the old tail buffer         */
  int64_t host_bytes;            /* bytes gathered from the host store             */
  int64_t cold_host_loads;       /* host loads of the first decode step            */
  int32_t max_host_loads_unit;   /* max host loads of one unit in one step (warm)  */
  int32_t min_hits;              /* min |Gamma ∩ R(t-1)| over units and warm steps */
  int64_t sum_hits;              /* sum of |Gamma ∩ R(t-1)| over the same          */
  int64_t hit_samples;           /* number of (unit, step) samples in sum_hits     */
  double gamma_min, gamma_mean;  /* min_hits / k and sum_hits / (k * hit_samples)  */
  int64_t near_ties;             /* top-k cuts whose k-th and (k+1)-th fp32 scores
                                    differ by < 1e-5 * max |score|                  */
  int32_t device_error;          /* nonzero: a bounded wait in a kernel gave up     */
  int32_t host_numa_node;        /* NUMA node the host store is bound to, -1: none  */
  /* Accumulated device time (microseconds) of each phase when NOSA_FLAG_TIMING.
   * The step is pipelined over chunks of units on internal streams, so the
   * phases overlap; each entry spans a phase's first start to its last end:
   * [0] append+pool, [1] scoring + selection + set-difference of all chunks,
   * [2] unused (0), [3] attention over the slots kept from the previous step,
   * [4] gather, [5] from the end of [3] to the end of the step (attention over
   * the filled slots, the merge), [6] unused (0), [7] whole step.
   * t_count = steps timed. */
  double t_us[8];
  int64_t t_count;
  int64_t launches;              /* kernels launched by decode steps (host count)    */
  int32_t host_store_kind;       /* how the host store was made: 0 cudaHostAlloc,
                                    1 a mapping bound to host_numa_node, 2 a mapping
                                    in transparent huge pages (unbound)             */
  int32_t host_store_pinned;     /* 1: the process holds long-term pins on the
                                    store's pages (they cannot move or be split)   */
} nosa_stats_t;

/*
 * Placement rule of the pinned host store (no counterpart in the NOSA pages; a
 * property of this implementation). The recall reads the store over the GPU's
 * host link, so on a host with several memory nodes nosa_create binds the
 * store's pages (preferred policy) to the GPU's own node before pinning them.
 * This pure function is the rule: it returns gpu_node when at least two nodes
 * with CPUs and memory exist (mem_nodes, n_mem), gpu_node is one of them and
 * the process may allocate on it (allowed, n_allowed); else -1 (nothing bound:
 * a plain pinned allocation). nosa_create feeds it the GPU's node from sysfs
 * (/sys/bus/pci/devices/<bus id>/numa_node), the nodes of
 * /sys/devices/system/node/has_memory that have CPUs, and Mems_allowed_list of
 * /proc/self/status; nosa_stats reports the outcome (host_numa_node). No GPU
 * is touched; NULL arrays return -1.
 */
int32_t nosa_numa_choose(int32_t gpu_node, const int32_t* mem_nodes, int32_t n_mem,
                         const int32_t* allowed, int32_t n_allowed);

/* Synchronises the handle's last stream and fills *out. */
nosa_status nosa_stats(nosa_handle* h, nosa_stats_t* out);

/* Clears the counters and timers of nosa_stats (not the state). */
nosa_status nosa_stats_reset(nosa_handle* h);

/*
 * Switches the per-phase timing of nosa_stats.t_us on (on != 0) or off for the
 * decode steps that follow (NOSA_FLAG_TIMING at create time starts with it
 * on). Timing records eight CUDA events per step, which costs some device
 * time: leave it off when measuring throughput. The events are created on the
 * first switch-on. Errors: INVALID_ARG (NULL handle), CUDA.
 */
nosa_status nosa_set_timing(nosa_handle* h, int32_t on);

/*
 * Debug read-back (synchronous, for tests). Copies `bytes` bytes starting at
 * byte `offset` of the chosen array into host memory `dst`. INVALID_ARG if the
 * range is outside the array. Arrays (U units, W = ceil(maxBlk / 32)):
 *   NOSA_DBG_SEL      int32 [U][k]   Gamma_e ascending then Gamma_q ascending, -1 pad
 *                     (derived at read time from the selection and eligibility masks)
 *   NOSA_DBG_NSEL     int32 [U][2]   |Gamma_e|, |Gamma_q|
 *   NOSA_DBG_ELIG     uint32 [U][W]  eligibility bitmask (bit i%32 of word i/32)
 *   NOSA_DBG_SLOTS    int32 [U][k]   block held by each slot, -1 empty
 *   NOSA_DBG_LOADS    int32 [U][k][3] load list (block, slot, src: 0 host, 1 tail)
 *   NOSA_DBG_NLOAD    int32 [U]      loads of the last step
 *   NOSA_DBG_POOLED   fp32 (bf16 with NOSA_FLAG_POOLED_BF16) [U][maxBlk][P][d] sub-block mean keys
 *   NOSA_DBG_SE       fp32 [U][maxBlk] block eviction scores (max of sub-block means)
 *   NOSA_DBG_SQ       fp32 [U][maxBlk] query-aware block scores of the last step
 *   NOSA_DBG_SLOTPOOL bytes [U][k][payload]  slot pool
 *   NOSA_DBG_HOST     bytes [U][maxBlk][payload] host store
 *   NOSA_DBG_TAIL     bytes [U][2][payload] tail buffers (block b uses buffer b % 2)
 *   NOSA_DBG_TRACE    uint64 [48][2] step trace of the last decode step: per traced
 *                     launch, the first CTA's start and the last CTA's end on the
 *                     device's global timer (ns; start UINT64_MAX = not run); slot 0
 *                     the append, 1 + c scoring (and selection) of unit chunk c,
 *                     9 + c a separate selection, 17 + c the gather, 25 + c the
 *                     attention over kept slots, 33 + c over filled slots (slot 0
 *                     is the fused front-end for nosa_decode_step_hidden). Points
 *                     (earliest and latest CTA): 41 / 42 the front-end's
 *                     accumulator complete / epilogue done; 43 - 47 the first
 *                     chunk's selection per unit: begins (scores complete), Gamma_e
 *                     and Gamma_q marked, lists written (45, 46, 47), set-difference
 *                     done (44). Present
 *                     (size > 0) only when the environment variable NOSA_TRACE=1 was
 *                     set at nosa_create; the records cost a few atomics per CTA.
 */
enum {
  NOSA_DBG_SEL = 0, NOSA_DBG_NSEL, NOSA_DBG_ELIG, NOSA_DBG_SLOTS, NOSA_DBG_LOADS,
  NOSA_DBG_NLOAD, NOSA_DBG_POOLED, NOSA_DBG_SE, NOSA_DBG_SQ, NOSA_DBG_SLOTPOOL,
  NOSA_DBG_HOST, NOSA_DBG_TAIL, NOSA_DBG_TRACE, NOSA_DBG_COUNT_
};
nosa_status nosa_debug_read(nosa_handle* h, int32_t what, size_t offset, void* dst, size_t bytes);

/* Size in bytes of a debug array (0 for an unknown id). */
size_t nosa_debug_size(const nosa_handle* h, int32_t what);

/* Releases everything the handle owns (synchronises its device first). NULL is a no-op. */
void nosa_destroy(nosa_handle* h);

/* Last error message of the handle ("" if none); valid until the next call on h.
 * With h == NULL: the last error of nosa_create on this thread. */
const char* nosa_last_error(const nosa_handle* h);

/*
 * Block-sparse decode attention (step 5 alone) over caller-owned block units,
 * the same split-K kernel nosa_decode_step runs. Async.
 *   units      : device array of n_units block units (layout above)
 *   n_units    : number of units in `units`
 *   block_tab  : device int32 [U][n_blocks] unit index of each attended block,
 *                -1 = skip; an index outside [0, n_units) is skipped and flagged
 *                in the workspace's error word (see below)
 *   tail       : device units [U] (the partial newest block of each unit) or NULL
 *   tail_len   : tokens valid in each tail unit (0..B; ignored if tail is NULL)
 *   q, out, lse: as in nosa_decode_step (lse may be NULL)
 *   workspace  : device scratch of nosa_attention_workspace_bytes(...) bytes,
 *                16-byte aligned; holds the split-K partials. Its last 16 bytes
 *                start with an int32 error word (0 = ok, 2 = bad block index,
 *                1 = a bounded wait gave up), cleared by each call.
 * U = batch * n_kv_heads from cfg; only the shape fields of cfg are used.
 */
size_t nosa_attention_workspace_bytes(const nosa_config* cfg, int32_t n_blocks);
nosa_status nosa_sparse_attention(const nosa_config* cfg, const void* units, int64_t n_units,
                                  const int32_t* block_tab, int32_t n_blocks, const void* tail,
                                  int32_t tail_len, const void* q, void* out, float* lse,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Self-test of the kernels' bounded waits (failure detection without a GPU
 * fault): launches one thread that waits, with the same bounded mbarrier wait
 * the attention kernel uses, on a barrier nothing ever completes. The wait must
 * give up after limit_ns (0 < limit_ns <= 10 s) and report it; the context stays
 * usable. Synchronous. *timed_out = 1 when the wait gave up, *waited_ms = the
 * time it waited. (No counterpart in the NOSA pages: a robustness check of this
 * implementation.)
 */
nosa_status nosa_selftest_bounded_wait(int32_t device, int64_t limit_ns, int32_t* timed_out,
                                       int32_t* waited_ms);

/*
 * nosa_sparse_attention without a caller workspace and without allocating.
 * (The NOSA pages have no counterpart of this call: it serves callers.)
 *
 * For callers that cannot allocate device memory: a serving engine or
 * framework that reserves all device memory up front in its own pool (an
 * allocation from inside this library could fail although the pool has free
 * memory, and would escape the pool's accounting), or a latency-critical loop
 * that must avoid cudaMalloc / cudaFree because they can synchronise the device.
 * Arguments are those of nosa_sparse_attention minus the workspace; the caller
 * still passes the inputs and outputs. The split-K scratch lives in one static
 * 16 MiB array in the library's device memory, held by every GPU that loads the
 * library until the process exits; nothing is allocated. The first call on a
 * device (with cfg->device made current for the lookup) finds that array's
 * device address; make it before any stream capture. The address is kept with
 * the device's context: the first call after a cudaDeviceReset (a new context)
 * looks it up again, so it too must come before any capture. All calls share the array
 * and it keeps the last call's contents (each call clears its counters and
 * error word); calls that overlap on the GPU race. Shapes whose scratch
 * (nosa_attention_workspace_bytes) exceeds 16 MiB are rejected with
 * NOSA_ERR_CAPACITY and a message in nosa_last_error(NULL). Async.
 */
nosa_status nosa_sparse_attention_noalloc(const nosa_config* cfg, const void* units,
                                          int64_t n_units, const int32_t* block_tab,
                                          int32_t n_blocks, const void* tail, int32_t tail_len,
                                          const void* q, void* out, float* lse, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NOSA_H */
