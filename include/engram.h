/*
 * engram.h -- C ABI of the GB300 (sm_103a) Engram conditional-memory forward path.
 *
 * The operation is the one described in "DeepSeek Engram 系列导读"
 * (foosynaptic.github.io, deepseek-tech-notes, chapter 07-Engram), section
 * "Engram 工作原理":
 *   Stage A (deterministic retrieval)
 *     Step 1  x'_t = P(x_t)                               vocabulary projection
 *     Step 2  g_{t,n} = (x'_{t-n+1}, ..., x'_t), n=2..N   suffix n-grams
 *     Step 3  z_{t,n,k} = phi_{n,k}(g_{t,n})              K multiplicative-XOR heads per order
 *     Step 4  e_t = concat_{n,k} E_{n,k}[z_{t,n,k}]       row gather + concat
 *   Stage B (context-aware gating and fusion)
 *     Step 5  k_t = W_K e_t,  v_t = W_V e_t
 *     Step 6  alpha_t = sigma(RMSNorm(h_t) . RMSNorm(k_t) / sqrt(d)),  v~_t = alpha_t v_t
 *     Step 7  Y = SiLU(Conv1D_{w, dilation N}(RMSNorm(V~))) + V~   (depthwise, causal)
 *     Step 8  H <- H + Y
 * and, for M hyper-connection branches, its section "多分支 backbone 上的变体":
 * a gate per branch from h^(m) and W_K^(m) e_t, a value W_V e_t shared by all.
 * Int8 tables with a per-row scale, read from HBM or from pinned host memory
 * by the same gather kernel, follow "Engram 嵌入扩展：面向高效 DRAM/SSD 卸载的
 * 协同设计" (web.reeddaily.com), section "AgentX Engram DRAM卸载提升性能".
 *
 * Concrete choices the pages leave open (hash form, window order, pad id,
 * RMSNorm form, conv layout):
 *   h = XOR_{i=0}^{n-1} (x'_{t-i} * m_{n,k,i})  (mod 2^64, unsigned)
 *   z = h mod p_{n,k}                            (p_{n,k} the table's row count)
 *   x'_{t-i} = 0 (pad) before the first token of a sequence
 *   RMSNorm(x) = x / sqrt(mean(x^2) + eps) * g   (one weight vector per use)
 *   conv tap j multiplies the input at lag (w-1-j)*dilation (PyTorch depthwise
 *   Conv1d layout), no bias, zeros before the sequence start.
 *
 * Conventions for every entry point
 *   - Every call is asynchronous and stream-ordered on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream).  Argument checks run on
 *     the host before any launch; a failed check launches nothing.
 *   - The caller owns every buffer and the stream.  The library owns only the
 *     plan: its small device parameter block and a device error word.
 *   - Arrays are dense, row-major, and (unless stated) in device memory.  Device
 *     pointers handed to the 16-byte vector paths must be 16-byte aligned.
 *   - No exception crosses the ABI.  A status code is returned; errors found
 *     inside kernels (an index out of range, a wait that timed out) are
 *     recorded in the plan's error word and reported by engram_get_error.
 *   - Indices are int32: every table has fewer than 2^31 rows.
 *   - Calls on one plan may run concurrently on different streams only if they
 *     write disjoint buffers.
 */
#ifndef ENGRAM_GB300_H
#define ENGRAM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* engram_stream_t; /* == cudaStream_t */

typedef enum {
  ENGRAM_OK = 0,
  ENGRAM_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, bad config */
  ENGRAM_ERR_UNSUPPORTED = 2,   /* valid but outside what this build implements */
  ENGRAM_ERR_NOT_MAPPED = 3,    /* a host pointer the GPU cannot address (not pinned/registered) */
  ENGRAM_ERR_INDEX_RANGE = 4,   /* a gather index >= its table's row count (row zero-filled) */
  ENGRAM_ERR_CUDA = 5,          /* a CUDA runtime call failed */
  ENGRAM_ERR_TIMEOUT = 6,       /* a bounded in-kernel wait gave up (results invalid) */
  ENGRAM_ERR_WORKSPACE = 7      /* workspace missing or smaller than engram_plan_workspace_bytes */
} engram_status_t;

typedef enum {
  ENGRAM_F32 = 0,               /* IEEE binary32 */
  ENGRAM_BF16 = 1,              /* bfloat16 */
  ENGRAM_I8_ROWSCALE_F16 = 2    /* table only: int8 rows + one fp16 scale per row */
} engram_dtype_t;

/* Layer configuration.  The two host arrays are copied by engram_plan_create. */
typedef struct {
  int N;                        /* max n-gram order; orders 2..N.  2 <= N <= 8 */
  int K;                        /* hash heads per order.  1 <= K, (N-1)*K <= 64 */
  int row_dim;                  /* elements per table row; row bytes a multiple of 16 */
  int d;                        /* hidden size; multiple of 8 (bf16) / 4 (f32) */
  int M;                        /* hyper-connection branches, 1 <= M <= 8 */
  int conv_w;                   /* conv taps, 1 <= conv_w <= 8 */
  int conv_dilation;            /* >= 1, (conv_w-1)*conv_dilation <= 192 (the pages use N) */
  engram_dtype_t table_dtype;   /* F32, BF16 or I8_ROWSCALE_F16 */
  engram_dtype_t act_dtype;     /* F32 or BF16: H, W_kv, e and the k/v buffer */
  float eps;                    /* RMSNorm epsilon, > 0 */
  const uint32_t* primes;       /* host [R = (N-1)*K]: rows of E_{n,k}, index (n-2)*K + k */
  const uint64_t* multipliers;  /* host [sum_{n=2..N} K*n]: m_{n,k,i} at
                                   sum_{n'<n} K*n' + k*n + i; any 64-bit values */
} engram_config_t;

typedef struct engram_plan engram_plan_t;

/* Per-layer parameters.  `table` is the concatenation of the R tables E_{n,k}
 * in (n, k) n-major order: table r starts at row sum_{r'<r} primes[r'].
 * `table` (and `scales`) may be device memory or pinned/registered host memory
 * (read over UVA: NVLink-C2C on Grace-Blackwell).  All others are device. */
typedef struct {
  const void* table;            /* [sum primes, row_dim] in table_dtype */
  const uint16_t* scales;       /* fp16 [sum primes] for I8 tables, else NULL */
  const void* w_kv;             /* act_dtype [(M+1)*d, d_mem], d_mem = R*row_dim:
                                   rows [0,d) = W_V, rows [(1+m)d, (2+m)d) = W_K^(m) */
  const float* g_h;             /* [M, d] RMSNorm weight on h, per branch */
  const float* g_k;             /* [M, d] RMSNorm weight on k, per branch */
  const float* g_c;             /* [d]    RMSNorm weight on v~ before the conv (shared) */
  const float* conv;            /* [d, conv_w] depthwise taps (shared by branches) */
  /* FP8 projection (BF16 layers, d_mem a multiple of 128), or both NULL.  With
   * them, Step 5 runs on e4m3 operands: W_kv as quantised by
   * engram_quantize_fp8 (one scale per output row), e quantised per token by
   * the call itself (engram_forward: by its gather, where engram_stage_a_e4m3
   * applies); w_kv is then not read and may be NULL. */
  const uint8_t* w_kv_fp8;      /* e4m3 [(M+1)*d, d_mem] */
  const float* w_kv_scale;      /* [(M+1)*d] */
} engram_weights_t;

/* Streaming state of B sequences (decode, chunked prefill).  Owned by the
 * caller, zero-initialised for fresh sequences, updated in place by
 * engram_forward after the chunk.  L = (conv_w - 1) * conv_dilation. */
typedef struct {
  int32_t* prev_ids;            /* [B, N-1] projected ids before the chunk, oldest first (0 = pad) */
  float* u_ring;                /* [B, L, M, d] RMSNorm(v~) (before its weight g_c) of the
                                   last L positions; position p lives in slot p mod L */
  int32_t* pos;                 /* [B] tokens already processed per sequence */
} engram_state_t;

/* Human-readable name of a status code (static string). */
const char* engram_status_string(engram_status_t s);

/* Validate `cfg`, copy its primes/multipliers, precompute per-table reduction
 * constants and row offsets, and allocate the plan's device block on the
 * current device.  `max_tokens` bounds B*T of later calls (> 0). */
engram_status_t engram_plan_create(const engram_config_t* cfg, int64_t max_tokens, engram_plan_t** out);

/* Free the plan (after all its work has finished).  NULL is accepted. */
engram_status_t engram_plan_destroy(engram_plan_t* plan);

/* Bytes of device workspace engram_forward needs for `ntok` = B*T tokens. */
engram_status_t engram_plan_workspace_bytes(const engram_plan_t* plan, int64_t ntok, size_t* bytes);

/* Steps 1-3.  ids: int32 [B, T] raw token ids in [0, V); proj: int32 [V]
 * canonical ids P; prev_ids: int32 [B, N-1] projected ids that precede
 * position 0 of each sequence, oldest first, or NULL for fresh sequences (pad 0).
 * idx_out: int32 [B*T, R], head (n,k) in column (n-2)*K + k, value in [0, p_{n,k}).
 * Raw ids outside [0, V) are an argument error the kernel cannot see; they are
 * clamped to 0 and flagged as ENGRAM_ERR_INDEX_RANGE. */
engram_status_t engram_hash(const engram_plan_t* plan, const int32_t* ids, int B, int T,
                            const int32_t* proj, int V, const int32_t* prev_ids,
                            int32_t* idx_out, engram_stream_t stream);

/* Step 4.  idx: int32 [ntok, R] from engram_hash.  e_out: [ntok, d_mem] in
 * act_dtype, segment (n,k) at columns [r*row_dim, (r+1)*row_dim), r=(n-2)K+k.
 * Copies rows (F32 -> F32, BF16 -> BF16), or dequantises I8 rows as
 * bf16(q * scale) with one rounding (the product is exact in binary32).
 * An index >= p_r writes a zero row and flags ENGRAM_ERR_INDEX_RANGE.
 * Host tables must be cudaHostAlloc'd or cudaHostRegister'd: otherwise
 * ENGRAM_ERR_NOT_MAPPED.  The first read of a newly pinned host table pays for
 * the GPU's first translation of its pages (measured: 50-70 ms for a 2.6 GB
 * int8 table); later reads run at the host link's rate whatever the tokens,
 * so a server warms a table with one call before it takes traffic. */
engram_status_t engram_gather(const engram_plan_t* plan, const int32_t* idx, int64_t ntok,
                              const void* table, const uint16_t* scales, void* e_out,
                              engram_stream_t stream);

/* Steps 1-4 in one kernel (Stage A of "DeepSeek Engram 系列导读", section
 * "Engram 工作原理"): the hash of each row is computed inside the gather as the
 * row is read, so the indices never reach memory.  ids/proj/V/prev_ids as in
 * engram_hash; table/scales as in engram_gather; e_out: [B*T, d_mem] act_dtype
 * exactly as engram_gather writes it (16-byte aligned).  Stage A depends on
 * the tokens only, so a caller can run it for a later layer on another stream
 * while earlier layers compute (prefetch), then call engram_stage_b.  For a
 * continued sequence prev_ids must already hold the ids before this chunk
 * (the state as the previous chunk's Stage B left it).  Errors as in
 * engram_hash and engram_gather. */
engram_status_t engram_stage_a(const engram_plan_t* plan, const int32_t* ids, int B, int T,
                               const int32_t* proj, int V, const int32_t* prev_ids,
                               const void* table, const uint16_t* scales, void* e_out,
                               engram_stream_t stream);

/* Stage A of several layers in one launch: engram_stage_a for layer l =
 * 0..n_layers-1 with plans[l], tables[l], scales[l] (or scales == NULL for
 * tables without scales), prev_ids[l] (or prev_ids == NULL: fresh sequences in
 * every layer) and e_out[l], all of one shape: the plans share N, K, row_dim,
 * table_dtype, act_dtype and the device, and the tables are either all in
 * device memory or all in pinned host memory.  ids, proj and V are common to
 * the layers (the token stream and P).  Indices depend on the tokens only
 * ("DeepSeek Engram 系列导读", section "Engram 工作原理", Stage A), so every
 * layer's lookups can be issued together: one grid (grid.y = layer) in place
 * of n_layers launches, which lets a step start its first Stage B sooner than
 * a chain of per-layer gathers that occupy the SMs in turn.  Writes exactly
 * what n_layers engram_stage_a calls write.  1 <= n_layers <= 8; plans that
 * differ in shape, or n_layers out of range: ENGRAM_ERR_INVALID_ARG.  Errors
 * found by the kernel go to each layer's own plan. */
engram_status_t engram_stage_a_layers(int n_layers, const engram_plan_t* const* plans,
                                      const int32_t* ids, int B, int T, const int32_t* proj, int V,
                                      const int32_t* const* prev_ids, const void* const* tables,
                                      const uint16_t* const* scales, void* const* e_out,
                                      engram_stream_t stream);

/* Step 5 alone (inspection / reuse of k and v).  e: [ntok, d_mem] act_dtype;
 * w_kv as in engram_weights_t; kv_out: [ntok, (M+1)*d] act_dtype =
 * e . w_kv^T (fp32 accumulation, one rounding to act_dtype), columns [0,d) = v,
 * [(1+m)d, (2+m)d) = k^(m).  BF16 runs on the tcgen05 tensor cores. */
engram_status_t engram_kv_projection(const engram_plan_t* plan, const void* e, int64_t ntok,
                                     const void* w_kv, void* kv_out, engram_stream_t stream);

/* Steps 5-8 from gathered rows (Stage B): for a caller that ran Stage A
 * (engram_stage_a, or engram_hash + engram_gather) ahead of time, e.g. on a side stream while
 * earlier layers computed -- the indices depend on the tokens only.
 * e: [B*T, d_mem] act_dtype as written by engram_gather; w: table/scales are
 * not read (may be NULL); H: [B, T, M, d] act_dtype, updated in place;
 * state: NULL or as in engram_forward, which then also needs ids/proj/V (the
 * chunk's raw ids, for the rolling n-gram state); with state == NULL, ids
 * and proj may be NULL.  workspace: device, >= engram_plan_workspace_bytes(
 * plan, B*T), 256-B aligned.  BF16 layers run the K/V projection on the
 * tcgen05 tensor cores with a fused epilogue that keeps v in fp32 and turns
 * the k tiles into gate partial sums (k itself is never stored). */
engram_status_t engram_stage_b(const engram_plan_t* plan, const int32_t* ids, int B, int T,
                               const int32_t* proj, int V, const void* e,
                               const engram_weights_t* w, void* H, engram_state_t* state,
                               void* workspace, size_t workspace_bytes, engram_stream_t stream);

/* Stage A for the FP8 projection: Steps 1-4 writing, instead of e, its e4m3
 * codes and per-token scales -- exactly what engram_quantize_fp8 would make of
 * the rows engram_stage_a writes (same rule, same bytes; see there) -- from
 * the row each warp holds in registers, so e never reaches memory and no
 * quantisation launch follows.  For BF16 tables and activations with at most
 * 32 rows and 128 16-byte chunks per token (R * row_dim * 2 <= 2048 bytes),
 * else ENGRAM_ERR_UNSUPPORTED.  e8_out: device uint8 [B*T, d_mem]; e_scale_out:
 * device float [B*T]; both 16-byte aligned.  Other arguments, errors and the
 * several-layer form as engram_stage_a and engram_stage_a_layers (there:
 * e8_out[l], e_scale_out[l] per layer). */
engram_status_t engram_stage_a_e4m3(const engram_plan_t* plan, const int32_t* ids, int B, int T,
                                    const int32_t* proj, int V, const int32_t* prev_ids, const void* table,
                                    uint8_t* e8_out, float* e_scale_out, engram_stream_t stream);
engram_status_t engram_stage_a_layers_e4m3(int n_layers, const engram_plan_t* const* plans,
                                           const int32_t* ids, int B, int T, const int32_t* proj, int V,
                                           const int32_t* const* prev_ids, const void* const* tables,
                                           uint8_t* const* e8_out, float* const* e_scale_out,
                                           engram_stream_t stream);

/* Stage B from the codes of engram_stage_a_e4m3: engram_stage_b with e given
 * as e4m3 codes e8 [B*T, d_mem] and scales e_scale [B*T] (device, 16-byte
 * aligned) instead of bf16 rows; the weights must carry the FP8 projection
 * (w_kv_fp8, w_kv_scale), else ENGRAM_ERR_INVALID_ARG.  The same bits as
 * engram_stage_b on the rows the codes were made from. */
engram_status_t engram_stage_b_e4m3(const engram_plan_t* plan, const int32_t* ids, int B, int T,
                                    const int32_t* proj, int V, const uint8_t* e8, const float* e_scale,
                                    const engram_weights_t* w, void* H, engram_state_t* state,
                                    void* workspace, size_t workspace_bytes, engram_stream_t stream);

/* Steps 1-8: the whole layer for B sequences of T new tokens each.
 * ids/proj/V as in engram_hash; w as in engram_weights_t; H: [B, T, M, d]
 * act_dtype, updated in place; state: NULL or engram_state_t (prev_ids is then
 * used instead of the pad, and u_ring/pos supply the convolution's history).
 * workspace: device, >= engram_plan_workspace_bytes(plan, B*T), 256-B aligned.
 * Capturable in a CUDA graph (no allocation, no synchronisation). */
engram_status_t engram_forward(const engram_plan_t* plan, const int32_t* ids, int B, int T,
                               const int32_t* proj, int V, const engram_weights_t* w,
                               void* H, engram_state_t* state,
                               void* workspace, size_t workspace_bytes, engram_stream_t stream);

/* engram_forward without a workspace argument.  No page describes this: it
 * exists for callers that cannot allocate device memory -- a host framework
 * that owns the device allocator and exposes none of it, a plugin host that
 * accepts only plain calls, a latency-critical path where cudaMalloc (which
 * may synchronise the device) is not allowed.  The scratch lives in a
 * file-scope __device__ array of 32 MiB inside the library image: every GPU
 * that loads the library holds it until the process exits, and this call
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library call).
 * Limit: engram_plan_workspace_bytes(plan, B*T) must not exceed 32 MiB (about
 * 4300 tokens of a d = 1024, d_mem = 1024 layer); larger calls return
 * ENGRAM_ERR_WORKSPACE before any launch.  The current device must be the
 * plan's.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.  The cached address belongs to the device's context of that
 * first call: after cudaDeviceReset (or anything else that destroys and
 * re-creates the primary context) this entry point must not be called again
 * in the same process.  All calls in the process share the one array and it keeps
 * the last call's contents (nothing in it needs to start at zero: the forward
 * writes every scratch byte before reading it), so calls that overlap on the
 * GPU -- on different streams, or from different threads -- race; serialise
 * them.  Other arguments and behaviour as in engram_forward. */
engram_status_t engram_forward_static_scratch(const engram_plan_t* plan, const int32_t* ids, int B, int T,
                                              const int32_t* proj, int V, const engram_weights_t* w,
                                              void* H, engram_state_t* state, engram_stream_t stream);

/* HBM hot-row cache in front of a table held in host memory (the UVA path).
 * The pages keep Engram tables in host DRAM and read rows over the host link
 * ("Engram 嵌入扩展：面向高效 DRAM/SSD 卸载的协同设计", section "AgentX Engram
 * DRAM卸载提升性能"), and keep Zipf-hot rows in device memory (the Ascend
 * RecSDK Engram blog).  The cache holds up to `capacity` rows of `plan`'s
 * table in HBM; which rows is decided by counting (LFU): engram_cache_observe
 * counts the rows a batch will read, engram_cache_build admits the most-counted
 * rows.  engram_stage_a_cached then reads cached rows from HBM and the rest
 * from the host table; its output equals engram_stage_a's bit for bit.
 * Device memory: 8 bytes per table row (counts and slot map) plus capacity
 * rows (plus the dedup region, below).  A cache belongs to one plan and one
 * table; calls on it are stream-ordered (never in flight on two streams at
 * once); engram_cache_build synchronises `stream`. */
typedef struct engram_cache engram_cache_t;

/* table: the plan's table in pinned or registered host memory (or on the
 * device); capacity: rows, 0 <= capacity <= total rows (0: no hot rows, for
 * the dedup alone).  Starts empty, counts 0, no dedup. */
engram_status_t engram_cache_create(const engram_plan_t* plan, int64_t capacity, const void* table,
                                    engram_cache_t** out);
engram_status_t engram_cache_destroy(engram_cache_t* cache);

/* Add one count to every table row the tokens read (ids/proj/V/prev_ids as
 * in engram_hash). */
engram_status_t engram_cache_observe(engram_cache_t* cache, const int32_t* ids, int B, int T,
                                     const int32_t* proj, int V, const int32_t* prev_ids,
                                     engram_stream_t stream);

/* Re-admit: the rows with the highest counts (all rows above a count
 * threshold, then rows one below it while slots remain) are copied into the
 * cache; every other row is read from the host table.  decay != 0 halves all
 * counts afterwards (aging).  cached_rows (optional): rows now cached. */
engram_status_t engram_cache_build(engram_cache_t* cache, int decay, engram_stream_t stream,
                                   int64_t* cached_rows);

/* Per-batch row dedup.  Under the Zipf-skewed n-gram statistics of text many
 * lookups of one batch read the same rows (about a quarter of them on the
 * int8 host-table workload); "Engram 嵌入扩展：面向高效 DRAM/SSD 卸载的协同设计"
 * names the host link as the cost.  With batch_rows > 0, every later
 * engram_stage_a_cached whose batch has at most batch_rows lookups (B*T*R)
 * first copies each distinct table row of the batch that is not cached over
 * the host link once, into a per-batch HBM region with a row per lookup
 * (after the cached rows, in the same slot map), serves every lookup of it
 * from HBM, and frees the slots again.  A batch of B >= 2 sequences runs in
 * up to four pieces of whole sequences so that the host-link copies of one
 * piece overlap the claims of the next and the HBM gather of the one before:
 * claims and the final release on the caller's stream, copies and gathers on
 * two streams the cache owns (made here), which the caller's stream waits for
 * before the call's work on it ends; stream-ordered and capturable.  A row
 * claimed by an earlier piece is not fetched again.  Larger batches run
 * without the dedup.  The output is
 * unchanged, bit for bit.  batch_rows = 0 turns it off.  Synchronises the
 * device and reallocates the cache's row buffer (cached rows are kept);
 * capacity + batch_rows <= INT32_MAX.  Device memory: batch_rows x (row
 * bytes + 4). */
engram_status_t engram_cache_set_dedup(engram_cache_t* cache, int64_t batch_rows);

/* engram_stage_a with the cache's table, cached rows read from HBM (and, with
 * the dedup on, every row of the batch fetched once).  scales: as in
 * engram_gather (fp16 per row, HBM or mapped host memory; I8 only). */
engram_status_t engram_stage_a_cached(const engram_cache_t* cache, const int32_t* ids, int B, int T,
                                      const int32_t* proj, int V, const int32_t* prev_ids,
                                      const uint16_t* scales, void* e_out, engram_stream_t stream);

/* Synchronise `stream` and read the counters of engram_stage_a_cached since
 * the last reset: table rows looked up, lookups served from HBM (cached rows
 * and the dedup's batch region), and rows read over the host link (lookups
 * read from the host table plus the dedup's one fetch per distinct row);
 * reset != 0 zeroes them.  cached_rows: rows the last build cached.  Any
 * output pointer may be NULL. */
engram_status_t engram_cache_stats(const engram_cache_t* cache, engram_stream_t stream, int reset,
                                   uint64_t* rows_looked_up, uint64_t* rows_from_hbm, uint64_t* rows_over_link,
                                   int64_t* cached_rows);

/* Per-row e4m3 quantisation of a bf16 array x [rows, cols] (device, 16-byte
 * aligned, cols a multiple of 16), for the FP8 projection that "DeepSeek
 * Engram 系列导读" (section "多分支 backbone 上的变体") suggests for the fused
 * [W_V; W_K^(1..M)] GEMM; the page fixes no scaling.  For every row i:
 *   scale[i] = amax_i / 448,  q[i, j] = e4m3(x[i, j] * (448 / amax_i))
 * (448: the largest finite e4m3 value; both quotients IEEE binary32; the
 * conversion rounds to nearest even and saturates to +-448); an all-zero row
 * gets scale 1 and zero codes.  q: device uint8 [rows, cols]; scale: device
 * float [rows].  Used once per layer for W_kv (rows = (M+1)*d, cols = d_mem);
 * the forward applies the same rule to each token's row of e. */
engram_status_t engram_quantize_fp8(const engram_plan_t* plan, const void* x, int64_t rows, int cols, uint8_t* q,
                                    float* scale, engram_stream_t stream);

/* Stage B of BF16 layers with one branch, conv_w = 4 and d = 1024 (eight
 * 128-column slices per projection quantity), for chunks of T > 1 positions,
 * can run as ONE cooperative launch (enable = 1): the K/V projection and the
 * conv share the GPU, each conv tile starting as soon as the 128-row blocks
 * it reads are projected (after a one-block kernel that zeroes the launch's
 * counters in the workspace).  The default (enable = 0) is the two-launch
 * form: projection, then the conv with the gate finalisation, which measures
 * faster on GB300 at 4096 tokens.  Both give the same bits.  Other layer
 * shapes always use separate launches.  enable: 0 or 1; applies to calls
 * made after it. */
engram_status_t engram_plan_set_fused_stage_b(engram_plan_t* plan, int enable);

/* Chunks of one position per sequence (decode, T = 1) of BF16 layers with
 * (N-1)*K <= 32 table rows per token, conv_w = 4 and e4m3-free weights can run
 * as ONE cooperative launch (enable = 1): engram_forward's gather (Steps
 * 1-4), the K/V projection on the tensor cores with its gate epilogue (Steps
 * 5-6) and the gate, conv, residual and state update of every sequence
 * (Steps 6-8), phases linked by counters in the workspace; engram_stage_b
 * runs the same launch without the gather.  The indices of Stage A depend on
 * the tokens only ("DeepSeek Engram 系列导读", section "Engram 工作原理"), so
 * nothing between them needs the host.  The default (enable = 0) is separate
 * launches (gather, projection, decode tail), which measure faster on GB300
 * for 256 sequences: they overlap the next layer's gather and each other's
 * launch, where the one launch runs its phases back to back.  Both give the
 * same bits.  A device that cannot hold one block per SM of the launch falls
 * back to separate launches.  enable: 0 or 1; applies to calls made after it. */
engram_status_t engram_plan_set_fused_decode(engram_plan_t* plan, int enable);

/* At most n_sms SMs for Stage B's persistent kernels (the K/V projection,
 * the conv, their tile shapes chosen for that many SMs) in its two-launch
 * form, the default; the one-launch cooperative form (set_fused_stage_b)
 * keeps one block per SM.  0 (the default): all of them.  For running Stage B beside other work that holds the remaining
 * SMs: chiefly the Stage A of the next piece of a batch over tables in pinned
 * host memory, whose gather occupies engram_plan_host_gather_sms(plan) whole
 * SMs while the host link sets its pace ("DeepSeek Engram 系列导读", section
 * "Engram 工作原理": the lookup depends on the tokens only and can run ahead).
 * The results do not depend on it.  n_sms >= 0; applies to calls made after it. */
engram_status_t engram_plan_set_sm_limit(engram_plan_t* plan, int n_sms);

/* The number of SMs a Stage A (engram_stage_a, engram_stage_a_layers,
 * engram_forward's gather) over tables in pinned host memory occupies: its
 * gather runs as one 1024-thread block per SM on that many SMs, leaving the
 * others to concurrent work.  0 for a null plan. */
int engram_plan_host_gather_sms(const engram_plan_t* plan);

/* The number of SMs (one 1024-thread block each) a Stage A over tables in
 * pinned host memory runs on: n_sms > 0 (capped at the device's SM count),
 * or 0 for the default, a quarter of the SMs.  For an SM split, set it to
 * the lookup group's SM count.  The results do not depend on it; n_sms >= 0;
 * applies to calls made after it. */
engram_status_t engram_plan_set_host_gather_sms(engram_plan_t* plan, int n_sms);

/* An SM split: the device's SMs in two disjoint sets, each with one
 * non-blocking stream whose kernels run on that set's SMs only (green
 * contexts of the driver).  For a batch in pieces over tables in pinned host
 * memory: each piece's Stage A on group 0's stream, sized to the host gather
 * (engram_plan_host_gather_sms), and the previous piece's Stage B on group 1's
 * stream with engram_plan_set_sm_limit(plan, engram_sm_split_sms(split, 1)),
 * so neither stage's blocks wait for SMs the other holds ("DeepSeek Engram
 * 系列导读", section "Engram 工作原理": the lookup depends on the tokens only
 * and can run ahead of the layers that use it).
 *
 * engram_sm_split_create: device ordinal; n_sms > 0, below the device's SM
 * count, is group 0's minimum (the driver rounds it up to its partition
 * granularity: 8 SMs on this architecture); group 1 holds the rest.  The
 * streams use the device's primary context, so memory allocated there (by
 * the CUDA runtime, or PyTorch) is used as is, and events order them against
 * any other stream.  A driver without green contexts, or a split the driver
 * refuses: ENGRAM_ERR_UNSUPPORTED.  The split owns both streams; destroy it
 * after the work on them has completed, and after any CUDA graph captured
 * from them (engram_forward_split inside a capture) has been destroyed.
 * engram_sm_split_sms: the SMs of group 0 or 1 (0 for a null split or
 * another group).  engram_sm_split_stream: that group's stream (a
 * cudaStream_t; null for a null split or another group). */
typedef struct engram_sm_split engram_sm_split_t;
engram_status_t engram_sm_split_create(int device, int n_sms, engram_sm_split_t** out);
int engram_sm_split_sms(const engram_sm_split_t* split, int group);
void* engram_sm_split_stream(const engram_sm_split_t* split, int group);
engram_status_t engram_sm_split_destroy(engram_sm_split_t* split);

/* engram_forward (Steps 1-8) of B sequences in n_pieces pieces of whole
 * sequences (with n_pieces >= 3 the first and the last piece hold half as
 * many sequences as the others, so that the pipeline fills and drains fast;
 * with 1 or 2, equal pieces) on an SM
 * split: every piece's Stage A on group 0's stream, each piece's Stage B on
 * group 1's stream as soon as its rows are in, so the lookup of piece i+1
 * runs beside the projection and conv of piece i ("DeepSeek Engram 系列导读",
 * section "Engram 工作原理": the lookup depends on the tokens only).  Made for
 * tables in pinned host memory, whose lookup is paced by the host link; any
 * table works.  Same arguments, layouts and results (bit for bit) as
 * engram_forward; the state, when given, is updated per piece.
 * The work is ordered after what `stream` holds before the call, and `stream`
 * waits for all of it (graph capture of `stream` captures both groups).
 * During the call the plan's SM limit and host-gather SMs are the split's
 * groups (1 and 0), and the call uses the two-launch Stage B on one SM per
 * CTA and records no tracing events; the plan's settings are restored before
 * it returns.  Not for concurrent calls on one split.  1 <= n_pieces <= B and
 * n_pieces <= 64, else ENGRAM_ERR_INVALID_ARG; other errors as engram_forward.
 * cache: NULL, or an HBM hot-row cache of this plan's table (engram_cache_*),
 * through which every piece's Stage A then reads (engram_stage_a_cached, the
 * same bits); a cache of another plan: ENGRAM_ERR_INVALID_ARG; a cache with
 * the per-batch dedup on (it runs its own pipeline): ENGRAM_ERR_UNSUPPORTED. */
engram_status_t engram_forward_split(engram_plan_t* plan, const engram_sm_split_t* split, int n_pieces,
                                     const engram_cache_t* cache, const int32_t* ids, int B, int T,
                                     const int32_t* proj, int V, const engram_weights_t* w, void* H,
                                     engram_state_t* state, void* workspace, size_t workspace_bytes,
                                     engram_stream_t stream);

/* The K/V projection (Step 5, bf16 layers) in 256 x 256 output tiles on CTA
 * pairs (enable = 1): two SMs of a thread-block cluster share one
 * tcgen05.mma.cta_group::2 tile, each staging its 128 rows of e and half of
 * the tile's rows of W_kv, so each SM loads a third less operand data per
 * FLOP.  Applies where the projection would use 256-column tiles on one SM
 * (enough tokens to give every SM such a tile: about 2400 or more at
 * d = 1024) and d is a multiple of 256; the results are the same bits.  The
 * default (enable = 0) keeps one SM per 128 x 256 tile, which measures faster
 * on GB300 at 4096 tokens.  enable: 0 or 1; applies to calls made after it. */
engram_status_t engram_plan_set_cta_pairs(engram_plan_t* plan, int enable);

/* Tracing.  With timing on, engram_forward / engram_stage_b record one of
 * the plan's CUDA events on `stream` before the first kernel and after every
 * kernel they launch.  engram_forward on BF16 layers: hash + gather (Steps
 * 1-4 in one kernel), K/V projection with the gate reductions, gate
 * (finalize), conv + residual; on F32 layers: hash + gather, K/V projection,
 * gate, conv + residual; then the state update when a state is given.  Chunks
 * of one position (T = 1, decode) run the gate, conv, residual and state
 * update as one kernel after the K/V projection, or, with the one-launch
 * decode (engram_plan_set_fused_decode, off by default), the whole step is
 * one traced interval.  Where the conv computes the
 * gate itself there is no finalize kernel; where Stage B is one cooperative
 * launch (engram_plan_set_fused_stage_b), its events bracket the counter
 * reset and that launch together.
 * engram_stage_b records the same list without the first kernel.  For use on
 * one stream at a time.  A call captured into a CUDA graph records its events
 * as event-record nodes: after each replay, engram_plan_kernel_times reads
 * that replay's times (until the plan's next call).  enable: 0 or 1. */
engram_status_t engram_plan_set_timing(engram_plan_t* plan, int enable);

/* Wait for the last call's events and write the device time of each kernel it
 * launched, in launch order, in milliseconds: ms_out[0..*count-1]. */
engram_status_t engram_plan_kernel_times(const engram_plan_t* plan, float* ms_out, int max_out, int* count);

/* Synchronise `stream`, then read and clear the plan's device error word.
 * Returns ENGRAM_OK, ENGRAM_ERR_INDEX_RANGE or ENGRAM_ERR_TIMEOUT (the first
 * set, in that order of precedence reversed: TIMEOUT wins).  `flags_out`
 * (optional) receives the raw bits: 1 = index range, 2 = timeout. */
engram_status_t engram_get_error(const engram_plan_t* plan, engram_stream_t stream, uint32_t* flags_out);

#ifdef __cplusplus
}
#endif

#endif /* ENGRAM_GB300_H */
