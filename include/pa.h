/*
 * pa.h -- C ABI of libpa: single-token decode attention over a paged KV
 * cache on one GB300 (sm_103a).
 *
 * What the library computes.  For every sequence b < num_seqs and query head
 * h < num_heads, with G = num_heads / num_kv_heads, kvh = h / G and
 * L = seq_lens[b]:
 *
 *   l_t      = scale * dot(q[b,h,:], K[blk(t), kvh, t % block_size, :]),
 *              blk(t) = block_tables[b * max_blocks_per_seq + t / block_size]
 *   out[b,h] = sum_t exp(l_t - max l) V[blk(t), kvh, t % block_size, :]
 *              / sum_t exp(l_t - max l)                       (t < L)
 *
 * Sources (commit pages of the project "project_6"):
 *   - the paged cache and its block table, and the [blocks, kv_heads,
 *     block_size, head_dim] layout both caches use: commit 4eb83a7e
 *     "qwen3_6_scripts", paragraph "Hardware testing confirmed";
 *   - the V2 split-KV scheme (per-partition QK^T, softmax and weighted V sum
 *     into tmp_output / exp_sums / max_logits, then a cross-partition
 *     log-sum-exp reduction): same page, paragraph "Implementation
 *     (paged_attention_v2_pytorch.py)", and commit 1a4e1005 "paged_attn.py",
 *     paragraph "Architecture follows CCCL's two-pass dispatch";
 *   - the V1 single pass and the 8192-token dispatch threshold: commit
 *     1a4e1005 "paged_attn.py", change 1 "Restore V1/V2 adaptive dispatch",
 *     and commit 4eb83a7e "qwen3_6_scripts", paragraph "forward_decode: V2
 *     enabled via original heuristic";
 *   - the preallocated V2 workspace: commit 1a4e1005 "paged_attn.py",
 *     change 2 "Pre-allocate V2 intermediate tensors".
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer, owned by the caller, valid
 *     for the whole asynchronous execution of the call.  The library never
 *     allocates, frees, synchronises or logs (pa_read_device_status is the
 *     one call that waits on the stream, and it says so).
 *   - All work is enqueued on `stream` and returns before it runs.  The
 *     decode calls make no allocation and no host synchronisation.
 *   - Host-side checks run before anything is enqueued; a failing check
 *     returns its status and enqueues nothing.
 *   - q, k_cache, v_cache and out must be 16-byte aligned; block_tables and
 *     seq_lens 4-byte aligned; the workspace 256-byte aligned.
 *   - The caller promises 0 <= seq_lens[b] <= max_seq_len and valid block ids
 *     for every token t < seq_lens[b].  A violation is caught on the device:
 *     the offending output row is written as NaN, no out-of-range memory is
 *     touched, and (for calls given a workspace) the status word records it.
 *   - A sequence of length 0 gets an all-zero output row.
 *   - The library keeps no per-call state; calls are thread-safe.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,         /* null pointer, bad shape or size          */
  PA_ERR_UNSUPPORTED = 2,         /* valid but not built: dtype, head_dim ... */
  PA_ERR_MISALIGNED = 3,          /* pointer alignment rule broken            */
  PA_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes < pa_workspace_size()    */
  PA_ERR_CUDA = 5,                /* a CUDA launch or copy failed             */
  PA_ERR_DEVICE_TIMEOUT = 6,      /* device status: a bounded wait gave up    */
  PA_ERR_BAD_BLOCK_ID = 7,        /* device status: block id outside the pool */
  PA_ERR_BAD_SEQ_LEN = 8,         /* device status: seq_len outside 0..max    */
  PA_ERR_WORKSPACE_NOT_INIT = 9   /* device status: pa_workspace_init missing */
} pa_status_t;

typedef enum pa_dtype { PA_F32 = 0, PA_BF16 = 1, PA_F16 = 2 } pa_dtype_t;

/* Flags (pa_params_t.flags). */
#define PA_FLAG_PORTABLE 1 /* use the CUDA-core kernels even where the
                              TMA / tensor-core kernels apply              */
#define PA_FLAG_SELFTEST_STALL 2 /* diagnostic: the tensor-core kernels
                              (either cache layout; prefill too) first wait
                              for an event that never happens, with a short
                              (~10 ms) bound, so their bounded-wait path
                              runs: the call's outputs become NaN and the
                              workspace status word (V2) reads
                              PA_ERR_DEVICE_TIMEOUT.  Ignored by the
                              CUDA-core kernels, which have no such waits. */
#define PA_FLAG_SPLIT_X 4 /* the caches are in the layout commit 4eb83a7e
                              "qwen3_6_scripts", paragraph "Hardware testing
                              confirmed", gives for its V1 kernel:
                                k_cache [num_blocks, num_kv_heads,
                                         head_dim / x, block_size, x]
                                v_cache [num_blocks, num_kv_heads,
                                         head_dim, block_size]
                              with x = 16 / element bytes (8 for bf16 / f16,
                              4 for f32).  Read directly, with no conversion
                              copy: for bf16 / f16 caches with block_size 16
                              or 32 and at most 8 query heads per KV head by
                              a tensor-core kernel (warp-level MMA fed by
                              ldmatrix from whole-block bulk copies; V2 in one
                              launch and V1 in clusters as on the standard
                              layout), else by the CUDA-core kernels; every
                              call accepts it. */

typedef struct pa_params {
  int32_t num_seqs;           /* B >= 0                                      */
  int32_t num_heads;          /* Hq >= 1                                     */
  int32_t num_kv_heads;       /* Hkv >= 1, divides Hq                        */
  int32_t head_dim;           /* D: 64, 128 or 256                           */
  int32_t block_size;         /* BS >= 1 tokens per physical block           */
  int32_t num_blocks;         /* NB >= 1: blocks in each cache pool          */
  int32_t max_blocks_per_seq; /* MB: row length of block_tables              */
  int32_t max_seq_len;        /* host-known upper bound of seq_lens, <= MB*BS */
  int32_t partition_size;     /* P: V2 tokens per partition, multiple of BS  */
  int32_t v1_max_seq_len;     /* pa_decode threshold, <= 0 means 8192        */
  pa_dtype_t kv_dtype;        /* element type of q, k_cache and v_cache      */
  pa_dtype_t out_dtype;       /* PA_F32, or the same type as kv_dtype        */
  float scale;                /* logit scale, usually 1/sqrt(head_dim)       */
  int32_t flags;              /* PA_FLAG_* bits, 0 by default                */
} pa_params_t;

/*
 * Tensor layouts (row-major, element type in brackets):
 *   q            [kv_dtype] [num_seqs, num_heads, head_dim]
 *   k_cache      [kv_dtype] [num_blocks, num_kv_heads, block_size, head_dim]
 *   v_cache      [kv_dtype] [num_blocks, num_kv_heads, block_size, head_dim]
 *   block_tables [int32]    [num_seqs, max_blocks_per_seq]
 *   seq_lens     [int32]    [num_seqs]
 *   out          [out_dtype][num_seqs, num_heads, head_dim]
 *
 * Workspace (V2 only), NP = ceil(max_seq_len / partition_size), each region
 * starting on a 256-byte boundary, in this order:
 *   control      1024 bytes (PA_WORKSPACE_CONTROL_BYTES), whatever the
 *                parameters: the int32 status word at offset 0, an
 *                initialisation marker at offset 4, and from offset 256 the
 *                counters of the one-launch V2 step
 *   max_logits   float32 [num_seqs, num_heads, NP]   m_p, natural-log units
 *   exp_sums     float32 [num_seqs, num_heads, NP]   s_p = sum exp(l_t - m_p)
 *   tmp_output   float32 [num_seqs, num_heads, NP, head_dim]
 *                o_p = sum exp(l_t - m_p) V_t / s_p
 * Only partitions p < ceil(seq_lens[b] / P) are written or read; the rest
 * may hold anything.  pa_decode_v2_partitions leaves every partition's
 * partials as defined above.  After pa_decode_v2 a sequence with a single
 * partition has no partials in the workspace.
 * The control block must be initialised once, by pa_workspace_init, before
 * the first V2 call; every V2 call leaves it ready for the next one, with
 * any parameters.
 */
#define PA_WORKSPACE_CONTROL_BYTES ((size_t)1024)

/* Bytes of workspace pa_decode_v2 / pa_decode need for these parameters
 * (0 if the parameters are invalid): the control block plus the partials.
 * Depends only on num_seqs, num_heads, head_dim, max_seq_len and
 * partition_size. */
PA_API size_t pa_workspace_size(const pa_params_t* params);

/*
 * V1: one pass per (sequence, KV head) over the whole sequence, normalised
 * straight into `out`.  No workspace: when there are fewer (sequence, KV
 * head) pairs than SMs, the tensor-core kernels (either cache layout) share
 * each pair across a thread-block cluster of up to 16 CTAs that merge their
 * partial results in distributed shared memory.
 * Source: commit 1a4e1005 "paged_attn.py", change 1 (V1 single-CTA
 * iteration); commit 4eb83a7e "qwen3_6_scripts", paragraph "V1
 * paged_attention (decode <= 8192)".
 */
PA_API pa_status_t pa_decode_v1(const pa_params_t* params, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* block_tables,
                         const int32_t* seq_lens, void* out, cudaStream_t stream);

/*
 * V2: split-KV.  Pass 1 runs per (sequence, KV-head group, partition of
 * partition_size tokens) and writes max_logits, exp_sums and tmp_output into
 * the workspace; pass 2 combines a row's partitions with weights
 * exp(m_p - max_p m_p) * s_p and writes `out`.
 * `workspace` must hold pa_workspace_size(params) bytes, its control block
 * initialised by pa_workspace_init.
 * One launch: when a tensor-core kernel (either cache layout) runs as a
 * persistent grid with at least one CTA per reduce unit (num_seqs * num_heads * head_dim / 32 units:
 * few long sequences, e.g. one 100K-token sequence), pass 2 runs in the same
 * launch.  Each CTA, after its partitions, counts itself finished in the
 * workspace; CTAs that finish once every CTA of the grid has started take
 * reduce units and run them when all are finished (no cooperative launch
 * and no wait on a CTA that has not started; the order of every sum is
 * fixed, so results are bit-identical from run to run).  Other batches and
 * the CUDA-core path use two kernels, pass 2 launched as a programmatic
 * dependent of pass 1 (pa_decode_launches() tells which).  In a workspace
 * that pa_workspace_init never initialised the one-launch step reduces
 * nothing: the status word reads PA_ERR_WORKSPACE_NOT_INIT and the rows of
 * sequences longer than one partition are NaN.
 * The V1 / V2 choice is also made per sequence inside the pass-1 launch: a
 * sequence of 1..partition_size tokens has a single partition, so pass 1
 * writes its normalised result straight into `out` (V1's contract), writes
 * no partials for it, and pass 2 skips its rows; longer sequences are split
 * and reduced.  (pa_decode_v2_partitions below always writes the partials.)
 * Source: commit 4eb83a7e "qwen3_6_scripts", paragraph "Implementation
 * (paged_attention_v2_pytorch.py)", Phase 1 and Phase 2; the per-sequence
 * choice follows the V1 / V2 tiers of commit 1a4e1005 "paged_attn.py",
 * change 1, with the partition size as the per-sequence threshold.
 */
PA_API pa_status_t pa_decode_v2(const pa_params_t* params, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* block_tables,
                         const int32_t* seq_lens, void* workspace, size_t workspace_bytes,
                         void* out, cudaStream_t stream);

/*
 * The two kernels of pa_decode_v2 as separate calls, for callers that want
 * to schedule or time them apart.  pa_decode_v2_partitions enqueues pass 1
 * and writes the workspace's partials for every partition of every
 * sequence (single-partition sequences included); pa_decode_v2_reduce
 * enqueues pass 2 (reads the workspace, writes every row of `out`) and must
 * follow pass 1 on the same stream with the same arguments.  Together they
 * give pa_decode_v2's result; pa_decode_v2 itself launches pass 2 as a
 * programmatic dependent of pass 1 and finishes single-partition sequences
 * in pass 1.
 */
PA_API pa_status_t pa_decode_v2_partitions(const pa_params_t* params, const void* q,
                                           const void* k_cache, const void* v_cache,
                                           const int32_t* block_tables, const int32_t* seq_lens,
                                           void* workspace, size_t workspace_bytes,
                                           cudaStream_t stream);
PA_API pa_status_t pa_decode_v2_reduce(const pa_params_t* params, const int32_t* seq_lens,
                                       const void* workspace, size_t workspace_bytes, void* out,
                                       cudaStream_t stream);

/*
 * Dispatch: V2 when max_seq_len > v1_max_seq_len (8192 by default), else
 * V1.  The workspace is only touched (and only required) when V2 runs.
 * Source: commit 1a4e1005 "paged_attn.py", change 1 (V2 for sequences
 * longer than 8192 tokens), and commit 4eb83a7e "qwen3_6_scripts",
 * paragraph "forward_decode: V2 enabled via original heuristic".
 */
PA_API pa_status_t pa_decode(const pa_params_t* params, const void* q, const void* k_cache,
                      const void* v_cache, const int32_t* block_tables, const int32_t* seq_lens,
                      void* workspace, size_t workspace_bytes, void* out, cudaStream_t stream);

/*
 * pa_decode_v2 for callers that cannot allocate device memory.  The pages
 * have no counterpart of this call: it exists for callers with no way to
 * call cudaMalloc or any allocator where they decode (a plugin of a host
 * runtime that owns every device allocation, a C program linking libpa
 * without torch, a real-time loop that must not stall on or fail an
 * allocation).  The caller still passes its inputs and `out`; the V2
 * workspace is instead a fixed array of PA_STATIC_WORKSPACE_BYTES (16 MiB)
 * that the library keeps in device memory, which every GPU that loads
 * libpa.so holds until the process exits.
 *   - Parameters whose pa_workspace_size() exceeds PA_STATIC_WORKSPACE_BYTES
 *     are rejected with PA_ERR_WORKSPACE_TOO_SMALL before anything is
 *     enqueued (16 MiB covers, e.g., one 24-head, head_dim-256 sequence of
 *     up to about 340K tokens at partition_size 512).
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it for the current context; a new
 *     context on that device (after cudaDeviceReset, or a driver-API context
 *     the caller made current) looks it up again.  Make the first call in a
 *     context before any stream capture.
 *   - All calls on a device share the array, and it keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls that overlap on
 *     the GPU race on it: order them on one stream.
 *   - It makes no allocation of its own and calls no allocating routine.
 *   - Device-detected input errors still show as NaN output rows; the status
 *     word is not reported by this call.
 */
#define PA_STATIC_WORKSPACE_BYTES ((size_t)16 << 20)
PA_API pa_status_t pa_decode_v2_static(const pa_params_t* params, const void* q,
                                       const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* seq_lens,
                                       void* out, cudaStream_t stream);

/*
 * The decode step from host memory.  The per-step inputs -- q, block_tables
 * and seq_lens -- are read from HOST buffers and `out` is written to a HOST
 * buffer; k_cache, v_cache and the workspace are device memory that stays
 * resident between steps.  The call enqueues on `stream` the three
 * host-to-device copies into `staging`, the pa_decode step (V1 or V2 by the
 * same threshold) and the device-to-host copy of the result, then WAITS for
 * the stream: `out_host` is complete when it returns PA_OK.  It is therefore
 * not for use inside stream capture.
 *   staging    caller-owned device memory of pa_host_staging_size(params)
 *              bytes, 256-byte aligned; it holds the copied inputs and the
 *              result (q | block_tables | seq_lens | out, each on a 256-byte
 *              boundary) and may hold anything between calls.
 *   host buffers: page-locked memory (cudaHostAlloc / pinned tensors) makes
 *              the copies asynchronous DMA; pageable memory also works, with
 *              the copies staged by the CUDA driver.  When block_tables_host
 *              and seq_lens_host sit at the staging offsets from q_host (a
 *              host mirror of the staging layout, pa_host_staging_offsets),
 *              the three inputs move in one copy.
 * Errors: the checks of pa_decode, a null or misaligned staging buffer
 * (PA_ERR_INVALID_ARG / PA_ERR_MISALIGNED), staging_bytes too small
 * (PA_ERR_WORKSPACE_TOO_SMALL), misaligned caches (PA_ERR_MISALIGNED), all
 * before anything is enqueued; a failed copy, launch or wait gives
 * PA_ERR_CUDA.  An error found after the copies were queued is returned only
 * once the stream has finished, so no copy still uses the host buffers when
 * the call returns.
 */
PA_API size_t pa_host_staging_size(const pa_params_t* params);
/* Byte offsets within the staging layout: offsets[0] = q (0), [1] =
 * block_tables, [2] = seq_lens, [3] = out, [4] = total (= staging size).
 * PA_ERR_INVALID_ARG for invalid parameters or a null array.  Pure host
 * function. */
PA_API pa_status_t pa_host_staging_offsets(const pa_params_t* params, size_t offsets[5]);
PA_API pa_status_t pa_decode_host(const pa_params_t* params, const void* q_host,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables_host, const int32_t* seq_lens_host,
                                  void* workspace, size_t workspace_bytes, void* staging,
                                  size_t staging_bytes, void* out_host, cudaStream_t stream);

/* Which path pa_decode takes for these parameters: 1 (V1), 2 (V2) or 0 if
 * the parameters are invalid.  Pure host function. */
PA_API int pa_decode_path(const pa_params_t* params);

/* Kernel launches one pa_decode call makes for these parameters on the
 * current device: 1 (V1, or V2 in one launch), 2 (V2 as pass 1 and a
 * dependent pass 2), 0 for invalid parameters or an empty batch.  Host
 * function; it queries the current device like pa_decode_kernel. */
PA_API int pa_decode_launches(const pa_params_t* params);

/* Which kernels the decode calls use for these parameters on the current
 * device: 2 = tensor-core kernels (bf16 / f16 caches, at most 8 query heads
 * per KV head; standard layout: TMA + tcgen05, head_dim 128 or 256 with
 * block_size 16 or 32, or head_dim 128 with block_size 64; PA_FLAG_SPLIT_X:
 * bulk copies + warp-level MMA, head_dim 64, 128 or 256 with block_size 16
 * or 32), 1 = CUDA-core kernels (every other valid case, or
 * PA_FLAG_PORTABLE), 0 = invalid parameters.  Host function; it queries the
 * current device's compute capability. */
PA_API int pa_decode_kernel(const pa_params_t* params);

/* Static description of a status code (never NULL). */
PA_API const char* pa_status_string(pa_status_t status);

/* Initialise the workspace's control block (enqueued on `stream`): zero the
 * status word and the arrival counters and write the initialisation marker
 * (the first min(workspace_bytes, PA_WORKSPACE_CONTROL_BYTES) bytes).  Call
 * once after allocating a workspace, before its first V2 call; device
 * errors then accumulate in the status word until read. */
PA_API pa_status_t pa_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Diagnostic: copy the status word to *status (PA_OK or the last device
 * error recorded), WAITING for `stream` to finish, then zero it when
 * `clear` is non-zero.  Not for use inside stream capture. */
PA_API pa_status_t pa_read_device_status(const void* workspace, int32_t* status, int clear,
                                  cudaStream_t stream);

/*
 * Paged prefix prefill (chunked prefill): sequence b attends a chunk of n_b
 * new tokens to its C_b cached tokens and, causally, to the chunk itself.
 * Source: commit 1a4e1005 "paged_attn.py", opening paragraph (prefill is
 * online softmax over key tiles); commit 4eb83a7e "qwen3_6_scripts",
 * paragraphs on the prefix attention's pre-allocated m_blk / m_new / corr
 * buffers (a tile loop over the cached context, then one over the chunk),
 * "Complete rewrite of qwen3_6_scripts/paged_attn.py" item 1 (the context
 * comes from the paged cache) and "Prefill (flash_attn_func)" (causal).
 *
 *   q    [kv_dtype] [T, num_heads, head_dim]    the chunk's queries
 *   k, v [kv_dtype] [T, num_kv_heads, head_dim] the chunk's keys / values
 *   k_cache, v_cache, block_tables: as for decode; only each sequence's
 *        first ctx_lens[b] tokens are read
 *   query_start [int32] [num_seqs + 1]: sequence b owns rows
 *        query_start[b] .. query_start[b+1] - 1 of q / k / v / out
 *   ctx_lens    [int32] [num_seqs]: C_b cached tokens
 *   out  [out_dtype] [T, num_heads, head_dim]
 * Row i of sequence b (0-based in its chunk), query head h, reads KV head
 * h / (num_heads / num_kv_heads) and gives
 *   softmax(scale * q . k_j) over j = the C_b context tokens and the chunk's
 *   tokens 0..i, applied to the matching values.
 * Tensor-core kernel only: bf16 or f16, head_dim 128 (block_size 16, 32, 64)
 * or 256 (block_size 16, 32); anything else is PA_ERR_UNSUPPORTED.
 * Device-side checks: a sequence whose chunk does not satisfy
 * 0 <= n_b <= max_query_len and query_start[b+1] <= total_tokens is skipped
 * (its rows are not written); a context length outside
 * 0..min(max_ctx_len, max_blocks_per_seq * block_size), or a context block
 * id outside the pool, makes the affected rows NaN.  Asynchronous on
 * `stream`; no workspace.
 */
typedef struct pa_prefill_params {
  int32_t num_seqs;           /* B >= 0                                      */
  int32_t num_heads;          /* Hq >= 1                                     */
  int32_t num_kv_heads;       /* Hkv >= 1, divides Hq                        */
  int32_t head_dim;           /* D: 128 or 256                               */
  int32_t block_size;         /* tokens per cache block                      */
  int32_t num_blocks;         /* blocks in each cache pool                   */
  int32_t max_blocks_per_seq; /* row length of block_tables                  */
  int32_t total_tokens;       /* T: rows of q / k / v / out                  */
  int32_t max_query_len;      /* host-known bound of every n_b               */
  int32_t max_ctx_len;        /* host-known bound of every C_b               */
  pa_dtype_t kv_dtype;        /* PA_BF16 or PA_F16: q, k, v and the caches   */
  pa_dtype_t out_dtype;       /* PA_F32 or kv_dtype                          */
  float scale;                /* logit scale, usually 1/sqrt(head_dim)       */
  int32_t flags;              /* 0                                           */
} pa_prefill_params_t;

PA_API pa_status_t pa_prefill(const pa_prefill_params_t* params, const void* q, const void* k,
                              const void* v, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, const int32_t* query_start,
                              const int32_t* ctx_lens, void* out, cudaStream_t stream);

/* ABI version: major * 10000 + minor * 100 + patch. */
PA_API int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
