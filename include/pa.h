/*
 * pa.h -- C ABI of the GB300 paged KV-cache library (libpa_gb300.so).
 *
 * The paged-attention operations of the pages, plus the plumbing around them:
 *
 *   pa_reshape_and_cache   write each new token's K/V rows into the physical
 *                          cache block its slot_mapping entry names
 *                          ("Inside vLLM CUDA Kernels: KV-Cache Writes and Paged
 *                          Attention", Part 2; "How vLLM CUDA Kernels Write and
 *                          Read the Paged KV Cache", "Writing K and V into the cache")
 *   pa_decode / _ex        single-query paged decode attention with GQA, online
 *                          softmax and split-KV partitions merged by a
 *                          log-sum-exp reduce ("Inside vLLM CUDA Kernels", Part 3;
 *                          "vLLM 源码完全拆解（七）", 参数与内存布局 through V1 与 V2)
 *
 *   pa_decode_step         the cache write and the decode of one step in one call
 *   pa_attention_varlen    several new query tokens per sequence, causal
 *                          ("Inside vLLM CUDA Kernels", Part 3, the varlen read path);
 *                          long chunks run on a tcgen05 query-tile kernel
 *   pa_*_opt               the same calls with per-head FP8 scales and ALiBi
 *   pa_bm_*, pa_copy_blocks  host block manager and device block copy ("tiny-vllm,
 *                          Part 6"; "PagedAttention kernel: paged KV cache & block
 *                          tables")
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensors are passed as pa_tensor descriptors: a data pointer, an element type,
 *    a rank and per-dimension extents and strides (strides in ELEMENTS).  All data
 *    pointers are DEVICE pointers on the current CUDA device unless a comment says
 *    otherwise.  The caller owns all memory; the library keeps no pointer after a
 *    call returns (pa_decode's internal workspace excepted, see below).
 *  - The block size (tokens per KV-cache block) is fixed at PA_BLOCK_SIZE = 16.
 *  - Cache layout ("HND"): k_cache and v_cache are each [num_blocks, num_kv_heads,
 *    16, head_size], innermost dimension contiguous.  One (block, kv head) page is
 *    16 x head_size elements; with the default contiguous strides it is one
 *    contiguous run of memory.  Other strides for the two outer dimensions are
 *    accepted (for instance K and V as views of one [num_blocks, 2, ...] tensor).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and never synchronise, except pa_check_device_error and
 *    pa_profile_read.
 *  - Return value: PA_OK (0) or a negative pa_status.  Argument errors are
 *    detected on the host before anything is launched; nothing is written then.
 *  - Faults that only the device can see (a slot, block id or sequence length out
 *    of range) never cause an out-of-bounds access: the affected work item writes
 *    nothing and sets a bit in the caller's device error word (when one is given),
 *    which pa_check_device_error reports.
 */
#ifndef PA_GB300_H
#define PA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_BLOCK_SIZE 16

typedef enum {
    PA_F32 = 0,
    PA_BF16 = 1,
    PA_F16 = 2,
    PA_FP8_E4M3 = 3, /* OCP OFP8 E4M3: bias 7, no infinities, max 448 */
    PA_I32 = 4,
    PA_I64 = 5
} pa_dtype;

typedef enum {
    PA_KV_AUTO = 0,     /* cache element type == key/value element type: bit copy */
    PA_KV_FP8_E4M3 = 1  /* quantise to E4M3 with a per-tensor scale */
} pa_kv_dtype;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,       /* null pointer, rank/extent mismatch, Hq % Hkv != 0 ... */
    PA_ERR_UNSUPPORTED_DTYPE = -2, /* element type (combination) not provided */
    PA_ERR_ALIGNMENT = -3,         /* a base pointer or stride breaks the 16-byte rule */
    PA_ERR_WORKSPACE = -4,         /* workspace missing or smaller than required */
    PA_ERR_CUDA = -5,              /* a CUDA runtime/driver call or launch failed */
    PA_ERR_DEVICE_BOUNDS = -6,     /* device error word: slot / block id / length out of range */
    PA_ERR_UNSUPPORTED_SHAPE = -7, /* head_size or block size outside what is built */
    PA_ERR_DEVICE_TIMEOUT = -8,    /* device error word: a bounded wait gave up */
    PA_ERR_NO_BLOCKS = -9          /* block manager: the pool has too few free blocks */
} pa_status;

/* Bits of the device error word (an int in device memory, owned by the caller). */
#define PA_DEVERR_SLOT_RANGE 0x1    /* slot_mapping entry >= num_blocks * 16 */
#define PA_DEVERR_BLOCK_RANGE 0x2   /* block_table entry read < 0 or >= num_blocks */
#define PA_DEVERR_SEQLEN_RANGE 0x4  /* seq_lens[s] < 0 or > max_blocks_per_seq * 16 */
#define PA_DEVERR_WAIT_TIMEOUT 0x8  /* a shared-memory pipeline wait exceeded its limit */

typedef void *pa_stream_t; /* cudaStream_t */

typedef struct {
    void *data;        /* device pointer to element [0, 0, ...] */
    int32_t dtype;     /* pa_dtype */
    int32_t ndim;      /* rank, 1..5 */
    int64_t shape[5];  /* extents */
    int64_t stride[5]; /* strides in elements */
} pa_tensor;

/*
 * pa_reshape_and_cache -- scatter this step's new K/V rows into the paged cache.
 *
 * Defined by: "Inside vLLM CUDA Kernels", Part 2 (reshape_and_cache_flash: one
 * destination slot per token, slot -> (block = slot / 16, offset = slot % 16),
 * negative slot = padding with no destination; k_op = copy, or scale and convert
 * for an FP8 cache).
 *
 *   key, value    [T, Hkv, D], PA_F32 / PA_BF16 / PA_F16 (same type for both);
 *                 innermost stride 1; the token and head strides are free.
 *   k_cache,      [num_blocks, Hkv, 16, D]; element type == key's for PA_KV_AUTO,
 *   v_cache       PA_FP8_E4M3 for PA_KV_FP8_E4M3.  Written in place.
 *   slot_mapping  PA_I64 [T].  Row t goes to cache slot slot_mapping[t];
 *                 a negative entry writes nothing for row t.  Entries
 *                 >= num_blocks * 16 write nothing and set PA_DEVERR_SLOT_RANGE.
 *                 Two rows naming the same slot: which one lands is unspecified.
 *   kv_dtype      PA_KV_AUTO: bit-exact copy.  PA_KV_FP8_E4M3: each element x is
 *                 stored as E4M3(fp32(x) / scale) -- one IEEE fp32 division
 *                 rounded to nearest, then round-to-nearest-even to E4M3 with
 *                 saturation to +-448 and NaN -> 0x7F.
 *   k_scale,      device pointers to one fp32 scale each (per tensor); NULL means
 *   v_scale       1.0.  Ignored for PA_KV_AUTO.
 *   device_error  device int to OR error bits into, or NULL.
 * Alignment: key/value/cache base pointers and all strides in bytes must be
 * multiples of 16 bytes, and D * element size a multiple of 16.
 * T == 0 is a no-op.
 */
int pa_reshape_and_cache(const pa_tensor *key, const pa_tensor *value, pa_tensor *k_cache,
                         pa_tensor *v_cache, const pa_tensor *slot_mapping, int kv_dtype,
                         const float *k_scale, const float *v_scale, int *device_error,
                         pa_stream_t stream);

/*
 * Options of the _opt entry points.  Zero-initialise the struct (every field then
 * takes its default) and set what the call needs.
 *
 * Per-head scales ("Inside vLLM CUDA Kernels", Part 2, why layout and quantization
 * scale produce two copy paths: kv_scale_stride == 0 means every head shares one
 * scale, otherwise head h uses scale[h * kv_scale_stride]).
 */
typedef struct {
    const float *k_scale;  /* device fp32 scale(s) of an FP8 cache; NULL = 1.0 */
    const float *v_scale;
    int64_t scale_stride;  /* 0: one scale for every KV head; > 0: KV head h uses
                              k_scale[h * scale_stride] and v_scale[h * scale_stride];
                              < 0: PA_ERR_INVALID_ARG */
    int *device_error;     /* device int to OR error bits into, or NULL */
} pa_write_options;

/*
 * pa_reshape_and_cache_opt -- pa_reshape_and_cache with per-head FP8 scales.
 * Arguments as pa_reshape_and_cache; `opt` may be NULL (all defaults).  An FP8
 * element x of KV head h is stored as E4M3(fp32(x) / scale_h), scale_h as above.
 * The cache may also be a strided view: an NHD cache [num_blocks, 16, Hkv, D]
 * is passed as its [num_blocks, Hkv, 16, D] permutation (strides 16*Hkv*D, D,
 * Hkv*D, 1).
 */
int pa_reshape_and_cache_opt(const pa_tensor *key, const pa_tensor *value, pa_tensor *k_cache,
                             pa_tensor *v_cache, const pa_tensor *slot_mapping, int kv_dtype,
                             const pa_write_options *opt, pa_stream_t stream);

/*
 * pa_decode -- single-query paged decode attention (one query token per sequence).
 *
 * Defined by: "Inside vLLM CUDA Kernels", Part 3 (scores = q k^T * scale,
 * softmax, probs v; online softmax m/l/acc; split-KV merged by max/LSE
 * rescaling) and "vLLM 源码完全拆解（七）" (query [num_seqs, num_heads,
 * head_size]; block_table walk over the first ceil(seq_len / 16) entries; GQA map
 * kv_head = q_head / (Hq / Hkv); tail tokens t >= seq_len excluded from max and
 * denominator; stale tail values never reach the output).
 *
 *   out           [S, Hq, D], same element type as q (may be the same memory as q).
 *   q             [S, Hq, D], PA_F32 / PA_BF16 / PA_F16, innermost stride 1.
 *   k_cache,      [num_blocks, Hkv, 16, D]; element type == q's, or PA_FP8_E4M3
 *   v_cache       with a PA_BF16 / PA_F16 query.
 *   block_table   PA_I32 [S, max_blocks_per_seq], innermost stride 1.  Only the
 *                 first ceil(seq_lens[s] / 16) entries of row s are used; the
 *                 rest may hold any value (padding).
 *   seq_lens      PA_I32 [S]: visible KV length of each sequence, counting the
 *                 token written in this step.  0 gives an all-zero output row.
 *   scale         softmax scale (usually 1 / sqrt(D)).
 *   num_kv_heads  Hkv; must equal k_cache->shape[1] and divide Hq.
 * Head sizes built: 64, 128, 256 (FP8 caches: 128, 256).
 * Uses a library-held workspace on the current device (grown on demand with
 * cudaMallocAsync and zero-filled on `stream`); calls that use it on different
 * streams must not overlap.  FP8 scales are 1.0 here; use pa_decode_ex for scales, a caller-owned
 * workspace, an explicit partition size or a device error word.
 */
int pa_decode(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
              const pa_tensor *block_table, const pa_tensor *seq_lens, float scale, int num_kv_heads,
              pa_stream_t stream);

/*
 * pa_decode_ex -- pa_decode with every knob.
 *
 * Split-KV ("vLLM 源码完全拆解（七）", V1 与 V2: why long contexts need partitions -- a
 * small batch gives too few (sequence, head) work items to fill the GPU, so the context is
 * cut into partitions computed in parallel whose partial results are rescaled and merged;
 * "Inside vLLM CUDA Kernels", Part 3: split-KV changes the work partition, not the
 * softmax identity).  The pages' fixed 512-token partition and 8192-token V1/V2 switch are
 * replaced by a plan measured on GB300 (pa_decode_plan).
 *
 *   k_scale, v_scale  device fp32 per-tensor dequantisation scales for an FP8 cache
 *                     (K and V element values are code_value * scale); NULL = 1.0.
 *   partition_size    how the KV range of a sequence is split: 0 = chosen by the
 *                     library's measured heuristic (pa_decode_plan); -1 = never split;
 *                     > 0 = partitions of that many tokens (rounded up to a multiple of
 *                     16), merged through the workspace; -2, -4 or -8 = every sequence
 *                     cut into 2, 4 or 8 equal parts processed by the CTAs of one
 *                     thread-block cluster and merged through distributed shared
 *                     memory (no workspace); PA_PARTITION_BALANCED = the balanced
 *                     split: the pages of all sequences, concatenated, cut into equal
 *                     ranges over one resident wave of CTAs per (kv head, head group),
 *                     the parts of a cut sequence merged through the workspace
 *                     (batches of at most 511 sequences, else
 *                     PA_ERR_UNSUPPORTED_SHAPE; the fp32 cache runs it unsplit).
 *   workspace,        device memory for split-KV partition states; at least
 *   workspace_bytes   pa_decode_workspace_size(...) bytes for the partition size
 *                     the call ends up using (0 bytes when it does not split or
 *                     uses the cluster split).
 *                     NULL with workspace_bytes == 0 is fine for the unsplit path.
 *                     Zero-fill it once before its first use: it holds per-unit
 *                     arrival counters that every call leaves at zero again.  The
 *                     library owns its contents between calls, and calls that
 *                     share one workspace must not run concurrently.
 *   device_error      device int to OR error bits into, or NULL.
 * Split-KV runs in the one decode launch: each partition's CTA stores its
 * (max, exp-sum, partial output) state and the last CTA of a (sequence, kv head)
 * unit merges them with log-sum-exp rescaling.  The decode kernel is launched as a
 * programmatic dependent of the preceding work on `stream` and waits for it before
 * reading any input.
 */
#define PA_PARTITION_BALANCED (-100)
int pa_decode_ex(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
                 const pa_tensor *block_table, const pa_tensor *seq_lens, float scale, int num_kv_heads,
                 const float *k_scale, const float *v_scale, int partition_size, void *workspace,
                 size_t workspace_bytes, int *device_error, pa_stream_t stream);

/*
 * Decode options (pa_decode_opt).  Zero-initialise, then set what is needed.
 *
 * ALiBi ("vLLM 源码完全拆解（七）", the QK step: the kernel adds a_h times the
 * (non-positive) distance of key token t from the current position seq_len - 1 to
 * the scaled logit, before the softmax): with alibi_slopes, the logit of query head
 * h for key token t is scale * q.k_t + alibi_slopes[h] * (t - (seq_len - 1)).
 */
typedef struct {
    const float *k_scale;        /* as pa_write_options: FP8 dequantisation scales, */
    const float *v_scale;        /* NULL = 1.0; element value = code value * scale_h */
    int64_t scale_stride;        /* 0: one scale; > 0: KV head h uses [h * scale_stride] */
    const float *alibi_slopes;   /* device fp32 [Hq], contiguous, or NULL (no bias) */
    int partition_size;          /* as pa_decode_ex (0 = the library's plan) */
    void *workspace;             /* as pa_decode_ex; NULL with 0 bytes = the library's */
    size_t workspace_bytes;      /*   internal workspace (pa_decode's) */
    int *device_error;           /* device int to OR error bits into, or NULL */
    /* Poll limit of the first shared-memory pipeline wait (decode: each warp's first page;
     * query tile: the first K/V group).  0 = the normal limit (about 2^20 polls); > 0 = that
     * many polls; < 0 = give up without polling.  For testing the timeout path: a wait that
     * gives up first waits (with the normal limit) for the copies it had in flight, sets
     * PA_DEVERR_WAIT_TIMEOUT and writes no output for its work item (nor for a split-KV unit
     * that any of its parts gave up on).  Every later wait keeps the normal limit. */
    int first_wait_limit;
} pa_decode_options;

/*
 * pa_decode_opt -- pa_decode with every option.  Arguments as pa_decode; `opt`
 * may be NULL (all defaults, as pa_decode).  Status codes as pa_decode_ex.  The
 * cache may be an NHD cache passed as its [num_blocks, Hkv, 16, D] permutation.
 */
int pa_decode_opt(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
                  const pa_tensor *block_table, const pa_tensor *seq_lens, float scale, int num_kv_heads,
                  const pa_decode_options *opt, pa_stream_t stream);

/*
 * pa_attention_varlen -- paged attention for several new query tokens per sequence
 * (speculative decoding, chunked prefill): the varlen read path of "Inside vLLM CUDA
 * Kernels", Part 3 (query_start_loc packs each request's tokens, seq_lens bounds its
 * visible history, block_table resolves the history's pages).
 *
 *   out, q           [Tq, Hq, D]: the new tokens of all sequences, packed; sequence s owns
 *                    rows query_start_loc[s] .. query_start_loc[s+1]-1 (n_s tokens).  out
 *                    may not alias q.  Rows of no sequence are not written.
 *   query_start_loc  PA_I32 [S + 1], non-decreasing (device).
 *   block_table,     as pa_decode, S rows; seq_lens[s] counts the history and the n_s new
 *   seq_lens         tokens (already written to the cache).
 *   max_query_len    host upper bound of every n_s; sizes the grid.
 * Query i of sequence s sits at position seq_lens[s] - n_s + i and attends to the tokens
 * 0 .. that position (causal; with alibi_slopes the logit gets slope_h * (t - position)).
 * n_s = 1 for every s is pa_decode.  A sequence whose rows fall outside [0, Tq), or with
 * n_s < 0, n_s > max_query_len or n_s > seq_lens[s], writes nothing and sets
 * PA_DEVERR_SEQLEN_RANGE.
 * opt: as pa_decode_opt; NULL = defaults.  The partition plan and the workspace size count
 * query columns as Hq * max_query_len heads: pa_decode_plan / pa_decode_workspace_size
 * with num_heads = Hq * max_query_len give them.  PA_PARTITION_BALANCED is refused
 * (PA_ERR_UNSUPPORTED_SHAPE).  Kernels: with fewer than 64 query columns per KV head
 * (max_query_len * Hq / Hkv; 32 at head size 64), an fp8 or fp32 cache, D other than 64 / 128, or a split
 * asked for (partition_size > 0 or a cluster split), the decode kernels run with 8
 * columns per CTA, each CTA reading the pages its columns see.  Otherwise (bf16 / f16
 * cache, partition_size 0 or -1) a query-tile kernel runs on the tcgen05 tensor cores:
 * 128 query rows per CTA share each page load, the page range is not split and no
 * workspace is used.
 */
int pa_attention_varlen(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
                        const pa_tensor *query_start_loc, const pa_tensor *block_table, const pa_tensor *seq_lens,
                        float scale, int num_kv_heads, int max_query_len, const pa_decode_options *opt,
                        pa_stream_t stream);

/*
 * pa_decode_step -- one decode step in one call: the cache write of the step's new rows
 * (pa_reshape_and_cache_opt) followed by pa_decode_opt over the updated cache, with the
 * decode reading everything the write does not touch while the write still runs.
 *
 * The pages call the two operations in this order for every layer ("How vLLM CUDA Kernels
 * Write and Read the Paged KV Cache": the new token's K/V go to their slot, then attention
 * reads the sequence's blocks through block_table).  Here the decode is launched behind the
 * write with a programmatic dependency.  With new_rows_start (several new rows per
 * sequence) it reads q, the tables and every page without a new position while the write
 * runs, and waits for the write only before a page that holds new positions and before it
 * writes out or its workspace; with one new row per sequence it starts behind the write as
 * pa_decode_opt does (the write is over before early reads could help).
 *
 *   out, q, k_cache, v_cache, block_table, seq_lens, scale, num_kv_heads, opt: as
 *                    pa_decode_opt (one query token per sequence; opt's scales and
 *                    scale_stride also quantise the rows written to an FP8 cache).
 *   key, value       [T, Hkv, D] new rows, slot_mapping int64 [T]: as pa_reshape_and_cache
 *                    (kv dtype: E4M3 when the cache is E4M3, else the cache keeps q's dtype).
 *   new_rows_start   NULL: T == S and row s is sequence s's newest token.  Else int32 [S + 1]
 *                    (device): rows new_rows_start[s] .. new_rows_start[s+1]-1 are sequence
 *                    s's newest n_s tokens, row i at position seq_lens[s] - n_s + i.
 * Precondition (not checked on the device): every row's slot is the one its position maps to
 * in its sequence's block table (or < 0: no write), and no other sequence of the batch reads
 * that block.  Every argument of both operations is validated before anything is launched;
 * the results equal those of the two calls made one after the other.
 */
int pa_decode_step(pa_tensor *out, const pa_tensor *q, const pa_tensor *key, const pa_tensor *value,
                   pa_tensor *k_cache, pa_tensor *v_cache, const pa_tensor *slot_mapping,
                   const pa_tensor *new_rows_start, const pa_tensor *block_table, const pa_tensor *seq_lens,
                   float scale, int num_kv_heads, const pa_decode_options *opt, pa_stream_t stream);

/*
 * pa_decode_noalloc -- pa_decode_ex for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for callers that have no
 * allocator where they run decode (a plugin that an inference runtime hands only
 * its input and output buffers) or must not allocate there (a serving loop that
 * has given all free device memory to its KV-cache pool, where an allocation can
 * fail and cudaMalloc/cudaFree can synchronise the device).  It takes the same
 * inputs and outputs as pa_decode_ex minus the workspace: the split-KV scratch is
 * a fixed buffer of PA_NOALLOC_SCRATCH_BYTES (32 MiB) inside the library, which
 * every GPU that loads the library keeps until the process exits.  The call makes
 * no cudaMalloc, cudaFree or other allocating call.
 *
 *   - A call whose plan needs more split-KV scratch than PA_NOALLOC_SCRATCH_BYTES
 *     (pa_decode_workspace_size for the partition size it would use) returns
 *     PA_ERR_WORKSPACE and launches nothing; use a larger partition_size, -1
 *     (never split, needs no scratch) or pa_decode_ex.
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress with that device current) and keeps it; make that
 *     first call before any stream capture.
 *   - All calls on a device share the one buffer, which keeps whatever the last
 *     call left there.  Each call first clears, on its stream, the part that must
 *     start at zero.  Calls that can overlap on the GPU (different streams without
 *     ordering between them) race on the buffer and give wrong results.
 * Returns the pa_decode_ex status codes.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)
int pa_decode_noalloc(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
                      const pa_tensor *block_table, const pa_tensor *seq_lens, float scale, int num_kv_heads,
                      const float *k_scale, const float *v_scale, int partition_size, int *device_error,
                      pa_stream_t stream);

/*
 * pa_decode_plan -- host-only: the split pa_decode_ex would use.
 *
 * The pages choose between the unpartitioned kernel and 512-token partitions by a fixed
 * rule (max_seq_len <= 8192 and one partition or num_seqs * num_heads > 512: unsplit) and
 * describe the choice as a trade-off between parallelism and the extra reduction, to be
 * weighed per shape ("vLLM 源码完全拆解（七）", V1 与 V2 and 性能模型).  This plan makes
 * the same trade on GB300 from the batch's work units against the GPU's resident CTA slots,
 * fitted to a measured sweep of partition sizes over the benchmark workloads.
 *   kv_dtype_code   pa_dtype of the cache; sm_count <= 0 queries the current device.
 *   partition_size  in: as for pa_decode_ex.  *partition_out: tokens per fixed
 *                   partition, 0 = unsplit, -C for the cluster split into C parts, or
 *                   PA_PARTITION_BALANCED; *num_partitions_out: partitions of the
 *                   longest possible sequence (max_blocks_per_seq * 16 tokens), C, or
 *                   the balanced split's CTAs per (kv head, head group).
 *                   With sm_count > 0 the CTAs resident per SM are the shared-memory
 *                   bound; with sm_count <= 0, the current device's occupancy.
 * Returns PA_OK or PA_ERR_INVALID_ARG.  No device memory is touched.
 */
int pa_decode_plan(int num_seqs, int num_heads, int num_kv_heads, int head_size, int max_blocks_per_seq,
                   int kv_dtype_code, int sm_count, int partition_size, int *partition_out,
                   int *num_partitions_out);

/*
 * pa_decode_workspace_size -- bytes of split-KV workspace for `partition_size`
 * tokens per partition (0 or -1 = unsplit -> 0 bytes; invalid arguments -> 0).
 * For PA_PARTITION_BALANCED: enough for any cache type on the current device
 * (0 when no device can be queried).  Host-only.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                int max_blocks_per_seq, int partition_size);

/*
 * Block manager -- host bookkeeping of the physical block pool ("tiny-vllm, Part 6:
 * the block table and physical block lifetime": one free list, blocks taken when a
 * token is the first of a logical block, all of a sequence's blocks returned when it
 * ends; "PagedAttention kernel: paged KV cache & block tables": identical blocks can
 * be shared across sequences).  Pure host code: no device memory, no stream.  One
 * manager is not thread safe.
 *
 * Blocks carry reference counts.  A forked sequence shares its source's blocks; when
 * a token is appended to a shared block that is not full, that block is first copied
 * to a fresh one (copy on write): the append reports the (source, destination) block
 * pair, and the caller copies it on the device (pa_copy_blocks) before writing the
 * token's K/V.
 */
typedef struct pa_block_manager pa_block_manager;

/* num_blocks physical blocks (ids 0 .. num_blocks-1), sequence ids 0 .. max_seqs-1,
 * at most max_blocks_per_seq blocks per sequence.  NULL on bad arguments or no memory. */
pa_block_manager *pa_bm_create(int num_blocks, int max_seqs, int max_blocks_per_seq);
void pa_bm_destroy(pa_block_manager *m);
int pa_bm_num_free(const pa_block_manager *m);          /* free blocks; -1 for NULL */
int pa_bm_block_refs(const pa_block_manager *m, int block);  /* references; -1 if invalid */
int64_t pa_bm_seq_len(const pa_block_manager *m, int seq);   /* tokens; -1 if not live */

/* Append n_tokens positions to sequence `seq` (it becomes live) and store their cache
 * slots (block * 16 + offset) in slots_out (host int64 [n_tokens]).  Blocks are taken
 * from the free list as tokens start new logical blocks.  copy_out (host int64 [2],
 * required when the sequence's last block is shared and not full) receives the
 * (source, destination) pair of a copy on write; *n_copies (nullable) gets 0 or 1.
 * PA_ERR_NO_BLOCKS (nothing changed) when the pool cannot supply the blocks;
 * PA_ERR_INVALID_ARG for a bad id, a negative count, more than max_blocks_per_seq blocks,
 * or a missing copy_out. */
int pa_bm_append(pa_block_manager *m, int seq, int n_tokens, int64_t *slots_out, int64_t *copy_out,
                 int *n_copies);

/* Sequence dst (not live) starts as a copy of src (live): same length, same blocks,
 * each block's reference count + 1. */
int pa_bm_fork(pa_block_manager *m, int src, int dst);

/* Drop all of a sequence's references; blocks nobody references go back to the free
 * list.  The sequence is no longer live (freeing one that is not live is a no-op). */
int pa_bm_free(pa_block_manager *m, int seq);

/* Block-table rows and lengths of sequences seqs[0..n-1] into host arrays: row i of
 * block_table_out (int32, row_stride >= max_blocks_per_seq entries, unused entries -1)
 * and seq_lens_out[i] (nullable; 0 for a sequence that is not live), ready for a
 * host-to-device copy and pa_decode. */
int pa_bm_export(const pa_block_manager *m, const int *seqs, int n, int row_stride, int32_t *block_table_out,
                 int32_t *seq_lens_out);

/* Copy whole cache blocks on the device: for each row (src, dst) of block_pairs
 * (PA_I64 [n, 2], contiguous, device), every (kv head, token) row of block src of
 * k_cache and v_cache ([num_blocks, Hkv, 16, D], any 16-byte-aligned strides, any cache
 * type) is copied to block dst.  Pairs naming a block outside [0, num_blocks) copy
 * nothing and set PA_DEVERR_BLOCK_RANGE.  Asynchronous on `stream`. */
int pa_copy_blocks(pa_tensor *k_cache, pa_tensor *v_cache, const pa_tensor *block_pairs, int *device_error,
                   pa_stream_t stream);

/*
 * pa_check_device_error -- synchronise `stream`, read the device error word,
 * store its bits in *bits_out (nullable) and reset the word to 0.
 * Returns PA_OK, PA_ERR_DEVICE_BOUNDS (any range bit), PA_ERR_DEVICE_TIMEOUT
 * (wait bit only) or PA_ERR_CUDA.
 */
int pa_check_device_error(int *device_error, int *bits_out, pa_stream_t stream);

/* Human-readable text for a pa_status value (static storage). */
const char *pa_status_string(int status);

/*
 * Profiling: when enabled, every kernel the library launches is bracketed by a
 * pair of CUDA events recorded on its launch stream.  pa_profile_read
 * synchronises on the recorded events, returns the summed device time (ms) and
 * the launch count for one kernel kind since the last read, and clears them.
 *   kind: 0 = cache write, 1 = decode (attention with the fused split-KV merge).
 */
#define PA_KERNEL_WRITE 0
#define PA_KERNEL_DECODE 1
int pa_profile_enable(int on);
int pa_profile_read(int kind, double *total_ms, long long *launches);

#ifdef __cplusplus
}
#endif

#endif /* PA_GB300_H */
