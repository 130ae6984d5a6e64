// pa_internal.h -- launch parameters shared by the host API and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/pa.h"

namespace pa {

constexpr int kBlock = PA_BLOCK_SIZE;  // tokens per KV-cache block (one "page")
constexpr int kFlatMaxSeqs = 511;      // batch limit of the balanced split (page offsets kept in smem)

// Cache element kinds of the decode kernels (query/output type in brackets).
enum DecodeKind : int {
  KIND_BF16 = 0,      // bf16 cache [bf16 q]
  KIND_F16 = 1,       // f16 cache [f16 q]
  KIND_FP8_BF16Q = 2, // e4m3 cache [bf16 q]
  KIND_FP8_F16Q = 3,  // e4m3 cache [f16 q]
  KIND_F32 = 4        // fp32 cache [fp32 q], CUDA-core path
};

struct WriteParams {
  const void *key, *value;
  void *k_cache, *v_cache;
  const int64_t *slot_mapping;
  int64_t T;
  int Hkv, D;
  int64_t key_ts, key_hs, val_ts, val_hs;          // elements
  int64_t kc_s0, kc_s1, kc_s2, vc_s0, vc_s1, vc_s2; // elements
  int64_t num_slots;                                // num_blocks * 16
  const float *k_scale, *v_scale;                   // nullable
  int64_t scale_stride;                             // 0: per tensor; else KV head h uses [h * stride]
  int *err;                                         // nullable
  int i32;                                          // every source offset, cache stride and offset
                                                    // within a block below 2^31 bytes
};

struct DecodeParams {
  void *out;
  const void *q;
  int64_t out_ss, out_hs, q_ss, q_hs;  // elements
  const int32_t *block_table;
  int64_t bt_ss;
  const int32_t *seq_lens;
  int S, Hq, Hkv, G, HG, D;            // HG = head groups of <= 8 query heads per KV head
  int num_blocks, max_blocks;
  float scale_log2;                    // softmax scale * log2(e)
  const float *k_scale, *v_scale;      // nullable (1.0)
  int64_t scale_stride;                // 0: per tensor; else KV head g uses k_scale[g * scale_stride]
  const float *alibi;                  // nullable: ALiBi slope per query head [Hq]
  int pages_per_part;                  // partition length in pages
  int max_parts;                       // partitions of the longest sequence (1 = unsplit); = cluster if > 1
  int cluster;                         // > 1: cluster split, each unit cut into `cluster` equal parts
  int *counters;                       // [S, Hkv, HG] arrival counters of split units (zero between calls)
  float2 *part_ml;                     // [S, Hq, max_parts] (m in log2 units, l)
  float *part_acc;                     // [S, Hq, max_parts, D]
  int *err;                            // nullable
  int lpt;                             // 1: CTA row z takes the z-th longest sequence (S <= kLptMax)
  // Query columns.  A CTA covers 8 "virtual heads" of one KV head; virtual head v is query
  // token v / G of its sequence at query head g G + v % G.  Decode: one token per sequence,
  // VH = G.  Several tokens (varlen): qsl = query_start_loc [S + 1], VH = nq_max * G.
  const int32_t *qsl;                  // nullable: sequence s owns q / out rows qsl[s] .. qsl[s+1]-1
  int nq_max;                          // largest number of query tokens per sequence (1 for decode)
  int64_t Tq;                          // rows of q / out
  int VH;                              // virtual heads per KV head; HG = ceil(VH / 8)
  int nhd;                             // caches token-major within a block (TMA coordinates (d, g, 0, blk))
  int q_tma;                           // query-tile kernel: Q tiles come by TMA (tmQ), else by loads
  // Early reads (pa_decode_step): the grid launched just before this one writes only the
  // newest n_s positions of each sequence s (n_s = new_start[s+1] - new_start[s], or 1 when
  // new_start is null).  The kernel then reads q, the tables and every other page before that
  // grid completes and waits for it only before a page holding new positions and before
  // writing any output.  0: wait for it first.
  int early;
  const int32_t *new_start;
  int flat;                            // > 0: balanced split, this many CTAs per head row (S <= kFlatMaxSeqs)
  // Poll limit of the first pipeline wait (decode: each warp's first page; query tile: the
  // first K/V group): 0 = the normal limit, > 0 = that many polls, < 0 = give up at once.
  // Tests use it to make a bounded wait run out; every later wait and drain keeps the normal limit.
  int first_wait_limit;
  // fp32 path only: direct cache pointers and strides (elements)
  const float *kc, *vc;
  int64_t kc_s0, kc_s1, kc_s2, vc_s0, vc_s1, vc_s2;
};

// The query columns of one CTA: virtual heads v0 .. v0+7 of KV head g (see DecodeParams).
// Column j is query token (v0 + j) / G of the sequence -- q / out row row0 + (v0 + j) / G --
// at query head g G + (v0 + j) % G.
struct Cols {
  int64_t row0;  // q / out row of the sequence's first query token
  int G, g, v0;
  __host__ __device__ __forceinline__ int64_t row(int j) const { return row0 + (v0 + j) / G; }
  __host__ __device__ __forceinline__ int head(int j) const { return g * G + (v0 + j) % G; }
  __host__ __device__ __forceinline__ int64_t out_off(const DecodeParams &p, int j) const {
    return row(j) * p.out_ss + static_cast<int64_t>(head(j)) * p.out_hs;
  }
  __host__ __device__ __forceinline__ int64_t q_off(const DecodeParams &p, int j) const {
    return row(j) * p.q_ss + static_cast<int64_t>(head(j)) * p.q_hs;
  }
};

// Error bits (mirror PA_DEVERR_* of pa.h).
constexpr int kErrSlot = PA_DEVERR_SLOT_RANGE;
constexpr int kErrBlock = PA_DEVERR_BLOCK_RANGE;
constexpr int kErrSeqLen = PA_DEVERR_SEQLEN_RANGE;
constexpr int kErrTimeout = PA_DEVERR_WAIT_TIMEOUT;

// Every check pa_decode_ex makes, without launching or allocating anything; on PA_OK,
// *ws_bytes is the split-KV workspace the call will need and *counter_bytes the size of the
// arrival-counter region at its start, which must be zero when the decode starts (both 0
// when the call does not split or uses the cluster split).  Used by pa_decode_noalloc.
int decode_ex_requirements(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
                           const pa_tensor *block_table, const pa_tensor *seq_lens, float scale, int num_kv_heads,
                           const float *k_scale, const float *v_scale, int partition_size, int *device_error,
                           size_t *ws_bytes, size_t *counter_bytes);

// Launchers (defined next to their kernels).  Return a cudaError_t.
// ctas_per_sm: the grid's CTAs per SM (1 .. 4; 0 = the standalone write's choice).
cudaError_t launch_write(const WriteParams &p, int in_dtype, int cache_dtype, int sm_count, int ctas_per_sm,
                         cudaStream_t st);

// Tensor-core kernel shape per (kind, head size): warps per CTA and pipeline
// stages per warp.  Shared memory = W * STAGES * 2 pages (+ alignment, barriers).
// A CTA's loads are served at a bounded rate for each warp's stages in flight
// (measured on GB300: one 2 KiB K+V page pair per warp about every 0.5 us with the
// page math, 2 to 4 stages alike), so the warps per CTA set how fast one long
// sequence streams.  Head size 64: 8 warps (3 CTAs per SM); 128 and 256: 4 warps,
// whose larger pages already fill HBM with 3 CTAs per SM.
constexpr int mma_warps(int kind, int D) { return (void)kind, D == 64 ? 8 : 4; }
// Two stages per warp: pages of 2-8 KiB give 35-131 KiB per CTA.  Measured on
// GB300: 3-4 stages with fewer CTAs per SM were slower on every benchmark workload.
constexpr int mma_stages(int kind, int D) { return (void)kind, (void)D, 2; }
// Resident CTAs per SM the register allocation must allow (ptxas launch bound): as
// many as the shared memory admits, so registers never cut the occupancy, except
// for the E4M3 head-size-128 kernel (6 by shared memory; held at 4 to avoid spills).
constexpr bool mma_fp8(int kind) { return kind == KIND_FP8_BF16Q || kind == KIND_FP8_F16Q; }
constexpr int mma_min_ctas(int kind, int D) {
  return D == 64 ? 3 : D == 128 ? (mma_fp8(kind) ? 4 : 3) : (mma_fp8(kind) ? 3 : 1);
}
constexpr size_t kMmaScratch = 2048;  // sequence-order ranking scratch (after the barriers)
constexpr size_t mma_smem(int kind, int D) {
  return 1024 + static_cast<size_t>(mma_warps(kind, D)) * mma_stages(kind, D) *
                    (2 * kBlock * D * ((kind == KIND_FP8_BF16Q || kind == KIND_FP8_F16Q) ? 1 : 2) + 8) +
         kMmaScratch;
}

cudaError_t launch_decode_mma_16(const DecodeParams &p, int kind, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                 cudaStream_t st);  // KIND_BF16, KIND_F16
cudaError_t launch_decode_mma_fp8(const DecodeParams &p, int kind, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                  cudaStream_t st);  // KIND_FP8_*
cudaError_t launch_decode_f32(const DecodeParams &p, cudaStream_t st);
// Query-tile kernel for chunks of query tokens (pa_attention_varlen) on tcgen05 tensor
// cores: bf16 / f16 caches, head sizes 64 and 128; never splits the page range.
// tmQ is read when p.q_tma is set (make_q_map).
cudaError_t launch_chunk_umma(const DecodeParams &p, int kind, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              const CUtensorMap &tmQ, cudaStream_t st);
// Query columns per KV head (max_query_len x G) from which varlen attention uses it: below
// that the column-group kernels are as fast or faster (256 sequences of 512-4096 tokens, 32/8
// heads: at 32 columns 644 vs 737 us at head size 128, but 453 vs 325 us at head size 64).
constexpr int chunk_min_columns(int D) { return D == 64 ? 32 : 64; }
// Query columns per KV head above which the query-tile kernel takes two 128-row tiles per
// CTA (head size 128).
constexpr int kChunkTwoTileColumns = 128;
// Resident CTAs per SM of a tensor-core instantiation (CUDA occupancy calculator:
// shared memory, registers and threads); 0 when it cannot be queried.
int occupancy_decode_mma_16(int kind, int D);
int occupancy_decode_mma_fp8(int kind, int D);

// Launch `kern` as a programmatic dependent of the previous work on `st`, in
// thread-block clusters of `cluster_x` CTAs along x when cluster_x > 1.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster_x,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster_x > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace pa
