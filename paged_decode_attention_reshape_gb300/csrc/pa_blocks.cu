// pa_blocks.cu -- host block manager for the paged KV cache, and the device block copy.
//
// What the pages describe ("tiny-vllm, Part 6: the block table and physical block
// lifetime"; "PagedAttention kernel: paged KV cache & block tables"): physical blocks
// come from one free list (allocation takes a block off it, returning puts it back),
// a sequence's block table maps its logical blocks to physical ones, a new block is
// taken only when a token is the first of a logical block, all of a sequence's blocks
// go back when it ends, and identical blocks can be shared by several sequences
// (prefix sharing).
//
// Here a block has a reference count.  pa_bm_fork makes a sequence share all of
// another's blocks (a common prefix: each block's count goes up); pa_bm_free drops a
// sequence's references and returns the blocks that nobody references any more.  A
// token appended to a shared block that is not full would change what the other
// sequences see, so that block is first copied to a fresh one (copy on write): the
// append reports the (source, destination) pair and the caller runs pa_copy_blocks on
// the device before writing the token.
//
// The manager is host code with no device state; one instance is not thread safe.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>
#include <numeric>
#include <vector>

#include "pa_internal.h"

#define PA_API extern "C" __attribute__((visibility("default")))

using pa::kBlock;

struct pa_block_manager {
  int num_blocks, max_seqs, max_blocks_per_seq;
  std::vector<int32_t> free_list;  // taken from the back
  std::vector<int32_t> refs;       // references per physical block
  struct Seq {
    bool live = false;
    int64_t len = 0;
    std::vector<int32_t> blocks;
  };
  std::vector<Seq> seqs;
};

namespace {

bool seq_ok(const pa_block_manager *m, int s) { return m && s >= 0 && s < m->max_seqs; }

int take_block(pa_block_manager *m) {
  const int32_t b = m->free_list.back();
  m->free_list.pop_back();
  m->refs[b] = 1;
  return b;
}

void drop_ref(pa_block_manager *m, int32_t b) {
  if (--m->refs[b] == 0) m->free_list.push_back(b);
}

}  // namespace

PA_API pa_block_manager *pa_bm_create(int num_blocks, int max_seqs, int max_blocks_per_seq) {
  if (num_blocks <= 0 || max_seqs <= 0 || max_blocks_per_seq <= 0) return nullptr;
  pa_block_manager *m = new (std::nothrow) pa_block_manager;
  if (!m) return nullptr;
  m->num_blocks = num_blocks;
  m->max_seqs = max_seqs;
  m->max_blocks_per_seq = max_blocks_per_seq;
  // ascending from the back: the first blocks handed out are 0, 1, 2, ...
  m->free_list.resize(num_blocks);
  std::iota(m->free_list.rbegin(), m->free_list.rend(), 0);
  m->refs.assign(num_blocks, 0);
  m->seqs.resize(max_seqs);
  return m;
}

PA_API void pa_bm_destroy(pa_block_manager *m) { delete m; }

PA_API int pa_bm_num_free(const pa_block_manager *m) { return m ? static_cast<int>(m->free_list.size()) : -1; }

PA_API int pa_bm_block_refs(const pa_block_manager *m, int block) {
  return (m && block >= 0 && block < m->num_blocks) ? m->refs[block] : -1;
}

PA_API int64_t pa_bm_seq_len(const pa_block_manager *m, int seq) {
  return (seq_ok(m, seq) && m->seqs[seq].live) ? m->seqs[seq].len : -1;
}

PA_API int pa_bm_append(pa_block_manager *m, int seq, int n_tokens, int64_t *slots_out, int64_t *copy_out,
                        int *n_copies) {
  if (!seq_ok(m, seq) || n_tokens < 0 || (n_tokens > 0 && !slots_out)) return PA_ERR_INVALID_ARG;
  pa_block_manager::Seq &q = m->seqs[seq];
  q.live = true;
  if (n_copies) *n_copies = 0;
  if (n_tokens == 0) return PA_OK;
  const int64_t len = q.len, end = len + n_tokens;
  const int64_t need_blocks = (end + kBlock - 1) / kBlock;
  if (need_blocks > m->max_blocks_per_seq) return PA_ERR_INVALID_ARG;
  // a token going into a shared, partly filled last block needs a private copy first
  const bool cow = len % kBlock != 0 && m->refs[q.blocks.back()] > 1;
  if (cow && !copy_out) return PA_ERR_INVALID_ARG;
  const int64_t fresh = need_blocks - static_cast<int64_t>(q.blocks.size()) + (cow ? 1 : 0);
  if (fresh > static_cast<int64_t>(m->free_list.size())) return PA_ERR_NO_BLOCKS;  // nothing changed
  if (cow) {
    const int32_t old = q.blocks.back(), nb = take_block(m);
    drop_ref(m, old);
    q.blocks.back() = nb;
    copy_out[0] = old;
    copy_out[1] = nb;
    if (n_copies) *n_copies = 1;
  }
  for (int64_t pos = len; pos < end; ++pos) {
    if (pos % kBlock == 0) q.blocks.push_back(take_block(m));  // first token of a logical block
    slots_out[pos - len] = static_cast<int64_t>(q.blocks[pos / kBlock]) * kBlock + pos % kBlock;
  }
  q.len = end;
  return PA_OK;
}

PA_API int pa_bm_fork(pa_block_manager *m, int src, int dst) {
  if (!seq_ok(m, src) || !seq_ok(m, dst) || src == dst || !m->seqs[src].live || m->seqs[dst].live)
    return PA_ERR_INVALID_ARG;
  pa_block_manager::Seq &d = m->seqs[dst];
  d = m->seqs[src];
  for (int32_t b : d.blocks) ++m->refs[b];
  return PA_OK;
}

PA_API int pa_bm_free(pa_block_manager *m, int seq) {
  if (!seq_ok(m, seq)) return PA_ERR_INVALID_ARG;
  pa_block_manager::Seq &q = m->seqs[seq];
  for (auto it = q.blocks.rbegin(); it != q.blocks.rend(); ++it) drop_ref(m, *it);
  q = pa_block_manager::Seq{};
  return PA_OK;
}

PA_API int pa_bm_export(const pa_block_manager *m, const int *seqs, int n, int row_stride, int32_t *block_table_out,
                        int32_t *seq_lens_out) {
  if (!m || n < 0 || (n > 0 && (!seqs || !block_table_out)) || row_stride < m->max_blocks_per_seq)
    return PA_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    if (!seq_ok(m, seqs[i])) return PA_ERR_INVALID_ARG;
    const pa_block_manager::Seq &q = m->seqs[seqs[i]];
    int32_t *row = block_table_out + static_cast<int64_t>(i) * row_stride;
    std::fill(row, row + row_stride, -1);
    std::copy(q.blocks.begin(), q.blocks.end(), row);
    if (seq_lens_out) seq_lens_out[i] = q.live ? static_cast<int32_t>(q.len) : 0;
  }
  return PA_OK;
}

// ------------------------------------------------------------- block copy

namespace pa {
namespace {

// One CTA per (pair, cache): copies every (kv head, token) row of block src to block dst,
// 16 bytes per thread and step.
__global__ void __launch_bounds__(256) copy_blocks_kernel(char *kc, char *vc, int64_t kc_s0, int64_t kc_s1,
                                                          int64_t kc_s2, int64_t vc_s0, int64_t vc_s1, int64_t vc_s2,
                                                          int Hkv, int row_bytes, const int64_t *pairs, int n,
                                                          int num_blocks, int *err) {
  const int i = blockIdx.x >> 1;
  const bool is_v = blockIdx.x & 1;
  if (i >= n) return;
  const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && !is_v && err) atomicOr(err, kErrBlock);
    return;
  }
  char *base = is_v ? vc : kc;
  const int64_t s0 = is_v ? vc_s0 : kc_s0, s1 = is_v ? vc_s1 : kc_s1, s2 = is_v ? vc_s2 : kc_s2;  // bytes
  const int packs = row_bytes / 16, per_block = Hkv * kBlock * packs;
  for (int j = threadIdx.x; j < per_block; j += blockDim.x) {
    const int pk = j % packs, r = j / packs, t = r % kBlock, h = r / kBlock;
    const int64_t off = h * s1 + t * s2 + static_cast<int64_t>(pk) * 16;
    *reinterpret_cast<uint4 *>(base + dst * s0 + off) = *reinterpret_cast<const uint4 *>(base + src * s0 + off);
  }
}

}  // namespace
}  // namespace pa

PA_API int pa_copy_blocks(pa_tensor *k_cache, pa_tensor *v_cache, const pa_tensor *block_pairs, int *device_error,
                          pa_stream_t stream) {
  using namespace pa;
  if (!k_cache || !v_cache || !block_pairs || k_cache->ndim != 4 || v_cache->ndim != 4 || block_pairs->ndim != 2)
    return PA_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i)
    if (k_cache->shape[i] != v_cache->shape[i]) return PA_ERR_INVALID_ARG;
  if (k_cache->dtype != v_cache->dtype || k_cache->shape[2] != kBlock) return PA_ERR_INVALID_ARG;
  if (block_pairs->dtype != PA_I64 || block_pairs->shape[1] != 2 || block_pairs->stride[1] != 1 ||
      block_pairs->stride[0] != 2)
    return PA_ERR_INVALID_ARG;
  const int64_t n = block_pairs->shape[0];
  if (n == 0) return PA_OK;
  if (n > (1 << 30) || !k_cache->data || !v_cache->data || !block_pairs->data) return PA_ERR_INVALID_ARG;
  const int eb = k_cache->dtype == PA_F32 ? 4 : (k_cache->dtype == PA_FP8_E4M3 ? 1 : 2);
  const int row_bytes = static_cast<int>(k_cache->shape[3]) * eb;
  if (k_cache->stride[3] != 1 || v_cache->stride[3] != 1 || row_bytes % 16) return PA_ERR_INVALID_ARG;
  const uintptr_t kb = reinterpret_cast<uintptr_t>(k_cache->data), vb = reinterpret_cast<uintptr_t>(v_cache->data);
  if (kb % 16 || vb % 16) return PA_ERR_ALIGNMENT;
  for (int i = 0; i < 3; ++i)
    if ((k_cache->stride[i] * eb) % 16 || (v_cache->stride[i] * eb) % 16) return PA_ERR_ALIGNMENT;
  copy_blocks_kernel<<<static_cast<unsigned>(2 * n), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<char *>(k_cache->data), static_cast<char *>(v_cache->data), k_cache->stride[0] * eb,
      k_cache->stride[1] * eb, k_cache->stride[2] * eb, v_cache->stride[0] * eb, v_cache->stride[1] * eb,
      v_cache->stride[2] * eb, static_cast<int>(k_cache->shape[1]), row_bytes,
      static_cast<const int64_t *>(block_pairs->data), static_cast<int>(n), static_cast<int>(k_cache->shape[0]),
      device_error);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
