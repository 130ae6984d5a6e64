// pa_api.cu -- the C ABI of include/pa.h: argument validation, the split-KV
// partition plan, TMA descriptors, workspace, device error word and profiling.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "pa_internal.h"

#define PA_API extern "C" __attribute__((visibility("default")))

namespace pa {
namespace {

// ------------------------------------------------------------------ helpers

int elem_bytes(int dt) {
  switch (dt) {
    case PA_F32: case PA_I32: return 4;
    case PA_BF16: case PA_F16: return 2;
    case PA_FP8_E4M3: return 1;
    case PA_I64: return 8;
    default: return 0;
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Descriptor sanity: non-null, rank, element type, positive extents.
int check_desc(const pa_tensor *t, int ndim) {
  if (!t || t->ndim != ndim) return PA_ERR_INVALID_ARG;
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0 || t->stride[i] < 0) return PA_ERR_INVALID_ARG;
  if (elem_bytes(t->dtype) == 0) return PA_ERR_UNSUPPORTED_DTYPE;
  return PA_OK;
}

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

// --------------------------------------------------------------- profiling

struct Profiler {
  std::mutex mu;
  bool on = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev[2];
  std::vector<cudaEvent_t> pool;
  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};
Profiler &prof() {
  static Profiler P;
  return P;
}

// Brackets one kernel launch with events when profiling is on.
struct ProfScope {
  int kind;
  cudaStream_t st;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  ProfScope(int k, cudaStream_t s) : kind(k), st(s) {
    Profiler &P = prof();
    std::lock_guard<std::mutex> g(P.mu);
    if (!P.on) return;
    e0 = P.get();
    e1 = P.get();
    cudaEventRecord(e0, st);
  }
  ~ProfScope() {
    if (!e0) return;
    cudaEventRecord(e1, st);
    Profiler &P = prof();
    std::lock_guard<std::mutex> g(P.mu);
    P.ev[kind].emplace_back(e0, e1);
  }
};

// ------------------------------------------------------------- tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 4-D TMA map of one cache, boxes of one (block, kv head) page: 16 token rows of one
// 128-byte swizzle span.  HND caches (token stride <= head stride) are described as
// (D, 16, Hkv, NB), box (span, 16, 1, 1); NHD caches (token-major within a block,
// [NB, 16, Hkv, D] seen through its [NB, Hkv, 16, D] permutation) in their own order,
// (D, Hkv, 16, NB), box (span, 1, 16, 1), which lands in shared memory as the same
// 16 x span tile.  *nhd tells the kernel which coordinate order to use.
int make_cache_map(const pa_tensor *c, CUtensorMap *map, int *nhd) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PA_ERR_CUDA;
  const int eb = elem_bytes(c->dtype);
  *nhd = c->stride[2] > c->stride[1] ? 1 : 0;
  const int mid_a = *nhd ? 1 : 2, mid_b = *nhd ? 2 : 1;  // dimension order after D
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(c->shape[3]), static_cast<cuuint64_t>(c->shape[mid_a]),
                              static_cast<cuuint64_t>(c->shape[mid_b]), static_cast<cuuint64_t>(c->shape[0])};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(c->stride[mid_a] * eb),
                                 static_cast<cuuint64_t>(c->stride[mid_b] * eb),
                                 static_cast<cuuint64_t>(c->stride[0] * eb)};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / eb), *nhd ? 1u : 16u, *nhd ? 16u : 1u, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt = eb == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  CUresult r = enc(map, dt, 4, c->data, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// 3-D TMA map of varlen queries [Tq, Hq, D] for the query-tile kernel: dims (D, Hq, Tq),
// box (64 elements, G heads, 128 / G tokens), 128-byte swizzle.  One box is 128 rows (query
// token-major, head-minor: the kernel's row order) of one 128-byte column span, the layout
// in which the kernel's MMAs read Q.  Needs G to divide 128; PA_ERR_INVALID_ARG otherwise
// (the kernel then loads Q itself).  The strides were checked 16-byte aligned by the caller.
int make_q_map(const pa_tensor *q, int G, CUtensorMap *map) {
  if (G <= 0 || 128 % G != 0) return PA_ERR_INVALID_ARG;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PA_ERR_CUDA;
  const int eb = elem_bytes(q->dtype);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(q->shape[2]), static_cast<cuuint64_t>(q->shape[1]),
                              static_cast<cuuint64_t>(q->shape[0])};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(q->stride[1] * eb), static_cast<cuuint64_t>(q->stride[0] * eb)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(G),
                             static_cast<cuuint32_t>(128 / G)};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, q->data, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// --------------------------------------------------------------- plan

int kind_of(int q_dtype, int cache_dtype) {
  if (cache_dtype == PA_FP8_E4M3) {
    if (q_dtype == PA_BF16) return KIND_FP8_BF16Q;
    if (q_dtype == PA_F16) return KIND_FP8_F16Q;
    return -1;
  }
  if (q_dtype != cache_dtype) return -1;
  if (q_dtype == PA_BF16) return KIND_BF16;
  if (q_dtype == PA_F16) return KIND_F16;
  if (q_dtype == PA_F32) return KIND_F32;
  return -1;
}

// Batches the tensor-core kernel runs longest-first (see lpt_sequence).
bool longest_first(int kind, int S) { return kind != KIND_F32 && S <= 128; }

// Resident CTAs per SM of the decode kernel for (kind, D).  With `device`, the CUDA
// occupancy calculator's answer for the current device (cached per shape); otherwise,
// or when that query fails, the shared-memory bound alone (a what-if plan for another
// GPU, or a host without one).
int ctas_per_sm(int kind, int D, bool device) {
  if (kind == KIND_F32) return 4;
  if (device) {
    static std::atomic<int> cache[5][3];
    const int di = D == 64 ? 0 : D == 128 ? 1 : 2;
    int n = cache[kind][di].load(std::memory_order_relaxed);
    if (n == 0) {
      n = (kind == KIND_BF16 || kind == KIND_F16) ? occupancy_decode_mma_16(kind, D) : occupancy_decode_mma_fp8(kind, D);
      if (n > 0) cache[kind][di].store(n, std::memory_order_relaxed);
    }
    if (n > 0) return n;
  }
  const size_t smem = mma_smem(kind, D);
  int n = static_cast<int>((227u * 1024u) / (smem + 1024));
  return std::max(1, std::min(n, 16));
}

// Partition size in tokens (0 = unsplit).  The plan cannot read seq_lens (no
// host sync), so it assumes lengths spread up to the block-table width (average
// about half of it).
//  - Batches of at most kLptMax sequences run longest-first (the kernel ranks the
//    lengths itself); when their (sequence, kv head, head group) units fill the
//    GPU's resident CTA slots at least once, that order balances the load and the
//    call does not split.  Any batch whose units fill the slots twice does not
//    split either.
//  - Otherwise the assumed work is cut into partitions of equal length, about two
//    resident waves' worth, never shorter than 64 pages (1024 tokens): below that
//    the per-CTA prologue and the partition merge cost more than the balance gains.
// Fitted on GB300 to sweeps over partition sizes for the benchmark workloads:
// 128 x 1k..8k tokens and 256 x 512..4096 run best unsplit, 64 x 1..2048 with its
// longest sequences cut in two (1024), 4 x 32k..128k near 2048 tokens.
int plan_partition(int S, int Hq, int Hkv, int D, int maxNB, int kind, int sm, bool device, int request) {
  if (request < 0) return 0;
  const int max_tokens = maxNB * kBlock;
  int P;
  if (request > 0) {
    P = (request + kBlock - 1) / kBlock * kBlock;
  } else {
    const int G = Hq / Hkv;
    const int64_t units = static_cast<int64_t>(S) * Hkv * ((G + 7) / 8);
    const int64_t slots = static_cast<int64_t>(std::max(sm, 1)) * ctas_per_sm(kind, D, device);
    if ((longest_first(kind, S) && units >= slots) || units >= 2 * slots) return 0;
    const int64_t work = units * std::max(1, maxNB / 2);  // pages, assuming half-full tables
    const int64_t pages = std::max<int64_t>(work / (2 * slots), 64);
    if (pages >= maxNB) return 0;
    P = static_cast<int>(pages * kBlock);
  }
  if (P >= max_tokens) return 0;
  return P;
}

// The full plan: fixed-size partitions (P tokens, merged through the workspace by the
// last-arriving CTA), the balanced split (request PA_PARTITION_BALANCED: one resident
// wave of CTAs per head row, each taking an equal share of the batch's pages), or, on
// request only (-2, -4 or -8), a cluster split: each unit cut into C equal parts whose
// CTAs form one thread-block cluster and merge through distributed shared memory, with
// no workspace.  The heuristic does not pick the cluster split: cutting every unit
// (short ones too) multiplies the CTAs beyond the resident slots, and on GB300 that
// cost more than the shorter critical path saved (64 x 1..2048 tokens: 33.2 us
// unsplit, 34.3 / 42.1 / 56.1 us for C = 2 / 4 / 8, 32.9 us with 1024-token partitions).
struct Plan {
  int P;        // tokens per fixed partition (0 = none)
  int cluster;  // parts per unit of the cluster split (0 = none)
  int flat;     // CTAs per head row of the balanced split (0 = none)
  int status;
};
int balanced_ctas(int Hq, int Hkv, int D, int kind, int sm, bool device) {
  const int64_t rows = static_cast<int64_t>(Hkv) * ((Hq / Hkv + 7) / 8);
  const int64_t slots = static_cast<int64_t>(std::max(sm, 1)) * ctas_per_sm(kind, D, device);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(slots / rows, 65535)));
}
Plan make_plan(int S, int Hq, int Hkv, int D, int maxNB, int kind, int sm, bool device, int request) {
  Plan pl{0, 0, 0, PA_OK};
  if (request == PA_PARTITION_BALANCED) {
    if (kind == KIND_F32) return pl;  // the CUDA-core kernel runs it unsplit
    if (S > kFlatMaxSeqs) pl.status = PA_ERR_UNSUPPORTED_SHAPE;
    else pl.flat = balanced_ctas(Hq, Hkv, D, kind, sm, device);
    return pl;
  }
  if (request <= -2) {
    const int C = -request;
    if (C != 2 && C != 4 && C != 8) pl.status = PA_ERR_INVALID_ARG;
    else pl.cluster = C;
    return pl;
  }
  pl.P = plan_partition(S, Hq, Hkv, D, maxNB, kind, sm, device, request);
  return pl;
}

// Split-KV workspace: [arrival counters, one int per (sequence, kv head, head group)]
// [partial (m, l): one float2 per row] [partial acc: D floats per row], each region
// starting on a 256-byte boundary.  Rows: one per (sequence, head, partition) for
// fixed-size partitions; 2 x 8 per CTA for the balanced split (`flat` CTAs per head row).
struct WsLayout {
  size_t ml_off, acc_off, total;
};
size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
WsLayout workspace_layout(int S, int Hq, int Hkv, int D, int maxNB, int P, int flat) {
  WsLayout L{0, 0, 0};
  if (P <= 0 && flat <= 0) return L;
  const int64_t head_rows = static_cast<int64_t>(Hkv) * ((Hq / Hkv + 7) / 8);
  const int64_t rows = flat > 0 ? head_rows * flat * 16
                                : static_cast<int64_t>(S) * Hq * ((static_cast<int64_t>(maxNB) * kBlock + P - 1) / P);
  const int64_t units = static_cast<int64_t>(S) * head_rows;
  L.ml_off = round256(static_cast<size_t>(units) * sizeof(int));
  L.acc_off = L.ml_off + round256(static_cast<size_t>(rows) * sizeof(float2));
  L.total = L.acc_off + static_cast<size_t>(rows) * D * sizeof(float);
  return L;
}

// ------------------------------------------------------ internal workspace

struct DevWorkspace {
  void *ptr = nullptr;
  size_t bytes = 0;
};
std::mutex g_ws_mu;
DevWorkspace g_ws[64];

// ------------------------------------------------------------- validation

int validate_cache_pair(const pa_tensor *kc, const pa_tensor *vc, int *NB, int *Hkv, int *D) {
  int r;
  if ((r = check_desc(kc, 4)) || (r = check_desc(vc, 4))) return r;
  for (int i = 0; i < 4; ++i)
    if (kc->shape[i] != vc->shape[i]) return PA_ERR_INVALID_ARG;
  if (kc->dtype != vc->dtype) return PA_ERR_INVALID_ARG;
  if (kc->shape[2] != kBlock) return PA_ERR_UNSUPPORTED_SHAPE;
  if (kc->stride[3] != 1 || vc->stride[3] != 1) return PA_ERR_INVALID_ARG;
  if (!kc->data || !vc->data) return PA_ERR_INVALID_ARG;
  const int eb = elem_bytes(kc->dtype);
  if (!aligned16(kc->data) || !aligned16(vc->data)) return PA_ERR_ALIGNMENT;
  for (int i = 0; i < 3; ++i)
    if ((kc->stride[i] * eb) % 16 || (vc->stride[i] * eb) % 16) return PA_ERR_ALIGNMENT;
  if (kc->shape[0] > INT32_MAX || kc->shape[1] > 65535) return PA_ERR_UNSUPPORTED_SHAPE;
  *NB = static_cast<int>(kc->shape[0]);
  *Hkv = static_cast<int>(kc->shape[1]);
  *D = static_cast<int>(kc->shape[3]);
  return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

// ===================================================================== ABI

PA_API const char *pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED_DTYPE: return "unsupported element type";
    case PA_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_CUDA: return "CUDA call or launch failed";
    case PA_ERR_DEVICE_BOUNDS: return "device reported an out-of-range slot, block id or sequence length";
    case PA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (block size, head size or extent)";
    case PA_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case PA_ERR_NO_BLOCKS: return "block pool has too few free blocks";
    default: return "unknown status";
  }
}

// The write with its grid's CTAs per SM (0: the standalone choice; pa_decode_step asks for
// fewer when the decode's early reads overlap it).
static int write_impl(const pa_tensor *key, const pa_tensor *value, pa_tensor *k_cache, pa_tensor *v_cache,
                      const pa_tensor *slot_mapping, int kv_dtype, const pa_write_options *opt, pa_stream_t stream,
                      int ctas_per_sm) {
  const pa_write_options o = opt ? *opt : pa_write_options{};
  if (o.scale_stride < 0) return PA_ERR_INVALID_ARG;
  int r;
  if ((r = check_desc(key, 3)) || (r = check_desc(value, 3)) || (r = check_desc(slot_mapping, 1))) return r;
  int NB, Hkv, D;
  if ((r = validate_cache_pair(k_cache, v_cache, &NB, &Hkv, &D))) return r;
  const int in_dt = key->dtype;
  if (value->dtype != in_dt) return PA_ERR_INVALID_ARG;
  if (in_dt != PA_F32 && in_dt != PA_BF16 && in_dt != PA_F16) return PA_ERR_UNSUPPORTED_DTYPE;
  if (slot_mapping->dtype != PA_I64) return PA_ERR_UNSUPPORTED_DTYPE;
  if (kv_dtype == PA_KV_AUTO) {
    if (k_cache->dtype != in_dt) return PA_ERR_UNSUPPORTED_DTYPE;
  } else if (kv_dtype == PA_KV_FP8_E4M3) {
    if (k_cache->dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED_DTYPE;
  } else {
    return PA_ERR_INVALID_ARG;
  }
  const int64_t T = key->shape[0];
  if (value->shape[0] != T || slot_mapping->shape[0] != T) return PA_ERR_INVALID_ARG;
  if (key->shape[1] != Hkv || key->shape[2] != D || value->shape[1] != Hkv || value->shape[2] != D)
    return PA_ERR_INVALID_ARG;
  if (key->stride[2] != 1 || value->stride[2] != 1 || slot_mapping->stride[0] != 1) return PA_ERR_INVALID_ARG;
  const int ib = elem_bytes(in_dt);
  if ((static_cast<int64_t>(D) * ib) % 16) return PA_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return PA_OK;
  if (!key->data || !value->data || !slot_mapping->data) return PA_ERR_INVALID_ARG;
  if (!aligned16(key->data) || !aligned16(value->data)) return PA_ERR_ALIGNMENT;
  for (int i = 0; i < 2; ++i)
    if ((key->stride[i] * ib) % 16 || (value->stride[i] * ib) % 16) return PA_ERR_ALIGNMENT;

  WriteParams p;
  p.key = key->data;
  p.value = value->data;
  p.k_cache = k_cache->data;
  p.v_cache = v_cache->data;
  p.slot_mapping = static_cast<const int64_t *>(slot_mapping->data);
  p.T = T;
  p.Hkv = Hkv;
  p.D = D;
  p.key_ts = key->stride[0];
  p.key_hs = key->stride[1];
  p.val_ts = value->stride[0];
  p.val_hs = value->stride[1];
  p.kc_s0 = k_cache->stride[0];
  p.kc_s1 = k_cache->stride[1];
  p.kc_s2 = k_cache->stride[2];
  p.vc_s0 = v_cache->stride[0];
  p.vc_s1 = v_cache->stride[1];
  p.vc_s2 = v_cache->stride[2];
  p.num_slots = static_cast<int64_t>(NB) * kBlock;
  p.k_scale = kv_dtype == PA_KV_FP8_E4M3 ? o.k_scale : nullptr;
  p.v_scale = kv_dtype == PA_KV_FP8_E4M3 ? o.v_scale : nullptr;
  p.scale_stride = o.scale_stride;
  p.err = o.device_error;
  {
    // 32-bit index arithmetic when every byte offset the kernel forms stays below 2^31: the
    // source rows (first to last element), the cache's block and token strides and the
    // extent of one block (the block offset itself is one widening multiply)
    const int64_t lim = INT32_MAX;
    const int cb = elem_bytes(k_cache->dtype);
    auto span = [&](const pa_tensor *t) { return ((T - 1) * t->stride[0] + (Hkv - 1) * t->stride[1] + D) * ib; };
    auto inner = [&](const pa_tensor *c) { return ((Hkv - 1) * c->stride[1] + (kBlock - 1) * c->stride[2] + D) * cb; };
    p.i32 = T <= lim && span(key) <= lim && span(value) <= lim && k_cache->stride[0] * cb <= lim &&
            v_cache->stride[0] * cb <= lim && inner(k_cache) <= lim && inner(v_cache) <= lim;
  }
  const int sm = device_sm_count();
  if (sm <= 0) return PA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  {
    ProfScope ps(PA_KERNEL_WRITE, st);
    e = launch_write(p, in_dt, k_cache->dtype, sm, ctas_per_sm, st);
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API int pa_reshape_and_cache_opt(const pa_tensor *key, const pa_tensor *value, pa_tensor *k_cache,
                                    pa_tensor *v_cache, const pa_tensor *slot_mapping, int kv_dtype,
                                    const pa_write_options *opt, pa_stream_t stream) {
  return write_impl(key, value, k_cache, v_cache, slot_mapping, kv_dtype, opt, stream, 0);
}

PA_API int pa_reshape_and_cache(const pa_tensor *key, const pa_tensor *value, pa_tensor *k_cache, pa_tensor *v_cache,
                                const pa_tensor *slot_mapping, int kv_dtype, const float *k_scale,
                                const float *v_scale, int *device_error, pa_stream_t stream) {
  pa_write_options o{};
  o.k_scale = k_scale;
  o.v_scale = v_scale;
  o.device_error = device_error;
  return pa_reshape_and_cache_opt(key, value, k_cache, v_cache, slot_mapping, kv_dtype, &o, stream);
}

PA_API int pa_decode_plan(int num_seqs, int num_heads, int num_kv_heads, int head_size, int max_blocks_per_seq,
                          int kv_dtype_code, int sm_count, int partition_size, int *partition_out,
                          int *num_partitions_out) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || head_size <= 0 ||
      max_blocks_per_seq < 0)
    return PA_ERR_INVALID_ARG;
  int kind;
  switch (kv_dtype_code) {
    case PA_FP8_E4M3: kind = KIND_FP8_BF16Q; break;
    case PA_BF16: kind = KIND_BF16; break;
    case PA_F16: kind = KIND_F16; break;
    case PA_F32: kind = KIND_F32; break;
    default: return PA_ERR_INVALID_ARG;
  }
  const bool device = sm_count <= 0;
  if (device) sm_count = device_sm_count();
  if (sm_count <= 0) return PA_ERR_CUDA;
  const Plan pl = make_plan(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq, kind, sm_count, device,
                            partition_size);
  if (pl.status != PA_OK) return pl.status;
  if (partition_out) *partition_out = pl.flat > 0 ? PA_PARTITION_BALANCED : pl.cluster > 1 ? -pl.cluster : pl.P;
  if (num_partitions_out)
    *num_partitions_out = pl.flat > 0       ? pl.flat
                          : pl.cluster > 1 ? pl.cluster
                          : pl.P > 0       ? (max_blocks_per_seq * kBlock + pl.P - 1) / pl.P
                                           : 1;
  return PA_OK;
}

PA_API size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                       int max_blocks_per_seq, int partition_size) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || head_size < 0 ||
      max_blocks_per_seq < 0)
    return 0;
  if (partition_size == PA_PARTITION_BALANCED) {
    // enough for any cache type on the current device: the E4M3 kernel's shared-memory
    // bound admits the most CTAs per SM
    const int sm = device_sm_count();
    if (sm <= 0 || num_seqs > kFlatMaxSeqs) return 0;
    const int kind = head_size >= 128 ? KIND_FP8_BF16Q : KIND_BF16;
    const int flat = balanced_ctas(num_heads, num_kv_heads, head_size, kind, sm, false);
    return workspace_layout(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq, 0, flat).total;
  }
  const int P = partition_size > 0 ? (partition_size + kBlock - 1) / kBlock * kBlock : 0;
  if (P >= max_blocks_per_seq * kBlock) return 0;
  return workspace_layout(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq, P, 0).total;
}

namespace {

// Decode (query_start_loc == NULL: one query token per sequence, q [S, Hq, D]) or varlen
// attention (q [Tq, Hq, D] packed, query_start_loc [S + 1], at most max_query_len tokens
// per sequence).
int decode_impl(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
                const pa_tensor *block_table, const pa_tensor *seq_lens, float scale, int num_kv_heads,
                const pa_decode_options &o, bool internal_ws, pa_stream_t stream,
                const pa_tensor *query_start_loc = nullptr, int max_query_len = 1,
                const pa_tensor *new_rows_start = nullptr, bool early = false, bool dry = false,
                size_t *ws_need = nullptr, size_t *ws_counters = nullptr) {
  const float *k_scale = o.k_scale, *v_scale = o.v_scale;
  const int partition_size = o.partition_size;
  void *workspace = o.workspace;
  size_t workspace_bytes = o.workspace_bytes;
  int *device_error = o.device_error;
  if (o.scale_stride < 0) return PA_ERR_INVALID_ARG;
  int r;
  if ((r = check_desc(out, 3)) || (r = check_desc(q, 3)) || (r = check_desc(block_table, 2)) ||
      (r = check_desc(seq_lens, 1)))
    return r;
  int NB, Hkv, D;
  if ((r = validate_cache_pair(k_cache, v_cache, &NB, &Hkv, &D))) return r;
  const bool varlen = query_start_loc != nullptr;
  const int64_t S64 = varlen ? seq_lens->shape[0] : q->shape[0], Hq64 = q->shape[1];
  if (num_kv_heads != Hkv || Hkv <= 0 || Hq64 <= 0 || Hq64 % Hkv) return PA_ERR_INVALID_ARG;
  if (varlen) {
    if ((r = check_desc(query_start_loc, 1))) return r;
    if (query_start_loc->dtype != PA_I32) return PA_ERR_UNSUPPORTED_DTYPE;
    if (query_start_loc->shape[0] != S64 + 1 || query_start_loc->stride[0] != 1 || !query_start_loc->data)
      return PA_ERR_INVALID_ARG;
    if (max_query_len < 1) return PA_ERR_INVALID_ARG;
    if (o.partition_size == PA_PARTITION_BALANCED) return PA_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(max_query_len) * (Hq64 / Hkv) > (1 << 20)) return PA_ERR_UNSUPPORTED_SHAPE;
  }
  if (q->shape[2] != D) return PA_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i)
    if (out->shape[i] != q->shape[i]) return PA_ERR_INVALID_ARG;
  if (out->dtype != q->dtype) return PA_ERR_INVALID_ARG;
  if (block_table->dtype != PA_I32 || seq_lens->dtype != PA_I32) return PA_ERR_UNSUPPORTED_DTYPE;
  if (block_table->shape[0] != S64 || seq_lens->shape[0] != S64) return PA_ERR_INVALID_ARG;
  if (block_table->stride[1] != 1 || seq_lens->stride[0] != 1 || q->stride[2] != 1 || out->stride[2] != 1)
    return PA_ERR_INVALID_ARG;
  const int kind = kind_of(q->dtype, k_cache->dtype);
  if (kind < 0) return PA_ERR_UNSUPPORTED_DTYPE;
  if (D != 64 && D != 128 && D != 256) return PA_ERR_UNSUPPORTED_SHAPE;
  if ((kind == KIND_FP8_BF16Q || kind == KIND_FP8_F16Q) && D < 128) return PA_ERR_UNSUPPORTED_SHAPE;
  if (S64 > 65535 || Hq64 > 65535 || block_table->shape[1] > (INT32_MAX / kBlock)) return PA_ERR_UNSUPPORTED_SHAPE;
  if (early && new_rows_start) {
    if ((r = check_desc(new_rows_start, 1))) return r;
    if (new_rows_start->dtype != PA_I32) return PA_ERR_UNSUPPORTED_DTYPE;
    if (new_rows_start->shape[0] != S64 + 1 || new_rows_start->stride[0] != 1) return PA_ERR_INVALID_ARG;
    if (S64 > 0 && !new_rows_start->data) return PA_ERR_INVALID_ARG;
  }
  if (S64 == 0 || q->shape[0] == 0) return PA_OK;
  if (!q->data || !out->data || !block_table->data || !seq_lens->data) return PA_ERR_INVALID_ARG;
  const int qb = elem_bytes(q->dtype);
  if (!aligned16(q->data) || !aligned16(out->data)) return PA_ERR_ALIGNMENT;
  for (int i = 0; i < 2; ++i)
    if ((q->stride[i] * qb) % 16 || (out->stride[i] * qb) % 16) return PA_ERR_ALIGNMENT;

  const int S = static_cast<int>(S64), Hq = static_cast<int>(Hq64);
  // query columns per KV head ("virtual heads"): G for decode, G per query token for varlen;
  // plans and workspace count them like query heads
  const int VH = (Hq / Hkv) * (varlen ? max_query_len : 1);
  const int Hqv = Hkv * VH;
  const int maxNB = static_cast<int>(block_table->shape[1]);
  const int sm = device_sm_count();
  if (sm <= 0) return PA_ERR_CUDA;
  // Chunks of query tokens run on the query-tile kernel (rows in the MMA M dimension, pages
  // shared by 64 rows, no split) unless a split was asked for.
  const bool chunk = varlen && (kind == KIND_BF16 || kind == KIND_F16) && (D == 64 || D == 128) &&
                     (partition_size == 0 || partition_size == -1) && VH >= chunk_min_columns(D);
  const Plan pl = make_plan(S, Hqv, Hkv, D, maxNB, kind, sm, true, chunk ? -1 : partition_size);
  if (pl.status != PA_OK) return pl.status;
  const int P = pl.P;
  const int max_parts = pl.cluster > 1 ? pl.cluster : P > 0 ? (maxNB * kBlock + P - 1) / P : 1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  DecodeParams p{};
  p.out = out->data;
  p.q = q->data;
  p.out_ss = out->stride[0];
  p.out_hs = out->stride[1];
  p.q_ss = q->stride[0];
  p.q_hs = q->stride[1];
  p.block_table = static_cast<const int32_t *>(block_table->data);
  p.bt_ss = block_table->stride[0];
  p.seq_lens = static_cast<const int32_t *>(seq_lens->data);
  p.S = S;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.VH = VH;
  p.HG = (VH + 7) / 8;
  p.qsl = varlen ? static_cast<const int32_t *>(query_start_loc->data) : nullptr;
  p.nq_max = varlen ? max_query_len : 1;
  p.Tq = q->shape[0];
  p.D = D;
  p.num_blocks = NB;
  p.max_blocks = maxNB;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.scale_stride = o.scale_stride;
  p.alibi = o.alibi_slopes;
  p.pages_per_part = P > 0 ? P / kBlock : std::max(maxNB, 1);
  p.max_parts = max_parts;
  p.cluster = pl.cluster;
  p.flat = pl.flat;
  p.first_wait_limit = o.first_wait_limit;
  p.early = early && !varlen ? 1 : 0;
  p.new_start = p.early && new_rows_start ? static_cast<const int32_t *>(new_rows_start->data) : nullptr;
  p.err = device_error;
  {
    // Order the batch longest-first only when its CTAs cannot all be resident at once:
    // with every CTA resident from the start the order buys nothing and the ranking
    // (a read of every length plus two block barriers) sits on each CTA's critical path.
    const int64_t ctas = static_cast<int64_t>(S) * Hkv * p.HG * max_parts;
    p.lpt = (pl.flat == 0 && longest_first(kind, S) && ctas > static_cast<int64_t>(sm) * ctas_per_sm(kind, D, true))
                ? 1
                : 0;
  }
  if (kind != KIND_FP8_BF16Q && kind != KIND_FP8_F16Q) p.k_scale = p.v_scale = nullptr;
  if (static_cast<int64_t>(p.Hkv) * p.HG > 65535) return PA_ERR_UNSUPPORTED_SHAPE;

  if (dry) {  // validation only (pa_decode_step checks everything before its first launch)
    if ((max_parts > 1 && pl.cluster <= 1) || pl.flat > 0) {
      const WsLayout lay = workspace_layout(S, Hqv, Hkv, D, maxNB, P, pl.flat);
      if (ws_need) *ws_need = lay.total;
      if (ws_counters) *ws_counters = lay.ml_off;
      if (!internal_ws) {
        if (!workspace || workspace_bytes < lay.total) return PA_ERR_WORKSPACE;
        if (!aligned16(workspace)) return PA_ERR_ALIGNMENT;
      }
    }
    return PA_OK;
  }
  if ((max_parts > 1 && pl.cluster <= 1) || pl.flat > 0) {
    const WsLayout lay = workspace_layout(S, Hqv, Hkv, D, maxNB, P, pl.flat);
    if (internal_ws) {
      int dev = 0;
      if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
      std::lock_guard<std::mutex> g(g_ws_mu);
      DevWorkspace &w = g_ws[dev];
      if (w.bytes < lay.total) {
        if (w.ptr) cudaFreeAsync(w.ptr, st);
        w.ptr = nullptr;
        w.bytes = 0;
        if (cudaMallocAsync(&w.ptr, lay.total, st) != cudaSuccess) return PA_ERR_CUDA;
        if (cudaMemsetAsync(w.ptr, 0, lay.total, st) != cudaSuccess) return PA_ERR_CUDA;
        w.bytes = lay.total;
      }
      workspace = w.ptr;
      workspace_bytes = w.bytes;
    }
    if (!workspace || workspace_bytes < lay.total) return PA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PA_ERR_ALIGNMENT;
    p.counters = static_cast<int *>(workspace);
    p.part_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) + lay.ml_off);
    p.part_acc = reinterpret_cast<float *>(static_cast<char *>(workspace) + lay.acc_off);
  }

  cudaError_t e;
  if (kind == KIND_F32) {
    p.kc = static_cast<const float *>(k_cache->data);
    p.vc = static_cast<const float *>(v_cache->data);
    p.kc_s0 = k_cache->stride[0];
    p.kc_s1 = k_cache->stride[1];
    p.kc_s2 = k_cache->stride[2];
    p.vc_s0 = v_cache->stride[0];
    p.vc_s1 = v_cache->stride[1];
    p.vc_s2 = v_cache->stride[2];
    ProfScope ps(PA_KERNEL_DECODE, st);
    e = launch_decode_f32(p, st);
  } else {
    CUtensorMap tmK, tmV;
    int nhd_k = 0, nhd_v = 0;
    if ((r = make_cache_map(k_cache, &tmK, &nhd_k)) || (r = make_cache_map(v_cache, &tmV, &nhd_v))) return r;
    if (nhd_k != nhd_v) return PA_ERR_INVALID_ARG;  // K and V in different layouts
    p.nhd = nhd_k;
    ProfScope ps(PA_KERNEL_DECODE, st);
    if (chunk) {
      CUtensorMap tmQ{};
      p.q_tma = make_q_map(q, p.G, &tmQ) == PA_OK ? 1 : 0;
      e = launch_chunk_umma(p, kind, tmK, tmV, tmQ, st);
    } else if (kind == KIND_BF16 || kind == KIND_F16) {
      e = launch_decode_mma_16(p, kind, tmK, tmV, st);
    } else {
      e = launch_decode_mma_fp8(p, kind, tmK, tmV, st);
    }
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

int pa::decode_ex_requirements(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
                           const pa_tensor *block_table, const pa_tensor *seq_lens, float scale, int num_kv_heads,
                           const float *k_scale, const float *v_scale, int partition_size, int *device_error,
                           size_t *ws_bytes, size_t *counter_bytes) {
  pa_decode_options o{};
  o.k_scale = k_scale;
  o.v_scale = v_scale;
  o.partition_size = partition_size;
  o.device_error = device_error;
  *ws_bytes = 0;
  *counter_bytes = 0;
  // internal_ws: the workspace is not checked here (the caller supplies it afterwards)
  return decode_impl(out, q, k_cache, v_cache, block_table, seq_lens, scale, num_kv_heads, o, true, nullptr,
                     nullptr, 1, nullptr, false, true, ws_bytes, counter_bytes);
}

PA_API int pa_decode_ex(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
                        const pa_tensor *block_table, const pa_tensor *seq_lens, float scale, int num_kv_heads,
                        const float *k_scale, const float *v_scale, int partition_size, void *workspace,
                        size_t workspace_bytes, int *device_error, pa_stream_t stream) {
  pa_decode_options o{};
  o.k_scale = k_scale;
  o.v_scale = v_scale;
  o.partition_size = partition_size;
  o.workspace = workspace;
  o.workspace_bytes = workspace_bytes;
  o.device_error = device_error;
  return decode_impl(out, q, k_cache, v_cache, block_table, seq_lens, scale, num_kv_heads, o, false, stream);
}

PA_API int pa_decode(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
                     const pa_tensor *block_table, const pa_tensor *seq_lens, float scale, int num_kv_heads,
                     pa_stream_t stream) {
  const pa_decode_options o{};
  return decode_impl(out, q, k_cache, v_cache, block_table, seq_lens, scale, num_kv_heads, o, true, stream);
}

PA_API int pa_decode_opt(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
                         const pa_tensor *block_table, const pa_tensor *seq_lens, float scale, int num_kv_heads,
                         const pa_decode_options *opt, pa_stream_t stream) {
  const pa_decode_options o = opt ? *opt : pa_decode_options{};
  const bool internal = !o.workspace && o.workspace_bytes == 0;
  return decode_impl(out, q, k_cache, v_cache, block_table, seq_lens, scale, num_kv_heads, o, internal, stream);
}

PA_API int pa_attention_varlen(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache, const pa_tensor *v_cache,
                               const pa_tensor *query_start_loc, const pa_tensor *block_table,
                               const pa_tensor *seq_lens, float scale, int num_kv_heads, int max_query_len,
                               const pa_decode_options *opt, pa_stream_t stream) {
  if (!query_start_loc) return PA_ERR_INVALID_ARG;
  const pa_decode_options o = opt ? *opt : pa_decode_options{};
  const bool internal = !o.workspace && o.workspace_bytes == 0;
  return decode_impl(out, q, k_cache, v_cache, block_table, seq_lens, scale, num_kv_heads, o, internal, stream,
                     query_start_loc, max_query_len);
}

PA_API int pa_decode_step(pa_tensor *out, const pa_tensor *q, const pa_tensor *key, const pa_tensor *value,
                          pa_tensor *k_cache, pa_tensor *v_cache, const pa_tensor *slot_mapping,
                          const pa_tensor *new_rows_start, const pa_tensor *block_table, const pa_tensor *seq_lens,
                          float scale, int num_kv_heads, const pa_decode_options *opt, pa_stream_t stream) {
  const pa_decode_options o = opt ? *opt : pa_decode_options{};
  const bool internal = !o.workspace && o.workspace_bytes == 0;
  int r;
  if ((r = check_desc(q, 3)) || (r = check_desc(key, 3)) || (r = check_desc(k_cache, 4))) return r;
  if (!new_rows_start && key->shape[0] != q->shape[0]) return PA_ERR_INVALID_ARG;  // one new row per sequence
  if (new_rows_start && ((r = check_desc(new_rows_start, 1)) || new_rows_start->shape[0] != q->shape[0] + 1))
    return r ? r : PA_ERR_INVALID_ARG;
  // every argument of both halves is checked before anything is launched
  if ((r = decode_impl(out, q, k_cache, v_cache, block_table, seq_lens, scale, num_kv_heads, o, internal, stream,
                       nullptr, 1, new_rows_start, true, true)))
    return r;
  const pa_write_options wo{o.k_scale, o.v_scale, o.scale_stride, o.device_error};
  const int kv = k_cache->dtype == PA_FP8_E4M3 ? PA_KV_FP8_E4M3 : PA_KV_AUTO;
  // Early reads pay when the write is long (several new rows per sequence: measured 202.8 ->
  // 198.7 us on 128 sequences x 64 rows into an E4M3 cache); a one-row write is over before
  // they help, and the early variant's in-loop wait costs more (c2: 33.3 vs 33.5 us).  With
  // early reads the write takes two CTAs per SM, leaving the decode's CTAs room beside it
  // (same step, graph replay: 4 / 3 / 2 / 1 write CTAs per SM 195.5 / 192.7 / 191.0 / 194.9 us).
  const int write_ctas = new_rows_start ? 2 : 0;
  if ((r = write_impl(key, value, k_cache, v_cache, slot_mapping, kv, &wo, stream, write_ctas))) return r;
  return decode_impl(out, q, k_cache, v_cache, block_table, seq_lens, scale, num_kv_heads, o, internal, stream,
                     nullptr, 1, new_rows_start, new_rows_start != nullptr);
}

PA_API int pa_check_device_error(int *device_error, int *bits_out, pa_stream_t stream) {
  if (!device_error) return PA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int bits = 0;
  if (cudaMemcpyAsync(&bits, device_error, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(device_error, 0, sizeof(int), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return PA_ERR_CUDA;
  if (bits_out) *bits_out = bits;
  if (bits & (PA_DEVERR_SLOT_RANGE | PA_DEVERR_BLOCK_RANGE | PA_DEVERR_SEQLEN_RANGE)) return PA_ERR_DEVICE_BOUNDS;
  if (bits & PA_DEVERR_WAIT_TIMEOUT) return PA_ERR_DEVICE_TIMEOUT;
  return PA_OK;
}

PA_API int pa_profile_enable(int on) {
  Profiler &P = prof();
  std::lock_guard<std::mutex> g(P.mu);
  P.on = on != 0;
  return PA_OK;
}

PA_API int pa_profile_read(int kind, double *total_ms, long long *launches) {
  if (kind < 0 || kind > 1) return PA_ERR_INVALID_ARG;
  Profiler &P = prof();
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev;
  {
    std::lock_guard<std::mutex> g(P.mu);
    ev.swap(P.ev[kind]);
  }
  double ms = 0.0;
  int rc = PA_OK;
  for (auto &pr : ev) {
    float t = 0.f;
    if (cudaEventSynchronize(pr.second) != cudaSuccess || cudaEventElapsedTime(&t, pr.first, pr.second) != cudaSuccess)
      rc = PA_ERR_CUDA;
    ms += t;
  }
  {
    std::lock_guard<std::mutex> g(P.mu);
    for (auto &pr : ev) {
      P.pool.push_back(pr.first);
      P.pool.push_back(pr.second);
    }
  }
  if (total_ms) *total_ms = ms;
  if (launches) *launches = static_cast<long long>(ev.size());
  return rc;
}
