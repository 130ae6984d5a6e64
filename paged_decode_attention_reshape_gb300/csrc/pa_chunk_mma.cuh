// pa_chunk_mma.cuh -- paged attention for chunks of query tokens (chunked prefill, long
// speculative windows) with the query rows in the tensor-core M dimension.
//
// What it computes is pa_attention_varlen's definition ("Inside vLLM CUDA Kernels",
// Part 3, FlashAttention over paged KV: a CTA owns a Q tile, resolves and loads the K/V
// tiles of its sequence through block_table while scanning the K dimension, and runs
// QK, online softmax and P.V on each): query i of a sequence with n new tokens sits at
// position len - n + i and sees the tokens up to it; the logit is scale q.k (+ the ALiBi
// bias slope_h (t - position)).
//
// Work unit (one CTA): sequence s, KV head g, and 64 query rows -- row r of the KV head
// is query token r / G at head g G + r % G -- 16 rows per warp.  All 4 warps consume
// every K/V page of the rows' visible range from one shared ring of R stage slots: warp
// 0 lane 0 resolves the physical block and issues the two TMA page loads (the same 4-D
// maps and 128-byte swizzle as the decode kernels) into the next slot once all warps
// have released it (an "empty" mbarrier with 4 arrivals); every warp waits on the slot's
// "full" mbarrier (bounded waits throughout).  Per page and warp:
//   S[16 rows x 16 tok] = Q[16 x D] . K_page^T      (mma m16n8k16, two n8 token tiles;
//                                                    K fragments by ldmatrix of the rows)
//   online softmax per row (log2 domain, the lazy running max of the decode kernels),
//   causal / length masking per row, the quad of lanes holding a row reducing it;
//   O[16 x D] += P[16 x 16] . V_page[16 x D]        (P taken from the S accumulators as
//                                                    hi + lo 16-bit A fragments; V by
//                                                    ldmatrix.trans, tail tokens zeroed)
// The outputs are written once at the end (no split of the page range).
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_merge.cuh"

namespace pa {

constexpr uint32_t kChunkWaitLimit = 1u << 20;  // mbarrier polls before a wait gives up
constexpr float kChunkSlack = 8.f;              // lazy running max, log2 units (p <= 256)
constexpr float kChunkEmpty = -1e30f;           // running max of a row with no visible token yet

template <int KIND, int D>
struct ChunkCfg {
  static constexpr bool BF = KIND == KIND_BF16;
  static constexpr int W = 4, THREADS = W * 32, ROWS = 16 * W;
  static constexpr int ROWB = D * 2;            // bytes of one token row of a page
  static constexpr int NBOX = ROWB / 128;       // 128-byte TMA boxes across a row
  static constexpr int BOXE = 64;               // elements per box row
  static constexpr int PAGEB = kBlock * ROWB;   // one (block, kv head) page
  static constexpr int STAGEB = 2 * PAGEB;      // K page + V page
  static constexpr int KT = D / 16;             // k-steps of Q.K^T
  static constexpr int NT = D / 8;              // n8 tiles of the output
  static constexpr int R = D == 64 ? 12 : 8;    // ring slots (48 / 64 KiB)
  static constexpr size_t BAR_OFF = static_cast<size_t>(R) * STAGEB;
  static constexpr size_t SMEM = 1024 + BAR_OFF + R * 16;
  static_assert(ROWB % 128 == 0, "page rows must be whole 128-byte swizzle spans");
};

template <int KIND, int D>
__global__ void __launch_bounds__(128) chunk_mma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK,
                                                        const __grid_constant__ CUtensorMap tmV) {
  using C = ChunkCfg<KIND, D>;
  using OutT = typename std::conditional<C::BF, __nv_bfloat16, __half>::type;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;  // 128B-swizzle boxes need 1 KiB alignment
  const uint32_t full0 = sbase + static_cast<uint32_t>(C::BAR_OFF), empty0 = full0 + C::R * 8;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rt = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int G = p.G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::R; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, C::W);
    }
    fence_barrier_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_l2(p.seq_lens + s);
    prefetch_l2(p.qsl + s);
  }
  __syncthreads();
  grid_dependency_wait();

  const int len = __ldg(p.seq_lens + s);
  const int a = __ldg(p.qsl + s), b = __ldg(p.qsl + s + 1);
  const int nq = b - a;
  if (len < 0 || len > p.max_blocks * kBlock || a < 0 || b > p.Tq || nq < 0 || nq > p.nq_max || nq > len) {
    if (threadIdx.x == 0 && rt == 0 && g == 0 && p.err) atomicOr(p.err, kErrSeqLen);
    return;
  }
  const int r0 = rt * C::ROWS;                       // first row of the CTA
  const int nrows = min(C::ROWS, nq * G - r0);       // rows with a query token
  if (nrows <= 0) return;
  const int pos0 = len - nq;                         // row r sees tokens 0 .. pos0 + r / G
  const int vis = pos0 + (r0 + nrows - 1) / G + 1;
  const int npages = (vis + kBlock - 1) / kBlock;
  const int32_t *bt = p.block_table + static_cast<int64_t>(s) * p.bt_ss;
  const uint64_t pol = policy_evict_first();

  bool bad = false, stalled = false;
  // ----------------------------------------------------------------- producer
  int pid_reg = 0;  // warp 0, lane i: physical block of page 32 c + i for the current chunk c
  int issued = 0;   // warp 0: pages issued so far
  auto issue = [&](int k) {  // warp 0, whole
    ++issued;
    if ((k & 31) == 0) {
      const int kk = k + lane;
      pid_reg = kk < npages ? __ldg(bt + kk) : 0;
    }
    int pid = __shfl_sync(0xffffffffu, pid_reg, k & 31);
    if (pid < 0 || pid >= p.num_blocks) {
      bad = true;
      if (lane == 0 && p.err) atomicOr(p.err, kErrBlock);
      pid = 0;  // load a valid block; the CTA writes nothing
    }
    if (lane == 0) {
      const int st = k % C::R;
      const uint32_t bar = full0 + 8 * st, dst = sbase + st * C::STAGEB;
      mbar_arrive_expect_tx(bar, C::STAGEB);
      const int c1 = p.nhd ? g : 0, c2 = p.nhd ? 0 : g;
#pragma unroll
      for (int bx = 0; bx < C::NBOX; ++bx) tma_load_4d(dst + bx * 2048, &tmK, bar, bx * C::BOXE, c1, c2, pid, pol);
#pragma unroll
      for (int bx = 0; bx < C::NBOX; ++bx)
        tma_load_4d(dst + C::PAGEB + bx * 2048, &tmV, bar, bx * C::BOXE, c1, c2, pid, pol);
    }
  };
  if (warp == 0)
    for (int k = 0; k < min(C::R, npages); ++k) issue(k);

  // ------------------------------------------------------- query fragments
  // A fragment of m16n8k16: rows g8 = lane / 4 and g8 + 8 of the warp's 16, k columns
  // 2 c4, 2 c4 + 1 (+ 8) of each 16-wide step, c4 = lane % 4.
  const int g8 = lane >> 2, c4 = lane & 3;
  const int ra = r0 + 16 * warp + g8, rb = ra + 8;  // the thread's two rows
  const bool va = ra < r0 + nrows, vb = rb < r0 + nrows;
  auto qrow = [&](int r) {
    return static_cast<const char *>(p.q) +
           ((static_cast<int64_t>(a) + r / G) * p.q_ss + static_cast<int64_t>(g * G + r % G) * p.q_hs) * 2;
  };
  const char *qa = qrow(va ? ra : r0), *qb = qrow(vb ? rb : r0);
  uint32_t qf[C::KT][4];
#pragma unroll
  for (int j = 0; j < C::KT; ++j) {
    const int e0 = 16 * j + 2 * c4, e1 = e0 + 8;
    qf[j][0] = va ? __ldg(reinterpret_cast<const uint32_t *>(qa + e0 * 2)) : 0u;
    qf[j][1] = vb ? __ldg(reinterpret_cast<const uint32_t *>(qb + e0 * 2)) : 0u;
    qf[j][2] = va ? __ldg(reinterpret_cast<const uint32_t *>(qa + e1 * 2)) : 0u;
    qf[j][3] = vb ? __ldg(reinterpret_cast<const uint32_t *>(qb + e1 * 2)) : 0u;
  }
  const int posA = va ? pos0 + ra / G : -1, posB = vb ? pos0 + rb / G : -1;
  float abA = 0.f, abB = 0.f;  // ALiBi slopes (log2 units)
  if (p.alibi) {
    if (va) abA = __ldg(p.alibi + g * G + ra % G) * 1.4426950408889634f;
    if (vb) abB = __ldg(p.alibi + g * G + rb % G) * 1.4426950408889634f;
  }

  float o[C::NT][4];
#pragma unroll
  for (int n = 0; n < C::NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float mA = kChunkEmpty, mB = kChunkEmpty, lA = 0.f, lB = 0.f;

  // ldmatrix lane roles: K (B operand of S): matrix lane / 8 = (token half, k half);
  // V (B operand of O, transposed): matrix lane / 8 = (token half, d half)
  const int krow = (lane & 7) | ((lane >> 4) << 3), khalf = (lane >> 3) & 1;
  const int vtok = (lane & 7) | (((lane >> 3) & 1) << 3), vhalf = lane >> 4;

  int k = 0;
  for (; k < npages; ++k) {
    const int st = k % C::R;
    // a warp leaves the loop as a whole: a vote makes the outcome of the wait uniform
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(full0 + 8 * st, (k / C::R) & 1, kChunkWaitLimit))) {
      bad = stalled = true;
      if (lane == 0 && p.err) atomicOr(p.err, kErrTimeout);
      break;
    }
    const uint32_t kb = sbase + st * C::STAGEB, vbase = kb + C::PAGEB;
    const int t0 = k * kBlock;  // first token of the page

    // ---- S = Q K^T: n-tile 0 = tokens 0-7, n-tile 1 = tokens 8-15
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < C::KT; ++j) {
      const int chunk = ((j & 3) << 1) | khalf;
      uint32_t bk[4];
      ldmatrix_x4(bk, kb + (j >> 2) * 2048 + krow * 128 + ((chunk ^ (krow & 7)) << 4));
      if constexpr (C::BF) {
        mma_bf16(s0, qf[j], bk[0], bk[1]);
        mma_bf16(s1, qf[j], bk[2], bk[3]);
      } else {
        mma_f16(s0, qf[j], bk[0], bk[1]);
        mma_f16(s1, qf[j], bk[2], bk[3]);
      }
    }
    // fragment tokens: s0[0..1] row A tokens 2c4, 2c4+1; s0[2..3] row B; s1 the same + 8
    const int ta = t0 + 2 * c4;
    float x[8];
    x[0] = ta <= posA ? fmaf(abA, static_cast<float>(ta - posA), s0[0] * p.scale_log2) : -INFINITY;
    x[1] = ta + 1 <= posA ? fmaf(abA, static_cast<float>(ta + 1 - posA), s0[1] * p.scale_log2) : -INFINITY;
    x[2] = ta <= posB ? fmaf(abB, static_cast<float>(ta - posB), s0[2] * p.scale_log2) : -INFINITY;
    x[3] = ta + 1 <= posB ? fmaf(abB, static_cast<float>(ta + 1 - posB), s0[3] * p.scale_log2) : -INFINITY;
    x[4] = ta + 8 <= posA ? fmaf(abA, static_cast<float>(ta + 8 - posA), s1[0] * p.scale_log2) : -INFINITY;
    x[5] = ta + 9 <= posA ? fmaf(abA, static_cast<float>(ta + 9 - posA), s1[1] * p.scale_log2) : -INFINITY;
    x[6] = ta + 8 <= posB ? fmaf(abB, static_cast<float>(ta + 8 - posB), s1[2] * p.scale_log2) : -INFINITY;
    x[7] = ta + 9 <= posB ? fmaf(abB, static_cast<float>(ta + 9 - posB), s1[3] * p.scale_log2) : -INFINITY;

    // ---- online softmax per row, lazy running max (a row's 16 tokens sit in one lane quad)
    const float lmA = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[4], x[5]));
    const float lmB = fmaxf(fmaxf(x[2], x[3]), fmaxf(x[6], x[7]));
    if (__any_sync(0xffffffffu, (lmA > mA + kChunkSlack) | (lmB > mB + kChunkSlack))) {
      float MA = lmA, MB = lmB;
      MA = fmaxf(MA, __shfl_xor_sync(0xffffffffu, MA, 1));
      MB = fmaxf(MB, __shfl_xor_sync(0xffffffffu, MB, 1));
      MA = fmaxf(MA, __shfl_xor_sync(0xffffffffu, MA, 2));
      MB = fmaxf(MB, __shfl_xor_sync(0xffffffffu, MB, 2));
      const float nA = fmaxf(mA, MA), nB = fmaxf(mB, MB);
      const float alA = ex2(mA - nA), alB = ex2(mB - nB);
      lA *= alA;
      lB *= alB;
#pragma unroll
      for (int n = 0; n < C::NT; ++n) {
        o[n][0] *= alA;
        o[n][1] *= alA;
        o[n][2] *= alB;
        o[n][3] *= alB;
      }
      mA = nA;
      mB = nB;
    }
    float pr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) pr[i] = ex2(x[i] - ((i & 2) ? mB : mA));
    lA += (pr[0] + pr[1]) + (pr[4] + pr[5]);
    lB += (pr[2] + pr[3]) + (pr[6] + pr[7]);

    // ---- P as the A fragment of O += P V: hi + lo 16-bit halves
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float u = pr[2 * i], v = pr[2 * i + 1];
      if constexpr (C::BF) {
        ph[i] = pack_bf16(u, v);
        const float2 f = unpack_bf16(ph[i]);
        pl[i] = pack_bf16(u - f.x, v - f.y);
      } else {
        ph[i] = pack_f16(u, v);
        const float2 f = unpack_f16(ph[i]);
        pl[i] = pack_f16(u - f.x, v - f.y);
      }
    }
    // A fragment order: (row A, tok 0-7), (row B, tok 0-7), (row A, tok 8-15), (row B, tok 8-15)
    const uint32_t ah[4] = {ph[0], ph[1], ph[2], ph[3]}, al[4] = {pl[0], pl[1], pl[2], pl[3]};

    // ---- O += P V; V rows of tokens >= len are zeroed (their P is 0, their data may be NaN)
    const int nv = min(kBlock, len - t0);
    const uint32_t m0 = (2 * c4 < nv ? 0x0000FFFFu : 0u) | (2 * c4 + 1 < nv ? 0xFFFF0000u : 0u);
    const uint32_t m1 = (2 * c4 + 8 < nv ? 0x0000FFFFu : 0u) | (2 * c4 + 9 < nv ? 0xFFFF0000u : 0u);
#pragma unroll
    for (int n2 = 0; n2 < C::NT / 2; ++n2) {  // two n8 output tiles (16 dims) per ldmatrix
      const int cidx = 2 * n2 + vhalf;       // 16-byte chunk of the row
      uint32_t bv[4];
      ldmatrix_x4_trans(bv, vbase + (cidx >> 3) * 2048 + vtok * 128 + (((cidx & 7) ^ (vtok & 7)) << 4));
      if (nv < kBlock) {
        bv[0] &= m0;
        bv[1] &= m1;
        bv[2] &= m0;
        bv[3] &= m1;
      }
      if constexpr (C::BF) {
        mma_bf16(o[2 * n2], ah, bv[0], bv[1]);
        mma_bf16(o[2 * n2], al, bv[0], bv[1]);
        mma_bf16(o[2 * n2 + 1], ah, bv[2], bv[3]);
        mma_bf16(o[2 * n2 + 1], al, bv[2], bv[3]);
      } else {
        mma_f16(o[2 * n2], ah, bv[0], bv[1]);
        mma_f16(o[2 * n2], al, bv[0], bv[1]);
        mma_f16(o[2 * n2 + 1], ah, bv[2], bv[3]);
        mma_f16(o[2 * n2 + 1], al, bv[2], bv[3]);
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);  // this warp is done with the slot
    if (warp == 0 && k + C::R < npages) {
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(empty0 + 8 * st, (k / C::R) & 1, kChunkWaitLimit))) {
        bad = stalled = true;
        if (lane == 0 && p.err) atomicOr(p.err, kErrTimeout);
        break;
      }
      fence_proxy_async_smem();
      issue(k + C::R);
    }
  }
  if (__syncthreads_or(stalled)) {
    // copies may still be in flight into the ring: the issuer waits (bounded) for the pages
    // it issued and did not consume -- each the latest use of its slot -- before the CTA's
    // shared memory goes away
    if (threadIdx.x == 0)
      for (int k2 = k; k2 < issued; ++k2)
        mbar_wait_bounded(full0 + 8 * (k2 % C::R), (k2 / C::R) & 1, kChunkWaitLimit);
    return;
  }
  if (__syncthreads_or(bad)) return;

  // ---- finish: row sums over the quad, normalise, store
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  const float iA = lA > 0.f ? 1.f / lA : 0.f, iB = lB > 0.f ? 1.f / lB : 0.f;
  OutT *outA = static_cast<OutT *>(p.out) +
               (static_cast<int64_t>(a) + ra / G) * p.out_ss + static_cast<int64_t>(g * G + ra % G) * p.out_hs;
  OutT *outB = static_cast<OutT *>(p.out) +
               (static_cast<int64_t>(a) + rb / G) * p.out_ss + static_cast<int64_t>(g * G + rb % G) * p.out_hs;
#pragma unroll
  for (int n = 0; n < C::NT; ++n) {
    const int d = 8 * n + 2 * c4;
    if (va) *reinterpret_cast<uint32_t *>(outA + d) = C::BF ? pack_bf16(o[n][0] * iA, o[n][1] * iA)
                                                            : pack_f16(o[n][0] * iA, o[n][1] * iA);
    if (vb) *reinterpret_cast<uint32_t *>(outB + d) = C::BF ? pack_bf16(o[n][2] * iB, o[n][3] * iB)
                                                            : pack_f16(o[n][2] * iB, o[n][3] * iB);
  }
}

template <int KIND, int D>
struct ChunkLaunch {
  using C = ChunkCfg<KIND, D>;
  static cudaError_t launch(const DecodeParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV, cudaStream_t st) {
    auto kern = chunk_mma_kernel<KIND, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    const int rows = p.nq_max * p.G;
    const dim3 grid((rows + C::ROWS - 1) / C::ROWS, p.Hkv, p.S);
    e = launch_pdl(kern, grid, dim3(C::THREADS), C::SMEM, st, 1, p, tmK, tmV);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
};

}  // namespace pa
