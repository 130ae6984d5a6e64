// pa_decode_mma.cuh -- paged decode attention on tensor cores (bf16 / f16 / e4m3 caches).
//
// What it computes ("Inside vLLM CUDA Kernels", Part 3; "vLLM 源码完全拆解（七）"):
// for each sequence s and query head h, o = sum_t softmax_t(scale * q . k_t) v_t
// over the first seq_lens[s] tokens, reading token t of KV head h / G from
// physical block block_table[s][t / 16], offset t % 16.
//
// Work unit (one CTA): sequence s, KV head g, a group of 8 query columns, and one
// split-KV partition of pages.  A column is a "virtual head": for single-query
// decode one of the KV head's query heads; with several query tokens per sequence
// (the varlen read path of "Inside vLLM CUDA Kernels", Part 3), column v is query
// token v / G at head g G + v % G, and sees the tokens up to its own position
// (causal, the new tokens at the end of the history).  All columns of the group
// share every K/V page the CTA loads, so each page is read once per KV head (and
// column group), not once per query head.
//
// Inside a CTA, warp w takes pages w, w+W, w+2W, ... of the partition and runs its
// own pipeline: lane 0 resolves the physical block through block_table and issues
// two TMA tensor loads (K page, V page) into one of STAGES shared-memory stages,
// completing on that stage's mbarrier; the warp waits on the barrier (bounded),
// computes, and refills the stage STAGES pages ahead.  One (block, kv head)
// page of the HND cache is 16 rows x D elements; TMA writes it with the 128-byte
// swizzle so the tensor-core fragment loads below are bank-conflict free.
//
// Per 16-token page and the CTA's 8 columns:
//   scores  S[16 tok x 8 cols] = K_page[16 x D] . Q^T[D x 8]      (mma m16n8k16, fp32 acc)
//           (+ the ALiBi bias slope_h * (t - position), one FMA per score)
//   online softmax per column (log2 domain): running max m, moved only when a score
//           exceeds it by more than 2^8 (otherwise the stale max is kept and p <= 256),
//           p = 2^(s-m), partial row sums kept per lane and reduced once at the end;
//           tokens a column cannot see get -inf (never in the max or the denominator)
//   output  O^T[D x 8 cols] += V_page^T[D x 16 tok] . P^T[16 tok x 8 cols]
//           with P split into hi + lo halves of the 16-bit type (two mmas), so the
//           probabilities keep ~16 bits; V rows t >= seq_len are zeroed before the
//           product, so stale or NaN tail values never reach the output.
// The score fragment is turned into the P^T operand with movmatrix (transpose of
// an 8x8 tile in registers); no shared-memory round trip.
//
// E4M3 caches: codes are widened to f16 exactly (cvt e4m3x2 -> f16x2) and the
// f16 tensor-core path is used; the query is scaled by a power of two per head so
// that its largest element lies in [2^14, 2^15) and rounded to f16 (exact for a
// bf16 query in that range); the power of two and k_scale are folded into the
// score scale, v_scale into the final output (per KV head with per-head scales).  K fragments use a permuted
// head-dimension order (each lane reads 32 contiguous bytes of a row) and the
// query uses the same permutation, which leaves q . k unchanged.
//
// After the last page, each warp writes its (m, l, acc) to its own shared-memory
// region; the CTA merges the W warp states with max/LSE rescaling and writes
// either the normalised output (a sequence with a single partition) or the
// partition's state to the workspace, where the unit's last CTA merges all
// partitions (pa_merge.cuh); a cluster split merges through distributed shared
// memory instead, and the balanced split runs several page ranges per CTA.
//
// The kernel is launched as a programmatic dependent of the previous grid on the
// stream: it waits for that grid before its first global read, so its launch
// overlaps the previous kernel's tail.  Three variants per shape: the general one
// (several query tokens, ALiBi), PLAIN (one query token, no ALiBi: one compare per score
// for the page tail), and PLAIN + EARLY for pa_decode_step's multi-row steps, which reads
// everything but the pages with new positions before that wait.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_merge.cuh"

namespace pa {

constexpr uint32_t kWaitLimit = 1u << 20;  // mbarrier polls before a wait gives up (>= ~20 ms)
constexpr float kMaxSlack = 8.f;            // log2 units: probabilities within a page stay <= 256
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kNoWaitPage = 0x7fffffff;     // run_pages: no page waits for the preceding grid
constexpr float kEmptyMax = -1e30f;         // running max of a column with no visible token yet

template <int KIND, int D, int W, int STAGES>
struct MmaCfg {
  static constexpr bool FP8 = KIND == KIND_FP8_BF16Q || KIND == KIND_FP8_F16Q;
  static constexpr bool QBF16 = KIND == KIND_BF16 || KIND == KIND_FP8_BF16Q;  // query/output bf16
  static constexpr bool MMA_BF16 = KIND == KIND_BF16;
  static constexpr int ELEM = FP8 ? 1 : 2;     // cache element bytes
  static constexpr int ROWB = D * ELEM;        // bytes of one token row of a page
  static constexpr int NBOX = ROWB / 128;      // 128-byte TMA boxes across a row
  static constexpr int BOXE = 128 / ELEM;      // elements per box row
  static constexpr int PAGEB = kBlock * ROWB;  // one (block, kv head) page
  static constexpr int STAGEB = 2 * PAGEB;     // K page + V page
  static constexpr int KT = D / 16;            // k-steps of Q.K^T = d-tiles of P.V
  static constexpr int THREADS = W * 32;
  static constexpr size_t SCRATCH_OFF = static_cast<size_t>(W) * STAGES * STAGEB + W * STAGES * 8;
  static constexpr size_t SMEM = 1024 + SCRATCH_OFF + kMmaScratch;
  static_assert(ROWB % 128 == 0, "page rows must be whole 128-byte swizzle spans");
  static_assert(STAGES * STAGEB >= 64 + 8 * D * 4, "warp region must hold the merge state");
  static_assert(static_cast<size_t>(W) * STAGES * STAGEB >= 8 * kMergeSmemParts * 4, "merge weights");
  static_assert(kMmaScratch >= kLptScratchBytes, "ranking scratch");
  static_assert(kMmaScratch >= (kFlatMaxSeqs + 1) * 4, "balanced-split page offsets");
};

// Runs pages [pb, pe) of sequence s (length len) for KV head g and the CTA's query
// columns 0 .. ng-1 (cm; column j sees the tokens up to position pos0 + (v0 + j) / G)
// through the warps' pipelines, and leaves each warp's state at the start of its own
// stage region: (m, l) per column, then acc[8][D].  `used` counts the
// pages this warp has already taken through its stages: the mbarrier phases go on
// from there, so a CTA can run several ranges in a row.  With `pid_ready`, pid_reg
// already holds lane i's table entry for the warp's i-th page (read early by the
// caller).  Returns true after a bad block id or a timed-out wait; `stalled` is set
// on a timeout, after which the CTA must not issue into its stages again.
template <int KIND, int D, int W, int STAGES, bool PLAIN, bool EARLY>
__device__ __forceinline__ bool run_pages(const DecodeParams &p, const CUtensorMap *tmK, const CUtensorMap *tmV,
                                          const uint32_t sbase, uint8_t *const sgen, int &used, bool &stalled,
                                          const int s, const int len, const Cols &cm, const int pos0,
                                          const int ng, const int pb, const int pe, int pid_reg,
                                          const bool pid_ready, const uint64_t pol, const int wait_page) {
  using C = MmaCfg<KIND, D, W, STAGES>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = cm.g;
  const int32_t *bt = p.block_table + static_cast<int64_t>(s) * p.bt_ss;
  const int nmine = (pe - pb > warp) ? (pe - pb - warp + W - 1) / W : 0;
  const uint32_t stage0 = sbase + static_cast<uint32_t>(warp * STAGES * C::STAGEB);
  const uint32_t bar0 = sbase + static_cast<uint32_t>(W * STAGES * C::STAGEB + warp * STAGES * 8);
  const int u0 = used;
  bool bad = false;

  bool waited = false;  // early reads: this warp has waited for the preceding write grid
  auto issue = [&](int kk) {  // whole warp; kk increases by one per call
    if constexpr (EARLY) {
      if (!waited && pb + warp + kk * W >= wait_page) {  // a page that may hold new positions
        grid_dependency_wait();
        waited = true;
      }
    }
    if ((kk & 31) == 0 && (kk > 0 || !pid_ready)) {
      const int k2 = kk + lane;
      pid_reg = (k2 < nmine) ? __ldg(bt + pb + warp + k2 * W) : 0;
    }
    int pid = __shfl_sync(0xffffffffu, pid_reg, kk & 31);
    if (pid < 0 || pid >= p.num_blocks) {
      bad = true;
      if (lane == 0 && p.err) atomicOr(p.err, kErrBlock);
      pid = 0;  // load a valid block; the CTA writes nothing
    }
    if (lane == 0) {
      const int st = (u0 + kk) % STAGES;
      const uint32_t bar = bar0 + 8 * st;
      const uint32_t kdst = stage0 + st * C::STAGEB;
      mbar_arrive_expect_tx(bar, C::STAGEB);
      const int c1 = p.nhd ? g : 0, c2 = p.nhd ? 0 : g;  // (token, head) or (head, token) order
#pragma unroll
      for (int b = 0; b < C::NBOX; ++b) tma_load_4d(kdst + b * 2048, tmK, bar, b * C::BOXE, c1, c2, pid, pol);
#pragma unroll
      for (int b = 0; b < C::NBOX; ++b)
        tma_load_4d(kdst + C::PAGEB + b * 2048, tmV, bar, b * C::BOXE, c1, c2, pid, pol);
    }
  };

  const int npre = min(STAGES, nmine);
  for (int kk = 0; kk < npre; ++kk) issue(kk);

  // ------------------------------------------------------- query fragments
  const int qh = lane >> 2, qc = lane & 3;  // fragment row (head / token) and column group
  const bool qvalid = qh < ng;
  const char *qrow = static_cast<const char *>(p.q) + cm.q_off(p, qvalid ? qh : 0) * 2;
  uint32_t qf[C::KT][2];
  float sc0, sc1;  // score scale (log2 units) of this lane's two head columns 2qc, 2qc+1
  if constexpr (!C::FP8) {
#pragma unroll
    for (int j = 0; j < C::KT; ++j) {
      const uint32_t lo = __ldg(reinterpret_cast<const uint32_t *>(qrow + (16 * j + 2 * qc) * 2));
      const uint32_t hi = __ldg(reinterpret_cast<const uint32_t *>(qrow + (16 * j + 8 + 2 * qc) * 2));
      qf[j][0] = qvalid ? lo : 0u;
      qf[j][1] = qvalid ? hi : 0u;
    }
    sc0 = sc1 = p.scale_log2;
  } else {
    // lane covers d = 128 b + 32 qc + [0, 32) of head qh, box b
    uint4 raw[C::NBOX][4];
    float mx = 0.f;
#pragma unroll
    for (int b = 0; b < C::NBOX; ++b) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        raw[b][i] = __ldg(reinterpret_cast<const uint4 *>(qrow + (128 * b + 32 * qc + 8 * i) * 2));
        const uint32_t w4[4] = {raw[b][i].x, raw[b][i].y, raw[b][i].z, raw[b][i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = C::QBF16 ? unpack_bf16(w4[e]) : unpack_f16(w4[e]);
          mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    int ex = 0;
    if (mx > 0.f && mx <= 3.0e38f) {
      frexpf(mx, &ex);  // mx = f * 2^ex, f in [0.5, 1)
      ex -= 1;          // floor(log2 mx)
    }
    const int sh = max(-120, min(120, 14 - ex));
    const float sfac = ldexpf(1.f, sh);  // max |q| * sfac in [2^14, 2^15)
#pragma unroll
    for (int b = 0; b < C::NBOX; ++b) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w4[4] = {raw[b][i].x, raw[b][i].y, raw[b][i].z, raw[b][i].w};
        // elements 8i .. 8i+7 of the lane's 32 = k-steps j = 2i, 2i+1 (4 elements each)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const float2 f0 = C::QBF16 ? unpack_bf16(w4[2 * jj]) : unpack_f16(w4[2 * jj]);
          const float2 f1 = C::QBF16 ? unpack_bf16(w4[2 * jj + 1]) : unpack_f16(w4[2 * jj + 1]);
          const int j = b * 8 + 2 * i + jj;
          qf[j][0] = qvalid ? pack_f16(f0.x * sfac, f0.y * sfac) : 0u;
          qf[j][1] = qvalid ? pack_f16(f1.x * sfac, f1.y * sfac) : 0u;
        }
      }
    }
    const float ks = p.k_scale ? __ldg(p.k_scale + g * p.scale_stride) : 1.f;  // this KV head's
    const float sf0 = __shfl_sync(0xffffffffu, sfac, (2 * qc) * 4);
    const float sf1 = __shfl_sync(0xffffffffu, sfac, (2 * qc + 1) * 4);
    sc0 = p.scale_log2 * ks / sf0;
    sc1 = p.scale_log2 * ks / sf1;
  }


  // --------------------------------------------------------------- main loop
  float acc[C::KT][4];
#pragma unroll
  for (int t = 0; t < C::KT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  // Running max of an empty column: a finite stand-in for -inf, so a page with every
  // token masked for a column (a causal column whose tokens end before this warp's first
  // page) gives p = 2^(-inf - m) = 0, never 2^(-inf + inf).
  float m0 = kEmptyMax, m1 = kEmptyMax, l0 = 0.f, l1 = 0.f;
  const int ra = lane >> 2;  // token row of score fragments (and +8)
  // The lane's two columns 2qc, 2qc+1: the last visible position (causal; -1 for a column
  // beyond the CTA's queries) and the ALiBi slope (log2 units; 0 without ALiBi), which
  // adds slope * (t - position) to the logit of token t.
  const int posA = 2 * qc < ng ? pos0 + (cm.v0 + 2 * qc) / cm.G : -1;
  const int posB = 2 * qc + 1 < ng ? pos0 + (cm.v0 + 2 * qc + 1) / cm.G : -1;
  float ab0 = 0.f, ab1 = 0.f;
  if (p.alibi) {
    if (2 * qc < ng) ab0 = __ldg(p.alibi + cm.head(2 * qc)) * kLog2e;
    if (2 * qc + 1 < ng) ab1 = __ldg(p.alibi + cm.head(2 * qc + 1)) * kLog2e;
  }

  for (int k = 0; k < nmine; ++k) {
    const int u = u0 + k;  // this page's use of the warp's stages
    const int st = u % STAGES;
    // the warp's first wait may carry a shorter limit (first_wait_limit: the timeout path's test)
    const uint32_t lim = (u == 0 && p.first_wait_limit != 0)
                             ? (p.first_wait_limit < 0 ? 0u : static_cast<uint32_t>(p.first_wait_limit))
                             : kWaitLimit;
    if (!mbar_wait_bounded(bar0 + 8 * st, (u / STAGES) & 1, lim)) {
      bad = true;
      stalled = true;
      if (lane == 0 && p.err) atomicOr(p.err, kErrTimeout);
      // Drain: the copies of pages k .. k+STAGES-1 (the one just given up on included) are in
      // flight; wait for every one of them, with the full limit, before the warp reuses its
      // stage region for its merge state or the CTA exits.
      for (int k2 = k; k2 < min(nmine, k + STAGES); ++k2)
        mbar_wait_bounded(bar0 + 8 * ((u0 + k2) % STAGES), ((u0 + k2) / STAGES) & 1, kWaitLimit);
      break;
    }
    const uint32_t kb = stage0 + st * C::STAGEB;
    const uint32_t vb = kb + C::PAGEB;
    const int page = pb + warp + k * W;
    const int nv = min(kBlock, len - page * kBlock);  // valid tokens in this page

    // ---- scores: two accumulation chains over the k-steps
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (!C::FP8) {
      const int lrow = (lane & 7) | (lane & 8);
      const int lhi = lane >> 4;
#pragma unroll
      for (int j = 0; j < C::KT; ++j) {
        const int chunk = ((j & 3) << 1) | lhi;
        uint32_t a[4];
        ldmatrix_x4(a, kb + (j >> 2) * 2048 + lrow * 128 + ((chunk ^ (lrow & 7)) << 4));
        if constexpr (C::MMA_BF16) {
          if (j & 1) mma_bf16(c1, a, qf[j][0], qf[j][1]); else mma_bf16(c0, a, qf[j][0], qf[j][1]);
        } else {
          if (j & 1) mma_f16(c1, a, qf[j][0], qf[j][1]); else mma_f16(c0, a, qf[j][0], qf[j][1]);
        }
      }
    } else {
#pragma unroll
      for (int b = 0; b < C::NBOX; ++b) {
        const uint32_t rowa = kb + b * 2048 + ra * 128, rowb = rowa + 8 * 128;
        const uint32_t ch0 = static_cast<uint32_t>(((2 * qc) ^ ra) << 4);
        const uint32_t ch1 = static_cast<uint32_t>(((2 * qc + 1) ^ ra) << 4);
        const uint4 A0 = lds128(rowa + ch0), A1 = lds128(rowa + ch1);
        const uint4 B0 = lds128(rowb + ch0), B1 = lds128(rowb + ch1);
        const uint32_t wa[8] = {A0.x, A0.y, A0.z, A0.w, A1.x, A1.y, A1.z, A1.w};
        const uint32_t wb[8] = {B0.x, B0.y, B0.z, B0.w, B1.x, B1.y, B1.z, B1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t a[4];
          e4m3x4_to_f16x2x2(wa[j], a[0], a[2]);  // row ra:   d 4j, 4j+1 | 4j+2, 4j+3
          e4m3x4_to_f16x2x2(wb[j], a[1], a[3]);  // row ra+8
          if (j & 1) mma_f16(c1, a, qf[b * 8 + j][0], qf[b * 8 + j][1]);
          else mma_f16(c0, a, qf[b * 8 + j][0], qf[b * 8 + j][1]);
        }
      }
    }

    // ---- online softmax (fragment: rows ra, ra+8 = tokens; columns 2qc, 2qc+1 = heads)
    float s0, s1, s2, s3;
    if constexpr (PLAIN) {  // one query token, no ALiBi: every column sees the tokens < len
      const bool va = ra < nv, vb8 = ra + 8 < nv;
      s0 = va ? (c0[0] + c1[0]) * sc0 : -INFINITY;
      s1 = va ? (c0[1] + c1[1]) * sc1 : -INFINITY;
      s2 = vb8 ? (c0[2] + c1[2]) * sc0 : -INFINITY;
      s3 = vb8 ? (c0[3] + c1[3]) * sc1 : -INFINITY;
    } else {
      const int ta = page * kBlock + ra, tb = ta + 8;  // the fragment's two tokens
      s0 = ta <= posA ? fmaf(ab0, static_cast<float>(ta - posA), (c0[0] + c1[0]) * sc0) : -INFINITY;
      s1 = ta <= posB ? fmaf(ab1, static_cast<float>(ta - posB), (c0[1] + c1[1]) * sc1) : -INFINITY;
      s2 = tb <= posA ? fmaf(ab0, static_cast<float>(tb - posA), (c0[2] + c1[2]) * sc0) : -INFINITY;
      s3 = tb <= posB ? fmaf(ab1, static_cast<float>(tb - posB), (c0[3] + c1[3]) * sc1) : -INFINITY;
    }
    // The running max of a head moves only when a score exceeds it by more than
    // kMaxSlack (log2 units); otherwise the page is weighted against the stale max,
    // p = 2^(s - m) <= 2^kMaxSlack, and the cross-lane max reduction and the rescale
    // are skipped.  (m, l, acc) stay consistent, so the merges are unchanged.
    const float lm0 = fmaxf(s0, s2), lm1 = fmaxf(s1, s3);
    if (__any_sync(0xffffffffu, (lm0 > m0 + kMaxSlack) | (lm1 > m1 + kMaxSlack))) {
      float mx0 = lm0, mx1 = lm1;
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);  // 0 on the first page (m = -inf)
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int t = 0; t < C::KT; ++t) {
        acc[t][0] *= al0;
        acc[t][1] *= al1;
        acc[t][2] *= al0;
        acc[t][3] *= al1;
      }
      m0 = mn0;
      m1 = mn1;
    }
    const float p0 = ex2(s0 - m0), p1 = ex2(s1 - m1), p2 = ex2(s2 - m0), p3 = ex2(s3 - m1);
    l0 += p0 + p2;
    l1 += p1 + p3;

    // ---- P^T operand: hi + lo 16-bit halves, transposed in registers
    uint32_t bh0, bh1, bl0, bl1;
    if constexpr (C::MMA_BF16) {
      const uint32_t ha = pack_bf16(p0, p1), hb = pack_bf16(p2, p3);
      const float2 fa = unpack_bf16(ha), fb = unpack_bf16(hb);
      bh0 = movmatrix_trans(ha);
      bh1 = movmatrix_trans(hb);
      bl0 = movmatrix_trans(pack_bf16(p0 - fa.x, p1 - fa.y));
      bl1 = movmatrix_trans(pack_bf16(p2 - fb.x, p3 - fb.y));
    } else {
      const uint32_t ha = pack_f16(p0, p1), hb = pack_f16(p2, p3);
      const float2 fa = unpack_f16(ha), fb = unpack_f16(hb);
      bh0 = movmatrix_trans(ha);
      bh1 = movmatrix_trans(hb);
      bl0 = movmatrix_trans(pack_f16(p0 - fa.x, p1 - fa.y));
      bl1 = movmatrix_trans(pack_f16(p2 - fb.x, p3 - fb.y));
    }

    // ---- O^T += V^T . P^T (tail rows of the last page zeroed first)
    if constexpr (!C::FP8) {
      const uint32_t mA = (2 * qc < nv ? 0x0000FFFFu : 0u) | (2 * qc + 1 < nv ? 0xFFFF0000u : 0u);
      const uint32_t mB = (2 * qc + 8 < nv ? 0x0000FFFFu : 0u) | (2 * qc + 9 < nv ? 0xFFFF0000u : 0u);
      const int vtok = (lane & 7) | ((lane >> 4) << 3);
      const int vhalf = (lane >> 3) & 1;
#pragma unroll
      for (int t = 0; t < C::KT; ++t) {
        const int cidx = 2 * t + vhalf;  // 16-byte chunk of the row
        uint32_t a[4];
        ldmatrix_x4_trans(a, vb + (cidx >> 3) * 2048 + vtok * 128 + (((cidx & 7) ^ (vtok & 7)) << 4));
        if (nv < kBlock) {
          a[0] &= mA;
          a[1] &= mA;
          a[2] &= mB;
          a[3] &= mB;
        }
        if constexpr (C::MMA_BF16) {
          mma_bf16(acc[t], a, bh0, bh1);
          mma_bf16(acc[t], a, bl0, bl1);
        } else {
          mma_f16(acc[t], a, bh0, bh1);
          mma_f16(acc[t], a, bl0, bl1);
        }
      }
    } else {
      const int t0 = 2 * qc, t1 = 2 * qc + 1, t2 = 2 * qc + 8, t3 = 2 * qc + 9;
#pragma unroll
      for (int b = 0; b < C::NBOX; ++b) {
        const uint32_t pgb = vb + b * 2048;
        uint4 w0 = lds128(pgb + t0 * 128 + ((ra ^ (t0 & 7)) << 4));
        uint4 w1 = lds128(pgb + t1 * 128 + ((ra ^ (t1 & 7)) << 4));
        uint4 w2 = lds128(pgb + t2 * 128 + ((ra ^ (t2 & 7)) << 4));
        uint4 w3 = lds128(pgb + t3 * 128 + ((ra ^ (t3 & 7)) << 4));
        if (nv < kBlock) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          if (t0 >= nv) w0 = z;
          if (t1 >= nv) w1 = z;
          if (t2 >= nv) w2 = z;
          if (t3 >= nv) w3 = z;
        }
        const uint32_t x0[4] = {w0.x, w0.y, w0.z, w0.w}, x1[4] = {w1.x, w1.y, w1.z, w1.w};
        const uint32_t x2[4] = {w2.x, w2.y, w2.z, w2.w}, x3[4] = {w3.x, w3.y, w3.z, w3.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          // d0 = 128b + 16ra + 2t (fragment row ra), d1 = d0 + 1 (row ra + 8)
          const uint32_t sel = (t & 1) ? 0x7362u : 0x5140u;
          const uint32_t p01 = __byte_perm(x0[t >> 1], x1[t >> 1], sel);
          const uint32_t p23 = __byte_perm(x2[t >> 1], x3[t >> 1], sel);
          uint32_t a[4];
          e4m3x4_to_f16x2x2(p01, a[0], a[1]);  // d0 | d1, tokens t0 t1
          e4m3x4_to_f16x2x2(p23, a[2], a[3]);  // d0 | d1, tokens t2 t3
          mma_f16(acc[b * 8 + t], a, bh0, bh1);
          mma_f16(acc[b * 8 + t], a, bl0, bl1);
        }
      }
    }

    __syncwarp();
    if (k + STAGES < nmine) {
      fence_proxy_async_smem();
      issue(k + STAGES);
    }
  }
  used = u0 + nmine;

  // ------------------------------------------------------ merge warp states
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  // warp region (its own stage buffers, no copies in flight): ml[8][2], then acc[8][D]
  float *wml = reinterpret_cast<float *>(sgen + warp * STAGES * C::STAGEB);
  float *wacc = wml + 16;
  if (ra == 0) {
    wml[2 * (2 * qc)] = m0;
    wml[2 * (2 * qc) + 1] = l0;
    wml[2 * (2 * qc + 1)] = m1;
    wml[2 * (2 * qc + 1) + 1] = l1;
  }
#pragma unroll
  for (int t = 0; t < C::KT; ++t) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int head = 2 * qc + (i & 1);
      int d;
      if constexpr (!C::FP8) d = 16 * t + ra + 8 * (i >> 1);
      else d = 128 * (t >> 3) + 16 * ra + 2 * (t & 7) + (i >> 1);
      wacc[head * D + d] = acc[t][i];
    }
  }
  return bad;
}

// Merges the W warp states of the CTA (max / log-sum-exp rescaling) and, for every
// (head, element) of the group, writes the normalised output (direct) or stores the
// CTA's state (m, l, unnormalised acc) in workspace row rows(hh).
template <int KIND, int D, int W, int STAGES, typename OutT, typename RowFn>
__device__ __forceinline__ void write_cta_state(const DecodeParams &p, const uint8_t *sgen, const Cols &cm, int ng,
                                                float vs, bool direct, RowFn rows) {
  using C = MmaCfg<KIND, D, W, STAGES>;
  for (int i = threadIdx.x; i < ng * D; i += C::THREADS) {
    const int hh = i / D, d = i - hh * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float *ml = reinterpret_cast<const float *>(sgen + w * STAGES * C::STAGEB);
      M = fmaxf(M, ml[2 * hh]);
    }
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float *ml = reinterpret_cast<const float *>(sgen + w * STAGES * C::STAGEB);
      const float mw = ml[2 * hh];
      const float sc = (mw == -INFINITY) ? 0.f : ex2(mw - M);
      den += sc * ml[2 * hh + 1];
      num += sc * ml[16 + hh * D + d];
    }
    if (direct) {
      OutT *o = static_cast<OutT *>(p.out) + cm.out_off(p, hh) + d;
      *o = OutT(den > 0.f ? num / den * vs : 0.f);
    } else {
      const int64_t r = rows(hh);
      p.part_acc[r * D + d] = num;
      if (d == 0) p.part_ml[r] = make_float2(M, den);
    }
  }
}

template <typename OutT>
__device__ __forceinline__ void zero_rows(const DecodeParams &p, const Cols &cm, int ng, int D, int threads) {
  for (int i = threadIdx.x; i < ng * D; i += threads) {
    OutT *o = static_cast<OutT *>(p.out) + cm.out_off(p, i / D) + i % D;
    *o = OutT(0.f);
  }
}

// PLAIN: one query token per sequence and no ALiBi (pa_decode), compiled without the
// per-column causal limits and the bias.  EARLY (with PLAIN only): the early reads of
// pa_decode_step (DecodeParams::early); a wait inside the page loop costs the other
// variants about 1.4 us on a 30 us decode, so only this one carries it.
template <int KIND, int D, int W, int STAGES, bool PLAIN, bool EARLY>
__global__ void __launch_bounds__(W * 32, mma_min_ctas(KIND, D))
    decode_mma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
  using C = MmaCfg<KIND, D, W, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;  // 128B-swizzle boxes need 1 KiB alignment
  uint8_t *const sgen = smem_raw + (sbase - raw_u32);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int part = blockIdx.x;
  const int g = blockIdx.y / p.HG, hg = blockIdx.y - g * p.HG;
  const int v0 = hg * 8;                // first column (virtual head) of this CTA
  const int h0 = g * p.G + v0;          // decode: its first query head
  int ng = min(8, p.VH - v0);           // columns in the group (fewer for a short query)
  const bool flat = p.flat > 0;
  using OutT = typename std::conditional<C::QBF16, __nv_bfloat16, __half>::type;

  if (lane == 0) {  // this warp's stage barriers, before any memory operation (the init fence is a release)
    const uint32_t bar0 = sbase + static_cast<uint32_t>(W * STAGES * C::STAGEB + warp * STAGES * 8);
    for (int st = 0; st < STAGES; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_barrier_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncwarp();
  // Warm L2 with the metadata this launch reads on its critical path.  A prefetch
  // returns no data, so it may run before the wait on the previous grid.
  if (warp == 0) {
    if (lane == 0) prefetch_l2(p.seq_lens + (flat ? 0 : blockIdx.z));
    if (lane == 1 && p.qsl) prefetch_l2(p.qsl + (flat ? 0 : blockIdx.z));
    if (flat) {  // CTA c: the table rows (first head row only) and query heads of sequences c, c + CTAs, ...
      for (int z = part; z < p.S; z += p.flat) {
        if (blockIdx.y == 0) {
          const int32_t *row = p.block_table + static_cast<int64_t>(z) * p.bt_ss;
          for (int pg = lane * 32; pg < p.max_blocks; pg += 32 * 32) prefetch_l2(row + pg);
        }
        const char *qr = static_cast<const char *>(p.q) +
                         (static_cast<int64_t>(z) * p.q_ss + static_cast<int64_t>(h0) * p.q_hs) * 2;
        if (lane * 128 < ng * D * 2 && p.q_hs == D) prefetch_l2(qr + lane * 128);
      }
    } else {
      // CTA row z prefetches sequence z's slice of the block table (the first head group
      // only) and its query heads (the first partition only); together the rows cover
      // every sequence, whichever row ends up working on it.
      const int z = blockIdx.z;
      if (blockIdx.y == 0) {
        const int pg0 = p.cluster > 1 ? part * p.max_blocks / p.cluster : part * p.pages_per_part;
        const int pg1 = p.cluster > 1 ? (part + 1) * p.max_blocks / p.cluster : min(p.max_blocks, pg0 + p.pages_per_part);
        const int32_t *row = p.block_table + static_cast<int64_t>(z) * p.bt_ss;
        for (int pg = pg0 + lane * 32; pg < pg1; pg += 32 * 32) prefetch_l2(row + pg);
      }
      if (part == 0 && !p.qsl) {
        const char *qr = static_cast<const char *>(p.q) +
                         (static_cast<int64_t>(z) * p.q_ss + static_cast<int64_t>(h0) * p.q_hs) * 2;
        if (lane * 128 < ng * D * 2 && p.q_hs == D) prefetch_l2(qr + lane * 128);
      }
    }
  }
  // Early reads apply to the one-unit path only (the balanced and cluster splits wait here).
  const bool early = EARLY && p.early && !flat && p.cluster <= 1;
  if (!early) grid_dependency_wait();

  // Pages are read once per CTA: evict them first.  (With several column groups of one KV
  // head reading the same pages, evict-normal measured 3 % slower on GB300: 4 query tokens
  // x 256 sequences x 32/8 heads, 395.6 vs 384.3 us.)
  const uint64_t pol = policy_evict_first();
  const float vs = (C::FP8 && p.v_scale) ? __ldg(p.v_scale + g * p.scale_stride) : 1.f;
  float *const smem_w = reinterpret_cast<float *>(sgen);  // merge weights (stage buffers, free by then)
  int used = 0;
  bool stalled = false;

  if (flat) {
    // ----------------------------------------------------------- balanced split
    // The pages of all sequences, concatenated in sequence order, are cut into
    // p.flat equal ranges, one per CTA of this head row; a range may end inside one
    // sequence and go on into the next.  A sequence held whole by one CTA is
    // written directly; the parts of a cut sequence are merged by the last of its
    // CTAs to finish.
    int *pref = reinterpret_cast<int *>(sgen + C::SCRATCH_OFF);  // page offsets of the sequences [S + 1]
    __shared__ int s_wsum[W];
    {
      constexpr int PER = (kFlatMaxSeqs + C::THREADS - 1) / C::THREADS;
      const int i0 = threadIdx.x * PER;
      int n[PER], sum = 0;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int i = i0 + j;
        const int L = i < p.S ? __ldg(p.seq_lens + i) : 0;
        const bool ok = L >= 0 && L <= p.max_blocks * kBlock;
        if (!ok && part == 0 && blockIdx.y == 0 && p.err) atomicOr(p.err, kErrSeqLen);
        n[j] = ok ? (L + kBlock - 1) / kBlock : 0;
        sum += n[j];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) s_wsum[warp] = incl;
      __syncthreads();
      int run = incl - sum, total = 0;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const int v = s_wsum[w];
        run += w < warp ? v : 0;
        total += v;
      }
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        if (i0 + j < p.S) pref[i0 + j] = run;
        run += n[j];
      }
      if (threadIdx.x == 0) pref[p.S] = total;
      __syncthreads();
    }
    for (int z = part; z < p.S; z += p.flat)  // empty sequences: zero output rows
      if (pref[z] == pref[z + 1] && __ldg(p.seq_lens + z) == 0)
        zero_rows<OutT>(p, Cols{z, p.G, g, v0}, ng, D, C::THREADS);

    const int T = pref[p.S];
    const int Ce = min(p.flat, T);  // CTAs with work: every range holds at least one page
    if (part >= Ce) return;
    const int a = static_cast<int>(static_cast<int64_t>(part) * T / Ce);
    const int b = static_cast<int>(static_cast<int64_t>(part + 1) * T / Ce);
    auto range_start = [&](int c) { return static_cast<int>(static_cast<int64_t>(c) * T / Ce); };
    auto owner = [&](int x) { return static_cast<int>((static_cast<int64_t>(x + 1) * Ce - 1) / T); };
    int z = 0;  // the sequence holding page a: the last z with pref[z] <= a (a non-empty one)
    {
      int hi = p.S - 1;
      while (z < hi) {
        const int mid = (z + hi + 1) >> 1;
        if (pref[mid] <= a) z = mid;
        else hi = mid - 1;
      }
    }
    const int64_t my_row = static_cast<int64_t>(blockIdx.y) * p.flat + part;
    bool dead = false;  // a wait timed out: no more copies into the stages
    for (int x = a; x < b;) {
      const int ps = pref[z], pn = pref[z + 1];
      const int y = min(b, pn);
      const Cols cm{z, p.G, g, v0};
      const int zlen = __ldg(p.seq_lens + z);
      bool bad = true;
      if (!dead)
        bad = run_pages<KIND, D, W, STAGES, PLAIN, false>(p, &tmK, &tmV, sbase, sgen, used, stalled, z, zlen, cm, zlen - 1, ng,
                                            x - ps, y - ps, 0, false, pol, kNoWaitPage);
      const bool any_bad = __syncthreads_or(bad);
      if (any_bad) dead = __syncthreads_or(stalled) || dead;
      if (x == ps && y == pn) {
        if (!any_bad) write_cta_state<KIND, D, W, STAGES, OutT>(p, sgen, cm, ng, vs, true, [](int) { return int64_t{0}; });
      } else {
        const int j = x == a ? 0 : 1;  // this CTA's first or last range
        if (!any_bad)
          write_cta_state<KIND, D, W, STAGES, OutT>(p, sgen, cm, ng, vs, false,
                                                    [&](int hh) { return (my_row * 2 + j) * 8 + hh; });
        // a CTA with an error still counts itself, so the unit's counter returns to zero
        const int c0 = owner(ps);
        merge_if_last<OutT, D>(p, cm, static_cast<int>(blockIdx.y) + p.Hkv * p.HG * z, ng, owner(pn - 1) - c0 + 1,
                               vs, any_bad, C::THREADS, smem_w,
                               FlatRows{static_cast<int64_t>(blockIdx.y) * p.flat + c0, range_start(c0) < ps ? 1 : 0});
      }
      x = y;
      if (x < b) {
        fence_proxy_async_smem();  // generic accesses to the stages before the next copies into them
        __syncthreads();
        do ++z;
        while (pref[z + 1] == pref[z]);  // next non-empty sequence (one exists: x < b)
      }
    }
    return;
  }

  // --------------------------------------------- one unit (or partition) per CTA
  const int s = p.lpt ? lpt_sequence(p.seq_lens, p.S, blockIdx.z, C::THREADS,
                                    reinterpret_cast<int *>(sgen + C::SCRATCH_OFF))
                      : static_cast<int>(blockIdx.z);
  const int32_t *bt = p.block_table + static_cast<int64_t>(s) * p.bt_ss;
  const int len = __ldg(p.seq_lens + s);
  const bool clustered = p.cluster > 1;  // rank `part` of a cluster splitting the unit equally
  const bool split = p.max_parts > 1;
  int pid_reg = 0;  // lane i: physical block of my page i; with fixed-size partitions it is
                    // read speculatively (bounded by the table width) alongside seq_len
  if (!clustered) {
    const int pg = part * p.pages_per_part + warp + lane * W;
    if (pg < p.max_blocks) pid_reg = __ldg(bt + pg);
  }
  if (len < 0 || len > p.max_blocks * kBlock) {  // (all ranks of a cluster see the same length)
    if (threadIdx.x == 0 && part == 0 && blockIdx.y == 0 && p.err) atomicOr(p.err, kErrSeqLen);
    return;
  }
  // The sequence's query tokens: one (decode), or rows qsl[s] .. qsl[s+1]-1 (varlen), the last
  // at position len - 1; column j sees the tokens up to pos0 + (v0 + j) / G.
  int64_t row0 = s;
  int nq = 1;
  if (p.qsl) {
    const int a = __ldg(p.qsl + s), b = __ldg(p.qsl + s + 1);
    row0 = a;
    nq = b - a;
    if (a < 0 || b > p.Tq || nq < 0 || nq > p.nq_max || nq > len) {  // rows outside q / out, or too many
      if (threadIdx.x == 0 && part == 0 && blockIdx.y == 0 && p.err) atomicOr(p.err, kErrSeqLen);
      return;
    }
  }
  ng = min(ng, nq * p.G - v0);  // columns past the sequence's last query token are empty
  if (ng <= 0) return;
  const Cols cm{row0, p.G, g, v0};
  const int pos0 = len - nq;
  const int vis = pos0 + (v0 + ng - 1) / p.G + 1;  // tokens the CTA's last column sees
  const int npages = (vis + kBlock - 1) / kBlock;
  int pb, pe;
  if (clustered) {
    pb = static_cast<int>(static_cast<int64_t>(part) * npages / p.cluster);
    pe = static_cast<int>(static_cast<int64_t>(part + 1) * npages / p.cluster);
    const int pg = pb + warp + lane * W;
    if (pg < pe) pid_reg = __ldg(bt + pg);
  } else {
    pb = part * p.pages_per_part;
    pe = min(npages, pb + p.pages_per_part);
  }
  if (pb >= pe && !clustered) {  // (an empty cluster rank stays: it takes part in the merge)
    if (npages == 0 && part == 0) {  // empty sequence (any split)
      if (early) grid_dependency_wait();
      zero_rows<OutT>(p, cm, ng, D, C::THREADS);
    }
    return;
  }
  // early reads: pages from the first new position on wait for the preceding write grid
  int wait_page = kNoWaitPage;
  if (early) {
    const int nnew = p.new_start ? __ldg(p.new_start + s + 1) - __ldg(p.new_start + s) : 1;
    wait_page = nnew <= 0 ? kNoWaitPage : max(0, len - nnew) / kBlock;
  }

  const bool bad = run_pages<KIND, D, W, STAGES, PLAIN, EARLY>(p, &tmK, &tmV, sbase, sgen, used, stalled, s, len, cm, pos0, ng,
                                                 pb, pe, pid_reg, true, pol, wait_page);
  if (early) grid_dependency_wait();  // before any output or workspace write
  const bool any_bad = __syncthreads_or(bad);

  if (clustered) {
    // CTA state in place: element (hh, d) of warp 0's accumulator region is read only by
    // the thread that overwrites it; (max, exp-sum) per head go to the scratch area
    float *cs = reinterpret_cast<float *>(sgen) + 16;
    float2 *cmd = reinterpret_cast<float2 *>(sgen + C::SCRATCH_OFF);
    if (!any_bad) {
      for (int i = threadIdx.x; i < ng * D; i += C::THREADS) {
        const int hh = i / D, d = i - hh * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, reinterpret_cast<const float *>(sgen + w * STAGES * C::STAGEB)[2 * hh]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float *ml = reinterpret_cast<const float *>(sgen + w * STAGES * C::STAGEB);
          const float mw = ml[2 * hh];
          const float sc = (mw == -INFINITY) ? 0.f : ex2(mw - M);
          den += sc * ml[2 * hh + 1];
          num += sc * ml[16 + hh * D + d];
        }
        cs[hh * D + d] = num;
        if (d == 0) cmd[hh] = make_float2(M, den);
      }
    }
    cluster_merge_write<OutT, D>(p, cm, ng, vs, any_bad, cs, D, cmd, reinterpret_cast<int *>(cmd + 8),
                                 C::THREADS);
    return;
  }
  const int nparts = split ? (npages + p.pages_per_part - 1) / p.pages_per_part : 1;
  const bool direct = nparts == 1;  // this CTA holds the whole sequence: write the output
  const FixedRows rows{(static_cast<int64_t>(s) * p.Hkv + g) * p.VH + v0, p.max_parts};
  if (!any_bad)
    write_cta_state<KIND, D, W, STAGES, OutT>(p, sgen, cm, ng, vs, direct, [&](int hh) { return rows(hh, part); });
  // a CTA with an error still counts itself (so the unit's counter returns to zero) and marks
  // the unit, whose merge then writes nothing
  if (!direct)
    merge_if_last<OutT, D>(p, cm, static_cast<int>(blockIdx.y) + p.Hkv * p.HG * s, ng, nparts, vs, any_bad,
                           C::THREADS, smem_w, rows);
}

// Host side of one (kind, head size) instantiation: function attributes, launch and
// resident CTAs per SM.
template <int KIND, int D>
struct MmaLaunch {
  static constexpr int W = mma_warps(KIND, D), ST = mma_stages(KIND, D);
  using C = MmaCfg<KIND, D, W, ST>;
  static_assert(C::SMEM == mma_smem(KIND, D), "shape table out of sync");

  template <bool PLAIN, bool EARLY>
  static cudaError_t attrs() {
    auto kern = decode_mma_kernel<KIND, D, W, ST, PLAIN, EARLY>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    // same shared/L1 split as the cache write that usually precedes it (no reconfiguration)
    return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  }
  static cudaError_t launch(const DecodeParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV, cudaStream_t st) {
    const bool plain = !p.qsl && !p.alibi;
    const bool early = plain && p.early;  // (the general variant ignores p.early: it waits first)
    cudaError_t e = early ? attrs<true, true>() : plain ? attrs<true, false>() : attrs<false, false>();
    if (e != cudaSuccess) return e;
    const dim3 grid = p.flat > 0 ? dim3(p.flat, p.Hkv * p.HG, 1) : dim3(p.max_parts, p.Hkv * p.HG, p.S);
    const dim3 block(C::THREADS);
    e = early   ? launch_pdl(decode_mma_kernel<KIND, D, W, ST, true, true>, grid, block, C::SMEM, st, p.cluster, p, tmK, tmV)
        : plain ? launch_pdl(decode_mma_kernel<KIND, D, W, ST, true, false>, grid, block, C::SMEM, st, p.cluster, p, tmK, tmV)
                : launch_pdl(decode_mma_kernel<KIND, D, W, ST, false, false>, grid, block, C::SMEM, st, p.cluster, p, tmK,
                             tmV);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  static int occupancy() {  // 0 when it cannot be queried
    int n = 0;
    if (attrs<false, false>() != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma_kernel<KIND, D, W, ST, false, false>, C::THREADS,
                                                      C::SMEM) !=
            cudaSuccess)
      return 0;
    return n;
  }
};

}  // namespace pa
