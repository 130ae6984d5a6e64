// pa_merge.cuh -- the split-KV log-sum-exp merge, fused into the decode kernels.
//
// "Inside vLLM CUDA Kernels", Part 3: split-KV changes the work partition, not
// the softmax identity -- each partition keeps a local maximum, exp-sum and
// unnormalised output, and the partial states are rescaled to a common maximum
// before merging.  "vLLM 源码完全拆解（七）", V1 与 V2, does this in a second
// kernel; here the merge runs in the decode kernel itself: every CTA of a split
// (sequence, kv head, head group) unit stores its state (m in log2 units, l,
// acc[D]) to the workspace and counts itself on the unit's arrival counter; the
// CTA whose arrival completes the count reads all partition states back from L2
// and writes
//     out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,   M = max_p m_p.
// The completing CTA also resets the counter to zero, so the counters are zero
// again at the end of every launch (the workspace contract: zero before first use).
#pragma once

#include <climits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// Up to this many partitions the merge keeps the per-partition weights in shared memory.
constexpr int kMergeSmemParts = 256;

// Workspace rows of the partial states.  Row r holds (m, l) at part_ml[r] and acc at
// part_acc[r * D .. r * D + D).
// Fixed-size partitions: one row per (sequence, KV head, virtual head, partition).
struct FixedRows {
  int64_t head0;  // (s * Hkv + g) * VH + v0: the unit's first column among all (sequence, column)
  int max_parts;
  __device__ __forceinline__ int64_t operator()(int hh, int i) const { return (head0 + hh) * max_parts + i; }
};
// Balanced split: each CTA owns two row groups (its first and its last page range),
// 8 heads each; the parts of one sequence belong to consecutive CTAs c0, c0+1, ...,
// and the first of them stores the sequence in its second group when the sequence
// is not where its range starts (j0 = 1).
struct FlatRows {
  int64_t c0;  // head row * CTAs per head row + first CTA of the sequence
  int j0;
  __device__ __forceinline__ int64_t operator()(int hh, int i) const {
    return ((c0 + i) * 2 + (i == 0 ? j0 : 0)) * 8 + hh;
  }
};

// A part that stored no state (a bad block id or a timed-out wait: `bad`) still arrives, so
// the counter returns to zero, but first sets kUnitBad in it; the last arriver then sees the
// flag and writes nothing for the unit (its error bit is already set).  Each thread's
// operations on one location are ordered, so a bad part's flag precedes its own arrival,
// and the last arrival follows every other.
constexpr int kUnitBad = 0x40000000;
constexpr int kArrivalMask = kUnitBad - 1;

// smem_w: shared memory for 8 * kMergeSmemParts floats, free for reuse by now.
// rows(hh, i): workspace row of column hh in the unit's i-th part; cm maps columns to outputs.
template <typename OutT, int D, typename Rows>
__device__ __forceinline__ void merge_if_last(const DecodeParams &p, const Cols &cm, int unit, int ng, int nparts,
                                              float vs, bool bad, int threads, float *smem_w, Rows rows) {
  __shared__ int s_last;
  float(*s_w)[kMergeSmemParts] = reinterpret_cast<float(*)[kMergeSmemParts]>(smem_w);  // weight per head, part
  __syncthreads();  // every partial store of this CTA precedes thread 0's release below
  if (threadIdx.x == 0) {
    if (bad) atomicOr(p.counters + unit, kUnitBad);
    int old;
    // release: this CTA's partial states become visible before the arrival counts;
    // acquire: the last arriver then sees every other partition's state
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(old) : "l"(p.counters + unit) : "memory");
    const int last = (old & kArrivalMask) == nparts - 1;
    if (last) atomicExch(p.counters + unit, 0);
    s_last = last && !(old & kUnitBad) && !bad;
  }
  __syncthreads();
  if (!s_last) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = threads >> 5;
  const bool in_smem = nparts <= kMergeSmemParts;
  for (int hh = warp; hh < ng; hh += nw) {
    float M = -INFINITY;
    for (int i = lane; i < nparts; i += 32) M = fmaxf(M, __ldcg(p.part_ml + rows(hh, i)).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float den = 0.f;
    for (int i = lane; i < nparts; i += 32) {
      const float2 v = __ldcg(p.part_ml + rows(hh, i));
      const float w = v.x == -INFINITY ? 0.f : ex2(v.x - M);
      den += w * v.y;
      if (in_smem) s_w[hh][i] = w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    const float inv = den > 0.f ? vs / den : 0.f;
    if (in_smem) {
      __syncwarp();
      for (int i = lane; i < nparts; i += 32) s_w[hh][i] *= inv;
    } else if (lane == 0) {
      s_w[hh][0] = M;
      s_w[hh][1] = inv;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < ng * D; i += threads) {
    const int hh = i / D, d = i - hh * D;
    float r = 0.f;
    if (in_smem) {
      for (int q = 0; q < nparts; ++q) r += s_w[hh][q] * __ldcg(p.part_acc + rows(hh, q) * D + d);
    } else {
      const float M = s_w[hh][0];
      for (int q = 0; q < nparts; ++q) {
        const int64_t r0 = rows(hh, q);
        const float m = __ldcg(p.part_ml + r0).x;
        r += (m == -INFINITY ? 0.f : ex2(m - M)) * __ldcg(p.part_acc + r0 * D + d);
      }
      r *= s_w[hh][1];
    }
    OutT *o = static_cast<OutT *>(p.out) + cm.out_off(p, hh) + d;
    *o = static_cast<OutT>(r);
  }
}

// The cluster split: the C CTAs of a thread-block cluster each take an equal share
// of one (sequence, kv head, head group) unit's pages.  Each CTA has already stored
// its state in its own shared memory -- the unnormalised output cs[hh * cs_stride + d]
// and (max in log2 units, exp-sum) cmd[hh] -- and here, after a cluster barrier, CTA
// rank r merges the d-slice [r D/C, (r+1) D/C) of every head, reading the C states
// through distributed shared memory, and writes the output.  A second barrier keeps
// each CTA's shared memory alive until the others have read it.  No global memory
// and no workspace are involved.
template <typename OutT, int D>
__device__ __forceinline__ void cluster_merge_write(const DecodeParams &p, const Cols &cm, int ng, float vs, bool bad,
                                                    const float *cs, int cs_stride, const float2 *cmd, int *cbad,
                                                    int threads) {
  if (threadIdx.x == 0) *cbad = bad ? 1 : 0;
  cluster_sync();
  const int C = p.cluster;
  const int r = static_cast<int>(cluster_rank());
  int anybad = 0;
  for (int j = 0; j < C; ++j) anybad |= ld_dsmem_s32(dsmem_addr(cbad, j));
  if (!anybad) {
    const int dsl = D / C;
    for (int i = threadIdx.x; i < ng * dsl; i += threads) {
      const int hh = i / dsl, d = r * dsl + (i - hh * dsl);
      float M = -INFINITY;
      for (int j = 0; j < C; ++j) M = fmaxf(M, ld_dsmem_f32x2(dsmem_addr(cmd + hh, j)).x);
      float num = 0.f, den = 0.f;
      for (int j = 0; j < C; ++j) {
        const float2 md = ld_dsmem_f32x2(dsmem_addr(cmd + hh, j));
        const float w = md.x == -INFINITY ? 0.f : ex2(md.x - M);
        den += w * md.y;
        num += w * ld_dsmem_f32(dsmem_addr(cs + hh * cs_stride + d, j));
      }
      OutT *o = static_cast<OutT *>(p.out) + cm.out_off(p, hh) + d;
      *o = static_cast<OutT>(den > 0.f ? num / den * vs : 0.f);
    }
  }
  cluster_sync();
}

// Longest-first order of sequences (for batches of at most kLptMax sequences).
// The block scheduler starts CTAs in increasing blockIdx order, so when CTA row z
// works on the z-th longest sequence, the long sequences start first and the last
// wave is made of short ones (longest-processing-time-first list scheduling).
// Warp 0 ranks all lengths with shuffles (ties by index) and the CTA takes the
// sequence of rank `rank`.
constexpr int kLptMax = 128;
constexpr int kLptScratchBytes = 4 * kLptMax * 4;

// smem_rank: shared memory for 4 * kLptMax ints.
__device__ __forceinline__ int lpt_sequence(const int32_t *seq_lens, int S, int rank, int threads, int *smem_rank) {
  int(*s_rank)[kLptMax] = reinterpret_cast<int(*)[kLptMax]>(smem_rank);
  __shared__ int s_pick;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = threads >> 5;
  int L[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = lane + 32 * k;
    L[k] = i < S ? __ldg(seq_lens + i) : INT_MIN;
  }
  // warp w counts, for every i, the j in its 32-block(s) that come before i in the order
  for (int jb = warp; jb < 4; jb += nw) {
    int rk[4] = {0, 0, 0, 0};
    const int Lb = jb == 0 ? L[0] : jb == 1 ? L[1] : jb == 2 ? L[2] : L[3];
    if (jb * 32 < S) {
#pragma unroll 8
      for (int jj = 0; jj < 32; ++jj) {
        const int Lj = __shfl_sync(0xffffffffu, Lb, jj);
        const int j = jb * 32 + jj;
#pragma unroll
        for (int k = 0; k < 4; ++k) rk[k] += (Lj > L[k]) | ((Lj == L[k]) & (j < lane + 32 * k));
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) s_rank[jb][lane + 32 * k] = rk[k];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < S; i += threads)
    if (s_rank[0][i] + s_rank[1][i] + s_rank[2][i] + s_rank[3][i] == rank) s_pick = i;
  __syncthreads();
  return s_pick;
}

// Programmatic dependent launch: wait for the grid this one depends on (no-op
// when the launch has no programmatic dependency) / let the next grid launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace pa
