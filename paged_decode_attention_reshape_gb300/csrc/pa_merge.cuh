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

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

template <typename OutT, int D>
__device__ __forceinline__ void merge_if_last(const DecodeParams &p, int s, int unit, int h0, int ng, int nparts,
                                              float vs, int threads) {
  __shared__ int s_last;
  __shared__ float s_md[8][2];
  __syncthreads();  // every partial store of this CTA has been issued
  if (threadIdx.x == 0) {
    __threadfence();  // ... and is visible device-wide before the arrival is counted
    const int old = atomicAdd(p.counters + unit, 1);
    const int last = old == nparts - 1;
    if (last) atomicExch(p.counters + unit, 0);
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = threads >> 5;
  for (int hh = warp; hh < ng; hh += nw) {
    const int64_t row0 = (static_cast<int64_t>(s) * p.Hq + h0 + hh) * p.max_parts;
    float M = -INFINITY;
    for (int i = lane; i < nparts; i += 32) M = fmaxf(M, __ldcg(p.part_ml + row0 + i).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float den = 0.f;
    for (int i = lane; i < nparts; i += 32) {
      const float2 v = __ldcg(p.part_ml + row0 + i);
      den += (v.x == -INFINITY ? 0.f : ex2(v.x - M)) * v.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (lane == 0) {
      s_md[hh][0] = M;
      s_md[hh][1] = den;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < ng * D; i += threads) {
    const int hh = i / D, d = i - hh * D;
    const float M = s_md[hh][0], den = s_md[hh][1];
    const int64_t row0 = (static_cast<int64_t>(s) * p.Hq + h0 + hh) * p.max_parts;
    float num = 0.f;
    for (int q = 0; q < nparts; ++q) {
      const float m = __ldcg(p.part_ml + row0 + q).x;
      const float w = m == -INFINITY ? 0.f : ex2(m - M);
      num += w * __ldcg(p.part_acc + (row0 + q) * D + d);
    }
    OutT *o = static_cast<OutT *>(p.out) + s * p.out_ss + static_cast<int64_t>(h0 + hh) * p.out_hs + d;
    *o = static_cast<OutT>(den > 0.f ? num / den * vs : 0.f);
  }
}

// Programmatic dependent launch: wait for the grid this one depends on (no-op
// when the launch has no programmatic dependency) / let the next grid launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace pa
