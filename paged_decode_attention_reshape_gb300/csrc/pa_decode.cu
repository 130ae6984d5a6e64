// pa_decode.cu -- the fp32 decode path (CUDA cores).
#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_merge.cuh"

namespace pa {

// ---------------------------------------------------------------- fp32 path
//
// CUDA-core decode for fp32 caches (exact fp32 products; no 16-bit operand).
// Same work unit and merge as the tensor-core kernel.  Each warp walks its pages
// token by token: the 32 lanes hold D/32 strided elements of the K/V rows
// (coalesced 128-byte loads), one butterfly reduction per (token, head) gives
// the score, and the per-head online-softmax state is kept in registers.

template <int D, int W>
__global__ void __launch_bounds__(W * 32) decode_f32_kernel(const DecodeParams p) {
  constexpr int PER = D / 32;
  __shared__ float sm[W][8][D + 2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int s = blockIdx.z, part = blockIdx.x;
  const int g = blockIdx.y / p.HG, hg = blockIdx.y - g * p.HG;
  const int v0 = hg * 8;  // first column (virtual head) of this CTA, see DecodeParams
  int ng = min(8, p.VH - v0);
  const bool split = p.max_parts > 1;
  grid_dependency_wait();
  const int len = __ldg(p.seq_lens + s);
  if (len < 0 || len > p.max_blocks * kBlock) {
    if (threadIdx.x == 0 && part == 0 && blockIdx.y == 0 && p.err) atomicOr(p.err, kErrSeqLen);
    return;
  }
  int64_t row0 = s;  // the sequence's query tokens: one (decode) or rows qsl[s] .. qsl[s+1]-1
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
  ng = min(ng, nq * p.G - v0);
  if (ng <= 0) return;
  const Cols cm{row0, p.G, g, v0};
  const int pos0 = len - nq;  // column hh sees the tokens up to pos0 + (v0 + hh) / G
  const int npages = (pos0 + (v0 + ng - 1) / p.G + 1 + kBlock - 1) / kBlock;
  const bool clustered = p.cluster > 1;  // rank `part` of a cluster splitting the unit equally
  const int pb = clustered ? static_cast<int>(static_cast<int64_t>(part) * npages / p.cluster) : part * p.pages_per_part;
  const int pe = clustered ? static_cast<int>(static_cast<int64_t>(part + 1) * npages / p.cluster)
                           : min(npages, pb + p.pages_per_part);
  if (pb >= pe && !clustered) {
    if (npages == 0 && part == 0)  // empty sequence (any split): zero output rows
      for (int i = threadIdx.x; i < ng * D; i += W * 32) static_cast<float *>(p.out)[cm.out_off(p, i / D) + i % D] = 0.f;
    return;
  }
  float q[8][PER], acc[8][PER], m[8], l[8], ab[8];
  int pos[8];
#pragma unroll
  for (int hh = 0; hh < 8; ++hh) {
    // last visible position (causal) and ALiBi slope in log2 units (0 without ALiBi):
    // logit += slope * (t - pos)
    pos[hh] = hh < ng ? pos0 + (v0 + hh) / p.G : -1;
    ab[hh] = (p.alibi && hh < ng) ? __ldg(p.alibi + cm.head(hh)) * 1.4426950408889634f : 0.f;
    const float *qr = static_cast<const float *>(p.q) + cm.q_off(p, min(hh, ng - 1));
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      q[hh][i] = hh < ng ? __ldg(qr + lane + 32 * i) : 0.f;
      acc[hh][i] = 0.f;
    }
    m[hh] = -INFINITY;
    l[hh] = 0.f;
  }
  bool bad = false;
  const int32_t *bt = p.block_table + static_cast<int64_t>(s) * p.bt_ss;
  for (int page = pb + warp; page < pe; page += W) {
    const int pid = __ldg(bt + page);
    if (pid < 0 || pid >= p.num_blocks) {
      bad = true;
      if (lane == 0 && p.err) atomicOr(p.err, kErrBlock);
      continue;
    }
    const int nv = min(kBlock, len - page * kBlock);
    const float *kbase = p.kc + static_cast<int64_t>(pid) * p.kc_s0 + static_cast<int64_t>(g) * p.kc_s1;
    const float *vbase = p.vc + static_cast<int64_t>(pid) * p.vc_s0 + static_cast<int64_t>(g) * p.vc_s1;
    for (int t = 0; t < nv; ++t) {
      float kr[PER], vr[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        kr[i] = __ldg(kbase + t * p.kc_s2 + lane + 32 * i);
        vr[i] = __ldg(vbase + t * p.vc_s2 + lane + 32 * i);
      }
      const int tt = page * kBlock + t;  // the token's position
#pragma unroll
      for (int hh = 0; hh < 8; ++hh) {
        if (tt <= pos[hh]) {  // visible to this column (never for hh >= ng)
          float z = 0.f;
#pragma unroll
          for (int i = 0; i < PER; ++i) z = fmaf(q[hh][i], kr[i], z);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
          z = fmaf(ab[hh], static_cast<float>(tt - pos[hh]), z * p.scale_log2);
          const float mn = fmaxf(m[hh], z);
          const float al = ex2(m[hh] - mn);
          const float pz = ex2(z - mn);
          l[hh] = l[hh] * al + pz;
#pragma unroll
          for (int i = 0; i < PER; ++i) acc[hh][i] = acc[hh][i] * al + pz * vr[i];
          m[hh] = mn;
        }
      }
    }
  }
#pragma unroll
  for (int hh = 0; hh < 8; ++hh) {
#pragma unroll
    for (int i = 0; i < PER; ++i) sm[warp][hh][lane + 32 * i] = acc[hh][i];
    if (lane == 0) {
      sm[warp][hh][D] = m[hh];
      sm[warp][hh][D + 1] = l[hh];
    }
  }
  const bool any_bad = __syncthreads_or(bad);
  if (clustered) {
    // CTA state in place over warp 0's slots (each element is read and overwritten by one thread)
    __shared__ float2 cmd[8];
    __shared__ int cbad;
    if (!any_bad) {
      for (int i = threadIdx.x; i < ng * D; i += W * 32) {
        const int hh = i / D, d = i - hh * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, sm[w][hh][D]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float mw = sm[w][hh][D];
          const float sc = (mw == -INFINITY) ? 0.f : ex2(mw - M);
          den += sc * sm[w][hh][D + 1];
          num += sc * sm[w][hh][d];
        }
        sm[0][hh][d] = num;
        if (d == 0) cmd[hh] = make_float2(M, den);
      }
    }
    cluster_merge_write<float, D>(p, cm, ng, 1.f, any_bad, &sm[0][0][0], D + 2, cmd, &cbad, W * 32);
    return;
  }
  const int nparts = split ? (npages + p.pages_per_part - 1) / p.pages_per_part : 1;
  const bool direct = nparts == 1;
  const FixedRows rows{(static_cast<int64_t>(s) * p.Hkv + g) * p.VH + v0, p.max_parts};
  if (!any_bad) {
    for (int i = threadIdx.x; i < ng * D; i += W * 32) {
      const int hh = i / D, d = i - hh * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < W; ++w) M = fmaxf(M, sm[w][hh][D]);
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float mw = sm[w][hh][D];
        const float sc = (mw == -INFINITY) ? 0.f : ex2(mw - M);
        den += sc * sm[w][hh][D + 1];
        num += sc * sm[w][hh][d];
      }
      if (direct) {
        static_cast<float *>(p.out)[cm.out_off(p, hh) + d] = den > 0.f ? num / den : 0.f;
      } else {
        const int64_t row = rows(hh, part);
        p.part_acc[row * D + d] = num;
        if (d == 0) p.part_ml[row] = make_float2(M, den);
      }
    }
  }
  static_assert(sizeof(sm) >= 8 * kMergeSmemParts * 4, "merge weights reuse sm");
  if (!direct)
    merge_if_last<float, D>(p, cm, static_cast<int>(blockIdx.y) + p.Hkv * p.HG * s, ng, nparts, 1.f, any_bad,
                            W * 32, &sm[0][0][0], rows);
}

cudaError_t launch_decode_f32(const DecodeParams &p, cudaStream_t st) {
  const dim3 grid(p.max_parts, p.Hkv * p.HG, p.S);
  cudaError_t e;
  switch (p.D) {
    case 64: e = launch_pdl(decode_f32_kernel<64, 4>, grid, dim3(128), 0, st, p.cluster, p); break;
    case 128: e = launch_pdl(decode_f32_kernel<128, 4>, grid, dim3(128), 0, st, p.cluster, p); break;
    case 256: e = launch_pdl(decode_f32_kernel<256, 2>, grid, dim3(64), 0, st, p.cluster, p); break;
    default: return cudaErrorInvalidValue;
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pa
