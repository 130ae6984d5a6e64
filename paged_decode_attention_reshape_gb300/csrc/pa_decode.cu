// pa_decode.cu -- fp32 decode path, split-KV reduce, and decode kernel dispatch.
//
// The split-KV reduce follows "Inside vLLM CUDA Kernels", Part 3 ("Split-KV
// changes the work partition, not the softmax identity": partial states are
// rescaled to a common maximum before merging) and "vLLM 源码完全拆解（七）",
// V1 与 V2 (one reduce work item per (sequence, head) combining the partitions'
// max logits, exp sums and partial outputs).  Per (s, h):
//   M = max_p m_p,  out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p
// with m in log2 units, as the decode kernels write it.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// -------------------------------------------------------------------- reduce

template <typename OutT, int D>
__device__ __forceinline__ void store_row(OutT *o, const float (&v)[D / 32]) {
  constexpr int PER = D / 32;
#pragma unroll
  for (int i = 0; i < PER; ++i) o[i] = static_cast<OutT>(v[i]);
}

template <typename OutT, int D>
__global__ void __launch_bounds__(128) reduce_kernel(const DecodeParams p) {
  constexpr int PER = D / 32;  // contiguous d values per lane
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (item >= p.S * p.Hq) return;
  const int s = item / p.Hq, h = item - s * p.Hq;
  OutT *o = static_cast<OutT *>(p.out) + s * p.out_ss + static_cast<int64_t>(h) * p.out_hs + lane * PER;
  const int len = __ldg(p.seq_lens + s);
  float r[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) r[i] = 0.f;
  if (len < 0 || len > p.max_blocks * kBlock) return;  // flagged by the decode kernel
  const int np = ((len + kBlock - 1) / kBlock + p.pages_per_part - 1) / p.pages_per_part;
  if (np == 0) {
    store_row<OutT, D>(o, r);
    return;
  }
  const int64_t row0 = (static_cast<int64_t>(s) * p.Hq + h) * p.max_parts;
  const float2 *ml = p.part_ml + row0;
  float M = -INFINITY;
  for (int i = lane; i < np; i += 32) M = fmaxf(M, ml[i].x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float den = 0.f;
  const float *acc = p.part_acc + row0 * D + lane * PER;
#pragma unroll 4
  for (int i = 0; i < np; ++i) {
    const float2 v = ml[i];
    const float w = ex2(v.x - M);
    den += w * v.y;
    const float *a = acc + static_cast<int64_t>(i) * D;
    if constexpr (PER % 4 == 0) {
#pragma unroll
      for (int e = 0; e < PER; e += 4) {
        const float4 x = *reinterpret_cast<const float4 *>(a + e);
        r[e] += w * x.x;
        r[e + 1] += w * x.y;
        r[e + 2] += w * x.z;
        r[e + 3] += w * x.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < PER; e += 2) {
        const float2 x = *reinterpret_cast<const float2 *>(a + e);
        r[e] += w * x.x;
        r[e + 1] += w * x.y;
      }
    }
  }
  const float vs = p.v_scale ? __ldg(p.v_scale) : 1.f;
  const float inv = den > 0.f ? vs / den : 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) r[i] *= inv;
  store_row<OutT, D>(o, r);
}

template <typename OutT>
cudaError_t launch_reduce_t(const DecodeParams &p, cudaStream_t st) {
  const int items = p.S * p.Hq;
  const dim3 grid((items + 3) / 4);
  switch (p.D) {
    case 64: reduce_kernel<OutT, 64><<<grid, 128, 0, st>>>(p); break;
    case 128: reduce_kernel<OutT, 128><<<grid, 128, 0, st>>>(p); break;
    case 256: reduce_kernel<OutT, 256><<<grid, 128, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_reduce(const DecodeParams &p, int out_dtype, cudaStream_t st) {
  switch (out_dtype) {
    case PA_F32: return launch_reduce_t<float>(p, st);
    case PA_BF16: return launch_reduce_t<__nv_bfloat16>(p, st);
    case PA_F16: return launch_reduce_t<__half>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

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
  const int h0 = g * p.G + hg * 8;
  const int ng = min(8, p.G - hg * 8);
  const bool split = p.max_parts > 1;
  const int len = __ldg(p.seq_lens + s);
  if (len < 0 || len > p.max_blocks * kBlock) {
    if (threadIdx.x == 0 && part == 0 && blockIdx.y == 0 && p.err) atomicOr(p.err, kErrSeqLen);
    return;
  }
  const int npages = (len + kBlock - 1) / kBlock;
  const int pb = part * p.pages_per_part;
  const int pe = min(npages, pb + p.pages_per_part);
  if (pb >= pe) {
    if (!split && part == 0)
      for (int i = threadIdx.x; i < ng * D; i += W * 32)
        static_cast<float *>(p.out)[s * p.out_ss + static_cast<int64_t>(h0 + i / D) * p.out_hs + i % D] = 0.f;
    return;
  }
  float q[8][PER], acc[8][PER], m[8], l[8];
#pragma unroll
  for (int hh = 0; hh < 8; ++hh) {
    const int h = h0 + min(hh, ng - 1);
    const float *qr = static_cast<const float *>(p.q) + s * p.q_ss + static_cast<int64_t>(h) * p.q_hs;
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
#pragma unroll
      for (int hh = 0; hh < 8; ++hh) {
        if (hh < ng) {
          float z = 0.f;
#pragma unroll
          for (int i = 0; i < PER; ++i) z = fmaf(q[hh][i], kr[i], z);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
          z *= p.scale_log2;
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
  if (__syncthreads_or(bad)) return;
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
    const int h = h0 + hh;
    if (!split) {
      static_cast<float *>(p.out)[s * p.out_ss + static_cast<int64_t>(h) * p.out_hs + d] = den > 0.f ? num / den : 0.f;
    } else {
      const int64_t row = (static_cast<int64_t>(s) * p.Hq + h) * p.max_parts + part;
      p.part_acc[row * D + d] = num;
      if (d == 0) p.part_ml[row] = make_float2(M, den);
    }
  }
}

cudaError_t launch_decode_f32(const DecodeParams &p, cudaStream_t st) {
  const dim3 grid(p.max_parts, p.Hkv * p.HG, p.S);
  switch (p.D) {
    case 64: decode_f32_kernel<64, 4><<<grid, 128, 0, st>>>(p); break;
    case 128: decode_f32_kernel<128, 4><<<grid, 128, 0, st>>>(p); break;
    case 256: decode_f32_kernel<256, 2><<<grid, 64, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace pa
