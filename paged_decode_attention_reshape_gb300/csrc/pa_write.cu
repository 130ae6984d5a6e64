// pa_write.cu -- the paged KV-cache write (slot_mapping scatter).
//
// Follows "Inside vLLM CUDA Kernels: KV-Cache Writes and Paged Attention",
// Part 2: each new token has one destination slot; slot < 0 means padding with
// no destination; slot -> (block = slot / 16, offset = slot % 16); the element
// conversion is a copy, or scale-and-convert for an FP8 cache.
//
// GB300 design: the work item is one 16-byte pack of one (token, kv head) row,
// for K and V together.  A 256-thread block covers whole tokens (adjacent threads
// take adjacent packs of the source: fully coalesced reads), so each thread's
// token and pack indices are fixed and the loop is a stride over tokens; each
// destination (block, head, offset) row is a contiguous run of D * elem bytes in
// the HND cache, so a warp's stores cover whole 32-byte sectors.  Sources are read
// once with no L1 allocation.  The grid is one resident wave (4 CTAs per SM) striding
// over tokens, each thread streaming its tokens through a two-deep software pipeline.
// The E4M3 path divides by the tensor's scale, or its KV head's
// (Part 2: kv_scale_stride == 0 shares one scale, otherwise head h uses
// scale[h * kv_scale_stride]), with a reciprocal-based, correctly rounded quotient
// (Divisor below), the same value as an IEEE division.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ __forceinline__ uint4 ld_once(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Element type codes for the template (match pa_dtype values).
template <int DT> struct In;
template <> struct In<PA_F32> { static constexpr int bytes = 4; };
template <> struct In<PA_BF16> { static constexpr int bytes = 2; };
template <> struct In<PA_F16> { static constexpr int bytes = 2; };

template <int DT>
__device__ __forceinline__ void unpack8(const uint4 &v, float (&x)[16 / In<DT>::bytes]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (DT == PA_F32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = __uint_as_float(w[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = (DT == PA_BF16) ? unpack_bf16(w[i]) : unpack_f16(w[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
}

// The correctly rounded quotient x / s for one divisor s shared by a whole tensor.
// With y = RN(1/s): q0 = RN(x y) is within 1.5 ulp of x/s; one correction
// q1 = RN(q0 + (x - q0 s) y) brings it within 1 ulp, and then (Markstein's theorem:
// y within half an ulp of 1/s, q1 within one ulp of x/s, residual x - q1 s exact by
// FMA) q2 = RN(q1 + (x - q1 s) y) is RN(x/s).  The theorem needs the operands and the
// residuals away from underflow and overflow, so zero, tiny, huge, infinite or NaN x
// (and divisors outside [2^-40, 2^40]) take the general IEEE division instead.
struct Divisor {
  float s, y;
  bool fast;
  __device__ __forceinline__ static bool in_range(float x) {
    const float ax = fabsf(x);
    return ax >= 0x1p-80f && ax <= 0x1p80f;  // false for zero, subnormals, inf, NaN
  }
  __device__ __forceinline__ float div(float x) const {
    if (fast && in_range(x)) {
      float q = __fmul_rn(x, y);
      float r = __fmaf_rn(-q, s, x);
      q = __fmaf_rn(r, y, q);
      r = __fmaf_rn(-q, s, x);
      return __fmaf_rn(r, y, q);
    }
    return __fdiv_rn(x, s);
  }
  // The same correctly rounded steps on two operands at once (packed fp32x2 operations,
  // each lane an IEEE round-to-nearest multiply / fused multiply-add); the caller has
  // checked fast and in_range for both.
  __device__ __forceinline__ float2 div2_fast(float a, float b) const {
    uint64_t x, sy, ns, q, r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
    asm("mov.b64 %0, {%1, %1};" : "=l"(sy) : "f"(y));
    asm("mov.b64 %0, {%1, %1};" : "=l"(ns) : "f"(-s));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q) : "l"(x), "l"(sy));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(q), "l"(ns), "l"(x));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(q) : "l"(r), "l"(sy));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(q), "l"(ns), "l"(x));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(q) : "l"(r), "l"(sy));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(q));
    return o;
  }
};

__device__ __forceinline__ Divisor make_divisor(float s) {
  Divisor d;
  d.s = s;
  d.y = __frcp_rn(s);
  const float as = fabsf(s);
  d.fast = as >= 0x1p-40f && as <= 0x1p40f;
  return d;
}

// min(|x|, 2^80), NaN for a NaN x.
__device__ __forceinline__ float clamp_mag(float x) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(fabsf(x)), "f"(0x1p80f));
  return r;
}

// E4M3 code pair of two quotients (cvt ... satfinite: round-to-nearest-even with
// saturation); low byte = a.
__device__ __forceinline__ uint32_t e4m3_pair(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// One 16-byte pack of inputs -> E4M3 codes of x / scale (correctly rounded quotient).
// 16-bit inputs: the codes of |x| / |s| are computed with |x| clamped to 2^80 (a NaN stays
// NaN), which keeps the fused steps exact for every input -- nothing overflows, and a |x|
// small enough for the steps to lose exactness gives a quotient far below the smallest E4M3
// value -- and the sign of x / s is put back on each code (round to nearest even and
// saturation are symmetric in the sign).  Zero, infinite and NaN inputs then need no branch.
template <int DT>
__device__ __forceinline__ void store_fp8(char *dst, const uint4 &v, const Divisor &dv) {
  constexpr int E = 16 / In<DT>::bytes;
  float x[E], q[E];
  unpack8<DT>(v, x);
  if constexpr (E == 8) {
    if (dv.fast) {
      const Divisor da{fabsf(dv.s), fabsf(dv.y), true};
#pragma unroll
      for (int i = 0; i < E; i += 2) {
        const float2 r = da.div2_fast(clamp_mag(x[i]), clamp_mag(x[i + 1]));
        q[i] = r.x;
        q[i + 1] = r.y;
      }
      // sign bits of elements 0..3 and 4..7 (bit 15 of each 16-bit input) into bit 7 of
      // each code byte, flipped for a negative scale
      const uint32_t neg = dv.s < 0.f ? 0x80808080u : 0u;
      uint2 o;
      o.x = e4m3_pair(q[0], q[1]) | (e4m3_pair(q[2], q[3]) << 16);
      o.y = e4m3_pair(q[4], q[5]) | (e4m3_pair(q[6], q[7]) << 16);
      o.x |= (__byte_perm(v.x, v.y, 0x7531) ^ neg) & 0x80808080u;
      o.y |= (__byte_perm(v.z, v.w, 0x7531) ^ neg) & 0x80808080u;
      *reinterpret_cast<uint2 *>(dst) = o;
      return;
    }
  }
  bool fast = dv.fast;
#pragma unroll
  for (int i = 0; i < E; ++i) fast &= Divisor::in_range(x[i]);
  if (fast) {
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const float2 r = dv.div2_fast(x[i], x[i + 1]);
      q[i] = r.x;
      q[i + 1] = r.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) q[i] = dv.div(x[i]);
  }
  if constexpr (E == 8) {
    uint2 o;
    o.x = e4m3_pair(q[0], q[1]) | (e4m3_pair(q[2], q[3]) << 16);
    o.y = e4m3_pair(q[4], q[5]) | (e4m3_pair(q[6], q[7]) << 16);
    *reinterpret_cast<uint2 *>(dst) = o;
  } else {
    *reinterpret_cast<uint32_t *>(dst) = e4m3_pair(q[0], q[1]) | (e4m3_pair(q[2], q[3]) << 16);
  }
}

// CTAs per SM of the grid (at most the resident ones, the launch bound), so that every CTA
// is in flight from the start and streams its tokens through the software pipeline.
// Measured on GB300, two-deep pipeline: the 8192-row E4M3 chunk with 1, 2, 3, 4 CTAs per SM
// 23.9, 16.5, 14.8, 15.4 us, the 32768-row bf16 copy with 3 or 4 45.5 / 43.9 us; two batched
// turns per thread over two waves 18.5 us; a three-deep pipeline no faster; 5 or 6 CTAs per SM
// (registers spill) 16.5 / 18.4 us.  (pa_decode_step asks for fewer when the decode overlaps
// the write.)
constexpr int kWriteCtasPerSmFp8 = 3, kWriteCtasPerSmCopy = 4;

template <int DT, bool FP8, bool I32>
__global__ void __launch_bounds__(256, 4) write_kernel(const WriteParams p) {
  // the decode that usually follows waits for this grid's completion before its first
  // read (griddepcontrol.wait), so it may be scheduled now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int IB = In<DT>::bytes;
  constexpr int EPP = 16 / IB;            // elements per 16-byte pack
  constexpr int CB = FP8 ? 1 : IB;        // cache element bytes
  const int ppr = p.D / EPP;              // packs per (token, head) row
  const int per_tok = p.Hkv * ppr;        // packs per token
  // thread -> (token within the block's rows, pack within the token), fixed for the kernel;
  // a token wider than the block is covered by an inner loop over packs
  const int width = min(per_tok, 256);
  const int rows = 256 / width;
  const int tl = threadIdx.x / width;
  const int j0 = threadIdx.x - tl * width;
  if (tl >= rows) return;  // spare threads when 256 is not a multiple of per_tok
  // FP8 scales: one per tensor, or one per KV head (head h at [h * scale_stride]).  A
  // thread's packs belong to one head unless a token is wider than the block.
  int hcur = j0 / ppr;
  Divisor kdiv{}, vdiv{};
  if (FP8) {
    kdiv = make_divisor(p.k_scale ? __ldg(p.k_scale + hcur * p.scale_stride) : 1.f);
    vdiv = make_divisor(p.v_scale ? __ldg(p.v_scale + hcur * p.scale_stride) : 1.f);
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * rows;  // tokens between a thread's turns
  if (per_tok <= 256) {
    // The thread's pack is fixed (head hcur, element e).
    const int64_t e = static_cast<int64_t>(j0 - hcur * ppr) * EPP;
    const char *ks = static_cast<const char *>(p.key) + (hcur * p.key_hs + e) * IB;
    const char *vs = static_cast<const char *>(p.value) + (hcur * p.val_hs + e) * IB;
    // Software pipeline over the thread's tokens: the slot and both source packs of the next
    // token are in flight while the current one is converted and stored.  (Padding rows are
    // loaded too; their sources are in bounds and nothing is written for them.)
    // byte offsets: within a block and between tokens they fit 32 bits (I32); a block's
    // offset is one widening multiply
    const int64_t kin = (hcur * p.kc_s1 + e) * CB, vin = (hcur * p.vc_s1 + e) * CB;
    auto process = [&](int64_t slot, const uint4 &kv, const uint4 &vv) {
      if (slot < 0) return;  // padding row (or past the end): no destination
      if (slot >= p.num_slots) {
        if (p.err && j0 == 0) atomicOr(p.err, kErrSlot);
        return;
      }
      char *kd, *vd;
      if constexpr (I32) {
        const int blk = static_cast<int>(slot >> 4), off = static_cast<int>(slot & 15);
        kd = static_cast<char *>(p.k_cache) + static_cast<int64_t>(blk) * static_cast<int>(p.kc_s0 * CB) +
             (static_cast<int>(kin) + off * static_cast<int>(p.kc_s2 * CB));
        vd = static_cast<char *>(p.v_cache) + static_cast<int64_t>(blk) * static_cast<int>(p.vc_s0 * CB) +
             (static_cast<int>(vin) + off * static_cast<int>(p.vc_s2 * CB));
      } else {
        const int64_t blk = slot / kBlock, off = slot % kBlock;
        kd = static_cast<char *>(p.k_cache) + (blk * p.kc_s0 + off * p.kc_s2) * CB + kin;
        vd = static_cast<char *>(p.v_cache) + (blk * p.vc_s0 + off * p.vc_s2) * CB + vin;
      }
      if constexpr (!FP8) {
        *reinterpret_cast<uint4 *>(kd) = kv;
        *reinterpret_cast<uint4 *>(vd) = vv;
      } else {
        store_fp8<DT>(kd, kv, kdiv);
        store_fp8<DT>(vd, vv, vdiv);
      }
    };
    auto src = [&](const char *base, int64_t tt, int64_t ts) {
      if constexpr (I32) return base + static_cast<int>(tt) * static_cast<int>(ts * IB);
      else return base + tt * ts * IB;
    };
    int64_t t = static_cast<int64_t>(blockIdx.x) * rows + tl;
    int64_t slot = -1;
    uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
    if (t < p.T) {
      slot = __ldg(p.slot_mapping + t);
      kv = ld_once(src(ks, t, p.key_ts));
      vv = ld_once(src(vs, t, p.val_ts));
    }
    while (t < p.T) {
      const int64_t tn = t + stride;
      int64_t slot_n = -1;
      uint4 kvn = kv, vvn = vv;
      if (tn < p.T) {
        slot_n = __ldg(p.slot_mapping + tn);
        kvn = ld_once(src(ks, tn, p.key_ts));
        vvn = ld_once(src(vs, tn, p.val_ts));
      }
      process(slot, kv, vv);
      t = tn;
      slot = slot_n;
      kv = kvn;
      vv = vvn;
    }
    return;
  }
  // a token wider than the block: an inner loop over its packs
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * rows + tl; t < p.T; t += stride) {
    const int64_t slot = __ldg(p.slot_mapping + t);
    if (slot < 0) continue;  // padding row: no destination
    if (slot >= p.num_slots) {
      if (p.err && j0 == 0) atomicOr(p.err, kErrSlot);
      continue;
    }
    const int64_t blk = slot / kBlock, off = slot % kBlock;
    for (int j = j0; j < per_tok; j += 256) {
      const int h = j / ppr;
      if (FP8 && p.scale_stride != 0 && h != hcur) {
        hcur = h;
        kdiv = make_divisor(p.k_scale ? __ldg(p.k_scale + h * p.scale_stride) : 1.f);
        vdiv = make_divisor(p.v_scale ? __ldg(p.v_scale + h * p.scale_stride) : 1.f);
      }
      const int64_t e = static_cast<int64_t>(j - h * ppr) * EPP;
      const uint4 kv = ld_once(static_cast<const char *>(p.key) + (t * p.key_ts + h * p.key_hs + e) * IB);
      const uint4 vv = ld_once(static_cast<const char *>(p.value) + (t * p.val_ts + h * p.val_hs + e) * IB);
      char *kd = static_cast<char *>(p.k_cache) + (blk * p.kc_s0 + h * p.kc_s1 + off * p.kc_s2 + e) * CB;
      char *vd = static_cast<char *>(p.v_cache) + (blk * p.vc_s0 + h * p.vc_s1 + off * p.vc_s2 + e) * CB;
      if constexpr (!FP8) {
        *reinterpret_cast<uint4 *>(kd) = kv;
        *reinterpret_cast<uint4 *>(vd) = vv;
      } else {
        store_fp8<DT>(kd, kv, kdiv);
        store_fp8<DT>(vd, vv, vdiv);
      }
    }
  }
}

template <int DT, bool FP8>
cudaError_t launch_one(const WriteParams &p, int sm_count, int ctas_per_sm, cudaStream_t st) {
  constexpr int EPP = 16 / In<DT>::bytes;
  const int per_tok = p.Hkv * (p.D / EPP);
  const int rows = 256 / (per_tok < 256 ? per_tok : 256);
  int64_t blocks = (p.T + rows - 1) / rows;
  const int per_sm = ctas_per_sm > 0 && ctas_per_sm <= 4 ? ctas_per_sm : FP8 ? kWriteCtasPerSmFp8 : kWriteCtasPerSmCopy;
  const int64_t cap = static_cast<int64_t>(sm_count) * per_sm;  // one resident wave, grid-stride
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  // the write uses no shared memory and reads around L1; keep the SM's shared/L1 split the
  // decode kernels ask for, so the usual write -> decode sequence does not reconfigure it
  auto kern = p.i32 ? write_kernel<DT, FP8, true> : write_kernel<DT, FP8, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(blocks), 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_write(const WriteParams &p, int in_dtype, int cache_dtype, int sm_count, int ctas_per_sm,
                         cudaStream_t st) {
  const bool fp8 = cache_dtype == PA_FP8_E4M3;
  const int c = ctas_per_sm;
  switch (in_dtype) {
    case PA_F32: return fp8 ? launch_one<PA_F32, true>(p, sm_count, c, st) : launch_one<PA_F32, false>(p, sm_count, c, st);
    case PA_BF16: return fp8 ? launch_one<PA_BF16, true>(p, sm_count, c, st) : launch_one<PA_BF16, false>(p, sm_count, c, st);
    case PA_F16: return fp8 ? launch_one<PA_F16, true>(p, sm_count, c, st) : launch_one<PA_F16, false>(p, sm_count, c, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
