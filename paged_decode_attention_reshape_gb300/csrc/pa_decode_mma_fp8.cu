// pa_decode_mma_fp8.cu -- instantiations of the tensor-core decode kernel for
// E4M3 caches with a bf16 or f16 query (see pa_decode_mma.cuh).
#include "pa_decode_mma.cuh"

namespace pa {
namespace {

template <int KIND, int D>
cudaError_t go(const DecodeParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV, cudaStream_t st) {
  constexpr int W = mma_warps(KIND, D), ST = mma_stages(KIND, D);
  using C = MmaCfg<KIND, D, W, ST>;
  static_assert(C::SMEM == mma_smem(KIND, D), "shape table out of sync");
  auto kern = decode_mma_kernel<KIND, D, W, ST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  // same shared/L1 split as the cache write that usually precedes it (no reconfiguration)
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.max_parts, p.Hkv * p.HG, p.S);
  e = launch_pdl(kern, grid, dim3(C::THREADS), C::SMEM, st, p.cluster, p, tmK, tmV);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int KIND>
cudaError_t by_d(const DecodeParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV, cudaStream_t st) {
  switch (p.D) {
    case 128: return go<KIND, 128>(p, tmK, tmV, st);
    case 256: return go<KIND, 256>(p, tmK, tmV, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_mma_fp8(const DecodeParams &p, int kind, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                  cudaStream_t st) {
  if (kind == KIND_FP8_BF16Q) return by_d<KIND_FP8_BF16Q>(p, tmK, tmV, st);
  if (kind == KIND_FP8_F16Q) return by_d<KIND_FP8_F16Q>(p, tmK, tmV, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
