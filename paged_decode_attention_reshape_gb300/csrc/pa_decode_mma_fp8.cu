// pa_decode_mma_fp8.cu -- instantiations of the tensor-core decode kernel for
// E4M3 caches with a bf16 or f16 query (see pa_decode_mma.cuh).
#include "pa_decode_mma.cuh"

namespace pa {
namespace {

// f(MmaLaunch<kind, D>) for the instantiated shapes, else `other`.
template <int KIND, typename R, typename F>
R by_d(int D, R other, F f) {
  switch (D) {
    case 128: return f(MmaLaunch<KIND, 128>{});
    case 256: return f(MmaLaunch<KIND, 256>{});
    default: return other;
  }
}

template <typename R, typename F>
R by_kind(int kind, int D, R other, F f) {
  if (kind == KIND_FP8_BF16Q) return by_d<KIND_FP8_BF16Q>(D, other, f);
  if (kind == KIND_FP8_F16Q) return by_d<KIND_FP8_F16Q>(D, other, f);
  return other;
}

}  // namespace

cudaError_t launch_decode_mma_fp8(const DecodeParams &p, int kind, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                 cudaStream_t st) {
  return by_kind(kind, p.D, cudaErrorInvalidValue, [&](auto L) { return decltype(L)::launch(p, tmK, tmV, st); });
}

int occupancy_decode_mma_fp8(int kind, int D) {
  return by_kind(kind, D, 0, [](auto L) { return decltype(L)::occupancy(); });
}

}  // namespace pa
