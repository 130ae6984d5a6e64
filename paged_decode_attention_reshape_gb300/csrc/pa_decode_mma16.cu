// pa_decode_mma16.cu -- instantiations of the tensor-core decode kernel for
// bf16 and f16 caches (see pa_decode_mma.cuh).
#include "pa_decode_mma.cuh"

namespace pa {
namespace {

// f(MmaLaunch<kind, D>) for the instantiated shapes, else `other`.
template <int KIND, typename R, typename F>
R by_d(int D, R other, F f) {
  switch (D) {
    case 64: return f(MmaLaunch<KIND, 64>{});
    case 128: return f(MmaLaunch<KIND, 128>{});
    case 256: return f(MmaLaunch<KIND, 256>{});
    default: return other;
  }
}

template <typename R, typename F>
R by_kind(int kind, int D, R other, F f) {
  if (kind == KIND_BF16) return by_d<KIND_BF16>(D, other, f);
  if (kind == KIND_F16) return by_d<KIND_F16>(D, other, f);
  return other;
}

}  // namespace

cudaError_t launch_decode_mma_16(const DecodeParams &p, int kind, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                 cudaStream_t st) {
  return by_kind(kind, p.D, cudaErrorInvalidValue, [&](auto L) { return decltype(L)::launch(p, tmK, tmV, st); });
}

int occupancy_decode_mma_16(int kind, int D) {
  return by_kind(kind, D, 0, [](auto L) { return decltype(L)::occupancy(); });
}

}  // namespace pa
