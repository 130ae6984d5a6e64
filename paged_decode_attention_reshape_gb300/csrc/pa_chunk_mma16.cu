// pa_chunk_mma16.cu -- instantiations of the tensor-memory query-tile kernel (see
// pa_chunk_umma.cuh) for bf16 and f16 caches, head sizes 64 and 128.
#include "pa_chunk_umma.cuh"

namespace pa {

cudaError_t launch_chunk_umma(const DecodeParams &p, int kind, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              cudaStream_t st) {
  if (kind == KIND_BF16 && p.D == 64) return UmmaLaunch<KIND_BF16, 64>::launch(p, tmK, tmV, st);
  if (kind == KIND_BF16 && p.D == 128) return UmmaLaunch<KIND_BF16, 128>::launch(p, tmK, tmV, st);
  if (kind == KIND_F16 && p.D == 64) return UmmaLaunch<KIND_F16, 64>::launch(p, tmK, tmV, st);
  if (kind == KIND_F16 && p.D == 128) return UmmaLaunch<KIND_F16, 128>::launch(p, tmK, tmV, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
