// pa_chunk_mma16.cu -- instantiations of the tensor-memory query-tile kernel (see
// pa_chunk_umma.cuh) for bf16 and f16 caches, head sizes 64 and 128, one or two row tiles.
#include "pa_chunk_umma.cuh"

namespace pa {

cudaError_t launch_chunk_umma(const DecodeParams &p, int kind, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              const CUtensorMap &tmQ, cudaStream_t st) {
  // head size 128 with more than one tile of query rows per KV head: two 128-row tiles per
  // CTA share each page (measured faster there; at head size 64 one tile per CTA is faster)
  const bool two = p.D == 128 && p.nq_max * p.G > kChunkTwoTileColumns;
  if (kind == KIND_BF16 && p.D == 64) return UmmaLaunch<KIND_BF16, 64, 1>::launch(p, tmK, tmV, tmQ, st);
  if (kind == KIND_BF16 && p.D == 128)
    return two ? UmmaLaunch<KIND_BF16, 128, 2>::launch(p, tmK, tmV, tmQ, st)
               : UmmaLaunch<KIND_BF16, 128, 1>::launch(p, tmK, tmV, tmQ, st);
  if (kind == KIND_F16 && p.D == 64) return UmmaLaunch<KIND_F16, 64, 1>::launch(p, tmK, tmV, tmQ, st);
  if (kind == KIND_F16 && p.D == 128)
    return two ? UmmaLaunch<KIND_F16, 128, 2>::launch(p, tmK, tmV, tmQ, st) : UmmaLaunch<KIND_F16, 128, 1>::launch(p, tmK, tmV, tmQ, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
