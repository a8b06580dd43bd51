// decode_mma.cu -- tensor-core consumer of the split-K paged decode (placeholder:
// forwards to the CUDA-core consumer until the mma.sync tiles land).
#include "decode.cuh"

namespace ekv {
cudaError_t launch_split_simt(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                              const DecodeParams& p, int D, int vmode, int grid, cudaStream_t st);

cudaError_t launch_split_mma(const CUtensorMap& tk, const CUtensorMap& t8, const CUtensorMap& t16,
                             const DecodeParams& p, int D, int vmode, int grid, cudaStream_t st) {
  return launch_split_simt(tk, t8, t16, p, D, vmode, grid, st);
}
}  // namespace ekv
