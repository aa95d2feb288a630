// Instantiation of the row-split attention kernel for one variant.
#include "fa_rowsplit.cuh"

namespace af {
cudaError_t rs_launch_fp8qkv(bool causal, const Tc05Params& prm, int grid, cudaStream_t stream) {
  return rs_launch_t<RsTraitsFp8Qkv>(causal, prm, grid, stream);
}
}  // namespace af
