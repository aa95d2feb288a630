// Instantiation of the tcgen05 attention kernel for one head-dimension variant.
#include "fa_tc05.cuh"

namespace af {
cudaError_t tc05_launch_fp8d128(int mask, const Tc05Params& prm, int grid, cudaStream_t stream) {
  return tc05_launch_t<TraitsFp8D128>(mask, prm, grid, stream);
}
}  // namespace af
