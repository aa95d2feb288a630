// Instantiation of the tcgen05 attention kernel for one head-dimension
// variant on CTA pairs.
#include "fa_tc05.cuh"

namespace af {
cudaError_t tc05_launch_d128r64pair(int mask, const Tc05Params& prm, int grid, cudaStream_t stream) {
  return tc05_launch_t<TraitsD128R64Pair>(mask, prm, grid, stream);
}
int tc05_max_clusters_d128r64pair() { return tc05_max_clusters_t<TraitsD128R64Pair>(); }
}  // namespace af
