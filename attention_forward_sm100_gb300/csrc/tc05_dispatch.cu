// Variant table of the tcgen05 kernel: static configuration and launch.
#include "fa_tc05.cuh"

namespace af {

Tc05Config tc05_config(int variant) {
  switch (variant) {
    case kVarD64: return tc05_config_t<TraitsD64>();
    case kVarD128: return tc05_config_t<TraitsD128>();
    case kVarD128Rope64: return tc05_config_t<TraitsD128R64>();
    case kVarFp8QkvD128: return tc05_config_t<TraitsFp8QkvD128>();
    case kVarD128Pair: return tc05_config_t<TraitsD128Pair>();
    case kVarD128Rope64Pair: return tc05_config_t<TraitsD128R64Pair>();
    default: return tc05_config_t<TraitsFp8D128>();
  }
}

cudaError_t tc05_launch(int variant, int mask, const Tc05Params& prm, int grid, cudaStream_t stream) {
  switch (variant) {
    case kVarD64: return tc05_launch_d64(mask, prm, grid, stream);
    case kVarD128: return tc05_launch_d128(mask, prm, grid, stream);
    case kVarD128Rope64: return tc05_launch_d128r64(mask, prm, grid, stream);
    case kVarFp8D128: return tc05_launch_fp8d128(mask, prm, grid, stream);
    case kVarFp8QkvD128: return tc05_launch_fp8qkvd128(mask, prm, grid, stream);
    case kVarD128Pair: return tc05_launch_d128pair(mask, prm, grid, stream);
    case kVarD128Rope64Pair: return tc05_launch_d128r64pair(mask, prm, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int tc05_max_clusters(int variant) {
  switch (variant) {
    case kVarD128Pair: return tc05_max_clusters_d128pair();
    case kVarD128Rope64Pair: return tc05_max_clusters_d128r64pair();
    default: return 0;
  }
}

}  // namespace af
