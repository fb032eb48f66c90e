// Warp-per-channel-group scan variants with SP = false, CONV = true.
#include "k_warp_opts.cuh"

namespace vssm {
VSSM_WARP_OPTS_DEFINE(false, true)
}  // namespace vssm
