// Warp-per-channel-group scan variants with SP = true, CONV = false.
#include "k_warp_opts.cuh"

namespace vssm {
VSSM_WARP_OPTS_DEFINE(true, false)
}  // namespace vssm
