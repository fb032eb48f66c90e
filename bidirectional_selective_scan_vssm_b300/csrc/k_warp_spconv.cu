// Warp-per-channel-group scan variants with SP = true, CONV = true.
#include "k_warp_opts.cuh"

namespace vssm {
VSSM_WARP_OPTS_DEFINE(true, true)
}  // namespace vssm
