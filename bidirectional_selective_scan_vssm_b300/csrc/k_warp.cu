// Launch dispatch of the warp-per-channel-group scan (scan_warp.cuh); the
// kernel variants are instantiated in the k_warp_*.cu translation units.
#include "k_warp_opts.cuh"

namespace vssm {

cudaError_t launch_warp(const WarpScanParams &p, int dirs, bool f32, bool carry, bool sp, bool conv,
                        long long ctas, long long summ_ctas, cudaStream_t s)
{
    if (conv)
        return sp ? launch_warp_opts<true, true>(p, dirs, f32, carry, ctas, summ_ctas, s)
                  : launch_warp_opts<false, true>(p, dirs, f32, carry, ctas, summ_ctas, s);
    return sp ? launch_warp_opts<true, false>(p, dirs, f32, carry, ctas, summ_ctas, s)
              : launch_warp_opts<false, false>(p, dirs, f32, carry, ctas, summ_ctas, s);
}

}  // namespace vssm
