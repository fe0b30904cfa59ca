// dh_coarse_tc.cu -- kernels (2)+(3), tcgen05 path (tensor memory accumulators).
#include "dh_common.cuh"
#include "dh_internal.h"

namespace dh {

int tc_npad(int M)
{
    return ((M + 15) / 16) * 16;
}

bool tc_supported(int M, int H)
{
    (void)M;
    (void)H;
    return false;
}

cudaError_t launch_coarse_tc(const CoarseArgs &a, cudaStream_t stream)
{
    (void)a;
    (void)stream;
    return cudaErrorNotSupported;
}

} // namespace dh
