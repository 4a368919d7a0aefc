// Down projection of the grouped experts with the output rotation and the
// route-weighted combine epilogue (see expert_gemm.cuh).
#include "expert_gemm.cuh"

namespace exl3 {

cudaError_t launch_gemm_down(bool additive, int nrb, const GemmArgs &a, int grid,
                              cudaStream_t s)
{
    if (additive)
        return gemm::launch_one<kModeDown, 1, true>(a, grid, s);
    if (nrb == 2)
        return gemm::launch_one<kModeDown, 2, false>(a, grid, s);
    return gemm::launch_one<kModeDown, 1, false>(a, grid, s);
}

cudaError_t gemm_down_set_attributes()
{
    cudaError_t e = gemm::set_attr_one<kModeDown, 1, true>();
    if (e == cudaSuccess)
        e = gemm::set_attr_one<kModeDown, 1, false>();
    return e != cudaSuccess ? e : gemm::set_attr_one<kModeDown, 2, false>();
}

}  // namespace exl3
