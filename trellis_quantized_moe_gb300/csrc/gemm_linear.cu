// The standalone EXL3 linear (one projection, rows in groups of 16; see
// expert_gemm.cuh).
#include "expert_gemm.cuh"

namespace exl3 {

cudaError_t launch_gemm_linear(const GemmArgs &a, int grid, cudaStream_t s)
{
    return gemm::launch_one<kModeLinear, 2, false>(a, grid, s);
}

cudaError_t gemm_linear_set_attributes()
{
    return gemm::set_attr_one<kModeLinear, 2, false>();
}

}  // namespace exl3
