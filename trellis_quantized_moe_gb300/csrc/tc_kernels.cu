// Prefill-regime (tcgen05 / TMEM) gate/up, down and linear kernels (see expert_tc.cuh).
#include "expert_tc.cuh"

namespace exl3 {

cudaError_t launch_tc_gateup(const GemmArgs &a, const TcMaps &maps, int grid, cudaStream_t s)
{
    return tc::launch_tc<kModeGateUp>(a, maps, grid, s);
}

cudaError_t launch_tc_down(const GemmArgs &a, const TcMaps &maps, int grid, cudaStream_t s)
{
    return tc::launch_tc<kModeDown>(a, maps, grid, s);
}

cudaError_t launch_tc_linear(const GemmArgs &a, const TcMaps &maps, int grid, cudaStream_t s)
{
    return tc::launch_tc<kModeLinear>(a, maps, grid, s);
}

cudaError_t tc_set_attributes()
{
    cudaError_t e = tc::set_attr_tc<kModeGateUp>();
    if (e == cudaSuccess)
        e = tc::set_attr_tc<kModeLinear>();
    return e != cudaSuccess ? e : tc::set_attr_tc<kModeDown>();
}

int tc_rows_per_item() { return tc::kNT; }

}  // namespace exl3
