// exl3_linear_noalloc: the EXL3 linear for callers that cannot allocate device
// memory themselves -- for example code running inside a CUDA graph that is
// re-instantiated without a memory pool, plug-in hosts that forbid cudaMalloc
// outside their own allocator, or latency-critical paths where an allocation
// would synchronise the device.  Instead of a caller-provided workspace it
// uses one fixed scratch array that lives in this library's device image.
//
// The scratch is a file-scope __device__ array.  Its host-side name is only a
// stand-in for the symbol, not a device address, so the address is looked up
// with cudaGetSymbolAddress once per device (on the first call made with that
// device current) and cached.  Make that first call before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"

namespace {

// 32 MiB per device, held by every GPU that loads the library until exit.
constexpr size_t kNoAllocScratchBytes = 32u << 20;
__device__ __align__(256) uint8_t g_linear_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
void *g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;

int scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return EXL3_E_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_linear_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return EXL3_E_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return EXL3_OK;
}

}  // namespace

extern "C" {

size_t exl3_linear_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

int exl3_linear_noalloc(const void *x, int act_dtype, int M, const exl3_proj *proj, void *y,
                        cudaStream_t stream)
{
    if (!proj)
        return EXL3_E_NULL;
    if (M < 0 || proj->in_features <= 0 || proj->out_features <= 0 ||
        proj->in_features % exl3::kHb || proj->out_features % exl3::kHb)
        return EXL3_E_SHAPE;
    const size_t need = exl3::linear_layout(M, proj->in_features, proj->out_features).total;
    if (need > kNoAllocScratchBytes)
        return EXL3_E_WORKSPACE;   // this M x in x out needs more than the fixed scratch
    void *scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc != EXL3_OK)
        return rc;
    return exl3_linear(x, act_dtype, M, proj, y, scratch, kNoAllocScratchBytes, stream);
}

// The device error word that the last exl3_linear_noalloc call on the current
// device left in the fixed scratch (0: no device-side error).  Waits for the
// stream, like exl3_workspace_error; never call it while capturing.
int exl3_linear_noalloc_error(int32_t *err_host, cudaStream_t stream)
{
    if (!err_host)
        return EXL3_E_NULL;
    void *scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc != EXL3_OK)
        return rc;
    return exl3_workspace_error(scratch, err_host, stream);
}

}  // extern "C"
