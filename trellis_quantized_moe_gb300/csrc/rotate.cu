// Input rotation a' = Hb(x * suh) ("EXL3 linear and grouped routed experts",
// TensorFold #837, "What this changes": the input rotation, each expert's
// rotation).  One warp per (row, projection); lane l holds 4 consecutive
// features of each 128-block; the 128-point Hadamard runs in registers and
// warp shuffles.  Output is fp16 (the MMA operand), one row per packed route.
#include "common.cuh"
#include "kernels.h"

namespace exl3 {

__global__ void __launch_bounds__(256) k_rotate(RotateArgs a)
{
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = blockIdx.x * 256 + tid; i < a.nzero; i += gridDim.x * 256)
        a.zero[i] = 0;
    if (a.hdr_reset && blockIdx.x == 0 && tid == 0)
        a.hdr_reset[kHdrError] = 0;
    if (a.hdr && a.hdr[kHdrError])
        return;
    const int wg = blockIdx.x * 8 + (tid >> 5);
    const int row = wg / a.nproj, p = wg % a.nproj;
    if (row >= a.rows)
        return;
    long token;
    const uint16_t *suh;
    if (a.packed) {
        const int f = a.packed[row];
        token = f / a.topk;
        const long long e = a.ids_dtype == EXL3_I64
                                ? static_cast<const int64_t *>(a.ids)[f]
                                : static_cast<const int32_t *>(a.ids)[f];
        suh = reinterpret_cast<const uint16_t *>(a.t_suh[e * 3 + p]);
    } else {
        token = row;
        suh = a.suh;
    }
    const int nblk = a.width / kHb;
    const size_t src = (size_t)token * a.width + 4 * lane;
    uint16_t *dst = a.out + ((size_t)row * a.nproj + p) * a.width + 4 * lane;
#pragma unroll 4
    for (int b = 0; b < nblk; b++) {
        float v[4], s[4];
        load_act4(a.x, src + b * kHb, a.act_dtype, v);
        load_half4(suh, b * kHb + 4 * lane, s);
#pragma unroll
        for (int i = 0; i < 4; i++)
            v[i] *= s[i];
        warp_hadamard128(v);
#pragma unroll
        for (int i = 0; i < 4; i++)
            v[i] *= kInvSqrt128;
        store_act4(dst + b * kHb, 0, EXL3_F16, v);
    }
}

cudaError_t launch_rotate(const RotateArgs &a, cudaStream_t s)
{
    long warps = (long)a.rows * a.nproj;
    long blocks = (warps + 7) / 8;
    if (blocks < 1)
        blocks = 1;
    k_rotate<<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace exl3
