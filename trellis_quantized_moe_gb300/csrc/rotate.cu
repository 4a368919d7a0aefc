// Input rotation a' = Hb(x * suh) ("EXL3 linear and grouped routed experts",
// TensorFold #837, "What this changes": the input rotation, each expert's
// rotation).  One warp per (row, projection, 4 consecutive 128-blocks), all
// loads of the group issued first; lane l holds 4 consecutive features of each
// block; the 128-point Hadamard runs in registers and warp shuffles.  Output
// is fp16 (the MMA operand), one row per packed route.
#include "common.cuh"
#include "kernels.h"

namespace exl3 {

constexpr int kGroup = 4;   // 128-blocks per warp

__global__ void __launch_bounds__(256) k_rotate(RotateArgs a)
{
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = blockIdx.x * 256 + tid; i < a.nzero; i += gridDim.x * 256)
        a.zero[i] = 0;
    if (a.hdr_reset && blockIdx.x == 0 && tid == 0)
        a.hdr_reset[kHdrError] = 0;
    if (a.hdr && a.hdr[kHdrError])
        return;
    // warp = (row, projection, group of kGroup 128-blocks)
    const int ngroups = (a.width / kHb + kGroup - 1) / kGroup;
    const long wg = (long)blockIdx.x * 8 + (tid >> 5);
    const int grp = (int)(wg % ngroups);
    const int p = (int)((wg / ngroups) % a.nproj);
    const int row = (int)(wg / ((long)ngroups * a.nproj));
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
    const int b0 = grp * kGroup;
    const size_t src = (size_t)token * a.width + 4 * lane;
    uint16_t *dst = a.out + ((size_t)row * a.nproj + p) * a.width + 4 * lane;
    float v[kGroup][4], s[kGroup][4];
#pragma unroll
    for (int k = 0; k < kGroup; k++) {          // all loads of the group first
        const int b = min(b0 + k, nblk - 1);
        load_act4(a.x, src + b * kHb, a.act_dtype, v[k]);
        load_half4(suh, b * kHb + 4 * lane, s[k]);
    }
#pragma unroll
    for (int k = 0; k < kGroup; k++) {
        if (b0 + k >= nblk)
            break;
#pragma unroll
        for (int i = 0; i < 4; i++)
            v[k][i] *= s[k][i];
        warp_hadamard128(v[k]);
#pragma unroll
        for (int i = 0; i < 4; i++)
            v[k][i] *= kInvSqrt128;
        store_act4(dst + (b0 + k) * kHb, 0, EXL3_F16, v[k]);
    }
}

cudaError_t launch_rotate(const RotateArgs &a, cudaStream_t s)
{
    long warps = (long)a.rows * a.nproj * ((a.width / kHb + kGroup - 1) / kGroup);
    long blocks = (warps + 7) / 8;
    if (blocks < 1)
        blocks = 1;
    k_rotate<<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace exl3
