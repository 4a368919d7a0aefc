// Input rotation a' = Hb(x * suh) ("EXL3 linear and grouped routed experts",
// TensorFold #837, "What this changes": the input rotation, each expert's
// rotation).  Four lanes per 128-block, eight blocks per warp: lane 4q+c holds
// features 32c..32c+31 of block q, so butterfly stages 0-4 of the 128-point
// Hadamard run in registers and only stages 5 and 6 cross lanes (2 shuffle
// stages instead of 5 with 4 features per lane).  Stages run in index-bit
// order 0..6 with the same pairings as warp_hadamard128, so every sum is the
// same fp32 operation.  Output is fp16 (the MMA operand), one row per packed
// route.
#include "common.cuh"
#include "kernels.h"

namespace exl3 {

constexpr int kBlocksPerWarp = 8;
constexpr int kFeat = 32;            // features per lane

// 32 activations of type dtype at p[i..i+31] -> fp32 (16-byte loads; x rows
// are 16-byte aligned by the API's checks and widths are multiples of 128)
__device__ __forceinline__ void load_act32(const void *p, size_t i, int dtype, float v[kFeat])
{
    if (dtype == EXL3_F32) {
        const float4 *q = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p) + i);
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const float4 f = q[k];
            v[4 * k] = f.x; v[4 * k + 1] = f.y; v[4 * k + 2] = f.z; v[4 * k + 3] = f.w;
        }
        return;
    }
    const uint4 *q = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p) + i);
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint4 raw = q[k];
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int h = 0; h < 4; h++) {
            float2 f;
            if (dtype == EXL3_BF16)
                f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[h]));
            else
                f = __half22float2(*reinterpret_cast<const __half2 *>(&w[h]));
            v[8 * k + 2 * h] = f.x;
            v[8 * k + 2 * h + 1] = f.y;
        }
    }
}

// 32 fp16 values at p[i..i+31] -> fp32 with 8-byte loads (the tables only
// guarantee 8-byte alignment of suh)
__device__ __forceinline__ void load_half32(const uint16_t *p, size_t i, float v[kFeat])
{
    const uint2 *q = reinterpret_cast<const uint2 *>(p + i);
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const uint2 raw = q[k];
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
        v[4 * k] = f0.x; v[4 * k + 1] = f0.y; v[4 * k + 2] = f1.x; v[4 * k + 3] = f1.y;
    }
}

__global__ void __launch_bounds__(256) k_rotate(RotateArgs a)
{
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = blockIdx.x * 256 + tid; i < a.nzero; i += gridDim.x * 256)
        a.zero[i] = 0;
    if (a.hdr_reset && blockIdx.x == 0 && tid == 0)
        a.hdr_reset[kHdrError] = 0;
    if (a.hdr && a.hdr[kHdrError])
        return;
    // warp = (row, projection, group of 8 128-blocks)
    const int nblk = a.width / kHb;
    const int ngroups = (nblk + kBlocksPerWarp - 1) / kBlocksPerWarp;
    const long wg = (long)blockIdx.x * 8 + (tid >> 5);
    const int grp = (int)(wg % ngroups);
    const int p = (int)((wg / ngroups) % a.nproj);
    const int row = (int)(wg / ((long)ngroups * a.nproj));
    if (row >= a.rows)
        return;
    const int blk = grp * kBlocksPerWarp + (lane >> 2);
    const int c = lane & 3;                      // quarter of the block
    const bool active = blk < nblk;              // uniform within each group of 4 lanes
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
    const int col = (active ? blk : 0) * kHb + kFeat * c;
    float v[kFeat], s[kFeat];
    load_act32(a.x, (size_t)token * a.width + col, a.act_dtype, v);
    load_half32(suh, col, s);
#pragma unroll
    for (int i = 0; i < kFeat; i++)
        v[i] *= s[i];
    // stages 0-4: index bits inside the lane's 32 features
#pragma unroll
    for (int m = 1; m < kFeat; m <<= 1) {
#pragma unroll
        for (int i = 0; i < kFeat; i++) {
            if ((i & m) == 0) {
                const float lo = v[i], hi = v[i + m];
                v[i] = lo + hi;
                v[i + m] = lo - hi;
            }
        }
    }
    // stages 5-6: the two lane bits of the quarter index
#pragma unroll
    for (int m = 1; m < 4; m <<= 1) {
        const bool upper = c & m;
#pragma unroll
        for (int i = 0; i < kFeat; i++) {
            const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
            v[i] = upper ? (o - v[i]) : (v[i] + o);
        }
    }
    if (!active)
        return;
    uint4 out[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; h++) {
            const __half2 t = __floats2half2_rn(v[8 * k + 2 * h] * kInvSqrt128, v[8 * k + 2 * h + 1] * kInvSqrt128);
            w[h] = *reinterpret_cast<const uint32_t *>(&t);
        }
        out[k] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((size_t)row * a.nproj + p) * a.width + col);
#pragma unroll
    for (int k = 0; k < 4; k++)
        dst[k] = out[k];
}

cudaError_t launch_rotate(const RotateArgs &a, cudaStream_t s)
{
    const long groups = (a.width / kHb + kBlocksPerWarp - 1) / kBlocksPerWarp;
    long warps = (long)a.rows * a.nproj * groups;
    long blocks = (warps + 7) / 8;
    if (blocks < 1)
        blocks = 1;
    k_rotate<<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace exl3
