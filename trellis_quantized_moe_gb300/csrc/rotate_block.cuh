// One 128-feature block of the input rotation a' = Hb(x * suh) / sqrt(128),
// computed by four lanes (lane quad c = lane & 3 holds features 32c..32c+31),
// shared by the rotate kernel and the decode-regime gate/up kernel so both
// produce the same fp16 bits ("EXL3 linear and grouped routed experts",
// TensorFold #837, "What this changes": the input rotation).  Butterfly
// stages 0-4 run in registers, stages 5-6 across the lane quad, in index-bit
// order 0..6 with the pairings of warp_hadamard128.  Every lane of the warp
// must call it (the shuffles use the full mask).
#pragma once
#include "common.cuh"

namespace exl3 {

constexpr int kRotFeat = 32;            // features per lane

// 32 activations of type dtype at p[i..i+31] -> fp32 (16-byte loads: x rows
// are 16-byte aligned by the API's checks and widths are multiples of 128)
__device__ __forceinline__ void load_act32(const void *p, size_t i, int dtype, float v[kRotFeat])
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
__device__ __forceinline__ void load_half32(const uint16_t *p, size_t i, float v[kRotFeat])
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

// v = this lane's 32 features of x * suh (fp32) -> 4 x uint4 of fp16 output
// features 32c..32c+31 of the rotated block.
__device__ __forceinline__ void rotate_block32(float v[kRotFeat], int c, uint4 out[4])
{
#pragma unroll
    for (int m = 1; m < kRotFeat; m <<= 1) {
#pragma unroll
        for (int i = 0; i < kRotFeat; i++) {
            if ((i & m) == 0) {
                const float lo = v[i], hi = v[i + m];
                v[i] = lo + hi;
                v[i + m] = lo - hi;
            }
        }
    }
#pragma unroll
    for (int m = 1; m < 4; m <<= 1) {
        // upper lane: o - v, lower lane: v + o, as one fma with a +-1 factor
        // (multiplying by +-1 is exact, so the single rounding is the same)
        const float sgn = (c & m) ? -1.0f : 1.0f;
#pragma unroll
        for (int i = 0; i < kRotFeat; i++) {
            const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
            v[i] = __fmaf_rn(sgn, v[i], o);
        }
    }
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
}

}  // namespace exl3
