// Device helpers shared by the kernels: dtype access, the warp-level 128-point
// Hadamard transform, mbarrier / bulk-copy wrappers and the legacy mma.sync.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/exl3.h"
#include "plan.h"

namespace exl3 {

#define EXL3_DEV __device__ __forceinline__

// ---------------------------------------------------------------- dtypes
EXL3_DEV float load_act(const void *p, size_t i, int dtype)
{
    if (dtype == EXL3_BF16)
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
    if (dtype == EXL3_F32)
        return reinterpret_cast<const float *>(p)[i];
    return __half2float(reinterpret_cast<const __half *>(p)[i]);
}

// Four consecutive activations (8-byte aligned for 16-bit types).
EXL3_DEV void load_act4(const void *p, size_t i, int dtype, float v[4])
{
    if (dtype == EXL3_F32) {
        float4 f = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p) + i);
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        return;
    }
    uint2 raw = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(p) + i);
    if (dtype == EXL3_BF16) {
        __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&raw.x);
        __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&raw.y);
        float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
        v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
    } else {
        __half2 a = *reinterpret_cast<__half2 *>(&raw.x);
        __half2 b = *reinterpret_cast<__half2 *>(&raw.y);
        float2 fa = __half22float2(a), fb = __half22float2(b);
        v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
    }
}

EXL3_DEV void store_act4(void *p, size_t i, int dtype, const float v[4])
{
    uint2 raw;
    if (dtype == EXL3_BF16) {
        __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
        raw.x = *reinterpret_cast<uint32_t *>(&a);
        raw.y = *reinterpret_cast<uint32_t *>(&b);
    } else {
        __half2 a = __floats2half2_rn(v[0], v[1]);
        __half2 b = __floats2half2_rn(v[2], v[3]);
        raw.x = *reinterpret_cast<uint32_t *>(&a);
        raw.y = *reinterpret_cast<uint32_t *>(&b);
    }
    *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(p) + i) = raw;
}

EXL3_DEV void load_half4(const uint16_t *p, size_t i, float v[4])
{
    load_act4(p, i, EXL3_F16, v);
}

// ---------------------------------------------------------------- Hadamard
// 128-point Sylvester transform of one vector held as 4 consecutive values per
// lane (lane l holds indices 4l..4l+3).  Unnormalised; the caller scales.
EXL3_DEV void warp_hadamard128(float v[4])
{
    float a = v[0] + v[1], b = v[0] - v[1], c = v[2] + v[3], d = v[2] - v[3];
    v[0] = a + c; v[1] = b + d; v[2] = a - c; v[3] = b - d;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        // upper lane: o - v, lower lane: v + o, as one fma with a +-1 factor
        // (exact product, same single rounding)
        const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
            v[i] = __fmaf_rn(sgn, v[i], o);
        }
    }
}

constexpr float kInvSqrt128 = 0.08838834764831845f;
constexpr float kInvSqrtMul1 = 0.006765875086793228f;   // 1 / sqrt(21845)
constexpr float kSqrtMul1 = 147.80054127099805f;        // sqrt(21845)

// ---------------------------------------------------------------- mbarrier / bulk copy
EXL3_DEV uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

EXL3_DEV void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

EXL3_DEV void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

EXL3_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// try_wait with a 1 ms suspend-time hint: a waiting thread sleeps until the
// phase completes (or the hint runs out) instead of re-polling, which leaves
// the issue slots of its SM sub-partition to the warps that have work.
EXL3_DEV bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

// x << N as an integer multiply: it issues on the FMA pipe, which the trellis
// decode otherwise leaves mostly idle while shifts and logic ops share the ALU
// pipe (both pipes take 16 lanes per cycle per SM sub-partition).
template <int N>
EXL3_DEV uint32_t shl_fma(uint32_t x)
{
    if constexpr (N == 0) {
        return x;
    } else {
        uint32_t d;
        asm("mul.lo.u32 %0, %1, %2;" : "=r"(d) : "r"(x), "n"(1u << N));
        return d;
    }
}

// The 16 bits of x starting N bits below its top (N <= 16): (x << N) >> 16,
// the left shift on the FMA pipe and the right shift on the ALU pipe.
template <int N>
EXL3_DEV uint32_t bits16_from_top(uint32_t x)
{
    return shl_fma<N>(x) >> 16;
}

// Programmatic dependent launch: wait until the preceding kernel in the stream
// has completed and its writes are visible; allow the next kernel to start
// launching.  Both are no-ops in a kernel launched without the attribute.
EXL3_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
EXL3_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Bounded wait: gives up after ~2^31 cycles and reports false.
EXL3_DEV bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait_sleep(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try_wait_sleep(bar, parity)) {
        if (clock64() - t0 > (1ll << 31))
            return false;
    }
    return true;
}

// One bulk global->shared copy completing on `bar` (16-byte aligned, size % 16 == 0).
EXL3_DEV void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

EXL3_DEV void named_barrier(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- mma.sync
// D = A(16x16, row) * B(16x8, col) + D, fp16 operands, fp32 accumulate.
EXL3_DEV void mma_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                        uint32_t b0, uint32_t b1)
{
    // not volatile: the scheduler may interleave it with the next tile's loads
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (x & mask) ^ flip as one LOP3 (truth table 0x6A).  A LOP3 takes at most
// one immediate, and an immediate constant that the compiler re-materialises
// inside an unrolled decode loop costs a second logic instruction per weight,
// so both constants are register operands here.
EXL3_DEV uint32_t and_xor(uint32_t x, uint32_t mask, uint32_t flip)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(x), "r"(mask), "r"(flip));
    return d;
}

// The mask and exponent flip that the mcg and 3inst codebooks apply to both
// 16-bit halves of the hashed state, as register values for a whole decode
// loop.  `zero` must be 0 at run time but unknown to the compiler (the low
// address bit of an int32 pointer argument), which stops it from folding the
// constants back into immediates.
struct HashConsts {
    uint32_t mask, flip;
};

EXL3_DEV HashConsts hash_consts(const int32_t *aligned_ptr)
{
    const uint32_t zero = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(aligned_ptr) & 1u);
    return {0x8FFF8FFFu ^ zero, 0x3B603B60u ^ zero};
}

EXL3_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

EXL3_DEV void set_error(int32_t *hdr, int bits)
{
    atomicOr(reinterpret_cast<int *>(hdr + kHdrError), bits);
}

}  // namespace exl3
