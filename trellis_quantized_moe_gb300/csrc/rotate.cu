// Input rotation a' = Hb(x * suh) ("EXL3 linear and grouped routed experts",
// TensorFold #837, "What this changes": the input rotation, each expert's
// rotation).  Four lanes per 128-block (rotate_block.cuh), eight blocks per
// warp.  Output is fp16 (the MMA operand), one row per packed route.
#include "common.cuh"
#include "kernels.h"
#include "rotate_block.cuh"

namespace exl3 {

constexpr int kBlocksPerWarp = 8;
constexpr int kFeat = kRotFeat;

// TRIGGER: the tcgen05 linear, launched after this kernel with programmatic
// dependent launch, may start once every CTA of this grid is running (its
// activation producer waits for this grid's completion).  A separate
// instantiation: the fused layer's rotate kernels do not contain the trigger.
template <int RPW, bool TRIGGER>
__global__ void __launch_bounds__(256) k_rotate(RotateArgs a)
{
    const int tid = threadIdx.x, lane = tid & 31;
    if constexpr (TRIGGER)
        grid_dep_launch();
    for (int i = blockIdx.x * 256 + tid; i < a.nzero; i += gridDim.x * 256)
        a.zero[i] = 0;
    if (a.hdr_reset && blockIdx.x == 0 && tid == 0)
        a.hdr_reset[kHdrError] = 0;
    if (a.hdr && a.hdr[kHdrError])
        return;
    // warp = (RPW consecutive rows, projection, group of 8 128-blocks)
    const int nblk = a.width / kHb;
    const int ngroups = (nblk + kBlocksPerWarp - 1) / kBlocksPerWarp;
    const long wg = (long)blockIdx.x * 8 + (tid >> 5);
    const int grp = (int)(wg % ngroups);
    const int p = (int)((wg / ngroups) % a.nproj);
    const int row0 = (int)(wg / ((long)ngroups * a.nproj)) * RPW;
    if (row0 >= a.rows)
        return;
    const int nr = min(RPW, a.rows - row0);
    const int blk = grp * kBlocksPerWarp + (lane >> 2);
    const int c = lane & 3;                      // quarter of the block
    const bool active = blk < nblk;              // uniform within each group of 4 lanes
    const int col = (active ? blk : 0) * kHb + kFeat * c;
    // the rows' tokens and suh vectors, looked up once, lane i for row i:
    // the dependent loads of all rows are in flight together
    long long tok_l = 0;
    unsigned long long suh_l = 0;
    if (lane < nr) {
        const int row = row0 + lane;
        if (a.packed) {
            const int f = a.packed[row];
            tok_l = f / a.topk;
            const long long e = a.ids_dtype == EXL3_I64 ? static_cast<const int64_t *>(a.ids)[f]
                                                        : static_cast<const int32_t *>(a.ids)[f];
            suh_l = static_cast<unsigned long long>(a.t_suh[e * 3 + p]);
        } else {
            tok_l = row;
            suh_l = reinterpret_cast<unsigned long long>(a.suh);
        }
    }
    // the next row's activations load while this row is rotated
    auto load_row = [&](int i, uint4 (&r)[4]) {
        const long long tok = __shfl_sync(0xffffffffu, tok_l, i);
        const uint4 *q = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.x) + tok * a.width + col);
#pragma unroll
        for (int k = 0; k < 4; k++)
            r[k] = q[k];
    };
    uint4 cur[4], nxt[4];
    load_row(0, cur);
    unsigned long long cur_suh = 0;
    uint32_t sh[kFeat / 2];                      // suh as fp16 pairs (fewer live registers)
#pragma unroll 1
    for (int i = 0; i < nr; i++) {
        if (i + 1 < nr)
            load_row(i + 1, nxt);
        const unsigned long long suh = __shfl_sync(0xffffffffu, suh_l, i);
        if (suh != cur_suh) {                    // warp-uniform
            const uint2 *q = reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(suh) + col);
#pragma unroll
            for (int k = 0; k < kFeat / 4; k++) {
                const uint2 r = q[k];
                sh[2 * k] = r.x;
                sh[2 * k + 1] = r.y;
            }
            cur_suh = suh;
        }
        float v[kFeat];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const uint32_t w[4] = {cur[k].x, cur[k].y, cur[k].z, cur[k].w};
#pragma unroll
            for (int h = 0; h < 4; h++) {
                float2 f;
                if (a.act_dtype == EXL3_BF16)
                    f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[h]));
                else
                    f = __half22float2(*reinterpret_cast<const __half2 *>(&w[h]));
                const float2 sf = __half22float2(*reinterpret_cast<const __half2 *>(&sh[4 * k + h]));
                v[8 * k + 2 * h] = f.x * sf.x;
                v[8 * k + 2 * h + 1] = f.y * sf.y;
            }
        }
        uint4 out[4];
        rotate_block32(v, c, out);
        if (active) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((size_t)(row0 + i) * a.nproj + p) * a.width + col);
#pragma unroll
            for (int k = 0; k < 4; k++)
                dst[k] = out[k];
        }
#pragma unroll
        for (int k = 0; k < 4; k++)
            cur[k] = nxt[k];
    }
}

// Large layers: a warp takes up to 16 consecutive packed rows (a.rpw, fewer
// when that would leave SMs short of warps) of one projection and 8 blocks;
// each lane streams its 64 bytes of the next rows' activations into
// a 3-deep per-warp ring in shared memory with cp.async (no registers held
// for the prefetch, so more warps fit), then rotates exactly as k_rotate.  The
// rotated row goes out through shared memory so that each store instruction
// writes 512 contiguous bytes (whole 32-byte sectors) instead of 16 bytes
// every 64.
constexpr int kRingRows = 16;      // rows per warp, at most
constexpr int kRingDepth = 3;      // rows in flight per warp
constexpr int kRingWarps = 6;      // 48 KB of static shared memory per CTA, 4 CTAs per SM

template <bool TRIGGER>
__global__ void __launch_bounds__(kRingWarps * 32, 4) k_rotate_ring(RotateArgs a)
{
    __shared__ __align__(16) uint8_t ring[kRingWarps][kRingDepth + 1][32 * 64];   // + the output row
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if constexpr (TRIGGER)
        grid_dep_launch();                       // as in k_rotate
    for (int i = blockIdx.x * blockDim.x + tid; i < a.nzero; i += gridDim.x * blockDim.x)
        a.zero[i] = 0;
    if (a.hdr_reset && blockIdx.x == 0 && tid == 0)
        a.hdr_reset[kHdrError] = 0;
    if (a.hdr && a.hdr[kHdrError])
        return;
    const int nblk = a.width / kHb;
    const int ngroups = (nblk + kBlocksPerWarp - 1) / kBlocksPerWarp;
    const long wg = (long)blockIdx.x * kRingWarps + warp;
    const int grp = (int)(wg % ngroups);
    const int p = (int)((wg / ngroups) % a.nproj);
    const int row0 = (int)(wg / ((long)ngroups * a.nproj)) * a.rpw;
    if (row0 >= a.rows)
        return;
    const int nr = min(a.rpw, a.rows - row0);
    const int blk = grp * kBlocksPerWarp + (lane >> 2);
    const int c = lane & 3;
    const bool active = blk < nblk;
    const int col = (active ? blk : 0) * kHb + kFeat * c;
    long long tok_l = 0;
    unsigned long long suh_l = 0;
    if (lane < nr) {
        const int row = row0 + lane;
        if (a.packed) {
            const int f = a.packed[row];
            tok_l = f / a.topk;
            const long long e = a.ids_dtype == EXL3_I64 ? static_cast<const int64_t *>(a.ids)[f]
                                                        : static_cast<const int32_t *>(a.ids)[f];
            suh_l = static_cast<unsigned long long>(a.t_suh[e * 3 + p]);
        } else {
            tok_l = row;
            suh_l = reinterpret_cast<unsigned long long>(a.suh);
        }
    }
    // lane l's 64 bytes of slot d, its four 16-byte chunks rotated by l so the
    // lanes of a shared-memory wavefront hit different banks
    auto chunk_at = [&](int d, int k) -> uint8_t * {
        return &ring[warp][d][lane * 64 + (((k + lane) & 3) << 4)];
    };
    auto fetch = [&](int i) {
        if (i < nr) {
            const long long tok = __shfl_sync(0xffffffffu, tok_l, i);
            const uint8_t *src = reinterpret_cast<const uint8_t *>(
                static_cast<const uint16_t *>(a.x) + tok * a.width + col);
#pragma unroll
            for (int k = 0; k < 4; k++)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                             ::"r"(smem_addr(chunk_at(i % kRingDepth, k))), "l"(src + 16 * k) : "memory");
        } else {
            __shfl_sync(0xffffffffu, tok_l, 0);   // keep the warp's shuffles in step
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
#pragma unroll
    for (int i = 0; i < kRingDepth; i++)
        fetch(i);
    unsigned long long cur_suh = 0;
    uint32_t sh[kFeat / 2];
#pragma unroll 1
    for (int i = 0; i < nr; i++) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kRingDepth - 1) : "memory");
        const unsigned long long suh = __shfl_sync(0xffffffffu, suh_l, i);
        if (suh != cur_suh) {                    // warp-uniform
            const uint2 *q = reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(suh) + col);
#pragma unroll
            for (int k = 0; k < kFeat / 4; k++) {
                const uint2 r = q[k];
                sh[2 * k] = r.x;
                sh[2 * k + 1] = r.y;
            }
            cur_suh = suh;
        }
        float v[kFeat];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(chunk_at(i % kRingDepth, k));
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int h = 0; h < 4; h++) {
                float2 f;
                if (a.act_dtype == EXL3_BF16)
                    f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[h]));
                else
                    f = __half22float2(*reinterpret_cast<const __half2 *>(&w[h]));
                const float2 sf = __half22float2(*reinterpret_cast<const __half2 *>(&sh[4 * k + h]));
                v[8 * k + 2 * h] = f.x * sf.x;
                v[8 * k + 2 * h + 1] = f.y * sf.y;
            }
        }
        // the slot's words are in registers (v depends on them): refill it
        fetch(i + kRingDepth);
        uint4 out[4];
        rotate_block32(v, c, out);
        // lane l's features 32c.. of block l/4 are bytes 64l.. of the warp's
        // 2 KB output span; written lane-major, read back 16 bytes per lane
        // at 16l + 512k
#pragma unroll
        for (int k = 0; k < 4; k++)
            *reinterpret_cast<uint4 *>(chunk_at(kRingDepth, k)) = out[k];
        __syncwarp();
        uint8_t *orow = reinterpret_cast<uint8_t *>(a.out + ((size_t)(row0 + i) * a.nproj + p) * a.width +
                                                    (size_t)grp * kBlocksPerWarp * kHb);
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int off = 16 * lane + 512 * k;               // byte in the span
            const int src_lane = off >> 6, ch = (off >> 4) & 3;
            if ((off >> 8) + grp * kBlocksPerWarp < nblk) {    // 256 bytes per block
                const uint4 val = *reinterpret_cast<const uint4 *>(
                    &ring[warp][kRingDepth][src_lane * 64 + (((ch + src_lane) & 3) << 4)]);
                *reinterpret_cast<uint4 *>(orow + off) = val;
            }
        }
        __syncwarp();
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
}

cudaError_t launch_rotate(const RotateArgs &a, cudaStream_t s)
{
    const long groups = (a.width / kHb + kBlocksPerWarp - 1) / kBlocksPerWarp;
    // from 4096 rows: up to 16 rows per warp with the cp.async ring, as many
    // as leave one full wave of resident warps (4 CTAs of kRingWarps per SM);
    // fewer rows take one row per warp
    if (a.rows >= 4096) {
        RotateArgs b = a;
        const long tasks = (long)a.rows * a.nproj * groups;
        const long slots = (long)(a.num_sms > 0 ? a.num_sms : 1) * 4 * kRingWarps;
        b.rpw = (int)((tasks + slots - 1) / slots);
        b.rpw = b.rpw < 1 ? 1 : (b.rpw > kRingRows ? kRingRows : b.rpw);
        const long warps = (long)((a.rows + b.rpw - 1) / b.rpw) * a.nproj * groups;
        const long blocks = (warps + kRingWarps - 1) / kRingWarps;
        if (a.trigger)
            k_rotate_ring<true><<<(unsigned)blocks, kRingWarps * 32, 0, s>>>(b);
        else
            k_rotate_ring<false><<<(unsigned)blocks, kRingWarps * 32, 0, s>>>(b);
        return cudaGetLastError();
    }
    const long warps = (long)a.rows * a.nproj * groups;
    long blocks = (warps + 7) / 8;
    if (blocks < 1)
        blocks = 1;
    if (a.trigger)
        k_rotate<1, true><<<(unsigned)blocks, 256, 0, s>>>(a);
    else
        k_rotate<1, false><<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace exl3
