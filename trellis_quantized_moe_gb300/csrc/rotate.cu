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

template <int RPW>
__global__ void __launch_bounds__(256) k_rotate(RotateArgs a)
{
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = blockIdx.x * 256 + tid; i < a.nzero; i += gridDim.x * 256)
        a.zero[i] = 0;
    if (a.hdr_reset && blockIdx.x == 0 && tid == 0)
        a.hdr_reset[kHdrError] = 0;
    if (a.hdr && a.hdr[kHdrError])
        return;
    // warp = (RPW consecutive rows, projection, group of 8 128-blocks): packed rows come in runs of one expert, so suh is loaded
    // once per run and reused for the warp's following rows
    const int nblk = a.width / kHb;
    const int ngroups = (nblk + kBlocksPerWarp - 1) / kBlocksPerWarp;
    const long wg = (long)blockIdx.x * 8 + (tid >> 5);
    const int grp = (int)(wg % ngroups);
    const int p = (int)((wg / ngroups) % a.nproj);
    const int row0 = (int)(wg / ((long)ngroups * a.nproj)) * RPW;
    if (row0 >= a.rows)
        return;
    const int blk = grp * kBlocksPerWarp + (lane >> 2);
    const int c = lane & 3;                      // quarter of the block
    const bool active = blk < nblk;              // uniform within each group of 4 lanes
    const int col = (active ? blk : 0) * kHb + kFeat * c;
    const uint16_t *cur_suh = nullptr;
    float s[kFeat];
#pragma unroll 1
    for (int row = row0; row < row0 + RPW && row < a.rows; row++) {
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
        if (suh != cur_suh) {                    // warp-uniform: depends on the row only
            load_half32(suh, col, s);
            cur_suh = suh;
        }
        float v[kFeat];
        load_act32(a.x, (size_t)token * a.width + col, a.act_dtype, v);
#pragma unroll
        for (int i = 0; i < kFeat; i++)
            v[i] *= s[i];
        uint4 out[4];
        rotate_block32(v, c, out);
        if (active) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((size_t)row * a.nproj + p) * a.width + col);
#pragma unroll
            for (int k = 0; k < 4; k++)
                dst[k] = out[k];
        }
    }
}

cudaError_t launch_rotate(const RotateArgs &a, cudaStream_t s)
{
    const long groups = (a.width / kHb + kBlocksPerWarp - 1) / kBlocksPerWarp;
    // 8 rows per warp once there are enough warps to hide load latency
    // (measured: 4096-route layers -21% rotate time, 1024 rows +27%)
    const int rpw = a.rows >= 4096 ? 8 : 1;
    long warps = (long)((a.rows + rpw - 1) / rpw) * a.nproj * groups;
    long blocks = (warps + 7) / 8;
    if (blocks < 1)
        blocks = 1;
    if (rpw == 8)
        k_rotate<8><<<(unsigned)blocks, 256, 0, s>>>(a);
    else
        k_rotate<1><<<(unsigned)blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace exl3
