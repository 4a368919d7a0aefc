// Per-row epilogues shared by the decode-regime (mma.sync) and prefill-regime
// (tcgen05) grouped GEMMs.  One warp handles one route row of one 128-output
// block; lane l owns outputs 4l..4l+3.  Inputs are the raw fp32 contraction
// results z (before the output Hadamard).
//
// "EXL3 linear and grouped routed experts" (TensorFold #837), "What this
// changes": output rotation, SwiGLU, down-input rotation, weighted combine.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace exl3 {

// Per-column factors of one (expert, 128-output block), lane l holding
// outputs 4l..4l+3: they depend on neither the route nor the row, so a kernel
// that runs many rows of one block loads them once.
struct GateUpConsts {
    float svg[4], scg[4], svu[4], scu[4], sud[4];
};

__device__ __forceinline__ void epi_gateup_consts(const GemmArgs &a, int e, int nbk, GateUpConsts &c)
{
    const int col = nbk * kHb + 4 * (threadIdx.x & 31);
    load_half4(reinterpret_cast<const uint16_t *>(a.t_svh[e * 3 + 0]), col, c.svg);
    load_half4(reinterpret_cast<const uint16_t *>(a.t_scale[e * 3 + 0]), col, c.scg);
    load_half4(reinterpret_cast<const uint16_t *>(a.t_svh[e * 3 + 1]), col, c.svu);
    load_half4(reinterpret_cast<const uint16_t *>(a.t_scale[e * 3 + 1]), col, c.scu);
    load_half4(reinterpret_cast<const uint16_t *>(a.t_suh[e * 3 + 2]), col, c.sud);
}

// gate/up: g' = Hb(g)*svh*scale, u' likewise, h = silu(g')*u', then the down
// projection's input rotation a_d = Hb(h * suh_down) over the same 128 block of
// the intermediate dimension; stored as the fp16 MMA operand of the down GEMM.
__device__ __forceinline__ void epi_gateup_row(const GemmArgs &a, const GateUpConsts &c, int nbk,
                                               int prow, float gv[4], float uv[4])
{
    const int lane = threadIdx.x & 31;
    const int col = nbk * kHb + 4 * lane;
    float h[4];
    warp_hadamard128(gv);
    warp_hadamard128(uv);
#pragma unroll
    for (int i = 0; i < 4; i++)
        gv[i] = gv[i] * kInvSqrt128 * c.svg[i] * c.scg[i];
#pragma unroll
    for (int i = 0; i < 4; i++)
        uv[i] = uv[i] * kInvSqrt128 * c.svu[i] * c.scu[i];
#pragma unroll
    for (int i = 0; i < 4; i++)
        h[i] = gv[i] / (1.0f + expf(-gv[i])) * uv[i] * c.sud[i];
    warp_hadamard128(h);
#pragma unroll
    for (int i = 0; i < 4; i++)
        h[i] *= kInvSqrt128;
    store_act4(a.ad, (size_t)prow * a.out_f + col, EXL3_F16, h);
}

__device__ __forceinline__ void epi_gateup_row(const GemmArgs &a, int e, int nbk, int prow,
                                               float gv[4], float uv[4])
{
    GateUpConsts c;
    epi_gateup_consts(a, e, nbk, c);
    epi_gateup_row(a, c, nbk, prow, gv, uv);
}

struct DownConsts {
    float sv[4], sc[4];
};

__device__ __forceinline__ void epi_down_consts(const GemmArgs &a, int e, int nbk, DownConsts &c)
{
    const int col = nbk * kHb + 4 * (threadIdx.x & 31);
    load_half4(reinterpret_cast<const uint16_t *>(a.t_svh[e * 3 + 2]), col, c.sv);
    load_half4(reinterpret_cast<const uint16_t *>(a.t_scale[e * 3 + 2]), col, c.sc);
}

// down: d = Hb(z)*svh*scale into the fp32 staging row of flat route f; the
// warp that completes all topk routes of a token's block combines them in j
// order (fp32 fma chain, rounded once) and resets the block's counter.
__device__ __forceinline__ void epi_down_row(const GemmArgs &a, int e, int nbk, int prow,
                                             float z[4])
{
    const int lane = threadIdx.x & 31;
    const int col = nbk * kHb + 4 * lane;
    const uint16_t *svh = reinterpret_cast<const uint16_t *>(a.t_svh[e * 3 + 2]);
    const uint16_t *scl = reinterpret_cast<const uint16_t *>(a.t_scale[e * 3 + 2]);
    float sv[4], sc[4];
    warp_hadamard128(z);
    load_half4(svh, col, sv);
    load_half4(scl, col, sc);
#pragma unroll
    for (int i = 0; i < 4; i++)
        z[i] = z[i] * kInvSqrt128 * sv[i] * sc[i];
    const int f = a.packed[prow];
    const int tok = f / a.topk;
    *reinterpret_cast<float4 *>(a.stage + (size_t)f * a.out_f + col) =
        make_float4(z[0], z[1], z[2], z[3]);
    __threadfence();
    __syncwarp();
    int old = 0;
    if (lane == 0)
        old = atomicAdd(&a.cnt_comb[tok * a.nb + nbk], 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == a.topk - 1) {
        __threadfence();
        float o4[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < a.topk; j++) {
            const float w = load_act(a.rw, (size_t)tok * a.topk + j, a.rw_dtype);
            const float4 d = __ldcg(reinterpret_cast<const float4 *>(
                a.stage + ((size_t)tok * a.topk + j) * a.out_f + col));
            o4[0] = __fmaf_rn(w, d.x, o4[0]);
            o4[1] = __fmaf_rn(w, d.y, o4[1]);
            o4[2] = __fmaf_rn(w, d.z, o4[2]);
            o4[3] = __fmaf_rn(w, d.w, o4[3]);
        }
        store_act4(a.out, (size_t)tok * a.out_f + col, a.act_dtype, o4);
        if (lane == 0)
            a.cnt_comb[tok * a.nb + nbk] = 0;
    }
}

// The down epilogue in two phases, for kernels that stage many rows and then
// publish them with a single fence: (1) d = Hb(z)*svh*scale into the staging
// row (epi_down_stage_row); (2) after a __threadfence by every staging thread,
// count the routes and combine each token block completed
// (epi_down_combine_rows).
__device__ __forceinline__ void epi_down_stage_row(const GemmArgs &a, const DownConsts &c, int nbk,
                                                   int prow, float z[4])
{
    const int lane = threadIdx.x & 31;
    const int col = nbk * kHb + 4 * lane;
    warp_hadamard128(z);
#pragma unroll
    for (int i = 0; i < 4; i++)
        z[i] = z[i] * kInvSqrt128 * c.sv[i] * c.sc[i];
    const int f = a.packed[prow];
    *reinterpret_cast<float4 *>(a.stage + (size_t)f * a.out_f + col) =
        make_float4(z[0], z[1], z[2], z[3]);
}

// Counters of many staged rows at once: warp w of nw takes rows w, w + nw, ...
// (at most 32 per warp), one lane per row, so the atomics are in flight
// together; each token block that a lane completed is then combined by the
// whole warp, in lane order.
__device__ __forceinline__ void epi_down_combine_rows(const GemmArgs &a, int nbk, int row0, int nrows,
                                                      int w, int nw)
{
    const int lane = threadIdx.x & 31;
    const int col = nbk * kHb + 4 * lane;
    for (int base = w; base < nrows; base += 32 * nw) {
        const int r = base + lane * nw;
        int tok = -1;
        if (r < nrows) {
            const int f = a.packed[row0 + r];
            const int t = f / a.topk;
            if (atomicAdd(&a.cnt_comb[t * a.nb + nbk], 1) == a.topk - 1)
                tok = t;
        }
        unsigned done = __ballot_sync(0xffffffffu, tok >= 0);
        if (done)
            __threadfence();
        while (done) {
            const int src = __ffs(done) - 1;
            done &= done - 1;
            const int t = __shfl_sync(0xffffffffu, tok, src);
            float o4[4] = {0.f, 0.f, 0.f, 0.f};
            for (int j = 0; j < a.topk; j++) {
                const float wj = load_act(a.rw, (size_t)t * a.topk + j, a.rw_dtype);
                const float4 d = __ldcg(reinterpret_cast<const float4 *>(
                    a.stage + ((size_t)t * a.topk + j) * a.out_f + col));
                o4[0] = __fmaf_rn(wj, d.x, o4[0]);
                o4[1] = __fmaf_rn(wj, d.y, o4[1]);
                o4[2] = __fmaf_rn(wj, d.z, o4[2]);
                o4[3] = __fmaf_rn(wj, d.w, o4[3]);
            }
            store_act4(a.out, (size_t)t * a.out_f + col, a.act_dtype, o4);
            if (lane == 0)
                a.cnt_comb[t * a.nb + nbk] = 0;
        }
    }
}

// linear (one projection): the per-column factors, loaded once per block
__device__ __forceinline__ void epi_linear_consts(const GemmArgs &a, int nbk, DownConsts &c)
{
    const int col = nbk * kHb + 4 * (threadIdx.x & 31);
    load_half4(a.lin.svh, col, c.sv);
    load_half4(a.lin.scale, col, c.sc);
}

__device__ __forceinline__ void epi_linear_row(const GemmArgs &a, const DownConsts &c, int nbk, int row,
                                               float z[4])
{
    const int lane = threadIdx.x & 31;
    const int col = nbk * kHb + 4 * lane;
    warp_hadamard128(z);
#pragma unroll
    for (int i = 0; i < 4; i++)
        z[i] = z[i] * kInvSqrt128 * c.sv[i] * c.sc[i];
    store_act4(a.out, (size_t)row * a.out_f + col, a.act_dtype, z);
}

// linear: y = Hb(z)*svh*scale, stored in the activation dtype.
__device__ __forceinline__ void epi_linear_row(const GemmArgs &a, int nbk, int row, float z[4])
{
    const int lane = threadIdx.x & 31;
    const int col = nbk * kHb + 4 * lane;
    float sv[4], sc[4];
    warp_hadamard128(z);
    load_half4(a.lin.svh, col, sv);
    load_half4(a.lin.scale, col, sc);
#pragma unroll
    for (int i = 0; i < 4; i++)
        z[i] = z[i] * kInvSqrt128 * sv[i] * sc[i];
    store_act4(a.out, (size_t)row * a.out_f + col, a.act_dtype, z);
}

}  // namespace exl3
