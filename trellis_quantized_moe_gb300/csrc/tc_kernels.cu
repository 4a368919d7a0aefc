// Prefill-regime (tcgen05 / TMEM) gate/up, down and linear kernels (see
// expert_tc.cuh), and the two elementwise steps of the prefill-regime layer
// around them: SwiGLU + down-input rotation, and the weighted combine.
#include "expert_tc.cuh"

namespace exl3 {

// SwiGLU and the down projection's input rotation of the prefill regime
// ("EXL3 linear and grouped routed experts", TensorFold #837, "What this
// changes"): the gate/up kernel staged g' = Hb(g)*svh*scale and u' likewise
// in fp32; here h = silu(g')*u'*suh_down, a_d = Hb(h)/sqrt(128) in fp16, the
// same operations in the same order as the decode regime's fused epilogue.
// One warp per (row group, 32-row chunk, 128 block); lane l owns outputs
// 4l..4l+3.
__global__ void __launch_bounds__(256) k_tc_gu_finish(GemmArgs a)
{
    if (a.hdr[kHdrRegime] != 1)
        return;
    const int lane = threadIdx.x & 31;
    const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nw = (int)((gridDim.x * blockDim.x) >> 5);
    const int ntask = a.hdr[kHdrNRg] * (tc::kNT / 32) * a.nb;
    const size_t ld = 2 * (size_t)a.out_f;
    for (int task = gw; task < ntask; task += nw) {
        const int nbk = task % a.nb, rest = task / a.nb;
        const int ch = rest % (tc::kNT / 32), rgi = rest / (tc::kNT / 32);
        const int4 r = static_cast<const int4 *>(a.rg)[rgi];
        const int rb = ch * 32;
        if (rb >= r.z)
            continue;
        const int col = nbk * kHb + 4 * lane;
        float sud[4];
        load_half4(reinterpret_cast<const uint16_t *>(a.t_suh[r.x * 3 + 2]), col, sud);
        const int rend = min(r.z, rb + 32);
        for (int i0 = rb; i0 < rend; i0 += 2) {
            float4 g[2], u[2];
#pragma unroll
            for (int j = 0; j < 2; j++) {
                if (i0 + j < rend) {
                    const float *row = a.stage + (size_t)(r.y + i0 + j) * ld;
                    g[j] = __ldcs(reinterpret_cast<const float4 *>(row + col));
                    u[j] = __ldcs(reinterpret_cast<const float4 *>(row + a.out_f + col));
                }
            }
#pragma unroll
            for (int j = 0; j < 2; j++) {
                if (i0 + j < rend) {
                    const float gv[4] = {g[j].x, g[j].y, g[j].z, g[j].w};
                    const float uv[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
                    float h[4];
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        h[i] = gv[i] / (1.0f + expf(-gv[i])) * uv[i] * sud[i];
                    warp_hadamard128(h);
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        h[i] *= kInvSqrt128;
                    store_act4(a.ad, (size_t)(r.y + i0 + j) * a.out_f + col, EXL3_F16, h);
                }
            }
        }
    }
}

// Route-weighted combine of the prefill regime (same page and section):
// out[t] = sum over j of w[t, j] * d[t*topk + j], an fp32 fma chain in j
// order rounded once to the activation dtype, as the decode regime's combine.
// One thread per 4 outputs of a token.  A layer whose plan carries an error
// writes zeros.
__global__ void __launch_bounds__(256) k_tc_combine(GemmArgs a)
{
    if (a.hdr[kHdrRegime] != 1)
        return;
    const bool err = a.hdr[kHdrError] != 0;
    const int h4 = a.out_f / 4;
    const size_t n = (size_t)a.M_tokens * h4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / h4), c = (int)(i % h4) * 4;
        float o4[4] = {0.f, 0.f, 0.f, 0.f};
        if (!err) {
            for (int j = 0; j < a.topk; j++) {
                const float wj = load_act(a.rw, (size_t)t * a.topk + j, a.rw_dtype);
                const float4 d = __ldcs(reinterpret_cast<const float4 *>(
                    a.stage + ((size_t)t * a.topk + j) * a.out_f + c));
                o4[0] = __fmaf_rn(wj, d.x, o4[0]);
                o4[1] = __fmaf_rn(wj, d.y, o4[1]);
                o4[2] = __fmaf_rn(wj, d.z, o4[2]);
                o4[3] = __fmaf_rn(wj, d.w, o4[3]);
            }
        }
        store_act4(a.out, (size_t)t * a.out_f + c, a.act_dtype, o4);
    }
}

cudaError_t launch_tc_gu_finish(const GemmArgs &a, int sms, cudaStream_t s)
{
    k_tc_gu_finish<<<sms * 8, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_tc_combine(const GemmArgs &a, int sms, cudaStream_t s)
{
    k_tc_combine<<<sms * 8, 256, 0, s>>>(a);
    return cudaGetLastError();
}

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
