// Kernel argument structs and launchers (host <-> device interface of the
// library; internal, not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stdint.h>

#include "../../include/exl3.h"
#include "plan.h"

#ifndef __CUDACC__
struct int4_host { int x, y, z, w; };
#endif

namespace exl3 {

struct RoutePackArgs {
    const void *ids;
    int R, E, capacity, rg_size, nw;
    // fused layer regime model: rows per prefill-regime item (0: that regime
    // is not allowed), rows per decode-regime row group of the plain forward
    // and its cost in hundredths of a microsecond (8 rows: 1050, 16 rows:
    // 1700).  A layer whose residual stages all have scale zero is the plain
    // forward, so the model never depends on the stages.
    int tc_rows, cost_rg, dec_unit_cost;
    int32_t *offsets, *packed, *tiles, *info;
    int32_t *zero;                  // words to clear (per-call counters), or null
    int nzero;
    // fused-layer planning (plan != 0)
    int plan;
    void *rg;                       // int4 [max_rg] = (expert, first row, rows, 0)
    int nb1, nb2, nchunks1, nchunks2, split_pairs1, split_pairs2, num_sms;
    const int64_t *t_trellis, *t_suh, *t_svh, *t_scale;
    const int32_t *t_K, *t_cb;
    int num_stages;
    const int64_t *s_trellis;
    const float *s_scale;
    const int32_t *s_K;
};

struct RotateArgs {
    const void *x;
    int act_dtype, rows, width, nproj;
    // fused layer: row i is packed slot i, token = packed[i] / topk, suh from the table
    const int32_t *packed;
    const void *ids;
    int ids_dtype, topk;
    const int64_t *t_suh;
    // linear: row i is token i, one suh
    const uint16_t *suh;
    uint16_t *out;                  // fp16 [rows][nproj][width]
    int32_t *hdr;                   // skip everything when the error word is set
    int32_t *zero;                  // words to clear
    int nzero;
    int32_t *hdr_reset;             // linear: header to reset (error word)
    int num_sms;                    // sizes the large-layer grid (rows per warp)
    int rpw;                        // large layers: rows per warp (set by launch_rotate)
    // let the next kernel (launched with programmatic dependent launch) start
    // once every CTA of this grid is running: the tcgen05 linear only (early
    // resident decode-regime CTAs crowd out the rotate's blocks)
    int trigger;
};

enum GemmMode { kModeGateUp = 0, kModeDown = 1, kModeLinear = 2 };

struct GemmArgs {
    int act_dtype;
    int in_f, out_f, nb, nchunks;
    int32_t *hdr;
    const void *rg;                 // int4 row groups (fused layer)
    // linear: host-planned work
    int M, n_items_host, split_host;
    const uint16_t *act;            // fp16 rows (rotated activations)
    long act_row_stride;            // halves between rows
    // gate/up of small decode-regime layers: rotate the raw activations x
    // (act_dtype, [M][in_f]) while loading each chunk instead of reading act
    const void *x;
    int fuse_rot;
    // launch with programmatic dependent launch (decode-regime layers): the
    // kernel waits for its predecessor itself, before reading its outputs
    int pdl;
    // expert tables (fused layer)
    const int64_t *t_trellis, *t_suh, *t_svh, *t_scale;
    const int32_t *t_K, *t_cb;
    // linear projection
    exl3_proj lin;
    // additive stages
    int num_stages, E;
    const int64_t *s_trellis;
    const float *s_scale;
    const int32_t *s_K;
    // split partials
    float *part;
    int32_t *cnt_split;
    // outputs
    uint16_t *ad;                   // gate/up: fp16 [R][inter]
    // fp32 staging: down [R][hidden] (flat route order); prefill-regime
    // gate/up [R][2][inter] (packed order: rotated gate, rotated up)
    float *stage;
    const int32_t *packed;
    int topk;
    const void *rw;
    int rw_dtype;
    int32_t *cnt_comb;
    void *out;                      // down: [M][hidden] act; linear: [M][out] act
    int M_tokens;
    // tcgen05 linear: rows per item (256; above that an item is two halves of
    // lin_rows / 2 rows sharing each decoded weight stage)
    int lin_rows;
    // tcgen05 linear: the kernel launched just before is the rotate kernel,
    // so only the activation producer needs to wait for it
    int tc_pdl;
};

int route_pack_hist_warps(int E, int R);
cudaError_t launch_route_pack(const RoutePackArgs &a, int ids_dtype, cudaStream_t s);
cudaError_t route_pack_set_attributes();
cudaError_t launch_rotate(const RotateArgs &a, cudaStream_t s);
cudaError_t launch_gemm_gateup(bool additive, int nrb, const GemmArgs &a, int grid, cudaStream_t s);
cudaError_t launch_gemm_down(bool additive, int nrb, const GemmArgs &a, int grid, cudaStream_t s);
cudaError_t launch_gemm_linear(const GemmArgs &a, int grid, cudaStream_t s);
// Prefill-regime activation tensor maps: 2D fp16 [rows][cols] views of the
// rotated activations, one map per box height 16 << i rows; a box {kTcKs,
// 16 << i} (128-byte rows, 128-byte swizzle) is one stage's B tile.  A
// launch of the linear's two-half items uses only act[0], of box {kTcKs,
// lin_rows / 2}.
constexpr int kTcMaps = 5;
constexpr int kTcKs = 64;
struct TcMaps {
    CUtensorMap act[kTcMaps];
};
cudaError_t launch_tc_gateup(const GemmArgs &a, const TcMaps &maps, int grid, cudaStream_t s);
cudaError_t launch_tc_down(const GemmArgs &a, const TcMaps &maps, int grid, cudaStream_t s);
cudaError_t launch_tc_linear(const GemmArgs &a, const TcMaps &maps, int grid, cudaStream_t s);
// Prefill-regime layer steps between and after the GEMMs (no-ops unless the
// route-pack plan chose that regime): SwiGLU + down-input rotation of the
// staged gate/up rows, and the route-weighted combine of the staged down rows.
cudaError_t launch_tc_gu_finish(const GemmArgs &a, int sms, cudaStream_t s);
cudaError_t launch_tc_combine(const GemmArgs &a, int sms, cudaStream_t s);
cudaError_t tc_set_attributes();
int tc_rows_per_item();
cudaError_t gemm_gateup_set_attributes();
cudaError_t gemm_down_set_attributes();
cudaError_t gemm_linear_set_attributes();
// resident CTAs per SM of the GEMM kernels: 8-row items (3, additive 2), 16-row items 1
constexpr int gemm_ctas_per_sm(int nrb, bool additive) { return nrb == 2 ? 1 : (additive ? 2 : 3); }

}  // namespace exl3
