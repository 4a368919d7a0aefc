// Host side of the C ABI (include/exl3.h): argument validation, workspace
// planning and kernel launches.  Nothing here allocates, frees or synchronises
// (except exl3_workspace_error, which is documented to synchronise).
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "kernels.h"

using namespace exl3;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kLinearTcMinRows = 128;  // linear: more rows than this take the tcgen05 kernel
constexpr int kPdlRoutes = 64;         // routes up to which gate/up -> down use programmatic dependent launch
constexpr int kFuseRotRoutes = 32;     // routes up to which gate/up rotates its own inputs (measured: M=1 -7 us, M=8 +25 us)

struct DeviceState {
    int num_sms = 0;
    bool ready = false;
};

DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
thread_local void *const *g_prof_events = nullptr;

void prof_mark(int i, cudaStream_t s)
{
    if (g_prof_events)
        cudaEventRecord(static_cast<cudaEvent_t>(g_prof_events[i]), s);
}

// True while the calling thread's call is being recorded into a CUDA graph:
// the stream-device and pointer-residency queries are skipped then (they fail
// on a capturing stream and would invalidate the capture); the eager calls
// that must precede any capture run them.
thread_local bool g_capturing = false;

// Device of the stream (must be the current device); lazily sets kernel attributes.
int setup_device(cudaStream_t s, int *dev_out, int *sms_out)
{
    int cur = -1, dev = -1;
    if (cudaGetDevice(&cur) != cudaSuccess)
        return EXL3_E_CUDA;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        return EXL3_E_DEVICE;
    }
    g_capturing = cs != cudaStreamCaptureStatusNone;
    if (g_capturing) {
        dev = cur;
    } else if (cudaStreamGetDevice(s, &dev) != cudaSuccess) {
        cudaGetLastError();
        return EXL3_E_DEVICE;
    }
    if (dev != cur || dev < 0 || dev >= kMaxDevices)
        return EXL3_E_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        if (g_capturing)
            return EXL3_E_CUDA;              // the first call per device sets kernel attributes
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return EXL3_E_CUDA;
        if (route_pack_set_attributes() != cudaSuccess || gemm_gateup_set_attributes() != cudaSuccess ||
            gemm_down_set_attributes() != cudaSuccess || gemm_linear_set_attributes() != cudaSuccess ||
            tc_set_attributes() != cudaSuccess)
            return EXL3_E_CUDA;
        d.ready = true;
    }
    *dev_out = dev;
    *sms_out = d.num_sms;
    return EXL3_OK;
}

bool on_device(const void *p, int dev)
{
    if (g_capturing)
        return true;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (the library
// does not link the driver library itself); looked up once.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// fp16 [rows][cols] (row pitch cols * 2 bytes) -> one map per box {kTcKs,
// 16 << i} with the 128-byte swizzle of a 128-byte row, or (half_rows > 0)
// only the map of box {kTcKs, half_rows}; rows past the end read as zero.
bool encode_act_maps(TcMaps &m, const void *base, int cols, int rows, int half_rows = 0)
{
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B;
    for (int i = 0; i < kTcMaps; i++) {
        // two-half linear items: only act[0], of box height half_rows
        if (half_rows > 0 && i > 0) {
            memset(&m.act[i], 0, sizeof(m.act[i]));
            continue;
        }
        const int box_rows = half_rows > 0 ? half_rows : 16 << i;
        CUtensorMap *dst = &m.act[i];
        const cuuint32_t box[2] = {(cuuint32_t)kTcKs, (cuuint32_t)box_rows};
        if (fn(dst, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

bool act_dtype_ok(int d) { return d == EXL3_F16 || d == EXL3_BF16; }
bool ids_dtype_ok(int d) { return d == EXL3_I32 || d == EXL3_I64; }
bool rw_dtype_ok(int d) { return d == EXL3_F16 || d == EXL3_BF16 || d == EXL3_F32; }
size_t rw_size(int d) { return d == EXL3_F32 ? 4 : 2; }

int check_moe_args(const void *x, int act_dtype, int M, int hidden, int inter, int E, int topk,
                   const void *ids, int ids_dtype, const void *rw, int rw_dtype,
                   const exl3_experts *ex, int capacity, void *ws, size_t ws_bytes, void *out,
                   int dev)
{
    if (!x || !ids || !rw || !ex || !ws || !out || !ex->trellis || !ex->suh || !ex->svh ||
        !ex->scale || !ex->K || !ex->codebook)
        return EXL3_E_NULL;
    if (!act_dtype_ok(act_dtype) || !ids_dtype_ok(ids_dtype) || !rw_dtype_ok(rw_dtype))
        return EXL3_E_DTYPE;
    if (M < 0 || hidden <= 0 || inter <= 0 || hidden % kHb || inter % kHb ||
        (long long)M * topk >= (1ll << 30) || (long long)M * hidden >= (1ll << 40))
        return EXL3_E_SHAPE;
    if (E < 1 || E > EXL3_MAX_EXPERTS || topk < 1 || topk > E || capacity < 1)
        return EXL3_E_ROUTING;
    if (!aligned(x, 16) || !aligned(out, 16) || !aligned(ws, 256) ||
        !aligned(ids, ids_dtype == EXL3_I64 ? 8 : 4) || !aligned(rw, rw_size(rw_dtype)) ||
        !aligned(ex->trellis, 8) || !aligned(ex->suh, 8) || !aligned(ex->svh, 8) ||
        !aligned(ex->scale, 8) || !aligned(ex->K, 4) || !aligned(ex->codebook, 4))
        return EXL3_E_ALIGN;
    const void *ptrs[] = {x, ids, rw, ws, out, ex->trellis, ex->suh, ex->svh, ex->scale, ex->K,
                          ex->codebook};
    for (const void *p : ptrs)
        if (!on_device(p, dev))
            return EXL3_E_DEVICE;
    MoeLayout L = moe_layout(M, topk, E, hidden, inter, capacity);
    if (ws_bytes < L.total)
        return EXL3_E_WORKSPACE;
    return EXL3_OK;
}

int run_moe(const void *x, int act_dtype, int M, int hidden, int inter, int E, int topk,
            const void *ids, int ids_dtype, const void *rw, int rw_dtype, const exl3_experts *ex,
            const exl3_stages *st, int capacity, void *ws, void *out, int sms, cudaStream_t s)
{
    const bool additive = st != nullptr && st->num_stages > 1;
    const MoeLayout L = moe_layout(M, topk, E, hidden, inter, capacity);
    uint8_t *w = static_cast<uint8_t *>(ws);
    int32_t *hdr = reinterpret_cast<int32_t *>(w + L.hdr);
    const int R = L.R;
    // Two regimes: decode (mma.sync; 16-row items at 1 CTA/SM when experts
    // carry more than 8 routes on average, else 8 rows; residual stages: 8
    // rows) and prefill (tcgen05, up to 256 routes per item; residual stages
    // as extra passes over the same accumulators).  With more than 128 tokens
    // both kernel pairs are launched and the route-pack kernel picks one from
    // the per-expert route counts (the other pair returns at once).  M <= 128
    // always takes the decode regime, so a row's bytes never depend on M
    // there.
    const int active = E < R ? E : R;
    const bool tc_ok = M > 128;
    const int nrb_plain = R > 8 * active ? 2 : 1;
    const int nrb = additive ? 1 : nrb_plain;
    const int ctas = gemm_ctas_per_sm(nrb, additive);
    // Small decode-regime layers rotate the inputs inside the gate/up kernel
    // (same fp16 bits as the rotate kernel), saving a launch; the route-pack
    // kernel then clears the per-call counters.
    const bool fuse_rot = !tc_ok && R <= kFuseRotRoutes;

    RoutePackArgs rp{};
    rp.ids = ids;
    rp.R = R;
    rp.E = E;
    rp.capacity = capacity;
    rp.rg_size = 8 * nrb;
    rp.tc_rows = tc_ok ? tc_rows_per_item() : 0;
    rp.cost_rg = 8 * nrb_plain;
    rp.dec_unit_cost = nrb_plain == 2 ? 1700 : 1050;
    rp.nw = route_pack_hist_warps(E, rp.R);
    rp.offsets = reinterpret_cast<int32_t *>(w + L.offsets);
    rp.packed = reinterpret_cast<int32_t *>(w + L.packed);
    rp.tiles = reinterpret_cast<int32_t *>(w + L.tiles);
    rp.info = hdr;
    rp.plan = 1;
    rp.rg = w + L.rg;
    rp.nb1 = L.nb1;
    rp.nb2 = L.nb2;
    rp.nchunks1 = L.nchunks1;
    rp.nchunks2 = L.nchunks2;
    rp.split_pairs1 = L.split_pairs1;
    rp.split_pairs2 = L.split_pairs2;
    rp.num_sms = sms;
    rp.t_trellis = ex->trellis;
    rp.t_suh = ex->suh;
    rp.t_svh = ex->svh;
    rp.t_scale = ex->scale;
    rp.t_K = ex->K;
    rp.t_cb = ex->codebook;
    rp.num_stages = additive ? st->num_stages : 1;
    rp.s_trellis = additive ? st->trellis : nullptr;
    rp.s_scale = additive ? st->scale : nullptr;
    rp.s_K = additive ? st->K : nullptr;
    rp.zero = fuse_rot ? reinterpret_cast<int32_t *>(w + L.cnt) : nullptr;
    rp.nzero = fuse_rot ? (int)((L.cnt2 - L.cnt) / 4) + L.split_pairs2 : 0;
    prof_mark(0, s);
    if (launch_route_pack(rp, ids_dtype, s) != cudaSuccess)
        return EXL3_E_CUDA;
    prof_mark(1, s);

    RotateArgs ra{};
    ra.x = x;
    ra.act_dtype = act_dtype;
    ra.rows = R;
    ra.num_sms = sms;
    ra.width = hidden;
    ra.nproj = 2;
    ra.packed = rp.packed;
    ra.ids = ids;
    ra.ids_dtype = ids_dtype;
    ra.topk = topk;
    ra.t_suh = ex->suh;
    ra.out = reinterpret_cast<uint16_t *>(w + L.arot);
    ra.hdr = hdr;
    ra.zero = reinterpret_cast<int32_t *>(w + L.cnt);
    ra.nzero = (int)((L.cnt2 - L.cnt) / 4) + L.split_pairs2;
    if (!fuse_rot && launch_rotate(ra, s) != cudaSuccess)
        return EXL3_E_CUDA;
    prof_mark(2, s);

    GemmArgs g{};
    g.act_dtype = act_dtype;
    g.hdr = hdr;
    g.rg = w + L.rg;
    g.t_trellis = ex->trellis;
    g.t_suh = ex->suh;
    g.t_svh = ex->svh;
    g.t_scale = ex->scale;
    g.t_K = ex->K;
    g.t_cb = ex->codebook;
    g.num_stages = rp.num_stages;
    g.E = E;
    g.s_trellis = rp.s_trellis;
    g.s_scale = rp.s_scale;
    g.s_K = rp.s_K;
    g.topk = topk;
    g.M_tokens = M;

    // gate/up: [R][2][hidden] -> SwiGLU -> rotated down inputs [R][inter]
    g.in_f = hidden;
    g.out_f = inter;
    g.nb = L.nb1;
    g.nchunks = L.nchunks1;
    g.act = ra.out;
    g.act_row_stride = 2L * hidden;
    g.x = x;
    g.fuse_rot = fuse_rot ? 1 : 0;
    // small decode-regime layers chain gate/up -> down with programmatic
    // dependent launch: down streams its first trellis words during gate/up's
    // tail (measured: M=1 -5%, 16-route layer -15%; above 64 routes the early
    // down CTAs slow gate/up's tail, a 288-expert layer at M=64 by 21%)
    g.pdl = (!tc_ok && R <= kPdlRoutes) ? 1 : 0;
    g.packed = rp.packed;
    g.part = reinterpret_cast<float *>(w + L.part1);
    g.cnt_split = reinterpret_cast<int32_t *>(w + L.cnt1);
    g.ad = reinterpret_cast<uint16_t *>(w + L.ad);
    g.stage = reinterpret_cast<float *>(w + L.stage);
    TcMaps maps1, maps2;
    if (tc_ok && (!encode_act_maps(maps1, g.act, 2 * hidden, R) || !encode_act_maps(maps2, g.ad, inter, R)))
        return EXL3_E_CUDA;
    // prefill regime: gate and up items stage their rotated outputs, then
    // SwiGLU + the down-input rotation run as one elementwise pass
    if ((tc_ok && launch_tc_gateup(g, maps1, sms, s) != cudaSuccess) ||
        launch_gemm_gateup(additive, nrb, g, sms * ctas, s) != cudaSuccess ||
        (tc_ok && launch_tc_gu_finish(g, sms, s) != cudaSuccess))
        return EXL3_E_CUDA;
    prof_mark(3, s);

    // down: [R][inter] -> [R][hidden] fp32 staging -> combine into out
    g.in_f = inter;
    g.out_f = hidden;
    g.nb = L.nb2;
    g.nchunks = L.nchunks2;
    g.act = g.ad;
    g.act_row_stride = inter;
    g.part = reinterpret_cast<float *>(w + L.part2);
    g.cnt_split = reinterpret_cast<int32_t *>(w + L.cnt2);
    g.packed = rp.packed;
    g.rw = rw;
    g.rw_dtype = rw_dtype;
    g.cnt_comb = reinterpret_cast<int32_t *>(w + L.cnt);
    g.out = out;
    // prefill regime: down items stage their rotated rows; the weighted
    // combine follows as one pass in token order
    if ((tc_ok && launch_tc_down(g, maps2, sms, s) != cudaSuccess) ||
        launch_gemm_down(additive, nrb, g, sms * ctas, s) != cudaSuccess ||
        (tc_ok && launch_tc_combine(g, sms, s) != cudaSuccess))
        return EXL3_E_CUDA;
    prof_mark(4, s);
    return EXL3_OK;
}

}  // namespace

extern "C" {

int exl3_abi_version(void) { return EXL3_ABI_VERSION; }

size_t exl3_moe_workspace_bytes(int M, int topk, int E, int hidden, int inter, int capacity)
{
    if (M < 0 || topk < 1 || E < 1 || E > EXL3_MAX_EXPERTS || hidden <= 0 || inter <= 0 ||
        hidden % kHb || inter % kHb || capacity < 1 || (long long)M * topk >= (1ll << 30))
        return 0;
    return moe_layout(M, topk, E, hidden, inter, capacity).total;
}

size_t exl3_linear_workspace_bytes(int M, int in_features, int out_features)
{
    if (M < 0 || in_features <= 0 || out_features <= 0 || in_features % kHb ||
        out_features % kHb)
        return 0;
    return linear_layout(M, in_features, out_features).total;
}

int exl3_route_pack_max_tiles(int M, int topk, int E, int capacity)
{
    if (M < 0 || topk < 1 || E < 1 || capacity < 1)
        return 0;
    const int R = M * topk;
    return R / capacity + (E < R ? E : R);
}

int exl3_route_pack(const void *ids, int ids_dtype, int M, int topk, int E, int capacity,
                    int32_t *offsets, int32_t *packed, int32_t *tiles, int32_t *info,
                    cudaStream_t stream)
{
    int dev, sms;
    if (!offsets || !info || (M > 0 && (!ids || !packed || !tiles)))
        return EXL3_E_NULL;
    if (!ids_dtype_ok(ids_dtype))
        return EXL3_E_DTYPE;
    if (M < 0 || (long long)M * topk >= (1ll << 30))
        return EXL3_E_SHAPE;
    if (E < 1 || E > EXL3_MAX_EXPERTS || topk < 1 || capacity < 1)
        return EXL3_E_ROUTING;
    if (!aligned(ids, ids_dtype == EXL3_I64 ? 8 : 4) || !aligned(offsets, 4) ||
        !aligned(packed, 4) || !aligned(tiles, 4) || !aligned(info, 4))
        return EXL3_E_ALIGN;
    int rc = setup_device(stream, &dev, &sms);
    if (rc != EXL3_OK)
        return rc;
    const void *ptrs[] = {ids, offsets, info, packed, tiles};
    for (const void *p : ptrs)
        if (p && M > 0 && !on_device(p, dev))
            return EXL3_E_DEVICE;
    if (!on_device(offsets, dev) || !on_device(info, dev))
        return EXL3_E_DEVICE;
    RoutePackArgs rp{};
    rp.ids = ids;
    rp.R = M * topk;
    rp.E = E;
    rp.capacity = capacity;
    rp.rg_size = kRowGroup;
    rp.nw = route_pack_hist_warps(E, rp.R);
    rp.offsets = offsets;
    rp.packed = packed;
    rp.tiles = tiles;
    rp.info = info;
    rp.plan = 0;
    return launch_route_pack(rp, ids_dtype, stream) == cudaSuccess ? EXL3_OK : EXL3_E_CUDA;
}

int exl3_linear(const void *x, int act_dtype, int M, const exl3_proj *p, void *y, void *ws,
                size_t ws_bytes, cudaStream_t stream)
{
    if (!x || !p || !y || !ws || !p->trellis || !p->suh || !p->svh || !p->scale)
        return EXL3_E_NULL;
    if (!act_dtype_ok(act_dtype))
        return EXL3_E_DTYPE;
    if (M < 0 || p->in_features <= 0 || p->out_features <= 0 || p->in_features % kHb ||
        p->out_features % kHb || (long long)M * p->in_features >= (1ll << 40))
        return EXL3_E_SHAPE;
    if (p->K < 1 || p->K > 8 || p->codebook < EXL3_CB_MUL1 || p->codebook > EXL3_CB_3INST)
        return EXL3_E_CODEBOOK;
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(ws, 256) || !aligned(p->trellis, 16) ||
        !aligned(p->suh, 8) || !aligned(p->svh, 8) || !aligned(p->scale, 8))
        return EXL3_E_ALIGN;
    int dev, sms;
    int rc = setup_device(stream, &dev, &sms);
    if (rc != EXL3_OK)
        return rc;
    const void *ptrs[] = {x, y, ws, p->trellis, p->suh, p->svh, p->scale};
    for (const void *q : ptrs)
        if (!on_device(q, dev))
            return EXL3_E_DEVICE;
    const LinearLayout L = linear_layout(M, p->in_features, p->out_features);
    if (ws_bytes < L.total)
        return EXL3_E_WORKSPACE;
    if (M == 0)
        return EXL3_OK;
    uint8_t *w = static_cast<uint8_t *>(ws);
    int32_t *hdr = reinterpret_cast<int32_t *>(w + L.hdr);

    RotateArgs ra{};
    ra.x = x;
    ra.act_dtype = act_dtype;
    ra.rows = M;
    ra.num_sms = sms;
    ra.width = p->in_features;
    ra.nproj = 1;
    ra.suh = p->suh;
    ra.out = reinterpret_cast<uint16_t *>(w + L.arot);
    ra.zero = reinterpret_cast<int32_t *>(w + L.cnt);
    ra.nzero = L.split_pairs;
    ra.hdr_reset = hdr;
    ra.trigger = M > kLinearTcMinRows ? 1 : 0;     // the tcgen05 kernel follows
    if (launch_rotate(ra, stream) != cudaSuccess)
        return EXL3_E_CUDA;

    GemmArgs g{};
    g.act_dtype = act_dtype;
    g.in_f = p->in_features;
    g.out_f = p->out_features;
    g.nb = L.nb;
    g.nchunks = L.nchunks;
    g.hdr = hdr;
    g.M = M;
    const int pairs = L.n_rg * L.nb;
    const int lim = kSplitMaxPairs < 4 * sms ? kSplitMaxPairs : 4 * sms;
    g.split_host = L.nchunks > 1 && pairs <= lim && pairs <= L.split_pairs;
    g.n_items_host = g.split_host ? pairs * L.nchunks : pairs;
    g.act = ra.out;
    g.act_row_stride = p->in_features;
    g.lin = *p;
    g.num_stages = 1;
    g.part = reinterpret_cast<float *>(w + L.part);
    g.cnt_split = reinterpret_cast<int32_t *>(w + L.cnt);
    g.out = y;
    if (M > kLinearTcMinRows) {
        // prompt-sized inputs: the tcgen05 kernel, items of up to 256 rows x
        // 128 outputs, the whole contraction per item (M <= 128 keeps the
        // decode regime, so a row's bytes never depend on M there).  When
        // those items would need a second wave, items of up to 512 rows in
        // two halves (each decoded weight stage feeds both) fill one wave.
        g.split_host = 0;
        g.tc_pdl = 1;
        g.lin_rows = tc_rows_per_item();
        const int rg_per_wave = sms / L.nb;
        if (ceil_div(M, g.lin_rows) * L.nb > sms && rg_per_wave > 0) {
            const int r = (ceil_div(M, rg_per_wave) + 31) / 32 * 32;
            if (r <= 2 * tc_rows_per_item())
                g.lin_rows = r;
        }
        TcMaps maps;
        const int half_rows = g.lin_rows > tc_rows_per_item() ? g.lin_rows / 2 : 0;
        if (!encode_act_maps(maps, ra.out, p->in_features, M, half_rows))
            return EXL3_E_CUDA;
        g.n_items_host = ceil_div(M, g.lin_rows) * L.nb;
        const int grid = sms < g.n_items_host ? sms : g.n_items_host;
        return launch_tc_linear(g, maps, grid, stream) == cudaSuccess ? EXL3_OK : EXL3_E_CUDA;
    }
    int grid = sms * gemm_ctas_per_sm(2, false);
    if (grid > g.n_items_host)
        grid = g.n_items_host;
    return launch_gemm_linear(g, grid, stream) == cudaSuccess ? EXL3_OK : EXL3_E_CUDA;
}

int exl3_moe_forward(const void *x, int act_dtype, int M, int hidden, int inter, int E, int topk,
                     const void *ids, int ids_dtype, const void *rw, int rw_dtype,
                     const exl3_experts *ex, int capacity, void *ws, size_t ws_bytes, void *out,
                     cudaStream_t stream)
{
    int dev, sms;
    int rc = setup_device(stream, &dev, &sms);
    if (rc != EXL3_OK)
        return rc;
    rc = check_moe_args(x, act_dtype, M, hidden, inter, E, topk, ids, ids_dtype, rw, rw_dtype, ex,
                        capacity, ws, ws_bytes, out, dev);
    if (rc != EXL3_OK || M == 0)
        return rc;
    return run_moe(x, act_dtype, M, hidden, inter, E, topk, ids, ids_dtype, rw, rw_dtype, ex,
                   nullptr, capacity, ws, out, sms, stream);
}

int exl3_moe_additive(const void *x, int act_dtype, int M, int hidden, int inter, int E, int topk,
                      const void *ids, int ids_dtype, const void *rw, int rw_dtype,
                      const exl3_experts *ex, const exl3_stages *st, int capacity, void *ws,
                      size_t ws_bytes, void *out, cudaStream_t stream)
{
    int dev, sms;
    int rc = setup_device(stream, &dev, &sms);
    if (rc != EXL3_OK)
        return rc;
    if (!st)
        return EXL3_E_NULL;
    if (st->num_stages < 1)
        return EXL3_E_SHAPE;
    if (st->num_stages > 1) {
        if (!st->trellis || !st->scale || !st->K)
            return EXL3_E_NULL;
        if (!aligned(st->trellis, 8) || !aligned(st->scale, 4) || !aligned(st->K, 4))
            return EXL3_E_ALIGN;
        if (!on_device(st->trellis, dev) || !on_device(st->scale, dev) || !on_device(st->K, dev))
            return EXL3_E_DEVICE;
    }
    rc = check_moe_args(x, act_dtype, M, hidden, inter, E, topk, ids, ids_dtype, rw, rw_dtype, ex,
                        capacity, ws, ws_bytes, out, dev);
    if (rc != EXL3_OK || M == 0)
        return rc;
    return run_moe(x, act_dtype, M, hidden, inter, E, topk, ids, ids_dtype, rw, rw_dtype, ex, st,
                   capacity, ws, out, sms, stream);
}

int exl3_profile_events(void *const *events)
{
    g_prof_events = events;
    return EXL3_OK;
}

int exl3_workspace_error(const void *ws, int32_t *err_host, cudaStream_t stream)
{
    if (!ws || !err_host)
        return EXL3_E_NULL;
    if (cudaMemcpyAsync(err_host, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return EXL3_E_CUDA;
    return cudaStreamSynchronize(stream) == cudaSuccess ? EXL3_OK : EXL3_E_CUDA;
}

}  // extern "C"
