// Route histogram, exclusive scan and stable packing of (token, expert) routes
// into per-expert spans, capacity tiles and row groups ("MoE: Add fused additive
// EXL3 kernels", exllamav3 #284, "Summary" and "Relationship to #246").
//
// One CTA of 1024 threads.  The routes are cut into nw contiguous chunks, one
// per warp.  Pass 1 builds a per-warp histogram in shared memory; the expert
// scan turns (expert-major, warp-minor) counts into per-warp write cursors;
// pass 2 walks each chunk in order, 32 routes at a time, ranking equal ids
// inside the step with __match_any_sync.  The result is the unique stable
// order (ascending flat route index inside each expert's span).
#include "common.cuh"
#include "kernels.h"

namespace exl3 {

namespace {

constexpr int kThreads = 1024;

// Exclusive scan of v over the block (one value per thread); returns the
// exclusive prefix and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int *warp_sums, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d)
            x += y;
    }
    if (lane == 31)
        warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
        int s = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, d);
            if (lane >= d)
                s += y;
        }
        warp_sums[lane] = s - w;          // exclusive warp offsets
        if (lane == 31)
            warp_sums[32] = s;
    }
    __syncthreads();
    int r = warp_sums[warp] + x - v;
    *total = warp_sums[32];
    __syncthreads();
    return r;
}

template <typename IdT>
__device__ __forceinline__ long long read_id(const IdT *ids, int f)
{
    return static_cast<long long>(ids[f]);
}

// The call's plan in the workspace header (one thread): tile, active-expert and
// row-group counts, the contraction split of each decode-regime kernel and the
// regime.  bad_table: an active expert's table entry is invalid.
__device__ void write_plan_header(const RoutePackArgs &a, int ntiles, int nact, int n_rg, bool bad_table,
                                  bool use_tc)
{
    a.info[kHdrNTiles] = ntiles;
    a.info[kHdrNumActive] = nact;
    if (!a.plan)
        return;
    if (bad_table) {
        a.info[kHdrError] |= EXL3_DERR_TABLE;
        n_rg = 0;
    }
    a.info[kHdrNRg] = n_rg;
    const int pairs1 = n_rg * a.nb1, pairs2 = n_rg * a.nb2;
    const int lim = min(kSplitMaxPairs, 4 * a.num_sms);
    // the prefill regime never splits the contraction
    const int split1 = !use_tc && a.nchunks1 > 1 && pairs1 <= min(lim, a.split_pairs1);
    const int split2 = !use_tc && a.nchunks2 > 1 && pairs2 <= min(lim, a.split_pairs2);
    a.info[kHdrSplit1] = split1;
    a.info[kHdrSplit2] = split2;
    // prefill-regime gate/up items are single projections: two per pair
    a.info[kHdrNItems1] = use_tc ? 2 * pairs1 : (split1 ? pairs1 * a.nchunks1 : pairs1);
    a.info[kHdrNItems2] = split2 ? pairs2 * a.nchunks2 : pairs2;
    a.info[kHdrRegime] = use_tc ? 1 : 0;
}

// Table entries of an active expert (the fused layer): widths, codebooks,
// 16-/8-byte aligned non-null pointers, and every residual stage of nonzero
// scale.  True when something is invalid.
__device__ bool bad_tables(const RoutePackArgs &a, int e)
{
    int K[3], cb[3];
    long long tr[3], su[3], sv[3], sc[3];
#pragma unroll
    for (int p = 0; p < 3; p++) {          // independent loads, issued together
        const int i = e * 3 + p;
        K[p] = a.t_K[i];
        cb[p] = a.t_cb[i];
        tr[p] = a.t_trellis[i];
        su[p] = a.t_suh[i];
        sv[p] = a.t_svh[i];
        sc[p] = a.t_scale[i];
    }
    bool bad = false;
#pragma unroll
    for (int p = 0; p < 3; p++) {
        bad |= (K[p] < 1) | (K[p] > 8) | (cb[p] < 0) | (cb[p] > 2) | (tr[p] == 0) |
               ((tr[p] & 15) != 0) | (su[p] == 0) | ((su[p] & 7) != 0) | (sv[p] == 0) |
               ((sv[p] & 7) != 0) | (sc[p] == 0) | ((sc[p] & 7) != 0);
    }
    for (int st = 1; st < a.num_stages; st++) {
#pragma unroll
        for (int p = 0; p < 3; p++) {
            const int j = ((st - 1) * a.E + e) * 3 + p;
            const float al = a.s_scale[j];
            const int Ks = a.s_K[j];
            const long long ts = a.s_trellis[j];
            if (al != 0.0f)
                bad |= (Ks < 1) | (Ks > 8) | (ts == 0) | ((ts & 15) != 0);
        }
    }
    return bad;
}

}  // namespace

// Layers of at most 32 routes (one decode step): one warp, no block barriers.
// Lane f holds route f; __match_any_sync groups equal experts, the rank inside
// a group is the count of lower lanes (the stable order), and every count,
// offset and tile position is a sum over the other lanes by shuffles.  Same
// outputs as k_route_pack.
template <typename IdT>
__global__ void __launch_bounds__(32, 1) k_route_pack_warp(RoutePackArgs a)
{
    const IdT *ids = static_cast<const IdT *>(a.ids);
    const int E = a.E, R = a.R, lane = threadIdx.x;
    for (int i = lane; i < a.nzero; i += 32)
        a.zero[i] = 0;
    const bool valid = lane < R;
    const long long id = valid ? static_cast<long long>(ids[lane]) : -1;
    if (lane == 0) {
        a.info[kHdrError] = 0;
        if (a.plan)
            a.info[kHdrRegime] = 0;
    }
    if (__any_sync(0xffffffffu, valid && (id < 0 || id >= E))) {
        if (lane == 0) {
            a.info[kHdrError] |= EXL3_DERR_ROUTE_ID;
            a.info[kHdrNTiles] = 0;
            a.info[kHdrNumActive] = 0;
            if (a.plan) {
                a.info[kHdrNRg] = 0;
                a.info[kHdrNItems1] = 0;
                a.info[kHdrNItems2] = 0;
            }
        }
        return;
    }
    const int e = valid ? static_cast<int>(id) : E;          // invalid lanes sort last
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    const unsigned peers = __match_any_sync(0xffffffffu, e) & vmask;
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int cnt = __popc(peers);
    const bool leader = valid && rank == 0;                  // lowest lane of its expert
    const int ntile_e = leader ? (cnt + a.capacity - 1) / a.capacity : 0;
    int nrg_e = 0;
    if (leader && a.plan)
        for (int s0 = 0; s0 < cnt; s0 += a.capacity)
            nrg_e += (min(a.capacity, cnt - s0) + a.rg_size - 1) / a.rg_size;
    // position of this expert's span, tiles and row groups: sums over the
    // routes / leaders of lower experts
    int off_e = 0, tile_off = 0, rg_off = 0, ntiles = 0, n_rg = 0;
    for (int f = 0; f < 32; f++) {
        const int ef = __shfl_sync(0xffffffffu, e, f);
        const int tf = __shfl_sync(0xffffffffu, ntile_e, f);
        const int gf = __shfl_sync(0xffffffffu, nrg_e, f);
        off_e += (f < R && ef < e) ? 1 : 0;
        tile_off += ef < e ? tf : 0;
        rg_off += ef < e ? gf : 0;
        ntiles += tf;
        n_rg += gf;
    }
    if (valid)
        a.packed[off_e + rank] = lane;
    // offsets[x] = routes with an expert below x, for every x in 0..E (the
    // loop bounds are warp-uniform, so every lane takes part in each shuffle)
    for (int x0 = 0; x0 <= E; x0 += 32) {
        const int x = x0 + lane;
        int c = 0;
        for (int f = 0; f < R; f++)
            c += __shfl_sync(0xffffffffu, e, f) < x ? 1 : 0;
        if (x <= E)
            a.offsets[x] = c;
    }
    const int nact = __popc(__ballot_sync(0xffffffffu, leader));
    if (leader) {
        for (int s0 = 0, t = 0; s0 < cnt; s0 += a.capacity, t++) {
            int *tt = a.tiles + 3 * (tile_off + t);
            tt[0] = e;
            tt[1] = off_e + s0;
            tt[2] = min(a.capacity, cnt - s0);
        }
        if (a.plan) {
            int k = rg_off;
            for (int s0 = 0; s0 < cnt; s0 += a.capacity) {
                const int len = min(a.capacity, cnt - s0);
                for (int r = 0; r < len; r += a.rg_size)
                    static_cast<int4 *>(a.rg)[k++] = make_int4(e, off_e + s0 + r, min(a.rg_size, len - r), 0);
            }
        }
    }
    const bool bad = a.plan && leader && bad_tables(a, e);
    const bool any_bad = __any_sync(0xffffffffu, bad);
    if (lane == 0)
        write_plan_header(a, ntiles, nact, n_rg, any_bad, false);
}

template <typename IdT>
__global__ void __launch_bounds__(kThreads, 1) k_route_pack(RoutePackArgs a)
{
    extern __shared__ int smem_i[];
    const IdT *ids = static_cast<const IdT *>(a.ids);
    const int E = a.E, R = a.R;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int nw = a.nw;                       // warps holding a histogram row
    int *hist = smem_i;                        // [nw][E]
    __shared__ int s_warp[40];
    __shared__ int s_err;

    for (int i = tid; i < nw * E; i += kThreads)
        hist[i] = 0;
    for (int i = tid; i < a.nzero; i += kThreads)
        a.zero[i] = 0;
    if (tid == 0) {
        s_err = 0;
        a.info[kHdrError] = 0;
        if (a.plan)
            a.info[kHdrRegime] = 0;
    }
    __syncthreads();

    // chunk of each warp: whole 32-route steps
    const int steps = (R + 31) / 32;
    const int per_warp = (steps + nw - 1) / nw;
    const int f_begin = warp * per_warp * 32;
    const int f_end = min(R, f_begin + per_warp * 32);

    // pass 1: validate and count
    if (warp < nw) {
        for (int f = f_begin + lane; f < f_end; f += 32) {
            long long e = read_id(ids, f);
            if (e < 0 || e >= E)
                s_err = 1;
            else
                atomicAdd(&hist[warp * E + (int)e], 1);
        }
    }
    __syncthreads();
    if (s_err) {
        if (tid == 0) {
            a.info[kHdrError] |= EXL3_DERR_ROUTE_ID;
            a.info[kHdrNTiles] = 0;
            a.info[kHdrNumActive] = 0;
            if (a.plan) {
                a.info[kHdrNRg] = 0;
                a.info[kHdrNItems1] = 0;
                a.info[kHdrNItems2] = 0;
            }
        }
        return;
    }

    // per-expert totals, spans and tile / row-group counts
    int cnt = 0;
    if (tid < E)
        for (int w = 0; w < nw; w++)
            cnt += hist[w * E + tid];
    int total;
    const int off = block_exclusive_scan(tid < E ? cnt : 0, s_warp, &total);
    const int ntile_e = (tid < E) ? (cnt + a.capacity - 1) / a.capacity : 0;
    int ntiles;
    const int tile_off = block_exclusive_scan(ntile_e, s_warp, &ntiles);
    // Regime choice (fused layer): both regimes decode a whole expert block
    // once per work item, the decode regime per row group of rg_size rows, the
    // prefill regime per item of up to tc_rows rows.  Measured cost per item
    // (hidden 5120, inter 1536, K 3-4; other shapes scale both alike): decode
    // regime 10.5 us (8-row groups) or 17 us (16-row groups), prefill regime
    // 12.0 + 8.1 * rows / 256 us (the earlier 14.4 + 9.8 scaled by the
    // measured GEMM time of the current prefill kernels on the 3072-token
    // layer, 2.90 -> 2.39 ms).  The regime with the smaller total wins; the
    // choice depends only on the routing.
    // (integer costs in hundredths, so the sums and the choice are exact)
    // Residual stages add the same decode work to both regimes and are left
    // out, so a call whose stage scales are all 0 chooses as the plain
    // forward does.
    __shared__ long long s_cost[2];
    __shared__ int s_tc;
    if (tid == 0) {
        s_cost[0] = 0;
        s_cost[1] = 0;
    }
    __syncthreads();
    if (tid < E && a.plan && a.tc_rows > 0 && cnt > 0) {
        long long cd = 0, ct = 0;
        for (int s = 0; s < ntile_e; s++) {
            const int len = min(a.capacity, cnt - s * a.capacity);
            cd += (long long)a.dec_unit_cost * ((len + a.cost_rg - 1) / a.cost_rg);
            for (int r = 0; r < len; r += a.tc_rows)
                ct += 1200 + 810 * min(a.tc_rows, len - r) / 256;
        }
        atomicAdd(reinterpret_cast<unsigned long long *>(&s_cost[0]), (unsigned long long)cd);
        atomicAdd(reinterpret_cast<unsigned long long *>(&s_cost[1]), (unsigned long long)ct);
    }
    __syncthreads();
    if (tid == 0)
        s_tc = a.plan && a.tc_rows > 0 && s_cost[1] < s_cost[0];
    __syncthreads();
    const bool use_tc = s_tc != 0;
    const int rg_size = use_tc ? a.tc_rows : a.rg_size;
    int nrg_e = 0;
    if (tid < E && a.plan) {
        for (int s = 0; s < ntile_e; s++) {
            int len = min(a.capacity, cnt - s * a.capacity);
            nrg_e += (len + rg_size - 1) / rg_size;
        }
    }
    int n_rg;
    const int rg_off = block_exclusive_scan(nrg_e, s_warp, &n_rg);
    int nact;
    block_exclusive_scan((tid < E && cnt > 0) ? 1 : 0, s_warp, &nact);
    if (tid < E) {
        a.offsets[tid] = off;
        // per-warp cursors: expert-major, warp-minor
        int run = off;
        for (int w = 0; w < nw; w++) {
            int c = hist[w * E + tid];
            hist[w * E + tid] = run;
            run += c;
        }
    }
    if (tid == 0)
        a.offsets[E] = total;
    __syncthreads();

    // pass 2: stable placement
    if (warp < nw) {
        const unsigned lt = (1u << lane) - 1u;
        for (int f0 = f_begin; f0 < f_end; f0 += 32) {
            const int f = f0 + lane;
            const bool valid = f < f_end;
            const unsigned vmask = __ballot_sync(0xffffffffu, valid);
            int e = valid ? (int)read_id(ids, f) : -1;
            unsigned peers = __match_any_sync(0xffffffffu, e);
            if (valid) {
                peers &= vmask;
                int rank = __popc(peers & lt);
                int base = hist[warp * E + e];
                a.packed[base + rank] = f;
            }
            __syncwarp();
            if (valid && (peers & lt) == 0)          // lowest lane of its group
                hist[warp * E + e] += __popc(peers);
            __syncwarp();
        }
    }

    // capacity tiles (and row groups for the fused layer)
    if (tid < E && cnt > 0) {
        for (int s = 0; s < ntile_e; s++) {
            const int start = off + s * a.capacity;
            const int len = min(a.capacity, cnt - s * a.capacity);
            int *t = a.tiles + 3 * (tile_off + s);
            t[0] = tid; t[1] = start; t[2] = len;
        }
        if (a.plan) {
            int k = rg_off;
            for (int s = 0; s < ntile_e; s++) {
                const int start = off + s * a.capacity;
                const int len = min(a.capacity, cnt - s * a.capacity);
                for (int r = 0; r < len; r += rg_size)
                    static_cast<int4 *>(a.rg)[k++] = make_int4(tid, start + r, min(rg_size, len - r), 0);
            }
        }
    }

    // the fused layer: validate the tables of every expert that receives routes
    if (a.plan && tid < E && cnt > 0 && bad_tables(a, tid))
        s_err = 2;
    __syncthreads();

    if (tid == 0)
        write_plan_header(a, ntiles, nact, n_rg, s_err != 0, use_tc);
}

// Warps holding a histogram row: at most 32, at most 16384 counters of shared
// memory, and no more than the 32-route steps there are (each warp walks the
// per-expert rows when it sums counts and sets cursors, so idle rows cost time).
int route_pack_hist_warps(int E, int R)
{
    int nw = 16384 / (E > 0 ? E : 1);
    const int steps = (R + 31) / 32;
    nw = nw < steps ? nw : steps;
    return nw < 1 ? 1 : (nw > 32 ? 32 : nw);
}

cudaError_t launch_route_pack(const RoutePackArgs &a, int ids_dtype, cudaStream_t s)
{
    if (a.R <= 32 && a.tc_rows == 0) {
        // one decode step: the one-warp kernel (the regime is the decode one)
        if (ids_dtype == EXL3_I64)
            k_route_pack_warp<int64_t><<<1, 32, 0, s>>>(a);
        else
            k_route_pack_warp<int32_t><<<1, 32, 0, s>>>(a);
        return cudaGetLastError();
    }
    const size_t smem = (size_t)a.nw * a.E * sizeof(int);
    if (ids_dtype == EXL3_I64) {
        k_route_pack<int64_t><<<1, kThreads, smem, s>>>(a);
    } else {
        k_route_pack<int32_t><<<1, kThreads, smem, s>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t route_pack_set_attributes()
{
    const int max_dyn = 16384 * (int)sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(k_route_pack<int32_t>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn);
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(k_route_pack<int64_t>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn);
}

}  // namespace exl3
