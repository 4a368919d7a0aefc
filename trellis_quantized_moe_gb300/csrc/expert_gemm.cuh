// Weight-streaming grouped GEMM over EXL3 trellis codes, for the gate/up
// projections (+ SwiGLU + down-input rotation), the down projection (+ output
// rotation + route-weighted combine) and the standalone linear.
//
// Follows "EXL3 linear and grouped routed experts" (TensorFold #837), "What this
// changes" (decode straight into tensor-core fragments, grouped experts, gate
// and up, SwiGLU, down, weighted combine, a width per expert) and "Receipt" (a
// row's bytes are the same for every row count, K split and member count), and
// "MoE: Add fused additive EXL3 kernels" (exllamav3 #284), "Summary" (FP32
// accumulation with output scaling for residual stages).
//
// Work item = (row group of <= 8*NRB routes of one expert, 128-output block,
// range of 512-input chunks).  Each of the 8 warps owns a fixed slice of every
// chunk, streams that slice's trellis words with cp.async.bulk into its own
// shared-memory ring of two 3 KB slots of whole tk rows (one mbarrier per
// slot), decodes each 16x16 tile
// in registers straight into mma.sync A fragments and multiplies by the rotated
// activations (B fragments, rows = routes).
//
// Decode: a thread decodes two runs of 4 consecutive trellis positions per
// tile (output columns g and g+8, input rows 4t..4t+3).  Both runs start at the
// same bit offset modulo 32, so 3 words + 2 funnel shifts give a 64-bit window
// from which each 16-bit state is one funnel shift and one shift.  mcg/3inst:
// the masked product holds two fp16 halves whose sum is the weight; instead of
// adding them, each half is one element of the MMA's k dimension against a
// duplicated activation, so the tensor core forms lo*a + hi*a exactly in fp32.
// mul1: __dp4a sums the four bytes onto the fp16 bit pattern of 1024, giving
// the exact integer byte sum - 510 after one half2 subtraction; 1/sqrt(21845)
// is applied to the warp's fp32 partial.
//
// Canonical reduction (identical for every row count and every chunk split,
// hence byte-invariant rows): per 512-input chunk each warp chains its MMAs
// over its tk slice in ascending order from zero; warp partials are combined
// by a fixed pairwise tree; chunk partials are added in ascending chunk order.
// Small launches split chunks over CTAs (fp32 partials in the workspace, the
// last-arriving CTA adds them in chunk order); large ones keep all chunks in
// one CTA.  Both perform the same fp32 operations.
#pragma once
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "rotate_block.cuh"

namespace exl3 {
namespace gemm {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 2;
constexpr int kSlotBytes = 3072;           // whole tk rows of 8 tiles (32*K bytes each), K <= 8
constexpr int kActLd = kChunk + 16;        // halves per activation row in smem
constexpr int kZsLd = kHb + 4;             // floats per row of the z tile

// resident CTAs per SM: 8-row items 3 (additive 2), 16-row items 1
__host__ __device__ constexpr int ctas_per_sm(int nrb, bool add) { return nrb == 2 ? 1 : (add ? 2 : 3); }

template <int MODE>
struct ModeTraits {
    static constexpr int nproj = (MODE == kModeGateUp) ? 2 : 1;
    static constexpr int group = (MODE == kModeGateUp) ? 4 : 8;   // warps per projection
    static constexpr int slice_tk = (MODE == kModeGateUp) ? 8 : 4;
};

template <int MODE, int NRB>
struct SmemPlan {
    static constexpr int rows = 8 * NRB;
    static constexpr int act_bytes_raw = ModeTraits<MODE>::nproj * rows * kActLd * 2;
    static constexpr int fold_bytes = 4 * NRB * 32 * 32 * 4;
    static constexpr int act_bytes =
        ((act_bytes_raw > fold_bytes ? act_bytes_raw : fold_bytes) + 127) / 128 * 128;
    static constexpr int bar_off = 0;
    static constexpr int ring_off = 256;
    static constexpr int act_off = ring_off + kWarps * kSlots * kSlotBytes;
    static constexpr int zs_off = act_off + act_bytes;
    static constexpr int zs_bytes = ModeTraits<MODE>::nproj * rows * kZsLd * 4;
    static constexpr int flag_off = zs_off + zs_bytes;
    static constexpr int ws_off = flag_off + 16;
    static constexpr int total = ws_off + kWarps * 128;
};

struct Item {
    int e, row0, nrows, nbk, c_begin, c_end, pair;
};

struct Pass {
    const uint32_t *trellis;
    int K, cb, tk0, tk1;
    float alpha;
};

template <int MODE, int NRB>
__device__ __forceinline__ void load_item(const GemmArgs &a, int item, bool split, Item &it)
{
    const int pair = split ? item / a.nchunks : item;
    const int c = split ? item % a.nchunks : 0;
    it.pair = pair;
    it.c_begin = c;
    it.c_end = split ? c + 1 : a.nchunks;
    const int rgi = pair / a.nb;
    it.nbk = pair % a.nb;
    if (MODE == kModeLinear) {
        it.e = 0;
        it.row0 = rgi * 8 * NRB;
        it.nrows = min(8 * NRB, a.M - it.row0);
    } else {
        const int4 r = static_cast<const int4 *>(a.rg)[rgi];
        it.e = r.x;
        it.row0 = r.y;
        it.nrows = r.z;
    }
}

// The warp's share of (chunk, pass): tk range, trellis, width, codebook.
// Returns false when the warp streams nothing for it.
template <int MODE>
__device__ __forceinline__ bool get_pass(const GemmArgs &a, const Item &it, int chunk, int pass,
                                         int warp, Pass &ps)
{
    using T = ModeTraits<MODE>;
    const int p = (MODE == kModeGateUp) ? (warp >> 2) : (MODE == kModeDown ? 2 : 0);
    const int slice = (MODE == kModeGateUp) ? (warp & 3) : warp;
    const int ntk = a.in_f / 16;
    ps.tk0 = chunk * kChunkTk + slice * T::slice_tk;
    ps.tk1 = min(ps.tk0 + T::slice_tk, ntk);
    if (ps.tk0 >= ps.tk1)
        return false;
    if (pass == 0) {
        if (MODE == kModeLinear) {
            ps.trellis = a.lin.trellis;
            ps.K = a.lin.K;
            ps.cb = a.lin.codebook;
        } else {
            const int i = it.e * 3 + p;
            ps.trellis = reinterpret_cast<const uint32_t *>(a.t_trellis[i]);
            ps.K = a.t_K[i];
            ps.cb = a.t_cb[i];
        }
        ps.alpha = 1.0f;
        return true;
    }
    const int j = ((pass - 1) * a.E + it.e) * 3 + p;
    ps.alpha = a.s_scale[j];
    if (ps.alpha == 0.0f)
        return false;                       // zero scale: no bytes, no MMA
    ps.trellis = reinterpret_cast<const uint32_t *>(a.s_trellis[j]);
    ps.K = a.s_K[j];
    ps.cb = EXL3_CB_MCG;
    return true;
}

// Enumerates, in consumption order, the trellis segments (one tk row of the 8
// tiles of a 128-output block) that one warp streams.
struct Producer {
    // fast path: rows left in the current (item, chunk, pass), next row, stride
    const uint32_t *row;
    int rows_left, rps, row_bytes, stride_words;
    // slow path: position in the enumeration
    int item, chunk, pass, n_items;
    bool split, done;
    Item it;
};

template <int MODE, int NRB, bool ADD>
__device__ __forceinline__ void producer_init(const GemmArgs &a, Producer &P, int n_items,
                                              bool split)
{
    P.n_items = n_items;
    P.split = split;
    P.item = blockIdx.x;
    P.rows_left = 0;
    P.done = P.item >= n_items;
    P.pass = -1;
    if (!P.done) {
        load_item<MODE, NRB>(a, P.item, split, P.it);
        P.chunk = P.it.c_begin;
    }
}

__host__ __device__ constexpr int rows_per_slot(int K) { return kSlotBytes / (256 * K); }

template <int MODE, int NRB, bool ADD>
__device__ __forceinline__ bool producer_next(const GemmArgs &a, Producer &P, int warp,
                                              const uint32_t **src, int *nrows, int *row_bytes,
                                              int *stride)
{
    const int npass = ADD ? a.num_stages : 1;
    while (P.rows_left <= 0) {              // advance to the next pass with rows
        if (P.done)
            return false;
        if (++P.pass < npass) {
            Pass ps;
            if (get_pass<MODE>(a, P.it, P.chunk, P.pass, warp, ps)) {
                P.stride_words = (a.out_f / 16) * 8 * ps.K;
                P.row = ps.trellis + (size_t)ps.tk0 * P.stride_words + (size_t)P.it.nbk * 64 * ps.K;
                P.rows_left = ps.tk1 - ps.tk0;
                P.rps = rows_per_slot(ps.K);
                P.row_bytes = 256 * ps.K;
            }
            continue;
        }
        P.pass = -1;
        if (++P.chunk < P.it.c_end)
            continue;
        P.item += gridDim.x;
        if (P.item >= P.n_items) {
            P.done = true;
            return false;
        }
        load_item<MODE, NRB>(a, P.item, P.split, P.it);
        P.chunk = P.it.c_begin;
    }
    // next slot of the current pass
    const int n = min(P.rps, P.rows_left);
    *src = P.row;
    *nrows = n;
    *row_bytes = P.row_bytes;
    *stride = P.stride_words;
    P.row += (size_t)n * P.stride_words;
    P.rows_left -= n;
    return true;
}

// Per-warp stream state.  The producer cursor lives in shared memory and only
// lane 0 advances it and issues copies; the consumer only counts slots.
struct WarpStream {
    Producer P;
    uint32_t issued;
    int dead;
};

static_assert(sizeof(WarpStream) <= 128, "WarpStream slot");

struct Ring {
    uint64_t *bar;
    uint8_t *buf;
    WarpStream *ws;
    uint32_t head;
    bool dead;
};

template <int MODE, int NRB, bool ADD>
__device__ __forceinline__ void ring_issue(Ring &r, const GemmArgs &a, int warp)
{
    if ((threadIdx.x & 31) != 0)
        return;
    WarpStream *w = r.ws;
    const uint32_t *src;
    int nrows, row_bytes, stride;
    if (w->dead)
        return;
    if (producer_next<MODE, NRB, ADD>(a, w->P, warp, &src, &nrows, &row_bytes, &stride)) {
        // one slot = nrows consecutive tk rows of the 8 tiles of the block,
        // one bulk copy each, all completing on the slot's mbarrier
        const int slot = w->issued % kSlots;
        mbar_arrive_expect_tx(&r.bar[slot], row_bytes * nrows);
        for (int i = 0; i < nrows; i++)
            bulk_g2s(r.buf + slot * kSlotBytes + i * row_bytes, src + (size_t)i * stride,
                     row_bytes, &r.bar[slot]);
        w->issued++;
    }
}

__device__ __forceinline__ const uint32_t *ring_wait(Ring &r, int32_t *hdr)
{
    if (r.dead)
        return nullptr;
    const int slot = r.head % kSlots;
    const uint32_t parity = (r.head / kSlots) & 1u;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&r.bar[slot], parity));
    if (!ok) {
        r.dead = true;
        if ((threadIdx.x & 31) == 0) {
            r.ws->dead = 1;
            set_error(hdr, EXL3_DERR_TIMEOUT);
        }
        return nullptr;
    }
    return reinterpret_cast<const uint32_t *>(r.buf + slot * kSlotBytes);
}

template <int MODE, int NRB, bool ADD>
__device__ __forceinline__ void ring_release(Ring &r, const GemmArgs &a, int warp)
{
    __syncwarp();
    r.head++;
    ring_issue<MODE, NRB, ADD>(r, a, warp);
}

// Before exit: wait (bounded) for copies still in flight into this warp's ring.
__device__ __forceinline__ void ring_drain(Ring &r)
{
    __syncwarp();
    if ((threadIdx.x & 31) != 0)
        return;
    uint32_t h = r.head;
    while (h < r.ws->issued) {
        const int slot = h % kSlots;
        mbar_wait(&r.bar[slot], (h / kSlots) & 1u);
        h++;
    }
}

__device__ __forceinline__ uint32_t hsub_1534(uint32_t v)
{
    __half2 h = *reinterpret_cast<__half2 *>(&v);
    h = __hsub2(h, __half2(__ushort_as_half(0x65FE), __ushort_as_half(0x65FE)));
    return *reinterpret_cast<uint32_t *>(&h);
}

// State i (0..3) of a run whose 64-bit window X0:X1 starts at the run's first
// window bit: bits [iK, iK+16).
template <int K, int I>
__device__ __forceinline__ uint32_t run_state(uint32_t X0, uint32_t X1)
{
    if constexpr (I * K + 16 <= 32)
        return bits16_from_top<I * K>(X0);
    else
        return __funnelshift_l(X1, X0, I * K) >> 16;
}

// codebook constants: x = a*s + b (mod 2^32)
template <int CB>
struct Codebook {
    static constexpr uint32_t a = CB == EXL3_CB_MUL1 ? 0x83DCD12Du
                                : (CB == EXL3_CB_3INST ? 89226354u : 0xCBAC1FEDu);
    static constexpr uint32_t b = CB == EXL3_CB_3INST ? 64248484u : 0u;
};

// Per-lane word offsets and bit shift of the decode of one tile row: thread
// (g, t) decodes, in every 16x16 tile, the two runs of 4 consecutive states
// at positions 16g+4t.. (column g, run A) and 16(g+8)+4t.. (column g+8, run
// B), whose windows start at the same bit offset modulo 32.
template <int K>
struct RowLanes {
    int oA0, oA1, oA2, oB0, oB1, oB2, o;
    __device__ __forceinline__ explicit RowLanes(int lane)
    {
        constexpr int NWD = 8 * K;                            // 32-bit words per tile
        const int g = lane >> 2, t = lane & 3;
        const int start = (16 * g + 4 * t + 1) * K - 16;      // first bit of run A's window
        const int w0 = start >> 5;                            // floor (may be -1)
        o = start & 31;
        oA0 = (w0 + NWD) % NWD;
        oA1 = (w0 + 1 + NWD) % NWD;
        oA2 = (w0 + 2 + NWD) % NWD;
        oB0 = (w0 + 4 * K) % NWD;
        oB1 = (w0 + 4 * K + 1) % NWD;
        oB2 = (w0 + 4 * K + 2) % NWD;
    }
};

// Activation (B) fragments of one tk row for NRB 8-row groups: the 4 inputs
// 16*tk + 4t.. of row g of each group, each fp16 duplicated into both halves
// of a word (mcg/3inst: one MMA k element per weight half) or kept as pairs
// (mul1).
template <int CB, int NRB>
__device__ __forceinline__ void load_bfrag(uint32_t (&bf)[NRB][4], const uint16_t *act, int ld,
                                           int kcol)
{
    const int g = (threadIdx.x & 31) >> 2;
#pragma unroll
    for (int nb = 0; nb < NRB; nb++) {
        const uint2 v = *reinterpret_cast<const uint2 *>(act + (8 * nb + g) * ld + kcol);
        if (CB == EXL3_CB_MUL1) {
            bf[nb][0] = v.x;
            bf[nb][1] = v.y;
        } else {
            bf[nb][0] = prmt(v.x, v.x, 0x1010);
            bf[nb][1] = prmt(v.x, v.x, 0x3232);
            bf[nb][2] = prmt(v.y, v.y, 0x1010);
            bf[nb][3] = prmt(v.y, v.y, 0x3232);
        }
    }
}

// Decode one 16-input row of the 8 tiles of a 128-output block (row = its
// 8 tiles' words in shared memory) and accumulate it into acc with mma.sync.
template <int K, int CB, int NRB>
__device__ __forceinline__ void decode_row(float (&acc)[NRB][8][4], const uint32_t *row,
                                           const uint32_t (&bf)[NRB][4], const RowLanes<K> &rl,
                                           const HashConsts &hc)
{
    constexpr int NWD = 8 * K;
    constexpr bool W3 = 16 + 3 * K > 33;      // a run's window needs a third word (K >= 6)
    constexpr bool MUL1 = CB == EXL3_CB_MUL1;
    constexpr uint32_t mul = Codebook<CB>::a, add = Codebook<CB>::b;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const uint32_t *tw = row + j * NWD;
        const uint32_t a0 = tw[rl.oA0], a1 = tw[rl.oA1];
        const uint32_t b0 = tw[rl.oB0], b1 = tw[rl.oB1];
        const uint32_t XA0 = __funnelshift_l(a1, a0, rl.o), XB0 = __funnelshift_l(b1, b0, rl.o);
        uint32_t XA1 = 0, XB1 = 0;
        if (W3) {
            const uint32_t a2 = tw[rl.oA2], b2 = tw[rl.oB2];
            XA1 = __funnelshift_l(a2, a1, rl.o);
            XB1 = __funnelshift_l(b2, b1, rl.o);
        }
        uint32_t sA[4], sB[4];
        sA[0] = run_state<K, 0>(XA0, XA1);
        sA[1] = run_state<K, 1>(XA0, XA1);
        sA[2] = run_state<K, 2>(XA0, XA1);
        sA[3] = run_state<K, 3>(XA0, XA1);
        sB[0] = run_state<K, 0>(XB0, XB1);
        sB[1] = run_state<K, 1>(XB0, XB1);
        sB[2] = run_state<K, 2>(XB0, XB1);
        sB[3] = run_state<K, 3>(XB0, XB1);
        if (MUL1) {
            uint32_t dA[4], dB[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                dA[i] = __dp4a(sA[i] * mul, 0x01010101u, 0x6400u);
                dB[i] = __dp4a(sB[i] * mul, 0x01010101u, 0x6400u);
            }
            const uint32_t A0 = hsub_1534(prmt(dA[0], dA[1], 0x5410));
            const uint32_t A1 = hsub_1534(prmt(dB[0], dB[1], 0x5410));
            const uint32_t A2 = hsub_1534(prmt(dA[2], dA[3], 0x5410));
            const uint32_t A3 = hsub_1534(prmt(dB[2], dB[3], 0x5410));
#pragma unroll
            for (int nb = 0; nb < NRB; nb++)
                mma_16816(acc[nb][j], A0, A1, A2, A3, bf[nb][0], bf[nb][1]);
        } else {
            uint32_t xA[4], xB[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                xA[i] = and_xor(sA[i] * mul + add, hc.mask, hc.flip);
                xB[i] = and_xor(sB[i] * mul + add, hc.mask, hc.flip);
            }
#pragma unroll
            for (int nb = 0; nb < NRB; nb++) {
                mma_16816(acc[nb][j], xA[0], xB[0], xA[1], xB[1], bf[nb][0], bf[nb][1]);
                mma_16816(acc[nb][j], xA[2], xB[2], xA[3], xB[3], bf[nb][2], bf[nb][3]);
            }
        }
    }
}

// Decode + MMA over the warp's tk slice of one (chunk, pass).
template <int K, int CB, int MODE, int NRB, bool ADD>
__device__ __forceinline__ void run_pass(float (&acc)[NRB][8][4], Ring &ring,
                                         const GemmArgs &a, int warp, const Pass &ps,
                                         int chunk, const uint16_t *act_s)
{
    const int lane = threadIdx.x & 31, t = lane & 3;
    const RowLanes<K> rl(lane);
    constexpr int RPS = rows_per_slot(K);
    const HashConsts hc = hash_consts(a.hdr);
    for (int tk_s = ps.tk0; tk_s < ps.tk1; tk_s += RPS) {
        const int nrows = min(RPS, ps.tk1 - tk_s);
        const uint32_t *seg = ring_wait(ring, a.hdr);
#pragma unroll 1
        for (int rr = 0; rr < nrows && seg != nullptr; rr++) {
            const int tk = tk_s + rr;
            const uint32_t *row = seg + rr * 64 * K;       // 8 tiles of 8K words
            uint32_t bf[NRB][4];
            load_bfrag<CB, NRB>(bf, act_s, kActLd, (tk - chunk * kChunkTk) * 16 + 4 * t);
            decode_row<K, CB, NRB>(acc, row, bf, rl, hc);
        }
        ring_release<MODE, NRB, ADD>(ring, a, warp);
    }
}

template <int MODE, int NRB, bool ADD>
__device__ __forceinline__ void dispatch_pass(float (&acc)[NRB][8][4], Ring &ring,
                                              const GemmArgs &a, int warp, const Pass &ps,
                                              int chunk, const uint16_t *act_s)
{
#define EXL3_K_CASE(KK)                                                                        \
    case KK:                                                                                   \
        if (ps.cb == EXL3_CB_MUL1)                                                             \
            run_pass<KK, EXL3_CB_MUL1, MODE, NRB, ADD>(acc, ring, a, warp, ps, chunk, act_s);  \
        else if (ps.cb == EXL3_CB_3INST)                                                       \
            run_pass<KK, EXL3_CB_3INST, MODE, NRB, ADD>(acc, ring, a, warp, ps, chunk, act_s); \
        else                                                                                   \
            run_pass<KK, EXL3_CB_MCG, MODE, NRB, ADD>(acc, ring, a, warp, ps, chunk, act_s);   \
        break;
    switch (ps.K) {
        EXL3_K_CASE(1)
        EXL3_K_CASE(2)
        EXL3_K_CASE(3)
        EXL3_K_CASE(4)
        EXL3_K_CASE(5)
        EXL3_K_CASE(6)
        EXL3_K_CASE(7)
        EXL3_K_CASE(8)
        default:
            break;
    }
#undef EXL3_K_CASE
}

constexpr int kPartStride = kRowGroup * kHb;   // floats per (pair, chunk, projection) partial

// Element e of the fragment-ordered partials [nproj][nb][j][r][lane] -> its
// index in zs[nproj][ROWS][kZsLd] (row = route, column = output in the block).
template <int ROWS>
__device__ __forceinline__ int zs_index(int e, int frag)
{
    const int p = e / (frag * 32);
    const int i = e % (frag * 32);
    const int lane = i & 31, q = i >> 5;
    const int r = q & 3, j = (q >> 2) & 7, nb = q >> 5;
    const int row = 8 * nb + 2 * (lane & 3) + (r & 1);
    const int col = 16 * j + (lane >> 2) + 8 * (r >> 1);
    return (p * ROWS + row) * kZsLd + col;
}

template <int MODE, int NRB, bool ADD>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(NRB, ADD)) k_expert_gemm(GemmArgs a)
{
    using T = ModeTraits<MODE>;
    using S = SmemPlan<MODE, NRB>;
    constexpr int ROWS = 8 * NRB;
    constexpr int FRAG = NRB * 32;           // accumulator floats per lane
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::bar_off);
    uint8_t *ring_base = smem + S::ring_off;
    uint16_t *act_s = reinterpret_cast<uint16_t *>(smem + S::act_off);
    float *fold = reinterpret_cast<float *>(smem + S::act_off);   // aliases act_s
    float *zs = reinterpret_cast<float *>(smem + S::zs_off);
    int *s_flag = reinterpret_cast<int *>(smem + S::flag_off);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // Programmatic dependent launch (decode-regime layers): gate/up and linear
    // wait for their predecessor at once and let the next kernel launch; down
    // first reads the plan (written by the route-pack kernel, complete before
    // gate/up passed its wait) and starts streaming its trellis words, then
    // waits for gate/up before touching its outputs.  Every CTA waits before
    // it exits, so each kernel completes after its predecessor.
    if (MODE != kModeDown) {
        grid_dep_wait();
        grid_dep_launch();
    }
    int n_items;
    bool split;
    if (MODE == kModeLinear) {
        n_items = a.n_items_host;
        split = a.split_host != 0;
    } else {
        if (a.hdr[kHdrRegime] != 0) {
            grid_dep_wait();
            return;                          // the prefill-regime kernels run this layer
        }
        n_items = a.hdr[MODE == kModeGateUp ? kHdrNItems1 : kHdrNItems2];
        split = a.hdr[MODE == kModeGateUp ? kHdrSplit1 : kHdrSplit2] != 0;
    }
    const bool work = (int)blockIdx.x < n_items;
    if (MODE != kModeDown && !work)
        return;

    Ring ring;
    ring.bar = bars + warp * kSlots;
    ring.buf = ring_base + warp * kSlots * kSlotBytes;   // shared memory
    ring.ws = reinterpret_cast<WarpStream *>(smem + S::ws_off) + warp;
    ring.head = 0;
    ring.dead = false;
    if (work) {
        if (lane == 0) {
            for (int s = 0; s < kSlots; s++)
                mbar_init(&ring.bar[s], 1);
            fence_mbar_init();
            producer_init<MODE, NRB, ADD>(a, ring.ws->P, n_items, split);
            ring.ws->issued = 0;
            ring.ws->dead = 0;
        }
        __syncwarp();
        for (int s = 0; s < kSlots; s++)
            ring_issue<MODE, NRB, ADD>(ring, a, warp);
    }
    if (MODE == kModeDown) {
        grid_dep_wait();
        if (a.hdr[kHdrError] != 0) {
            // device-detected contract violation: zero-filled output (every
            // CTA of the grid takes part)
            const size_t n = (size_t)a.M_tokens * a.out_f;
            for (size_t i = (size_t)blockIdx.x * kThreads + tid; i < n;
                 i += (size_t)gridDim.x * kThreads)
                reinterpret_cast<uint16_t *>(a.out)[i] = 0;
            if (work)
                ring_drain(ring);
            return;
        }
        if (!work)
            return;
    }

    const int npass = ADD ? a.num_stages : 1;
    const int my_proj = (MODE == kModeGateUp) ? (warp >> 2) : 0;
    const bool root = (warp % T::group) == 0;

    // fused input rotation: units per chunk = nproj x ROWS x 4 blocks, 8 per
    // warp per pass; each lane's (projection, row) is fixed within an item,
    // so its token and suh pointer are looked up once per item
    constexpr int kRotUnits = T::nproj * ROWS * (kChunk / kHb);
    constexpr int kRotPasses = MODE == kModeGateUp ? kRotUnits / (kWarps * 8) : 1;
    static_assert(MODE != kModeGateUp || kRotPasses * kWarps * 8 == kRotUnits, "rotation units");
    int rot_tok[kRotPasses];
    const uint16_t *rot_suh[kRotPasses];

    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        Item it;
        load_item<MODE, NRB>(a, item, split, it);
        if (MODE == kModeGateUp && a.fuse_rot) {
#pragma unroll
            for (int q = 0; q < kRotPasses; q++) {
                const int u = (q * kWarps + warp) * 8 + (lane >> 2);
                const int r = (u / (kChunk / kHb)) % ROWS;
                const int p = u / (ROWS * (kChunk / kHb));
                rot_tok[q] = r < it.nrows ? a.packed[it.row0 + r] / a.topk : -1;
                rot_suh[q] = reinterpret_cast<const uint16_t *>(a.t_suh[it.e * 3 + p]);
            }
        }

        for (int chunk = it.c_begin; chunk < it.c_end; chunk++) {
            // ---- activations of this chunk: [nproj][ROWS][512] fp16
            named_barrier(1, kThreads);
            if (MODE == kModeGateUp && a.fuse_rot) {
                // rotate x rows here: unit = (projection, row, 128-block of
                // the chunk), four lanes per unit, the same arithmetic as the
                // rotate kernel (identical fp16 bits)
                const int c = lane & 3;
#pragma unroll
                for (int q = 0; q < kRotPasses; q++) {
                    const int u = (q * kWarps + warp) * 8 + (lane >> 2);
                    const int b = u % (kChunk / kHb);
                    const int r = (u / (kChunk / kHb)) % ROWS;
                    const int p = u / (ROWS * (kChunk / kHb));
                    const int col = chunk * kChunk + b * kHb;
                    const bool valid = rot_tok[q] >= 0 && col < a.in_f;
                    float v[kRotFeat], sv[kRotFeat];
                    if (valid) {
                        const int tok = rot_tok[q];
                        const uint16_t *suh = rot_suh[q];
                        load_act32(a.x, (size_t)tok * a.in_f + col + kRotFeat * c, a.act_dtype, v);
                        load_half32(suh, col + kRotFeat * c, sv);
#pragma unroll
                        for (int i = 0; i < kRotFeat; i++)
                            v[i] *= sv[i];
                    } else {
#pragma unroll
                        for (int i = 0; i < kRotFeat; i++)
                            v[i] = 0.0f;
                    }
                    uint4 o[4];
                    rotate_block32(v, c, o);
                    uint4 *dst = reinterpret_cast<uint4 *>(act_s + (p * ROWS + r) * kActLd + b * kHb + kRotFeat * c);
#pragma unroll
                    for (int k = 0; k < 4; k++)
                        dst[k] = o[k];
                }
            } else {
                const int c0 = chunk * kChunk;
                const int nvec = T::nproj * ROWS * (kChunk / 8);
                for (int v = tid; v < nvec; v += kThreads) {
                    const int col = (v % (kChunk / 8)) * 8;
                    const int r = (v / (kChunk / 8)) % ROWS;
                    const int p = v / (ROWS * (kChunk / 8));
                    uint4 val = make_uint4(0, 0, 0, 0);
                    if (r < it.nrows && c0 + col < a.in_f) {
                        const uint16_t *src = a.act + (size_t)(it.row0 + r) * a.act_row_stride +
                                              (size_t)p * a.in_f + c0 + col;
                        val = __ldg(reinterpret_cast<const uint4 *>(src));
                    }
                    *reinterpret_cast<uint4 *>(act_s + (p * ROWS + r) * kActLd + col) = val;
                }
            }
            named_barrier(1, kThreads);

            // ---- this warp's partial over its slice, base + residual stages
            float acc[NRB][8][4];
#pragma unroll
            for (int nb = 0; nb < NRB; nb++)
#pragma unroll
                for (int j = 0; j < 8; j++)
#pragma unroll
                    for (int r = 0; r < 4; r++)
                        acc[nb][j][r] = 0.0f;
            const uint16_t *act_p = act_s + my_proj * ROWS * kActLd;
            for (int pass = 0; pass < npass; pass++) {
                Pass ps;
                if (!get_pass<MODE>(a, it, chunk, pass, warp, ps))
                    continue;
                if (!ADD) {
                    dispatch_pass<MODE, NRB, ADD>(acc, ring, a, warp, ps, chunk, act_p);
                    if (ps.cb == EXL3_CB_MUL1) {
#pragma unroll
                        for (int nb = 0; nb < NRB; nb++)
#pragma unroll
                            for (int j = 0; j < 8; j++)
#pragma unroll
                                for (int r = 0; r < 4; r++)
                                    acc[nb][j][r] *= kInvSqrtMul1;
                    }
                } else {
                    float tmp[NRB][8][4];
#pragma unroll
                    for (int nb = 0; nb < NRB; nb++)
#pragma unroll
                        for (int j = 0; j < 8; j++)
#pragma unroll
                            for (int r = 0; r < 4; r++)
                                tmp[nb][j][r] = 0.0f;
                    dispatch_pass<MODE, NRB, ADD>(tmp, ring, a, warp, ps, chunk, act_p);
                    const float f = (ps.cb == EXL3_CB_MUL1) ? kInvSqrtMul1 : 1.0f;
#pragma unroll
                    for (int nb = 0; nb < NRB; nb++)
#pragma unroll
                        for (int j = 0; j < 8; j++)
#pragma unroll
                            for (int r = 0; r < 4; r++) {
                                if (pass == 0)
                                    acc[nb][j][r] = (f == 1.0f) ? tmp[nb][j][r] : tmp[nb][j][r] * f;
                                else
                                    acc[nb][j][r] = __fmaf_rn(ps.alpha, tmp[nb][j][r], acc[nb][j][r]);
                            }
                }
            }

            // ---- fixed pairwise tree over the warps of each projection
#pragma unroll
            for (int s = 1; s < T::group; s <<= 1) {
                named_barrier(1, kThreads);
                const int wl = warp % T::group;
                if (wl % (2 * s) == s) {
                    float *slot = fold + ((warp - s) / (2 * s)) * FRAG * 32;
#pragma unroll
                    for (int nb = 0; nb < NRB; nb++)
#pragma unroll
                        for (int j = 0; j < 8; j++)
#pragma unroll
                            for (int r = 0; r < 4; r++)
                                slot[((nb * 8 + j) * 4 + r) * 32 + lane] = acc[nb][j][r];
                }
                named_barrier(1, kThreads);
                if (wl % (2 * s) == 0) {
                    const float *slot = fold + (warp / (2 * s)) * FRAG * 32;
#pragma unroll
                    for (int nb = 0; nb < NRB; nb++)
#pragma unroll
                        for (int j = 0; j < 8; j++)
#pragma unroll
                            for (int r = 0; r < 4; r++)
                                acc[nb][j][r] = acc[nb][j][r] + slot[((nb * 8 + j) * 4 + r) * 32 + lane];
                }
            }

            // ---- chunk partial of each projection: root warp -> shared memory
            //      (fragment order), then elementwise: running sum in zs, or
            //      out to the workspace when chunks are split over CTAs
            named_barrier(1, kThreads);
            if (root) {
                float *pb = fold + my_proj * FRAG * 32;
#pragma unroll
                for (int nb = 0; nb < NRB; nb++)
#pragma unroll
                    for (int j = 0; j < 8; j++)
#pragma unroll
                        for (int r = 0; r < 4; r++)
                            pb[((nb * 8 + j) * 4 + r) * 32 + lane] = acc[nb][j][r];
            }
            named_barrier(1, kThreads);
            if (split) {
                float *dst = a.part + (size_t)(it.pair * a.nchunks + chunk) * T::nproj * kPartStride;
                for (int e = tid; e < T::nproj * FRAG * 32; e += kThreads)
                    dst[(e / (FRAG * 32)) * kPartStride + e % (FRAG * 32)] = fold[e];
            } else {
                const bool first = chunk == it.c_begin;
                for (int e = tid; e < T::nproj * FRAG * 32; e += kThreads) {
                    float &zz = zs[zs_index<ROWS>(e, FRAG)];
                    zz = first ? fold[e] : zz + fold[e];
                }
            }
        }

        if (split) {
            // last CTA of this (row group, block) adds the chunk partials in order
            __threadfence();
            named_barrier(1, kThreads);
            if (tid == 0) {
                const int old = atomicAdd(&a.cnt_split[it.pair], 1);
                *s_flag = (old == a.nchunks - 1);
            }
            named_barrier(1, kThreads);
            if (*s_flag == 0)
                continue;
            __threadfence();
            const float *src = a.part + (size_t)it.pair * a.nchunks * T::nproj * kPartStride;
            constexpr int PER = T::nproj * FRAG * 32 / kThreads;   // elements per thread
            float run[PER];
#pragma unroll 2
            for (int c = 0; c < a.nchunks; c++) {
                const float *sc = src + (size_t)c * T::nproj * kPartStride;
                float v[PER];
#pragma unroll
                for (int k = 0; k < PER; k++) {
                    const int e = tid + k * kThreads;
                    v[k] = __ldcg(sc + (e / (FRAG * 32)) * kPartStride + e % (FRAG * 32));
                }
#pragma unroll
                for (int k = 0; k < PER; k++)
                    run[k] = (c == 0) ? v[k] : run[k] + v[k];
            }
#pragma unroll
            for (int k = 0; k < PER; k++)
                zs[zs_index<ROWS>(tid + k * kThreads, FRAG)] = run[k];
            if (tid == 0)
                a.cnt_split[it.pair] = 0;
        }
        named_barrier(1, kThreads);

        // ---- epilogue: one warp per row, lane l owns outputs 4l..4l+3 of the block
        for (int r = warp; r < it.nrows; r += kWarps) {
            if (MODE == kModeGateUp) {
                float gv[4], uv[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    gv[i] = zs[r * kZsLd + 4 * lane + i];
                    uv[i] = zs[(ROWS + r) * kZsLd + 4 * lane + i];
                }
                epi_gateup_row(a, it.e, it.nbk, it.row0 + r, gv, uv);
            } else {
                float z[4];
#pragma unroll
                for (int i = 0; i < 4; i++)
                    z[i] = zs[r * kZsLd + 4 * lane + i];
                if (MODE == kModeLinear)
                    epi_linear_row(a, it.nbk, it.row0 + r, z);
                else
                    epi_down_row(a, it.e, it.nbk, it.row0 + r, z);
            }
        }
        named_barrier(1, kThreads);
    }
    ring_drain(ring);
}

template <int MODE, int NRB, bool ADD>
cudaError_t launch_one(const GemmArgs &a, int grid, cudaStream_t s)
{
    if (!a.pdl) {
        k_expert_gemm<MODE, NRB, ADD><<<grid, kThreads, SmemPlan<MODE, NRB>::total, s>>>(a);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SmemPlan<MODE, NRB>::total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_expert_gemm<MODE, NRB, ADD>, a);
}

template <int MODE, int NRB, bool ADD>
cudaError_t set_attr_one()
{
    cudaError_t e = cudaFuncSetAttribute(k_expert_gemm<MODE, NRB, ADD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SmemPlan<MODE, NRB>::total);
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(k_expert_gemm<MODE, NRB, ADD>,
                                cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

}  // namespace gemm
}  // namespace exl3
