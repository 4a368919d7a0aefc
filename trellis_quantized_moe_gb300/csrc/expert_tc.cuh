// Prefill-regime grouped GEMM on the 5th-generation tensor cores (tcgen05 +
// TMEM), for the gate/up and down projections of the fused EXL3 MoE layer and
// for the prompt-sized linear.
//
// Follows "EXL3 linear and grouped routed experts" (TensorFold #837), "What this
// changes" (trellis decode, grouped experts, gate and up, SwiGLU, down, the
// weighted combine, a width per expert).  The pages' kernels decode into
// mma.m16n8k16 fragments; on sm_103a the decoded tile goes to shared memory
// and one thread drives tcgen05.mma, so the integer decode, the tensor work
// and the epilogue of the previous item run concurrently.
//
// Work item = (up to 256 routes of one expert, 128-output block, one
// projection): gate and up are separate items.  An item's accumulator takes
// 256 TMEM columns (128 lanes = outputs x routes), so two items' accumulators
// fit: while the epilogue warps drain one, the MMAs of the next fill the
// other.  One persistent CTA per SM.  A stage covers 128 inputs: every
// barrier wait, tcgen05.commit and activation copy then serves 8 MMAs (the
// single issuing thread's own instruction latencies, not the tensor pipe,
// bound 64-input stages).  Roles:
//   warp 0      streams trellis rows with cp.async.bulk (lane t: row t) into a 24 KB
//               ring of word slots (4 rows each, two per stage) sized by the
//               layer's largest K, mbarrier complete_tx, running into the
//               next item as slots free up;
//   warp 1      owns TMEM (2 x 256 columns); lane 0 issues tcgen05.mma
//               (M=128, N=routes rounded up to 16, K=16) per stage into the
//               item's buffer, tcgen05.commit to release the stage's
//               operands, and at the item's end to hand the buffer over;
//   warps 2-17  decode: each thread turns two 16-state trellis column runs
//               (inputs 16t.. and 64+16t.. of one output) into 16 fp16
//               weights each (the two halves of the mcg/3inst word summed in
//               fp16, mul1 as the exact integer byte sum - 510) and stores
//               them, 16 bytes at a time, into a K-major no-swizzle A tile;
//   warp 18     loads the activation (B) tiles with 2D TMA, two boxes per
//               stage (lanes 0 and 1), into a byte ring that runs as far
//               ahead of the MMAs as it has room;
//   warps 19-26 epilogue: warps 19-22 read the finished buffer (tcgen05.ld,
//               one TMEM lane quarter each), all eight transpose 16 routes at
//               a time through shared
//               memory and run the per-row output rotation: gate/up write
//               Hb(z)*svh*scale in fp32 (the SwiGLU and the down-input
//               rotation follow in k_tc_gu_finish), down writes its rotated
//               rows to the fp32 staging (the weighted combine follows in
//               k_tc_combine), the linear writes its output.
// Linear launches whose 256-row items would take more than one wave use
// items of up to 512 rows instead, split into two halves with one
// accumulator buffer each: every decoded A stage then feeds the MMAs of both
// halves (half the decode work per row) and the items fit in one wave.
// Additive layers: each residual stage with a nonzero scale on the item's
// projection is one more pass of stages that every role walks in the same
// order, accumulating into the same TMEM columns.
// A layout (K-major, no swizzle): element (r, k) of a stage tile sits at
// (r/8)*SBO + (k/8)*128 + (r%8)*16 + (k%8)*2 bytes, SBO = (KS/8)*128.
// B layout (K-major, 128-byte swizzle; two 2D TMA boxes {64 inputs, RB rows}
// per stage, one after the other): route r's 64 inputs of a box are one
// 128-byte row, 8-row groups 1 KB apart; the swizzle permutes the 16-byte
// chunks of row r by r % 8 and is undone by the MMA.
#pragma once
#include <string.h>
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace exl3 {
namespace tc {

constexpr int kNT = 256;          // routes per work item (MMA N upper bound), TMEM columns per buffer
constexpr int kStages = 2;        // decoded-weight (A) stages
constexpr int kTwSlots = 16;      // trellis word slots (at most; sized by the layer's largest K)
constexpr int kBRingBytes = 128 * 1024;   // activation (B) stages, sized per item
constexpr int kMaxBSlots = 16;
constexpr int kTwRingBytes = 24 * 1024;
constexpr int kDecWarps = 16;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kBWarp = 2 + kDecWarps;     // activation producer
constexpr int kEpiWarp0 = kBWarp + 1;     // first of eight epilogue warps
constexpr int kEpiThreads = 256;
constexpr int kThreads = kDecThreads + 96 + kEpiThreads;
constexpr int kEpiRows = 16;      // routes per epilogue interval
constexpr int kZsLd = kHb + 4;
constexpr int kKS = 2 * kTcKs;    // inputs per stage: two 64-input activation boxes
constexpr int kT = kKS / 16;      // trellis rows per stage, in two word slots
constexpr int kTH = kT / 2;       // trellis rows per word slot

struct Smem {
    static constexpr int SBO = (kKS / 8) * 128;
    static constexpr int a_bytes = 128 * kKS * 2;               // one stage's A tile
    static constexpr int tmem_cols = 2 * kNT;                   // two accumulator buffers
    static constexpr int off_a = 0;
    static constexpr int off_b = off_a + kStages * a_bytes;
    static constexpr int off_tw = off_b + kBRingBytes;
    static constexpr int off_zs = off_tw + kTwRingBytes;        // epilogue transpose, 16 routes
    static constexpr int off_rows = off_zs + kEpiRows * kZsLd * 4;   // down: staging row of each item row
    static constexpr int off_bar = off_rows + kNT * 4;
    static constexpr int nbar = 2 * kStages + 2 * kTwSlots + 2 * kMaxBSlots + 4;
    static constexpr int off_misc = off_bar + nbar * 8;
    static constexpr int total = off_misc + 64;
};
static_assert(Smem::total <= 227 * 1024, "prefill kernel shared memory");
static_assert(Smem::off_b % 1024 == 0, "128-byte swizzled B ring alignment");

struct Bars {
    uint64_t *full, *empty, *twfull, *twempty, *bfull, *bempty, *tfull, *tempty;
};

// The activation tensor maps: one per TMA box height RB = 16, 32, ..., 256;
// a launch of two-half linear items has one, act[0], of box {64, lin_rows / 2}.
struct TcMapsDev {
    CUtensorMap act[kTcMaps];
};

// Activation geometry of one work item: RB = the item's routes rounded up to
// a power of two (>= 16); a stage is two TMA boxes of RB rows x 128 bytes.
// (Rounding to a power of two fetches about 5% more rows than rounding to 16
// on a Zipf-routed layer.)
struct BGeom {
    int rb, map, stage_bytes;
};

__device__ __forceinline__ BGeom b_geom(int nrows)
{
    BGeom g;
    g.map = 0;
    while ((16 << g.map) < nrows)
        g.map++;
    g.rb = 16 << g.map;
    g.stage_bytes = g.rb * kKS * 2;
    return g;
}

// Placement of activation stages in the B byte ring: stages of any geometry
// follow each other, each at the first offset after the previous one that
// leaves room for it (else at 0); at most kMaxBSlots are in flight, stage i
// signalling barrier i % kMaxBSlots.  The producer and the MMA thread replay
// the same sequence of sizes, so they agree on every offset without
// exchanging them, and items of different sizes never drain the ring.
struct BRing {
    uint32_t head = 0;      // next free byte
    uint32_t n = 0;         // stages placed
    __device__ __forceinline__ uint32_t place(uint32_t bytes)
    {
        const uint32_t o = head + bytes > (uint32_t)kBRingBytes ? 0u : head;
        head = o + bytes;
        n++;
        return o;
    }
};

// Bounded mbarrier wait shared by every role: gives up after ~2^31 cycles or
// as soon as another thread has given up, and then reports false.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort,
                                         int32_t *hdr)
{
    if (mbar_try_wait_sleep(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try_wait_sleep(bar, parity)) {
        if (*abort)
            return false;
        if (clock64() - t0 > (1ll << 31)) {
            *abort = 1;
            set_error(hdr, EXL3_DERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Warp-uniform forms for the roles whose 32 lanes run together (decode,
// epilogue): every lane waits, and the warp goes on only if all lanes saw the
// phase, so no lane is left behind at a warp-collective after a timeout.
__device__ __forceinline__ bool warp_wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort,
                                              int32_t *hdr)
{
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort, hdr));
}

__device__ __forceinline__ bool warp_aborted(volatile int *abort)
{
    return __any_sync(0xffffffffu, *abort != 0);
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// no-swizzle K-major operand: lbo = bytes between core matrices adjacent in
// k, sbo = bytes between 8-row groups
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;                              // tcgen05 descriptor version
    return d;                                            // no swizzle
}

// swizzled K-major operand (rows of 64 or 128 bytes): sbo = bytes between
// 8-row groups; the k offset inside the row is added to the start address
__device__ __forceinline__ uint64_t smem_desc_swz(uint32_t addr, uint32_t sbo, int row_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;                              // unused for swizzled K-major
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;                              // tcgen05 descriptor version
    d |= (uint64_t)(row_bytes == 128 ? 2 : 4) << 61;     // 128-byte / 64-byte swizzle
    return d;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
          "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t instr_desc(int n)
{
    // f32 accumulate, f16 A and B, both K-major, M = 128, N = n
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t dtmem, uint64_t ad, uint64_t bd, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 ::"r"(dtmem), "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate));
}

// The same with the descriptors given as 32-bit halves: the address fields
// of a stage's eight MMAs differ by small constants, so the issuing thread
// adds to the low words only (fewer instructions in the single-thread loop).
__device__ __forceinline__ void mma_f16_lo(uint32_t dtmem, uint32_t alo, uint32_t ahi, uint32_t blo, uint32_t bhi,
                                           uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n .reg .pred p;\n .reg .b64 ad, bd;\n mov.b64 ad, {%1, %2};\n mov.b64 bd, {%3, %4};\n"
                 " setp.ne.b32 p, %6, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p;\n}\n"
                 ::"r"(dtmem), "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

template <int NREG>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&v)[NREG])
{
    if constexpr (NREG == 16) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                       "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                       "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                     : "r"(taddr));
    } else if constexpr (NREG == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                       "=r"(v[6]), "=r"(v[7])
                     : "r"(taddr));
    } else {
        static_assert(NREG == 4, "tcgen05.ld width");
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                     : "r"(taddr));
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// tcgen05.ld of 16 columns without the wait, and the wait that completes it:
// the wait names the destination registers as in/out operands, so no use of
// them can be scheduled before it.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16_wait(uint32_t (&v)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15])
                 :: "memory");
}

__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b)
{
    __half2 x = *reinterpret_cast<__half2 *>(&a), y = *reinterpret_cast<__half2 *>(&b);
    x = __hadd2(x, y);
    return *reinterpret_cast<uint32_t *>(&x);
}

__device__ __forceinline__ uint32_t hsub1534(uint32_t v)
{
    __half2 h = *reinterpret_cast<__half2 *>(&v);
    h = __hsub2(h, __half2(__ushort_as_half(0x65FE), __ushort_as_half(0x65FE)));
    return *reinterpret_cast<uint32_t *>(&h);
}

// Word offsets (inside a tile) and bit shift of the window holding the 16
// consecutive trellis states of tile column c (inputs 0..15 of one output);
// the window is cyclic, so column 0 starts in the tile's last word.
template <int K>
struct ColumnWindow {
    static constexpr int NWD = 8 * K;
    static constexpr int LEN = 16 + 15 * K;     // window bits of the 16 states
    static constexpr int NX = (LEN + 31) / 32;  // normalised 32-bit words
    int idx[NX + 1];
    int o;
    __device__ __forceinline__ explicit ColumnWindow(int c)
    {
        const int start = (16 * c + 1) * K - 16;
        const int w0 = start >> 5;
        o = start & 31;
#pragma unroll
        for (int j = 0; j <= NX; j++) {
            int v = w0 + j;
            idx[j] = v < 0 ? v + NWD : (v >= NWD ? v - NWD : v);
        }
    }
};

// State i of the window (bits [iK, iK+16) of the normalised words X): one
// FMA-pipe shift and one ALU shift when the state sits in one word.
template <int K, int I>
struct ColumnStates {
    static __device__ __forceinline__ void run(const uint32_t *X, uint32_t *st)
    {
        constexpr int bit = I * K, q = bit >> 5, r = bit & 31;
        if constexpr (r + 16 <= 32)
            st[I] = bits16_from_top<r>(X[q]);
        else
            st[I] = __funnelshift_l(X[q + 1], X[q], r) >> 16;
        ColumnStates<K, I + 1>::run(X, st);
    }
};
template <int K>
struct ColumnStates<K, 16> {
    static __device__ __forceinline__ void run(const uint32_t *, uint32_t *) {}
};

// The 16 states of the window -> 16 fp16 weights in k order (8 half2 words):
// mcg/3inst sum their two fp16 halves in fp16 (one rounding), mul1 gives the
// exact integer byte sum - 510.
// The window of the column's 16 states as normalised words X (bit 0 of state
// 0 at the top of X[0]): the shared-memory reads of a column run.  Once X is
// in registers the word slot may be refilled.
template <int K>
__device__ __forceinline__ void column_bits(const uint32_t *tile, const ColumnWindow<K> &cw,
                                            uint32_t (&X)[ColumnWindow<K>::NX + 1])
{
    constexpr int NX = ColumnWindow<K>::NX;
    uint32_t W[NX + 1];
#pragma unroll
    for (int j = 0; j <= NX; j++)
        W[j] = tile[cw.idx[j]];
#pragma unroll
    for (int j = 0; j < NX; j++)
        X[j] = __funnelshift_l(W[j + 1], W[j], cw.o);
    X[NX] = 0;
}

template <int K, int CB>
__device__ __forceinline__ void decode_bits(const uint32_t (&X)[ColumnWindow<K>::NX + 1], const HashConsts &hc,
                                            uint32_t w[8])
{
    constexpr uint32_t A = CB == EXL3_CB_MUL1 ? 0x83DCD12Du : (CB == EXL3_CB_3INST ? 89226354u : 0xCBAC1FEDu);
    constexpr uint32_t B = CB == EXL3_CB_3INST ? 64248484u : 0u;
    uint32_t x[16];
    uint32_t st[16];
    ColumnStates<K, 0>::run(X, st);
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const uint32_t s = st[i];
        if (CB == EXL3_CB_MUL1)
            x[i] = __dp4a(s * A, 0x01010101u, 0x6400u);
        else
            x[i] = and_xor(s * A + B, hc.mask, hc.flip);
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
        if (CB == EXL3_CB_MUL1)
            w[i] = hsub1534(prmt(x[2 * i], x[2 * i + 1], 0x5410));
        else
            w[i] = hadd2_u32(prmt(x[2 * i], x[2 * i + 1], 0x5410), prmt(x[2 * i], x[2 * i + 1], 0x7632));
    }
}

__device__ __forceinline__ void warp_arrive(uint64_t *bar)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        mbar_arrive(bar);
}

// Position in a ring of N slots: the slot and the parity of its current use
// (flips whenever the slot index wraps).  A consumer waits for parity `phase`
// on a slot's full barrier; a producer waits for `phase ^ 1` on its empty
// barrier, which a freshly initialised barrier already satisfies.
template <int N>
struct RingPos {
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ void next()
    {
        if (++slot == N) {
            slot = 0;
            phase ^= 1;
        }
    }
};

// The same for a ring whose slot count is known at run time.
struct RingPosN {
    uint32_t slot = 0, phase = 0, n = 1;
    __device__ __forceinline__ void next()
    {
        if (++slot == n) {
            slot = 0;
            phase ^= 1;
        }
    }
};

// Trellis ring geometry: one slot holds a stage's nproj * T trellis rows
// (4 rows in both modes), each 256 * kmax bytes.
struct TwGeom {
    int row_bytes, slot_bytes, nslots;
};

__device__ __forceinline__ TwGeom tw_geom(int kmax)
{
    TwGeom g;
    g.row_bytes = 256 * kmax;
    g.slot_bytes = 4 * g.row_bytes;
    g.nslots = min(kTwSlots, kTwRingBytes / g.slot_bytes);
    return g;
}

struct TcItem {
    int e, row0, nrows, nbk, p;   // p: gate (0) or up (1) of a gate/up item
};

// Item -> (row group, block, projection).  Fused layer: row groups of <= 256
// routes from the route-pack plan (one expert's packed routes), gate and up
// of one (row group, block) adjacent; linear: 256 token rows.
template <int MODE>
__device__ __forceinline__ TcItem tc_item(const GemmArgs &a, int item)
{
    TcItem it;
    it.p = 0;
    if (MODE == kModeGateUp) {
        it.p = item & 1;
        item >>= 1;
    }
    const int rgi = item / a.nb;
    it.nbk = item % a.nb;
    if (MODE == kModeLinear) {
        it.e = 0;
        it.row0 = rgi * a.lin_rows;
        it.nrows = min(a.lin_rows, a.M - it.row0);
        return it;
    }
    const int4 r = static_cast<const int4 *>(a.rg)[rgi];
    it.e = r.x;
    it.row0 = r.y;
    it.nrows = r.z;
    return it;
}

template <int MODE>
__device__ __forceinline__ int proj_index(int p) { return MODE == kModeGateUp ? p : 2; }

// The accumulators of one item: one (up to 256 routes or rows), or, for the
// linear's items of more than 256 rows, two halves of lin_rows / 2 rows
// (rows past the item's end leave the second half short or empty).  Half h
// takes the TMEM buffer of the CTA's sub-item count + h.
struct Halves {
    int n, hr;          // halves; rows between their first rows
    int rows[2];
};

template <int MODE>
__device__ __forceinline__ bool tc_two_halves(const GemmArgs &a)
{
    return MODE == kModeLinear && a.lin_rows > kNT;
}

template <int MODE>
__device__ __forceinline__ Halves item_halves(const GemmArgs &a, const TcItem &it)
{
    Halves h;
    if (tc_two_halves<MODE>(a)) {
        h.n = 2;
        h.hr = a.lin_rows / 2;
        h.rows[0] = min(it.nrows, h.hr);
        h.rows[1] = it.nrows - h.rows[0];
    } else {
        h.n = 1;
        h.hr = 0;
        h.rows[0] = it.nrows;
        h.rows[1] = 0;
    }
    return h;
}

// Rows of half 0 of a CTA's last two-half item that the eight epilogue warps
// drain; the sixteen decode warps take the rest of half 0 and all of half 1
// (about 40% and 60% of the rows: sixteen warps drain a 16-row interval in
// about two thirds of the eight epilogue warps' time).  A multiple of 16.
__device__ __forceinline__ int shared_split(const Halves &hv)
{
    return min(hv.rows[0], ((hv.rows[0] + hv.rows[1]) * 2 / 5 + 15) & ~15);
}

// Projection p of expert e: trellis words, width, codebook (linear: its one
// projection).
struct ProjRef {
    const uint32_t *trellis;
    int K, cb;
};

template <int MODE>
__device__ __forceinline__ ProjRef proj_ref(const GemmArgs &a, int e, int p)
{
    ProjRef r;
    if (MODE == kModeLinear) {
        r.trellis = a.lin.trellis;
        r.K = a.lin.K;
        r.cb = a.lin.codebook;
    } else {
        const int i = e * 3 + proj_index<MODE>(p);
        r.trellis = reinterpret_cast<const uint32_t *>(a.t_trellis[i]);
        r.K = a.t_K[i];
        r.cb = a.t_cb[i];
    }
    return r;
}

// Residual stages ("MoE: Add fused additive EXL3 kernels", exllamav3 #284,
// "Summary"): pass 0 of an item is the base weights, pass s = 1..num_stages-1
// residual stage s, included when the item's projection has a nonzero scale
// there.  Every role walks the same passes, stage by stage.
template <int MODE>
__device__ __forceinline__ int tc_num_passes(const GemmArgs &a)
{
    return MODE == kModeLinear ? 1 : a.num_stages;
}

// Scale of projection p in pass s (1 for the base; 0 = stage skipped).
template <int MODE>
__device__ __forceinline__ float pass_alpha(const GemmArgs &a, int e, int p, int s)
{
    if (MODE == kModeLinear || s == 0)
        return 1.0f;
    return a.s_scale[((s - 1) * a.E + e) * 3 + proj_index<MODE>(p)];
}

// Trellis words, width and codebook of projection p in pass s (residuals are
// mcg); only read where the pass's scale is nonzero.
template <int MODE>
__device__ __forceinline__ ProjRef pass_ref(const GemmArgs &a, int e, int p, int s)
{
    if (s == 0)
        return proj_ref<MODE>(a, e, p);
    const int j = ((s - 1) * a.E + e) * 3 + proj_index<MODE>(p);
    ProjRef r;
    r.trellis = reinterpret_cast<const uint32_t *>(a.s_trellis[j]);
    r.K = a.s_K[j];
    r.cb = EXL3_CB_MCG;
    return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, __half2 b)
{
    __half2 x = *reinterpret_cast<__half2 *>(&a);
    x = __hmul2(x, b);
    return *reinterpret_cast<uint32_t *>(&x);
}

// All stages of one pass of a work item for one decode thread: trellis words
// -> decoded A tile (times the pass's scale), one arrival per warp on the
// stage barrier.  K and the codebook are compile-time.  RES: a residual pass.
template <int MODE, int K, int CB, bool RES>
__device__ __forceinline__ bool tc_stages(const GemmArgs &a, uint8_t *smem, const Bars &B,
                                          volatile int *abort, RingPos<kStages> &ra, RingPosN &rt,
                                          const TwGeom &tg, int t, int m, float alpha)
{
    using S = Smem;
    const int nst = a.in_f / kKS;
    const __half2 alpha2 = __float2half2_rn(alpha);
    const ColumnWindow<K> cw(m & 15);
    const HashConsts hc = hash_consts(a.hdr);
    const int tile_off = t * tg.row_bytes + (m >> 4) * 32 * K;          // bytes
    const int a_off = (m >> 3) * S::SBO + (m & 7) * 16 + 2 * t * 128;
    // one stage = two word slots (trellis rows t and t + 4 of this thread)
    for (int s = 0; s < nst; s++) {
        RingPosN rt1 = rt;
        rt1.next();
        if (!warp_wait_bar(&B.twfull[rt.slot], rt.phase, abort, a.hdr) ||
            !warp_wait_bar(&B.twfull[rt1.slot], rt1.phase, abort, a.hdr))
            return false;
        uint32_t X0[ColumnWindow<K>::NX + 1], X1[ColumnWindow<K>::NX + 1];
        column_bits<K>(reinterpret_cast<const uint32_t *>(smem + S::off_tw + rt.slot * tg.slot_bytes + tile_off), cw, X0);
        column_bits<K>(reinterpret_cast<const uint32_t *>(smem + S::off_tw + rt1.slot * tg.slot_bytes + tile_off), cw, X1);
        // the words are in registers (X depends on them): the slots can be refilled
        warp_arrive(&B.twempty[rt.slot]);
        warp_arrive(&B.twempty[rt1.slot]);
        uint32_t w0[8], w1[8];
        decode_bits<K, CB>(X0, hc, w0);
        decode_bits<K, CB>(X1, hc, w1);
        if (RES) {
#pragma unroll
            for (int i = 0; i < 8; i++) {
                w0[i] = hmul2_u32(w0[i], alpha2);
                w1[i] = hmul2_u32(w1[i], alpha2);
            }
        }
        // an A slot is free once the MMAs of its previous stage completed; the
        // decode above does not need it
        if (!warp_wait_bar(&B.empty[ra.slot], ra.phase ^ 1, abort, a.hdr))
            return false;
        uint8_t *abuf = smem + S::off_a + ra.slot * S::a_bytes + a_off;
        *reinterpret_cast<uint4 *>(abuf) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
        *reinterpret_cast<uint4 *>(abuf + 128) = make_uint4(w0[4], w0[5], w0[6], w0[7]);
        *reinterpret_cast<uint4 *>(abuf + 8 * 128) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
        *reinterpret_cast<uint4 *>(abuf + 9 * 128) = make_uint4(w1[4], w1[5], w1[6], w1[7]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        warp_arrive(&B.full[ra.slot]);
        ra.next();
        rt1.next();
        rt = rt1;
    }
    return true;
}

template <int MODE, int K>
__device__ __forceinline__ bool tc_stages_cb(int cb, const GemmArgs &a, uint8_t *smem, const Bars &B,
                                             volatile int *abort, RingPos<kStages> &ra, RingPosN &rt,
                                             const TwGeom &tg, int t, int m)
{
    if (cb == EXL3_CB_MUL1)
        return tc_stages<MODE, K, EXL3_CB_MUL1, false>(a, smem, B, abort, ra, rt, tg, t, m, 1.0f);
    if (cb == EXL3_CB_3INST)
        return tc_stages<MODE, K, EXL3_CB_3INST, false>(a, smem, B, abort, ra, rt, tg, t, m, 1.0f);
    return tc_stages<MODE, K, EXL3_CB_MCG, false>(a, smem, B, abort, ra, rt, tg, t, m, 1.0f);
}

// One decode thread's share of one work item: the base pass, then each
// residual pass of the item's projection.  A mul1 base is scaled by
// 1/sqrt(21845) in the epilogue while the (mcg) residuals are not, so their
// scale carries sqrt(21845) for such a projection.
template <int MODE>
__device__ __forceinline__ bool tc_item_decode(const GemmArgs &a, uint8_t *smem, const Bars &B,
                                               volatile int *abort, const TcItem &it,
                                               RingPos<kStages> &ra, RingPosN &rt, const TwGeom &tg,
                                               int t, int m)
{
    const ProjRef base = proj_ref<MODE>(a, it.e, it.p);
    bool ok;
    switch (base.K) {
        case 1: ok = tc_stages_cb<MODE, 1>(base.cb, a, smem, B, abort, ra, rt, tg, t, m); break;
        case 2: ok = tc_stages_cb<MODE, 2>(base.cb, a, smem, B, abort, ra, rt, tg, t, m); break;
        case 3: ok = tc_stages_cb<MODE, 3>(base.cb, a, smem, B, abort, ra, rt, tg, t, m); break;
        case 4: ok = tc_stages_cb<MODE, 4>(base.cb, a, smem, B, abort, ra, rt, tg, t, m); break;
        case 5: ok = tc_stages_cb<MODE, 5>(base.cb, a, smem, B, abort, ra, rt, tg, t, m); break;
        case 6: ok = tc_stages_cb<MODE, 6>(base.cb, a, smem, B, abort, ra, rt, tg, t, m); break;
        case 7: ok = tc_stages_cb<MODE, 7>(base.cb, a, smem, B, abort, ra, rt, tg, t, m); break;
        default: ok = tc_stages_cb<MODE, 8>(base.cb, a, smem, B, abort, ra, rt, tg, t, m); break;
    }
    if (!ok || warp_aborted(abort))
        return false;
    const int npass = tc_num_passes<MODE>(a);
    for (int s = 1; s < npass; s++) {
        const float al = pass_alpha<MODE>(a, it.e, it.p, s);
        if (al == 0.0f)
            continue;
        const int K = pass_ref<MODE>(a, it.e, it.p, s).K;
        const float alpha = base.cb == EXL3_CB_MUL1 ? al * kSqrtMul1 : al;
#define EXL3_RES_CASE(KK)                                                                            \
    case KK:                                                                                         \
        ok = tc_stages<MODE, KK, EXL3_CB_MCG, true>(a, smem, B, abort, ra, rt, tg, t, m, alpha);     \
        break;
        switch (K) {
            EXL3_RES_CASE(1)
            EXL3_RES_CASE(2)
            EXL3_RES_CASE(3)
            EXL3_RES_CASE(4)
            EXL3_RES_CASE(5)
            EXL3_RES_CASE(6)
            EXL3_RES_CASE(7)
            default:
                ok = tc_stages<MODE, 8, EXL3_CB_MCG, true>(a, smem, B, abort, ra, rt, tg, t, m, alpha);
                break;
        }
#undef EXL3_RES_CASE
        if (!ok || warp_aborted(abort))
            return false;
    }
    return true;
}

// Output rotation of one route row of a gate/up item (lane l owns outputs
// 4l..4l+3 of the block): Hb(z)*svh*scale in fp32, into the staging row of the
// packed route (gate at columns 0..inter, up at inter..2*inter); k_gu_finish
// takes it from there.
__device__ __forceinline__ void epi_gu_half_row(const GemmArgs &a, const DownConsts &c, int p, int nbk, int prow,
                                                float z[4])
{
    const int lane = threadIdx.x & 31;
    warp_hadamard128(z);
#pragma unroll
    for (int i = 0; i < 4; i++)
        z[i] = z[i] * kInvSqrt128 * c.sv[i] * c.sc[i];
    *reinterpret_cast<float4 *>(a.stage + (size_t)prow * (2 * a.out_f) + p * a.out_f + nbk * kHb + 4 * lane) =
        make_float4(z[0], z[1], z[2], z[3]);
}

// A team of NW warps' share of one item: rows [r_begin, it.nrows) of buffer
// `buf` of TMEM -> 16 routes at a time through shared memory -> per-row
// output rotation.  Warps ew 0..3 read TMEM lane quarter q = their warp index
// % 4; each warp runs 16/NW routes of each interval.  The next interval's
// tcgen05.ld is in flight while the current one is processed; down items look
// their staging rows up once per item (a dependent global load per row would
// stall every interval).  The team meets at named barrier `bar`.
template <int MODE, int NW>
__device__ __forceinline__ void tc_item_epilogue(const GemmArgs &a, const TcItem &it, uint32_t tbuf, float *zs,
                                                 int *rowmap, int ew, int q, int r_begin, int bar)
{
    constexpr int kRpw = kEpiRows / NW;         // routes per warp and interval
    static_assert(kRpw * NW == kEpiRows, "epilogue team size");
    const int lane = threadIdx.x & 31;
    DownConsts cd;
    const int pi = proj_index<MODE>(it.p);
    if (MODE == kModeLinear) {
        epi_linear_consts(a, it.nbk, cd);
    } else {
        const int col = it.nbk * kHb + 4 * lane;
        load_half4(reinterpret_cast<const uint16_t *>(a.t_svh[it.e * 3 + pi]), col, cd.sv);
        load_half4(reinterpret_cast<const uint16_t *>(a.t_scale[it.e * 3 + pi]), col, cd.sc);
    }
    if (MODE == kModeDown)
        for (int r = ew * 32 + lane; r < it.nrows; r += NW * 32)
            rowmap[r] = a.packed[it.row0 + r];
    const float fac = (proj_ref<MODE>(a, it.e, it.p).cb == EXL3_CB_MUL1) ? kInvSqrtMul1 : 1.0f;
    const uint32_t taddr = tbuf + ((uint32_t)(32 * q) << 16);
    uint32_t v[16];
    const bool loader = ew < 4;                 // one warp per TMEM lane quarter loads
    if (loader && r_begin < it.nrows)
        tmem_ld16_issue(taddr + r_begin, v);
    for (int r0 = r_begin; r0 < it.nrows; r0 += kEpiRows) {
        if (loader) {
            tmem_ld16_wait(v);
#pragma unroll
            for (int j = 0; j < 16; j++)
                zs[j * kZsLd + 32 * q + lane] = __uint_as_float(v[j]) * fac;
        }
        named_barrier(bar, NW * 32);
        if (loader && r0 + kEpiRows < it.nrows)
            tmem_ld16_issue(taddr + r0 + kEpiRows, v);
#pragma unroll
        for (int h = 0; h < kRpw; h++) {
            const int rr = kRpw * ew + h, r = r0 + rr;
            if (r < it.nrows) {
                float z[4];
#pragma unroll
                for (int i = 0; i < 4; i++)
                    z[i] = zs[rr * kZsLd + 4 * lane + i];
                if (MODE == kModeGateUp) {
                    epi_gu_half_row(a, cd, it.p, it.nbk, it.row0 + r, z);
                } else if (MODE == kModeLinear) {
                    epi_linear_row(a, cd, it.nbk, it.row0 + r, z);
                } else {
                    warp_hadamard128(z);
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        z[i] = z[i] * kInvSqrt128 * cd.sv[i] * cd.sc[i];
                    *reinterpret_cast<float4 *>(a.stage + (size_t)rowmap[r] * a.out_f + it.nbk * kHb + 4 * lane) =
                        make_float4(z[0], z[1], z[2], z[3]);
                }
            }
        }
        named_barrier(bar, NW * 32);
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_expert_tc(GemmArgs a, const __grid_constant__ TcMapsDev maps)
{
    using S = Smem;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Bars B;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::off_bar);
    B.full = bars;
    B.empty = bars + kStages;
    B.twfull = bars + 2 * kStages;
    B.twempty = bars + 2 * kStages + kTwSlots;
    B.bfull = bars + 2 * kStages + 2 * kTwSlots;
    B.bempty = B.bfull + kMaxBSlots;
    B.tfull = B.bempty + kMaxBSlots;           // [2]
    B.tempty = B.tfull + 2;                    // [2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::off_misc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + S::off_misc + 8);
    int *kmax_slot = reinterpret_cast<int *>(smem + S::off_misc + 16);

    if (MODE != kModeLinear && a.hdr[kHdrRegime] != 1)
        return;                              // the decode-regime kernels run this layer
    const int n_items = MODE == kModeLinear ? a.n_items_host
                                            : a.hdr[MODE == kModeGateUp ? kHdrNItems1 : kHdrNItems2];
    if (MODE == kModeDown && a.hdr[kHdrError] != 0)
        return;                              // k_tc_combine writes zeros
    if ((int)blockIdx.x >= n_items)
        return;
    const int nst = a.in_f / kKS;                   // stages per item
    const int ntn = a.out_f / 16;

    if (tid == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&B.full[s], kDecWarps);
            mbar_init(&B.empty[s], 1);
        }
        for (int s = 0; s < kTwSlots; s++) {
            mbar_init(&B.twfull[s], 1);
            mbar_init(&B.twempty[s], kDecWarps);
        }
        for (int s = 0; s < kMaxBSlots; s++) {
            mbar_init(&B.bfull[s], 1);
            mbar_init(&B.bempty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&B.tfull[b], 1);
            mbar_init(&B.tempty[b], kEpiThreads / 32);
        }
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        // the largest K of this kernel's projections sizes the trellis slots
        int km = 1;
        if (MODE == kModeLinear)
            km = max(1, min(8, a.lin.K));
        else
            for (int e = lane; e < a.E; e += 32)
                for (int p = 0; p < (MODE == kModeGateUp ? 2 : 1); p++) {
                    km = max(km, min(8, a.t_K[e * 3 + proj_index<MODE>(p)]));
                    for (int st = 1; st < tc_num_passes<MODE>(a); st++)
                        if (pass_alpha<MODE>(a, e, p, st) != 0.0f)
                            km = max(km, min(8, a.s_K[((st - 1) * a.E + e) * 3 + proj_index<MODE>(p)]));
                }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            km = max(km, __shfl_xor_sync(0xffffffffu, km, o));
        if (lane == 0)
            *kmax_slot = km;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_addr(tmem_slot)), "r"(S::tmem_cols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    const TwGeom tg = tw_geom(*kmax_slot);

    if (warp == 0) {
        // ---------------- producer: trellis rows -> word slots (the whole warp
        // runs the loop; lanes 0..3 each issue one row's bulk copy, so a slot
        // costs one copy instruction issue)
        RingPosN rt;
        rt.n = tg.nslots;
        const int npass = tc_num_passes<MODE>(a);
        bool ok = true;
        for (int item = blockIdx.x; ok && item < n_items && !warp_aborted(abort); item += gridDim.x) {
            const TcItem it = tc_item<MODE>(a, item);
            for (int ps = 0; ok && ps < npass; ps++) {
                if (pass_alpha<MODE>(a, it.e, it.p, ps) == 0.0f)
                    continue;
                const ProjRef pr = pass_ref<MODE>(a, it.e, it.p, ps);
                const uint32_t *tr0 = pr.trellis + (size_t)it.nbk * 8 * (8 * pr.K);
                const uint32_t bytes = kTH * 256 * pr.K;
                for (int h = 0; h < 2 * nst; h++, rt.next()) {      // word slots: rows kTH*h ..
                    const int slot = rt.slot;
                    if (!(ok = warp_wait_bar(&B.twempty[slot], rt.phase ^ 1, abort, a.hdr)))
                        break;
                    uint8_t *dst = smem + S::off_tw + slot * tg.slot_bytes;
                    if (lane == 0)
                        mbar_arrive_expect_tx(&B.twfull[slot], bytes);
                    __syncwarp();
                    if (lane < kTH)
                        bulk_g2s(dst + lane * tg.row_bytes, tr0 + (size_t)(h * kTH + lane) * ntn * (8 * pr.K),
                                 256 * pr.K, &B.twfull[slot]);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            RingPos<kStages> ra;
            uint32_t nit = 0, bphase = 0;            // bphase: parity bit per B stage barrier
            BRing br;
            // descriptors of A slot 0 / B ring byte 0; offsets are added in
            // 16-byte units to the address field
            const uint64_t adesc0 = smem_desc(smem_addr(smem + S::off_a), 128, S::SBO);
            const uint64_t bdesc0 = smem_desc_swz(smem_addr(smem + S::off_b), 1024, 128);
            const uint32_t adlo = (uint32_t)adesc0, adhi = (uint32_t)(adesc0 >> 32);
            const uint32_t bdlo = (uint32_t)bdesc0, bdhi = (uint32_t)(bdesc0 >> 32);
            for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
                const TcItem it = tc_item<MODE>(a, item);
                const Halves hv = item_halves<MODE>(a, it);
                const BGeom bg = b_geom(it.nrows);
                const uint32_t bsub16 = (uint32_t)(bg.rb * 128) >> 4;   // second box of a stage
                // the epilogue has drained the buffers' previous items
                uint32_t dt[2], idesc[2];
                bool ok = true;
                for (int h = 0; h < hv.n; h++) {
                    const uint32_t sub = nit + h, buf = sub & 1, use = sub >> 1;
                    if (use > 0 && !(ok = wait_bar(&B.tempty[buf], (use - 1) & 1, abort, a.hdr)))
                        break;
                    dt[h] = tmem + buf * kNT;
                    idesc[h] = instr_desc(max(16, (hv.rows[h] + 15) & ~15));
                }
                if (!ok)
                    break;
                fence_after();
                // pass 0 (base) opens the accumulator; residual passes add to it
                bool first = true;
                for (int ps = 0; ps < tc_num_passes<MODE>(a) && !*abort; ps++) {
                    if (pass_alpha<MODE>(a, it.e, it.p, ps) == 0.0f)
                        continue;
                    for (int s = 0; s < nst; s++, ra.next()) {
                        const int slot = ra.slot;
                        if (!wait_bar(&B.full[slot], ra.phase, abort, a.hdr))
                            break;
                        // address fields stay below 2^14 (shared memory < 256 KB): 32-bit adds
                        const uint32_t alo = adlo + (uint32_t)(slot * (S::a_bytes >> 4));
                        if (hv.n == 1) {
                            const int bs = (int)(br.n % kMaxBSlots);
                            const uint32_t boff = br.place((uint32_t)bg.stage_bytes);
                            if (!wait_bar(&B.bfull[bs], (bphase >> bs) & 1, abort, a.hdr))
                                break;
                            bphase ^= 1u << bs;
                            fence_after();
                            const uint32_t blo = bdlo + (boff >> 4);
                            const uint32_t blo2 = blo + bsub16;
                            mma_f16_lo(dt[0], alo, adhi, blo, bdhi, idesc[0], first ? 0u : 1u);
#pragma unroll
                            for (int ks = 1; ks < kKS / 16; ks++)
                                mma_f16_lo(dt[0], alo + (uint32_t)(ks * 16), adhi,
                                           (ks >= kKS / 32 ? blo2 : blo) + (uint32_t)((ks % (kKS / 32)) * 2), bdhi,
                                           idesc[0], 1u);
                            // the A slot first: the decode warps wait for it
                            mma_commit(&B.empty[slot]);
                            mma_commit(&B.bempty[bs]);
                        } else {
                            // two entries per stage (inputs 0..63, 64..127), each
                            // the two halves' boxes; every A sub-tile feeds both
                            const uint32_t ebytes = (uint32_t)hv.hr * 256u;
                            bool bok = true;
                            for (int e = 0; e < 2; e++) {
                                const int bs = (int)(br.n % kMaxBSlots);
                                const uint32_t boff = br.place(ebytes);
                                if (!(bok = wait_bar(&B.bfull[bs], (bphase >> bs) & 1, abort, a.hdr)))
                                    break;
                                bphase ^= 1u << bs;
                                fence_after();
                                for (int h = 0; h < 2; h++) {
                                    if (hv.rows[h] == 0)
                                        continue;
                                    const uint32_t blo = bdlo + ((boff + (uint32_t)(h * hv.hr * 128)) >> 4);
#pragma unroll
                                    for (int j = 0; j < kKS / 32; j++) {
                                        const int ks = e * (kKS / 32) + j;
                                        mma_f16_lo(dt[h], alo + (uint32_t)(ks * 16), adhi, blo + (uint32_t)(j * 2),
                                                   bdhi, idesc[h], (first && ks == 0) ? 0u : 1u);
                                    }
                                }
                                if (e == 1)
                                    mma_commit(&B.empty[slot]);
                                mma_commit(&B.bempty[bs]);
                            }
                            if (!bok)
                                break;
                        }
                        first = false;
                    }
                }
                for (int h = 0; h < hv.n; h++)
                    mma_commit(&B.tfull[(nit + h) & 1]);
                nit += hv.n;
            }
        }
    } else if (warp == kBWarp) {
        // ---------------- activation producer: 2D TMA boxes into the B ring
        // (the whole warp runs the loop; lanes 0 and 1 issue a stage's boxes;
        // lane j < kMaxBSlots tracks the bytes of in-flight stage barrier j)
        {
            uint32_t ph = 0;                          // bempty parity bit per stage barrier
            uint32_t my_off = 0, my_end = 0;          // lane j: bytes of the stage on barrier j
            bool my_busy = false;
            uint32_t tail = 0;                        // oldest stage in flight
            BRing br;
            bool ok = true;
            // the linear, launched during the rotate kernel's tail
            // (programmatic dependent launch): the trellis stream, the decode
            // and TMEM setup need nothing from it, the activations do.  Only
            // the linear's kernel contains the wait (with the dependent-launch
            // instructions in every instantiation, here and in the rotate
            // kernels, the additive layer ran 2.5% slower although its kernels
            // never execute them).
            if constexpr (MODE == kModeLinear) {
                if (a.tc_pdl)
                    grid_dep_wait();
            }
            for (int item = blockIdx.x; ok && item < n_items && !warp_aborted(abort); item += gridDim.x) {
                const TcItem it = tc_item<MODE>(a, item);
                const Halves hv = item_halves<MODE>(a, it);
                const BGeom bg = b_geom(it.nrows);
                // one entry per stage (its two 64-input boxes), or for a two-half
                // item two entries per stage (per 64 inputs, both halves' boxes)
                const CUtensorMap *map = &maps.act[hv.n == 1 ? bg.map : 0];
                const int nent = hv.n == 1 ? 1 : 2;
                const uint32_t ebytes = hv.n == 1 ? (uint32_t)bg.stage_bytes : (uint32_t)hv.hr * 256u;
                const int x0 = (MODE == kModeGateUp) ? it.p * a.in_f : 0;
                // the same activation tiles again for every residual pass
                for (int ps = 0; ok && ps < tc_num_passes<MODE>(a); ps++) {
                    if (pass_alpha<MODE>(a, it.e, it.p, ps) == 0.0f)
                        continue;
                    for (int se = 0; ok && se < nst * nent; se++) {
                        const int s = se / nent, en = se % nent;
                        const int bs = (int)(br.n % kMaxBSlots);
                        const uint32_t o = br.place(ebytes);
                        const uint32_t e = o + ebytes;
                        // retire the oldest stages until none in flight overlaps [o, e)
                        // and barrier bs is free
                        while (ok) {
                            const bool clash = my_busy && my_off < e && o < my_end;
                            const bool full = br.n - 1 - tail >= (uint32_t)kMaxBSlots;
                            if (!__any_sync(0xffffffffu, clash) && !full)
                                break;
                            const int ts = (int)(tail % kMaxBSlots);
                            if (!(ok = warp_wait_bar(&B.bempty[ts], (ph >> ts) & 1, abort, a.hdr)))
                                break;
                            ph ^= 1u << ts;
                            if (lane == ts)
                                my_busy = false;
                            tail++;
                        }
                        if (!ok)
                            break;
                        if (lane == bs) {
                            my_off = o;
                            my_end = e;
                            my_busy = true;
                        }
                        uint8_t *dst = smem + S::off_b + o;
                        if (lane == 0)
                            mbar_arrive_expect_tx(&B.bfull[bs], ebytes);
                        __syncwarp();
                        if (lane < 2) {
                            if (hv.n == 1)
                                tma_load_2d(dst + lane * bg.rb * 128, map, x0 + s * kKS + lane * (kKS / 2), it.row0,
                                            &B.bfull[bs]);
                            else
                                tma_load_2d(dst + lane * hv.hr * 128, map, s * kKS + en * (kKS / 2),
                                            it.row0 + lane * hv.hr, &B.bfull[bs]);
                        }
                    }
                }
            }
            // every load this warp issued is consumed by an MMA before the
            // CTA ends; nothing to wait for here
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------- epilogue (warps 19..26): finished buffers, in item order
        const int ew = warp - kEpiWarp0, q = warp & 3;   // TMEM lane quarter = warp % 4
        float *zs = reinterpret_cast<float *>(smem + S::off_zs);
        int *rowmap = reinterpret_cast<int *>(smem + S::off_rows);
        volatile int *go = reinterpret_cast<volatile int *>(smem + S::off_misc + 24);
        uint32_t nit = 0;
        bool ok = true;
        for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
            const TcItem it = tc_item<MODE>(a, item);
            const Halves hv = item_halves<MODE>(a, it);
            // the CTA's last two-half item: the decode warps, idle by then,
            // take the tail of half 0 and all of half 1
            const bool shared = tc_two_halves<MODE>(a) && item + (int)gridDim.x >= n_items;
            for (int h = 0; h < hv.n; h++, nit++) {
                const uint32_t buf = nit & 1, use = nit >> 1;
                if (shared && h == 1)
                    break;
                // one thread waits for the buffer; the eight warps learn the
                // outcome together at the named barrier, so all of them take
                // the same barriers until the end
                if (ew == 0 && lane == 0)
                    *go = !*abort && wait_bar(&B.tfull[buf], use & 1, abort, a.hdr);
                named_barrier(2, kEpiThreads);
                ok = *go != 0;
                named_barrier(2, kEpiThreads);
                if (!ok)
                    break;
                fence_after();
                TcItem hi = it;
                hi.row0 = it.row0 + h * hv.hr;
                hi.nrows = shared ? shared_split(hv) : hv.rows[h];
                if (hi.nrows > 0)
                    tc_item_epilogue<MODE, kEpiThreads / 32>(a, hi, tmem + buf * kNT, zs, rowmap, ew, q, 0, 2);
                fence_before();
                warp_arrive(&B.tempty[buf]);
            }
        }
    } else {
        // ---------------- decode (warps 2..17)
        const int dt = tid - 64;                 // 0..511
        const int t = dt >> 7;                   // trellis row of the stage
        const int m = dt & 127;                  // output of the block
        RingPos<kStages> ra;
        RingPosN rt;
        rt.n = tg.nslots;
        for (int item = blockIdx.x; item < n_items && !warp_aborted(abort); item += gridDim.x) {
            const TcItem it = tc_item<MODE>(a, item);
            if (!tc_item_decode<MODE>(a, smem, B, abort, it, ra, rt, tg, t, m))
                break;
        }
        if constexpr (MODE == kModeLinear) {
            // the CTA's last two-half item: rows [split, rows0) of half 0 and
            // all of half 1, as a team of 16 warps (named barrier 3)
            // transposing through the A ring, free once the item's MMAs have
            // completed.  Every decode warp takes this path (the item is fixed
            // by the launch, not by how far the loop above got), so the team's
            // barriers always fill; after a timeout the go flag ends it.
            const int last = (int)blockIdx.x + (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x * (int)gridDim.x;
            if (tc_two_halves<MODE>(a)) {
                const TcItem it = tc_item<MODE>(a, last);
                const Halves hv = item_halves<MODE>(a, it);
                const int split = shared_split(hv);
                const uint32_t use = (uint32_t)((last - (int)blockIdx.x) / (int)gridDim.x);   // items before it
                const int ew = warp - 2, q = warp & 3;
                float *zs = reinterpret_cast<float *>(smem + S::off_a);
                volatile int *go = reinterpret_cast<volatile int *>(smem + S::off_misc + 32);
                for (int h = 0; h < 2; h++) {
                    const int r_begin = h == 0 ? split : 0;
                    if (r_begin >= hv.rows[h])
                        continue;
                    // its sub-items are 2*use (buffer 0) and 2*use + 1 (buffer 1)
                    if (ew == 0 && lane == 0)
                        *go = !*abort && wait_bar(&B.tfull[h], use & 1, abort, a.hdr);
                    named_barrier(3, kDecThreads);
                    const bool go_on = *go != 0;
                    named_barrier(3, kDecThreads);
                    if (!go_on)
                        break;
                    fence_after();
                    TcItem hi = it;
                    hi.row0 = it.row0 + h * hv.hr;
                    hi.nrows = hv.rows[h];
                    tc_item_epilogue<MODE, kDecWarps>(a, hi, tmem + (uint32_t)h * kNT, zs, nullptr, ew, q, r_begin, 3);
                    fence_before();
                }
            }
        }
    }

    // after a timeout, give copies and MMAs still in flight time to land
    // before the shared memory and TMEM are released
    if (*abort) {
        const long long t0 = clock64();
        while (clock64() - t0 < (1ll << 21)) {
        }
    }
    // teardown: the MMA warp frees TMEM once the last accumulator was read
    __syncwarp();
    fence_before();
    __syncthreads();
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem), "r"(Smem::tmem_cols) : "memory");
    }
}

template <int MODE>
cudaError_t launch_tc(const GemmArgs &a, const TcMaps &maps, int grid, cudaStream_t s)
{
    TcMapsDev m;
    static_assert(sizeof(m.act) == sizeof(maps.act), "tensor map table");
    memcpy(m.act, maps.act, sizeof(m.act));
    if (!a.tc_pdl) {
        k_expert_tc<MODE><<<grid, kThreads, Smem::total, s>>>(a, m);
        return cudaGetLastError();
    }
    // the linear, right after the rotate kernel: programmatic dependent
    // launch, the activation producer waits for it (every other role reads
    // only the weights and TMEM)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Smem::total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_expert_tc<MODE>, a, m);
}

template <int MODE>
cudaError_t set_attr_tc()
{
    cudaError_t e = cudaFuncSetAttribute(k_expert_tc<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Smem::total);
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(k_expert_tc<MODE>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

}  // namespace tc
}  // namespace exl3
