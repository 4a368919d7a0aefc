// Workspace layout of the MoE layer and of the linear.  The single definition
// used both by the host (sizing, validation, launch arguments) and by every
// kernel (through the Layout struct passed by value), so writer and reader of
// each region can never disagree.
#pragma once
#include <stddef.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define EXL3_HD __host__ __device__
#else
#define EXL3_HD
#endif

namespace exl3 {

constexpr int kHb = 128;           // Hadamard block / output block per work item
constexpr int kChunk = 512;        // inputs per canonical reduction chunk
constexpr int kChunkTk = kChunk / 16;
constexpr int kRowGroup = 16;      // rows per work item (forward, linear)
constexpr int kRowGroupAdd = 8;    // rows per work item (additive stages)
constexpr int kSplitMaxPairs = 640;  // cap on (row group, block) pairs split by chunk

// Header words (int32) at the start of the workspace.
enum HdrWord {
    kHdrError = 0,     // sticky device error word (exl3_device_error bits)
    kHdrNTiles = 1,
    kHdrNumActive = 2,
    kHdrNRg = 3,       // row groups
    kHdrSplit1 = 4,    // gate/up items split by chunk (0/1)
    kHdrSplit2 = 5,    // down / linear items split by chunk (0/1)
    kHdrNItems1 = 6,
    kHdrNItems2 = 7,
    kHdrRegime = 8,    // fused layer: 0 = decode-regime kernels run, 1 = prefill (tcgen05) kernels
    kHdrWords = 64
};

EXL3_HD inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
EXL3_HD inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

struct MoeLayout {
    int M, topk, E, hidden, inter, capacity, R;
    int max_tiles, max_rg, nb1, nb2, nchunks1, nchunks2, split_pairs1, split_pairs2;
    size_t hdr, offsets, packed, tiles, rg, arot, ad, stage, cnt, cnt1, cnt2, part1, part2;
    size_t total;
};

// Row groups of <= rg_size rows never straddle a capacity tile, so their count
// is at most R/rg_size + (number of tiles).
EXL3_HD inline MoeLayout moe_layout(int M, int topk, int E, int hidden, int inter,
                                    int capacity)
{
    MoeLayout L{};
    L.M = M; L.topk = topk; L.E = E; L.hidden = hidden; L.inter = inter;
    L.capacity = capacity;
    L.R = M * topk;
    int active_max = E < L.R ? E : L.R;
    L.max_tiles = L.R / capacity + active_max;
    L.max_rg = L.R / kRowGroupAdd + L.max_tiles;
    L.nb1 = inter / kHb;
    L.nb2 = hidden / kHb;
    L.nchunks1 = ceil_div(hidden, kChunk);
    L.nchunks2 = ceil_div(inter, kChunk);
    long p1 = (long)L.max_rg * L.nb1, p2 = (long)L.max_rg * L.nb2;
    L.split_pairs1 = (int)(p1 < kSplitMaxPairs ? p1 : kSplitMaxPairs);
    L.split_pairs2 = (int)(p2 < kSplitMaxPairs ? p2 : kSplitMaxPairs);
    size_t o = 0;
    L.hdr = o;      o = align_up(o + kHdrWords * 4, 256);
    L.offsets = o;  o = align_up(o + (size_t)(E + 1) * 4, 256);
    L.packed = o;   o = align_up(o + (size_t)L.R * 4, 256);
    L.tiles = o;    o = align_up(o + (size_t)L.max_tiles * 12, 256);
    L.rg = o;       o = align_up(o + (size_t)L.max_rg * 16, 256);
    L.arot = o;     o = align_up(o + (size_t)L.R * 2 * hidden * 2, 256);
    L.ad = o;       o = align_up(o + (size_t)L.R * inter * 2, 256);
    // fp32 staging: the down rows [R][hidden]; above 128 tokens also the
    // prefill regime's rotated gate and up rows [R][2][inter]
    const size_t stage_w = (M > 128 && 2 * inter > hidden) ? 2 * (size_t)inter : (size_t)hidden;
    L.stage = o;    o = align_up(o + (size_t)L.R * stage_w * 4, 256);
    // counters (cleared by every call): combine, gate/up split, down split
    L.cnt = o;      o += (size_t)M * L.nb2 * 4;
    L.cnt1 = o;     o += (size_t)L.split_pairs1 * 4;
    L.cnt2 = o;     o = align_up(o + (size_t)L.split_pairs2 * 4, 256);
    L.part1 = o;    o = align_up(o + (size_t)L.split_pairs1 * L.nchunks1 * kRowGroup * 2 * kHb * 4, 256);
    L.part2 = o;    o = align_up(o + (size_t)L.split_pairs2 * L.nchunks2 * kRowGroup * kHb * 4, 256);
    L.total = o;
    return L;
}

struct LinearLayout {
    int M, in, out, n_rg, nb, nchunks, split_pairs;
    size_t hdr, arot, part, cnt, total;
};

EXL3_HD inline LinearLayout linear_layout(int M, int in_f, int out_f)
{
    LinearLayout L{};
    L.M = M; L.in = in_f; L.out = out_f;
    L.n_rg = ceil_div(M, kRowGroup);
    L.nb = out_f / kHb;
    L.nchunks = ceil_div(in_f, kChunk);
    long p = (long)L.n_rg * L.nb;
    L.split_pairs = (int)(p < kSplitMaxPairs ? p : kSplitMaxPairs);
    size_t o = 0;
    L.hdr = o;   o = align_up(o + kHdrWords * 4, 256);
    L.arot = o;  o = align_up(o + (size_t)M * in_f * 2, 256);
    L.part = o;  o = align_up(o + (size_t)L.split_pairs * L.nchunks * kRowGroup * kHb * 4, 256);
    L.cnt = o;   o = align_up(o + (size_t)L.split_pairs * 4, 256);
    L.total = o;
    return L;
}

}  // namespace exl3
