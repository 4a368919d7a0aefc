/*
 * exl3.h -- C ABI of the GB300 (sm_103a) fused EXL3 routed-expert MoE library.
 *
 * The operations follow four pull-request pages on EXL3 trellis-quantised MoE
 * kernels:
 *   - "MoE: Add fused additive EXL3 kernels" (exllamav3 #284): "Summary" (route
 *     histogram / scan / stable packing, capacity-tiled spans, additive stages,
 *     ABI version), "API contract" (pointer-table lifetime, mcg residuals that
 *     reuse the base suh/svh, zero scale skips a GEMM, num_active is a hint).
 *   - "EXL3 linear and grouped routed experts, every codebook and width, a width
 *     per expert" (TensorFold #837): "What this changes" (trellis decode, input
 *     rotation, row-invariant linear, grouped experts with gate/up, SwiGLU,
 *     down and weighted combine, per-expert widths) and "Receipt" (a row's
 *     bytes do not depend on the row count, the K split or member counts).
 *
 * Definitions the pages leave open (fixed once, identical in the CPU oracle):
 *   - Trellis tile: 16x16 weights, K bits each (K = 1..8), stored as 8*K
 *     little-endian uint32 words; the 256*K-bit string is read most significant
 *     bit first.  State of position p = the 16-bit window ending at bit
 *     (p+1)*K - 1, cyclic (tail-biting).  Position p holds the weight at input
 *     row (p % 16), output column (p / 16) of its tile.  A projection with
 *     `in` inputs and `out` outputs stores tiles as uint32 [in/16][out/16][8*K].
 *   - Codebooks (enum exl3_codebook): 3inst x = 89226354*s + 64248484; mcg
 *     x = 0xCBAC1FED*s; both then x = (x & 0x8FFF8FFF) ^ 0x3B603B60 and the
 *     weight is fp16(x[15:0]) + fp16(x[31:16]).  mul1 x = 0x83DCD12D*s and the
 *     weight is (sum of the four bytes of x - 510) / sqrt(21845).
 *   - Rotations: a' = Hb(a * suh); y = Hb(a' W) * svh * scale, Hb the
 *     block-diagonal 128-point Sylvester Hadamard scaled by 1/sqrt(128).
 *     Every feature count must be a multiple of 128.
 *   - SwiGLU: h = silu(g) * u with silu(g) = g / (1 + exp(-g)).
 *   - Combine: out[t] = sum over j = 0..topk-1 (ascending) of rw[t,j] * d[t,j].
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers on the device that owns `stream`,
 *     row-major and contiguous, unless marked "host".  The caller owns all
 *     memory.  The library never allocates, frees, synchronises or retains a
 *     pointer after it returns; every call only enqueues kernels on `stream`,
 *     so calls can be captured in a CUDA graph.  The first call on a device
 *     sets kernel attributes and reads device attributes; make it outside
 *     stream capture (inside one it returns EXL3_E_CUDA).  While `stream` is
 *     capturing, the checks that pointers live on the stream's device are
 *     skipped (those queries cannot run on a capturing stream); an eager
 *     call with the same arguments performs them.
 *   - A negative return is a contract violation found on the host; nothing
 *     was written to device memory and nothing was launched.
 *   - Contracts that only the device can check (route ids in [0, E), each
 *     expert table entry: K in 1..8, codebook in range, non-null 16-byte
 *     aligned pointers) set a sticky error word in the workspace (see
 *     exl3_workspace_error); later kernels of the call then skip their work and
 *     the output is zero-filled.
 */
#ifndef EXL3_GB300_H
#define EXL3_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exact-match compatibility contract (exllamav3 #284, "API contract"): bumped
 * for any incompatible change of signature, pointer layout, workspace, residual
 * encoding or capacity semantics. */
#define EXL3_ABI_VERSION 1

/* Largest expert count a call accepts. */
#define EXL3_MAX_EXPERTS 1024

enum exl3_status {
    EXL3_OK = 0,
    EXL3_E_NULL = -1,       /* a required pointer is NULL */
    EXL3_E_DEVICE = -2,     /* a pointer is not device memory of the stream's device */
    EXL3_E_DTYPE = -3,      /* unknown dtype enum */
    EXL3_E_SHAPE = -4,      /* a size is out of range or not a multiple of 128 */
    EXL3_E_ALIGN = -5,      /* a pointer is not 16-byte aligned (workspace: 256) */
    EXL3_E_WORKSPACE = -6,  /* ws_bytes below the *_workspace_bytes() result */
    EXL3_E_ROUTING = -7,    /* bad topk / capacity / expert count */
    EXL3_E_CODEBOOK = -8,   /* K outside 1..8 or unknown codebook (host-checked cases) */
    EXL3_E_CUDA = -9        /* a CUDA runtime call failed */
};

/* Device error word bits (exl3_workspace_error). */
enum exl3_device_error {
    EXL3_DERR_ROUTE_ID = 1,   /* a route id outside [0, E) */
    EXL3_DERR_TABLE = 2,      /* a used expert / stage table entry is invalid */
    EXL3_DERR_TIMEOUT = 4     /* a bounded wait on an asynchronous copy gave up */
};

enum exl3_dtype { EXL3_F16 = 0, EXL3_BF16 = 1, EXL3_F32 = 2, EXL3_I32 = 3, EXL3_I64 = 4 };
enum exl3_codebook { EXL3_CB_MUL1 = 0, EXL3_CB_MCG = 1, EXL3_CB_3INST = 2 };
enum exl3_projection { EXL3_GATE = 0, EXL3_UP = 1, EXL3_DOWN = 2 };

/* One projection (host struct holding device pointers).
 *   trellis: uint32 [in/16][out/16][8*K]; suh: fp16 [in]; svh, scale: fp16 [out];
 *   in_features, out_features: multiples of 128. */
typedef struct exl3_proj {
    const uint32_t *trellis;
    const uint16_t *suh;
    const uint16_t *svh;
    const uint16_t *scale;
    int32_t in_features;
    int32_t out_features;
    int32_t K;
    int32_t codebook;
} exl3_proj;

/* Per-expert descriptor tables (host struct holding DEVICE table pointers).
 * Entry (e, p) sits at index e*3 + p, p = gate, up, down.  Pointer tables hold
 * device addresses as int64 and do not retain their pointees: the caller keeps
 * every referenced allocation alive, unmoved and on this device until the
 * call completes, and for the lifetime of any graph that captured it
 * (exllamav3 #284, "API contract").  Gate/up are [hidden -> inter], down is
 * [inter -> hidden].  Only entries of experts that receive routes are read. */
typedef struct exl3_experts {
    const int64_t *trellis;   /* [E*3] */
    const int64_t *suh;       /* [E*3] fp16 vectors */
    const int64_t *svh;       /* [E*3] */
    const int64_t *scale;     /* [E*3] */
    const int32_t *K;         /* [E*3] */
    const int32_t *codebook;  /* [E*3] */
} exl3_experts;

/* Additive residual stages (exllamav3 #284, "Summary" and "API contract").
 * Stage-major device tables for stages s = 1..num_stages-1 (stage 0 is the
 * base): entry (s, e, p) at index ((s-1)*E + e)*3 + p.  Residual trellises use
 * the mcg codebook at their own K and reuse the base projection's suh, svh and
 * scale.  A zero scale skips that projection's GEMM: its trellis pointer is
 * not read and may be NULL, and its K is not checked. */
typedef struct exl3_stages {
    int32_t num_stages;       /* >= 1 (1 = base only) */
    const int64_t *trellis;   /* [(S-1)*E*3] */
    const float *scale;       /* [(S-1)*E*3] alpha, applied in fp32 */
    const int32_t *K;         /* [(S-1)*E*3] */
} exl3_stages;

int exl3_abi_version(void);

/* Bytes of workspace exl3_moe_forward / exl3_moe_additive need.  Depends only
 * on the arguments (M tokens, topk, E experts, hidden, inter, capacity).
 * Returns 0 for invalid arguments. */
size_t exl3_moe_workspace_bytes(int M, int topk, int E, int hidden, int inter, int capacity);

/* Bytes of workspace exl3_linear needs for M rows of in -> out. */
size_t exl3_linear_workspace_bytes(int M, int in_features, int out_features);

/* Upper bound of the number of span tiles exl3_route_pack can write:
 * floor(M*topk / capacity) + min(E, M*topk). */
int exl3_route_pack_max_tiles(int M, int topk, int E, int capacity);

/* Route histogram, exclusive scan and stable packing (exllamav3 #284,
 * "Summary" and "Relationship to #246").
 *   ids: [M][topk] int32 or int64 (ids_dtype), expert of flat route f = t*topk + j
 *        (ids, packed and tiles may be NULL when M == 0).
 *   offsets: int32 [E+1], offsets[e] = first packed slot of expert e.
 *   packed:  int32 [M*topk], packed[offsets[e] + r] = the r-th smallest f with
 *            id e (stable in f; bit-exact).
 *   tiles:   int32 [max_tiles][3] = (expert, first packed slot, length), one tile
 *            per `capacity` routes of each expert's span, ascending (expert, slot).
 *   info:    int32 [4] = (device error word, number of tiles, num_active =
 *            experts with >= 1 route, 0).
 * num_active is only a launch-size hint (exllamav3 #284, "API contract"). */
int exl3_route_pack(const void *ids, int ids_dtype, int M, int topk, int E, int capacity,
                    int32_t *offsets, int32_t *packed, int32_t *tiles, int32_t *info,
                    cudaStream_t stream);

/* One EXL3 projection for M rows: y = Hb(Hb(x * suh) W) * svh * scale
 * (TensorFold #837, "What this changes": the linear and the input rotation).
 *   x: [M][in] act_dtype (f16 or bf16); y: [M][out] act_dtype.
 *   proj: host struct, validated on the host.  A row's output bytes do not
 *   depend on M. */
int exl3_linear(const void *x, int act_dtype, int M, const exl3_proj *proj, void *y,
                void *workspace, size_t ws_bytes, cudaStream_t stream);

/* The fused routed-expert MoE layer (TensorFold #837 "What this changes";
 * exllamav3 #284 "Summary"): route packing, per route r = (t, j) with
 * e = ids[t][j]: g = gate_e(x_t), u = up_e(x_t), h = silu(g) * u,
 * d = down_e(h); out[t] = sum_j rw[t][j] * d_{t,j}.
 *   x: [M][hidden] act_dtype (f16/bf16); ids: [M][topk] int32/int64;
 *   rw: [M][topk] f16/bf16/f32; out: [M][hidden] act_dtype.
 *   capacity: routes per span tile; results do not depend on it.
 *   workspace: >= exl3_moe_workspace_bytes(...), 256-byte aligned; its
 *   contents need not be initialised.  Two calls must not share a workspace
 *   concurrently. */
int exl3_moe_forward(const void *x, int act_dtype, int M, int hidden, int inter, int E,
                     int topk, const void *ids, int ids_dtype, const void *rw, int rw_dtype,
                     const exl3_experts *experts, int capacity, void *workspace,
                     size_t ws_bytes, void *out, cudaStream_t stream);

/* exl3_moe_forward plus additive residual stages (exllamav3 #284 "Summary":
 * exl3_moe_additive_fused).  For every projection the weights become
 * W_base + sum_s alpha_{s,e,p} W_{s,e,p}, accumulated in fp32: up to 128
 * tokens each stage's partial sum is scaled by alpha in fp32 and added to the
 * accumulator; above 128 tokens, when the tensor-core kernels run the layer,
 * a stage is one more pass over the same fp32 accumulators with its decoded
 * fp16 weights multiplied by alpha.  Entries with alpha == 0 read no bytes and
 * run no MMA, so all-zero stages reproduce exl3_moe_forward bit for bit.
 * stages: host struct holding device tables. */
int exl3_moe_additive(const void *x, int act_dtype, int M, int hidden, int inter, int E,
                      int topk, const void *ids, int ids_dtype, const void *rw, int rw_dtype,
                      const exl3_experts *experts, const exl3_stages *stages, int capacity,
                      void *workspace, size_t ws_bytes, void *out, cudaStream_t stream);

/* exl3_linear for callers that cannot allocate device memory (graph replays
 * without a memory pool, hosts whose allocator forbids cudaMalloc, paths where
 * an allocation would synchronise).  Same result as exl3_linear, but its
 * workspace is one fixed scratch array inside the library's device image
 * (exl3_linear_noalloc_max_scratch_bytes() bytes, resident on every GPU that
 * loads the library until the process exits).  Allocates nothing.  The first
 * call on a device looks up the scratch address for that device (make it
 * before any stream capture).  Calls whose exl3_linear_workspace_bytes(M, in,
 * out) exceeds the scratch size return EXL3_E_WORKSPACE without launching.
 * All calls share the scratch: calls that may overlap on the GPU (different
 * streams, or graphs replayed concurrently) race and must be serialised by the
 * caller.  The pages have no counterpart; this entry point is an addition. */
size_t exl3_linear_noalloc_max_scratch_bytes(void);
int exl3_linear_noalloc(const void *x, int act_dtype, int M, const exl3_proj *proj, void *y,
                        cudaStream_t stream);
/* The failure channel of exl3_linear_noalloc, whose workspace the caller never
 * sees: waits for `stream`, then stores in *err_host the device error word
 * (exl3_device_error bits, 0 = none) that the last exl3_linear_noalloc call on
 * the current device left in the scratch.  Synchronises; never call it while
 * the stream is capturing.  Returns EXL3_E_NULL for a null err_host. */
int exl3_linear_noalloc_error(int32_t *err_host, cudaStream_t stream);

/* Benchmark instrumentation: when `events` is non-NULL, the following calls of
 * exl3_moe_forward / exl3_moe_additive on this host thread record the five
 * cudaEvent_t in events[0..4] on their stream before the route pack, after the
 * route pack, after the input rotation, after the gate/up GEMM and after the
 * down GEMM + combine, so that each kernel's time can be read with
 * cudaEventElapsedTime.  NULL switches recording off.  The events stay owned
 * by the caller.  Always returns EXL3_OK. */
int exl3_profile_events(void *const *events);

/* Reads the device error word of the last call that used `workspace`.
 * SYNCHRONISES `stream`; for tests and debugging, never inside a capture. */
int exl3_workspace_error(const void *workspace, int32_t *err_host, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* EXL3_GB300_H */
