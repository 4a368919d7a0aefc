"""GPU parity of the CUDA path (through the C ABI) against the float64 oracle.

Route packing must be bit-exact; layer outputs within relative L2 2e-3 and
max-abs 1e-2 of the oracle; a row's bytes identical across batch sizes,
chunk splits, member counts and capacities (TensorFold #837, "Receipt";
exllamav3 #284, "Validation")."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import trellis_quantized_moe_gb300 as X  # noqa: E402
from oracle import exl3_oracle as O  # noqa: E402
from workloads import (CB_3INST, CB_MCG, CB_MUL1, LinearWorkload, MoEWorkload,  # noqa: E402
                       act_to_f64, config)
from gpu_common import (assert_close, assert_close_linear, covering_tokens, moe_inputs,  # noqa: E402
                        oracle_rows, out_tensor, to_device, to_f64)


# --------------------------------------------------------------------------- route pack
def _pack_on_gpu(ids_np, E, cap, dtype):
    ids = torch.from_numpy(ids_np.astype(np.int64 if dtype == "i64" else np.int32)).cuda()
    M, topk = ids_np.shape
    R = M * topk
    nt = X.exl3_route_pack_max_tiles(M, topk, E, cap)
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    packed = torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda")
    tiles = torch.full((max(nt, 1), 3), -7, dtype=torch.int32, device="cuda")
    info = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    X.exl3_route_pack(ids, E, cap, off, packed, tiles, info)
    torch.cuda.synchronize()
    info = info.cpu().numpy()
    return (off.cpu().numpy(), packed.cpu().numpy()[:R], tiles.cpu().numpy()[:info[1]], info)


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_route_pack_bit_exact_on_configs(cfg):
    s = config(cfg, M={1: 128}.get(cfg))
    w = MoEWorkload(s)
    off, packed, tiles, info = _pack_on_gpu(w.ids, s.E, s.capacity, s.ids_dtype)
    r_off, r_packed, r_tiles, r_nact = O.route_pack(w.ids, s.E, s.capacity)
    assert info[0] == 0
    assert np.array_equal(off, r_off) and np.array_equal(packed, r_packed)
    assert np.array_equal(tiles, r_tiles) and info[2] == r_nact


@pytest.mark.parametrize("M,topk,E,cap,dt", [
    (16, 2, 8, 32, "i32"),          # topk=2, capacity = rows
    (9, 4, 3, 11, "i64"),           # one expert gets exactly capacity + 1
    (300, 8, 5, 64, "i32"),         # multi-tile spans, multi-step warps
    (4000, 8, 1000, 7, "i64"),      # many experts, many warps
    (1, 1, 1, 1, "i32"),
    (0, 8, 16, 4, "i32"),           # empty batch
    # at most 32 routes: the one-warp kernel
    (1, 8, 192, 512, "i32"),        # one decode token over 192 experts
    (4, 8, 192, 1, "i64"),          # capacity 1: every route its own tile
    (31, 1, 3, 2, "i32"),           # 31 routes over 3 experts, multi-tile spans
    (8, 4, 5, 3, "i64"),            # 32 routes, ragged tiles
])
def test_route_pack_edge_cases(M, topk, E, cap, dt):
    rng = np.random.default_rng(M + E)
    ids = rng.integers(0, E, size=(M, topk))
    if M == 9:
        ids[:, :] = np.arange(M * topk).reshape(M, topk) % 3
        ids[ids == 0] = 1
        ids.reshape(-1)[:cap + 1] = 0
    if (M, topk) == (8, 4):
        ids[2, :] = 4                   # one token listing an expert four times
    off, packed, tiles, info = _pack_on_gpu(ids, E, cap, dt)
    r_off, r_packed, r_tiles, r_nact = O.route_pack(ids, E, cap)
    assert np.array_equal(off, r_off) and np.array_equal(packed, r_packed)
    assert np.array_equal(tiles, r_tiles) and info[2] == r_nact and info[0] == 0


def test_route_pack_bad_id_sets_error_word():
    ids = np.array([[0, 1], [5, 2]])
    _, _, _, info = _pack_on_gpu(ids, 4, 2, "i32")
    assert info[0] & X.binding.DERR_ROUTE_ID


# --------------------------------------------------------------------------- linear
def _linear_gpu(lw, dev_proj=None):
    p = dev_proj or X.DeviceProjection(lw.proj)
    x = to_device(lw.x, lw.act)
    y = torch.empty((lw.M, lw.proj.out_features), dtype=x.dtype, device="cuda")
    ws = torch.empty(X.exl3_linear_workspace_bytes(lw.M, lw.proj.in_features,
                                                    lw.proj.out_features), dtype=torch.uint8,
                     device="cuda")
    X.exl3_linear(x, p, y, ws)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("cb", [CB_MUL1, CB_MCG, CB_3INST])
def test_linear_every_width_and_codebook(K, cb):
    lw = LinearWorkload(M=5, in_f=640, out_f=384, K=K, cb=cb, act="f16", seed=K * 3 + cb)
    y = to_f64(_linear_gpu(lw))
    ref = O.linear(act_to_f64(lw.x, "f16"), lw.proj)
    assert_close_linear(y, ref, "f16", f"linear K={K} cb={cb}")


@pytest.mark.parametrize("M,in_f,out_f,act", [(1, 4096, 1408, "bf16"), (37, 1408, 4096, "f16"),
                                              (128, 512, 256, "bf16"), (200, 256, 128, "f16")])
def test_linear_shapes(M, in_f, out_f, act):
    lw = LinearWorkload(M=M, in_f=in_f, out_f=out_f, K=4, cb=CB_MCG, act=act, seed=M)
    y = to_f64(_linear_gpu(lw))
    rows = np.arange(min(M, 24))
    ref = O.linear(act_to_f64(lw.x, act)[rows], lw.proj)
    assert_close_linear(y[rows], ref, act, f"linear {M}x{in_f}x{out_f}")


@pytest.mark.parametrize("M,K,cb,act", [(300, 3, CB_MCG, "bf16"), (600, 5, CB_3INST, "f16"),
                                        (129, 2, CB_MUL1, "f16")])
def test_linear_prompt_rows_tcgen05(M, K, cb, act):
    # more than 128 rows: the tcgen05 kernel (items of 256 rows; 300 and 600
    # leave ragged last tiles, 129 a one-row tile); sampled rows from every tile
    lw = LinearWorkload(M=M, in_f=1024, out_f=640, K=K, cb=cb, act=act, seed=M + K)
    y = to_f64(_linear_gpu(lw))
    rows = np.unique(np.array([0, 1, 127, 128, 255, 256, M // 2, M - 2, M - 1]) % M)
    ref = O.linear(act_to_f64(lw.x, act)[rows], lw.proj)
    assert_close_linear(y[rows], ref, act, f"linear tcgen05 M={M} K={K} cb={cb}")


@pytest.mark.parametrize("M", [4900, 5056, 5220])
def test_linear_two_half_items(M):
    # 256-row items would need a second wave (on 152 SMs: 20 or 21 row tiles x
    # 8 blocks), so the launch takes items of 288 rows in two 144-row halves,
    # one wave: 4900 leaves a 4-row last item (empty second half), 5056 a
    # 160-row one (a 16-row second half), 5220 a 36-row one.  Every row
    # against the oracle, and the bytes equal those of a launch of 256-row
    # items
    lw = LinearWorkload(M=M, in_f=256, out_f=1024, K=3, cb=CB_MCG, act="bf16", seed=M)
    dp = X.DeviceProjection(lw.proj)
    y = _linear_gpu(lw, dp)
    ref = O.linear(act_to_f64(lw.x, "bf16"), lw.proj)
    assert_close_linear(to_f64(y), ref, "bf16", f"linear two-half items M={M}")
    few = LinearWorkload(M=1024, in_f=256, out_f=1024, K=3, cb=CB_MCG, act="bf16", seed=M)
    few.x = lw.x[:1024]
    y_few = _linear_gpu(few, dp).view(torch.int16).cpu().numpy()
    assert np.array_equal(y.view(torch.int16).cpu().numpy()[:1024], y_few)


@pytest.mark.parametrize("M", [10000, 10100])
def test_linear_more_row_tiles_than_sms(M):
    # too many rows for one wave of 512-row items (on 152 SMs, 19 row groups x
    # 8 blocks): 256-row items, CTAs run two or three each, alternating between
    # the two TMEM accumulators (10100: a 116-row last tile); every row against
    # the oracle, and the bytes equal those of a launch with fewer items
    lw = LinearWorkload(M=M, in_f=256, out_f=1024, K=3, cb=CB_MCG, act="bf16", seed=M)
    dp = X.DeviceProjection(lw.proj)
    y = _linear_gpu(lw, dp)
    ref = O.linear(act_to_f64(lw.x, "bf16"), lw.proj)
    assert_close_linear(to_f64(y), ref, "bf16", f"linear multi-item M={M}")
    few = LinearWorkload(M=1024, in_f=256, out_f=1024, K=3, cb=CB_MCG, act="bf16", seed=M)
    few.x = lw.x[:1024]
    y_few = _linear_gpu(few, dp).view(torch.int16).cpu().numpy()
    assert np.array_equal(y.view(torch.int16).cpu().numpy()[:1024], y_few)


def test_linear_prompt_rows_do_not_depend_on_row_count():
    # above 128 rows every output column is computed by the same tcgen05
    # contraction whatever the tile's row count
    big = LinearWorkload(M=600, in_f=1024, out_f=512, K=4, cb=CB_MCG, act="bf16", seed=5)
    dp = X.DeviceProjection(big.proj)
    y_big = _linear_gpu(big, dp).view(torch.int16).cpu().numpy()
    for M in (129, 300, 513):
        small = LinearWorkload(M=M, in_f=1024, out_f=512, K=4, cb=CB_MCG, act="bf16", seed=5)
        small.x = big.x[:M]
        y = _linear_gpu(small, dp).view(torch.int16).cpu().numpy()
        assert np.array_equal(y, y_big[:M]), M


def test_linear_rows_are_byte_invariant_across_row_counts():
    big = LinearWorkload(M=128, in_f=5120, out_f=1536, K=3, cb=CB_MCG, act="bf16", seed=77)
    dp = X.DeviceProjection(big.proj)
    y_big = _linear_gpu(big, dp).view(torch.int16).cpu().numpy()
    for M in (1, 2, 7, 16, 17, 64):
        small = LinearWorkload(M=M, in_f=5120, out_f=1536, K=3, cb=CB_MCG, act="bf16", seed=77)
        small.x = big.x[:M]
        y = _linear_gpu(small, dp).view(torch.int16).cpu().numpy()
        assert np.array_equal(y, y_big[:M]), M


# --------------------------------------------------------------------------- fused layer
_EXPERTS = {}


def _experts(cfg):
    if cfg not in _EXPERTS:
        _EXPERTS.clear()
        torch.cuda.empty_cache()
        w = MoEWorkload(config(cfg, M=1))
        _EXPERTS[cfg] = X.DeviceExperts.from_workload(w)
    return _EXPERTS[cfg]


def _stages(w):
    s = w.spec
    return X.DeviceStages(w.residual, w.alpha, s.residual_K, s.E)


# regime of the last run_layer call: workspace header word 8, written by the
# route-pack kernel (0 = decode-regime kernels ran, 1 = tcgen05 kernels ran)
LAST = {}


def run_layer(w, experts, capacity=None, stages=None, ws=None):
    s = w.spec
    x, ids, rw = moe_inputs(w)
    out = out_tensor(w)
    cap = capacity or s.capacity
    if ws is None:
        ws = torch.empty(X.exl3_moe_workspace_bytes(s.M, s.topk, s.E, s.hidden, s.inter, cap),
                         dtype=torch.uint8, device="cuda")
    if stages is None:
        X.exl3_moe_forward(x, ids, rw, experts, cap, ws, out)
    else:
        X.exl3_moe_additive(x, ids, rw, experts, stages, cap, ws, out)
    torch.cuda.synchronize()
    assert X.exl3_workspace_error(ws) == 0
    LAST["regime"] = int(ws[:64 * 4].view(torch.int32)[8].item())
    return out


def test_tiny_layer_full_parity():
    w = MoEWorkload(config(0))
    out = to_f64(run_layer(w, _experts(0)))
    assert_close(out, oracle_rows(w), w.spec.act, "config 0")


def test_tiny_layer_capacity_does_not_change_bytes():
    w = MoEWorkload(config(0))
    outs = [run_layer(w, _experts(0), capacity=c).view(torch.int16).cpu().numpy()
            for c in (1, 3, 5, 512)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("M,n", [(1, None), (8, None), (32, 8), (128, 8)])
def test_decode_layer_parity(M, n):
    w = MoEWorkload(config(1, M=M))
    out = to_f64(run_layer(w, _experts(1)))
    rows = np.arange(M) if n is None else covering_tokens(w, n, seed=M, cover=False)
    assert_close(out[rows], oracle_rows(w, tokens=rows), w.spec.act, f"config 1 M={M}")


@pytest.mark.parametrize("cfg,M", [(1, 1), (1, 32), (0, 16)])
def test_layer_replayed_from_a_cuda_graph_matches_eager(cfg, M):
    # the forward allocates and synchronises nothing, so it can be captured;
    # the replay (with the dependent launches of small layers inside the
    # graph) writes the same bytes as the eager call
    w = MoEWorkload(config(cfg, M=M))
    s = w.spec
    ex = _experts(cfg)
    x, ids, rw = moe_inputs(w)
    ws = torch.empty(X.exl3_moe_workspace_bytes(s.M, s.topk, s.E, s.hidden, s.inter, s.capacity),
                     dtype=torch.uint8, device="cuda")
    eager = out_tensor(w)
    X.exl3_moe_forward(x, ids, rw, ex, s.capacity, ws, eager)
    torch.cuda.synchronize()
    out = out_tensor(w)
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            X.exl3_moe_forward(x, ids, rw, ex, s.capacity, ws, out)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert X.exl3_workspace_error(ws) == 0
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_decode_layer_rows_byte_invariant_across_batch_sizes():
    # tokens are prefixes of one stream, so every row of the smaller batch is
    # compared with the same row of the next larger one
    prev = None
    for M in (1, 2, 8, 32, 128):
        w = MoEWorkload(config(1, M=M))
        o = run_layer(w, _experts(1)).view(torch.int16).cpu().numpy()
        if prev is not None:
            assert np.array_equal(o[:prev.shape[0]], prev), M
        prev = o


def _small_layer(M, act, seed, E=8, topk=2):
    from workloads import MoESpec
    Ks = [1, 2, 3, 4, 5, 6, 7, 8][:E]
    cbs = [CB_MCG, CB_3INST, CB_MUL1, CB_MCG, CB_3INST, CB_MUL1, CB_MCG, CB_3INST][:E]
    spec = MoESpec("small", 512, 256, E, topk, M, act, "i32", "f16", np.array(Ks), np.array(cbs),
                   seed=seed)
    return MoEWorkload(spec)


@pytest.mark.parametrize("act", ["f16", "bf16"])
def test_small_layer_rows_byte_invariant_across_batch_sizes(act):
    # every width 1..8 and all three codebooks: a token's row at 16 tokens
    # (32 routes: inputs rotated inside the gate/up kernel, chunks split over
    # CTAs, 8-row items) equals its row at 40 tokens (80 routes: the rotate
    # kernel, 16-row items) byte for byte, and both are within tolerance
    small = _small_layer(16, act, 123)
    large = _small_layer(40, act, 123)
    ex = X.DeviceExperts.from_workload(large)
    a = run_layer(small, ex).view(torch.int16).cpu().numpy()
    b = run_layer(large, ex).view(torch.int16).cpu().numpy()
    assert np.array_equal(a, b[:16])
    got = to_f64(run_layer(small, ex))
    assert_close(got, oracle_rows(small), act, f"16 tokens {act}")


@pytest.mark.parametrize("M,act", [(512, "f16"), (1100, "bf16")])
def test_prefill_path_small_layer_full_parity(M, act):
    # M > 128 with > 64 routes per expert: the tcgen05 path; M=1100 puts more
    # than 256 routes on some experts (several row tiles per expert)
    w = _small_layer(M, act, seed=40 + M)
    ex = X.DeviceExperts.from_workload(w)
    assert np.bincount(w.ids.reshape(-1), minlength=8).max() > (256 if M > 1000 else 64)
    out = to_f64(run_layer(w, ex))
    assert LAST["regime"] == 1
    # outputs are O(1) here (8 experts, top-2): worst element within one output
    # ulp plus 1e-2 of the output rms, rel-L2 2e-3
    assert_close_linear(out, oracle_rows(w), act, f"prefill path M={M}")


def test_prefill_path_rows_do_not_depend_on_capacity():
    w = _small_layer(600, "f16", seed=7)
    ex = X.DeviceExperts.from_workload(w)
    a = run_layer(w, ex, capacity=512).view(torch.int16).cpu().numpy()
    assert LAST["regime"] == 1
    b = run_layer(w, ex, capacity=97).view(torch.int16).cpu().numpy()
    assert LAST["regime"] == 1
    assert np.array_equal(a, b)


def test_prefill_rows_do_not_depend_on_row_group_boundaries():
    # more than 256 routes per expert: capacity 512 cuts each expert's span
    # into 256 + 256 + ... row groups, 2048 into 256-route groups from the
    # span's start, 200 into groups of <= 200.  A route's bytes are the same
    # in any group.
    w = _small_layer(1100, "bf16", seed=1140)
    assert np.bincount(w.ids.reshape(-1), minlength=8).min() > 256
    ex = X.DeviceExperts.from_workload(w)
    outs = []
    for cap in (512, 2048, 200):
        outs.append(run_layer(w, ex, capacity=cap).view(torch.int16).cpu().numpy())
        assert LAST["regime"] == 1
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


@pytest.mark.parametrize("cfg,M,regime", [(1, 136, 0), (3, 160, 1)])
def test_regime_choice_above_128_tokens(cfg, M, regime):
    # both kernel pairs are launched above 128 tokens; the route-pack kernel
    # picks one from the route counts: few routes per expert (uniform routing)
    # keep the decode regime, Zipf-concentrated routing takes the tcgen05 path
    w = MoEWorkload(config(cfg, M=M))
    out = to_f64(run_layer(w, _experts(cfg)))
    assert LAST["regime"] == regime
    rows = np.array([0, M // 2, M - 1])
    assert_close(out[rows], oracle_rows(w, tokens=rows), w.spec.act, f"config {cfg} M={M}")


def test_mixed_width_layer_parity():
    w = MoEWorkload(config(2))
    out = to_f64(run_layer(w, _experts(2)))
    rows = covering_tokens(w, 32, seed=2, cover=False)
    assert_close(out[rows], oracle_rows(w, tokens=rows), w.spec.act, "config 2")


def test_prefill_layer_parity_sampled():
    w = MoEWorkload(config(3))
    out = to_f64(run_layer(w, _experts(3)))
    assert LAST["regime"] == 1
    # >= 64 tokens, with a checked route in every 256-route half of every
    # capacity tile (the multi-tile spans of the Zipf-heavy experts included)
    rows = covering_tokens(w, 64, seed=3)
    assert len(rows) >= 64
    assert_close(out[rows], oracle_rows(w, tokens=rows), w.spec.act, "config 3")
    assert np.all(np.isfinite(out))


def test_additive_layer_parity_and_zero_scale_identity():
    w = MoEWorkload(config(4))
    ex = _experts(4)
    st = _stages(w)
    out = run_layer(w, ex, stages=st)
    assert LAST["regime"] == 1            # ~14 routes per expert: the tcgen05 kernels
    rows = covering_tokens(w, 32, seed=4, cover=False)
    assert_close(to_f64(out)[rows], oracle_rows(w, tokens=rows), w.spec.act, "config 4")
    # every stage at scale 0: bit-identical to the base-only forward
    zero = _stages(w)
    zero.t_scale.zero_()
    a = run_layer(w, ex, stages=zero).view(torch.int16).cpu().numpy()
    b = run_layer(w, ex).view(torch.int16).cpu().numpy()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("M", [24, 300, 1100])
def test_three_residual_stages_of_mixed_widths(M):
    # S = 4 (base + stages of K = 3, 1, 5, mcg, base rotations), some alpha
    # exactly 0, bases of all three codebooks (a mul1 base scales its mcg
    # residuals differently); above 128 tokens the tcgen05 kernels run the
    # stages as extra passes over their accumulators (1100 tokens: ~275
    # routes per expert, so each down item is two 256-route halves)
    from workloads import MoESpec
    E = 8
    spec = MoESpec("stages", 512, 256, E, 2, M, "f16", "i32", "f32", np.full(E, 4),
                   np.array([CB_MCG, CB_3INST, CB_MUL1, CB_MCG] * 2), seed=90 + M,
                   residual_K=[3, 1, 5], residual_zero_frac=0.3)
    w = MoEWorkload(spec)
    ex = X.DeviceExperts.from_workload(w)
    st = _stages(w)
    out = to_f64(run_layer(w, ex, stages=st))
    assert LAST["regime"] == (0 if M <= 128 else 1)
    assert_close_linear(out, oracle_rows(w), "f16", f"three stages M={M}")
    zero = _stages(w)
    zero.t_scale.zero_()
    a = run_layer(w, ex, stages=zero).view(torch.int16).cpu().numpy()
    b = run_layer(w, ex).view(torch.int16).cpu().numpy()
    assert np.array_equal(a, b)


def _dense_moe(w, get_dense, tokens):
    """Float64 layer from dense per-(expert, projection) weights W[in, out]:
    the oracle's routing, rotations, SwiGLU and j-ordered combine."""
    s = w.spec
    x = act_to_f64(w.x, s.act)
    from workloads import rw_to_f64
    rw = rw_to_f64(w.rw, s.rw_dtype)
    out = np.zeros((len(tokens), s.hidden))
    for i, t in enumerate(tokens):
        for j in range(s.topk):
            e = int(w.ids[t, j])
            pr = [w.projection(e, q, cache=True) for q in range(3)]
            g = O.linear_from_dense(x[t:t + 1], get_dense(e, 0), pr[0].suh, pr[0].svh, pr[0].scale)
            u = O.linear_from_dense(x[t:t + 1], get_dense(e, 1), pr[1].suh, pr[1].svh, pr[1].scale)
            d = O.linear_from_dense(O.silu(g) * u, get_dense(e, 2), pr[2].suh, pr[2].svh, pr[2].scale)
            out[i] += float(rw[t, j]) * d[0]
    return out


def test_prefill_additive_rounding_stays_within_its_bound():
    # Above 128 tokens a residual stage is one more pass over the base
    # accumulator with its decoded fp16 weights multiplied by fp16(alpha')
    # (alpha' = alpha * sqrt(21845) over a mul1 base, whose accumulator is
    # scaled by 1/sqrt(21845) at the end), i.e. W_res -> fp16(fp16(W_res) *
    # fp16(alpha')) / c: two extra roundings of 2^-11 each per residual
    # weight, where the decode regime scales the fp32 partial instead.
    # (1) the kernel equals that model within the layer tolerance, and (2)
    # the model's departure from the exact stage sum is at most 2^-8 of the
    # residual stages' own contribution (4x the 2^-10 per-weight bound).
    from workloads import MoESpec
    E = 8
    spec = MoESpec("stages", 512, 256, E, 2, 300, "f16", "i32", "f32", np.full(E, 4),
                   np.array([CB_MCG, CB_3INST, CB_MUL1, CB_MCG] * 2), seed=391,
                   residual_K=[3, 1, 5], residual_zero_frac=0.3)
    w = MoEWorkload(spec)
    ex = X.DeviceExperts.from_workload(w)
    gpu = to_f64(run_layer(w, ex, stages=_stages(w)))
    assert LAST["regime"] == 1
    tokens = np.arange(0, 300, 7)
    f16 = lambda a: np.asarray(a, np.float64).astype(np.float16).astype(np.float64)  # noqa: E731
    cache = {}

    def dense(e, p, mode):
        key = (e, p, mode)
        if key not in cache:
            pr = w.projection(e, p, cache=True)
            base = O.decode_projection(pr.trellis, pr.K, pr.codebook)
            c = np.sqrt(21845.0) if pr.codebook == CB_MUL1 else 1.0
            W = base if pr.codebook == CB_MUL1 else f16(base)      # the kernel's fp16 weight sums
            if mode == "base":
                cache[key] = W
                return W
            for st in range(1, spec.num_stages):
                a = float(w.alpha[st - 1, e, p])
                if a == 0.0:
                    continue
                R = O.decode_projection(w.residual(st, e, p), int(spec.residual_K[st - 1]), O.MCG)
                if mode == "exact":
                    W = W + a * R
                else:
                    W = W + f16(f16(R) * f16(a * c)) / c
            cache[key] = W
        return cache[key]

    model = _dense_moe(w, lambda e, p: dense(e, p, "model"), tokens)
    exact = _dense_moe(w, lambda e, p: dense(e, p, "exact"), tokens)
    base = _dense_moe(w, lambda e, p: dense(e, p, "base"), tokens)
    assert_close_linear(gpu[tokens], model, "f16", "prefill additive vs its rounding model")
    dev = np.linalg.norm(model - exact)
    contrib = np.linalg.norm(exact - base)
    assert contrib > 0.05 * np.linalg.norm(exact), "residual stages too small to test"
    assert dev <= 2.0 ** -8 * contrib, (dev, contrib)
    assert np.max(np.abs(model - exact)) <= 2.0 ** -8 * np.max(np.abs(exact - base)) + 1e-6


# --------------------------------------------------------------------------- contracts
def test_host_contract_violation_writes_nothing():
    import ctypes
    w = MoEWorkload(config(0))
    s = w.spec
    x, ids, rw = moe_inputs(w)
    out = torch.full((s.M, s.hidden), 3.0, dtype=torch.float16, device="cuda")
    nbytes = X.exl3_moe_workspace_bytes(s.M, s.topk, s.E, s.hidden, s.inter, 4)
    ws = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device="cuda")
    ex = _experts(0)
    st = ex.struct()
    lib = X.binding.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(act=0, hidden=s.hidden, E=s.E, topk=s.topk, cap=4, wsb=nbytes, ids_dt=3, xp=None):
        return lib.exl3_moe_forward(xp if xp is not None else x.data_ptr(), act, s.M, hidden,
                                    s.inter, E, topk, ids.data_ptr(), ids_dt, rw.data_ptr(), 0,
                                    ctypes.byref(st), cap, ws.data_ptr(), wsb, out.data_ptr(),
                                    stream)
    assert call(wsb=nbytes - 1) == -6          # workspace short
    assert call(act=7) == -3                   # unknown dtype
    assert call(ids_dt=2) == -3                # float ids
    assert call(hidden=500) == -4              # not a multiple of 128
    assert call(cap=0) == -7                   # capacity
    assert call(topk=9) == -7                  # topk > E
    assert call(E=2000) == -7                  # too many experts
    assert call(xp=x.data_ptr() + 2) == -5     # misaligned activations
    assert call(xp=0) == -1                    # null
    host = torch.zeros(16, dtype=torch.float16).pin_memory()
    assert call(xp=host.data_ptr()) == -2      # host memory
    torch.cuda.synchronize()
    assert torch.all(out == 3.0) and torch.all(ws == 0x5A)


def test_device_detected_bad_route_zero_fills_output():
    w = MoEWorkload(config(0))
    s = w.spec
    w.ids[3, 1] = s.E + 4
    x, ids, rw = moe_inputs(w)
    out = torch.full((s.M, s.hidden), 3.0, dtype=torch.float16, device="cuda")
    ws = torch.empty(X.exl3_moe_workspace_bytes(s.M, s.topk, s.E, s.hidden, s.inter, 4),
                     dtype=torch.uint8, device="cuda")
    X.exl3_moe_forward(x, ids, rw, _experts(0), 4, ws, out)
    torch.cuda.synchronize()
    assert X.exl3_workspace_error(ws) & X.binding.DERR_ROUTE_ID
    assert torch.all(out == 0)


def test_empty_batch_is_a_no_op():
    # M = 0 (valid pointers, nothing to compute): every entry point returns OK
    # and writes neither the output nor the workspace
    import ctypes
    w = MoEWorkload(config(0))
    s = w.spec
    x, ids, rw = moe_inputs(w)
    ex = _experts(0)
    st = ex.struct()
    out = torch.full((s.M, s.hidden), 3.0, dtype=torch.float16, device="cuda")
    nbytes = X.exl3_moe_workspace_bytes(16, s.topk, s.E, s.hidden, s.inter, s.capacity)
    ws = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device="cuda")
    lib = X.binding.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.exl3_moe_forward(x.data_ptr(), 0, 0, s.hidden, s.inter, s.E, s.topk, ids.data_ptr(),
                              3, rw.data_ptr(), 0, ctypes.byref(st), s.capacity, ws.data_ptr(),
                              nbytes, out.data_ptr(), stream)
    assert rc == 0
    lw = LinearWorkload(M=4, in_f=256, out_f=128, K=3, cb=CB_MCG, act="f16", seed=5)
    dp = X.DeviceProjection(lw.proj)
    ps = dp.struct()
    xl = to_device(lw.x, lw.act)
    y = torch.full((4, 128), 3.0, dtype=torch.float16, device="cuda")
    lws = torch.full((X.exl3_linear_workspace_bytes(4, 256, 128),), 0x5A, dtype=torch.uint8,
                     device="cuda")
    rc = lib.exl3_linear(xl.data_ptr(), 0, 0, ctypes.byref(ps), y.data_ptr(), lws.data_ptr(),
                         lws.numel(), stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.all(out == 3.0) and torch.all(ws == 0x5A)
    assert torch.all(y == 3.0) and torch.all(lws == 0x5A)
