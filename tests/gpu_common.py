"""Helpers shared by the GPU parity tests: upload seeded workloads, run the CUDA
path through the C ABI, and compare with the float64 oracle."""
import numpy as np
import torch

from workloads import act_to_f64, rw_to_f64

REL_L2 = 2e-3     # layer tolerance: relative L2 to the float64 oracle
MAX_ABS = 1e-2    # and worst element

_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
          "i32": torch.int32, "i64": torch.int64}


def to_device(a: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16).copy()).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def assert_close(got: np.ndarray, ref: np.ndarray, act: str, what: str = ""):
    """Layer tolerance: rel-L2 <= 2e-3 and max-abs <= 1e-2 of the computed value
    before its final rounding to the activation dtype; on the stored output that
    reads |got - ref| <= 1e-2 + half an ulp of the output dtype at |got| (a
    correctly rounded exact result is itself up to half an ulp away)."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what
    r = rel_l2(got, ref)
    excess = np.abs(got - ref) - 0.5 * ulp(got, act)
    m = float(np.max(excess)) if got.size else 0.0
    mabs = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert r <= REL_L2 and m <= MAX_ABS, (
        f"{what}: rel_l2={r:.3e} max_abs={mabs:.3e} beyond half an output ulp={m:.3e}")
    return r, m


def ulp(ref: np.ndarray, act: str) -> np.ndarray:
    """One unit in the last place of the output dtype at |ref|."""
    mant = 7 if act == "bf16" else 10
    e = np.floor(np.log2(np.maximum(np.abs(ref), 1e-30)))
    return np.exp2(e - mant)


def assert_close_linear(got: np.ndarray, ref: np.ndarray, act: str, what: str = ""):
    """Tolerance for outputs of magnitude O(1): a single projection, or a test
    layer of 8 experts with top-2 routing.  rel-L2 <= 2e-3, and every element
    within one ulp of the output dtype at |ref| plus 1e-2 of the output RMS.

    The layer bound max-abs <= 1e-2 presumes outputs of the configs' size
    (|out| ~ 0.05).  At |y| in [2, 4) one bf16 ulp is 2^-6 = 0.0156, so the
    correctly rounded exact result alone can miss an absolute 1e-2 by half an
    ulp (0.0078) plus the fp32 accumulation error; the ulp term absorbs the
    final rounding and the RMS term is the layer bound's 1e-2 relative to the
    output scale.  Layer tests at the configs' scales use assert_close."""
    assert got.shape == ref.shape and np.all(np.isfinite(got)), what
    r = rel_l2(got, ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    excess = np.abs(got - ref) - ulp(ref, act)
    worst = float(np.max(excess)) / rms if got.size else 0.0
    assert r <= REL_L2 and worst <= MAX_ABS, f"{what}: rel_l2={r:.3e} worst/rms={worst:.3e}"
    return r, worst


def covering_tokens(w, n: int, seed: int = 0, cover: bool = True) -> np.ndarray:
    """At least n tokens of workload w, chosen so that every 256-route half of
    every capacity tile (the down items of the prefill regime), hence every
    tile of every multi-tile expert, holds at least one checked route, and so
    that the first and last tokens are checked; the rest are drawn at random
    (seeded).  Tokens are picked greedily by the number of uncovered halves
    they route into.  cover=False: first, last and random tokens only.
    Sorted, unique."""
    from oracle import exl3_oracle as O
    s = w.spec
    _, packed, tiles, _ = O.route_pack(w.ids, s.E, s.capacity)
    unit_of_route = np.empty(s.M * s.topk, np.int64)
    nunits = 0
    for _, start, ln in tiles:
        for h0 in range(0, ln, 256):
            unit_of_route[packed[start + h0:start + min(ln, h0 + 256)]] = nunits
            nunits += 1
    units = unit_of_route.reshape(s.M, s.topk)
    covered = np.zeros(nunits, bool)
    pick = [0, s.M - 1]
    covered[units[pick].ravel()] = True
    while cover and not covered.all():
        gain = (~covered[units]).sum(axis=1)
        t = int(np.argmax(gain))
        pick.append(t)
        covered[units[t]] = True
    rng = np.random.default_rng(seed)
    for t in rng.permutation(s.M):
        if len(set(pick)) >= n:
            break
        pick.append(int(t))
    return np.array(sorted(set(pick)), dtype=np.int64)


def moe_inputs(w):
    s = w.spec
    x = to_device(w.x, s.act)
    ids = to_device(w.ids, s.ids_dtype)
    rw = to_device(w.rw, s.rw_dtype)
    return x, ids, rw


def out_tensor(w):
    s = w.spec
    return torch.empty((s.M, s.hidden), dtype=_TORCH[s.act], device="cuda")


def oracle_rows(w, tokens=None, impl="c", residuals=True):
    from oracle import exl3_oracle as O
    s = w.spec
    get_res = None
    if residuals and len(s.residual_K):
        def get_res(e, p):
            out = []
            for st in range(1, s.num_stages):
                a = float(w.alpha[st - 1, e, p])
                if a != 0.0:
                    out.append((a, w.residual(st, e, p), int(s.residual_K[st - 1])))
            return out
    return O.moe_forward(act_to_f64(w.x, s.act), w.ids, rw_to_f64(w.rw, s.rw_dtype),
                         w.projection, tokens=tokens, impl=impl, get_residuals=get_res)
