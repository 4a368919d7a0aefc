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


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what
    r = rel_l2(got, ref)
    m = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert r <= REL_L2 and m <= MAX_ABS, f"{what}: rel_l2={r:.3e} max_abs={m:.3e}"
    return r, m


def ulp(ref: np.ndarray, act: str) -> np.ndarray:
    """One unit in the last place of the output dtype at |ref|."""
    mant = 7 if act == "bf16" else 10
    e = np.floor(np.log2(np.maximum(np.abs(ref), 1e-30)))
    return np.exp2(e - mant)


def assert_close_linear(got: np.ndarray, ref: np.ndarray, act: str, what: str = ""):
    """Single projection (outputs O(1), unlike the layer's O(0.05)): rel-L2 2e-3
    and a worst-element bound of one output ulp plus 1e-2 of the output RMS."""
    assert got.shape == ref.shape and np.all(np.isfinite(got)), what
    r = rel_l2(got, ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    excess = np.abs(got - ref) - ulp(ref, act)
    worst = float(np.max(excess)) / rms if got.size else 0.0
    assert r <= REL_L2 and worst <= MAX_ABS, f"{what}: rel_l2={r:.3e} worst/rms={worst:.3e}"
    return r, worst


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
