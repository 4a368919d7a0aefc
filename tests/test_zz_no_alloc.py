"""exl3_linear_noalloc (for callers that cannot allocate device memory) gives
the same result as exl3_linear with a caller workspace, call after call, using
only the library's fixed device scratch.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import trellis_quantized_moe_gb300 as X  # noqa: E402
from workloads import CB_MCG, CB_MUL1, LinearWorkload  # noqa: E402
from gpu_common import assert_close_linear, to_device, to_f64  # noqa: E402


def _noalloc():
    lib = X.binding.lib()
    f = lib.exl3_linear_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                  ctypes.POINTER(X.binding.exl3_proj), ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    lib.exl3_linear_noalloc_max_scratch_bytes.restype = ctypes.c_size_t
    return f, lib.exl3_linear_noalloc_max_scratch_bytes()


def _noalloc_error(stream):
    lib = X.binding.lib()
    g = lib.exl3_linear_noalloc_error
    g.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]
    g.restype = ctypes.c_int
    err = ctypes.c_int32(-1)
    assert g(ctypes.byref(err), stream) == 0
    return err.value


def _with_workspace(lw, dp, x):
    y = torch.empty((lw.M, lw.proj.out_features), dtype=x.dtype, device="cuda")
    ws = torch.empty(X.exl3_linear_workspace_bytes(lw.M, lw.proj.in_features,
                                                    lw.proj.out_features),
                     dtype=torch.uint8, device="cuda")
    X.exl3_linear(x, dp, y, ws)
    return y


@pytest.mark.parametrize("Ms", [(7, 3), (300, 256)])
def test_noalloc_linear_matches_the_workspace_linear_on_consecutive_calls(Ms):
    # (7, 3): the decode-regime kernel; (300, 256): prompt-sized rows, the
    # tcgen05 kernel, whose activation tensor maps then point into the scratch
    f, cap = _noalloc()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [LinearWorkload(M=Ms[0], in_f=1408, out_f=4096, K=4, cb=CB_MCG, act="bf16", seed=31),
             LinearWorkload(M=Ms[1], in_f=1408, out_f=4096, K=4, cb=CB_MCG, act="bf16", seed=32)]
    cases[1].proj = cases[0].proj                  # same weights, new rows
    dp = X.DeviceProjection(cases[0].proj)
    st = dp.struct()
    for lw in cases:                               # two calls in a row
        assert X.exl3_linear_workspace_bytes(lw.M, 1408, 4096) <= cap
        x = to_device(lw.x, lw.act)
        ref = _with_workspace(lw, dp, x)
        y = torch.full_like(ref, float("nan"))
        rc = f(x.data_ptr(), X.EXL3_BF16, lw.M, ctypes.byref(st), y.data_ptr(), stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert _noalloc_error(stream) == 0
        assert_close_linear(to_f64(y), to_f64(ref), "bf16", "noalloc vs workspace")
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


def test_noalloc_linear_rejects_sizes_beyond_its_scratch():
    f, cap = _noalloc()
    lw = LinearWorkload(M=4, in_f=256, out_f=128, K=2, cb=CB_MUL1, act="f16", seed=5)
    dp = X.DeviceProjection(lw.proj)
    st = dp.struct()
    big_m = 1
    while X.exl3_linear_workspace_bytes(big_m, 256, 128) <= cap:
        big_m *= 2
    x = torch.zeros((big_m, 256), dtype=torch.float16, device="cuda")
    y = torch.full((big_m, 128), 7.0, dtype=torch.float16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert f(x.data_ptr(), X.EXL3_F16, big_m, ctypes.byref(st), y.data_ptr(), stream) == -6
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
