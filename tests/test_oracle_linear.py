"""Pins for the oracle's rotations and linear (exllamav3 #284 "API contract":
suh/svh rotations; TensorFold #837 "What this changes": the EXL3 linear)."""

import math

import numpy as np
import pytest
import scipy.linalg

from oracle import exl3_oracle as O
from workloads import make_projection, CB_MCG, CB_MUL1, CB_3INST


def test_hadamard_is_sylvester_and_orthonormal():
    H = O.hadamard(128)
    assert np.array_equal(H * math.sqrt(128), scipy.linalg.hadamard(128).astype(float))
    assert np.allclose(H @ H, np.eye(128), atol=1e-13)
    assert np.array_equal(H, H.T)


def test_block_hadamard_is_block_diagonal():
    a = np.random.default_rng(0).standard_normal((3, 384))
    H = scipy.linalg.block_diag(*([scipy.linalg.hadamard(128) / math.sqrt(128)] * 3))
    assert np.allclose(O.block_hadamard_rows(a), a @ H, atol=1e-12)


@pytest.mark.parametrize("cb,K", [(CB_MCG, 3), (CB_MUL1, 5), (CB_3INST, 8)])
def test_rotation_form_equals_dense_dequantised_matmul(cb, K):
    p = make_projection([9, cb, K], 256, 384, K, cb)
    x = np.random.default_rng(1).standard_normal((5, 256))
    y = O.linear(x, p)
    y_dense = x @ O.dense_matrix(p)
    assert y.shape == (5, 384)
    assert np.allclose(y, y_dense, rtol=1e-11, atol=1e-11)


def test_linear_brute_force_loops():
    """Pure-Python sums with H[i][j] = (-1)^popcount(i & j) / sqrt(128)."""
    p = make_projection([10], 128, 128, 2, CB_MCG)
    W = O.decode_projection(p.trellis, 2, CB_MCG)
    x = np.random.default_rng(2).standard_normal((2, 128))
    y = O.linear(x, p)
    r = 1 / math.sqrt(128)
    h = [[(-1) ** bin(i & j).count("1") * r for j in range(128)] for i in range(128)]
    suh, svh, sc = (v.astype(float) for v in (p.suh, p.svh, p.scale))
    for m in range(2):
        a = [sum(x[m, i] * suh[i] * h[i][k] for i in range(128)) for k in range(128)]
        z = [sum(a[k] * W[k, n] for k in range(128)) for n in range(128)]
        for o in range(0, 128, 17):
            yo = sum(z[n] * h[n][o] for n in range(128)) * svh[o] * sc[o]
            assert abs(yo - y[m, o]) < 1e-10


def test_unit_rotations_reduce_to_hadamard_sandwich():
    p = make_projection([11], 128, 256, 4, CB_MCG)
    p.suh[:] = 1
    p.svh[:] = 1
    p.scale[:] = 1
    W = O.decode_projection(p.trellis, 4, CB_MCG)
    H = scipy.linalg.hadamard(128) / math.sqrt(128)
    Hout = scipy.linalg.block_diag(H, H)
    x = np.eye(128)[:3]
    assert np.allclose(O.linear(x, p), H[:3] @ W @ Hout, atol=1e-12)


def test_scale_and_svh_apply_per_output_channel():
    p = make_projection([12], 128, 128, 3, CB_MCG)
    x = np.random.default_rng(3).standard_normal((2, 128))
    y = O.linear(x, p)
    q = make_projection([12], 128, 128, 3, CB_MCG)
    q.scale = (q.scale.astype(np.float64) * 2).astype(np.float16)
    q.svh[5] = -q.svh[5]
    y2 = O.linear(x, q)
    ratio = y2 / y
    expect = np.full(128, 2.0)
    expect[5] = -2.0
    assert np.allclose(ratio, expect[None, :], rtol=1e-12)
