"""Float64 CPU oracle for the fused EXL3 routed-expert MoE layer.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference legs of ``bench.py`` may import or run anything in
this directory.  It shares no code with the CUDA path and imports nothing from
the product package.  It is deliberately plain and slow.

What it computes (the pages name the method but never print the trellis math;
every constant or layout they leave open is fixed here once, as a reading):

* Trellis tiles -- "EXL3 linear and grouped routed experts" (TensorFold #837),
  "What this changes": 16x16 tiles of K-bit codes, K = 1..8, decoded by the
  codebooks mul1, mcg and 3inst.
  Readings: a tile's 256*K bits are stored as 8*K little-endian 32-bit words and
  read most significant bit first; the state of position p is the 16-bit window
  of the cyclic bit string that ends at bit (p+1)*K - 1 (the 16-bit bitshift
  trellis of QTIP, Tseng et al. 2024, tail-biting); position p sits at input
  row p mod 16 and output column p div 16 of its tile; tiles are stored
  [in/16][out/16].
* Codebooks (reading; constants not on the pages): 3inst is QTIP's published
  3INST (x = a*s + b mod 2^32, mask/xor, sum of the two fp16 halves); mcg is the
  same without the increment and with an odd multiplier; mul1 multiplies and
  sums the four bytes, centred and scaled to unit variance.
* Rotations -- "MoE: Add fused additive EXL3 kernels" (exllamav3 #284),
  "API contract" (suh/svh rotations): a' = Hb(a * suh), y = Hb(z) * svh * scale,
  Hb the block-diagonal 128-point Sylvester Hadamard scaled by 1/sqrt(128)
  (reading: block size and normalisation are not on the pages).
* Grouped experts -- TensorFold #837, "What this changes": per expert, gate and
  up, SwiGLU, down, and the route-weighted combine.
* Route packing -- exllamav3 #284, "Summary" and "Relationship to #246": route
  histogram, exclusive scan, stable packing; oversized spans tiled by capacity.
* Additive residual stages -- exllamav3 #284, "Summary" and "API contract":
  stage-major residual trellises in the mcg codebook reusing the base
  projection's suh/svh; a zero scale skips the stage.

Parity unpinned: that these codebook constants and this bit layout equal
ExLlamaV3's own (no checkpoint or printed decoded value exists to compare
with).  Everything else is pinned by tests/test_oracle_*.py.
"""

from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

MUL1, MCG, INST3 = 0, 1, 2

# 3INST constants as published with QTIP; mcg / mul1 multipliers are readings.
A_3INST = 89226354
B_3INST = 64248484
A_MCG = 0xCBAC1FED
A_MUL1 = 0x83DCD12D
HALF_MASK = 0x8FFF8FFF
HALF_XOR = 0x3B603B60
MUL1_MEAN = 510.0                  # mean of a sum of four uniform bytes
MUL1_STD = math.sqrt(21845.0)      # sd of that sum: sqrt(4 * (256^2 - 1) / 12)
HB = 128                           # Hadamard block (reading)

_U32 = np.uint64(0xFFFFFFFF)


# ----------------------------------------------------------------------------
# Trellis states (TensorFold #837, "What this changes": the trellis decode)
# ----------------------------------------------------------------------------

def tile_bits(words: np.ndarray, K: int) -> np.ndarray:
    """Bit string of tiles: [..., 8K] uint32 words -> [..., 256K] bits, MSB first."""
    words = np.asarray(words, dtype=np.uint64)
    assert words.shape[-1] == 8 * K
    b = np.arange(256 * K)
    shift = (31 - (b % 32)).astype(np.uint64)
    return (words[..., b // 32] >> shift) & np.uint64(1)


def tile_states(words: np.ndarray, K: int) -> np.ndarray:
    """States s_p, p = 0..255: the 16 bits ending at bit (p+1)K-1, cyclic, MSB first."""
    bits = tile_bits(words, K)
    nbits = 256 * K
    p = np.arange(256)
    window = ((p[:, None] + 1) * K - 16 + np.arange(16)[None, :]) % nbits   # [256, 16]
    place = (np.uint64(1) << (15 - np.arange(16)).astype(np.uint64))
    return (bits[..., window] * place).sum(axis=-1).astype(np.int64)


# ----------------------------------------------------------------------------
# Codebooks (TensorFold #837, "What this changes": mul1, mcg, 3inst)
# ----------------------------------------------------------------------------

def _f16_bits_to_f64(h: np.ndarray) -> np.ndarray:
    return np.asarray(h, dtype=np.uint16).view(np.float16).astype(np.float64)


def codebook_halves(states: np.ndarray, cb: int):
    """For mcg/3inst: the two fp16 halves (low, high) of the masked product."""
    s = np.asarray(states, dtype=np.uint64)
    if cb == MCG:
        x = (np.uint64(A_MCG) * s) & _U32
    elif cb == INST3:
        x = (np.uint64(A_3INST) * s + np.uint64(B_3INST)) & _U32
    else:
        raise ValueError("halves exist for mcg and 3inst only")
    x = (x & np.uint64(HALF_MASK)) ^ np.uint64(HALF_XOR)
    lo = _f16_bits_to_f64((x & np.uint64(0xFFFF)).astype(np.uint16))
    hi = _f16_bits_to_f64((x >> np.uint64(16)).astype(np.uint16))
    return lo, hi


def codebook_values(states: np.ndarray, cb: int) -> np.ndarray:
    """Decoded weight of each 16-bit state, exact in float64."""
    if cb == MUL1:
        s = np.asarray(states, dtype=np.uint64)
        x = (np.uint64(A_MUL1) * s) & _U32
        byte_sum = sum(((x >> np.uint64(8 * i)) & np.uint64(0xFF)).astype(np.float64)
                       for i in range(4))
        return (byte_sum - MUL1_MEAN) / MUL1_STD
    lo, hi = codebook_halves(states, cb)
    return lo + hi


# ----------------------------------------------------------------------------
# Projection decode
# ----------------------------------------------------------------------------

def decode_projection_numpy(trellis: np.ndarray, K: int, cb: int,
                            batch: int = 1024) -> np.ndarray:
    """Dense weights W[in, out] of one projection, numpy path."""
    ntk, ntn, nw = trellis.shape
    assert nw == 8 * K
    flat = trellis.reshape(ntk * ntn, nw)
    vals = np.empty((ntk * ntn, 256), np.float64)
    for i in range(0, flat.shape[0], batch):
        vals[i:i + batch] = codebook_values(tile_states(flat[i:i + batch], K), cb)
    # position p -> (row r = p % 16, col c = p // 16)
    v = vals.reshape(ntk, ntn, 16, 16)          # [tk, tn, c, r]
    return v.transpose(0, 3, 1, 2).reshape(ntk * 16, ntn * 16)


_lib = None
_lib_lock = threading.Lock()
_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")


def build_c_oracle(force: bool = False) -> str:
    """Compile the C decoder (plain C, float64, OpenMP) next to this file."""
    src = os.path.join(_HERE, "exl3_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def c_oracle():
    global _lib
    with _lib_lock:
        if _lib is None:
            lib = ctypes.CDLL(build_c_oracle())
            lib.oracle_decode_projection.argtypes = [
                ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_void_p]
            lib.oracle_decode_projection.restype = ctypes.c_int
            lib.oracle_tile_states.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
            lib.oracle_tile_states.restype = None
            lib.oracle_codebook.argtypes = [ctypes.c_uint32, ctypes.c_int]
            lib.oracle_codebook.restype = ctypes.c_double
            lib.oracle_threads.argtypes = []
            lib.oracle_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def decode_projection_c(trellis: np.ndarray, K: int, cb: int) -> np.ndarray:
    t = np.ascontiguousarray(trellis, dtype=np.uint32)
    ntk, ntn, nw = t.shape
    assert nw == 8 * K
    W = np.empty((ntk * 16, ntn * 16), np.float64)
    rc = c_oracle().oracle_decode_projection(t.ctypes.data, ntk * 16, ntn * 16, K, cb,
                                             W.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle decode rejected K={K} cb={cb}")
    return W


def decode_projection(trellis: np.ndarray, K: int, cb: int, impl: str = "c") -> np.ndarray:
    if impl == "numpy":
        return decode_projection_numpy(trellis, K, cb)
    return decode_projection_c(trellis, K, cb)


def oracle_threads() -> int:
    return int(c_oracle().oracle_threads())


# ----------------------------------------------------------------------------
# Rotations (exllamav3 #284, "API contract": suh/svh; TensorFold #837: input rotation)
# ----------------------------------------------------------------------------

def hadamard(n: int = HB) -> np.ndarray:
    """Sylvester Hadamard matrix of order n (power of two), scaled to be orthonormal."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    assert h.shape[0] == n
    return h / math.sqrt(n)


def block_hadamard_rows(a: np.ndarray) -> np.ndarray:
    """Apply Hb (block-diagonal, 128-blocks) to each row vector of a."""
    a = np.asarray(a, np.float64)
    n = a.shape[-1]
    assert n % HB == 0
    H = hadamard(HB)
    return (a.reshape(*a.shape[:-1], n // HB, HB) @ H).reshape(a.shape)


def rotate_in(a: np.ndarray, suh: np.ndarray) -> np.ndarray:
    return block_hadamard_rows(np.asarray(a, np.float64) * suh.astype(np.float64))


def rotate_out(z: np.ndarray, svh: np.ndarray, scale: np.ndarray) -> np.ndarray:
    return block_hadamard_rows(z) * svh.astype(np.float64) * scale.astype(np.float64)


# ----------------------------------------------------------------------------
# Linear (TensorFold #837, "What this changes": the EXL3 linear)
# ----------------------------------------------------------------------------

def linear_from_dense(a: np.ndarray, W: np.ndarray, suh, svh, scale) -> np.ndarray:
    """y = Hb( Hb(a * suh) @ W ) * svh * scale for row vectors a."""
    return rotate_out(rotate_in(a, suh) @ W, svh, scale)


def linear(a: np.ndarray, proj, impl: str = "c", residuals=()) -> np.ndarray:
    """One projection.  ``residuals`` = [(alpha, trellis, K)], mcg, base rotations."""
    W = decode_projection(proj.trellis, proj.K, proj.codebook, impl)
    for alpha, trellis, K in residuals:
        if alpha != 0.0:
            W = W + float(alpha) * decode_projection(trellis, K, MCG, impl)
    return linear_from_dense(a, W, proj.suh, proj.svh, proj.scale)


def dense_matrix(proj, impl: str = "c") -> np.ndarray:
    """The equivalent dense matrix diag(suh) Hb W Hb diag(svh * scale)."""
    W = decode_projection(proj.trellis, proj.K, proj.codebook, impl)
    n_in, n_out = W.shape
    Hin = np.kron(np.eye(n_in // HB), hadamard(HB))
    Hout = np.kron(np.eye(n_out // HB), hadamard(HB))
    return (np.diag(proj.suh.astype(np.float64)) @ Hin @ W @ Hout
            @ np.diag(proj.svh.astype(np.float64) * proj.scale.astype(np.float64)))


# ----------------------------------------------------------------------------
# Routing (exllamav3 #284, "Summary": stable route packing, span tiling)
# ----------------------------------------------------------------------------

def route_pack(ids: np.ndarray, E: int, capacity: int):
    """Histogram, exclusive scan and stable packing of flat routes f = t*topk + j.

    Returns (offsets[E+1], packed[R], tiles[n][3] = (expert, start, length),
    num_active).  Raises ValueError on an id outside [0, E).
    """
    flat = np.asarray(ids).reshape(-1).astype(np.int64)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("route id out of range")
    counts = np.zeros(E, np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    packed = np.empty(flat.size, np.int64)
    cursor = offsets[:-1].copy()
    for f, e in enumerate(flat):
        packed[cursor[e]] = f
        cursor[e] += 1
    tiles = []
    for e in range(E):
        start = 0
        while start < counts[e]:
            n = min(capacity, counts[e] - start)
            tiles.append((e, offsets[e] + start, n))
            start += n
    num_active = int((counts > 0).sum())
    return offsets, packed, np.array(tiles, np.int64).reshape(-1, 3), num_active


# ----------------------------------------------------------------------------
# Grouped experts (TensorFold #837: gate and up, SwiGLU, down, weighted combine)
# ----------------------------------------------------------------------------

def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def moe_forward(x: np.ndarray, ids: np.ndarray, rw: np.ndarray, get_proj,
                tokens=None, impl: str = "c", get_residuals=None) -> np.ndarray:
    """out[t] = sum_j rw[t,j] * down_e(silu(gate_e(x_t)) * up_e(x_t)), e = ids[t,j].

    x, rw: float64 arrays [M, H], [M, topk].  get_proj(e, p) -> projection with
    trellis/suh/svh/scale/K/codebook, p in (0 gate, 1 up, 2 down).
    get_residuals(e, p) -> [(alpha, trellis, K)] additive mcg stages.
    tokens: optional subset of rows to evaluate (each row depends only on its
    own routes).  Returns float64 [len(tokens), H].
    """
    M, topk = ids.shape
    tokens = np.arange(M) if tokens is None else np.asarray(tokens)
    out = np.zeros((len(tokens), x.shape[1]), np.float64)
    by_expert = {}
    for i, t in enumerate(tokens):
        for j in range(topk):
            by_expert.setdefault(int(ids[t, j]), []).append((i, t, j))
    contrib = {}
    for e, members in sorted(by_expert.items()):
        rows = np.array([t for _, t, _ in members])
        res = (lambda p: get_residuals(e, p)) if get_residuals else (lambda p: ())
        g = linear(x[rows], get_proj(e, 0), impl, res(0))
        u = linear(x[rows], get_proj(e, 1), impl, res(1))
        d = linear(silu(g) * u, get_proj(e, 2), impl, res(2))
        for k, (i, t, j) in enumerate(members):
            contrib[(i, j)] = d[k]
    for i, t in enumerate(tokens):
        for j in range(topk):          # j ascending
            out[i] += float(rw[t, j]) * contrib[(i, j)]
    return out
