"""Thin ctypes binding of the C ABI in include/exl3.h.

Functions keep the C names and only marshal arguments (torch tensors -> device
pointers, torch streams -> cudaStream_t).  Every step of the layer runs in the
CUDA library; if it is not built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libexl3_gb300.so")

EXL3_F16, EXL3_BF16, EXL3_F32, EXL3_I32, EXL3_I64 = 0, 1, 2, 3, 4
EXL3_CB_MUL1, EXL3_CB_MCG, EXL3_CB_3INST = 0, 1, 2
STATUS = {0: "OK", -1: "E_NULL", -2: "E_DEVICE", -3: "E_DTYPE", -4: "E_SHAPE", -5: "E_ALIGN",
          -6: "E_WORKSPACE", -7: "E_ROUTING", -8: "E_CODEBOOK", -9: "E_CUDA"}
DERR_ROUTE_ID, DERR_TABLE, DERR_TIMEOUT = 1, 2, 4

_DTYPE = {torch.float16: EXL3_F16, torch.bfloat16: EXL3_BF16, torch.float32: EXL3_F32,
          torch.int32: EXL3_I32, torch.int64: EXL3_I64}


class Exl3Error(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {code} ({STATUS.get(code, '?')})")
        self.code = code


class exl3_proj(ctypes.Structure):
    _fields_ = [("trellis", ctypes.c_void_p), ("suh", ctypes.c_void_p),
                ("svh", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("in_features", ctypes.c_int32), ("out_features", ctypes.c_int32),
                ("K", ctypes.c_int32), ("codebook", ctypes.c_int32)]


class exl3_experts(ctypes.Structure):
    _fields_ = [("trellis", ctypes.c_void_p), ("suh", ctypes.c_void_p),
                ("svh", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("K", ctypes.c_void_p), ("codebook", ctypes.c_void_p)]


class exl3_stages(ctypes.Structure):
    _fields_ = [("num_stages", ctypes.c_int32), ("trellis", ctypes.c_void_p),
                ("scale", ctypes.c_void_p), ("K", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() "
                          "(the library has no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    V, I, Z, P = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.POINTER
    lib.exl3_abi_version.restype = I
    lib.exl3_moe_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.exl3_moe_workspace_bytes.restype = Z
    lib.exl3_linear_workspace_bytes.argtypes = [I, I, I]
    lib.exl3_linear_workspace_bytes.restype = Z
    lib.exl3_route_pack_max_tiles.argtypes = [I, I, I, I]
    lib.exl3_route_pack_max_tiles.restype = I
    lib.exl3_route_pack.argtypes = [V, I, I, I, I, I, V, V, V, V, V]
    lib.exl3_route_pack.restype = I
    lib.exl3_linear.argtypes = [V, I, I, P(exl3_proj), V, V, Z, V]
    lib.exl3_linear.restype = I
    lib.exl3_moe_forward.argtypes = [V, I, I, I, I, I, I, V, I, V, I, P(exl3_experts), I, V, Z, V, V]
    lib.exl3_moe_forward.restype = I
    lib.exl3_moe_additive.argtypes = [V, I, I, I, I, I, I, V, I, V, I, P(exl3_experts),
                                      P(exl3_stages), I, V, Z, V, V]
    lib.exl3_moe_additive.restype = I
    lib.exl3_profile_events.argtypes = [V]
    lib.exl3_profile_events.restype = I
    lib.exl3_workspace_error.argtypes = [V, P(ctypes.c_int32), V]
    lib.exl3_workspace_error.restype = I
    return lib


_lib = _load()
EXPORTED = ["exl3_abi_version", "exl3_moe_workspace_bytes", "exl3_linear_workspace_bytes",
            "exl3_route_pack_max_tiles", "exl3_route_pack", "exl3_linear", "exl3_moe_forward",
            "exl3_moe_additive", "exl3_profile_events", "exl3_workspace_error"]


def lib():
    return _lib


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(fn, rc, raise_on_error):
    if rc != 0 and raise_on_error:
        raise Exl3Error(fn, rc)
    return rc


# --------------------------------------------------------------------------- sizes
def exl3_abi_version() -> int:
    return _lib.exl3_abi_version()


def exl3_moe_workspace_bytes(M, topk, E, hidden, inter, capacity) -> int:
    return _lib.exl3_moe_workspace_bytes(M, topk, E, hidden, inter, capacity)


def exl3_linear_workspace_bytes(M, in_features, out_features) -> int:
    return _lib.exl3_linear_workspace_bytes(M, in_features, out_features)


def exl3_route_pack_max_tiles(M, topk, E, capacity) -> int:
    return _lib.exl3_route_pack_max_tiles(M, topk, E, capacity)


# --------------------------------------------------------------------------- device weights
def _to_dev(a: np.ndarray, device) -> torch.Tensor:
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    elif a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DeviceProjection:
    """One projection in device memory (from a workloads.Projection)."""

    def __init__(self, proj, device="cuda"):
        self.trellis = _to_dev(proj.trellis.reshape(-1), device)
        self.suh = _to_dev(proj.suh, device)
        self.svh = _to_dev(proj.svh, device)
        self.scale = _to_dev(proj.scale, device)
        self.K, self.codebook = int(proj.K), int(proj.codebook)
        self.in_features, self.out_features = proj.in_features, proj.out_features

    def struct(self) -> exl3_proj:
        return exl3_proj(self.trellis.data_ptr(), self.suh.data_ptr(), self.svh.data_ptr(),
                         self.scale.data_ptr(), self.in_features, self.out_features, self.K,
                         self.codebook)


class DeviceExperts:
    """All experts of a layer: one trellis arena, one fp16 vector arena and the
    int64 pointer / int32 width and codebook tables of exl3_experts.

    get_proj(e, p) returns a workloads.Projection; K_of(e, p) its width (used to
    size the arena before any projection is generated)."""

    def __init__(self, get_proj, E, hidden, inter, K_of, device="cuda"):
        shape = {0: (hidden, inter), 1: (hidden, inter), 2: (inter, hidden)}
        words = [[(shape[p][0] // 16) * (shape[p][1] // 16) * 8 * int(K_of(e, p))
                  for p in range(3)] for e in range(E)]
        host = np.empty(sum(sum(r) for r in words), np.uint32)
        vec = np.empty(E * (2 * (2 * hidden + 2 * inter) + 2 * hidden + inter), np.float16)
        toff, voff, Ks, cbs = [], [], [], []
        o = v = 0
        for e in range(E):
            for p in range(3):
                pr = get_proj(e, p)
                n = pr.trellis.size
                assert n == words[e][p] and (pr.in_features, pr.out_features) == shape[p]
                host[o:o + n] = pr.trellis.reshape(-1)
                toff.append(o)
                o += n
                offs = []
                for arr in (pr.suh, pr.svh, pr.scale):
                    vec[v:v + arr.size] = arr
                    offs.append(v)
                    v += arr.size
                voff.append(offs)
                Ks.append(pr.K)
                cbs.append(pr.codebook)
        self.arena = _to_dev(host, device)
        self.vectors = torch.from_numpy(vec[:v]).to(device)
        base, vb = self.arena.data_ptr(), self.vectors.data_ptr()
        i64 = dict(dtype=torch.int64, device=device)
        self.t_trellis = torch.tensor([base + 4 * x for x in toff], **i64)
        self.t_suh = torch.tensor([vb + 2 * x[0] for x in voff], **i64)
        self.t_svh = torch.tensor([vb + 2 * x[1] for x in voff], **i64)
        self.t_scale = torch.tensor([vb + 2 * x[2] for x in voff], **i64)
        self.t_K = torch.tensor(Ks, dtype=torch.int32, device=device)
        self.t_cb = torch.tensor(cbs, dtype=torch.int32, device=device)
        self.E, self.hidden, self.inter = E, hidden, inter
        self.trellis_words = [w for r in words for w in r]

    @classmethod
    def from_workload(cls, w, device="cuda"):
        s = w.spec
        return cls(w.projection, s.E, s.hidden, s.inter, lambda e, p: s.K[e], device)

    def struct(self) -> exl3_experts:
        return exl3_experts(self.t_trellis.data_ptr(), self.t_suh.data_ptr(),
                            self.t_svh.data_ptr(), self.t_scale.data_ptr(),
                            self.t_K.data_ptr(), self.t_cb.data_ptr())


class DeviceStages:
    """Stage-major residual tables of exl3_stages (stages 1..S-1)."""

    def __init__(self, get_residual, alpha: np.ndarray, Ks, E, device="cuda"):
        nres = alpha.shape[0]
        self.num_stages = 1 + nres
        arrays, ptr_index = [], []
        for s in range(nres):
            for e in range(E):
                for p in range(3):
                    t = get_residual(s + 1, e, p)
                    ptr_index.append(None if t is None else len(arrays))
                    if t is not None:
                        arrays.append(t.reshape(-1))
        total = sum(a.size for a in arrays)
        host = np.empty(max(total, 4), np.uint32)
        offs, o = [], 0
        for a in arrays:
            host[o:o + a.size] = a
            offs.append(o)
            o += a.size
        self.arena = _to_dev(host, device)
        base = self.arena.data_ptr()
        ptrs = [0 if i is None else base + 4 * offs[i] for i in ptr_index]
        self.t_trellis = torch.tensor(ptrs, dtype=torch.int64, device=device)
        self.t_scale = torch.from_numpy(np.ascontiguousarray(alpha, np.float32).reshape(-1)).to(device)
        self.t_K = torch.tensor(np.repeat(np.asarray(Ks, np.int32), E * 3), device=device)
        self.trellis_bytes = 4 * total

    def struct(self) -> exl3_stages:
        return exl3_stages(self.num_stages, self.t_trellis.data_ptr(), self.t_scale.data_ptr(),
                           self.t_K.data_ptr())


# --------------------------------------------------------------------------- entry points
def exl3_route_pack(ids, E, capacity, offsets, packed, tiles, info, stream=None,
                    raise_on_error=True) -> int:
    M, topk = ids.shape
    rc = _lib.exl3_route_pack(_ptr(ids), _DTYPE[ids.dtype], M, topk, E, capacity, _ptr(offsets),
                              _ptr(packed), _ptr(tiles), _ptr(info), _stream(stream))
    return _check("exl3_route_pack", rc, raise_on_error)


def exl3_linear(x, proj: DeviceProjection, y, workspace, stream=None, raise_on_error=True) -> int:
    st = proj.struct()
    rc = _lib.exl3_linear(_ptr(x), _DTYPE[x.dtype], x.shape[0], ctypes.byref(st), _ptr(y),
                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                          _stream(stream))
    return _check("exl3_linear", rc, raise_on_error)


def exl3_moe_forward(x, ids, rw, experts: DeviceExperts, capacity, workspace, out, stream=None,
                     raise_on_error=True) -> int:
    st = experts.struct()
    M, topk = ids.shape
    rc = _lib.exl3_moe_forward(_ptr(x), _DTYPE[x.dtype], M, experts.hidden, experts.inter,
                               experts.E, topk, _ptr(ids), _DTYPE[ids.dtype], _ptr(rw),
                               _DTYPE[rw.dtype], ctypes.byref(st), capacity, _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _ptr(out),
                               _stream(stream))
    return _check("exl3_moe_forward", rc, raise_on_error)


def exl3_moe_additive(x, ids, rw, experts: DeviceExperts, stages: DeviceStages, capacity,
                      workspace, out, stream=None, raise_on_error=True) -> int:
    st = experts.struct()
    ss = stages.struct()
    M, topk = ids.shape
    rc = _lib.exl3_moe_additive(_ptr(x), _DTYPE[x.dtype], M, experts.hidden, experts.inter,
                                experts.E, topk, _ptr(ids), _DTYPE[ids.dtype], _ptr(rw),
                                _DTYPE[rw.dtype], ctypes.byref(st), ctypes.byref(ss), capacity,
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _ptr(out), _stream(stream))
    return _check("exl3_moe_additive", rc, raise_on_error)


class ProfileEvents:
    """Five torch CUDA events recorded between the fused layer's kernels
    (route pack | rotation | gate/up GEMM | down GEMM + combine)."""

    def __init__(self):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        for e in self.events:          # creates the underlying cudaEvent_t
            e.record()
        torch.cuda.synchronize()
        self._arr = (ctypes.c_void_p * 5)(*[ctypes.c_void_p(e.cuda_event) for e in self.events])

    def __enter__(self):
        _lib.exl3_profile_events(ctypes.cast(self._arr, ctypes.c_void_p))
        return self

    def __exit__(self, *exc):
        _lib.exl3_profile_events(None)

    def times_ms(self):
        """(route pack, rotation, gate/up, down + combine) in ms for the last call."""
        e = self.events
        return [e[i].elapsed_time(e[i + 1]) for i in range(4)]


def exl3_workspace_error(workspace, stream=None) -> int:
    err = ctypes.c_int32(0)
    rc = _lib.exl3_workspace_error(_ptr(workspace), ctypes.byref(err), _stream(stream))
    _check("exl3_workspace_error", rc, True)
    return int(err.value)
