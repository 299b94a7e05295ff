"""Thin Python binding of libslimkv (ctypes): argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels; torch is used
for device memory and streams. The names follow ``include/slimkv.h``.
There is no CPU fallback: without the built library on a CUDA device every call
raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libslimkv.so")

SLIMKV_F32, SLIMKV_BF16 = 0, 1
SLIMKV_LATENT, SLIMKV_RECONSTRUCT, SLIMKV_FULL_KV, SLIMKV_PREFILL = 0, 1, 2, 3
STATUS = {0: "SLIMKV_OK", 1: "SLIMKV_ERR_NULL", 2: "SLIMKV_ERR_SHAPE", 3: "SLIMKV_ERR_DTYPE",
          4: "SLIMKV_ERR_ALIGN", 5: "SLIMKV_ERR_WORKSPACE", 6: "SLIMKV_ERR_CUDA",
          7: "SLIMKV_ERR_TOO_LARGE"}
NOALLOC_SCRATCH_BYTES = 64 << 20   # SLIMKV_NOALLOC_SCRATCH_BYTES

# every symbol include/slimkv.h declares
EXPORTS = ("slimkv_workspace_bytes", "slimkv_decode_attn", "slimkv_decode_attn_alibi", "slimkv_decode_attn_reconstruct",
           "slimkv_decode_attn_reconstruct_rope", "slimkv_decode_attn_full_kv", "slimkv_status_str", "slimkv_abi_version",
           "slimkv_kernel_path", "slimkv_force_simt", "slimkv_time_next_decode",
           "slimkv_decode_attn_noalloc", "slimkv_append_kv", "slimkv_prefill_attn",
           "slimkv_abort_count", "slimkv_test_withhold_first_load")


class SlimkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
                ("d", ctypes.c_int), ("N_b", ctypes.c_int), ("r_k", ctypes.c_int),
                ("r_v", ctypes.c_int), ("W", ctypes.c_int), ("scale", ctypes.c_float),
                ("rope_base", ctypes.c_double), ("dtype", ctypes.c_int)]


_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libslimkv.so (built in-tree by ``latent_kv_cache_decode_b300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libslimkv.so not built ({path}); run "
                           "`python -m latent_kv_cache_decode_b300.build`")
    lib = ctypes.CDLL(path)
    vp, sz, i32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p
    sp = ctypes.POINTER(Shape)
    lib.slimkv_workspace_bytes.argtypes = [sp, ctypes.c_int]
    lib.slimkv_workspace_bytes.restype = sz
    lib.slimkv_decode_attn.argtypes = [sp] + [vp] * 7 + [i32p, vp, vp, sz, vp]
    lib.slimkv_decode_attn.restype = ctypes.c_int
    lib.slimkv_decode_attn_reconstruct.argtypes = [sp] + [vp] * 7 + [i32p, vp, vp, sz, vp]
    lib.slimkv_decode_attn_reconstruct.restype = ctypes.c_int
    lib.slimkv_decode_attn_alibi.argtypes = [sp] + [vp] * 7 + [i32p, vp, ctypes.c_int, vp, vp, sz, vp]
    lib.slimkv_decode_attn_alibi.restype = ctypes.c_int
    lib.slimkv_decode_attn_reconstruct_rope.argtypes = [sp] + [vp] * 7 + [i32p, ctypes.c_int, vp, vp, sz, vp]
    lib.slimkv_decode_attn_reconstruct_rope.restype = ctypes.c_int
    lib.slimkv_decode_attn_full_kv.argtypes = [sp, vp, vp, vp, i32p, vp, vp, sz, vp]
    lib.slimkv_decode_attn_full_kv.restype = ctypes.c_int
    lib.slimkv_decode_attn_noalloc.argtypes = [sp] + [vp] * 7 + [i32p, vp, vp]
    lib.slimkv_decode_attn_noalloc.restype = ctypes.c_int
    lib.slimkv_append_kv.argtypes = [sp, vp, vp, vp, vp, i32p, vp]
    lib.slimkv_abort_count.restype = ctypes.c_longlong
    lib.slimkv_abort_count.argtypes = [ctypes.c_int]
    lib.slimkv_test_withhold_first_load.restype = None
    lib.slimkv_test_withhold_first_load.argtypes = [ctypes.c_int]
    lib.slimkv_prefill_attn.restype = ctypes.c_int
    lib.slimkv_prefill_attn.argtypes = [sp] + [vp] * 7 + [i32p, vp, vp, sz, vp]
    lib.slimkv_append_kv.restype = ctypes.c_int
    lib.slimkv_status_str.argtypes = [ctypes.c_int]
    lib.slimkv_status_str.restype = ctypes.c_char_p
    lib.slimkv_abi_version.argtypes = []
    lib.slimkv_abi_version.restype = ctypes.c_int
    lib.slimkv_kernel_path.argtypes = [sp, ctypes.c_int]
    lib.slimkv_kernel_path.restype = ctypes.c_int
    lib.slimkv_force_simt.argtypes = [ctypes.c_int]
    lib.slimkv_force_simt.restype = ctypes.c_int
    lib.slimkv_time_next_decode.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.slimkv_time_next_decode.restype = None
    _lib = lib
    return lib


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return SLIMKV_F32
    if t == torch.bfloat16:
        return SLIMKV_BF16
    raise TypeError(f"unsupported storage dtype {t}")


def make_shape(B, Hq, Hkv, d, N_b, r_k, r_v, W, dtype, scale=None, rope_base=10000.0) -> Shape:
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return Shape(B, Hq, Hkv, d, N_b, r_k, r_v, W, scale, rope_base, code)


_SHAPES: dict = {}


def _shape_and_bytes(which: int, B, Hq, Hkv, d, N_b, r_k, r_v, W, dtype, scale, rope_base):
    """(Shape, workspace bytes) for one argument signature, built once and reused:
    a decode step calls the library once per layer with the same few signatures."""
    key = (which, B, Hq, Hkv, d, N_b, r_k, r_v, W, dtype, scale, rope_base)
    hit = _SHAPES.get(key)
    if hit is None:
        sh = make_shape(B, Hq, Hkv, d, N_b, r_k, r_v, W, dtype, scale, rope_base)
        nb = int(load().slimkv_workspace_bytes(ctypes.byref(sh), which))
        if len(_SHAPES) > 1024:
            _SHAPES.clear()
        hit = _SHAPES[key] = (sh, nb)
    return hit


def workspace_bytes(shape: Shape, which: int) -> int:
    return int(load().slimkv_workspace_bytes(ctypes.byref(shape), which))


def kernel_path(shape: Shape, which: int) -> int:
    return int(load().slimkv_kernel_path(ctypes.byref(shape), which))


def force_simt(on: bool) -> bool:
    return bool(load().slimkv_force_simt(1 if on else 0))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on the CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(status: int, what: str):
    if status != 0:
        raise SlimkvError(status, what)


class Workspace:
    """A reusable device workspace (grows on demand)."""

    def __init__(self, device=None):
        self.device = device
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device or "cuda")
        return self.buf


def decode_attn(q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, *, scale=None, rope_base=10000.0,
                out=None, workspace: Optional[Workspace] = None, stream=None, shape=None):
    """slimkv_decode_attn on torch CUDA tensors; returns out [B,Hq,d] float32."""
    lib = load()
    B, Hq, d = q.shape
    N_b = C_K.shape[1] if C_K is not None else 0
    W = K_raw.shape[1] if K_raw is not None else 0
    Hkv = U_K.shape[0] // d if U_K is not None else K_raw.shape[2]
    r_k = C_K.shape[2] if C_K is not None else 0
    r_v = C_V.shape[2] if C_V is not None else 0
    if shape is not None:
        sh = shape
        nb = lib.slimkv_workspace_bytes(ctypes.byref(sh), SLIMKV_LATENT)
    else:
        sh, nb = _shape_and_bytes(SLIMKV_LATENT, B, Hq, Hkv, d, N_b, r_k, r_v, W, q.dtype, scale, rope_base)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    if nb == 0:
        _check(2, "slimkv_decode_attn")
    ws = (workspace or Workspace(q.device)).get(nb)
    st = lib.slimkv_decode_attn(ctypes.byref(sh), _ptr(q), _ptr(C_K), _ptr(C_V), _ptr(K_raw),
                                _ptr(V_raw), _ptr(U_K), _ptr(U_V), _ptr(q_pos), _ptr(out),
                                _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "slimkv_decode_attn")
    return out


def decode_attn_reconstruct(q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, *, scale=None,
                            rope_base=10000.0, out=None, workspace: Optional[Workspace] = None,
                            stream=None):
    """slimkv_decode_attn_reconstruct on torch CUDA tensors."""
    lib = load()
    B, Hq, d = q.shape
    W = K_raw.shape[1] if K_raw is not None else 0
    sh, nb = _shape_and_bytes(SLIMKV_RECONSTRUCT, B, Hq, U_K.shape[0] // d, d, C_K.shape[1], C_K.shape[2],
                              C_V.shape[2], W, q.dtype, scale, rope_base)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    if nb == 0:
        _check(2, "slimkv_decode_attn_reconstruct")
    ws = (workspace or Workspace(q.device)).get(nb)
    st = lib.slimkv_decode_attn_reconstruct(ctypes.byref(sh), _ptr(q), _ptr(C_K), _ptr(C_V),
                                            _ptr(K_raw), _ptr(V_raw), _ptr(U_K), _ptr(U_V),
                                            _ptr(q_pos), _ptr(out), _ptr(ws), ws.numel(),
                                            _stream(stream))
    _check(st, "slimkv_decode_attn_reconstruct")
    return out


def alibi_slopes(n_heads: int):
    """The usual ALiBi slopes for n_heads heads: 2^(-8 i / n) for i = 1 .. n when n is a
    power of two; otherwise those of the largest power of two m < n, followed by every
    other slope of 2m heads (the first n - m of them)."""
    def pow2(n):
        return [2.0 ** (-8.0 * (i + 1) / n) for i in range(n)]
    m = 1 << (n_heads.bit_length() - 1)
    if m == n_heads:
        return pow2(n_heads)
    return pow2(m) + pow2(2 * m)[0::2][: n_heads - m]


def decode_attn_alibi(q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, slopes, beacon_ratio, *, scale=None,
                      rope_base=10000.0, out=None, workspace: Optional[Workspace] = None, stream=None):
    """slimkv_decode_attn_alibi on torch CUDA tensors; `slopes` is a sequence of Hq floats."""
    lib = load()
    B, Hq, d = q.shape
    N_b = C_K.shape[1] if C_K is not None else 0
    W = K_raw.shape[1] if K_raw is not None else 0
    Hkv = U_K.shape[0] // d if U_K is not None else K_raw.shape[2]
    r_k = C_K.shape[2] if C_K is not None else 0
    r_v = C_V.shape[2] if C_V is not None else 0
    sh, nb = _shape_and_bytes(SLIMKV_LATENT, B, Hq, Hkv, d, N_b, r_k, r_v, W, q.dtype, scale, rope_base)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    if nb == 0:
        _check(2, "slimkv_decode_attn_alibi")
    sl = (ctypes.c_float * Hq)(*[float(x) for x in slopes])
    ws = (workspace or Workspace(q.device)).get(nb)
    st = lib.slimkv_decode_attn_alibi(ctypes.byref(sh), _ptr(q), _ptr(C_K), _ptr(C_V), _ptr(K_raw), _ptr(V_raw),
                                      _ptr(U_K), _ptr(U_V), _ptr(q_pos), ctypes.cast(sl, ctypes.c_void_p),
                                      int(beacon_ratio), _ptr(out), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "slimkv_decode_attn_alibi")
    return out


def decode_attn_reconstruct_rope(q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, beacon_ratio, *, scale=None,
                                 rope_base=10000.0, out=None, workspace: Optional[Workspace] = None,
                                 stream=None):
    """slimkv_decode_attn_reconstruct_rope on torch CUDA tensors."""
    lib = load()
    B, Hq, d = q.shape
    W = K_raw.shape[1] if K_raw is not None else 0
    sh, nb = _shape_and_bytes(SLIMKV_RECONSTRUCT, B, Hq, U_K.shape[0] // d, d, C_K.shape[1], C_K.shape[2],
                              C_V.shape[2], W, q.dtype, scale, rope_base)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    if nb == 0:
        _check(2, "slimkv_decode_attn_reconstruct_rope")
    ws = (workspace or Workspace(q.device)).get(nb)
    st = lib.slimkv_decode_attn_reconstruct_rope(ctypes.byref(sh), _ptr(q), _ptr(C_K), _ptr(C_V),
                                                 _ptr(K_raw), _ptr(V_raw), _ptr(U_K), _ptr(U_V),
                                                 _ptr(q_pos), int(beacon_ratio), _ptr(out), _ptr(ws),
                                                 ws.numel(), _stream(stream))
    _check(st, "slimkv_decode_attn_reconstruct_rope")
    return out


def decode_attn_full_kv(q, K, V, q_pos, *, scale=None, rope_base=10000.0, out=None,
                        workspace: Optional[Workspace] = None, stream=None):
    """slimkv_decode_attn_full_kv on torch CUDA tensors."""
    lib = load()
    B, Hq, d = q.shape
    sh, nb = _shape_and_bytes(SLIMKV_FULL_KV, B, Hq, K.shape[2], d, 0, 0, 0, K.shape[1], q.dtype, scale,
                              rope_base)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    if nb == 0:
        _check(2, "slimkv_decode_attn_full_kv")
    ws = (workspace or Workspace(q.device)).get(nb)
    st = lib.slimkv_decode_attn_full_kv(ctypes.byref(sh), _ptr(q), _ptr(K), _ptr(V), _ptr(q_pos),
                                        _ptr(out), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "slimkv_decode_attn_full_kv")
    return out


def prefill_attn(q, C_K, C_V, K_chunk, V_chunk, U_K, U_V, p0, *, scale=None, rope_base=10000.0,
                 out=None, workspace: Optional[Workspace] = None, stream=None):
    """slimkv_prefill_attn on torch CUDA tensors: a chunk q [B,T,Hq,d] over the beacons
    and, causally, the chunk's own keys K_chunk / V_chunk [B,T,Hkv,d]; p0 [B] int32 is
    the position of chunk token 0. Returns out [B,T,Hq,d] float32."""
    lib = load()
    B, T, Hq, d = q.shape
    N_b = C_K.shape[1] if C_K is not None else 0
    Hkv = K_chunk.shape[2]
    r_k = C_K.shape[2] if C_K is not None else 0
    r_v = C_V.shape[2] if C_V is not None else 0
    sh, nb = _shape_and_bytes(SLIMKV_PREFILL, B, Hq, Hkv, d, N_b, r_k, r_v, T, q.dtype, scale, rope_base)
    if out is None:
        out = torch.empty((B, T, Hq, d), dtype=torch.float32, device=q.device)
    if nb == 0:
        _check(2, "slimkv_prefill_attn")
    ws = (workspace or Workspace(q.device)).get(nb)
    st = lib.slimkv_prefill_attn(ctypes.byref(sh), _ptr(q), _ptr(C_K), _ptr(C_V), _ptr(K_chunk),
                                 _ptr(V_chunk), _ptr(U_K), _ptr(U_V), _ptr(p0), _ptr(out),
                                 _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "slimkv_prefill_attn")
    return out


def decode_attn_noalloc(q, C_K, C_V, K_raw, V_raw, U_K, U_V, q_pos, *, scale=None,
                        rope_base=10000.0, out=None, stream=None):
    """slimkv_decode_attn_noalloc on torch CUDA tensors: the library uses its own fixed
    device scratch array instead of a caller workspace (for callers that cannot
    allocate device memory). ``out`` may be preallocated; nothing else is allocated."""
    lib = load()
    B, Hq, d = q.shape
    N_b = C_K.shape[1] if C_K is not None else 0
    W = K_raw.shape[1] if K_raw is not None else 0
    Hkv = U_K.shape[0] // d if U_K is not None else K_raw.shape[2]
    r_k = C_K.shape[2] if C_K is not None else 0
    r_v = C_V.shape[2] if C_V is not None else 0
    sh = make_shape(B, Hq, Hkv, d, N_b, r_k, r_v, W, q.dtype, scale, rope_base)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    st = lib.slimkv_decode_attn_noalloc(ctypes.byref(sh), _ptr(q), _ptr(C_K), _ptr(C_V),
                                        _ptr(K_raw), _ptr(V_raw), _ptr(U_K), _ptr(U_V),
                                        _ptr(q_pos), _ptr(out), _stream(stream))
    _check(st, "slimkv_decode_attn_noalloc")
    return out


def abort_count(reset: bool = False) -> int:
    """Thread blocks of the tensor-core kernels on the current device that gave up on a
    bounded wait (their results are NaN) since load or the last reset; synchronises."""
    n = int(load().slimkv_abort_count(1 if reset else 0))
    if n < 0:
        raise SlimkvError(6, "slimkv_abort_count")
    return n


def withhold_first_load_for_test(cta: int):
    """Test hook: the next tensor-core decode launch of this thread skips CTA `cta`'s
    first key load, so that a bounded wait runs out and the abort path runs."""
    load().slimkv_test_withhold_first_load(int(cta))


def status_str(status: int) -> str:
    return load().slimkv_status_str(status).decode()


def append_kv(k_new, v_new, K_raw, V_raw, pos, *, rope_base=10000.0, stream=None):
    """slimkv_append_kv: the current token into the window ring (slot pos mod W),
    its key rotated at pos. K_raw / V_raw [B, W, Hkv, d] are updated in place."""
    lib = load()
    B, W, Hkv, d = K_raw.shape
    sh = make_shape(B, 1, 1, d, 0, 0, 0, W, K_raw.dtype, 1.0, rope_base)
    sh.Hkv = Hkv
    st = lib.slimkv_append_kv(ctypes.byref(sh), _ptr(k_new), _ptr(v_new), _ptr(K_raw), _ptr(V_raw), _ptr(pos),
                              _stream(stream))
    _check(st, "slimkv_append_kv")
