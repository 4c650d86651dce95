"""Position-free paged attention for GB300 (sm_103a): Python binding.

This module only marshals arguments to the C ABI of ``libminipic.so`` (declared
in ``include/minipic.h``); every step of the attention runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current CUDA stream.
There is no CPU fallback: if the library is missing or fails to load, every
call raises ``MiniPICError``.

Conventions (see the header for the full contract): the paged pools are
``[num_blocks, num_kv_heads, block_size, head_dim]`` and hold UNROTATED keys;
request r's key j lives in block ``block_tables[r, j // 16]`` at logical
position ``block_starts[r, j // 16] + j % 16``; queries are passed unrotated
with their positions; the kernels rotate both with the cos/sin table built by
``rope_table`` (half-rotation RoPE, theta_i = base^(-2i/d)).
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

__all__ = [
    "MiniPICError",
    "library_path",
    "load",
    "RopeTable",
    "rope_table",
    "rope_table_f16",
    "rope_table_bf16",
    "decode_workspace_size",
    "attn_decode",
    "attn_decode_prerotated",
    "prefill_workspace_size",
    "attn_prefill",
    "attn_prefill_prerotated",
    "attn_mixed",
    "kv_append",
    "kv_swap_out",
    "kv_swap_in",
    "device_error",
    "block_hashes",
    "PrefixCache",
    "STATUS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libminipic.so")

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
          3: "workspace missing or too small", 4: "CUDA error", 5: "device data out of range",
          6: "prefix cache full"}
F32, BF16 = 0, 1


class MiniPICError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, 'unknown')} (status {self.status})")


class _KV(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class _Append(ctypes.Structure):
    _fields_ = [("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p), ("cu_new_lens", ctypes.c_void_p),
                ("kv_start", ctypes.c_void_p), ("block_tables", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("total_new", ctypes.c_int32), ("max_new_len", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32)]


class _Rope(ctypes.Structure):
    _fields_ = [("cos_sin", ctypes.c_void_p), ("max_pos", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("cos_sin_f16", ctypes.c_void_p), ("cos_sin_bf16", ctypes.c_void_p)]


class _Decode(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("block_tables", ctypes.c_void_p),
                ("block_starts", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("q_pos", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("out", ctypes.c_void_p),
                ("lse", ctypes.c_void_p)]


class _Prefill(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("cu_q_lens", ctypes.c_void_p), ("q_pos", ctypes.c_void_p),
                ("block_tables", ctypes.c_void_p), ("block_starts", ctypes.c_void_p),
                ("kv_lens", ctypes.c_void_p), ("batch", ctypes.c_int32), ("total_q", ctypes.c_int32),
                ("max_q_len", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _LIB_PATH


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libminipic.so (once) and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise MiniPICError(4, f"libminipic.so not found at {p}; build it with "
                                  "position_independent_kv_paged_gb300._build.build()")
        L = ctypes.CDLL(p)
        c_i32, c_sz, c_vp, c_f, c_d = ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float, ctypes.c_double
        L.minipic_status_string.restype = ctypes.c_char_p
        L.minipic_status_string.argtypes = [ctypes.c_int]
        L.minipic_rope_table.restype = ctypes.c_int
        L.minipic_rope_table.argtypes = [c_vp, c_i32, c_i32, c_d, c_vp]
        L.minipic_rope_table_f16.restype = ctypes.c_int
        L.minipic_rope_table_f16.argtypes = [c_vp, c_i32, c_i32, c_d, c_vp]
        L.minipic_rope_table_bf16.restype = ctypes.c_int
        L.minipic_rope_table_bf16.argtypes = [c_vp, c_i32, c_i32, c_d, c_vp]
        L.minipic_rope_tables.restype = ctypes.c_int
        L.minipic_rope_tables.argtypes = [c_vp, c_vp, c_vp, c_i32, c_i32, c_d, c_vp]
        L.minipic_attn_decode_workspace_size.restype = c_sz
        L.minipic_attn_decode_workspace_size.argtypes = [c_i32] * 6
        L.minipic_attn_decode.restype = ctypes.c_int
        L.minipic_attn_decode.argtypes = [ctypes.c_int, c_i32, ctypes.POINTER(_KV), ctypes.POINTER(_Rope),
                                          ctypes.POINTER(_Decode), c_f, c_vp, c_sz, c_vp]
        L.minipic_attn_decode_prerotated.restype = ctypes.c_int
        L.minipic_attn_decode_prerotated.argtypes = [ctypes.c_int, c_i32, ctypes.POINTER(_KV),
                                                     ctypes.POINTER(_Decode), c_f, c_vp, c_sz, c_vp]
        L.minipic_attn_prefill_workspace_size.restype = c_sz
        L.minipic_attn_prefill_workspace_size.argtypes = [c_i32] * 7
        L.minipic_attn_prefill.restype = ctypes.c_int
        L.minipic_attn_prefill.argtypes = [ctypes.c_int, c_i32, ctypes.POINTER(_KV), ctypes.POINTER(_Rope),
                                           ctypes.POINTER(_Prefill), c_f, c_vp, c_sz, c_vp]
        L.minipic_attn_prefill_prerotated.restype = ctypes.c_int
        L.minipic_attn_prefill_prerotated.argtypes = [ctypes.c_int, c_i32, ctypes.POINTER(_KV),
                                                      ctypes.POINTER(_Prefill), c_f, c_vp]
        L.minipic_attn_mixed.restype = ctypes.c_int
        L.minipic_attn_mixed.argtypes = [ctypes.c_int, c_i32, ctypes.POINTER(_KV), ctypes.POINTER(_Rope),
                                         ctypes.POINTER(_Prefill), ctypes.POINTER(_Decode), c_f, c_vp, c_sz, c_vp]
        L.minipic_kv_append.restype = ctypes.c_int
        L.minipic_kv_append.argtypes = [ctypes.c_int, ctypes.POINTER(_KV), ctypes.POINTER(_Append), c_vp]
        for fn in (L.minipic_kv_swap_out, L.minipic_kv_swap_in):
            fn.restype = ctypes.c_int
            fn.argtypes = [ctypes.c_int, ctypes.POINTER(_KV), c_vp, c_i32, c_vp, c_vp, c_vp]
        L.minipic_device_error.restype = ctypes.c_int
        L.minipic_device_error.argtypes = [ctypes.POINTER(c_i32), c_i32, c_vp]
        L.minipic_block_hashes.restype = ctypes.c_int
        L.minipic_block_hashes.argtypes = [c_vp, c_i32, c_i32, c_i32, c_i32, ctypes.c_uint64, c_vp, c_i32,
                                           ctypes.POINTER(c_i32)]
        L.minipic_prefix_cache_create.restype = ctypes.c_int
        L.minipic_prefix_cache_create.argtypes = [c_i32, ctypes.POINTER(c_vp)]
        L.minipic_prefix_cache_destroy.restype = None
        L.minipic_prefix_cache_destroy.argtypes = [c_vp]
        L.minipic_prefix_cache_assign.restype = ctypes.c_int
        L.minipic_prefix_cache_assign.argtypes = [c_vp, c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp]
        L.minipic_prefix_cache_release.restype = ctypes.c_int
        L.minipic_prefix_cache_release.argtypes = [c_vp, c_vp, c_i32]
        _lib = L
        return L


# ---------------------------------------------------------------- helpers

def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")


def _need(t, name, dtype=None, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _check(status: int, where: str):
    if status != 0:
        raise MiniPICError(status, where)


def _kv(k_pool, v_pool) -> _KV:
    _need(k_pool, "k_pool", ndim=4)
    _need(v_pool, "v_pool", dtype=k_pool.dtype, ndim=4)
    if tuple(k_pool.shape) != tuple(v_pool.shape):
        raise ValueError("k_pool and v_pool shapes differ")
    nb, hkv, bs, d = k_pool.shape
    return _KV(k_pool.data_ptr(), v_pool.data_ptr(), nb, hkv, bs, d)


# ---------------------------------------------------------------- API

class RopeTable:
    """The rotary cos/sin table in the three forms the kernels read:
    ``cos_sin`` (float32 [max_pos, head_dim]: the fp32 decode and the prefill's
    query rotation), ``cos_sin_f16`` (the same values rounded to float16: the
    prefill's key rotation) and ``cos_sin_bf16`` (bfloat16 [max_pos, 2,
    3 head_dim / 2]: cos | sin | -sin of +p theta and of -p theta, the bf16
    decode's rotation).  Built by ``rope_table``."""

    def __init__(self, cos_sin, cos_sin_f16=None, cos_sin_bf16=None):
        self.cos_sin = cos_sin
        self.cos_sin_f16 = cos_sin_f16
        self.cos_sin_bf16 = cos_sin_bf16

    @property
    def max_pos(self) -> int:
        return int(self.cos_sin.shape[0])

    @property
    def head_dim(self) -> int:
        return int(self.cos_sin.shape[1])


def rope_table_f16(max_pos: int, head_dim: int, base: float, device=None, stream=None, out=None):
    """Build the float16 cos/sin table [max_pos, head_dim] on the GPU."""
    torch = _torch()
    L = load()
    if out is None:
        out = torch.empty((max_pos, head_dim), dtype=torch.float16,
                          device=device if device is not None else "cuda")
    _need(out, "out", dtype=torch.float16, ndim=2)
    _check(L.minipic_rope_table_f16(out.data_ptr(), int(max_pos), int(head_dim), float(base), _stream(stream)),
           "minipic_rope_table_f16")
    return out


def rope_table_bf16(max_pos: int, head_dim: int, base: float, device=None, stream=None, out=None):
    """Build the bfloat16 rows [max_pos, 2, 3 head_dim / 2] on the GPU: [p, 0] is
    cos | sin | -sin of +p theta_i, [p, 1] the same of -p theta_i."""
    torch = _torch()
    L = load()
    if out is None:
        out = torch.empty((max_pos, 2, 3 * head_dim // 2), dtype=torch.bfloat16,
                          device=device if device is not None else "cuda")
    _need(out, "out", dtype=torch.bfloat16, ndim=3)
    if tuple(out.shape) != (max_pos, 2, 3 * head_dim // 2):
        raise ValueError("out must be [max_pos, 2, 3 * head_dim / 2]")
    _check(L.minipic_rope_table_bf16(out.data_ptr(), int(max_pos), int(head_dim), float(base), _stream(stream)),
           "minipic_rope_table_bf16")
    return out


def rope_table(max_pos: int, head_dim: int, base: float, device=None, stream=None) -> RopeTable:
    """Build the cos/sin table (float32, float16 and bfloat16 forms) on the GPU
    in one pass."""
    torch = _torch()
    L = load()
    dev = device if device is not None else "cuda"
    f32 = torch.empty((max_pos, head_dim), dtype=torch.float32, device=dev)
    f16 = torch.empty((max_pos, head_dim), dtype=torch.float16, device=f32.device)
    b16 = torch.empty((max_pos, 2, 3 * head_dim // 2), dtype=torch.bfloat16, device=f32.device)
    _check(L.minipic_rope_tables(f32.data_ptr(), f16.data_ptr(), b16.data_ptr(), int(max_pos), int(head_dim),
                                 float(base), _stream(stream)), "minipic_rope_tables")
    return RopeTable(f32, f16, b16)


def _rope_struct(rope, need_f16: bool, need_bf16: bool = False) -> _Rope:
    """ABI view of a RopeTable (or, for the fp32 decode, of a bare float32 table)."""
    torch = _torch()
    if isinstance(rope, RopeTable):
        f32, f16, b16 = rope.cos_sin, rope.cos_sin_f16, rope.cos_sin_bf16
    else:
        f32, f16, b16 = rope, None, None
    _need(f32, "rope", dtype=torch.float32, ndim=2)
    if f16 is not None:
        _need(f16, "rope f16", dtype=torch.float16, ndim=2)
        if tuple(f16.shape) != tuple(f32.shape):
            raise ValueError("the float16 and float32 tables differ in shape")
    elif need_f16:
        raise TypeError("prefill needs the RopeTable built by rope_table() (it carries the float16 table)")
    if b16 is not None:
        _need(b16, "rope bf16", dtype=torch.bfloat16, ndim=3)
        if tuple(b16.shape) != (f32.shape[0], 2, 3 * f32.shape[1] // 2):
            raise ValueError("the bfloat16 table must be [max_pos, 2, 3 * head_dim / 2]")
    elif need_bf16:
        raise TypeError("the bf16 decode needs the RopeTable built by rope_table() (it carries the bfloat16 table)")
    return _Rope(f32.data_ptr(), f32.shape[0], f32.shape[1], None if f16 is None else f16.data_ptr(),
                 None if b16 is None else b16.data_ptr())


def decode_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                          max_blocks_per_seq: int, block_size: int = 16) -> int:
    return int(load().minipic_attn_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                         max_blocks_per_seq, block_size))


def _decode(q, k_pool, v_pool, block_tables, block_starts, seq_lens, q_pos, rope, scale, out, lse,
            workspace, stream, prerotated):
    torch = _torch()
    L = load()
    _need(q, "q", ndim=3)
    kv = _kv(k_pool, v_pool)
    if k_pool.dtype != q.dtype:
        raise TypeError("q and the pools must share a dtype")
    B, Hq, d = q.shape
    for name, t in (("block_tables", block_tables), ("block_starts", block_starts)):
        _need(t, name, dtype=torch.int32, ndim=2)
    _need(seq_lens, "seq_lens", dtype=torch.int32, ndim=1)
    _need(q_pos, "q_pos", dtype=torch.int32, ndim=1)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", dtype=q.dtype)
    if lse is not None:
        _need(lse, "lse", dtype=torch.float32)
    mb = block_tables.shape[1]
    if workspace is None:
        n = decode_workspace_size(B, Hq, kv.num_kv_heads, d, mb, kv.block_size)
        workspace = torch.zeros(max(n, 1), dtype=torch.uint8, device=q.device)
    db = _Decode(q.data_ptr(), block_tables.data_ptr(), block_starts.data_ptr(), seq_lens.data_ptr(),
                 q_pos.data_ptr(), B, mb, out.data_ptr(), _ptr(lse))
    ws_ptr, ws_n = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if prerotated:
        st = L.minipic_attn_decode_prerotated(_dtype_code(q), Hq, ctypes.byref(kv), ctypes.byref(db),
                                              float(scale), ws_ptr, ws_n, _stream(stream))
        _check(st, "minipic_attn_decode_prerotated")
    else:
        rp = _rope_struct(rope, False, need_bf16=q.dtype == torch.bfloat16)
        st = L.minipic_attn_decode(_dtype_code(q), Hq, ctypes.byref(kv), ctypes.byref(rp), ctypes.byref(db),
                                   float(scale), ws_ptr, ws_n, _stream(stream))
        _check(st, "minipic_attn_decode")
    return out, lse


def attn_decode(q, k_pool, v_pool, block_tables, block_starts, seq_lens, q_pos, rope, scale: float = 0.0,
                out=None, lse=None, workspace=None, stream=None):
    """One decode token per request over the position-free paged cache.

    Returns (out, lse); out has q's shape/dtype, lse is the optional float
    [B, Hq] log-sum-exp buffer passed in (None if not given)."""
    return _decode(q, k_pool, v_pool, block_tables, block_starts, seq_lens, q_pos, rope, scale, out, lse,
                   workspace, stream, False)


def attn_decode_prerotated(q, k_pool, v_pool, block_tables, block_starts, seq_lens, q_pos,
                           scale: float = 0.0, out=None, lse=None, workspace=None, stream=None):
    """Same kernel with rotation compiled out (keys and q already rotated)."""
    return _decode(q, k_pool, v_pool, block_tables, block_starts, seq_lens, q_pos, None, scale, out, lse,
                   workspace, stream, True)


def prefill_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_q_len, max_blocks_per_seq,
                           block_size=16) -> int:
    return int(load().minipic_attn_prefill_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                          max_q_len, max_blocks_per_seq, block_size))


def _prefill(q, cu_q_lens, q_pos, k_pool, v_pool, block_tables, block_starts, kv_lens, rope, max_q_len, scale,
             out, lse, workspace, stream, prerotated):
    torch = _torch()
    L = load()
    _need(q, "q", ndim=3)
    kv = _kv(k_pool, v_pool)
    total_q, Hq, d = q.shape
    for name, t in (("block_tables", block_tables), ("block_starts", block_starts)):
        _need(t, name, dtype=torch.int32, ndim=2)
    for name, t in (("cu_q_lens", cu_q_lens), ("q_pos", q_pos), ("kv_lens", kv_lens)):
        _need(t, name, dtype=torch.int32, ndim=1)
    if out is None:
        out = torch.empty_like(q)
    if lse is not None:
        _need(lse, "lse", dtype=torch.float32)
    B = kv_lens.shape[0]
    mb = block_tables.shape[1]
    pb = _Prefill(q.data_ptr(), cu_q_lens.data_ptr(), q_pos.data_ptr(), block_tables.data_ptr(),
                  block_starts.data_ptr(), kv_lens.data_ptr(), B, total_q, int(max_q_len), mb,
                  out.data_ptr(), _ptr(lse))
    if prerotated:
        st = L.minipic_attn_prefill_prerotated(_dtype_code(q), Hq, ctypes.byref(kv), ctypes.byref(pb),
                                               float(scale), _stream(stream))
        _check(st, "minipic_attn_prefill_prerotated")
        return out, lse
    rp = _rope_struct(rope, True)
    if workspace is None:
        n = prefill_workspace_size(B, Hq, kv.num_kv_heads, d, max_q_len, mb, kv.block_size)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    st = L.minipic_attn_prefill(_dtype_code(q), Hq, ctypes.byref(kv), ctypes.byref(rp), ctypes.byref(pb),
                                float(scale), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "minipic_attn_prefill")
    return out, lse


def attn_prefill(q, cu_q_lens, q_pos, k_pool, v_pool, block_tables, block_starts, kv_lens, rope,
                 max_q_len: int, scale: float = 0.0, out=None, lse=None, workspace=None, stream=None):
    """Chunked prefill (bf16) over cached span blocks plus the chunk's own keys."""
    return _prefill(q, cu_q_lens, q_pos, k_pool, v_pool, block_tables, block_starts, kv_lens, rope, max_q_len,
                    scale, out, lse, workspace, stream, False)


def attn_prefill_prerotated(q, cu_q_lens, q_pos, k_pool, v_pool, block_tables, block_starts, kv_lens,
                            max_q_len: int, scale: float = 0.0, out=None, lse=None, stream=None):
    """Same prefill kernel with rotation compiled out (keys and q already rotated)."""
    return _prefill(q, cu_q_lens, q_pos, k_pool, v_pool, block_tables, block_starts, kv_lens, None, max_q_len,
                    scale, out, lse, None, stream, True)


def attn_mixed(prefill: dict, decode: dict, k_pool, v_pool, rope, scale: float = 0.0, workspace=None,
               stream=None):
    """Span-prefill chunks and decode tokens over one pool in ONE launch.

    ``prefill``: dict with q, cu_q_lens, q_pos, block_tables, block_starts,
    kv_lens, max_q_len and optional out / lse.  ``decode``: dict with q,
    block_tables, block_starts, seq_lens, q_pos and optional out / lse.
    Returns (prefill_out, prefill_lse, decode_out, decode_lse)."""
    torch = _torch()
    L = load()
    kv = _kv(k_pool, v_pool)
    rp = _rope_struct(rope, True, need_bf16=True)
    pq, dq = prefill["q"], decode["q"]
    _need(pq, "prefill q", dtype=k_pool.dtype, ndim=3)
    _need(dq, "decode q", dtype=k_pool.dtype, ndim=3)
    for nm in ("cu_q_lens", "q_pos", "kv_lens"):
        _need(prefill[nm], "prefill " + nm, dtype=torch.int32, ndim=1)
    for nm in ("block_tables", "block_starts"):
        _need(prefill[nm], "prefill " + nm, dtype=torch.int32, ndim=2)
        _need(decode[nm], "decode " + nm, dtype=torch.int32, ndim=2)
    for nm in ("seq_lens", "q_pos"):
        _need(decode[nm], "decode " + nm, dtype=torch.int32, ndim=1)
    pout = prefill.get("out") if prefill.get("out") is not None else torch.empty_like(pq)
    dout = decode.get("out") if decode.get("out") is not None else torch.empty_like(dq)
    plse, dlse = prefill.get("lse"), decode.get("lse")
    Hq = pq.shape[1]
    pb = _Prefill(pq.data_ptr(), prefill["cu_q_lens"].data_ptr(), prefill["q_pos"].data_ptr(),
                  prefill["block_tables"].data_ptr(), prefill["block_starts"].data_ptr(),
                  prefill["kv_lens"].data_ptr(), prefill["kv_lens"].shape[0], pq.shape[0],
                  int(prefill["max_q_len"]), prefill["block_tables"].shape[1], pout.data_ptr(), _ptr(plse))
    db = _Decode(dq.data_ptr(), decode["block_tables"].data_ptr(), decode["block_starts"].data_ptr(),
                 decode["seq_lens"].data_ptr(), decode["q_pos"].data_ptr(), dq.shape[0],
                 decode["block_tables"].shape[1], dout.data_ptr(), _ptr(dlse))
    if workspace is None:
        n = decode_workspace_size(dq.shape[0], Hq, kv.num_kv_heads, kv.head_dim, decode["block_tables"].shape[1],
                                  kv.block_size)
        workspace = torch.zeros(max(n, 1), dtype=torch.uint8, device=dq.device)
    st = L.minipic_attn_mixed(_dtype_code(pq), Hq, ctypes.byref(kv), ctypes.byref(rp), ctypes.byref(pb),
                              ctypes.byref(db), float(scale), workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "minipic_attn_mixed")
    return pout, plse, dout, dlse


def device_error(clear: bool = True, stream=None) -> int:
    """Device error word (MINIPIC_DEVERR_* bits) after the stream's work."""
    flags = ctypes.c_int32(0)
    st = load().minipic_device_error(ctypes.byref(flags), 1 if clear else 0, _stream(stream))
    if st not in (0, 5):
        raise MiniPICError(st, "minipic_device_error")
    return int(flags.value)


def kv_append(k_new, v_new, cu_new_lens, kv_start, block_tables, k_pool, v_pool, max_new_len=None,
              stream=None):
    """Write new unrotated keys and values into their paged slots, in place:
    token i of request r (rows cu_new_lens[r] + i of k_new / v_new) becomes key
    index kv_start[r] + i, block block_tables[r][j // 16], slot j % 16.
    ``max_new_len`` bounds every request's count (read from cu_new_lens if None,
    which synchronizes)."""
    torch = _torch()
    L = load()
    kv = _kv(k_pool, v_pool)
    _need(k_new, "k_new", dtype=k_pool.dtype, ndim=3)
    _need(v_new, "v_new", dtype=k_pool.dtype, ndim=3)
    if tuple(k_new.shape) != tuple(v_new.shape) or k_new.shape[1:] != (kv.num_kv_heads, kv.head_dim):
        raise ValueError("k_new / v_new must be [total_new, num_kv_heads, head_dim]")
    for name, t in (("cu_new_lens", cu_new_lens), ("kv_start", kv_start)):
        _need(t, name, dtype=torch.int32, ndim=1)
    _need(block_tables, "block_tables", dtype=torch.int32, ndim=2)
    B = kv_start.shape[0]
    if cu_new_lens.shape[0] != B + 1 or block_tables.shape[0] != B:
        raise ValueError("cu_new_lens must have batch + 1 entries and block_tables batch rows")
    if max_new_len is None:
        max_new_len = int((cu_new_lens[1:] - cu_new_lens[:-1]).max().item()) if B else 0
    ab = _Append(k_new.data_ptr(), v_new.data_ptr(), cu_new_lens.data_ptr(), kv_start.data_ptr(),
                 block_tables.data_ptr(), B, k_new.shape[0], int(max_new_len), block_tables.shape[1])
    _check(L.minipic_kv_append(_dtype_code(k_pool), ctypes.byref(kv), ctypes.byref(ab), _stream(stream)),
           "minipic_kv_append")


def kv_swap_out(k_pool, v_pool, block_ids, host_k=None, host_v=None, stream=None):
    """Copy whole blocks (K and V, every kv head) to page-locked host memory:
    host[i] = pool[block_ids[i]].  Returns (host_k, host_v), allocated pinned
    when not given; they are complete once the stream reaches this call."""
    torch = _torch()
    L = load()
    kv = _kv(k_pool, v_pool)
    _need(block_ids, "block_ids", dtype=torch.int32, ndim=1)
    n = block_ids.shape[0]
    shape = (n,) + tuple(k_pool.shape[1:])
    if host_k is None:
        host_k = torch.empty(shape, dtype=k_pool.dtype, pin_memory=True)
    if host_v is None:
        host_v = torch.empty(shape, dtype=k_pool.dtype, pin_memory=True)
    for name, t in (("host_k", host_k), ("host_v", host_v)):
        if tuple(t.shape) != shape or t.dtype != k_pool.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {tuple(shape)} tensor of the pool's dtype")
    _check(L.minipic_kv_swap_out(_dtype_code(k_pool), ctypes.byref(kv), block_ids.data_ptr(), n,
                                 host_k.data_ptr(), host_v.data_ptr(), _stream(stream)), "minipic_kv_swap_out")
    return host_k, host_v


def kv_swap_in(host_k, host_v, block_ids, k_pool, v_pool, stream=None):
    """Copy host blocks back into the pools: pool[block_ids[i]] = host[i] (ids
    need not be the ones the blocks left from; remap the block tables)."""
    torch = _torch()
    L = load()
    kv = _kv(k_pool, v_pool)
    _need(block_ids, "block_ids", dtype=torch.int32, ndim=1)
    n = block_ids.shape[0]
    shape = (n,) + tuple(k_pool.shape[1:])
    for name, t in (("host_k", host_k), ("host_v", host_v)):
        if tuple(t.shape) != shape or t.dtype != k_pool.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {tuple(shape)} tensor of the pool's dtype")
    _check(L.minipic_kv_swap_in(_dtype_code(k_pool), ctypes.byref(kv), block_ids.data_ptr(), n,
                                host_k.data_ptr(), host_v.data_ptr(), _stream(stream)), "minipic_kv_swap_in")


# ---------------------------------------------------------------- span reuse (host)

def block_hashes(tokens, block_size: int, ssep_token: int, pdep_token: int, h0: int = 0):
    """uint64 hashes of the full blocks of one prompt (SSEP restarts the chain,
    PDEP ties a block to the whole prompt before it); see the header."""
    import numpy as np
    L = load()
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    n_full = t.size // int(block_size) if block_size > 0 else 0
    out = np.zeros(max(n_full, 1), dtype=np.uint64)
    n = ctypes.c_int32(0)
    _check(L.minipic_block_hashes(t.ctypes.data if t.size else None, int(t.size), int(block_size), int(ssep_token),
                                  int(pdep_token), ctypes.c_uint64(int(h0) & ((1 << 64) - 1)),
                                  out.ctypes.data, int(out.size), ctypes.byref(n)), "minipic_block_hashes")
    return out[:n.value]


class PrefixCache:
    """Hash -> physical block map over a pool of num_blocks blocks (host)."""

    def __init__(self, num_blocks: int):
        self._L = load()
        self._h = ctypes.c_void_p(None)
        _check(self._L.minipic_prefix_cache_create(int(num_blocks), ctypes.byref(self._h)),
               "minipic_prefix_cache_create")

    def assign(self, hashes, n_blocks: int, block_size: int):
        """(block_table, block_starts, is_new) of one request: int32, int32,
        uint8 arrays of n_blocks entries.  Raises MiniPICError (status 6)
        when the pool is full; the cache is then unchanged."""
        import numpy as np
        h = np.ascontiguousarray(hashes, dtype=np.uint64)
        n = int(n_blocks)
        tab = np.zeros(max(n, 1), dtype=np.int32)
        st = np.zeros(max(n, 1), dtype=np.int32)
        new = np.zeros(max(n, 1), dtype=np.uint8)
        _check(self._L.minipic_prefix_cache_assign(self._h, h.ctypes.data if h.size else None, int(h.size), n,
                                                    int(block_size), tab.ctypes.data, st.ctypes.data,
                                                    new.ctypes.data), "minipic_prefix_cache_assign")
        return tab[:n], st[:n], new[:n]

    def release(self, block_ids):
        import numpy as np
        b = np.ascontiguousarray(block_ids, dtype=np.int32)
        _check(self._L.minipic_prefix_cache_release(self._h, b.ctypes.data if b.size else None, int(b.size)),
               "minipic_prefix_cache_release")

    def close(self):
        if self._h:
            self._L.minipic_prefix_cache_destroy(self._h)
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
