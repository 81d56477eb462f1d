"""CPU oracle of the decode-batch QKV front (plain C, loaded with ctypes).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the product library
(``kv_insert_gb300``) never does, and shares no code with it.

The C source ``qkv_oracle.c`` states each step with the page section it
follows.  This module only compiles it (gcc, no fast-math, no FP contraction)
and marshals numpy arrays in and out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

HEAD_DIM = 64
Q_PER_KV = 8
PAGE_SLOTS = 16
SLOT_WIDTH = 128
EPS = 1e-6

HEAD_Q, HEAD_K, HEAD_V, HEAD_GATE = 0, 1, 2, 3
ERR_SLOT, ERR_POSITION, ERR_SHAPE, ERR_ATTN_REQUEST = 1, 2, 4, 8

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so``; returns its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = f32
        lib.oracle_f32_to_bf16.argtypes = [f32]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_project_f32.argtypes = [vp, vp, i32, i32, i32, vp]
        lib.oracle_project_f32.restype = None
        lib.oracle_head_kind.argtypes = [i32, i32]
        lib.oracle_head_kind.restype = i32
        lib.oracle_rms_norm_head.argtypes = [vp, f32, vp]
        lib.oracle_rms_norm_head.restype = None
        lib.oracle_rope_head.argtypes = [vp, vp, vp]
        lib.oracle_rope_head.restype = None
        lib.oracle_kv_insert_token.argtypes = [vp, i64, vp, i32]
        lib.oracle_kv_insert_token.restype = None
        lib.oracle_qkv_front.argtypes = [vp, vp, vp, vp, vp, i64, vp, vp, i64,
                                         i32, i32, i32, i32, vp]
        lib.oracle_qkv_front.restype = i32
        lib.oracle_qknorm_rope_kv_insert.argtypes = [vp, vp, vp, vp, i64, vp, i64, i32, i32, i32]
        lib.oracle_qknorm_rope_kv_insert.restype = i32
        lib.oracle_layer_front.argtypes = [vp, i32, vp, vp, vp, vp, i32, i32, f32]
        lib.oracle_layer_front.restype = None
        lib.oracle_attn2.argtypes = [vp, i32, i32, vp, i64, vp, i32, vp, i32, i32,
                                     ctypes.c_double, ctypes.c_double, vp]
        lib.oracle_attn2.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


# ---- element steps ---------------------------------------------------------

def f32_to_bf16_bits(values) -> np.ndarray:
    """uint16 BF16 bit patterns of float32 values, round-to-nearest-even."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.fromiter((lib.oracle_f32_to_bf16(float(f)) for f in v),
                       dtype=np.uint16, count=v.size).reshape(np.shape(values))


def bf16_bits_to_f32(bits) -> np.ndarray:
    """float32 values of uint16 BF16 bit patterns (exact widening)."""
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.fromiter((lib.oracle_bf16_to_f32(int(h)) for h in b),
                       dtype=np.float32, count=b.size).reshape(np.shape(bits))


def project_f32(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """FP32 accumulators acc[M, N] = x @ W^T, sequential in k."""
    x = _c(x_bits, np.uint16)
    w = _c(w_bits, np.uint16)
    M, K = x.shape
    N, K2 = w.shape
    if K != K2:
        raise ValueError("x and W disagree on K")
    acc = np.empty((M, N), dtype=np.float32)
    _load().oracle_project_f32(_ptr(x), _ptr(w), M, N, K, _ptr(acc))
    return acc


def head_kind(head: int, num_kv_heads: int) -> int:
    return int(_load().oracle_head_kind(head, num_kv_heads))


def rms_norm_head(p, eps: float = EPS) -> np.ndarray:
    p = _c(np.asarray(p, dtype=np.float32), np.float32)
    if p.shape != (HEAD_DIM,):
        raise ValueError("one head of 64 values")
    u = np.empty(HEAD_DIM, dtype=np.float32)
    _load().oracle_rms_norm_head(_ptr(p), float(eps), _ptr(u))
    return u


def rope_head(u, cs_row) -> np.ndarray:
    u = _c(np.asarray(u, dtype=np.float32), np.float32)
    cs = _c(np.asarray(cs_row, dtype=np.float32), np.float32)
    if u.shape != (HEAD_DIM,) or cs.shape != (HEAD_DIM,):
        raise ValueError("one head of 64 values and one table row of 64")
    y = np.empty(HEAD_DIM, dtype=np.float32)
    _load().oracle_rope_head(_ptr(u), _ptr(cs), _ptr(y))
    return y


def kv_insert_token(out_row_bits: np.ndarray, slot: int, kv_cache_bits: np.ndarray,
                    num_kv_heads: int) -> None:
    """In place: writes one token's K and V rows into the cache array."""
    row = _c(out_row_bits, np.uint16)
    if not kv_cache_bits.flags.c_contiguous or kv_cache_bits.dtype != np.uint16:
        raise TypeError("cache must be a contiguous uint16 array")
    _load().oracle_kv_insert_token(_ptr(row), int(slot), _ptr(kv_cache_bits), num_kv_heads)


# ---- the whole front -------------------------------------------------------

def qkv_front(x_bits, w_bits, positions, slots, cos_sin, kv_cache_bits, num_kv_heads,
              out_bits=None):
    """Run the oracle.  All arrays are numpy (bf16 as uint16 bit patterns).

    ``kv_cache_bits`` (uint16 [pages, nkv, 16, 128]) is updated in place.
    Returns ``(out_bits [M, N] uint16, err)``.  ``out_bits`` may be given to
    start from a known content (elements the op skips keep it).
    """
    x = _c(x_bits, np.uint16)
    w = _c(w_bits, np.uint16)
    pos = _c(np.asarray(positions, dtype=np.int64), np.int64)
    sl = _c(np.asarray(slots, dtype=np.int64), np.int64)
    cs = _c(cos_sin, np.float32)
    if not kv_cache_bits.flags.c_contiguous or kv_cache_bits.dtype != np.uint16:
        raise TypeError("cache must be a contiguous uint16 array")
    M, K = x.shape
    N = w.shape[0]
    if out_bits is None:
        out = np.zeros((M, N), dtype=np.uint16)
    else:
        out = _c(out_bits, np.uint16).copy()
    acc = np.empty((max(M, 1), N), dtype=np.float32)
    num_pages = kv_cache_bits.shape[0]
    if M == 0:
        return out, 0
    err = _load().oracle_qkv_front(_ptr(x), _ptr(w), _ptr(pos), _ptr(sl), _ptr(cs),
                                   cs.shape[0], _ptr(out), _ptr(kv_cache_bits), num_pages,
                                   M, N, K, num_kv_heads, _ptr(acc))
    return out, int(err)


def qknorm_rope_kv_insert(qkv_bits, positions, slots, cos_sin, kv_cache_bits, num_kv_heads):
    """The unfused epilogue on a BF16 projection output.  Returns
    ``(qkv_out_bits [T, N], err)``; ``kv_cache_bits`` is updated in place and
    ``qkv_bits`` is left unchanged (the result is a copy)."""
    q = _c(qkv_bits, np.uint16).copy()
    pos = _c(np.asarray(positions, dtype=np.int64), np.int64)
    sl = _c(np.asarray(slots, dtype=np.int64), np.int64)
    cs = _c(cos_sin, np.float32)
    if not kv_cache_bits.flags.c_contiguous or kv_cache_bits.dtype != np.uint16:
        raise TypeError("cache must be a contiguous uint16 array")
    T, N = q.shape
    if T == 0:
        return q, 0
    err = _load().oracle_qknorm_rope_kv_insert(_ptr(q), _ptr(pos), _ptr(sl), _ptr(cs), cs.shape[0],
                                               _ptr(kv_cache_bits), kv_cache_bits.shape[0], T, N,
                                               num_kv_heads)
    return q, int(err)


def layer_front(x, weight_bits=None, keep_aux=False, eps: float = EPS):
    """The predecessor: x (uint16 bf16 bits or float32) [rows, hidden] ->
    (stream f32, aux f32 or None, out bf16 bits)."""
    x = np.ascontiguousarray(x)
    if x.dtype not in (np.uint16, np.float32):
        raise TypeError("x must be bf16 bits (uint16) or float32")
    rows, hidden = x.shape
    stream = np.empty((rows, hidden), np.float32)
    aux = np.empty((rows, hidden), np.float32) if keep_aux else None
    out = np.empty((rows, hidden), np.uint16)
    w = None if weight_bits is None else _c(weight_bits, np.uint16)
    if w is not None and w.shape != (hidden,):
        raise ValueError("weight must be [hidden]")
    _load().oracle_layer_front(_ptr(x), 1 if x.dtype == np.float32 else 0,
                               None if w is None else _ptr(w), _ptr(stream),
                               None if aux is None else _ptr(aux), _ptr(out), rows, hidden,
                               float(eps))
    return stream, aux, out


def attn2(qkv_bits, kv_cache_bits, block_table, context_lens, num_kv_heads, window=0,
          scale=0.125, eps=EPS, out_bits=None):
    """Paged verify-step attention with o-norm and sigmoid gate.  qkv: uint16
    [8 R, N]; block_table int32 [R, max_blocks]; context_lens int32 [R].
    Returns (out uint16 [8 R, 8 nkv 64], err)."""
    q = _c(qkv_bits, np.uint16)
    cache = _c(kv_cache_bits, np.uint16)
    bt = _c(np.asarray(block_table, dtype=np.int32), np.int32)
    cl = _c(np.asarray(context_lens, dtype=np.int32), np.int32)
    R = cl.shape[0]
    T, N = q.shape
    if T != 8 * R:
        raise ValueError("qkv must hold 8 rows per request")
    cols = Q_PER_KV * num_kv_heads * HEAD_DIM
    out = np.zeros((T, cols), np.uint16) if out_bits is None else _c(out_bits, np.uint16).copy()
    if R == 0:
        return out, 0
    err = _load().oracle_attn2(_ptr(q), N, num_kv_heads, _ptr(cache), cache.shape[0], _ptr(bt),
                               bt.shape[1], _ptr(cl), R, int(window), float(scale), float(eps),
                               _ptr(out))
    return out, int(err)
