"""Python binding of libqkvfront: argument marshalling over the C ABI only.

Every step of the op runs in the library's CUDA kernel.  Tensors are torch
CUDA tensors (torch supplies device memory and streams); this module checks
their dtypes, shapes and contiguity, passes raw pointers and sizes, and turns
error codes into exceptions.  There is no CPU path: without the compiled
library every call raises.

Names follow the pages' API (page "vllm.models.muse_spark.nvidia.
specialized_decode.cutedsl.attention.qkv_front": qkv_front, launch,
unsupported, prepare, variant, hidden_rows_ok, kv_cache_layout_ok,
supports_shape, token_tiles; page "...runtime.cute_ops": split_qkv,
supports_call).
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import _build

HIDDEN = 8192
HEAD_DIM = 64
Q_PER_KV = 8
PAGE_SLOTS = 16
SLOT_WIDTH = 128
MAX_TOKENS = 16

CONSUMER_DEFAULT, CONSUMER_MMA_SYNC, CONSUMER_TCGEN05, CONSUMER_RESIDENT = 0, 1, 2, 3

STATUS_BAD_SLOT = 1
STATUS_BAD_POSITION = 2
STATUS_WAIT_TIMEOUT = 4
STATUS_BAD_REQUEST = 8

HEADER = os.path.join(_build.ROOT, "include", "qkvfront.h")

_lock = threading.Lock()
_lib = None


class QkvFrontError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"qkv_front error {code}: {message}")
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        front_args = [vp, vp, vp, vp, vp, i64, vp, vp, i64, i32, i32, i32]
        lib.qkv_front.argtypes = front_args + [vp]
        lib.qkv_front.restype = i32
        lib.qkv_front_launch.argtypes = front_args + [vp]
        lib.qkv_front_launch.restype = i32
        lib.qkv_front_unsupported.argtypes = front_args
        lib.qkv_front_unsupported.restype = ctypes.c_char_p
        lib.qkv_front_launch_variant.argtypes = front_args + [i32, i32, i32, i32, vp]
        lib.qkv_front_launch_variant.restype = i32
        lib.qkv_front_variant.argtypes = [i32, i32] + [ctypes.POINTER(i32)] * 5
        lib.qkv_front_variant.restype = i32
        lib.qkv_front_prepare.argtypes = [i32, i32]
        lib.qkv_front_prepare.restype = i32
        lib.qkv_front_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.qkv_front_status.restype = i32
        lib.qkv_front_strerror.argtypes = [i32]
        lib.qkv_front_strerror.restype = ctypes.c_char_p
        lib.qkv_front_selftest_wait.argtypes = [i64, vp]
        lib.qkv_front_selftest_wait.restype = i32
        lib.qkv_front_set_wait_limit.argtypes = [i64]
        lib.qkv_front_set_wait_limit.restype = i32
        lib.qkv_front_from_host.argtypes = [vp, vp, vp, vp, vp, vp, i64, vp, i64, vp,
                                            ctypes.c_uint64, i32, i32, i32, vp]
        lib.qkv_front_from_host.restype = i32
        lib.qkv_front_staging_bytes.argtypes = [i32, i32]
        lib.qkv_front_staging_bytes.restype = ctypes.c_uint64
        epi_args = [vp, vp, vp, vp, i64, vp, i64, i32, i32, i32]
        lib.qknorm_rope_kv_insert.argtypes = epi_args + [vp]
        lib.qknorm_rope_kv_insert.restype = i32
        lib.qknorm_rope_kv_insert_unsupported.argtypes = epi_args
        lib.qknorm_rope_kv_insert_unsupported.restype = ctypes.c_char_p
        lib.layer_front.argtypes = [vp, i32, vp, vp, vp, vp, i32, ctypes.c_float, vp]
        lib.layer_front.restype = i32
        a2 = [vp, vp, i64, vp, i32, vp, i32, i32, i32, i32, ctypes.c_float, ctypes.c_float, vp]
        lib.attn2.argtypes = a2 + [vp]
        lib.attn2.restype = i32
        lib.attn2_unsupported.argtypes = a2
        lib.attn2_unsupported.restype = ctypes.c_char_p
        lib.attn2_launch_splits.argtypes = a2 + [i32, vp]
        lib.attn2_launch_splits.restype = i32
        lib.attn2_splits.argtypes = [i32, i32, i32, i32]
        lib.attn2_splits.restype = i32
        lib.attn2_split_kv.argtypes = a2 + [i32, vp, ctypes.c_size_t, vp]
        lib.attn2_split_kv.restype = i32
        lib.attn2_split_kv_workspace_bytes.argtypes = [i32, i32, i32]
        lib.attn2_split_kv_workspace_bytes.restype = ctypes.c_size_t
        lib.attn2_split_kv_splits.argtypes = [i32, i32, i32, i32]
        lib.attn2_split_kv_splits.restype = i32
        lib.attn2_split_kv_noalloc.argtypes = a2 + [i32, vp]
        lib.attn2_split_kv_noalloc.restype = i32
        lib.qkv_front_set_pdl.argtypes = [i32]
        lib.qkv_front_set_pdl.restype = i32
        _lib = lib
        return lib


def header_functions() -> list[str]:
    """Names of the functions include/qkvfront.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(
        r"\b((?:qkv_front|qknorm_rope_kv_insert|layer_front|attn2)\w*)\s*\(", text)))


def strerror(code: int) -> str:
    return load().qkv_front_strerror(code).decode()


def _check(code: int) -> None:
    if code != 0:
        raise QkvFrontError(code, strerror(code))


# ---- host-side checks (shapes and dtypes the C ABI cannot see) -------------

def hidden_rows_ok(t: torch.Tensor) -> bool:
    """Whether t is a contiguous, 16-byte aligned bf16 [rows, 8192] CUDA tensor."""
    return (t.dtype == torch.bfloat16 and t.dim() == 2 and t.shape[1] == HIDDEN
            and t.is_contiguous() and t.data_ptr() % 16 == 0)


def kv_cache_layout_ok(kv_cache: torch.Tensor) -> bool:
    """Whether a cache is bf16 [pages, num_kv_heads, 16, 128], contiguous, 16-byte aligned."""
    return (kv_cache.dtype == torch.bfloat16 and kv_cache.dim() == 4
            and kv_cache.shape[2] == PAGE_SLOTS and kv_cache.shape[3] == SLOT_WIDTH
            and kv_cache.is_contiguous() and kv_cache.data_ptr() % 16 == 0)


def supports_shape(n: int, num_kv_heads: int) -> bool:
    """Whether the kernel computes an n-wide projection with these KV heads."""
    return num_kv_heads >= 1 and n == 2 * (Q_PER_KV + 1) * num_kv_heads * HEAD_DIM


def token_tiles(m: int) -> int:
    """8-token mma column tiles for m tokens."""
    return (m + 7) // 8


def head_spans(num_kv_heads: int) -> dict:
    """Column range [start, end) of each head kind in an output row: the
    kinds follow one another as q, k, v, gate, with Q_PER_KV q and gate
    heads and one k and one v head per KV head, HEAD_DIM columns each."""
    counts = (("q", Q_PER_KV), ("k", 1), ("v", 1), ("gate", Q_PER_KV))
    spans, col = {}, 0
    for kind, per_kv in counts:
        width = per_kv * num_kv_heads * HEAD_DIM
        spans[kind] = (col, col + width)
        col += width
    return spans


def split_qkv(qkv: torch.Tensor, num_kv_heads: int):
    """Views of the q heads and of the gate heads of the front's output rows
    (what attn2 reads), taken from the row layout of head_spans."""
    spans = head_spans(num_kv_heads)
    row = spans["gate"][1]
    if qkv.dim() != 2 or qkv.shape[1] != row:
        raise ValueError(f"split_qkv: a layer with {num_kv_heads} KV heads has output rows of "
                         f"{row} columns; this tensor has shape {tuple(qkv.shape)}")
    (q0, q1), (g0, g1) = spans["q"], spans["gate"]
    return qkv[:, q0:q1], qkv[:, g0:g1]


def _tensor_reason(x, weight, positions, cos_sin, slots, kv_cache, out):
    if not all(t.is_cuda for t in (x, weight, positions, cos_sin, slots, kv_cache)):
        return "tensors on a CUDA device"
    dev = x.device
    if any(t.device != dev for t in (weight, positions, cos_sin, slots, kv_cache)):
        return "tensors on different devices"
    if not hidden_rows_ok(x) or not hidden_rows_ok(weight):
        return f"x and weight other than contiguous 16-byte aligned bf16 [rows, {HIDDEN}]"
    M = x.shape[0]
    if not 0 <= M <= MAX_TOKENS:
        return f"{M} tokens (the kernel takes 1 to {MAX_TOKENS})"
    for name, t in (("positions", positions), ("slots", slots)):
        if t.dtype != torch.int64 or t.dim() != 1 or t.shape[0] != M or not t.is_contiguous():
            return f"{name} other than contiguous int64 [{M}]"
    if (cos_sin.dtype != torch.float32 or cos_sin.dim() != 2 or cos_sin.shape[1] != HEAD_DIM
            or not cos_sin.is_contiguous()):
        return "a rotary table other than a contiguous fp32 [*, 64] one"
    if not kv_cache_layout_ok(kv_cache):
        return "a KV cache other than contiguous bf16 [pages, num_kv_heads, 16, 128]"
    nkv = kv_cache.shape[1]
    if not supports_shape(weight.shape[0], nkv):
        return f"a projection of {weight.shape[0]} rows for {nkv} KV heads"
    if out is not None:
        if (out.dtype != torch.bfloat16 or out.shape != (M, weight.shape[0])
                or not out.is_contiguous() or out.device != dev):
            return f"out other than contiguous bf16 [{M}, {weight.shape[0]}]"
    return None


def _args(x, weight, positions, slots, cos_sin, out, kv_cache):
    return (x.data_ptr(), weight.data_ptr(), positions.data_ptr(), slots.data_ptr(),
            cos_sin.data_ptr(), cos_sin.shape[0], out.data_ptr() if out is not None else None,
            kv_cache.data_ptr(), kv_cache.shape[0], x.shape[0], weight.shape[0],
            kv_cache.shape[1])


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def unsupported(x, weight, positions, cos_sin, slots, kv_cache, out=None) -> str | None:
    """Why the kernel cannot take this call (with out, also its output), or None."""
    why = _tensor_reason(x, weight, positions, cos_sin, slots, kv_cache, out)
    if why is not None:
        return why
    if out is None:
        return None
    with torch.cuda.device(x.device):
        r = load().qkv_front_unsupported(*_args(x, weight, positions, slots, cos_sin, out, kv_cache))
    return None if r is None else r.decode()


def supports_call(x, weight, positions, cos_sin, slots, kv_cache, num_kv_heads, out=None) -> bool:
    """Whether the front takes this call of a layer with num_kv_heads: the
    cache must hold exactly the layer's KV heads, and every check of
    `unsupported` must pass (otherwise the caller keeps its unfused path)."""
    if kv_cache.dim() != 4 or kv_cache.shape[1] != num_kv_heads:
        return False
    return not unsupported(x, weight, positions, cos_sin, slots, kv_cache, out)


def qkv_front(x, weight, positions, slots, cos_sin, kv_cache, out=None, stream=None):
    """out[M, N] = x @ weight^T with the q and k heads normed and rotated, and
    the k / v heads inserted into kv_cache at slots.  Returns out."""
    if out is None:
        out = torch.empty(x.shape[0], weight.shape[0], dtype=torch.bfloat16, device=x.device)
    why = _tensor_reason(x, weight, positions, cos_sin, slots, kv_cache, out)
    if why is not None:
        raise ValueError(f"qkv_front does not support {why}")
    with torch.cuda.device(x.device):
        _check(load().qkv_front(*_args(x, weight, positions, slots, cos_sin, out, kv_cache),
                                _stream(stream)))
    return out


def launch(x, weight, positions, slots, cos_sin, kv_cache, out, stream=None):
    """qkv_front without its checks, for a call `unsupported` accepted with out."""
    _check(load().qkv_front_launch(*_args(x, weight, positions, slots, cos_sin, out, kv_cache),
                                   _stream(stream)))
    return out


def launch_variant(x, weight, positions, slots, cos_sin, kv_cache, out, splits, stages, kb=0,
                   consumer=CONSUMER_DEFAULT, stream=None):
    """qkv_front at an explicit (splits, stages, kb, consumer) variant."""
    why = _tensor_reason(x, weight, positions, cos_sin, slots, kv_cache, out)
    if why is not None:
        raise ValueError(f"qkv_front does not support {why}")
    with torch.cuda.device(x.device):
        _check(load().qkv_front_launch_variant(
            *_args(x, weight, positions, slots, cos_sin, out, kv_cache), int(splits), int(stages),
            int(kb), int(consumer), _stream(stream)))
    return out


def variant(n: int, m: int) -> tuple[int, int, int, int]:
    """(tiles, stages, splits, fixed_m) of the kernel for n columns, m rows
    (fixed_m is 0: one build serves every m of its tile count)."""
    v = variant_full(n, m)
    return v["tiles"], v["stages"], v["splits"], 0


def variant_full(n: int, m: int) -> dict:
    """Every field of the launch shape for n columns, m rows."""
    f = [ctypes.c_int() for _ in range(5)]
    _check(load().qkv_front_variant(n, m, *[ctypes.byref(v) for v in f]))
    names = ("tiles", "stages", "splits", "kb", "consumer")
    out = {k: v.value for k, v in zip(names, f)}
    out["consumer"] = {CONSUMER_MMA_SYNC: "mma.sync", CONSUMER_TCGEN05: "tcgen05",
                       CONSUMER_RESIDENT: "resident"}[out["consumer"]]
    return out


def k_split(n: int) -> int:
    """CTAs per head splitting the 8192-long K (a power of two <= 16 with
    heads x splits within the SM count): 1 at N = 9216, 8 at N = 1152."""
    return variant_full(n, 1)["splits"]


def ring_stages(n: int, m: int) -> int:
    """Ring slots of the W / x stream for n columns and m tokens."""
    return variant_full(n, m)["stages"]


def prepare(n: int, num_kv_heads: int) -> None:
    """Set the kernel attributes the variants of n columns need (before graph capture)."""
    _check(load().qkv_front_prepare(n, num_kv_heads))


def compile_qkv_front(n: int, num_kv_heads: int) -> None:
    """The kernels are compiled ahead of time for sm_103a (build()); what is
    left to do before the first call or a graph capture is prepare()."""
    prepare(n, num_kv_heads)


def sm100_family(device=None) -> bool:
    """Whether the device is a compute capability 10.x part.  This library is
    built for 10.3 (GB300) only; other 10.x parts are refused at the first call."""
    if not torch.cuda.is_available():
        return False
    return torch.cuda.get_device_capability(device)[0] == 10


def unsupported_projection(weight, bias=None, is_neox_style: bool = False, cos_sin=None,
                           gather_output: bool = False, quantized: bool = False):
    """Why a QKV projection layer cannot use the fused front, or None: the
    front takes unquantized BF16 weights [N, 8192] with no bias, interleaved
    RoPE (pairs 2i, 2i + 1) from an FP32 [positions, 64] cos | sin table, and
    keeps its column shard (no gathered output)."""
    if quantized:
        return "quantized weights (the front streams BF16 weights)"
    if weight.dtype != torch.bfloat16:
        return f"{weight.dtype} weights (the front streams BF16 weights)"
    if weight.dim() != 2 or weight.shape[1] != HIDDEN:
        return f"weight shape {tuple(weight.shape)} (the front takes [N, {HIDDEN}])"
    if bias is not None:
        return "a bias on the projection"
    if is_neox_style:
        return "neox-style RoPE (the front rotates interleaved pairs 2i, 2i + 1)"
    if cos_sin is not None and (cos_sin.dtype != torch.float32 or cos_sin.dim() != 2
                                or cos_sin.shape[1] != HEAD_DIM):
        return f"a cos | sin table other than FP32 [positions, {HEAD_DIM}]"
    if gather_output:
        return "a gathered output (the front keeps each rank's column shard)"
    if weight.shape[0] % (2 * (Q_PER_KV + 1) * HEAD_DIM) != 0:
        return f"N = {weight.shape[0]} (the front takes 1152 columns per KV head)"
    return None


def status() -> int:
    """Read and clear the device status word (synchronizes the device)."""
    v = ctypes.c_uint()
    _check(load().qkv_front_status(ctypes.byref(v)))
    return v.value


def staging_bytes(m: int, n: int) -> int:
    """Device staging bytes qkv_front_from_host needs for m tokens, n columns."""
    return int(load().qkv_front_staging_bytes(m, n))


def qkv_front_from_host(x_host, positions_host, slots_host, out_host, weight, cos_sin, kv_cache,
                        staging, stream=None):
    """The whole call from host buffers: x / positions / slots in, the front
    run, out back, all on one stream in one library call.  Pinned host tensors
    are read and written by the kernels directly, pageable ones are copied;
    `staging` is a device uint8 tensor of at least staging_bytes(M, N) bytes."""
    for name, t in (("x_host", x_host), ("positions_host", positions_host),
                    ("slots_host", slots_host), ("out_host", out_host)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    M, N = x_host.shape[0], weight.shape[0]
    if (x_host.dtype != torch.bfloat16 or tuple(x_host.shape) != (M, HIDDEN)
            or out_host.dtype != torch.bfloat16 or tuple(out_host.shape) != (M, N)
            or positions_host.dtype != torch.int64 or slots_host.dtype != torch.int64
            or positions_host.numel() != M or slots_host.numel() != M):
        raise ValueError("host buffers must be bf16 x [M, 8192], int64 positions / slots [M], "
                         "bf16 out [M, N]")
    if not staging.is_cuda or staging.device != weight.device:
        raise ValueError("staging must be on the weights' device")
    _check(load().qkv_front_from_host(
        x_host.data_ptr(), positions_host.data_ptr(), slots_host.data_ptr(), out_host.data_ptr(),
        weight.data_ptr(), cos_sin.data_ptr(), cos_sin.shape[0], kv_cache.data_ptr(),
        kv_cache.shape[0], staging.data_ptr(), staging.numel() * staging.element_size(), M, N,
        kv_cache.shape[1], _stream(stream)))
    return out_host


def _epi_reason(qkv, positions, slots, cos_sin, kv_cache):
    if not all(t.is_cuda for t in (qkv, positions, slots, cos_sin, kv_cache)):
        return "tensors on a CUDA device"
    if any(t.device != qkv.device for t in (positions, slots, cos_sin, kv_cache)):
        return "tensors on different devices"
    if qkv.dtype != torch.bfloat16 or qkv.dim() != 2 or not qkv.is_contiguous():
        return "qkv other than a contiguous bf16 [tokens, N]"
    T = qkv.shape[0]
    for name, t in (("positions", positions), ("slots", slots)):
        if t.dtype != torch.int64 or t.dim() != 1 or t.shape[0] != T or not t.is_contiguous():
            return f"{name} other than contiguous int64 [{T}]"
    if (cos_sin.dtype != torch.float32 or cos_sin.dim() != 2 or cos_sin.shape[1] != HEAD_DIM
            or not cos_sin.is_contiguous()):
        return "a rotary table other than a contiguous fp32 [*, 64] one"
    if not kv_cache_layout_ok(kv_cache):
        return "a KV cache other than contiguous bf16 [pages, num_kv_heads, 16, 128]"
    if not supports_shape(qkv.shape[1], kv_cache.shape[1]):
        return f"{qkv.shape[1]} columns for {kv_cache.shape[1]} KV heads"
    return None


def _epi_args(qkv, positions, slots, cos_sin, kv_cache):
    return (qkv.data_ptr(), positions.data_ptr(), slots.data_ptr(), cos_sin.data_ptr(),
            cos_sin.shape[0], kv_cache.data_ptr(), kv_cache.shape[0], qkv.shape[0], qkv.shape[1],
            kv_cache.shape[1])


def qknorm_rope_kv_insert_unsupported(qkv, positions, slots, cos_sin, kv_cache) -> str | None:
    """Why the standalone epilogue cannot take this call, or None."""
    why = _epi_reason(qkv, positions, slots, cos_sin, kv_cache)
    if why is not None:
        return why
    with torch.cuda.device(qkv.device):
        r = load().qknorm_rope_kv_insert_unsupported(*_epi_args(qkv, positions, slots, cos_sin,
                                                                 kv_cache))
    return None if r is None else r.decode()


def qknorm_rope_kv_insert(qkv, positions, slots, cos_sin, kv_cache, stream=None):
    """In place on a bf16 projection output qkv [T, N]: q and k heads normed and
    rotated, each token's k / v heads inserted into kv_cache.  Returns qkv."""
    why = _epi_reason(qkv, positions, slots, cos_sin, kv_cache)
    if why is not None:
        raise ValueError(f"qknorm_rope_kv_insert does not support {why}")
    with torch.cuda.device(qkv.device):
        _check(load().qknorm_rope_kv_insert(*_epi_args(qkv, positions, slots, cos_sin, kv_cache),
                                            _stream(stream)))
    return qkv


def layer_front(x, stream_out, out, aux=None, weight=None, eps: float = 1e-6, stream=None):
    """The first layer's front (page layer_front, LayerFront.run): stream_out =
    x as fp32, aux = stream_out (if given), out = bf16 RMS norm of the row
    (times weight, if given).  x: bf16 or fp32 [rows, 8192].  Returns out."""
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("x must be bf16 or fp32")
    rows = x.shape[0]
    checks = [(x, x.dtype, "x"), (stream_out, torch.float32, "stream"),
              (out, torch.bfloat16, "out")] + ([(aux, torch.float32, "aux")] if aux is not None else [])
    for t, dt, name in checks:
        if (not t.is_cuda or t.dtype != dt or tuple(t.shape) != (rows, HIDDEN)
                or not t.is_contiguous() or t.device != x.device):
            raise ValueError(f"{name} must be a contiguous {dt} CUDA tensor [{rows}, {HIDDEN}]")
    if weight is not None and (weight.dtype != torch.bfloat16 or tuple(weight.shape) != (HIDDEN,)
                               or not weight.is_contiguous() or weight.device != x.device):
        raise ValueError(f"weight must be a contiguous bf16 CUDA tensor [{HIDDEN}]")
    with torch.cuda.device(x.device):
        _check(load().layer_front(x.data_ptr(), 1 if x.dtype == torch.float32 else 0,
                                  None if weight is None else weight.data_ptr(),
                                  stream_out.data_ptr(), None if aux is None else aux.data_ptr(),
                                  out.data_ptr(), rows, float(eps), _stream(stream)))
    return out


def _attn2_args(qkv, kv_cache, block_table, context_lens, out, window, scale, eps):
    """Checks the torch arguments of attn2 and returns (out, C arguments)."""
    R = context_lens.shape[0]
    nkv = kv_cache.shape[1]
    N = qkv.shape[1]
    cols = Q_PER_KV * nkv * HEAD_DIM
    if out is None:
        out = torch.empty(8 * R, cols, dtype=torch.bfloat16, device=qkv.device)
    for t, dt, shape, name in ((qkv, torch.bfloat16, (8 * R, N), "qkv"),
                               (out, torch.bfloat16, (8 * R, cols), "out"),
                               (context_lens, torch.int32, (R,), "context_lens")):
        if (not t.is_cuda or t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous()
                or t.device != qkv.device):
            raise ValueError(f"{name} must be a contiguous {dt} CUDA tensor {shape}")
    if (block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != R
            or not block_table.is_contiguous() or not block_table.is_cuda):
        raise ValueError("block_table must be a contiguous int32 CUDA tensor [R, max_blocks]")
    if not kv_cache_layout_ok(kv_cache) or not supports_shape(N, nkv):
        raise ValueError("cache must be bf16 [pages, nkv, 16, 128] and N = 1152 nkv")
    args = (qkv.data_ptr(), kv_cache.data_ptr(), kv_cache.shape[0], block_table.data_ptr(),
            block_table.shape[1], context_lens.data_ptr(), R, N, nkv, int(window), float(scale),
            float(eps), out.data_ptr())
    return out, args


def unsupported_attn2(layer) -> str | None:
    """Why attn2 cannot compute this attention layer, or None (page cute_ops,
    unsupported_attn2).  `layer` is any object with the attention layer's
    attributes use_o_norm, use_o_gate, head_dim, num_heads, num_kv_heads,
    scaling and rms_norm_eps.  attn2 is the o-norm + sigmoid-gate variant of
    the verify-step attention with 64-wide heads and 8 q heads per KV head;
    its scale and eps are call arguments (scale > 0, eps in (0, 1])."""
    if not layer.use_o_norm or not layer.use_o_gate:
        return "a layer without both the output RMS norm and the sigmoid output gate"
    if layer.head_dim != HEAD_DIM:
        return f"heads of {layer.head_dim} dims (attn2 has {HEAD_DIM})"
    if layer.num_kv_heads < 1 or layer.num_heads != Q_PER_KV * layer.num_kv_heads:
        return (f"{layer.num_heads} q heads over {layer.num_kv_heads} KV heads "
                f"(attn2 has {Q_PER_KV} q heads per KV head)")
    if not layer.scaling > 0:
        return f"a softmax scale of {layer.scaling} (attn2 takes a positive scale)"
    if not 0 < layer.rms_norm_eps <= 1:
        return f"an o-norm eps of {layer.rms_norm_eps} (attn2 takes eps in (0, 1])"
    return None


def attn2_unsupported_call(qkv, kv_cache, block_table, context_lens, out, window: int = 0,
                           scale: float = 0.125, eps: float = 1e-6) -> str | None:
    """Why attn2 would refuse this call into `out` (the binding's tensor
    checks, then the C ABI's host checks), or None."""
    try:
        out, args = _attn2_args(qkv, kv_cache, block_table, context_lens, out, window, scale, eps)
    except ValueError as e:
        return str(e)
    with torch.cuda.device(qkv.device):
        r = load().attn2_unsupported(*args)
    return None if r is None else r.decode()


def attn2(qkv, kv_cache, block_table, context_lens, out=None, window: int = 0,
          scale: float = 0.125, eps: float = 1e-6, splits=None, stream=None):
    """Verify-step paged attention with o-norm and sigmoid gate (the o_proj
    input).  qkv bf16 [8 R, N]; block_table int32 [R, max_blocks];
    context_lens int32 [R]; returns out bf16 [8 R, 512 num_kv_heads]."""
    out, args = _attn2_args(qkv, kv_cache, block_table, context_lens, out, window, scale, eps)
    with torch.cuda.device(qkv.device):
        if splits is None:
            _check(load().attn2(*args, _stream(stream)))
        else:
            _check(load().attn2_launch_splits(*args, int(splits), _stream(stream)))
    return out


def attn2_splits(num_reqs: int, num_kv_heads: int, max_blocks: int, window: int = 0) -> int:
    return int(load().attn2_splits(num_reqs, num_kv_heads, max_blocks, window))


def attn2_split_kv_workspace_bytes(num_reqs: int, num_kv_heads: int, splits: int) -> int:
    return int(load().attn2_split_kv_workspace_bytes(num_reqs, num_kv_heads, splits))


def attn2_split_kv_splits(num_reqs: int, num_kv_heads: int, max_blocks: int, window: int = 0) -> int:
    return int(load().attn2_split_kv_splits(num_reqs, num_kv_heads, max_blocks, window))


def attn2_split_kv_noalloc(qkv, kv_cache, block_table, context_lens, out=None, window: int = 0,
                           scale: float = 0.125, eps: float = 1e-6, splits: int = 0, stream=None):
    """attn2_split_kv for callers that cannot allocate device memory: the
    partials go to the library's own device array (256 slots; more raises
    QkvFrontError with QKVF_ERR_SIZES).  Pass `out` to keep the call free of
    allocations: with out=None this wrapper allocates the output with torch."""
    out, args = _attn2_args(qkv, kv_cache, block_table, context_lens, out, window, scale, eps)
    with torch.cuda.device(qkv.device):
        _check(load().attn2_split_kv_noalloc(*args, int(splits), _stream(stream)))
    return out


def attn2_split_kv(qkv, kv_cache, block_table, context_lens, workspace, out=None, window: int = 0,
                   scale: float = 0.125, eps: float = 1e-6, splits: int = 0, stream=None):
    """attn2 with the split-KV engine: partials in `workspace` (a uint8 CUDA
    tensor of at least attn2_split_kv_workspace_bytes bytes), merged by a
    second grid."""
    out, args = _attn2_args(qkv, kv_cache, block_table, context_lens, out, window, scale, eps)
    if (not workspace.is_cuda or workspace.dtype != torch.uint8 or not workspace.is_contiguous()
            or workspace.device != qkv.device):
        raise ValueError("workspace must be a contiguous uint8 CUDA tensor on qkv's device")
    with torch.cuda.device(qkv.device):
        _check(load().attn2_split_kv(*args, int(splits), workspace.data_ptr(), workspace.numel(),
                                     _stream(stream)))
    return out


def selftest_wait(timeout_ns: int, stream=None) -> None:
    _check(load().qkv_front_selftest_wait(int(timeout_ns), _stream(stream)))


def set_pdl(enable: bool) -> None:
    """Launch the library's kernels with PDL (default) or plainly stream-ordered."""
    _check(load().qkv_front_set_pdl(1 if enable else 0))


def set_wait_limit(ns: int) -> None:
    _check(load().qkv_front_set_wait_limit(int(ns)))
