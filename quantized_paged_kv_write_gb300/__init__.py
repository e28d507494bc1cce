"""Python binding of libkvq (include/kvq.h): quantize-on-write into a paged KV
cache and paged decode attention over it, on NVIDIA GB300 (sm_103a).

This module only marshals arguments: every step of the path runs in the CUDA
kernels of ``libkvq.so``.  PyTorch provides device memory and streams.  There
is no fallback: if the library is missing or the device is not CUDA, the
calls raise.

The function names follow the C ABI: ``kvq_quantize_write``,
``kvq_decode_workspace_size``, ``kvq_paged_decode``, ``kvq_device_errors``,
``kvq_status_string``.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

# enum values of include/kvq.h
KVQ_OK = 0
KVQ_ERR_INVALID_ARG = -1
KVQ_ERR_UNSUPPORTED = -2
KVQ_ERR_WORKSPACE = -3
KVQ_ERR_CUDA = -4

DTYPES = {"int8": 0, "int4": 1, "fp8_e4m3fn": 2, "int2": 3}
GRANS = {"token_head": 0, "token_group": 1, "block_channel": 2}

DEVERR_SLOT_RANGE = 1 << 0
DEVERR_BLOCK_RANGE = 1 << 1
DEVERR_CONTEXT_RANGE = 1 << 2
DEVERR_TIMEOUT = 1 << 3
DEVERR_CHANNEL_RUN = 1 << 4

EXPORTED_SYMBOLS = (
    "kvq_quantize_write", "kvq_decode_workspace_size", "kvq_paged_decode",
    "kvq_device_errors", "kvq_status_string", "kvq_version", "kvq_paged_decode_noalloc",
    "kvq_write_decode", "kvq_prefetch_blocks", "kvq_kivi_append", "kvq_kivi_decode", "kvq_build_id",
)

# size of the static scratch of kvq_paged_decode_noalloc (include/kvq.h)
NOALLOC_SCRATCH_BYTES = 32 << 20


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {kvq_status_string(status)} ({status})")


class _Format(ctypes.Structure):
    _fields_ = [
        ("k_dtype", ctypes.c_int32), ("v_dtype", ctypes.c_int32),
        ("k_gran", ctypes.c_int32), ("v_gran", ctypes.c_int32),
        ("k_group", ctypes.c_int32), ("v_group", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32), ("rotation", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64), ("rotation_signs", ctypes.c_uint32 * 4),
    ]


class _Caches(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p)]


class _Scales(ctypes.Structure):
    _fields_ = [("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


_lib = None
_lib_lock = threading.Lock()


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libkvq.so (built in-tree by ``build.py``)."""
    global _lib
    with _lib_lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it with `python -m quantized_paged_kv_write_gb300.build` "
                "(nvcc for sm_103a); there is no fallback implementation")
        lib = ctypes.CDLL(p)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        fmtp = ctypes.POINTER(_Format)
        lib.kvq_quantize_write.argtypes = [vp, vp, vp, i64, fmtp, _Caches, _Scales, vp]
        lib.kvq_quantize_write.restype = ctypes.c_int
        lib.kvq_decode_workspace_size.argtypes = [fmtp, i32, i32, i32, ctypes.POINTER(ctypes.c_size_t)]
        lib.kvq_decode_workspace_size.restype = ctypes.c_int
        lib.kvq_paged_decode.argtypes = [vp, i32, i32, fmtp, _Caches, _Scales, vp, i32, vp, i32, vp, vp,
                                         ctypes.c_size_t, vp]
        lib.kvq_paged_decode.restype = ctypes.c_int
        lib.kvq_write_decode.argtypes = [vp, vp, vp, i32, i32, fmtp, _Caches, _Scales, vp, i32, vp, i32, vp, vp,
                                         ctypes.c_size_t, vp]
        lib.kvq_write_decode.restype = ctypes.c_int
        lib.kvq_kivi_append.argtypes = [vp, vp, i32, fmtp, _Caches, _Scales, vp, i32, vp, vp, vp, vp]
        lib.kvq_kivi_append.restype = ctypes.c_int
        lib.kvq_kivi_decode.argtypes = [vp, i32, i32, fmtp, _Caches, _Scales, vp, i32, vp, i32, vp, vp, vp, vp,
                                        ctypes.c_size_t, vp]
        lib.kvq_kivi_decode.restype = ctypes.c_int
        lib.kvq_prefetch_blocks.argtypes = [fmtp, _Caches, _Scales, i64, vp, vp, i32, _Caches, _Scales, vp]
        lib.kvq_prefetch_blocks.restype = ctypes.c_int
        lib.kvq_paged_decode_noalloc.argtypes = [vp, i32, i32, fmtp, _Caches, _Scales, vp, i32, vp, i32, vp, vp]
        lib.kvq_paged_decode_noalloc.restype = ctypes.c_int
        lib.kvq_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32, vp]
        lib.kvq_device_errors.restype = ctypes.c_int
        lib.kvq_status_string.argtypes = [i32]
        lib.kvq_status_string.restype = ctypes.c_char_p
        lib.kvq_version.argtypes = []
        lib.kvq_version.restype = i32
        lib.kvq_build_id.argtypes = []
        lib.kvq_build_id.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


@dataclasses.dataclass(frozen=True)
class CacheFormat:
    """Host description of one layer's paged cache (kvq_format)."""
    k_dtype: str
    v_dtype: str
    k_gran: str
    v_gran: str
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    block_size: int = 16
    k_group: int = 0
    v_group: int = 0
    # randomized Walsh-Hadamard rotation of K and V rows (include/kvq.h):
    # None, or 4 words of sign bits (bit c set -> sigma_c = -1)
    rotation_signs: Optional[tuple] = None

    def as_c(self) -> _Format:
        rot = self.rotation_signs is not None
        signs = (ctypes.c_uint32 * 4)(*(tuple(int(w) & 0xFFFFFFFF for w in self.rotation_signs) if rot
                                        else (0, 0, 0, 0)))
        return _Format(DTYPES[self.k_dtype], DTYPES[self.v_dtype], GRANS[self.k_gran], GRANS[self.v_gran],
                       self.k_group, self.v_group, self.num_kv_heads, self.head_dim, self.block_size,
                       1 if rot else 0, self.num_blocks, signs)

    def code_row_bytes(self, which: str) -> int:
        dt = self.k_dtype if which == "k" else self.v_dtype
        return {"int4": self.head_dim // 2, "int2": self.head_dim // 4}.get(dt, self.head_dim)

    def scale_shape(self, which: str):
        gran = self.k_gran if which == "k" else self.v_gran
        group = self.k_group if which == "k" else self.v_group
        nb, bs, h, d = self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim
        if gran == "token_head":
            return (nb, bs, h)
        if gran == "token_group":
            return (nb, bs, h, d // group)
        return (nb, h, d)


def cache_format(k_fmt, v_fmt, num_kv_heads: int, head_dim: int, num_blocks: int,
                 block_size: int = 16, rotation_signs=None) -> CacheFormat:
    """Build a CacheFormat from two objects with .dtype/.gran/.group names;
    rotation_signs (4 words of sign bits) turns on the Walsh-Hadamard rotation."""
    rs = None if rotation_signs is None else tuple(int(w) for w in rotation_signs)
    return CacheFormat(k_fmt.dtype, v_fmt.dtype, k_fmt.gran, v_fmt.gran, num_kv_heads, head_dim,
                       num_blocks, block_size, k_fmt.group, v_fmt.group, rs)


def allocate_cache(fmt: CacheFormat, device="cuda", zero: bool = True) -> dict:
    """Device buffers of one layer's cache: codes (uint8) and FP32 scales."""
    alloc = torch.zeros if zero else torch.empty
    out = {}
    for w in ("k", "v"):
        out[w + "_cache"] = alloc((fmt.num_blocks, fmt.block_size, fmt.num_kv_heads, fmt.code_row_bytes(w)),
                                  dtype=torch.uint8, device=device)
        out[w + "_scale"] = alloc(fmt.scale_shape(w), dtype=torch.float32, device=device)
    return out


def allocate_host_pool(fmt: CacheFormat, num_blocks: int) -> dict:
    """A pool of num_blocks cache blocks in pinned host memory, with the
    per-block layout of fmt (for kvq_prefetch_blocks)."""
    out = {}
    for w in ("k", "v"):
        out[w + "_cache"] = torch.zeros((num_blocks, fmt.block_size, fmt.num_kv_heads, fmt.code_row_bytes(w)),
                                        dtype=torch.uint8).pin_memory()
        shape = (num_blocks,) + tuple(fmt.scale_shape(w)[1:])
        out[w + "_scale"] = torch.zeros(shape, dtype=torch.float32).pin_memory()
    return out


def _host_ptr(t: torch.Tensor, dtype, what: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if t.is_cuda or not t.is_pinned():
        raise ValueError(f"{what} must be a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _ptr(t: torch.Tensor, dtype=None, what: str = "tensor") -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device: a pointer into another
        # GPU's memory would be read by the wrong device's kernels
        raise ValueError(f"{what} is on {t.device} but the current device is cuda:{torch.cuda.current_device()} "
                         "(torch.cuda.set_device)")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _caches(c: dict) -> tuple:
    return (_Caches(_ptr(c["k_cache"], torch.uint8, "k_cache"), _ptr(c["v_cache"], torch.uint8, "v_cache")),
            _Scales(_ptr(c["k_scale"], torch.float32, "k_scale"), _ptr(c["v_scale"], torch.float32, "v_scale")))


def kvq_status_string(status: int) -> str:
    return load_library().kvq_status_string(int(status)).decode()


def kvq_version() -> int:
    return int(load_library().kvq_version())


def kvq_build_id() -> str:
    """Hash of the sources the loaded library was built from (build.source_hash)."""
    return load_library().kvq_build_id().decode()


def kvq_quantize_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, fmt: CacheFormat,
                       cache: dict, stream=None) -> None:
    """Quantize BF16 K, V [num_tokens, H_kv, head_dim] into the cache at
    slot_mapping (int64 [num_tokens]); asynchronous on ``stream``."""
    lib = load_library()
    n = int(slot_mapping.shape[0])
    exp = (n, fmt.num_kv_heads, fmt.head_dim)
    if tuple(k.shape) != exp or tuple(v.shape) != exp:
        raise ValueError(f"k and v must have shape {exp}")
    cf = fmt.as_c()
    caches, scales = _caches(cache)
    st = lib.kvq_quantize_write(_ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"),
                                _ptr(slot_mapping, torch.int64, "slot_mapping"), n, ctypes.byref(cf),
                                caches, scales, _stream(stream))
    if st != KVQ_OK:
        raise KvqError(st, "kvq_quantize_write")


def kvq_decode_workspace_size(fmt: CacheFormat, batch: int, num_q_heads: int, max_context_len: int) -> int:
    lib = load_library()
    out = ctypes.c_size_t(0)
    cf = fmt.as_c()
    st = lib.kvq_decode_workspace_size(ctypes.byref(cf), int(batch), int(num_q_heads), int(max_context_len),
                                       ctypes.byref(out))
    if st != KVQ_OK:
        raise KvqError(st, "kvq_decode_workspace_size")
    return int(out.value)


def kvq_paged_decode(q: torch.Tensor, fmt: CacheFormat, cache: dict, block_tables: torch.Tensor,
                     context_lens: torch.Tensor, max_context_len: int, out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One decode step: q BF16 [B, H_q, d] -> out FP32 [B, H_q, d]."""
    lib = load_library()
    bsz, hq, d = (int(x) for x in q.shape)
    if d != fmt.head_dim:
        raise ValueError("q head_dim does not match the cache format")
    if out is None:
        out = torch.empty((bsz, hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = kvq_decode_workspace_size(fmt, bsz, hq, max_context_len)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    if block_tables.dim() != 2 or block_tables.shape[0] != bsz or context_lens.shape != (bsz,):
        raise ValueError("block_tables must be [B, max_blocks] and context_lens [B]")
    cf = fmt.as_c()
    caches, scales = _caches(cache)
    st = lib.kvq_paged_decode(_ptr(q, torch.bfloat16, "q"), bsz, hq, ctypes.byref(cf), caches, scales,
                              _ptr(block_tables, torch.int32, "block_tables"), int(block_tables.shape[1]),
                              _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len),
                              _ptr(out, torch.float32, "out"), _ptr(workspace, torch.uint8, "workspace"),
                              int(workspace.numel()), _stream(stream))
    if st != KVQ_OK:
        raise KvqError(st, "kvq_paged_decode")
    return out


def kvq_write_decode(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, fmt: CacheFormat, cache: dict,
                     block_tables: torch.Tensor, context_lens: torch.Tensor, max_context_len: int,
                     out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """One decode step that first writes each sequence's new token: k_new and
    v_new BF16 [B, H_kv, d] go to position context_lens[b] - 1 (slot from the
    block table), then q BF16 [B, H_q, d] attends over [0, context_lens[b]).
    Same results as kvq_quantize_write on those slots + kvq_paged_decode."""
    lib = load_library()
    bsz, hq, d = (int(x) for x in q.shape)
    if d != fmt.head_dim:
        raise ValueError("q head_dim does not match the cache format")
    want = (bsz, fmt.num_kv_heads, fmt.head_dim)
    if tuple(k_new.shape) != want or tuple(v_new.shape) != want:
        raise ValueError(f"k_new and v_new must be {list(want)}")
    if out is None:
        out = torch.empty((bsz, hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = kvq_decode_workspace_size(fmt, bsz, hq, max_context_len)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    if block_tables.dim() != 2 or block_tables.shape[0] != bsz or context_lens.shape != (bsz,):
        raise ValueError("block_tables must be [B, max_blocks] and context_lens [B]")
    cf = fmt.as_c()
    caches, scales = _caches(cache)
    st = lib.kvq_write_decode(_ptr(q, torch.bfloat16, "q"), _ptr(k_new, torch.bfloat16, "k_new"),
                              _ptr(v_new, torch.bfloat16, "v_new"), bsz, hq, ctypes.byref(cf), caches, scales,
                              _ptr(block_tables, torch.int32, "block_tables"), int(block_tables.shape[1]),
                              _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len),
                              _ptr(out, torch.float32, "out"), _ptr(workspace, torch.uint8, "workspace"),
                              int(workspace.numel()), _stream(stream))
    if st != KVQ_OK:
        raise KvqError(st, "kvq_write_decode")
    return out


def kvq_paged_decode_noalloc(q: torch.Tensor, fmt: CacheFormat, cache: dict, block_tables: torch.Tensor,
                             context_lens: torch.Tensor, max_context_len: int, out: torch.Tensor,
                             stream=None) -> torch.Tensor:
    """kvq_paged_decode with the library's static scratch instead of a
    workspace, for callers that cannot allocate device memory at the call.
    ``out`` must be given (the call allocates nothing).  Calls share the
    scratch: order them if their work could overlap on the GPU."""
    lib = load_library()
    bsz, hq, d = (int(x) for x in q.shape)
    if d != fmt.head_dim:
        raise ValueError("q head_dim does not match the cache format")
    if block_tables.dim() != 2 or block_tables.shape[0] != bsz or context_lens.shape != (bsz,):
        raise ValueError("block_tables must be [B, max_blocks] and context_lens [B]")
    cf = fmt.as_c()
    caches, scales = _caches(cache)
    st = lib.kvq_paged_decode_noalloc(_ptr(q, torch.bfloat16, "q"), bsz, hq, ctypes.byref(cf), caches, scales,
                                      _ptr(block_tables, torch.int32, "block_tables"),
                                      int(block_tables.shape[1]), _ptr(context_lens, torch.int32, "context_lens"),
                                      int(max_context_len), _ptr(out, torch.float32, "out"), _stream(stream))
    if st != KVQ_OK:
        raise KvqError(st, "kvq_paged_decode_noalloc")
    return out


def allocate_residual(fmt: CacheFormat, batch: int, device="cuda") -> dict:
    """The full-precision tail of a per-channel K cache (kvq_kivi_append /
    kvq_kivi_decode): BF16 K and V rows [batch, 16, H_kv, d]."""
    shape = (batch, fmt.block_size, fmt.num_kv_heads, fmt.head_dim)
    return {"k": torch.zeros(shape, dtype=torch.bfloat16, device=device),
            "v": torch.zeros(shape, dtype=torch.bfloat16, device=device)}


def kvq_kivi_append(k_new: torch.Tensor, v_new: torch.Tensor, fmt: CacheFormat, cache: dict,
                    block_tables: torch.Tensor, context_lens: torch.Tensor, residual: dict, stream=None) -> None:
    """One token per sequence (k_new, v_new BF16 [B, H_kv, d]) at position
    context_lens[b] - 1; a block that it completes is quantized into the cache."""
    lib = load_library()
    bsz = int(k_new.shape[0])
    cf = fmt.as_c()
    caches, scales = _caches(cache)
    st = lib.kvq_kivi_append(_ptr(k_new, torch.bfloat16, "k_new"), _ptr(v_new, torch.bfloat16, "v_new"), bsz,
                             ctypes.byref(cf), caches, scales, _ptr(block_tables, torch.int32, "block_tables"),
                             int(block_tables.shape[1]), _ptr(context_lens, torch.int32, "context_lens"),
                             _ptr(residual["k"], torch.bfloat16, "residual k"),
                             _ptr(residual["v"], torch.bfloat16, "residual v"), _stream(stream))
    if st != KVQ_OK:
        raise KvqError(st, "kvq_kivi_append")


def kvq_kivi_decode(q: torch.Tensor, fmt: CacheFormat, cache: dict, block_tables: torch.Tensor,
                    context_lens: torch.Tensor, max_context_len: int, residual: dict,
                    out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """Decode over the quantized complete blocks and the residual's tail."""
    lib = load_library()
    bsz, hq, d = (int(x) for x in q.shape)
    if out is None:
        out = torch.empty((bsz, hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = kvq_decode_workspace_size(fmt, bsz, hq, max_context_len)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    cf = fmt.as_c()
    caches, scales = _caches(cache)
    st = lib.kvq_kivi_decode(_ptr(q, torch.bfloat16, "q"), bsz, hq, ctypes.byref(cf), caches, scales,
                             _ptr(block_tables, torch.int32, "block_tables"), int(block_tables.shape[1]),
                             _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len),
                             _ptr(residual["k"], torch.bfloat16, "residual k"),
                             _ptr(residual["v"], torch.bfloat16, "residual v"),
                             _ptr(out, torch.float32, "out"), _ptr(workspace, torch.uint8, "workspace"),
                             int(workspace.numel()), _stream(stream))
    if st != KVQ_OK:
        raise KvqError(st, "kvq_kivi_decode")
    return out


def kvq_prefetch_blocks(host_pool: dict, src_blocks: torch.Tensor, dst_blocks: torch.Tensor, fmt: CacheFormat,
                        cache: dict, stream=None) -> None:
    """Copy host pool block src_blocks[i] into device cache block
    dst_blocks[i] (int32 CUDA tensors), asynchronously on `stream`."""
    lib = load_library()
    n = int(src_blocks.numel())
    if dst_blocks.numel() != n:
        raise ValueError("src_blocks and dst_blocks differ in length")
    hc = _Caches(_host_ptr(host_pool["k_cache"], torch.uint8, "host k_cache"),
                 _host_ptr(host_pool["v_cache"], torch.uint8, "host v_cache"))
    hs = _Scales(_host_ptr(host_pool["k_scale"], torch.float32, "host k_scale"),
                 _host_ptr(host_pool["v_scale"], torch.float32, "host v_scale"))
    cf = fmt.as_c()
    caches, scales = _caches(cache)
    st = lib.kvq_prefetch_blocks(ctypes.byref(cf), hc, hs, int(host_pool["k_cache"].shape[0]),
                                 _ptr(src_blocks, torch.int32, "src_blocks"), _ptr(dst_blocks, torch.int32, "dst_blocks"),
                                 n, caches, scales, _stream(stream))
    if st != KVQ_OK:
        raise KvqError(st, "kvq_prefetch_blocks")


def kvq_device_errors(clear: bool = True, stream=None) -> int:
    """Synchronize the stream and return the sticky device error bits."""
    lib = load_library()
    bits = ctypes.c_uint32(0)
    st = lib.kvq_device_errors(ctypes.byref(bits), 1 if clear else 0, _stream(stream))
    if st != KVQ_OK:
        raise KvqError(st, "kvq_device_errors")
    return int(bits.value)


__all__ = [n for n in dir() if n.startswith("kvq_")] + [
    "CacheFormat", "cache_format", "allocate_cache", "allocate_host_pool", "allocate_residual", "load_library", "KvqError", "LIB_PATH",
    "EXPORTED_SYMBOLS"]
