"""ctypes binding of libdecode_attn.so (include/decode_attn.h), same names as the C ABI.

Argument marshalling only: each function turns ``torch.Tensor`` arguments into
``da_tensor_t`` descriptors (data pointer, dtype, shape, strides in elements),
passes the current CUDA stream, and raises :class:`DecodeAttnError` on a
nonzero status. Every step of the computation runs in the library's kernels.
The library must have been built (``decode_attention_output_gb300.build``);
there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import struct
import threading

import torch

from . import build as _build

DA_DTYPE_BF16, DA_DTYPE_F32, DA_DTYPE_I32, DA_DTYPE_E4M3 = 1, 2, 3, 4
_DTYPES = {torch.bfloat16: DA_DTYPE_BF16, torch.float32: DA_DTYPE_F32, torch.int32: DA_DTYPE_I32,
           torch.float8_e4m3fn: DA_DTYPE_E4M3}

# every symbol declared in include/decode_attn.h
EXPORTS = ("decode_attn_fwd", "decode_attn_only", "decode_attn_only_noalloc", "decode_attn_fwd_paged",
           "decode_attn_only_paged", "decode_attn_fwd_fp8", "decode_attn_only_fp8", "decode_attn_scores", "decode_attn_oproj", "decode_attn_set_option", "decode_attn_get_option", "decode_attn_last_device_error", "decode_attn_device_error",
           "decode_attn_release", "decode_attn_status_str")


class da_tensor_t(ctypes.Structure):  # noqa: N801 - mirrors the C name
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class DecodeAttnError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


_lib = None
_lock = threading.Lock()


def load_library(path: str) -> ctypes.CDLL:
    """Loads a build of the library at ``path`` with its argument types declared, without
    making it the one the entry points below call (see :func:`use_library`)."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run decode_attention_output_gb300.build.build() first")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p  # a packed da_tensor_t (see _pack), a pointer to one, or NULL
    vp, f32, i64 = ctypes.c_void_p, ctypes.c_float, ctypes.c_int64
    lib.decode_attn_fwd.argtypes = [P, P, P, P, P, P, f32, vp]
    lib.decode_attn_only.argtypes = [P, P, P, P, P, f32, vp]
    lib.decode_attn_only_noalloc.argtypes = [P, P, P, P, P, f32, vp]
    lib.decode_attn_fwd_paged.argtypes = [P, P, P, P, P, P, P, f32, vp]
    lib.decode_attn_only_paged.argtypes = [P, P, P, P, P, P, f32, vp]
    lib.decode_attn_fwd_fp8.argtypes = [P, P, P, P, P, P, f32, f32, f32, vp]
    lib.decode_attn_only_fp8.argtypes = [P, P, P, P, P, f32, f32, f32, vp]
    lib.decode_attn_scores.argtypes = [P, P, P, P, vp]
    lib.decode_attn_oproj.argtypes = [P, P, P, vp]
    lib.decode_attn_set_option.argtypes = [ctypes.c_char_p, i64]
    lib.decode_attn_get_option.argtypes = [ctypes.c_char_p, ctypes.POINTER(i64)]
    lib.decode_attn_last_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    lib.decode_attn_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    lib.decode_attn_release.argtypes = []
    lib.decode_attn_release.restype = None
    lib.decode_attn_status_str.argtypes = [ctypes.c_int]
    lib.decode_attn_status_str.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name not in ("decode_attn_release", "decode_attn_status_str"):
            getattr(lib, name).restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads the library (once). Fails loudly if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(path or _build.lib_path())
    return _lib


def use_library(lib: ctypes.CDLL | None) -> ctypes.CDLL | None:
    """Makes ``lib`` (from :func:`load_library`) the library every entry point below calls
    and returns the previous one; the tests use it to run the bounds-checked build."""
    global _lib
    with _lock:
        prev, _lib = _lib, lib
    return prev


def describe(t: torch.Tensor | None) -> da_tensor_t | None:
    """da_tensor_t view of a tensor (no copy)."""
    if t is None:
        return None
    return da_tensor_t.from_buffer_copy(_pack(t))


# da_tensor_t as bytes: data pointer, dtype, ndim, shape[4], stride[4] (little endian,
# no padding: the C struct has none either). Packing the fields in one call costs a
# third of filling a ctypes structure field by field, and the calls below are made
# once per tensor per step.
_DESC = struct.Struct("<Qii4q4q")
_PAD = ((0, 0, 0, 0), (0, 0, 0), (0, 0), (0,), ())
assert _DESC.size == ctypes.sizeof(da_tensor_t)


def _pack(t: torch.Tensor) -> bytes:
    code = _DTYPES.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    shape = t.shape
    n = len(shape)
    if n > 4:
        raise ValueError("at most 4 dimensions")
    pad = _PAD[n]
    return _DESC.pack(t.data_ptr() if t.numel() else 0, code, n, *shape, *pad, *t.stride(), *pad)


def _ref(t):
    """Argument for a `const da_tensor_t*` parameter: packed bytes, or NULL for None."""
    return None if t is None else _pack(t)


# The raw handle of the current stream without building a torch.cuda.Stream object
# (0.3 us against 2.9 us per call); the public route where torch lacks the accessor.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int | None:
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise DecodeAttnError(fn, code, status_str(code))


def status_str(code: int) -> str:
    return load().decode_attn_status_str(int(code)).decode()


def decode_attn_fwd(q, k_cache, v_cache, seq_lens, o_weight, out, scale: float, stream=None) -> torch.Tensor:
    """out[B, N] = (softmax(scale * q K^T) V)_flat . o_weight; returns ``out``."""
    lib = _lib or load()  # the lock only until the library is loaded
    ds = [_ref(x) for x in (q, k_cache, v_cache, seq_lens, o_weight, out)]
    _check("decode_attn_fwd", lib.decode_attn_fwd(*ds, float(scale), _stream(stream)))
    return out


def decode_attn_only(q, k_cache, v_cache, seq_lens, attn_out, scale: float, stream=None) -> torch.Tensor:
    """attn_out[B, Hq, D] = softmax(scale * q K^T) V (bf16); returns ``attn_out``."""
    lib = _lib or load()  # the lock only until the library is loaded
    ds = [_ref(x) for x in (q, k_cache, v_cache, seq_lens, attn_out)]
    _check("decode_attn_only", lib.decode_attn_only(*ds, float(scale), _stream(stream)))
    return attn_out


def decode_attn_only_noalloc(q, k_cache, v_cache, seq_lens, attn_out, scale: float, stream=None) -> torch.Tensor:
    """decode_attn_only without any device allocation by the library: for callers that
    must not allocate GPU memory at run time (memory reserved up front by their own
    pool, or no device-wide synchronisation allowed on the request path). Uses a
    fixed 8 MiB scratch array inside the library; calls that overlap on the GPU race
    on it. Raises DecodeAttnError (DA_ERR_SCRATCH) when a call needs more scratch."""
    lib = _lib or load()  # the lock only until the library is loaded
    ds = [_ref(x) for x in (q, k_cache, v_cache, seq_lens, attn_out)]
    _check("decode_attn_only_noalloc",
           lib.decode_attn_only_noalloc(*ds, float(scale), _stream(stream)))
    return attn_out


def decode_attn_fwd_paged(q, k_pages, v_pages, block_table, seq_lens, o_weight, out, scale: float,
                          stream=None) -> torch.Tensor:
    """decode_attn_fwd over a paged cache: k_pages / v_pages [num_blocks, Hkv, block_size, D],
    block_table [B, max_blocks] int32; returns ``out``."""
    lib = _lib or load()  # the lock only until the library is loaded
    ds = [_ref(x) for x in (q, k_pages, v_pages, block_table, seq_lens, o_weight, out)]
    _check("decode_attn_fwd_paged", lib.decode_attn_fwd_paged(*ds, float(scale), _stream(stream)))
    return out


def decode_attn_only_paged(q, k_pages, v_pages, block_table, seq_lens, attn_out, scale: float,
                           stream=None) -> torch.Tensor:
    """decode_attn_only over a paged cache (see decode_attn_fwd_paged); returns ``attn_out``."""
    lib = _lib or load()  # the lock only until the library is loaded
    ds = [_ref(x) for x in (q, k_pages, v_pages, block_table, seq_lens, attn_out)]
    _check("decode_attn_only_paged",
           lib.decode_attn_only_paged(*ds, float(scale), _stream(stream)))
    return attn_out


def decode_attn_fwd_fp8(q, k_cache, v_cache, seq_lens, o_weight, out, scale: float, k_scale: float, v_scale: float,
                        stream=None) -> torch.Tensor:
    """decode_attn_fwd over an fp8 cache: k_cache / v_cache torch.float8_e4m3fn, the keys
    and values being k_cache * k_scale and v_cache * v_scale; returns ``out``."""
    lib = _lib or load()  # the lock only until the library is loaded
    ds = [_ref(x) for x in (q, k_cache, v_cache, seq_lens, o_weight, out)]
    _check("decode_attn_fwd_fp8", lib.decode_attn_fwd_fp8(*ds, float(scale), float(k_scale),
                                                          float(v_scale), _stream(stream)))
    return out


def decode_attn_only_fp8(q, k_cache, v_cache, seq_lens, attn_out, scale: float, k_scale: float, v_scale: float,
                         stream=None) -> torch.Tensor:
    """decode_attn_only over an fp8 cache (see decode_attn_fwd_fp8); returns ``attn_out``."""
    lib = _lib or load()  # the lock only until the library is loaded
    ds = [_ref(x) for x in (q, k_cache, v_cache, seq_lens, attn_out)]
    _check("decode_attn_only_fp8", lib.decode_attn_only_fp8(*ds, float(scale), float(k_scale),
                                                            float(v_scale), _stream(stream)))
    return attn_out


def decode_attn_scores(q, k_cache, seq_lens, scores, stream=None) -> torch.Tensor:
    """scores[B, Hq, Lcap] (fp32) = q K^T for t < seq_lens[b]; returns ``scores``."""
    lib = _lib or load()  # the lock only until the library is loaded
    ds = [_ref(x) for x in (q, k_cache, seq_lens, scores)]
    _check("decode_attn_scores", lib.decode_attn_scores(*ds, _stream(stream)))
    return scores


def decode_attn_oproj(attn_flat, o_weight, out, stream=None) -> torch.Tensor:
    """out[B, N] = attn_flat[B, K] . o_weight[K, N] (bf16); returns ``out``."""
    lib = _lib or load()  # the lock only until the library is loaded
    ds = [_ref(x) for x in (attn_flat, o_weight, out)]
    _check("decode_attn_oproj", lib.decode_attn_oproj(*ds, _stream(stream)))
    return out


def decode_attn_set_option(key: str, value: int) -> None:
    _check("decode_attn_set_option", load().decode_attn_set_option(key.encode(), int(value)))


def decode_attn_get_option(key: str) -> int:
    v = ctypes.c_int64(0)
    _check("decode_attn_get_option", load().decode_attn_get_option(key.encode(), ctypes.byref(v)))
    return int(v.value)


def decode_attn_last_device_error(stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device error word (the
    workspace's and the no-allocation scratch's, OR-ed); a non-zero word also resets
    the completion counters beside it."""
    code = ctypes.c_int32(0)
    _check("decode_attn_last_device_error",
           load().decode_attn_last_device_error(_stream(stream), ctypes.byref(code)))
    return int(code.value)


def decode_attn_device_error(stream=None) -> int:
    """decode_attn_last_device_error under its earlier name."""
    code = ctypes.c_int32(0)
    _check("decode_attn_device_error", load().decode_attn_device_error(_stream(stream), ctypes.byref(code)))
    return int(code.value)


def decode_attn_release() -> None:
    load().decode_attn_release()
