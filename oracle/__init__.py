"""fp64 CPU oracle for the decode-attention + output-projection step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. The
library (``decode_attention_output_gb300``) never imports it, and this module
imports nothing from the library.

The arithmetic lives in ``decode_oracle.c`` (plain C, double precision,
OpenMP over (batch, head)); this file only compiles it with gcc and marshals
numpy arrays through ctypes. Inputs are bf16 bit patterns held in ``uint16``
arrays, so the oracle reads exactly the bits the GPU reads.

What it computes: the three contractions of the page "PyPTO 开箱性能调优实战
Decode Attention 多 Matmul 独立 TileShape 配置 F-16", section "代码对比"
(scores = q_grouped . k_cache^T, scale + softmax, attn = weights . v_cache,
out = attn_flat . o_weight), with the shapes of its table "三个 Matmul 的 Shape
特征分析".
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "decode_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
CFLAGS = ["-O2", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC", "-std=c99"]


def build(src: str = SRC, out_dir: str = BUILD_DIR, tag: str = "liboracle") -> str:
    """Compile ``src`` into ``out_dir/<tag>-<hash>.so`` (skipped when up to date)."""
    with open(src, "rb") as f:
        digest = hashlib.sha1(f.read() + " ".join(CFLAGS).encode()).hexdigest()[:12]
    os.makedirs(out_dir, exist_ok=True)
    out = os.path.join(out_dir, f"{tag}-{digest}.so")
    if not os.path.exists(out):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, out)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


_i64 = ctypes.c_int64
_dbl = ctypes.c_double
_p = ctypes.c_void_p


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u16(a, name: str) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"{name}: expected uint16 bf16 bit patterns, got {a.dtype}")
    return a


class Oracle:
    """ctypes front end of ``decode_oracle.c``; ``lib_path`` defaults to a fresh build."""

    def __init__(self, lib_path: str | None = None):
        self.lib_path = lib_path or build()
        lib = ctypes.CDLL(self.lib_path)
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_group_scores.argtypes = [_p, _i64, _p, _i64, _i64, _i64, _i64, _p]
        lib.oracle_group_scores.restype = None
        lib.oracle_group_attention.argtypes = [_p, _i64, _p, _i64, _p, _i64, _i64, _i64, _i64, _dbl, _p]
        lib.oracle_group_attention.restype = ctypes.c_int
        lib.oracle_group_attention_split.argtypes = [_p, _i64, _p, _i64, _p, _i64, _i64, _i64, _i64, _dbl,
                                                     _i64, _p]
        lib.oracle_group_attention_split.restype = ctypes.c_int
        lib.oracle_oproj.argtypes = [_p, _p, _i64, _i64, _i64, _p]
        lib.oracle_oproj.restype = None
        lib.oracle_scores.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, _p]
        lib.oracle_scores.restype = ctypes.c_int
        lib.oracle_attention.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _dbl, _p]
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _dbl, _p, _p]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_gather_pages.argtypes = [_p, _i64, _i64, _i64, _i64, _p, _i64, _i64, _p, _p]
        lib.oracle_gather_pages.restype = ctypes.c_int
        lib.oracle_e4m3_to_bf16.argtypes = [_p, _i64, _p]
        lib.oracle_e4m3_to_bf16.restype = ctypes.c_int64
        self._lib = lib

    def num_threads(self) -> int:
        return int(self._lib.oracle_num_threads())

    # ---- one (batch, KV-head) group -------------------------------------------------
    def group_scores(self, q: np.ndarray, k: np.ndarray) -> np.ndarray:
        """q [G, D], k [L, D] (uint16 bf16 bits) -> unscaled scores [G, L] float64."""
        q, k = _u16(q, "q"), _u16(k, "k")
        G, D = q.shape
        L = k.shape[0]
        if k.shape[1] != D:
            raise ValueError("q and k disagree on D")
        s = np.zeros((G, L), np.float64)
        self._lib.oracle_group_scores(_ptr(q), D, _ptr(k), D, G, L, D, _ptr(s))
        return s

    def group_attention(self, q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
        """q [G, D], k/v [L, D] -> softmax(scale * q k^T) v, [G, D] float64."""
        q, k, v = _u16(q, "q"), _u16(k, "k"), _u16(v, "v")
        G, D = q.shape
        L = k.shape[0]
        if k.shape != (L, D) or v.shape != (L, D):
            raise ValueError("bad k/v shapes")
        out = np.zeros((G, D), np.float64)
        rc = self._lib.oracle_group_attention(_ptr(q), D, _ptr(k), D, _ptr(v), D, G, L, D, float(scale),
                                              _ptr(out))
        if rc != 0:
            raise RuntimeError("oracle_group_attention failed")
        return out

    def group_attention_split(self, q, k, v, scale: float, chunk: int) -> np.ndarray:
        """Split-KV form of :meth:`group_attention` with chunks of ``chunk`` tokens."""
        q, k, v = _u16(q, "q"), _u16(k, "k"), _u16(v, "v")
        G, D = q.shape
        L = k.shape[0]
        out = np.zeros((G, D), np.float64)
        rc = self._lib.oracle_group_attention_split(_ptr(q), D, _ptr(k), D, _ptr(v), D, G, L, D, float(scale),
                                                    int(chunk), _ptr(out))
        if rc != 0:
            raise RuntimeError("oracle_group_attention_split failed")
        return out

    # ---- whole batch -------------------------------------------------------------------
    @staticmethod
    def _dims(q, k, seq_lens):
        B, Hq, D = q.shape
        Bk, Hkv, Lcap, Dk = k.shape
        if Bk != B or Dk != D or seq_lens.shape != (B,):
            raise ValueError("inconsistent shapes")
        return B, Hq, Hkv, Lcap, D

    def scores(self, q, k, seq_lens) -> np.ndarray:
        """Unscaled scores [B, Hq, Lcap] float64; NaN where t >= seq_lens[b]."""
        q, k = _u16(q, "q"), _u16(k, "k")
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, Hq, Hkv, Lcap, D = self._dims(q, k, seq_lens)
        s = np.full((B, Hq, Lcap), np.nan, np.float64)
        if self._lib.oracle_scores(_ptr(q), _ptr(k), _ptr(seq_lens), B, Hq, Hkv, Lcap, D, _ptr(s)) != 0:
            raise ValueError("oracle_scores rejected its arguments")
        return s

    def attention(self, q, k, v, seq_lens, scale: float) -> np.ndarray:
        """Attention output [B, Hq, D] float64."""
        q, k, v = _u16(q, "q"), _u16(k, "k"), _u16(v, "v")
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, Hq, Hkv, Lcap, D = self._dims(q, k, seq_lens)
        if v.shape != k.shape:
            raise ValueError("k and v shapes differ")
        attn = np.zeros((B, Hq, D), np.float64)
        if self._lib.oracle_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, Hq, Hkv, Lcap, D,
                                      float(scale), _ptr(attn)) != 0:
            raise ValueError("oracle_attention rejected its arguments")
        return attn

    def oproj(self, x: np.ndarray, w) -> np.ndarray:
        """x [B, K] float64 (or bf16 bits), w [K, N] bf16 bits -> y [B, N] float64."""
        x = np.asarray(x)
        if x.dtype == np.uint16:
            x = bf16_bits_to_f64(x)
        x = np.ascontiguousarray(x, dtype=np.float64)
        w = _u16(w, "w")
        B, K = x.shape
        if w.shape[0] != K:
            raise ValueError("x and w disagree on K")
        N = w.shape[1]
        y = np.zeros((B, N), np.float64)
        self._lib.oracle_oproj(_ptr(x), _ptr(w), B, K, N, _ptr(y))
        return y

    def decode(self, q, k, v, seq_lens, w, scale: float):
        """Whole step -> (attn [B, Hq, D], out [B, N]) both float64."""
        q, k, v, w = _u16(q, "q"), _u16(k, "k"), _u16(v, "v"), _u16(w, "w")
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, Hq, Hkv, Lcap, D = self._dims(q, k, seq_lens)
        if w.shape[0] != Hq * D:
            raise ValueError("o_weight rows must equal Hq * D")
        N = w.shape[1]
        attn = np.zeros((B, Hq, D), np.float64)
        out = np.zeros((B, N), np.float64)
        if self._lib.oracle_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), _ptr(w), B, Hq, Hkv, Lcap, D, N,
                                   float(scale), _ptr(attn), _ptr(out)) != 0:
            raise ValueError("oracle_decode rejected its arguments")
        return attn, out


    # ---- paged cache -------------------------------------------------------------------
    def gather_pages(self, pages, table, seq_lens) -> np.ndarray:
        """pages [num_blocks, Hkv, bs, D] (bf16 bits), table [B, max_blocks] int32 ->
        the contiguous cache [B, Hkv, max_blocks * bs, D] (bf16 bits) the table describes."""
        pages = _u16(pages, "pages")
        table = np.ascontiguousarray(table, dtype=np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        nblk, Hkv, bs, D = pages.shape
        B, mb = table.shape
        if seq_lens.shape != (B,):
            raise ValueError("seq_lens must be [B]")
        cache = np.zeros((B, Hkv, mb * bs, D), np.uint16)
        if self._lib.oracle_gather_pages(_ptr(pages), nblk, Hkv, bs, D, _ptr(table), B, mb, _ptr(seq_lens),
                                         _ptr(cache)) != 0:
            raise ValueError("oracle_gather_pages rejected its arguments")
        return cache

    def decode_paged(self, q, k_pages, v_pages, table, seq_lens, w, scale: float):
        """Whole step over a paged cache: the step on the caches the table describes."""
        k = self.gather_pages(k_pages, table, seq_lens)
        v = self.gather_pages(v_pages, table, seq_lens)
        return self.decode(q, k, v, seq_lens, w, scale)


    # ---- fp8 (e4m3) cache ------------------------------------------------------------------
    def e4m3_to_bf16_bits(self, codes) -> np.ndarray:
        """e4m3 codes (uint8) -> bf16 bit patterns of the same values (exact)."""
        codes = np.ascontiguousarray(codes)
        if codes.dtype != np.uint8:
            raise TypeError(f"expected uint8 e4m3 codes, got {codes.dtype}")
        out = np.zeros(codes.shape, np.uint16)
        self._lib.oracle_e4m3_to_bf16(_ptr(codes), codes.size, _ptr(out))
        return out

    def decode_fp8(self, q, k_codes, v_codes, seq_lens, w, scale: float, k_scale: float, v_scale: float):
        """Whole step over an fp8 cache whose keys and values are k_codes * k_scale and
        v_codes * v_scale. The codes widen exactly to bf16; k_scale multiplies every
        score (it joins `scale`) and v_scale every attention output (the projection is
        linear), so the step is the bf16 one on the widened codes, in fp64."""
        kb = self.e4m3_to_bf16_bits(k_codes)
        vb = self.e4m3_to_bf16_bits(v_codes)
        attn, out = self.decode(q, kb, vb, seq_lens, w, float(scale) * float(k_scale))
        return attn * float(v_scale), out * float(v_scale)


_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from the committed source."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
