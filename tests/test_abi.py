"""The C-ABI library on the host (no GPU needed): it builds, loads, exports every
symbol include/decode_attn.h declares, and rejects bad arguments on the host
with the documented status codes before touching the device.

The argument-validation cases use fake device addresses. They are skipped when
a GPU is visible, so that a validation bug can never turn into a launch on
made-up pointers.
"""
import ctypes
import os
import re

import pytest
import torch

import decode_attention_output_gb300 as da
from decode_attention_output_gb300 import binding
from decode_attention_output_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "decode_attn.h")

OK, NULL, DTYPE, SHAPE, STRIDE, ALIGN, UNSUP = 0, -1, -2, -3, -4, -5, -6


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return binding.load()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(decode_attn_\w+)\s*\(", text)))


def test_header_declares_what_binding_wraps():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"


def test_status_strings(lib):
    for code in range(-10, 1):
        assert binding.status_str(code) != binding.status_str(-99)
    assert binding.status_str(-99) == "unknown status"


def test_options_roundtrip(lib):
    old = da.decode_attn_get_option("attn_ctas")
    da.decode_attn_set_option("attn_ctas", 7)
    assert da.decode_attn_get_option("attn_ctas") == 7
    da.decode_attn_set_option("attn_ctas", old)


# every documented option, its default and a value that must be refused
OPTION_DEFAULTS = {"attn_ctas": 0, "oproj_path": 0, "oproj_splitk": 0, "gemm_min_batch": 1, "pdl": 1,
                   "l2_prefetch": 0, "attn_stages": 4, "fused": 0, "fused_attn_ctas": 0, "oproj_prefetch": 0,
                   "oproj_cluster": 1, "attn_cluster": 1, "attn_pdl": 1, "attn_trigger": 3, "grid_wait_us": 0,
                   "grid_wait_extra": 0}
OPTION_BAD = {"attn_ctas": 513, "oproj_path": 4, "pdl": 2, "l2_prefetch": -1, "attn_stages": 5, "fused": 2,
              "oproj_prefetch": 2, "oproj_cluster": 2, "attn_cluster": 3, "gemm_min_batch": 0, "attn_pdl": 2,
              "attn_trigger": -1, "grid_wait_us": 2000001, "grid_wait_extra": 2}


@pytest.mark.parametrize("key", sorted(OPTION_DEFAULTS))
def test_option_defaults_and_range(lib, key):
    assert da.decode_attn_get_option(key) == OPTION_DEFAULTS[key]
    if key in OPTION_BAD:
        with pytest.raises(da.DecodeAttnError):
            da.decode_attn_set_option(key, OPTION_BAD[key])
        assert da.decode_attn_get_option(key) == OPTION_DEFAULTS[key]
    da.decode_attn_set_option(key, OPTION_DEFAULTS[key])
    assert da.decode_attn_get_option(key) == OPTION_DEFAULTS[key]
    with pytest.raises(da.DecodeAttnError):
        da.decode_attn_set_option("no_such_option", 1)
    with pytest.raises(da.DecodeAttnError):
        da.decode_attn_set_option("oproj_path", 5)


# ---------------------------------------------------------------- validation
FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


def desc(shape, dtype=binding.DA_DTYPE_BF16, strides=None, addr=FAKE):
    d = binding.da_tensor_t()
    d.data = addr
    d.dtype = dtype
    d.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, strides)):
        d.shape[i] = s
        d.stride[i] = st
    return d


def fwd_args(B=2, Hq=8, Hkv=2, L=64, N=256, **over):
    a = dict(q=desc([B, Hq, 128]), k=desc([B, Hkv, L, 128]), v=desc([B, Hkv, L, 128]),
             lens=desc([B], binding.DA_DTYPE_I32), w=desc([Hq * 128, N]), out=desc([B, N]))
    a.update(over)
    return a


def call_fwd(lib, a, scale=0.1):
    r = lambda d: ctypes.byref(d) if d is not None else None  # noqa: E731
    return lib.decode_attn_fwd(r(a["q"]), r(a["k"]), r(a["v"]), r(a["lens"]), r(a["w"]), r(a["out"]),
                               ctypes.c_float(scale), None)


cpu_only = pytest.mark.skipif(torch.cuda.is_available(), reason="fake-pointer cases run only without a GPU")

BAD_FWD = [
    ("q_dtype", dict(q=desc([2, 8, 128], binding.DA_DTYPE_F32)), DTYPE),
    ("lens_dtype", dict(lens=desc([2], binding.DA_DTYPE_F32)), DTYPE),
    ("head_dim_64", dict(q=desc([2, 8, 64])), SHAPE),
    ("kv_head_dim_64", dict(k=desc([2, 2, 64, 64]), v=desc([2, 2, 64, 64])), SHAPE),
    ("head_dim_192", dict(q=desc([2, 8, 192]), k=desc([2, 2, 64, 192]), v=desc([2, 2, 64, 192]),
                          w=desc([8 * 192, 256])), SHAPE),
    ("q_256_cache_128", dict(q=desc([2, 8, 256]), w=desc([8 * 256, 256])), SHAPE),
    ("d256_w_rows_for_128", dict(q=desc([2, 8, 256]), k=desc([2, 2, 64, 256]), v=desc([2, 2, 64, 256])), SHAPE),
    ("heads_not_multiple", dict(q=desc([2, 6, 128]), k=desc([2, 4, 64, 128]), v=desc([2, 4, 64, 128]),
                                w=desc([6 * 128, 256])), SHAPE),
    ("group_32", dict(q=desc([2, 64, 128]), w=desc([64 * 128, 256])), UNSUP),
    ("batch_mismatch", dict(k=desc([3, 2, 64, 128]), v=desc([3, 2, 64, 128])), SHAPE),
    ("v_shape", dict(v=desc([2, 2, 32, 128])), SHAPE),
    ("w_rows", dict(w=desc([4 * 128, 256])), SHAPE),
    ("out_cols", dict(out=desc([2, 128])), SHAPE),
    ("n_not_multiple_of_8", dict(w=desc([8 * 128, 260], strides=[264, 1]), out=desc([2, 260])), SHAPE),
    ("q_misaligned", dict(q=desc([2, 8, 128], addr=FAKE + 2)), ALIGN),
    ("k_misaligned", dict(k=desc([2, 2, 64, 128], addr=FAKE + 8)), ALIGN),
    ("q_inner_stride", dict(q=desc([2, 8, 128], strides=[2048, 256, 2])), STRIDE),
    ("k_row_stride_odd", dict(k=desc([2, 2, 64, 128], strides=[2 * 64 * 130, 64 * 130, 130, 1])), STRIDE),
    ("w_row_stride_odd", dict(w=desc([1024, 256], strides=[260, 1])), STRIDE),
    ("null_q", dict(q=None), NULL),
    ("null_lens", dict(lens=None), NULL),
    ("lens_strided", dict(lens=desc([2], binding.DA_DTYPE_I32, strides=[2])), STRIDE),
    ("batch_too_large", dict(q=desc([2048, 8, 128]), k=desc([2048, 2, 64, 128]), v=desc([2048, 2, 64, 128]),
                             lens=desc([2048], binding.DA_DTYPE_I32), out=desc([2048, 256])), UNSUP),
    ("empty_cache", dict(k=desc([2, 2, 0, 128]), v=desc([2, 2, 0, 128])), SHAPE),
]


@cpu_only
@pytest.mark.parametrize("name,over,code", BAD_FWD, ids=[c[0] for c in BAD_FWD])
def test_fwd_rejects(lib, name, over, code):
    assert call_fwd(lib, fwd_args(**over)) == code


@cpu_only
def test_fwd_rejects_nonfinite_scale(lib):
    assert call_fwd(lib, fwd_args(), scale=float("nan")) == UNSUP
    assert call_fwd(lib, fwd_args(), scale=float("inf")) == UNSUP


@cpu_only
def test_empty_batch_is_a_noop(lib):
    a = fwd_args(B=0)
    for key in ("q", "k", "v", "lens", "out"):  # zero-element tensors carry no storage
        a[key].data = None
    assert call_fwd(lib, a) == OK


@cpu_only
def test_only_and_scores_and_oproj_reject(lib):
    r = ctypes.byref
    a = fwd_args()
    bad_attn = desc([2, 8, 64])
    assert lib.decode_attn_only(r(a["q"]), r(a["k"]), r(a["v"]), r(a["lens"]), r(bad_attn), ctypes.c_float(1.0),
                                None) == SHAPE
    bad_scores = desc([2, 8, 63], binding.DA_DTYPE_F32)
    assert lib.decode_attn_scores(r(a["q"]), r(a["k"]), r(a["lens"]), r(bad_scores), None) == SHAPE
    scores_bf16 = desc([2, 8, 64])
    assert lib.decode_attn_scores(r(a["q"]), r(a["k"]), r(a["lens"]), r(scores_bf16), None) == DTYPE
    x, w, out = desc([2, 1024]), desc([1000, 256]), desc([2, 256])
    assert lib.decode_attn_oproj(r(x), r(w), r(out), None) == SHAPE
    x, w, out = desc([2, 1020]), desc([1020, 256]), desc([2, 256])
    assert lib.decode_attn_oproj(r(x), r(w), r(out), None) == STRIDE  # row stride 1020 is not a multiple of 8


@cpu_only
def test_binding_raises_with_code(lib):
    q = torch.zeros((2, 8, 128), dtype=torch.float32)  # wrong dtype: rejected before any device access
    k = torch.zeros((2, 2, 64, 128), dtype=torch.bfloat16)
    lens = torch.zeros((2,), dtype=torch.int32)
    attn = torch.zeros((2, 8, 128), dtype=torch.bfloat16)
    with pytest.raises(da.DecodeAttnError) as ei:
        da.decode_attn_only(q, k, k, lens, attn, 0.1, stream=0)
    assert ei.value.code == DTYPE


# ---------------------------------------------------------- paged-cache entry points
def paged_args(B=2, Hq=8, Hkv=2, D=128, nblk=10, bs=16, mb=4, N=256, **over):
    a = dict(q=desc([B, Hq, D]), kp=desc([nblk, Hkv, bs, D]), vp=desc([nblk, Hkv, bs, D]),
             table=desc([B, mb], binding.DA_DTYPE_I32), lens=desc([B], binding.DA_DTYPE_I32),
             w=desc([Hq * D, N]), out=desc([B, N]), attn=desc([B, Hq, D]))
    a.update(over)
    return a


def call_paged(lib, a, scale=0.1):
    r = lambda d: ctypes.byref(d) if d is not None else None  # noqa: E731
    rc_fwd = lib.decode_attn_fwd_paged(r(a["q"]), r(a["kp"]), r(a["vp"]), r(a["table"]), r(a["lens"]), r(a["w"]),
                                       r(a["out"]), ctypes.c_float(scale), None)
    rc_only = lib.decode_attn_only_paged(r(a["q"]), r(a["kp"]), r(a["vp"]), r(a["table"]), r(a["lens"]),
                                         r(a["attn"]), ctypes.c_float(scale), None)
    return rc_fwd, rc_only


BAD_PAGED = [
    ("block_size_24", dict(kp=desc([10, 2, 24, 128]), vp=desc([10, 2, 24, 128])), UNSUP),
    ("block_size_4", dict(kp=desc([10, 2, 4, 128]), vp=desc([10, 2, 4, 128])), UNSUP),
    ("block_size_96", dict(kp=desc([10, 2, 96, 128]), vp=desc([10, 2, 96, 128])), UNSUP),
    ("block_size_192", dict(kp=desc([10, 2, 192, 128]), vp=desc([10, 2, 192, 128])), UNSUP),
    ("table_not_16_aligned", dict(table=desc([2, 4], binding.DA_DTYPE_I32, addr=FAKE + 4)), ALIGN),
    ("d256_block_size_48", dict(q=desc([2, 8, 256]), kp=desc([10, 2, 48, 256]), vp=desc([10, 2, 48, 256]),
                                w=desc([8 * 256, 256]), attn=desc([2, 8, 256])), UNSUP),
    ("table_dtype", dict(table=desc([2, 4], binding.DA_DTYPE_F32)), DTYPE),
    ("table_rows", dict(table=desc([3, 4], binding.DA_DTYPE_I32)), SHAPE),
    ("table_1d", dict(table=desc([8], binding.DA_DTYPE_I32)), SHAPE),
    ("table_inner_stride", dict(table=desc([2, 4], binding.DA_DTYPE_I32, strides=[8, 2])), STRIDE),
    ("table_rows_overlap", dict(table=desc([2, 4], binding.DA_DTYPE_I32, strides=[2, 1])), STRIDE),
    ("table_misaligned", dict(table=desc([2, 4], binding.DA_DTYPE_I32, addr=FAKE + 2)), ALIGN),
    ("null_table", dict(table=None), NULL),
    ("v_pages_shape", dict(vp=desc([9, 2, 16, 128])), SHAPE),
    ("pages_head_dim", dict(kp=desc([10, 2, 16, 256]), vp=desc([10, 2, 16, 256])), SHAPE),
    ("pages_misaligned", dict(kp=desc([10, 2, 16, 128], addr=FAKE + 8)), ALIGN),
    ("pages_token_stride_odd", dict(kp=desc([10, 2, 16, 128], strides=[2 * 16 * 132, 16 * 132, 132, 1])),
     STRIDE),
    ("group_32", dict(q=desc([2, 64, 128]), w=desc([64 * 128, 256]), attn=desc([2, 64, 128])), UNSUP),
    ("empty_pool", dict(kp=desc([0, 2, 16, 128]), vp=desc([0, 2, 16, 128])), SHAPE),
]


@cpu_only
@pytest.mark.parametrize("name,over,code", BAD_PAGED, ids=[c[0] for c in BAD_PAGED])
def test_paged_rejects(lib, name, over, code):
    assert call_paged(lib, paged_args(**over)) == (code, code)


@cpu_only
def test_paged_accepts_valid_block_sizes_on_the_host(lib):
    """Valid shapes pass validation; with B = 0 nothing is launched."""
    for D, bs in ((128, 8), (128, 16), (128, 32), (128, 64), (128, 4096), (256, 8), (256, 16), (256, 32),
                  (256, 128)):
        a = paged_args(B=0, D=D, bs=bs)
        for key in ("q", "table", "lens", "out", "attn"):
            a[key].data = None
        assert call_paged(lib, a) == (OK, OK), (D, bs)


# ------------------------------------------------------------- fp8-cache entry points
E4M3 = binding.DA_DTYPE_E4M3


def fp8_args(**over):
    a = fwd_args(k=desc([2, 2, 64, 128], E4M3), v=desc([2, 2, 64, 128], E4M3))
    a["attn"] = desc([2, 8, 128])
    a.update(over)
    return a


def call_fp8(lib, a, scale=0.1, k_scale=0.02, v_scale=0.02):
    r = lambda d: ctypes.byref(d) if d is not None else None  # noqa: E731
    f = ctypes.c_float
    rc_fwd = lib.decode_attn_fwd_fp8(r(a["q"]), r(a["k"]), r(a["v"]), r(a["lens"]), r(a["w"]), r(a["out"]), f(scale),
                                     f(k_scale), f(v_scale), None)
    rc_only = lib.decode_attn_only_fp8(r(a["q"]), r(a["k"]), r(a["v"]), r(a["lens"]), r(a["attn"]), f(scale),
                                       f(k_scale), f(v_scale), None)
    return rc_fwd, rc_only


BAD_FP8 = [
    ("kv_bf16", dict(k=desc([2, 2, 64, 128]), v=desc([2, 2, 64, 128])), DTYPE),
    ("v_bf16", dict(v=desc([2, 2, 64, 128])), DTYPE),
    ("q_fp8", dict(q=desc([2, 8, 128], E4M3)), DTYPE),
    ("head_dim_256", dict(q=desc([2, 8, 256]), k=desc([2, 2, 64, 256], E4M3), v=desc([2, 2, 64, 256], E4M3),
                          w=desc([8 * 256, 256]), attn=desc([2, 8, 256])), UNSUP),
    ("row_stride_136_bytes", dict(k=desc([2, 2, 64, 128], E4M3, strides=[2 * 64 * 136, 64 * 136, 136, 1])), STRIDE),
    ("k_misaligned", dict(k=desc([2, 2, 64, 128], E4M3, addr=FAKE + 8)), ALIGN),
    ("v_shape", dict(v=desc([2, 2, 32, 128], E4M3)), SHAPE),
]


@cpu_only
@pytest.mark.parametrize("name,over,code", BAD_FP8, ids=[c[0] for c in BAD_FP8])
def test_fp8_rejects(lib, name, over, code):
    assert call_fp8(lib, fp8_args(**over)) == (code, code)


@cpu_only
def test_fp8_rejects_nonfinite_scales(lib):
    assert call_fp8(lib, fp8_args(), k_scale=float("inf")) == (UNSUP, UNSUP)
    assert call_fp8(lib, fp8_args(), v_scale=float("nan")) == (UNSUP, UNSUP)


@cpu_only
def test_fp8_row_stride_of_16_bytes_passes_validation(lib):
    """A 144-byte row stride (16-byte multiple, not a multiple of 128) is accepted; B = 0."""
    a = fp8_args(q=desc([0, 8, 128]), k=desc([0, 2, 64, 128], E4M3, strides=[2 * 64 * 144, 64 * 144, 144, 1]),
                 v=desc([0, 2, 64, 128], E4M3), lens=desc([0], binding.DA_DTYPE_I32), out=desc([0, 256]),
                 attn=desc([0, 8, 128]))
    for key in ("q", "k", "v", "lens", "out", "attn"):
        a[key].data = None
    assert call_fp8(lib, a) == (OK, OK)
