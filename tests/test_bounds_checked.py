"""The bounds-checked build of the library (-DDA_BOUNDS_CHECK), on small GPU cases.

In that build every guarded index of the kernels (global outputs, split-KV partials,
completion counters, shared-memory stages and merge scratch, distributed shared
memory of clusters, tile cursors, block-table entries, projection partials) is
tested against the extent of its buffer before the access; a failure sets bit 256
of the device error word and skips the access, with no trap and no assert. This
stands in for a memory checker on this GPU. Each case also surrounds every output
with canaries (a NaN bit pattern the kernels never write): an extra slice before
and after the batch dimension and spare elements around each innermost row, so
that an output view with padded strides is written exactly where it should be.

Checked for every case: the error word is 0, every canary is intact, and the
outputs match the fp64 oracle within the bf16 tolerances. The cases cover the
flat and cluster grids, empty and one-token sequences, group widths 1/4/16, head
dim 256, a single CTA doing all the work, the paged and fp8 caches, the fused
step, the scores hook, both projection paths with split-K through a cluster and
through global partials, batch chunks of the tensor-core projection, and the
no-allocation entry point.
"""
import numpy as np
import pytest
import torch

import decode_attention_output_gb300 as da
from decode_attention_output_gb300 import binding, synth
from gpu_helpers import RTOL_SCORES, assert_bf16_close, f64, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CANARY = {torch.bfloat16: 0x7FA5, torch.float32: 0x7FC0DEAD}  # NaN payloads no kernel writes
BOUNDS_BIT = 256


@pytest.fixture(scope="module", autouse=True)
def _checked_library():
    from decode_attention_output_gb300 import build

    torch.cuda.set_device(0)
    build.build()
    da.load()
    chk = binding.load_library(build.build(checked=True))
    prev = binding.use_library(chk)
    yield
    binding.use_library(prev)


class Padded:
    """An output tensor of `shape` inside a canary-filled buffer: one extra slice before and
    after dim 0 and 16 bytes of spare elements on both sides of every innermost row."""

    def __init__(self, shape, dtype):
        self.dtype, self.shape = dtype, tuple(shape)
        self.pad = 16 // torch.tensor([], dtype=dtype).element_size()
        big_shape = (shape[0] + 2, *shape[1:-1], shape[-1] + 2 * self.pad)
        self.big = torch.empty(big_shape, dtype=dtype, device=DEV)
        self._int().fill_(CANARY[dtype])
        self.view = self.big[(slice(1, shape[0] + 1),) + (slice(None),) * (len(shape) - 2) +
                             (slice(self.pad, self.pad + shape[-1]),)]

    def _int(self):
        return self.big.view(torch.int16 if self.dtype == torch.bfloat16 else torch.int32)

    def canaries_intact(self) -> bool:
        mask = torch.ones(self.big.shape, dtype=torch.bool, device=DEV)
        mask[(slice(1, self.shape[0] + 1),) + (slice(None),) * (len(self.shape) - 2) +
             (slice(self.pad, self.pad + self.shape[-1]),)] = False
        bits = self._int()[mask]
        return bool((bits == CANARY[self.dtype]).all())


class _Opt:
    def __init__(self, **kv):
        self.kv = kv

    def __enter__(self):
        self.old = {k: da.decode_attn_get_option(k) for k in self.kv}
        for k, v in self.kv.items():
            da.decode_attn_set_option(k, v)

    def __exit__(self, *exc):
        for k, v in self.old.items():
            da.decode_attn_set_option(k, v)


def W(name, B, Hq, Hkv, Lcap, N, lens, D=128, kv="bf16"):
    return synth.Workload(name, B=B, Hq=Hq, Hkv=Hkv, Lcap=Lcap, N=N, fixed_lens=tuple(lens), D=D, kv=kv)


def _finish(orc, x, outs, what):
    torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0, f"{what}: device error word set"
    for name, po in outs.items():
        assert po.canaries_intact(), f"{what}: {name} written outside its view"
    ref_attn, ref_out = oracle_decode(orc, x)
    if "attn" in outs:
        assert_bf16_close(f64(outs["attn"].view), ref_attn, f"{what} attention")
    if "out" in outs:
        assert_bf16_close(f64(outs["out"].view), ref_out, f"{what} output")


STEP_CASES = [
    (W("flat_g4_zero", 3, 8, 2, 300, 256, (300, 0, 129)), {}),
    (W("g16", 2, 32, 2, 150, 256, (150, 64)), {}),
    (W("g1_one_token", 2, 4, 4, 100, 128, (100, 1)), {}),
    (W("cluster_equal", 8, 32, 8, 1024, 512, (1024,) * 8), {}),
    (W("cluster_ragged", 8, 32, 8, 1024, 512, (1024, 0, 1, 700, 64, 1000, 333, 129)), {}),
    (W("one_cta", 6, 8, 2, 200, 256, (200, 3, 0, 64, 65, 199)), {"attn_ctas": 1}),
    (W("d256", 3, 8, 2, 300, 256, (300, 0, 129), D=256), {}),
    (W("fused", 3, 8, 2, 300, 256, (300, 0, 129)), {"fused": 1}),
    (W("gemv", 5, 8, 2, 130, 264, (130, 7, 0, 64, 129)), {"oproj_path": 1}),
    (W("splitk_partials", 4, 32, 8, 256, 512, (256, 100, 1, 255)), {"oproj_cluster": 0, "oproj_splitk": 16}),
    (W("batch130", 130, 8, 2, 40, 256, tuple(int(v) for v in np.random.default_rng(2).integers(0, 41, 130))), {}),
    (W("onchip_b1", 1, 32, 8, 1024, 2048, (1000,)), {"oproj_path": 3}),
]


@pytest.mark.parametrize("w,opts", STEP_CASES, ids=[c[0].name for c in STEP_CASES])
def test_step_in_bounds(orc, w, opts):
    x = synth.make_inputs(w, seed=5, device=DEV)
    attn = Padded((w.B, w.Hq, w.D), torch.bfloat16)
    out = Padded((w.B, w.N), torch.bfloat16)
    with _Opt(**opts):
        da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn.view, x["scale"])
        da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out.view, x["scale"])
    _finish(orc, x, {"attn": attn, "out": out}, w.name)


@pytest.mark.parametrize("bs", [16, 64])
def test_paged_in_bounds(orc, bs):
    w = W("paged", 3, 8, 2, 256, 256, (256, 0, 77))
    x = synth.make_inputs(w, seed=6, device=DEV)
    mb = w.Lcap // bs
    g = torch.Generator().manual_seed(bs)
    perm = torch.randperm(w.B * mb + 2, generator=g)[: w.B * mb].view(w.B, mb)
    pools = []
    for key in ("k_cache", "v_cache"):
        pool = torch.zeros((w.B * mb + 2, w.Hkv, bs, w.D), dtype=torch.bfloat16, device=DEV)
        for b in range(w.B):
            for i in range(mb):
                pool[perm[b, i]] = x[key][b, :, i * bs:(i + 1) * bs]
        pools.append(pool)
    table = perm.to(torch.int32).to(DEV).contiguous()
    attn = Padded((w.B, w.Hq, w.D), torch.bfloat16)
    out = Padded((w.B, w.N), torch.bfloat16)
    da.decode_attn_only_paged(x["q"], pools[0], pools[1], table, x["seq_lens"], attn.view, x["scale"])
    da.decode_attn_fwd_paged(x["q"], pools[0], pools[1], table, x["seq_lens"], x["o_weight"], out.view, x["scale"])
    _finish(orc, x, {"attn": attn, "out": out}, f"paged block {bs}")


def test_fp8_in_bounds(orc):
    w = W("fp8", 3, 8, 2, 400, 256, (400, 0, 129), kv="e4m3")
    x = synth.make_inputs(w, seed=7, device=DEV)
    attn = Padded((w.B, w.Hq, w.D), torch.bfloat16)
    out = Padded((w.B, w.N), torch.bfloat16)
    da.decode_attn_only_fp8(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn.view, x["scale"], x["k_scale"],
                            x["v_scale"])
    da.decode_attn_fwd_fp8(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out.view, x["scale"],
                           x["k_scale"], x["v_scale"])
    _finish(orc, x, {"attn": attn, "out": out}, "fp8 cache")


def test_noalloc_in_bounds(orc):
    w = W("noalloc", 4, 16, 2, 500, 128, (500, 3, 0, 257))
    x = synth.make_inputs(w, seed=8, device=DEV)
    attn = Padded((w.B, w.Hq, w.D), torch.bfloat16)
    da.decode_attn_only_noalloc(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn.view, x["scale"])
    _finish(orc, x, {"attn": attn}, "no-allocation entry point")


def test_scores_in_bounds(orc):
    """The scores hook writes t < seq_lens[b] only: entries past each length keep their canary."""
    w = W("scores", 3, 8, 2, 200, 128, (200, 0, 77))
    x = synth.make_inputs(w, seed=9, device=DEV)
    sc = Padded((w.B, w.Hq, w.Lcap), torch.float32)
    da.decode_attn_scores(x["q"], x["k_cache"], x["seq_lens"], sc.view)
    torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    assert sc.canaries_intact()
    lens = x["seq_lens"].cpu().numpy()
    ref = orc.scores(synth.to_bits(x["q"]), synth.to_bits(x["k_cache"]), lens)
    got = sc.view.cpu().numpy().astype(np.float64)
    bits = sc.view.view(torch.int32).cpu().numpy()
    for b in range(w.B):
        L = int(lens[b])
        assert np.all(bits[b, :, L:] == CANARY[torch.float32]), f"row {b}: scores written past the length"
        for h in range(w.Hq):
            if L:
                err = np.linalg.norm(got[b, h, :L] - ref[b, h, :L]) / np.linalg.norm(ref[b, h, :L])
                assert err <= RTOL_SCORES, (b, h, err)
