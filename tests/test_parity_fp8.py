"""Parity of the fp8 (e4m3) KV-cache entry points through the C ABI.

The keys and values are k_cache * k_scale and v_cache * v_scale with e4m3 codes; the
oracle widens the codes exactly and runs the bf16 definition in fp64 with the scales
folded in. The cases span several 64-token tiles, ragged tails, every group width the
kernel specialises on, empty sequences and CTA counts from one to more than the tiles,
with the bf16 tolerances. Exact checks: V = 1 gives v_scale; a dominant key copies its
value row; NaN codes past a sequence's length never reach the output; and on caches
whose dequantized values are bf16 numbers, the fp8 path agrees with the bf16 path.
"""
import numpy as np
import pytest
import torch

import decode_attention_output_gb300 as da
from decode_attention_output_gb300 import synth
from gpu_helpers import assert_bf16_close, f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
E4M3_ONE = 0x38


@pytest.fixture(scope="module", autouse=True)
def _library():
    from decode_attention_output_gb300 import build

    build.build()
    da.load()
    torch.cuda.set_device(0)
    yield
    assert da.decode_attn_last_device_error() == 0


def W(name, B, Hq, Hkv, Lcap, N, lens, k_mult=1.0):
    return synth.Workload(name, B=B, Hq=Hq, Hkv=Hkv, Lcap=Lcap, N=N, fixed_lens=tuple(lens), k_mult=k_mult, kv="e4m3")


def oracle_fp8(orc, x):
    lens = x["seq_lens"].cpu().numpy().astype(np.int64).clip(0, x["k_cache"].shape[2]).astype(np.int32)
    return orc.decode_fp8(synth.to_bits(x["q"]), synth.to_bits(x["k_cache"]), synth.to_bits(x["v_cache"]), lens,
                          synth.to_bits(x["o_weight"]), x["scale"], x["k_scale"], x["v_scale"])


def run_fp8(w, x, ctas=0):
    old = da.decode_attn_get_option("attn_ctas")
    da.decode_attn_set_option("attn_ctas", ctas)
    try:
        attn = torch.full((w.B, w.Hq, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
        out = torch.full((w.B, w.N), float("nan"), dtype=torch.bfloat16, device=DEV)
        da.decode_attn_only_fp8(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"], x["k_scale"],
                                x["v_scale"])
        da.decode_attn_fwd_fp8(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"],
                               x["k_scale"], x["v_scale"])
        torch.cuda.synchronize()
    finally:
        da.decode_attn_set_option("attn_ctas", old)
    assert da.decode_attn_last_device_error() == 0
    return attn, out


CASES = [
    W("f8_g4_ragged", 3, 8, 2, 300, 256, (300, 1, 129)),
    W("f8_g4_tiles", 2, 32, 8, 640, 1024, (640, 511)),
    W("f8_g8", 2, 16, 2, 200, 512, (200, 77)),
    W("f8_g16", 2, 32, 2, 150, 256, (150, 64)),
    W("f8_g1_mha", 2, 4, 4, 100, 128, (100, 16)),
    W("f8_g3", 2, 6, 2, 257, 264, (257, 130)),
    W("f8_g5_sharp", 2, 10, 2, 190, 640, (190, 33), k_mult=2.0),
    W("f8_g4_very_sharp", 2, 8, 2, 700, 256, (700, 77), k_mult=60.0),
    W("f8_zero_len", 3, 8, 2, 130, 256, (0, 130, 65)),
    W("f8_tiny", 1, 2, 1, 1, 8, (1,)),
    W("f8_tile_plus_one", 1, 8, 2, 65, 256, (65,)),
    W("f8_many_batches", 40, 8, 1, 70, 128, tuple(int(x) for x in np.random.default_rng(8).integers(0, 71, 40))),
    # clusters of two and four CTAs (on-chip merges; a ragged mix partly through L2)
    W("f8_equal_cs2", 8, 32, 8, 2048, 512, (2048,) * 8),
    W("f8_ragged_cs4", 4, 32, 8, 4096, 256, (4096, 100, 3000, 129)),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_fp8_matches_oracle(orc, w):
    x = synth.make_inputs(w, seed=31, device=DEV)
    attn, out = run_fp8(w, x)
    ref_attn, ref_out = oracle_fp8(orc, x)
    assert_bf16_close(f64(attn), ref_attn, f"{w.name} attention")
    assert_bf16_close(f64(out), ref_out, f"{w.name} output")


CLUSTER_CASES = [c for c in CASES if c.name in ("f8_equal_cs2", "f8_ragged_cs4", "f8_g4_ragged", "f8_zero_len")]


@pytest.mark.parametrize("w", CLUSTER_CASES, ids=[c.name for c in CLUSTER_CASES])
def test_fp8_flat_grid(orc, w):
    """The flat grid (option attn_cluster = 0) on the cases that take clusters by default."""
    x = synth.make_inputs(w, seed=33, device=DEV)
    old = da.decode_attn_get_option("attn_cluster")
    da.decode_attn_set_option("attn_cluster", 0)
    try:
        attn, out = run_fp8(w, x)
    finally:
        da.decode_attn_set_option("attn_cluster", old)
    ref_attn, ref_out = oracle_fp8(orc, x)
    assert_bf16_close(f64(attn), ref_attn, f"{w.name} attention")
    assert_bf16_close(f64(out), ref_out, f"{w.name} output")


@pytest.mark.parametrize("ctas", [1, 7, 300])
def test_fp8_cta_counts(orc, ctas):
    w = W("f8_splits", 3, 16, 2, 700, 256, (700, 333, 64))
    x = synth.make_inputs(w, seed=32, device=DEV)
    attn, out = run_fp8(w, x, ctas=ctas)
    ref_attn, ref_out = oracle_fp8(orc, x)
    assert_bf16_close(f64(attn), ref_attn, f"ctas={ctas} attention")
    assert_bf16_close(f64(out), ref_out, f"ctas={ctas} output")


def test_fp8_range_starts_at_every_kind_of_tile(orc):
    """As for bf16, over 128-token tiles: every CTA count from 1 past the number of tiles
    (ranges of one tile, ranges starting on a sequence's last tile or mid-sequence, empty
    rows) equals the oracle."""
    # tiles of 128 tokens per row: 0, 1, 1, 3, 2; two KV heads: 14 tiles
    w = W("f8_firsttiles", 5, 8, 2, 300, 256, (0, 128, 1, 300, 129))
    x = synth.make_inputs(w, seed=41, device=DEV)
    ref_attn, _ = oracle_fp8(orc, x)
    old = da.decode_attn_get_option("attn_cluster")
    try:
        da.decode_attn_set_option("attn_cluster", 0)
        for ctas in range(1, 17):
            attn, _ = run_fp8(w, x, ctas=ctas)
            assert_bf16_close(f64(attn), ref_attn, f"ctas={ctas} attention")
    finally:
        da.decode_attn_set_option("attn_cluster", old)


@pytest.mark.parametrize("rise", [3.0, 30.0, 600.0, -60.0])
def test_fp8_running_maximum_moving_along_the_sequence(orc, rise):
    """As for bf16: a ramp in dim 0 of the K codes (k_scale 1, q[0] = 16) makes the scores rise
    or fall along the sequence by about `rise` log2 units, so that the running reference of the
    online softmax moves every few tiles, on every tile (600: ~17 per warp's 32 tokens), never
    after the first or hardly at all; each equals the oracle on one CTA and on many."""
    w = W("f8_ramp", 2, 8, 2, 1100, 256, (1100, 777))
    x = synth.make_inputs(w, seed=9, device=DEV)
    x["q"][..., 0] = 16.0
    x["k_scale"] = 1.0
    per_unit = 16.0 * x["scale"] * np.log2(np.e)
    kc = x["k_cache"].float()
    kc[:, :, :, 0] = torch.arange(w.Lcap, device=DEV, dtype=torch.float32) * (rise / per_unit / w.Lcap)
    x["k_cache"] = kc.to(torch.float8_e4m3fn)
    ref_attn, _ = oracle_fp8(orc, x)
    for ctas in (1, 0):
        attn, _ = run_fp8(w, x, ctas=ctas)
        assert_bf16_close(f64(attn), ref_attn, f"rise {rise}, ctas {ctas}")


def test_fp8_ones_give_v_scale():
    """V codes = 1.0 and v_scale = 2^-6: every attention output is exactly 2^-6."""
    w = W("f8_ones", 2, 16, 2, 333, 256, (333, 70))
    x = synth.make_inputs(w, seed=33, device=DEV)
    x["v_cache"].view(torch.uint8).fill_(E4M3_ONE)
    x["v_scale"] = 2.0 ** -6
    attn, _ = run_fp8(w, x)
    assert torch.all(attn.float() == 2.0 ** -6)


def test_fp8_dominant_key_copies_its_value_row():
    w = W("f8_dominant", 1, 8, 2, 300, 256, (300,))
    x = synth.make_inputs(w, seed=34, device=DEV)
    q = torch.zeros_like(x["q"])
    q[..., 5] = 8.0
    x["q"] = q
    kc = x["k_cache"].float().clamp(-2, 2)
    kc[:, :, 211, 5] = 128.0  # k_scale 0.5: key 64, scaled score 45.3 vs <= 0.71 for the others
    x["k_cache"] = kc.to(torch.float8_e4m3fn)
    x["k_scale"], x["v_scale"] = 0.5, 0.25
    attn, _ = run_fp8(w, x)
    ref = (x["v_cache"][:, :, 211].float() * 0.25).to(torch.bfloat16).repeat_interleave(4, dim=1)
    assert torch.equal(attn, ref)


def test_fp8_nan_codes_past_seq_len_are_ignored():
    w = W("f8_garbage", 2, 8, 2, 200, 256, (70, 129))
    x = synth.make_inputs(w, seed=35, device=DEV)
    a0, o0 = run_fp8(w, x)
    for cache in ("k_cache", "v_cache"):
        codes = x[cache].view(torch.uint8)
        codes[0, :, 70:] = 0x7F  # e4m3 NaN
        codes[1, :, 129:] = 0xFF
    a1, o1 = run_fp8(w, x)
    assert torch.equal(a0, a1) and torch.equal(o0, o1)


def test_fp8_agrees_with_the_bf16_path():
    """Power-of-two scales: the dequantized caches are exactly bf16 numbers, so the bf16
    path sees the very same keys and values; the two differ only in the rounding of P
    (f16 against bf16), inside the bf16 tolerance."""
    w = W("f8_vs_bf16", 4, 32, 8, 700, 512, (700, 1, 333, 64))
    x = synth.make_inputs(w, seed=36, device=DEV)
    x["k_scale"], x["v_scale"] = 2.0 ** -5, 2.0 ** -6
    attn8, out8 = run_fp8(w, x)
    kb = (x["k_cache"].float() * x["k_scale"]).to(torch.bfloat16)
    vb = (x["v_cache"].float() * x["v_scale"]).to(torch.bfloat16)
    assert torch.equal(kb.float(), x["k_cache"].float() * x["k_scale"])
    attn = torch.empty_like(attn8)
    out = torch.empty_like(out8)
    da.decode_attn_only(x["q"], kb, vb, x["seq_lens"], attn, x["scale"])
    da.decode_attn_fwd(x["q"], kb, vb, x["seq_lens"], x["o_weight"], out, x["scale"])
    torch.cuda.synchronize()
    assert_bf16_close(f64(attn8), f64(attn), "fp8 vs bf16 attention")
    assert_bf16_close(f64(out8), f64(out), "fp8 vs bf16 output")


def test_fp8_repeated_calls_are_deterministic():
    w = W("f8_repeat", 4, 32, 8, 1000, 512, (1000, 999, 500, 3))
    x = synth.make_inputs(w, seed=37, device=DEV)
    runs = [run_fp8(w, x)[1] for _ in range(3)]
    assert torch.equal(runs[0], runs[1]) and torch.equal(runs[1], runs[2])


def test_fp8_trigger_point_does_not_change_the_result():
    """The projection's launch point (option attn_trigger) is timing only on the fp8 path too."""
    w = W("f8_trig", 2, 32, 8, 1024, 512, (1024, 77))
    x = synth.make_inputs(w, seed=23, device=DEV)
    old = da.decode_attn_get_option("attn_trigger")
    outs = []
    try:
        for trig in (0, 3):
            da.decode_attn_set_option("attn_trigger", trig)
            outs.append(run_fp8(w, x)[1])
    finally:
        da.decode_attn_set_option("attn_trigger", old)
    assert torch.equal(outs[0], outs[1])


SIX_STAGE_CASES = [c for c in CASES if c.name in ("f8_g4_ragged", "f8_g16", "f8_zero_len", "f8_equal_cs2",
                                                   "f8_many_batches", "f8_tile_plus_one")]


@pytest.mark.parametrize("w", SIX_STAGE_CASES, ids=[c.name for c in SIX_STAGE_CASES])
def test_fp8_six_stage_ring(orc, w):
    """The 6-stage ring (option attn_stages = 6) gives bit for bit the 4-stage result: the
    ring depth changes when tiles arrive, not which CTA reads which tile or the merge order."""
    x = synth.make_inputs(w, seed=34, device=DEV)
    attn4, out4 = run_fp8(w, x)
    old = da.decode_attn_get_option("attn_stages")
    da.decode_attn_set_option("attn_stages", 6)
    try:
        attn6, out6 = run_fp8(w, x)
    finally:
        da.decode_attn_set_option("attn_stages", old)
    assert torch.equal(attn4, attn6) and torch.equal(out4, out6)
    ref_attn, ref_out = oracle_fp8(orc, x)
    assert_bf16_close(f64(attn6), ref_attn, f"{w.name} attention, 6 stages")
