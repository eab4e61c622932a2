"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, element by
element, on seeded inputs that span several 64-token tiles, ragged tails, every
GQA group width the kernels specialise on, and the degenerate cases: empty
sequences, one token, lengths past the cache (clamped), a single persistent CTA
doing all the work and more CTAs than tiles.
"""
import math

import numpy as np
import pytest
import torch

import decode_attention_output_gb300 as da
from decode_attention_output_gb300 import synth
from gpu_helpers import RTOL_SCORES, assert_bf16_close, f64, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from decode_attention_output_gb300 import build

    build.build()
    da.load()
    torch.cuda.set_device(0)
    yield
    assert da.decode_attn_last_device_error() == 0


def W(name, B, Hq, Hkv, Lcap, N, lens, k_mult=1.0):
    return synth.Workload(name, B=B, Hq=Hq, Hkv=Hkv, Lcap=Lcap, N=N, fixed_lens=tuple(lens), k_mult=k_mult)


CASES = [
    W("g4_ragged", 3, 8, 2, 300, 256, (300, 1, 129)),
    W("g4_tiles", 2, 32, 8, 640, 1024, (640, 511)),
    W("g8", 2, 16, 2, 200, 512, (200, 77)),
    W("g16", 2, 32, 2, 150, 256, (150, 64)),
    W("g1_mha", 2, 4, 4, 100, 128, (100, 16)),
    W("g3", 2, 6, 2, 257, 264, (257, 130)),
    W("g5_sharp", 2, 10, 2, 190, 640, (190, 33), k_mult=2.0),
    # scores spread over hundreds of log2 units: the softmax is nearly one-hot in places and its
    # running maximum jumps by far more than the lagging reference's slack
    W("g4_very_sharp", 2, 8, 2, 700, 256, (700, 77), k_mult=60.0),
    W("zero_len", 3, 8, 2, 130, 256, (0, 130, 65)),
    W("all_zero_len", 2, 8, 2, 70, 256, (0, 0)),
    W("tiny", 1, 2, 1, 1, 8, (1,)),
    W("one_tile", 1, 8, 2, 64, 256, (64,)),
    W("tile_plus_one", 1, 8, 2, 65, 256, (65,)),
    W("many_batches", 40, 8, 1, 70, 128, tuple(int(x) for x in np.random.default_rng(3).integers(0, 71, 40))),
    W("b9_gemv_chunks", 9, 8, 2, 96, 256, (96, 1, 2, 3, 64, 65, 95, 33, 17)),
    # batch 1 and 2 with the full hidden size (the projection's full 32 x 8 grid)
    W("b1_hidden4096", 1, 32, 8, 2048, 4096, (2048,)),
    W("b1_hidden4096_short", 1, 32, 8, 2048, 4096, (777,)),
    W("b2_hidden4096", 2, 32, 8, 2048, 4096, (2048, 1000)),
]


def _run(w, seed=0, ctas=0):
    x = synth.make_inputs(w, seed=seed, device=DEV)
    old = da.decode_attn_get_option("attn_ctas")
    da.decode_attn_set_option("attn_ctas", ctas)
    try:
        attn = torch.full((w.B, w.Hq, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
        da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"])
        out = torch.full((w.B, w.N), float("nan"), dtype=torch.bfloat16, device=DEV)
        da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"])
        torch.cuda.synchronize()
    finally:
        da.decode_attn_set_option("attn_ctas", old)
    assert da.decode_attn_last_device_error() == 0
    return x, attn, out


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_decode_matches_oracle(orc, w):
    x, attn, out = _run(w)
    ref_attn, ref_out = oracle_decode(orc, x)
    assert_bf16_close(f64(attn), ref_attn, f"{w.name} attention")
    assert_bf16_close(f64(out), ref_out, f"{w.name} output")


CLUSTER_CASES = [c for c in CASES if c.name in ("g4_ragged", "zero_len", "all_zero_len", "tiny", "one_tile",
                                                 "tile_plus_one", "g16", "g3")] + [
    W("b1_l2k", 1, 32, 8, 2048, 512, (2048,)),
    W("b2_ragged_short", 2, 32, 8, 700, 256, (700, 5)),
    W("b1_g8_d", 1, 64, 8, 1500, 256, (1333,)),
    # clusters of two (64 sequences) and four (32): every sequence on chip with equal lengths,
    # a mix of on-chip and L2 merges with ragged ones (balanced split either way)
    W("b8_equal_cs2", 8, 32, 8, 1024, 512, (1024,) * 8),
    W("b8_ragged_cs2", 8, 32, 8, 2048, 512, (2048, 0, 1, 1500, 64, 2000, 777, 129)),
    W("b4_equal_cs4", 4, 32, 8, 4096, 256, (4096,) * 4),
    W("b4_ragged_cs4", 4, 32, 8, 4096, 256, (4096, 100, 3000, 65)),
    W("b2_g16_cs8", 2, 32, 2, 2000, 256, (2000, 999)),
]


@pytest.mark.parametrize("w", CLUSTER_CASES, ids=[c.name for c in CLUSTER_CASES])
def test_cluster_mode_matches_flat_and_oracle(orc, w):
    """Where there is room, the attention runs in thread-block clusters; with equal lengths each
    sequence's parts share a cluster and merge in distributed shared memory, with unequal ones
    the tiles are split over the whole grid and merged through global partials, as on the flat
    grid (option attn_cluster = 0). Both against the oracle, and against each other within the
    bf16 rounding of the merge order."""
    res = {}
    for mode in (1, 0):  # clusters where they fit (the default), never
        old = da.decode_attn_get_option("attn_cluster")
        da.decode_attn_set_option("attn_cluster", mode)
        try:
            res[mode] = _run(w, seed=21)
        finally:
            da.decode_attn_set_option("attn_cluster", old)
    x = res[1][0]
    ref_attn, ref_out = oracle_decode(orc, x)
    for mode, (_, attn, out) in res.items():
        assert_bf16_close(f64(attn), ref_attn, f"{w.name} attention, cluster mode {mode}")
        assert_bf16_close(f64(out), ref_out, f"{w.name} output, cluster mode {mode}")
    for mode in (1,):
        for i, what in ((1, "attention"), (2, "output")):
            diff = (res[mode][i].float() - res[0][i].float()).abs()
            tol = 2.0 ** -7 * res[0][i].float().abs() + 1e-3  # the two merges round differently
            assert torch.all(diff <= tol), f"{w.name}: {what}, cluster mode {mode} and flat differ by {diff.max().item():.3e}"


MAX_CASES = [
    W("max_batch_g16", 1024, 16, 1, 70, 128, tuple(int(x) for x in np.random.default_rng(11).integers(0, 71, 1024))),
    W("max_batch_g2", 1024, 8, 4, 40, 136, tuple(int(x) for x in np.random.default_rng(12).integers(0, 41, 1024))),
]


@pytest.mark.parametrize("w", MAX_CASES, ids=[c.name for c in MAX_CASES])
def test_maximum_batch_matches_oracle(orc, w):
    """The largest batch the entry points accept (1024), with the widest GQA group (16) and
    with 4096 (batch, KV head) sequences; ragged lengths with empty sequences; the
    projection pads the batch to 128 rows in 8 chunks."""
    x, attn, out = _run(w, seed=5)
    ref_attn, ref_out = oracle_decode(orc, x)
    assert_bf16_close(f64(attn), ref_attn, f"{w.name} attention")
    assert_bf16_close(f64(out), ref_out, f"{w.name} output")


TRIGGER_CASES = [
    W("b1_l2k", 1, 32, 8, 2048, 512, (2048,)),
    W("trig_ragged", 3, 8, 2, 300, 256, (300, 1, 129)),
    W("trig_zero_len", 3, 8, 2, 130, 256, (0, 130, 65)),
    W("trig_b8_equal_clusters", 8, 32, 8, 1024, 512, (1024,) * 8),  # clusters of two, idle CTAs
]


@pytest.mark.parametrize("w", TRIGGER_CASES, ids=[c.name for c in TRIGGER_CASES])
@pytest.mark.parametrize("ctas", [0, 1, 7])
def test_projection_trigger_point_does_not_change_the_result(orc, w, ctas):
    """decode_attn_fwd lets the projection kernel launch a few tiles before each attention
    CTA's end (option attn_trigger); the projection still waits for the whole attention grid,
    so every trigger point (at set-up, one tile before the end, three, and more than any CTA
    holds) gives the same bits, equal to the oracle within tolerance."""
    outs = {}
    old = da.decode_attn_get_option("attn_trigger")
    try:
        for trig in (0, 1, 3, 1000):
            da.decode_attn_set_option("attn_trigger", trig)
            x, _, out = _run(w, seed=31, ctas=ctas)
            outs[trig] = out
    finally:
        da.decode_attn_set_option("attn_trigger", old)
    for trig, out in outs.items():
        assert torch.equal(out, outs[0]), f"{w.name}: trigger point {trig} changed the output"
    _, ref_out = oracle_decode(orc, x)
    assert_bf16_close(f64(outs[3]), ref_out, f"{w.name} output")


@pytest.mark.parametrize("ctas", [1, 2, 7, 300])
def test_cta_count_does_not_change_the_result(orc, ctas):
    """Split-KV over any number of persistent CTAs (1 = no split at all, 300 = more
    CTAs than many sequences have tiles) equals the oracle and the default plan."""
    w = W("splits", 3, 16, 2, 700, 256, (700, 333, 64))
    x, attn, out = _run(w, seed=5, ctas=ctas)
    _, attn0, out0 = _run(w, seed=5, ctas=0)
    ref_attn, ref_out = oracle_decode(orc, x)
    assert_bf16_close(f64(attn), ref_attn, f"ctas={ctas} attention")
    assert_bf16_close(f64(out), ref_out, f"ctas={ctas} output")
    # Each split rounds its weights P to bf16 against its own running maximum
    # (relative error <= 2^-9 per weight), and the outputs are rounded to bf16
    # (<= 2^-9 relative). So |split - unsplit| <= 2 * 2^-9 * (sum_t p_t |v_t| + |o|),
    # bounded here by 2^-8 * (max|v| + |o|) elementwise.
    a, b = f64(attn), f64(attn0)
    vmax = float(x["v_cache"].abs().max())
    assert np.all(np.abs(a - b) <= 2.0 ** -8 * (vmax + np.maximum(np.abs(a), np.abs(b))))
    assert np.sqrt(np.sum((a - b) ** 2) / np.sum(b * b)) <= 2e-3


def test_range_starts_at_every_kind_of_tile(orc):
    """The set-up warp computes each CTA's range and the cursor at its first tile, copies the
    first tile of each consumer group (the second only inside the same sequence), and the
    consumers read the first segment's q themselves. Sweeping the CTA count moves the range
    boundaries over every position: a range of one tile, a range that starts on a sequence's
    last tile (its second tile opens the next sequence and carries q), ranges that start
    mid-sequence, empty rows between (equal prefix entries), one tile per CTA (more CTAs
    than tiles). Every split must equal the oracle."""
    # tiles of 64 tokens per row: 0, 1, 1, 5, 2, 2, 0, 3; two KV heads: 28 tiles
    w = W("firsttiles", 8, 8, 2, 300, 256, (0, 64, 1, 300, 65, 128, 0, 150))
    x = synth.make_inputs(w, seed=23, device=DEV)
    ref_attn, _ = oracle_decode(orc, x)
    old_ctas, old_cl = da.decode_attn_get_option("attn_ctas"), da.decode_attn_get_option("attn_cluster")
    try:
        da.decode_attn_set_option("attn_cluster", 0)
        for ctas in list(range(1, 31)) + [57]:
            da.decode_attn_set_option("attn_ctas", ctas)
            attn = torch.full((w.B, w.Hq, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
            da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"])
            torch.cuda.synchronize()
            assert da.decode_attn_last_device_error() == 0
            assert_bf16_close(f64(attn), ref_attn, f"ctas={ctas} attention")
    finally:
        da.decode_attn_set_option("attn_ctas", old_ctas)
        da.decode_attn_set_option("attn_cluster", old_cl)


def test_step_with_clusters_at_every_size(orc):
    """attn_cluster = 2: decode_attn_fwd takes the cluster mode for small problems too."""
    w = W("fwd_clusters", 1, 32, 8, 2048, 1024, (2048,))
    x = synth.make_inputs(w, seed=29, device=DEV)
    _, ref_out = oracle_decode(orc, x)
    old = da.decode_attn_get_option("attn_cluster")
    try:
        da.decode_attn_set_option("attn_cluster", 2)
        out = torch.full((w.B, w.N), float("nan"), dtype=torch.bfloat16, device=DEV)
        da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"])
        torch.cuda.synchronize()
    finally:
        da.decode_attn_set_option("attn_cluster", old)
    assert da.decode_attn_last_device_error() == 0
    assert_bf16_close(f64(out), ref_out, "clusters at batch 1: output")


def test_lengths_are_clamped_to_the_cache(orc):
    w = W("clamp", 3, 8, 2, 100, 256, (150, -5, 100))
    x, attn, out = _run(w)
    ref_attn, ref_out = oracle_decode(orc, x)  # the helper clamps to [0, Lcap] for the oracle
    assert_bf16_close(f64(attn), ref_attn, "clamped attention")
    assert np.all(f64(attn)[1] == 0.0)
    assert_bf16_close(f64(out), ref_out, "clamped output")


def test_garbage_past_seq_len_is_ignored():
    """Inf and NaN in cache rows t >= seq_len must not reach the output."""
    w = W("garbage", 2, 8, 2, 200, 256, (70, 129))
    x = synth.make_inputs(w, seed=1, device=DEV)
    a0 = torch.empty((2, 8, 128), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], a0, x["scale"])
    x["k_cache"][0, :, 70:] = float("inf")
    x["v_cache"][0, :, 70:] = float("nan")
    x["k_cache"][1, :, 129:] = float("nan")
    x["v_cache"][1, :, 129:] = float("inf")
    a1 = torch.empty_like(a0)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], a1, x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(a0, a1)


def test_softmax_rows_sum_to_one():
    """V = 1: every attention output is exactly 1.0 after the bf16 store."""
    w = W("ones", 2, 16, 2, 333, 256, (333, 70))
    x = synth.make_inputs(w, seed=2, device=DEV)
    x["v_cache"].fill_(1.0)
    attn = torch.empty((2, 16, 128), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"])
    assert torch.all(attn.float() == 1.0)


def test_identical_keys_give_the_mean_of_v():
    w = W("same_keys", 1, 8, 2, 250, 256, (250,))
    x = synth.make_inputs(w, seed=3, device=DEV)
    x["k_cache"][:] = x["k_cache"][:, :, :1]
    attn = torch.empty((1, 8, 128), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"])
    mean = x["v_cache"].double().mean(dim=2)  # [1, Hkv, 128]
    ref = mean.repeat_interleave(4, dim=1)
    assert torch.max(torch.abs(attn.double() - ref)).item() <= 2.0 ** -8 * ref.abs().max().item() + 1e-3


def test_dominant_key_copies_its_value_row():
    w = W("dominant", 1, 8, 2, 300, 256, (300,))
    x = synth.make_inputs(w, seed=4, device=DEV)
    q = torch.zeros_like(x["q"])
    q[..., 0] = 8.0
    x["q"] = q
    x["k_cache"].clamp_(-2, 2)
    tstar = 211
    x["k_cache"][:, :, tstar, 0] = 64.0  # scaled score 45.25 vs <= 1.42 for the others
    attn = torch.empty((1, 8, 128), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"])
    ref = x["v_cache"][:, :, tstar].repeat_interleave(4, dim=1)  # [1, 8, 128]
    assert torch.equal(attn, ref)


@pytest.mark.parametrize("rise", [3.0, 30.0, 600.0, -60.0])
@pytest.mark.parametrize("D", [128, 256])
def test_running_maximum_moving_along_the_sequence(orc, rise, D):
    """Scores that rise (or fall) along the sequence by about `rise` log2 units in all (a ramp
    in dim 0 of K, q[0] = 4): the running reference of the online softmax then moves every
    few tiles (30), on every tile (600: ~8.7 per 16 tokens), never after the first tile (-60)
    or hardly at all (3). Every case equals the oracle, on one CTA and on many."""
    w = synth.Workload("ramp", B=2, Hq=8, Hkv=2, Lcap=1100, N=256, fixed_lens=(1100, 777), D=D)
    x = synth.make_inputs(w, seed=9, device=DEV)
    x["q"][..., 0] = 4.0
    per_unit = 4.0 * x["scale"] * math.log2(math.e)  # log2 units per unit of k[0]
    ramp = torch.arange(w.Lcap, device=DEV, dtype=torch.float32) * (rise / per_unit / w.Lcap)
    x["k_cache"][:, :, :, 0] = ramp.to(torch.bfloat16)
    ref_attn, _ = oracle_decode(orc, x)
    old = da.decode_attn_get_option("attn_ctas")
    try:
        for ctas in (1, 0):
            da.decode_attn_set_option("attn_ctas", ctas)
            attn = torch.full((w.B, w.Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
            da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"])
            torch.cuda.synchronize()
            assert_bf16_close(f64(attn), ref_attn, f"rise {rise}, D {D}, ctas {ctas}")
    finally:
        da.decode_attn_set_option("attn_ctas", old)


# ------------------------------------------------------------- fp32 scores
@pytest.mark.parametrize("G,Hkv", [(4, 2), (8, 1), (16, 1), (3, 2)])
def test_scores_match_oracle(orc, G, Hkv):
    B, Lcap = 2, 203
    w = W("scores", B, G * Hkv, Hkv, Lcap, 8, (203, 90))
    x = synth.make_inputs(w, seed=9, device=DEV)
    s = torch.full((B, w.Hq, Lcap), float("nan"), dtype=torch.float32, device=DEV)
    da.decode_attn_scores(x["q"], x["k_cache"], x["seq_lens"], s)
    ref = orc.scores(synth.to_bits(x["q"]), synth.to_bits(x["k_cache"]), x["seq_lens"].cpu().numpy())
    got = s.cpu().numpy().astype(np.float64)
    for b in range(B):
        L = int(x["seq_lens"][b])
        assert np.all(np.isnan(got[b, :, L:])), "scores past seq_len must be left untouched"
        num = np.linalg.norm(got[b, :, :L] - ref[b, :, :L], axis=1)
        den = np.linalg.norm(ref[b, :, :L], axis=1)
        assert np.all(num <= RTOL_SCORES * den), f"b={b}: worst rel {np.max(num / den):.2e}"


def test_integer_scores_are_exact(orc):
    """Integer-valued q and K: every fp32 partial sum is exact, so the scores equal
    the oracle bit for bit (the integer-valued golden check of the CANN page "自动调优流程")."""
    B, Hq, Hkv, Lcap = 2, 8, 2, 150
    g = torch.Generator(device="cpu").manual_seed(21)
    q = torch.randint(-4, 5, (B, Hq, 128), generator=g).to(torch.bfloat16).to(DEV)
    k = torch.randint(-4, 5, (B, Hkv, Lcap, 128), generator=g).to(torch.bfloat16).to(DEV)
    lens = torch.tensor([150, 77], dtype=torch.int32, device=DEV)
    s = torch.full((B, Hq, Lcap), float("nan"), dtype=torch.float32, device=DEV)
    da.decode_attn_scores(q, k, lens, s)
    ref = orc.scores(synth.to_bits(q), synth.to_bits(k), lens.cpu().numpy())
    got = s.cpu().numpy().astype(np.float64)
    mask = ~np.isnan(ref)
    assert np.array_equal(got[mask], ref[mask])


# ------------------------------------------------------------ output projection
@pytest.mark.parametrize("B", [1, 2, 3, 4, 5, 8, 9, 16])
def test_oproj_integer_exact(B):
    """Integer attention rows and W in {-1, 0, 1}: fp32 sums are exact, so the result
    is the round-to-nearest-even bf16 of the exact integer matmul."""
    K, N = 1032, 264  # ragged k-slices and a partial 256-column block
    g = torch.Generator(device="cpu").manual_seed(100 + B)
    xi = torch.randint(-8, 9, (B, K), generator=g)
    wi = torch.randint(-1, 2, (K, N), generator=g)
    ref = (xi.long() @ wi.long()).double().to(torch.bfloat16)
    out = torch.full((B, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_oproj(xi.to(torch.bfloat16).to(DEV), wi.to(torch.bfloat16).to(DEV), out)
    assert torch.equal(out.cpu(), ref)


@pytest.mark.parametrize("B,K,N", [(1, 4096, 4096), (4, 512, 1024), (8, 1024, 768), (32, 256, 512)])
def test_oproj_matches_oracle(orc, B, K, N):
    g = torch.Generator(device="cpu").manual_seed(7)
    x = torch.randn((B, K), generator=g).to(torch.bfloat16)
    w = (torch.randn((K, N), generator=g) / math.sqrt(K)).to(torch.bfloat16)
    out = torch.empty((B, N), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_oproj(x.to(DEV), w.to(DEV), out)
    ref = orc.oproj(synth.to_bits(x), synth.to_bits(w))
    assert_bf16_close(f64(out), ref, "o_proj")


def test_strided_views():
    """Non-contiguous but legal views (padded rows, a sliced cache) give the same bits."""
    w = W("strided", 2, 8, 2, 130, 256, (130, 50))
    x = synth.make_inputs(w, seed=11, device=DEV)
    ref = torch.empty((2, w.N), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], ref, x["scale"])
    big_k = torch.zeros((2, 3, 160, 136), dtype=torch.bfloat16, device=DEV)
    big_v = torch.zeros((2, 3, 160, 136), dtype=torch.bfloat16, device=DEV)
    big_k[:, 1:3, 5:135, :128] = x["k_cache"]
    big_v[:, 1:3, 5:135, :128] = x["v_cache"]
    k_view = big_k[:, 1:3, 5:135, :128]
    v_view = big_v[:, 1:3, 5:135, :128]
    q_big = torch.zeros((2, 8, 136), dtype=torch.bfloat16, device=DEV)
    q_big[..., :128] = x["q"]
    w_big = torch.zeros((w.Hq * 128, 272), dtype=torch.bfloat16, device=DEV)
    w_big[:, :256] = x["o_weight"]
    out_big = torch.zeros((2, 300), dtype=torch.bfloat16, device=DEV)
    out_view = out_big[:, 8:264]
    da.decode_attn_fwd(q_big[..., :128], k_view, v_view, x["seq_lens"], w_big[:, :256], out_view, x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out_view, ref)
    assert torch.all(out_big[:, :8] == 0) and torch.all(out_big[:, 264:] == 0)


def test_repeated_calls_are_deterministic():
    w = W("repeat", 4, 32, 8, 1000, 512, (1000, 999, 500, 3))
    x = synth.make_inputs(w, seed=12, device=DEV)
    outs = []
    for _ in range(3):
        o = torch.empty((4, 512), dtype=torch.bfloat16, device=DEV)
        da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], o, x["scale"])
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


# ------------------------------------------------- tensor-core projection path
class _Path:
    def __init__(self, path):
        self.path = path

    def __enter__(self):
        self.old = da.decode_attn_get_option("oproj_path")
        da.decode_attn_set_option("oproj_path", self.path)

    def __exit__(self, *exc):
        da.decode_attn_set_option("oproj_path", self.old)


# every batch on the small shapes; the full-size W (4096 x 4096) at a few batch sizes
GEMM_EXACT = [(B, K, N) for K, N in [(1088, 384), (256, 264)] for B in (1, 2, 3, 8, 9, 16, 17, 32, 33, 64, 65, 128, 130)]
GEMM_EXACT += [(B, 4096, 4096) for B in (1, 8, 16, 64)]


@pytest.mark.parametrize("B,K,N", GEMM_EXACT)
@pytest.mark.parametrize("path", [1, 2])
def test_oproj_gemm_integer_exact(path, B, K, N):
    """Both projection paths (1: CUDA-core GEMV, 2: tcgen05): integer operands make every
    fp32 sum exact, so the result is the bf16 rounding of the exact integer matmul
    (batch padding, batch chunks, ragged split-K, partial column tiles)."""
    g = torch.Generator(device="cpu").manual_seed(300 + B + K)
    xi = torch.randint(-8, 9, (B, K), generator=g)
    wi = torch.randint(-1, 2, (K, N), generator=g)
    ref = (xi.long() @ wi.long()).double().to(torch.bfloat16)
    out = torch.full((B, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    with _Path(path):
        da.decode_attn_oproj(xi.to(torch.bfloat16).to(DEV), wi.to(torch.bfloat16).to(DEV), out)
    torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    assert torch.equal(out.cpu(), ref)


@pytest.mark.parametrize("B,K,N", [(8, 4096, 4096), (32, 4096, 4096), (64, 1024, 2048), (5, 512, 640),
                                   (1, 4096, 4096), (16, 8192, 8192), (12, 1000, 776)])
@pytest.mark.parametrize("path", [1, 2])
def test_oproj_gemm_matches_oracle(orc, path, B, K, N):
    g = torch.Generator(device="cpu").manual_seed(8)
    x = torch.randn((B, K), generator=g).to(torch.bfloat16)
    w = (torch.randn((K, N), generator=g) / math.sqrt(K)).to(torch.bfloat16)
    out = torch.empty((B, N), dtype=torch.bfloat16, device=DEV)
    with _Path(path):
        da.decode_attn_oproj(x.to(DEV), w.to(DEV), out)
    ref = orc.oproj(synth.to_bits(x), synth.to_bits(w))
    assert_bf16_close(f64(out), ref, f"o_proj path {path}")


@pytest.mark.parametrize("path", [1, 2])
def test_fused_step_on_each_projection_path(orc, path):
    w = W("paths", 12, 16, 4, 300, 512, (300, 1, 64, 65, 299, 128, 0, 7, 200, 100, 50, 3))
    with _Path(path):
        x, attn, out = _run(w, seed=13)
    ref_attn, ref_out = oracle_decode(orc, x)
    assert_bf16_close(f64(attn), ref_attn, f"path {path} attention")
    assert_bf16_close(f64(out), ref_out, f"path {path} output")


# ------------------------------------------------------------- fused decode step
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


FUSED_CASES = [
    W("f_b1_g4", 1, 32, 8, 700, 4096, (700,)),
    W("f_b3_g4_ragged", 3, 8, 2, 300, 256, (300, 0, 129)),
    W("f_b8_g8", 8, 16, 2, 200, 384, (200, 1, 64, 65, 199, 128, 3, 100)),
    W("f_b17_g16", 17, 32, 2, 130, 264, tuple([130, 1] * 8 + [64])),
    W("f_b40_g4", 40, 8, 2, 90, 512, tuple(int(x) for x in np.random.default_rng(5).integers(0, 91, 40))),
    W("f_b100_g1", 100, 4, 4, 70, 128, tuple(int(x) for x in np.random.default_rng(6).integers(1, 71, 100))),
]


@pytest.mark.parametrize("w", FUSED_CASES, ids=[c.name for c in FUSED_CASES])
def test_fused_step_matches_oracle_and_two_launches(orc, w):
    """decode_attn_fwd as one persistent launch (attention, grid barrier, tcgen05
    projection) against the oracle and against the two-launch path."""
    with _Opt(fused=1):
        x, attn, out = _run(w, seed=17)
    with _Opt(fused=0):
        out2 = torch.full_like(out, float("nan"))
        da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out2, x["scale"])
        torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    ref_attn, ref_out = oracle_decode(orc, x)
    assert_bf16_close(f64(out), ref_out, f"{w.name} fused output")
    assert_bf16_close(f64(out2), ref_out, f"{w.name} two-launch output")


def test_fused_step_integer_exact():
    """Integer attention outputs (V rows constant per KV head make every output an
    integer) and W in {-1, 0, 1}: the fused projection is the exact integer product."""
    B, Hq, Hkv, L, N = 8, 32, 8, 333, 384
    w = W("f_int", B, Hq, Hkv, L, N, (L,) * B)
    x = synth.make_inputs(w, seed=3, device=DEV)
    vals = torch.randint(-3, 4, (B, Hkv, 1, 128), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    x["v_cache"][:] = vals.to(DEV)  # softmax weights sum to one: attention = that row exactly
    wi = torch.randint(-1, 2, (Hq * 128, N), generator=torch.Generator().manual_seed(5))
    attn_ref = vals[:, :, 0].repeat_interleave(Hq // Hkv, dim=1).reshape(B, Hq * 128).long()
    ref = (attn_ref @ wi.long()).double().to(torch.bfloat16)
    out = torch.full((B, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    with _Opt(fused=1):
        da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], wi.to(torch.bfloat16).to(DEV), out,
                           x["scale"])
    torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    assert torch.equal(out.cpu(), ref)


def test_graph_replays_and_eager_calls_agree_with_the_oracle(orc):
    """decode_attn_fwd captured in a CUDA graph and replayed, interleaved with eager calls,
    on inputs refilled in place between calls: every result matches the oracle (the
    workspace's completion counters return to zero after every call, whichever way it
    was launched)."""
    w = W("graph", 2, 32, 8, 1000, 512, (1000, 517))
    x = synth.make_inputs(w, seed=31, device=DEV)
    out = torch.full((w.B, w.N), float("nan"), dtype=torch.bfloat16, device=DEV)
    st = torch.cuda.Stream(DEV)
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"])
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"])
        for i in range(6):
            y = synth.make_inputs(w, seed=40 + i, device=DEV)
            for k in ("q", "k_cache", "v_cache"):
                x[k].copy_(y[k])
            out.fill_(float("nan"))
            if i % 2:
                da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"])
            else:
                g.replay()
            st.synchronize()
            assert da.decode_attn_last_device_error(st) == 0
            _, ref_out = oracle_decode(orc, x)
            assert_bf16_close(f64(out), ref_out, f"call {i} ({'eager' if i % 2 else 'graph'})")
    del g


# ------------------------------------------- batch-1 projection staged on chip (option 3)
ONCHIP_CASES = [
    W("oc_b1_h4096", 1, 32, 8, 2048, 4096, (2048,)),
    W("oc_b1_short", 1, 32, 8, 2048, 4096, (301,)),
    W("oc_b1_n2048", 1, 32, 8, 1024, 2048, (1000,)),
    W("oc_b1_g8", 1, 64, 8, 512, 4096, (512,)),
    W("oc_b1_empty", 1, 32, 8, 256, 4096, (0,)),
]


@pytest.mark.parametrize("w", ONCHIP_CASES, ids=[c.name for c in ONCHIP_CASES])
def test_onchip_projection_matches_oracle(orc, w):
    """Batch 1 with the projection staged on chip behind the attention (option oproj_path = 3,
    where the free SMs can hold W) against the oracle, and
    against the tcgen05 projection within the bf16 tolerance (their sums run in other orders).
    Called three times in a row: the strip counters return to zero after every call."""
    x = synth.make_inputs(w, seed=19, device=DEV)
    outs = {}
    for path in (3, 2):
        with _Opt(oproj_path=path):
            out = torch.full((w.B, w.N), float("nan"), dtype=torch.bfloat16, device=DEV)
            for _ in range(3):
                da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"])
            torch.cuda.synchronize()
            assert da.decode_attn_last_device_error() == 0
            outs[path] = out
    _, ref_out = oracle_decode(orc, x)
    assert_bf16_close(f64(outs[3]), ref_out, f"{w.name} on-chip projection")
    assert_bf16_close(f64(outs[3]), f64(outs[2]), f"{w.name} on-chip vs tcgen05 projection")


def test_onchip_projection_integer_exact():
    """Integer attention outputs (V rows constant per KV head) and W in {-1, 0, 1}: the
    on-chip projection's fp32 sums are exact, so the result is the exact integer product."""
    B, Hq, Hkv, L, N = 1, 32, 8, 777, 4096
    w = W("oc_int", B, Hq, Hkv, L, N, (L,))
    x = synth.make_inputs(w, seed=3, device=DEV)
    vals = torch.randint(-3, 4, (B, Hkv, 1, 128), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    x["v_cache"][:] = vals.to(DEV)
    wi = torch.randint(-1, 2, (Hq * 128, N), generator=torch.Generator().manual_seed(5))
    attn_ref = vals[:, :, 0].repeat_interleave(Hq // Hkv, dim=1).reshape(B, Hq * 128).long()
    ref = (attn_ref @ wi.long()).double().to(torch.bfloat16)
    out = torch.full((B, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    with _Opt(oproj_path=3):
        da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], wi.to(torch.bfloat16).to(DEV), out,
                           x["scale"])
    torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    assert torch.equal(out.cpu(), ref)
