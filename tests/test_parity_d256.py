"""Parity of the head-dim-256 attention path (through the C ABI) with the fp64 oracle.

Head dim 256 is the second decode-attention shape of the page "PyPTO 开箱性能调优实战
Decode Attention 多 Matmul 独立 TileShape 配置 F-16", section "仓库源码佐证": a GQA
decode whose QK^T contracts D = 256 in two 128-wide halves and whose attn.V has
N = D = 256. The kernel streams 32-token tiles there, so these cases span several
such tiles, ragged tails (1, 31, 33 tokens), every group width the kernel
specialises on (G <= 8 and G <= 16), empty sequences and CTA counts from one to
more than the tiles.
"""
import numpy as np
import pytest
import torch

import decode_attention_output_gb300 as da
from decode_attention_output_gb300 import synth
from gpu_helpers import RTOL_SCORES, assert_bf16_close, f64, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
D = 256


@pytest.fixture(scope="module", autouse=True)
def _library():
    from decode_attention_output_gb300 import build

    build.build()
    da.load()
    torch.cuda.set_device(0)
    yield
    assert da.decode_attn_last_device_error() == 0


def W(name, B, Hq, Hkv, Lcap, N, lens, k_mult=1.0):
    return synth.Workload(name, B=B, Hq=Hq, Hkv=Hkv, Lcap=Lcap, N=N, fixed_lens=tuple(lens), k_mult=k_mult, D=D)


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


CASES = [
    W("d256_g4_ragged", 3, 8, 2, 300, 256, (300, 1, 129)),
    W("d256_g4_tiles", 2, 32, 8, 640, 1024, (640, 511)),
    W("d256_g8", 2, 16, 2, 200, 512, (200, 77)),
    W("d256_g16", 2, 32, 2, 150, 256, (150, 31)),
    W("d256_g1_mha", 2, 4, 4, 100, 128, (100, 16)),
    W("d256_g3", 2, 6, 2, 257, 264, (257, 33)),
    W("d256_g5_sharp", 2, 10, 2, 190, 640, (190, 32), k_mult=2.0),
    W("d256_zero_len", 3, 8, 2, 130, 256, (0, 130, 65)),
    W("d256_tiny", 1, 2, 1, 1, 8, (1,)),
    W("d256_one_tile", 1, 8, 2, 32, 256, (32,)),
    W("d256_many_batches", 40, 8, 1, 70, 128, tuple(int(x) for x in np.random.default_rng(7).integers(0, 71, 40))),
    # clusters of two and four CTAs (on-chip merges), and G = 16, which merges through L2
    W("d256_equal_cs2", 8, 32, 8, 1024, 512, (1024,) * 8),
    W("d256_ragged_cs4", 4, 32, 8, 2048, 256, (2048, 5, 1500, 33)),
    W("d256_g16_flat", 2, 32, 2, 1000, 256, (1000, 400)),
]


def _run(w, seed=0, ctas=0):
    x = synth.make_inputs(w, seed=seed, device=DEV)
    with _Opt(attn_ctas=ctas):
        attn = torch.full((w.B, w.Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
        da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"])
        out = torch.full((w.B, w.N), float("nan"), dtype=torch.bfloat16, device=DEV)
        da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"])
        torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    return x, attn, out


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_decode_d256_matches_oracle(orc, w):
    x, attn, out = _run(w)
    ref_attn, ref_out = oracle_decode(orc, x)
    assert_bf16_close(f64(attn), ref_attn, f"{w.name} attention")
    assert_bf16_close(f64(out), ref_out, f"{w.name} output")


CLUSTER_CASES = [c for c in CASES if c.name in ("d256_equal_cs2", "d256_ragged_cs4", "d256_g16_flat", "d256_g4_ragged",
                                                 "d256_zero_len", "d256_tiny")]


@pytest.mark.parametrize("w", CLUSTER_CASES, ids=[c.name for c in CLUSTER_CASES])
def test_d256_cluster_and_flat_grids(orc, w):
    """Clusters of two to eight CTAs with on-chip merges (the default where they fit; G = 16
    at D = 256 has no room for the parked states and merges through L2) and the flat grid
    (option attn_cluster = 0), both against the oracle."""
    for mode in (1, 0):
        with _Opt(attn_cluster=mode):
            x, attn, out = _run(w, seed=3)
        ref_attn, ref_out = oracle_decode(orc, x)
        assert_bf16_close(f64(attn), ref_attn, f"{w.name} attention, attn_cluster {mode}")
        assert_bf16_close(f64(out), ref_out, f"{w.name} output, attn_cluster {mode}")


@pytest.mark.parametrize("ctas", [1, 2, 7, 300])
def test_d256_cta_count_does_not_change_the_result(orc, ctas):
    w = W("d256_splits", 3, 16, 2, 700, 256, (700, 333, 32))
    x, attn, out = _run(w, seed=5, ctas=ctas)
    _, attn0, _ = _run(w, seed=5, ctas=0)
    ref_attn, ref_out = oracle_decode(orc, x)
    assert_bf16_close(f64(attn), ref_attn, f"ctas={ctas} attention")
    assert_bf16_close(f64(out), ref_out, f"ctas={ctas} output")
    # the same bound as at head dim 128: bf16 weights per split and the bf16 store
    a, b = f64(attn), f64(attn0)
    vmax = float(x["v_cache"].abs().max())
    assert np.all(np.abs(a - b) <= 2.0 ** -8 * (vmax + np.maximum(np.abs(a), np.abs(b))))


@pytest.mark.parametrize("G,Hkv", [(4, 2), (8, 1), (16, 1), (3, 2)])
def test_d256_scores_match_oracle(orc, G, Hkv):
    B, Lcap = 2, 203
    w = W("d256_scores", B, G * Hkv, Hkv, Lcap, 8, (203, 45))
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


def test_d256_integer_scores_are_exact(orc):
    """Integer q and K in [-4, 4]: |partial sums| <= 256 * 16, exact in fp32, so both
    128-dim halves and their sum match the oracle bit for bit."""
    B, Hq, Hkv, Lcap = 2, 8, 2, 101
    g = torch.Generator(device="cpu").manual_seed(23)
    q = torch.randint(-4, 5, (B, Hq, D), generator=g).to(torch.bfloat16).to(DEV)
    k = torch.randint(-4, 5, (B, Hkv, Lcap, D), generator=g).to(torch.bfloat16).to(DEV)
    lens = torch.tensor([101, 33], dtype=torch.int32, device=DEV)
    s = torch.full((B, Hq, Lcap), float("nan"), dtype=torch.float32, device=DEV)
    da.decode_attn_scores(q, k, lens, s)
    ref = orc.scores(synth.to_bits(q), synth.to_bits(k), lens.cpu().numpy())
    got = s.cpu().numpy().astype(np.float64)
    mask = ~np.isnan(ref)
    assert np.array_equal(got[mask], ref[mask])


def test_d256_softmax_rows_sum_to_one():
    w = W("d256_ones", 2, 16, 2, 333, 256, (333, 70))
    x = synth.make_inputs(w, seed=2, device=DEV)
    x["v_cache"].fill_(1.0)
    attn = torch.empty((2, 16, D), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"])
    assert torch.all(attn.float() == 1.0)


def test_d256_dominant_key_copies_its_value_row():
    """A key whose scaled score beats the rest by > 40 in the upper half of the dims
    only: the output is that key's V row in both halves (a dropped half would miss it)."""
    w = W("d256_dominant", 1, 8, 2, 300, 256, (300,))
    x = synth.make_inputs(w, seed=4, device=DEV)
    q = torch.zeros_like(x["q"])
    q[..., 200] = 8.0
    x["q"] = q
    x["k_cache"].clamp_(-2, 2)
    tstar = 117
    x["k_cache"][:, :, tstar, 200] = 128.0  # scaled score 64 vs <= 1 for the others
    attn = torch.empty((1, 8, D), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"])
    ref = x["v_cache"][:, :, tstar].repeat_interleave(4, dim=1)
    assert torch.equal(attn, ref)


def test_d256_garbage_past_seq_len_is_ignored():
    w = W("d256_garbage", 2, 8, 2, 200, 256, (70, 129))
    x = synth.make_inputs(w, seed=1, device=DEV)
    a0 = torch.empty((2, 8, D), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], a0, x["scale"])
    x["k_cache"][0, :, 70:] = float("inf")
    x["v_cache"][0, :, 70:] = float("nan")
    x["k_cache"][1, :, 129:] = float("nan")
    x["v_cache"][1, :, 129:] = float("inf")
    a1 = torch.empty_like(a0)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], a1, x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(a0, a1)


def test_d256_strided_views():
    """A cache padded to 264 dims and offset in tokens and heads gives the same bits."""
    w = W("d256_strided", 2, 8, 2, 130, 256, (130, 50))
    x = synth.make_inputs(w, seed=11, device=DEV)
    ref = torch.empty((2, 8, D), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], ref, x["scale"])
    big_k = torch.zeros((2, 3, 160, 264), dtype=torch.bfloat16, device=DEV)
    big_v = torch.zeros((2, 3, 160, 264), dtype=torch.bfloat16, device=DEV)
    big_k[:, 1:3, 5:135, :D] = x["k_cache"]
    big_v[:, 1:3, 5:135, :D] = x["v_cache"]
    q_big = torch.zeros((2, 8, 264), dtype=torch.bfloat16, device=DEV)
    q_big[..., :D] = x["q"]
    out_big = torch.zeros((2, 8, 272), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only(q_big[..., :D], big_k[:, 1:3, 5:135, :D], big_v[:, 1:3, 5:135, :D], x["seq_lens"],
                        out_big[..., 8:264], x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out_big[..., 8:264], ref)
    assert torch.all(out_big[..., :8] == 0) and torch.all(out_big[..., 264:] == 0)


def test_d256_fused_option_takes_two_launches():
    """The fused step is built for head dim 128; with the option on, head dim 256 runs
    the two-launch step and gives the same bits."""
    w = W("d256_fused", 3, 8, 2, 300, 256, (300, 0, 129))
    x = synth.make_inputs(w, seed=3, device=DEV)
    ref = torch.empty((3, 256), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], ref, x["scale"])
    out = torch.empty_like(ref)
    with _Opt(fused=1):
        da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_d256_no_alloc_entry_point_matches():
    w = W("d256_noalloc", 4, 16, 2, 400, 256, (400, 1, 0, 255))
    x = synth.make_inputs(w, seed=6, device=DEV)
    ref = torch.empty((4, 16, D), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], ref, x["scale"])
    got = torch.full_like(ref, float("nan"))
    da.decode_attn_only_noalloc(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], got, x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
