"""Parity of the paged-cache entry points (block table) through the C ABI.

A paged cache is the contiguous computation on the cache its block table describes,
so each case builds a contiguous cache, scatters it into a shuffled pool of blocks
(with spare blocks of noise), and checks the paged call against the fp64 oracle on
the gathered cache (within the bf16 tolerances) and against the contiguous call on
the same logical cache bit for bit: the kernel reads the same tiles in the same
order, and what lies past a sequence's length is masked either way. Block sizes
cover boxes cut from blocks (8, 16, 32 tokens) and blocks holding whole tiles.
"""
import numpy as np
import pytest
import torch

import decode_attention_output_gb300 as da
from decode_attention_output_gb300 import synth
from gpu_helpers import assert_bf16_close, f64

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


def scatter(cache: torch.Tensor, bs: int, seed: int, spare: int = 3):
    """cache [B, Hkv, Lcap, D] -> (pool [nblk, Hkv, bs, D], table [B, Lcap / bs] int32)."""
    B, Hkv, Lcap, D = cache.shape
    mb = Lcap // bs
    nblk = B * mb + spare
    g = torch.Generator(device="cpu").manual_seed(seed)
    perm = torch.randperm(nblk, generator=g)[: B * mb].view(B, mb)
    pool = torch.randn((nblk, Hkv, bs, D), generator=g).to(torch.bfloat16).to(cache.device)
    for b in range(B):
        for i in range(mb):
            pool[perm[b, i]] = cache[b, :, i * bs:(i + 1) * bs]
    return pool, perm.to(torch.int32).to(cache.device)


def W(name, B, Hq, Hkv, Lcap, N, lens, D=128):
    return synth.Workload(name, B=B, Hq=Hq, Hkv=Hkv, Lcap=Lcap, N=N, fixed_lens=tuple(lens), D=D)


CASES = [  # (workload, block size); Lcap is a multiple of the block size
    (W("p_g4_bs16", 3, 8, 2, 320, 256, (320, 1, 129)), 16),
    (W("p_g4_bs8", 2, 8, 2, 200, 256, (200, 63)), 8),
    (W("p_g8_bs32", 2, 16, 2, 224, 512, (224, 65)), 32),
    (W("p_g16_bs64", 2, 32, 2, 192, 256, (192, 64)), 64),
    (W("p_g4_bs128", 3, 8, 2, 384, 256, (384, 0, 200)), 128),
    (W("p_g1_bs256", 2, 4, 4, 512, 128, (300, 512)), 256),
    (W("p_many_bs16", 24, 8, 1, 96, 128, tuple(int(x) for x in np.random.default_rng(9).integers(0, 97, 24))), 16),
    (W("p_d256_bs16", 3, 8, 2, 320, 256, (320, 1, 129), D=256), 16),
    (W("p_d256_bs32", 2, 16, 2, 192, 256, (192, 33), D=256), 32),
    (W("p_d256_bs64_g16", 2, 32, 2, 256, 256, (256, 31), D=256), 64),
    (W("p_d256_bs8", 2, 8, 2, 96, 128, (96, 9), D=256), 8),
    # clusters of two CTAs (on-chip merges; a ragged mix partly through L2)
    (W("p_equal_cs2_bs16", 8, 32, 8, 1024, 512, (1024,) * 8), 16),
    (W("p_ragged_cs2_bs64", 8, 32, 8, 2048, 512, (2048, 0, 1, 1500, 64, 2000, 777, 129)), 64),
]


def _contiguous(w, x):
    attn = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device=DEV)
    out = torch.empty((w.B, w.N), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"])
    da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"])
    return attn, out


def _paged(w, x, kp, vp, table):
    attn = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = torch.full((w.B, w.N), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only_paged(x["q"], kp, vp, table, x["seq_lens"], attn, x["scale"])
    da.decode_attn_fwd_paged(x["q"], kp, vp, table, x["seq_lens"], x["o_weight"], out, x["scale"])
    return attn, out


@pytest.mark.parametrize("w,bs", CASES, ids=[c[0].name for c in CASES])
def test_paged_matches_oracle_and_contiguous(orc, w, bs):
    x = synth.make_inputs(w, seed=21, device=DEV)
    kp, table = scatter(x["k_cache"], bs, seed=1)
    vp, _ = scatter(x["v_cache"], bs, seed=1)
    attn, out = _paged(w, x, kp, vp, table)
    attn0, out0 = _contiguous(w, x)
    torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    assert torch.equal(attn, attn0), "paged attention differs from the contiguous path"
    assert torch.equal(out, out0), "paged output differs from the contiguous path"
    lens = x["seq_lens"].cpu().numpy().astype(np.int32)
    ref_attn, ref_out = orc.decode_paged(synth.to_bits(x["q"]), synth.to_bits(kp), synth.to_bits(vp),
                                         table.cpu().numpy(), lens, synth.to_bits(x["o_weight"]), x["scale"])
    assert_bf16_close(f64(attn), ref_attn, f"{w.name} attention")
    assert_bf16_close(f64(out), ref_out, f"{w.name} output")


@pytest.mark.parametrize("ctas", [1, 5, 300])
def test_paged_cta_counts(orc, ctas):
    w = W("p_splits", 3, 16, 2, 640, 256, (640, 333, 17))
    x = synth.make_inputs(w, seed=22, device=DEV)
    kp, table = scatter(x["k_cache"], 16, seed=2)
    vp, _ = scatter(x["v_cache"], 16, seed=2)
    old = da.decode_attn_get_option("attn_ctas")
    da.decode_attn_set_option("attn_ctas", ctas)
    try:
        attn, out = _paged(w, x, kp, vp, table)
        attn0, out0 = _contiguous(w, x)
        torch.cuda.synchronize()
    finally:
        da.decode_attn_set_option("attn_ctas", old)
    assert torch.equal(attn, attn0) and torch.equal(out, out0)


def test_paged_token_major_pool_view():
    """A pool stored as [num_blocks, block_size, Hkv, D] is passed as a permuted view."""
    w = W("p_view", 2, 8, 2, 256, 256, (256, 100))
    x = synth.make_inputs(w, seed=23, device=DEV)
    kp, table = scatter(x["k_cache"], 32, seed=3)
    vp, _ = scatter(x["v_cache"], 32, seed=3)
    kp_tok = kp.permute(0, 2, 1, 3).contiguous()  # [nblk, bs, Hkv, D] in memory
    vp_tok = vp.permute(0, 2, 1, 3).contiguous()
    attn = torch.empty((2, 8, 128), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only_paged(x["q"], kp_tok.permute(0, 2, 1, 3), vp_tok.permute(0, 2, 1, 3), table, x["seq_lens"],
                              attn, x["scale"])
    attn0, _ = _contiguous(w, x)
    torch.cuda.synchronize()
    assert torch.equal(attn, attn0)


def test_paged_table_row_stride_and_unused_entries():
    """A padded table (row stride > max_blocks) works, and entries past a sequence's
    last block are never read (they hold out-of-pool ids here, without an error)."""
    w = W("p_table", 2, 8, 2, 160, 256, (40, 160))
    x = synth.make_inputs(w, seed=24, device=DEV)
    kp, table = scatter(x["k_cache"], 16, seed=4)
    vp, _ = scatter(x["v_cache"], 16, seed=4)
    big = torch.full((2, 16), 1 << 30, dtype=torch.int32, device=DEV)
    big[:, :10] = table
    big[0, 3:10] = -1  # row 0 has 40 tokens: entries 3.. are unused
    attn = torch.empty((2, 8, 128), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only_paged(x["q"], kp, vp, big[:, :10], x["seq_lens"], attn, x["scale"])
    attn0, _ = _contiguous(w, x)
    torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    assert torch.equal(attn, attn0)


def test_paged_out_of_pool_block_is_reported(orc):
    """A used table entry outside the pool sets bit 64 of the device error word and
    its tokens read as zeros (as the oracle's gather defines)."""
    w = W("p_bad", 2, 8, 2, 64, 256, (64, 64))
    x = synth.make_inputs(w, seed=25, device=DEV)
    kp, table = scatter(x["k_cache"], 16, seed=5)
    vp, _ = scatter(x["v_cache"], 16, seed=5)
    table[1, 2] = kp.shape[0] + 7
    attn = torch.empty((2, 8, 128), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only_paged(x["q"], kp, vp, table, x["seq_lens"], attn, x["scale"])
    assert da.decode_attn_last_device_error() == 64
    assert da.decode_attn_last_device_error() == 0  # reading the word cleared it
    lens = x["seq_lens"].cpu().numpy().astype(np.int32)
    ref = orc.attention(synth.to_bits(x["q"]), orc.gather_pages(synth.to_bits(kp), table.cpu().numpy(), lens),
                        orc.gather_pages(synth.to_bits(vp), table.cpu().numpy(), lens), lens, x["scale"])
    assert_bf16_close(f64(attn), ref, "out-of-pool block")


def test_paged_empty_batch_is_a_noop():
    q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device=DEV)
    kp = torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16, device=DEV)
    table = torch.empty((0, 3), dtype=torch.int32, device=DEV)
    lens = torch.empty((0,), dtype=torch.int32, device=DEV)
    attn = torch.empty((0, 8, 128), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_only_paged(q, kp, kp, table, lens, attn, 0.1)
    torch.cuda.synchronize()


def test_paged_trigger_point_does_not_change_the_result():
    """The projection's launch point (option attn_trigger) is timing only on the paged path too."""
    w = W("p_trig_bs16", 2, 32, 8, 1024, 512, (1024, 77))
    x = synth.make_inputs(w, seed=23, device=DEV)
    kp, table = scatter(x["k_cache"], 16, seed=2)
    vp, _ = scatter(x["v_cache"], 16, seed=2)
    old = da.decode_attn_get_option("attn_trigger")
    outs = []
    try:
        for trig in (0, 3):
            da.decode_attn_set_option("attn_trigger", trig)
            outs.append(_paged(w, x, kp, vp, table)[1])
    finally:
        da.decode_attn_set_option("attn_trigger", old)
    torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    assert torch.equal(outs[0], outs[1])


CLUSTER_CASES = [c for c in CASES if c[0].name in ("p_equal_cs2_bs16", "p_ragged_cs2_bs64", "p_g4_bs16", "p_d256_bs16")]


@pytest.mark.parametrize("w,bs", CLUSTER_CASES, ids=[c[0].name for c in CLUSTER_CASES])
def test_paged_flat_grid(orc, w, bs):
    """The flat grid (option attn_cluster = 0) on the cases that take clusters by default: the
    paged path equals the contiguous one under the same plan, and the oracle."""
    x = synth.make_inputs(w, seed=24, device=DEV)
    kp, table = scatter(x["k_cache"], bs, seed=3)
    vp, _ = scatter(x["v_cache"], bs, seed=3)
    old = da.decode_attn_get_option("attn_cluster")
    da.decode_attn_set_option("attn_cluster", 0)
    try:
        attn, out = _paged(w, x, kp, vp, table)
        attn0, out0 = _contiguous(w, x)
        torch.cuda.synchronize()
    finally:
        da.decode_attn_set_option("attn_cluster", old)
    assert da.decode_attn_last_device_error() == 0
    assert torch.equal(attn, attn0) and torch.equal(out, out0)
    lens = x["seq_lens"].cpu().numpy().astype(np.int32)
    ref_attn, ref_out = orc.decode_paged(synth.to_bits(x["q"]), synth.to_bits(kp), synth.to_bits(vp),
                                         table.cpu().numpy(), lens, synth.to_bits(x["o_weight"]), x["scale"])
    assert_bf16_close(f64(attn), ref_attn, f"{w.name} attention")
    assert_bf16_close(f64(out), ref_out, f"{w.name} output")
