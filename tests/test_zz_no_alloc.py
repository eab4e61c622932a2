"""decode_attn_only_noalloc: the attention step for callers that must not allocate
GPU memory at run time (a process whose device memory is reserved up front by its
own pool, or a request path that may not take the device-wide synchronisation of
growing a workspace). The entry point keeps its scratch in a fixed array inside
the library, so these tests check that it returns exactly what decode_attn_only
returns (the same plan and kernel, so bit for bit), on two calls in a row (the
array keeps the previous call's contents, so the second call checks that the
per-call clearing works), that the first call also matches the fp64 oracle
within the bf16 tolerances, and that a call needing more scratch than the array
holds is refused without a launch.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test. It also passes on its own in a fresh
process.
"""
import pytest
import torch

import decode_attention_output_gb300 as da
from decode_attention_output_gb300 import synth
from gpu_helpers import assert_bf16_close, f64, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DA_ERR_SCRATCH = -11


@pytest.fixture(scope="module", autouse=True)
def _library():
    from decode_attention_output_gb300 import build

    build.build()
    da.load()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (32, 2)], ids=["G4", "G16"])
def test_noalloc_matches_decode_attn_only_twice(orc, Hq, Hkv):
    for call, seed in enumerate((21, 22)):  # two calls in a row, different inputs
        w = synth.Workload("noalloc", B=5, Hq=Hq, Hkv=Hkv, Lcap=700, N=256, fixed_lens=(700, 1, 333, 0, 129))
        x = synth.make_inputs(w, seed=seed, device=DEV)
        ref = torch.empty((w.B, w.Hq, 128), dtype=torch.bfloat16, device=DEV)
        da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], ref, x["scale"])
        got = torch.full_like(ref, float("nan"))
        da.decode_attn_only_noalloc(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], got, x["scale"])
        torch.cuda.synchronize()
        assert da.decode_attn_last_device_error() == 0
        # the same plan and kernel as decode_attn_only: bit for bit the same result
        assert torch.equal(got, ref), f"no-alloc call {call + 1}, G={w.G}: differs from decode_attn_only"
        if call == 0:  # and an absolute anchor: the fp64 oracle
            ref_attn, _ = oracle_decode(orc, x)
            assert_bf16_close(f64(got), ref_attn, f"no-alloc call {call + 1}, G={w.G} vs oracle")


def test_noalloc_refuses_calls_beyond_its_scratch():
    B, Hkv, G = 1024, 8, 8  # 8192 (sequence, KV head) pairs: far more partial slots than 8 MiB holds
    q = torch.zeros((B, Hkv * G, 128), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((B, Hkv, 1, 128), dtype=torch.bfloat16, device=DEV)
    lens = torch.ones((B,), dtype=torch.int32, device=DEV)
    out = torch.zeros((B, Hkv * G, 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(da.DecodeAttnError) as ei:
        da.decode_attn_only_noalloc(q, k, k, lens, out, 0.1)
    assert ei.value.code == DA_ERR_SCRATCH
    torch.cuda.synchronize()
    assert torch.all(out == 0)
