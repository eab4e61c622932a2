"""The library's workspace on the GPU: it is grown in stream order (cudaFreeAsync of the old
block, cudaMallocAsync of the new one, its header zeroed by cudaMemsetAsync, all on the
call's stream) when a call needs more scratch than it holds, and released by
decode_attn_release. The calls before and after a growth, on a side stream, and after a
release all match the fp64 oracle.
"""
import pytest
import torch

import decode_attention_output_gb300 as da
from decode_attention_output_gb300 import synth
from gpu_helpers import assert_bf16_close, f64, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from decode_attention_output_gb300 import build

    build.build()
    da.load()
    torch.cuda.set_device(0)


def _attention(x, w, stream):
    attn = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    with torch.cuda.stream(stream):
        da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"], stream=stream)
    return attn


def test_growth_on_a_side_stream_and_release(orc):
    small = synth.Workload("ws_small", B=3, Hq=8, Hkv=2, Lcap=300, N=256, fixed_lens=(300, 0, 129))
    # 1024 x 16 sequences: about 68 MB of split-KV partials, more than the first allocation
    big = synth.Workload("ws_big", B=1024, Hq=16, Hkv=16, Lcap=8, N=128,
                         fixed_lens=tuple((i * 7) % 9 for i in range(1024)))
    xs = synth.make_inputs(small, seed=51, device=DEV)
    xb = synth.make_inputs(big, seed=52, device=DEV)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream())
    a1 = _attention(xs, small, side)   # first allocation (or the existing workspace)
    a2 = _attention(xb, big, side)     # grows the workspace on `side`
    a3 = _attention(xs, small, side)   # after the growth
    side.synchronize()
    assert da.decode_attn_last_device_error(side) == 0
    ref_s, _ = oracle_decode(orc, xs)
    ref_b, _ = oracle_decode(orc, xb)
    assert_bf16_close(f64(a1), ref_s, "before the growth")
    assert_bf16_close(f64(a2), ref_b, "the call that grew the workspace")
    assert torch.equal(a1, a3), "the same call after the growth"
    da.decode_attn_release()
    a4 = _attention(xs, small, torch.cuda.current_stream())  # allocates again
    torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    assert torch.equal(a1, a4), "the same call after decode_attn_release"
