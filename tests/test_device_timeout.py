"""A bounded device wait that runs out, on purpose, with no bad address and nothing
left hanging: two test hooks of the options tell the fused step's grid barrier to
wait for one CTA more than the grid holds, with a 200 microsecond limit. Every CTA
then gives up after the limit, records the grid-barrier code (bit 32) in the error
word and completes the kernel (its result is not valid).

Checked: the call returns and the stream drains; decode_attn_last_device_error
reports the code and clears it (a second query reads 0); a repeat of the failing
call fails the same way; and the next normal call matches the fp64 oracle and the
two-launch path, which needs the error query to have reset the barrier's counters
(the CTAs that gave up left them short of the count at which the last CTA resets
them, and a stale count would let the next call pass its barrier early).
"""
import pytest
import torch

import decode_attention_output_gb300 as da
from decode_attention_output_gb300 import synth
from gpu_helpers import assert_bf16_close, f64, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ERR_GRID_SYNC = 32


@pytest.fixture(scope="module", autouse=True)
def _library():
    from decode_attention_output_gb300 import build

    build.build()
    da.load()
    torch.cuda.set_device(0)
    yield
    for k, v in {"fused": 0, "grid_wait_us": 0, "grid_wait_extra": 0}.items():
        da.decode_attn_set_option(k, v)


def _fwd(x, w):
    out = torch.full((w.B, w.N), float("nan"), dtype=torch.bfloat16, device=DEV)
    da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"])
    return out


@pytest.mark.parametrize("lens", [(300, 0, 129), (700,) * 4], ids=["ragged_b3", "b4"])
def test_grid_barrier_timeout_is_reported_and_the_next_call_is_clean(orc, lens):
    w = synth.Workload("timeout", B=len(lens), Hq=8, Hkv=2, Lcap=max(lens), N=256, fixed_lens=lens)
    x = synth.make_inputs(w, seed=29, device=DEV)
    assert da.decode_attn_last_device_error() == 0
    da.decode_attn_set_option("fused", 1)
    try:
        da.decode_attn_set_option("grid_wait_us", 200)
        da.decode_attn_set_option("grid_wait_extra", 1)
        for _ in range(2):  # the failure repeats the same way
            _fwd(x, w)
            torch.cuda.synchronize()  # the call ended: every CTA gave up and completed
            assert da.decode_attn_last_device_error() == ERR_GRID_SYNC
            assert da.decode_attn_last_device_error() == 0  # the query cleared it
        da.decode_attn_set_option("grid_wait_extra", 0)
        da.decode_attn_set_option("grid_wait_us", 0)
        out = _fwd(x, w)
        torch.cuda.synchronize()
        assert da.decode_attn_last_device_error() == 0
    finally:
        da.decode_attn_set_option("grid_wait_extra", 0)
        da.decode_attn_set_option("grid_wait_us", 0)
        da.decode_attn_set_option("fused", 0)
    out2 = _fwd(x, w)  # two launches, no grid barrier
    torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    _, ref_out = oracle_decode(orc, x)
    assert_bf16_close(f64(out), ref_out, "fused step after the timeout")
    assert_bf16_close(f64(out2), ref_out, "two-launch step")
