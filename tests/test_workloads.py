"""The synthetic decode workloads at full size, run exactly as bench.py runs
them (default plan, one decode_attn_fwd call), compared with the oracle on the
whole output: every batch row, every attention head and every output column,
with the same tolerances as the small cases. For the ragged workload the
longest and the shortest sequences' attention rows are also checked on their
own, so that their errors are not averaged away by the others. Properties that
hold at any size are checked too (finite outputs; the two-launch step agrees
with projecting the attention-only result).
"""
import numpy as np
import pytest
import torch

import decode_attention_output_gb300 as da
from decode_attention_output_gb300 import synth
from gpu_helpers import assert_bf16_close, f64, oracle_decode, run_fwd, run_only

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from decode_attention_output_gb300 import build

    build.build()
    da.load()
    torch.cuda.set_device(0)
    yield
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", synth.ORDER)
def test_workload_full_output(orc, name):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w, seed=0, device=DEV)
    out = torch.full((w.B, w.N), float("nan"), dtype=torch.bfloat16, device=DEV)
    run_fwd(x, out)
    attn = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    run_only(x, attn)
    torch.cuda.synchronize()
    assert da.decode_attn_last_device_error() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(attn.float()).all()
    # the whole step agrees with projecting the attention-only result (split-K orders
    # may differ, so within the bf16 tolerance rather than bit for bit)
    out2 = torch.empty_like(out)
    da.decode_attn_oproj(attn.view(w.B, w.Hq * w.D), x["o_weight"], out2)
    torch.cuda.synchronize()
    assert_bf16_close(f64(out), f64(out2), f"{name} one step vs attention then projection")

    ref_attn, ref_out = oracle_decode(orc, x)  # every batch row
    assert_bf16_close(f64(attn), ref_attn, f"{name} attention, all {w.B} rows")
    assert_bf16_close(f64(out), ref_out, f"{name} output, all {w.B} rows")
    lens = x["seq_lens"].cpu().numpy()
    if w.lens == "ragged":
        for b in (int(np.argmax(lens)), int(np.argmin(lens))):
            assert_bf16_close(f64(attn[b]), ref_attn[b], f"{name} attention row {b} (length {lens[b]})")
    del x, out, attn, out2
    torch.cuda.empty_cache()
