"""Shared helpers of the GPU parity tests: tolerances, error measures, oracle calls."""
from __future__ import annotations

import numpy as np
import torch

from decode_attention_output_gb300 import synth

# bf16 outputs: max |gpu - oracle| <= 2e-2 and ||gpu - oracle|| / ||oracle|| <= 5e-3 (whole tensor)
ATOL_BF16 = 2e-2
RRMS_BF16 = 5e-3
# fp32 scores: per (b, h) row ||gpu - oracle|| / ||oracle|| <= 1e-4
RTOL_SCORES = 1e-4


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    max_abs = float(np.max(np.abs(got - ref))) if got.size else 0.0
    den = float(np.sqrt(np.sum(ref * ref)))
    rrms = float(np.sqrt(np.sum((got - ref) ** 2)) / den) if den > 0 else max_abs
    return max_abs, rrms


def assert_bf16_close(got, ref, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    max_abs, rrms = errors(got, ref)
    assert max_abs <= ATOL_BF16 and rrms <= RRMS_BF16, f"{what}: max abs {max_abs:.3e}, rel rms {rrms:.3e}"
    return max_abs, rrms


def oracle_decode(orc, x: dict, rows=None):
    """Runs the oracle on host copies of the inputs (optionally a subset of batch rows)."""
    q, k, v, lens = x["q"], x["k_cache"], x["v_cache"], x["seq_lens"]
    if rows is not None:
        idx = torch.tensor(rows, device=q.device)
        q, k, v, lens = q[idx], k[idx], v[idx], lens[idx]
    lcap = k.shape[2]
    lens_h = lens.cpu().numpy().astype(np.int64).clip(0, lcap).astype(np.int32)
    if "k_scale" in x:  # fp8 (e4m3) cache
        return orc.decode_fp8(synth.to_bits(q), synth.to_bits(k), synth.to_bits(v), lens_h,
                              synth.to_bits(x["o_weight"]), x["scale"], x["k_scale"], x["v_scale"])
    return orc.decode(synth.to_bits(q), synth.to_bits(k), synth.to_bits(v), lens_h, synth.to_bits(x["o_weight"]),
                      x["scale"])


def run_fwd(x, out, stream=None):
    """decode_attn_fwd, or decode_attn_fwd_fp8 for an e4m3 cache."""
    import decode_attention_output_gb300 as da

    if "k_scale" in x:
        return da.decode_attn_fwd_fp8(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out,
                                      x["scale"], x["k_scale"], x["v_scale"], stream=stream)
    return da.decode_attn_fwd(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], x["o_weight"], out, x["scale"],
                              stream=stream)


def run_only(x, attn, stream=None):
    """decode_attn_only, or decode_attn_only_fp8 for an e4m3 cache."""
    import decode_attention_output_gb300 as da

    if "k_scale" in x:
        return da.decode_attn_only_fp8(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"],
                                       x["k_scale"], x["v_scale"], stream=stream)
    return da.decode_attn_only(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], attn, x["scale"], stream=stream)
