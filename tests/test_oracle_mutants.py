"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant is a one-line textual edit of ``oracle/decode_oracle.c`` (a wrong
KV-head index, a dropped term, a flipped sign, a transposed operand, a wrong
merge weight ...). The copy is compiled into a temporary library and the whole
pin battery of ``_pins.py`` runs against it in a child process (so that a
mutant that crashes also counts as caught). The committed oracle is never
modified. This is the evidence that the pins constrain every step the oracle
takes, not only the ones a given pin was written for.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))

# (name, original text, replacement, occurrence index to replace or None for all)
MUTANTS = [
    ("kv_head_modulo_in_attention", "j = h / G;\n    const uint16_t* kb", "j = h % Hkv;\n    const uint16_t* kb", None),
    ("kv_head_modulo_in_scores", "j = h / G;\n    int64_t L = seq_lens[b];", "j = h % Hkv;\n    int64_t L = seq_lens[b];", None),
    ("scale_dropped", "z[t] = scale * z[t];", "z[t] = z[t];", None),
    ("no_normalisation", "z[t] = z[t] / zsum;", "z[t] = z[t];", None),
    ("exp_sign_flipped", "z[t] = exp(z[t] - zmax);", "z[t] = exp(zmax - z[t]);", None),
    ("sum_counts_terms", "zsum += z[t];", "zsum += 1.0;", None),
    ("last_d_dropped_in_scores", "for (int64_t d = 0; d < D; ++d) {\n        acc +=",
     "for (int64_t d = 0; d < D - 1; ++d) {\n        acc +=", None),
    ("last_token_dropped_in_pv", "for (int64_t t = 0; t < L; ++t) acc += z[t]", "for (int64_t t = 0; t + 1 < L; ++t) acc += z[t]", None),
    ("w_transposed", "yb[n] += xk * bf16_bits_to_double(wk[n]);", "yb[n] += xk * bf16_bits_to_double(w[n * Kdim + kk]);", None),
    ("x_index_transposed", "double xk = x[b * Kdim + kk];", "double xk = x[kk * B + b];", None),
    ("scores_stored_transposed", "s[g * L + t] = acc;", "s[t * G + g] = acc;", None),
    ("split_denominator_unweighted", "denom += exp(m_c[c] - big_m) * l_c[c];", "denom += l_c[c];", None),
    ("split_weight_sign", "num += exp(m_c[c] - big_m) * o_c[c * D + d];", "num += exp(big_m - m_c[c]) * o_c[c * D + d];", None),
    ("split_chunk_max_ignored", "m_c[c] = m;", "m_c[c] = 0.0;", None),
    ("bf16_widening_shift", "((uint32_t)bits) << 16", "((uint32_t)bits) << 15", None),
    ("k_batch_stride_wrong", "const uint16_t* kb = k + (b * Hkv + j) * Lcap * D;", "const uint16_t* kb = k + (b * Hkv + j) * D;", None),
    ("q_uses_kv_head", "if (oracle_group_attention(q + (b * Hq + h) * D", "if (oracle_group_attention(q + (b * Hq + j) * D", None),
    ("v_read_from_k", "const uint16_t* vb = v + (b * Hkv + j) * Lcap * D;", "const uint16_t* vb = k + (b * Hkv + j) * Lcap * D;", None),
    ("seq_len_ignored", "1, seq_lens[b], D, scale,", "1, Lcap, D, scale,", None),
    ("v_row_offset", "acc += z[t] * bf16_bits_to_double(v[t * v_row_stride + d]);",
     "acc += z[t] * bf16_bits_to_double(v[t * v_row_stride + (d + 1) % D]);", None),
    ("paged_block_index_modulo", "table[b * max_blocks + t / bs]", "table[b * max_blocks + t % max_blocks]", None),
    ("paged_row_index_divided", "const int64_t row = t % bs;", "const int64_t row = (t / bs) % bs;", None),
    ("paged_head_ignored", "pages + ((blk * Hkv + j) * bs + row) * D", "pages + ((blk * Hkv) * bs + row) * D", None),
    ("paged_table_stride", "table[b * max_blocks + t / bs]", "table[b + t / bs]", None),
    ("e4m3_bias_8", "ldexp(1.0 + (double)m / 8.0, (int)e - 7)", "ldexp(1.0 + (double)m / 8.0, (int)e - 8)", None),
    ("e4m3_subnormal_as_normal", "e == 0 ? ldexp((double)m, -9)", "e == 0 ? ldexp(1.0 + (double)m / 8.0, -7)", None),
    ("e4m3_mantissa_quarters", "(1.0 + (double)m / 8.0, (int)e - 7)", "(1.0 + (double)m / 4.0, (int)e - 7)", None),
    ("e4m3_sign_dropped", "(float)(s ? -mag : mag)", "(float)(mag)", None),
]


def _mutate(src: str, old: str, new: str) -> str:
    assert src.count(old) >= 1, f"mutation target not found: {old!r}"
    return src.replace(old, new)


@pytest.mark.parametrize("name,old,new,_occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, _occ):
    with open(oracle.SRC) as f:
        src = f.read()
    mut = tmp_path / f"{name}.c"
    mut.write_text(_mutate(src, old, new))
    lib = oracle.build(src=str(mut), out_dir=str(tmp_path), tag=name)
    proc = subprocess.run([sys.executable, os.path.join(HERE, "_pins.py"), "--lib", lib],
                          capture_output=True, text=True, timeout=300)
    if proc.returncode != 0:
        return  # the mutant crashed the pin run: caught
    res = json.loads(proc.stdout.strip().splitlines()[-1])
    failed = [k for k, v in res.items() if v != "ok"]
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(tmp_path):
    """Control: the same child-process route on the committed source passes every pin."""
    lib = oracle.build(out_dir=str(tmp_path), tag="control")
    proc = subprocess.run([sys.executable, os.path.join(HERE, "_pins.py"), "--lib", lib],
                          capture_output=True, text=True, timeout=300)
    assert proc.returncode == 0, proc.stderr
    res = json.loads(proc.stdout.strip().splitlines()[-1])
    assert all(v == "ok" for v in res.values()), res
