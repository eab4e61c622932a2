"""Pins for the fp64 oracle: checks against facts that do not come from the oracle.

Each ``pin_*`` function takes an :class:`oracle.Oracle` and raises
``AssertionError`` when the oracle disagrees with what the pages or the
mathematics fix: closed forms, invariants, special cases that reduce to a
library routine (integer matmul in numpy), a brute-force evaluation in
60-digit decimal arithmetic on tiny inputs, and the shape table printed on the
page "PyPTO 开箱性能调优实战 Decode Attention 多 Matmul 独立 TileShape 配置
F-16" (section "三个 Matmul 的 Shape 特征分析").

The same battery runs against deliberately broken copies of the oracle
(``test_oracle_mutants.py``), each of which must fail at least one pin.
Run as a script (``python tests/_pins.py --lib path.so``) it prints a JSON
map pin -> "ok" | error text, which is how the mutant test calls it.
"""
from __future__ import annotations

import decimal
import json
import math
import os
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

D = 128


# ---------------------------------------------------------------------------
# input helpers (bf16 bit patterns; no arithmetic of the method)
# ---------------------------------------------------------------------------
def to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even) and return the bits."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bits_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_bits(rng, shape, std=1.0) -> np.ndarray:
    return to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def int_bits(rng, shape, lo, hi) -> np.ndarray:
    """Integer-valued bf16 tensors (exact for |x| <= 256)."""
    return to_bf16_bits(rng.integers(lo, hi + 1, size=shape).astype(np.float32))


def _close(a, b, tol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max |diff| {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------------------
# brute force in 60-digit decimal arithmetic (independent of the C oracle)
# ---------------------------------------------------------------------------
_CTX = decimal.Context(prec=60)


def _dec(x: float) -> decimal.Decimal:
    return _CTX.create_decimal_from_float(float(x))


def brute_decode(q, k, v, seq_lens, w, scale):
    """Whole step in Decimal: q [B,Hq,D], k/v [B,Hkv,Lcap,D], w [Hq*D,N] (float64 values)."""
    B, Hq, Dd = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    N = w.shape[1]
    sc = _dec(scale)
    attn = [[[decimal.Decimal(0)] * Dd for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        L = int(seq_lens[b])
        for h in range(Hq):
            j = h // G
            if L == 0:
                continue
            z = []
            for t in range(L):
                s = sum((_dec(q[b, h, d]) * _dec(k[b, j, t, d]) for d in range(Dd)), decimal.Decimal(0))
                z.append(_CTX.multiply(sc, s))
            m = max(z)
            e = [_CTX.exp(_CTX.subtract(zt, m)) for zt in z]
            tot = sum(e, decimal.Decimal(0))
            p = [_CTX.divide(et, tot) for et in e]
            for d in range(Dd):
                attn[b][h][d] = sum((_CTX.multiply(p[t], _dec(v[b, j, t, d])) for t in range(L)),
                                    decimal.Decimal(0))
    y = [[decimal.Decimal(0)] * N for _ in range(B)]
    for b in range(B):
        flat = [attn[b][h][d] for h in range(Hq) for d in range(Dd)]
        for n in range(N):
            y[b][n] = sum((_CTX.multiply(flat[kk], _dec(w[kk, n])) for kk in range(Hq * Dd)), decimal.Decimal(0))
    a = np.array([[[float(x) for x in row] for row in hb] for hb in attn], np.float64)
    yy = np.array([[float(x) for x in row] for row in y], np.float64)
    return a, yy


# ---------------------------------------------------------------------------
# the pins
# ---------------------------------------------------------------------------
def pin_bruteforce_whole_step(orc):
    """Tiny batch, ragged lengths, G = 2, non-square o_proj: oracle == 60-digit brute force."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, Lcap, N = 2, 4, 2, 6, 24
    q = rand_bits(rng, (B, Hq, D))
    k = rand_bits(rng, (B, Hkv, Lcap, D))
    v = rand_bits(rng, (B, Hkv, Lcap, D))
    w = rand_bits(rng, (Hq * D, N), std=1 / math.sqrt(Hq * D))
    lens = np.array([5, 2], np.int32)
    scale = 1 / math.sqrt(D)
    attn, y = orc.decode(q, k, v, lens, w, scale)
    ba, by = brute_decode(bits_to_f64(q), bits_to_f64(k), bits_to_f64(v), lens, bits_to_f64(w), scale)
    _close(attn, ba, 1e-13, "attention vs brute force")
    _close(y, by, 1e-13, "output vs brute force")


def pin_bruteforce_whole_step_d256(orc):
    """Head dim 256 (the page's other GQA decode): oracle == 60-digit brute force."""
    rng = np.random.default_rng(31)
    D2 = 256
    B, Hq, Hkv, Lcap, N = 1, 2, 1, 3, 8
    q = rand_bits(rng, (B, Hq, D2))
    k = rand_bits(rng, (B, Hkv, Lcap, D2))
    v = rand_bits(rng, (B, Hkv, Lcap, D2))
    w = rand_bits(rng, (Hq * D2, N), std=1 / math.sqrt(Hq * D2))
    lens = np.array([3], np.int32)
    scale = 1 / math.sqrt(D2)
    attn, y = orc.decode(q, k, v, lens, w, scale)
    ba, by = brute_decode(bits_to_f64(q), bits_to_f64(k), bits_to_f64(v), lens, bits_to_f64(w), scale)
    _close(attn, ba, 1e-13, "attention (D=256) vs brute force")
    _close(y, by, 1e-13, "output (D=256) vs brute force")


def pin_integer_scores_exact_d256(orc):
    """Integer q, k at head dim 256: scores equal the int64 matmul over all 256 dims
    (a contraction that stopped at 128 would differ)."""
    rng = np.random.default_rng(32)
    B, Hq, Hkv, Lcap = 1, 4, 2, 5
    G = Hq // Hkv
    qi = rng.integers(-4, 5, size=(B, Hq, 256))
    ki = rng.integers(-4, 5, size=(B, Hkv, Lcap, 256))
    lens = np.array([5], np.int32)
    s = orc.scores(to_bf16_bits(qi.astype(np.float32)), to_bf16_bits(ki.astype(np.float32)), lens)
    for h in range(Hq):
        ref = ki[0, h // G] @ qi[0, h]
        assert np.array_equal(s[0, h], ref.astype(np.float64)), f"scores (D=256) h={h}"
        assert not np.array_equal(ref, ki[0, h // G, :, :128] @ qi[0, h, :128]), "test needs both halves"


def pin_bruteforce_group(orc):
    """One group of G = 3 heads over 7 keys, unusual scale: group_attention == brute force."""
    rng = np.random.default_rng(12)
    G, L = 3, 7
    q = rand_bits(rng, (G, D))
    k = rand_bits(rng, (L, D))
    v = rand_bits(rng, (L, D))
    scale = 0.3
    got = orc.group_attention(q, k, v, scale)
    ba, _ = brute_decode(bits_to_f64(q)[None], bits_to_f64(k)[None, None], bits_to_f64(v)[None, None],
                         np.array([L]), np.zeros((G * D, 1)), scale)
    _close(got, ba[0], 1e-13, "group attention vs brute force")


def pin_integer_scores_exact(orc):
    """Integer-valued q, k: unscaled scores equal the int64 matmul, with KV head h // G."""
    rng = np.random.default_rng(13)
    B, Hq, Hkv, Lcap = 2, 6, 2, 9
    G = Hq // Hkv
    qi = rng.integers(-4, 5, size=(B, Hq, D))
    ki = rng.integers(-4, 5, size=(B, Hkv, Lcap, D))
    lens = np.array([9, 4], np.int32)
    s = orc.scores(to_bf16_bits(qi.astype(np.float32)), to_bf16_bits(ki.astype(np.float32)), lens)
    for b in range(B):
        for h in range(Hq):
            ref = ki[b, h // G] @ qi[b, h]  # int64
            L = lens[b]
            assert np.array_equal(s[b, h, :L], ref[:L].astype(np.float64)), f"scores b={b} h={h}"
            assert np.all(np.isnan(s[b, h, L:])), "entries past seq_len must be untouched"


def pin_group_scores_layout(orc):
    """group_scores returns [G, L] with s[g, t] = q[g] . k[t] (integer case, np.matmul)."""
    rng = np.random.default_rng(14)
    G, L = 3, 5
    qi = rng.integers(-3, 4, size=(G, D))
    ki = rng.integers(-3, 4, size=(L, D))
    s = orc.group_scores(to_bf16_bits(qi.astype(np.float32)), to_bf16_bits(ki.astype(np.float32)))
    assert np.array_equal(s, (qi @ ki.T).astype(np.float64)), "group scores layout"


def pin_oproj_integer_exact(orc):
    """Integer attention and W in {-1,0,1}, K != N: y equals the int64 matmul exactly."""
    rng = np.random.default_rng(15)
    B, K, N = 3, 256, 40
    xi = rng.integers(-8, 9, size=(B, K))
    wi = rng.integers(-1, 2, size=(K, N))
    y = orc.oproj(xi.astype(np.float64), to_bf16_bits(wi.astype(np.float32)))
    assert np.array_equal(y, (xi @ wi).astype(np.float64)), "o_proj integer case"


def pin_oproj_all_ones(orc):
    """All-ones operands give y = K everywhere (the golden check of the basic_matmul
    example on the CANN page "自动调优流程": all-ones operands compared with np.matmul)."""
    B, K, N = 2, 384, 16
    y = orc.oproj(np.ones((B, K)), to_bf16_bits(np.ones((K, N), np.float32)))
    assert np.array_equal(y, np.full((B, N), float(K))), "all-ones o_proj"


def pin_single_token(orc):
    """L = 1: the softmax of one score is 1, so the output row is V[0] exactly."""
    rng = np.random.default_rng(16)
    q, k, v = rand_bits(rng, (4, D)), rand_bits(rng, (1, D)), rand_bits(rng, (1, D))
    out = orc.group_attention(q, k, v, 1 / math.sqrt(D))
    assert np.array_equal(out, np.broadcast_to(bits_to_f64(v[0]), (4, D))), "single token"


def pin_rows_sum_to_one(orc):
    """V = 1 everywhere: every output is sum_t p_t = 1 (softmax rows sum to 1)."""
    rng = np.random.default_rng(17)
    q, k = rand_bits(rng, (4, D), std=3.0), rand_bits(rng, (37, D), std=3.0)
    v = to_bf16_bits(np.ones((37, D), np.float32))
    out = orc.group_attention(q, k, v, 1 / math.sqrt(D))
    _close(out, np.ones((4, D)), 4e-16 * 37, "rows sum to one")


def pin_constant_rows(orc):
    """Every V row equal to u: output = u (convex combination of equal rows)."""
    rng = np.random.default_rng(18)
    q, k = rand_bits(rng, (3, D)), rand_bits(rng, (20, D))
    u = rand_bits(rng, (1, D))
    v = np.repeat(u, 20, axis=0)
    out = orc.group_attention(q, k, v, 1 / math.sqrt(D))
    _close(out, np.broadcast_to(bits_to_f64(u[0]), (3, D)), 1e-14, "constant V rows")


def pin_identical_keys_mean(orc):
    """All keys equal: p = 1/L, so the output is the mean of the V rows."""
    rng = np.random.default_rng(19)
    L = 23
    q = rand_bits(rng, (4, D))
    k = np.repeat(rand_bits(rng, (1, D)), L, axis=0)
    v = rand_bits(rng, (L, D))
    out = orc.group_attention(q, k, v, 1 / math.sqrt(D))
    _close(out, np.broadcast_to(bits_to_f64(v).mean(axis=0), (4, D)), 1e-14, "identical keys")


def pin_zero_scale_mean(orc):
    """scale = 0: uniform weights whatever the keys, output = mean of V rows."""
    rng = np.random.default_rng(20)
    L = 11
    q, k, v = rand_bits(rng, (2, D)), rand_bits(rng, (L, D), std=5.0), rand_bits(rng, (L, D))
    out = orc.group_attention(q, k, v, 0.0)
    _close(out, np.broadcast_to(bits_to_f64(v).mean(axis=0), (2, D)), 1e-14, "zero scale")


def pin_dominant_key(orc):
    """One scaled score above the others by > 40: the output copies that V row
    to within exp(-40) * L."""
    rng = np.random.default_rng(21)
    L, tstar = 30, 17
    qf = np.zeros((1, D), np.float32)
    qf[0, 0] = 8.0
    kf = rng.integers(-2, 3, size=(L, D)).astype(np.float32)
    kf[tstar, 0] = 64.0  # score 512 -> scaled 45.25; others |score| <= 16 -> <= 1.42
    v = rand_bits(rng, (L, D))
    out = orc.group_attention(to_bf16_bits(qf), to_bf16_bits(kf), v, 1 / math.sqrt(D))
    _close(out[0], bits_to_f64(v[tstar]), 4 * L * math.exp(-40), "dominant key")


def pin_two_tokens_closed_form(orc):
    """L = 2: out = V0 + sigmoid(z1 - z0) (V1 - V0), z = scale * q.k (numpy dot)."""
    rng = np.random.default_rng(22)
    q, k, v = rand_bits(rng, (3, D)), rand_bits(rng, (2, D)), rand_bits(rng, (2, D))
    scale = 1 / math.sqrt(D)
    qf, kf, vf = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    z = scale * (qf @ kf.T)
    sig = 1.0 / (1.0 + np.exp(-(z[:, 1] - z[:, 0])))
    ref = vf[0][None, :] + sig[:, None] * (vf[1] - vf[0])[None, :]
    out = orc.group_attention(q, k, v, scale)
    _close(out, ref, 1e-14, "two-token closed form")


def pin_head_mapping(orc):
    """Query head h reads KV head h // G: V of KV head j filled with j + 1."""
    rng = np.random.default_rng(23)
    B, Hq, Hkv, Lcap = 2, 6, 3, 5
    q = rand_bits(rng, (B, Hq, D))
    k = rand_bits(rng, (B, Hkv, Lcap, D))
    vf = np.zeros((B, Hkv, Lcap, D), np.float32)
    for j in range(Hkv):
        vf[:, j] = j + 1
    lens = np.array([5, 3], np.int32)
    attn = orc.attention(q, k, to_bf16_bits(vf), lens, 1 / math.sqrt(D))
    G = Hq // Hkv
    for h in range(Hq):
        _close(attn[:, h, :], np.full((B, D), float(h // G + 1)), 1e-15 * 8, f"head {h} -> kv head")


def pin_batch_indexing(orc):
    """Batch b reads its own cache rows: V of batch b filled with 10 b + 1."""
    rng = np.random.default_rng(24)
    B, Hq, Hkv, Lcap = 3, 4, 2, 4
    vf = np.zeros((B, Hkv, Lcap, D), np.float32)
    for b in range(B):
        vf[b] = 10 * b + 1
    attn = orc.attention(rand_bits(rng, (B, Hq, D)), rand_bits(rng, (B, Hkv, Lcap, D)), to_bf16_bits(vf),
                         np.array([4, 1, 3], np.int32), 1 / math.sqrt(D))
    for b in range(B):
        _close(attn[b], np.full((Hq, D), 10.0 * b + 1), 1e-13, f"batch {b}")


def pin_permutation_invariance(orc):
    """Reordering the (key, value) pairs leaves the output unchanged."""
    rng = np.random.default_rng(25)
    L = 19
    q, k, v = rand_bits(rng, (4, D)), rand_bits(rng, (L, D)), rand_bits(rng, (L, D))
    perm = rng.permutation(L)
    a = orc.group_attention(q, k, v, 1 / math.sqrt(D))
    b = orc.group_attention(q, k[perm], v[perm], 1 / math.sqrt(D))
    _close(a, b, 1e-14, "permutation invariance")


def pin_shift_invariance(orc):
    """Adding one vector u to every key adds q.u to every score of a head;
    the softmax does not change (integer data keeps the bf16 values exact)."""
    rng = np.random.default_rng(26)
    L = 13
    qi = rng.integers(-2, 3, size=(3, D)).astype(np.float32)
    ki = rng.integers(-3, 4, size=(L, D)).astype(np.float32)
    u = rng.integers(-3, 4, size=(1, D)).astype(np.float32)
    v = rand_bits(rng, (L, D))
    a = orc.group_attention(to_bf16_bits(qi), to_bf16_bits(ki), v, 0.05)
    b = orc.group_attention(to_bf16_bits(qi), to_bf16_bits(ki + u), v, 0.05)
    _close(a, b, 1e-13, "shift invariance")


def pin_linearity_in_v(orc):
    """The output is linear in V: o(2V) = 2 o(V) and o(V + W) = o(V) + o(W)."""
    rng = np.random.default_rng(27)
    L = 9
    q, k = rand_bits(rng, (2, D)), rand_bits(rng, (L, D))
    vi = rng.integers(-5, 6, size=(L, D)).astype(np.float32)
    wi = rng.integers(-5, 6, size=(L, D)).astype(np.float32)
    s = 1 / math.sqrt(D)
    ov = orc.group_attention(q, k, to_bf16_bits(vi), s)
    ow = orc.group_attention(q, k, to_bf16_bits(wi), s)
    _close(orc.group_attention(q, k, to_bf16_bits(2 * vi), s), 2 * ov, 1e-13, "o(2V)")
    _close(orc.group_attention(q, k, to_bf16_bits(vi + wi), s), ov + ow, 1e-13, "o(V+W)")


def pin_split_equals_unsplit(orc):
    """Split-KV with a log-sum-exp merge equals the unsplit softmax, for any chunk."""
    rng = np.random.default_rng(28)
    L = 130
    q, k, v = rand_bits(rng, (4, D), std=2.0), rand_bits(rng, (L, D), std=2.0), rand_bits(rng, (L, D))
    s = 1 / math.sqrt(D)
    ref = orc.group_attention(q, k, v, s)
    for chunk in (1, 3, 64, 129, 130, 1000):
        _close(orc.group_attention_split(q, k, v, s, chunk), ref, 1e-14, f"split chunk={chunk}")


def pin_split_matches_brute(orc):
    """The split form also matches the brute force directly (not only the unsplit oracle)."""
    rng = np.random.default_rng(29)
    L = 6
    q, k, v = rand_bits(rng, (2, D)), rand_bits(rng, (L, D)), rand_bits(rng, (L, D))
    ba, _ = brute_decode(bits_to_f64(q)[None], bits_to_f64(k)[None, None], bits_to_f64(v)[None, None],
                         np.array([L]), np.zeros((2 * D, 1)), 0.2)
    _close(orc.group_attention_split(q, k, v, 0.2, 4), ba[0], 1e-13, "split vs brute force")


def pin_seq_len_masks_tail(orc):
    """Cache rows at t >= seq_len do not matter: huge values there change nothing."""
    rng = np.random.default_rng(30)
    B, Hq, Hkv, Lcap = 2, 4, 2, 12
    q = rand_bits(rng, (B, Hq, D))
    k = rand_bits(rng, (B, Hkv, Lcap, D))
    v = rand_bits(rng, (B, Hkv, Lcap, D))
    lens = np.array([7, 12], np.int32)
    a = orc.attention(q, k, v, lens, 1 / math.sqrt(D))
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 7:] = to_bf16_bits(np.full((Hkv, 5, D), 3.0e4, np.float32))
    v2[0, :, 7:] = to_bf16_bits(np.full((Hkv, 5, D), -7.0e4, np.float32))
    b = orc.attention(q, k2, v2, lens, 1 / math.sqrt(D))
    assert np.array_equal(a, b), "rows past seq_len changed the output"


def pin_zero_length(orc):
    """seq_len = 0 attends to nothing: the attention row is 0 (and so is its projection)."""
    rng = np.random.default_rng(31)
    B, Hq, Hkv, Lcap, N = 2, 4, 2, 5, 8
    q = rand_bits(rng, (B, Hq, D))
    k = rand_bits(rng, (B, Hkv, Lcap, D))
    v = rand_bits(rng, (B, Hkv, Lcap, D))
    w = rand_bits(rng, (Hq * D, N))
    attn, y = orc.decode(q, k, v, np.array([0, 5], np.int32), w, 1 / math.sqrt(D))
    assert np.array_equal(attn[0], np.zeros((Hq, D))) and np.array_equal(y[0], np.zeros(N)), "empty sequence"
    assert np.any(attn[1] != 0), "non-empty sequence must not be zero"


def pin_page1_shape_table(orc):
    """The page's shape table (golden file) matches the oracle's contractions on the
    configuration it describes: GQA group 4, head_dim 128, kv_len 2048, batch 1, hidden 4096."""
    shapes = {}
    with open(os.path.join(_HERE, "golden", "page1_matmul_shapes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, m, kk, n = line.split()
                shapes[name] = (int(m), int(kk), int(n))
    Hq, Hkv, L, B, hidden = 32, 8, 2048, 1, 4096
    G = Hq // Hkv
    q = np.zeros((G, D), np.uint16)
    kc = np.zeros((L, D), np.uint16)
    s = orc.group_scores(q, kc)  # M x N = G x L, reduced over K = D
    assert (s.shape[0], q.shape[1], s.shape[1]) == shapes["qk_t"], "QK^T shape"
    o = orc.group_attention(q, kc, kc, 1.0)  # M x N = G x D, reduced over K = L
    assert (o.shape[0], kc.shape[0], o.shape[1]) == shapes["attn_v"], "attn.V shape"
    x = np.zeros((B, Hq * D))
    y = orc.oproj(x, np.zeros((Hq * D, hidden), np.uint16))
    assert (y.shape[0], x.shape[1], y.shape[1]) == shapes["output_proj"], "output_proj shape"


def pin_bf16_widening(orc):
    """Powers of two and sign survive the bf16 -> double widening (o_proj with W = 1 x 1)."""
    vals = np.array([1.0, -2.0, 0.5, 3.0e38, -1.0e-38, 0.0, 1.5, 65504.0], np.float32)
    bits = to_bf16_bits(vals)
    y = orc.oproj(np.ones((1, 1)), bits[None, :])
    assert np.array_equal(y[0], bits_to_f64(bits)), "bf16 widening"


def _scatter_to_pages(rng, cache, bs, spare):
    """Cuts a contiguous cache [B, Hkv, Lcap, D] into blocks of bs tokens, stores them in
    a pool at random places (with `spare` extra blocks of noise) and returns (pool, table).
    Block-granular slicing, the inverse of the oracle's per-token gather."""
    B, Hkv, Lcap, D = cache.shape
    mb = Lcap // bs
    nblk = B * mb + spare
    pool = rng.integers(0, 1 << 16, size=(nblk, Hkv, bs, D)).astype(np.uint16)
    perm = rng.permutation(nblk)[: B * mb].reshape(B, mb)
    for b in range(B):
        for i in range(mb):
            pool[perm[b, i]] = cache[b, :, i * bs:(i + 1) * bs, :]
    return pool, perm.astype(np.int32)


def pin_gather_pages_roundtrip(orc):
    """Scattering a cache into shuffled blocks and gathering it back through the table
    returns the cache exactly (rows t < seq_len), and zeros past seq_len."""
    rng = np.random.default_rng(41)
    for bs, D in ((16, 128), (8, 256), (64, 128)):
        B, Hkv, mb = 3, 2, 4
        cache = rng.integers(0, 1 << 16, size=(B, Hkv, mb * bs, D)).astype(np.uint16)
        pool, table = _scatter_to_pages(rng, cache, bs, spare=5)
        lens = np.array([mb * bs, 1, bs + 3], np.int32)
        got = orc.gather_pages(pool, table, lens)
        for b in range(B):
            L = lens[b]
            assert np.array_equal(got[b, :, :L], cache[b, :, :L]), f"gather bs={bs} b={b}"
            assert np.all(got[b, :, L:] == 0), "rows past seq_len are zero"


def pin_gather_pages_reads_only_used_entries(orc):
    """Table entries past ceil(L / bs) are never used, and an entry outside the pool
    gives zero rows for its tokens only."""
    rng = np.random.default_rng(42)
    bs, D, B, Hkv, mb = 16, 128, 2, 1, 3
    cache = rng.integers(0, 1 << 16, size=(B, Hkv, mb * bs, D)).astype(np.uint16)
    pool, table = _scatter_to_pages(rng, cache, bs, spare=0)
    lens = np.array([20, 48], np.int32)
    table[0, 2] = 1 << 30  # past ceil(20 / 16) = 2 entries: unused
    table[1, 1] = -7       # outside the pool: tokens 16..31 of row 1 read as zero
    got = orc.gather_pages(pool, table, lens)
    assert np.array_equal(got[0, :, :20], cache[0, :, :20])
    assert np.array_equal(got[1, :, :16], cache[1, :, :16]) and np.all(got[1, :, 16:32] == 0)
    assert np.array_equal(got[1, :, 32:48], cache[1, :, 32:48])


def pin_paged_decode_equals_contiguous(orc):
    """The whole step over a paged cache equals the step over the cache it describes."""
    rng = np.random.default_rng(43)
    B, Hq, Hkv, bs, mb, N = 2, 4, 2, 16, 3, 16
    q = rand_bits(rng, (B, Hq, D))
    k = rand_bits(rng, (B, Hkv, mb * bs, D))
    v = rand_bits(rng, (B, Hkv, mb * bs, D))
    w = rand_bits(rng, (Hq * D, N), std=1 / math.sqrt(Hq * D))
    lens = np.array([48, 17], np.int32)
    kp, table = _scatter_to_pages(np.random.default_rng(44), k, bs, spare=2)
    vp, table_v = _scatter_to_pages(np.random.default_rng(44), v, bs, spare=2)
    assert np.array_equal(table, table_v)
    a1, y1 = orc.decode_paged(q, kp, vp, table, lens, w, 1 / math.sqrt(D))
    a0, y0 = orc.decode(q, k, v, lens, w, 1 / math.sqrt(D))
    assert np.array_equal(a1, a0) and np.array_equal(y1, y0)


def pin_e4m3_known_values(orc):
    """e4m3 codes whose values the format's definition fixes by hand (bias 7, 3 mantissa
    bits, subnormals m * 2^-9, S.1111.111 = NaN)."""
    table = {0x00: 0.0, 0x80: -0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5,
             0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x48: 4.0, 0x58: 16.0, 0x7E: 448.0,
             0xB8: -1.0, 0xFE: -448.0, 0x77: 240.0, 0x70: 128.0}
    codes = np.array(sorted(table), np.uint8)
    got = bits_to_f64(orc.e4m3_to_bf16_bits(codes))
    for c, g in zip(codes, got):
        want = table[int(c)]
        assert g == want and math.copysign(1, g) == math.copysign(1, want), f"code {c:#04x}: {g} != {want}"
    nan = bits_to_f64(orc.e4m3_to_bf16_bits(np.array([0x7F, 0xFF], np.uint8)))
    assert np.all(np.isnan(nan)), "S.1111.111 is NaN"


def pin_e4m3_all_codes_match_library(orc):
    """All 256 codes widen to the values torch's float8_e4m3fn conversion gives."""
    import torch

    codes = np.arange(256, dtype=np.uint8)
    got = bits_to_f64(orc.e4m3_to_bf16_bits(codes))
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "NaN codes"
    assert np.array_equal(got[~nan], ref[~nan]), "e4m3 values"


def pin_fp8_decode_bruteforce(orc):
    """The fp8-cache step (scales folded into the softmax scale and the outputs) equals a
    60-digit brute force on the dequantized keys and values, k_codes * k_scale and
    v_codes * v_scale, computed here from the e4m3 definition independently."""
    import torch

    rng = np.random.default_rng(51)
    B, Hq, Hkv, Lcap, N = 1, 4, 2, 5, 16
    q = rand_bits(rng, (B, Hq, D))
    kc = rng.integers(0, 256, size=(B, Hkv, Lcap, D)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(B, Hkv, Lcap, D)).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x3A  # no NaN codes in a valid cache
    vc[(vc & 0x7F) == 0x7F] = 0x41
    w = rand_bits(rng, (Hq * D, N), std=1 / math.sqrt(Hq * D))
    lens = np.array([4], np.int32)
    scale, k_scale, v_scale = 1 / math.sqrt(D), 0.0123, 0.75
    attn, y = orc.decode_fp8(q, kc, vc, lens, w, scale, k_scale, v_scale)
    kf = torch.from_numpy(kc).view(torch.float8_e4m3fn).double().numpy() * k_scale
    vf = torch.from_numpy(vc).view(torch.float8_e4m3fn).double().numpy() * v_scale
    ba, by = brute_decode(bits_to_f64(q), kf, vf, lens, bits_to_f64(w), scale)
    _close(attn, ba, 1e-12, "fp8 attention vs brute force")
    _close(y, by, 1e-12, "fp8 output vs brute force")


PINS = [v for kname, v in sorted(globals().items()) if kname.startswith("pin_") and callable(v)]


def run_all(orc) -> dict:
    res = {}
    for p in PINS:
        try:
            p(orc)
            res[p.__name__] = "ok"
        except Exception as e:  # noqa: BLE001 - every failure is a detected mistake
            res[p.__name__] = f"{type(e).__name__}: {e}"[:300]
    return res


if __name__ == "__main__":
    import argparse

    ap = argparse.ArgumentParser()
    ap.add_argument("--lib", required=True)
    args = ap.parse_args()
    from oracle import Oracle

    print(json.dumps(run_all(Oracle(args.lib))))
