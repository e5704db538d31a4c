"""Pins for the oracle's attention (CPU only).

Each test checks ``oracle.attention`` against something other than itself:
exact arithmetic on the worked example printed on the page, closed forms,
invariants the pages state, and an independent library implementation.
"""

import math
import os
from fractions import Fraction

import mpmath
import numpy as np
import pytest
import torch

from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example_kvcache.txt")


def _read_golden():
    sections, cur = {}, None
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("["):
            cur = line.strip("[]")
            sections[cur] = []
            continue
        sections[cur].append([Fraction(tok) for tok in line.split()])
    return sections


def _matmul(a, b):
    return [[sum(a[i][k] * b[k][j] for k in range(len(b))) for j in range(len(b[0]))]
            for i in range(len(a))]


def _exact_causal(X, WQ, WK, WV, div):
    """Exact rationals for Q, K, V and scores; 50-digit exp for the softmax."""
    mpmath.mp.dps = 50
    Q, K, V = _matmul(X, WQ), _matmul(X, WK), _matmul(X, WV)
    n = len(X)
    out = []
    for i in range(n):
        scores = [sum(Q[i][j] * K[t][j] for j in range(4)) / div for t in range(i + 1)]
        e = [mpmath.exp(mpmath.mpf(s.numerator) / s.denominator) for s in scores]
        z = sum(e)
        row = [sum(e[t] * mpmath.mpf(V[t][j].numerator) / V[t][j].denominator for t in range(i + 1)) / z
               for j in range(4)]
        out.append([float(x) for x in row])
    return Q, K, V, np.array(out)


def test_worked_example_steps_match_exact_arithmetic():
    g = _read_golden()
    X, WQ, WK, WV = g["X"], g["W_Q"], g["W_K"], g["W_V"]
    div = g["divisor"][0][0]
    scale = float(1 / div)
    # step 1: two tokens; step 2: three tokens (the page recomputes everything)
    for n in (2, 3):
        Q, K, V, exact = _exact_causal(X[:n], WQ, WK, WV, div)
        Qf = np.array([[float(x) for x in r] for r in Q])
        Kf = np.array([[float(x) for x in r] for r in K])
        Vf = np.array([[float(x) for x in r] for r in V])
        got = A.causal_attention(Qf, Kf, Vf, scale)
        np.testing.assert_allclose(got, exact, rtol=0, atol=1e-15)
    # row 1 attends to itself only: output row 1 == V row 1 (exactly)
    _, _, V, exact2 = _exact_causal(X[:2], WQ, WK, WV, div)
    assert exact2[0].tolist() == [float(x) for x in V[0]]


def test_worked_example_cached_decode_equals_recompute():
    """Step 2 with a cache: q of the new token against cached K/V rows 1..3 equals row 3
    of the full recompute ([KV Cache篇] §2.2), and rows 1..2 of step 2 equal step 1."""
    g = _read_golden()
    X, WQ, WK, WV = g["X"], g["W_Q"], g["W_K"], g["W_V"]
    div = g["divisor"][0][0]
    Q, K, V, exact3 = _exact_causal(X, WQ, WK, WV, div)
    _, _, _, exact2 = _exact_causal(X[:2], WQ, WK, WV, div)
    np.testing.assert_allclose(exact3[:2], exact2, rtol=0, atol=1e-15)
    Qf = np.array([[float(x) for x in r] for r in Q])
    Kf = np.array([[float(x) for x in r] for r in K])
    Vf = np.array([[float(x) for x in r] for r in V])
    got = A.decode_attention_one(Qf[2], Kf, Vf, float(1 / div))
    np.testing.assert_allclose(got, exact3[2], rtol=0, atol=1e-15)


def test_worked_example_as_paged_cache():
    """The same three cached tokens stored in two permuted physical blocks of size 2."""
    g = _read_golden()
    X, WQ, WK, WV = g["X"], g["W_Q"], g["W_K"], g["W_V"]
    div = g["divisor"][0][0]
    Q, K, V, exact3 = _exact_causal(X, WQ, WK, WV, div)
    Kf = np.array([[float(x) for x in r] for r in K])
    Vf = np.array([[float(x) for x in r] for r in V])
    q = np.array([[[float(x) for x in Q[2]]]])           # [batch 1, H 1, d 4]
    B, nb = 2, 5
    kp = np.full((nb, 1, B, 4), np.nan)
    vp = np.full((nb, 1, B, 4), np.nan)
    table = [3, 1]                                         # logical 0 -> 3, logical 1 -> 1
    for t in range(3):
        kp[table[t // B], 0, t % B] = Kf[t]
        vp[table[t // B], 0, t % B] = Vf[t]
    got = A.paged_decode_attention(q, kp, vp, np.array([table]), [3], float(1 / div), B)
    np.testing.assert_allclose(got[0, 0], exact3[2], rtol=0, atol=1e-15)


# ---------------------------------------------------------------- closed forms

def test_single_token_returns_its_value_exactly():
    rng = np.random.default_rng(11)
    q, K, V = rng.standard_normal(64), rng.standard_normal((1, 64)), rng.standard_normal((1, 64))
    assert np.array_equal(A.decode_attention_one(q, K, V, 0.125), V[0])


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(12)
    K, V = rng.standard_normal((37, 64)), rng.standard_normal((37, 64))
    got = A.decode_attention_one(np.zeros(64), K, V, 0.125)
    np.testing.assert_allclose(got, V.mean(axis=0), rtol=0, atol=1e-14)


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(13)
    K = np.tile(rng.standard_normal(64), (20, 1))
    V = rng.standard_normal((20, 64))
    got = A.decode_attention_one(rng.standard_normal(64), K, V, 0.3)
    np.testing.assert_allclose(got, V.mean(axis=0), rtol=0, atol=1e-14)


def test_constant_values_are_returned():
    rng = np.random.default_rng(14)
    c = rng.standard_normal(64)
    V = np.tile(c, (50, 1))
    got = A.decode_attention_one(rng.standard_normal(64), rng.standard_normal((50, 64)), V, 0.125)
    np.testing.assert_allclose(got, c, rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(15)
    q = rng.standard_normal(64)
    K = rng.standard_normal((30, 64)) * 0.01
    K[17] = q * 1000.0
    V = rng.standard_normal((30, 64))
    got = A.decode_attention_one(q, K, V, 1.0)
    np.testing.assert_allclose(got, V[17], rtol=0, atol=1e-14)


def test_two_keys_closed_form():
    """Two keys: p = sigmoid(x0 - x1), out = p V0 + (1-p) V1."""
    rng = np.random.default_rng(16)
    q, K, V = rng.standard_normal(8), rng.standard_normal((2, 8)), rng.standard_normal((2, 8))
    s = 0.7
    x0, x1 = s * q @ K[0], s * q @ K[1]
    p0 = 1.0 / (1.0 + math.exp(x1 - x0))
    np.testing.assert_allclose(A.decode_attention_one(q, K, V, s), p0 * V[0] + (1 - p0) * V[1],
                               rtol=0, atol=1e-15)


def test_score_shift_invariance():
    """Adding u with q.u = c to every key shifts every score by scale*c: output unchanged."""
    rng = np.random.default_rng(17)
    q, K, V = rng.standard_normal(64), rng.standard_normal((40, 64)), rng.standard_normal((40, 64))
    u = 3.0 * q / (q @ q)
    a = A.decode_attention_one(q, K, V, 0.2)
    b = A.decode_attention_one(q, K + u, V, 0.2)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_empty_context_is_zero():
    got = A.decode_attention_one(np.ones(64), np.zeros((0, 64)), np.zeros((0, 64)), 0.125)
    assert np.array_equal(got, np.zeros(64))


def test_scale_is_applied_to_scores():
    """With two keys the output depends on scale only through scale*(x0-x1)."""
    rng = np.random.default_rng(18)
    q, K, V = rng.standard_normal(16), rng.standard_normal((2, 16)), rng.standard_normal((2, 16))
    a = A.decode_attention_one(q, K, V, 0.5)
    b = A.decode_attention_one(2.0 * q, K, V, 0.25)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-15)
    c = A.decode_attention_one(q, K, V, 1.0)
    assert not np.allclose(a, c)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("n,d", [(1, 4), (5, 64), (37, 64), (129, 128)])
def test_cached_decode_equals_last_row_of_causal_recompute(n, d):
    rng = np.random.default_rng(100 + n)
    Q, K, V = (rng.standard_normal((n, d)) for _ in range(3))
    s = 1 / math.sqrt(d)
    full = A.causal_attention(Q, K, V, s)
    for i in range(n):
        np.testing.assert_allclose(A.decode_attention_one(Q[i], K[:i + 1], V[:i + 1], s), full[i],
                                   rtol=0, atol=1e-13)


@pytest.mark.parametrize("B", [1, 2, 8, 16, 32])
def test_paged_equals_contiguous_under_block_permutation(B):
    rng = np.random.default_rng(200 + B)
    H, d = 3, 16
    lens = [0, 1, B - 1 if B > 1 else 1, B, B + 1, 3 * B + 5, 70]
    total = sum(-(-n // B) for n in lens)
    nb = total + 7
    perm = rng.permutation(nb)
    kp = np.full((nb, H, B, d), np.nan)
    vp = np.full((nb, H, B, d), np.nan)
    tables = np.full((len(lens), max(1, max(-(-n // B) for n in lens))), -1)
    ks, vs, pos = [], [], 0
    for s, n in enumerate(lens):
        Ks, Vs = rng.standard_normal((n, H, d)), rng.standard_normal((n, H, d))
        ks.append(Ks)
        vs.append(Vs)
        for j in range(-(-n // B)):
            tables[s, j] = perm[pos]
            pos += 1
        for t in range(n):
            kp[tables[s, t // B], :, t % B] = Ks[t]
            vp[tables[s, t // B], :, t % B] = Vs[t]
    q = rng.standard_normal((len(lens), H, d))
    want = A.decode_attention(q, ks, vs, 0.25)
    got = A.paged_decode_attention(q, kp, vp, tables, lens, 0.25, B)
    assert np.array_equal(got, want)          # same values, same order of operations
    assert np.all(np.isfinite(got))           # NaN in unused slots never read


def test_matches_torch_sdpa_float64():
    rng = np.random.default_rng(300)
    b, H, d = 3, 4, 32
    lens = [1, 17, 64]
    q = rng.standard_normal((b, H, d))
    ks = [rng.standard_normal((n, H, d)) for n in lens]
    vs = [rng.standard_normal((n, H, d)) for n in lens]
    got = A.decode_attention(q, ks, vs, 1 / math.sqrt(d))
    for s in range(b):
        qt = torch.from_numpy(q[s]).view(H, 1, d)
        kt = torch.from_numpy(ks[s]).permute(1, 0, 2)
        vt = torch.from_numpy(vs[s]).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).view(H, d).numpy()
        np.testing.assert_allclose(got[s], ref, rtol=0, atol=1e-13)


def test_fp8_paged_dequantises_with_block_scale():
    """FP8 pool: element value = decode(code) * scale[physical block].  Pinned through an
    independent route: torch's own float8_e4m3fn type widens the codes, torch indexing
    picks each token's block and block scale, and torch's float64 SDPA attends.  The
    scales differ per block (K and V too) and the table is permuted, so a scale taken by
    logical block, or K's scale used for V, fails; unused slots hold the NaN code."""
    from oracle import fp8
    rng = np.random.default_rng(400)
    B, H, d, nb = 4, 2, 8, 6
    # codes of magnitudes below 2 (exponent field <= 7) and both signs: with block scales
    # in [0.25, 2] the softmax weights stay spread, so every scale matters
    sign = lambda: (rng.integers(0, 2, (nb, H, B, d)) << 7).astype(np.uint8)
    codes_k = rng.integers(0, 0x40, (nb, H, B, d), dtype=np.uint8) | sign()
    codes_v = rng.integers(0, 0x40, (nb, H, B, d), dtype=np.uint8) | sign()
    ks = rng.uniform(0.25, 2.0, nb)
    vs = rng.uniform(0.25, 2.0, nb)
    table = np.array([[4, 0, 2]])
    n = 10                                                  # block 2 holds 2 of its 4 slots
    codes_k[2, :, 2:] = 0x7F
    codes_v[2, :, 2:] = 0x7F
    q = rng.standard_normal((1, H, d))
    got = A.paged_decode_attention(q, codes_k, codes_v, table, [n], 0.3, B, ks, vs, fp8.decode)
    assert np.all(np.isfinite(got))

    def widened(codes, scale):                              # [n, H, d] float64, torch only
        t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
        tok = torch.arange(n)
        phys = torch.from_numpy(table[0])[tok // B]
        return t[phys, :, tok % B, :] * torch.from_numpy(scale)[phys].view(n, 1, 1)

    K, V = widened(codes_k, ks), widened(codes_v, vs)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q[0]).view(H, 1, d), K.permute(1, 0, 2), V.permute(1, 0, 2), scale=0.3).view(H, d)
    np.testing.assert_allclose(got[0], ref.numpy(), rtol=0, atol=1e-13)


# ---------------------------------------------------------------- grouped-query attention

@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_gqa_equals_mha_on_replicated_kv_heads(G):
    """Sharing a K/V head among G query heads is MHA over K/V heads repeated G times."""
    rng = np.random.default_rng(500 + G)
    Hkv, d, lens = 3, 16, [1, 9, 40]
    q = rng.standard_normal((len(lens), Hkv * G, d))
    ks = [rng.standard_normal((n, Hkv, d)) for n in lens]
    vs = [rng.standard_normal((n, Hkv, d)) for n in lens]
    got = A.decode_attention_gqa(q, ks, vs, 0.3)
    want = A.decode_attention(q, [np.repeat(k, G, axis=1) for k in ks], [np.repeat(v, G, axis=1) for v in vs], 0.3)
    assert np.array_equal(got, want)
    if G == 1:
        assert np.array_equal(got, A.decode_attention(q, ks, vs, 0.3))


def test_gqa_matches_torch_sdpa_enable_gqa():
    rng = np.random.default_rng(510)
    Hkv, G, d, n = 2, 4, 32, 21
    q = rng.standard_normal((1, Hkv * G, d))
    k = rng.standard_normal((n, Hkv, d))
    v = rng.standard_normal((n, Hkv, d))
    got = A.decode_attention_gqa(q, [k], [v], 1 / math.sqrt(d))[0]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q[0]).view(1, Hkv * G, 1, d), torch.from_numpy(k).permute(1, 0, 2)[None],
        torch.from_numpy(v).permute(1, 0, 2)[None], enable_gqa=True).view(Hkv * G, d).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- sliding window

def test_window_closed_forms():
    rng = np.random.default_rng(520)
    H, d, lens = 2, 16, [1, 5, 40]
    q = rng.standard_normal((3, H, d))
    ks = [rng.standard_normal((n, H, d)) for n in lens]
    vs = [rng.standard_normal((n, H, d)) for n in lens]
    full = A.decode_attention(q, ks, vs, 0.25)
    # a window at least as long as every context, or none, changes nothing
    assert np.array_equal(A.decode_attention_window(q, ks, vs, 0.25, 40), full)
    assert np.array_equal(A.decode_attention_window(q, ks, vs, 0.25, 0), full)
    # a window of one token returns that token's value row exactly
    w1 = A.decode_attention_window(q, ks, vs, 0.25, 1)
    for s, n in enumerate(lens):
        assert np.array_equal(w1[s], vs[s][n - 1])
    # window W equals full attention over the last W rows, and differs from the full context
    w7 = A.decode_attention_window(q, ks, vs, 0.25, 7)
    np.testing.assert_allclose(w7[2], A.decode_attention(q[2:], [ks[2][-7:]], [vs[2][-7:]], 0.25)[0],
                               rtol=0, atol=0)
    assert not np.allclose(w7[2], full[2])
