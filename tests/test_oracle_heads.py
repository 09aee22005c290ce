"""Pins of the oracle's Medusa heads and top-k (Medusa Heads glossary page,
"How heads predict later tokens")."""
import numpy as np
import pytest

import workloads as W
from oracle import oracle as O


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_init_heads_reproduce_lm_head_exactly(dtype):
    # The page's check: W1 and b1 start at zero and W2 is a copy of lm_head, so
    # every head prints True against lm_head's own logits (hidden 256, vocab
    # 1000, 3 heads, h ~ N(0,1)).  z = h + SiLU(0) = h exactly, so the float64
    # logits must be bitwise equal.
    x = W.heads_inputs(seed=1, B=1, H=256, V=1000, K=3, dtype=dtype, zero_init=True)
    heads = O.heads_logits(x["h"], x["w1"], x["b1"], x["w2"], dtype)
    lm = O.lm_head_logits(x["h"], x["lm_head"], dtype)
    assert [bool(np.array_equal(heads[:, k], lm)) for k in range(3)] == [True, True, True]


def _numpy_heads(h, w1, b1, w2):
    # Library restatement on float64 arrays: W2 (h + silu(W1 h + b1)).
    u = np.einsum("kij,bj->bki", w1, h) + b1[None]
    z = h[:, None, :] + u / (1.0 + np.exp(-u))
    return np.einsum("kvi,bki->bkv", w2, z), z


def test_heads_match_numpy_restatement_fp32():
    rng = np.random.default_rng(0)
    B, K, H, V = 3, 2, 24, 37
    h = rng.standard_normal((B, H)).astype(np.float32)
    w1 = (rng.standard_normal((K, H, H)) * 0.3).astype(np.float32)  # not symmetric
    b1 = rng.standard_normal((K, H)).astype(np.float32)              # nonzero bias
    w2 = rng.standard_normal((K, V, H)).astype(np.float32)
    got, z = O.heads_logits(h, w1, b1, w2, "f32", return_z=True)
    ref, zr = _numpy_heads(*(a.astype(np.float64) for a in (h, w1, b1, w2)))
    np.testing.assert_allclose(z, zr, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-11)


def test_heads_bf16_decoding_is_exact():
    rng = np.random.default_rng(1)
    B, K, H, V = 2, 2, 16, 9
    h32 = rng.standard_normal((B, H)).astype(np.float32)
    w1 = rng.standard_normal((K, H, H)).astype(np.float32) * 0.2
    b1 = rng.standard_normal((K, H)).astype(np.float32)
    w2 = rng.standard_normal((K, V, H)).astype(np.float32)
    bits = [W.f32_to_bf16_bits(a) for a in (h32, w1, b1, w2)]
    got = O.heads_logits(*bits, "bf16")
    ref, _ = _numpy_heads(*(W.bf16_bits_to_f32(b).astype(np.float64) for b in bits))
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-11)


def test_silu_limits():
    # large |u|: SiLU(u) -> u for u >> 0 and -> 0 for u << 0 (no NaN from exp overflow)
    H = 2
    h = np.zeros((1, H), np.float32)
    w1 = np.zeros((1, H, H), np.float32)
    b1 = np.array([[800.0, -800.0]], np.float32)
    w2 = np.eye(H, dtype=np.float32)[None]
    got, z = O.heads_logits(h, w1, b1, w2, "f32", return_z=True)
    assert z[0, 0, 0] == 800.0 and z[0, 0, 1] == 0.0 and np.isfinite(got).all()


def test_topk_matches_stable_sort_with_ties():
    rng = np.random.default_rng(2)
    x = rng.integers(-5, 6, size=(7, 300)).astype(np.float64)  # many exact ties
    idx, val = O.topk(x, 9)
    for r in range(x.shape[0]):
        order = np.lexsort((np.arange(x.shape[1]), -x[r]))[:9]  # value desc, index asc
        assert idx[r].tolist() == order.tolist()
        assert val[r].tolist() == x[r, order].tolist()


def test_topk_k_equals_n_is_a_permutation():
    x = np.array([[3.0, 1.0, 3.0, 2.0]])
    idx, _ = O.topk(x, 4)
    assert idx[0].tolist() == [0, 2, 3, 1]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_lm_head_logits_closed_forms(dtype):
    # The verifier's next-token logits are lm_head h (Medusa Heads glossary page,
    # "Tree attention and acceptance": the base model scores each candidate).
    # Closed forms that a transposed operand or a shifted index would break:
    #  (1) h = e_j picks column j of lm_head: logits[v] = lm[v, j];
    #  (2) lm row v = c_v e_{pi(v)} picks one entry of h: logits[v] = c_v h[pi(v)];
    #  (3) constant h = s and lm = t_v 1: logits[v] = H s t_v.
    H, V = 24, 37
    rng = np.random.default_rng(5)
    lm = (rng.integers(-8, 9, (V, H)) / 4.0).astype(np.float32)  # exact in bf16
    hs = np.zeros((H, H), np.float32)
    hs[np.arange(H), np.arange(H)] = 1.0
    conv = (lambda a: W.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    got = O.lm_head_logits(conv(hs), conv(lm), dtype)                     # [H, V]
    np.testing.assert_array_equal(got, lm.T.astype(np.float64))
    pi = rng.permutation(V) % H
    c = (rng.integers(1, 5, V) / 2.0).astype(np.float32)
    lm2 = np.zeros((V, H), np.float32)
    lm2[np.arange(V), pi] = c
    h2 = (rng.integers(-16, 17, (3, H)) / 8.0).astype(np.float32)
    got2 = O.lm_head_logits(conv(h2), conv(lm2), dtype)
    np.testing.assert_array_equal(got2, (h2[:, pi] * c[None]).astype(np.float64))
    t = (rng.integers(-4, 5, V) / 4.0).astype(np.float32)
    got3 = O.lm_head_logits(conv(np.full((1, H), 0.5, np.float32)),
                            conv(np.repeat(t[:, None], H, 1)), dtype)
    np.testing.assert_array_equal(got3[0], H * 0.5 * t.astype(np.float64))


def _perm_case(seed, B=3, K=3, H=12, V=17):
    """Heads whose W1_k = s * P_k for permutation matrices P_k (row i holds a 1
    at column pi_k(i), so (W1_k h)_i = s * h[pi_k(i)]) and whose W2_k rows are
    one-hot: W2_k[v] = e_{rho_k(v)}.  No P_k is symmetric, and pi_k != rho_k."""
    rng = np.random.default_rng(seed)
    pis = [rng.permutation(H) for _ in range(K)]
    for p in pis:
        assert not np.array_equal(p[p], np.arange(H))  # P_k is not its own transpose
    rhos = [rng.integers(0, H, V) for _ in range(K)]
    h = (rng.integers(-24, 25, (B, H)) / 8.0).astype(np.float32)  # exact in bf16 too
    w2 = np.zeros((K, V, H), np.float32)
    for k in range(K):
        w2[k, np.arange(V), rhos[k]] = 1.0
    def w1(sign):
        a = np.zeros((K, H, H), np.float32)
        for k in range(K):
            a[k, np.arange(H), pis[k]] = sign
        return a
    return h, w1, w2, pis, rhos


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_silu_odd_part_pins_w1_orientation_and_heads(dtype):
    # SiLU(x) - SiLU(-x) = x sigma(x) + x sigma(-x) = x for every x.  With
    # W1_k = +P_k and W1_k = -P_k (b1 = 0) the two z's differ by exactly
    # h[pi_k]; through the one-hot W2_k the logits differ by h[pi_k[rho_k(v)]].
    # A transposed W1 would give h[pi_k^-1], a head offset another pi, a dropped
    # residual or SiLU term a difference other than x.
    h, w1, w2, pis, rhos = _perm_case(11)
    K, H = w2.shape[0], h.shape[1]
    b1 = np.zeros((K, H), np.float32)
    conv = (lambda a: W.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    lp = O.heads_logits(conv(h), conv(w1(1.0)), conv(b1), conv(w2), dtype)
    lm = O.heads_logits(conv(h), conv(w1(-1.0)), conv(b1), conv(w2), dtype)
    for k in range(K):
        np.testing.assert_allclose(lp[:, k] - lm[:, k], h[:, pis[k][rhos[k]]].astype(np.float64),
                                   rtol=0, atol=1e-12)


def test_silu_even_part_pins_the_sigmoid():
    # SiLU(x) + SiLU(-x) = x (sigma(x) - sigma(-x)) = x tanh(x / 2), so the two
    # z's above sum to 2 h + h[pi] tanh(h[pi] / 2).  The odd part alone cannot
    # tell x sigma(x) from x sigma(-x); this sum changes sign between them.
    h, w1, w2, pis, rhos = _perm_case(12)
    K, H = w2.shape[0], h.shape[1]
    b1 = np.zeros((K, H), np.float32)
    lp = O.heads_logits(h, w1(1.0), b1, w2, "f32")
    lm = O.heads_logits(h, w1(-1.0), b1, w2, "f32")
    hd = h.astype(np.float64)
    for k in range(K):
        x = hd[:, pis[k]]
        want = 2.0 * hd + x * np.tanh(x / 2.0)
        np.testing.assert_allclose(lp[:, k] + lm[:, k], want[:, rhos[k]], rtol=0, atol=1e-12)


def test_bias_odd_part_pins_bias_orientation():
    # W1 = 0 and b1 = +c vs -c: z differs by exactly c_k (the bias of head k,
    # feature i), whatever h is; through one-hot W2_k rows that is c_k[rho_k(v)].
    h, _, w2, _, rhos = _perm_case(13)
    K, H = w2.shape[0], h.shape[1]
    rng = np.random.default_rng(14)
    c = (rng.integers(-40, 41, (K, H)) / 16.0).astype(np.float32)
    w1 = np.zeros((K, H, H), np.float32)
    lp = O.heads_logits(h, w1, c, w2, "f32")
    lm = O.heads_logits(h, w1, -c, w2, "f32")
    for k in range(K):
        np.testing.assert_allclose(lp[:, k] - lm[:, k], np.broadcast_to(c[k, rhos[k]], lp[:, k].shape),
                                   rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_lm_head_matmul_form_equals_the_loop(dtype):
    # the matrix-product form of the lm_head logits (for large row counts) gives
    # the C loop's float64 values on shapes with ragged sizes
    rng = np.random.default_rng(6)
    h = rng.standard_normal((7, 40)).astype(np.float32)
    lm = (rng.standard_normal((53, 40)) * 0.1).astype(np.float32)
    conv = (lambda a: W.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    a = O.lm_head_logits(conv(h), conv(lm), dtype)
    b = O.lm_head_logits_matmul(conv(h), conv(lm), dtype)
    np.testing.assert_allclose(b, a, rtol=1e-13, atol=1e-13)
