"""GPU parity of medusa_verify_accept_chain against the oracle (e-book page "Giai
ma dau co: doan truoc roi kiem mot luot", "Faster without changing the result"
and "Why a round always yields exactly k + 1 tokens")."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import analytic as A
from oracle import oracle as O
from util import CHAIN_RACE_BAND, to_dev, to_np

pytestmark = pytest.mark.gpu


def _gpu(M, x, seed, rnd):
    gamma = x["p"].shape[1] - 1
    n_acc, out = M.verify_accept_chain(to_dev(x["p"]), to_dev(x["q"]) if gamma else None,
                                       to_dev(x["draft"]) if gamma else None, seed, rnd)
    torch.cuda.synchronize()
    return to_np(n_acc), to_np(out)


def _compare(n_acc, out, ref, band=CHAIN_RACE_BAND):
    """Acceptance counts are exact; the drawn token may differ only where the
    oracle's two best race keys are within `band` (relative): the float32 keys'
    own error bound, 8 units of 2^-24 (tests/util.py)."""
    assert np.array_equal(n_acc, ref["n_acc"])
    near = 0
    for b in range(len(n_acc)):
        if np.array_equal(out[b], ref["out_tok"][b]):
            continue
        k = n_acc[b]
        assert np.array_equal(out[b, :k], ref["out_tok"][b, :k])
        assert ref["race_gap"][b] < band, (b, out[b], ref["out_tok"][b])
        near += 1
    return near


@pytest.mark.parametrize("B,gamma,V,sigma", [(16, 0, 1000, 0.5), (16, 1, 1000, 0.1), (32, 4, 5000, 1.0),
                                             (8, 8, 20000, 0.5)])
def test_chain_small(medusa, B, gamma, V, sigma):
    x = W.chain_inputs(seed=gamma + 3, B=B, gamma=gamma, V=V, sigma=sigma)
    for rnd in range(3):
        n_acc, out = _gpu(medusa, x, 1234, rnd)
        ref = O.verify_chain(x["p"], x["q"], x["draft"], 1234, rnd)
        assert _compare(n_acc, out, ref) <= 1
        assert ((out >= 0).sum(1) == n_acc + 1).all()  # k + 1 tokens


@pytest.mark.parametrize("B,gamma,V,sigma", [
    # scalar path (vocab not a multiple of 4: rows not 16-byte aligned)
    (5, 3, 999, 0.5), (3, 0, 1001, 0.1),
    # 16-byte path at its edges: rows shorter than a warp's first group, a
    # single chunk per sequence, a ragged last chunk, chunks ending inside a
    # warp's groups
    (1, 2, 8, 0.5), (3, 1, 4, 1.0), (2, 5, 2044, 0.5), (7, 2, 2052, 0.5), (64, 1, 2048, 0.3),
    (4, 3, 8196, 0.5)])
def test_chain_paths_and_edges(medusa, B, gamma, V, sigma):
    x = W.chain_inputs(seed=B * 13 + gamma, B=B, gamma=gamma, V=V, sigma=sigma)
    for rnd in range(3):
        n_acc, out = _gpu(medusa, x, 4321, rnd)
        ref = O.verify_chain(x["p"], x["q"], x["draft"], 4321, rnd)
        assert _compare(n_acc, out, ref) <= 1
        assert ((out >= 0).sum(1) == n_acc + 1).all()


def test_chain_misaligned_rows_take_the_scalar_path(medusa):
    # p and q one float past a 16-byte boundary: the same results
    B, gamma, V = 6, 3, 4096
    x = W.chain_inputs(seed=17, B=B, gamma=gamma, V=V, sigma=0.5)
    P = torch.empty(x["p"].size + 1, device="cuda")[1:].view(B, gamma + 1, V)
    Q = torch.empty(x["q"].size + 1, device="cuda")[1:].view(B, gamma, V)
    P.copy_(to_dev(x["p"]))
    Q.copy_(to_dev(x["q"]))
    for rnd in range(2):
        n_acc, out = medusa.verify_accept_chain(P, Q, to_dev(x["draft"]), 7, rnd)
        torch.cuda.synchronize()
        ref = O.verify_chain(x["p"], x["q"], x["draft"], 7, rnd)
        assert _compare(to_np(n_acc), to_np(out), ref) <= 1


@pytest.mark.parametrize("gamma,sigma", [(0, 0.1), (1, 0.5), (4, 1.0), (8, 0.1), (32, 0.5)])
def test_chain_full_size(medusa, gamma, sigma):
    c = W.WORKLOADS["chain_b64_v128256"]
    x = W.chain_inputs(seed=5, B=c["B"], gamma=gamma, V=c["V"], sigma=sigma)
    for rnd in range(2):
        n_acc, out = _gpu(medusa, x, 99, rnd)
        ref = O.verify_chain(x["p"], x["q"], x["draft"], 99, rnd)
        assert _compare(n_acc, out, ref) <= 1


def test_identical_distributions_give_gamma_plus_one(medusa):
    x = W.chain_inputs(seed=9, B=16, gamma=6, V=3000, sigma=0.0)
    x["p"][:, :6] = x["q"]
    n_acc, out = _gpu(medusa, x, 5, 0)
    assert (n_acc == 6).all() and (out >= 0).all()
    ref = O.verify_chain(x["p"], x["q"], x["draft"], 5, 0)
    _compare(n_acc, out, ref)


def test_measured_alpha_and_expected_tokens(medusa):
    # One fixed (p, q) pair on every position: the measured acceptance rate
    # matches sum min(p, q) = 1 - TV, and the mean tokens per round matches
    # E = (1 - alpha^(gamma+1)) / (1 - alpha) ("Expected tokens per round").
    V, B, gamma, R = 2048, 64, 6, 40
    rng = np.random.default_rng(11)
    ql = rng.standard_normal(V) * 2.0
    q = np.exp(ql - ql.max()); q /= q.sum()
    y = ql + rng.standard_normal(V) * 0.5
    p = np.exp(y - y.max()); p /= p.sum()
    p32, q32 = p.astype(np.float32), q.astype(np.float32)
    alpha = float(np.minimum(p32.astype(np.float64), q32.astype(np.float64)).sum())
    P = to_dev(np.ascontiguousarray(np.broadcast_to(p32, (B, gamma + 1, V))))
    Q = to_dev(np.ascontiguousarray(np.broadcast_to(q32, (B, gamma, V))))
    c = np.cumsum(q32.astype(np.float64))
    acc = exam = 0
    toks = []
    for r in range(R):
        u = rng.random((B, gamma)) * c[-1]
        draft = np.minimum(np.searchsorted(c, u, side="right"), V - 1).astype(np.int32)
        n_acc, out = medusa.verify_accept_chain(P, Q, to_dev(draft), 77, r)
        n_acc = to_np(n_acc)
        acc += int(n_acc.sum())
        exam += int(np.minimum(n_acc + 1, gamma).sum())
        toks.append(n_acc + 1)
    toks = np.concatenate(toks)
    a_hat = acc / exam
    assert abs(a_hat - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / exam)
    E = A.expected_tokens(alpha, gamma)
    assert abs(toks.mean() - E) < 4 * toks.std() / np.sqrt(len(toks))
    print(f"\nalpha={alpha:.4f} measured={a_hat:.4f}  E={E:.4f} mean tokens={toks.mean():.4f}")
