"""Pins of the oracle's XA block-mask estimation (antidiagonal scoring and the
threshold selection) against library routines, closed forms and brute force.

The pages name the scoring (antidiagonal, stride 16, threshold 0.9) without
writing it out; the oracle follows a stated reading of those words.  These
checks pin that reading's arithmetic: the cell indexing (antidiagonal, not
diagonal), the softmax normalisation over causal cells, the block sums over
the query heads of a KV head, and the selection rule.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle

BLOCK = oracle.BLOCK


def _bf16(*shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("S,T,Hq,Hkv", [(300, 64, 4, 2), (256, 32, 2, 2)])
def test_stride_one_is_block_sums_of_softmax_attention(S, T, Hq, Hkv):
    """With stride 1 a cell is one (query, key) pair: the scores must be the
    block sums of causal softmax attention probabilities (torch, fp64)."""
    Q = _bf16(1, S, Hq, 128, seed=1)
    K = _bf16(1, S, Hkv, 128, seed=2)
    g = Hq // Hkv
    scale = 1.0 / np.sqrt(128)
    nB = (S + T - 1) // T
    causal = torch.ones(S, S, dtype=torch.bool).tril()
    for h in range(Hkv):
        W = oracle.xa_block_scores(Q, K, 0, h, stride=1, T=T)
        ref = torch.zeros(nB, nB, dtype=torch.float64)
        for qh in range(h * g, (h + 1) * g):
            logits = (Q[0, :, qh].double() @ K[0, :, h].double().T) * scale
            P = torch.softmax(logits.masked_fill(~causal, float("-inf")), dim=-1)
            pad = nB * T - S
            Pp = torch.nn.functional.pad(P, (0, pad, 0, pad))
            ref += Pp.reshape(nB, T, nB, T).sum(dim=(1, 3))
        np.testing.assert_allclose(W, ref.numpy(), rtol=1e-12, atol=1e-12)


def _uniform_scores(S, s, T, g):
    """Closed form when every cell score is equal: P[a][c] = 1/(a+1) for c <= a."""
    nA = (S + s - 1) // s
    nB = (S + T - 1) // T
    W = np.zeros((nB, nB))
    for a in range(nA):
        for c in range(a + 1):
            W[a * s // T, c * s // T] += g / (a + 1)
    return W


def test_zero_queries_give_the_uniform_closed_form():
    S, s, T = 512, 16, 128
    Q = torch.zeros(1, S, 4, 128, dtype=torch.bfloat16)
    K = _bf16(1, S, 2, 128, seed=3)
    W = oracle.xa_block_scores(Q, K, 0, 1, stride=s, T=T)
    np.testing.assert_allclose(W, _uniform_scores(S, s, T, 2), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("u0,v0", [(3, 12), (0, 15), (15, 0), (3, 3), (5, 11), (0, 0)])
def test_one_nonzero_pair_lights_only_its_antidiagonal_cell(u0, v0):
    """Q and K are zero except one query token a0*s+u0 and one key token c0*s+v0.
    The cell (a0, c0) departs from the uniform closed form iff u0 + v0 = s - 1
    (the pair lies on the cell's antidiagonal), by the closed form
    P[a0][c0] = e^x / (e^x + a0) with x = scale * <q, k> / s."""
    S, s, T, d = 512, 16, 128, 128
    a0, c0 = 19, 4
    Q = torch.zeros(1, S, 2, d, dtype=torch.bfloat16)
    K = torch.zeros(1, S, 1, d, dtype=torch.bfloat16)
    Q[0, a0 * s + u0, 1, :] = 1.0
    K[0, c0 * s + v0, 0, :] = 2.0
    W = oracle.xa_block_scores(Q, K, 0, 0, stride=s, T=T)
    ref = _uniform_scores(S, s, T, 2)
    if u0 + v0 == s - 1:
        x = (1.0 / np.sqrt(d)) * (2.0 * d) / s
        p_hit, p_other = np.exp(x) / (np.exp(x) + a0), 1.0 / (np.exp(x) + a0)
        qb = a0 * s // T
        for c in range(a0 + 1):
            ref[qb, c * s // T] += (p_hit if c == c0 else p_other) - 1.0 / (a0 + 1)
        assert not np.allclose(ref, _uniform_scores(S, s, T, 2))
    np.testing.assert_allclose(W, ref, rtol=1e-13, atol=1e-13)


def test_row_totals_count_the_softmax_rows():
    """Each cell row's probabilities add to 1: a block row's total is the number of
    cell rows in it times the heads of the group (ragged last block included)."""
    S, s, T = 400, 16, 128
    Q = _bf16(1, S, 4, 128, seed=4)
    K = _bf16(1, S, 1, 128, seed=5)
    W = oracle.xa_block_scores(Q, K, 0, 0, stride=s, T=T)
    nA = (S + s - 1) // s
    rows = np.bincount(np.arange(nA) * s // T, minlength=W.shape[0])
    np.testing.assert_allclose(W.sum(axis=1), 4 * rows, rtol=1e-12)
    assert np.all(np.triu(W, 1) == 0)


def _brute_force_select(row, tau):
    """Fewest blocks whose scores reach tau * total; among those, the largest sum."""
    n = len(row)
    total = sum(row)
    for size in range(0, n + 1):
        best = None
        for X in itertools.combinations(range(n), size):
            t = sum(row[i] for i in X)
            if t >= tau * total and (best is None or t > best[0]):
                best = (t, X)
        if best is not None:
            return set(best[1])
    return set(range(n))


@pytest.mark.parametrize("tau", [0.3, 0.5, 0.9, 0.97])
def test_selection_matches_brute_force_over_subsets(tau):
    rng = np.random.default_rng(7)
    nB = 7
    W = np.tril(rng.exponential(size=(nB, nB)))
    mask = oracle.xa_select(W, tau)
    for qb in range(nB):
        expect = _brute_force_select(list(W[qb, :qb + 1]), tau) | {qb}
        got = set(np.nonzero(mask[qb])[0].tolist())
        assert got == expect, (qb, got, expect)


def test_selection_edge_thresholds_and_planted_block():
    rng = np.random.default_rng(8)
    nB = 6
    W = np.tril(rng.uniform(0.1, 1.0, size=(nB, nB)))
    assert np.array_equal(oracle.xa_select(W, 0.0), np.eye(nB, dtype=np.uint8))
    assert np.array_equal(oracle.xa_select(W, 1.0), np.tril(np.ones((nB, nB), dtype=np.uint8)))
    W2 = W.copy()
    W2[5, 2] = 100.0                      # one block holds almost all of row 5's mass
    m = oracle.xa_select(W2, 0.9)
    assert set(np.nonzero(m[5])[0].tolist()) == {2, 5}
    # equal scores: lower key blocks first
    W3 = np.tril(np.ones((4, 4)))
    m3 = oracle.xa_select(W3, 0.5)
    assert m3[3].tolist() == [1, 1, 0, 1]


def test_estimate_touches_block_heads_only():
    S = 256
    Q = _bf16(1, S, 4, 128, seed=9)
    K = _bf16(1, S, 2, 128, seed=10)
    W, M = oracle.xa_estimate(Q, K, np.array([[0, BLOCK]], dtype=np.uint8), stride=16, tau=0.9)
    assert np.all(W[0, 0] == 0) and np.all(M[0, 0] == 0)
    assert np.all(np.diag(M[0, 1]) == 1)
    np.testing.assert_allclose(W[0, 1], oracle.xa_block_scores(Q, K, 0, 1, stride=16))


def test_ragged_last_cell():
    """S = 410 with stride 16: the last cell holds 10 tokens.  Zero queries give
    the uniform closed form over ceil(S/16) = 26 cells; a pair inside the last
    cell on its antidiagonal (query offset 2, key offset 13: both below S) moves
    only that cell, by the closed form."""
    S, s, T, d = 410, 16, 128, 128
    Q = torch.zeros(1, S, 1, d, dtype=torch.bfloat16)
    K = _bf16(1, S, 1, d, seed=12)
    W = oracle.xa_block_scores(Q, K, 0, 0, stride=s, T=T)
    np.testing.assert_allclose(W, _uniform_scores(S, s, T, 1), rtol=1e-13, atol=1e-13)
    a0 = c0 = S // s                      # the partial cell, 25 (tokens 400 .. 409)
    Q = torch.zeros(1, S, 1, d, dtype=torch.bfloat16)
    K = torch.zeros(1, S, 1, d, dtype=torch.bfloat16)
    Q[0, a0 * s + 2, 0, :] = 1.0          # its antidiagonal partner in cell 25 (token 413) does not exist
    W = oracle.xa_block_scores(Q, K, 0, 0, stride=s, T=T)
    np.testing.assert_allclose(W, _uniform_scores(S, s, T, 1), rtol=1e-13, atol=1e-13)
    K[0, (c0 - 1) * s + 13, 0, :] = 1.0   # the partner one cell to the left (token 397)
    W = oracle.xa_block_scores(Q, K, 0, 0, stride=s, T=T)
    x = (1.0 / np.sqrt(d)) * d / s
    ref = _uniform_scores(S, s, T, 1)
    qb = a0 * s // T
    for c in range(a0 + 1):
        hit = c == c0 - 1
        ref[qb, c * s // T] += (np.exp(x) if hit else 1.0) / (np.exp(x) + a0) - 1.0 / (a0 + 1)
    np.testing.assert_allclose(W, ref, rtol=1e-13, atol=1e-13)
