"""Parity of the XA block-mask estimation (CUDA, through the C ABI) with the
fp64 oracle: block scores element by element, the selection bit for bit when
applied to the kernel's own scores, and every mask row that differs from the
oracle's shown to be a near-tie of the fp64 scores.  Covers several cell-row
tiles and key tiles with a ragged tail, group sizes 1 to 4, several batch rows,
the threshold edge cases, too many BLOCK heads for the workspace, and sampled
rows of the 256K workload."""
import numpy as np
import pytest
import torch

import oracle
import sparse_head_attention_gb300 as ea
from sparse_head_attention_gb300 import workloads as wl
from gpu_helpers import check_no_device_error, gpu_device

pytestmark = pytest.mark.gpu
FULL, SSA, BLOCK = ea.FULL, ea.SSA, ea.BLOCK

# fp32 scores from bf16 products accumulated in fp32 and SFU exponentials:
# relative 1e-3 of the score, plus 1e-6 of the row total.
SCORE_RTOL = 1e-3
SCORE_ATOL_OF_TOTAL = 1e-6
# a mask row may differ from the oracle's only where the fp64 scores decide it
# by less than this share of the row total
TIE_TOL = 1e-4


@pytest.fixture(scope="module")
def dev():
    return gpu_device()


def run(dev, Q, K, m, tau=0.9, max_units=None, fill=0, check=True):
    B, S, Hq, _ = Q.shape
    Hkv = K.shape[2]
    nB = (S + 127) // 128
    if max_units is None:
        max_units = B * Hkv
    ws = ea.xa_workspace(B, S, Hq, Hkv, max_units, device=dev)
    bm = torch.full((B, Hkv, nB, nB), fill, dtype=torch.uint8, device=dev)
    bm, sc = ea.ea_xa_estimate(Q.to(dev), K.to(dev), torch.as_tensor(m, dtype=torch.uint8).to(dev),
                               threshold=tau, max_units=max_units, block_mask=bm,
                               want_scores=True, workspace=ws)
    torch.cuda.synchronize()
    if check:
        check_no_device_error(ws)
    return bm.cpu().numpy(), sc.cpu().numpy(), ws


def check_scores(sc, W, rows, what):
    for qb in rows:
        total = W[qb, :qb + 1].sum()
        err = np.abs(sc[qb, :qb + 1] - W[qb, :qb + 1])
        lim = SCORE_RTOL * np.abs(W[qb, :qb + 1]) + SCORE_ATOL_OF_TOTAL * total
        assert (err <= lim).all(), "%s row %d: max score error %g" % (what, qb, err.max())
        assert (sc[qb, qb + 1:] == 0).all(), what + ": scores above the diagonal"


def near_tie(row, sel, tau):
    """Is `sel` (bool over kb <= qb) a valid threshold run of `row` up to TIE_TOL?
    Valid: every kept block (but the forced diagonal) scores at least every
    dropped one, the kept mass reaches tau * total, and dropping the lowest kept
    block (not the diagonal) would fall short of it, each within the tolerance."""
    total = row.sum()
    tol = TIE_TOL * total
    qb = len(row) - 1
    free = sel.copy()
    free[qb] = False
    kept, dropped = row[free], row[~sel]
    if kept.size and dropped.size and dropped.max() > kept.min() + tol:
        return False
    mass = row[sel].sum()
    if mass < tau * total - tol:
        return False
    if kept.size and row[free].sum() - kept.min() >= tau * total + tol:
        return False
    return True


def check_masks(mask, sc, W, tau, rows, what):
    """mask: kernel's uint8 [nB, nB]; sc: kernel's scores; W: oracle scores."""
    nB = W.shape[0]
    assert (np.triu(mask, 1) == 0).all(), what + ": kept blocks above the diagonal"
    assert (np.diagonal(mask)[rows] == 1).all(), what + ": diagonal not kept"
    # the selection rule, bit for bit, on the kernel's own scores
    rows = list(rows)
    own = oracle.xa_select(np.tril(sc.astype(np.float64)), tau, qb_rows=rows)
    ref = oracle.xa_select(W, tau, qb_rows=rows)
    n_diff = 0
    for qb in rows:
        if not np.array_equal(mask[qb], own[qb]):
            row = sc[qb, :qb + 1].astype(np.float64)
            assert near_tie(row, mask[qb, :qb + 1].astype(bool), tau), \
                "%s row %d: selection differs from the rule on the kernel's scores" % (what, qb)
        if not np.array_equal(mask[qb], ref[qb]):
            n_diff += 1
            assert near_tie(W[qb, :qb + 1], mask[qb, :qb + 1].astype(bool), tau), \
                "%s row %d: kernel's selection is not a valid run of the oracle's scores" % (what, qb)
    return n_diff


def oracle_all(Q, K, m, tau):
    W, M = oracle.xa_estimate(Q, K, m, stride=16, tau=tau)
    return W, M


@pytest.mark.parametrize("S,Hq,Hkv,planted", [
    (1024, 4, 2, True),       # one cell-row tile, one key tile
    (4800, 8, 2, True),       # 300 cell rows: 3 row tiles (last ragged), 2 key tiles
    (4800, 8, 2, False),      # plain N(0, 1): many near-ties
    (8192, 4, 1, True),       # 512 cell rows: 4 row tiles, 2 key tiles
    (2048, 2, 2, True),       # one query head per KV head
    (3200, 6, 2, True),       # three query heads per KV head (pair + single)
])
def test_scores_and_masks_match_oracle(dev, S, Hq, Hkv, planted):
    if planted:
        Q, K = wl.xa_planted_qk(1, S, Hq, Hkv, 128, seed=S % 97)
    else:
        Q, K, _ = wl.qkv(1, S, Hq, Hkv, 128, seed=5)
    m = np.full((1, Hkv), BLOCK, dtype=np.uint8)
    if Hkv > 1:
        m[0, 0] = SSA if S == 4800 else BLOCK
    bm, sc, _ = run(dev, Q, K, m)
    W, _ = oracle_all(Q, K, m, 0.9)
    nB = W.shape[2]
    for h in range(Hkv):
        if m[0, h] != BLOCK:
            assert (bm[0, h] == 0).all() and (sc[0, h] == 0).all()
            continue
        what = "S=%d Hq=%d Hkv=%d h=%d" % (S, Hq, Hkv, h)
        check_scores(sc[0, h], W[0, h], range(nB), what)
        n_diff = check_masks(bm[0, h], sc[0, h], W[0, h], 0.9, range(nB), what)
        if planted:
            assert n_diff <= max(1, nB // 20), "%s: %d rows differ from the oracle" % (what, n_diff)


def test_several_batch_rows_and_untouched_heads(dev):
    B, S, Hq, Hkv = 2, 2048, 4, 2
    Q, K = wl.xa_planted_qk(B, S, Hq, Hkv, 128, seed=3)
    m = np.array([[BLOCK, FULL], [SSA, BLOCK]], dtype=np.uint8)
    bm, sc, _ = run(dev, Q, K, m, fill=7)
    W, _ = oracle_all(Q, K, m, 0.9)
    nB = S // 128
    assert (bm[0, 1] == 7).all() and (bm[1, 0] == 7).all(), "rows of non-BLOCK heads were written"
    for b, h in ((0, 0), (1, 1)):
        check_scores(sc[b, h], W[b, h], range(nB), "b=%d h=%d" % (b, h))
        check_masks(bm[b, h], sc[b, h], W[b, h], 0.9, range(nB), "b=%d h=%d" % (b, h))


@pytest.mark.parametrize("tau", [0.0, 0.5, 1.0, 2.0])
def test_threshold_edges(dev, tau):
    S = 2048
    Q, K = wl.xa_planted_qk(1, S, 4, 1, 128, seed=11)
    m = np.array([[BLOCK]], dtype=np.uint8)
    bm, sc, _ = run(dev, Q, K, m, tau=tau)
    nB = S // 128
    mask = bm[0, 0]
    if tau == 0.0:
        assert np.array_equal(mask, np.eye(nB, dtype=np.uint8))
    elif tau >= 1.0:
        expect = (np.tril(sc[0, 0]) > 0).astype(np.uint8)
        np.fill_diagonal(expect, 1)
        assert np.array_equal(mask, expect)
    else:
        W, _ = oracle_all(Q, K, m, tau)
        check_masks(mask, sc[0, 0], W[0, 0], tau, range(nB), "tau=%g" % tau)


def test_too_many_block_heads_is_reported(dev):
    S = 1024
    Q, K = wl.xa_planted_qk(1, S, 4, 2, 128, seed=13)
    m = np.array([[BLOCK, BLOCK]], dtype=np.uint8)
    bm, sc, ws = run(dev, Q, K, m, max_units=1, fill=5, check=False)
    assert ea.ea_check_errors(ws) == 6   # EA_ERR_DEVICE_CHECK
    assert (bm[0, 1] == 5).all(), "the unit beyond max_units was written"
    W, _ = oracle_all(Q, K, np.array([[BLOCK, FULL]], dtype=np.uint8), 0.9)
    check_scores(sc[0, 0], W[0, 0], range(S // 128), "first unit")
    # the workspace is usable again after the error word was read
    run(dev, Q, K, np.array([[BLOCK, FULL]], dtype=np.uint8))


def test_repeat_calls_are_bitwise_identical(dev):
    S = 4800
    Q, K = wl.xa_planted_qk(1, S, 8, 2, 128, seed=17)
    m = np.array([[BLOCK, BLOCK]], dtype=np.uint8)
    a = run(dev, Q, K, m)
    b = run(dev, Q, K, m)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_xa_ssa_256k_sampled_rows(dev):
    """The 256K XA-SSA layer (2 BLOCK + 6 SSA KV heads, 32 query heads): sampled
    query-block rows against the oracle; row totals and the diagonal on every row."""
    cfg = wl.XA_SSA_256K
    Q, K = wl.xa_planted_qk(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.d, seed=0, device=dev)
    _, m = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads, cfg.fa_impl, cfg.sa_impl)
    blocks = [h for h in range(cfg.Hkv) if int(m[0, h]) == BLOCK]
    bm, sc, _ = run(dev, Q, K, m.numpy(), max_units=len(blocks))
    nB = cfg.S // 128
    g = cfg.Hq // cfg.Hkv
    Qc, Kc = Q.cpu(), K.cpu()
    del Q, K
    for h in blocks:
        tot = np.tril(sc[0, h]).sum(axis=1)
        np.testing.assert_allclose(tot, g * 8, rtol=1e-3)
        assert (np.diagonal(bm[0, h]) == 1).all() and (np.triu(bm[0, h], 1) == 0).all()
        rows = [0, 1, 333, 1024, nB - 1]
        W = oracle.xa_block_scores(Qc, Kc, 0, h, stride=16, qb_rows=rows)
        check_scores(sc[0, h], W, rows, "256K h=%d" % h)
        check_masks(bm[0, h], sc[0, h], W, 0.9, rows, "256K h=%d" % h)


def test_maximum_sequence_sampled_rows(dev):
    """S = 2^21 (the largest supported length), one KV head read by two query
    heads: sampled query-block rows against the oracle, the row totals and the
    diagonal on every row."""
    S, Hq, Hkv = 1 << 21, 2, 1
    Q, K = wl.xa_planted_qk(1, S, Hq, Hkv, 128, seed=23, device=dev)
    m = np.array([[BLOCK]], dtype=np.uint8)
    bm, sc, _ = run(dev, Q, K, m, max_units=1)
    nB = S // 128
    tot = np.tril(sc[0, 0]).sum(axis=1)
    np.testing.assert_allclose(tot, 2 * 8, rtol=1e-3)
    assert (np.diagonal(bm[0, 0]) == 1).all() and (np.triu(bm[0, 0], 1) == 0).all()
    rows = [0, 5, nB - 1]
    W = oracle.xa_block_scores(Q.cpu(), K.cpu(), 0, 0, stride=16, qb_rows=rows)
    check_scores(sc[0, 0], W, rows, "S=2^21")
    check_masks(bm[0, 0], sc[0, 0], W, 0.9, rows, "S=2^21")


@pytest.mark.parametrize("S", [16, 144, 400])
def test_short_sequences(dev, S):
    """S = 16 (one cell, one block), 144 (a last block of one cell), 400."""
    Q, K = wl.xa_planted_qk(2, S, 4, 2, 128, seed=S)
    m = np.array([[BLOCK, BLOCK], [SSA, BLOCK]], dtype=np.uint8)
    bm, sc, _ = run(dev, Q, K, m)
    W, _ = oracle_all(Q, K, m, 0.9)
    nB = (S + 127) // 128
    for b, h in ((0, 0), (0, 1), (1, 1)):
        check_scores(sc[b, h], W[b, h], range(nB), "S=%d b=%d h=%d" % (S, b, h))
        check_masks(bm[b, h], sc[b, h], W[b, h], 0.9, range(nB), "S=%d b=%d h=%d" % (S, b, h))
    assert (bm[1, 0] == 0).all()
