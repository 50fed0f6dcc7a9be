"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each check comes from outside the oracle's own formula: a library routine
(torch SDPA / logsumexp in fp64 on the CPU), a closed form, a special case that
reduces to a simpler problem, or a hand-computed value stored under
tests/golden/.  Chosen so that a dropped term, a wrong sign or index or a
transposed operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_head_attention_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FULL, SSA, BLOCK = oracle.FULL, oracle.SSA, oracle.BLOCK


def _f64(t):
    return t.to(torch.float64)


def _sdpa_reference(Q, K, V, mask_fn, scale):
    """Library check: SDPA in fp64 with a dense boolean mask built per KV head."""
    B, S, Hq, d = Q.shape
    Hkv = K.shape[2]
    g = Hq // Hkv
    O = torch.zeros(B, S, Hq, d, dtype=torch.float64)
    LSE = torch.zeros(B, Hq, S, dtype=torch.float64)
    for b in range(B):
        for qh in range(Hq):
            h = qh // g
            allow = mask_fn(b, h)                               # [S, S] bool
            q = _f64(Q[b, :, qh])
            k = _f64(K[b, :, h])
            v = _f64(V[b, :, h])
            o = torch.nn.functional.scaled_dot_product_attention(
                q[None, None], k[None, None], v[None, None], attn_mask=allow[None, None],
                scale=scale)[0, 0]
            s = (q @ k.T) * scale
            lse = torch.logsumexp(s.masked_fill(~allow, -math.inf), dim=-1)
            O[b, :, qh] = o
            LSE[b, qh] = lse
    return O.numpy(), LSE.numpy()


def _ssa_dense(S, sink, window):
    """SSA mask as a band (tril minus a shifted tril) plus sink columns."""
    ones = torch.ones(S, S, dtype=torch.bool)
    band = torch.tril(ones) & ~torch.tril(ones, diagonal=-window)
    sinkcols = torch.zeros(S, S, dtype=torch.bool)
    sinkcols[:, :sink] = True
    return band | (sinkcols & torch.tril(ones))


def _block_dense(bm_head, S, T):
    """BLOCK mask by expanding the block matrix with kron, then causal."""
    e = np.kron(bm_head.astype(bool), np.ones((T, T), dtype=bool))[:S, :S]
    return torch.from_numpy(e) & torch.tril(torch.ones(S, S, dtype=torch.bool))


@pytest.mark.parametrize("S,sink,window", [(70, 5, 9), (37, 0, 1), (64, 16, 16), (50, 3, 200)])
def test_prefill_matches_sdpa_fp64_fa_ssa(S, sink, window):
    B, Hq, Hkv, d = 2, 4, 2, 16
    Q, K, V = wl.qkv(B, S, Hq, Hkv, d, seed=7)
    modes = np.array([[FULL, SSA], [SSA, FULL]], dtype=np.uint8)
    scale = 1.0 / math.sqrt(d)
    O, LSE = oracle.prefill_full(Q, K, V, modes, sink=sink, window=window, T=16, scale=scale)

    def mask_fn(b, h):
        if modes[b, h] == FULL:
            return torch.tril(torch.ones(S, S, dtype=torch.bool))
        return _ssa_dense(S, sink, window)

    Oref, LSEref = _sdpa_reference(Q, K, V, mask_fn, scale)
    np.testing.assert_allclose(O, Oref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, LSEref, atol=1e-12, rtol=0)


def test_prefill_matches_sdpa_fp64_block():
    B, S, Hq, Hkv, d, T = 1, 75, 4, 2, 16, 16
    Q, K, V = wl.qkv(B, S, Hq, Hkv, d, seed=3)
    bm = wl.block_mask(B, Hkv, S, density=0.4, seed=5, T=T).numpy()
    bm[0, 1, 3, 3] = 0          # drop one diagonal block: its rows keep fewer keys
    modes = np.array([[BLOCK, BLOCK]], dtype=np.uint8)
    scale = 0.3
    O, LSE = oracle.prefill_full(Q, K, V, modes, block_mask=bm, T=T, scale=scale)
    Oref, LSEref = _sdpa_reference(Q, K, V, lambda b, h: _block_dense(bm[b, h], S, T), scale)
    np.testing.assert_allclose(O, Oref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, LSEref, atol=1e-12, rtol=0)


def test_softmax_rows_are_probabilities_and_masked_keys_get_zero():
    # V = identity rows: O_i is then the softmax row p_i itself.
    S, d, sink, window = 16, 16, 2, 5
    Q, K, _ = wl.qkv(1, S, 2, 1, d, seed=11)
    V = torch.eye(S, d, dtype=torch.bfloat16)[None, :, None, :]
    for mode in (FULL, SSA):
        O, LSE = oracle.prefill_full(Q, K, V, np.array([[mode]], np.uint8), sink=sink,
                                     window=window, T=16)
        P = O[0, :, 0, :S]                                   # [i, j]
        np.testing.assert_allclose(P.sum(-1), 1.0, atol=1e-12)
        for i in range(S):
            for j in range(S):
                kept = j <= i and (mode == FULL or j < sink or i - j < window)
                if not kept:
                    assert P[i, j] == 0.0
                else:
                    s = float(_f64(Q[0, i, 0]) @ _f64(K[0, j, 0])) / math.sqrt(d)
                    assert abs(P[i, j] - math.exp(s - LSE[0, 0, i])) < 1e-12


@pytest.mark.parametrize("sink,window", [(0, 1), (3, 4), (7, 1), (2, 30)])
def test_zero_query_gives_mean_of_kept_values(sink, window):
    # Q = 0: every kept score is 0, O_i = mean of kept V rows, LSE_i = ln(count).
    # The kept set is written as two index ranges, not as the mask predicate.
    S, d = 40, 8
    _, K, V = wl.qkv(1, S, 1, 1, d, seed=2)
    Q = torch.zeros(1, S, 1, d, dtype=torch.bfloat16)
    O, LSE = oracle.prefill_full(Q, K, V, np.array([[SSA]], np.uint8), sink=sink,
                                 window=window, T=8)
    v = _f64(V[0, :, 0]).numpy()
    csum = np.concatenate([np.zeros((1, d)), np.cumsum(v, axis=0)])
    for i in range(S):
        lo = max(0, i - window + 1)
        sink_end = min(sink, lo)                  # sink keys below the window
        count = (i + 1 - lo) + sink_end
        closed = min(i + 1, window) + max(0, min(sink, i + 1 - window))
        assert count == closed
        mean = (csum[i + 1] - csum[lo] + csum[sink_end]) / count
        np.testing.assert_allclose(O[0, i, 0], mean, atol=1e-12)
        assert abs(LSE[0, 0, i] - math.log(count)) < 1e-12


def test_constant_values_and_single_key():
    S, d = 33, 8
    Q, K, _ = wl.qkv(1, S, 2, 1, d, seed=4)
    c = torch.linspace(-2, 2, d).to(torch.bfloat16)
    V = c.expand(1, S, 1, d).contiguous()
    O, _ = oracle.prefill_full(Q, K, V, np.array([[FULL]], np.uint8))
    np.testing.assert_allclose(O, np.broadcast_to(_f64(c).numpy(), O.shape), atol=1e-12)
    # sink 0, window 1: only the diagonal key -> O_i = V_i, LSE_i = its score
    _, _, V2 = wl.qkv(1, S, 2, 1, d, seed=5)
    O, LSE = oracle.prefill_full(Q, K, V2, np.array([[SSA]], np.uint8), sink=0, window=1)
    for qh in range(2):
        np.testing.assert_array_equal(O[0, :, qh], _f64(V2[0, :, 0]).numpy())
        s = (_f64(Q[0, :, qh]) * _f64(K[0, :, 0])).sum(-1) / math.sqrt(d)
        np.testing.assert_allclose(LSE[0, qh], s.numpy(), atol=1e-12)


def test_reductions_to_full_attention():
    B, S, Hq, Hkv, d, T = 1, 96, 4, 2, 16, 32
    Q, K, V = wl.qkv(B, S, Hq, Hkv, d, seed=9)
    full = np.array([[FULL, FULL]], np.uint8)
    O_fa, L_fa = oracle.prefill_full(Q, K, V, full, T=T)
    # SSA with sink + window >= S keeps every causal pair
    O_s, L_s = oracle.prefill_full(Q, K, V, np.array([[SSA, SSA]], np.uint8), sink=40,
                                   window=S - 40, T=T)
    np.testing.assert_array_equal(O_s, O_fa)
    np.testing.assert_array_equal(L_s, L_fa)
    # all-ones block mask is FA
    nB = S // T
    ones = np.ones((B, Hkv, nB, nB), np.uint8)
    O_b, L_b = oracle.prefill_full(Q, K, V, np.array([[BLOCK, BLOCK]], np.uint8),
                                   block_mask=ones, T=T)
    np.testing.assert_array_equal(O_b, O_fa)
    np.testing.assert_array_equal(L_b, L_fa)


def test_diagonal_block_mask_is_blockwise_causal_attention():
    # Only diagonal blocks kept: each block of T queries is FA over its own T keys,
    # i.e. FA run separately on each chunk.
    B, S, Hq, Hkv, d, T = 1, 80, 2, 1, 8, 16
    Q, K, V = wl.qkv(B, S, Hq, Hkv, d, seed=13)
    nB = S // T
    diag = np.eye(nB, dtype=np.uint8)[None, None]
    O_b, L_b = oracle.prefill_full(Q, K, V, np.array([[BLOCK]], np.uint8), block_mask=diag, T=T)
    for c in range(nB):
        sl = slice(c * T, (c + 1) * T)
        O_c, L_c = oracle.prefill_full(Q[:, sl].contiguous(), K[:, sl].contiguous(),
                                       V[:, sl].contiguous(), np.array([[FULL]], np.uint8), T=T)
        np.testing.assert_array_equal(O_b[:, sl], O_c)
        np.testing.assert_array_equal(L_b[:, :, sl], L_c)


def test_empty_row_is_zero_with_minus_inf_lse():
    B, S, Hq, Hkv, d, T = 1, 32, 1, 1, 8, 16
    Q, K, V = wl.qkv(B, S, Hq, Hkv, d, seed=1)
    bm = np.array([[[[1, 0], [0, 0]]]], np.uint8)          # second query block keeps nothing
    O, LSE = oracle.prefill_full(Q, K, V, np.array([[BLOCK]], np.uint8), block_mask=bm, T=T)
    assert np.all(O[0, 16:] == 0.0)
    assert np.all(np.isneginf(LSE[0, 0, 16:]))
    assert np.all(np.isfinite(LSE[0, 0, :16]))


def test_gqa_grouping_and_concatenation():
    # query head qh reads KV head qh // (Hq/Hkv) and lands in its own slice of O:
    # permuting the KV heads permutes contiguous groups of query heads.
    B, S, Hq, Hkv, d = 1, 24, 6, 3, 8
    Q, K, V = wl.qkv(B, S, Hq, Hkv, d, seed=21)
    modes = np.array([[FULL, SSA, FULL]], np.uint8)
    O, _ = oracle.prefill_full(Q, K, V, modes, sink=2, window=3)
    for qh in range(Hq):
        h = qh // 2
        Oh, _ = oracle.prefill_full(Q[:, :, qh:qh + 1].contiguous(), K[:, :, h:h + 1].contiguous(),
                                    V[:, :, h:h + 1].contiguous(),
                                    np.array([[modes[0, h]]], np.uint8), sink=2, window=3)
        np.testing.assert_array_equal(O[:, :, qh], Oh[:, :, 0])


@pytest.mark.parametrize("mode", [FULL, SSA, BLOCK])
def test_decode_is_last_prefill_row(mode):
    B, Hq, Hkv, d, Lmax, sink, window, T = 3, 4, 2, 16, 50, 3, 7, 8
    cfg = wl.DecodeConfig("t", B=B, Hq=Hq, Hkv=Hkv, d=d, L=Lmax, sink=sink, window=window)
    seqlens = [50, 1, 23]
    q, Kc, Vc, sl = wl.decode_inputs(cfg, seqlens=seqlens)
    modes = np.full((B, Hkv), mode, np.uint8)
    nB = (Lmax + T - 1) // T
    bm = wl.block_mask(B, Hkv, Lmax, density=0.4, seed=5, T=T).numpy() if mode == BLOCK else None
    O, LSE = oracle.decode(q, Kc, Vc, sl, modes, sink=sink, window=window, block_mask=bm, T=T)
    for b, L in enumerate(seqlens):
        Qp = torch.zeros(1, L, Hq, d, dtype=torch.bfloat16)
        Qp[0, L - 1] = q[b]
        rows = np.array([[0, qh, L - 1] for qh in range(Hq)])
        nBL = (L + T - 1) // T
        bmL = None if bm is None else np.ascontiguousarray(bm[b:b + 1, :, :nBL, :nBL])
        Op, Lp = oracle.prefill_rows(Qp, Kc[b:b + 1, :L].contiguous(), Vc[b:b + 1, :L].contiguous(),
                                     modes[b:b + 1], rows, sink=sink, window=window, block_mask=bmL,
                                     T=T)
        np.testing.assert_array_equal(O[b], Op)
        np.testing.assert_array_equal(LSE[b], Lp)
        # library check on the same row
        g = Hq // Hkv
        for qh in range(Hq):
            k = _f64(Kc[b, :L, qh // g])
            s = (k @ _f64(q[b, qh])) / math.sqrt(d)
            j = torch.arange(L)
            if mode == FULL:
                keep = torch.ones(L, dtype=torch.bool)
            elif mode == SSA:
                keep = (j < sink) | ((L - 1) - j < window)
            else:
                keep = torch.as_tensor(bm[b, qh // g, (L - 1) // T][j // T] != 0)
            p = torch.softmax(s.masked_fill(~keep, -math.inf), 0)
            np.testing.assert_allclose(O[b, qh], (p @ _f64(Vc[b, :L, qh // g])).numpy(), atol=1e-12)


def test_decode_block_heads_need_a_mask_and_empty_rows_are_zero():
    cfg = wl.DecodeConfig("t", B=1, Hq=2, Hkv=1, d=8, L=40, sink=1, window=2)
    q, Kc, Vc, sl = wl.decode_inputs(cfg)
    with pytest.raises(ValueError):
        oracle.decode(q, Kc, Vc, sl, np.array([[BLOCK]], np.uint8))
    bm = np.zeros((1, 1, 5, 5), np.uint8)            # row (L - 1) / 8 keeps nothing
    O, LSE = oracle.decode(q, Kc, Vc, sl, np.array([[BLOCK]], np.uint8), block_mask=bm, T=8)
    assert (O == 0).all() and np.isneginf(LSE).all()


@pytest.mark.parametrize("S,T,sink,window", [(70, 16, 5, 9), (128, 16, 16, 17), (100, 32, 0, 1),
                                              (300, 64, 70, 130)])
def test_visited_tiles_closed_form(S, T, sink, window):
    B, Hkv = 1, 3
    nB = (S + T - 1) // T
    bm = wl.block_mask(B, Hkv, S, density=0.3, seed=S, T=T).numpy()
    bm[0, 2, nB - 1, nB - 1] = 0
    modes = np.array([[FULL, SSA, BLOCK]], np.uint8)
    vis = oracle.visited(B, S, Hkv, modes, sink=sink, window=window, block_mask=bm, T=T)
    qb = np.arange(nB)[:, None]
    kb = np.arange(nB)[None, :]
    fa = kb <= qb
    # SSA: a sink key in the tile, the window reaching the tile's last key, or the diagonal
    ssa = fa & ((kb * T < sink) | ((qb - kb - 1) * T + 1 < window) | (kb == qb))
    blk = fa & (bm[0, 2] != 0)
    np.testing.assert_array_equal(vis[0, 0], fa.astype(np.uint8))
    np.testing.assert_array_equal(vis[0, 1], ssa.astype(np.uint8))
    np.testing.assert_array_equal(vis[0, 2], blk.astype(np.uint8))


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden("router_hand_examples.json")["cases"], ids=lambda c: c["name"])
def test_router_hand_examples(case):
    K = torch.tensor(case["K"], dtype=torch.float32).to(torch.bfloat16)[None]  # [1, S, H, d]
    assert K.shape[1] == case["S"]
    Ws = [np.array(w, np.float32) for w in case["W"]]
    bs = [np.array(b, np.float32) for b in case["b"]]
    r, m, logits, pooled = oracle.route(K, Ws, bs, pool_head=case["pool_head"],
                                        pool_tail=case["pool_tail"], fa_impl=FULL, sa_impl=SSA)
    np.testing.assert_array_equal(pooled[0], np.array(case["pooled"], np.float64))
    np.testing.assert_array_equal(logits[0], np.array(case["logits"], np.float64))
    np.testing.assert_array_equal(r[0], np.array(case["r"], np.uint8))
    np.testing.assert_array_equal(m[0], np.where(np.array(case["r"]) == 1, SSA, FULL))
    # XA-SSA policy: r = 0 executes as BLOCK
    _, m2, _, _ = oracle.route(K, Ws, bs, pool_head=case["pool_head"], pool_tail=case["pool_tail"],
                               fa_impl=BLOCK, sa_impl=SSA)
    np.testing.assert_array_equal(m2[0], np.where(np.array(case["r"]) == 1, SSA, BLOCK))


def _mlp_variant(x, Ws, bs, transpose_layer=None, trailing_relu=False):
    # dense layers on a pooled vector with one planted mistake: weights of one
    # layer read as W[c][o] (the flat [out][in] array indexed the other way) or
    # a ReLU after the last layer
    for li, (W, b) in enumerate(zip(Ws, bs)):
        nout, nin = W.shape
        flat = W.reshape(-1)
        y = []
        for o in range(nout):
            acc = float(b[o])
            for c in range(nin):
                w = flat[c * nout + o] if li == transpose_layer else flat[o * nin + c]
                acc += float(w) * x[c]
            y.append(acc)
        if li + 1 < len(Ws) or trailing_relu:
            y = [v if v > 0 else 0.0 for v in y]
        x = y
    return x


@pytest.mark.parametrize("case", [c for c in _golden("router_hand_examples.json")["cases"]
                                  if "_catches" in c], ids=lambda c: c["name"])
def test_router_hand_examples_catch_planted_mistakes(case):
    """The non-square, asymmetric cases are chosen so that each plausible slip
    in the dense-layer evaluation changes the expected result: a ReLU after the
    last layer (negative logits become 0 and the SA head ties, so r flips to FA),
    the second layer's weights read transposed (r flips), the first layer's read
    transposed (the logits change).  Evaluated here on the hand-pooled vectors,
    so each mistake is shown to fail the oracle pin above."""
    Ws = [np.array(w, np.float64) for w in case["W"]]
    bs = [np.array(b, np.float64) for b in case["b"]]
    want = np.array(case["logits"], np.float64)
    r_want = np.array(case["r"])
    flips = {"trailing": False, "t1": False, "t0": False}
    for h, x in enumerate(case["pooled"]):
        ok = _mlp_variant(list(map(float, x)), Ws, bs)
        np.testing.assert_array_equal(ok, want[h])   # the hand working is self-consistent
        for key, kw in (("trailing", dict(trailing_relu=True)), ("t1", dict(transpose_layer=1)),
                        ("t0", dict(transpose_layer=0))):
            z = _mlp_variant(list(map(float, x)), Ws, bs, **kw)
            assert not np.array_equal(z, want[h]) or key == "t0"
            flips[key] |= int(z[1] > z[0]) != r_want[h]
    # across the heads: each planted mistake changes some logit, the first two flip a decision
    assert flips["trailing"] and flips["t1"]
    assert any(not np.array_equal(_mlp_variant(list(map(float, x)), Ws, bs, transpose_layer=0), want[h])
               for h, x in enumerate(case["pooled"]))


def test_router_pools_only_boundary_tokens():
    # changing a middle token leaves the decision inputs unchanged; changing a
    # boundary token moves the pooled mean by exactly delta / 200
    B, S, Hkv, d = 1, 500, 2, 16
    _, K, _ = wl.qkv(B, S, 2, Hkv, d, seed=17)
    W, b = wl.router_weights(0, d=d, hidden=8)
    _, _, lg0, p0 = oracle.route(K, W, b)
    K2 = K.clone()
    K2[0, 250] += 4.0
    _, _, lg1, p1 = oracle.route(K2, W, b)
    np.testing.assert_array_equal(p0, p1)
    np.testing.assert_array_equal(lg0, lg1)
    K3 = K.clone()
    K3[0, 450, 1, 3] = K[0, 450, 1, 3].float() + 8.0
    _, _, _, p3 = oracle.route(K3, W, b)
    delta = float(K3[0, 450, 1, 3]) - float(K[0, 450, 1, 3])
    assert abs((p3 - p0)[0, 1, 3] - delta / 200.0) < 1e-12
    assert np.count_nonzero(p3 - p0) == 1


@pytest.mark.parametrize("case", _golden("sparsity_ratio_hand_examples.json")["cases"],
                         ids=lambda c: c["name"])
def test_sparsity_ratio_hand_examples(case):
    bms = np.array(case["block_masks"], np.uint8) if "block_masks" in case else None
    msr, esr, kept = oracle.sparsity_ratios(np.array(case["r"], np.uint8),
                                            np.array(case["m"], np.uint8), case["S"],
                                            sink=case["sink"], window=case["window"],
                                            block_masks=bms, T=case["T"])
    np.testing.assert_array_equal(kept, np.array(case["kept"]))
    assert msr == case["msr"]
    assert esr == case["esr_num"] / case["esr_den"]


@pytest.mark.parametrize("S,sink,window", [(1024, 64, 256), (300, 0, 300), (257, 128, 100),
                                           (999, 5, 1)])
def test_ssa_rho_closed_form(S, sink, window):
    _, esr, kept = oracle.sparsity_ratios(np.array([[1]], np.uint8), np.array([[SSA]], np.uint8),
                                          S, sink=sink, window=window)
    closed = sum(min(i + 1, window) + max(0, min(sink, i + 1 - window)) for i in range(S))
    assert kept[0, 0] == closed
    causal = S * (S + 1) // 2
    assert esr == (causal - closed) / causal


def test_tiny_config_rho_matches_hand_count():
    # Tiny workload (S=1024, sink 64, window 256): 229504 window + 47136 sink pairs kept,
    # so the SSA head prunes 47.29% of the 524800 causal pairs
    _, esr, kept = oracle.sparsity_ratios(np.array([[1]], np.uint8), np.array([[SSA]], np.uint8),
                                          1024, sink=64, window=256)
    assert kept[0, 0] == 276640
    assert round(esr, 4) == 0.4729
