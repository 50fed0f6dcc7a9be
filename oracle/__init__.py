"""fp64 CPU oracle for Elastic Attention's hybrid-head attention path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code with
the CUDA library (``sparse_head_attention_gb300``) and never imports it; the two
meet only through the seeded input generators in
``sparse_head_attention_gb300.workloads``, which hold none of the method's
arithmetic.

Every function is a thin ctypes marshaller around ``ea_oracle.c``; the
arithmetic, and the citation of the passage each function follows, is there.
Inputs are bf16 tensors on the CPU (torch) or uint16 numpy arrays of bf16 bit
patterns; outputs are float64 numpy arrays.

Parity status of each function (what pins it, see ``tests/test_oracle_pins.py``):
  prefill_rows   - pinned: library SDPA in fp64 with a dense mask, closed forms
                   (Q = 0, constant V, single kept key), SSA/BLOCK reductions to FA
                   and to block-local causal attention.
  decode         - pinned: equals the prefill oracle's last row (FA, SSA and BLOCK
                   with the same block mask); library SDPA.
  visited        - pinned: closed-form tile sets for FA/SSA, block mask for BLOCK.
  route          - pinned: hand-computed examples (tests/golden), exact in binary:
                   symmetric and square layers, plus non-square asymmetric layers
                   with negative final logits, chosen so that a transposed weight
                   read or an activation after the last layer changes the result.
  sparsity_ratios- pinned: hand-counted masks (tests/golden), closed form for SSA.
  xa_block_scores- pinned: stride 1 equals block sums of library softmax attention
                   probabilities; a single nonzero query/key pair lights exactly the
                   antidiagonal cell; Q = 0 gives the closed-form uniform scores; row
                   totals equal the number of softmax rows.  The scoring itself is a
                   reading (the pages name antidiagonal scoring without defining it).
  xa_select      - pinned: tau = 0 keeps only the diagonal, tau = 1 keeps every block
                   with mass, a planted dominant block is chosen, brute force over all
                   subsets on small rows.
"""
import ctypes
import math
import os

import numpy as np

from . import build as _build

FULL, SSA, BLOCK = 0, 1, 2

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.ea_oracle_prefill_rows.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, f64,
                                             P, i32, i32, P, i32, i64, P, P, P]
        L.ea_oracle_decode.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, f64,
                                       P, i32, i32, P, i32, P, P]
        L.ea_oracle_visited.argtypes = [i32, i32, i32, P, i32, i32, P, i32, i32, i32, P]
        L.ea_oracle_route.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32, P, P, P,
                                      i32, i32, P, P, P, P]
        L.ea_oracle_sparsity_ratios.argtypes = [P, P, i32, i32, i32, i32, i32, P, i32,
                                                P, P, P]
        L.ea_oracle_xa_block_scores.argtypes = [P, P, P, P, i32, i32, i32, i32, f64, i32, i32,
                                                i32, i32, P, P]
        L.ea_oracle_xa_select.argtypes = [P, i64, f64, P, P]
        for f in (L.ea_oracle_prefill_rows, L.ea_oracle_decode, L.ea_oracle_visited,
                  L.ea_oracle_route, L.ea_oracle_sparsity_ratios, L.ea_oracle_xa_block_scores,
                  L.ea_oracle_xa_select):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def _bf16_bits(t):
    """(uint16 array of bf16 bit patterns, element strides) of a tensor/array."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        a = t
    else:  # torch tensor
        import torch
        assert t.dtype == torch.bfloat16, t.dtype
        a = t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    strides = np.array([s // a.itemsize for s in a.strides], dtype=np.int64)
    return a, strides


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _u8(a, n=None):
    if a is None:
        return None
    if not isinstance(a, np.ndarray):
        a = a.detach().cpu().numpy()
    a = np.ascontiguousarray(a, dtype=np.uint8)
    if n is not None:
        assert a.size == n, (a.size, n)
    return a


def prefill_rows(Q, K, V, modes, rows, *, sink=0, window=1, block_mask=None, T=128,
                 scale=None):
    """O (float64 [n, d]) and LSE (float64 [n]) of the hybrid-head prefill for the
    requested rows (int array [n, 3] of (b, q head, query index)).

    Q: bf16 [B, S, Hq, d]; K, V: bf16 [B, S, Hkv, d] (same strides);
    modes: uint8 [B, Hkv] in {FULL, SSA, BLOCK}; block_mask: uint8
    [B, Hkv, nB, nB] when any mode is BLOCK."""
    q, qs = _bf16_bits(Q)
    k, ks = _bf16_bits(K)
    v, vs = _bf16_bits(V)
    assert (ks == vs).all()
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    m = _u8(modes, B * Hkv)
    bm = _u8(block_mask)
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
    n = rows.shape[0]
    O = np.zeros((n, d), dtype=np.float64)
    LSE = np.zeros((n,), dtype=np.float64)
    rc = lib().ea_oracle_prefill_rows(_ptr(q), _ptr(qs), _ptr(k), _ptr(v), _ptr(ks),
                                      B, S, Hq, Hkv, d, scale, _ptr(m), sink, window,
                                      _ptr(bm), T, n, _ptr(rows), _ptr(O), _ptr(LSE))
    if rc != 0:
        raise ValueError("oracle prefill_rows rejected its arguments (rc=%d)" % rc)
    return O, LSE


def prefill_full(Q, K, V, modes, **kw):
    """Every row: O float64 [B, S, Hq, d], LSE float64 [B, Hq, S] (small cases)."""
    B, S, Hq, d = Q.shape
    b, s, h = np.meshgrid(np.arange(B), np.arange(S), np.arange(Hq), indexing="ij")
    rows = np.stack([b.ravel(), h.ravel(), s.ravel()], axis=1)
    O, LSE = prefill_rows(Q, K, V, modes, rows, **kw)
    return O.reshape(B, S, Hq, d), LSE.reshape(B, S, Hq).transpose(0, 2, 1).copy()


def decode(q, Kc, Vc, seqlens, modes, *, sink=0, window=1, block_mask=None, T=128, scale=None):
    """O float64 [B, Hq, d], LSE float64 [B, Hq] of one decode step.
    q: bf16 [B, Hq, d]; Kc, Vc: bf16 [B, Lmax, Hkv, d]; seqlens int [B];
    block_mask uint8 [B, Hkv, nB, nB] (nB = ceil(Lmax / T)) when any mode is BLOCK."""
    qq, qs = _bf16_bits(q)
    k, ks = _bf16_bits(Kc)
    v, vs = _bf16_bits(Vc)
    assert (ks == vs).all()
    B, Hq, d = qq.shape
    Lmax, Hkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    sl = np.ascontiguousarray(np.asarray(seqlens), dtype=np.int32)
    m = _u8(modes, B * Hkv)
    O = np.zeros((B, Hq, d), dtype=np.float64)
    LSE = np.zeros((B, Hq), dtype=np.float64)
    bm = _u8(block_mask)
    rc = lib().ea_oracle_decode(_ptr(qq), _ptr(qs), _ptr(k), _ptr(v), _ptr(ks), _ptr(sl),
                                B, Hq, Hkv, d, Lmax, scale, _ptr(m), sink, window,
                                _ptr(bm), T, _ptr(O), _ptr(LSE))
    if rc != 0:
        raise ValueError("oracle decode rejected its arguments (rc=%d)" % rc)
    return O, LSE


def visited(B, S, Hkv, modes, *, sink=0, window=1, block_mask=None, T=128,
            qb_begin=0, qb_end=None):
    """uint8 [B, Hkv, qb_end - qb_begin, nB]: 1 where the tile holds a kept pair."""
    nB = (S + T - 1) // T
    if qb_end is None:
        qb_end = nB
    m = _u8(modes, B * Hkv)
    bm = _u8(block_mask)
    vis = np.zeros((B, Hkv, qb_end - qb_begin, nB), dtype=np.uint8)
    rc = lib().ea_oracle_visited(B, S, Hkv, _ptr(m), sink, window, _ptr(bm), T,
                                 qb_begin, qb_end, _ptr(vis))
    if rc != 0:
        raise ValueError("oracle visited rejected its arguments (rc=%d)" % rc)
    return vis


def route(K, weights, biases, *, pool_head=100, pool_tail=100, fa_impl=FULL, sa_impl=SSA):
    """Router forward in fp64.  weights: list of float32 [out, in] arrays, biases:
    list of float32 [out].  Returns (r uint8 [B, Hkv], m uint8 [B, Hkv],
    logits float64 [B, Hkv, 2], pooled float64 [B, Hkv, d])."""
    k, ks = _bf16_bits(K)
    B, S, Hkv, d = k.shape
    Ws = [np.ascontiguousarray(np.asarray(w if isinstance(w, np.ndarray) else w.cpu().numpy()),
                               dtype=np.float32) for w in weights]
    bs = [np.ascontiguousarray(np.asarray(b if isinstance(b, np.ndarray) else b.cpu().numpy()),
                               dtype=np.float32) for b in biases]
    dims = [Ws[0].shape[1]] + [w.shape[0] for w in Ws]
    dims_a = np.array(dims, dtype=np.int32)
    W_all = np.concatenate([w.ravel() for w in Ws]).astype(np.float32)
    b_all = np.concatenate([b.ravel() for b in bs]).astype(np.float32)
    r = np.zeros((B, Hkv), dtype=np.uint8)
    m = np.zeros((B, Hkv), dtype=np.uint8)
    logits = np.zeros((B, Hkv, 2), dtype=np.float64)
    pooled = np.zeros((B, Hkv, d), dtype=np.float64)
    rc = lib().ea_oracle_route(_ptr(k), _ptr(ks), B, S, Hkv, d, pool_head, pool_tail,
                               len(Ws), _ptr(dims_a), _ptr(W_all), _ptr(b_all),
                               fa_impl, sa_impl, _ptr(r), _ptr(m), _ptr(logits), _ptr(pooled))
    if rc != 0:
        raise ValueError("oracle route rejected its arguments (rc=%d)" % rc)
    return r, m, logits, pooled


def sparsity_ratios(r, m, S, *, sink=0, window=1, block_masks=None, T=128):
    """(Omega_MSR, Omega_ESR, kept int64 [L, Hkv]) by brute-force pair counts.
    r, m: uint8 [L, Hkv]; block_masks uint8 [L, Hkv, nB, nB] when any m is BLOCK."""
    ra = _u8(r)
    ma = _u8(m)
    L, Hkv = ra.shape
    bm = _u8(block_masks)
    msr = ctypes.c_double()
    esr = ctypes.c_double()
    kept = np.zeros((L, Hkv), dtype=np.int64)
    rc = lib().ea_oracle_sparsity_ratios(_ptr(ra), _ptr(ma), L, Hkv, S, sink, window,
                                         _ptr(bm), T, ctypes.byref(msr), ctypes.byref(esr),
                                         _ptr(kept))
    if rc != 0:
        raise ValueError("oracle sparsity_ratios rejected its arguments (rc=%d)" % rc)
    return msr.value, esr.value, kept


def xa_block_scores(Q, K, b, h, *, stride=16, T=128, scale=None, qb_rows=None):
    """XA antidiagonal block scores (float64 [nB, nB], zero above the diagonal) of
    KV head h of batch row b, summed over the query heads that read it.
    Q: bf16 [B, S, Hq, d]; K: bf16 [B, S, Hkv, d].  qb_rows: compute only these
    query-block rows (the rest stay zero)."""
    q, qs = _bf16_bits(Q)
    k, ks = _bf16_bits(K)
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    nB = (S + T - 1) // T
    W = np.zeros((nB, nB), dtype=np.float64)
    sel = None
    if qb_rows is not None:
        sel = np.zeros(nB, dtype=np.uint8)
        sel[np.asarray(qb_rows, dtype=np.int64)] = 1
    rc = lib().ea_oracle_xa_block_scores(_ptr(q), _ptr(qs), _ptr(k), _ptr(ks), S, Hq, Hkv, d,
                                         scale, stride, T, b, h, _ptr(sel), _ptr(W))
    if rc != 0:
        raise ValueError("oracle xa_block_scores rejected its arguments (rc=%d)" % rc)
    return W


def xa_select(W, tau, qb_rows=None):
    """XA threshold selection: uint8 [nB, nB] block mask from float64 scores [nB, nB]
    (only the rows qb_rows when given; the others stay zero)."""
    W = np.ascontiguousarray(W, dtype=np.float64)
    nB = W.shape[0]
    assert W.shape == (nB, nB)
    mask = np.zeros((nB, nB), dtype=np.uint8)
    sel = None
    if qb_rows is not None:
        sel = np.zeros(nB, dtype=np.uint8)
        sel[np.asarray(qb_rows, dtype=np.int64)] = 1
    rc = lib().ea_oracle_xa_select(_ptr(W), nB, float(tau), _ptr(sel), _ptr(mask))
    if rc != 0:
        raise ValueError("oracle xa_select rejected its arguments (rc=%d)" % rc)
    return mask


def xa_estimate(Q, K, modes, *, stride=16, tau=0.9, T=128, scale=None):
    """Scores float64 [B, Hkv, nB, nB] and block masks uint8 [B, Hkv, nB, nB] for the
    heads whose mode is BLOCK (other heads' entries stay zero)."""
    B, S, Hq, d = Q.shape
    Hkv = K.shape[2]
    m = _u8(modes, B * Hkv).reshape(B, Hkv)
    nB = (S + T - 1) // T
    W = np.zeros((B, Hkv, nB, nB), dtype=np.float64)
    M = np.zeros((B, Hkv, nB, nB), dtype=np.uint8)
    for b in range(B):
        for h in range(Hkv):
            if m[b, h] == BLOCK:
                W[b, h] = xa_block_scores(Q, K, b, h, stride=stride, T=T, scale=scale)
                M[b, h] = xa_select(W[b, h], tau)
    return W, M
