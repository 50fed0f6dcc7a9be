"""Prefill of sequences of different lengths packed back to back
(ea_hybrid_attn_prefill_varlen): every sequence must equal, bit for bit, the
fixed-length prefill of that sequence alone, and the fp64 oracle within the
tolerances; no sequence may see another."""
import numpy as np
import pytest
import torch

import oracle
import sparse_head_attention_gb300 as ea
from sparse_head_attention_gb300 import workloads as wl
from gpu_helpers import assert_close, check_no_device_error, gpu_device

pytestmark = pytest.mark.gpu
FULL, SSA, BLOCK = ea.FULL, ea.SSA, ea.BLOCK


@pytest.fixture(scope="module")
def dev():
    return gpu_device()


def packed_inputs(lens, Hq, Hkv, seed, use_bm):
    """Per-sequence Q/K/V (seeded), their packed forms, cu_seqlens, modes and
    (optionally) per-sequence block masks packed back to back."""
    seqs = [wl.qkv(1, L, Hq, Hkv, 128, seed=seed + i) if L > 0 else None for i, L in enumerate(lens)]
    d = 128

    def cat(k, H):
        parts = [s[k][0] for s in seqs if s is not None]
        return torch.cat(parts, 0) if parts else torch.empty(0, H, d, dtype=torch.bfloat16)

    Q, K, V = cat(0, Hq), cat(1, Hkv), cat(2, Hkv)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    cycle = [FULL, SSA, BLOCK, SSA] if use_bm else [FULL, SSA, SSA, FULL]
    m = torch.tensor([[cycle[(b + h) % 4] for h in range(Hkv)] for b in range(len(lens))], dtype=torch.uint8)
    masks = [wl.block_mask(1, Hkv, L, density=0.35, seed=seed + 50 + i)[0] if (use_bm and L > 0) else None
             for i, L in enumerate(lens)]
    packed_bm = None
    if use_bm:
        packed_bm = torch.cat([mk.reshape(-1) for mk in masks if mk is not None])
    return seqs, Q, K, V, cu, m, masks, packed_bm


@pytest.mark.parametrize("lens,Hq,Hkv,use_bm", [
    ([1000, 1, 0, 129, 700], 8, 2, False),
    ([128, 256, 127, 1], 12, 4, True),
    ([3000], 8, 2, True),
    ([5, 300, 0, 0, 2049, 17], 6, 2, False),
    # lengths at 32-row boundaries: a warp's 32 rows either all inside the
    # sequence (stored through shared memory and TMA) or crossing its end
    ([160, 96, 32, 64, 224, 33, 31], 8, 2, True),
])
def test_each_sequence_equals_its_own_prefill(dev, lens, Hq, Hkv, use_bm):
    sink, window = 64, 300
    seqs, Q, K, V, cu, m, masks, packed_bm = packed_inputs(lens, Hq, Hkv, 70 + len(lens), use_bm)
    total = int(cu[-1])
    ws = ea.prefill_varlen_workspace(len(lens), total, max(lens), Hq, Hkv, device=dev)
    O, LSE = ea.ea_hybrid_attn_prefill_varlen(
        Q.to(dev), K.to(dev), V.to(dev), cu.to(dev), m.to(dev), max_seqlen=max(lens), sink=sink,
        window=window, block_mask=None if packed_bm is None else packed_bm.to(dev), workspace=ws)
    torch.cuda.synchronize()
    check_no_device_error(ws)
    O, LSE = O.cpu(), LSE.cpu()
    for b, L in enumerate(lens):
        if L == 0:
            continue
        q, k, v = seqs[b]
        mb = m[b:b + 1]
        bm = None if masks[b] is None else masks[b][None]
        Ob, Lb = ea.ea_hybrid_attn_prefill(q.to(dev), k.to(dev), v.to(dev), mb.to(dev), sink=sink,
                                           window=window, block_mask=None if bm is None else bm.to(dev))
        torch.cuda.synchronize()
        c0 = int(cu[b])
        assert torch.equal(O[c0:c0 + L], Ob[0].cpu()), "sequence %d O" % b
        assert torch.equal(LSE[:, c0:c0 + L], Lb[0].cpu()), "sequence %d LSE" % b
        if L <= 1000:
            Oo, Lo = oracle.prefill_full(q, k, v, mb.numpy(), sink=sink, window=window,
                                         block_mask=None if bm is None else bm.numpy())
            assert_close(O[c0:c0 + L][None].float().numpy(), LSE[:, c0:c0 + L][None].numpy(), Oo, Lo,
                         "sequence %d" % b)


def test_strided_views_and_bad_sequence(dev):
    # Q/K/V as column slices of one packed QKV projection; sequence 1 longer
    # than max_seqlen: skipped and reported, the others still exact
    lens, Hq, Hkv = [400, 900, 300], 8, 2
    total = sum(lens)
    qkv = wl.randn_bf16((total, Hq + 2 * Hkv, 128), seed=91).to(dev)
    Q, K, V = qkv[:, :Hq], qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    cu = torch.tensor([0, 400, 1300, 1600], dtype=torch.int32, device=dev)
    m = torch.tensor([[FULL, SSA]] * 3, dtype=torch.uint8, device=dev)
    wide = torch.full((total, Hq + 3, 128), 7.0, dtype=torch.bfloat16, device=dev)
    O = wide[:, 1:1 + Hq]
    ws = ea.prefill_varlen_workspace(3, total, 500, Hq, Hkv, device=dev)
    _, LSE = ea.ea_hybrid_attn_prefill_varlen(Q, K, V, cu, m, max_seqlen=500, sink=16, window=200, O=O,
                                              workspace=ws)
    assert ea.ea_check_errors(ws) == 6            # sequence 1 (900 > 500) reported
    assert (O[400:1300].float() == 7.0).all()     # and not written
    # the heads beside the view are untouched (staged stores write whole warps of rows)
    assert (wide[:, 0].float() == 7.0).all() and (wide[:, 1 + Hq:].float() == 7.0).all()
    for b, (c0, L) in enumerate([(0, 400), (1300, 300)]):
        Ob, Lb = ea.ea_hybrid_attn_prefill(Q[c0:c0 + L][None], K[c0:c0 + L][None], V[c0:c0 + L][None],
                                           m[:1], sink=16, window=200)
        torch.cuda.synchronize()
        assert torch.equal(O[c0:c0 + L], Ob[0]), b
        assert torch.equal(LSE[:, c0:c0 + L], Lb[0]), b


def test_many_short_sequences_one_launch(dev):
    # a serving-like batch: 64 sequences of 1..700 tokens
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 701, size=64)]
    Hq, Hkv = 32, 8
    seqs, Q, K, V, cu, m, _, _ = packed_inputs(lens, Hq, Hkv, 300, False)
    O, LSE = ea.ea_hybrid_attn_prefill_varlen(Q.to(dev), K.to(dev), V.to(dev), cu.to(dev), m.to(dev),
                                              max_seqlen=max(lens), sink=32, window=256)
    torch.cuda.synchronize()
    O, LSE = O.cpu(), LSE.cpu()
    for b in (0, 17, 63):
        L, c0 = lens[b], int(cu[b])
        q, k, v = seqs[b]
        Oo, Lo = oracle.prefill_full(q, k, v, m[b:b + 1].numpy(), sink=32, window=256)
        assert_close(O[c0:c0 + L][None].float().numpy(), LSE[:, c0:c0 + L][None].numpy(), Oo, Lo, "b=%d" % b)
