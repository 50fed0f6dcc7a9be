"""Decode over a paged KV cache (ea_hybrid_attn_decode_paged): the pages of
each sequence are scattered through a shared pool by a block table; the result
must match the fp64 oracle on the contiguous cache those pages spell out."""
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


def paged_from_contiguous(Kc, Vc, seqlens, page_size, seed, spare=3):
    """Scatter the first ceil(L_b / page_size) pages of every sequence into a
    shuffled pool (with `spare` unused pages); returns the pools and the block
    table [B, max_pages] (unused entries -1)."""
    B, Lmax, Hkv, d = Kc.shape
    max_pages = (Lmax + page_size - 1) // page_size
    need = [(int(L) + page_size - 1) // page_size for L in seqlens]
    n_pool = sum(need) + spare
    perm = torch.randperm(n_pool, generator=torch.Generator().manual_seed(seed))
    Kp = wl.randn_bf16((n_pool, page_size, Hkv, d), seed=seed + 1)   # junk in unused rows
    Vp = wl.randn_bf16((n_pool, page_size, Hkv, d), seed=seed + 2)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    nxt = 0
    for b in range(B):
        for p in range(need[b]):
            page = int(perm[nxt])
            nxt += 1
            table[b, p] = page
            r0, r1 = p * page_size, min((p + 1) * page_size, Lmax)
            Kp[page, : r1 - r0] = Kc[b, r0:r1]
            Vp[page, : r1 - r0] = Vc[b, r0:r1]
    return Kp, Vp, table


@pytest.mark.parametrize("page_size,num_splits", [(64, 0), (128, 0), (256, 0), (64, 7), (256, 1)])
def test_matches_oracle(dev, page_size, num_splits):
    cfg = wl.DecodeConfig("t", B=6, Hq=8, Hkv=2, d=128, L=3000, sink=100, window=1000)
    lens = [3000, 1, 0, 1000, 64 * 7, 2049]
    q, Kc, Vc, sl = wl.decode_inputs(cfg, seqlens=lens)
    modes = np.array([[FULL, SSA], [SSA, FULL], [SSA, SSA], [SSA, SSA], [FULL, SSA], [SSA, FULL]],
                     np.uint8)
    Kp, Vp, table = paged_from_contiguous(Kc, Vc, lens, page_size, seed=40 + page_size)
    ws = ea.decode_workspace(cfg.B, cfg.Hq, cfg.Hkv, table.shape[1] * page_size, num_splits, device=dev)
    O, LSE = ea.ea_hybrid_attn_decode_paged(q.to(dev), Kp.to(dev), Vp.to(dev), table.to(dev), sl.to(dev),
                                            torch.as_tensor(modes).to(dev), sink=cfg.sink,
                                            window=cfg.window, num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    check_no_device_error(ws)
    Oref, Lref = oracle.decode(q, Kc, Vc, sl, modes, sink=cfg.sink, window=cfg.window)
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "page %d" % page_size)


@pytest.mark.parametrize("page_size,num_splits", [(64, 0), (256, 0), (128, 5)])
def test_block_heads_on_a_paged_cache(dev, page_size, num_splits):
    """BLOCK heads read the kept blocks of their decode row through the block
    table; the mask spans max_pages * page_size positions."""
    cfg = wl.DecodeConfig("t", B=4, Hq=8, Hkv=2, d=128, L=3000, sink=100, window=1000)
    lens = [3000, 1, 2049, 64 * 7]
    q, Kc, Vc, sl = wl.decode_inputs(cfg, seqlens=lens)
    modes = np.array([[BLOCK, SSA], [BLOCK, BLOCK], [FULL, BLOCK], [BLOCK, FULL]], np.uint8)
    Kp, Vp, table = paged_from_contiguous(Kc, Vc, lens, page_size, seed=70 + page_size)
    Lp = table.shape[1] * page_size
    nBp, nBc = (Lp + 127) // 128, (cfg.L + 127) // 128
    bm = wl.block_mask(cfg.B, cfg.Hkv, Lp, density=0.3, seed=page_size).numpy()
    bm[2, 1, (lens[2] - 1) // 128, (lens[2] - 1) // 128] = 0     # diagonal block dropped
    ws = ea.decode_workspace(cfg.B, cfg.Hq, cfg.Hkv, Lp, num_splits, device=dev)
    O, LSE = ea.ea_hybrid_attn_decode_paged(q.to(dev), Kp.to(dev), Vp.to(dev), table.to(dev), sl.to(dev),
                                            torch.as_tensor(modes).to(dev), sink=cfg.sink,
                                            window=cfg.window, num_splits=num_splits, workspace=ws,
                                            block_mask=torch.as_tensor(bm).to(dev))
    torch.cuda.synchronize()
    check_no_device_error(ws)
    assert nBp >= nBc
    bmc = np.ascontiguousarray(bm[:, :, :nBc, :nBc])
    Oref, Lref = oracle.decode(q, Kc, Vc, sl, modes, sink=cfg.sink, window=cfg.window, block_mask=bmc)
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "page %d" % page_size)


@pytest.mark.parametrize("sink,window", [(0, 64), (64, 64), (130, 70), (5000, 1), (1, 5000)])
def test_sink_window_edges(dev, sink, window):
    cfg = wl.DecodeConfig("t", B=3, Hq=12, Hkv=4, d=128, L=1500, sink=sink, window=window)
    lens = [1500, 777, 129]
    q, Kc, Vc, sl = wl.decode_inputs(cfg, seqlens=lens)
    modes = np.array([[SSA, SSA, FULL, SSA]] * 3, np.uint8)
    Kp, Vp, table = paged_from_contiguous(Kc, Vc, lens, 128, seed=sink + window)
    O, LSE = ea.ea_hybrid_attn_decode_paged(q.to(dev), Kp.to(dev), Vp.to(dev), table.to(dev), sl.to(dev),
                                            torch.as_tensor(modes).to(dev), sink=sink, window=window)
    torch.cuda.synchronize()
    Oref, Lref = oracle.decode(q, Kc, Vc, sl, modes, sink=sink, window=window)
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "sink %d window %d" % (sink, window))


def test_bad_table_entry_is_reported(dev):
    cfg = wl.DecodeConfig("t", B=2, Hq=8, Hkv=2, d=128, L=512, sink=16, window=128)
    q, Kc, Vc, sl = wl.decode_inputs(cfg)
    Kp, Vp, table = paged_from_contiguous(Kc, Vc, [512, 512], 128, seed=9)
    table[1, 2] = Kp.shape[0] + 5          # outside the pool: reads zeros, reported
    ws = ea.decode_workspace(2, 8, 2, 512, device=dev)
    ea.ea_hybrid_attn_decode_paged(q.to(dev), Kp.to(dev), Vp.to(dev), table.to(dev), sl.to(dev),
                                   torch.tensor([[FULL, FULL]] * 2, dtype=torch.uint8, device=dev),
                                   sink=16, window=128, workspace=ws)
    assert ea.ea_check_errors(ws) == 6
    assert ea.ea_check_errors(ws) == 0     # read and cleared


def test_full_workload_sampled_sequences(dev):
    cfg = wl.DECODE_128K
    q, Kc, Vc, sl = wl.decode_inputs(cfg, device=dev)
    _, m = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads)
    page_size = 256
    # a permuted pool on the device: page p of sequence b sits in slot
    # perm[b * per_seq + p]
    per_seq = cfg.L // page_size
    perm = torch.randperm(cfg.B * per_seq, generator=torch.Generator().manual_seed(3)).to(dev)
    table = perm.view(cfg.B, per_seq).to(torch.int32)
    Kp = torch.empty(cfg.B * per_seq, page_size, cfg.Hkv, cfg.d, dtype=torch.bfloat16, device=dev)
    Vp = torch.empty_like(Kp)
    Kp[perm] = Kc.view(cfg.B * per_seq, page_size, cfg.Hkv, cfg.d)
    Vp[perm] = Vc.view(cfg.B * per_seq, page_size, cfg.Hkv, cfg.d)
    ws = ea.decode_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.L, device=dev)
    O, LSE = ea.ea_hybrid_attn_decode_paged(q, Kp, Vp, table, sl, m.to(dev), sink=cfg.sink,
                                            window=cfg.window, workspace=ws)
    torch.cuda.synchronize()
    check_no_device_error(ws)
    for b in (0, 17, cfg.B - 1):
        Oref, Lref = oracle.decode(q[b:b + 1].cpu(), Kc[b:b + 1].cpu(), Vc[b:b + 1].cpu(),
                                   sl[b:b + 1].cpu(), m[b:b + 1], sink=cfg.sink, window=cfg.window)
        assert_close(O[b:b + 1].float().cpu().numpy(), LSE[b:b + 1].cpu().numpy(), Oref, Lref, "b=%d" % b)
