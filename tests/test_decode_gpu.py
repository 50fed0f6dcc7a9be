"""Parity of the split-KV hybrid decode (CUDA, through the C ABI) with the fp64
oracle, split-count invariance, edge cases, and the full B=32 / 128K workload
on sampled sequences."""
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


def run(dev, q, Kc, Vc, sl, modes, sink, window, num_splits=0, bm=None):
    B, Hq, _ = q.shape
    Lmax, Hkv = Kc.shape[1], Kc.shape[2]
    ws = ea.decode_workspace(B, Hq, Hkv, Lmax, num_splits, device=dev)
    O, LSE = ea.ea_hybrid_attn_decode(q.to(dev), Kc.to(dev), Vc.to(dev), sl.to(dev),
                                      torch.as_tensor(modes, dtype=torch.uint8).to(dev),
                                      sink=sink, window=window, num_splits=num_splits, workspace=ws,
                                      block_mask=None if bm is None else torch.as_tensor(bm).to(dev))
    torch.cuda.synchronize()
    check_no_device_error(ws)
    return O, LSE


@pytest.mark.parametrize("num_splits", [0, 1, 2, 7, 64])
def test_small_batch_all_heads(dev, num_splits):
    cfg = wl.DecodeConfig("t", B=4, Hq=8, Hkv=2, d=128, L=5000, sink=128, window=1000)
    q, Kc, Vc, sl = wl.decode_inputs(cfg, seqlens=[5000, 1, 4097, 1129])
    modes = np.array([[FULL, SSA], [SSA, FULL], [SSA, SSA], [FULL, FULL]], np.uint8)
    O, LSE = run(dev, q, Kc, Vc, sl, modes, cfg.sink, cfg.window, num_splits)
    Oref, Lref = oracle.decode(q, Kc, Vc, sl, modes, sink=cfg.sink, window=cfg.window)
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "splits=%d" % num_splits)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (16, 2), (6, 2), (12, 4)])
def test_group_sizes(dev, Hq, Hkv):
    cfg = wl.DecodeConfig("t", B=2, Hq=Hq, Hkv=Hkv, d=128, L=3000, sink=7, window=333)
    q, Kc, Vc, sl = wl.decode_inputs(cfg, seqlens=[3000, 2049])
    modes = np.where(np.arange(Hkv)[None, :] % 2 == 0, FULL, SSA).repeat(2, 0).astype(np.uint8)
    O, LSE = run(dev, q, Kc, Vc, sl, modes, cfg.sink, cfg.window)
    Oref, Lref = oracle.decode(q, Kc, Vc, sl, modes, sink=cfg.sink, window=cfg.window)
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "g=%d" % (Hq // Hkv))


def _decode_mask(B, Hkv, Lmax, seqlens, seed):
    """Random block mask over the decode rows, with one unit's decode row emptied
    and one unit's diagonal block dropped (its last kept block is then a full one)."""
    bm = wl.block_mask(B, Hkv, Lmax, density=0.3, seed=seed).numpy()
    L0 = seqlens[0]
    bm[0, 0, (L0 - 1) // 128, :] = 0                 # no kept key at all
    L2 = seqlens[2]
    bm[2, 1, (L2 - 1) // 128, (L2 - 1) // 128] = 0   # diagonal block dropped
    return bm


@pytest.mark.parametrize("num_splits", [0, 1, 7])
def test_block_heads_match_oracle(dev, num_splits):
    cfg = wl.DecodeConfig("t", B=4, Hq=8, Hkv=2, d=128, L=5000, sink=128, window=1000)
    seqlens = [5000, 1, 4097, 1129]
    q, Kc, Vc, sl = wl.decode_inputs(cfg, seqlens=seqlens)
    modes = np.array([[BLOCK, BLOCK], [BLOCK, SSA], [FULL, BLOCK], [BLOCK, FULL]], np.uint8)
    bm = _decode_mask(4, 2, cfg.L, seqlens, seed=31)
    O, LSE = run(dev, q, Kc, Vc, sl, modes, cfg.sink, cfg.window, num_splits, bm=bm)
    Oref, Lref = oracle.decode(q, Kc, Vc, sl, modes, sink=cfg.sink, window=cfg.window, block_mask=bm)
    assert np.isneginf(Lref[0, :4]).all(), "the emptied decode row must have no kept key"
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "splits=%d" % num_splits)


@pytest.mark.parametrize("num_splits", [0, 3])
def test_few_kept_keys_with_large_values(dev, num_splits):
    # Units keeping 1 to 128 keys, |V| in [2.2, 3.8) with one sign per (head,
    # dim): |O| stays in [2, 4), where correct rounding alone errs by up to
    # 0.0078, and a P rounded to bf16 would add up to 2^-9 |O|.  Units of at
    # most 512 keys take P V in two bf16 parts: every element within a flat 1e-2.
    seqlens = [1, 2, 3, 5, 17, 64, 100, 128]
    B, Hq, Hkv, Lmax, sink, window = len(seqlens), 8, 2, 128, 2, 3
    cfg = wl.DecodeConfig("t", B=B, Hq=Hq, Hkv=Hkv, d=128, L=Lmax, sink=sink, window=window)
    q, Kc, _, sl = wl.decode_inputs(cfg, seqlens=seqlens)
    Vc = wl.offset_values(B, Lmax, Hkv, 128, seed=43)
    modes = np.array([[FULL, SSA], [SSA, BLOCK], [BLOCK, FULL]] * 3, np.uint8)[:B]
    bm = np.ones((B, Hkv, 1, 1), np.uint8)
    O, LSE = run(dev, q, Kc, Vc, sl, modes, sink, window, num_splits, bm=bm)
    Oref, Lref = oracle.decode(q, Kc, Vc, sl, modes, sink=sink, window=window, block_mask=bm)
    assert np.abs(Oref).min() >= 2.0
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref,
                 "few keys, splits=%d" % num_splits, flat=True)


def test_single_sequence_planned_in_kernel_equals_planner(dev):
    # B * Hkv <= 8 is planned inside the split kernel; the same sequence as row 0
    # of a two-sequence batch goes through the planner launch.  Both plans use
    # the 2048-key minimum chunk here, so the chunks, partials and merge are the
    # same: the outputs must be bitwise equal (and match the oracle).
    cfg = wl.DecodeConfig("t", B=2, Hq=32, Hkv=8, d=128, L=5000, sink=128, window=1000)
    q, Kc, Vc, _ = wl.decode_inputs(cfg, seqlens=[5000, 5000])
    q[1], Kc[1], Vc[1] = q[0], Kc[0], Vc[0]
    modes = np.array([[FULL, SSA, SSA, FULL, SSA, SSA, SSA, SSA]] * 2, np.uint8)
    sl2 = torch.tensor([5000, 5000], dtype=torch.int32)
    O2, L2 = run(dev, q, Kc, Vc, sl2, modes, cfg.sink, cfg.window)
    O1, L1 = run(dev, q[:1], Kc[:1], Vc[:1], sl2[:1], modes[:1], cfg.sink, cfg.window)
    assert torch.equal(O1[0], O2[0]) and torch.equal(L1[0], L2[0])
    Oref, Lref = oracle.decode(q[:1], Kc[:1], Vc[:1], sl2[:1], modes[:1], sink=cfg.sink, window=cfg.window)
    assert_close(O1.float().cpu().numpy(), L1.cpu().numpy(), Oref, Lref, "single sequence")


def test_block_decode_equals_last_prefill_row_on_gpu(dev):
    B, S, Hq, Hkv = 1, 1500, 8, 2
    Q, K, V = wl.qkv(B, S, Hq, Hkv, 128, seed=14)
    bm = torch.as_tensor(wl.block_mask(B, Hkv, S, density=0.4, seed=15)).to(dev)
    modes = torch.tensor([[BLOCK, SSA]], dtype=torch.uint8, device=dev)
    O, LSE = ea.ea_hybrid_attn_prefill(Q.to(dev), K.to(dev), V.to(dev), modes, sink=64, window=300,
                                       block_mask=bm)
    Od, Ld = ea.ea_hybrid_attn_decode(Q[:, S - 1].contiguous().to(dev), K.to(dev), V.to(dev),
                                      torch.tensor([S], dtype=torch.int32, device=dev), modes,
                                      sink=64, window=300, block_mask=bm)
    torch.cuda.synchronize()
    assert (Od[0].float() - O[0, S - 1].float()).abs().max().item() <= 1.6e-2
    assert (Ld[0] - LSE[0, :, S - 1]).abs().max().item() <= 1e-3


def test_empty_sequence_and_block_without_mask(dev):
    cfg = wl.DecodeConfig("t", B=2, Hq=8, Hkv=2, d=128, L=256, sink=4, window=16)
    q, Kc, Vc, sl = wl.decode_inputs(cfg, seqlens=[0, 256])
    O, LSE = run(dev, q, Kc, Vc, sl, [[FULL, SSA], [FULL, SSA]], cfg.sink, cfg.window)
    assert (O[0].float() == 0).all()
    assert torch.isneginf(LSE[0]).all()
    ws = ea.decode_workspace(2, 8, 2, 256, device=dev)
    ea.ea_hybrid_attn_decode(q.to(dev), Kc.to(dev), Vc.to(dev), sl.to(dev),
                             torch.tensor([[BLOCK, SSA], [FULL, SSA]], dtype=torch.uint8, device=dev),
                             sink=4, window=16, workspace=ws)
    assert ea.ea_check_errors(ws) == 6


def test_decode_equals_last_prefill_row_on_gpu(dev):
    B, S, Hq, Hkv, sink, window = 1, 1500, 8, 2, 64, 300
    Q, K, V = wl.qkv(B, S, Hq, Hkv, 128, seed=12)
    modes = torch.tensor([[FULL, SSA]], dtype=torch.uint8, device=dev)
    O, LSE = ea.ea_hybrid_attn_prefill(Q.to(dev), K.to(dev), V.to(dev), modes, sink=sink, window=window)
    Od, Ld = ea.ea_hybrid_attn_decode(Q[:, S - 1].contiguous().to(dev), K.to(dev), V.to(dev),
                                      torch.tensor([S], dtype=torch.int32, device=dev), modes,
                                      sink=sink, window=window)
    torch.cuda.synchronize()
    assert (Od[0].float() - O[0, S - 1].float()).abs().max().item() <= 1.6e-2
    assert (Ld[0] - LSE[0, :, S - 1]).abs().max().item() <= 1e-3


def test_full_workload_sampled_sequences(dev):
    cfg = wl.DECODE_128K
    q, Kc, Vc, sl = wl.decode_inputs(cfg, device=dev)
    _, m = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads)
    ws = ea.decode_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.L, device=dev)
    O, LSE = ea.ea_hybrid_attn_decode(q, Kc, Vc, sl, m.to(dev), sink=cfg.sink, window=cfg.window,
                                      workspace=ws)
    torch.cuda.synchronize()
    check_no_device_error(ws)
    for b in (0, 13, cfg.B - 1):
        Oref, Lref = oracle.decode(q[b:b + 1].cpu(), Kc[b:b + 1].cpu(), Vc[b:b + 1].cpu(),
                                   sl[b:b + 1].cpu(), m[b:b + 1], sink=cfg.sink, window=cfg.window)
        assert_close(O[b:b + 1].float().cpu().numpy(), LSE[b:b + 1].cpu().numpy(), Oref, Lref,
                     "b=%d" % b, flat=True)


def test_strided_query_cache_and_output(dev):
    # q as a slice of a wider projection, the cache as a view of a larger
    # [B, Lmax, heads, d] buffer, O written into a slice of a wider output.
    B, Hq, Hkv, d, Lmax = 2, 8, 2, 128, 1500
    proj = wl.randn_bf16((B, Hq + 4, d), seed=61)
    cache = wl.randn_bf16((B, Lmax, Hkv + 2, d), seed=62)
    q = proj[:, 2:2 + Hq]
    Kc, Vc = cache[:, :, :Hkv], cache[:, :, 2:]
    seqlens = torch.tensor([1500, 777], dtype=torch.int32)
    modes = np.array([[FULL, SSA], [SSA, FULL]], np.uint8)
    pd, cd = proj.to(dev), cache.to(dev)
    Ob = torch.full((B, Hq + 3, d), 5.0, dtype=torch.bfloat16, device=dev)
    ws = ea.decode_workspace(B, Hq, Hkv, Lmax, device=dev)
    ea.ea_hybrid_attn_decode(pd[:, 2:2 + Hq], cd[:, :, :Hkv], cd[:, :, 2:], seqlens.to(dev),
                             torch.as_tensor(modes).to(dev), sink=32, window=400, O=Ob[:, 1:1 + Hq],
                             workspace=ws)
    torch.cuda.synchronize()
    check_no_device_error(ws)
    Oref, _ = oracle.decode(q, Kc, Vc, seqlens, modes, sink=32, window=400)
    assert np.abs(Ob[:, 1:1 + Hq].float().cpu().numpy() - Oref).max() <= 1e-2
    assert (Ob[:, 0].float() == 5.0).all() and (Ob[:, 1 + Hq:].float() == 5.0).all()


def test_block_decode_at_the_longest_cache(dev):
    """Lmax = 2^21 keys (16384 mask blocks per row), a sparse decode row."""
    cfg = wl.DecodeConfig("t", B=1, Hq=4, Hkv=1, d=128, L=1 << 21, sink=0, window=1)
    q, Kc, Vc, sl = wl.decode_inputs(cfg, device=dev, seqlens=[(1 << 21) - 77])
    nB = cfg.L // 128
    row = torch.rand(nB, generator=torch.Generator().manual_seed(3)) < 0.01
    row[(int(sl[0]) - 1) // 128] = True
    bm = torch.zeros(1, 1, nB, nB, dtype=torch.uint8)
    bm[0, 0, (int(sl[0]) - 1) // 128] = row.to(torch.uint8)
    m = torch.tensor([[BLOCK]], dtype=torch.uint8)
    ws = ea.decode_workspace(1, 4, 1, cfg.L, device=dev)
    O, LSE = ea.ea_hybrid_attn_decode(q, Kc, Vc, sl, m.to(dev), sink=0, window=1,
                                      block_mask=bm.to(dev), workspace=ws)
    torch.cuda.synchronize()
    check_no_device_error(ws)
    Oref, Lref = oracle.decode(q.cpu(), Kc.cpu(), Vc.cpu(), sl.cpu(), m, sink=0, window=1,
                               block_mask=bm)
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "Lmax=2^21")


def test_random_configurations_offset_values(dev):
    # decode counterpart of the prefill's offset-value sweep: every element
    # within a flat 1e-2 (units of up to 512 kept keys take P V in two parts)
    rng = np.random.default_rng(4343)
    for case in range(20):
        B = int(rng.integers(1, 6))
        Hkv = int(rng.integers(1, 4))
        Hq = Hkv * int(rng.integers(1, 5))
        Lmax = int(rng.integers(1, 3000))
        sink, window = int(rng.integers(0, 300)), int(rng.integers(1, 1200))
        seqlens = [int(rng.integers(1, Lmax + 1)) for _ in range(B)]
        cfg = wl.DecodeConfig("t", B=B, Hq=Hq, Hkv=Hkv, d=128, L=Lmax, sink=sink, window=window)
        q, Kc, _, sl = wl.decode_inputs(cfg, seqlens=seqlens)
        Vc = wl.offset_values(B, Lmax, Hkv, 128, seed=7100 + case)
        modes = rng.integers(0, 3, size=(B, Hkv)).astype(np.uint8)
        bm = wl.block_mask(B, Hkv, Lmax, density=float(rng.uniform(0.1, 0.9)), seed=200 + case).numpy()
        ns = int(rng.choice([0, 0, 1, 3, 9]))
        O, LSE = run(dev, q, Kc, Vc, sl, modes, sink, window, ns, bm=bm)
        Oref, Lref = oracle.decode(q, Kc, Vc, sl, modes, sink=sink, window=window, block_mask=bm)
        assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref,
                     "offset V, case %d (B=%d Hq=%d Hkv=%d Lmax=%d splits=%d)" % (case, B, Hq, Hkv, Lmax, ns),
                     flat=True)
