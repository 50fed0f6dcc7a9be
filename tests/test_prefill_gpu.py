"""Parity of the fused hybrid-head prefill (CUDA, through the C ABI) with the
fp64 oracle: element by element on small and ragged shapes, on sampled rows at
the full workload sizes, bit-exact visited-tile sets, and the device checks."""
import numpy as np
import pytest
import torch

import oracle
import sparse_head_attention_gb300 as ea
from sparse_head_attention_gb300 import workloads as wl
from gpu_helpers import (assert_close, bitmap_to_tiles, check_no_device_error, gpu_device,
                         sample_rows)

pytestmark = pytest.mark.gpu
FULL, SSA, BLOCK = ea.FULL, ea.SSA, ea.BLOCK


@pytest.fixture(scope="module")
def dev():
    return gpu_device()


def run(dev, Q, K, V, modes, sink, window, bm=None, visited=False, **kw):
    B, S, Hq, _ = Q.shape
    Hkv = K.shape[2]
    nB = (S + 127) // 128
    ws = ea.prefill_workspace(B, S, Hq, Hkv, device=dev)
    vis = None
    if visited:
        vis = torch.zeros((B * Hkv * nB * nB + 31) // 32, dtype=torch.int32, device=dev)
    O, LSE = ea.ea_hybrid_attn_prefill(Q.to(dev), K.to(dev), V.to(dev),
                                       torch.as_tensor(modes, dtype=torch.uint8).to(dev),
                                       sink=sink, window=window,
                                       block_mask=None if bm is None else torch.as_tensor(bm).to(dev),
                                       workspace=ws, visited_bitmap=vis, **kw)
    torch.cuda.synchronize()
    check_no_device_error(ws)
    return O, LSE, vis


def test_tiny_workload_all_rows(dev):
    cfg = wl.TINY
    Q, K, V = wl.qkv(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.d, seed=cfg.seed)
    _, m = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads)
    O, LSE, vis = run(dev, Q, K, V, m, cfg.sink, cfg.window, visited=True)
    Oref, Lref = oracle.prefill_full(Q, K, V, m, sink=cfg.sink, window=cfg.window)
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "tiny", flat=True)
    nB = cfg.S // 128
    tiles = bitmap_to_tiles(vis, cfg.B, cfg.Hkv, nB)
    ref = oracle.visited(cfg.B, cfg.S, cfg.Hkv, m, sink=cfg.sink, window=cfg.window)
    np.testing.assert_array_equal(tiles, ref)
    assert tiles[0, 0].sum() == 36 and tiles[0, 1].sum() == 26   # FA / SSA tiles per head


SHAPES = [
    # B, S, Hq, Hkv, modes, sink, window
    (3, 129, 8, 2, [[FULL, SSA], [SSA, FULL], [SSA, SSA]], 5, 17),
    (1, 1000, 4, 1, [[SSA]], 0, 1),
    (1, 1, 8, 2, [[FULL, SSA]], 64, 256),
    (2, 300, 6, 2, [[FULL, SSA], [SSA, FULL]], 100, 3),          # odd group size 3
    (1, 513, 4, 4, [[FULL, SSA, FULL, SSA]], 130, 129),          # one query head per KV head
    (1, 700, 8, 2, [[SSA, SSA]], 2000, 1),                       # sink covers everything
    (1, 640, 8, 2, [[SSA, FULL]], 128, 128),                     # tile-aligned sink / window
    (1, 700, 16, 2, [[FULL, SSA]], 64, 300),                     # group size 8 (four head pairs)
    (2, 450, 14, 2, [[SSA, FULL], [FULL, SSA]], 32, 200),        # group size 7 (last head paired with itself)
]


@pytest.mark.parametrize("B,S,Hq,Hkv,modes,sink,window", SHAPES)
def test_ragged_shapes_all_rows(dev, B, S, Hq, Hkv, modes, sink, window):
    Q, K, V = wl.qkv(B, S, Hq, Hkv, 128, seed=S + Hq)
    O, LSE, vis = run(dev, Q, K, V, modes, sink, window, visited=True)
    Oref, Lref = oracle.prefill_full(Q, K, V, np.array(modes, np.uint8), sink=sink, window=window)
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "S=%d" % S)
    nB = (S + 127) // 128
    tiles = bitmap_to_tiles(vis, B, Hkv, nB)
    np.testing.assert_array_equal(tiles, oracle.visited(B, S, Hkv, np.array(modes, np.uint8),
                                                        sink=sink, window=window))


def test_block_masks_with_empty_rows(dev):
    B, S, Hq, Hkv = 2, 1000, 12, 3
    Q, K, V = wl.qkv(B, S, Hq, Hkv, 128, seed=5)
    bm = wl.block_mask(B, Hkv, S, density=0.3, seed=9).numpy()
    bm[0, 0, 3, :] = 0                   # query block 3 of (b0, h0) keeps nothing
    bm[1, 2, 5, 5] = 0                   # diagonal dropped
    bm[1, 1] = np.tril(np.ones_like(bm[1, 1]))   # all kept: equals FA
    modes = [[BLOCK, SSA, BLOCK], [FULL, BLOCK, BLOCK]]
    O, LSE, vis = run(dev, Q, K, V, modes, 64, 300, bm=bm, visited=True)
    Oref, Lref = oracle.prefill_full(Q, K, V, np.array(modes, np.uint8), sink=64, window=300,
                                     block_mask=bm)
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "block")
    assert np.isneginf(LSE[0, 0, 3 * 128:4 * 128].cpu().numpy()).all()
    assert (O[0, 3 * 128:4 * 128, 0:4].float().cpu().numpy() == 0).all()
    nB = (S + 127) // 128
    np.testing.assert_array_equal(
        bitmap_to_tiles(vis, B, Hkv, nB),
        oracle.visited(B, S, Hkv, np.array(modes, np.uint8), sink=64, window=300, block_mask=bm))


FEW_KEY_CASES = [
    # S, modes, sink, window: every query block's first row keeps at most 128 keys
    (128, [[SSA, FULL]], 0, 3),      # FA rows keep 1..128 keys, SSA rows 1..3
    (300, [[SSA, SSA]], 2, 2),       # two sink keys plus a window of 2
    (300, [[BLOCK, SSA]], 1, 1),     # diagonal block only; sink + window of 1
]


@pytest.mark.parametrize("S,modes,sink,window", FEW_KEY_CASES)
def test_few_kept_keys_with_large_values(dev, S, modes, sink, window):
    # |V| in [2.2, 3.8) with one sign per (head, dim), so |O| stays in [2, 4),
    # where a correctly rounded bf16 output errs by at most 2^-7 = 0.0078.
    # With one to a few kept keys a P rounded to bf16 (2^-9 relative) would
    # add up to 2^-9 |O| more and cross 1e-2 (an fp64 model of that arithmetic
    # puts 464 to 1063 elements of these cases above it); rows keeping at most
    # 512 keys take P V in two bf16 parts, which keeps every element within a
    # flat 1e-2.
    B, Hq, Hkv = 1, 4, 2
    Q, K, _ = wl.qkv(B, S, Hq, Hkv, 128, seed=41)
    V = wl.offset_values(B, S, Hkv, 128, seed=42)
    nB = (S + 127) // 128
    bm = np.zeros((B, Hkv, nB, nB), np.uint8)
    bm[:, :, np.arange(nB), np.arange(nB)] = 1
    O, LSE, _ = run(dev, Q, K, V, modes, sink, window, bm=bm)
    Oref, Lref = oracle.prefill_full(Q, K, V, np.array(modes, np.uint8), sink=sink, window=window,
                                     block_mask=bm)
    assert np.abs(Oref).min() >= 2.0
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref,
                 "few keys S=%d %s sink=%d window=%d" % (S, modes, sink, window), flat=True)


def test_strided_views_and_concatenation(dev):
    # Q, K, V as views of one packed projection [B, S, Hq + 2 Hkv, d]; O written
    # into the first Hq heads of a wider buffer (eq. 3 concatenation in place).
    B, S, Hq, Hkv, d = 2, 333, 8, 2, 128
    packed = wl.randn_bf16((B, S, Hq + 2 * Hkv, d), seed=77)
    Q, K, V = packed[:, :, :Hq], packed[:, :, Hq:Hq + Hkv], packed[:, :, Hq + Hkv:]
    modes = np.array([[SSA, FULL], [FULL, SSA]], np.uint8)
    pg = packed.to(dev)
    Ob = torch.full((B, S, Hq + 8, d), 7.0, dtype=torch.bfloat16, device=dev)
    Oview = Ob[:, :, :Hq]
    ws = ea.prefill_workspace(B, S, Hq, Hkv, device=dev)
    ea.ea_hybrid_attn_prefill(pg[:, :, :Hq], pg[:, :, Hq:Hq + Hkv], pg[:, :, Hq + Hkv:],
                              torch.as_tensor(modes).to(dev), sink=3, window=50, O=Oview,
                              workspace=ws)
    torch.cuda.synchronize()
    check_no_device_error(ws)
    Oref, _ = oracle.prefill_full(Q, K, V, modes, sink=3, window=50)
    err = np.abs(Oview.float().cpu().numpy() - Oref).max()
    assert err <= 1e-2, err
    assert (Ob[:, :, Hq:].float() == 7.0).all()       # neighbours untouched


def test_repeated_calls_are_bitwise_identical(dev):
    B, S, Hq, Hkv = 1, 2000, 8, 2
    Q, K, V = wl.qkv(B, S, Hq, Hkv, 128, seed=3)
    O1, L1, _ = run(dev, Q, K, V, [[FULL, SSA]], 64, 256)
    O2, L2, _ = run(dev, Q, K, V, [[FULL, SSA]], 64, 256)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


def test_device_checks_report_bad_modes_and_missing_masks(dev):
    B, S, Hq, Hkv = 1, 256, 4, 2
    Q, K, V = wl.qkv(B, S, Hq, Hkv, 128, seed=1)
    for modes in ([[FULL, 7]], [[BLOCK, SSA]]):       # unknown mode; BLOCK without a mask
        ws = ea.prefill_workspace(B, S, Hq, Hkv, device=dev)
        ea.ea_hybrid_attn_prefill(Q.to(dev), K.to(dev), V.to(dev),
                                  torch.tensor(modes, dtype=torch.uint8, device=dev),
                                  sink=0, window=16, workspace=ws)
        assert ea.ea_check_errors(ws) == 6
        assert ea.ea_check_errors(ws) == 0            # the word is cleared by the read


def _full_size(dev, cfg, m, bm=None, n_random=64):
    """Run one layer of a full-size workload and check sampled rows."""
    Qd, Kd, Vd = wl.qkv(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.d, seed=cfg.seed, device=dev)
    nB = (cfg.S + 127) // 128
    vis = torch.zeros((cfg.B * cfg.Hkv * nB * nB + 31) // 32, dtype=torch.int32, device=dev)
    ws = ea.prefill_workspace(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, device=dev)
    O, LSE = ea.ea_hybrid_attn_prefill(Qd, Kd, Vd, m.to(dev), sink=cfg.sink, window=cfg.window,
                                       block_mask=None if bm is None else bm.to(dev),
                                       workspace=ws, visited_bitmap=vis)
    torch.cuda.synchronize()
    check_no_device_error(ws)
    Q, K, V = Qd.cpu(), Kd.cpu(), Vd.cpu()
    del Qd, Kd, Vd
    srows = sample_rows(cfg.S, cfg.sink, cfg.window, n_random=n_random, edge=64)
    rows = np.array([[b, qh, i] for b in range(cfg.B) for qh in range(cfg.Hq) for i in srows])
    Oref, Lref = oracle.prefill_rows(Q, K, V, m, rows, sink=cfg.sink, window=cfg.window,
                                     block_mask=bm)
    idx = torch.from_numpy(rows).to(O.device)
    Og = O[idx[:, 0], idx[:, 2], idx[:, 1]].float().cpu().numpy()
    Lg = LSE[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy()
    assert_close(Og, Lg, Oref, Lref, cfg.name, flat=True)   # a benchmark workload: flat 1e-2
    # visited tiles of a few query blocks, bit-exact
    tiles = bitmap_to_tiles(vis, cfg.B, cfg.Hkv, nB)
    for qb in (0, 1, nB // 2, nB - 1):
        ref = oracle.visited(cfg.B, cfg.S, cfg.Hkv, m, sink=cfg.sink, window=cfg.window,
                             block_mask=bm, qb_begin=qb, qb_end=qb + 1)
        np.testing.assert_array_equal(tiles[:, :, qb:qb + 1], ref)
    return O, LSE


def test_llama_32k_layer_sampled_rows(dev):
    cfg = wl.LLAMA_32K
    _, m = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads)
    _full_size(dev, cfg, m)


def test_xa_ssa_256k_sampled_rows(dev):
    cfg = wl.XA_SSA_256K
    _, m = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads, fa_impl=BLOCK, sa_impl=SSA)
    bm = wl.block_mask(cfg.B, cfg.Hkv, cfg.S, density=cfg.block_density, seed=cfg.seed)
    _full_size(dev, cfg, m, bm=bm, n_random=32)


def test_serial_dispatch_matches_fused_launch(dev):
    # Algorithm 1(a) (split heads, one launch per group, scatter back) must give
    # exactly what the single fused launch gives: every head's computation is
    # the same, only the dispatch differs.
    import bench
    B, S, Hq, Hkv = 1, 1500, 16, 4
    Q, K, V = (t.to(dev) for t in wl.qkv(B, S, Hq, Hkv, 128, seed=31))
    m_cpu = torch.tensor([[SSA, FULL, SSA, SSA]], dtype=torch.uint8)
    O1, L1 = ea.ea_hybrid_attn_prefill(Q, K, V, m_cpu.to(dev), sink=64, window=300)
    O2 = torch.empty_like(O1)
    L2 = torch.empty_like(L1)
    wss = [ea.prefill_workspace(B, S, Hq, Hkv, device=dev) for _ in range(2)]
    bench.serial_dispatch(ea, Q, K, V, m_cpu, 64, 300, O2, L2, *wss)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    # and both against the oracle, every row
    Oref, Lref = oracle.prefill_full(Q.cpu(), K.cpu(), V.cpu(), m_cpu, sink=64, window=300)
    assert_close(O2.float().cpu().numpy(), L2.cpu().numpy(), Oref, Lref, "serial dispatch")


def test_qwen3_64k_routed_layer_sampled_rows(dev):
    # One layer of the 36-layer 64K workload: the modes come from the oracle
    # router on that layer's K (boundary tokens), then the fused prefill runs
    # with them at full size; sampled rows are checked.  The first layer whose
    # routing is mixed (some FA and some SA heads) is used.
    import dataclasses
    cfg = wl.QWEN_64K_36L
    for layer in range(cfg.layers):
        Kd = wl.randn_bf16((cfg.B, cfg.S, cfg.Hkv, cfg.d), seed=3 * (cfg.seed + layer) + 1, device=dev)
        W, b = wl.router_weights(layer, d=cfg.d, hidden=64, seed=cfg.seed, beta=0.0015)
        Kb = torch.cat([Kd[:, :100], Kd[:, -100:]], dim=1).cpu()
        r, m, _, _ = oracle.route(Kb, W, b, pool_head=100, pool_tail=100)
        if 0 < int(r.sum()) < cfg.Hkv:
            break
    else:
        pytest.skip("no layer with mixed routing at this output bias")
    del Kd
    c = dataclasses.replace(cfg, seed=cfg.seed + layer)
    _full_size(dev, c, torch.from_numpy(m), n_random=32)


def test_one_plan_feeds_several_launches(dev):
    # ea_prefill_plan once, ea_prefill_attend twice on other inputs: the queue
    # re-arms itself after each launch and both results match the oracle.
    B, S, Hq, Hkv = 1, 700, 8, 2
    modes = torch.tensor([[FULL, SSA]], dtype=torch.uint8, device=dev)
    ws = ea.prefill_workspace(B, S, Hq, Hkv, device=dev)
    ea.ea_prefill_plan(B, S, Hq, Hkv, modes, sink=16, window=200, workspace=ws)
    for seed in (41, 42):
        Q, K, V = wl.qkv(B, S, Hq, Hkv, 128, seed=seed)
        O, LSE = ea.ea_prefill_attend(Q.to(dev), K.to(dev), V.to(dev), modes, sink=16, window=200,
                                      workspace=ws)
        torch.cuda.synchronize()
        check_no_device_error(ws)
        Oref, Lref = oracle.prefill_full(Q, K, V, modes.cpu(), sink=16, window=200)
        assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "seed %d" % seed)


def test_random_small_configurations(dev):
    # Seeded sweep over ragged lengths, group sizes, mixed modes per head,
    # sink/window settings and block masks; every row against the oracle.
    rng = np.random.default_rng(2024)
    for case in range(12):
        B = int(rng.integers(1, 3))
        S = int(rng.integers(1, 700))
        Hkv = int(rng.integers(1, 4))
        g = int(rng.integers(1, 5))
        Hq = Hkv * g
        sink = int(rng.integers(0, 200))
        window = int(rng.integers(1, 400))
        modes = rng.integers(0, 3, size=(B, Hkv)).astype(np.uint8)
        Q, K, V = wl.qkv(B, S, Hq, Hkv, 128, seed=1000 + case)
        bm = wl.block_mask(B, Hkv, S, density=float(rng.uniform(0.1, 0.9)), seed=case).numpy()
        bm[rng.random(bm.shape) < 0.1] = 0            # drop some diagonal / first blocks too
        O, LSE, vis = run(dev, Q, K, V, modes, sink, window, bm=bm, visited=True)
        Oref, Lref = oracle.prefill_full(Q, K, V, modes, sink=sink, window=window, block_mask=bm)
        what = "case %d (B=%d S=%d Hq=%d Hkv=%d sink=%d window=%d modes=%s)" % (
            case, B, S, Hq, Hkv, sink, window, modes.tolist())
        assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, what)
        nB = (S + 127) // 128
        np.testing.assert_array_equal(
            bitmap_to_tiles(vis, B, Hkv, nB),
            oracle.visited(B, S, Hkv, modes, sink=sink, window=window, block_mask=bm), err_msg=what)


def test_longest_supported_sequence(dev):
    # S = 2^21 (the planner's limit): streaming heads only, sampled rows.
    B, S, Hq, Hkv, sink, window = 1, 1 << 21, 2, 1, 128, 300
    Qd, Kd, Vd = wl.qkv(B, S, Hq, Hkv, 128, seed=77, device=dev)
    m = torch.tensor([[SSA]], dtype=torch.uint8)
    ws = ea.prefill_workspace(B, S, Hq, Hkv, device=dev)
    O, LSE = ea.ea_hybrid_attn_prefill(Qd, Kd, Vd, m.to(dev), sink=sink, window=window, workspace=ws)
    torch.cuda.synchronize()
    check_no_device_error(ws)
    rows_i = np.array([0, 1, 127, 128, 299, 300, 301, 4095, S // 2, S - 129, S - 1], dtype=np.int64)
    rows = np.array([[0, qh, i] for qh in range(Hq) for i in rows_i])
    Oref, Lref = oracle.prefill_rows(Qd.cpu(), Kd.cpu(), Vd.cpu(), m, rows, sink=sink, window=window)
    idx = torch.from_numpy(rows).to(dev)
    assert_close(O[idx[:, 0], idx[:, 2], idx[:, 1]].float().cpu().numpy(),
                 LSE[idx[:, 0], idx[:, 1], idx[:, 2]].cpu().numpy(), Oref, Lref, "S=2^21")
    with pytest.raises(ValueError):
        ea.prefill_workspace(B, S + 1, Hq, Hkv, device=dev)


def test_random_configurations_wider(dev):
    # A second seeded sweep, longer sequences and group sizes up to 5; it holds
    # rows whose outputs reach |O| > 2 (few kept keys), where bf16 output
    # rounding matters for the tolerance.
    rng = np.random.default_rng(777)
    for case in range(30):
        B = int(rng.integers(1, 4))
        S = int(rng.integers(1, 1200))
        Hkv = int(rng.integers(1, 4))
        g = int(rng.integers(1, 6))
        Hq = Hkv * g
        sink = int(rng.integers(0, 300))
        window = int(rng.integers(1, 700))
        modes = rng.integers(0, 3, size=(B, Hkv)).astype(np.uint8)
        density = float(rng.uniform(0.1, 0.9))
        drop = rng.random((B, Hkv, (S + 127) // 128, (S + 127) // 128)) < 0.1
        Q, K, V = wl.qkv(B, S, Hq, Hkv, 128, seed=5000 + case)
        bm = wl.block_mask(B, Hkv, S, density=density, seed=case).numpy()
        bm[drop] = 0
        O, LSE, vis = run(dev, Q, K, V, modes, sink, window, bm=bm, visited=True)
        Oref, Lref = oracle.prefill_full(Q, K, V, modes, sink=sink, window=window, block_mask=bm)
        what = "case %d (B=%d S=%d Hq=%d Hkv=%d sink=%d window=%d)" % (case, B, S, Hq, Hkv, sink, window)
        assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, what)
        nB = (S + 127) // 128
        np.testing.assert_array_equal(
            bitmap_to_tiles(vis, B, Hkv, nB),
            oracle.visited(B, S, Hkv, modes, sink=sink, window=window, block_mask=bm), err_msg=what)


def test_random_configurations_offset_values(dev):
    # V with a large common offset (|v| in [2.2, 3.8), one sign per head
    # dimension): the softmax average keeps |O| near 3, where the output's own
    # rounding leaves least room under 1e-2, and each probability's rounding
    # error reaches O with the offset's weight unless it averages out over many
    # keys.  Every element must be within a flat 1e-2 (rows of up to 512 kept
    # keys take P V in two bf16 parts).
    rng = np.random.default_rng(4242)
    for case in range(30):
        B = int(rng.integers(1, 3))
        S = int(rng.integers(1, 1200))
        Hkv = int(rng.integers(1, 4))
        Hq = Hkv * int(rng.integers(1, 6))
        sink = int(rng.integers(0, 400))
        window = int(rng.integers(1, 900))
        modes = rng.integers(0, 3, size=(B, Hkv)).astype(np.uint8)
        Q, K, _ = wl.qkv(B, S, Hq, Hkv, 128, seed=6000 + case)
        V = wl.offset_values(B, S, Hkv, 128, seed=6500 + case)
        bm = wl.block_mask(B, Hkv, S, density=float(rng.uniform(0.05, 0.9)), seed=case).numpy()
        bm[rng.random(bm.shape) < 0.15] = 0
        O, LSE, _ = run(dev, Q, K, V, modes, sink, window, bm=bm)
        Oref, Lref = oracle.prefill_full(Q, K, V, modes, sink=sink, window=window, block_mask=bm)
        assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref,
                     "offset V, case %d (B=%d S=%d Hq=%d Hkv=%d sink=%d window=%d)"
                     % (case, B, S, Hq, Hkv, sink, window), flat=True)




def test_dominant_key_beyond_the_running_maximum(dev):
    # Rows 600..1023 keep key 0 (score 0, the first tile's maximum), key 600,
    # whose score is 5.005 higher (log2 units; within the lazy rescale's
    # threshold, so the running maximum stays at key 0's score), and keys far
    # below.  Key 600's probability 2^5.005 = 32.115 is rounded to 32.0 in bf16
    # (-0.36 %) and carries 97 % of the weight; with v = -3.875 against key 0's
    # +3.875 a copy of the kernel without the normaliser's correction is 0.0152
    # off the oracle (an fp64 model of that arithmetic: 0.0151).  These query
    # blocks keep more than 512 keys, so no remainder product applies; the
    # normaliser takes the rounding of the tile's largest probability, which
    # makes the weights exact: every element within a flat 1e-2.
    S, d = 1024, 128
    Q = torch.zeros(1, S, 1, d)
    K = torch.zeros(1, S, 1, d)
    V = torch.zeros(1, S, 1, d)
    Q[0, :, 0, 0] = 1.0
    K[0, 1:, 0, 0] = -128.0         # every other key far below
    K[0, 600, 0, 0] = 39.25         # 39.25 / sqrt(128) * log2(e) = 5.005
    V[0, 0, 0, :] = 3.875
    V[0, 600, 0, :] = -3.875
    Q, K, V = (t.to(torch.bfloat16) for t in (Q, K, V))
    modes = [[FULL]]
    O, LSE, _ = run(dev, Q, K, V, modes, 0, S)
    Oref, Lref = oracle.prefill_full(Q, K, V, np.array(modes, np.uint8), sink=0, window=S)
    assert_close(O.float().cpu().numpy(), LSE.cpu().numpy(), Oref, Lref, "dominant key", flat=True)
    assert abs(float(O[0, 700, 0, 0]) + 3.64) < 0.05    # the dominant key's value does dominate
