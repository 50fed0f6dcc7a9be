"""The entry points inside CUDA graphs: a call captured once and replayed with
new input values (written into the same buffers) must give exactly what an
eager call on those values gives.  Serving engines run decode steps this way."""
import numpy as np
import pytest
import torch

import sparse_head_attention_gb300 as ea
from sparse_head_attention_gb300 import workloads as wl
from gpu_helpers import check_no_device_error, gpu_device

pytestmark = pytest.mark.gpu
FULL, SSA = ea.FULL, ea.SSA


@pytest.fixture(scope="module")
def dev():
    return gpu_device()


def capture(fn):
    """Warm up on a side stream (first-call attribute setup happens outside
    the capture), then capture one call."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_step_replayed(dev):
    cfg = wl.DecodeConfig("t", B=4, Hq=16, Hkv=4, d=128, L=3000, sink=64, window=700)
    q, Kc, Vc, sl = wl.decode_inputs(cfg, device=dev, seqlens=[3000, 17, 1500, 2049])
    m = torch.tensor([[FULL, SSA, SSA, FULL]] * 4, dtype=torch.uint8, device=dev)
    ws = ea.decode_workspace(cfg.B, cfg.Hq, cfg.Hkv, cfg.L, device=dev)
    O = torch.empty_like(q)
    LSE = torch.empty(cfg.B, cfg.Hq, dtype=torch.float32, device=dev)

    def step():
        ea.ea_hybrid_attn_decode(q, Kc, Vc, sl, m, sink=cfg.sink, window=cfg.window, O=O, LSE=LSE,
                                 workspace=ws)

    g = capture(step)
    for seed in (5, 6, 7):
        q.copy_(wl.randn_bf16(q.shape, seed=seed, device=dev))
        sl.copy_(torch.tensor([3000 - seed, 1 + seed, 1500, 2049 + seed], dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        Og, Lg = O.clone(), LSE.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(Og, O) and torch.equal(Lg, LSE), seed
    check_no_device_error(ws)


def test_prefill_replayed(dev):
    B, S, Hq, Hkv = 1, 1500, 8, 2
    Q, K, V = (t.to(dev) for t in wl.qkv(B, S, Hq, Hkv, 128, seed=40))
    m = torch.tensor([[FULL, SSA]], dtype=torch.uint8, device=dev)
    ws = ea.prefill_workspace(B, S, Hq, Hkv, device=dev)
    O = torch.empty_like(Q)
    LSE = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)

    def step():
        ea.ea_hybrid_attn_prefill(Q, K, V, m, sink=32, window=400, O=O, LSE=LSE, workspace=ws)

    g = capture(step)
    for seed in (41, 42):
        Q.copy_(wl.randn_bf16(Q.shape, seed=seed, device=dev))
        m.copy_(torch.tensor([[SSA, FULL]] if seed == 42 else [[FULL, SSA]], dtype=torch.uint8))
        g.replay()
        torch.cuda.synchronize()
        Og, Lg = O.clone(), LSE.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(Og, O) and torch.equal(Lg, LSE), seed
    check_no_device_error(ws)


def test_varlen_prefill_and_router_replayed(dev):
    lens = [700, 1, 300]
    total, Hq, Hkv = sum(lens), 8, 2
    Q = wl.randn_bf16((total, Hq, 128), seed=50, device=dev)
    K = wl.randn_bf16((total, Hkv, 128), seed=51, device=dev)
    V = wl.randn_bf16((total, Hkv, 128), seed=52, device=dev)
    cu = torch.tensor([0, 700, 701, 1001], dtype=torch.int32, device=dev)
    m = torch.tensor([[FULL, SSA]] * 3, dtype=torch.uint8, device=dev)
    ws = ea.prefill_varlen_workspace(3, total, 700, Hq, Hkv, device=dev)
    O = torch.empty_like(Q)
    LSE = torch.empty(Hq, total, dtype=torch.float32, device=dev)
    Kr = wl.randn_bf16((1, 4096, 8, 128), seed=53, device=dev)
    W, b = wl.router_weights(0, d=128, hidden=64, device=dev)
    r = torch.empty(1, 8, dtype=torch.uint8, device=dev)
    mr = torch.empty_like(r)
    lg = torch.empty(1, 8, 2, dtype=torch.float64, device=dev)

    def step():
        ea.ea_hybrid_attn_prefill_varlen(Q, K, V, cu, m, max_seqlen=700, sink=16, window=128, O=O,
                                         LSE=LSE, workspace=ws)
        ea.ea_route(Kr, W, b, r_out=r, m_out=mr, logits_out=lg)

    g = capture(step)
    for seed in (54, 55):
        Q.copy_(wl.randn_bf16(Q.shape, seed=seed, device=dev))
        Kr.copy_(wl.randn_bf16(Kr.shape, seed=seed + 10, device=dev))
        g.replay()
        torch.cuda.synchronize()
        Og, Lg, lgg = O.clone(), LSE.clone(), lg.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(Og, O) and torch.equal(Lg, LSE) and torch.equal(lgg, lg), seed
    check_no_device_error(ws)


def test_xa_ssa_estimation_prefill_and_decode_replayed(dev):
    """XA-SSA in one graph: block-mask estimation from Q and K, the fused prefill
    on the estimated masks, then a decode step whose BLOCK head reads them."""
    BLOCK = ea.BLOCK
    B, S, Hq, Hkv = 1, 2048, 8, 2
    Qc, Kc = wl.xa_planted_qk(B, S, Hq, Hkv, 128, seed=50)
    Q, K = Qc.to(dev), Kc.to(dev)
    V = wl.randn_bf16((B, S, Hkv, 128), seed=51, device=dev)
    m = torch.tensor([[BLOCK, SSA]], dtype=torch.uint8, device=dev)
    nB = S // 128
    xws = ea.xa_workspace(B, S, Hq, Hkv, 1, device=dev)
    pws = ea.prefill_workspace(B, S, Hq, Hkv, device=dev)
    dws = ea.decode_workspace(B, Hq, Hkv, S, device=dev)
    bm = torch.zeros(B, Hkv, nB, nB, dtype=torch.uint8, device=dev)
    sc = torch.zeros(B, Hkv, nB, nB, dtype=torch.float32, device=dev)
    O = torch.empty_like(Q)
    LSE = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
    q = torch.empty(B, Hq, 128, dtype=torch.bfloat16, device=dev)
    sl = torch.tensor([S], dtype=torch.int32, device=dev)
    Od = torch.empty_like(q)
    Ld = torch.empty(B, Hq, dtype=torch.float32, device=dev)

    def step():
        ea.ea_xa_estimate(Q, K, m, max_units=1, block_mask=bm, block_scores=sc, workspace=xws)
        ea.ea_hybrid_attn_prefill(Q, K, V, m, sink=64, window=256, block_mask=bm, O=O, LSE=LSE,
                                  workspace=pws)
        ea.ea_hybrid_attn_decode(q, K, V, sl, m, sink=64, window=256, block_mask=bm, O=Od, LSE=Ld,
                                 workspace=dws)

    q.copy_(Q[:, S - 1])
    g = capture(step)
    for seed in (52, 53):
        Qn, Kn = wl.xa_planted_qk(B, S, Hq, Hkv, 128, seed=seed)
        Q.copy_(Qn.to(dev))
        K.copy_(Kn.to(dev))
        q.copy_(Q[:, S - 1])
        sl.fill_(S - seed)
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (bm, sc, O, LSE, Od, Ld)]
        step()
        torch.cuda.synchronize()
        for a_, b_ in zip(got, (bm, sc, O, LSE, Od, Ld)):
            assert torch.equal(a_, b_), seed
    for ws in (xws, pws, dws):
        check_no_device_error(ws)


def test_several_layers_in_one_launch_replayed(dev):
    # ea_hybrid_attn_prefill_layers inside a graph: the layers' pointers and
    # tensor maps travel as kernel parameters, so a replay with new values in
    # the same buffers equals an eager call
    L, B, S, Hq, Hkv = 3, 1, 700, 8, 2
    Qs, Ks, Vs = [], [], []
    for l in range(L):
        Q, K, V = (t.to(dev) for t in wl.qkv(B, S, Hq, Hkv, 128, seed=500 + l))
        Qs.append(Q), Ks.append(K), Vs.append(V)
    ms = [torch.tensor([[FULL, SSA]], dtype=torch.uint8, device=dev) for _ in range(L)]
    Os = [torch.empty_like(q) for q in Qs]
    LSEs = [torch.empty(B, Hq, S, dtype=torch.float32, device=dev) for _ in range(L)]
    ws = ea.prefill_layers_workspace(L, B, S, Hq, Hkv, device=dev)

    def step():
        ea.ea_hybrid_attn_prefill_layers(Qs, Ks, Vs, ms, sink=16, window=200, Os=Os, LSEs=LSEs,
                                         workspace=ws)

    g = capture(step)
    for seed in (510, 511):
        for l in range(L):
            Qs[l].copy_(wl.randn_bf16(Qs[l].shape, seed=seed + l, device=dev))
            ms[l].copy_(torch.tensor([[SSA, FULL]] if (seed + l) % 2 else [[FULL, SSA]],
                                     dtype=torch.uint8))
        g.replay()
        torch.cuda.synchronize()
        got = [(o.clone(), s.clone()) for o, s in zip(Os, LSEs)]
        step()
        torch.cuda.synchronize()
        for l in range(L):
            assert torch.equal(got[l][0], Os[l]) and torch.equal(got[l][1], LSEs[l]), (seed, l)
    check_no_device_error(ws)
