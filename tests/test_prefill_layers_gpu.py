"""Several layers in one planner + one persistent launch
(ea_hybrid_attn_prefill_layers): every layer's output must equal, bit for bit,
the single-layer prefill of that layer (the same items computed the same way,
only queued together), and match the fp64 oracle."""
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


def _same(a, b):
    assert torch.equal(a, b)


def test_mixed_layers_equal_single_layer_calls_and_oracle(dev):
    L, B, S, Hq, Hkv, sink, window = 5, 2, 700, 12, 3, 20, 150
    rng = np.random.default_rng(5)
    Qs, Ks, Vs, ms, bms = [], [], [], [], []
    for l in range(L):
        Q, K, V = wl.qkv(B, S, Hq, Hkv, 128, seed=300 + l)
        Qs.append(Q), Ks.append(K), Vs.append(V)
        ms.append(torch.from_numpy(rng.integers(0, 3 if l % 2 == 0 else 2, size=(B, Hkv)).astype(np.uint8)))
        bms.append(wl.block_mask(B, Hkv, S, density=0.4, seed=l) if l % 2 == 0 else None)
    d = lambda t: None if t is None else t.to(dev)
    ws = ea.prefill_layers_workspace(L, B, S, Hq, Hkv, device=dev)
    Os, LSEs = ea.ea_hybrid_attn_prefill_layers([d(q) for q in Qs], [d(k) for k in Ks], [d(v) for v in Vs],
                                                [d(m) for m in ms], sink=sink, window=window,
                                                block_masks=[d(b) for b in bms], workspace=ws)
    torch.cuda.synchronize()
    check_no_device_error(ws)
    for l in range(L):
        O1, L1 = ea.ea_hybrid_attn_prefill(d(Qs[l]), d(Ks[l]), d(Vs[l]), d(ms[l]), sink=sink, window=window,
                                           block_mask=d(bms[l]))
        torch.cuda.synchronize()
        _same(Os[l], O1)
        _same(LSEs[l], L1)
    for l in (0, 3):
        Oref, Lref = oracle.prefill_full(Qs[l], Ks[l], Vs[l], ms[l], sink=sink, window=window,
                                         block_mask=None if bms[l] is None else bms[l].numpy())
        assert_close(Os[l].float().cpu().numpy(), LSEs[l].cpu().numpy(), Oref, Lref, "layer %d" % l)


def test_36_layers_at_4k_equal_single_layer_calls(dev):
    # the 36-layer stack's shape at a short length: one launch for all layers
    L, B, S, Hq, Hkv = 36, 1, 4096, 32, 8
    Qs = [wl.randn_bf16((B, S, Hq, 128), seed=3 * l, device=dev) for l in range(L)]
    Ks = [wl.randn_bf16((B, S, Hkv, 128), seed=3 * l + 1, device=dev) for l in range(L)]
    Vs = [wl.randn_bf16((B, S, Hkv, 128), seed=3 * l + 2, device=dev) for l in range(L)]
    g = torch.Generator().manual_seed(9)
    ms = [(torch.rand(B, Hkv, generator=g) < 0.75).to(torch.uint8).to(dev) for _ in range(L)]  # SSA share ~0.75
    Os, LSEs = ea.ea_hybrid_attn_prefill_layers(Qs, Ks, Vs, ms, sink=128, window=2048)
    torch.cuda.synchronize()
    for l in range(L):
        O1, L1 = ea.ea_hybrid_attn_prefill(Qs[l], Ks[l], Vs[l], ms[l], sink=128, window=2048)
        torch.cuda.synchronize()
        _same(Os[l], O1)
        _same(LSEs[l], L1)


def test_too_many_layers_and_bad_layer_are_rejected(dev):
    B, S, Hq, Hkv = 1, 256, 8, 2
    Q, K, V = (t.to(dev) for t in wl.qkv(B, S, Hq, Hkv, 128, seed=1))
    m = torch.zeros(B, Hkv, dtype=torch.uint8, device=dev)
    n = ea.MAX_PREFILL_LAYERS + 1
    with pytest.raises(ValueError):        # no workspace size for that many layers
        ea.prefill_layers_workspace(n, B, S, Hq, Hkv, device=dev)
    ws = ea.prefill_layers_workspace(2, B, S, Hq, Hkv, device=dev)
    with pytest.raises(ea.EAError) as e:   # the library refuses the layer count itself
        ea.ea_hybrid_attn_prefill_layers([Q] * n, [K] * n, [V] * n, [m] * n, sink=0, window=64,
                                         workspace=ws)
    assert e.value.status == 2
    with pytest.raises(ValueError):
        ea.ea_hybrid_attn_prefill_layers([Q, Q[:, :128]], [K, K], [V, V], [m, m], sink=0, window=64)
