"""Parity of the router pre-pass (CUDA, through the C ABI) with the fp64 oracle:
hand-computed examples and the 36-layer 64K workload.  Routing decisions, modes
and the logits themselves are compared bit for bit (both sides pool exactly and
evaluate the MLP in fp64 in index order without fused multiply-adds)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import sparse_head_attention_gb300 as ea
from sparse_head_attention_gb300 import workloads as wl
from gpu_helpers import gpu_device

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def dev():
    return gpu_device()


def _cases():
    with open(os.path.join(GOLDEN, "router_hand_examples.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_examples(dev, case):
    # head dim 2 is below the library's attention limit but the router takes any d
    K = torch.tensor(case["K"], dtype=torch.float32).to(torch.bfloat16)[None].to(dev)
    Ws = [torch.tensor(w, dtype=torch.float32, device=dev) for w in case["W"]]
    bs = [torch.tensor(b, dtype=torch.float32, device=dev) for b in case["b"]]
    r, m, logits = ea.ea_route(K, Ws, bs, pool_head=case["pool_head"], pool_tail=case["pool_tail"],
                               policy=(ea.BLOCK, ea.SSA))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(r[0].cpu().numpy(), np.array(case["r"], np.uint8))
    np.testing.assert_array_equal(m[0].cpu().numpy(), np.where(np.array(case["r"]) == 1, ea.SSA, ea.BLOCK))
    np.testing.assert_array_equal(logits[0].cpu().numpy(), np.array(case["logits"], np.float64))


def test_36_layer_64k_workload_bit_exact(dev):
    cfg = wl.QWEN_64K_36L
    for layer in range(cfg.layers):
        K = wl.randn_bf16((cfg.B, cfg.S, cfg.Hkv, cfg.d), seed=3 * (cfg.seed + layer) + 1, device=dev)
        W, b = wl.router_weights(layer, d=cfg.d, hidden=64, seed=cfg.seed, beta=0.0015, device=dev)
        r, m, logits = ea.ea_route(K, W, b)
        torch.cuda.synchronize()
        # the oracle pools the same 200 boundary tokens, handed over as a 200-token sequence
        Kb = torch.cat([K[:, :100], K[:, -100:]], dim=1).cpu()
        ro, mo, lo, _ = oracle.route(Kb, [w.cpu() for w in W], [x.cpu() for x in b],
                                     pool_head=100, pool_tail=100)
        np.testing.assert_array_equal(logits.cpu().numpy(), lo)
        np.testing.assert_array_equal(r.cpu().numpy(), ro)
        np.testing.assert_array_equal(m.cpu().numpy(), mo)
        assert np.abs(lo[..., 1] - lo[..., 0]).min() > 1e-9     # decisions are not near ties


def test_route_layers_two_launches_mixed_mlps(dev):
    # 70 layers take two launches (64 + 6); layers alternate between a 1-layer,
    # a 2-layer and a 3-layer MLP, and pooling windows overlap (S < 200).
    L, B, S, Hkv, d = 70, 3, 150, 2, 128
    stack = wl.randn_bf16((L, B, S, Hkv, d), seed=77, device=dev)
    Ks = [stack[l] for l in range(L)]
    Ws, bs = [], []
    g = torch.Generator().manual_seed(78)
    for l in range(L):
        dims = [[d, 2], [d, 64, 2], [d, 32, 16, 2]][l % 3]
        Ws.append([(torch.randn(o, i, generator=g) * 0.05).float().to(dev)
                   for i, o in zip(dims[:-1], dims[1:])])
        bs.append([(torch.randn(o, generator=g) * 0.01).float().to(dev) for o in dims[1:]])
    r, m, logits = ea.ea_route_layers(Ks, Ws, bs, policy=(ea.BLOCK, ea.SSA))
    torch.cuda.synchronize()
    r, m, logits = r.cpu().numpy(), m.cpu().numpy(), logits.cpu().numpy()
    for l in range(L):
        ro, mo, lo, _ = oracle.route(Ks[l].cpu(), [w.cpu() for w in Ws[l]], [x.cpu() for x in bs[l]],
                                     pool_head=100, pool_tail=100, fa_impl=ea.BLOCK, sa_impl=ea.SSA)
        np.testing.assert_array_equal(logits[l], lo, err_msg="layer %d" % l)
        np.testing.assert_array_equal(r[l], ro, err_msg="layer %d" % l)
        np.testing.assert_array_equal(m[l], mo, err_msg="layer %d" % l)


def test_route_layers_equals_per_layer_route_on_64k_workload(dev):
    cfg = wl.QWEN_64K_36L
    Ks = [wl.randn_bf16((cfg.B, cfg.S, cfg.Hkv, cfg.d), seed=3 * (cfg.seed + l) + 1, device=dev)
          for l in range(cfg.layers)]
    wb = [wl.router_weights(l, d=cfg.d, hidden=64, seed=cfg.seed, beta=0.0015, device=dev)
          for l in range(cfg.layers)]
    r, m, logits = ea.ea_route_layers(Ks, [w for w, _ in wb], [b for _, b in wb])
    for l in range(cfg.layers):
        r1, m1, lg1 = ea.ea_route(Ks[l], *wb[l])
        torch.cuda.synchronize()
        assert torch.equal(logits[l], lg1) and torch.equal(r[l], r1) and torch.equal(m[l], m1), l
    # one layer against the oracle as well, on its 200 boundary tokens
    Kb = torch.cat([Ks[5][:, :100], Ks[5][:, -100:]], dim=1).cpu()
    _, _, lo, _ = oracle.route(Kb, [w.cpu() for w in wb[5][0]], [x.cpu() for x in wb[5][1]])
    np.testing.assert_array_equal(logits[5].cpu().numpy(), lo)


def _extreme_K(seed, B=2, S=300, Hkv=2, d=128):
    """K whose channels span the cases of the router's exact pooling: ordinary
    N(0, 1) values, exponent spreads wide enough that the sequential fp64 sum
    rounds, a spread just inside 2^53, bf16 subnormals, and signed zeros."""
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((B, S, Hkv, d)).astype(np.float32)
    # channels 8..39: magnitudes 2^-120 .. 2^120 with random signs
    K[..., 8:40] = (rng.choice([-1.0, 1.0], size=K[..., 8:40].shape) *
                    np.exp2(rng.integers(-120, 121, size=K[..., 8:40].shape))).astype(np.float32)
    # channel 40: 2^40 once among 2^-7 values -> beyond 2^53 quanta, fp64 rounds
    K[..., 40] = 2.0 ** -7
    K[:, 150, :, 40] = 2.0 ** 40
    # channel 41: 2^30 among 2^-10 values -> exact in fp64 (not in fp32)
    K[..., 41] = 2.0 ** -10
    K[:, 20, :, 41] = 2.0 ** 30
    # channel 42: bf16 subnormals and the smallest normal
    K[..., 42] = rng.choice([2.0 ** -133, -3 * 2.0 ** -133, 2.0 ** -126, 0.0], size=K[..., 42].shape)
    # channel 43: signed zeros only; channel 44: +x and -x pairs that cancel exactly
    K[..., 43] = rng.choice([0.0, -0.0], size=K[..., 43].shape)
    K[:, 0::2, :, 44] = 3.25
    K[:, 1::2, :, 44] = -3.25
    return torch.from_numpy(K).to(torch.bfloat16)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_pooling_extreme_values_bit_exact(dev, seed):
    K = _extreme_K(seed)
    W, b = wl.router_weights(seed, d=128, hidden=64, device=dev)
    r, m, logits = ea.ea_route(K.to(dev), W, b)
    torch.cuda.synchronize()
    ro, mo, lo, _ = oracle.route(K, [w.cpu() for w in W], [x.cpu() for x in b])
    np.testing.assert_array_equal(logits.cpu().numpy(), lo)
    np.testing.assert_array_equal(r.cpu().numpy(), ro)
    # the same through a 1-layer MLP that passes two pooled channels straight
    # to the logits, so each pooled value is compared on its own
    for c0, c1 in ((40, 41), (42, 43), (44, 8), (9, 10), (0, 1)):
        W1 = torch.zeros(2, 128)
        W1[0, c0] = 1.0
        W1[1, c1] = 1.0
        _, _, lg = ea.ea_route(K.to(dev), [W1.to(dev)], [torch.zeros(2, device=dev)])
        torch.cuda.synchronize()
        _, _, lo1, pooled = oracle.route(K, [W1], [torch.zeros(2)])
        np.testing.assert_array_equal(lg.cpu().numpy(), lo1, err_msg="channels %d,%d" % (c0, c1))
        np.testing.assert_array_equal(lg.cpu().numpy()[..., 0], pooled[..., c0])


def test_pooling_infinite_and_nan_values(dev):
    K = _extreme_K(5).float()
    K[0, 10, 0, 3] = float("inf")
    K[1, 290, 1, 4] = float("nan")
    K[1, 20, 0, 5] = float("-inf")
    K = K.to(torch.bfloat16)
    for c0, c1 in ((3, 4), (5, 6)):
        W1 = torch.zeros(2, 128)
        W1[0, c0] = 1.0
        W1[1, c1] = 1.0
        _, _, lg = ea.ea_route(K.to(dev), [W1.to(dev)], [torch.zeros(2, device=dev)])
        torch.cuda.synchronize()
        _, _, lo1, _ = oracle.route(K, [W1], [torch.zeros(2)])
        got, want = lg.cpu().numpy(), lo1
        assert np.array_equal(np.isnan(got), np.isnan(want))
        np.testing.assert_array_equal(np.nan_to_num(got), np.nan_to_num(want))
