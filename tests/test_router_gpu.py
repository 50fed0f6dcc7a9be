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
