"""The prefill on host tensors (ea_hybrid_attn_prefill_host): chunked copies
overlapped with the attention must give exactly what the device-buffer entry
point gives, for every chunk count, ragged lengths, batches, block masks,
pageable and page-locked memory, and the full 32K workload."""
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


def _device_reference(dev, Q, K, V, m, sink, window, bm):
    O, LSE = ea.ea_hybrid_attn_prefill(Q.to(dev), K.to(dev), V.to(dev), m.to(dev), sink=sink,
                                       window=window, block_mask=None if bm is None else bm.to(dev))
    torch.cuda.synchronize()
    return O.cpu(), LSE.cpu()


@pytest.mark.parametrize("B,S,Hq,Hkv,n_chunks,pinned,use_bm", [
    (1, 1000, 8, 2, 0, True, False),
    (1, 1000, 8, 2, 1, True, False),
    (1, 1000, 8, 2, 3, False, False),
    (2, 700, 12, 4, 6, True, True),
    (2, 700, 12, 4, 0, False, True),
    (1, 129, 4, 4, 2, True, False),
    (3, 513, 6, 2, 5, True, True),
])
def test_equals_device_entry_point(dev, B, S, Hq, Hkv, n_chunks, pinned, use_bm):
    Q, K, V = wl.qkv(B, S, Hq, Hkv, 128, seed=31 + S)
    modes = [FULL, SSA, BLOCK, SSA] if use_bm else [FULL, SSA, SSA, FULL]
    m = torch.tensor([[modes[(b + h) % 4] for h in range(Hkv)] for b in range(B)], dtype=torch.uint8)
    bm = wl.block_mask(B, Hkv, S, density=0.4, seed=7) if use_bm else None
    sink, window = 64, 300
    Oref, Lref = _device_reference(dev, Q, K, V, m, sink, window, bm)
    if pinned:
        Q, K, V = Q.pin_memory(), K.pin_memory(), V.pin_memory()
    buf = ea.prefill_host_buffer(B, S, Hq, Hkv, with_block_mask=use_bm, device=dev)
    O, LSE = ea.ea_hybrid_attn_prefill_host(Q, K, V, m, sink=sink, window=window, block_mask=bm,
                                            n_chunks=n_chunks, device_buffer=buf)
    torch.cuda.synchronize()
    check_no_device_error(buf)
    assert torch.equal(O, Oref)
    assert torch.equal(LSE, Lref)
    # and against the oracle, on every row
    Oo, Lo = oracle.prefill_full(Q, K, V, m.numpy(), sink=sink, window=window,
                                 block_mask=None if bm is None else bm.numpy())
    assert_close(O.float().numpy(), LSE.numpy(), Oo, Lo, "host pipeline")


def test_without_lse_and_repeated_calls(dev):
    B, S, Hq, Hkv = 1, 640, 8, 2
    Q, K, V = (t.pin_memory() for t in wl.qkv(B, S, Hq, Hkv, 128, seed=5))
    m = torch.tensor([[FULL, SSA]], dtype=torch.uint8)
    buf = ea.prefill_host_buffer(B, S, Hq, Hkv, device=dev)
    O1, L1 = ea.ea_hybrid_attn_prefill_host(Q, K, V, m, sink=16, window=200, device_buffer=buf,
                                            want_lse=False)
    assert L1 is None
    outs = []
    for n_chunks in (0, 5, 5):     # the same buffer again, back to back on one stream
        O, _ = ea.ea_hybrid_attn_prefill_host(Q, K, V, m, sink=16, window=200, device_buffer=buf,
                                              n_chunks=n_chunks)
        outs.append(O)
    torch.cuda.synchronize()
    for O in outs:
        assert torch.equal(O, O1)


def test_full_32k_workload_pinned(dev):
    cfg = wl.LLAMA_32K
    Q, K, V = wl.qkv(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.d, seed=cfg.seed)
    _, m = wl.routing_from_sa_heads(cfg.B, cfg.Hkv, cfg.sa_heads, cfg.fa_impl, cfg.sa_impl)
    Oref, Lref = _device_reference(dev, Q, K, V, m, cfg.sink, cfg.window, None)
    Q, K, V = Q.pin_memory(), K.pin_memory(), V.pin_memory()
    O, LSE = ea.ea_hybrid_attn_prefill_host(Q, K, V, m, sink=cfg.sink, window=cfg.window)
    torch.cuda.synchronize()
    assert torch.equal(O, Oref)
    assert torch.equal(LSE, Lref)
