"""The allocation-free prefill entry point, called through the C ABI, must give
exactly the output of the workspace entry point (same planner, same kernel),
bit for bit, on two calls in a row, and once more through the Python binding.

It exists for callers that cannot allocate device memory for the library (an
engine that owns all device memory through its own allocator, or a path that
cannot afford cudaMalloc's device synchronisation); its scratch is a fixed
array inside the library, shared by every call, so the second call also checks
that nothing left over from the first one leaks into it.  This file sorts last
so that a failure here never hides the other GPU tests."""
import ctypes

import numpy as np
import pytest
import torch

import sparse_head_attention_gb300 as ea
from sparse_head_attention_gb300 import workloads as wl
from gpu_helpers import check_no_device_error, gpu_device

pytestmark = pytest.mark.gpu


def _noalloc_c(L, Q, K, V, O, LSE, m, sink, window, bm):
    B, S, Hq, d = Q.shape
    Hkv = K.shape[2]
    st = lambda t: (ctypes.c_int64 * 4)(*t.stride())
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return L.ea_hybrid_attn_prefill_noalloc(
        P(Q), P(K), P(V), P(O), P(LSE), st(Q), st(K), st(O), B, S, Hq, Hkv, d,
        ctypes.c_float(d ** -0.5), P(m), sink, window, P(bm), 128, None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _same(O, LSE, Oref, Lref):
    # the same planner and kernel on the same inputs: bit for bit, -inf included
    assert torch.equal(O, Oref)
    assert torch.equal(LSE.view(torch.int32), Lref.view(torch.int32))


def test_noalloc_prefill_matches_workspace_prefill_on_two_calls():
    dev = gpu_device()
    L = ea.lib()
    cases = [
        # B, S, Hq, Hkv, modes, sink, window, seed
        (1, 1000, 8, 2, [[ea.FULL, ea.SSA]], 64, 256, 1),
        (2, 777, 12, 3, [[ea.BLOCK, ea.SSA, ea.FULL], [ea.SSA, ea.BLOCK, ea.BLOCK]], 5, 300, 2),
    ]
    for (B, S, Hq, Hkv, modes, sink, window, seed) in cases:
        Q, K, V = (t.to(dev) for t in wl.qkv(B, S, Hq, Hkv, 128, seed=seed))
        m = torch.tensor(modes, dtype=torch.uint8, device=dev)
        bm = wl.block_mask(B, Hkv, S, density=0.3, seed=seed).to(dev)
        ws = ea.prefill_workspace(B, S, Hq, Hkv, device=dev)
        Oref, Lref = ea.ea_hybrid_attn_prefill(Q, K, V, m, sink=sink, window=window,
                                               block_mask=bm, workspace=ws)
        O = torch.full_like(Q, float("nan"))
        LSE = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device=dev)
        assert _noalloc_c(L, Q, K, V, O, LSE, m, sink, window, bm) == 0
        torch.cuda.synchronize()
        check_no_device_error(ws)
        _same(O, LSE, Oref, Lref)
    # the Python binding of the same entry point (argument marshalling only)
    O2, L2 = ea.ea_hybrid_attn_prefill_noalloc(Q, K, V, m, sink=sink, window=window, block_mask=bm)
    torch.cuda.synchronize()
    _same(O2, L2, Oref, Lref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    gpu_device()
    L = ea.lib()
    # 2^21 tokens x 64 KV heads needs far more than the fixed 4 MiB plan array;
    # rejected on the host before any pointer is touched.
    fake = ctypes.c_void_p(0x1000)
    s4 = (ctypes.c_int64 * 4)(1, 1, 1, 1)
    st = L.ea_hybrid_attn_prefill_noalloc(fake, fake, fake, fake, None, s4, s4, s4, 1, 1 << 21,
                                          64, 64, 128, ctypes.c_float(0.1), fake, 0, 1, None, 128,
                                          None, None)
    assert st == 2
