"""Host-side checks of the C ABI (no GPU needed): the library loads and exports
every entry point include/ea.h declares, argument validation rejects bad calls
before anything is enqueued, workspace sizing, and the host-only sparsity
ratios, which must equal the oracle's bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
import sparse_head_attention_gb300 as ea
from sparse_head_attention_gb300 import build as ea_build
from sparse_head_attention_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    ea_build.build()
    return ea.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "ea.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ea_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_abi():
    names = _declared_functions()
    assert set(names) == set(ea.EXPORTS), names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_multi_layer_prefill_host_checks(L):
    # workspace: the single-layer plan of B * n_layers rows; 1 .. 48 layers
    assert L.ea_prefill_layers_workspace_size(36, 1, 4096, 32, 8, 128) == \
        L.ea_prefill_workspace_size(36, 4096, 32, 8, 128)
    assert L.ea_prefill_layers_workspace_size(0, 1, 4096, 32, 8, 128) == 0
    assert L.ea_prefill_layers_workspace_size(49, 1, 4096, 32, 8, 128) == 0
    assert L.ea_prefill_layers_workspace_size(2, 40000, 128, 32, 8, 128) == 0   # B * layers > 65535
    s4 = (ctypes.c_int64 * 4)(32 * 128 * 256, 32 * 128, 128, 1)
    k4 = (ctypes.c_int64 * 4)(8 * 128 * 256, 8 * 128, 128, 1)
    # rejected before anything is enqueued (no GPU needed): no layers, too many, a null tensor
    assert L.ea_hybrid_attn_prefill_layers(None, 1, s4, k4, s4, 1, 256, 32, 8, 128,
                                           ctypes.c_float(0.1), 0, 64, 128, None, 0, None) == 1
    arr = (ea._PrefillLayer * 49)()
    assert L.ea_hybrid_attn_prefill_layers(ctypes.cast(arr, ctypes.c_void_p), 49, s4, k4, s4, 1, 256, 32,
                                           8, 128, ctypes.c_float(0.1), 0, 64, 128, None, 0, None) == 2
    assert L.ea_hybrid_attn_prefill_layers(ctypes.cast(arr, ctypes.c_void_p), 2, s4, k4, s4, 1, 256, 32,
                                           8, 128, ctypes.c_float(0.1), 0, 64, 128, None, 0, None) == 1


def test_status_strings(L):
    for code in range(7):
        s = L.ea_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert L.ea_status_string(0) == b"ok"


def test_workspace_sizes(L):
    assert L.ea_prefill_workspace_size(1, 1024, 8, 2, 128) > 256
    assert L.ea_prefill_workspace_size(1, 1024, 8, 2, 64) == 0       # head dim 128 only
    assert L.ea_prefill_workspace_size(1, 1024, 8, 3, 128) == 0      # Hq % Hkv != 0
    assert L.ea_prefill_workspace_size(0, 1024, 8, 2, 128) == 0
    assert L.ea_decode_workspace_size(32, 32, 8, 128, 131072, 0) > 256
    assert L.ea_decode_workspace_size(32, 32, 8, 128, 131072, 2000) == 0
    # bigger problems never need less
    assert L.ea_prefill_workspace_size(1, 32768, 32, 8, 128) > L.ea_prefill_workspace_size(1, 1024, 32, 8, 128)
    # the allocation-free prefill's fixed 4 MiB plan array: every length up to
    # 2^21 fits at B = 1 with 32 query heads over 8 KV heads, and B = 2 still
    # does; B = 3 is rejected
    assert L.ea_prefill_workspace_size(1, 1 << 21, 32, 8, 128) == 1573120
    assert L.ea_prefill_workspace_size(2, 1 << 21, 32, 8, 128) <= 4 << 20
    assert L.ea_prefill_workspace_size(3, 1 << 21, 32, 8, 128) > 4 << 20


def _fake(n=0x1000):
    return ctypes.c_void_p(n)


def _str(*v):
    return (ctypes.c_int64 * len(v))(*v)


def _prefill(L, **kw):
    a = dict(Q=_fake(), K=_fake(), V=_fake(), O=_fake(), LSE=None,
             qs=_str(8 * 1024 * 128, 8 * 128, 128, 1), kvs=_str(2 * 1024 * 128, 2 * 128, 128, 1),
             os_=_str(8 * 1024 * 128, 8 * 128, 128, 1), B=1, S=1024, Hq=8, Hkv=2, d=128, scale=0.088,
             m=_fake(), sink=64, window=256, bm=None, bs=128, ws=_fake(0x100000), wsb=1 << 30,
             vis=None, stream=None)
    a.update(kw)
    return L.ea_hybrid_attn_prefill(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["qs"], a["kvs"], a["os_"],
                                    a["B"], a["S"], a["Hq"], a["Hkv"], a["d"], a["scale"], a["m"],
                                    a["sink"], a["window"], a["bm"], a["bs"], a["ws"], a["wsb"],
                                    a["vis"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(Q=None), 1), (dict(m=None), 1), (dict(B=0), 1), (dict(Hkv=3), 1), (dict(window=0), 1),
    (dict(sink=-1), 1), (dict(scale=0.0), 1), (dict(bs=64), 1), (dict(d=64), 2),
    (dict(S=(1 << 21) + 1), 2), (dict(qs=_str(8 * 1024 * 128, 8 * 128, 128, 2)), 1),
    (dict(kvs=_str(2 * 1024 * 128, 2 * 128, 100, 1)), 1), (dict(Q=_fake(0x1008)), 1),
    (dict(ws=None), 3), (dict(ws=_fake(0x100010)), 3), (dict(wsb=16), 3),
])
def test_prefill_rejects_bad_arguments_on_host(L, kw, expect):
    assert _prefill(L, **kw) == expect


def _decode(L, **kw):
    a = dict(q=_fake(), K=_fake(), V=_fake(), O=_fake(), LSE=None, qs=_str(32 * 128, 128, 1),
             kvs=_str(4096 * 8 * 128, 8 * 128, 128, 1), os_=_str(32 * 128, 128, 1), sl=_fake(),
             B=4, Hq=32, Hkv=8, d=128, Lmax=4096, scale=0.088, m=_fake(), sink=128, window=4096,
             bm=None, bs=128, ns=0, ws=_fake(0x100000), wsb=1 << 30, stream=None)
    a.update(kw)
    return L.ea_hybrid_attn_decode(a["q"], a["K"], a["V"], a["O"], a["LSE"], a["qs"], a["kvs"], a["os_"],
                                   a["sl"], a["B"], a["Hq"], a["Hkv"], a["d"], a["Lmax"], a["scale"], a["m"],
                                   a["sink"], a["window"], a["bm"], a["bs"], a["ns"], a["ws"], a["wsb"],
                                   a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), 1), (dict(sl=None), 1), (dict(Hq=30), 1), (dict(ns=-1), 1), (dict(ns=1025), 1),
    (dict(window=0), 1), (dict(Hkv=2), 2), (dict(d=96), 2), (dict(kvs=_str(4096 * 8 * 128, 8 * 128, 128, 2)), 1),
    (dict(ws=None), 3), (dict(wsb=1024), 3), (dict(bs=64), 1), (dict(bs=64, bm=_fake()), 1),
    (dict(bm=_fake(), Lmax=65536 * 128), 2),      # more than 65535 blocks per row
])
def test_decode_rejects_bad_arguments_on_host(L, kw, expect):
    assert _decode(L, **kw) == expect


def test_route_rejects_bad_mlp(L):
    dims = (ctypes.c_int * 3)(128, 64, 3)          # last layer must have 2 outputs
    W = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    b = (ctypes.c_void_p * 2)(0x3000, 0x4000)
    mlp = ea._Mlp(2, dims, W, b)
    st = L.ea_route(_fake(), _str(65536 * 8 * 128, 8 * 128, 128, 1), 1, 65536, 8, 128, 100, 100,
                    ctypes.byref(mlp), ea._Policy(0, 1), _fake(), _fake(), None, None)
    assert st == 1
    mlp5 = ea._Mlp(5, dims, W, b)
    st = L.ea_route(_fake(), _str(65536 * 8 * 128, 8 * 128, 128, 1), 1, 65536, 8, 128, 100, 100,
                    ctypes.byref(mlp5), ea._Policy(0, 1), _fake(), _fake(), None, None)
    assert st == 2


# ---------------------------------------------------------------- ratios
def test_sparsity_ratios_equal_oracle_on_hand_cases(L):
    import json
    cases = json.load(open(os.path.join(ROOT, "tests", "golden", "sparsity_ratio_hand_examples.json")))
    for c in cases["cases"]:
        if c["T"] != 128:
            continue  # the library's block size is fixed at 128
        msr, esr = ea.ea_sparsity_ratios(np.array(c["r"], np.uint8), np.array(c["m"], np.uint8), c["S"],
                                         sink=c["sink"], window=c["window"])
        assert msr == c["msr"]
        assert esr == c["esr_num"] / c["esr_den"]


@pytest.mark.parametrize("S,sink,window", [(1000, 64, 256), (257, 0, 1), (1300, 200, 129), (129, 128, 1)])
def test_sparsity_ratios_bit_exact_vs_oracle(L, S, sink, window):
    Lyr, Hkv = 3, 4
    g = torch.Generator().manual_seed(S)
    r = (torch.rand(Lyr, Hkv, generator=g) < 0.6).to(torch.uint8).numpy()
    pol = np.array([[ea.FULL, ea.SSA], [ea.BLOCK, ea.SSA]], np.uint8)
    m = np.where(r == 1, ea.SSA, np.where(np.arange(Hkv)[None, :] % 2 == 0, ea.FULL, ea.BLOCK)).astype(np.uint8)
    bms = wl.block_mask(Lyr, Hkv, S, density=0.3, seed=S).numpy()           # [L, Hkv, nB, nB]
    bms[0, 1, -1, -1] = 0
    msr_o, esr_o, _ = oracle.sparsity_ratios(r, m, S, sink=sink, window=window, block_masks=bms)
    msr, esr = ea.ea_sparsity_ratios(r, m, S, sink=sink, window=window, block_masks=list(bms))
    assert msr == msr_o
    assert esr == esr_o


def test_sparsity_ratios_at_256k_match_closed_forms(L):
    # XA-SSA 256K workload: 2 BLOCK heads (r = 0) and 6 SSA heads (sink 128, window 4096).
    cfg = wl.XA_SSA_256K
    S, T = cfg.S, 128
    r, m = wl.routing_from_sa_heads(1, cfg.Hkv, cfg.sa_heads, fa_impl=ea.BLOCK, sa_impl=ea.SSA)
    bm = wl.block_mask(1, cfg.Hkv, S, density=cfg.block_density, seed=cfg.seed).numpy()[0]
    msr, esr = ea.ea_sparsity_ratios(r.numpy(), m.numpy(), S, sink=cfg.sink, window=cfg.window,
                                     block_masks=[bm])
    assert msr == 0.75
    causal = S * (S + 1) // 2
    i = np.arange(S, dtype=np.int64)
    ssa_kept = int((np.minimum(i + 1, cfg.window) +
                    np.maximum(0, np.minimum(cfg.sink, i + 1 - cfg.window))).sum())
    pruned = 0
    for h in range(cfg.Hkv):
        if m[0, h] == ea.SSA:
            pruned += causal - ssa_kept
        else:
            # rows of query block qb keep 128 keys per kept block below the diagonal
            # plus (t + 1) keys of the diagonal block for row t
            nB = S // T
            below = np.tril(bm[h], -1).sum(axis=1).astype(np.int64)
            kept = int((below * T * T).sum()) + int(bm[h].diagonal().sum()) * (T * (T + 1) // 2)
            pruned += causal - kept
    assert esr == pruned / (1 * cfg.Hkv * causal)
    assert 0.9 < esr < 0.96


def test_device_entry_points_fail_loudly_without_gpu():
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    Q = torch.zeros(1, 128, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ea.ea_hybrid_attn_prefill(Q, Q[:, :, :2], Q[:, :, :2], torch.zeros(1, 2, dtype=torch.uint8),
                                  sink=0, window=1)


def test_route_layers_rejects_bad_arguments(L):
    good_dims = (ctypes.c_int * 3)(128, 64, 2)
    bad_dims = (ctypes.c_int * 3)(128, 64, 3)
    W = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    b = (ctypes.c_void_p * 2)(0x3000, 0x4000)
    strides = _str(65536 * 8 * 128, 8 * 128, 128, 1)

    def call(n, mlps, ptrs, **kw):
        a = dict(S=65536, ph=100, pt=100, r=_fake(), m=_fake())
        a.update(kw)
        return L.ea_route_layers(ptrs, n, strides, 1, a["S"], 8, 128, a["ph"], a["pt"], mlps,
                                 ea._Policy(0, 1), a["r"], a["m"], None, None)

    # layer 70 of 72 (in the second launch's chunk) has a bad MLP: the call
    # fails before the first launch (the fake pointers are never dereferenced)
    mlps = (ea._Mlp * 72)(*[ea._Mlp(2, bad_dims if l == 70 else good_dims, W, b) for l in range(72)])
    ptrs = (ctypes.c_void_p * 72)(*([0x1000] * 72))
    assert call(72, mlps, ptrs) == 1
    good = (ea._Mlp * 2)(ea._Mlp(2, good_dims, W, b), ea._Mlp(2, good_dims, W, b))
    assert call(0, good, (ctypes.c_void_p * 2)(0x1000, 0x1000)) == 1          # no layers
    assert call(2, good, (ctypes.c_void_p * 2)(0x1000, None)) == 1            # a null K
    assert call(2, good, (ctypes.c_void_p * 2)(0x1000, 0x1000), ph=0, pt=0) == 1
    assert call(2, good, (ctypes.c_void_p * 2)(0x1000, 0x1000), r=None) == 1
    deep = (ctypes.c_int * 6)(128, 64, 64, 64, 64, 2)                          # 5 dense layers
    W5 = (ctypes.c_void_p * 5)(*([0x1000] * 5))
    assert call(1, (ea._Mlp * 1)(ea._Mlp(5, deep, W5, W5)), (ctypes.c_void_p * 1)(0x1000)) == 2


def test_prefill_host_rejects_bad_arguments(L):
    B, S, Hq, Hkv = 1, 1024, 8, 2
    need = L.ea_prefill_host_buffer_size(B, S, Hq, Hkv, 128, 0)
    assert need > L.ea_prefill_host_buffer_size(B, S // 2, Hq, Hkv, 128, 0)
    assert L.ea_prefill_host_buffer_size(B, S, Hq, Hkv, 128, 1) > need     # room for the mask
    assert L.ea_prefill_host_buffer_size(B, S, Hq, Hkv, 64, 0) == 0

    def call(**kw):
        a = dict(Q=_fake(), K=_fake(), V=_fake(), O=_fake(), LSE=None, B=B, S=S, Hq=Hq, Hkv=Hkv,
                 d=128, scale=0.088, m=_fake(), sink=64, window=256, bm=None, bs=128,
                 buf=_fake(0x100000), nbytes=need, nch=0)
        a.update(kw)
        return L.ea_hybrid_attn_prefill_host(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["S"],
                                             a["Hq"], a["Hkv"], a["d"], a["scale"], a["m"], a["sink"],
                                             a["window"], a["bm"], a["bs"], a["buf"], a["nbytes"],
                                             a["nch"], None)

    for kw, expect in [(dict(Q=None), 1), (dict(m=None), 1), (dict(O=None), 1), (dict(scale=0.0), 1),
                       (dict(Hkv=3), 1), (dict(window=0), 1), (dict(bs=64), 1), (dict(d=64), 2),
                       (dict(nch=-1), 1), (dict(nch=9), 1), (dict(nch=65, S=1 << 14), 1),
                       (dict(buf=None), 3), (dict(buf=_fake(0x100010)), 3), (dict(nbytes=need - 1), 3),
                       (dict(bm=_fake()), 3)]:      # a mask needs the larger buffer
        assert call(**kw) == expect, kw


def test_paged_decode_rejects_bad_arguments(L):
    def call(**kw):
        a = dict(q=_fake(), K=_fake(), V=_fake(), O=_fake(), LSE=None, qs=_str(32 * 128, 128, 1),
                 kvs=_str(256 * 8 * 128, 8 * 128, 128, 1), os_=_str(32 * 128, 128, 1), bt=_fake(),
                 bts=16, maxp=16, ps=256, nump=1024, sl=_fake(), B=4, Hq=32, Hkv=8, d=128,
                 scale=0.088, m=_fake(), sink=128, window=4096, bm=None, bs=128, ns=0,
                 ws=_fake(0x100000), wsb=1 << 30)
        a.update(kw)
        return L.ea_hybrid_attn_decode_paged(a["q"], a["K"], a["V"], a["O"], a["LSE"], a["qs"], a["kvs"],
                                             a["os_"], a["bt"], a["bts"], a["maxp"], a["ps"], a["nump"],
                                             a["sl"], a["B"], a["Hq"], a["Hkv"], a["d"], a["scale"], a["m"],
                                             a["sink"], a["window"], a["bm"], a["bs"], a["ns"], a["ws"],
                                             a["wsb"], None)

    for kw, expect in [(dict(bt=None), 1), (dict(maxp=0), 1), (dict(nump=0), 1), (dict(bts=8), 1),
                       (dict(ps=100), 2), (dict(ps=32), 2), (dict(ps=0), 2),
                       (dict(maxp=1 << 20, bts=1 << 20, ps=1 << 12), 2),   # 2^32 rows per sequence
                       (dict(q=None), 1), (dict(Hq=30), 1), (dict(d=64), 2), (dict(ws=None), 3),
                       (dict(wsb=1024), 3), (dict(bs=0), 1)]:
        assert call(**kw) == expect, kw


def test_varlen_prefill_rejects_bad_arguments(L):
    B, total, maxS, Hq, Hkv = 3, 5000, 3000, 8, 2
    need = L.ea_prefill_varlen_workspace_size(B, total, maxS, Hq, Hkv, 128)
    assert need > 256 and L.ea_prefill_varlen_workspace_size(B, total, maxS, Hq, Hkv, 64) == 0
    assert L.ea_prefill_varlen_workspace_size(B, total, (1 << 21) + 1, Hq, Hkv, 128) == 0

    def call(**kw):
        a = dict(Q=_fake(), K=_fake(), V=_fake(), O=_fake(), LSE=None, qs=_str(Hq * 128, 128, 1),
                 kvs=_str(Hkv * 128, 128, 1), os_=_str(Hq * 128, 128, 1), cu=_fake(), B=B, total=total,
                 maxS=maxS, Hq=Hq, Hkv=Hkv, d=128, scale=0.088, m=_fake(), sink=64, window=256, bm=None,
                 bs=128, ws=_fake(0x100000), wsb=need)
        a.update(kw)
        return L.ea_hybrid_attn_prefill_varlen(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["qs"], a["kvs"],
                                               a["os_"], a["cu"], a["B"], a["total"], a["maxS"], a["Hq"],
                                               a["Hkv"], a["d"], a["scale"], a["m"], a["sink"], a["window"],
                                               a["bm"], a["bs"], a["ws"], a["wsb"], None)

    for kw, expect in [(dict(cu=None), 1), (dict(Q=None), 1), (dict(B=0), 1), (dict(total=0), 1),
                       (dict(maxS=0), 1), (dict(Hkv=3), 1), (dict(window=0), 1), (dict(bs=64), 1),
                       (dict(scale=0.0), 1), (dict(d=64), 2), (dict(maxS=(1 << 21) + 1), 2),
                       (dict(qs=_str(Hq * 128, 128, 2)), 1), (dict(kvs=_str(Hkv * 128, 100, 1)), 1),
                       (dict(Q=_fake(0x1008)), 1), (dict(ws=None), 3), (dict(wsb=need - 1), 3)]:
        assert call(**kw) == expect, kw


def test_xa_estimate_rejects_bad_arguments(L):
    B, S, Hq, Hkv = 1, 4096, 8, 2
    need = L.ea_xa_workspace_size(B, S, Hq, Hkv, 128, 16, 2)
    assert need > 256
    assert L.ea_xa_workspace_size(B, S, Hq, Hkv, 128, 16, 3) == 0      # more units than heads
    assert L.ea_xa_workspace_size(B, S + 8, Hq, Hkv, 128, 16, 2) == 0  # S not a multiple of 16
    assert L.ea_xa_workspace_size(B, S, Hq, Hkv, 128, 8, 2) == 0       # stride 16 only
    assert L.ea_xa_workspace_size(B, S, Hq, Hkv, 64, 16, 2) == 0
    assert L.ea_xa_workspace_size(B, S, Hq, Hkv, 128, 16, 1) < need    # one unit needs less
    assert L.ea_xa_workspace_size(B, 4 * S, Hq, Hkv, 128, 16, 2) > need

    def call(**kw):
        a = dict(Q=_fake(), K=_fake(), qs=_str(S * Hq * 128, Hq * 128, 128, 1),
                 ks=_str(S * Hkv * 128, Hkv * 128, 128, 1), B=B,
                 S=S, Hq=Hq, Hkv=Hkv, d=128, scale=0.088, m=_fake(), stride=16, tau=0.9, bs=128,
                 units=2, bm=_fake(), sc=None, ws=_fake(0x100000), wsb=need)
        a.update(kw)
        return L.ea_xa_estimate(a["Q"], a["K"], a["qs"], a["ks"], a["B"], a["S"], a["Hq"], a["Hkv"],
                                a["d"], a["scale"], a["m"], a["stride"], a["tau"], a["bs"],
                                a["units"], a["bm"], a["sc"], a["ws"], a["wsb"], None)

    for kw, expect in [(dict(Q=None), 1), (dict(K=None), 1), (dict(m=None), 1), (dict(bm=None), 1),
                       (dict(B=0), 1), (dict(Hkv=3), 1), (dict(bs=64), 1), (dict(scale=0.0), 1),
                       (dict(tau=-0.1), 1), (dict(tau=float("nan")), 1), (dict(units=0), 1),
                       (dict(units=3), 1), (dict(d=64), 2), (dict(stride=8), 2), (dict(S=S + 8), 2),
                       (dict(S=(1 << 21) + 16), 2), (dict(qs=_str(S * Hq * 128, Hq * 128, 128, 2)), 1),
                       (dict(ks=_str(S * Hkv * 128, Hkv * 128, 100, 1)), 1), (dict(K=_fake(0x1008)), 1),
                       (dict(ws=None), 3), (dict(ws=_fake(0x100010)), 3), (dict(wsb=need - 1), 3)]:
        assert call(**kw) == expect, kw
