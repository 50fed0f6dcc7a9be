"""Shared helpers of the GPU parity tests (imported by tests/test_*_gpu.py)."""
import numpy as np
import pytest
import torch

import oracle
import sparse_head_attention_gb300 as ea
from sparse_head_attention_gb300 import build as ea_build

# Tolerances (the benchmark configuration's figures): bf16 output max abs error
# 1e-2, LSE abs error 1e-3 (fp32 vs fp64).
O_TOL = 1e-2
LSE_TOL = 1e-3

# Every assert_close call records (what, elements above a flat O_TOL, elements
# compared, max |O - oracle|); tests/conftest.py prints the non-zero counts at
# the end of the run.
FLAT_EXCESS = []


def bf16_half_ulp(x):
    """Half a bf16 unit in the last place at |x| (8-bit significand): the error
    of the correctly rounded bf16 value of x, at most."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)


def gpu_device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ea_build.build()
    oracle.lib()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def assert_close(O, LSE, Oref, Lref, what="", flat=False):
    """O: bf16/float array vs float64 reference; LSE: -inf must match -inf.

    The output is bf16, and the correctly rounded bf16 value of O is only
    within half a bf16 step of O: half a step is 2^-8 = 0.0039 on [1, 2),
    2^-7 = 0.0078 on [2, 4) and 2^-6 = 0.0156 on [4, 8).  Below |O| = 4 a flat
    1e-2 is attainable and is the bound checked.  From |O| = 4 on, exact
    arithmetic followed by correct rounding can miss a flat 1e-2, so there the
    bound is 1e-2 plus half a bf16 step at the oracle's magnitude (a stated
    departure from a flat 1e-2, for such elements only).  Every call also counts
    the elements above a flat 1e-2, records the count in FLAT_EXCESS and prints
    it; with flat=True (the benchmark workloads) that count must be zero."""
    O = np.asarray(O, dtype=np.float64)
    LSE = np.asarray(LSE, dtype=np.float64)
    assert O.shape == Oref.shape, (O.shape, Oref.shape)
    assert np.isfinite(O).all(), what + ": non-finite output"
    diff = np.abs(O - Oref)
    err_o = diff.max() if O.size else 0.0
    bound = np.where(np.abs(Oref) < 4.0, O_TOL, O_TOL + bf16_half_ulp(Oref))
    excess = (diff - bound).max() if O.size else -1.0
    n_flat = int(np.count_nonzero(diff > O_TOL))
    FLAT_EXCESS.append((what, n_flat, int(O.size), float(err_o)))
    print("%s: %d of %d elements above a flat 1e-2 (max |O - oracle| %.5f)" % (
        what, n_flat, O.size, err_o))
    ninf = np.isneginf(Lref)
    assert (np.isneginf(LSE) == ninf).all(), what + ": -inf LSE pattern differs"
    err_l = np.abs(LSE[~ninf] - Lref[~ninf]).max() if (~ninf).any() else 0.0
    assert excess <= 0.0, (
        "%s: max |O - oracle| = %g exceeds 1e-2 (|O| < 4) or 1e-2 + half a bf16 step (|O| >= 4) by %g"
        % (what, err_o, excess))
    if flat:
        assert n_flat == 0, "%s: %d elements above a flat 1e-2 (max %g)" % (what, n_flat, err_o)
    assert err_l <= LSE_TOL, "%s: max |LSE - oracle| = %g" % (what, err_l)
    return err_o, err_l


def check_no_device_error(ws):
    st = ea.ea_check_errors(ws)
    assert st == 0, "device error word: status %d" % st


def bitmap_to_tiles(bitmap, B, Hkv, nB):
    """Unpack the visited-tile bitmap (uint32 words) to uint8 [B, Hkv, nB, nB]."""
    words = bitmap.cpu().numpy().view(np.uint32)
    bits = np.unpackbits(words.view(np.uint8), bitorder="little")
    return bits[: B * Hkv * nB * nB].reshape(B, Hkv, nB, nB)


def sample_rows(S, sink, window, T=128, block_mask_row0=None, n_random=128, seed=0, edge=128):
    """Deterministic query-row sample of a long sequence: the first and last
    `edge` rows, rows around the sink / window / sink+window boundaries (and
    their tile edges), and seeded random rows."""
    rows = set(range(min(edge, S))) | set(range(max(0, S - edge), S))
    for x in (sink, window, sink + window, T, 2 * T):
        for t in (x - 1, x, x + 1, (x // T) * T, (x // T) * T + T - 1):
            if 0 <= t < S:
                rows.add(t)
    g = np.random.default_rng(seed)
    rows |= set(int(v) for v in g.integers(0, S, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)
