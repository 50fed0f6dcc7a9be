"""The benchmark's work accounting (host logic, no GPU): the closed forms that
turn a timed step into useful FLOP/s, visited-tile FLOP/s and kept-byte GB/s
must equal the fp64 oracle's brute-force counts, and a profile's traffic figure
is used only while the kernel source it was captured from is unchanged."""
import hashlib

import numpy as np
import pytest

import bench
import oracle
from sparse_head_attention_gb300 import workloads as wl

FULL, SSA, BLOCK = oracle.FULL, oracle.SSA, oracle.BLOCK


@pytest.mark.parametrize("S,sink,window", [(1000, 64, 256), (4096, 128, 2048), (300, 0, 1),
                                           (700, 5000, 1), (1024, 128, 5000), (129, 3, 130)])
def test_visited_tiles_and_kept_pairs_equal_brute_force(S, sink, window):
    Hkv = 3
    bm = wl.block_mask(1, Hkv, S, density=0.3, seed=S).numpy()
    modes = np.array([[FULL, SSA, BLOCK]], np.uint8)
    vis = oracle.visited(1, S, Hkv, modes, sink=sink, window=window, block_mask=bm)
    _, _, kept = oracle.sparsity_ratios(np.zeros((1, Hkv), np.uint8), modes, S, sink=sink,
                                        window=window, block_masks=bm)
    for h in range(Hkv):
        mode = int(modes[0, h])
        assert bench.visited_tiles_per_kv_head(mode, S, sink, window, bm[0, h]) == int(vis[0, h].sum())
        assert bench.kept_pairs_per_kv_head(mode, S, sink, window, bm[0, h]) == int(kept[0, h])


def test_decode_kept_bytes_equal_the_last_row_of_brute_force_counts():
    """Kept keys of the decode query (position L - 1) = kept pairs over L rows
    minus kept pairs over L - 1 rows, both counted by the oracle."""
    L, Hkv, B = 1000, 3, 2          # ceil(L / 128) == ceil((L - 1) / 128): one mask for both
    cfg = wl.DecodeConfig("t", B=B, Hq=6, Hkv=Hkv, d=128, L=L, sink=100, window=300)
    bm = wl.block_mask(B, Hkv, L, density=0.4, seed=4).numpy()
    m = np.array([[FULL, SSA, BLOCK], [BLOCK, FULL, SSA]], np.uint8)
    keys = 0
    for b in range(B):
        counts = []
        for S in (L, L - 1):
            _, _, kept = oracle.sparsity_ratios(np.zeros((1, Hkv), np.uint8), m[b:b + 1], S,
                                                sink=cfg.sink, window=cfg.window,
                                                block_masks=bm[b:b + 1])
            counts.append(kept[0])
        keys += int((counts[0] - counts[1]).sum())
    rows = bm[:, :, (L - 1) // 128, :]
    assert bench.decode_kept_bytes(cfg, m, rows) == keys * 2 * cfg.d * 2


def test_profile_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// a kernel\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "p.md").write_text(
        "summary\n\ntraffic_bytes_per_launch: 12345\nsource_sha256: %s\n" % digest)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("p.md", str(src)) == 12345.0
    src.write_text("// a changed kernel\n")
    assert bench.profile_traffic("p.md", str(src)) is None
    assert bench.profile_traffic("missing.md", str(src)) is None

