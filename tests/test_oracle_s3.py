"""Pins for the oracle's SwapIn / BackUp (S3): byte identity of every copied
row, untouched rows unchanged (the HiCache TMA transfer PR's accuracy tests),
and the out-of-range source rule of hisparse_swap_in_kernel Phase 5 (zero the
hot row, revoke the slot's ownership)."""
import numpy as np

import oracle
from golden_io import load


def test_lru_trace_copies():
    g = load("s2_lru_trace.txt")
    hs = g["hot_size"]
    rb = 656  # the page walks Phase 5 with a 656-byte fp8_ds_mla row (41 x 16 B)
    rng = np.random.default_rng(0)
    host = rng.integers(0, 256, size=(2000, rb), dtype=np.uint8)
    hot = rng.integers(0, 256, size=(hs + 1, rb), dtype=np.uint8)
    hot0 = hot.copy()
    msrc = np.array([g["copy_src"]], np.int32)
    mdst = np.array([g["copy_dst"]], np.int64)
    oracle.swap_in(host.reshape(-1), hot.reshape(-1), rb, msrc, mdst, np.array([2], np.int32))
    for s, d in zip(g["copy_src"], g["copy_dst"]):
        assert (hot[d] == host[s]).all()
    untouched = [i for i in range(hs + 1) if i not in g["copy_dst"]]
    assert (hot[untouched] == hot0[untouched]).all()


def test_out_of_range_source_zeroes_and_revokes():
    rb, hs, region = 32, 4, 5
    host = np.arange(10 * rb, dtype=np.uint8).reshape(10, rb)
    hot = np.full((2 * region, rb), 7, np.uint8)
    dgi = np.array([[1, 2, 3, 4], [5, 6, 77, 8]], np.int32)
    msrc = np.array([[1, -1], [77, 3]], np.int32)
    mdst = np.array([[0, 1], [region + 2, region + 3]], np.int64)
    oracle.swap_in(host.reshape(-1), hot.reshape(-1), rb, msrc, mdst,
                   np.array([2, 2], np.int32), dgi=dgi, hot_size=hs, region_stride=region)
    assert (hot[0] == host[1]).all()
    assert (hot[1] == 0).all() and dgi[0, 1] == -1
    assert (hot[region + 2] == 0).all() and dgi[1, 2] == -1
    assert (hot[region + 3] == host[3]).all() and dgi[1, 3] == 8
    assert (hot[2] == 7).all()


def test_random_swap_byte_identity():
    rng = np.random.default_rng(3)
    rb, rows, cap, region = 48, 3, 20, 25
    host = rng.integers(0, 256, size=(500, rb), dtype=np.uint8)
    hot = rng.integers(0, 256, size=(rows * region, rb), dtype=np.uint8)
    hot0 = hot.copy()
    counts = rng.integers(0, cap + 1, size=rows).astype(np.int32)
    msrc = np.full((rows, cap), -1, np.int32)
    mdst = np.full((rows, cap), -1, np.int64)
    for r in range(rows):
        n = counts[r]
        msrc[r, :n] = rng.choice(500, size=n, replace=False)
        mdst[r, :n] = r * region + rng.choice(region - 1, size=n, replace=False)
    oracle.swap_in(host.reshape(-1), hot.reshape(-1), rb, msrc, mdst, counts)
    touched = set()
    for r in range(rows):
        for m in range(counts[r]):
            assert (hot[mdst[r, m]] == host[msrc[r, m]]).all()
            touched.add(int(mdst[r, m]))
    rest = [i for i in range(rows * region) if i not in touched]
    assert (hot[rest] == hot0[rest]).all()


def test_backup():
    rng = np.random.default_rng(4)
    rb = 64
    src = rng.integers(0, 256, size=(10, rb), dtype=np.uint8)
    host = np.zeros((20, rb), np.uint8)
    bad = oracle.backup(src.reshape(-1), np.array([9, 4, 0]), host.reshape(-1),
                        np.array([3, 25, 11]), rb)
    assert bad == 1
    assert (host[3] == src[9]).all() and (host[11] == src[0]).all()
    assert (np.delete(host, [3, 11], axis=0) == 0).all()


def test_backup_padding_destination():
    """A destination of -1 is padding (an inactive request of a fixed-size
    batch): nothing is written and nothing is counted; -2 is still an error."""
    rng = np.random.default_rng(5)
    rb = 32
    src = rng.integers(1, 256, size=(6, rb), dtype=np.uint8)
    host = np.zeros((8, rb), np.uint8)
    bad = oracle.backup(src.reshape(-1), np.array([0, 1, 2, 3]), host.reshape(-1),
                        np.array([-1, 5, -1, -2]), rb)
    assert bad == 1
    assert (host[5] == src[1]).all()
    assert (np.delete(host, [5], axis=0) == 0).all()
