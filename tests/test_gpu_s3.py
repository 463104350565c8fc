"""S3 parity: hs_swap_in / hs_backup against the oracle, byte-exact on the
whole destination buffer (copied rows equal their source, untouched rows are
unchanged, out-of-range sources zero the row and revoke the slot)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import cuda, np_i32, u8
from sparse_top_kv_gb300 import hs, inputs

pytestmark = pytest.mark.gpu


def pinned_random(rows, rb, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    t = torch.randint(0, 256, (rows, rb), generator=g, dtype=torch.uint8)
    return t.pin_memory()


def swap_both(pool, hot_init, rb, msrc, mdst, mcount, dgi=None, hot_size=0, region=0,
              ticket=None, max_ctas=0):
    hot_ref = hot_init.copy()
    dgi_ref = None if dgi is None else dgi.copy()
    oracle.swap_in(pool.numpy().reshape(-1), hot_ref.reshape(-1), rb, msrc, mdst, mcount,
                   dgi=dgi_ref, hot_size=hot_size, region_stride=region)
    hot = cuda(hot_init)
    gdgi = None if dgi is None else cuda(dgi)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs.swap_in(hs.host_device_pointer(pool), pool.shape[0], hot, rb, cuda(msrc), cuda(mdst),
               cuda(mcount), dgi=gdgi, hot_size=hot_size, region_stride=region,
               max_ctas=max_ctas, ticket=ticket, status=status)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(u8(hot), hot_ref)
    if ticket is not None:
        assert ticket.tolist()[:2] == [0, 0]  # left zero for the next call
    if dgi is not None:
        np.testing.assert_array_equal(np_i32(gdgi), dgi_ref)
    return int(status.item())


@pytest.mark.parametrize("rb,claim", [(16, False), (656, False), (1152, False), (4096, False),
                                      (1152, True), (16, True)])
def test_runs_scattered_and_bad_sources(rb, claim):
    """claim: groups claimed through ticket counters, on a budget of 3 SMs
    (one counter pair serves both calls: each call leaves it zero)."""
    rng = np.random.default_rng(rb)
    pool_rows, rows, hot_size = 5000, 6, 300
    region = hot_size + 1
    cap = hot_size
    pool = pinned_random(pool_rows, rb, rb)
    hot_init = rng.integers(0, 256, size=(rows * region, rb), dtype=np.uint8)
    msrc = np.full((rows, cap), -1, np.int32)
    mdst = np.full((rows, cap), -1, np.int64)
    counts = np.zeros(rows, np.int32)
    for r in range(rows):
        n = int(rng.integers(0, cap + 1)) if r else cap
        dst = rng.permutation(hot_size)[:n]
        if r % 3 == 0:  # long contiguous runs in both source and destination
            start = int(rng.integers(0, pool_rows - n))
            src = start + np.arange(n)
            dst = np.sort(dst)
            dst = np.arange(n) if r == 0 else dst
        elif r % 3 == 1:  # pages of 64
            src = (rng.choice(pool_rows // 64, size=(n + 63) // 64, replace=False)[:, None] * 64
                   + np.arange(64)[None]).reshape(-1)[:n]
        else:  # scattered, a few out of range
            src = rng.choice(pool_rows, size=n, replace=False)
            if n > 4:
                src[:3] = [-5, pool_rows, pool_rows + 100]
        msrc[r, :n] = src
        mdst[r, :n] = r * region + dst
        counts[r] = n
    dgi = rng.integers(0, 10**6, size=(rows, hot_size)).astype(np.int32)
    ticket = torch.zeros(2, dtype=torch.int32, device="cuda") if claim else None
    for _ in range(2 if claim else 1):
        status = swap_both(pool, hot_init, rb, msrc, mdst, counts, dgi=dgi, hot_size=hot_size,
                           region=region, ticket=ticket, max_ctas=3 if claim else 0)
        assert status == 0


def test_backup_and_bad_destination():
    rb = 1152
    pool = torch.zeros(1000, rb, dtype=torch.uint8).pin_memory()
    src = cuda(np.random.default_rng(3).integers(0, 256, size=(50, rb), dtype=np.uint8))
    src_rows = np.array([4, 9, 49, 0, 17], np.int64)
    dst = np.array([10, 999, 5000, 0, -3], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = pool.numpy().copy()
    bad = oracle.backup(u8(src).reshape(-1), src_rows, ref.reshape(-1), dst, rb)
    hs.backup(src, cuda(src_rows), hs.host_device_pointer(pool), cuda(dst), rb, 1000,
              status=status)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(pool.numpy(), ref)
    assert bad == 2 and status.item() == 6  # HS_ERR_BAD_INDEX


def test_swapin_config_full_size():
    """64 requests x 4096 misses (302 MB): half contiguous 64-row pages, half
    scattered rows, into a fresh 64 x 4097-row hot buffer; then the BackUp of
    one row per request."""
    cfg = inputs.swapin()
    R, M, rb = cfg["num_reqs"], cfg["misses"], cfg["row_bytes"]
    region = cfg["hot_rows_per_req"]
    pool = cfg["pool"]
    msrc = cfg["src"]
    mdst = (np.arange(R, dtype=np.int64)[:, None] * region + np.arange(M)[None]).astype(np.int64)
    counts = np.full(R, M, np.int32)
    hot_init = np.zeros((R * region, rb), np.uint8)
    assert swap_both(pool, hot_init, rb, msrc, mdst, counts) == 0
    # The step's launch: 24 SMs, groups claimed through ticket counters.
    ticket = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert swap_both(pool, hot_init, rb, msrc, mdst, counts, ticket=ticket, max_ctas=24) == 0
    # BackUp: the reserved row of each request -> random host slots.
    src = cuda(np.random.default_rng(5).integers(0, 256, size=(R * region, rb), dtype=np.uint8))
    src_rows = np.arange(R, dtype=np.int64) * region + M
    ref = pool.numpy().copy()
    oracle.backup(u8(src).reshape(-1), src_rows, ref.reshape(-1), cfg["backup_dst"], rb)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs.backup(src, cuda(src_rows), hs.host_device_pointer(pool), cuda(cfg["backup_dst"]), rb,
              pool.shape[0], status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    np.testing.assert_array_equal(pool.numpy(), ref)


def test_backup_padding_destination():
    """-1 destinations (inactive requests) are skipped without an error."""
    rb = 1152
    pool = torch.zeros(100, rb, dtype=torch.uint8).pin_memory()
    src = cuda(np.random.default_rng(4).integers(1, 256, size=(8, rb), dtype=np.uint8))
    src_rows = np.array([1, 2, 3, 4], np.int64)
    dst = np.array([-1, 7, -1, 60], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = pool.numpy().copy()
    bad = oracle.backup(u8(src).reshape(-1), src_rows, ref.reshape(-1), dst, rb)
    hs.backup(src, cuda(src_rows), hs.host_device_pointer(pool), cuda(dst), rb, 100,
              status=status)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(pool.numpy(), ref)
    assert bad == 0 and status.item() == 0
