"""S2 + S3 in one kernel (hs_hot_lookup_swap_in, the walkthrough's
hisparse_swap_in_kernel shape) against the oracle's lookup followed by the
oracle's SwapIn: every S2 output, dgi/lru/stats, and the whole hot buffer byte
for byte, over multi-step runs (hits, misses, evictions, repeats, padding,
sources outside the pool)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import cuda, np_i32, u8
from sparse_top_kv_gb300 import hs

pytestmark = pytest.mark.gpu


class FusedPair:
    def __init__(self, rows, hot_size, region, pool_rows, row_bytes, rng):
        self.hs, self.region, self.rb = hot_size, region, row_bytes
        self.pool = torch.from_numpy(
            rng.integers(0, 256, (pool_rows, row_bytes), dtype=np.uint8)).pin_memory()
        self.pool_dev = hs.host_device_pointer(self.pool)
        self.dgi = np.full((rows, hot_size), -1, np.int32)
        self.lru = np.tile(np.arange(hot_size, dtype=np.int16), (rows, 1))
        self.stats = np.zeros(2, np.int64)
        self.hot = rng.integers(0, 256, (rows * region, row_bytes), dtype=np.uint8)
        self.gdgi = torch.empty(rows, hot_size, dtype=torch.int32, device="cuda")
        self.glru = torch.empty(rows, hot_size, dtype=torch.int16, device="cuda")
        hs.hot_state_reset(self.gdgi, self.glru)
        self.gstats = torch.zeros(2, dtype=torch.int64, device="cuda")
        self.ghot = torch.from_numpy(self.hot.copy()).cuda()

    def step(self, slot, count, newest, num_real_rows=None):
        ref = oracle.hot_lookup_assign(slot, count, newest, self.dgi, self.lru, self.hs,
                                       self.region, num_real_rows=num_real_rows,
                                       stats=self.stats)
        oracle.swap_in(self.pool.numpy().reshape(-1), self.hot.reshape(-1), self.rb, ref[2],
                       ref[3], ref[4], dgi=self.dgi, hot_size=self.hs,
                       region_stride=self.region)
        got = hs.hot_lookup_assign(cuda(slot), None if count is None else cuda(count),
                                   None if newest is None else cuda(newest), self.gdgi,
                                   self.glru, self.region, self.gstats,
                                   num_real_rows=num_real_rows, with_split_lists=True,
                                   swap=(self.pool_dev, self.pool.shape[0], self.ghot, self.rb))
        torch.cuda.synchronize()
        names = ("hot_idx", "miss_mask", "miss_src", "miss_dst", "miss_count")
        for name, r, g in zip(names, ref[:5], got[:5]):
            np.testing.assert_array_equal(np_i32(g), r, err_msg=name)
        np.testing.assert_array_equal(np_i32(got[5]), ref[6], err_msg="err")
        np.testing.assert_array_equal(np_i32(self.gdgi), self.dgi, err_msg="dgi")
        np.testing.assert_array_equal(np_i32(self.glru), self.lru, err_msg="lru")
        np.testing.assert_array_equal(np_i32(self.gstats), self.stats, err_msg="stats")
        np.testing.assert_array_equal(u8(self.ghot), self.hot, err_msg="hot bytes")
        return ref


@pytest.mark.parametrize("seed,row_bytes", [(0, 1152), (1, 656), (2, 2048), (3, 16), (4, 1152)])
def test_random_steps(seed, row_bytes):
    """Random ids over a universe larger than the pool (some misses have no
    source row: the hot row is zeroed and the slot revoked), repeats, -1
    padding, counts, a padded request row."""
    rng = np.random.default_rng(3000 + seed)
    rows = int(rng.integers(1, 6))
    hot = int(rng.choice([16, 100, 1024, 3000]))
    cap = int(rng.integers(1, hot + 1))
    region = hot + 1 + int(rng.integers(0, 130))
    universe = int(rng.integers(cap + 2, 4 * hot))
    p = FusedPair(rows, hot, region, max(1, universe - 7), row_bytes, rng)
    for k in range(6):
        slot = rng.integers(-1, universe, size=(rows, cap)).astype(np.int32)
        count = rng.integers(0, cap + 1, size=rows).astype(np.int32)
        newest = (universe + k + np.arange(rows)).astype(np.int32)
        newest[0] = slot[0, 0]
        p.step(slot, count if k % 2 else None, newest, num_real_rows=rows - (k == 3))


def test_small_miss_steps_full_hot_size():
    """64 requests, hot 4096, cap 2048, 1152-byte rows: a cold step, then steps
    that keep all but a few dozen ids (the small-miss regime the fused kernel
    is for)."""
    rng = np.random.default_rng(11)
    rows, cap, hot = 64, 2048, 4096
    p = FusedPair(rows, hot, hot + 1, 200000, 1152, rng)
    slot = np.stack([rng.choice(200000, size=cap, replace=False) for _ in range(rows)])
    for k in range(4):
        if k:
            for r in range(rows):
                fresh = rng.choice(200000, size=24, replace=False)
                slot[r, rng.choice(cap, size=24, replace=False)] = fresh
        p.step(slot.astype(np.int32), None, np.full(rows, 300000 + k, np.int32))
