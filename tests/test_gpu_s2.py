"""S2 parity: hs_hot_lookup_assign against the oracle, bit-exact on hot
indices, miss masks, miss lists, dgi/lru state, stats and error counts, over
multi-step runs."""
import numpy as np
import pytest
import torch

import oracle
from golden_io import load
from gpu_util import cuda, np_i32
from sparse_top_kv_gb300 import hs

pytestmark = pytest.mark.gpu


class Pair:
    """The same hot-buffer state on both sides."""

    def __init__(self, rows, hot_size, region):
        self.hs, self.region = hot_size, region
        self.dgi = np.full((rows, hot_size), -1, np.int32)
        self.lru = np.tile(np.arange(hot_size, dtype=np.int16), (rows, 1))
        self.stats = np.zeros(2, np.int64)
        self.gdgi = torch.empty(rows, hot_size, dtype=torch.int32, device="cuda")
        self.glru = torch.empty(rows, hot_size, dtype=torch.int16, device="cuda")
        hs.hot_state_reset(self.gdgi, self.glru)
        self.gstats = torch.zeros(2, dtype=torch.int64, device="cuda")

    def set_state(self, dgi, lru):
        self.dgi[:] = dgi
        self.lru[:] = lru
        self.gdgi.copy_(torch.from_numpy(dgi))
        self.glru.copy_(torch.from_numpy(lru))

    def step(self, slot, count, newest, num_real_rows=None):
        ref = oracle.hot_lookup_assign(slot, count, newest, self.dgi, self.lru, self.hs,
                                       self.region, num_real_rows=num_real_rows,
                                       stats=self.stats)
        got = hs.hot_lookup_assign(cuda(slot), None if count is None else cuda(count),
                                   None if newest is None else cuda(newest), self.gdgi,
                                   self.glru, self.region, self.gstats,
                                   num_real_rows=num_real_rows, with_split_lists=True)
        torch.cuda.synchronize()
        names = ("hot_idx", "miss_mask", "miss_src", "miss_dst", "miss_count")
        for name, r, g in zip(names, ref[:5], got[:5]):
            np.testing.assert_array_equal(np_i32(g), r, err_msg=name)
        np.testing.assert_array_equal(np_i32(got[5]), ref[6], err_msg="err")
        np.testing.assert_array_equal(np_i32(got[6]), np.where(ref[1] == 0, ref[0], -1),
                                      err_msg="hit_idx")
        mr = np_i32(got[7])
        for r in range(slot.shape[0]):
            m = int(ref[4][r])
            np.testing.assert_array_equal(mr[r, :m], ref[3][r, :m], err_msg="miss_rows")
            assert (mr[r, m:] == -1).all()
        np.testing.assert_array_equal(np_i32(self.gdgi), self.dgi, err_msg="dgi")
        np.testing.assert_array_equal(np_i32(self.glru), self.lru, err_msg="lru")
        np.testing.assert_array_equal(np_i32(self.gstats), self.stats, err_msg="stats")
        return ref


def test_worked_trace():
    g = load("s2_lru_trace.txt")
    p = Pair(1, g["hot_size"], g["hot_size"] + 1)
    p.set_state(np.array([g["device_global_indices"]], np.int32),
                np.array([g["lru_slots"]], np.int16))
    ref = p.step(np.array([g["global_indices"]], np.int32), None,
                 np.array([g["newest_global"]], np.int32))
    assert list(ref[0][0]) == g["row_out"]


@pytest.mark.parametrize("seed", range(10))
def test_random_steps(seed):
    rng = np.random.default_rng(2000 + seed)
    rows = int(rng.integers(1, 6))
    hot = int(rng.choice([16, 100, 1024, 3000]))
    cap = int(rng.integers(1, hot + 1))
    region = hot + 1 + int(rng.integers(0, 130))
    p = Pair(rows, hot, region)
    universe = int(rng.integers(cap + 2, 4 * hot))
    for k in range(6):
        slot = rng.integers(-1, universe, size=(rows, cap)).astype(np.int32)
        count = rng.integers(0, cap + 1, size=rows).astype(np.int32)
        newest = (universe + k + np.arange(rows)).astype(np.int32)
        newest[0] = slot[0, 0]  # sometimes the newest id also appears in the row
        p.step(slot, count if k % 2 else None, newest, num_real_rows=rows - (k == 3))


def test_full_size_lookup():
    """64 requests, cap 2048, hot 4096 (the full_hisparse shape), 5 steps with
    85 % reuse so that hits, misses and evictions all occur."""
    rng = np.random.default_rng(9)
    rows, cap, hot = 64, 2048, 4096
    p = Pair(rows, hot, hot + 1)
    prev = None
    for k in range(5):
        if prev is None:
            slot = np.stack([rng.choice(10**6, size=cap, replace=False) for _ in range(rows)])
        else:
            slot = prev.copy()
            for r in range(rows):
                new = rng.choice(10**6, size=cap - 1741, replace=False)
                slot[r, rng.choice(cap, size=cap - 1741, replace=False)] = new
        slot = slot.astype(np.int32)
        p.step(slot, None, np.full(rows, 2 * 10**6 + k, np.int32))
        prev = slot


def test_cap_equals_hot_size_all_miss_then_all_hit():
    p = Pair(2, 64, 65)
    slot = np.arange(128, dtype=np.int32).reshape(2, 64)
    ref = p.step(slot, None, None)
    assert (ref[4] == 64).all()
    ref = p.step(slot[:, ::-1].copy(), None, None)
    assert (ref[4] == 0).all()
