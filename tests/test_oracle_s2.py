"""Pins for the oracle's hot-buffer lookup and LRU assignment (S2).

Fixed by: the full worked trace of hisparse_swap_in_kernel printed on the vLLM
HiSparse walkthrough (Phase 1 .. Phase 5, tests/golden/s2_lru_trace.txt), and a
timestamp model of the LRU policy over random multi-step runs (every slot
carries the key (step of last use, class, order); the new LRU list is the slots
sorted by key, and misses take the non-hit slots with the smallest keys).
"""
import numpy as np
import pytest

import oracle
from golden_io import load


def test_worked_trace():
    g = load("s2_lru_trace.txt")
    hs = g["hot_size"]
    region = hs + 1
    dgi = np.array([g["device_global_indices"]], np.int32)
    lru = np.array([g["lru_slots"]], np.int16)
    slot = np.array([g["global_indices"]], np.int32)
    newest = np.array([g["newest_global"]], np.int32)
    hot_idx, mm, msrc, mdst, mcount, stats, err = oracle.hot_lookup_assign(
        slot, None, newest, dgi, lru, hs, region)
    assert list(hot_idx[0]) == g["row_out"]
    assert list(mm[0]) == g["miss_mask"]
    assert list(dgi[0]) == g["device_global_indices_after"]
    assert list(lru[0]) == g["row_lru_after"]
    assert int(stats[0]) == g["total_hits"] and int(stats[1]) == g["total_misses"]
    assert int(mcount[0]) == g["total_misses"]
    assert list(msrc[0, :2]) == g["copy_src"]
    assert list(mdst[0, :2]) == g["copy_dst"]
    # The hits, read back from the new LRU tail, in LRU order.
    assert list(lru[0, -g["total_hits"]:]) == g["hit_slots_lru_order"]
    assert [int(hot_idx[0, i]) for i in g["miss_entries"]] == g["miss_slots"]
    assert int(err[0]) == 0


class TimestampLRU:
    """Each slot holds (g, key); key = (step, cls, order) with cls 1 = loaded,
    cls 2 = hit at that step; untouched slots keep their key."""

    def __init__(self, hot_size):
        self.g = [-1] * hot_size
        self.key = [(-1, 0, s) for s in range(hot_size)]  # identity order, all empty

    def order(self):
        return sorted(range(len(self.g)), key=lambda s: self.key[s])

    def step(self, k, entries, newest):
        order = self.order()
        rank = {s: i for i, s in enumerate(order)}
        where = {self.g[s]: s for s in range(len(self.g)) if self.g[s] >= 0}
        seen, out, hits, misses = set(), [], [], []
        for i, g in enumerate(entries):
            if g < 0 or g == newest or g in seen:
                out.append(None)
                continue
            seen.add(g)
            if g in where:
                hits.append(where[g])
                out.append(("hit", where[g]))
            else:
                misses.append(i)
                out.append(("miss", None))
        hit_set = set(hits)
        free = [s for s in order if s not in hit_set]
        for m, i in enumerate(misses):
            s = free[m]
            self.g[s] = entries[i]
            self.key[s] = (k, 1, m)
            out[i] = ("miss", s)
        for s in hits:
            self.key[s] = (k, 2, rank[s])
        return out


@pytest.mark.parametrize("seed", range(12))
def test_against_timestamp_model(seed):
    rng = np.random.default_rng(100 + seed)
    rows = 2
    hs = int(rng.choice([8, 16, 32]))
    cap = int(rng.integers(1, hs + 1))
    region = hs + 1 + int(rng.integers(0, 3))
    dgi = np.full((rows, hs), -1, np.int32)
    lru = np.tile(np.arange(hs, dtype=np.int16), (rows, 1))
    models = [TimestampLRU(hs) for _ in range(rows)]
    universe = int(rng.integers(cap + 1, 3 * hs))
    stats = np.zeros(2, np.int64)
    for k in range(8):
        slot = np.full((rows, cap), -1, np.int32)
        newest = np.zeros(rows, np.int32)
        count = np.zeros(rows, np.int32)
        for r in range(rows):
            n = int(rng.integers(0, cap + 1))
            vals = rng.integers(-1, universe, size=n)
            slot[r, :n] = vals
            count[r] = n
            newest[r] = universe + k if rng.random() < 0.5 else int(rng.integers(0, universe))
        before = stats.copy()
        hot_idx, mm, msrc, mdst, mcount, stats, err = oracle.hot_lookup_assign(
            slot, count, newest, dgi, lru, hs, region, stats=stats)
        tot_h = tot_m = 0
        for r in range(rows):
            base = r * region
            exp = models[r].step(k, [int(x) for x in slot[r, :count[r]]], int(newest[r]))
            assert list(lru[r]) == models[r].order()
            assert list(dgi[r]) == models[r].g
            m = 0
            for i in range(cap):
                g = int(slot[r, i]) if i < count[r] else -1
                if i >= count[r] or exp[i] is None:
                    if i < count[r] and g == newest[r] and g >= 0:
                        assert hot_idx[r, i] == base + hs
                    else:
                        assert hot_idx[r, i] == -1
                    assert mm[r, i] == 0
                    continue
                kind, s = exp[i]
                assert hot_idx[r, i] == base + s
                assert dgi[r, s] == g
                if kind == "hit":
                    tot_h += 1
                    assert mm[r, i] == 0
                else:
                    assert mm[r, i] == 1
                    assert msrc[r, m] == g and mdst[r, m] == base + s
                    m += 1
            assert mcount[r] == m
            tot_m += m
            # Invariants: permutation, unique valid ids.
            assert sorted(lru[r].tolist()) == list(range(hs))
            valid = dgi[r][dgi[r] >= 0]
            assert len(set(valid.tolist())) == len(valid)
        assert stats[0] - before[0] == tot_h and stats[1] - before[1] == tot_m


def test_padding_rows_untouched():
    hs, region = 8, 9
    dgi = np.arange(16, dtype=np.int32).reshape(2, 8)
    lru = np.tile(np.arange(8, dtype=np.int16), (2, 1))
    slot = np.array([[1, 2, 99], [9, 10, 98]], np.int32)
    d0, l0 = dgi.copy(), lru.copy()
    hot_idx, mm, msrc, mdst, mcount, stats, err = oracle.hot_lookup_assign(
        slot, None, None, dgi, lru, hs, region, num_real_rows=1)
    assert (hot_idx[1] == -1).all() and mcount[1] == 0
    assert (dgi[1] == d0[1]).all() and (lru[1] == l0[1]).all()
    assert list(hot_idx[0, :2]) == [1, 2] and mcount[0] == 1


def test_duplicate_entries_first_wins():
    hs, region = 8, 9
    dgi = np.full((1, hs), -1, np.int32)
    lru = np.arange(hs, dtype=np.int16)[None].copy()
    slot = np.array([[5, 7, 5, 7, 5]], np.int32)
    hot_idx, mm, msrc, mdst, mcount, stats, err = oracle.hot_lookup_assign(
        slot, None, None, dgi, lru, hs, region)
    assert list(hot_idx[0]) == [0, 1, -1, -1, -1]
    assert int(err[0]) == 3 and int(mcount[0]) == 2
