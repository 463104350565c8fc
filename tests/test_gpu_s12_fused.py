"""S1 and S2 in one kernel (hs_normalize_lookup_assign) against the oracle's
normalize followed by its lookup, bit-exact on every output and on the LRU
state, over several steps of evolving state: windows and sinks, repeated and
out-of-range candidates, foreign and out-of-pool pages, empty rows, the
newest token inside the set, block-table rows beyond the staged limit."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import cuda, np_i32
from sparse_top_kv_gb300 import hs

pytestmark = pytest.mark.gpu


def run(rng, num_reqs, B, max_blocks, n_cand, window, sinks, hot_size, steps, owner_frac=0.0,
        num_pages=None):
    num_pages = num_reqs * max_blocks + 7 if num_pages is None else num_pages
    table = rng.permutation(num_pages)[: num_reqs * max_blocks].reshape(num_reqs, max_blocks)
    table = table.astype(np.int32)
    table[0, max_blocks // 2] = num_pages + 3          # a page outside the pool
    owner = None
    if owner_frac > 0:
        owner = np.full(num_pages, -1, np.int32)
        for q in range(num_reqs):
            ok = (table[q] >= 0) & (table[q] < num_pages)
            owner[table[q][ok]] = q
        owner[table[-1, 1]] = 0 if num_reqs > 1 else 5  # a foreign page
    cap = n_cand + window + sinks
    region = hot_size + 1
    dgi = torch.empty(num_reqs, hot_size, dtype=torch.int32, device="cuda")
    lru = torch.empty(num_reqs, hot_size, dtype=torch.int16, device="cuda")
    hs.hot_state_reset(dgi, lru)
    o_dgi = np.full((num_reqs, hot_size), -1, np.int32)
    o_lru = np.tile(np.arange(hot_size, dtype=np.int16), (num_reqs, 1))
    stats = torch.zeros(2, dtype=torch.int64, device="cuda")
    o_stats = np.zeros(2, np.int64)
    row_req = np.arange(num_reqs, dtype=np.int32)
    T_max = max_blocks * B
    for s in range(steps):
        seq = rng.integers(max(1, T_max // 2), T_max + 1, size=num_reqs).astype(np.int32)
        seq[-1] = 0 if s == steps - 1 and num_reqs > 2 else seq[-1]   # an empty context
        cand = rng.integers(-2, T_max + 4, size=(num_reqs, n_cand)).astype(np.int32)
        if n_cand > 8:
            cand[:, :4] = cand[:, 4:8]                      # repeats
        newest_pos = np.maximum(seq - 1, 0)
        newest = oracle.normalize_indices(newest_pos[:, None], row_req, seq, table, B,
                                          num_pages=num_pages)[1][:, 0].copy()
        if s % 2 == 1:
            cand[:, -1] = newest_pos                         # the newest token in the set
        ref1 = oracle.normalize_indices(cand, row_req, seq, table, B, window=window,
                                        num_sinks=sinks, page_owner=owner,
                                        num_pages=num_pages)
        ref2 = oracle.hot_lookup_assign(ref1[1], ref1[2], newest, o_dgi, o_lru, hot_size,
                                        region, stats=o_stats)
        o_stats = ref2[5]
        s1, s2 = hs.normalize_lookup_assign(
            cuda(cand), cuda(row_req), cuda(seq), cuda(table), B, cuda(newest), dgi, lru, region,
            stats, window=window, num_sinks=sinks,
            page_owner=None if owner is None else cuda(owner), num_pages=num_pages)
        torch.cuda.synchronize()
        for name, g, r in zip(("tok", "slot", "count", "err"), s1, ref1):
            np.testing.assert_array_equal(np_i32(g), r, err_msg=f"step {s} {name}")
        hot_idx, mm, msrc, mdst, mcount, lerr, hit_idx, miss_rows = s2
        r_hot, r_mm, r_msrc, r_mdst, r_mcount, _, r_err = ref2
        np.testing.assert_array_equal(np_i32(hot_idx), r_hot, err_msg=f"step {s} hot_idx")
        np.testing.assert_array_equal(np_i32(mm), r_mm, err_msg=f"step {s} miss_mask")
        np.testing.assert_array_equal(np_i32(mcount), r_mcount, err_msg=f"step {s} miss_count")
        np.testing.assert_array_equal(np_i32(lerr), r_err, err_msg=f"step {s} lookup err")
        for r in range(num_reqs):
            m = int(r_mcount[r])
            np.testing.assert_array_equal(np_i32(msrc)[r, :m], r_msrc[r, :m])
            np.testing.assert_array_equal(np_i32(mdst)[r, :m], r_mdst[r, :m])
            np.testing.assert_array_equal(np_i32(miss_rows)[r, :m], r_mdst[r, :m])
        np.testing.assert_array_equal(np_i32(hit_idx), np.where(r_mm == 0, r_hot, -1))
        np.testing.assert_array_equal(np_i32(dgi), o_dgi, err_msg=f"step {s} dgi")
        np.testing.assert_array_equal(np_i32(lru), o_lru, err_msg=f"step {s} lru")
        np.testing.assert_array_equal(np_i32(stats), o_stats, err_msg=f"step {s} stats")


@pytest.mark.parametrize("seed", range(6))
def test_random_steps(seed):
    rng = np.random.default_rng(4000 + seed)
    B = int(rng.choice([4, 16, 64]))
    run(rng, num_reqs=int(rng.integers(1, 5)), B=B, max_blocks=int(rng.integers(4, 40)),
        n_cand=int(rng.integers(8, 300)), window=int(rng.integers(0, 20)),
        sinks=int(rng.integers(0, 5)), hot_size=640, steps=4, owner_frac=seed % 2)


def test_headline_shape():
    """64 requests, top_k 2048 of 131072 positions, hot 4096 (+1) rows."""
    rng = np.random.default_rng(77)
    run(rng, num_reqs=64, B=64, max_blocks=2048, n_cand=2048, window=0, sinks=0,
        hot_size=4096, steps=3)


def test_unstaged_block_table():
    """Block-table rows longer than the staged limit (20000 blocks of 12)."""
    rng = np.random.default_rng(78)
    run(rng, num_reqs=2, B=12, max_blocks=20000, n_cand=1500, window=40, sinks=3,
        hot_size=2048, steps=2, owner_frac=1)
