"""S1 parity: hs_normalize_indices against the oracle, bit-exact on every
output (sorted tokens, slots, counts, error counters)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import cuda, np_i32
from sparse_top_kv_gb300 import hs, inputs

pytestmark = pytest.mark.gpu


def run_both(cand, row_req, seq_lens, table, B, window=0, sinks=0, owner=None, num_pages=None):
    num_pages = int(table.max()) + 1 if num_pages is None else num_pages
    ref = oracle.normalize_indices(cand, row_req, seq_lens, table, B, window=window,
                                   num_sinks=sinks, page_owner=owner, num_pages=num_pages)
    got = hs.normalize_indices(cuda(cand), cuda(row_req), cuda(seq_lens), cuda(table), B,
                               window=window, num_sinks=sinks,
                               page_owner=None if owner is None else cuda(owner),
                               num_pages=num_pages)
    torch.cuda.synchronize()
    for name, r, g in zip(("tok", "slot", "count", "err"), ref, got):
        np.testing.assert_array_equal(np_i32(g), r, err_msg=name)
    return ref


@pytest.mark.parametrize("seed", range(24))
def test_random_small(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.choice([1, 4, 16, 64]))
    num_reqs = int(rng.integers(1, 6))
    max_blocks = int(rng.integers(1, 40))
    num_pages = num_reqs * max_blocks + 5
    table = rng.permutation(num_pages)[: num_reqs * max_blocks].reshape(num_reqs, max_blocks)
    table = table.astype(np.int32)
    table[0, -1] = num_pages + 7  # one page outside the pool
    owner = None
    if seed % 2:
        owner = np.full(num_pages, -1, np.int32)
        for q in range(num_reqs):
            for b in range(max_blocks):
                if 0 <= table[q, b] < num_pages:
                    owner[table[q, b]] = q
        owner[table[-1, 0]] = 99  # a foreign page
    seq_lens = rng.integers(0, max_blocks * B + 5, size=num_reqs).astype(np.int32)
    rows = int(rng.integers(1, 9))
    row_req = rng.integers(-1, num_reqs + 1, size=rows).astype(np.int32)
    n_cand = int(rng.integers(0, 700))
    cand = rng.integers(-3, max_blocks * B + 8, size=(rows, n_cand)).astype(np.int32)
    if n_cand > 10:
        cand[:, :5] = cand[:, 5:10]  # duplicates
    run_both(cand, row_req, seq_lens, table, B, window=int(rng.integers(0, 40)),
             sinks=int(rng.integers(0, 6)), owner=owner, num_pages=num_pages)


def test_several_bitmap_windows():
    """Contexts longer than one shared-memory bitmap window (131072 positions)."""
    rng = np.random.default_rng(7)
    B = 64
    T = 300_001
    max_blocks = (T + B - 1) // B
    table = rng.permutation(max_blocks + 10)[:max_blocks][None].astype(np.int32)
    edges = np.array([0, 1, 131071, 131072, 131073, 262143, 262144, T - 1, T, T + 5, -1, -2])
    cand = np.concatenate([edges, rng.integers(0, T, size=3000)]).astype(np.int32)[None]
    run_both(cand, np.zeros(1, np.int32), np.array([T], np.int32), table, B, window=70000,
             sinks=9, num_pages=max_blocks + 10)


def test_edge_cases():
    table = np.arange(12, dtype=np.int32).reshape(3, 4)
    seq = np.array([0, 64, 10], np.int32)
    # Empty dynamic set with window/sinks; a row with no request; an empty context.
    cand = np.full((4, 3), -1, np.int32)
    cand[1] = [5, 5, 200]
    run_both(cand, np.array([1, 7, 0, 2], np.int32), seq, table, 16, window=4, sinks=2,
             num_pages=12)
    run_both(np.zeros((2, 0), np.int32), np.array([1, 2], np.int32), seq, table, 16, window=3,
             num_pages=12)


def test_full_size_configs():
    cfg3 = inputs.mla_decode(with_data=False)
    run_both(cfg3["cand"], np.arange(32, dtype=np.int32), np.full(32, cfg3["ctx"], np.int32),
             cfg3["block_table"], 64, num_pages=cfg3["num_pages"])
    cfg5 = inputs.gqa_union(with_data=False)
    ref = run_both(cfg5["cand"], cfg5["row_req"], np.full(16, cfg5["ctx"], np.int32),
                   cfg5["block_table"], 16, window=256, sinks=4, num_pages=cfg5["num_pages"])
    assert (ref[3][:, 3] > 0).all()  # the deliberate overlaps were counted


@pytest.mark.parametrize("B", [16, 12])
def test_block_table_rows_beyond_the_staged_limit(B):
    """Block-table rows longer than the kernel stages in shared memory
    (16384 blocks): page lookups go to global memory; power-of-two and
    other page sizes, several bitmap windows, foreign and out-of-pool pages,
    positions past the table."""
    rng = np.random.default_rng(900 + B)
    max_blocks = 20000
    num_reqs = 2
    num_pages = num_reqs * max_blocks + 50
    table = rng.permutation(num_pages)[: num_reqs * max_blocks].reshape(num_reqs, max_blocks)
    table = table.astype(np.int32)
    table[0, 17000] = num_pages + 3   # outside the pool
    table[1, 16384] = -1
    owner = np.full(num_pages, -1, np.int32)
    for q in range(num_reqs):
        ok = (table[q] >= 0) & (table[q] < num_pages)
        owner[table[q][ok]] = q
    owner[table[1, 19999]] = 0        # a foreign page
    T = max_blocks * B
    seq = np.array([T, T - 5], np.int32)
    edges = np.array([0, 16383 * B, 16384 * B, 16384 * B + 1, 17000 * B + 2, 19999 * B,
                      T - 1, T, T + 3, -1])
    cand = np.concatenate([edges, rng.integers(0, T + 10, size=4000)]).astype(np.int32)
    cand = np.stack([cand, rng.permutation(cand)])
    cand[:, 20:40] = cand[:, 40:60]   # repeats
    run_both(cand, np.array([0, 1], np.int32), seq, table, B, window=3000, sinks=7,
             owner=owner, num_pages=num_pages)
