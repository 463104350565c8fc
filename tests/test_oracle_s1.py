"""Pins for the oracle's index normalisation (S1).

Each check is fixed by something other than the oracle itself: the two worked
examples printed in PaperTrace 5.1.1 section 1.2 (tests/golden), and a
brute-force membership test over every position 0 <= t < T on tiny random
inputs (random page tables, duplicates, cross-page candidates, partly filled
tail pages, window/sink overlaps and every kind of invalid entry).
"""
import numpy as np
import pytest

import oracle
from golden_io import load


def test_worked_example_page64():
    g = load("s1_page64_example.txt")
    B = g["page_size"]
    table = np.array([g["block_table"]], np.int32)
    cand = np.array([g["candidates"]], np.int32)
    # The example has one query whose context covers both logical blocks.
    tok, slot, count, err = oracle.normalize_indices(
        cand, row_req=[0], seq_lens=[2 * B], block_table=table, page_size=B, num_pages=64)
    n = int(count[0])
    assert n == 6
    assert list(tok[0, :n]) == g["candidates"]
    assert (tok[0, n:] == -1).all() and (slot[0, n:] == -1).all()
    blocks = tok[0, :n] // B
    assert sorted(set(blocks.tolist())) == g["logical_blocks"]
    pages = slot[0, :n] // B
    offs = slot[0, :n] % B
    page_of_block = dict(zip(g["logical_blocks"], g["physical_pages"]))
    assert [page_of_block[b] for b in blocks] == list(pages)
    assert list(offs[blocks == 0]) == g["offsets_block0"]
    assert list(offs[blocks == 1]) == g["offsets_block1"]
    assert (err == 0).all()
    # The printed values imply slots 2625, 2626, 2687, 448, 449, 511.
    assert list(slot[0, :n]) == [2625, 2626, 2687, 448, 449, 511]


def test_worked_example_page16():
    g = load("s1_page16_example.txt")
    B = g["page_size"]
    req = g["request"]
    nlog = g["num_logical_pages"]
    x = 97  # the page elides pageTable[4]; any free value
    rng = np.random.default_rng(5)
    table = rng.permutation(np.arange(200, 200 + 3 * nlog)).reshape(3, nlog).astype(np.int32)
    table[req, :4] = g["block_table_prefix"]
    table[req, 4] = x
    seq_lens = np.array([nlog * B] * 3, np.int32)
    cand = np.array([g["tokens"]], np.int32)
    tok, slot, count, err = oracle.normalize_indices(
        cand, row_req=[req], seq_lens=seq_lens, block_table=table, page_size=B, num_pages=1000)
    n = int(count[0])
    assert list(tok[0, :n]) == g["tokens"]
    lp = tok[0, :n] // B
    assert sorted(set(lp.tolist())) == g["logical_pages"]
    offs = slot[0, :n] % B
    assert list(offs[lp == 1]) == g["offsets_page1"]
    assert list(offs[lp == 4]) == g["offsets_page4"]
    pages = slot[0, :n] // B
    assert set(pages[lp == 1].tolist()) == {g["physical_page_of_logical_page1"]}
    assert set(pages[lp == 4].tolist()) == {x}
    assert (err == 0).all()


def _brute(cand, row_req, seq_lens, table, B, window, sinks, owner, num_pages):
    """Membership decided position by position over 0 <= t < T."""
    rows = cand.shape[0]
    num_reqs, max_blocks = table.shape
    results = []
    for r in range(rows):
        q = int(row_req[r])
        D = [int(t) for t in cand[r] if t != -1]
        if q < 0 or q >= num_reqs:
            results.append(([], [], [len(D), 0, 0, 0]))
            continue
        T = max(int(seq_lens[q]), 0)

        def page_of(t):
            b = t // B
            if b >= max_blocks:
                return None, "range"
            p = int(table[q, b])
            if p < 0 or p >= num_pages:
                return None, "range"
            if owner is not None and int(owner[p]) != q:
                return None, "owner"
            return p, None

        struct = set(range(0, min(sinks, T))) | set(range(max(0, T - window), T))
        toks, slots = [], []
        for t in range(T):
            if t in struct or t in D:
                p, why = page_of(t)
                if p is not None:
                    toks.append(t)
                    slots.append(p * B + t % B)
        err = [0, 0, 0, 0]
        for t in sorted(struct):
            _, why = page_of(t)
            if why == "range":
                err[0] += 1
            elif why == "owner":
                err[2] += 1
        valid_d = 0
        for t in D:
            if t < 0:
                err[0] += 1
            elif t >= T:
                err[1] += 1
            else:
                _, why = page_of(t)
                if why == "range":
                    err[0] += 1
                elif why == "owner":
                    err[2] += 1
                else:
                    valid_d += 1
        # Every valid dynamic entry either adds a new member or repeats one.
        new_from_d = len([t for t in toks if t not in struct])
        err[3] = valid_d - new_from_d
        results.append((toks, slots, err))
    return results


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.choice([1, 2, 4, 16]))
    num_reqs = int(rng.integers(1, 4))
    max_blocks = int(rng.integers(1, 7))
    num_pages = num_reqs * max_blocks + int(rng.integers(0, 4))
    table = rng.permutation(num_pages)[: num_reqs * max_blocks].reshape(num_reqs, max_blocks)
    table = table.astype(np.int32)
    # A few table entries out of range, to exercise that check.
    if rng.random() < 0.3:
        table[rng.integers(num_reqs), rng.integers(max_blocks)] = num_pages + 3
    owner = None
    if rng.random() < 0.5:
        owner = np.full(num_pages, -1, np.int32)
        for q in range(num_reqs):
            for b in range(max_blocks):
                p = table[q, b]
                if 0 <= p < num_pages:
                    owner[p] = q
        # One foreign page.
        owner[rng.integers(num_pages)] = num_reqs + 1
    # Partly filled tail pages: T not a multiple of B, sometimes past the table.
    seq_lens = rng.integers(0, max_blocks * B + 3, size=num_reqs).astype(np.int32)
    rows = int(rng.integers(1, 5))
    row_req = rng.integers(-1, num_reqs + 1, size=rows).astype(np.int32)
    n_cand = int(rng.integers(0, 12))
    hi = max_blocks * B + 4
    cand = rng.integers(-3, hi, size=(rows, n_cand)).astype(np.int32)
    # Duplicates on purpose.
    if n_cand > 2:
        cand[:, -1] = cand[:, 0]
    window = int(rng.integers(0, 5))
    sinks = int(rng.integers(0, 3))
    tok, slot, count, err = oracle.normalize_indices(
        cand, row_req, seq_lens, table, B, window=window, num_sinks=sinks, page_owner=owner,
        num_pages=num_pages)
    ref = _brute(cand, row_req, seq_lens, table, B, window, sinks, owner, num_pages)
    cap = tok.shape[1]
    for r in range(rows):
        toks, slots, e = ref[r]
        n = int(count[r])
        assert n == len(toks)
        assert list(tok[r, :n]) == toks
        assert list(slot[r, :n]) == slots
        assert (tok[r, n:cap] == -1).all() and (slot[r, n:cap] == -1).all()
        assert list(err[r]) == e


def test_capacity_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.normalize_indices(np.zeros((1, 4), np.int32), [0], [8], np.zeros((1, 1), np.int32),
                                 8, window=2, cap=5)
