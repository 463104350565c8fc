"""Oracle pins for the HiCache layer transfer (SGLang PR "[HiCache] TMA-staged
host<->device KV transfer kernel (sm_90+)", Modifications: page-first and
layer-first host views, per-layer device pools through a pointer table, int32
and int64 indices, H2D and D2H).  The C oracle is checked against numpy views
of the host pool as [buffer, page, layer, token in page, row] (page-first) or
[buffer, layer, token, row] (layer-first), indexed directly."""
import numpy as np
import pytest

import oracle


def host_view(host, nbuf, layers, host_tokens, page_size, page_first, rb):
    if page_first:
        return host.reshape(nbuf, host_tokens // page_size, layers, page_size, rb)
    return host.reshape(nbuf, layers, host_tokens, rb)


def host_row(view, b, l, t, page_size, page_first):
    if page_first:
        return view[b, t // page_size, l, t % page_size]
    return view[b, l, t]


@pytest.mark.parametrize("page_first", [True, False])
@pytest.mark.parametrize("idx_dtype", [np.int32, np.int64])
def test_h2d_rows_land_at_their_device_slots(page_first, idx_dtype):
    rng = np.random.default_rng(3)
    nbuf, layers, P, rb = 2, 3, 8, 48
    host_tokens, dev_tokens = 64, 40
    host = rng.integers(0, 256, nbuf * layers * host_tokens * rb, dtype=np.uint8)
    dev = [[rng.integers(0, 256, dev_tokens * rb, dtype=np.uint8) for _ in range(layers)]
           for _ in range(nbuf)]
    before = [[d.copy() for d in bl] for bl in dev]
    src = rng.choice(host_tokens, size=20, replace=False).astype(idx_dtype)
    dst = rng.choice(dev_tokens, size=20, replace=False).astype(idx_dtype)
    assert oracle.layer_transfer(dev, host, host_tokens, rb, src, dst, page_size=P,
                                 page_first=page_first, direction=0) == 0
    view = host_view(host, nbuf, layers, host_tokens, P, page_first, rb)
    for b in range(nbuf):
        for l in range(layers):
            got = dev[b][l].reshape(dev_tokens, rb)
            exp = before[b][l].reshape(dev_tokens, rb).copy()
            for s, d in zip(src, dst):
                exp[d] = host_row(view, b, l, int(s), P, page_first)
            np.testing.assert_array_equal(got, exp)


@pytest.mark.parametrize("page_first", [True, False])
def test_d2h_writes_only_the_listed_host_rows(page_first):
    rng = np.random.default_rng(4)
    nbuf, layers, P, rb = 1, 2, 4, 32
    host_tokens, dev_tokens = 32, 16
    host = rng.integers(0, 256, nbuf * layers * host_tokens * rb, dtype=np.uint8)
    exp = host.copy()
    dev = [[rng.integers(0, 256, dev_tokens * rb, dtype=np.uint8) for _ in range(layers)]]
    src = np.array([3, 0, 15, 7], np.int64)
    dst = np.array([31, 4, 5, 12], np.int64)
    assert oracle.layer_transfer(dev, host, host_tokens, rb, src, dst, page_size=P,
                                 page_first=page_first, direction=1) == 0
    view = host_view(exp, nbuf, layers, host_tokens, P, page_first, rb)
    for l in range(layers):
        rows = dev[0][l].reshape(dev_tokens, rb)
        for s, d in zip(src, dst):
            host_row(view, 0, l, int(d), P, page_first)[...] = rows[s]
    np.testing.assert_array_equal(host, exp)


def test_page_first_page_is_contiguous_per_layer():
    """In the page-first view the rows of one page and one layer are one
    contiguous run of page_size rows (what makes a page one copy)."""
    nbuf, layers, P, rb, T = 1, 3, 4, 16, 12
    host = np.arange(nbuf * layers * T * rb, dtype=np.int64).astype(np.uint32).view(np.uint8)
    host = np.ascontiguousarray(host[: nbuf * layers * T * rb])
    dev = [[np.zeros(T * rb, np.uint8) for _ in range(layers)]]
    src = np.arange(4, 8, dtype=np.int32)  # page 1
    dst = np.arange(0, 4, dtype=np.int32)
    oracle.layer_transfer(dev, host, T, rb, src, dst, page_size=P, page_first=True,
                          direction=0)
    for l in range(layers):
        start = (1 * layers * P + l * P) * rb
        np.testing.assert_array_equal(dev[0][l][: P * rb], host[start:start + P * rb])


def test_out_of_range_indices_are_skipped_and_counted():
    rng = np.random.default_rng(5)
    nbuf, layers, P, rb = 2, 2, 4, 16
    host_tokens, dev_tokens = 16, 8
    host = rng.integers(0, 256, nbuf * layers * host_tokens * rb, dtype=np.uint8)
    dev = [[np.zeros(dev_tokens * rb, np.uint8) for _ in range(layers)] for _ in range(nbuf)]
    src = np.array([1, -1, 16, 2], np.int32)
    dst = np.array([0, 1, 2, 8], np.int32)
    bad = oracle.layer_transfer(dev, host, host_tokens, rb, src, dst, page_size=P,
                                page_first=False, direction=0)
    assert bad == 3 * nbuf * layers
    view = host_view(host, nbuf, layers, host_tokens, P, False, rb)
    for b in range(nbuf):
        for l in range(layers):
            rows = dev[b][l].reshape(dev_tokens, rb)
            np.testing.assert_array_equal(rows[0], view[b, l, 1])
            assert not rows[1:].any()


def test_round_trip_restores_the_host_rows():
    rng = np.random.default_rng(6)
    nbuf, layers, P, rb = 2, 4, 8, 64
    host_tokens, dev_tokens = 64, 64
    host = rng.integers(0, 256, nbuf * layers * host_tokens * rb, dtype=np.uint8)
    orig = host.copy()
    dev = [[np.zeros(dev_tokens * rb, np.uint8) for _ in range(layers)] for _ in range(nbuf)]
    src = rng.permutation(host_tokens)[:40].astype(np.int32)
    dst = rng.permutation(dev_tokens)[:40].astype(np.int32)
    oracle.layer_transfer(dev, host, host_tokens, rb, src, dst, page_size=P, page_first=True,
                          direction=0)
    host[:] = 0
    oracle.layer_transfer(dev, host, host_tokens, rb, dst, src, page_size=P, page_first=True,
                          direction=1)
    view_o = host_view(orig, nbuf, layers, host_tokens, P, True, rb)
    view_h = host_view(host, nbuf, layers, host_tokens, P, True, rb)
    for b in range(nbuf):
        for l in range(layers):
            for t in src:
                np.testing.assert_array_equal(host_row(view_h, b, l, int(t), P, True),
                                              host_row(view_o, b, l, int(t), P, True))
