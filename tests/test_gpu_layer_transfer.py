"""HiCache layer transfer parity: hs_layer_transfer against the oracle, byte for
byte on the whole host pool and every device pool (copied rows equal their
source, untouched rows unchanged): host -> device and device -> host,
page-first and layer-first host views, int32 and int64 indices, whole pages
and scattered tokens, a ragged tail, MLA single-buffer rows, ids outside
their pool."""
import numpy as np
import pytest
import torch

import oracle
from sparse_top_kv_gb300 import hs

pytestmark = pytest.mark.gpu


def run_both(nbuf, layers, P, rb, host_tokens, dev_tokens, src, dst, page_first, direction,
             seed, max_ctas=0):
    rng = np.random.default_rng(seed)
    host_np = rng.integers(0, 256, nbuf * layers * host_tokens * rb, dtype=np.uint8)
    dev_np = [[rng.integers(0, 256, dev_tokens * rb, dtype=np.uint8) for _ in range(layers)]
              for _ in range(nbuf)]
    host = torch.from_numpy(host_np.copy()).pin_memory()
    dev = [[torch.from_numpy(d.copy()).cuda().view(dev_tokens, rb) for d in bl]
           for bl in dev_np]
    table = hs.layer_pointer_table(dev)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs.layer_transfer(table, nbuf, layers, dev_tokens, rb, host, host_tokens,
                      torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(),
                      page_size=P, page_first=page_first, direction=direction,
                      max_ctas=max_ctas, status=status)
    torch.cuda.synchronize()
    bad = oracle.layer_transfer(dev_np, host_np, host_tokens, rb, src, dst, page_size=P,
                                page_first=page_first, direction=direction)
    np.testing.assert_array_equal(host.numpy(), host_np, err_msg="host pool")
    for b in range(nbuf):
        for l in range(layers):
            np.testing.assert_array_equal(dev[b][l].cpu().numpy().reshape(-1), dev_np[b][l],
                                          err_msg=f"device pool {b} {l}")
    return int(status.item()), bad


def pages(rng, n_pages_pool, n_pages, P, dtype):
    pg = np.sort(rng.choice(n_pages_pool, size=n_pages, replace=False))
    return (pg[:, None] * P + np.arange(P)[None]).reshape(-1).astype(dtype)


@pytest.mark.parametrize("page_first", [True, False])
@pytest.mark.parametrize("dtype", [np.int32, np.int64])
def test_h2d_whole_pages(page_first, dtype):
    """K and V, 4 layers, 512-byte rows, 16-token pages: whole pages of the
    host pool into a contiguous run of device slots."""
    rng = np.random.default_rng(1)
    P, rb, host_tokens, dev_tokens = 16, 512, 1024, 512
    src = pages(rng, host_tokens // P, 20, P, dtype)
    dst = np.arange(src.size, dtype=dtype) + 7
    st, bad = run_both(2, 4, P, rb, host_tokens, dev_tokens, src, dst, page_first, 0, 2)
    assert st == 0 and bad == 0


@pytest.mark.parametrize("page_first", [True, False])
def test_d2h_whole_pages_all_layers(page_first):
    rng = np.random.default_rng(3)
    P, rb, host_tokens, dev_tokens = 32, 512, 2048, 1024
    src = np.arange(5 * P, dtype=np.int64) + 64
    dst = pages(rng, host_tokens // P, 5, P, np.int64)
    st, bad = run_both(2, 6, P, rb, host_tokens, dev_tokens, src, dst, page_first, 1, 4)
    assert st == 0 and bad == 0


@pytest.mark.parametrize("direction", [0, 1])
@pytest.mark.parametrize("page_first", [True, False])
def test_scattered_tokens_ragged_tail(direction, page_first):
    """Single scattered tokens, n not a multiple of a stage's rows."""
    rng = np.random.default_rng(5 + direction)
    P, rb, host_tokens, dev_tokens = 8, 272, 512, 256
    n = 101
    h = rng.choice(host_tokens, size=n, replace=False).astype(np.int32)
    d = rng.choice(dev_tokens, size=n, replace=False).astype(np.int32)
    src, dst = (h, d) if direction == 0 else (d, h)
    st, bad = run_both(2, 3, P, rb, host_tokens, dev_tokens, src, dst, page_first, direction,
                       6)
    assert st == 0 and bad == 0


@pytest.mark.parametrize("layers", [1, 4])
def test_mla_single_buffer(layers):
    """MLA rows (1152 B, one buffer), page-first host, pages and single
    tokens mixed, on a budget of 4 SMs."""
    rng = np.random.default_rng(7)
    P, rb, host_tokens, dev_tokens = 64, 1152, 1024, 512
    src = np.concatenate([pages(rng, host_tokens // P, 3, P, np.int64),
                          rng.choice(np.arange(host_tokens), size=30, replace=False)])
    dst = np.arange(src.size, dtype=np.int64) + 100  # distinct slots
    st, bad = run_both(1, layers, P, rb, host_tokens, dev_tokens, src, dst, True, 0, 8,
                       max_ctas=4)
    assert st == 0 and bad == 0


def test_ids_outside_their_pool_are_skipped():
    rng = np.random.default_rng(9)
    P, rb, host_tokens, dev_tokens = 16, 256, 256, 64
    src = rng.choice(host_tokens, size=40, replace=False).astype(np.int32)
    dst = rng.choice(dev_tokens, size=40, replace=False).astype(np.int32)
    src[[3, 17]] = [-2, host_tokens]
    dst[25] = dev_tokens + 5
    st, bad = run_both(2, 2, P, rb, host_tokens, dev_tokens, src, dst, False, 0, 10)
    assert bad == 3 * 2 * 2
    assert hs.status_string(st) == "HS_ERR_BAD_INDEX"
