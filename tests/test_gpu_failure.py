"""Failure detection without a GPU fault: the bounded wait every mbarrier
wait of libhs goes through gives up after its time limit (or at once when
its CTA raised the abort flag) and reports HS_ERR_TIMEOUT; the context stays
usable and the next calls compute correct results."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bits, check_attention, cuda
from sparse_top_kv_gb300 import hs, inputs

pytestmark = pytest.mark.gpu


def test_wait_that_nothing_completes_times_out():
    st, ns = hs.wait_selftest(0, 2_000_000)  # 2 ms limit
    assert hs.status_string(st) == "HS_ERR_TIMEOUT"
    assert 2_000_000 <= ns < 1_000_000_000


def test_completed_wait_returns_at_once():
    st, ns = hs.wait_selftest(1, 2_000_000)
    assert st == 0 and ns < 1_000_000


def test_abort_flag_ends_the_wait_early():
    st, ns = hs.wait_selftest(2, 1_000_000_000)  # 1 s limit, abort after ~20 us
    assert hs.status_string(st) == "HS_ERR_TIMEOUT"
    assert ns < 100_000_000


def test_context_usable_after_timeouts():
    for mode in (0, 2, 0):
        hs.wait_selftest(mode, 1_000_000)
    rng = np.random.default_rng(5)
    n_kv, cap = 500, 200
    cache = inputs.randn_bf16((n_kv, 576), 70, device="cuda")
    q = inputs.randn_bf16((2, 16, 576), 71, device="cuda")
    kv_rows = np.stack([rng.choice(n_kv, cap, replace=False) for _ in range(2)])[:, None]
    kv_rows = kv_rows.astype(np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = hs.sparse_decode(q, cache, cache, 576, 0, n_kv, cuda(kv_rows), None, 1 / 24, 512,
                                status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kb = bits(cache).reshape(-1)
    ref_out, ref_lse = oracle.sparse_decode(bits(q), kb, kb, 576, 0, kv_rows, None, 1 / 24,
                                            d_v=512)
    check_attention(out, lse, ref_out, ref_lse)
