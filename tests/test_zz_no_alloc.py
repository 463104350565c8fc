"""The allocation-free S4 entry point (hs_sparse_decode_noalloc).

Some callers cannot allocate device memory while decoding -- plugin code
inside a host engine that owns every device allocation, or latency-critical
loops where a cudaMalloc (which may synchronise the device) is not allowed.
For them libhs keeps the split-KV scratch in an array compiled into the
library.  These tests call that entry point through the C ABI and check it
against hs_sparse_decode with a caller-allocated workspace, and against the
oracle, on two calls in a row (the second call reuses the array that the
first one left behind); that it allocates no device memory; and that a shape
too large for the array is refused.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bits, check_attention
from sparse_top_kv_gb300 import hs, inputs

pytestmark = pytest.mark.gpu


def test_capacity_limit_is_rejected_on_the_host():
    # The workspace of this shape (eight splits of each 128-head row, merged
    # through partial states in the workspace, on a GPU with 64 or more SMs)
    # exceeds the built-in array; the call is refused before any device
    # work, whatever the pointers.
    rows, heads, cap = 8, 128, 65536
    need = hs.sparse_decode_workspace_bytes(rows, heads, 1, cap, 576, 512)
    assert need > hs.NOALLOC_WORKSPACE_BYTES
    P = None
    rc = hs.lib().hs_sparse_decode_noalloc(P, P, P, 576, 0, 10, P, P, rows, cap, heads, 1, 576,
                                           512, 1.0, P, P, P, P)
    assert rc == 3  # HS_ERR_CAPACITY


@pytest.mark.parametrize("rows,heads,cap", [(4, 16, 2048), (2, 128, 1024)])
def test_noalloc_matches_workspace_entry_point(rows, heads, cap):
    need = hs.sparse_decode_workspace_bytes(rows, heads, 1, cap, 576, 512)
    assert 0 < need <= hs.NOALLOC_WORKSPACE_BYTES  # the built-in array is used
    rng = np.random.default_rng(rows * 1000 + heads)
    n_kv = 8192
    cache = inputs.randn_bf16((n_kv, 576), 70, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        q = inputs.randn_bf16((rows, heads, 576), 71 + call, device="cuda")
        kv = np.stack([rng.choice(n_kv, size=cap, replace=False) for _ in range(rows)])
        kv_rows = torch.from_numpy(kv.astype(np.int32))[:, None, :].contiguous().cuda()
        count = torch.full((rows, 1), cap - 3 * call, dtype=torch.int32, device="cuda")
        ref_out, ref_lse = hs.sparse_decode(q, cache, cache, 576, 0, n_kv, kv_rows, count,
                                            1 / math.sqrt(576), 512, status=status)
        out = torch.empty_like(ref_out)
        lse = torch.empty_like(ref_lse)
        hs.sparse_decode_noalloc(q, cache, cache, 576, 0, n_kv, kv_rows, count,
                                 1 / math.sqrt(576), 512, out=out, lse=lse, status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        check_attention(out, lse, ref_out.double().cpu().numpy(),
                        ref_lse.double().cpu().numpy(), label=f"call {call}")
        kb = bits(cache).reshape(-1)
        o_out, o_lse = oracle.sparse_decode(bits(q), kb, kb, 576, 0, kv[:, None, :].astype(
            np.int32), count.cpu().numpy(), 1 / math.sqrt(576), d_v=512)
        check_attention(out, lse, o_out, o_lse, label=f"call {call} vs oracle")


def test_noalloc_allocates_no_device_memory():
    # cudaMemGetInfo sees every device allocation of the process (torch's
    # caching allocator cannot see the library's own): after a first call
    # (the per-device set-up), further calls leave the free bytes unchanged.
    rows, heads, cap, n_kv = 4, 16, 2048, 8192
    assert hs.sparse_decode_workspace_bytes(rows, heads, 1, cap, 576, 512) > 0
    rng = np.random.default_rng(5)
    cache = inputs.randn_bf16((n_kv, 576), 80, device="cuda")
    q = inputs.randn_bf16((rows, heads, 576), 81, device="cuda")
    kv = np.stack([rng.choice(n_kv, size=cap, replace=False) for _ in range(rows)])
    kv_rows = torch.from_numpy(kv.astype(np.int32))[:, None, :].contiguous().cuda()
    out = torch.empty(rows, heads, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(rows, heads, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs.sparse_decode_noalloc(q, cache, cache, 576, 0, n_kv, kv_rows, None, 1 / 24, 512,
                             out=out, lse=lse, status=status)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(4):
        hs.sparse_decode_noalloc(q, cache, cache, 576, 0, n_kv, kv_rows, None, 1 / 24, 512,
                                 out=out, lse=lse, status=status)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert status.item() == 0
