"""The allocation-free S4 entry point (hs_sparse_decode_noalloc).

Some callers cannot allocate device memory while decoding -- plugin code
inside a host engine that owns every device allocation, or latency-critical
loops where a cudaMalloc (which may synchronise the device) is not allowed.
For them libhs keeps the split-KV scratch in an array compiled into the
library.  These tests call that entry point through the C ABI and check it
against hs_sparse_decode with a caller-allocated workspace, on two calls in a
row (the second call reuses the array that the first one left behind).
"""
import math

import numpy as np
import pytest
import torch

from gpu_util import check_attention
from sparse_top_kv_gb300 import hs, inputs


def test_capacity_limit_is_rejected_on_the_host():
    # A shape whose scratch would exceed the built-in array is refused before
    # any device work (no GPU needed for this check).
    L = hs.lib()
    assert hs.sparse_decode_workspace_bytes(64, 16, 1, 2048, 576, 512) <= \
        hs.NOALLOC_WORKSPACE_BYTES
    P = None
    rc = L.hs_sparse_decode_noalloc(P, P, P, 576, 0, 10, P, P, 2, 65536, 128, 1, 576, 512,
                                    1.0, P, P, P, P)
    need = hs.sparse_decode_workspace_bytes(2, 128, 1, 65536, 576, 512)
    if need > hs.NOALLOC_WORKSPACE_BYTES:
        assert rc == 3  # HS_ERR_CAPACITY
    else:
        assert rc == 1  # null pointers


@pytest.mark.gpu
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
