"""The C ABI without a GPU: libhs.so builds, loads and exports every function
include/hs_api.h declares; host-side argument checks return their status
codes before any device work."""
import ctypes
import os
import re

import pytest

from sparse_top_kv_gb300 import hs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "hs_api.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*(hs_[a-z_0-9]+)\s*\(",
                                 src, flags=re.M)))


def test_exports_every_declared_function():
    names = declared_functions()
    assert "hs_sparse_decode" in names and "hs_normalize_indices" in names
    L = hs.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) <= set(hs.EXPORTS) | set(names)
    assert set(hs.EXPORTS) <= set(names)


def test_status_strings():
    assert hs.status_string(0) == "HS_OK"
    assert hs.status_string(5) == "HS_ERR_TIMEOUT"
    assert hs.status_string(12345) == "HS_ERR_UNKNOWN"
    # The wait self-test checks its mode and outputs before launching.
    L = hs.lib()
    assert L.hs_wait_selftest(3, 1000, None, None, None) == 1
    assert L.hs_wait_selftest(0, 1000, None, None, None) == 1


def test_host_side_argument_checks():
    L = hs.lib()
    P = None
    # Negative rows / capacity below n_cand + window + sinks.
    assert L.hs_normalize_indices(P, -1, 4, 0, 0, P, P, P, 4, 4, P, 1, 1, 64, 4, P, P, P, P,
                                  P) == 1
    assert L.hs_normalize_indices(P, 1, 4, 2, 1, P, P, P, 4, 4, P, 1, 1, 64, 6, P, P, P, P,
                                  P) == 3
    # cap > hot_size, region stride too small, hot_size beyond int16 slots.
    assert L.hs_hot_lookup_assign(P, P, 1, 9, 1, P, P, P, 8, 9, P, P, P, P, P, P, P, P, P,
                                  P) == 3
    assert L.hs_hot_lookup_assign(P, P, 1, 4, 1, P, P, P, 8, 8, P, P, P, P, P, P, P, P, P,
                                  P) == 1
    assert L.hs_hot_state_reset(P, P, 1, 40000, P) == 1
    # Lookup + copy in one kernel: rows not a multiple of 16, rows over 2048 B.
    assert L.hs_hot_lookup_swap_in(P, P, 1, 4, 1, P, P, P, 8, 9, P, P, P, P, P, P, P, P, P, P,
                                   100, P, 1000, P) == 2
    assert L.hs_hot_lookup_swap_in(P, P, 1, 4, 1, P, P, P, 8, 9, P, P, P, P, P, P, P, P, P, P,
                                   100, P, 2064, P) == 3
    assert L.hs_hot_lookup_swap_in(P, P, 1, 4, 1, P, P, P, 8, 9, P, P, P, P, P, P, P, P, P, P,
                                   100, P, 1152, P) == 1
    # fp8 SwapIn: short rows, misaligned stride.
    assert L.hs_swap_in_fp8ds(P, 10, 640, P, 10, P, P, P, 1, 1, P, 0, 0, 0, P, P, P) == 1
    assert L.hs_swap_in_fp8ds(P, 10, 664, P, 10, P, P, P, 1, 1, P, 0, 0, 0, P, P, P) == 2
    # Rows not a multiple of 16 bytes.
    assert L.hs_swap_in(P, 10, P, 100, P, P, P, 1, 1, P, 0, 0, 0, P, P, P) == 2
    assert L.hs_swap_in(P, 10, P, 96, P, P, P, 1, 1, P, 0, 0, -1, P, P, P) == 1
    assert L.hs_backup(P, P, P, P, 1, 24, 10, P, P) == 2
    # Layer transfer: rows not a multiple of 16, index width, direction,
    # too many layers, a page-first pool that is not whole pages.
    assert L.hs_layer_transfer(P, P, 64, 0, 1, 1, 16, 0, 64, 100, P, P, 4, 1, 0, 0, P,
                               P) == 2
    assert L.hs_layer_transfer(P, P, 64, 0, 1, 1, 16, 0, 64, 96, P, P, 2, 1, 0, 0, P, P) == 1
    assert L.hs_layer_transfer(P, P, 64, 0, 1, 1, 16, 0, 64, 96, P, P, 4, 1, 2, 0, P, P) == 1
    assert L.hs_layer_transfer(P, P, 64, 0, 2, 4000, 16, 0, 64, 96, P, P, 4, 1, 0, 0, P,
                               P) == 1
    assert L.hs_layer_transfer(P, P, 60, 0, 1, 1, 16, 1, 64, 96, P, P, 4, 1, 0, 0, P, P) == 1
    assert L.hs_layer_transfer(P, P, 64, 0, 1, 1, 16, 0, 64, 16384, P, P, 4, 1, 0, 0, P,
                               P) == 3
    # fp8_ds_mla rows: rows shorter than 656 B, a stride that is not a
    # multiple of 16, a missing workspace, negative sizes.
    assert L.hs_fp8ds_gather(P, 640, 10, P, P, 1, 4, P, P, P, P) == 1
    assert L.hs_fp8ds_gather(P, 664, 10, P, P, 1, 4, P, P, P, P) == 2
    assert L.hs_fp8ds_gather(P, 656, 10, P, P, 0, 4, P, P, P, P) == 0
    assert L.hs_sparse_decode_fp8ds_workspace_bytes(-1, 16, 64) == -1
    assert L.hs_sparse_decode_fp8ds(P, P, 656, 10, P, P, 1, 64, 16, 1.0, P, P, P, 0, P, P) == 3
    # Unsupported attention shape, null pointers.
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf) % 16), ctypes.c_void_p)
    assert L.hs_sparse_decode(p, p, p, 96, 0, 10, p, P, 1, 4, 4, 1, 96, 96, 1.0, p, P, P, 0, P,
                              P) == 7
    assert L.hs_sparse_decode(P, p, p, 576, 0, 10, p, P, 1, 4, 4, 1, 576, 512, 1.0, p, P, P, 0,
                              P, P) == 1
    assert L.hs_merge_states(P, P, P, 1, 0, 8, P, P, P) == 1
    # Partial states: null outputs, and columns beyond parts_total.
    assert L.hs_sparse_decode_partial(p, p, p, 576, 0, 10, p, P, 1, 4, 16, 1, 576, 512, 1.0, P,
                                      P, P, 1, 0, P, P) == 1
    assert L.hs_sparse_decode_partial(p, p, p, 576, 0, 10, p, P, 1, 4, 16, 1, 576, 512, 1.0, p,
                                      p, p, 1, 1, P, P) == 1


@pytest.mark.parametrize("rows,heads,cap", [(32, 128, 2048), (64, 16, 2048), (1, 16, 64)])
def test_workspace_query_is_pure(rows, heads, cap):
    # Works without a device (falls back to 1 SM for the split policy).
    a = hs.sparse_decode_workspace_bytes(rows, heads, 1, cap, 576, 512)
    b = hs.sparse_decode_workspace_bytes(rows, heads, 1, cap, 576, 512)
    assert a == b and a >= 0


def test_fused_normalize_lookup_argument_checks():
    L = hs.lib()
    P = None
    # S1's checks: negative rows; cap below n_cand + window + sinks.
    assert L.hs_normalize_lookup_assign(P, -1, 4, 0, 0, P, P, P, 4, 4, P, 1, 1, 64, 4, P, P, P, P,
                                        P, P, P, 8, 9, P, P, P, P, P, P, P, P, P, P) == 1
    assert L.hs_normalize_lookup_assign(P, 1, 4, 2, 1, P, P, P, 4, 4, P, 1, 1, 64, 6, P, P, P, P,
                                        P, P, P, 8, 9, P, P, P, P, P, P, P, P, P, P) == 3
    # S2's checks: cap > hot_size; region stride below hot_size + 1.
    assert L.hs_normalize_lookup_assign(P, 1, 4, 0, 0, P, P, P, 4, 4, P, 1, 1, 64, 9, P, P, P, P,
                                        P, P, P, 8, 9, P, P, P, P, P, P, P, P, P, P) == 3
    assert L.hs_normalize_lookup_assign(P, 1, 4, 0, 0, P, P, P, 4, 4, P, 1, 1, 64, 4, P, P, P, P,
                                        P, P, P, 8, 8, P, P, P, P, P, P, P, P, P, P) == 1
    # Null outputs with rows > 0.
    assert L.hs_normalize_lookup_assign(P, 1, 4, 0, 0, P, P, P, 4, 4, P, 1, 1, 64, 4, P, P, P, P,
                                        P, P, P, 8, 9, P, P, P, P, P, P, P, P, P, P) == 1
