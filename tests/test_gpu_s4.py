"""S4 parity: hs_sparse_decode (and the eq. (7) merge kernel) against the fp64
oracle, within max |err| <= 1e-2 and relative L2 <= 5e-3 for bf16 inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bits, check_attention, cuda
from sparse_top_kv_gb300 import hs, inputs

pytestmark = pytest.mark.gpu


def decode_both(q, k, v, kv_rows, count, scale, d_v, row_stride, head_stride, sample_rows=None):
    """q bf16 cuda [rows, H, d_qk]; k/v bf16 cuda caches (v may be k)."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = hs.sparse_decode(q, k, v, row_stride, head_stride, k.numel() // row_stride,
                                cuda(kv_rows), None if count is None else cuda(count), scale,
                                d_v, status=status)
    torch.cuda.synchronize()
    rows = np.arange(q.shape[0]) if sample_rows is None else np.asarray(sample_rows)
    kb = bits(k).reshape(-1)
    vb = kb if v.data_ptr() == k.data_ptr() else bits(v).reshape(-1)
    ref_out, ref_lse = oracle.sparse_decode(bits(q)[rows], kb, vb, row_stride, head_stride,
                                            kv_rows[rows],
                                            None if count is None else count[rows], scale,
                                            d_v=d_v)
    check_attention(out[torch.from_numpy(rows).cuda()], lse[torch.from_numpy(rows).cuda()],
                    ref_out, ref_lse)
    return int(status.item())


def random_sets(rng, rows, kv_heads, cap, n_kv, holes=True, empty_row=True):
    kv_rows = np.full((rows, kv_heads, cap), -1, np.int32)
    count = np.zeros((rows, kv_heads), np.int32)
    for r in range(rows):
        for g in range(kv_heads):
            n = int(rng.integers(1, cap + 1))
            if empty_row and r == rows - 1 and g == 0:
                n = 0
            kv_rows[r, g, :n] = rng.choice(n_kv, size=n, replace=False)
            if holes and n > 4:
                kv_rows[r, g, rng.integers(0, n, size=2)] = -1
            count[r, g] = n
    return kv_rows, count


@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_gqa_small(group):
    rng = np.random.default_rng(group)
    rows, kv_heads, d, n_kv, cap = 3, 2, 128, 700, 300
    heads = group * kv_heads
    q = inputs.randn_bf16((rows, heads, d), 10 + group, device="cuda")
    k = inputs.randn_bf16((n_kv, kv_heads, d), 20 + group, device="cuda")
    v = inputs.randn_bf16((n_kv, kv_heads, d), 30 + group, device="cuda")
    kv_rows, count = random_sets(rng, rows, kv_heads, cap, n_kv)
    assert decode_both(q, k, v, kv_rows, count, 1 / math.sqrt(d), d, kv_heads * d, d) == 0


@pytest.mark.parametrize("group", [4, 8])
def test_gqa_long_lists_one_split(group):
    """Enough (row, KV head) units that no list is split, each longer than the
    kernel stages at once (2048 ids): several id chunks per CTA, ragged tail."""
    rng = np.random.default_rng(70 + group)
    rows, kv_heads, d, n_kv, cap = 40, 8, 128, 9000, 4500
    heads = group * kv_heads
    q = inputs.randn_bf16((rows, heads, d), 71 + group, device="cuda")
    k = inputs.randn_bf16((n_kv, kv_heads, d), 72 + group, device="cuda")
    v = inputs.randn_bf16((n_kv, kv_heads, d), 73 + group, device="cuda")
    kv_rows, count = random_sets(rng, rows, kv_heads, cap, n_kv)
    count[:4] = cap - np.arange(4)[:, None]
    for r in range(4):
        for g in range(kv_heads):
            kv_rows[r, g] = rng.choice(n_kv, size=cap, replace=False)
            kv_rows[r, g, count[r, g]:] = -1
    assert decode_both(q, k, v, kv_rows, count, 1 / math.sqrt(d), d, kv_heads * d, d,
                       sample_rows=[0, 1, 2, 3, 17, rows - 1]) == 0


@pytest.mark.parametrize("heads", [16, 128])
def test_mla_small(heads):
    rng = np.random.default_rng(heads)
    rows, n_kv, cap = 3, 2000, 600
    q = inputs.randn_bf16((rows, heads, 576), 40, device="cuda")
    cache = inputs.randn_bf16((n_kv, 576), 41, device="cuda")
    kv_rows, count = random_sets(rng, rows, 1, cap, n_kv)
    assert decode_both(q, cache, cache, kv_rows, count, 1 / 24, 512, 576, 0) == 0


@pytest.mark.parametrize("rows,heads,cap", [(152, 16, 384), (76, 128, 256), (200, 32, 300)])
def test_mla_many_tiles_per_cta(rows, heads, cap):
    """Enough rows that each CTA walks several 128-row tiles of its list."""
    rng = np.random.default_rng(rows + heads)
    n_kv = 20000
    q = inputs.randn_bf16((rows, heads, 576), 42, device="cuda")
    cache = inputs.randn_bf16((n_kv, 576), 43, device="cuda")
    kv_rows, count = random_sets(rng, rows, 1, cap, n_kv)
    count[:, 0] = np.maximum(count[:, 0], cap - 5)
    assert decode_both(q, cache, cache, kv_rows, count, 1 / 24, 512, 576, 0,
                       sample_rows=[0, 1, rows // 2, rows - 1]) == 0


@pytest.mark.parametrize("rows", [6, 37])
def test_mla_128_heads_two_splits(rows):
    """128 heads with lists of 257..512 rows: two splits per row.  Up to the
    number of co-resident clusters of four CTAs (6 rows), a row's two CTA
    pairs are one cluster and merge through distributed shared memory; 37
    rows run as separate pairs merged through global memory.  Rows with an
    empty list, with one tile only (the second split empty), a ragged tail
    and the full 512 rows, every row checked."""
    rng = np.random.default_rng(700 + rows)
    n_kv, cap = 6000, 500
    q = inputs.randn_bf16((rows, 128, 576), 70 + rows, device="cuda")
    cache = inputs.randn_bf16((n_kv, 576), 71, device="cuda")
    kv_rows = np.full((rows, 1, cap), -1, np.int32)
    count = np.zeros((rows, 1), np.int32)
    sizes = [0, 1, 128, 129, 300, cap] + [int(x) for x in rng.integers(200, cap + 1, rows)]
    for r in range(rows):
        n = sizes[r]
        kv_rows[r, 0, :n] = rng.choice(n_kv, size=n, replace=False)
        count[r, 0] = n
    assert decode_both(q, cache, cache, kv_rows, count, 1 / 24, 512, 576, 0) == 0


def test_mla_16_heads_two_splits():
    """16 heads, 64 rows of up to 300 candidates: two splits per row, merged
    with eq. (7) by the split that finishes last.  Empty, 1-row, one-tile,
    two-tile and ragged lists, every row checked."""
    rng = np.random.default_rng(640)
    rows, n_kv, cap = 64, 6000, 300
    q = inputs.randn_bf16((rows, 16, 576), 72, device="cuda")
    cache = inputs.randn_bf16((n_kv, 576), 73, device="cuda")
    kv_rows = np.full((rows, 1, cap), -1, np.int32)
    count = np.zeros((rows, 1), np.int32)
    sizes = [0, 1, 128, 129, 256, 257, cap] + [int(x) for x in rng.integers(1, cap + 1, rows)]
    for r in range(rows):
        n = sizes[r]
        kv_rows[r, 0, :n] = rng.choice(n_kv, size=n, replace=False)
        count[r, 0] = n
    assert decode_both(q, cache, cache, kv_rows, count, 1 / 24, 512, 576, 0) == 0


def test_single_candidate_and_tail_sizes():
    rng = np.random.default_rng(11)
    n_kv = 400
    cache = inputs.randn_bf16((n_kv, 576), 50, device="cuda")
    for cap in (1, 15, 16, 17, 63, 64, 65, 129):
        q = inputs.randn_bf16((2, 16, 576), 51 + cap, device="cuda")
        kv_rows = np.stack([rng.choice(n_kv, size=cap, replace=False) for _ in range(2)])
        decode_both(q, cache, cache, kv_rows[:, None].astype(np.int32), None, 1 / 24, 512, 576, 0)


def test_out_of_range_rows_flagged_and_skipped():
    cache = inputs.randn_bf16((100, 576), 60, device="cuda")
    q = inputs.randn_bf16((1, 16, 576), 61, device="cuda")
    kv_rows = np.array([[[3, 7, 100, 55, 1000]]], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = hs.sparse_decode(q, cache, cache, 576, 0, 100, cuda(kv_rows), None, 1 / 24, 512,
                                status=status)
    torch.cuda.synchronize()
    assert status.item() == 6
    ref_out, ref_lse = oracle.sparse_decode(bits(q), bits(cache).reshape(-1),
                                            bits(cache).reshape(-1), 576, 0,
                                            np.array([[[3, 7, -1, 55, -1]]], np.int32), None,
                                            1 / 24, d_v=512)
    check_attention(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("heads,d", [(16, 576), (128, 576), (4, 128)])
def test_partial_passes_merge_to_the_full_set(heads, d):
    """Two partial passes over disjoint halves of each candidate list (as the
    pipeline does for resident and swapped rows), merged by eq. (7), equal
    the oracle over the whole list."""
    rng = np.random.default_rng(heads + d)
    rows, n_kv, cap = 40, 5000, 700
    mla = d == 576
    kv_heads = 1 if mla else 2
    q = inputs.randn_bf16((rows, heads * (1 if mla else kv_heads), d), 90, device="cuda")
    H = q.shape[1]
    if mla:
        k = v = inputs.randn_bf16((n_kv, 576), 91, device="cuda")
        rs, hsd, d_v = 576, 0, 512
    else:
        k = inputs.randn_bf16((n_kv, kv_heads, d), 92, device="cuda")
        v = inputs.randn_bf16((n_kv, kv_heads, d), 93, device="cuda")
        rs, hsd, d_v = kv_heads * d, d, d
    full, count = random_sets(rng, rows, kv_heads, cap, n_kv)
    a = np.full_like(full, -1)
    b = np.full_like(full, -1)
    ca = np.zeros_like(count)
    cb = np.zeros_like(count)
    for r in range(rows):
        for g in range(kv_heads):
            n = count[r, g]
            sel = rng.random(n) < 0.8
            ia = full[r, g, :n][sel]
            ib = full[r, g, :n][~sel]
            a[r, g, :n] = np.where(sel, full[r, g, :n], -1)  # in place, holes elsewhere
            b[r, g, :len(ib)] = ib                           # compact
            ca[r, g], cb[r, g] = n, len(ib)
    pa = hs.sparse_decode_partial_splits(rows, H, kv_heads, cap, d, d_v)
    pb = hs.sparse_decode_partial_splits(rows, H, kv_heads, cap, d, d_v)
    P = pa + pb + 1
    pm = torch.full((rows * H, P), -np.inf, dtype=torch.float32, device="cuda")
    pl = torch.zeros(rows * H, P, dtype=torch.float32, device="cuda")
    po = torch.zeros(rows * H, P, d_v, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nkv = k.numel() // rs
    assert hs.sparse_decode_partial(q, k, v, rs, hsd, nkv, cuda(a), cuda(ca), 1 / math.sqrt(d),
                                    d_v, pm, pl, po, 0, status=status) == pa
    hs.sparse_decode_partial(q, k, v, rs, hsd, nkv, cuda(b), cuda(cb), 1 / math.sqrt(d), d_v,
                             pm, pl, po, pa, status=status)
    out, lse = hs.merge_states(pm, pl, po)  # the extra empty column (l = 0) is skipped
    # The fused last pass: the second half attended and merged in one call.
    out2, lse2 = hs.sparse_decode_finish(q, k, v, rs, hsd, nkv, cuda(b), cuda(cb),
                                         1 / math.sqrt(d), d_v, pm, pl, po, pa, status=status)
    # The split last pass: several CTAs per row, the last to arrive merges.
    # The counters are zero on entry and every call leaves them zero: two
    # calls in a row, no reset in between.
    sync = torch.zeros((rows * H,), dtype=torch.int32, device="cuda")
    for _ in range(2):
        out3, lse3 = hs.sparse_decode_finish(q, k, v, rs, hsd, nkv, cuda(b), cuda(cb),
                                             1 / math.sqrt(d), d_v, pm, pl, po, pa, sync=sync,
                                             status=status)
    torch.cuda.synchronize()
    assert int(sync.abs().sum().item()) == 0
    assert status.item() == 0
    sample = [0, 7, rows - 1]
    kb = bits(k).reshape(-1)
    vb = kb if mla else bits(v).reshape(-1)
    ref_out, ref_lse = oracle.sparse_decode(bits(q)[sample], kb, vb, rs, hsd, full[sample],
                                            count[sample], 1 / math.sqrt(d), d_v=d_v)
    idx = torch.tensor(sample, device="cuda")
    check_attention(out.view(rows, H, d_v)[idx], lse.view(rows, H)[idx], ref_out, ref_lse)
    check_attention(out2[idx], lse2[idx], ref_out, ref_lse, label="finish")
    check_attention(out3[idx], lse3[idx], ref_out, ref_lse, label="finish with split merge")


def test_merge_states_kernel():
    rng = np.random.default_rng(12)
    n, parts, d = 37, 5, 512
    m = rng.normal(size=(n, parts)) * 4
    l = rng.uniform(0.5, 30, size=(n, parts))
    o = rng.normal(size=(n, parts, d)) * l[..., None]
    l[3, :] = 0  # an all-empty state
    m[3, :] = -np.inf
    l[5, 2] = 0  # one empty part
    m[5, 2] = -np.inf
    mt = torch.tensor(m, dtype=torch.float32, device="cuda")
    lt = torch.tensor(l, dtype=torch.float32, device="cuda")
    ot = torch.tensor(o, dtype=torch.float32, device="cuda")
    out, lse = hs.merge_states(mt, lt, ot)
    torch.cuda.synchronize()
    # The kernel takes m in log2 units: convert for the natural-log oracle.
    m32 = mt.double().cpu().numpy()
    M, L, O = oracle.merge(m32 * math.log(2), lt.double().cpu().numpy(), ot.double().cpu().numpy())
    ref = np.where(L[:, None] > 0, O / np.where(L > 0, L, 1)[:, None], 0.0)
    ref_lse = np.where(L > 0, M + np.log(np.where(L > 0, L, 1)), -np.inf)
    check_attention(out, lse, ref, ref_lse)


def test_mla_decode_config_sampled():
    """Full size (32 requests x 128 heads x 2048 rows from a 1.2 GB paged
    cache), after S1; outputs of 3 sampled requests checked against the oracle."""
    cfg = inputs.mla_decode()
    R = cfg["num_reqs"]
    tok, slot, count, err = hs.normalize_indices(
        cuda(cfg["cand"]), torch.arange(R, dtype=torch.int32, device="cuda"),
        torch.full((R,), cfg["ctx"], dtype=torch.int32, device="cuda"),
        cuda(cfg["block_table"]), 64, num_pages=cfg["num_pages"])
    kv_rows = slot.cpu().numpy()[:, None, :]
    cnt = count.cpu().numpy()[:, None]
    assert decode_both(cfg["q"], cfg["cache"], cfg["cache"], kv_rows, cnt, cfg["scale"], 512,
                       576, 0, sample_rows=[0, 17, 31]) == 0


def test_gqa_union_config_sampled():
    """Full size (16 requests, 8 KV heads, 4.3 GB of bshd K/V), S1 union with
    window and sinks then S4; 2 sampled requests checked against the oracle."""
    cfg = inputs.gqa_union()
    rows = cfg["cand"].shape[0]
    R, G = cfg["num_reqs"], cfg["kv_heads"]
    tok, slot, count, err = hs.normalize_indices(
        cuda(cfg["cand"]), cuda(cfg["row_req"]),
        torch.full((R,), cfg["ctx"], dtype=torch.int32, device="cuda"), cuda(cfg["block_table"]),
        16, window=256, num_sinks=4, num_pages=cfg["num_pages"])
    kv_rows = slot.cpu().numpy().reshape(R, G, -1)
    cnt = count.cpu().numpy().reshape(R, G)
    d = cfg["d"]
    assert rows == R * G
    assert decode_both(cfg["q"], cfg["k_cache"], cfg["v_cache"], kv_rows, cnt, cfg["scale"], d,
                       G * d, d, sample_rows=[0, 15]) == 0
