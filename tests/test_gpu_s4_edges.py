"""S4 numeric edge cases against the fp64 oracle (PaperTrace 5.1.1 section
6.1, the correctness matrix: very large positive and negative logits,
all-equal logits, fully masked rows), on every S4 entry point: the one-call
decode (split over CTAs, merged by the last CTA), the allocation-free call,
and the partial + finishing passes (with and without the split merge).

The inputs steer the kernels into their rarely taken branches:
  * logits that grow by more than 2^8 (log2 units) from one 128-row tile to
    the next, per head and only for some heads, so that the tcgen05 kernel
    rescales O inside tensor memory at t > 0, several times per CTA;
  * CTA ranges whose first tile (or first two tiles) hold no valid row, so
    that the first rescale multiplies by a factor of exactly 0;
  * a single row whose logit exceeds the rest by ~1500 (log2 units), rows at
    ~-1500 next to ordinary ones, and q = 0 (every logit equal).
The MLA rows take the large values only in their 64 RoPE columns (K = all 576
columns, V = the first 512), so V stays N(0, 1) and the bf16 output keeps its
resolution while the logits are extreme.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bits, check_attention, cuda
from sparse_top_kv_gb300 import hs, inputs

pytestmark = pytest.mark.gpu

TILE = 128  # candidate rows per tile of the tcgen05 kernel


def rope_case(rows, heads, cap, rope_of_pos, seed, q_zero=False):
    """MLA inputs: request r owns cache rows [r * cap, (r + 1) * cap) in list
    order; row j's RoPE columns are rope_of_pos(j) * rvec (rvec = +-1), q's
    RoPE columns are sign_h * rvec with sign_h cycling over +1, 0, -1 by head.
    Returns (q, cache, kv_rows [rows, 1, cap])."""
    rng = np.random.default_rng(seed)
    n_kv = rows * cap
    cache = inputs.randn_bf16((n_kv, 576), seed).float()
    rvec = torch.from_numpy(rng.choice([-1.0, 1.0], size=64).astype(np.float32))
    a = torch.from_numpy(np.asarray([rope_of_pos(j) for j in range(cap)], np.float32))
    cache.view(rows, cap, 576)[:, :, 512:] = a[None, :, None] * rvec[None, None, :]
    q = inputs.randn_bf16((rows, heads, 576), seed + 1).float()
    sign = torch.tensor([(1.0, 0.0, -1.0)[h % 3] for h in range(heads)])
    q[:, :, 512:] = sign[None, :, None] * rvec[None, None, :]
    if q_zero:
        q.zero_()
    kv_rows = (np.arange(rows, dtype=np.int64)[:, None] * cap +
               np.arange(cap)[None]).astype(np.int32)[:, None, :]
    return q.to(torch.bfloat16).cuda(), cache.to(torch.bfloat16).cuda(), kv_rows


def oracle_ref(q, cache, kv_rows, count, sample):
    kb = bits(cache).reshape(-1)
    return oracle.sparse_decode(bits(q)[sample], kb, kb, 576, 0, kv_rows[sample],
                                None if count is None else count[sample], 1 / 24, d_v=512)


def all_entry_points(q, cache, kv_rows, count, sample, label):
    """hs_sparse_decode, hs_sparse_decode_noalloc, and partial + finish over a
    split of every list into its first and second half, each against the
    oracle over the whole list."""
    rows, heads, _ = q.shape
    cap = kv_rows.shape[-1]
    n_kv = cache.shape[0]
    ref_out, ref_lse = oracle_ref(q, cache, kv_rows, count, sample)
    idx = torch.tensor(sample, device="cuda")
    kv_d = cuda(kv_rows)
    cnt_d = None if count is None else cuda(count)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    out, lse = hs.sparse_decode(q, cache, cache, 576, 0, n_kv, kv_d, cnt_d, 1 / 24, 512,
                                status=status)
    check_attention(out[idx], lse[idx], ref_out, ref_lse, label=f"{label} decode")

    out_n = torch.empty_like(out)
    lse_n = torch.empty_like(lse)
    hs.sparse_decode_noalloc(q, cache, cache, 576, 0, n_kv, kv_d, cnt_d, 1 / 24, 512,
                             out=out_n, lse=lse_n, status=status)
    check_attention(out_n[idx], lse_n[idx], ref_out, ref_lse, label=f"{label} noalloc")

    # First half of each list (in place, -1 elsewhere) as partial states,
    # the second half (compacted) in the finishing pass.
    n = np.full((rows, 1), cap, np.int32) if count is None else count
    first = np.full_like(kv_rows, -1)
    second = np.full_like(kv_rows, -1)
    c2 = np.zeros_like(n)
    for r in range(rows):
        h = int(n[r, 0]) // 2
        first[r, 0, :h] = kv_rows[r, 0, :h]
        rest = kv_rows[r, 0, h:int(n[r, 0])]
        second[r, 0, :len(rest)] = rest
        c2[r, 0] = len(rest)
    pa = hs.sparse_decode_partial_splits(rows, heads, 1, cap, 576, 512)
    pb = hs.sparse_decode_partial_splits(rows, heads, 1, cap, 576, 512)
    P = pa + pb
    pm = torch.full((rows * heads, P), -np.inf, dtype=torch.float32, device="cuda")
    pl = torch.zeros(rows * heads, P, dtype=torch.float32, device="cuda")
    po = torch.zeros(rows * heads, P, 512, dtype=torch.float32, device="cuda")
    hs.sparse_decode_partial(q, cache, cache, 576, 0, n_kv, cuda(first), cuda(n), 1 / 24, 512,
                             pm, pl, po, 0, status=status)
    out_f, lse_f = hs.sparse_decode_finish(q, cache, cache, 576, 0, n_kv, cuda(second),
                                           cuda(c2), 1 / 24, 512, pm, pl, po, pa,
                                           status=status)
    sync = torch.zeros(rows * heads, dtype=torch.int32, device="cuda")
    out_s, lse_s = hs.sparse_decode_finish(q, cache, cache, 576, 0, n_kv, cuda(second),
                                           cuda(c2), 1 / 24, 512, pm, pl, po, pa, sync=sync,
                                           status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert int(sync.abs().sum().item()) == 0
    check_attention(out_f[idx], lse_f[idx], ref_out, ref_lse, label=f"{label} finish")
    check_attention(out_s[idx], lse_s[idx], ref_out, ref_lse, label=f"{label} finish+sync")
    return ref_out, ref_lse


# Shapes: (rows, heads, cap).  rows * heads / HG units against the SM count
# decide the splits; every shape leaves at least two tiles per CTA.  With
# 128 heads, 40 rows run one split per CTA pair and 30 rows two splits (the
# pairs of a row merge inside one cluster); with 16 heads, 64 rows run two
# splits per row (the split that finishes last merges, in the finishing
# pass together with two earlier partial columns).
SHAPES = [(40, 16, 2048), (64, 16, 1024), (40, 32, 1536), (40, 128, 1024), (30, 128, 1024),
          (6, 20, 700)]


@pytest.mark.parametrize("rows,heads,cap", SHAPES)
def test_logits_growing_across_tiles(rows, heads, cap):
    """Every tile's largest logit exceeds the previous tile's by ~11.5 (log2
    units) for the heads with sign +1, decreases for sign -1, stays flat for
    sign 0: the O rescale in tensor memory runs at every t > 0 for a subset
    of the heads of one CTA."""
    q, cache, kv = rope_case(rows, heads, cap, lambda j: 3.0 * (j // TILE), 100 + heads)
    all_entry_points(q, cache, kv, None, [0, 1, rows // 2, rows - 1], "growing")


@pytest.mark.parametrize("rows,heads,cap", SHAPES)
def test_single_dominant_row_and_extreme_negatives(rows, heads, cap):
    """One row late in each list has RoPE 400 (logit ~ +1540 log2 units for
    the +1 heads, ~ -1540 for the -1 heads); every third row has RoPE -400
    (the reverse).  Weights that underflow to 0 next to weights of 1."""
    def a(j):
        if j == cap - 37:
            return 400.0
        return -400.0 if j % 3 == 1 else 0.0
    q, cache, kv = rope_case(rows, heads, cap, a, 200 + heads)
    ref_out, _ = all_entry_points(q, cache, kv, None, [0, rows - 1], "extreme")
    # Closed form for the +1 heads: the spike row's V (its logit exceeds the
    # next one by > 1000 log2 units, so every other weight is exactly 0 in
    # fp64), rounded to bf16 by the kernel.
    spike = cache[kv[0, 0, cap - 37]].float().cpu().numpy().astype(np.float64)[:512]
    np.testing.assert_allclose(ref_out[0, 0], spike, rtol=0, atol=1e-12)


@pytest.mark.parametrize("rows,heads,cap", SHAPES)
def test_all_equal_logits(rows, heads, cap):
    """q = 0: every logit is 0, the output is the mean of V over the valid
    rows and LSE = ln |S| (holes and a short count included)."""
    q, cache, kv = rope_case(rows, heads, cap, lambda j: 0.0, 300 + heads, q_zero=True)
    kv = kv.copy()
    kv[:, :, 5::17] = -1
    count = np.full((rows, 1), cap, np.int32)
    count[1, 0] = cap - 77
    ref_out, ref_lse = all_entry_points(q, cache, kv, count, [0, 1], "equal")
    valid = kv[1, 0, :count[1, 0]]
    valid = valid[valid >= 0]
    v = cache[torch.from_numpy(valid).long().cuda()].float().cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(ref_out[1, 3], v[:, :512].mean(axis=0), rtol=0, atol=1e-9)
    assert abs(ref_lse[1, 3] - math.log(len(valid))) < 1e-9


@pytest.mark.parametrize("rows,heads,cap", SHAPES)
def test_leading_tiles_fully_masked(rows, heads, cap):
    """The first tile (row 0: the first two tiles) of every CTA's range of
    the list holds only -1, so the first valid tile rescales an empty O by a
    factor of 0; one list is -1 throughout (zero output, LSE = -inf); logits
    grow across the valid tiles as well."""
    q, cache, kv = rope_case(rows, heads, cap, lambda j: 3.0 * (j // TILE), 400 + heads)
    kv = kv.copy()
    splits = hs.sparse_decode_partial_splits(rows, heads, 1, cap, 576, 512)
    ntiles = (cap + TILE - 1) // TILE
    per = (ntiles + splits - 1) // splits
    for r in range(rows):
        lead = 2 if r == 0 else 1
        for s in range(splits):
            t0 = s * per
            if t0 >= ntiles:
                break
            kv[r, 0, t0 * TILE:min(cap, (t0 + lead) * TILE)] = -1
    kv[rows - 1] = -1
    out = all_entry_points(q, cache, kv, None, [0, 1, rows - 1], "masked")
    assert np.all(np.isneginf(out[1][-1]))
    assert np.all(out[0][-1] == 0.0)


# GQA (d = 128, separate K and V caches): the same growth and extremes
# through the warp-level MMA kernel, whose online softmax rescales per block
# of 16 candidates.
@pytest.mark.parametrize("group", [4, 8])
@pytest.mark.parametrize("case", ["growing", "extreme", "equal", "masked"])
def test_gqa_edges(group, case):
    rng = np.random.default_rng(500 + group)
    rows, kv_heads, d, cap = 6, 2, 128, 1100
    heads = group * kv_heads
    n_kv = rows * cap
    u = torch.from_numpy(rng.choice([-1.0, 1.0], size=d).astype(np.float32))
    k = inputs.randn_bf16((n_kv, kv_heads, d), 501 + group).float()
    v = inputs.randn_bf16((n_kv, kv_heads, d), 502 + group).cuda()
    j = np.arange(cap)
    if case == "growing":
        a = (j // 16).astype(np.float32)          # +16 log2 units per block of 16
    elif case == "extreme":
        a = np.where(j % 3 == 1, -60.0, 0.0).astype(np.float32)
        a[cap - 5] = 60.0
    else:
        a = np.zeros(cap, np.float32)
    k.view(rows, cap, kv_heads, d)[:] += torch.from_numpy(a)[None, :, None, None] * u
    q = inputs.randn_bf16((rows, heads, d), 503 + group).float()
    sign = torch.tensor([(1.0, 0.0, -1.0)[h % 3] for h in range(heads)])
    q += sign[None, :, None] * u[None, None, :]
    if case == "equal":
        q.zero_()
    q = q.to(torch.bfloat16).cuda()
    k = k.to(torch.bfloat16).cuda()
    kv_rows = np.broadcast_to((np.arange(rows)[:, None, None] * cap + j[None, None, :]),
                              (rows, kv_heads, cap)).astype(np.int32).copy()
    if case == "masked":
        kv_rows[:, :, :300] = -1     # the first blocks of every warp and split
        kv_rows[rows - 1] = -1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = hs.sparse_decode(q, k, v, kv_heads * d, d, n_kv, cuda(kv_rows), None,
                                1 / math.sqrt(d), d, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ref_out, ref_lse = oracle.sparse_decode(bits(q), bits(k).reshape(-1), bits(v).reshape(-1),
                                            kv_heads * d, d, kv_rows, None, 1 / math.sqrt(d),
                                            d_v=d)
    check_attention(out, lse, ref_out, ref_lse, label=f"gqa {case}")
