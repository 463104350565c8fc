"""Pins for the oracle's sparse decode attention (S4) and the split-KV merge.

Fixed by: library routines that compute the same function another way
(torch's scaled_dot_product_attention with a -inf mask over the dense context,
torch.logsumexp), closed forms (one candidate gives V_j exactly; all-equal
logits give the mean of V and LSE = ln |S|; an empty set gives 0 and -inf), the
multiset rule of PaperTrace 5.1.1 section 7.3 (a repeated key adds ln 2 to its
logit), and the eq. (7) / eq. (14) merge values printed in PaperTrace 5.1.1
sections 3.2 and 7.1 (tests/golden/merge_examples.txt).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from golden_io import load


def bf16_bits(t):
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def make_case(seed, rows, heads, kv_heads, d_qk, d_v, n_kv, cap, shared_kv):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(rows, heads, d_qk, generator=g).to(torch.bfloat16)
    if shared_kv:
        kv = torch.randn(n_kv, kv_heads, d_qk, generator=g).to(torch.bfloat16)
        k, v = kv, kv[..., :d_v]
    else:
        k = torch.randn(n_kv, kv_heads, d_qk, generator=g).to(torch.bfloat16)
        v = torch.randn(n_kv, kv_heads, d_v, generator=g).to(torch.bfloat16)
    return q, k, v


def sdpa_reference(q, k, v, sets, scale, kv_heads):
    """Dense attention over all n_kv rows with -inf outside each set."""
    rows, heads, _ = q.shape
    group = heads // kv_heads
    n_kv = k.shape[0]
    out = torch.zeros(rows, heads, v.shape[-1], dtype=torch.float64)
    lse = torch.zeros(rows, heads, dtype=torch.float64)
    for r in range(rows):
        for g in range(kv_heads):
            mask = torch.full((n_kv,), float("-inf"), dtype=torch.float64)
            mask[sets[r][g]] = 0.0
            qh = q[r, g * group:(g + 1) * group].double()          # [group, d_qk]
            kh = k[:, g].double()                                   # [n_kv, d_qk]
            vh = v[:, g].double()
            o = F.scaled_dot_product_attention(qh[None, :, None], kh[None, None].expand(1, group, -1, -1),
                                               vh[None, None].expand(1, group, -1, -1),
                                               attn_mask=mask[None, None, None], scale=scale)
            out[r, g * group:(g + 1) * group] = o[0, :, 0]
            logits = (qh @ kh.T) * scale + mask
            lse[r, g * group:(g + 1) * group] = torch.logsumexp(logits, dim=-1)
    return out, lse


def run_oracle(q, k, v, kv_rows, count, scale, d_v, shared_kv):
    n_kv, kv_heads, d_qk = k.shape
    kb = bf16_bits(k).reshape(-1)
    if shared_kv:
        vb = kb
        row_stride, head_stride = kv_heads * d_qk, d_qk
    else:
        vb = bf16_bits(v).reshape(-1)
        assert v.shape[-1] == d_qk  # same strides for K and V in these cases
        row_stride, head_stride = kv_heads * d_qk, d_qk
    return oracle.sparse_decode(bf16_bits(q), kb, vb, row_stride, head_stride, kv_rows, count,
                                scale, d_v=d_v)


@pytest.mark.parametrize("case", [
    # (heads, kv_heads, d_qk, d_v, shared_kv)  -- GQA with separate K/V, MLA-like shared row
    (8, 2, 32, 32, False),
    (4, 1, 48, 32, True),
    (6, 3, 16, 16, False),
])
def test_sparse_equals_masked_dense(case):
    heads, kv_heads, d_qk, d_v, shared = case
    rows, n_kv, cap = 3, 40, 12
    q, k, v = make_case(1, rows, heads, kv_heads, d_qk, d_v, n_kv, cap, shared)
    rng = np.random.default_rng(2)
    kv_rows = np.full((rows, kv_heads, cap), -1, np.int32)
    count = np.zeros((rows, kv_heads), np.int32)
    sets = []
    for r in range(rows):
        sr = []
        for g in range(kv_heads):
            n = int(rng.integers(1, cap + 1))
            idx = rng.choice(n_kv, size=n, replace=False)
            kv_rows[r, g, :n] = idx
            count[r, g] = n
            # Some -1 holes inside the counted prefix are skipped.
            if n > 3:
                kv_rows[r, g, 1] = -1
                idx = np.delete(idx, 1)
            sr.append(idx.tolist())
        sets.append(sr)
    scale = 1.0 / math.sqrt(d_qk)
    out, lse = run_oracle(q, k, v, kv_rows, count, scale, d_v, shared)
    ref_out, ref_lse = sdpa_reference(q, k, v, sets, scale, kv_heads)
    np.testing.assert_allclose(out, ref_out.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_full_set_is_textbook_decode():
    rows, heads, d, n_kv = 2, 4, 64, 33
    q, k, v = make_case(3, rows, heads, 1, d, d, n_kv, n_kv, False)
    kv_rows = np.tile(np.arange(n_kv, dtype=np.int32), (rows, 1, 1))
    out, _ = run_oracle(q, k, v, kv_rows, None, 0.125, d, False)
    ref = F.scaled_dot_product_attention(q.double()[:, :, None], k[:, 0].double()[None, None],
                                         v[:, 0].double()[None, None], scale=0.125)[:, :, 0]
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_single_candidate_is_exact_row():
    q, k, v = make_case(4, 1, 2, 1, 32, 32, 10, 1, False)
    kv_rows = np.array([[[7]]], np.int32)
    out, lse = run_oracle(q, k, v, kv_rows, None, 0.3, 32, False)
    assert (out[0] == v[7, 0].double().numpy()[None]).all()
    s = (q[0].double() @ k[7, 0].double()) * 0.3
    np.testing.assert_allclose(lse[0], s.numpy(), rtol=1e-13)


def test_equal_logits_mean_and_log_count():
    _, k, v = make_case(5, 1, 2, 1, 16, 16, 20, 5, False)
    q = torch.zeros(1, 2, 16)
    idx = [3, 9, 11, 17, 2]
    kv_rows = np.array([[idx]], np.int32)
    out, lse = run_oracle(q, k, v, kv_rows, None, 0.7, 16, False)
    mean = v[idx, 0].double().mean(0).numpy()
    np.testing.assert_allclose(out[0, 0], mean, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse[0], math.log(5), rtol=1e-14)


def test_empty_set():
    q, k, v = make_case(6, 2, 2, 1, 16, 16, 8, 4, False)
    kv_rows = np.full((2, 1, 4), -1, np.int32)
    kv_rows[1, 0, :2] = [1, 2]
    count = np.array([[4], [0]], np.int32)  # row 1 has entries but count 0
    out, lse = run_oracle(q, k, v, kv_rows, count, 0.25, 16, False)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_multiset_adds_log2():
    q, k, v = make_case(7, 1, 1, 1, 16, 16, 8, 3, False)
    out_dup, lse_dup = run_oracle(q, k, v, np.array([[[2, 2, 5]]], np.int32), None, 0.5, 16, False)
    s = (k[:, 0].double() @ q[0, 0].double()) * 0.5
    logits = torch.stack([s[2] + math.log(2), s[5]])
    w = torch.softmax(logits, 0)
    ref = w[0] * v[2, 0].double() + w[1] * v[5, 0].double()
    np.testing.assert_allclose(out_dup[0, 0], ref.numpy(), rtol=1e-12)
    np.testing.assert_allclose(lse_dup[0, 0], torch.logsumexp(logits, 0).item(), rtol=1e-13)


def test_normalised_duplicates_match_unique():
    """S1 then S4: duplicated candidates count once (PaperTrace 5.1.1 section 1.1)."""
    B, T = 4, 32
    table = np.array([np.random.default_rng(8).permutation(8)], np.int32)
    q, k, v = make_case(8, 1, 2, 1, 16, 16, 32, 12, False)
    c_dup = np.array([[3, 9, 3, 20, 9, 9, 31]], np.int32)
    c_uni = np.array([[3, 9, 20, 31, -1, -1, -1]], np.int32)
    res = []
    for c in (c_dup, c_uni):
        _, slot, count, err = oracle.normalize_indices(c, [0], [T], table, B, num_pages=8)
        res.append(run_oracle(q, k, v, slot[:, None, :], count[:, None], 0.25, 16, False))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    np.testing.assert_array_equal(res[0][1], res[1][1])


def test_merge_worked_examples():
    g = load("merge_examples.txt")
    m = np.array([g["eq7_parts_m"]], np.float64)
    l = np.array([g["eq7_parts_l"]], np.float64)
    o = np.array(g["eq7_parts_o"], np.float64).reshape(1, 2, 1)
    mo, lo, oo = oracle.merge(m, l, o)
    assert mo[0] == 2
    assert abs(lo[0] - g["eq7_l_approx"]) < 5e-4
    assert abs(oo[0, 0] - g["eq7_o_approx"]) < 5e-4
    assert abs(oo[0, 0] / lo[0] - g["eq7_out_approx"]) < 1e-12
    assert abs(oo[0, 0] / lo[0] - g["eq7_wrong_sum"]) > 1.0
    m = np.array([g["eq14_parts_m"]], np.float64)
    l = np.array([g["eq14_parts_l"]], np.float64)
    mo, lo, _ = oracle.merge(m, l, np.zeros((1, 4, 1)))
    assert mo[0] == g["eq14_m"]
    assert abs(lo[0] - g["eq14_l_approx"]) < 5e-3


@pytest.mark.parametrize("parts", [1, 2, 8])
def test_split_merge_equals_unsplit(parts):
    """Split counts 1/2/8 against no split (PaperTrace 5.1.1 section 6.1 test matrix);
    an empty split (l = 0) is skipped."""
    rows, heads, d, n_kv, cap = 2, 3, 32, 64, 40
    q, k, v = make_case(9, rows, heads, 1, d, d, n_kv, cap, False)
    rng = np.random.default_rng(9)
    idx = np.stack([rng.choice(n_kv, size=cap, replace=False) for _ in range(rows)]).astype(np.int32)
    full_out, full_lse = run_oracle(q, k, v, idx[:, None], None, 0.2, d, False)
    bounds = np.linspace(0, cap, parts + 1).astype(int)
    ms, ls, os_ = [], [], []
    for p in range(parts):
        sub = np.full((rows, 1, cap), -1, np.int32)
        sub[:, 0, : bounds[p + 1] - bounds[p]] = idx[:, bounds[p]:bounds[p + 1]]
        o_p, lse_p = run_oracle(q, k, v, sub, None, 0.2, d, False)
        ms.append(lse_p)
        ls.append(np.ones_like(lse_p))
        os_.append(o_p)
    # One extra empty part.
    ms.append(np.full_like(ms[0], -np.inf))
    ls.append(np.zeros_like(ls[0]))
    os_.append(np.zeros_like(os_[0]))
    m = np.stack(ms, -1).reshape(rows * heads, -1)
    l = np.stack(ls, -1).reshape(rows * heads, -1)
    o = np.stack(os_, -2).reshape(rows * heads, len(ms), d)
    mo, lo, oo = oracle.merge(m, l, o)
    np.testing.assert_allclose((oo / lo[:, None]).reshape(rows, heads, d), full_out, rtol=1e-12,
                               atol=1e-13)
    np.testing.assert_allclose((mo + np.log(lo)).reshape(rows, heads), full_lse, rtol=1e-12)
