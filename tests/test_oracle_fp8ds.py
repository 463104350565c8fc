"""Oracle pins for fp8_ds_mla rows (vLLM HiSparse walkthrough: the
FlashMLASparseBackend cache shape and FP8_DS_MLA_ROW_BYTES = 656, i.e. 512 B
of quantised latent columns + 16 B of scales + 128 B of RoPE; PaperTrace
5.1.1 section 7.2: the scale is applied to the stored codes before the
products).  The decoder is checked against torch's float8_e4m3fn conversion
and against hand-computed values of the format's definition; the row layout
against rows written byte by byte; the rounding against torch's binary32
product and bf16 conversion; the attention against a numpy brute force."""
import math
import struct

import numpy as np
import pytest
import torch

import oracle


def bf16_bits(x):
    """float values -> bf16 bit patterns via torch (round to nearest even)."""
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def make_row(codes, scales, rope_bits):
    row = bytearray(656)
    row[:512] = bytes(np.asarray(codes, np.uint8))
    row[512:528] = struct.pack("<4f", *scales)
    row[528:] = np.asarray(rope_bits, "<u2").tobytes()
    return np.frombuffer(bytes(row), np.uint8)


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF]
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    # Signed zeros keep their sign.
    assert math.copysign(1.0, ours[0x80]) == -1.0 and math.copysign(1.0, ours[0x00]) == 1.0


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x39, 1.125), (0x3C, 1.5), (0x40, 2.0), (0x77, 240.0), (0x7E, 448.0),
    (0xB8, -1.0), (0xFE, -448.0), (0x81, -(2.0 ** -9)),
])
def test_e4m3_definition_values(code, value):
    assert oracle.e4m3_decode(np.array([code], np.uint8))[0] == value


def test_row_layout_scale_groups_and_rope():
    """All codes 1.0; each 128-column group has its own scale; RoPE bits are
    copied unchanged (bytes 528.. little-endian)."""
    rope = np.arange(64, dtype=np.uint16) * 997 + 0x3F00
    row = make_row(np.full(512, 0x38), (1.0, 2.0, 0.5, 4.0), rope)
    out = oracle.fp8ds_dequant(row[None])[0]
    vals = bits_to_f64(out[:512])
    for g, sc in enumerate((1.0, 2.0, 0.5, 4.0)):
        np.testing.assert_array_equal(vals[128 * g:128 * (g + 1)], sc)
    np.testing.assert_array_equal(out[512:], rope)


def test_codes_sit_in_column_order():
    """Code byte d is latent column d (a reversal or a stride would fail)."""
    codes = np.zeros(512, np.uint8)
    codes[[0, 1, 127, 128, 300, 511]] = [0x38, 0x40, 0x3C, 0xB8, 0x7E, 0x01]
    out = bits_to_f64(oracle.fp8ds_dequant(make_row(codes, (1, 1, 1, 1), np.zeros(64))[None])[0])
    exp = np.zeros(512)
    exp[[0, 1, 127, 128, 300, 511]] = [1.0, 2.0, 1.5, -1.0, 448.0, 2.0 ** -9]
    np.testing.assert_array_equal(out[:512], exp)


def test_product_rounds_to_nearest_even_bf16():
    # 1.0 * (1 + 2^-8) is half-way between bf16 1.0 and 1 + 2^-7 -> even (1.0);
    # 1.0 * (1 + 3 * 2^-8) is half-way between 1 + 2^-7 and 1 + 2^-6 -> 1 + 2^-6;
    # 1.125 * 1.01171875 = 1.13818359375 -> 1.140625.
    for scale, want in ((1 + 2.0 ** -8, 1.0), (1 + 3 * 2.0 ** -8, 1 + 2.0 ** -6)):
        row = make_row(np.full(512, 0x38), (scale,) * 4, np.zeros(64))
        assert bits_to_f64(oracle.fp8ds_dequant(row[None])[0][:1])[0] == want
    row = make_row(np.full(512, 0x39), (1.01171875,) * 4, np.zeros(64))
    assert bits_to_f64(oracle.fp8ds_dequant(row[None])[0][:1])[0] == 1.140625


def test_random_rows_match_torch_binary32_product():
    rng = np.random.default_rng(11)
    n = 64
    codes = rng.integers(0, 256, (n, 512), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3A  # no NaN codes
    scales = (rng.standard_normal((n, 4)) * 4).astype(np.float32)
    rope = rng.integers(0, 1 << 16, (n, 64), dtype=np.uint16)
    rows = np.stack([make_row(codes[i], scales[i], rope[i]) for i in range(n)])
    ids = rng.permutation(n)[:40]
    got = oracle.fp8ds_dequant(rows, ids)
    cf = torch.from_numpy(codes[ids].copy()).view(torch.float8_e4m3fn).to(torch.float32)
    sc = torch.from_numpy(np.repeat(scales[ids], 128, axis=1))
    want = (cf * sc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got[:, :512], want)
    np.testing.assert_array_equal(got[:, 512:], rope[ids])


def test_attention_on_fp8_rows_matches_brute_force():
    """Tiny case: softmax(q . K^T * scale) V over the reconstructed rows, in
    numpy fp64, with a padded entry, an id beyond the rows and a count."""
    rng = np.random.default_rng(12)
    n_rows, heads, cap = 40, 3, 9
    vals = torch.from_numpy(rng.standard_normal((n_rows, 576)).astype(np.float32))
    from sparse_top_kv_gb300 import inputs
    rows8 = inputs.fp8ds_encode(vals).numpy()
    q = bf16_bits(rng.standard_normal((2, heads, 576))).reshape(2, heads, 576)
    kv = rng.integers(0, n_rows, (2, 1, cap)).astype(np.int32)
    kv[0, 0, 2] = -1
    kv[1, 0, 4] = n_rows + 3
    count = np.array([[cap], [6]], np.int32)
    scale = 1 / 24
    out, lse = oracle.sparse_decode_fp8ds(q, rows8, kv, count, scale)
    deq = bits_to_f64(oracle.fp8ds_dequant(rows8)).reshape(n_rows, 576)
    qf = bits_to_f64(q).reshape(2, heads, 576)
    for r in range(2):
        ids = [int(i) for i in kv[r, 0, :count[r, 0]] if 0 <= i < n_rows]
        K = deq[ids]
        for h in range(heads):
            s = K @ qf[r, h] * scale
            m = s.max()
            p = np.exp(s - m)
            np.testing.assert_allclose(out[r, h], p @ K[:, :512] / p.sum(), rtol=1e-12,
                                       atol=1e-12)
            assert abs(lse[r, h] - (m + math.log(p.sum()))) < 1e-12


def test_swap_in_fp8ds_is_byte_swap_then_reconstruction():
    """The reconstructing SwapIn equals the byte-level SwapIn of the 656-byte
    rows into a staging buffer followed by fp8ds_dequant of the staged rows;
    a source outside the pool zeroes the hot row and revokes its slot."""
    rng = np.random.default_rng(13)
    host_rows, R, region, hot_size = 50, 2, 9, 8
    vals = torch.from_numpy(rng.standard_normal((host_rows, 576)).astype(np.float32))
    from sparse_top_kv_gb300 import inputs
    pool = inputs.fp8ds_encode(vals).numpy()
    msrc = np.array([[3, 49, 7, 0], [12, -1, 30, 0]], np.int32)
    mdst = np.array([[0, 5, 2, 0], [9 + 1, 9 + 4, 9 + 7, 0]], np.int64)
    mcount = np.array([3, 3], np.int32)
    hot = rng.integers(0, 1 << 16, (R * region, 576), dtype=np.uint16)
    expect = hot.copy()
    dgi = np.arange(R * hot_size, dtype=np.int32).reshape(R, hot_size)
    dgi_exp = dgi.copy()
    oracle.swap_in_fp8ds(pool, hot, msrc, mdst, mcount, dgi=dgi, hot_size=hot_size,
                         region_stride=region)
    staged = np.zeros((R * region, 656), np.uint8)
    oracle.swap_in(pool.reshape(-1), staged.reshape(-1), 656,
                   np.where(msrc >= 0, msrc, 0), mdst, mcount)
    for r in range(R):
        for m in range(mcount[r]):
            d = mdst[r, m]
            if msrc[r, m] >= 0:
                expect[d] = oracle.fp8ds_dequant(staged, [d])[0]
            else:
                expect[d] = 0
                dgi_exp[r, d - r * region] = -1
    np.testing.assert_array_equal(hot, expect)
    np.testing.assert_array_equal(dgi, dgi_exp)
