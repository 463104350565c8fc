"""fp8_ds_mla rows on the GPU: the row reconstruction bit for bit against the
oracle (every E4M3 code, subnormals, signed zeros, group scales, RoPE bytes,
padding, ids beyond the rows, counts), S4 over fp8 rows within the attention
tolerance against the fp64 oracle on the reconstructed rows (several tiles,
ragged tails, empty lists, 16 / 64 / 128 heads, the full-size paged decode
sampled), and SwapIn / BackUp of 656-byte rows byte for byte."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import bits, check_attention, cuda, np_i32, u8
from sparse_top_kv_gb300 import hs, inputs

pytestmark = pytest.mark.gpu

RB = 656


def random_fp8_rows(rng, n, nan_free=True):
    """Rows of random bytes (every code value occurs), with finite random
    scales (some tiny, some large) and random RoPE bits."""
    rows = rng.integers(0, 256, (n, RB), dtype=np.uint8)
    if nan_free:
        lat = rows[:, :512]
        lat[(lat & 0x7F) == 0x7F] = 0x5A
    sc = (rng.standard_normal((n, 4)) * np.exp2(rng.integers(-20, 20, (n, 4)))).astype(np.float32)
    rows[:, 512:528] = sc.view(np.uint8).reshape(n, 16)
    rope = rng.standard_normal((n, 64)).astype(np.float32)
    rows[:, 528:] = bits(torch.from_numpy(rope).to(torch.bfloat16)).view(np.uint8).reshape(n, 128)
    return rows


def gather_both(rows8, kv_rows, count, row_bytes=RB):
    n_rows = rows8.shape[0]
    dev = torch.zeros(n_rows, row_bytes, dtype=torch.uint8, device="cuda")
    dev[:, :RB] = cuda(rows8)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, ids = hs.fp8ds_gather(dev, cuda(kv_rows), None if count is None else cuda(count),
                               status=status)
    torch.cuda.synchronize()
    got = bits(out).reshape(kv_rows.shape[0], kv_rows.shape[1], 576)
    got_ids = np_i32(ids).reshape(kv_rows.shape)
    R, cap = kv_rows.shape
    n = np.full(R, cap) if count is None else np.clip(count, 0, cap)
    for r in range(R):
        for j in range(n[r]):
            i = int(kv_rows[r, j])
            if 0 <= i < n_rows:
                assert got_ids[r, j] == r * cap + j
                np.testing.assert_array_equal(got[r, j], oracle.fp8ds_dequant(rows8, [i])[0],
                                              err_msg=f"row {r} entry {j} id {i}")
            else:
                assert got_ids[r, j] == -1
    return int(status.item())


@pytest.mark.parametrize("row_bytes", [656, 672, 1024])
def test_gather_every_code_and_layout(row_bytes):
    rng = np.random.default_rng(row_bytes)
    rows8 = random_fp8_rows(rng, 300)
    # Every code in one row, a zero-scale row, signed zeros and subnormals.
    rows8[0, :256] = np.arange(256)
    rows8[0, 256:512] = np.arange(256)[::-1]
    rows8[0, :512][(rows8[0, :512] & 0x7F) == 0x7F] = 0x01
    rows8[0, 512:528] = np.array([1.0, -2.0, 2.0 ** -30, 3.0e9], np.float32).view(np.uint8)
    rows8[1, 512:528] = 0
    kv_rows = np.stack([rng.choice(300, 70, replace=False) for _ in range(5)]).astype(np.int32)
    kv_rows[:, 0] = [0, 1, 2, 299, 0]
    kv_rows[1, 5] = -1
    count = np.array([70, 33, 0, 69, 1], np.int32)
    assert gather_both(rows8, kv_rows, count, row_bytes) == 0


def test_gather_nan_codes_stay_nan():
    rng = np.random.default_rng(3)
    rows8 = random_fp8_rows(rng, 4, nan_free=False)
    rows8[2, :512:7] = 0x7F
    rows8[2, 3:512:7] = 0xFF
    kv_rows = np.array([[2, 0, 3, 1]], np.int32)
    dev = cuda(rows8)
    out, _ = hs.fp8ds_gather(dev, cuda(kv_rows), None)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()[0]
    ref = oracle.fp8ds_dequant(rows8, [2])[0]
    ref_f = (ref.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref_f))
    fin = ~np.isnan(ref_f)
    np.testing.assert_array_equal(bits(out)[0][fin], ref[fin])


def test_gather_ids_beyond_rows_flagged():
    rng = np.random.default_rng(4)
    rows8 = random_fp8_rows(rng, 50)
    kv_rows = np.array([[3, 50, 7, -1, 1000, 49]], np.int32)
    assert hs.status_string(gather_both(rows8, kv_rows, None)) == "HS_ERR_BAD_INDEX"


def decode_fp8_both(q, rows8_np, rows8_dev, kv_rows, count, scale, sample_rows=None):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = hs.sparse_decode_fp8ds(q, rows8_dev, cuda(kv_rows),
                                      None if count is None else cuda(count), scale,
                                      status=status)
    torch.cuda.synchronize()
    rows = np.arange(q.shape[0]) if sample_rows is None else np.asarray(sample_rows)
    ref_out, ref_lse = oracle.sparse_decode_fp8ds(
        bits(q)[rows], rows8_np, kv_rows[rows], None if count is None else count[rows], scale)
    sel = torch.from_numpy(rows).cuda()
    check_attention(out[sel], lse[sel], ref_out, ref_lse)
    return int(status.item())


@pytest.mark.parametrize("heads", [16, 20, 64, 128])
def test_decode_small(heads):
    """Lists of up to 600 rows (several 128-row tiles, ragged tails), holes,
    one empty list; 20 heads attend on the CUDA-core MLA kernel."""
    rng = np.random.default_rng(20 + heads)
    rows, n_kv, cap = 3, 2000, 600
    vals = torch.from_numpy(rng.standard_normal((n_kv, 576)).astype(np.float32))
    rows8 = inputs.fp8ds_encode(vals).numpy()
    q = inputs.randn_bf16((rows, heads, 576), 21, device="cuda")
    kv_rows = np.full((rows, 1, cap), -1, np.int32)
    count = np.zeros((rows, 1), np.int32)
    for r, n in enumerate((cap, 301, 0)):
        kv_rows[r, 0, :n] = rng.choice(n_kv, n, replace=False)
        count[r, 0] = n
    kv_rows[0, 0, [5, 77]] = -1
    assert decode_fp8_both(q, rows8, cuda(rows8), kv_rows, count, 1 / 24) == 0


@pytest.mark.parametrize("rows,heads,cap", [(152, 16, 384), (76, 128, 256), (40, 32, 1000)])
def test_decode_many_tiles_per_cta(rows, heads, cap):
    """Enough rows that each attention CTA walks several 128-row tiles of the
    reconstructed rows."""
    rng = np.random.default_rng(rows + heads)
    n_kv = 20000
    vals = torch.from_numpy(rng.standard_normal((n_kv, 576)).astype(np.float32))
    rows8 = inputs.fp8ds_encode(vals).numpy()
    q = inputs.randn_bf16((rows, heads, 576), 44, device="cuda")
    kv_rows = np.stack([rng.choice(n_kv, cap, replace=False) for _ in range(rows)])
    count = np.maximum(rng.integers(1, cap + 1, rows), cap - 5).astype(np.int32)
    assert decode_fp8_both(q, rows8, cuda(rows8), kv_rows[:, None].astype(np.int32),
                           count[:, None], 1 / 24, sample_rows=[0, 1, rows // 2, rows - 1]) == 0


def test_decode_tail_sizes_and_bad_ids():
    rng = np.random.default_rng(30)
    n_kv = 400
    vals = torch.from_numpy(rng.standard_normal((n_kv, 576)).astype(np.float32))
    rows8 = inputs.fp8ds_encode(vals).numpy()
    dev = cuda(rows8)
    for cap in (1, 17, 64, 129):
        q = inputs.randn_bf16((2, 16, 576), 31 + cap, device="cuda")
        kv_rows = np.stack([rng.choice(n_kv, cap, replace=False) for _ in range(2)])
        assert decode_fp8_both(q, rows8, dev, kv_rows[:, None].astype(np.int32), None,
                               1 / 24) == 0
    q = inputs.randn_bf16((1, 16, 576), 40, device="cuda")
    st = decode_fp8_both(q, rows8, dev, np.array([[[3, 400, 9, -1, 7]]], np.int32), None, 1 / 24)
    assert hs.status_string(st) == "HS_ERR_BAD_INDEX"


def test_mla_decode_fp8_config_sampled():
    """Full size (32 requests x 128 heads x 2048 rows from a 688 MB paged
    fp8_ds_mla cache), after S1; 3 sampled requests against the oracle."""
    cfg = inputs.mla_decode_fp8()
    R = cfg["num_reqs"]
    tok, slot, count, err = hs.normalize_indices(
        cuda(cfg["cand"]), torch.arange(R, dtype=torch.int32, device="cuda"),
        torch.full((R,), cfg["ctx"], dtype=torch.int32, device="cuda"),
        cuda(cfg["block_table"]), 64, num_pages=cfg["num_pages"])
    kv_rows = slot.cpu().numpy()[:, None, :]
    cnt = count.cpu().numpy()[:, None]
    sample = [0, 17, 31]
    # The oracle reads only the referenced rows: copy those to the host.
    ids = np.unique(kv_rows[sample][kv_rows[sample] >= 0])
    host = np.zeros((cfg["cache8"].shape[0], RB), np.uint8)
    host[ids] = u8(cfg["cache8"][torch.from_numpy(ids).cuda().long()])
    assert decode_fp8_both(cfg["q"], host, cfg["cache8"], kv_rows, cnt, cfg["scale"],
                           sample_rows=sample) == 0


def test_swap_in_and_backup_of_656_byte_rows():
    """The hot buffer moves fp8_ds_mla rows as opaque 656-byte rows."""
    rng = np.random.default_rng(50)
    pool_rows, R, M = 5000, 4, 300
    pool = torch.from_numpy(random_fp8_rows(rng, pool_rows, nan_free=False)).pin_memory()
    region = M + 1
    hot = torch.zeros(R * region, RB, dtype=torch.uint8, device="cuda")
    src = np.stack([rng.choice(pool_rows, M, replace=False) for _ in range(R)]).astype(np.int32)
    dst = (np.arange(R)[:, None] * region + rng.permuted(np.tile(np.arange(M), (R, 1)),
                                                         axis=1)).astype(np.int64)
    cnt = np.array([M, 0, 151, 1], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs.swap_in(hs.host_device_pointer(pool), pool_rows, hot, RB, cuda(src), cuda(dst),
               cuda(cnt), status=status)
    torch.cuda.synchronize()
    exp = np.zeros((R * region, RB), np.uint8)
    for r in range(R):
        for m in range(cnt[r]):
            exp[dst[r, m]] = pool.numpy()[src[r, m]]
    np.testing.assert_array_equal(u8(hot), exp)
    assert status.item() == 0
    # BackUp: one hot row per request to a host slot.
    brows = np.array([0, region + 5, 2 * region + 7, 3 * region], np.int64)
    bdst = rng.choice(pool_rows, R, replace=False).astype(np.int32)
    before = pool.numpy().copy()
    hs.backup(hot, cuda(brows), hs.host_device_pointer(pool), cuda(bdst), RB, pool_rows,
              status=status)
    torch.cuda.synchronize()
    before[bdst] = exp[brows]
    np.testing.assert_array_equal(pool.numpy(), before)


@pytest.mark.parametrize("max_ctas,claim", [(0, False), (4, True), (24, True)])
def test_swap_in_fp8ds_matches_oracle(max_ctas, claim):
    """Reconstructing SwapIn from a pinned fp8_ds_mla pool into bf16 hot rows:
    whole hot buffer and dgi byte for byte against the oracle, with contiguous
    runs (one bulk load each), scattered rows, a source outside the pool
    (zeroed, slot revoked) and a ragged count, on every SM or a budget, with
    groups dealt round-robin or claimed by ticket."""
    rng = np.random.default_rng(60 + max_ctas)
    pool_rows, R, M, hot_size = 4000, 5, 257, 300
    region = hot_size + 1
    pool = torch.from_numpy(random_fp8_rows(rng, pool_rows)).pin_memory()
    src = np.stack([np.sort(rng.choice(pool_rows, M, replace=False)) for _ in range(R)])
    src[0] = np.arange(1000, 1000 + M)
    src = src.astype(np.int32)
    src[2, 17] = pool_rows + 5
    dst = np.stack([r * region + rng.permutation(hot_size)[:M] for r in range(R)]).astype(
        np.int64)
    cnt = np.array([M, 0, 200, 1, 131], np.int32)
    dgi0 = rng.integers(0, 1 << 20, (R, hot_size)).astype(np.int32)
    hot_np = rng.integers(0, 1 << 16, (R * region, 576), dtype=np.uint16)
    hot = torch.from_numpy(hot_np.view(np.int16).copy()).view(torch.bfloat16).cuda()
    dgi = cuda(dgi0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ticket = torch.zeros(2, dtype=torch.int32, device="cuda") if claim else None
    hs.swap_in_fp8ds(hs.host_device_pointer(pool), pool_rows, RB, hot, cuda(src), cuda(dst),
                     cuda(cnt), dgi=dgi, hot_size=hot_size, region_stride=region,
                     max_ctas=max_ctas, ticket=ticket, status=status)
    torch.cuda.synchronize()
    exp = hot_np.copy()
    dgi_exp = dgi0.copy()
    oracle.swap_in_fp8ds(pool.numpy(), exp, src, dst, cnt, dgi=dgi_exp, hot_size=hot_size,
                         region_stride=region)
    np.testing.assert_array_equal(bits(hot), exp)
    np.testing.assert_array_equal(np_i32(dgi), dgi_exp)
    assert status.item() == 0
    if ticket is not None:
        assert (np_i32(ticket) == 0).all()
