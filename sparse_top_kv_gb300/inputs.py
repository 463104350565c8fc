"""Seeded synthetic inputs shaped like the pages' workloads.

This module only DRAWS inputs (token positions, page tables, KV rows, query
vectors); it computes nothing of the method itself (no slot mapping, no
lookup, no attention).  The CUDA path and the oracle both consume what it
returns.  Every function is deterministic in its seed.

Workloads (names used by the tests and the bench):
  tiny_hisparse   1 request, 16 heads, MLA rows (576 bf16 = 1152 B), page 64,
                  1024 positions (1020 prefilled), 4 decode steps, top_k 64,
                  hot region 2*64+1 = 129 rows; step 0 uniform, later steps keep
                  round(0.7*64) = 45 of the previous set and draw 19 fresh.
  swapin          pinned pool 1,048,576 x 1152 B random bytes; 64 requests x
                  4096 misses into 64 x 4097 hot rows; requests 0-31 pull 64
                  distinct random 64-row pages (contiguous runs), requests
                  32-63 pull 4096 distinct uniform slot ids; BackUp of one row
                  per request to random host slots.
  mla_decode      32 requests x 128 heads, q [32,128,576], paged HBM cache of
                  16384 pages x 64 x 576 bf16, random page table (512 pages per
                  request), context 32768, 2048 unique uniform positions.
  full_hisparse   64 requests, 16 heads, MLA rows, page 64, context 131072
                  (all but the decoded positions prefilled in a pinned pool of
                  64 x 2048 pages), top_k 2048, hot 4096+1 rows per request;
                  step 0 uniform, later steps keep round(0.85*2048) = 1741 and
                  draw the rest Zipf(s=1.1) over recency rank r = T-1-t.
  mla_decode_fp8  mla_decode with the paged cache stored as fp8_ds_mla rows of
                  656 B (the same N(0,1) values, encoded by fp8ds_encode).
  gqa_union       16 requests, 32 query / 8 KV heads, d = 128, bshd caches of
                  65536 pages x 16 x 8 x 128 for K and V, random page table,
                  context 65536; one index row per (request, KV head): 922
                  distinct uniform positions (about 5 % inside the 256-token
                  window, 2 inside the 4 sinks) plus 102 repeats of them; W=256,
                  A=4.
"""
import math

import numpy as np
import torch

SEEDS = {"tiny_hisparse": 0, "swapin": 1, "mla_decode": 2, "full_hisparse": 3, "gqa_union": 4,
         "hicache": 5}


def _rng(seed):
    return np.random.default_rng(seed)


def randn_bf16(shape, seed, device="cpu"):
    """N(0, 1) values rounded to bf16 (torch's generator, seeded)."""
    g = torch.Generator(device=device).manual_seed(seed)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def pinned_empty(shape, dtype):
    """Pinned host tensor whose pages are first touched by the CPU."""
    out = torch.empty(*shape, dtype=dtype, pin_memory=True)
    flat = out.view(-1).view(torch.uint8)
    flat[::4096].zero_()
    return out


def host_read_pass(t):
    """Read every 64-byte line of a host tensor on the CPU.

    Measured on GB300 (Grace host, NVLink-C2C): host lines last written by
    the GPU (D2H copies) are read back by GPU kernels 10-40x slower than
    lines the CPU has read since (first GPU read of a row 2-6 ms for 19K
    rows instead of 0.15 ms).  A pool that the GPU filled is passed over
    once by the CPU before use."""
    flat = t.view(-1).view(torch.uint8)
    n = flat.numel() // 64 * 64
    return int(flat[:n].view(-1, 64)[:, 0].sum())


def fill_randn_bf16_pinned(rows, width, seed, chunk_rows=1 << 20):
    """A pinned host tensor [rows, width] bf16 of N(0,1) values, generated on the
    GPU in chunks (seeded) and copied down; used for the multi-GB host pools."""
    out = pinned_empty((rows, width), torch.bfloat16)
    g = torch.Generator(device="cuda").manual_seed(seed)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        blk = torch.randn(r1 - r0, width, generator=g, device="cuda").to(torch.bfloat16)
        out[r0:r1].copy_(blk)
    torch.cuda.synchronize()
    host_read_pass(out)
    return out


def fill_randn_fp8ds_pinned(rows, seed, chunk_rows=1 << 19):
    """A pinned host tensor [rows, 656] uint8 of fp8_ds_mla rows encoding N(0,1)
    values (fp8ds_encode), generated on the GPU in chunks and copied down."""
    out = pinned_empty((rows, FP8DS_ROW_BYTES), torch.uint8)
    g = torch.Generator(device="cuda").manual_seed(seed)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1].copy_(fp8ds_encode(torch.randn(r1 - r0, 576, generator=g, device="cuda")))
    torch.cuda.synchronize()
    host_read_pass(out)
    return out


def page_table(num_reqs, pages_per_req, num_pages, seed):
    """Random physical pages: a permutation of the pool, dealt out to requests."""
    perm = _rng(seed).permutation(num_pages)[: num_reqs * pages_per_req]
    return perm.reshape(num_reqs, pages_per_req).astype(np.int32)


# ----------------------------------------------------------------------------
# HiSparse decode-step index streams (configs tiny_hisparse, full_hisparse).

def hisparse_index_steps(num_reqs, top_k, prefill, steps, keep, seed, zipf_s=None):
    """Per step s (context T_s = prefill + s + 1, the newest position is T_s - 1):
    int32 [steps, num_reqs, top_k] candidate positions.  Step 0 draws top_k
    distinct uniform positions; later steps keep `keep` of the previous set
    (uniformly chosen) and draw the rest fresh, uniform or Zipf(zipf_s) over the
    recency rank r = T_s - 1 - t, rejecting repeats."""
    rng = _rng(seed)
    out = np.empty((steps, num_reqs, top_k), np.int32)
    prev = [None] * num_reqs
    cdf = None
    for s in range(steps):
        T = prefill + s + 1
        if zipf_s is not None:
            w = (np.arange(T, dtype=np.float64) + 1.0) ** (-zipf_s)
            cdf = np.cumsum(w)
            cdf /= cdf[-1]
        for r in range(num_reqs):
            if s == 0:
                cur = rng.choice(T, size=top_k, replace=False)
            else:
                kept = rng.choice(prev[r], size=keep, replace=False)
                chosen = set(kept.tolist())
                fresh = []
                while len(chosen) < top_k:
                    need = top_k - len(chosen)
                    if zipf_s is None:
                        cand = rng.integers(0, T, size=2 * need + 8)
                    else:
                        rank = np.searchsorted(cdf, rng.random(2 * need + 8), side="right")
                        cand = T - 1 - np.minimum(rank, T - 1)
                    for t in cand.tolist():
                        if t not in chosen:
                            chosen.add(t)
                            fresh.append(t)
                            if len(chosen) == top_k:
                                break
                cur = np.concatenate([kept, np.array(fresh, dtype=np.int64)])
                rng.shuffle(cur)
            out[s, r] = cur
            prev[r] = cur
    return out


def tiny_hisparse(row_format="bf16"):
    """Config tiny_hisparse; row_format "fp8ds": the pool and the new rows as
    fp8_ds_mla rows (the same values, encoded)."""
    seed = SEEDS["tiny_hisparse"]
    cfg = dict(name="tiny_hisparse", num_reqs=1, heads=16, d_qk=576, d_v=512, page_size=64,
               total_positions=1024, steps=4, top_k=64, hot_size=128, region_stride=129,
               scale=1.0 / math.sqrt(576.0), seed=seed)
    cfg["prefill"] = cfg["total_positions"] - cfg["steps"]
    pages = cfg["total_positions"] // cfg["page_size"]
    cfg["num_pages"] = pages
    cfg["block_table"] = page_table(1, pages, pages, seed)
    cfg["pool"] = randn_bf16((pages * cfg["page_size"], 576), seed + 100)
    cfg["cand"] = hisparse_index_steps(1, 64, cfg["prefill"], cfg["steps"], keep=round(0.7 * 64),
                                       seed=seed)
    cfg["q"] = randn_bf16((cfg["steps"], 1, 16, 576), seed + 200)
    cfg["new_rows"] = randn_bf16((cfg["steps"], 1, 576), seed + 300)
    cfg["newest_pos"] = np.array([[cfg["prefill"] + s] for s in range(cfg["steps"])], np.int32)
    cfg["row_format"] = row_format
    if row_format == "fp8ds":
        cfg["pool"] = fp8ds_encode(cfg["pool"].float())
        cfg["new_rows"] = fp8ds_encode(cfg["new_rows"].float().reshape(-1, 576)).reshape(
            cfg["steps"], 1, FP8DS_ROW_BYTES)
    return cfg


def full_hisparse(steps=16, num_reqs=64, top_k=2048, heads=16, pool_on_gpu_seed=True,
                  row_format="bf16"):
    """Config full_hisparse.  The 9.66 GB pool is generated on the GPU and copied
    into pinned host memory (requires CUDA).  row_format "fp8ds": the pool
    (5.5 GB) and the new rows as fp8_ds_mla rows of N(0,1) values."""
    seed = SEEDS["full_hisparse"]
    B = 64
    total = 131072
    pages_per_req = total // B
    num_pages = num_reqs * pages_per_req
    cfg = dict(name="full_hisparse", num_reqs=num_reqs, heads=heads, d_qk=576, d_v=512,
               page_size=B, total_positions=total, steps=steps, top_k=top_k,
               hot_size=2 * top_k, region_stride=2 * top_k + 1,
               scale=1.0 / math.sqrt(576.0), seed=seed, num_pages=num_pages)
    cfg["prefill"] = total - steps
    cfg["block_table"] = page_table(num_reqs, pages_per_req, num_pages, seed)
    if row_format == "fp8ds":
        cfg["pool"] = fill_randn_fp8ds_pinned(num_pages * B, seed + 100)
    else:
        cfg["pool"] = fill_randn_bf16_pinned(num_pages * B, 576, seed + 100)
    cfg["row_format"] = row_format
    cfg["cand"] = hisparse_index_steps(num_reqs, top_k, cfg["prefill"], steps,
                                       keep=round(0.85 * top_k), seed=seed, zipf_s=1.1)
    g = torch.Generator(device="cpu").manual_seed(seed + 200)
    cfg["q"] = torch.randn(steps, num_reqs, heads, 576, generator=g).to(torch.bfloat16)
    cfg["new_rows"] = torch.randn(steps, num_reqs, 576, generator=g).to(torch.bfloat16)
    if row_format == "fp8ds":
        cfg["new_rows"] = fp8ds_encode(cfg["new_rows"].float().reshape(-1, 576)).reshape(
            steps, num_reqs, FP8DS_ROW_BYTES)
    cfg["newest_pos"] = np.array([[cfg["prefill"] + s] * num_reqs for s in range(steps)],
                                 np.int32)
    return cfg


def multi_layer_hisparse(layers=4, num_reqs=64, total=32768, top_k=2048, steps=16, heads=16,
                         page_size=64, keep_frac=0.85, zipf_s=1.1, seed=None):
    """Several HiSparse layers that share each step's index stream (one top-k
    row per request and step, drawn as in full_hisparse: step 0 uniform, then
    round(keep_frac * top_k) kept and the rest Zipf(zipf_s) over recency).
    Layer l has its own pool of N(0, 1) bf16 rows (pinned; drawn on the GPU
    when it is large), its own queries and its own new rows, all seeded from
    seed + 1000 l.  Returns the shared fields plus per-layer lists
    pools, q and new_rows."""
    seed = SEEDS["full_hisparse"] + 10 if seed is None else seed
    pages_per_req = total // page_size
    num_pages = num_reqs * pages_per_req
    cfg = dict(name="multi_layer_hisparse", layers=layers, num_reqs=num_reqs, heads=heads,
               d_qk=576, d_v=512, page_size=page_size, total_positions=total, steps=steps,
               top_k=top_k, hot_size=2 * top_k, region_stride=2 * top_k + 1,
               scale=1.0 / math.sqrt(576.0), seed=seed, num_pages=num_pages)
    cfg["prefill"] = total - steps
    cfg["block_table"] = page_table(num_reqs, pages_per_req, num_pages, seed)
    cfg["cand"] = hisparse_index_steps(num_reqs, top_k, cfg["prefill"], steps,
                                       keep=round(keep_frac * top_k), seed=seed, zipf_s=zipf_s)
    cfg["newest_pos"] = np.array([[cfg["prefill"] + s] * num_reqs for s in range(steps)],
                                 np.int32)
    rows = num_pages * page_size
    pools, qs, news = [], [], []
    for l in range(layers):
        ls = seed + 1000 * l
        if rows * 576 * 2 > (256 << 20):
            pools.append(fill_randn_bf16_pinned(rows, 576, ls + 100))
        else:
            pools.append(randn_bf16((rows, 576), ls + 100).pin_memory())
        g = torch.Generator(device="cpu").manual_seed(ls + 200)
        qs.append(torch.randn(steps, num_reqs, heads, 576, generator=g).to(torch.bfloat16))
        news.append(torch.randn(steps, num_reqs, 576, generator=g).to(torch.bfloat16))
    cfg["pools"], cfg["q"], cfg["new_rows"] = pools, qs, news
    return cfg


# ----------------------------------------------------------------------------

def swapin(num_reqs=64, misses=4096, pool_rows=1 << 20, row_bytes=1152, seed=None):
    """Config swapin.  Returns the host pool (pinned uint8), the per-request
    miss source ids (sorted), and BackUp destinations."""
    seed = SEEDS["swapin"] if seed is None else seed
    rng = _rng(seed)
    pool = pinned_empty((pool_rows, row_bytes), torch.uint8)
    g = torch.Generator(device="cuda").manual_seed(seed)
    chunk = 1 << 18
    for r0 in range(0, pool_rows, chunk):
        r1 = min(pool_rows, r0 + chunk)
        pool[r0:r1].copy_(torch.randint(0, 256, (r1 - r0, row_bytes), generator=g,
                                        device="cuda", dtype=torch.uint8))
    torch.cuda.synchronize()
    host_read_pass(pool)
    src = np.empty((num_reqs, misses), np.int32)
    half = num_reqs // 2
    run = 64
    for r in range(num_reqs):
        if r < half:
            pages = np.sort(rng.choice(pool_rows // run, size=misses // run, replace=False))
            src[r] = (pages[:, None] * run + np.arange(run)[None, :]).reshape(-1)
        else:
            src[r] = np.sort(rng.choice(pool_rows, size=misses, replace=False))
    backup_dst = rng.choice(pool_rows, size=num_reqs, replace=False).astype(np.int32)
    return dict(name="swapin", pool=pool, src=src, num_reqs=num_reqs, misses=misses,
                row_bytes=row_bytes, hot_rows_per_req=misses + 1, backup_dst=backup_dst)


def mla_decode(num_reqs=32, heads=128, top_k=2048, num_pages=16384, ctx=32768, device="cuda",
               with_data=True):
    """Config mla_decode: device-resident paged cache [num_pages, 64, 576]
    (with_data=False: indices and page table only)."""
    seed = SEEDS["mla_decode"]
    B = 64
    rng = _rng(seed)
    ppr = ctx // B
    cfg = dict(name="mla_decode", num_reqs=num_reqs, heads=heads, d_qk=576, d_v=512,
               page_size=B, ctx=ctx, top_k=top_k, num_pages=num_pages,
               scale=1.0 / math.sqrt(576.0))
    cfg["block_table"] = page_table(num_reqs, ppr, num_pages, seed)
    if with_data:
        cfg["cache"] = randn_bf16((num_pages * B, 576), seed + 100, device=device)
        cfg["q"] = randn_bf16((num_reqs, heads, 576), seed + 200, device=device)
    cfg["cand"] = np.stack([rng.choice(ctx, size=top_k, replace=False)
                            for _ in range(num_reqs)]).astype(np.int32)
    return cfg


FP8DS_ROW_BYTES = 656


def fp8ds_encode(values):
    """Encode float rows [n, 576] as fp8_ds_mla rows, uint8 [n, 656]: columns
    0..511 as E4M3 codes of value / scale (torch's float8_e4m3fn conversion),
    with one fp32 scale per 128 columns = the group's largest magnitude / 448
    (1 for an all-zero group) at bytes 512..527, and columns 512..575 as bf16
    at bytes 528..655.  Input synthesis only: reading the rows back (the
    dequantization the attention performs) is not done here."""
    v = values.to(torch.float32)
    n = v.shape[0]
    lat = v[:, :512].reshape(n, 4, 128)
    amax = lat.abs().amax(dim=2)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (lat / scale[:, :, None]).reshape(n, 512).to(torch.float8_e4m3fn)
    out = torch.empty(n, FP8DS_ROW_BYTES, dtype=torch.uint8, device=v.device)
    out[:, :512] = codes.view(torch.uint8)
    out[:, 512:528] = scale.contiguous().view(torch.uint8).reshape(n, 16)
    out[:, 528:] = v[:, 512:].to(torch.bfloat16).contiguous().view(torch.uint8).reshape(n, 128)
    return out


def mla_decode_fp8(device="cuda", with_data=True, **kw):
    """Config mla_decode_fp8: mla_decode's indices, page table and query, with
    the paged cache [num_pages * 64, 656] in fp8_ds_mla rows (encoded in
    chunks on `device`)."""
    cfg = mla_decode(device=device, with_data=False, **kw)
    cfg["name"] = "mla_decode_fp8"
    seed = SEEDS["mla_decode"]
    if with_data:
        n = cfg["num_pages"] * cfg["page_size"]
        cache = torch.empty(n, FP8DS_ROW_BYTES, dtype=torch.uint8, device=device)
        g = torch.Generator(device=device).manual_seed(seed + 100)
        step = 1 << 17
        for r0 in range(0, n, step):
            r1 = min(n, r0 + step)
            vals = torch.randn(r1 - r0, 576, generator=g, device=device, dtype=torch.float32)
            cache[r0:r1] = fp8ds_encode(vals)
        cfg["cache8"] = cache
        cfg["q"] = randn_bf16((cfg["num_reqs"], cfg["heads"], 576), seed + 200, device=device)
    return cfg


def gqa_union(num_reqs=16, heads=32, kv_heads=8, d=128, ctx=65536, page=16, n_unique=922,
              n_dup=102, window=256, sinks=4, device="cuda", with_data=True):
    """Config gqa_union: bshd K/V caches [num_pages, page, kv_heads, d]
    (with_data=False: indices and page table only)."""
    seed = SEEDS["gqa_union"]
    rng = _rng(seed)
    ppr = ctx // page
    num_pages = num_reqs * ppr
    cfg = dict(name="gqa_union", num_reqs=num_reqs, heads=heads, kv_heads=kv_heads, d=d,
               ctx=ctx, page_size=page, num_pages=num_pages, window=window, sinks=sinks,
               scale=1.0 / math.sqrt(d))
    cfg["block_table"] = page_table(num_reqs, ppr, num_pages, seed)
    if with_data:
        cfg["k_cache"] = randn_bf16((num_pages * page, kv_heads, d), seed + 100, device=device)
        cfg["v_cache"] = randn_bf16((num_pages * page, kv_heads, d), seed + 101, device=device)
        cfg["q"] = randn_bf16((num_reqs, heads, d), seed + 200, device=device)
    rows = num_reqs * kv_heads
    n_win = round(0.05 * n_unique)
    cand = np.empty((rows, n_unique + n_dup), np.int32)
    for i in range(rows):
        in_sink = rng.choice(sinks, size=2, replace=False)
        in_win = rng.choice(np.arange(ctx - window, ctx), size=n_win, replace=False)
        middle = rng.choice(np.arange(sinks, ctx - window), size=n_unique - 2 - n_win,
                            replace=False)
        uniq = np.concatenate([in_sink, in_win, middle])
        dup = rng.choice(uniq, size=n_dup, replace=True)
        row = np.concatenate([uniq, dup])
        rng.shuffle(row)
        cand[i] = row
    cfg["cand"] = cand
    cfg["row_req"] = np.repeat(np.arange(num_reqs, dtype=np.int32), kv_heads)
    return cfg


def hicache(nbuf=2, layers=4, page_size=128, row_bytes=512, host_tokens=65536, n=32768):
    """HiCache layer-transfer workload (K and V rows of 512 B = 4 KV heads x 64
    bf16, 128-token pages): a pinned host pool of random bytes holding nbuf
    pools of host_tokens * layers rows, and n // page_size whole random pages
    (sorted) as the token ids to move."""
    seed = SEEDS["hicache"]
    rng = _rng(seed)
    pool = pinned_empty((nbuf * layers * host_tokens * row_bytes,), torch.uint8)
    chunk = 1 << 24
    g = torch.Generator(device="cuda").manual_seed(seed)
    for o in range(0, pool.numel(), chunk):
        e = min(pool.numel(), o + chunk)
        pool[o:e].copy_(torch.randint(0, 256, (e - o,), generator=g, device="cuda",
                                      dtype=torch.uint8))
    torch.cuda.synchronize()
    host_read_pass(pool)
    pg = np.sort(rng.choice(host_tokens // page_size, size=n // page_size, replace=False))
    tokens = (pg[:, None] * page_size + np.arange(page_size)[None]).reshape(-1).astype(np.int64)
    return dict(name="hicache", pool=pool, tokens=tokens, nbuf=nbuf, layers=layers,
                page_size=page_size, row_bytes=row_bytes, host_tokens=host_tokens, n=n)
