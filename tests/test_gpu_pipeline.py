"""Whole-step parity: the GPU decode step (sparse_top_kv_gb300.pipeline) against
the oracle's step (oracle.pipeline), every stage compared after every step:
S1 outputs, S2 outputs and dgi/lru state, the whole hot buffer and the host
pool byte for byte, and attention within tolerance."""
import numpy as np
import pytest
import torch

from gpu_util import bits, check_attention, cuda, np_i32, u8
from oracle.pipeline import OracleHiSparse
from sparse_top_kv_gb300 import inputs
from sparse_top_kv_gb300.pipeline import HiSparseDecoder

pytestmark = pytest.mark.gpu


def run_steps(cfg, pool, attend_sample=None, steps=None):
    R = cfg["num_reqs"]
    B = cfg["page_size"]
    fmt = cfg.get("row_format", "bf16")
    rb = pool.shape[1] * pool.element_size()  # bytes of a pool row (and of a new row)
    dec = HiSparseDecoder(host_pool=pool, block_table=torch.from_numpy(cfg["block_table"]),
                          num_pages=cfg["num_pages"], page_size=B, top_k=cfg["top_k"],
                          hot_size=cfg["hot_size"], region_stride=cfg["region_stride"],
                          heads=cfg["heads"], scale=cfg["scale"], row_format=fmt)
    # The oracle reads the same pinned pool: both sides write identical
    # BackUp rows, and step s only reads positions < T_s, which no later
    # BackUp overwrites.
    ora = OracleHiSparse(host_pool_u8=pool.view(torch.uint8).numpy(),
                         block_table=cfg["block_table"], num_pages=cfg["num_pages"],
                         page_size=B, top_k=cfg["top_k"], hot_size=cfg["hot_size"],
                         region_stride=cfg["region_stride"], row_bytes=rb, scale=cfg["scale"],
                         row_format=fmt)
    hit_rates = []
    nsteps = cfg["steps"] if steps is None else steps
    for s in range(nsteps):
        T = cfg["prefill"] + s + 1
        seq = np.full(R, T, np.int32)
        newest_pos = np.full(R, cfg["prefill"] + s, np.int32)
        g_newest = dec.newest_slots(cuda(newest_pos), cuda(seq))
        o_newest = ora.newest_slots(newest_pos, seq)
        np.testing.assert_array_equal(np_i32(g_newest), o_newest)
        q = cfg["q"][s]
        new_row = cfg["new_rows"][s]
        stats0 = ora.stats.copy()
        out, lse = dec.step(cuda(cfg["cand"][s]), cuda(seq), g_newest, new_row.cuda(), q.cuda())
        torch.cuda.synchronize()
        ref = ora.step(cfg["cand"][s], seq, o_newest, u8(new_row).reshape(R, rb), bits(q),
                       attend_rows=attend_sample)
        tok, slot, count, err = dec.s1_out
        for name, g in (("tok", tok), ("slot", slot), ("count", count), ("err", err)):
            np.testing.assert_array_equal(np_i32(g), ref[name], err_msg=f"step {s} {name}")
        hot_idx, mm, msrc, mdst, mcount, lerr, hit_idx, miss_rows = dec.s2_out
        # The split lists: resident rows keep their hot row, the swapped ones
        # are listed compactly.
        exp_hit = np.where(ref["miss_mask"] == 0, ref["hot_idx"], -1)
        np.testing.assert_array_equal(np_i32(hit_idx), exp_hit, err_msg=f"step {s} hit_idx")
        for r in range(R):
            m = int(ref["miss_count"][r])
            np.testing.assert_array_equal(np_i32(miss_rows)[r, :m], ref["miss_dst"][r, :m])
            assert (np_i32(miss_rows)[r, m:] == -1).all()
        for name, g in (("hot_idx", hot_idx), ("miss_mask", mm), ("miss_count", mcount),
                        ("lookup_err", lerr)):
            np.testing.assert_array_equal(np_i32(g), ref[name], err_msg=f"step {s} {name}")
        for r in range(R):
            m = int(ref["miss_count"][r])
            np.testing.assert_array_equal(np_i32(msrc)[r, :m], ref["miss_src"][r, :m])
            np.testing.assert_array_equal(np_i32(mdst)[r, :m], ref["miss_dst"][r, :m])
        np.testing.assert_array_equal(np_i32(dec.dgi), ora.dgi, err_msg=f"step {s} dgi")
        np.testing.assert_array_equal(np_i32(dec.lru), ora.lru, err_msg=f"step {s} lru")
        np.testing.assert_array_equal(np_i32(dec.stats), ora.stats, err_msg=f"step {s} stats")
        np.testing.assert_array_equal(u8(dec.hot), ora.hot, err_msg=f"step {s} hot bytes")
        assert dec.status.item() == 0
        rows = torch.from_numpy(ref["rows"]).cuda()
        check_attention(out[rows], lse[rows], ref["out"], ref["lse"], label=f"step {s}")
        d = ora.stats - stats0
        hit_rates.append(d[0] / max(1, d[0] + d[1]))
    return hit_rates


def test_tiny_hisparse_all_steps():
    cfg = inputs.tiny_hisparse()
    pool = cfg["pool"].pin_memory()
    run_steps(cfg, pool)


def test_tiny_hisparse_fp8_all_steps():
    """fp8_ds_mla pool and new rows: the hot buffer holds their bf16
    reconstruction, compared byte for byte with the oracle's every step."""
    cfg = inputs.tiny_hisparse("fp8ds")
    pool = cfg["pool"].pin_memory()
    run_steps(cfg, pool)


def test_full_hisparse_fp8_steps_sampled_attention():
    """The full-size step with the 5.5 GB fp8_ds_mla pool: six steps, S1-S3,
    the reconstructed hot buffer, the pool and the state compared in full,
    S4 on two sampled requests per step."""
    cfg = inputs.full_hisparse(row_format="fp8ds")
    rates = run_steps(cfg, cfg["pool"], attend_sample=[0, 63], steps=6)
    assert rates[0] == 0.0 and min(rates[1:]) > 0.5


def test_full_hisparse_all_steps_sampled_attention():
    """64 requests, context 131072, top_k 2048, hot 4097 rows, the pinned
    9.66 GB pool; S1-S3 and the state compared in full at every step, S4 on
    two sampled requests per step."""
    cfg = inputs.full_hisparse()
    rates = run_steps(cfg, cfg["pool"], attend_sample=[0, 63])
    assert rates[0] == 0.0 and min(rates[1:]) > 0.5


@pytest.mark.parametrize("row_format", ["bf16", "fp8ds"])
def test_captured_step_matches_eager(row_format):
    """The captured step, replayed with a staged copy of the inputs
    (replay_packed), as one graph per input slot read in place
    (capture(slot=...)) and as one graph per pinned host input buffer with
    the results copied back to pinned host tensors (host_in / host_out),
    gives the eager step's outputs and state bit for bit at every step (the
    decoders write identical BackUp rows into the shared pool)."""
    cfg = inputs.tiny_hisparse(row_format)
    pool = cfg["pool"].pin_memory()
    R = cfg["num_reqs"]

    def make():
        return HiSparseDecoder(host_pool=pool, block_table=torch.from_numpy(cfg["block_table"]),
                               num_pages=cfg["num_pages"], page_size=cfg["page_size"],
                               top_k=cfg["top_k"], hot_size=cfg["hot_size"],
                               region_stride=cfg["region_stride"], heads=cfg["heads"],
                               scale=cfg["scale"], row_format=row_format)

    decs = [make(), make(), make(), make()]
    steps = []
    for s in range(cfg["steps"]):
        T = cfg["prefill"] + s + 1
        seq = cuda(np.full(R, T, np.int32))
        newest = decs[0].newest_slots(cuda(np.full(R, cfg["prefill"] + s, np.int32)), seq)
        steps.append((cuda(cfg["cand"][s]), seq, newest, cfg["new_rows"][s].cuda(),
                      cfg["q"][s].cuda()))
    packed = [decs[0].pack_inputs(*st) for st in steps]
    for d in decs:  # step 0 eagerly: the one-time set-up
        d.step(*steps[0])
    torch.cuda.synchronize()
    decs[1].capture()
    slot_graphs = [None] + [decs[2].capture(slot=packed[s]) for s in range(1, cfg["steps"])]
    # Inputs from pinned host buffers and results into pinned host tensors,
    # both copied by the graph.
    host_in = [p.cpu().pin_memory() for p in packed]
    out_h = torch.empty(decs[3].out.shape, dtype=decs[3].out.dtype).pin_memory()
    lse_h = torch.empty(decs[3].lse.shape, dtype=decs[3].lse.dtype).pin_memory()
    dev_slot = torch.empty_like(packed[0])
    host_graphs = [None] + [decs[3].capture(slot=dev_slot, host_in=host_in[s],
                                            host_out=(out_h, lse_h))
                            for s in range(1, cfg["steps"])]
    torch.cuda.synchronize()
    for s in range(1, cfg["steps"]):
        out0, lse0 = decs[0].step(*steps[s])
        out1, lse1 = decs[1].replay_packed(packed[s])
        out1, lse1 = out1.clone(), lse1.clone()
        slot_graphs[s].replay()
        host_graphs[s].replay()
        torch.cuda.synchronize()
        out2, lse2 = decs[2].out, decs[2].lse
        for o, l in ((out1, lse1), (out2, lse2), (out_h.cuda(), lse_h.cuda())):
            assert torch.equal(o.view(torch.int16), out0.view(torch.int16)), f"step {s} out"
            assert torch.equal(l, lse0), f"step {s} lse"
        for d in decs[1:]:
            for name in ("dgi", "lru", "stats", "hot"):
                assert torch.equal(getattr(d, name), getattr(decs[0], name)), f"step {s} {name}"
            assert d.status.item() == 0


def test_inactive_requests_in_a_captured_step():
    """Graph-stable stepping with a changing set of active requests: one
    captured step serves every step of a fixed-size batch; an inactive
    request's row is padding (no candidates, context length 0, newest slot
    -1).  Every step is compared with the oracle's step on the same inputs;
    an inactive request gets a zero output and LSE -inf and keeps its dgi and
    lru."""
    cfg = inputs.full_hisparse(steps=6, num_reqs=4, top_k=256)
    pool = cfg["pool"]
    R, B, rb = cfg["num_reqs"], cfg["page_size"], 576 * 2
    dec = HiSparseDecoder(host_pool=pool, block_table=torch.from_numpy(cfg["block_table"]),
                          num_pages=cfg["num_pages"], page_size=B, top_k=cfg["top_k"],
                          hot_size=cfg["hot_size"], region_stride=cfg["region_stride"],
                          heads=cfg["heads"], scale=cfg["scale"])
    ora = OracleHiSparse(host_pool_u8=pool.view(torch.uint8).numpy(),
                         block_table=cfg["block_table"], num_pages=cfg["num_pages"],
                         page_size=B, top_k=cfg["top_k"], hot_size=cfg["hot_size"],
                         region_stride=cfg["region_stride"], row_bytes=rb, scale=cfg["scale"])
    active = [[1, 1, 1, 1], [1, 0, 1, 1], [0, 1, 1, 0], [1, 1, 0, 1], [1, 1, 1, 1], [0, 0, 1, 1]]
    for s in range(cfg["steps"]):
        act = np.array(active[s], bool)
        T = cfg["prefill"] + s + 1
        seq = np.where(act, T, 0).astype(np.int32)
        newest_pos = np.where(act, cfg["prefill"] + s, -1).astype(np.int32)
        cand = cfg["cand"][s].copy()
        cand[~act] = -1
        g_newest = dec.newest_slots(cuda(newest_pos), cuda(seq))
        o_newest = ora.newest_slots(newest_pos, seq)
        np.testing.assert_array_equal(np_i32(g_newest), o_newest)
        assert (o_newest[~act] == -1).all()
        q, new_row = cfg["q"][s], cfg["new_rows"][s]
        dgi0, lru0 = np_i32(dec.dgi).copy(), np_i32(dec.lru).copy()
        if s == 0:  # the eager first step performs the one-time set-up
            out, lse = dec.step(cuda(cand), cuda(seq), g_newest, new_row.cuda(), q.cuda())
            dec.capture()
        else:
            out, lse = dec.replay_packed(dec.pack_inputs(cuda(cand), cuda(seq), g_newest,
                                                         new_row.cuda(), q.cuda()))
        torch.cuda.synchronize()
        ref = ora.step(cand, seq, o_newest, u8(new_row).reshape(R, rb), bits(q))
        tok, slot, count, err = dec.s1_out
        for name, g in (("tok", tok), ("slot", slot), ("count", count), ("err", err)):
            np.testing.assert_array_equal(np_i32(g), ref[name], err_msg=f"step {s} {name}")
        hot_idx, mm, msrc, mdst, mcount = dec.s2_out[:5]
        for name, g in (("hot_idx", hot_idx), ("miss_mask", mm), ("miss_count", mcount)):
            np.testing.assert_array_equal(np_i32(g), ref[name], err_msg=f"step {s} {name}")
        np.testing.assert_array_equal(np_i32(dec.dgi), ora.dgi, err_msg=f"step {s} dgi")
        np.testing.assert_array_equal(np_i32(dec.lru), ora.lru, err_msg=f"step {s} lru")
        np.testing.assert_array_equal(u8(dec.hot), ora.hot, err_msg=f"step {s} hot bytes")
        assert dec.status.item() == 0 and ref["backup_bad"] == 0
        for r in np.flatnonzero(~act):
            np.testing.assert_array_equal(np_i32(dec.dgi)[r], dgi0[r])
            np.testing.assert_array_equal(np_i32(dec.lru)[r], lru0[r])
            assert int(np_i32(count)[r]) == 0
            assert not out[r].float().abs().sum().item()
            assert torch.isinf(lse[r]).all() and (lse[r] < 0).all()
        rows = torch.from_numpy(np.flatnonzero(act)).cuda()
        check_attention(out[rows], lse[rows], ref["out"][act], ref["lse"][act], label=f"step {s}")
