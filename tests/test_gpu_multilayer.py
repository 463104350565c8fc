"""Several layers sharing each step's index row, overlapped layer by layer
(pipeline.MultiLayerHiSparse): every layer's S2 outputs, state, hot buffer,
host pool and attention against that layer's own oracle step, at every step,
eagerly and through the captured graph."""
import numpy as np
import pytest
import torch

from gpu_util import bits, check_attention, cuda, np_i32, u8
from oracle.pipeline import OracleHiSparse
from sparse_top_kv_gb300 import inputs
from sparse_top_kv_gb300.pipeline import HiSparseDecoder, MultiLayerHiSparse

pytestmark = pytest.mark.gpu


def build(cfg):
    decs, oras = [], []
    for pool in cfg["pools"]:
        decs.append(HiSparseDecoder(host_pool=pool,
                                    block_table=torch.from_numpy(cfg["block_table"]),
                                    num_pages=cfg["num_pages"], page_size=cfg["page_size"],
                                    top_k=cfg["top_k"], hot_size=cfg["hot_size"],
                                    region_stride=cfg["region_stride"], heads=cfg["heads"],
                                    scale=cfg["scale"]))
        oras.append(OracleHiSparse(host_pool_u8=pool.view(torch.uint8).numpy(),
                                   block_table=cfg["block_table"], num_pages=cfg["num_pages"],
                                   page_size=cfg["page_size"], top_k=cfg["top_k"],
                                   hot_size=cfg["hot_size"], region_stride=cfg["region_stride"],
                                   row_bytes=1152, scale=cfg["scale"]))
    return MultiLayerHiSparse(decs), oras


def compare(ml, oras, cfg, s, outs, seq, o_newest, attend=None):
    R = cfg["num_reqs"]
    for l, (dec, ora) in enumerate(zip(ml.layers, oras)):
        ref = ora.step(cfg["cand"][s], seq, o_newest,
                       u8(cfg["new_rows"][l][s]).reshape(R, 1152), bits(cfg["q"][l][s]),
                       attend_rows=attend)
        hot_idx, mm, msrc, mdst, mcount, lerr = dec.s2_out[:6]
        for name, g in (("hot_idx", hot_idx), ("miss_mask", mm), ("miss_count", mcount),
                        ("lookup_err", lerr)):
            np.testing.assert_array_equal(np_i32(g), ref[name], err_msg=f"step {s} layer {l} {name}")
        np.testing.assert_array_equal(np_i32(dec.dgi), ora.dgi, err_msg=f"step {s} layer {l} dgi")
        np.testing.assert_array_equal(np_i32(dec.lru), ora.lru, err_msg=f"step {s} layer {l} lru")
        np.testing.assert_array_equal(u8(dec.hot), ora.hot, err_msg=f"step {s} layer {l} hot")
        assert dec.status.item() == 0
        out, lse = outs[l]
        rows = torch.from_numpy(ref["rows"]).cuda()
        check_attention(out[rows], lse[rows], ref["out"], ref["lse"], label=f"step {s} layer {l}")


@pytest.mark.parametrize("captured", [False, True])
def test_layers_share_the_index_row(captured):
    cfg = inputs.multi_layer_hisparse(layers=3, num_reqs=3, total=2048, top_k=96, steps=5,
                                      heads=16)
    R = cfg["num_reqs"]
    ml, oras = build(cfg)
    d0 = ml.layers[0]
    graph = None
    cand_d = torch.empty(R, cfg["top_k"], dtype=torch.int32, device="cuda")
    seq_d = torch.empty(R, dtype=torch.int32, device="cuda")
    newest_d = torch.empty(R, dtype=torch.int32, device="cuda")
    news_d = [torch.empty(R, 576, dtype=torch.bfloat16, device="cuda") for _ in ml.layers]
    qs_d = [torch.empty(R, cfg["heads"], 576, dtype=torch.bfloat16, device="cuda")
            for _ in ml.layers]
    for s in range(cfg["steps"]):
        T = cfg["prefill"] + s + 1
        seq = np.full(R, T, np.int32)
        newest_pos = np.full(R, T - 1, np.int32)
        g_newest = d0.newest_slots(cuda(newest_pos), cuda(seq))
        o_newest = oras[0].newest_slots(newest_pos, seq)
        cand_d.copy_(cuda(cfg["cand"][s]))
        seq_d.copy_(cuda(seq))
        newest_d.copy_(g_newest)
        for l in range(len(ml.layers)):
            news_d[l].copy_(cfg["new_rows"][l][s].cuda())
            qs_d[l].copy_(cfg["q"][l][s].cuda())
        if captured and s >= 1:
            if graph is None:
                graph = ml.capture(cand_d, seq_d, newest_d, news_d, qs_d)
            graph.replay()
            outs = [(d.out, d.lse) for d in ml.layers]
        else:
            outs = ml.step(cand_d, seq_d, newest_d, news_d, qs_d)
        torch.cuda.synchronize()
        compare(ml, oras, cfg, s, outs, seq, o_newest)
