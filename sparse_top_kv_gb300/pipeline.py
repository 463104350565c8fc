"""One HiSparse decode step on the GPU, through the C ABI of libhs.

Stage order per step (vLLM HiSparse walkthrough, "swap_in 方法流程详解" and the
BackUp interface of its overview):
  (model)  the new token's KV row lands in the request's reserved hot row
  S1 + S2  hs_normalize_lookup_assign  candidates -> sorted unique slots ->
           hot rows, misses, LRU update (one kernel)
  S3       hs_swap_in            missed rows host -> hot;  hs_backup  reserved row -> host
  S4       hs_sparse_decode      attention over the hot rows
Torch provides device memory, pinned host memory and the stream; every stage is
a libhs kernel.
"""
import torch

from . import hs


class HiSparseDecoder:
    """Per-layer hot buffer of `num_reqs` regions of `region_stride` rows of
    `row_width` bf16 elements, backed by a pinned host pool (the only
    full-size store, keyed by global slot id).

    row_format "fp8ds": the pool holds fp8_ds_mla rows (uint8 [rows, 656],
    vLLM HiSparse walkthrough's FP8_DS_MLA_ROW_BYTES), and so do the new rows
    a step receives; the hot buffer holds their bf16 reconstruction (576
    columns), written by the SwapIn's store step (hs_swap_in_fp8ds), so the
    host link carries 656 bytes per miss and the attention is unchanged."""

    def __init__(self, *, host_pool, block_table, num_pages, page_size, top_k, hot_size,
                 region_stride, heads, d_qk=576, d_v=512, scale, window=0, num_sinks=0,
                 device="cuda", row_format="bf16"):
        if not host_pool.is_pinned():
            raise ValueError("host pool must be pinned")
        if row_format not in ("bf16", "fp8ds"):
            raise ValueError("row_format: bf16 or fp8ds")
        self.fp8 = row_format == "fp8ds"
        if self.fp8 and (host_pool.dtype != torch.uint8 or host_pool.shape[1] < hs.FP8DS_ROW_BYTES
                         or d_qk != 576):
            raise ValueError("fp8ds: host pool uint8 [rows, >= 656], MLA rows (d_qk 576)")
        self.device = torch.device(device)
        self.num_reqs = block_table.shape[0]
        self.row_width = d_qk if self.fp8 else host_pool.shape[1]
        # Bytes of one pool row (what the host link and the BackUp move).
        self.row_bytes = host_pool.shape[1] * host_pool.element_size()
        self.host_pool = host_pool
        self.host_rows = host_pool.shape[0]
        self.host_dev = hs.host_device_pointer(host_pool)
        self.block_table = block_table.to(self.device, torch.int32).contiguous()
        self.num_pages, self.page_size = num_pages, page_size
        self.top_k, self.hot_size, self.region_stride = top_k, hot_size, region_stride
        self.heads, self.d_qk, self.d_v, self.scale = heads, d_qk, d_v, scale
        self.window, self.num_sinks = window, num_sinks
        R = self.num_reqs
        dev = self.device
        self.hot = torch.zeros(R * region_stride, self.row_width,
                               dtype=torch.bfloat16 if self.fp8 else host_pool.dtype, device=dev)
        self.dgi = torch.empty(R, hot_size, dtype=torch.int32, device=dev)
        self.lru = torch.empty(R, hot_size, dtype=torch.int16, device=dev)
        hs.hot_state_reset(self.dgi, self.lru)
        self.stats = torch.zeros(2, dtype=torch.int64, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.row_req = torch.arange(R, dtype=torch.int32, device=dev)
        self.reserved_rows = (torch.arange(R, dtype=torch.int64, device=dev) * region_stride
                              + hot_size)
        if self.fp8:
            # The new rows' reconstruction into the reserved rows: row r of
            # the step's new-row buffer -> reserved row r.
            self.new_src = torch.arange(R, dtype=torch.int32, device=dev).view(R, 1)
            self.new_dst = self.reserved_rows.view(R, 1).clone()
            self.new_cnt = torch.ones(R, dtype=torch.int32, device=dev)
            self.new_rows_idx = torch.arange(R, dtype=torch.int64, device=dev)
        cap = top_k + window + num_sinks
        self.cap = cap
        i32 = dict(dtype=torch.int32, device=dev)
        self.s1_out = (torch.empty(R, cap, **i32), torch.empty(R, cap, **i32),
                       torch.empty(R, **i32), torch.empty(R, 4, **i32))
        self.s2_out = (torch.empty(R, cap, **i32),
                       torch.empty(R, cap, dtype=torch.uint8, device=dev),
                       torch.empty(R, cap, **i32),
                       torch.empty(R, cap, dtype=torch.int64, device=dev),
                       torch.empty(R, **i32), torch.empty(R, **i32),
                       torch.empty(R, cap, **i32), torch.empty(R, cap, **i32))
        self.out = torch.empty(R, heads, d_v, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(R, heads, dtype=torch.float32, device=dev)
        ws = hs.sparse_decode_workspace_bytes(R, heads, 1, cap, d_qk, d_v)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        # Partial states of the two attention passes (resident rows, swapped rows).
        self.parts_hit = hs.sparse_decode_partial_splits(R, heads, 1, cap, d_qk, d_v)
        self.parts_miss = self.parts_hit
        P = self.parts_hit + self.parts_miss
        f32 = dict(dtype=torch.float32, device=dev)
        # Arrival counters of the finishing pass's last-CTA merge.
        self.sync = torch.zeros(R * heads, dtype=torch.int32, device=dev)
        self.ticket = torch.zeros(2, dtype=torch.int32, device=dev)  # SwapIn group claims
        self.part_m = torch.empty(R * heads, P, **f32)
        self.part_l = torch.empty(R * heads, P, **f32)
        self.part_o = torch.empty(R * heads, P, d_v, **f32)
        self.side = torch.cuda.Stream(device=dev)
        self.ev_lists = torch.cuda.Event()
        self.ev_attn = torch.cuda.Event()
        self.ev_fork = torch.cuda.Event()
        # SMs left to the SwapIn while the resident-row attention runs (one
        # attention CTA per SM, one copy CTA per SM).
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        hg = 64 if heads % 64 == 0 else (32 if heads % 32 == 0 else 16)
        attn_ctas = R * max(1, heads // hg) * max(1, self.parts_hit)
        self.swap_ctas = max(16, sms - attn_ctas)


    def warm_pool(self, page_bytes=4096):
        """One-time set-up pass: read one row of every `page_bytes` of the host
        pool (every 4 KB page by default) into the (still empty) hot buffer
        with hs_swap_in, in chunks of at most the hot buffer's rows.

        On GB300 virtual machines whose GPU reaches host memory through the
        IOMMU, the first GPU reads of a page of a freshly allocated pinned
        pool run far below the link rate (measured); a decoder whose
        pool had only one row per 64 KB read beforehand ran its first steps
        3x slower than a later decoder over the same pool.  A server pays that
        once at start-up; this pass pays it at set-up so that a decode step
        sees the steady state.  Must run before the first step (it overwrites
        hot rows, which are empty until then)."""
        stride = max(1, page_bytes // self.row_bytes)
        chunk = self.hot.shape[0]
        for r0 in range(0, self.host_rows, stride * chunk):
            src = torch.arange(r0, min(self.host_rows, r0 + stride * chunk), stride,
                               dtype=torch.int32, device=self.device)
            n = src.numel()
            src = src.view(1, n).contiguous()
            dst = torch.arange(n, dtype=torch.int64, device=self.device).view(1, n)
            cnt = torch.full((1,), n, dtype=torch.int32, device=self.device)
            if self.fp8:
                hs.swap_in_fp8ds(self.host_dev, self.host_rows, self.row_bytes, self.hot, src,
                                 dst, cnt, status=self.status)
            else:
                hs.swap_in(self.host_dev, self.host_rows, self.hot, self.row_bytes, src, dst,
                           cnt, status=self.status)
        self.hot.zero_()
        torch.cuda.synchronize(self.device)

    def newest_slots(self, newest_pos, seq_lens):
        """Slot mapping of the newest positions, int32 [R] (S1 on one candidate)."""
        tok, slot, count, err = hs.normalize_indices(
            newest_pos.view(-1, 1), self.row_req, seq_lens, self.block_table, self.page_size,
            num_pages=self.num_pages)
        return slot.view(-1).clone()

    def step(self, cand, seq_lens, newest_slot, new_row, q, stream=None, events=None,
             out=None, lse=None):
        """cand int32 [R, top_k] positions; seq_lens int32 [R]; newest_slot int32
        [R]; new_row [R, row_width] (the new token's KV row; uint8 [R, 656]
        fp8_ds_mla rows with row_format "fp8ds"); q bf16 [R, H, d_qk].
        Returns (out bf16 [R, H, d_v], lse fp32 [R, H]); state is updated.
        cand, seq_lens and newest_slot may be pinned host tensors (the kernels
        read them over the link); `out` / `lse`, if given (device or pinned
        host tensors of those shapes), receive the results instead of the
        decoder's own buffers.

        The SwapIn runs concurrently with the attention over the rows that
        were already resident (hit_idx, side stream); the attention over the
        swapped rows (miss_rows) follows the SwapIn, and the two sets of
        partial states are merged with eq. (7).  The new rows' write and
        their BackUp run on the side stream ahead of that attention.
        `events`, if given, is a list of 7 CUDA events recorded before S1 + S2
        (one kernel), after it (twice), before and after SwapIn, after the
        resident-row attention (side stream) and at the end of the step."""
        R = self.num_reqs
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        side = self.side
        rec = (lambda i, st: events[i].record(st)) if events is not None else (lambda i, st: None)
        rec(0, main)
        # S1 and S2 in one kernel (one CTA per request; S1's set stays in
        # shared memory for the lookup).
        (tok, slot, count, err), (hot_idx, miss_mask, miss_src, miss_dst, miss_count, lerr,
                                  hit_idx, miss_rows) = hs.normalize_lookup_assign(
            cand, self.row_req, seq_lens, self.block_table, self.page_size, newest_slot,
            self.dgi, self.lru, self.region_stride, self.stats, window=self.window,
            num_sinks=self.num_sinks, num_pages=self.num_pages, s1_out=self.s1_out,
            s2_out=self.s2_out, stream=main)
        rec(1, main)
        rec(2, main)
        self.ev_lists.record(main)
        # Main stream: the SwapIn of the misses right behind S2, then the
        # swapped rows' attention right behind the SwapIn; these three are
        # the step's critical path and each may start (set-up only) while its
        # predecessor runs (programmatic dependent launch).
        rec(3, main)
        if self.fp8:
            hs.swap_in_fp8ds(self.host_dev, self.host_rows, self.row_bytes, self.hot, miss_src,
                             miss_dst, miss_count, dgi=self.dgi, hot_size=self.hot_size,
                             region_stride=self.region_stride, max_ctas=self.swap_ctas,
                             ticket=self.ticket, status=self.status, stream=main)
        else:
            hs.swap_in(self.host_dev, self.host_rows, self.hot, self.row_bytes, miss_src,
                       miss_dst, miss_count, dgi=self.dgi, hot_size=self.hot_size,
                       region_stride=self.region_stride, max_ctas=self.swap_ctas,
                       ticket=self.ticket, status=self.status, stream=main)
        rec(4, main)
        # Side stream, once S2 has listed the misses (kernels beside S1 and
        # S2 slowed them by ~5 us in the captured step, measured): the
        # model's KV write of the newest token (stand-in: the reserved hot
        # rows; only the attention passes read them, and both follow this
        # stream), the BackUp of those rows to their host rows (this step's
        # SwapIn never reads them: S2 maps the newest token to its reserved
        # row, never to a miss), then the HBM traffic over the resident rows,
        # on the SMs the SwapIn leaves free.
        qv = self.q_view(q)
        nkv = self.hot.shape[0]
        side.wait_event(self.ev_lists)
        if self.fp8:
            # fp8 rows: the new rows are reconstructed into the reserved rows
            # and backed up in their 656-byte form.
            hs.swap_in_fp8ds(hs.device_address(new_row), self.num_reqs, self.row_bytes, self.hot,
                             self.new_src, self.new_dst, self.new_cnt, max_ctas=0,
                             status=self.status, stream=side)
        else:
            with torch.cuda.stream(side):
                self.hot.index_copy_(0, self.reserved_rows, new_row)
        if not torch.cuda.is_current_stream_capturing():
            new_row.record_stream(side)  # the caller's tensor is read on the side stream
        if self.fp8:
            hs.backup(new_row, self.new_rows_idx, self.host_dev, newest_slot, self.row_bytes,
                      self.host_rows, status=self.status, stream=side)
        else:
            hs.backup(self.hot, self.reserved_rows, self.host_dev, newest_slot, self.row_bytes,
                      self.host_rows, status=self.status, stream=side)
        hs.sparse_decode_partial(qv, self.hot, self.hot, self.row_width, 0, nkv,
                                 hit_idx.view(R, 1, self.cap), count.view(R, 1), self.scale,
                                 self.d_v, self.part_m, self.part_l, self.part_o, 0,
                                 status=self.status, stream=side)
        rec(5, side)
        self.ev_attn.record(side)
        main.wait_event(self.ev_attn)  # also joins the side stream: its last work
        # The swapped rows, merged with the resident-row states (eq. 7).
        hs.sparse_decode_finish(qv, self.hot, self.hot, self.row_width, 0, nkv,
                                miss_rows.view(R, 1, self.cap), miss_count.view(R, 1),
                                self.scale, self.d_v, self.part_m, self.part_l, self.part_o,
                                self.parts_hit, sync=self.sync,
                                out=self.out if out is None else out,
                                lse=self.lse if lse is None else lse,
                                status=self.status, stream=main)
        rec(6, main)
        return (self.out if out is None else out), (self.lse if lse is None else lse)

    def _input_layout(self):
        """Byte layout of one step's inputs packed in one buffer: (name,
        offset, shape, dtype) per input, 256-byte aligned."""
        R = self.num_reqs
        new_row = ((R, self.row_bytes), torch.uint8) if self.fp8 else ((R, self.row_width),
                                                                        self.hot.dtype)
        specs = [("cand", (R, self.top_k), torch.int32), ("seq", (R,), torch.int32),
                 ("newest", (R,), torch.int32), ("new_row",) + new_row,
                 ("q", (R, self.heads, self.d_qk), torch.bfloat16)]
        out, off = [], 0
        for name, shape, dt in specs:
            n = 1
            for x in shape:
                n *= x
            nbytes = n * torch.empty(0, dtype=dt).element_size()
            out.append((name, off, shape, dt, nbytes))
            off += (nbytes + 255) // 256 * 256
        return out, off

    def pack_inputs(self, cand, seq_lens, newest_slot, new_row, q, out=None):
        """One step's inputs in the packed layout of `replay_packed` (a uint8
        tensor on the same device as the given tensors)."""
        layout, total = self._input_layout()
        if out is None:
            out = torch.empty(total, dtype=torch.uint8, device=cand.device)
        for (name, off, shape, dt, nbytes), t in zip(layout, (cand, seq_lens, newest_slot,
                                                              new_row, q)):
            out[off:off + nbytes].view(dt).view(shape).copy_(t.reshape(shape))
        return out

    def capture(self, events=None, slot=None, host_in=None, host_out=None):
        """Capture one decode step over static input buffers (`self.graph_in`,
        views of the packed buffer `self.graph_in_packed`) as a CUDA graph,
        both streams included.  `replay(...)` / `replay_packed(...)` then copy
        a step's inputs into those buffers and run the step with one graph
        launch.  Run at least one eager step first (it performs the one-time
        library set-up that capture must not do).  `events`, if given, are
        timing events recorded inside the graph (see `step`).  Returns the
        graph (also kept as self.graph, the one replay uses).

        `slot`, if given, is a device buffer in the packed layout
        (`pack_inputs`) that the graph reads its inputs from in place: an
        engine that keeps each step's inputs in graph-stable slots (the model
        writes the next step's inputs into a slot) replays one such graph per
        slot with no staging copy.  That graph is returned and not kept.

        `host_in`, if given, is a pinned host buffer in the packed layout:
        S1, S2 and the BackUp read the index inputs (cand, seq, newest) from
        it in place over the link, and the graph copies the new rows and q
        into its device input buffer on the side stream, in parallel with S1
        and S2 (they are first read after S2).  `host_out`, if given, is a
        pair of pinned tensors (out, lse) that the finishing pass writes the
        step's results into directly."""
        dev = self.device
        if slot is None:
            if getattr(self, "graph_in_packed", None) is None:
                layout, total = self._input_layout()
                self.graph_in_packed = torch.empty(total, dtype=torch.uint8, device=dev)
                self.graph_in = self.input_views(self.graph_in_packed)
            gi = self.graph_in
        else:
            gi = self.input_views(slot)
        dev_buf = self.graph_in_packed if slot is None else slot
        g = torch.cuda.CUDAGraph()
        self.side.wait_stream(torch.cuda.current_stream(dev))
        idx = gi
        if host_in is not None:
            idx = self.input_views(host_in)
        out, lse = (None, None) if host_out is None else host_out
        with torch.cuda.graph(g):
            if host_in is not None:
                main = torch.cuda.current_stream(dev)
                layout, total = self._input_layout()
                cut = dict((name, off) for name, off, _, _, _ in layout)["new_row"]
                self.ev_fork.record(main)
                self.side.wait_event(self.ev_fork)
                with torch.cuda.stream(self.side):
                    dev_buf[cut:total].copy_(host_in[cut:total], non_blocking=True)
            self.step(idx["cand"], idx["seq"], idx["newest"], gi["new_row"], gi["q"],
                      events=events, out=out, lse=lse)
        if slot is None:
            self.graph = g
        return g

    def input_views(self, packed):
        """The step's inputs as views into a buffer in the packed layout."""
        layout, total = self._input_layout()
        if packed.numel() * packed.element_size() < total or packed.dtype != torch.uint8:
            raise ValueError("packed input buffer: uint8 of at least %d bytes" % total)
        return {name: packed[off:off + nb].view(dt).view(shape)
                for name, off, shape, dt, nb in layout}

    def replay(self, cand, seq_lens, newest_slot, new_row, q):
        """One decode step through the captured graph (see `capture`)."""
        gi = self.graph_in
        gi["cand"].copy_(cand, non_blocking=True)
        gi["seq"].copy_(seq_lens, non_blocking=True)
        gi["newest"].copy_(newest_slot, non_blocking=True)
        gi["new_row"].copy_(new_row, non_blocking=True)
        gi["q"].copy_(q, non_blocking=True)
        self.graph.replay()
        return self.out, self.lse

    def replay_packed(self, packed):
        """One decode step through the captured graph, the step's inputs given
        as one packed buffer (`pack_inputs`; device or pinned host memory):
        one copy, one graph launch."""
        self.graph_in_packed.copy_(packed, non_blocking=True)
        self.graph.replay()
        return self.out, self.lse

    @staticmethod
    def q_view(q):
        return q if q.dtype == torch.bfloat16 else q.view(torch.bfloat16)

    # Kernels of libhs launched by one step (index_copy_ above is torch's):
    # BackUp, S1 + S2 (one kernel), SwapIn, resident-row attention,
    # swapped-row attention with the merge in its epilogue.
    def launches_per_step(self):
        return 5


class MultiLayerHiSparse:
    """Several layers of HiSparse state (one HiSparseDecoder each: its own
    pinned pool, hot buffer and LRU state) that share each step's index row,
    overlapped layer by layer (the layerwise offload of the vLLM HiSparse
    walkthrough's overview and of the SGLang HiCache PR's motivation).

    One step: S1 once (the index row is shared); on an index stream, each
    layer's S2 right after S1; on a copy stream, per layer and in layer
    order, the new row's write, its BackUp and the SwapIn of that layer's
    misses, so the host link stays busy from the first SwapIn to the last;
    on the main stream, per layer and in layer order (a layer's query
    depends on the previous layer's output), the attention over the rows
    that were resident (while that layer's SwapIn copies) and then over the
    swapped rows, merged with eq. (7), as in HiSparseDecoder.step."""

    def __init__(self, decoders):
        if not decoders:
            raise ValueError("at least one layer")
        d0 = decoders[0]
        for d in decoders[1:]:
            if (d.num_reqs, d.cap, d.page_size, d.num_pages, d.heads, d.fp8) != (
                    d0.num_reqs, d0.cap, d0.page_size, d0.num_pages, d0.heads, d0.fp8):
                raise ValueError("layers must share the index geometry")
        self.layers = list(decoders)
        dev = d0.device
        self.index_stream = torch.cuda.Stream(device=dev)
        self.copy_stream = torch.cuda.Stream(device=dev)
        L = len(decoders)
        self.ev_s1 = torch.cuda.Event()
        self.ev_s2 = [torch.cuda.Event() for _ in range(L)]
        self.ev_new = [torch.cuda.Event() for _ in range(L)]
        self.ev_swap = [torch.cuda.Event() for _ in range(L)]

    def step(self, cand, seq_lens, newest_slot, new_rows, qs, stream=None):
        """cand int32 [R, top_k], seq_lens int32 [R], newest_slot int32 [R]
        (shared by every layer); new_rows[l] and qs[l] as in
        HiSparseDecoder.step.  Returns [(out, lse)] per layer."""
        d0 = self.layers[0]
        R = d0.num_reqs
        main = stream if stream is not None else torch.cuda.current_stream(d0.device)
        idx_s, cp_s = self.index_stream, self.copy_stream
        tok, slot, count, err = hs.normalize_indices(
            cand, d0.row_req, seq_lens, d0.block_table, d0.page_size, window=d0.window,
            num_sinks=d0.num_sinks, num_pages=d0.num_pages, out=d0.s1_out, stream=main)
        self.ev_s1.record(main)
        idx_s.wait_event(self.ev_s1)
        lists = []
        for l, dec in enumerate(self.layers):
            lists.append(hs.hot_lookup_assign(slot, count, newest_slot, dec.dgi, dec.lru,
                                              dec.region_stride, dec.stats, out=dec.s2_out,
                                              stream=idx_s))
            self.ev_s2[l].record(idx_s)
        for l, dec in enumerate(self.layers):
            (hot_idx, miss_mask, miss_src, miss_dst, miss_count, lerr, hit_idx,
             miss_rows) = lists[l]
            cp_s.wait_event(self.ev_s2[l])
            new_row = new_rows[l]
            if dec.fp8:
                hs.swap_in_fp8ds(hs.device_address(new_row), R, dec.row_bytes, dec.hot,
                                 dec.new_src, dec.new_dst, dec.new_cnt, max_ctas=0,
                                 status=dec.status, stream=cp_s)
                hs.backup(new_row, dec.new_rows_idx, dec.host_dev, newest_slot, dec.row_bytes,
                          dec.host_rows, status=dec.status, stream=cp_s)
            else:
                with torch.cuda.stream(cp_s):
                    dec.hot.index_copy_(0, dec.reserved_rows, new_row)
                hs.backup(dec.hot, dec.reserved_rows, dec.host_dev, newest_slot,
                          dec.row_bytes, dec.host_rows, status=dec.status, stream=cp_s)
            self.ev_new[l].record(cp_s)
            if dec.fp8:
                hs.swap_in_fp8ds(dec.host_dev, dec.host_rows, dec.row_bytes, dec.hot, miss_src,
                                 miss_dst, miss_count, dgi=dec.dgi, hot_size=dec.hot_size,
                                 region_stride=dec.region_stride, max_ctas=dec.swap_ctas,
                                 ticket=dec.ticket, status=dec.status, stream=cp_s)
            else:
                hs.swap_in(dec.host_dev, dec.host_rows, dec.hot, dec.row_bytes, miss_src,
                           miss_dst, miss_count, dgi=dec.dgi, hot_size=dec.hot_size,
                           region_stride=dec.region_stride, max_ctas=dec.swap_ctas,
                           ticket=dec.ticket, status=dec.status, stream=cp_s)
            if not torch.cuda.is_current_stream_capturing():
                new_row.record_stream(cp_s)
            self.ev_swap[l].record(cp_s)
        outs = []
        for l, dec in enumerate(self.layers):
            hit_idx, miss_rows, miss_count = lists[l][6], lists[l][7], lists[l][4]
            qv = HiSparseDecoder.q_view(qs[l])
            nkv = dec.hot.shape[0]
            main.wait_event(self.ev_new[l])
            hs.sparse_decode_partial(qv, dec.hot, dec.hot, dec.row_width, 0, nkv,
                                     hit_idx.view(R, 1, dec.cap), count.view(R, 1), dec.scale,
                                     dec.d_v, dec.part_m, dec.part_l, dec.part_o, 0,
                                     status=dec.status, stream=main)
            main.wait_event(self.ev_swap[l])
            out, lse = hs.sparse_decode_finish(qv, dec.hot, dec.hot, dec.row_width, 0, nkv,
                                               miss_rows.view(R, 1, dec.cap),
                                               miss_count.view(R, 1), dec.scale, dec.d_v,
                                               dec.part_m, dec.part_l, dec.part_o,
                                               dec.parts_hit, sync=dec.sync, out=dec.out,
                                               lse=dec.lse, status=dec.status, stream=main)
            outs.append((out, lse))
        return outs

    def capture(self, cand, seq_lens, newest_slot, new_rows, qs):
        """The step over these (device) input tensors as one CUDA graph, every
        stream included; run one eager step first.  Returns the graph."""
        g = torch.cuda.CUDAGraph()
        cur = torch.cuda.current_stream(self.layers[0].device)
        self.index_stream.wait_stream(cur)
        self.copy_stream.wait_stream(cur)
        with torch.cuda.graph(g):
            self.step(cand, seq_lens, newest_slot, new_rows, qs)
        return g

    # Kernels of libhs per step: S1, then per layer S2, BackUp, SwapIn and
    # the two attention passes (index_copy_ is torch's).
    def launches_per_step(self):
        return 1 + 5 * len(self.layers)
