"""One split-KV attention pass through the C ABI, for a batch of sequences.

``SplitKVAttention`` strings the library calls together in the path's order:

    splitkv_block_costs -> splitkv_plan -> splitkv_build_work   (host)
    copy work descriptor to the device
    splitkv_attn_partial -> splitkv_merge                        (device, one stream)

(the first two lines are one call, splitkv_plan_batch, for the plain LPT plan).

It owns the device buffers the calls need (work descriptor, partials, outputs),
allocated with torch and reused across calls of the same shape.  It computes
nothing itself.

Streams: ``plan(stream=s)`` uploads the work descriptor on ``s`` (default: the
current stream) into one of two device buffers, used in turn.  A device call on
another stream first waits for that upload, and an upload into a buffer waits
for the last device call that read it, so plans and calls may use different
streams: planning batch i+1 on a copy stream overlaps batch i's kernels.  The
partial buffers are shared by ``partial`` and ``merge``: calls of one batch on
different streams are ordered by the caller, as with any stream API.
"""

import numpy as np
import torch

from . import splitkv as _k


class SplitKVAttention:
    def __init__(self, q_len, kv_len, block_len, causal, n_shards, Hq, Hkv, d, dtype,
                 device="cuda", kernel=_k.KERNEL_AUTO, fused=False, planner="lpt", dcp_alpha=1.0,
                 dcp_beta=0.0, dcp_gamma=0.0, item_blocks=0, tail_pieces=None, tail_slots=None):
        self.q_len = [int(x) for x in q_len]
        self.kv_len = [int(x) for x in kv_len]
        self.B = len(self.q_len)
        self.block_len = int(block_len)
        self.causal = bool(causal)
        self.n_shards = int(n_shards)
        self.Hq, self.Hkv, self.d = int(Hq), int(Hkv), int(d)
        self.dtype = dtype
        self.device = torch.device(device)
        self.kernel = kernel
        self.fused = bool(fused)
        if planner not in ("lpt", "dcp"):
            raise ValueError("planner must be 'lpt' or 'dcp'")
        self.planner = planner
        self.dcp_alpha, self.dcp_beta, self.dcp_gamma = float(dcp_alpha), float(dcp_beta), float(dcp_gamma)
        self.n_shards_used = self.n_shards
        self.item_blocks = int(item_blocks)  # > 0: work items of at most this many blocks
        self.tail_pieces = tail_pieces  # > 1: the last partial wave's items cut into this many (set below)
        self.tail_slots = tail_slots  # resident CTAs assumed by the cut (None: the library's count)
        self._slots = None
        self._tickets = None
        self._grad_pools = None
        self.total_q = sum(self.q_len)
        self.max_q_len = max(self.q_len) if self.q_len else 0
        # tail_pieces None: decided after the first plan (_choose_tail)
        self._tail_auto = self.tail_pieces is None
        self.tail_pieces = 0 if self._tail_auto else int(self.tail_pieces)
        self._q_len_np = np.asarray(self.q_len, dtype=np.int32)
        self._kv_len_np = np.asarray(self.kv_len, dtype=np.int32)
        # pinned staging buffers for the work list, used in turn, so planning the
        # next batches on the host runs up to len(ring) uploads ahead of the device
        # (a few KB each; eight steps absorb a host stall of about a millisecond on
        # the shortest workloads)
        self._ring = [[None, None] for _ in range(8)]  # [pinned buffer, upload-done event]
        n_blocks = _k.splitkv_num_blocks(self._kv_len_np, self.block_len)
        self._words = _k.splitkv_work_words(n_blocks, self.B)
        self.block_cost = np.zeros(n_blocks, dtype=np.int64)  # outputs of the one-call plan
        self.shard_of_block = np.zeros(n_blocks, dtype=np.int32)
        self.shard_load = np.zeros(self.n_shards, dtype=np.int64)
        self._ring_next = 0
        self._work_dev = [None, None]  # device descriptors, used in turn
        self._cur = 1                  # the buffer the device calls read (flipped by each plan)
        self._o_part = None
        self._lse_part = None
        self._upload = None            # (event, stream) of the last work upload
        self._last_use = [None, None]  # per buffer: event after the last device call that read it
        self._use_ev = [torch.cuda.Event(), torch.cuda.Event()]
        self.plan()
        if self._tail_auto and self._choose_tail():
            self.plan()

    # host steps -------------------------------------------------------------
    def plan(self, stream=None):
        """Block costs, LPT plan and work lists on the host; copy the work to the device on
        ``stream`` (default: the current stream).  The LPT plan, with or without the tail cut,
        takes one library call (splitkv_plan_batch), which also queues the copy; split selection
        and items of bounded length take the separate calls."""
        if self.tail_pieces > 1 and self.item_blocks > 0:
            raise ValueError("tail_pieces and item_blocks are exclusive")
        one_call = self.planner == "lpt" and self.item_blocks <= 0
        if not one_call:
            work = self._plan_steps()
        else:
            upi, slots = self._tail_slots() if self.tail_pieces > 1 else (0, 0)
        slot = self._ring[self._ring_next]
        self._ring_next = (self._ring_next + 1) % len(self._ring)
        if slot[1] is None:
            slot[0] = torch.empty(self._words, dtype=torch.int32, pin_memory=True)
            slot[1] = torch.cuda.Event()
        else:
            slot[1].synchronize()  # this buffer's last upload has left it
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        b = 1 - self._cur
        buf = self._work_dev[b]
        if buf is None:
            buf = self._work_dev[b] = torch.empty(self._words, dtype=torch.int32, device=self.device)
        elif self._last_use[b] is not None:
            st.wait_event(self._last_use[b])  # the calls of two batches back have read this buffer
        if one_call:
            self.n_items, self.part_rows = _k.splitkv_plan_batch(
                self._q_len_np, self._kv_len_np, self.block_len, self.causal, self.n_shards, self.block_cost,
                self.shard_of_block, self.shard_load, slot[0], buf, st, upi, slots, self.tail_pieces)
        else:
            slot[0].copy_(torch.from_numpy(work))
            with torch.cuda.stream(st):
                buf.copy_(slot[0], non_blocking=True)
        self._cur = b
        slot[1].record(st)
        self._upload = (slot[1], st)
        self._host_slot = slot[0]
        if self._o_part is None or self._o_part.shape[0] < self.part_rows:
            self._o_part = torch.empty((max(self.part_rows, 1), self.Hq, self.d), dtype=torch.float32,
                                       device=self.device)
            self._lse_part = torch.empty((max(self.part_rows, 1), self.Hq), dtype=torch.float32,
                                         device=self.device)
        return self

    def _plan_steps(self):
        """The host steps as separate library calls."""
        self.block_cost = _k.splitkv_block_costs(self._q_len_np, self._kv_len_np, self.block_len,
                                                 self.causal)
        if self.planner == "lpt":
            self.shard_of_block, self.shard_load = _k.splitkv_plan(self.block_cost, self.n_shards)
        else:
            self.n_shards_used, self.shard_of_block, self.shard_load, self.modeled_time = _k.splitkv_plan_dcp(
                self._q_len_np, self._kv_len_np, self.block_len, self.causal, self.n_shards, self.dcp_alpha,
                self.dcp_beta, self.dcp_gamma)
        if self.tail_pieces > 1:
            per_item, slots = self._tail_slots()
            work, self.n_items, self.part_rows = _k.splitkv_build_work_tail(
                self._q_len_np, self._kv_len_np, self.block_len, self.block_cost, self.shard_of_block,
                self.n_shards, per_item, slots, self.tail_pieces)
        elif self.item_blocks > 0:
            work, self.n_items, self.part_rows = _k.splitkv_build_work_split(
                self._q_len_np, self._kv_len_np, self.block_len, self.block_cost, self.shard_of_block,
                self.n_shards, self.item_blocks)
        else:
            work, self.n_items, self.part_rows = _k.splitkv_build_work(
                self._q_len_np, self._kv_len_np, self.block_len, self.block_cost, self.shard_of_block,
                self.n_shards)
        return work

    def _choose_tail(self):
        """Default tail cut: when the launch's last wave of CTAs is at most half full, its
        items are cut into 4 pieces (decode kernel: 184 -> 176 us; tensor-core kernel on the
        1M-context shape: 2.64 -> 2.59 ms).  A fuller last wave gains nothing from the cut and
        pays its extra partial rows (short query: 0.785 -> 0.798 ms; 16 query rows per K/V
        head: 200 -> 208 us).  Returns whether a cut was chosen."""
        if self.item_blocks > 0 or self.kernel_used() not in (_k.KERNEL_DECODE, _k.KERNEL_TC):
            return False
        per_item, slots = self._tail_slots()
        units = self.n_items * per_item
        rem = units % slots if slots > 0 else 0
        if units > slots and 0 < rem <= slots // 2:
            self.tail_pieces = 4
            return True
        return False

    def _tail_slots(self):
        """(CTAs per work item, resident CTAs) for the tail cut."""
        if self._slots is None:  # the shape and kernel are fixed: ask once
            code = _k.SPLITKV_F32 if self.dtype == torch.float32 else _k.SPLITKV_BF16
            with torch.cuda.device(self.device):
                self._slots = _k.splitkv_partial_slots(self.Hq, self.Hkv, self.d, self.block_len,
                                                       self.max_q_len, code, self.kernel)
        slots, per_item = self._slots
        return per_item, (int(self.tail_slots) if self.tail_slots is not None else slots)

    @property
    def work_host(self):
        """A copy of the current plan's work descriptor (int32 numpy)."""
        return self._host_slot.numpy().copy()

    @property
    def imbalance(self):
        """max / mean - 1 of the shard loads of the current plan (from the library)."""
        return _k.splitkv_imbalance(self.shard_load[: self.n_shards_used])

    @property
    def o_part(self):
        return self._o_part[: self.part_rows]

    @property
    def lse_part(self):
        return self._lse_part[: self.part_rows]

    @property
    def work_device(self):
        return self._work_dev[self._cur]

    def kernel_used(self):
        if self.kernel != _k.KERNEL_AUTO:
            return self.kernel
        code = _k.SPLITKV_F32 if self.dtype == torch.float32 else _k.SPLITKV_BF16
        return _k.splitkv_auto_kernel(self.Hq, self.Hkv, self.d, self.block_len, self.max_q_len, code)

    def fuses_in_one_launch(self):
        """Whether splitkv_attn_fused merges inside the partial kernel's launch for this shape."""
        code = _k.SPLITKV_F32 if self.dtype == torch.float32 else _k.SPLITKV_BF16
        return _k.splitkv_fused_launches(self.Hq, self.Hkv, self.d, self.block_len, self.max_q_len, self.n_items,
                                         code, self.kernel) == 1

    # device steps -----------------------------------------------------------
    def wait_plan(self, stream=None):
        """Makes ``stream`` (default: the current stream) wait for the last descriptor upload;
        the device calls do this themselves when needed, so this only moves the wait earlier
        (e.g. ahead of an event that should time the kernel alone)."""
        return self._begin(stream)

    def _begin(self, stream):
        """The stream of a device call, made to wait for the work upload if that ran elsewhere."""
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        ev, up = self._upload
        if st != up:
            st.wait_event(ev)
        return st

    def _end(self, st):
        ev = self._use_ev[self._cur]  # re-recorded: a later wait sees the last device call
        ev.record(st)
        self._last_use[self._cur] = ev

    def partial(self, q, k_pool, v_pool, block_table, scale, stream=None):
        st = self._begin(stream)
        _k.splitkv_attn_partial(q, k_pool, v_pool, block_table, self.work_device, self.n_items, self.B,
                                self.total_q, self.max_q_len, self.block_len, scale, self.causal,
                                self._o_part, self._lse_part, kernel=self.kernel, stream=st)
        self._end(st)

    def merge(self, out, lse, stream=None):
        st = self._begin(stream)
        _k.splitkv_merge(self._o_part, self._lse_part, self.work_device, self.B, self.total_q, out, lse,
                         stream=st)
        self._end(st)

    def backward(self, q, k_pool, v_pool, block_table, scale, out, lse, dout, stream=None):
        """Gradients of the forward pass that produced (out, lse) for upstream gradient dout.
        Returns (dq fp32 [total_q, Hq, d], dk_pool, dv_pool fp32 like the pools; zero where no key).
        dk_pool / dv_pool are this object's buffers, rewritten by the next call: every key slot is
        written by every call and the slots without a key stay zero, so they are cleared only when
        the pool shape or the block table (storage or in-place version) changes."""
        dev = q.device
        st = self._begin(stream)
        with torch.cuda.stream(st):  # this call's buffers are allocated on the stream that uses them
            return self._backward(q, k_pool, v_pool, block_table, scale, out, lse, dout, st, dev)

    def _backward(self, q, k_pool, v_pool, block_table, scale, out, lse, dout, stream, dev):
        delta = torch.empty((self.total_q, self.Hq), dtype=torch.float32, device=dev)
        _k.splitkv_bwd_delta(out, dout, delta, stream=stream)
        dq_part = torch.empty((max(self.part_rows, 1), self.Hq, self.d), dtype=torch.float32, device=dev)
        key = (tuple(k_pool.shape), dev, block_table.data_ptr(), block_table._version)
        if self._grad_pools is None or self._grad_pools[0] != key:
            self._grad_pools = (key, torch.zeros(tuple(k_pool.shape), dtype=torch.float32, device=dev),
                                torch.zeros(tuple(v_pool.shape), dtype=torch.float32, device=dev))
        dk, dv = self._grad_pools[1], self._grad_pools[2]
        _k.splitkv_attn_backward(q, k_pool, v_pool, block_table, self.work_device, self.n_items, self.B,
                                 self.total_q, self.max_q_len, self.block_len, scale, self.causal, dout, lse,
                                 delta, dq_part, dk, dv, stream=stream)
        dq = torch.empty((self.total_q, self.Hq, self.d), dtype=torch.float32, device=dev)
        _k.splitkv_dq_reduce(dq_part, self.work_device, self.B, self.total_q, dq, stream=stream)
        self._end(stream)
        return dq, dk, dv

    def fused_call(self, q, k_pool, v_pool, block_table, scale, out, lse, stream=None):
        st = self._begin(stream)
        if self._tickets is None:
            n = _k.splitkv_ticket_count(self.B, self.Hq, self.Hkv, self.max_q_len)
            with torch.cuda.stream(st):
                self._tickets = torch.zeros(n, dtype=torch.int32, device=self.device)
        _k.splitkv_attn_fused(q, k_pool, v_pool, block_table, self.work_device, self.n_items, self.B,
                              self.total_q, self.max_q_len, self.block_len, scale, self.causal, self._o_part,
                              self._lse_part, self._tickets, out, lse, kernel=self.kernel, stream=st)
        self._end(st)

    @property
    def tickets(self):
        return self._tickets

    def __call__(self, q, k_pool, v_pool, block_table, scale, out=None, lse=None, stream=None):
        if out is None:
            out = torch.empty((self.total_q, self.Hq, self.d), dtype=q.dtype, device=q.device)
        if lse is None:
            lse = torch.empty((self.total_q, self.Hq), dtype=torch.float32, device=q.device)
        if self.fused:
            self.fused_call(q, k_pool, v_pool, block_table, scale, out, lse, stream=stream)
        else:
            self.partial(q, k_pool, v_pool, block_table, scale, stream=stream)
            self.merge(out, lse, stream=stream)
        return out, lse
