"""Python binding of libsplitkv.so: argument marshalling only.

Every function here has the name of the C entry point it calls (see
include/splitkv.h) and does nothing but turn numpy arrays / torch tensors into
pointers and sizes, call the library, and raise on a negative status.  All
arithmetic of the path - block costs, the LPT plan, the work lists, partial
attention, the merge - runs in the library.  There is no fallback: if the
library is missing or a call fails, an exception is raised.
"""

import ctypes
import os

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsplitkv.so")
_lib = None

SPLITKV_F32 = 0
SPLITKV_BF16 = 1
KERNEL_AUTO, KERNEL_SIMT, KERNEL_DECODE, KERNEL_TC = 0, 1, 2, 3
KERNEL_NAMES = {KERNEL_SIMT: "simt", KERNEL_DECODE: "decode", KERNEL_TC: "tcgen05"}

_i32, _i64, _f32, _p, _u32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_uint32

_SIGNATURES = {
    "splitkv_num_blocks": (_i64, [_p, _i32, _i32]),
    "splitkv_block_costs": (ctypes.c_int, [_p, _p, _i32, _i32, _i32, _p, _i64]),
    "splitkv_plan": (ctypes.c_int, [_p, _i64, _i32, _p, _p]),
    "splitkv_imbalance": (ctypes.c_int, [_p, _i32, _p]),
    "splitkv_plan_dcp": (ctypes.c_int, [_p, _p, _i32, _i32, _i32, _i32, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_double, _p, _i64, _p, _p, _p]),
    "splitkv_work_words": (_i64, [_i64, _i32]),
    "splitkv_build_work": (ctypes.c_int, [_p, _p, _i32, _i32, _p, _p, _i64, _i32, _p, _i64, _p, _p]),
    "splitkv_build_work_split": (ctypes.c_int, [_p, _p, _i32, _i32, _p, _p, _i64, _i32, _i32, _p, _i64, _p, _p]),
    "splitkv_build_work_tail": (ctypes.c_int, [_p, _p, _i32, _i32, _p, _p, _i64, _i32, _i32, _i32, _i32, _p, _i64,
                                               _p, _p]),
    "splitkv_plan_batch": (ctypes.c_int, [_p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _p, _p, _i64, _p, _p, _p,
                                          _i64, _p, _p, _p]),
    "splitkv_partial_slots": (ctypes.c_int, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _p]),
    "splitkv_auto_kernel": (ctypes.c_int, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "splitkv_backward_kernel": (ctypes.c_int, [_i32, _i32, _i32, _i32, _i32]),
    "splitkv_attn_partial": (ctypes.c_int, [_p, _p, _p, _i64, _p, _i32, _p, _i32, _i32, _i32, _i32,
                                             _i32, _i32, _i32, _i32, _f32, _i32, _i32, _p, _p, _i64,
                                             _i32, _p]),
    "splitkv_merge": (ctypes.c_int, [_p, _p, _i64, _p, _i32, _i32, _i32, _i32, _i32, _p, _p, _p]),
    "splitkv_ticket_count": (_i64, [_i32, _i32, _i32, _i32]),
    "splitkv_fused_launches": (ctypes.c_int, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "splitkv_attn_fused": (ctypes.c_int, [_p, _p, _p, _i64, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32, _i32,
                                          _i32, _i32, _f32, _i32, _i32, _p, _p, _i64, _p, _i64, _p, _p, _i32,
                                          _p]),
    "splitkv_attention_noalloc": (ctypes.c_int, [_p, _p, _p, _i64, _p, _i32, _p, _i64, _i32, _i32, _i32,
                                                  _i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _i64, _p,
                                                  _p, _p]),
    "splitkv_bwd_delta": (ctypes.c_int, [_p, _p, _i32, _i32, _i32, _i32, _p, _p]),
    "splitkv_attn_backward": (ctypes.c_int, [_p, _p, _p, _i64, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32, _i32,
                                             _i32, _i32, _f32, _i32, _i32, _p, _p, _p, _p, _i64, _p, _p, _p]),
    "splitkv_dq_reduce": (ctypes.c_int, [_p, _i64, _p, _i32, _i32, _i32, _i32, _p, _p]),
    "splitkv_device_status": (ctypes.c_int, [_p, _i32]),
    "splitkv_last_error": (ctypes.c_char_p, []),
}


class SplitKVError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


def library_path():
    return _LIB_PATH


def lib():
    """The loaded library (loaded on first use; raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libsplitkv.so not found at {_LIB_PATH}; build it first "
                "(python -m context_long_attention_lpt_gb300.build)")
        L = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGNATURES)


def splitkv_last_error():
    return lib().splitkv_last_error().decode()


def _check(fn, status):
    if status < 0:
        raise SplitKVError(fn, status, splitkv_last_error())
    return status


def _np(a, dtype):
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ host calls


def splitkv_num_blocks(kv_len, block_len):
    kv = _np(kv_len, np.int32)
    return _check("splitkv_num_blocks", lib().splitkv_num_blocks(_ptr(kv), len(kv), block_len))


def splitkv_block_costs(q_len, kv_len, block_len, causal):
    q, kv = _np(q_len, np.int32), _np(kv_len, np.int32)
    n = splitkv_num_blocks(kv, block_len)
    out = np.zeros(n, dtype=np.int64)
    _check("splitkv_block_costs", lib().splitkv_block_costs(_ptr(q), _ptr(kv), len(q), block_len,
                                                           int(bool(causal)), _ptr(out), n))
    return out


def splitkv_plan(block_cost, n_shards):
    c = _np(block_cost, np.int64)
    sob = np.zeros(len(c), dtype=np.int32)
    load = np.zeros(n_shards, dtype=np.int64)
    _check("splitkv_plan", lib().splitkv_plan(_ptr(c), len(c), n_shards, _ptr(sob), _ptr(load)))
    return sob, load


def splitkv_imbalance(shard_load):
    """max / mean - 1 of the shard loads, computed by the library."""
    load = _np(shard_load, np.int64)
    r = ctypes.c_double(0.0)
    _check("splitkv_imbalance", lib().splitkv_imbalance(_ptr(load), len(load), ctypes.byref(r)))
    return r.value


def splitkv_plan_dcp(q_len, kv_len, block_len, causal, max_shards, alpha, beta, gamma=0.0):
    """Returns (n_shards_used, shard_of_block, shard_load[max_shards], modeled_time)."""
    q, kv = _np(q_len, np.int32), _np(kv_len, np.int32)
    n = splitkv_num_blocks(kv, block_len)
    sob = np.zeros(n, dtype=np.int32)
    load = np.zeros(max_shards, dtype=np.int64)
    used = ctypes.c_int32(0)
    t = ctypes.c_double(0.0)
    _check("splitkv_plan_dcp", lib().splitkv_plan_dcp(_ptr(q), _ptr(kv), len(q), block_len, int(bool(causal)),
                                                     max_shards, float(alpha), float(beta), float(gamma),
                                                     _ptr(sob), n,
                                                     _ptr(load), ctypes.byref(used), ctypes.byref(t)))
    return used.value, sob, load, t.value


def splitkv_work_words(n_blocks, B):
    return _check("splitkv_work_words", lib().splitkv_work_words(n_blocks, B))


def splitkv_build_work(q_len, kv_len, block_len, block_cost, shard_of_block, n_shards):
    """Returns (work int32 array, n_items, part_rows)."""
    q, kv = _np(q_len, np.int32), _np(kv_len, np.int32)
    c, sob = _np(block_cost, np.int64), _np(shard_of_block, np.int32)
    words = splitkv_work_words(len(c), len(q))
    work = np.zeros(words, dtype=np.int32)
    n_items = ctypes.c_int32(0)
    part_rows = ctypes.c_int64(0)
    _check("splitkv_build_work",
           lib().splitkv_build_work(_ptr(q), _ptr(kv), len(q), block_len, _ptr(c), _ptr(sob), len(c),
                                    n_shards, _ptr(work), words, ctypes.byref(n_items),
                                    ctypes.byref(part_rows)))
    return work, n_items.value, part_rows.value


def splitkv_build_work_split(q_len, kv_len, block_len, block_cost, shard_of_block, n_shards, max_item_blocks):
    """Returns (work int32 array, n_items, part_rows); items of at most max_item_blocks blocks."""
    q, kv = _np(q_len, np.int32), _np(kv_len, np.int32)
    c, sob = _np(block_cost, np.int64), _np(shard_of_block, np.int32)
    words = splitkv_work_words(len(c), len(q))
    work = np.zeros(words, dtype=np.int32)
    n_items = ctypes.c_int32(0)
    part_rows = ctypes.c_int64(0)
    _check("splitkv_build_work_split",
           lib().splitkv_build_work_split(_ptr(q), _ptr(kv), len(q), block_len, _ptr(c), _ptr(sob), len(c),
                                          n_shards, int(max_item_blocks), _ptr(work), words,
                                          ctypes.byref(n_items), ctypes.byref(part_rows)))
    return work, n_items.value, part_rows.value


def splitkv_build_work_tail(q_len, kv_len, block_len, block_cost, shard_of_block, n_shards, units_per_item, slots,
                            pieces):
    """Returns (work int32 array, n_items, part_rows); the items of the last partial wave
    (units_per_item CTAs per item, `slots` resident CTAs) cut into up to `pieces` items."""
    q, kv = _np(q_len, np.int32), _np(kv_len, np.int32)
    c, sob = _np(block_cost, np.int64), _np(shard_of_block, np.int32)
    words = splitkv_work_words(len(c), len(q))
    work = np.zeros(words, dtype=np.int32)
    n_items = ctypes.c_int32(0)
    part_rows = ctypes.c_int64(0)
    _check("splitkv_build_work_tail",
           lib().splitkv_build_work_tail(_ptr(q), _ptr(kv), len(q), block_len, _ptr(c), _ptr(sob), len(c),
                                         n_shards, int(units_per_item), int(slots), int(pieces), _ptr(work), words,
                                         ctypes.byref(n_items), ctypes.byref(part_rows)))
    return work, n_items.value, part_rows.value


def _host_out(a, dtype, name):
    if not (isinstance(a, np.ndarray) and a.dtype == dtype and a.flags.c_contiguous and a.flags.writeable):
        raise TypeError(f"{name} must be a writeable contiguous {np.dtype(dtype).name} numpy array")
    return a.ctypes.data


def splitkv_plan_batch(q_len, kv_len, block_len, causal, n_shards, block_cost, shard_of_block, shard_load,
                       work_host, work_dev=None, stream=None, units_per_item=0, slots=0, pieces=0):
    """Block costs, LPT plan, work lists and the descriptor upload in one library call.
    q_len, kv_len: [B] sequence lengths; block_cost (int64 [n_blocks]), shard_of_block (int32
    [n_blocks]) and shard_load (int64 [n_shards]) are numpy outputs; work_host is the int32
    descriptor output, a CPU tensor (page-locked for an asynchronous copy) or a numpy array;
    work_dev an int32 device tensor of the same length, or None for no copy.  The copy runs on
    ``stream`` (default: the current stream).  units_per_item, slots, pieces: the tail cut of
    splitkv_build_work_tail (pieces <= 1: none).  Returns (n_items, part_rows)."""
    q_len, kv_len = _np(q_len, np.int32), _np(kv_len, np.int32)
    if len(q_len) != len(kv_len):
        raise ValueError("q_len and kv_len must have one entry per sequence")
    n_blocks = len(block_cost)
    if len(shard_of_block) != n_blocks or len(shard_load) != n_shards:
        raise ValueError("shard_of_block must have n_blocks entries and shard_load n_shards")
    if isinstance(work_host, np.ndarray):
        wh, words = _host_out(work_host, np.int32, "work_host"), work_host.size
    else:
        if work_host.device.type != "cpu" or not work_host.is_contiguous() or work_host.element_size() != 4:
            raise TypeError("work_host must be a contiguous int32 CPU tensor or numpy array")
        wh, words = work_host.data_ptr(), work_host.numel()
    wd, sh = None, None
    if work_dev is not None:
        if work_dev.numel() != words or not work_dev.is_contiguous() or work_dev.element_size() != 4:
            raise ValueError("work_dev must be a contiguous int32 tensor as long as work_host")
        wd, sh = work_dev.data_ptr(), _stream_handle(stream)
    n_items, part_rows = ctypes.c_int32(0), ctypes.c_int64(0)
    _check("splitkv_plan_batch", lib().splitkv_plan_batch(
        q_len.ctypes.data, kv_len.ctypes.data, len(q_len), block_len, int(bool(causal)), n_shards,
        int(units_per_item), int(slots), int(pieces), _host_out(block_cost, np.int64, "block_cost"),
        _host_out(shard_of_block, np.int32, "shard_of_block"), n_blocks, _host_out(shard_load, np.int64, "shard_load"),
        wh, wd, words, ctypes.byref(n_items), ctypes.byref(part_rows), sh))
    return n_items.value, part_rows.value


def splitkv_partial_slots(Hq, Hkv, d, block_len, max_q_len, dtype, kernel=KERNEL_AUTO):
    """(CTAs one partial launch keeps resident on the current device, CTAs it launches per
    work item) for the decode and tensor-core kernels."""
    per_item = ctypes.c_int32(0)
    slots = _check("splitkv_partial_slots", lib().splitkv_partial_slots(Hq, Hkv, d, block_len, max_q_len, dtype,
                                                                        kernel, ctypes.byref(per_item)))
    return slots, per_item.value


def splitkv_auto_kernel(Hq, Hkv, d, block_len, max_q_len, dtype):
    return _check("splitkv_auto_kernel", lib().splitkv_auto_kernel(Hq, Hkv, d, block_len, max_q_len, dtype))


def splitkv_backward_kernel(Hq, Hkv, d, block_len, dtype):
    return _check("splitkv_backward_kernel", lib().splitkv_backward_kernel(Hq, Hkv, d, block_len, dtype))


# ---------------------------------------------------------------- device calls


def _dtype_code(t):
    import torch

    if t.dtype == torch.float32:
        return SPLITKV_F32
    if t.dtype == torch.bfloat16:
        return SPLITKV_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream_handle(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def splitkv_attn_partial(q, k_pool, v_pool, block_table, work, n_items, B, total_q, max_q_len,
                         block_len, scale, causal, o_part, lse_part, kernel=KERNEL_AUTO, stream=None):
    """q [total_q, Hq, d], k_pool/v_pool [n_pool, block_len, Hkv, d], block_table int32 [B, max_blk],
    work int32 (device), o_part fp32 [part_rows, Hq, d], lse_part fp32 [part_rows, Hq]."""
    for name, t in (("q", q), ("k_pool", k_pool), ("v_pool", v_pool), ("block_table", block_table),
                    ("work", work), ("o_part", o_part), ("lse_part", lse_part)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    _, hq, d = q.shape
    n_pool, bl, hkv, d2 = k_pool.shape
    if d2 != d or bl != block_len:
        raise ValueError("k_pool shape does not match q / block_len")
    _check("splitkv_attn_partial", lib().splitkv_attn_partial(
        q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), n_pool, block_table.data_ptr(),
        block_table.shape[1], work.data_ptr(), n_items, B, total_q, max_q_len, hq, hkv, d, block_len,
        float(scale), int(bool(causal)), _dtype_code(q), o_part.data_ptr(), lse_part.data_ptr(),
        o_part.shape[0], kernel, _stream_handle(stream)))


def splitkv_ticket_count(B, Hq, Hkv, max_q_len):
    return _check("splitkv_ticket_count", lib().splitkv_ticket_count(B, Hq, Hkv, max_q_len))


def splitkv_fused_launches(Hq, Hkv, d, block_len, max_q_len, n_items, dtype, kernel=KERNEL_AUTO):
    """1 when splitkv_attn_fused merges inside the partial kernel's launch, else 2."""
    return _check("splitkv_fused_launches",
                  lib().splitkv_fused_launches(Hq, Hkv, d, block_len, max_q_len, n_items, dtype, kernel))


def splitkv_attn_fused(q, k_pool, v_pool, block_table, work, n_items, B, total_q, max_q_len, block_len, scale,
                       causal, o_part, lse_part, tickets, out, lse_out, kernel=KERNEL_AUTO, stream=None):
    """Partial attention + merge (one launch with the decode and tensor-core kernels); tickets: zeroed int32/uint32 device
    tensor of at least splitkv_ticket_count(...) elements, left zeroed."""
    for name, t in (("q", q), ("k_pool", k_pool), ("v_pool", v_pool), ("block_table", block_table),
                    ("work", work), ("o_part", o_part), ("lse_part", lse_part), ("tickets", tickets),
                    ("out", out), ("lse_out", lse_out)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    _, hq, d = q.shape
    n_pool, bl, hkv, d2 = k_pool.shape
    if d2 != d or bl != block_len:
        raise ValueError("k_pool shape does not match q / block_len")
    _check("splitkv_attn_fused", lib().splitkv_attn_fused(
        q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), n_pool, block_table.data_ptr(),
        block_table.shape[1], work.data_ptr(), n_items, B, total_q, max_q_len, hq, hkv, d, block_len,
        float(scale), int(bool(causal)), _dtype_code(q), o_part.data_ptr(), lse_part.data_ptr(),
        o_part.shape[0], tickets.data_ptr(), tickets.numel(), out.data_ptr(), lse_out.data_ptr(), kernel,
        _stream_handle(stream)))


def splitkv_merge(o_part, lse_part, work, B, total_q, out, lse_out, stream=None):
    """out [total_q, Hq, d] (bf16 or fp32), lse_out fp32 [total_q, Hq]."""
    _, hq, d = out.shape
    _check("splitkv_merge", lib().splitkv_merge(
        o_part.data_ptr(), lse_part.data_ptr(), o_part.shape[0], work.data_ptr(), B, total_q, hq, d,
        _dtype_code(out),
        out.data_ptr(), lse_out.data_ptr(), _stream_handle(stream)))


def splitkv_attention_noalloc(q, k_pool, v_pool, block_table, work_host, n_items, B, total_q, max_q_len,
                              block_len, scale, causal, part_rows, out, lse_out, stream=None):
    """Partial attention + merge with the library's fixed scratch array; work_host is the
    numpy int32 descriptor from splitkv_build_work.  out [total_q, Hq, d], lse_out fp32 [total_q, Hq]."""
    for name, t in (("q", q), ("k_pool", k_pool), ("v_pool", v_pool), ("block_table", block_table),
                    ("out", out), ("lse_out", lse_out)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    work = _np(work_host, np.int32)
    _, hq, d = q.shape
    n_pool, bl, hkv, _ = k_pool.shape
    if bl != block_len:
        raise ValueError("k_pool shape does not match block_len")
    _check("splitkv_attention_noalloc", lib().splitkv_attention_noalloc(
        q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), n_pool, block_table.data_ptr(),
        block_table.shape[1], _ptr(work), work.size, n_items, B, total_q, max_q_len, hq, hkv, d, block_len,
        float(scale), int(bool(causal)), _dtype_code(q), part_rows, out.data_ptr(), lse_out.data_ptr(),
        _stream_handle(stream)))


def splitkv_bwd_delta(o, dout, delta, stream=None):
    total_q, hq, d = o.shape
    _check("splitkv_bwd_delta", lib().splitkv_bwd_delta(o.data_ptr(), dout.data_ptr(), total_q, hq, d,
                                                       _dtype_code(o), delta.data_ptr(), _stream_handle(stream)))


def splitkv_attn_backward(q, k_pool, v_pool, block_table, work, n_items, B, total_q, max_q_len, block_len, scale,
                          causal, dout, lse, delta, dq_part, dk_pool, dv_pool, stream=None):
    for name, t in (("q", q), ("k_pool", k_pool), ("v_pool", v_pool), ("dout", dout), ("lse", lse),
                    ("delta", delta), ("dq_part", dq_part), ("dk_pool", dk_pool), ("dv_pool", dv_pool)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    _, hq, d = q.shape
    n_pool, bl, hkv, _ = k_pool.shape
    _check("splitkv_attn_backward", lib().splitkv_attn_backward(
        q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), n_pool, block_table.data_ptr(), block_table.shape[1],
        work.data_ptr(), n_items, B, total_q, max_q_len, hq, hkv, d, block_len, float(scale), int(bool(causal)),
        _dtype_code(q), dout.data_ptr(), lse.data_ptr(), delta.data_ptr(), dq_part.data_ptr(), dq_part.shape[0],
        dk_pool.data_ptr(), dv_pool.data_ptr(), _stream_handle(stream)))


def splitkv_dq_reduce(dq_part, work, B, total_q, dq, stream=None):
    _, hq, d = dq.shape
    _check("splitkv_dq_reduce", lib().splitkv_dq_reduce(dq_part.data_ptr(), dq_part.shape[0], work.data_ptr(), B,
                                                       total_q, hq, d, dq.data_ptr(), _stream_handle(stream)))


def splitkv_device_status(clear=False):
    v = ctypes.c_uint32(0)
    _check("splitkv_device_status", lib().splitkv_device_status(ctypes.byref(v), int(bool(clear))))
    return v.value
