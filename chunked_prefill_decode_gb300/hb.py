"""ctypes binding of libhb.so (the C ABI declared in include/hb.h).

Argument marshalling only: every function here turns torch tensors / numpy
arrays into the pointers and sizes the C calls take, calls them, and raises
HbError on a non-zero status.  All computation runs in the library's CUDA
kernels; there is no fallback, and loading fails loudly when the library is
missing.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libhb.so")
_lib = None

HB_OK = 0
HB_NUM_KERNEL_IDS = 3
KERNEL_NAMES = ("kv_append", "attention", "linear")

STATUS_NAMES = {
    0: "HB_OK", 1: "HB_ERR_INVALID_ARG", 2: "HB_ERR_SHAPE", 3: "HB_ERR_UNSUPPORTED",
    4: "HB_ERR_WORKSPACE", 5: "HB_ERR_CUDA", 6: "HB_ERR_DEVICE_INDEX",
    7: "HB_ERR_TIMEOUT", 8: "HB_ERR_OUT_OF_PAGES",
}


class HbError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class HbBatch(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("total_q", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("sliding_window", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("cu_q_len", ctypes.c_void_p),
        ("context_len", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
    ]


EXPORTED = (
    "hb_last_error", "hb_status_string", "hb_kv_append", "hb_plan", "hb_attention",
    "hb_attention_new_kv",
    "hb_check", "hb_timing_enable", "hb_timing_read", "hb_launch_count",
    "hb_builder_create", "hb_builder_destroy", "hb_builder_add_request",
    "hb_builder_step", "hb_builder_complete", "hb_builder_counts",
    "hb_builder_free_list", "hb_builder_last_error", "hb_decode_attention_noalloc",
    "hb_selftest_wait_timeout", "hb_selftest_flag_timeout", "hb_linear", "hb_linear_workspace_size",
    "hb_timing_durations", "hb_step_layout", "hb_step_slot_create", "hb_step_slot_destroy",
    "hb_step_slot_sync", "hb_step",
)

LINEAR_STORE, LINEAR_GATED, LINEAR_RESIDUAL = 0, 1, 2


class HbStepBuffers(ctypes.Structure):
    _fields_ = [("h_in", ctypes.c_void_p), ("d_in", ctypes.c_void_p),
                ("h_out", ctypes.c_void_p), ("d_out", ctypes.c_void_p),
                ("h_plan", ctypes.c_void_p), ("plan_bytes", ctypes.c_size_t),
                ("d_workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


HB_STEP_SECTIONS = 6


class HbLinearOut(ctypes.Structure):
    _fields_ = [("y", ctypes.c_void_p * 3), ("cols", ctypes.c_int32 * 3)]


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libhb.so (raising if it has not been built) and declare its calls."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    P = ctypes.POINTER
    L.hb_last_error.restype = ctypes.c_char_p
    L.hb_last_error.argtypes = []
    L.hb_builder_last_error.restype = ctypes.c_char_p
    L.hb_builder_last_error.argtypes = []
    L.hb_status_string.restype = ctypes.c_char_p
    L.hb_status_string.argtypes = [ctypes.c_int]
    L.hb_kv_append.restype = ctypes.c_int
    L.hb_kv_append.argtypes = [P(HbBatch), vp, vp, vp, vp, vp]
    L.hb_plan.restype = ctypes.c_int
    L.hb_plan.argtypes = [P(HbBatch), vp, vp, i32, vp, P(sz), vp, P(sz), vp]
    L.hb_attention.restype = ctypes.c_int
    L.hb_attention.argtypes = [P(HbBatch), vp, vp, vp, vp, ctypes.c_float, vp, vp, vp]
    L.hb_attention_new_kv.restype = ctypes.c_int
    L.hb_attention_new_kv.argtypes = [P(HbBatch), vp, vp, vp, vp, vp, vp, ctypes.c_float, vp,
                                      vp, vp]
    L.hb_decode_attention_noalloc.restype = ctypes.c_int
    L.hb_decode_attention_noalloc.argtypes = [P(HbBatch), vp, vp, vp, vp, vp, ctypes.c_float,
                                              vp, vp]
    L.hb_linear.restype = ctypes.c_int
    L.hb_linear.argtypes = [vp, vp, i32, i32, i32, i32, P(HbLinearOut), vp, sz, vp]
    L.hb_linear_workspace_size.restype = sz
    L.hb_linear_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.hb_selftest_wait_timeout.restype = ctypes.c_int
    L.hb_selftest_wait_timeout.argtypes = [vp]
    L.hb_selftest_flag_timeout.restype = ctypes.c_int
    L.hb_selftest_flag_timeout.argtypes = [vp]
    L.hb_check.restype = ctypes.c_int
    L.hb_check.argtypes = [vp]
    L.hb_timing_enable.restype = ctypes.c_int
    L.hb_timing_enable.argtypes = [i32]
    L.hb_timing_read.restype = ctypes.c_int
    L.hb_timing_read.argtypes = [P(ctypes.c_double), P(i32)]
    L.hb_timing_durations.restype = ctypes.c_int
    L.hb_timing_durations.argtypes = [i32, P(ctypes.c_float), i32, P(i32)]
    L.hb_step_layout.restype = ctypes.c_int
    L.hb_step_layout.argtypes = [P(HbBatch), P(sz), P(sz)]
    L.hb_step_slot_create.restype = ctypes.c_int
    L.hb_step_slot_create.argtypes = [P(vp)]
    L.hb_step_slot_destroy.restype = None
    L.hb_step_slot_destroy.argtypes = [vp]
    L.hb_step_slot_sync.restype = ctypes.c_int
    L.hb_step_slot_sync.argtypes = [vp]
    L.hb_step.restype = ctypes.c_int
    L.hb_step.argtypes = [P(HbBatch), vp, vp, i32, vp, P(HbStepBuffers), vp, vp,
                          ctypes.c_float, vp, vp, vp]
    L.hb_launch_count.restype = i64
    L.hb_launch_count.argtypes = []
    L.hb_builder_create.restype = ctypes.c_int
    L.hb_builder_create.argtypes = [i32, i32, i32, i32, vp, P(vp)]
    L.hb_builder_destroy.restype = None
    L.hb_builder_destroy.argtypes = [vp]
    L.hb_builder_add_request.restype = ctypes.c_int
    L.hb_builder_add_request.argtypes = [vp, i64, i32, i32]
    L.hb_builder_step.restype = ctypes.c_int
    L.hb_builder_step.argtypes = [vp, i32, P(i32), vp, vp, vp, vp, vp, P(i32)]
    L.hb_builder_complete.restype = ctypes.c_int
    L.hb_builder_complete.argtypes = [vp, i32, P(i32), vp]
    L.hb_builder_counts.restype = ctypes.c_int
    L.hb_builder_counts.argtypes = [vp, P(i32), P(i32), P(i32)]
    L.hb_builder_free_list.restype = ctypes.c_int
    L.hb_builder_free_list.argtypes = [vp, i32, P(i32), vp]
    _lib = L
    return L


def _check(status, builder=False):
    if status != HB_OK:
        L = load()
        msg = (L.hb_builder_last_error() if builder else L.hb_last_error()) or b""
        raise HbError(status, msg.decode(errors="replace"))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return ctypes.c_void_p(t.data_ptr()) if t.numel() else None
    if isinstance(t, np.ndarray):
        return t.ctypes.data_as(ctypes.c_void_p)
    return t


def _stream(stream):
    if stream is None:
        if torch.cuda.is_available():
            return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        return None
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def make_batch(num_seqs, total_q, max_pages_per_seq, num_pages, num_q_heads,
               num_kv_heads, head_dim, cu_q_len, context_len, block_table,
               page_size=16, sliding_window=0) -> HbBatch:
    """hb_batch over device int32 tensors (kept alive by the caller)."""
    for name, t in (("cu_q_len", cu_q_len), ("context_len", context_len),
                    ("block_table", block_table)):
        if t is not None and isinstance(t, torch.Tensor):
            if t.dtype != torch.int32 or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous int32 tensor")
    b = HbBatch()
    b.num_seqs, b.total_q = int(num_seqs), int(total_q)
    b.max_pages_per_seq, b.num_pages = int(max_pages_per_seq), int(num_pages)
    b.num_q_heads, b.num_kv_heads = int(num_q_heads), int(num_kv_heads)
    b.head_dim, b.page_size = int(head_dim), int(page_size)
    b.sliding_window, b.reserved = int(sliding_window), 0
    b.cu_q_len = _ptr(cu_q_len).value if _ptr(cu_q_len) is not None else None
    b.context_len = _ptr(context_len).value if _ptr(context_len) is not None else None
    b.block_table = _ptr(block_table).value if _ptr(block_table) is not None else None
    return b


def _bf16(t, name):
    if t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bfloat16 tensor")
    return _ptr(t)


def hb_kv_append(batch, k_new, v_new, k_cache, v_cache, stream=None):
    _check(load().hb_kv_append(ctypes.byref(batch), _bf16(k_new, "k_new"),
                               _bf16(v_new, "v_new"), _bf16(k_cache, "k_cache"),
                               _bf16(v_cache, "v_cache"), _stream(stream)))


def hb_plan_sizes(batch, q_len, context_len, num_sms):
    """(plan_bytes, workspace_bytes) for the batch; host-only."""
    ql = np.ascontiguousarray(q_len, dtype=np.int32)
    cl = np.ascontiguousarray(context_len, dtype=np.int32)
    pb, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load().hb_plan(ctypes.byref(batch), _ptr(ql), _ptr(cl), int(num_sms), None,
                          ctypes.byref(pb), None, ctypes.byref(wb), None))
    return pb.value, wb.value


def hb_plan(batch, q_len, context_len, num_sms, workspace=None, stream=None,
            plan=None, upload=True):
    """Write the plan; returns (plan as a host uint8 array, device workspace).

    `workspace` (a uint8 device tensor) is allocated when None or too small.
    With upload=False only the host plan is built (no CUDA call)."""
    ql = np.ascontiguousarray(q_len, dtype=np.int32)
    cl = np.ascontiguousarray(context_len, dtype=np.int32)
    if plan is not None and (workspace is not None or not upload):
        # buffers given: plan straight into them; ask for sizes only if they
        # turn out too small
        ws = workspace if upload else None
        pb = ctypes.c_size_t(plan.nbytes)
        wb = ctypes.c_size_t(ws.numel() if ws is not None else 0)
        st = load().hb_plan(ctypes.byref(batch), _ptr(ql), _ptr(cl), int(num_sms), _ptr(plan),
                            ctypes.byref(pb), _ptr(ws), ctypes.byref(wb),
                            _stream(stream) if upload else None)
        if st == 0:
            return plan, ws
        if st != 4:   # anything but HB_ERR_WORKSPACE
            _check(st)
    need_p, need_w = hb_plan_sizes(batch, ql, cl, num_sms)
    if plan is None or plan.nbytes < need_p:
        plan = np.zeros(need_p, dtype=np.uint8)
    if upload and (workspace is None or workspace.numel() < need_w):
        workspace = torch.empty(need_w, dtype=torch.uint8, device="cuda")
    if not upload:
        workspace = None
    pb = ctypes.c_size_t(plan.nbytes)
    wb = ctypes.c_size_t(workspace.numel() if workspace is not None else 0)
    _check(load().hb_plan(ctypes.byref(batch), _ptr(ql), _ptr(cl), int(num_sms),
                          _ptr(plan), ctypes.byref(pb), _ptr(workspace),
                          ctypes.byref(wb), _stream(stream) if upload else None))
    return plan, workspace


HEADER_BYTES = 176
DECODE_ITEM_INTS = 12
CHUNK_ITEM_INTS = 16


def plan_header(plan):
    """Decode the header of a host plan (for tests and reports)."""
    h = np.frombuffer(plan[:88].tobytes(), dtype=np.int32)
    keys = ("magic", "version", "num_seqs", "total_q", "num_q_heads", "num_kv_heads",
            "head_dim", "page_size", "max_pages_per_seq", "num_sms",
            "num_decode_items", "num_chunk_items", "num_partial_slots",
            "num_merge_counters", "decode_grid", "decode_kvh_block",
            "chunk_tokens_per_tile", "num_chunk_slots", "num_chunk_merges", "sliding_window",
            "num_decode_dynamic", "chunk_pairs_only")
    out = {k: int(v) for k, v in zip(keys, h)}
    u = np.frombuffer(plan[88:HEADER_BYTES].tobytes(), dtype=np.uint64)
    for k, v in zip(("ws_decode_offsets", "items_bytes", "ws_counters", "ws_partial_o",
                     "ws_partial_ml", "ws_total", "plan_bytes", "ws_chunk_counters",
                     "ws_chunk_o", "ws_chunk_ml"), u):
        out[k] = int(v)
    return out


def plan_items(plan):
    """(decode items [n, 12] int32 in interval order, chunk items [m, 16]
    int32, decode interval offsets [grid + num_decode_dynamic + 1]) of a host
    plan: interval b < grid is decode CTA b's static range, the rest are the
    dynamic tail.

    Chunk item columns: seq, kv_head, tok0, ntok, kv_tiles (end), q0, q_len,
    ctx, kv_begin, split, n_splits, slot, merge_id, 3 x padding."""
    hd = plan_header(plan)
    body = plan[HEADER_BYTES:]
    nd, nc = hd["num_decode_items"], hd["num_chunk_items"]
    n_int = nd * DECODE_ITEM_INTS + nc * CHUNK_ITEM_INTS
    ints = np.frombuffer(body[: 4 * n_int].tobytes(), dtype=np.int32)
    dec = ints[: nd * DECODE_ITEM_INTS].reshape(nd, DECODE_ITEM_INTS)
    chk = ints[nd * DECODE_ITEM_INTS: n_int].reshape(nc, CHUNK_ITEM_INTS)
    off = hd["ws_decode_offsets"]
    n_int = hd["decode_grid"] + hd["num_decode_dynamic"]
    offs = np.frombuffer(body[off: off + 4 * (n_int + 1)].tobytes(), dtype=np.int32) \
        if n_int > 0 else np.zeros(1, np.int32)
    return dec, chk, offs


def hb_attention(batch, plan, q, k_cache, v_cache, scale, out, workspace, stream=None):
    _check(load().hb_attention(ctypes.byref(batch), _ptr(plan), _bf16(q, "q"),
                               _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache"),
                               ctypes.c_float(scale), _bf16(out, "out"), _ptr(workspace),
                               _stream(stream)))


def hb_attention_new_kv(batch, plan, q, k_new, v_new, k_cache, v_cache, scale, out, workspace,
                        stream=None):
    """hb_attention that reads the chunks' new K/V rows from k_new / v_new (the
    append's inputs) instead of waiting for the append to write them."""
    _check(load().hb_attention_new_kv(ctypes.byref(batch), _ptr(plan), _bf16(q, "q"),
                                      _bf16(k_new, "k_new"), _bf16(v_new, "v_new"),
                                      _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache"),
                                      ctypes.c_float(scale), _bf16(out, "out"), _ptr(workspace),
                                      _stream(stream)))


def hb_decode_attention_noalloc(batch, q_len, context_len, q, k_cache, v_cache, scale,
                                out, stream=None):
    """Decode-row attention with the library's static scratch (no workspace,
    no device allocation by the library); all rows must have q_len == 1."""
    ql = np.ascontiguousarray(q_len, dtype=np.int32)
    cl = np.ascontiguousarray(context_len, dtype=np.int32)
    _check(load().hb_decode_attention_noalloc(
        ctypes.byref(batch), _ptr(ql), _ptr(cl), _bf16(q, "q"), _bf16(k_cache, "k_cache"),
        _bf16(v_cache, "v_cache"), ctypes.c_float(scale), _bf16(out, "out"),
        _stream(stream)))


def hb_check(stream=None):
    _check(load().hb_check(_stream(stream)))


def hb_selftest_wait_timeout(stream=None):
    _check(load().hb_selftest_wait_timeout(_stream(stream)))


def hb_selftest_flag_timeout(stream=None):
    _check(load().hb_selftest_flag_timeout(_stream(stream)))


def hb_timing_enable(on: bool, keep: bool = False):
    """Start (clearing earlier records; with keep=True resuming) or stop
    recording launch durations."""
    _check(load().hb_timing_enable((2 if keep else 1) if on else 0))


def hb_timing_read():
    """{kernel name: (total ms, launches)} since timing was enabled."""
    ms = (ctypes.c_double * HB_NUM_KERNEL_IDS)()
    n = (ctypes.c_int32 * HB_NUM_KERNEL_IDS)()
    _check(load().hb_timing_read(ms, n))
    return {KERNEL_NAMES[i]: (ms[i], n[i]) for i in range(HB_NUM_KERNEL_IDS)}


def hb_timing_durations(kernel):
    """Per-launch durations (ms, launch order) recorded for one kernel name."""
    k = KERNEL_NAMES.index(kernel)
    n = ctypes.c_int32(0)
    _check(load().hb_timing_durations(k, None, 0, ctypes.byref(n)))
    buf = (ctypes.c_float * max(1, n.value))()
    _check(load().hb_timing_durations(k, buf, n.value, ctypes.byref(n)))
    return [float(buf[i]) for i in range(n.value)]


def hb_step_layout(batch):
    """(section offsets [q, k_new, v_new, cu_q_len, context_len, block_table],
    total bytes) of hb_step's packed input block for this batch's sizes."""
    offs = (ctypes.c_size_t * HB_STEP_SECTIONS)()
    n = ctypes.c_size_t(0)
    _check(load().hb_step_layout(ctypes.byref(batch), offs, ctypes.byref(n)))
    return list(offs), n.value


class StepSlot:
    """hb_step_slot: the events that order one set of staging buffers' copies
    and kernels (created on the current device)."""

    def __init__(self):
        h = ctypes.c_void_p()
        _check(load().hb_step_slot_create(ctypes.byref(h)))
        self._h = h

    def sync(self):
        _check(load().hb_step_slot_sync(self._h))

    def close(self):
        if self._h:
            load().hb_step_slot_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def hb_step(batch, q_len, context_len, num_sms, slot, buffers, k_cache, v_cache, scale,
            copy_in_stream, stream, copy_out_stream):
    """One step from host memory (see hb.h).  `buffers` is an HbStepBuffers;
    q_len / context_len are host int32 arrays (kept contiguous by the
    caller for repeated calls)."""
    _check(load().hb_step(ctypes.byref(batch), _ptr(q_len), _ptr(context_len), int(num_sms),
                          slot._h, ctypes.byref(buffers), _bf16(k_cache, "k_cache"),
                          _bf16(v_cache, "v_cache"), ctypes.c_float(scale),
                          _stream(copy_in_stream), _stream(stream), _stream(copy_out_stream)))


def hb_launch_count() -> int:
    return int(load().hb_launch_count())


class Builder:
    """The library's stall-free batch builder (host only)."""

    def __init__(self, budget, page_size, num_pages, max_pages_per_seq, page_order=None):
        self.max_pages_per_seq = max_pages_per_seq
        handle = ctypes.c_void_p()
        order = None
        if page_order is not None:
            order = np.ascontiguousarray(page_order, dtype=np.int32)
        _check(load().hb_builder_create(budget, page_size, num_pages, max_pages_per_seq,
                                        _ptr(order), ctypes.byref(handle)), builder=True)
        self._h = handle
        self._max_rows = 64

    def close(self):
        if self._h:
            load().hb_builder_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_request(self, rid, prompt_len, max_new):
        _check(load().hb_builder_add_request(self._h, int(rid), int(prompt_len),
                                             int(max_new)), builder=True)

    def step(self):
        """Next batch as a dict of numpy arrays, or None when there is nothing to run."""
        while True:
            mr, mp = self._max_rows, self.max_pages_per_seq
            # the library writes every entry of the rows it returns (block
            # table entries past a row's pages as -1); the rest is not read
            ql = np.empty(mr, np.int32)
            cl = np.empty(mr, np.int32)
            bt = np.empty((mr, mp), np.int32)
            ids = np.empty(mr, np.int64)
            kind = np.empty(mr, np.int32)
            n, over = ctypes.c_int32(0), ctypes.c_int32(0)
            st = load().hb_builder_step(self._h, mr, ctypes.byref(n), _ptr(ql), _ptr(cl),
                                        _ptr(bt), _ptr(ids), _ptr(kind), ctypes.byref(over))
            if st == 4 and n.value > mr:      # HB_ERR_WORKSPACE: grow and retry
                self._max_rows = n.value
                continue
            _check(st, builder=True)
            k = n.value
            if k == 0:
                return None
            return {"q_len": ql[:k], "context_len": cl[:k], "block_table": bt[:k],
                    "ids": ids[:k], "kind": kind[:k], "over_budget": bool(over.value)}

    def complete(self):
        out = np.zeros(max(self._max_rows, 1), np.int64)
        n = ctypes.c_int32(0)
        _check(load().hb_builder_complete(self._h, out.size, ctypes.byref(n), _ptr(out)),
               builder=True)
        return [int(x) for x in out[: n.value]]

    def counts(self):
        w, r, f = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(load().hb_builder_counts(self._h, ctypes.byref(w), ctypes.byref(r),
                                        ctypes.byref(f)), builder=True)
        return w.value, r.value, f.value

    def free_list(self):
        _, _, nfree = self.counts()
        out = np.zeros(max(nfree, 1), np.int32)
        n = ctypes.c_int32(0)
        _check(load().hb_builder_free_list(self._h, out.size, ctypes.byref(n), _ptr(out)),
               builder=True)
        return [int(x) for x in out[: n.value]]


_linear_ws = {}


def linear_workspace(M, N, K, epilogue, device=None):
    """A zero-filled device workspace big enough for hb_linear's split-K on
    this problem (cached per device and grown as needed), or None."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    need = int(load().hb_linear_workspace_size(int(M), int(N), int(K), int(epilogue), sms))
    if need == 0:
        return None
    ws = _linear_ws.get(dev)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(need, dtype=torch.uint8, device=dev)
        _linear_ws[dev] = ws
    return ws


def hb_linear(x, w, outs, epilogue=LINEAR_STORE, stream=None, workspace="auto"):
    """y = x w^T on the tensor cores.  x [M, K], w [N, K] bf16 device tensors;
    outs: the destination tensors ([M, cols_i] bf16 each; their column
    counts split N for STORE / RESIDUAL, one [M, N / 2] tensor for GATED).
    workspace: "auto" (a cached zero-filled device buffer for split-K when
    the problem has few tiles), None (no split), or a uint8 device tensor."""
    if len(outs) > 3:
        raise ValueError("at most three destinations")
    o = HbLinearOut()
    for i, t in enumerate(outs):
        _bf16(t, "out")
        if t.dim() != 2 or not t.is_contiguous():
            raise ValueError("each destination must be a contiguous 2-D tensor")
        o.y[i] = t.data_ptr()
        o.cols[i] = t.shape[1]
    M, N, K = int(x.shape[0]), int(w.shape[0]), int(x.shape[1])
    if isinstance(workspace, str):
        workspace = linear_workspace(M, N, K, epilogue, x.device) if M > 0 else None
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().hb_linear(_bf16(x, "x"), _bf16(w, "w"), M, N, K, int(epilogue),
                            ctypes.byref(o), ws_ptr, ws_bytes, _stream(stream)))
