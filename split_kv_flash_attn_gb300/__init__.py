"""Split-KV flash attention over a partitioned KV cache, for GB300 (sm_103a).

A thin Python layer over libsplitkv.so (C ABI: include/splitkv.h).  The
functions below carry the C names without the ``skv_`` prefix and only
marshal arguments (torch tensors -> device pointers, streams); all compute
runs in the library's CUDA kernels.  PyTorch provides device memory and
streams.

    h = Handle(0)
    o, lse = attn_partial(h, q, k, v, Hk=8, kv_rows=rows)        # unified cache
    o, lse = attn_window_tail(h, q, k_win, v_win, k_tail, v_tail, Hk=8, ...)
    o, lse = attn_combine(h, o_parts, lse_parts)
    x = kv_dequant_q8_0(h, blocks, n_values)
"""
from __future__ import annotations

import ctypes
import math

from . import _lib
from ._lib import F16, Q4_0, Q8_0, SkvShape

__all__ = ["Handle", "SplitKVError", "F16", "Q8_0", "Q4_0", "attn_partial", "attn_combine", "attn_window_tail",
           "attn_paged", "BlockCache", "kv_dequant_q8_0", "kv_dequant_q4_0", "gather_rows", "kv_append", "plan_splits", "plan_prefill_splits",
           "segment_bytes"]


class SplitKVError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_lib.STATUS.get(status, status)}: {msg}")
        self.status = status


def segment_bytes(type_: int, D: int) -> int:
    return {F16: 2 * D, Q8_0: 34 * (D // 32), Q4_0: 18 * (D // 32)}[type_]


def _torch():
    import torch
    return torch


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Handle:
    """Owns the library handle: copy stream, events, workspace, tail ring."""

    def __init__(self, device: int = 0):
        self._h = ctypes.c_void_p()
        rc = _lib.lib().skv_create(int(device), ctypes.byref(self._h))
        if rc != 0:
            raise SplitKVError(rc, "skv_create failed")
        self.device = device

    @property
    def ptr(self):
        return self._h

    def check(self, rc: int):
        if rc != 0:
            msg = _lib.lib().skv_last_error(self._h).decode(errors="replace")
            raise SplitKVError(rc, msg)

    def reserve(self, workspace_bytes: int = 0, ring_bytes_per_slot: int = 0, n_slots: int = 0):
        self.check(_lib.lib().skv_reserve(self._h, workspace_bytes, ring_bytes_per_slot, n_slots))

    def scratch_info(self):
        ws, ring, n = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_int32()
        self.check(_lib.lib().skv_scratch_info(self._h, ctypes.byref(ws), ctypes.byref(ring), ctypes.byref(n)))
        return ws.value, ring.value, n.value

    def sm_count(self) -> int:
        n = ctypes.c_int32()
        self.check(_lib.lib().skv_sm_count(self._h, ctypes.byref(n)))
        return n.value

    def status(self) -> int:
        """Synchronise and read/clear the device status word (raises on a timeout)."""
        code = ctypes.c_int32()
        self.check(_lib.lib().skv_status(self._h, ctypes.byref(code)))
        return code.value

    def set_profile_events(self, before=None, after=None):
        """Bracket later attention-kernel launches with these torch.cuda.Events."""
        b = ctypes.c_void_p(before.cuda_event) if before is not None else None
        a = ctypes.c_void_p(after.cuda_event) if after is not None else None
        self.check(_lib.lib().skv_set_profile_events(self._h, b, a))

    def close(self):
        if self._h:
            _lib.lib().skv_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def plan_prefill_splits(S, nq, H, Hk, n_keys, sm_count, *, k_type=F16, v_type=F16, D=128, rows=False):
    """The split plan a prefill call of this shape gets on the tensor-core
    path (no GPU needed): returns (split_len, n_splits, n_ctas)."""
    sh = SkvShape(int(S), int(nq), int(H), int(Hk), int(D), 1.0 / math.sqrt(D), int(k_type), int(v_type),
                  int(Hk) * segment_bytes(k_type, D), int(Hk) * segment_bytes(v_type, D))
    sl, ns, nc = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int64()
    rc = _lib.lib().skv_plan_prefill_splits(ctypes.byref(sh), int(n_keys), int(sm_count), int(bool(rows)),
                                            ctypes.byref(sl), ctypes.byref(ns), ctypes.byref(nc))
    if rc != 0:
        raise SplitKVError(rc, "skv_plan_prefill_splits rejected its arguments")
    return sl.value, ns.value, nc.value


def plan_splits(n_keys, n_units, sm_count, ctas_per_sm, tile=64, max_split=0):
    """Host-side split planner (no GPU needed): returns (split_len, n_splits)."""
    sl, ns = ctypes.c_int64(), ctypes.c_int32()
    rc = _lib.lib().skv_plan_splits(int(n_keys), int(n_units), int(sm_count), int(ctas_per_sm), int(tile),
                                    int(max_split), ctypes.byref(sl), ctypes.byref(ns))
    if rc != 0:
        raise SplitKVError(rc, "skv_plan_splits rejected its arguments")
    return sl.value, ns.value


def plan_window(per_cell_bytes, kv_size, free_bytes, target_bytes=0, reserve_bytes=1536 << 20, n_pad=256):
    """Host-side resident-window sizing (no GPU needed): cells kept on the device."""
    out = ctypes.c_int64()
    rc = _lib.lib().skv_plan_window(int(per_cell_bytes), int(kv_size), int(free_bytes), int(target_bytes),
                                    int(reserve_bytes), int(n_pad), ctypes.byref(out))
    if rc != 0:
        raise SplitKVError(rc, "skv_plan_window rejected its arguments")
    return out.value


def plan_tail_tile(n_keys, per_key_bytes, n_slots=4, slot_cap_bytes=512 << 20, target_keys=32768, align=256):
    """Host-side tail-tile sizing (no GPU needed): (tile_rows, n_tiles)."""
    rows, n = ctypes.c_int64(), ctypes.c_int32()
    rc = _lib.lib().skv_plan_tail_tile(int(n_keys), int(per_key_bytes), int(n_slots), int(slot_cap_bytes),
                                       int(target_keys), int(align), ctypes.byref(rows), ctypes.byref(n))
    if rc != 0:
        raise SplitKVError(rc, "skv_plan_tail_tile rejected its arguments")
    return rows.value, n.value


def _shape(q, Hk, k_type, v_type, k_row_bytes, v_row_bytes, scale):
    S, nq, H, D = (int(x) for x in q.shape)
    if k_row_bytes is None:
        k_row_bytes = Hk * segment_bytes(k_type, D)
    if v_row_bytes is None:
        v_row_bytes = Hk * segment_bytes(v_type, D)
    sc = 1.0 / math.sqrt(D) if scale is None else float(scale)
    return SkvShape(S, nq, H, int(Hk), D, sc, int(k_type), int(v_type), int(k_row_bytes), int(v_row_bytes))


def _outputs(q, o, lse):
    torch = _torch()
    S, nq, H, D = q.shape
    if o is None:
        o = torch.empty((S, nq, H, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((S, nq, H), dtype=torch.float32, device=q.device)
    return o, lse


def attn_partial(h: Handle, q, k, v, *, Hk, k_type=F16, v_type=F16, k_row_bytes=None, v_row_bytes=None,
                 scale=None, kv_begin=0, kv_end=None, kv_rows=None, kv_rows_per_head=False,
                 mask=None, q_pos=None, key_pos0=0, o=None, lse=None, stream=None):
    """skv_attn_partial: attention over logical keys [kv_begin, kv_end)."""
    sh = _shape(q, Hk, k_type, v_type, k_row_bytes, v_row_bytes, scale)
    if kv_end is None:
        kv_end = int(kv_rows.shape[-1]) if kv_rows is not None else int(k.shape[0])
    rows_ld = int(kv_rows.shape[-1]) if kv_rows is not None else 0
    mask_ld = int(mask.shape[-1]) if mask is not None else 0
    o, lse = _outputs(q, o, lse)
    h.check(_lib.lib().skv_attn_partial(h.ptr, ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(mask), mask_ld,
                                        _ptr(q_pos), int(key_pos0), _ptr(kv_rows), rows_ld,
                                        int(bool(kv_rows_per_head)), int(kv_begin), int(kv_end), _ptr(o),
                                        _ptr(lse), _stream(stream)))
    return o, lse


def attn_combine(h: Handle, o_parts, lse_parts, *, o=None, lse=None, stream=None):
    """skv_attn_combine: o_parts [P, rows, D] fp32, lse_parts [P, rows] -> (o [rows, D], lse [rows])."""
    torch = _torch()
    P, rows, D = (int(x) for x in o_parts.shape)
    if o is None:
        o = torch.empty((rows, D), dtype=torch.float32, device=o_parts.device)
    if lse is None:
        lse = torch.empty((rows,), dtype=torch.float32, device=o_parts.device)
    h.check(_lib.lib().skv_attn_combine(h.ptr, P, _ptr(o_parts), _ptr(lse_parts), rows, D, _ptr(o), _ptr(lse),
                                        _stream(stream)))
    return o, lse


def attn_window_tail(h: Handle, q, k_win, v_win, k_tail_host, v_tail_host, *, Hk, n_win=None, n_tail=None,
                     tile_rows=0, k_type=F16, v_type=F16, k_row_bytes=None, v_row_bytes=None, scale=None,
                     mask=None, q_pos=None, o=None, lse=None, stream=None):
    """skv_attn_window_tail: window rows on the device, tail rows in pinned host memory.

    tile_rows <= 0 lets the library size the tail tiles (skv_plan_tail_tile)."""
    sh = _shape(q, Hk, k_type, v_type, k_row_bytes, v_row_bytes, scale)
    if n_win is None:
        n_win = int(k_win.shape[0]) if k_win is not None else 0
    if n_tail is None:
        n_tail = int(k_tail_host.shape[0]) if k_tail_host is not None else 0
    mask_ld = int(mask.shape[-1]) if mask is not None else 0
    o, lse = _outputs(q, o, lse)
    h.check(_lib.lib().skv_attn_window_tail(h.ptr, ctypes.byref(sh), _ptr(q), _ptr(k_win), _ptr(v_win), int(n_win),
                                            _ptr(k_tail_host), _ptr(v_tail_host), int(n_tail), int(tile_rows),
                                            _ptr(mask), mask_ld, _ptr(q_pos), _ptr(o), _ptr(lse), _stream(stream)))
    return o, lse


def attn_paged(h: Handle, q, k_pages, v_pages, page_ids, *, Hk, page_rows, scale=None, o=None, lse=None,
               stream=None):
    """skv_attn_paged: page_ids int32 [S, Hk, pages_per_list] into pools of
    page_rows x D fp16 pages (one KV head per page)."""
    sh = _shape(q, Hk, F16, F16, None, None, scale)
    o, lse = _outputs(q, o, lse)
    h.check(_lib.lib().skv_attn_paged(h.ptr, ctypes.byref(sh), _ptr(q), _ptr(k_pages), _ptr(v_pages),
                                      int(page_rows), _ptr(page_ids), int(page_ids.shape[-1]), _ptr(o), _ptr(lse),
                                      _stream(stream)))
    return o, lse


class BlockCache:
    """Device block cache over a pinned paged host copy [n_blocks][Hk][block_rows][D] fp16."""

    def __init__(self, h: Handle, host_k, host_v, *, n_blocks, block_rows, Hk, D, n_slots=0, max_lookups=0,
                 ring_blocks=0, max_seqs=1):
        """ring_blocks > 0 makes a ring (static table block -> block % ring_blocks)."""
        self.h = h
        self.Hk, self.D, self.block_rows = int(Hk), int(D), int(block_rows)
        self.ring_blocks = int(ring_blocks)
        self._c = ctypes.c_void_p()
        if self.ring_blocks > 0:
            h.check(_lib.lib().skv_bcache_create_ring(h.ptr, int(n_blocks), int(block_rows), int(Hk), int(D),
                                                      self.ring_blocks, int(max_seqs), _ptr(host_k), _ptr(host_v),
                                                      ctypes.byref(self._c)))
        else:
            h.check(_lib.lib().skv_bcache_create(h.ptr, int(n_blocks), int(block_rows), int(Hk), int(D),
                                                 int(n_slots), int(max_lookups), _ptr(host_k), _ptr(host_v),
                                                 ctypes.byref(self._c)))
        self._keep = (host_k, host_v)

    def ring_restore(self, n_keys, stream=None):
        self.h.check(_lib.lib().skv_bcache_ring_restore(self._c, int(n_keys), _stream(stream)))

    def ring_attn(self, q, n_keys, window=0, *, scale=None, o=None, lse=None, stream=None):
        sh = _shape(q, self.Hk, F16, F16, None, None, scale)
        o, lse = _outputs(q, o, lse)
        self.h.check(_lib.lib().skv_bcache_ring_attn(self._c, ctypes.byref(sh), _ptr(q), int(n_keys), int(window),
                                                     _ptr(o), _ptr(lse), _stream(stream)))
        return o, lse

    def reset(self, stream=None):
        self.h.check(_lib.lib().skv_bcache_reset(self._c, _stream(stream)))

    def resolve(self, sel, page_ids=None, stream=None):
        S, _, n_sel = (int(x) for x in sel.shape)
        self.h.check(_lib.lib().skv_bcache_resolve(self._c, _ptr(sel), S, n_sel, _ptr(page_ids), _stream(stream)))
        return page_ids

    def append(self, k_new, v_new, positions, stream=None):
        """Write-through append of fp32 rows [n][Hk][D] at cache positions."""
        self.h.check(_lib.lib().skv_bcache_append(self._c, _ptr(k_new), _ptr(v_new), _ptr(positions),
                                                  int(positions.numel()), _stream(stream)))

    def attn(self, q, sel, *, scale=None, o=None, lse=None, stream=None):
        sh = _shape(q, self.Hk, F16, F16, None, None, scale)
        o, lse = _outputs(q, o, lse)
        self.h.check(_lib.lib().skv_bcache_attn(self._c, ctypes.byref(sh), _ptr(q), _ptr(sel), int(sel.shape[-1]),
                                                _ptr(o), _ptr(lse), _stream(stream)))
        return o, lse

    def stats(self):
        c = _lib.SkvBcacheCounters()
        self.h.check(_lib.lib().skv_bcache_stats(self._c, ctypes.byref(c)))
        return {k: getattr(c, k) for k, _ in c._fields_}

    def check(self) -> int:
        v = ctypes.c_int32()
        self.h.check(_lib.lib().skv_bcache_check(self._c, ctypes.byref(v)))
        return v.value

    def pool(self):
        k, v, n, ids = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_int64(), ctypes.c_void_p()
        self.h.check(_lib.lib().skv_bcache_pool(self._c, ctypes.byref(k), ctypes.byref(v), ctypes.byref(n),
                                                ctypes.byref(ids)))
        return k.value, v.value, n.value, ids.value

    def close(self):
        if self._c:
            _lib.lib().skv_bcache_destroy(self._c)
            self._c = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _dequant(fn, h, blocks, n_values, out, stream):
    torch = _torch()
    if out is None:
        out = torch.empty((n_values,), dtype=torch.float32, device=blocks.device)
    h.check(fn(h.ptr, _ptr(blocks), int(n_values), _ptr(out), _stream(stream)))
    return out


def kv_dequant_q8_0(h: Handle, blocks, n_values, *, out=None, stream=None):
    return _dequant(_lib.lib().skv_kv_dequant_q8_0, h, blocks, n_values, out, stream)


def kv_dequant_q4_0(h: Handle, blocks, n_values, *, out=None, stream=None):
    return _dequant(_lib.lib().skv_kv_dequant_q4_0, h, blocks, n_values, out, stream)


def gather_rows(h: Handle, src, rows, *, row_bytes=None, out=None, stream=None):
    """dst[i] = src[rows[i]]; negative rows give zero rows."""
    torch = _torch()
    n = int(rows.numel())
    if row_bytes is None:
        row_bytes = src[0].numel() * src.element_size()
    if out is None:
        out = torch.empty((n, row_bytes), dtype=torch.uint8, device=src.device)
    h.check(_lib.lib().skv_gather_rows(h.ptr, _ptr(src), int(row_bytes), _ptr(rows), n, _ptr(out),
                                       _stream(stream)))
    return out


def selftest_wait_timeout(h: Handle, budget_ns: int = 5_000_000, stream=None):
    """skv_selftest_wait_timeout: a bounded device-side wait that nothing
    completes gives up after budget_ns and marks the handle's status word."""
    h.check(_lib.lib().skv_selftest_wait_timeout(h.ptr, int(budget_ns), _stream(stream)))


def kv_append(h: Handle, x, positions, dst0, dst1=None, *, type_=F16, n_rows0=None, n_rows1=None, row_bytes=None,
              stream=None):
    """Write x (fp32 [n][Hk][D], device) into a two-region cell-major cache:
    position p < n_rows0 goes to row p of dst0, otherwise row p - n_rows0 of
    dst1 (device or page-locked host).  Rows are converted to fp16 or
    quantised to q8_0 / q4_0 according to type_."""
    n, Hk, D = (int(s) for s in x.shape)
    if row_bytes is None:
        row_bytes = Hk * segment_bytes(type_, D)
    if n_rows0 is None:
        n_rows0 = 0 if dst0 is None else dst0.numel() * dst0.element_size() // row_bytes
    if n_rows1 is None:
        n_rows1 = 0 if dst1 is None else dst1.numel() * dst1.element_size() // row_bytes
    h.check(_lib.lib().skv_kv_append(h.ptr, int(type_), Hk, D, int(row_bytes), _ptr(x), _ptr(positions), n,
                                     _ptr(dst0), int(n_rows0), _ptr(dst1), int(n_rows1), _stream(stream)))
