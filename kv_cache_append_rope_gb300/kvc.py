"""Python face of libkvc (include/kvc.h): the same entry points, marshalling only.

``KVCache`` wraps a ``kvc_handle``; each method calls the C entry point of the
same name (``append_attend`` -> ``kvc_append_attend`` ...).  Tensors must be
contiguous CUDA tensors; host int arrays are copied into ctypes arrays.  Work
is enqueued on ``stream`` (default: torch's current stream).
"""
import ctypes

import numpy as np
import torch

from . import _lib as L
from ._lib import KVCError  # noqa: F401  (re-export)

TORCH_DTYPE = {torch.bfloat16: 0, torch.float32: 1, torch.float64: 2}
STORAGE_TORCH = {0: torch.bfloat16, 1: torch.float32, 2: torch.float64}
NAME_CODE = {"bf16": 0, "f32": 1, "f64": 2}


def tensor_desc(t):
    """kvc_tensor descriptor of a contiguous CUDA tensor (rank <= 4)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("libkvc takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libkvc takes contiguous tensors")
    if t.dtype not in TORCH_DTYPE:
        raise ValueError(f"unsupported dtype {t.dtype}")
    if t.dim() > 4:
        raise ValueError("rank must be at most 4")
    d = L.kvc_tensor()
    d.data = t.data_ptr()
    d.dtype = TORCH_DTYPE[t.dtype]
    d.ndim = t.dim()
    for i, s in enumerate(t.shape):
        d.shape[i] = s
    return d


def host_tensor_desc(t):
    """kvc_tensor descriptor of a contiguous CPU tensor (pinned for overlapped copies)."""
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError("the host-buffer call takes CPU tensors")
    if not t.is_contiguous():
        raise ValueError("libkvc takes contiguous tensors")
    if t.dtype not in TORCH_DTYPE:
        raise ValueError(f"unsupported dtype {t.dtype}")
    if t.dim() > 4:
        raise ValueError("rank must be at most 4")
    d = L.kvc_tensor()
    d.data = t.data_ptr()
    d.dtype = TORCH_DTYPE[t.dtype]
    d.ndim = t.dim()
    for i, s in enumerate(t.shape):
        d.shape[i] = s
    return d


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ref(desc):
    return ctypes.byref(desc) if desc is not None else None


class _DeviceArray:
    """Exposes a device pointer to torch through __cuda_array_interface__."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


class KVCache:
    """A kvc_handle: per-layer [B, H_kv, C, d_h] key/value storage on one GPU."""

    def __init__(self, batch, heads_q, capacity, head_dim, layers=1, heads_kv=None, dtype="bf16",
                 rope_base=10000.0, rope_max_positions=0, checked=False, device=0, window=0,
                 block_rows=0, blocks=0):
        cfg = L.kvc_config()
        cfg.batch, cfg.heads_q = batch, heads_q
        cfg.heads_kv = heads_q if heads_kv is None else heads_kv
        cfg.capacity, cfg.head_dim, cfg.layers = capacity, head_dim, layers
        cfg.dtype = NAME_CODE[dtype] if isinstance(dtype, str) else int(dtype)
        cfg.rope_max_positions = rope_max_positions
        cfg.rope_base = float(rope_base)
        cfg.checked = int(bool(checked))
        cfg.device = device
        cfg.window = window
        cfg.block_rows, cfg.blocks = block_rows, blocks
        self._h = ctypes.c_void_p()
        L.check(L.lib.kvc_create_ex(ctypes.byref(cfg), ctypes.byref(self._h)))
        got = L.kvc_config()
        L.check(L.lib.kvc_get_config(self._h, ctypes.byref(got)), self._h)
        self.config = got
        self.device = torch.device("cuda", device)

    # -- lifetime -------------------------------------------------------------
    def destroy(self):
        if self._h:
            L.lib.kvc_destroy(self._h)
            self._h = ctypes.c_void_p()

    close = destroy

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    # -- properties -------------------------------------------------------------
    @property
    def storage_dtype(self):
        return STORAGE_TORCH[self.config.dtype]

    @property
    def out_dtype(self):
        return torch.float64 if self.config.dtype == 2 else torch.float32

    def _check(self, status):
        L.check(status, self._h)

    # -- entry points -------------------------------------------------------------
    def append_attend(self, layer, q, k, v, out=None, stream=None):
        """kvc_append_attend: one decode step; returns ``out`` [B, H_q, 1, d_h]."""
        if out is None:
            out = torch.empty(q.shape, dtype=self.out_dtype, device=q.device)
        dq, dk, dv, do = tensor_desc(q), tensor_desc(k), tensor_desc(v), tensor_desc(out)
        self._check(L.lib.kvc_append_attend(self._h, layer, ctypes.byref(dq), ctypes.byref(dk),
                                            ctypes.byref(dv), ctypes.byref(do), _stream(stream)))
        return out

    def bind_append_attend(self, layer, q, k, v, out, stream=None):
        """A kvc_append_attend call on fixed tensors, its descriptors and stream built once:
        returns a function that enqueues one decode step (for loops that reuse the same
        buffers every step, where building the arguments would cost more host time than
        the call itself)."""
        descs = tuple(tensor_desc(t) for t in (q, k, v, out))
        refs = tuple(ctypes.byref(d) for d in descs)
        st, fn, h, check = _stream(stream), L.lib.kvc_append_attend, self._h, self._check
        keep = (descs, q, k, v, out)

        def call():
            check(fn(h, layer, refs[0], refs[1], refs[2], refs[3], st))
            return keep[-1]
        return call

    def prepare_attend(self, layer, q, k, v, out=None, stream=None):
        """kvc_prepare_attend: a decode step without its commit; returns (out, ticket)."""
        if out is None:
            out = torch.empty(q.shape, dtype=self.out_dtype, device=q.device)
        dq, dk, dv, do = tensor_desc(q), tensor_desc(k), tensor_desc(v), tensor_desc(out)
        ticket = L.kvc_ticket()
        self._check(L.lib.kvc_prepare_attend(self._h, layer, ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv),
                                             ctypes.byref(do), ctypes.byref(ticket), _stream(stream)))
        return out, ticket

    def commit(self, tickets, stream=None):
        """kvc_commit: advance every ticket's layer by one row, or none of them."""
        arr = (L.kvc_ticket * len(tickets))(*tickets)
        self._check(L.lib.kvc_commit(self._h, arr, len(tickets), _stream(stream)))

    def prefill_suffix(self, layer, q, k, v, start_pos=None, seqlen=None, out=True, stream=None):
        """kvc_prefill_suffix.  ``out``: a tensor, True (allocate) or None/False (append only)."""
        if out is True:
            out = torch.zeros(q.shape, dtype=self.out_dtype, device=q.device) if q is not None else None
        elif out is False:
            out = None
        dq = tensor_desc(q) if q is not None else None
        dk, dv = tensor_desc(k), tensor_desc(v)
        do = tensor_desc(out) if out is not None else None
        sp = L.int_array(start_pos) if start_pos is not None else None
        sl = L.int_array(seqlen) if seqlen is not None else None
        self._check(L.lib.kvc_prefill_suffix(self._h, layer, _ref(dq), ctypes.byref(dk),
                                             ctypes.byref(dv), sp, sl, _ref(do), _stream(stream)))
        return out

    def prefill_suffix_host(self, layer, q, k, v, start_pos=None, seqlen=None, out=True, chunk_sequences=0,
                            stream=None, sync=True):
        """kvc_prefill_suffix_host: q, k, v (and out) are CPU tensors, ideally pinned.  ``out``: a
        CPU tensor, True (allocate a pinned one) or None/False (append only).  With ``sync`` the
        stream is synchronised before returning, else ``out`` is valid once the stream completes."""
        if out is True:
            out = torch.empty(q.shape, dtype=self.out_dtype).pin_memory() if q is not None else None
        elif out is False:
            out = None
        dq = host_tensor_desc(q) if q is not None else None
        dk, dv = host_tensor_desc(k), host_tensor_desc(v)
        do = host_tensor_desc(out) if out is not None else None
        sp = L.int_array(start_pos) if start_pos is not None else None
        sl = L.int_array(seqlen) if seqlen is not None else None
        st = _stream(stream)
        self._check(L.lib.kvc_prefill_suffix_host(self._h, layer, _ref(dq), ctypes.byref(dk), ctypes.byref(dv),
                                                  sp, sl, _ref(do), int(chunk_sequences), st))
        if sync:
            (stream or torch.cuda.current_stream()).synchronize()
        return out

    def reset(self, stream=None):
        self._check(L.lib.kvc_reset(self._h, _stream(stream)))

    def truncate(self, cut, stream=None):
        self._check(L.lib.kvc_truncate(self._h, L.int_array(cut), _stream(stream)))

    def get_lengths(self, layer=0):
        B = self.config.batch
        ln, nx = (ctypes.c_int32 * B)(), (ctypes.c_int32 * B)()
        self._check(L.lib.kvc_get_lengths(self._h, layer, ln, nx))
        return list(ln), list(nx)

    def get_len(self, layer=0):
        """kvc_get_len: the host mirror of one layer's logical lengths."""
        ln = (ctypes.c_int32 * self.config.batch)()
        self._check(L.lib.kvc_get_len(self._h, layer, ln))
        return list(ln)

    def read_rows(self, layer=0, rows=None, stream=None):
        """kvc_read_rows: the logical snapshot of one layer -- keys and values [B, H_kv, R, d_h]
        in the storage dtype and positions [B, R] int32 (R = ``rows``, default C); rows at or past a
        sequence's length are zero (positions -1)."""
        c = self.config
        R = c.capacity if rows is None else int(rows)
        shape = (c.batch, c.heads_kv, R, c.head_dim)
        K = torch.empty(shape, dtype=self.storage_dtype, device=self.device)
        V = torch.empty(shape, dtype=self.storage_dtype, device=self.device)
        P = torch.empty((c.batch, R), dtype=torch.int32, device=self.device)
        dk, dv = tensor_desc(K), tensor_desc(V)
        self._check(L.lib.kvc_read_rows(self._h, layer, ctypes.byref(dk), ctypes.byref(dv),
                                        ctypes.c_void_p(P.data_ptr()), _stream(stream)))
        return K, V, P

    def poison(self):
        """Test only (KVC_OPT_TEST_POISON): every stored row no sequence holds gets keys 0 and
        values 1e4, so that a kernel reading past a length shows in its output."""
        self.set_option(L.OPT_TEST_POISON, 1)

    def share_prefix(self, dst, src, rows, stream=None):
        """kvc_share_prefix: sequence dst (empty) takes src's first rows by sharing its blocks."""
        self._check(L.lib.kvc_share_prefix(self._h, dst, src, rows, _stream(stream)))

    def block_table(self):
        """kvc_block_table: (host block table [B, ceil(C/P)] as numpy int32, free blocks)."""
        c = self.config
        nblk = -(-c.capacity // c.block_rows)
        table = np.zeros((c.batch, nblk), dtype=np.int32)
        free = ctypes.c_int32()
        self._check(L.lib.kvc_block_table(self._h, table.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                          ctypes.byref(free)))
        return table, free.value

    def sync_lengths(self):
        """kvc_sync_lengths: read the device lengths back into the host mirrors."""
        self._check(L.lib.kvc_sync_lengths(self._h))

    def storage(self, layer=0):
        """Views of one layer's device storage: keys, values [B, H_kv, C, d_h] (paged: the pool
        [blocks, H_kv, P, d_h]), positions [B, C]."""
        k, v, p = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
        self._check(L.lib.kvc_storage(self._h, layer, ctypes.byref(k), ctypes.byref(v), ctypes.byref(p)))
        c = self.config
        shape = ((c.blocks, c.heads_kv, c.block_rows, c.head_dim) if c.block_rows
                 else (c.batch, c.heads_kv, c.capacity, c.head_dim))
        code = {0: "<u2", 1: "<f4", 2: "<f8"}[c.dtype]
        with torch.cuda.device(self.device):
            K = torch.as_tensor(_DeviceArray(k.value, shape, code), device=self.device)
            V = torch.as_tensor(_DeviceArray(v.value, shape, code), device=self.device)
            P = torch.as_tensor(_DeviceArray(p.value, (c.batch, c.capacity), "<i4"), device=self.device)
        if c.dtype == 0:
            K, V = K.view(torch.bfloat16), V.view(torch.bfloat16)
        return K, V, P

    def check(self, stream=None):
        """kvc_check: synchronise and verify the device error word and lengths."""
        self._check(L.lib.kvc_check(self._h, _stream(stream)))

    def set_option(self, option, value):
        self._check(L.lib.kvc_set_option(self._h, option, int(value)))

    def kernel_stats(self, kernel=-1):
        """kvc_kernel_stats: (device ms with timing on, launches) of one family (name or id) or all."""
        kid = L.KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
        ms, n = ctypes.c_double(), ctypes.c_int64()
        self._check(L.lib.kvc_kernel_stats(self._h, kid, ctypes.byref(ms), ctypes.byref(n)))
        return ms.value, n.value

    def reset_stats(self):
        self._check(L.lib.kvc_reset_stats(self._h))


def create(batch, heads, capacity, head_dim, layers):
    """kvc_create: bf16, H_q = H_kv = heads, RoPE base 10000."""
    return KVCache(batch, heads, capacity, head_dim, layers=layers)


def _ids(ids):
    """int32 pointer to token ids (numpy int32 arrays are passed without a copy)."""
    if isinstance(ids, np.ndarray) and ids.dtype == np.int32 and ids.flags.c_contiguous:
        return ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if ids.size else None, ids
    return (L.int_array(ids) if len(ids) else None), None


def lcp(cached_ids, query_ids, window=0):
    """kvc_lcp: cut = min(longest common prefix, len(query) - 1), on the host;
    kvc_lcp_window for a sliding-window cache (window > 0)."""
    cut = ctypes.c_int32()
    a, keep_a = _ids(cached_ids)
    b, keep_b = _ids(query_ids)
    if window:
        L.check(L.lib.kvc_lcp_window(a, len(cached_ids), b, len(query_ids), int(window), ctypes.byref(cut)))
    else:
        L.check(L.lib.kvc_lcp(a, len(cached_ids), b, len(query_ids), ctypes.byref(cut)))
    return cut.value
