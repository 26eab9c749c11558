"""Quantized KV cache for NVIDIA B300: Python binding of the C-ABI library.

The compute lives in ``libkvq.so`` (hand-written CUDA for sm_103a plus a thin
C++ host layer); this module only marshals arguments.  The functions below
have the names of the C entry points declared in ``include/kvq.h``:

    kvq_append, kvq_decode_attn, kvq_alloc_bits, kvq_page_bytes,
    kvq_decode_workspace_bytes, kvq_get_status, kvq_reset_status,
    kvq_last_error, kvq_version

``Cache`` owns the device memory of a paged cache (allocated with PyTorch) and
forwards to them.  There is no fallback: if ``libkvq.so`` is missing, every
call raises ``KvqLibraryMissing``; build it with
``python -m quantized_decode_attention_diag_b300.build``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED, KVQ_ECUDA, KVQ_EBUDGET, KVQ_EDEVICE, KVQ_EWORKSPACE = range(7)
DEV_BAD_PAGE, DEV_BAD_LENGTH, DEV_NONFINITE, DEV_COPY_TIMEOUT = 0x1, 0x2, 0x4, 0x8
STATUS_NAMES = {KVQ_OK: "KVQ_OK", KVQ_EINVAL: "KVQ_EINVAL", KVQ_EUNSUPPORTED: "KVQ_EUNSUPPORTED",
                KVQ_ECUDA: "KVQ_ECUDA", KVQ_EBUDGET: "KVQ_EBUDGET", KVQ_EDEVICE: "KVQ_EDEVICE",
                KVQ_EWORKSPACE: "KVQ_EWORKSPACE"}


class KvqLibraryMissing(RuntimeError):
    pass


class KvqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class kvq_cache(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("had_block", ctypes.c_int),
        ("window", ctypes.c_int),
        ("max_batch", ctypes.c_int),
        ("num_pages", ctypes.c_int),
        ("bits_host", ctypes.POINTER(ctypes.c_int8)),
        ("layer_pools", ctypes.POINTER(ctypes.c_void_p)),
        ("window_bufs", ctypes.POINTER(ctypes.c_void_p)),
        ("status_dev", ctypes.c_void_p),
        ("launch_flags", ctypes.c_int),
        ("logquant_w", ctypes.c_int),
        ("key_per_channel", ctypes.c_int),
    ]


_lib = None
_I, _LL, _P, _SZ, _F = ctypes.c_int, ctypes.c_longlong, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
_SIGS = {
    "kvq_page_bytes": (_SZ, [ctypes.POINTER(kvq_cache), _I]),
    "kvq_append": (_I, [ctypes.POINTER(kvq_cache), _I, _P, _P, _P, _I, _P, _I, _I, _P]),
    "kvq_decode_workspace_bytes": (_SZ, [ctypes.POINTER(kvq_cache), _I, _I, _I]),
    "kvq_decode_attn": (_I, [ctypes.POINTER(kvq_cache), _I, _P, _I, _P, _I, _P, _I, _I, _F, _P,
                             _P, _SZ, _P]),
    "kvq_decode_attn_static": (_I, [ctypes.POINTER(kvq_cache), _I, _P, _I, _P, _I, _P, _I, _I,
                                    _F, _P, _P]),
    "kvq_decode_step": (_I, [ctypes.POINTER(kvq_cache), _I, _P, _P, _P, _I, _P, _I, _P, _I, _I, _F,
                             _P, _P, _SZ, _P]),
    "kvq_alloc_bits": (_I, [_P, _P, _I, _LL, _P, _P, _P]),
    "kvq_distortion": (_I, [_I, _I, _I, _P, _LL, _P, _I, _P, _P]),
    "kvq_fit_distortion": (_I, [_P, _P, _I, _I, _P, _P]),
    "kvq_logquant_rows": (_I, [_I]),
    "kvq_logquant_members": (_LL, [_LL, _I, _P, _LL]),
    "kvq_window_bytes": (_SZ, [ctypes.POINTER(kvq_cache)]),
    "kvq_get_status": (_I, [ctypes.POINTER(kvq_cache), ctypes.POINTER(ctypes.c_int)]),
    "kvq_reset_status": (_I, [ctypes.POINTER(kvq_cache), _P]),
    "kvq_last_error": (ctypes.c_char_p, []),
    "kvq_version": (ctypes.c_char_p, []),
}


def lib() -> ctypes.CDLL:
    """The loaded ``libkvq.so`` (raises ``KvqLibraryMissing`` when not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise KvqLibraryMissing(
                f"{LIB_PATH} is not built; run python -m quantized_decode_attention_diag_b300.build")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status: int) -> None:
    if status != KVQ_OK:
        raise KvqError(status, kvq_last_error())


def _ptr(t) -> int:
    """Device (or host) address of a tensor / ndarray / int."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


# ------------------------------------------------------------------ C entry points

def kvq_version() -> str:
    return lib().kvq_version().decode()


def kvq_last_error() -> str:
    return lib().kvq_last_error().decode()


def kvq_page_bytes(desc: kvq_cache, layer: int) -> int:
    n = lib().kvq_page_bytes(ctypes.byref(desc), layer)
    if n == 0:
        raise KvqError(KVQ_EINVAL, kvq_last_error())
    return int(n)


def kvq_append(desc: kvq_cache, layer: int, K, V, page_table, max_pages: int, seq_lens, B: int,
               T_new: int, stream=None) -> None:
    _check(lib().kvq_append(ctypes.byref(desc), layer, _ptr(K), _ptr(V), _ptr(page_table),
                            max_pages, _ptr(seq_lens), B, T_new, _stream(stream)))


def kvq_decode_workspace_bytes(desc: kvq_cache, B: int, Hq: int, max_pages: int) -> int:
    n = lib().kvq_decode_workspace_bytes(ctypes.byref(desc), B, Hq, max_pages)
    if n == 0:
        raise KvqError(KVQ_EINVAL, kvq_last_error())
    return int(n)


def kvq_decode_attn(desc: kvq_cache, layer: int, q, q_is_fp32: bool, page_table, max_pages: int,
                    seq_lens, B: int, Hq: int, softmax_scale: float, o, workspace,
                    ws_bytes: int, stream=None) -> None:
    _check(lib().kvq_decode_attn(ctypes.byref(desc), layer, _ptr(q), int(bool(q_is_fp32)),
                                 _ptr(page_table), max_pages, _ptr(seq_lens), B, Hq,
                                 float(softmax_scale), _ptr(o), _ptr(workspace), int(ws_bytes),
                                 _stream(stream)))


def kvq_decode_step(desc: kvq_cache, layer: int, K_new, V_new, q, q_is_fp32: bool, page_table,
                    max_pages: int, seq_lens, B: int, Hq: int, softmax_scale: float, o, workspace,
                    ws_bytes: int, stream=None) -> None:
    """Append of one token per sequence fused with the decode (seq_lens include the token)."""
    _check(lib().kvq_decode_step(ctypes.byref(desc), layer, _ptr(K_new), _ptr(V_new), _ptr(q),
                                 int(bool(q_is_fp32)), _ptr(page_table), max_pages,
                                 _ptr(seq_lens), B, Hq, float(softmax_scale), _ptr(o),
                                 _ptr(workspace), int(ws_bytes), _stream(stream)))


STATIC_WORKSPACE_BYTES = 8 * 1024 * 1024   # KVQ_STATIC_WORKSPACE_BYTES in kvq.h
LAUNCH_OVERLAP = 0x1                        # KVQ_LAUNCH_OVERLAP in kvq.h


def kvq_decode_attn_static(desc: kvq_cache, layer: int, q, q_is_fp32: bool, page_table,
                           max_pages: int, seq_lens, B: int, Hq: int, softmax_scale: float, o,
                           stream=None) -> None:
    """kvq_decode_attn with the library's own fixed scratch instead of a workspace.

    For callers that may not allocate device memory (a plugin whose host owns
    every device byte, a path that must not hit cudaMalloc).  Make the first
    call on a device before any stream capture; calls that overlap on the GPU
    share the scratch and race."""
    _check(lib().kvq_decode_attn_static(ctypes.byref(desc), layer, _ptr(q), int(bool(q_is_fp32)),
                                        _ptr(page_table), max_pages, _ptr(seq_lens), B, Hq,
                                        float(softmax_scale), _ptr(o), _stream(stream)))


def kvq_alloc_bits(w: Sequence[float], beta: Sequence[float], budget: int,
                   allowed_mask: Optional[Sequence[int]] = None) -> tuple[list, int]:
    """RateQuant greedy allocation; returns (bits, leftover)."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    beta = np.ascontiguousarray(beta, dtype=np.float64)
    n = int(w.shape[0])
    if beta.shape[0] != n:
        raise ValueError("w and beta differ in length")
    mask = None if allowed_mask is None else np.ascontiguousarray(allowed_mask, dtype=np.uint16)
    out = np.zeros(n, dtype=np.int32)
    left = ctypes.c_longlong(0)
    _check(lib().kvq_alloc_bits(w.ctypes.data, beta.ctypes.data, n, int(budget),
                                None if mask is None else mask.ctypes.data, out.ctypes.data,
                                ctypes.addressof(left)))
    return out.tolist(), int(left.value)


def kvq_distortion(head_dim: int, had_block: int, X, widths: Sequence[int], mse=None,
                   stream=None):
    """Per-head quantization MSE at each width: X bf16 [T][Hkv][head_dim] on the
    device; returns (or fills) a float64 device tensor [Hkv][len(widths)]."""
    import torch
    T, hkv = int(X.shape[0]), int(X.shape[1])
    if X.dim() != 3 or int(X.shape[2]) != head_dim or X.dtype != torch.bfloat16:
        raise ValueError("X must be bf16 [T][Hkv][head_dim]")
    if not X.is_contiguous():
        raise ValueError("X must be contiguous")
    w = np.ascontiguousarray(widths, dtype=np.int32)
    if mse is None:
        mse = torch.empty((hkv, int(w.shape[0])), dtype=torch.float64, device=X.device)
    _check(lib().kvq_distortion(head_dim, had_block, hkv, _ptr(X), T, w.ctypes.data,
                                int(w.shape[0]), _ptr(mse), _stream(stream)))
    return mse


def kvq_fit_distortion(mse, widths: Sequence[int]) -> tuple[np.ndarray, np.ndarray]:
    """(alpha, beta) per row of mse [n][len(widths)] (host) for D(b) = alpha beta^-b."""
    d = np.ascontiguousarray(mse, dtype=np.float64)
    w = np.ascontiguousarray(widths, dtype=np.int32)
    if d.ndim != 2 or d.shape[1] != w.shape[0]:
        raise ValueError("mse must be [n][len(widths)]")
    alpha = np.zeros(d.shape[0], np.float64)
    beta = np.zeros(d.shape[0], np.float64)
    _check(lib().kvq_fit_distortion(d.ctypes.data, w.ctypes.data, int(w.shape[0]),
                                    int(d.shape[0]), alpha.ctypes.data, beta.ctypes.data))
    return alpha, beta


def kvq_logquant_rows(w: int) -> int:
    """Rows of one plane of the LogQuant reserve for base window w (0 if unsupported)."""
    return int(lib().kvq_logquant_rows(int(w)))


def kvq_logquant_members(n: int, w: int) -> np.ndarray:
    """Positions kept at full precision after n appends with base window w."""
    count = lib().kvq_logquant_members(int(n), int(w), None, 0)
    if count < 0:
        raise KvqError(KVQ_EINVAL, kvq_last_error())
    out = np.zeros(max(count, 1), dtype=np.int64)
    lib().kvq_logquant_members(int(n), int(w), out.ctypes.data, count)
    return out[:count]


def kvq_window_bytes(desc: kvq_cache) -> int:
    return int(lib().kvq_window_bytes(ctypes.byref(desc)))


def kvq_get_status(desc: kvq_cache) -> int:
    v = ctypes.c_int(0)
    st = lib().kvq_get_status(ctypes.byref(desc), ctypes.byref(v))
    if st not in (KVQ_OK, KVQ_EDEVICE):
        raise KvqError(st, kvq_last_error())
    return int(v.value)


def kvq_reset_status(desc: kvq_cache, stream=None) -> None:
    _check(lib().kvq_reset_status(ctypes.byref(desc), _stream(stream)))


def mask_of(widths: Sequence[int]) -> int:
    m = 0
    for b in widths:
        m |= 1 << int(b)
    return m


# ------------------------------------------------------------------ device-memory owner

class Cache:
    """Paged quantized KV cache whose device memory PyTorch allocates.

    ``bits`` is an int array [num_layers][num_kv_heads][2] of (bK, bV).
    Pools are uint8 [num_pages * page_bytes(layer)]; window buffers are bf16
    [max_batch][Hkv][2][rows][head_dim] with rows the window R, the LogQuant
    reserve's rows, or R + 16 with per-channel keys; the status word is one int32.
    """

    def __init__(self, num_layers: int, num_kv_heads: int, head_dim: int, had_block: int,
                 bits, num_pages: int, window: int = 0, max_batch: int = 0, device="cuda",
                 overlap: bool = False, logquant_w: int = 0, key_per_channel: bool = False):
        import torch
        self.bits = np.ascontiguousarray(np.asarray(bits).reshape(num_layers, num_kv_heads, 2),
                                         dtype=np.int8)
        self.num_layers, self.num_kv_heads, self.head_dim = num_layers, num_kv_heads, head_dim
        self.had_block, self.window, self.num_pages = had_block, window, num_pages
        self.max_batch = max_batch
        self.desc = kvq_cache()
        d = self.desc
        d.num_layers, d.num_kv_heads, d.head_dim, d.page_size = num_layers, num_kv_heads, head_dim, 16
        d.had_block, d.window, d.max_batch, d.num_pages = had_block, window, max_batch, num_pages
        d.logquant_w = logquant_w
        d.key_per_channel = 1 if key_per_channel else 0
        self.logquant_w = logquant_w
        self.key_per_channel = bool(key_per_channel)
        d.bits_host = self.bits.ctypes.data_as(ctypes.POINTER(ctypes.c_int8))
        self.page_bytes = [kvq_page_bytes(d, l) for l in range(num_layers)]
        self.pools = [torch.zeros(num_pages * pb, dtype=torch.uint8, device=device)
                      for pb in self.page_bytes]
        self._pool_ptrs = (ctypes.c_void_p * num_layers)(*[p.data_ptr() for p in self.pools])
        d.layer_pools = self._pool_ptrs
        self.windows = None
        self._win_ptrs = None
        if window or logquant_w or key_per_channel:
            rows = self.ring_rows
            self.windows = [torch.zeros((max_batch, num_kv_heads, 2, rows, head_dim),
                                        dtype=torch.bfloat16, device=device)
                            for _ in range(num_layers)]
            self._win_ptrs = (ctypes.c_void_p * num_layers)(*[w.data_ptr() for w in self.windows])
            d.window_bufs = self._win_ptrs
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        d.status_dev = self.status.data_ptr()
        # decode launches may overlap the preceding kernel (programmatic dependent
        # launch); that kernel must not write these pools, the page table or the lengths
        d.launch_flags = LAUNCH_OVERLAP if overlap else 0
        self._ws = {}

    # -- calls ------------------------------------------------------------------------------
    def append(self, layer: int, K, V, page_table, seq_lens, stream=None,
               window_row: int = 0) -> None:
        """K, V bf16 [B][T_new][Hkv][d]; page_table int32 [B][max_pages]; seq_lens int32 [B].

        Sequence b of the call uses window row window_row + b: a call for fewer
        sequences than the batch (a one-sequence prefill) addresses its rows
        through a descriptor whose window pointers are offset."""
        B, T = int(K.shape[0]), int(K.shape[1])
        desc = self.desc
        if window_row and self.windows:
            desc = self._shifted(window_row)
        kvq_append(desc, layer, K, V, page_table, int(page_table.shape[1]), seq_lens, B, T,
                   stream)

    @property
    def ring_rows(self) -> int:
        """Rows per (sequence, KV head, K|V) of the window buffers."""
        if self.logquant_w:
            return kvq_logquant_rows(self.logquant_w)
        return self.window + 16 if self.key_per_channel else self.window

    def _shifted(self, row: int) -> kvq_cache:
        """A copy of the descriptor whose window buffers start at window row `row`."""
        d = kvq_cache.from_buffer_copy(self.desc)
        rows = self.ring_rows
        step = self.num_kv_heads * 2 * rows * self.head_dim * 2
        self._tmp_win = (ctypes.c_void_p * self.num_layers)(
            *[w.data_ptr() + row * step for w in self.windows])
        d.window_bufs = self._tmp_win
        return d

    def workspace(self, B: int, Hq: int, max_pages: int):
        import torch
        n = kvq_decode_workspace_bytes(self.desc, B, Hq, max_pages)
        ws = self._ws.get(n)
        if ws is None:
            ws = torch.zeros(n, dtype=torch.uint8, device=self.pools[0].device)
            self._ws[n] = ws
        return ws

    def decode(self, layer: int, q, page_table, seq_lens, o=None, softmax_scale: float = 0.0,
               workspace=None, stream=None):
        """q [B][Hq][d] (bf16 or fp32) -> o fp32 [B][Hq][d]."""
        import torch
        B, Hq = int(q.shape[0]), int(q.shape[1])
        max_pages = int(page_table.shape[1])
        if o is None:
            o = torch.empty((B, Hq, self.head_dim), dtype=torch.float32, device=q.device)
        ws = workspace if workspace is not None else self.workspace(B, Hq, max_pages)
        kvq_decode_attn(self.desc, layer, q, q.dtype == torch.float32, page_table, max_pages,
                        seq_lens, B, Hq, softmax_scale, o, ws, ws.numel(), stream)
        return o

    def decode_step(self, layer: int, K_new, V_new, q, page_table, seq_lens, o=None,
                    softmax_scale: float = 0.0, workspace=None, stream=None):
        """Append K_new, V_new (bf16 [B][Hkv][d]) at position seq_lens - 1 and decode.

        seq_lens (int32 [B]) count the new token; returns o fp32 [B][Hq][d]."""
        import torch
        B, Hq = int(q.shape[0]), int(q.shape[1])
        max_pages = int(page_table.shape[1])
        if o is None:
            o = torch.empty((B, Hq, self.head_dim), dtype=torch.float32, device=q.device)
        ws = workspace if workspace is not None else self.workspace(B, Hq, max_pages)
        kvq_decode_step(self.desc, layer, K_new, V_new, q, q.dtype == torch.float32, page_table,
                        max_pages, seq_lens, B, Hq, softmax_scale, o, ws, ws.numel(), stream)
        return o

    def get_status(self) -> int:
        return kvq_get_status(self.desc)

    def reset_status(self, stream=None) -> None:
        kvq_reset_status(self.desc, stream)

    # -- host copies (tests, diagnostics) ----------------------------------------------------
    def pool_host(self, layer: int) -> np.ndarray:
        return self.pools[layer].cpu().numpy().reshape(self.num_pages, self.page_bytes[layer])

    def window_host(self, layer: int) -> Optional[np.ndarray]:
        if not self.windows:
            return None
        import torch
        w = self.windows[layer].cpu().view(torch.int16).numpy().view(np.uint16)
        return (w.astype(np.uint32) << 16).view(np.float32)


__all__ = [
    "KVQ_OK", "KVQ_EINVAL", "KVQ_EUNSUPPORTED", "KVQ_ECUDA", "KVQ_EBUDGET", "KVQ_EDEVICE",
    "KVQ_EWORKSPACE", "LAUNCH_OVERLAP", "DEV_BAD_PAGE", "DEV_BAD_LENGTH", "DEV_NONFINITE", "DEV_COPY_TIMEOUT",
    "KvqError", "KvqLibraryMissing", "kvq_cache", "lib", "kvq_version", "kvq_last_error",
    "kvq_page_bytes", "kvq_append", "kvq_decode_workspace_bytes", "kvq_decode_attn",
    "kvq_decode_attn_static", "kvq_decode_step", "STATIC_WORKSPACE_BYTES",
    "kvq_distortion", "kvq_fit_distortion", "kvq_logquant_rows", "kvq_logquant_members",
    "kvq_window_bytes",
    "kvq_alloc_bits", "kvq_get_status", "kvq_reset_status", "mask_of", "Cache",
]
