"""Thin Python binding of the C ABI in include/mkv.h (ctypes).

Argument marshalling only: every step of compression and decode runs in the
CUDA library libmkv.so.  Functions keep the C names.  Tensor arguments are
torch tensors on the ctx's device; the CUDA stream defaults to torch's current
stream.  A missing library is an ImportError, never a fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import (POINTER, Structure, c_char_p, c_double, c_float, c_int, c_int32, c_int64,
                    c_uint8, c_uint16, c_uint32, c_uint64, c_void_p)

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmkv.so")

MKV_OK = 0
MKV_ERR_INVALID_ARG = 1
MKV_ERR_STATE = 2
MKV_ERR_OOM = 3
MKV_ERR_CUDA = 4
MKV_ERR_DEVICE_CHECK = 5
MKV_ERR_TIMEOUT = 6

MKV_STRATEGY_SM, MKV_STRATEGY_PV, MKV_STRATEGY_DENSE, MKV_STRATEGY_PVB = 0, 1, 2, 3
MKV_FLAG_KERNEL_TIMING = 1
MKV_FLAG_SCORE_TIMING = 2
MKV_FLAG_NO_PDL = 4
MKV_FLAG_BITMASK_PV = 8
MKV_BASIS_STATIC_MAX_BYTES = 16 << 20
(MKV_KERNEL_QROT, MKV_KERNEL_SCORE, MKV_KERNEL_TOPK, MKV_KERNEL_ATTN, MKV_KERNEL_MERGE,
 MKV_KERNEL_GRAM, MKV_KERNEL_EIG, MKV_KERNEL_ANALYZE, MKV_KERNEL_LAYOUT, MKV_KERNEL_PACK) = range(10)
KERNEL_NAMES = ["qrot", "score", "topk", "attn", "merge"]          # decode kernels
COMPRESS_KERNEL_NAMES = ["gram", "eig", "analyze", "layout", "pack"]  # ids 5..9


class mkv_config(Structure):
    _fields_ = [("batch", c_int32), ("n_kv_heads", c_int32), ("n_q_heads", c_int32),
                ("head_dim", c_int32), ("max_ctx", c_int64), ("segment", c_int32),
                ("c", c_int32), ("tau", c_float), ("top_k", c_int32), ("attn_chunk", c_int32),
                ("max_pool_bytes", c_uint64), ("flags", c_uint32), ("device", c_int32)]


class mkv_segment_header(Structure):
    _fields_ = [("off16", c_uint32), ("strategy", c_uint8), ("reserved", c_uint8),
                ("rows", c_uint16)]


class mkv_stats_t(Structure):
    _fields_ = [("ctx_len", c_int64), ("n_segments", c_int64),
                ("strategy_count", (c_int64 * 4) * 2), ("payload_bytes", c_uint64 * 2),
                ("header_bytes", c_uint64), ("uncompressed_bytes", c_uint64),
                ("pool_capacity", c_uint64), ("decode_calls", c_int64),
                ("kernel_launches", c_int64)]


HEADER_NP = np.dtype([("off16", "<u4"), ("strategy", "u1"), ("rsv", "u1"), ("rows", "<u2")])


class MkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {mkv_status_string(status)}"
        if status == MKV_ERR_CUDA or status == MKV_ERR_OOM:
            msg += f" ({mkv_last_error_string()})"
        super().__init__(msg)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run two_compressed_kv_gb300.build_lib.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P = c_void_p
    sig = {
        "mkv_validate_config": (c_int, [POINTER(mkv_config)]),
        "mkv_segment_bytes": (c_uint64, [c_int, c_int, c_int]),
        "mkv_create": (c_int, [POINTER(mkv_config), POINTER(P)]),
        "mkv_compress": (c_int, [P, P, P, c_int64, P]),
        "mkv_decode": (c_int, [P, P, P, P, P]),
        "mkv_decode_layers": (c_int, [P, c_int, P, P, P, P]),
        "mkv_free": (None, [P]),
        "mkv_status_string": (c_char_p, [c_int]),
        "mkv_last_error_string": (c_char_p, []),
        "mkv_stats": (c_int, [P, POINTER(mkv_stats_t)]),
        "mkv_export": (c_int, [P, c_int, c_int, c_int, P, P, P, P, POINTER(c_uint64)]),
        "mkv_kernel_time": (c_int, [P, c_int, POINTER(c_double), POINTER(c_int64), c_int]),
        "mkv_check_device": (c_int, [P]),
        "mkv_basis_static": (c_int, [P, P, c_int, c_int, c_int64, P, P, P]),
        "mkv_debug_wait_test": (c_int, [P, c_uint64, P]),
        "mkv_append": (c_int, [P, P, P, c_int32, P]),
        "mkv_set_flags": (c_int, [P, c_uint32]),
        "mkv_debug_set_pdl": (c_int, [P, c_uint32]),
        "mkv_debug_set_check_extent": (c_int, [P, c_uint64]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()
lib = _lib


def _check(status: int, where: str):
    if status != MKV_OK:
        raise MkvError(status, where)


def _stream_ptr(stream, device=None):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dptr(t, dtype, name, shape=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def mkv_status_string(status: int) -> str:
    return _lib.mkv_status_string(status).decode()


def mkv_last_error_string() -> str:
    return _lib.mkv_last_error_string().decode()


def make_config(batch, n_kv_heads, n_q_heads, max_ctx, segment, c, tau, top_k,
                attn_chunk=0, max_pool_bytes=0, flags=0, device=0, head_dim=128) -> mkv_config:
    return mkv_config(batch=batch, n_kv_heads=n_kv_heads, n_q_heads=n_q_heads, head_dim=head_dim,
                      max_ctx=max_ctx, segment=segment, c=c, tau=tau, top_k=top_k,
                      attn_chunk=attn_chunk, max_pool_bytes=max_pool_bytes, flags=flags,
                      device=device)


def mkv_validate_config(cfg: mkv_config) -> int:
    return _lib.mkv_validate_config(ctypes.byref(cfg))


def mkv_segment_bytes(strategy: int, rows: int, c: int) -> int:
    return int(_lib.mkv_segment_bytes(strategy, rows, c))


def mkv_create(cfg: mkv_config) -> c_void_p:
    h = c_void_p()
    _check(_lib.mkv_create(ctypes.byref(cfg), ctypes.byref(h)), "mkv_create")
    return h


def mkv_free(ctx) -> None:
    _lib.mkv_free(ctx)


def mkv_compress(ctx, k, v, ctx_len=None, stream=None) -> None:
    import torch
    ctx_len = k.shape[2] if ctx_len is None else ctx_len
    pk = _dptr(k, torch.float16, "k")
    pv = _dptr(v, torch.float16, "v", k.shape)
    _check(_lib.mkv_compress(ctx, pk, pv, ctx_len, _stream_ptr(stream, k.device)), "mkv_compress")


def mkv_decode(ctx, q, out, sel=None, stream=None) -> None:
    import torch
    pq = _dptr(q, torch.float16, "q")
    po = _dptr(out, torch.float32, "out", q.shape)
    ps = None if sel is None else _dptr(sel, torch.int32, "sel")
    _check(_lib.mkv_decode(ctx, pq, po, ps, _stream_ptr(stream, q.device)), "mkv_decode")


MKV_MAX_FUSED_LAYERS = 64


def mkv_decode_layers(ctxs, qs, outs, sels=None, stream=None) -> None:
    """mkv_decode of several ctxs (same shape and state) in one launch per
    decode kernel.  ctxs: ctx handles; qs, outs (and sels, or None): one
    tensor per ctx, as for mkv_decode."""
    import torch
    n = len(ctxs)
    if len(qs) != n or len(outs) != n or (sels is not None and len(sels) != n):
        raise ValueError("ctxs, qs, outs and sels must have the same length")
    devs = {t.device for t in list(qs) + list(outs) + list(sels or []) if t is not None}
    if len(devs) > 1:
        raise ValueError("all tensors of one call must be on one device")
    arr = lambda vals: (c_void_p * max(1, n))(*vals)
    pc = arr([c if isinstance(c, int) else getattr(c, "value", c) for c in ctxs])
    pq = arr([_dptr(q, torch.float16, "q") for q in qs])
    po = arr([_dptr(o, torch.float32, "out", q.shape) for o, q in zip(outs, qs)])
    ps = None if sels is None else arr([None if t is None else _dptr(t, torch.int32, "sel")
                                        for t in sels])
    dev = qs[0].device if n else None
    with torch.cuda.device(dev):
        _check(_lib.mkv_decode_layers(pc, n, pq, po, ps, _stream_ptr(stream, dev)),
               "mkv_decode_layers")


def mkv_decode_layers_raw(ctxs, n: int, q_ptrs, out_ptrs, sel_ptrs=None, stream_ptr: int = 0) -> int:
    """Pointer-level call (no checks beyond the library's own); returns the status.
    Any of the arrays may be None (a NULL array)."""
    arr = lambda vals: None if vals is None else (c_void_p * max(1, len(vals)))(*vals)
    return _lib.mkv_decode_layers(arr(ctxs), n, arr(q_ptrs), arr(out_ptrs), arr(sel_ptrs),
                                  stream_ptr or None)


def mkv_append(ctx, k, v, stream=None) -> None:
    """k, v: fp16 [B][H][n][128] new tokens of every stream."""
    import torch
    pk = _dptr(k, torch.float16, "k")
    pv = _dptr(v, torch.float16, "v", k.shape)
    _check(_lib.mkv_append(ctx, pk, pv, int(k.shape[2]), _stream_ptr(stream, k.device)),
           "mkv_append")


def mkv_decode_raw(ctx, q_ptr: int, out_ptr: int, sel_ptr: int = 0, stream_ptr: int = 0) -> int:
    """Pointer-level call (no checks beyond the library's own); returns the status."""
    return _lib.mkv_decode(ctx, q_ptr, out_ptr, sel_ptr or None, stream_ptr or None)


def mkv_stats(ctx) -> dict:
    st = mkv_stats_t()
    _check(_lib.mkv_stats(ctx, ctypes.byref(st)), "mkv_stats")
    return {
        "ctx_len": st.ctx_len, "n_segments": st.n_segments,
        "strategy_count": [[st.strategy_count[x][i] for i in range(4)] for x in range(2)],
        "payload_bytes": [st.payload_bytes[0], st.payload_bytes[1]],
        "header_bytes": st.header_bytes, "uncompressed_bytes": st.uncompressed_bytes,
        "pool_capacity": st.pool_capacity, "decode_calls": st.decode_calls,
        "kernel_launches": st.kernel_launches,
    }


def mkv_export(ctx, b: int, h: int, which: int, n_segments: int):
    """(basis [128,128] fp32, eigvals [128] fp32, headers (structured), payload bytes)."""
    basis = np.zeros((128, 128), dtype=np.float32)
    lam = np.zeros(128, dtype=np.float32)
    hdr = np.zeros(n_segments, dtype=HEADER_NP)
    nbytes = c_uint64(0)
    _check(_lib.mkv_export(ctx, b, h, which, None, None, None, None, ctypes.byref(nbytes)),
           "mkv_export(size)")
    payload = np.zeros(max(1, nbytes.value), dtype=np.uint8)
    _check(_lib.mkv_export(ctx, b, h, which, basis.ctypes.data, lam.ctypes.data,
                           hdr.ctypes.data, payload.ctypes.data, ctypes.byref(nbytes)),
           "mkv_export")
    return basis, lam, hdr, payload[:nbytes.value].tobytes()


def mkv_export_headers(ctx, b: int, h: int, which: int, n_segments: int) -> np.ndarray:
    """Only the segment headers of one stream (off16 relative to the stream)."""
    hdr = np.zeros(n_segments, dtype=HEADER_NP)
    nbytes = c_uint64(0)
    _check(_lib.mkv_export(ctx, b, h, which, None, None, hdr.ctypes.data, None,
                           ctypes.byref(nbytes)), "mkv_export(headers)")
    return hdr


def mkv_check_device(ctx) -> int:
    """MKV_OK, or MKV_ERR_TIMEOUT when a bounded device wait gave up (synchronous)."""
    return _lib.mkv_check_device(ctx)


def mkv_set_flags(ctx, flags: int) -> None:
    _check(_lib.mkv_set_flags(ctx, int(flags)), "mkv_set_flags")


def mkv_debug_set_pdl(ctx, mask: int) -> None:
    """Measurement hook: decode kernels launched with PDL (bit k), bit 8 = no early signal."""
    _check(_lib.mkv_debug_set_pdl(ctx, int(mask)), "mkv_debug_set_pdl")


def mkv_debug_wait_test(ctx, limit_ns: int, stream=None) -> None:
    """Test hook: one CTA waits on an mbarrier nobody arrives on, for limit_ns."""
    _check(_lib.mkv_debug_wait_test(ctx, int(limit_ns), _stream_ptr(stream)),
           "mkv_debug_wait_test")


def mkv_debug_set_check_extent(ctx, nbytes: int) -> None:
    """Test hook: check pool accesses against min(nbytes, pool size); 0 resets."""
    _check(_lib.mkv_debug_set_check_extent(ctx, int(nbytes)), "mkv_debug_set_check_extent")


def mkv_kernel_time(ctx, kernel_id: int, reset: bool = False):
    ms = c_double(0.0)
    n = c_int64(0)
    _check(_lib.mkv_kernel_time(ctx, kernel_id, ctypes.byref(ms), ctypes.byref(n), int(reset)),
           "mkv_kernel_time")
    return ms.value, n.value


def mkv_basis_static(k, v, basis, eigvals, stream=None) -> None:
    """Bases and eigenvalues of every K and V stream, with no ctx and no
    allocation inside the library (its scratch is a static device buffer).
    k, v: fp16 [B][H][T][128]; basis: fp32 [2][B*H][128][128]; eigvals: fp32
    [2][B*H][128], all on the current CUDA device."""
    import torch
    devs = {t.device for t in (k, v, basis, eigvals)}
    if len(devs) != 1:
        raise ValueError("k, v, basis and eigvals must be on one device, got "
                         f"{sorted(map(str, devs))}")
    B, H, T, _ = k.shape
    pk = _dptr(k, torch.float16, "k", (B, H, T, 128))
    pv = _dptr(v, torch.float16, "v", (B, H, T, 128))
    pb = _dptr(basis, torch.float32, "basis", (2, B * H, 128, 128))
    pe = _dptr(eigvals, torch.float32, "eigvals", (2, B * H, 128))
    # the library works on the current device: make it the tensors' own
    with torch.cuda.device(k.device):
        _check(_lib.mkv_basis_static(pk, pv, B, H, T, pb, pe, _stream_ptr(stream, k.device)),
               "mkv_basis_static")


class Mkv:
    """Owns one ctx (one layer); frees it on close()."""

    def __init__(self, cfg: mkv_config):
        self.cfg = cfg
        self.ctx = mkv_create(cfg)
        self.T = 0

    @property
    def group(self) -> int:
        return self.cfg.n_q_heads // self.cfg.n_kv_heads

    def compress(self, k, v, stream=None):
        mkv_compress(self.ctx, k, v, k.shape[2], stream)
        self.T = k.shape[2]

    def append(self, k, v, stream=None):
        mkv_append(self.ctx, k, v, stream)
        self.T += k.shape[2]

    def decode(self, q, out=None, sel=None, stream=None):
        import torch
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        mkv_decode(self.ctx, q, out, sel, stream)
        return out

    def n_segments(self) -> int:
        return int(mkv_stats(self.ctx)["n_segments"])

    def export(self, b, h, which):
        return mkv_export(self.ctx, b, h, which, self.n_segments())

    def stats(self):
        return mkv_stats(self.ctx)

    def close(self):
        if self.ctx is not None:
            mkv_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()
