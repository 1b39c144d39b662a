"""ctypes binding of libmaskattn (include/maskattn.h), same names as the C ABI.

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch supplies device memory and the current stream.  If the
library cannot be built or loaded, every call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import threading
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE, ATTN_ERR_CUDA, \
    ATTN_ERR_TIMEOUT = range(6)
ATTN_F16, ATTN_BF16 = 0, 1
ATTN_MASK_NONE, ATTN_MASK_CAUSAL, ATTN_MASK_SLIDING, ATTN_MASK_BLOCK = range(4)

# Every symbol include/maskattn.h declares.
EXPORTS = ("attn_workspace_size", "attn_fwd", "attn_bwd", "attn_bwd_noalloc",
           "attn_get_device_status", "attn_noalloc_get_device_status", "attn_profile_enable",
           "attn_profile_read", "attn_status_string")


class attn_shape_t(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
                ("Sq", ctypes.c_int), ("Skv", ctypes.c_int), ("D", ctypes.c_int),
                ("dtype", ctypes.c_int), ("flags", ctypes.c_int)]


ATTN_FLAG_COMPENSATED = 1
ATTN_FLAG_SINGLE_PASS = 2


class attn_mask_desc_t(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("window", ctypes.c_int), ("bx", ctypes.c_int),
                ("by", ctypes.c_int), ("block_mask", ctypes.c_void_p),
                ("seqlen_q", ctypes.c_void_p), ("seqlen_k", ctypes.c_void_p),
                ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
                ("total_q", ctypes.c_int), ("total_k", ctypes.c_int)]


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {attn_status_string(code)}")


_lock = threading.Lock()
_lib = None


def load(build: bool = True) -> ctypes.CDLL:
    """Load libmaskattn.so (building it first when sources are newer)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build else _build.LIB
            lib = ctypes.CDLL(path)
            vp, sz = ctypes.c_void_p, ctypes.c_size_t
            ps, pm = ctypes.POINTER(attn_shape_t), ctypes.POINTER(attn_mask_desc_t)
            lib.attn_workspace_size.argtypes = [ps, pm, ctypes.POINTER(sz)]
            lib.attn_workspace_size.restype = ctypes.c_int
            lib.attn_fwd.argtypes = [ps, vp, vp, vp, vp, pm, ctypes.c_float, vp, vp, vp, sz, vp]
            lib.attn_fwd.restype = ctypes.c_int
            lib.attn_bwd.argtypes = [ps, vp, vp, vp, vp, vp, vp, vp, pm, ctypes.c_float,
                                     vp, vp, vp, vp, vp, sz, vp]
            lib.attn_bwd.restype = ctypes.c_int
            lib.attn_bwd_noalloc.argtypes = [ps, vp, vp, vp, vp, vp, vp, vp, pm, ctypes.c_float,
                                             vp, vp, vp, vp, vp]
            lib.attn_bwd_noalloc.restype = ctypes.c_int
            lib.attn_get_device_status.argtypes = [vp, vp]
            lib.attn_get_device_status.restype = ctypes.c_int
            lib.attn_noalloc_get_device_status.argtypes = [vp]
            lib.attn_noalloc_get_device_status.restype = ctypes.c_int
            lib.attn_profile_enable.argtypes = [ctypes.c_int]
            lib.attn_profile_enable.restype = ctypes.c_int
            lib.attn_profile_read.argtypes = [ctypes.POINTER(ctypes.c_char_p),
                                              ctypes.POINTER(ctypes.c_float), ctypes.c_int,
                                              ctypes.POINTER(ctypes.c_int)]
            lib.attn_profile_read.restype = ctypes.c_int
            lib.attn_status_string.argtypes = [ctypes.c_int]
            lib.attn_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


# ------------------------------------------------------------------ raw C ABI

def attn_status_string(code: int) -> str:
    return load().attn_status_string(int(code)).decode()


def attn_workspace_size(shape: attn_shape_t, mask: attn_mask_desc_t):
    n = ctypes.c_size_t(0)
    r = load().attn_workspace_size(ctypes.byref(shape), ctypes.byref(mask), ctypes.byref(n))
    return r, n.value


def attn_fwd(shape, q, k, v, sink, mask, scale, o, lse, ws, ws_bytes, stream) -> int:
    return load().attn_fwd(ctypes.byref(shape), q, k, v, sink, ctypes.byref(mask),
                           ctypes.c_float(scale), o, lse, ws, ws_bytes, stream)


def attn_bwd(shape, q, k, v, o, dO, lse, sink, mask, scale, dq, dk, dv, dsink, ws, ws_bytes,
             stream) -> int:
    return load().attn_bwd(ctypes.byref(shape), q, k, v, o, dO, lse, sink, ctypes.byref(mask),
                           ctypes.c_float(scale), dq, dk, dv, dsink, ws, ws_bytes, stream)


def attn_bwd_noalloc(shape, q, k, v, o, dO, lse, sink, mask, scale, dq, dk, dv, dsink,
                     stream) -> int:
    """attn_bwd with the library's fixed device scratch instead of a workspace."""
    return load().attn_bwd_noalloc(ctypes.byref(shape), q, k, v, o, dO, lse, sink,
                                   ctypes.byref(mask), ctypes.c_float(scale), dq, dk, dv, dsink,
                                   stream)


def attn_get_device_status(ws, stream) -> int:
    return load().attn_get_device_status(ws, stream)


def attn_noalloc_get_device_status(stream) -> int:
    """Status word of the last attn_bwd_noalloc call on the current device."""
    return load().attn_noalloc_get_device_status(stream)


def attn_profile_enable(on: bool) -> int:
    return load().attn_profile_enable(1 if on else 0)


def attn_profile_read(capacity: int = 16):
    """[(kernel name, ms)] of the most recent profiled call."""
    names = (ctypes.c_char_p * capacity)()
    ms = (ctypes.c_float * capacity)()
    n = ctypes.c_int(0)
    r = load().attn_profile_read(names, ms, capacity, ctypes.byref(n))
    if r != ATTN_OK:
        raise AttnError(r, "attn_profile_read")
    return [(names[i].decode(), float(ms[i])) for i in range(min(n.value, capacity))]


# ------------------------------------------------------------- torch helpers

@dataclass
class Mask:
    kind: int = ATTN_MASK_NONE
    window: int = 0
    bx: int = 1
    by: int = 1
    block_mask: Optional[torch.Tensor] = None   # uint8 [B,Hq,nQB,nKB] on the device
    seqlen_q: Optional[torch.Tensor] = None     # int32 [B] on the device: valid query rows
    seqlen_k: Optional[torch.Tensor] = None     # int32 [B] on the device: valid keys
    # packed layout: int32 [B + 1] cumulative offsets on the device, the
    # longest lengths (the shape's Sq, Skv) and the tensors' token counts
    cu_seqlens_q: Optional[torch.Tensor] = None
    cu_seqlens_k: Optional[torch.Tensor] = None
    max_seqlen_q: int = 0
    max_seqlen_k: int = 0
    total_q: int = 0
    total_k: int = 0

    @property
    def packed(self) -> bool:
        return self.cu_seqlens_q is not None

    def desc(self) -> attn_mask_desc_t:
        def ptr(t):
            return t.data_ptr() if t is not None else None
        for t, n in ((self.seqlen_q, "seqlen_q"), (self.seqlen_k, "seqlen_k"),
                     (self.cu_seqlens_q, "cu_seqlens_q"), (self.cu_seqlens_k, "cu_seqlens_k")):
            if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
                raise ValueError(f"{n} must be a contiguous int32 tensor")
        return attn_mask_desc_t(self.kind, self.window, self.bx, self.by, ptr(self.block_mask),
                                ptr(self.seqlen_q), ptr(self.seqlen_k), ptr(self.cu_seqlens_q),
                                ptr(self.cu_seqlens_k), self.total_q, self.total_k)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return ATTN_F16
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def shape_of(q: torch.Tensor, k: torch.Tensor, flags: int = 0,
             mask: Optional[Mask] = None) -> attn_shape_t:
    """BHSD tensors [B,H,S,D]; or, with a packed mask, token-major [T,H,D]
    tensors whose batch and longest lengths come from the mask."""
    if mask is not None and mask.packed:
        _, Hq, D = q.shape
        _, Hkv, _ = k.shape
        B = mask.cu_seqlens_q.numel() - 1
        return attn_shape_t(B, Hq, Hkv, mask.max_seqlen_q, mask.max_seqlen_k, D, _dtype_code(q),
                            flags)
    B, Hq, Sq, D = q.shape
    _, Hkv, Skv, _ = k.shape
    return attn_shape_t(B, Hq, Hkv, Sq, Skv, D, _dtype_code(q), flags)


def packed_mask(kind: int, seqlens_q, seqlens_k, device, window: int = 0, bx: int = 1,
                by: int = 1, block_mask: Optional[torch.Tensor] = None) -> Mask:
    """Mask for the packed layout from per-sequence lengths (host integers)."""
    import itertools
    lq, lk = [int(x) for x in seqlens_q], [int(x) for x in seqlens_k]
    cq = [0] + list(itertools.accumulate(lq))
    ck = [0] + list(itertools.accumulate(lk))
    return Mask(kind=kind, window=window, bx=bx, by=by, block_mask=block_mask,
                cu_seqlens_q=torch.tensor(cq, dtype=torch.int32, device=device),
                cu_seqlens_k=torch.tensor(ck, dtype=torch.int32, device=device),
                max_seqlen_q=max(lq), max_seqlen_k=max(lk), total_q=cq[-1], total_k=ck[-1])


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def workspace(shape: attn_shape_t, mask: Mask, device) -> torch.Tensor:
    r, n = attn_workspace_size(shape, mask.desc())
    if r != ATTN_OK:
        raise AttnError(r, "attn_workspace_size")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def _check(t: torch.Tensor, name: str):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def fwd(q, k, v, sink, mask: Mask, scale: float, ws: Optional[torch.Tensor] = None,
        stream=None):
    """Forward; returns (o, lse)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    shape = shape_of(q, k, mask=mask)
    o = torch.empty_like(q)
    lse_shape = (q.shape[1], q.shape[0]) if mask.packed else q.shape[:3]   # [Hq, T] when packed
    lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(shape, mask, q.device)
    r = attn_fwd(shape, _ptr(q), _ptr(k), _ptr(v), _ptr(sink), mask.desc(), scale, _ptr(o),
                 _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    if r != ATTN_OK:
        raise AttnError(r, "attn_fwd")
    return o, lse


def bwd(q, k, v, o, dO, lse, sink, mask: Mask, scale: float, ws: Optional[torch.Tensor] = None,
        out=None, stream=None, compensated: bool = False, single_pass: bool = False):
    """Backward; returns (dq, dk, dv, dsink) (dsink is None without a sink).
    compensated: P and dS enter the contractions as high part + remainder.
    single_pass: dq from partials of the key-stationary kernel, summed by a
    reduction kernel (ATTN_FLAG_SINGLE_PASS) instead of the dq kernel."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO"), (lse, "lse")):
        _check(t, n)
    flags = (ATTN_FLAG_COMPENSATED if compensated else 0) | \
        (ATTN_FLAG_SINGLE_PASS if single_pass else 0)
    shape = shape_of(q, k, flags, mask=mask)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dsink = torch.empty_like(sink) if sink is not None else None
    else:
        dq, dk, dv, dsink = out
    if ws is None:
        ws = workspace(shape, mask, q.device)
    r = attn_bwd(shape, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(sink),
                 mask.desc(), scale, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dsink), _ptr(ws),
                 ws.numel(), _stream(stream))
    if r != ATTN_OK:
        raise AttnError(r, "attn_bwd")
    return dq, dk, dv, dsink


def device_status(ws: torch.Tensor, stream=None) -> int:
    return attn_get_device_status(_ptr(ws), _stream(stream))


class HostBackward:
    """Backward from pinned host tensors to pinned host tensors, with the
    host<->device copies overlapped with the kernels.

    The heads of a GQA group are independent of every other group, so the
    call is split into runs of whole key/value heads: `chunks` equal runs, or
    a list of the key/value heads in each run (a short first run shortens the
    copy nothing hides, a short last run the copy out that follows the last
    kernel, and longer runs in between leave fewer grid tails).  Chunk c's
    inputs are copied in on one stream while earlier chunks run attn_bwd and
    their gradients are copied out on another; every chunk is one attn_bwd
    call on pointer offsets into device buffers that are allocated once here
    (the library itself allocates nothing).  Consecutive chunks rotate over
    three compute streams, each with a workspace of its own, so that the SMs
    a chunk leaves idle while its largest key tiles finish take the next
    chunks' work; small chunks also shorten the first copy, which nothing
    hides.  With B > 1 a run of heads is not contiguous across the
    batch, and dSink sums over the batch, so the call is not split
    (chunks = 1).

    __call__ enqueues everything behind the caller's current stream and makes
    that stream wait for the last copy out, so synchronising it covers the
    whole call."""

    def __init__(self, B, Hq, Hkv, Sq, Skv, dtype, mask: Mask, scale: float, has_sink: bool,
                 device, chunks=8, compensated: bool = False):
        self.B, self.Hq, self.Hkv, self.Sq, self.Skv = B, Hq, Hkv, Sq, Skv
        self.dtype, self.mask, self.scale, self.has_sink = dtype, mask, scale, has_sink
        self.device = torch.device(device)
        if isinstance(chunks, int):
            sizes = [Hkv // chunks] * chunks if chunks > 0 and Hkv % chunks == 0 else [Hkv]
        else:
            sizes = [int(x) for x in chunks]
            if any(x <= 0 for x in sizes) or sum(sizes) != Hkv:
                raise ValueError(f"runs of key/value heads {sizes} do not cover the {Hkv} heads")
        if B != 1:
            sizes = [Hkv]
        self.sizes = sizes
        self.chunks = len(sizes)
        self.g = Hq // Hkv
        D = 128
        e = dict(dtype=dtype, device=self.device)
        self.dev = {
            "q": torch.empty(B, Hq, Sq, D, **e), "o": torch.empty(B, Hq, Sq, D, **e),
            "dO": torch.empty(B, Hq, Sq, D, **e), "k": torch.empty(B, Hkv, Skv, D, **e),
            "v": torch.empty(B, Hkv, Skv, D, **e),
            "lse": torch.empty(B, Hq, Sq, dtype=torch.float32, device=self.device),
            "dq": torch.empty(B, Hq, Sq, D, **e), "dk": torch.empty(B, Hkv, Skv, D, **e),
            "dv": torch.empty(B, Hkv, Skv, D, **e),
        }
        if has_sink:
            self.dev["sink"] = torch.empty(Hq, dtype=torch.float32, device=self.device)
            self.dev["dsink"] = torch.empty(Hq, dtype=torch.float32, device=self.device)
        code = ATTN_BF16 if dtype == torch.bfloat16 else ATTN_F16
        flags = ATTN_FLAG_COMPENSATED if compensated else 0
        self.cshapes = [attn_shape_t(B, self.g * kv, kv, Sq, Skv, D, code, flags) for kv in sizes]
        nws = min(3, self.chunks)
        # each workspace is sized for the largest run, so any run may use it
        big = attn_shape_t(B, self.g * max(sizes), max(sizes), Sq, Skv, D, code, flags)
        self.ws = [workspace(big, mask, self.device) for _ in range(nws)]
        self.s_comp = [torch.cuda.Stream(self.device) for _ in range(nws)]
        self.s_in = torch.cuda.Stream(self.device)
        self.s_out = torch.cuda.Stream(self.device)
        self.ev_in = [torch.cuda.Event() for _ in range(self.chunks)]
        self.ev_done = [torch.cuda.Event() for _ in range(self.chunks)]
        self.ev_start = torch.cuda.Event()
        self.ev_out = torch.cuda.Event()
        self.ev_comp = [torch.cuda.Event() for _ in range(len(self.s_comp))]

    def bytes_per_call(self, host_in, host_out):
        h2d = sum(t.numel() * t.element_size() for t in host_in.values() if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in host_out if t is not None)
        return h2d, d2h

    def __call__(self, host_in: dict, host_out):
        """host_in: pinned q, k, v, o, dO, lse (and sink); host_out: pinned
        (dq, dk, dv, dsink)."""
        cur = torch.cuda.current_stream(self.device)
        self.ev_start.record(cur)
        self.s_in.wait_event(self.ev_start)
        for sc in self.s_comp:
            sc.wait_event(self.ev_start)
        g = self.g
        d = self.dev
        k_lo = 0
        for c, kv in enumerate(self.sizes):
            ks = slice(k_lo, k_lo + kv)
            qs = slice(k_lo * g, (k_lo + kv) * g)
            k_lo += kv
            with torch.cuda.stream(self.s_in):
                for n in ("q", "o", "dO", "lse"):
                    d[n][:, qs].copy_(host_in[n][:, qs], non_blocking=True)
                for n in ("k", "v"):
                    d[n][:, ks].copy_(host_in[n][:, ks], non_blocking=True)
                if self.has_sink:
                    d["sink"][qs].copy_(host_in["sink"][qs], non_blocking=True)
                self.ev_in[c].record(self.s_in)
            sc = self.s_comp[c % len(self.s_comp)]
            ws = self.ws[c % len(self.ws)]
            sc.wait_event(self.ev_in[c])
            mask = self.mask
            if mask.block_mask is not None:
                mask = Mask(mask.kind, mask.window, mask.bx, mask.by, mask.block_mask[:, qs],
                            mask.seqlen_q, mask.seqlen_k)
            sink = d["sink"][qs] if self.has_sink else None
            dsink = d["dsink"][qs] if self.has_sink else None
            r = attn_bwd(self.cshapes[c], _ptr(d["q"][:, qs]), _ptr(d["k"][:, ks]),
                         _ptr(d["v"][:, ks]), _ptr(d["o"][:, qs]), _ptr(d["dO"][:, qs]),
                         _ptr(d["lse"][:, qs]), _ptr(sink), mask.desc(), self.scale,
                         _ptr(d["dq"][:, qs]), _ptr(d["dk"][:, ks]), _ptr(d["dv"][:, ks]),
                         _ptr(dsink), _ptr(ws), ws.numel(), _stream(sc))
            if r != ATTN_OK:
                raise AttnError(r, "attn_bwd")
            self.ev_done[c].record(sc)
            self.s_out.wait_event(self.ev_done[c])
            with torch.cuda.stream(self.s_out):
                dq, dk, dv, dsink_h = host_out
                dq[:, qs].copy_(d["dq"][:, qs], non_blocking=True)
                dk[:, ks].copy_(d["dk"][:, ks], non_blocking=True)
                dv[:, ks].copy_(d["dv"][:, ks], non_blocking=True)
                if self.has_sink:
                    dsink_h[qs].copy_(d["dsink"][qs], non_blocking=True)
        self.ev_out.record(self.s_out)
        cur.wait_event(self.ev_out)
        # the compute streams are idle once the last copy out has begun; keep
        # the caller's stream ordered after them too (nothing is pending)
        for sc, ev in zip(self.s_comp, self.ev_comp):
            ev.record(sc)
            cur.wait_event(ev)
