"""fp64 CPU oracle for masked attention forward/backward (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  It shares no code with the CUDA library and the CUDA
library never calls it.

The arithmetic lives in ``oracle.c`` (plain loops in double precision, one
output row or column at a time).  This module compiles it with the host C
compiler, loads it with ctypes and converts arguments: every floating-point
input is widened exactly to float64 before the call, so the oracle sees the
very values the GPU sees.

Sources restated by the oracle:
  * tilelang-ascend PR #1 "Add GQA Sink Backward BHSD" -- Summary (online
    softmax with an attention sink and a sliding-window mask) and the commit
    notes of its 2-kernel design (Phase0 Delta = sum(O*dO), five contractions
    + softmax + dS in the KV loop, Phase5 dSink).
  * cannbot-knowledge PR #174, BlockSparseAttentionGrad runbook -- task
    features (uint8 block mask [B,N,ceil(Sq/bx),ceil(Skv/by)]), optimisations
    1-2 (device-side mask transpose, select tables built by prefix count) and
    the precision notes (p = exp(s - lse), ds = p*(dp - delta)).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

MASK_NONE, MASK_CAUSAL, MASK_SLIDING, MASK_BLOCK, MASK_TOKEN = 0, 1, 2, 3, 4


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("Hq", ctypes.c_int64), ("Hkv", ctypes.c_int64),
        ("Sq", ctypes.c_int64), ("Skv", ctypes.c_int64), ("D", ctypes.c_int64),
        ("mask_kind", ctypes.c_int64), ("window", ctypes.c_int64),
        ("bx", ctypes.c_int64), ("by", ctypes.c_int64),
        ("block_mask", ctypes.c_void_p), ("token_mask", ctypes.c_void_p),
        ("sink", ctypes.c_void_p), ("scale", ctypes.c_double),
        ("seqlen_q", ctypes.c_void_p), ("seqlen_k", ctypes.c_void_p),
    ]


def compile_source(src: str, out: str) -> str:
    """Compile a C source of the oracle's interface into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (OpenMP if available)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _bind(lib):
    """Declare the argument types of every entry point of a loaded build."""
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    pp = ctypes.POINTER(_Problem)
    lib.om_forward_rows.argtypes = [pp, vp, vp, vp, i64, vp, vp, vp]
    lib.om_delta.argtypes = [pp, vp, vp, vp]
    lib.om_dq_rows.argtypes = [pp, vp, vp, vp, vp, vp, vp, i64, vp, vp]
    lib.om_dkdv_cols.argtypes = [pp, vp, vp, vp, vp, vp, vp, i64, vp, vp, vp]
    lib.om_dsink.argtypes = [pp, vp, vp, vp]
    lib.om_mask_transpose.argtypes = [i64, i64, i64, vp, vp]
    lib.om_select_tables.argtypes = [i64, i64, i64, i64, i64, vp,
                                     i64, i64, vp, vp, i64, i64, vp, vp]
    lib.om_count_visible.argtypes = [pp]
    lib.om_count_visible.restype = ctypes.c_int64
    lib.om_num_threads.restype = ctypes.c_int
    return lib


def use_library(path: str) -> None:
    """Route every later call of this process to another build of oracle.c.

    Used by the mutation test, which compiles altered copies of the source in
    a child process and checks that each one fails at least one pin."""
    global _lib
    with _lock:
        _lib = _bind(ctypes.CDLL(path))


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def num_threads() -> int:
    return int(_load().om_num_threads())


def _f64(x) -> np.ndarray:
    """Exact widening of a torch tensor / array to a contiguous float64 array."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _u8(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.uint8)


def _ptr(a) -> Optional[int]:
    return None if a is None else a.ctypes.data


@dataclass
class Problem:
    """Shapes, mask and sink of one attention problem (BHSD, contiguous)."""
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int
    scale: float
    mask_kind: int = MASK_NONE
    window: int = 0
    bx: int = 1
    by: int = 1
    block_mask: Optional[np.ndarray] = None   # uint8 [B,Hq,nQB,nKB]
    token_mask: Optional[np.ndarray] = None   # uint8 [B,Hq,Sq,Skv]
    sink: Optional[np.ndarray] = None         # float64 [Hq] (may hold -inf)
    seqlen_q: Optional[np.ndarray] = None     # int [B]: valid query rows per batch
    seqlen_k: Optional[np.ndarray] = None     # int [B]: valid keys per batch

    def _c(self):
        self._bm = _u8(self.block_mask)
        self._tm = _u8(self.token_mask)
        self._sk = _f64(self.sink)
        self._lq = (np.ascontiguousarray(np.asarray(self.seqlen_q, dtype=np.int64))
                    if self.seqlen_q is not None else None)
        self._lk = (np.ascontiguousarray(np.asarray(self.seqlen_k, dtype=np.int64))
                    if self.seqlen_k is not None else None)
        for a in (self._lq, self._lk):
            assert a is None or a.size == self.B
        if self.mask_kind == MASK_BLOCK:
            nqb = -(-self.Sq // self.bx)
            nkb = -(-self.Skv // self.by)
            assert self._bm is not None and self._bm.size == self.B * self.Hq * nqb * nkb
        if self.mask_kind == MASK_TOKEN:
            assert self._tm is not None and self._tm.size == self.B * self.Hq * self.Sq * self.Skv
        assert self.Hq % self.Hkv == 0
        return ctypes.byref(_Problem(
            self.B, self.Hq, self.Hkv, self.Sq, self.Skv, self.D,
            self.mask_kind, self.window, self.bx, self.by,
            _ptr(self._bm), _ptr(self._tm), _ptr(self._sk), float(self.scale),
            _ptr(self._lq), _ptr(self._lk)))


def forward(pb: Problem, q, k, v, rows=None):
    """O [n,D] and LSE [n] for the given flat query rows (default: all rows).

    With rows=None the results are shaped [B,Hq,Sq,D] and [B,Hq,Sq].
    """
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    full = rows is None
    if full:
        rows = np.arange(pb.B * pb.Hq * pb.Sq, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    O = np.zeros((rows.size, pb.D), np.float64)
    LSE = np.zeros(rows.size, np.float64)
    lib.om_forward_rows(pb._c(), _ptr(q), _ptr(k), _ptr(v), rows.size,
                        _ptr(rows), _ptr(O), _ptr(LSE))
    if full:
        return O.reshape(pb.B, pb.Hq, pb.Sq, pb.D), LSE.reshape(pb.B, pb.Hq, pb.Sq)
    return O, LSE


def delta(pb: Problem, O_in, dO) -> np.ndarray:
    lib = _load()
    O_in, dO = _f64(O_in), _f64(dO)
    out = np.zeros(pb.B * pb.Hq * pb.Sq, np.float64)
    lib.om_delta(pb._c(), _ptr(O_in), _ptr(dO), _ptr(out))
    return out.reshape(pb.B, pb.Hq, pb.Sq)


def dq_rows(pb: Problem, q, k, v, dO, lse_in, delta_, rows) -> np.ndarray:
    lib = _load()
    q, k, v, dO, lse_in, delta_ = map(_f64, (q, k, v, dO, lse_in, delta_))
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, pb.D), np.float64)
    lib.om_dq_rows(pb._c(), _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse_in),
                   _ptr(delta_), rows.size, _ptr(rows), _ptr(out))
    return out


def dkdv_cols(pb: Problem, q, k, v, dO, lse_in, delta_, cols):
    lib = _load()
    q, k, v, dO, lse_in, delta_ = map(_f64, (q, k, v, dO, lse_in, delta_))
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    dK = np.zeros((cols.size, pb.D), np.float64)
    dV = np.zeros((cols.size, pb.D), np.float64)
    lib.om_dkdv_cols(pb._c(), _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse_in),
                     _ptr(delta_), cols.size, _ptr(cols), _ptr(dK), _ptr(dV))
    return dK, dV


def dsink(pb: Problem, lse_in, delta_) -> np.ndarray:
    lib = _load()
    lse_in, delta_ = _f64(lse_in), _f64(delta_)
    out = np.zeros(pb.Hq, np.float64)
    lib.om_dsink(pb._c(), _ptr(lse_in), _ptr(delta_), _ptr(out))
    return out


def backward(pb: Problem, q, k, v, O_in, dO, lse_in):
    """Full backward (parity mode: O_in and lse_in are taken as given).

    Returns dict with dq [B,Hq,Sq,D], dk, dv [B,Hkv,Skv,D], dsink [Hq],
    delta [B,Hq,Sq].
    """
    q, k, v, O_in, dO, lse_in = map(_f64, (q, k, v, O_in, dO, lse_in))
    dl = delta(pb, O_in, dO)
    rows = np.arange(pb.B * pb.Hq * pb.Sq, dtype=np.int64)
    cols = np.arange(pb.B * pb.Hkv * pb.Skv, dtype=np.int64)
    dQ = dq_rows(pb, q, k, v, dO, lse_in, dl, rows)
    dK, dV = dkdv_cols(pb, q, k, v, dO, lse_in, dl, cols)
    ds = dsink(pb, lse_in, dl)
    return {
        "dq": dQ.reshape(pb.B, pb.Hq, pb.Sq, pb.D),
        "dk": dK.reshape(pb.B, pb.Hkv, pb.Skv, pb.D),
        "dv": dV.reshape(pb.B, pb.Hkv, pb.Skv, pb.D),
        "dsink": ds,
        "delta": dl,
    }


def backward_exact(pb: Problem, q, k, v, dO):
    """Exact mode: the oracle's own fp64 O and LSE feed the backward."""
    O, lse = forward(pb, q, k, v)
    out = backward(pb, q, k, v, O, dO, lse)
    out["o"], out["lse"] = O, lse
    return out


def mask_transpose(mask: np.ndarray) -> np.ndarray:
    """uint8 [B,H,nQB,nKB] -> [B,H,nKB,nQB]."""
    lib = _load()
    m = _u8(mask)
    B, H, nqb, nkb = m.shape
    out = np.zeros((B, H, nkb, nqb), np.uint8)
    lib.om_mask_transpose(B * H, nqb, nkb, _ptr(m), _ptr(out))
    return out


def select_tables(mask, Sq: int, Skv: int, bx: int, by: int,
                  tq_k: int, tk_k: int, tq_q: int, tk_q: int):
    """Select tables for the kv-major (sel_k) and q-major (sel_q) walks.

    sel_k[b,h,kt,:cnt_k] lists ascending query tiles (size tq_k) that share an
    active mask block with key tile kt (size tk_k); sel_q is the transpose
    relation for query tiles of size tq_q and key tiles of size tk_q.  Unused
    entries are -1.
    """
    lib = _load()
    m = _u8(mask)
    B, H, nqb, nkb = m.shape
    assert nqb == -(-Sq // bx) and nkb == -(-Skv // by)
    nqt_k, nkt_k = -(-Sq // tq_k), -(-Skv // tk_k)
    nqt_q, nkt_q = -(-Sq // tq_q), -(-Skv // tk_q)
    sel_k = np.zeros((B, H, nkt_k, nqt_k), np.int32)
    cnt_k = np.zeros((B, H, nkt_k), np.int32)
    sel_q = np.zeros((B, H, nqt_q, nkt_q), np.int32)
    cnt_q = np.zeros((B, H, nqt_q), np.int32)
    lib.om_select_tables(B * H, Sq, Skv, bx, by, _ptr(m), tq_k, tk_k,
                         _ptr(sel_k), _ptr(cnt_k), tq_q, tk_q, _ptr(sel_q), _ptr(cnt_q))
    return sel_k, cnt_k, sel_q, cnt_q


def count_visible(pb: Problem) -> int:
    return int(_load().om_count_visible(pb._c()))


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)
