"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before anything is
enqueued (so the fake device addresses below are never dereferenced)."""
import ctypes
import os
import re

import pytest

from masked_attention_backward_gb300 import binding as mab
from masked_attention_backward_gb300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Aligned addresses that are never touched: every call below fails validation first.
FAKE = ctypes.c_void_p(0x7F0000000000)
MISALIGNED = ctypes.c_void_p(0x7F0000000008)


@pytest.fixture(scope="module")
def lib():
    return mab.load()


def _shape(B=1, Hq=4, Hkv=2, Sq=256, Skv=256, D=128, dtype=mab.ATTN_BF16, flags=0):
    return mab.attn_shape_t(B, Hq, Hkv, Sq, Skv, D, dtype, flags)


def test_exports_every_declared_symbol(lib):
    hdr = open(os.path.join(ROOT, "include", "maskattn.h")).read()
    declared = set(re.findall(r"^\s*(?:attn_status_t|const char\*)\s+(attn_\w+)\s*\(", hdr, re.M))
    assert declared == set(mab.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in enumerate(["ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED",
                                 "ATTN_ERR_WORKSPACE", "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT"]):
        assert mab.attn_status_string(code) == name


@pytest.mark.parametrize("shape,mask,want", [
    (_shape(D=64), mab.attn_mask_desc_t(0, 0, 1, 1, None), mab.ATTN_ERR_UNSUPPORTED),
    (_shape(Hq=6, Hkv=4), mab.attn_mask_desc_t(0, 0, 1, 1, None), mab.ATTN_ERR_INVALID_ARG),
    (_shape(Sq=0), mab.attn_mask_desc_t(0, 0, 1, 1, None), mab.ATTN_ERR_INVALID_ARG),
    (_shape(Sq=100, Skv=120), mab.attn_mask_desc_t(1, 0, 1, 1, None), mab.ATTN_ERR_INVALID_ARG),
    (_shape(), mab.attn_mask_desc_t(2, 0, 1, 1, None), mab.ATTN_ERR_INVALID_ARG),
    (_shape(), mab.attn_mask_desc_t(3, 0, 0, 16, None), mab.ATTN_ERR_INVALID_ARG),
    (_shape(), mab.attn_mask_desc_t(7, 0, 1, 1, None), mab.ATTN_ERR_INVALID_ARG),
    (_shape(dtype=5), mab.attn_mask_desc_t(0, 0, 1, 1, None), mab.ATTN_ERR_INVALID_ARG),
    (_shape(flags=4), mab.attn_mask_desc_t(0, 0, 1, 1, None), mab.ATTN_ERR_INVALID_ARG),
    (_shape(flags=mab.ATTN_FLAG_SINGLE_PASS), mab.attn_mask_desc_t(1, 0, 1, 1, None), mab.ATTN_OK),
    # the single-pass kernels have no compensated and no packed form
    (_shape(flags=mab.ATTN_FLAG_SINGLE_PASS | mab.ATTN_FLAG_COMPENSATED),
     mab.attn_mask_desc_t(1, 0, 1, 1, None), mab.ATTN_ERR_UNSUPPORTED),
    (_shape(flags=mab.ATTN_FLAG_SINGLE_PASS),
     mab.attn_mask_desc_t(0, 0, 1, 1, None, None, None, 4096, 8192, 100, 90),
     mab.ATTN_ERR_UNSUPPORTED),
    (_shape(flags=-1), mab.attn_mask_desc_t(0, 0, 1, 1, None), mab.ATTN_ERR_INVALID_ARG),
    (_shape(flags=mab.ATTN_FLAG_COMPENSATED), mab.attn_mask_desc_t(1, 0, 1, 1, None), mab.ATTN_OK),
    (_shape(B=1024, Hq=128, Hkv=128), mab.attn_mask_desc_t(0, 0, 1, 1, None),
     mab.ATTN_ERR_INVALID_ARG),
    # per-batch length arrays must be 4-byte aligned
    (_shape(), mab.attn_mask_desc_t(0, 0, 1, 1, None, 4098, None), mab.ATTN_ERR_INVALID_ARG),
    (_shape(), mab.attn_mask_desc_t(0, 0, 1, 1, None, None, 4097), mab.ATTN_ERR_INVALID_ARG),
    # packed layout: both offset arrays, aligned, no per-batch lengths beside
    # them, and token totals of at least one
    (_shape(), mab.attn_mask_desc_t(0, 0, 1, 1, None, None, None, 4096, 8192, 100, 90),
     mab.ATTN_OK),
    (_shape(), mab.attn_mask_desc_t(0, 0, 1, 1, None, None, None, 4096, None, 100, 90),
     mab.ATTN_ERR_INVALID_ARG),
    (_shape(), mab.attn_mask_desc_t(0, 0, 1, 1, None, None, None, None, 8192, 100, 90),
     mab.ATTN_ERR_INVALID_ARG),
    (_shape(), mab.attn_mask_desc_t(0, 0, 1, 1, None, 4096, None, 4096, 8192, 100, 90),
     mab.ATTN_ERR_INVALID_ARG),
    (_shape(), mab.attn_mask_desc_t(0, 0, 1, 1, None, None, None, 4098, 8192, 100, 90),
     mab.ATTN_ERR_INVALID_ARG),
    (_shape(), mab.attn_mask_desc_t(0, 0, 1, 1, None, None, None, 4096, 8192, 0, 90),
     mab.ATTN_ERR_INVALID_ARG),
    (_shape(), mab.attn_mask_desc_t(0, 0, 1, 1, None, None, None, 4096, 8192, 100, -1),
     mab.ATTN_ERR_INVALID_ARG),
])
def test_workspace_size_validation(lib, shape, mask, want):
    r, _ = mab.attn_workspace_size(shape, mask)
    assert r == want


def test_workspace_size_matches_layout(lib):
    from parity import ws_layout
    for wl in WORKLOADS:
        shape = mab.attn_shape_t(wl.B, wl.Hq, wl.Hkv, wl.Sq, wl.Skv, wl.D,
                                 mab.ATTN_F16 if wl.dtype == "f16" else mab.ATTN_BF16)
        mask = mab.attn_mask_desc_t(wl.mask_kind, wl.window, wl.bx, wl.by, None)
        r, n = mab.attn_workspace_size(shape, mask)
        assert r == mab.ATTN_OK
        assert n == ws_layout(wl)["total"], wl.name


def test_single_pass_workspace_size(lib):
    """The single-pass regions: one flag byte and one 64 x 128 fp32 partial
    per (query head, key tile, query sub-tile) pair that holds a visible pair
    (counted from the mask's definition), every pair for block masks."""
    from parity import single_pass_steps_head, ws_layout
    from masked_attention_backward_gb300.workloads import Workload
    extra = [
        Workload("causal_ragged", "bf16", B=2, Hq=4, Hkv=2, Sq=333, Skv=333, mask_kind=1),
        Workload("swa1", "f16", B=1, Hq=2, Hkv=1, Sq=300, Skv=300, mask_kind=2, window=1),
        Workload("swa100", "bf16", B=1, Hq=2, Hkv=1, Sq=1000, Skv=1000, mask_kind=2, window=100),
        Workload("dense_uneven", "f16", B=1, Hq=2, Hkv=1, Sq=200, Skv=333, mask_kind=0),
    ]
    for wl in list(WORKLOADS) + extra:
        flags = mab.ATTN_FLAG_SINGLE_PASS
        shape = mab.attn_shape_t(wl.B, wl.Hq, wl.Hkv, wl.Sq, wl.Skv, wl.D,
                                 mab.ATTN_F16 if wl.dtype == "f16" else mab.ATTN_BF16, flags)
        mask = mab.attn_mask_desc_t(wl.mask_kind, wl.window, wl.bx, wl.by, None)
        r, n = mab.attn_workspace_size(shape, mask)
        assert r == mab.ATTN_OK
        L = ws_layout(wl, single_pass=True)
        assert n == L["total"], wl.name
        assert L["total"] - ws_layout(wl)["total"] >= \
            wl.B * wl.Hq * single_pass_steps_head(wl) * (64 * 128 * 4 + 1)
    # the causal count in closed form: key tile t meets the sub-tiles from 2t on
    wl = WORKLOADS[4]
    nkt, nqt = wl.Skv // 128, wl.Sq // 64
    assert single_pass_steps_head(wl) == sum(nqt - 2 * t for t in range(nkt))


def _bwd(shape, mask, ws_bytes=1 << 30, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, dO=FAKE, lse=FAKE, sink=None, dq=FAKE, dk=FAKE,
                dv=FAKE, dsink=None, ws=FAKE)
    args.update(over)
    return mab.attn_bwd(shape, args["q"], args["k"], args["v"], args["o"], args["dO"], args["lse"],
                        args["sink"], mask, 0.088, args["dq"], args["dk"], args["dv"],
                        args["dsink"], args["ws"], ws_bytes, None)


def test_bwd_argument_errors(lib):
    shape, mask = _shape(), mab.attn_mask_desc_t(1, 0, 1, 1, None)
    assert _bwd(shape, mask, q=None) == mab.ATTN_ERR_INVALID_ARG
    assert _bwd(shape, mask, dv=None) == mab.ATTN_ERR_INVALID_ARG
    assert _bwd(shape, mask, q=MISALIGNED) == mab.ATTN_ERR_INVALID_ARG
    assert _bwd(shape, mask, sink=FAKE, dsink=None) == mab.ATTN_ERR_INVALID_ARG
    assert _bwd(shape, mask, ws_bytes=1024) == mab.ATTN_ERR_WORKSPACE
    assert _bwd(_shape(D=64), mask) == mab.ATTN_ERR_UNSUPPORTED
    blk = mab.attn_mask_desc_t(3, 0, 16, 16, None)
    assert _bwd(shape, blk) == mab.ATTN_ERR_INVALID_ARG  # block mask pointer missing


def test_fwd_argument_errors(lib):
    shape, mask = _shape(), mab.attn_mask_desc_t(0, 0, 1, 1, None)
    r = mab.attn_fwd(shape, FAKE, FAKE, None, None, mask, 0.088, FAKE, FAKE, FAKE, 1 << 30, None)
    assert r == mab.ATTN_ERR_INVALID_ARG
    r = mab.attn_fwd(shape, FAKE, FAKE, FAKE, None, mask, 0.088, FAKE, FAKE, FAKE, 16, None)
    assert r == mab.ATTN_ERR_WORKSPACE


def test_visible_pair_count_matches_oracle():
    import numpy as np
    import oracle
    from masked_attention_backward_gb300 import measure
    from masked_attention_backward_gb300.workloads import Workload, make_inputs
    cases = [Workload("c", "f16", 2, 3, 1, 37, 37, 8, mask_kind=1),
             Workload("s", "f16", 1, 2, 2, 41, 41, 8, mask_kind=2, window=6),
             Workload("s2", "f16", 1, 2, 2, 5, 5, 8, mask_kind=2, window=9),
             Workload("n", "f16", 1, 2, 1, 13, 29, 8, mask_kind=0),
             Workload("b", "f16", 2, 2, 2, 50, 70, 8, mask_kind=3, bx=6, by=9,
                      block_pattern="random", density=0.4, seed=3),
             # variable lengths (lengths 0 .. S drawn by the workload generator)
             Workload("cv", "f16", 5, 3, 1, 37, 37, 8, mask_kind=1, varlen=True, seed=4),
             Workload("sv", "f16", 4, 2, 2, 41, 41, 8, mask_kind=2, window=6, varlen=True,
                      seed=5),
             Workload("nv", "f16", 4, 2, 1, 13, 29, 8, mask_kind=0, varlen=True, seed=6),
             Workload("bv", "f16", 4, 2, 2, 50, 70, 8, mask_kind=3, bx=6, by=9,
                      block_pattern="random", density=0.4, varlen=True, seed=7)]
    for wl in cases:
        inp = make_inputs(wl)
        pb = oracle.Problem(B=wl.B, Hq=wl.Hq, Hkv=wl.Hkv, Sq=wl.Sq, Skv=wl.Skv, D=wl.D,
                            scale=wl.scale, mask_kind=wl.mask_kind, window=wl.window, bx=wl.bx,
                            by=wl.by, block_mask=None if inp.block_mask is None
                            else inp.block_mask.numpy(),
                            seqlen_q=None if inp.seqlen_q is None else inp.seqlen_q.numpy(),
                            seqlen_k=None if inp.seqlen_k is None else inp.seqlen_k.numpy())
        assert (measure.visible_pairs(wl, inp.block_mask, inp.seqlen_q, inp.seqlen_k)
                == oracle.count_visible(pb)), wl.name


def test_host_pipeline_runs_validation():
    # uneven runs must cover the key/value heads exactly (checked before any allocation)
    for runs in ([1, 2], [2, 2, 1], [0, 4], [-1, 5]):
        with pytest.raises(ValueError):
            mab.HostBackward(1, 8, 4, 64, 64, None, mab.Mask(), 0.088, False, "cpu",
                             chunks=runs)
