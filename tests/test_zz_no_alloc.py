"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Callers such as operator or plugin interfaces that receive only their input
and output buffers (no workspace), or services that forbid device allocation
once running, use attn_bwd_noalloc, which keeps its scratch in a fixed array
inside the library.  These tests call it through the C ABI and check it
against attn_bwd with a caller-allocated workspace, under the same tolerance
gate as the other parity tests, on two calls in a row with different masks
and shapes (so that anything the first call left in the shared array would
show up in the second).  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from masked_attention_backward_gb300 import binding as mab
from masked_attention_backward_gb300.workloads import (MASK_BLOCK, MASK_SLIDING, Workload,
                                                        make_inputs)
from parity import compare, forward_stats, gpu_mask

pytestmark = pytest.mark.gpu

CALLS = [
    Workload("noalloc_blocks_f16", "f16", B=1, Hq=4, Hkv=2, Sq=333, Skv=290, mask_kind=MASK_BLOCK,
             bx=48, by=80, block_pattern="random", density=0.4, sink=True, seed=71),
    Workload("noalloc_swa_bf16", "bf16", B=2, Hq=4, Hkv=1, Sq=300, Skv=300,
             mask_kind=MASK_SLIDING, window=90, sink=True, seed=72),
]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _device_case(wl):
    inp = make_inputs(wl)
    O, lse = forward_stats(wl, inp)
    dev = "cuda"
    t = {n: x.to(dev) for n, x in (("q", inp.q), ("k", inp.k), ("v", inp.v), ("o", O),
                                   ("dO", inp.dO), ("lse", lse))}
    t["sink"] = inp.sink.to(dev)
    return t, gpu_mask(wl, inp, dev)


def _outputs(t):
    outs = [torch.full_like(t["q"], float("nan")), torch.full_like(t["k"], float("nan")),
            torch.full_like(t["v"], float("nan")), torch.full_like(t["sink"], float("nan"))]
    return outs


def test_noalloc_matches_workspace_backward_on_two_calls(cuda_lib):
    for wl in CALLS:
        t, mask = _device_case(wl)
        shape = mab.shape_of(t["q"], t["k"])
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        # reference: the existing entry point with a caller workspace
        ref = _outputs(t)
        ws = mab.workspace(shape, mask, "cuda")
        r = mab.attn_bwd(shape, _ptr(t["q"]), _ptr(t["k"]), _ptr(t["v"]), _ptr(t["o"]),
                         _ptr(t["dO"]), _ptr(t["lse"]), _ptr(t["sink"]), mask.desc(), wl.scale,
                         _ptr(ref[0]), _ptr(ref[1]), _ptr(ref[2]), _ptr(ref[3]), _ptr(ws),
                         ws.numel(), stream)
        assert r == mab.ATTN_OK, mab.attn_status_string(r)
        # the allocation-free entry point
        got = _outputs(t)
        r = mab.attn_bwd_noalloc(shape, _ptr(t["q"]), _ptr(t["k"]), _ptr(t["v"]), _ptr(t["o"]),
                                 _ptr(t["dO"]), _ptr(t["lse"]), _ptr(t["sink"]), mask.desc(),
                                 wl.scale, _ptr(got[0]), _ptr(got[1]), _ptr(got[2]),
                                 _ptr(got[3]), stream)
        assert r == mab.ATTN_OK, mab.attn_status_string(r)
        torch.cuda.synchronize()
        st = mab.attn_noalloc_get_device_status(stream)
        assert st == mab.ATTN_OK, mab.attn_status_string(st)
        for name, a, b in zip(("dq", "dk", "dv", "dsink"), got, ref):
            compare(name, a, b.double().cpu().numpy(), wl.dtype,
                    min_frac=1.0 if name == "dsink" else 0.999)


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_lib):
    # B*Hq*S rows of statistics well past 32 MiB of scratch; rejected on the
    # host before anything is enqueued, so the addresses are never touched
    shape = mab.attn_shape_t(1, 64, 8, 131072, 131072, 128, mab.ATTN_BF16)
    mask = mab.attn_mask_desc_t(mab.ATTN_MASK_CAUSAL, 0, 1, 1, None)
    fake = ctypes.c_void_p(0x7F0000000000)
    r = mab.attn_bwd_noalloc(shape, fake, fake, fake, fake, fake, fake, None, mask, 0.088, fake,
                             fake, fake, None, None)
    assert r == mab.ATTN_ERR_WORKSPACE


def _noalloc_call(shape, t, mask, scale, outs, stream):
    return mab.attn_bwd_noalloc(shape, _ptr(t["q"]), _ptr(t["k"]), _ptr(t["v"]), _ptr(t["o"]),
                                _ptr(t["dO"]), _ptr(t["lse"]), _ptr(t["sink"]), mask.desc(),
                                scale, _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]),
                                _ptr(outs[3]), stream)


def test_noalloc_largest_accepted_shape(cuda_lib):
    # a long sliding-window problem whose scratch is just under the 32 MiB
    # limit (the per-row statistics grow with B * Hq * S): accepted, and the
    # same gradients as attn_bwd with a caller workspace
    limit = 32 << 20
    B, Hq, Hkv, W = 2, 16, 2, 128
    mask = mab.Mask(kind=mab.ATTN_MASK_SLIDING, window=W)
    S = 131072
    while True:
        shape = mab.attn_shape_t(B, Hq, Hkv, S, S, 128, mab.ATTN_BF16)
        r, need = mab.attn_workspace_size(shape, mask.desc())
        assert r == mab.ATTN_OK
        if need <= limit:
            break
        S -= 128
    assert need > limit - (1 << 20), need
    g = torch.Generator(device="cuda").manual_seed(7)
    dev = "cuda"
    t = {"q": torch.randn(B, Hq, S, 128, generator=g, device=dev).to(torch.bfloat16),
         "k": torch.randn(B, Hkv, S, 128, generator=g, device=dev).to(torch.bfloat16),
         "v": torch.randn(B, Hkv, S, 128, generator=g, device=dev).to(torch.bfloat16),
         "dO": torch.randn(B, Hq, S, 128, generator=g, device=dev).to(torch.bfloat16),
         "sink": torch.randn(Hq, generator=g, device=dev)}
    scale = 128 ** -0.5
    t["o"], t["lse"] = mab.fwd(t["q"], t["k"], t["v"], t["sink"], mask, scale)
    ref = mab.bwd(t["q"], t["k"], t["v"], t["o"], t["dO"], t["lse"], t["sink"], mask, scale)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    got = _outputs(t)
    r = _noalloc_call(shape, t, mask, scale, got, stream)
    assert r == mab.ATTN_OK, mab.attn_status_string(r)
    torch.cuda.synchronize()
    assert mab.attn_noalloc_get_device_status(stream) == mab.ATTN_OK
    for name, a, b in zip(("dq", "dk", "dv", "dsink"), got, ref):
        assert torch.equal(a, b), name
    # one row more per sequence crosses the limit
    big = mab.attn_shape_t(B, Hq, Hkv, S + 128, S + 128, 128, mab.ATTN_BF16)
    assert mab.attn_workspace_size(big, mask.desc())[1] > limit
    fake = ctypes.c_void_p(0x7F0000000000)
    r = mab.attn_bwd_noalloc(big, fake, fake, fake, fake, fake, fake, fake, mask.desc(), scale,
                             fake, fake, fake, fake, stream)
    assert r == mab.ATTN_ERR_WORKSPACE


def test_noalloc_wait_timeout_is_readable(cuda_lib, monkeypatch):
    # with the loader warps idle every device wait runs out: the status word in
    # the library's scratch says so, and the next call clears it
    wl = CALLS[1]
    t, mask = _device_case(wl)
    shape = mab.shape_of(t["q"], t["k"])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    monkeypatch.setenv("MASKATTN_WAIT_TIMEOUT_NS", "20000000")
    monkeypatch.setenv("MASKATTN_TEST_NO_LOADS", "1")
    assert _noalloc_call(shape, t, mask, wl.scale, _outputs(t), stream) == mab.ATTN_OK
    torch.cuda.synchronize()
    assert mab.attn_noalloc_get_device_status(stream) == mab.ATTN_ERR_TIMEOUT
    monkeypatch.delenv("MASKATTN_TEST_NO_LOADS")
    monkeypatch.delenv("MASKATTN_WAIT_TIMEOUT_NS")
    got = _outputs(t)
    assert _noalloc_call(shape, t, mask, wl.scale, got, stream) == mab.ATTN_OK
    torch.cuda.synchronize()
    assert mab.attn_noalloc_get_device_status(stream) == mab.ATTN_OK
    ref = mab.bwd(t["q"], t["k"], t["v"], t["o"], t["dO"], t["lse"], t["sink"], mask, wl.scale)
    for name, a, b in zip(("dq", "dk", "dv", "dsink"), got, ref):
        assert torch.equal(a, b), name
