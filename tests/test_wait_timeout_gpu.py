"""The bounded waits end a call that cannot make progress with ATTN_ERR_TIMEOUT
in the workspace status, and the GPU context stays usable.

MASKATTN_TEST_NO_LOADS=1 makes the kernels' loader warps issue nothing, so
every other warp waits on barriers that nothing will complete, with no copy
or MMA in flight; MASKATTN_WAIT_TIMEOUT_NS shortens each wait to 20 ms.  The
next call, with the hook off, must give the oracle's gradients again.
"""
import pytest
import torch

import oracle
from masked_attention_backward_gb300 import binding as mab
from masked_attention_backward_gb300.workloads import MASK_BLOCK, MASK_CAUSAL, Workload, make_inputs
from parity import compare, forward_stats, gpu_mask, oracle_problem, run_gpu_bwd

pytestmark = pytest.mark.gpu

CASES = [
    Workload("stall_causal", "bf16", B=1, Hq=4, Hkv=1, Sq=300, Skv=300, mask_kind=MASK_CAUSAL,
             sink=True, seed=51),
    Workload("stall_blocks", "f16", B=1, Hq=2, Hkv=2, Sq=260, Skv=200, mask_kind=MASK_BLOCK,
             bx=64, by=64, block_pattern="random", density=0.5, seed=52),
]


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_wait_timeout_reported_and_recovered(cuda_lib, monkeypatch, wl):
    inp = make_inputs(wl)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    dev = "cuda"
    q, k, v, dO = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dO))
    o, l = O.to(dev), lse.to(dev)
    sink = inp.sink.to(dev) if inp.sink is not None else None
    mask = gpu_mask(wl, inp, dev)
    ws = mab.workspace(mab.shape_of(q, k), mask, dev)

    monkeypatch.setenv("MASKATTN_WAIT_TIMEOUT_NS", "20000000")
    monkeypatch.setenv("MASKATTN_TEST_NO_LOADS", "1")
    mab.bwd(q, k, v, o, dO, l, sink, mask, wl.scale, ws=ws)
    torch.cuda.synchronize()
    assert mab.device_status(ws) == mab.ATTN_ERR_TIMEOUT
    mab.fwd(q, k, v, sink, mask, wl.scale, ws=ws)
    torch.cuda.synchronize()
    assert mab.device_status(ws) == mab.ATTN_ERR_TIMEOUT

    monkeypatch.delenv("MASKATTN_TEST_NO_LOADS")
    monkeypatch.delenv("MASKATTN_WAIT_TIMEOUT_NS")
    # the same workspace: every call starts from a clean status
    dq, dk, dv, dsink = mab.bwd(q, k, v, o, dO, l, sink, mask, wl.scale, ws=ws)
    torch.cuda.synchronize()
    assert mab.device_status(ws) == mab.ATTN_OK
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        compare(name, t, ref[name], wl.dtype)
    run = run_gpu_bwd(wl, inp, O, lse)   # a fresh workspace too
    assert torch.equal(run.dq, dq) and torch.equal(run.dk, dk) and torch.equal(run.dv, dv)
