"""GPU parity of the single-pass backward (ATTN_FLAG_SINGLE_PASS): dq from the
key-stationary kernel's per-step partials, summed by the reduction kernel.

dq is checked against the fp64 oracle element by element on the same cases
as the split design; dk and dv come from the same contractions in the same
order as the split design's key-stationary kernel, so they must agree with it
bit for bit (and dsink too: the same preprocess kernel).  The reduction sums
in a fixed order, so two runs agree bit for bit.
"""
import pytest
import torch

import oracle
from masked_attention_backward_gb300 import binding as mab
from masked_attention_backward_gb300.workloads import (MASK_BLOCK, MASK_CAUSAL, MASK_SLIDING,
                                                        Workload, make_inputs)
from parity import (compare, forward_stats, full_parity, gpu_mask, oracle_problem, run_gpu_bwd)
from test_bwd_gpu import CASES

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_single_pass_parity(cuda_lib, wl):
    reps, run, _ = full_parity(wl, single_pass=True)
    print({r["name"]: (round(r["frac"], 6), r["max_err"]) for r in reps})
    inp = make_inputs(wl)
    O, lse = forward_stats(wl, inp)
    split = run_gpu_bwd(wl, inp, O, lse)
    assert torch.equal(run.dk, split.dk) and torch.equal(run.dv, split.dv)
    if run.dsink is not None:
        assert torch.equal(run.dsink, split.dsink)


@pytest.mark.parametrize("S", [1, 2, 63, 64, 65, 127, 128, 129])
def test_single_pass_tiny_lengths(cuda_lib, S):
    wl = Workload(f"causal_sink_S{S}", "bf16", B=1, Hq=4, Hkv=1, Sq=S, Skv=S,
                  mask_kind=MASK_CAUSAL, sink=True, seed=20 + S)
    full_parity(wl, single_pass=True)


def test_single_pass_deterministic(cuda_lib):
    wl = Workload("swa_gqa_det", "bf16", B=1, Hq=8, Hkv=2, Sq=1000, Skv=1000,
                  mask_kind=MASK_SLIDING, window=300, sink=True, seed=61)
    inp = make_inputs(wl)
    O, lse = forward_stats(wl, inp)
    a = run_gpu_bwd(wl, inp, O, lse, single_pass=True)
    b = run_gpu_bwd(wl, inp, O, lse, single_pass=True)
    assert torch.equal(a.dq, b.dq) and torch.equal(a.dk, b.dk) and torch.equal(a.dv, b.dv)


def test_single_pass_varlen(cuda_lib):
    # per-batch lengths on the padded layout: rows and keys past them get zeros
    wl = Workload("varlen_causal_sp", "bf16", B=3, Hq=4, Hkv=2, Sq=400, Skv=400,
                  mask_kind=MASK_CAUSAL, sink=True, seed=62)
    inp = make_inputs(wl)
    inp.seqlen_q = torch.tensor([400, 130, 1], dtype=torch.int32)
    inp.seqlen_k = torch.tensor([400, 257, 64], dtype=torch.int32)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    run = run_gpu_bwd(wl, inp, O, lse, single_pass=True)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name in ("dq", "dk", "dv"):
        compare(name, getattr(run, name), ref[name], wl.dtype)
    compare("dsink", run.dsink, ref["dsink"], wl.dtype, min_frac=1.0)
    assert torch.all(run.dq[1, :, 130:].cpu() == 0) and torch.all(run.dq[2, :, 1:].cpu() == 0)
    assert torch.all(run.dk[1, :, 257:].cpu() == 0) and torch.all(run.dv[2, :, 64:].cpu() == 0)


def test_single_pass_empty_rows_and_key_tiles(cuda_lib):
    wl = Workload("holes_sp", "f16", B=1, Hq=2, Hkv=2, Sq=400, Skv=400, mask_kind=MASK_BLOCK,
                  bx=64, by=64, block_pattern="ones", seed=31)
    inp = make_inputs(wl)
    inp.block_mask[0, 1, 2, :] = 0
    inp.block_mask[0, 1, :, 4:] = 0
    inp.block_mask[0, 0, :, :] = 0
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    run = run_gpu_bwd(wl, inp, O, lse, single_pass=True)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name in ("dq", "dk", "dv"):
        compare(name, getattr(run, name), ref[name], wl.dtype)
    assert torch.all(run.dq[0, 1, 128:192].cpu() == 0)
    assert torch.all(run.dq[0, 0].cpu() == 0)


def test_single_pass_timeout_reported_and_recovered(cuda_lib, monkeypatch):
    """A call whose waits run out reports ATTN_ERR_TIMEOUT and writes zeros
    (no partial of it is summed); the next call on the same workspace is
    correct again."""
    wl = Workload("stall_sp", "bf16", B=1, Hq=4, Hkv=1, Sq=300, Skv=300, mask_kind=MASK_CAUSAL,
                  sink=True, seed=53)
    inp = make_inputs(wl)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    dev = "cuda"
    q, k, v, dO = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dO))
    o, l = O.to(dev), lse.to(dev)
    sink = inp.sink.to(dev)
    mask = gpu_mask(wl, inp, dev)
    ws = mab.workspace(mab.shape_of(q, k, mab.ATTN_FLAG_SINGLE_PASS), mask, dev)
    monkeypatch.setenv("MASKATTN_WAIT_TIMEOUT_NS", "20000000")
    monkeypatch.setenv("MASKATTN_TEST_NO_LOADS", "1")
    dq, dk, dv, _ = mab.bwd(q, k, v, o, dO, l, sink, mask, wl.scale, ws=ws, single_pass=True)
    torch.cuda.synchronize()
    assert mab.device_status(ws) == mab.ATTN_ERR_TIMEOUT
    assert torch.all(dq == 0) and torch.all(dk == 0) and torch.all(dv == 0)
    monkeypatch.delenv("MASKATTN_TEST_NO_LOADS")
    monkeypatch.delenv("MASKATTN_WAIT_TIMEOUT_NS")
    dq, dk, dv, _ = mab.bwd(q, k, v, o, dO, l, sink, mask, wl.scale, ws=ws, single_pass=True)
    torch.cuda.synchronize()
    assert mab.device_status(ws) == mab.ATTN_OK
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        compare(name, t, ref[name], wl.dtype)


def test_single_pass_rejects_unsupported_combinations(cuda_lib):
    wl = Workload("c", "bf16", B=1, Hq=2, Hkv=1, Sq=128, Skv=128, mask_kind=MASK_CAUSAL, seed=1)
    inp = make_inputs(wl)
    O, lse = forward_stats(wl, inp)
    with pytest.raises(mab.AttnError) as e:
        run_gpu_bwd(wl, inp, O, lse, compensated=True, single_pass=True)
    assert e.value.code == mab.ATTN_ERR_UNSUPPORTED
