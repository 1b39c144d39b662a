"""GPU parity of the persistent dK/dV kernel (k_dkdv_units), which the library
picks for short walks on the BHSD layout; MASKATTN_DKDV_SCHEDULE forces it
(or the per-tile kernel) on any shape.

Both forms run the same contractions in the same order, so dK and dV must
agree bit for bit; each is also gated against the fp64 oracle.  The shapes
with more units than the GPU has SMs make CTAs claim several units in turn.
"""
import pytest
import torch

import oracle
from masked_attention_backward_gb300 import binding as mab
from masked_attention_backward_gb300.workloads import (MASK_BLOCK, MASK_CAUSAL, MASK_SLIDING,
                                                        Workload, make_inputs)
from parity import compare, forward_stats, gpu_mask, oracle_problem, run_gpu_bwd
from test_bwd_gpu import CASES

pytestmark = pytest.mark.gpu

MANY_UNITS = [
    # 16 key tiles x 16 (b, kv head) = 256 units
    Workload("swa128_units256", "bf16", B=4, Hq=8, Hkv=4, Sq=2048, Skv=2048,
             mask_kind=MASK_SLIDING, window=128, sink=True, seed=71),
    # 12 x 16 = 192 units, one query head per kv head
    Workload("random30_units192", "f16", B=1, Hq=16, Hkv=16, Sq=1500, Skv=1500,
             mask_kind=MASK_BLOCK, bx=64, by=64, block_pattern="random", density=0.3, seed=72),
]


def _run_both(monkeypatch, wl, inp, O, lse, **kw):
    monkeypatch.setenv("MASKATTN_DKDV_SCHEDULE", "units")
    units = run_gpu_bwd(wl, inp, O, lse, **kw)
    monkeypatch.setenv("MASKATTN_DKDV_SCHEDULE", "tile")
    tile = run_gpu_bwd(wl, inp, O, lse, **kw)
    monkeypatch.delenv("MASKATTN_DKDV_SCHEDULE")
    return units, tile


@pytest.mark.parametrize("wl", CASES + MANY_UNITS, ids=[w.name for w in CASES + MANY_UNITS])
def test_units_parity_and_equal_to_tile(cuda_lib, monkeypatch, wl):
    inp = make_inputs(wl)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    units, tile = _run_both(monkeypatch, wl, inp, O, lse)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name in ("dq", "dk", "dv"):
        compare(name, getattr(units, name), ref[name], wl.dtype)
    if inp.sink is not None:
        compare("dsink", units.dsink, ref["dsink"], wl.dtype, min_frac=1.0)
        assert torch.equal(units.dsink, tile.dsink)
    assert torch.equal(units.dk, tile.dk) and torch.equal(units.dv, tile.dv)
    assert torch.equal(units.dq, tile.dq)


@pytest.mark.parametrize("S", [1, 63, 64, 65, 128, 129, 300])
def test_units_tiny_lengths(cuda_lib, monkeypatch, S):
    wl = Workload(f"causal_sink_S{S}", "bf16", B=2, Hq=4, Hkv=2, Sq=S, Skv=S,
                  mask_kind=MASK_CAUSAL, sink=True, seed=30 + S)
    inp = make_inputs(wl)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    units, tile = _run_both(monkeypatch, wl, inp, O, lse)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name in ("dq", "dk", "dv"):
        compare(name, getattr(units, name), ref[name], wl.dtype)
    assert torch.equal(units.dk, tile.dk) and torch.equal(units.dv, tile.dv)


def test_units_varlen_and_empty_key_tiles(cuda_lib, monkeypatch):
    # per-batch lengths leave whole key tiles without steps (zeros) between
    # units with steps, in the same CTA's sequence of units
    wl = Workload("varlen_swa_units", "f16", B=3, Hq=4, Hkv=2, Sq=700, Skv=700,
                  mask_kind=MASK_SLIDING, window=90, sink=True, seed=73)
    inp = make_inputs(wl)
    inp.seqlen_q = torch.tensor([700, 129, 0], dtype=torch.int32)
    inp.seqlen_k = torch.tensor([650, 300, 5], dtype=torch.int32)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    units, tile = _run_both(monkeypatch, wl, inp, O, lse)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name in ("dq", "dk", "dv"):
        compare(name, getattr(units, name), ref[name], wl.dtype)
    compare("dsink", units.dsink, ref["dsink"], wl.dtype, min_frac=1.0)
    assert torch.equal(units.dk, tile.dk) and torch.equal(units.dv, tile.dv)
    assert torch.all(units.dk[1, :, 300:].cpu() == 0) and torch.all(units.dv[2].cpu() == 0)


COMPENSATED = [
    Workload("swa_comp_units", "f16", B=1, Hq=4, Hkv=2, Sq=600, Skv=600,
             mask_kind=MASK_SLIDING, window=128, sink=True, seed=74),
    # 64 x 64 blocks: whole softmax-warp regions masked (zero high and low parts)
    Workload("blocks_comp_units", "f16", B=1, Hq=4, Hkv=4, Sq=700, Skv=650,
             mask_kind=MASK_BLOCK, bx=64, by=64, block_pattern="random", density=0.35,
             sink=True, seed=75),
]


@pytest.mark.parametrize("wl", COMPENSATED, ids=[w.name for w in COMPENSATED])
def test_units_compensated_equal_to_tile(cuda_lib, monkeypatch, wl):
    inp = make_inputs(wl)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    units, tile = _run_both(monkeypatch, wl, inp, O, lse, compensated=True)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name in ("dk", "dv"):
        compare(name, getattr(units, name), ref[name], wl.dtype)
    assert torch.equal(units.dk, tile.dk) and torch.equal(units.dv, tile.dv)


def test_units_timeout_reported_and_recovered(cuda_lib, monkeypatch):
    wl = MANY_UNITS[0]
    inp = make_inputs(wl)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    dev = "cuda"
    q, k, v, dO = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dO))
    o, l = O.to(dev), lse.to(dev)
    sink = inp.sink.to(dev)
    mask = gpu_mask(wl, inp, dev)
    ws = mab.workspace(mab.shape_of(q, k), mask, dev)
    monkeypatch.setenv("MASKATTN_DKDV_SCHEDULE", "units")
    monkeypatch.setenv("MASKATTN_WAIT_TIMEOUT_NS", "20000000")
    monkeypatch.setenv("MASKATTN_TEST_NO_LOADS", "1")
    mab.bwd(q, k, v, o, dO, l, sink, mask, wl.scale, ws=ws)
    torch.cuda.synchronize()
    assert mab.device_status(ws) == mab.ATTN_ERR_TIMEOUT
    monkeypatch.delenv("MASKATTN_TEST_NO_LOADS")
    monkeypatch.delenv("MASKATTN_WAIT_TIMEOUT_NS")
    dq, dk, dv, dsink = mab.bwd(q, k, v, o, dO, l, sink, mask, wl.scale, ws=ws)
    torch.cuda.synchronize()
    assert mab.device_status(ws) == mab.ATTN_OK
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        compare(name, t, ref[name], wl.dtype)
