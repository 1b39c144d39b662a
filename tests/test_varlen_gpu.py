"""GPU parity of the variable-length batch (per-batch valid lengths on the
padded BHSD layout) against the fp64 oracle, forward and backward.

Rows past a batch element's query length and keys past its key length are
outside the problem: O = 0 and LSE = +inf, dQ = 0, dK = dV = 0, no part in
dSink -- exactly, not within a tolerance.  Lengths include 0, 1, lengths that
end inside a tile, and the full length; one case has more (head, query tile)
units than SMs.
"""
import numpy as np
import pytest
import torch

import oracle
from masked_attention_backward_gb300 import binding as mab
from masked_attention_backward_gb300.workloads import (MASK_BLOCK, MASK_CAUSAL, MASK_NONE,
                                                        MASK_SLIDING, Workload, make_inputs)
from parity import compare, forward_stats, gpu_mask, oracle_problem, run_gpu_bwd

pytestmark = pytest.mark.gpu

CASES = [
    (Workload("vl_causal_bf16", "bf16", B=4, Hq=4, Hkv=2, Sq=300, Skv=300,
              mask_kind=MASK_CAUSAL, sink=True, seed=61), [0, 1, 130, 300], None),
    (Workload("vl_swa_f16", "f16", B=3, Hq=2, Hkv=1, Sq=257, Skv=257, mask_kind=MASK_SLIDING,
              window=100, sink=True, seed=62), [65, 257, 200], None),
    (Workload("vl_dense_f16", "f16", B=2, Hq=2, Hkv=2, Sq=200, Skv=333, mask_kind=MASK_NONE,
              seed=63), [0, 150], [17, 333]),
    (Workload("vl_blocks_bf16", "bf16", B=2, Hq=2, Hkv=1, Sq=260, Skv=190, mask_kind=MASK_BLOCK,
              bx=32, by=48, block_pattern="random", density=0.4, sink=True, seed=64),
     [259, 70], [190, 100]),
    (Workload("vl_claims_bf16", "bf16", B=4, Hq=8, Hkv=2, Sq=700, Skv=700,
              mask_kind=MASK_CAUSAL, sink=True, seed=65), [700, 333, 1, 512], None),
]
IDS = [c[0].name for c in CASES]


def _inputs(wl, lq, lk):
    inp = make_inputs(wl)
    inp.seqlen_q = torch.tensor(lq, dtype=torch.int32)
    inp.seqlen_k = torch.tensor(lk if lk is not None else lq, dtype=torch.int32)
    return inp


@pytest.mark.parametrize("wl,lq,lk", CASES, ids=IDS)
def test_varlen_bwd_parity(cuda_lib, wl, lq, lk):
    inp = _inputs(wl, lq, lk)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    run = run_gpu_bwd(wl, inp, O, lse)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name in ("dq", "dk", "dv"):
        compare(name, getattr(run, name), ref[name], wl.dtype)
    if inp.sink is not None:
        compare("dsink", run.dsink, ref["dsink"], wl.dtype, min_frac=1.0)
    for b in range(wl.B):
        Lq, Lk = int(inp.seqlen_q[b]), int(inp.seqlen_k[b])
        assert torch.all(run.dq[b, :, Lq:].cpu() == 0)
        assert torch.all(run.dk[b, :, Lk:].cpu() == 0) and torch.all(run.dv[b, :, Lk:].cpu() == 0)


@pytest.mark.parametrize("wl,lq,lk", CASES, ids=IDS)
def test_varlen_fwd_parity(cuda_lib, wl, lq, lk):
    inp = _inputs(wl, lq, lk)
    pb = oracle_problem(wl, inp)
    O_ref, lse_ref = oracle.forward(pb, inp.q, inp.k, inp.v)
    dev = "cuda"
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    sink = inp.sink.to(dev) if inp.sink is not None else None
    o, lse = mab.fwd(q, k, v, sink, gpu_mask(wl, inp, dev), wl.scale)
    torch.cuda.synchronize()
    compare("o", o, O_ref, wl.dtype)
    g = lse.double().cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.all(np.abs(g[fin] - lse_ref[fin]) <= 1e-4 * (1 + np.abs(lse_ref[fin])))
    for b in range(wl.B):
        Lq = int(inp.seqlen_q[b])
        assert torch.all(o[b, :, Lq:].cpu() == 0)
        assert np.all(np.isposinf(g[b, :, Lq:]))


def test_varlen_bwd_ignores_rows_past_the_length(cuda_lib):
    # O, dO and LSE of rows outside the problem may hold anything
    wl, lq, lk = CASES[0]
    inp = _inputs(wl, lq, lk)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    clean = run_gpu_bwd(wl, inp, O, lse)
    g = torch.Generator().manual_seed(70)
    O2, lse2 = O.clone(), lse.clone()
    for b, L in enumerate(lq):
        O2[b, :, L:] = torch.randn(O2[b, :, L:].shape, generator=g).to(O2.dtype)
        inp.dO[b, :, L:] = torch.randn(inp.dO[b, :, L:].shape, generator=g).to(inp.dO.dtype)
        lse2[b, :, L:] = -torch.rand(lse2[b, :, L:].shape, generator=g) * 10
    dirty = run_gpu_bwd(wl, inp, O2, lse2)
    for name in ("dq", "dk", "dv", "dsink"):
        assert torch.equal(getattr(clean, name), getattr(dirty, name)), name
