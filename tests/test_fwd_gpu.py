"""GPU parity of attn_fwd (O and LSE) against the fp64 oracle forward."""
import numpy as np
import pytest
import torch

import oracle
from masked_attention_backward_gb300 import binding as mab
from masked_attention_backward_gb300.workloads import make_inputs
from parity import compare, gpu_mask, oracle_problem
from test_bwd_gpu import CASES

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_fwd_parity(cuda_lib, wl):
    inp = make_inputs(wl)
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
