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


def _fwd_case(wl, inp):
    pb = oracle_problem(wl, inp)
    O_ref, lse_ref = oracle.forward(pb, inp.q, inp.k, inp.v)
    dev = "cuda"
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    sink = inp.sink.to(dev) if inp.sink is not None else None
    o, lse = mab.fwd(q, k, v, sink, gpu_mask(wl, inp, dev), wl.scale)
    torch.cuda.synchronize()
    return o, lse, O_ref, lse_ref


@pytest.mark.parametrize("with_sink", [False, True])
def test_fwd_empty_rows(cuda_lib, with_sink):
    # rows that see no key: O = 0; LSE = +inf without a sink, the sink itself with one
    from masked_attention_backward_gb300.workloads import MASK_BLOCK, Workload
    wl = Workload("fwd_holes", "bf16", B=1, Hq=2, Hkv=1, Sq=300, Skv=260, mask_kind=MASK_BLOCK,
                  bx=64, by=64, block_pattern="ones", sink=with_sink, seed=41)
    inp = make_inputs(wl)
    inp.block_mask[0, 1, 1, :] = 0   # query rows 64..127 of head 1 see nothing
    inp.block_mask[0, 0, :, 2:] = 0  # head 0 sees keys 0..127 only
    o, lse, O_ref, lse_ref = _fwd_case(wl, inp)
    compare("o", o, O_ref, wl.dtype)
    assert torch.all(o[0, 1, 64:128].float().cpu() == 0)
    g = lse.double().cpu().numpy()
    if with_sink:
        assert np.allclose(g[0, 1, 64:128], float(inp.sink[1]), rtol=1e-6, atol=1e-6)
    else:
        assert np.all(np.isinf(g[0, 1, 64:128]) & (g[0, 1, 64:128] > 0))
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.all(np.abs(g[fin] - lse_ref[fin]) <= 1e-4 * (1 + np.abs(lse_ref[fin])))


def test_fwd_sink_minus_inf_is_no_sink(cuda_lib):
    from masked_attention_backward_gb300.workloads import MASK_CAUSAL, Workload
    wl = Workload("fwd_sinkinf", "f16", B=1, Hq=4, Hkv=2, Sq=257, Skv=257, mask_kind=MASK_CAUSAL,
                  sink=True, seed=42)
    inp = make_inputs(wl)
    inp.sink = torch.full((wl.Hq,), float("-inf"))
    o, lse, _, _ = _fwd_case(wl, inp)
    inp.sink = None
    o2, lse2, O_ref, lse_ref = _fwd_case(wl, inp)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    compare("o", o2, O_ref, wl.dtype)


def test_fwd_large_logits_fp16(cuda_lib):
    # q entries near +-32000 in fp16: the row maximum must be taken exactly,
    # every P stays finite and O matches the oracle
    from masked_attention_backward_gb300.workloads import MASK_SLIDING, Workload
    wl = Workload("fwd_big", "f16", B=1, Hq=2, Hkv=1, Sq=190, Skv=190, mask_kind=MASK_SLIDING,
                  window=70, sink=True, seed=43)
    inp = make_inputs(wl)
    spikes = torch.rand(inp.q.shape, generator=torch.Generator().manual_seed(9)) < 0.01
    inp.q = torch.where(spikes, inp.q.float().sign() * 32000, inp.q.float()).half()
    o, lse, O_ref, lse_ref = _fwd_case(wl, inp)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    # logits reach ~3e3 after scaling, so fp32 score accumulation alone moves
    # P by ~1e-3: check what holds at any magnitude -- each O row is a convex
    # combination of V rows, and LSE agrees to 1e-3 relative
    vmax = float(inp.v.float().abs().max())
    assert float(o.float().abs().max()) <= vmax * (1 + 1e-2)
    g = lse.double().cpu().numpy()
    assert np.all(np.abs(g - lse_ref) <= 1e-3 * (1 + np.abs(lse_ref)))
