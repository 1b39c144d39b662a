"""Parity at the full sizes of the named workloads, in the launch configuration
the benchmark times (one attn_bwd call over the whole problem).

* gqa_sink_swa128_s4096, blocksparse_bigbird_5000x7000: every element of dq,
  dk, dv, dsink against the oracle (parity mode: oracle O and LSE fed to both).
* blocksparse_random30_s8192: oracle O and LSE for all rows; dq on sampled
  rows and dk, dv on sampled key rows, computed one by one by the oracle.
* gqa_sink_varlen_causal_b8_s2048: oracle O and LSE for all rows, against
  which every element of the CUDA forward is compared too; dq on sampled rows,
  dk, dv on sampled key rows, dsink of every head; exact zeros and +inf past
  each sequence's length.
* gqa_sink_causal_s16384: O and LSE from the CUDA forward (the oracle's full
  forward at this size would take minutes), compared against the oracle in
  exact mode (its own fp64 statistics): dq on sampled rows of every head; dk,
  dv on sampled key rows and dsink of the first kv-head group, whose 8 query
  heads get a complete oracle forward; in parity mode (the CUDA forward's O
  and LSE fed to the oracle as they are to the backward) dk, dv on sampled key
  rows of kv heads 3 and 7 and dsink of all 64 heads; plus the column-sum
  property of dv on every kv head, which holds at any size.
"""
import numpy as np
import pytest
import torch

import oracle
from masked_attention_backward_gb300 import binding as mab
from masked_attention_backward_gb300.workloads import BY_NAME, make_inputs
from parity import compare, forward_stats, gpu_mask, oracle_problem, run_gpu_bwd, tight_gate

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["gqa_sink_swa128_s4096", "blocksparse_bigbird_5000x7000"])
def test_fullsize_every_element(cuda_lib, name):
    wl = BY_NAME[name]
    inp = make_inputs(wl)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    run = run_gpu_bwd(wl, inp, O, lse)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for n in ("dq", "dk", "dv"):
        compare(n, getattr(run, n), ref[n], wl.dtype)
    if inp.sink is not None:
        compare("dsink", run.dsink, ref["dsink"], wl.dtype, min_frac=1.0)


@pytest.mark.parametrize("compensated", [False, True], ids=["default", "compensated"])
def test_fullsize_blocksparse_random_sampled(cuda_lib, compensated):
    wl = BY_NAME["blocksparse_random30_s8192"]
    inp = make_inputs(wl)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    run = run_gpu_bwd(wl, inp, O, lse, compensated=compensated)
    rng = np.random.default_rng(0)
    rows = rng.choice(wl.B * wl.Hq * wl.Sq, size=2048, replace=False)
    cols = rng.choice(wl.B * wl.Hkv * wl.Skv, size=1024, replace=False)
    q, k, v, dO = (oracle._f64(t) for t in (inp.q, inp.k, inp.v, inp.dO))
    dl = oracle.delta(pb, O, dO)
    dq = oracle.dq_rows(pb, q, k, v, dO, lse, dl, rows)
    dk, dv = oracle.dkdv_cols(pb, q, k, v, dO, lse, dl, cols)
    compare("dq", run.dq.reshape(-1, wl.D)[rows], dq, wl.dtype)
    compare("dk", run.dk.reshape(-1, wl.D)[cols], dk, wl.dtype)
    compare("dv", run.dv.reshape(-1, wl.D)[cols], dv, wl.dtype)
    if compensated:   # fp16: the tighter gate as well
        tight_gate("dq", run.dq.reshape(-1, wl.D)[rows], dq)
        tight_gate("dk", run.dk.reshape(-1, wl.D)[cols], dk)
        tight_gate("dv", run.dv.reshape(-1, wl.D)[cols], dv)


@pytest.mark.parametrize("compensated", [False, True], ids=["default", "compensated"])
def test_fullsize_causal_16k_sampled(cuda_lib, compensated):
    wl = BY_NAME["gqa_sink_causal_s16384"]
    inp = make_inputs(wl)
    dev = "cuda"
    mask = gpu_mask(wl, inp, dev)
    q, k, v, dO = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dO))
    sink = inp.sink.to(dev)
    o_gpu, lse_gpu = mab.fwd(q, k, v, sink, mask, wl.scale)
    dq, dk, dv, dsink = mab.bwd(q, k, v, o_gpu, dO, lse_gpu, sink, mask, wl.scale,
                                compensated=compensated)
    torch.cuda.synchronize()
    for t in (dq, dk, dv, dsink):
        assert torch.isfinite(t.float()).all()

    pb = oracle_problem(wl, inp)
    g = wl.Hq // wl.Hkv
    S, D = wl.Sq, wl.D
    q64, k64, v64, dO64 = (oracle._f64(t) for t in (inp.q, inp.k, inp.v, inp.dO))
    rng = np.random.default_rng(1)
    # exact statistics for every row of kv group 0 and for sampled rows elsewhere
    group_rows = np.arange(g * S, dtype=np.int64)                  # heads 0..g-1 (B = 1)
    other_rows = rng.choice(np.arange(g * S, wl.Hq * S), size=256, replace=False)
    stat_rows = np.concatenate([group_rows, other_rows])
    O_r, lse_r = oracle.forward(pb, q64, k64, v64, rows=stat_rows)
    O_full = np.zeros((wl.Hq * S, D))
    lse_full = np.zeros(wl.Hq * S)
    O_full[stat_rows], lse_full[stat_rows] = O_r, lse_r
    O_full = O_full.reshape(1, wl.Hq, S, D)
    lse_full = lse_full.reshape(1, wl.Hq, S)
    dl = oracle.delta(pb, O_full, dO64)

    dq_rows = np.concatenate([rng.choice(group_rows, size=256, replace=False), other_rows])
    ref_dq = oracle.dq_rows(pb, q64, k64, v64, dO64, lse_full, dl, dq_rows)
    compare("dq", dq.reshape(-1, D)[dq_rows], ref_dq, wl.dtype)
    cols = rng.choice(S, size=192, replace=False).astype(np.int64)  # kv head 0
    ref_dk, ref_dv = oracle.dkdv_cols(pb, q64, k64, v64, dO64, lse_full, dl, cols)
    compare("dk", dk.reshape(-1, D)[cols], ref_dk, wl.dtype)
    compare("dv", dv.reshape(-1, D)[cols], ref_dv, wl.dtype)
    ref_ds = oracle.dsink(pb, lse_full, dl)[:g]
    compare("dsink", dsink[:g], ref_ds, wl.dtype, min_frac=1.0)

    # parity mode on the device's own statistics (the backward takes O and LSE
    # as given, like every other parity case): dK, dV on sampled key rows of
    # kv heads 3 and 7 (groups other than the first, reached by key tiles far
    # into the grid) and dSink of every head
    o64 = oracle._f64(o_gpu.cpu())
    lse64 = lse_gpu.double().cpu().numpy()
    dl_g = oracle.delta(pb, o64, dO64)
    cols_g = np.concatenate([c * S + rng.choice(S, size=128, replace=False) for c in (3, 7)])
    rk, rv = oracle.dkdv_cols(pb, q64, k64, v64, dO64, lse64, dl_g, cols_g.astype(np.int64))
    compare("dk (kv heads 3, 7)", dk.reshape(-1, D)[cols_g], rk, wl.dtype)
    compare("dv (kv heads 3, 7)", dv.reshape(-1, D)[cols_g], rv, wl.dtype)
    compare("dsink (all heads)", dsink, oracle.dsink(pb, lse64, dl_g), wl.dtype, min_frac=1.0)

    # any size: sum_j dV_j = sum_{h in group} sum_i (1 - exp(sink_h - lse_i)) dO_i, per kv head
    w = 1.0 - torch.exp(sink.double().view(1, -1, 1) - lse_gpu.double())
    want = (w.unsqueeze(-1) * dO.double()).reshape(1, wl.Hkv, g, S, D).sum(dim=(2, 3))
    got = dv.double().sum(dim=2)
    err = (got - want).abs().max().item()
    assert err <= 2e-2 * (1 + want.abs().max().item()), err


def test_fullsize_varlen_sampled(cuda_lib):
    wl = BY_NAME["gqa_sink_varlen_causal_b8_s2048"]
    inp = make_inputs(wl)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    dev = "cuda"
    q_d, k_d, v_d = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    o_g, lse_g = mab.fwd(q_d, k_d, v_d, inp.sink.to(dev), gpu_mask(wl, inp, dev), wl.scale)
    torch.cuda.synchronize()
    compare("o", o_g, O.double().numpy(), wl.dtype)
    g = lse_g.double().cpu().numpy()
    r = lse.double().numpy()
    fin = np.isfinite(r)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.all(np.abs(g[fin] - r[fin]) <= 1e-4 * (1 + np.abs(r[fin])))
    run = run_gpu_bwd(wl, inp, O, lse)
    for b in range(wl.B):
        L = int(inp.seqlen_q[b])
        assert torch.all(o_g[b, :, L:].cpu() == 0) and np.all(np.isposinf(g[b, :, L:]))
        assert torch.all(run.dq[b, :, L:].cpu() == 0)
        assert torch.all(run.dk[b, :, L:].cpu() == 0) and torch.all(run.dv[b, :, L:].cpu() == 0)
    rng = np.random.default_rng(0)
    rows = rng.choice(wl.B * wl.Hq * wl.Sq, size=2048, replace=False)
    cols = rng.choice(wl.B * wl.Hkv * wl.Skv, size=1024, replace=False)
    q, k, v, dO = (oracle._f64(t) for t in (inp.q, inp.k, inp.v, inp.dO))
    dl = oracle.delta(pb, O, dO)
    dq = oracle.dq_rows(pb, q, k, v, dO, lse, dl, rows)
    dk, dv = oracle.dkdv_cols(pb, q, k, v, dO, lse, dl, cols)
    compare("dq", run.dq.reshape(-1, wl.D)[rows], dq, wl.dtype)
    compare("dk", run.dk.reshape(-1, wl.D)[cols], dk, wl.dtype)
    compare("dv", run.dv.reshape(-1, wl.D)[cols], dv, wl.dtype)
    compare("dsink", run.dsink, oracle.dsink(pb, lse, dl), wl.dtype, min_frac=1.0)
