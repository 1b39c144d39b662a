"""GPU parity of attn_bwd against the fp64 oracle, element by element.

Sizes span several tiles of both walks (128-row key tiles with 64-row query
sub-tiles; 128-row query tiles with 64-row key sub-tiles) and end on ragged
tails; every mask family of the workloads appears, in both dtypes.
"""
import numpy as np
import pytest
import torch

import oracle
from masked_attention_backward_gb300.workloads import (MASK_BLOCK, MASK_CAUSAL, MASK_NONE,
                                                        MASK_SLIDING, WORKLOADS, Workload,
                                                        make_inputs)
from parity import (compare, forward_stats, full_parity, oracle_problem, run_gpu_bwd, ws_layout,
                    ws_view)

pytestmark = pytest.mark.gpu

CASES = [
    WORKLOADS[0],  # the tiny workload exactly: fp16 B1 Hq2 Hkv1 S256 window 64 + sink
    Workload("swa_sink_bf16_ragged", "bf16", B=2, Hq=4, Hkv=2, Sq=333, Skv=333,
             mask_kind=MASK_SLIDING, window=100, sink=True, seed=11),
    Workload("causal_sink_bf16_gqa8", "bf16", B=1, Hq=8, Hkv=1, Sq=515, Skv=515,
             mask_kind=MASK_CAUSAL, sink=True, seed=12),
    Workload("causal_f16_nosink", "f16", B=1, Hq=2, Hkv=2, Sq=300, Skv=300,
             mask_kind=MASK_CAUSAL, seed=13),
    Workload("random_blocks_f16", "f16", B=1, Hq=2, Hkv=2, Sq=700, Skv=700, mask_kind=MASK_BLOCK,
             bx=64, by=64, block_pattern="random", density=0.3, seed=14),
    Workload("bigbird_f16_uneven", "f16", B=2, Hq=2, Hkv=2, Sq=500, Skv=700, mask_kind=MASK_BLOCK,
             bx=48, by=80, block_pattern="bigbird", seed=15),
    Workload("blocks_bf16_small_bxby", "bf16", B=1, Hq=4, Hkv=2, Sq=257, Skv=190,
             mask_kind=MASK_BLOCK, bx=16, by=32, block_pattern="random", density=0.2, sink=True,
             seed=16),
    Workload("dense_f16_uneven", "f16", B=1, Hq=2, Hkv=1, Sq=200, Skv=333, mask_kind=MASK_NONE,
             seed=17),
    Workload("dense_bf16_sink", "bf16", B=2, Hq=2, Hkv=2, Sq=129, Skv=129, mask_kind=MASK_NONE,
             sink=True, seed=18),
    # a window of one key (the diagonal alone) and one narrower than a 64-row sub-tile
    Workload("swa1_f16_sink", "f16", B=1, Hq=2, Hkv=1, Sq=300, Skv=300, mask_kind=MASK_SLIDING,
             window=1, sink=True, seed=19),
    Workload("swa1_bf16_nosink", "bf16", B=1, Hq=2, Hkv=2, Sq=200, Skv=200,
             mask_kind=MASK_SLIDING, window=1, seed=21),
    Workload("swa17_bf16_gqa", "bf16", B=2, Hq=4, Hkv=2, Sq=333, Skv=333, mask_kind=MASK_SLIDING,
             window=17, sink=True, seed=22),
    # blocks larger than every tile: 256 x 256, and 192 x 320 (neither divides the lengths)
    Workload("blocks256_f16", "f16", B=1, Hq=2, Hkv=2, Sq=900, Skv=1000, mask_kind=MASK_BLOCK,
             bx=256, by=256, block_pattern="random", density=0.5, seed=23),
    Workload("blocks192x320_bf16", "bf16", B=1, Hq=4, Hkv=2, Sq=1000, Skv=1100,
             mask_kind=MASK_BLOCK, bx=192, by=320, block_pattern="random", density=0.5, sink=True,
             seed=24),
    # blocks that hold no whole softmax-warp region: the producers publish each
    # step's mask bits (24 x 40), or the softmax warps read the mask (8 x 8)
    Workload("blocks24x40_f16", "f16", B=1, Hq=4, Hkv=2, Sq=500, Skv=460, mask_kind=MASK_BLOCK,
             bx=24, by=40, block_pattern="random", density=0.4, seed=25),
    Workload("blocks8x8_bf16", "bf16", B=1, Hq=2, Hkv=1, Sq=200, Skv=190, mask_kind=MASK_BLOCK,
             bx=8, by=8, block_pattern="random", density=0.3, sink=True, seed=26),
]


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_bwd_parity(cuda_lib, wl):
    reps, _, _ = full_parity(wl)
    print({r["name"]: (round(r["frac"], 6), r["max_err"]) for r in reps})


@pytest.mark.parametrize("S", [1, 2, 63, 64, 65, 127, 128, 129])
def test_bwd_tiny_lengths(cuda_lib, S):
    wl = Workload(f"causal_sink_S{S}", "bf16", B=1, Hq=4, Hkv=1, Sq=S, Skv=S,
                  mask_kind=MASK_CAUSAL, sink=True, seed=20 + S)
    full_parity(wl)


def test_bwd_sink_minus_inf_matches_no_sink(cuda_lib):
    wl = Workload("swa_f16", "f16", B=1, Hq=2, Hkv=1, Sq=200, Skv=200, mask_kind=MASK_SLIDING,
                  window=50, sink=True, seed=30)
    inp = make_inputs(wl)
    inp.sink = torch.full((wl.Hq,), float("-inf"))
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    run = run_gpu_bwd(wl, inp, O, lse)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name in ("dq", "dk", "dv"):
        compare(name, getattr(run, name), ref[name], wl.dtype)
    assert torch.all(run.dsink.cpu() == 0)


def test_bwd_empty_rows_and_empty_key_tiles(cuda_lib):
    # head 1 has whole query blocks and whole key blocks switched off: rows that
    # see nothing get dQ = 0, key tiles that nobody sees get dK = dV = 0
    wl = Workload("holes_f16", "f16", B=1, Hq=2, Hkv=2, Sq=400, Skv=400, mask_kind=MASK_BLOCK,
                  bx=64, by=64, block_pattern="ones", seed=31)
    inp = make_inputs(wl)
    inp.block_mask[0, 1, 2, :] = 0      # query rows 128..191 of head 1 see nothing
    inp.block_mask[0, 1, :, 4:] = 0     # keys 256.. of head 1 are seen by nobody
    inp.block_mask[0, 0, :, :] = 0      # head 0: nothing at all
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    run = run_gpu_bwd(wl, inp, O, lse)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name in ("dq", "dk", "dv"):
        compare(name, getattr(run, name), ref[name], wl.dtype)
    assert torch.all(run.dq[0, 1, 128:192].cpu() == 0)
    assert torch.all(run.dq[0, 0].cpu() == 0)
    assert torch.all(run.dk[0, 1, 256:].cpu() == 0) and torch.all(run.dv[0, 1, 256:].cpu() == 0)
    assert torch.all(run.dk[0, 0].cpu() == 0)


def _rounding_bounds(wl, inp, O, lse):
    """Per-element bounds on what fp32 arithmetic on the device must leave in
    dV and dK (beyond the plain gate) for one kv head of a causal problem
    without per-batch lengths, computed in float64 from the inputs.

    The device forms each logit as an fp32 dot product of 128 fp16 products:
    its accumulated rounding error is at most 2^-17 times the sum of the
    products' magnitudes (128 additions at 2^-24 each), and the exponent's
    argument is rounded once more (2^-23 of its size, for the logit and for
    -LSE log2 e).  P then carries that relative error, plus 2^-11 from its
    rounding to fp16 before the dV contraction.  dS = P (dP - Delta) adds the
    same accumulation bound for dP and Delta and 2^-11 from its own rounding;
    dK multiplies dS by q, so a q entry of 32000 multiplies it too.  Rows
    without large entries get bounds far below the gate's tolerance."""
    q, k, v, dO = (x.double().numpy()[0] for x in (inp.q, inp.k, inp.v, inp.dO))
    o, l = O.double().numpy()[0], lse.double().numpy()[0]
    S, g = wl.Sq, wl.Hq // wl.Hkv
    causal = np.tril(np.ones((S, S), dtype=bool))
    bdv = np.zeros((wl.Hkv, S, wl.D))
    bdk = np.zeros((wl.Hkv, S, wl.D))
    for h in range(wl.Hq):
        c = h // g
        s = wl.scale * q[h] @ k[c].T
        P = np.exp(np.where(causal, s - l[h][:, None], -np.inf))
        A = wl.scale * np.abs(q[h]) @ np.abs(k[c]).T                  # |terms| of each logit
        dx = 2.0 ** -17 * A + 2.0 ** -23 * (np.abs(s) + np.abs(l[h])[:, None]) * 2
        dP = dO[h] @ v[c].T
        delta = (dO[h] * o[h]).sum(1)
        terms = np.abs(dO[h]) @ np.abs(v[c]).T + (np.abs(dO[h]) * np.abs(o[h])).sum(1)[:, None]
        eP = P * (dx + 2.0 ** -11)                                    # |error of P|
        eS = P * dx * np.abs(dP - delta[:, None]) + P * 2.0 ** -17 * terms \
            + 2.0 ** -11 * P * np.abs(dP - delta[:, None])            # |error of dS|
        bdv[c] += eP.T @ np.abs(dO[h])
        bdk[c] += wl.scale * eS.T @ np.abs(q[h])
    return bdv, bdk


def test_bwd_extreme_logits_fp16(cuda_lib):
    # a few q entries near +-32000 in fp16 (0.2 % of them, in about a quarter
    # of the rows) keep every logit finite in fp32 (scaled logits reach about
    # 3e3; in most of those rows one key takes all of the softmax).  dQ against the oracle under the plain
    # gate; dV and dK under the plain gate widened by the rounding that fp32
    # arithmetic on such logits must leave (_rounding_bounds): the oracle
    # computes the same formulas from the same inputs in float64, so what the
    # widening admits is the device's fp32 rounding, not a different result
    wl = Workload("big_f16", "f16", B=1, Hq=2, Hkv=1, Sq=130, Skv=130, mask_kind=MASK_CAUSAL,
                  sink=True, seed=32)
    inp = make_inputs(wl)
    spikes = (torch.rand(inp.q.shape, generator=torch.Generator().manual_seed(5)) < 0.002)
    inp.q = torch.where(spikes, inp.q.float().sign() * 32000, inp.q.float()).half()
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    run = run_gpu_bwd(wl, inp, O, lse)
    for t in (run.dq, run.dk, run.dv):
        assert torch.isfinite(t.float()).all()
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    compare("dq", run.dq, ref["dq"], wl.dtype)
    bdv, bdk = _rounding_bounds(wl, inp, O, lse)
    tol = 2e-3
    for name, got, bound in (("dv", run.dv, bdv), ("dk", run.dk, bdk)):
        r = ref[name][0]
        err = np.abs(got.double().cpu().numpy()[0] - r)
        ok = err <= tol + tol * np.abs(r) + bound
        assert ok.mean() >= 0.999, (name, ok.mean(), float(err.max()))
        # the widening is confined to the rows that hold large entries: on at
        # least half of the elements it stays below the plain tolerance
        assert np.median(bound) < tol, (name, float(np.median(bound)))


def test_bwd_deterministic(cuda_lib):
    wl = CASES[4]
    inp = make_inputs(wl)
    O, lse = forward_stats(wl, inp)
    a = run_gpu_bwd(wl, inp, O, lse)
    for _ in range(3):
        b = run_gpu_bwd(wl, inp, O, lse)
        for name in ("dq", "dk", "dv"):
            assert torch.equal(getattr(a, name), getattr(b, name)), name


@pytest.mark.parametrize("compensated", [False, True], ids=["default", "compensated"])
def test_bwd_more_units_than_sms(cuda_lib, compensated):
    # 2 x 12 x 11 = 264 query tiles: more than one per SM, so the persistent
    # kernels hand out work units at run time; some tiles see no key at all.
    # Every element against the oracle, and bitwise the same on every run
    wl = Workload("claims_bf16", "bf16", B=2, Hq=12, Hkv=4, Sq=1300, Skv=1100,
                  mask_kind=MASK_BLOCK, bx=64, by=64, block_pattern="random", density=0.25,
                  sink=True, seed=33)
    inp = make_inputs(wl)
    inp.block_mask[0, 3, 4:8, :] = 0    # query rows 256..511 of (0, 3) see nothing
    inp.block_mask[1, 7, :, :] = 0      # (1, 7) sees nothing
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    a = run_gpu_bwd(wl, inp, O, lse, compensated=compensated)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    for name in ("dq", "dk", "dv"):
        compare(name, getattr(a, name), ref[name], wl.dtype)
    compare("dsink", a.dsink, ref["dsink"], wl.dtype, min_frac=1.0)
    assert torch.all(a.dq[0, 3, 256:512].cpu() == 0) and torch.all(a.dq[1, 7].cpu() == 0)
    for _ in range(2):
        b = run_gpu_bwd(wl, inp, O, lse, compensated=compensated)
        for name in ("dq", "dk", "dv", "dsink"):
            assert torch.equal(getattr(a, name), getattr(b, name)), name


@pytest.mark.parametrize("wl", [CASES[4], CASES[5], CASES[6], CASES[12], CASES[13]],
                         ids=lambda w: w.name)
def test_tables_bit_exact(cuda_lib, wl):
    inp = make_inputs(wl)
    O, lse = forward_stats(wl, inp)
    run = run_gpu_bwd(wl, inp, O, lse)
    L = ws_layout(wl)
    assert run.ws.numel() == L["total"]
    BH = wl.B * wl.Hq
    ws = run.ws.cpu()
    maskT = ws_view(ws, L["maskT"], BH * wl.nqb * wl.nkb, torch.uint8).numpy()
    want = oracle.mask_transpose(inp.block_mask.numpy())
    assert np.array_equal(maskT.reshape(want.shape), want)
    sel_k, cnt_k, sel_q, cnt_q = oracle.select_tables(inp.block_mask.numpy(), wl.Sq, wl.Skv, wl.bx,
                                                      wl.by, 64, 128, 128, 64)
    g_sel_k = ws_view(ws, L["sel_k"], sel_k.size, torch.int32).numpy().reshape(sel_k.shape)
    g_cnt_k = ws_view(ws, L["cnt_k"], cnt_k.size, torch.int32).numpy().reshape(cnt_k.shape)
    g_sel_q = ws_view(ws, L["sel_q"], sel_q.size, torch.int32).numpy().reshape(sel_q.shape)
    g_cnt_q = ws_view(ws, L["cnt_q"], cnt_q.size, torch.int32).numpy().reshape(cnt_q.shape)
    assert np.array_equal(g_cnt_k, cnt_k) and np.array_equal(g_sel_k, sel_k)
    assert np.array_equal(g_cnt_q, cnt_q) and np.array_equal(g_sel_q, sel_q)


def test_preprocess_delta_and_nlse2(cuda_lib):
    wl = CASES[1]
    inp = make_inputs(wl)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    run = run_gpu_bwd(wl, inp, O, lse)
    L = ws_layout(wl)
    BH, Sp = wl.B * wl.Hq, L["Sq_pad"]
    ws = run.ws.cpu()
    delta = ws_view(ws, L["delta"], BH * Sp, torch.float32).reshape(BH, Sp).double().numpy()
    nlse2 = ws_view(ws, L["nlse2"], BH * Sp, torch.float32).reshape(BH, Sp).double().numpy()
    ref = oracle.delta(pb, O, inp.dO).reshape(BH, wl.Sq)
    assert np.all(np.abs(delta[:, :wl.Sq] - ref) <= 1e-5 * (1 + np.abs(ref)))
    assert np.all(delta[:, wl.Sq:] == 0) and np.all(np.isneginf(nlse2[:, wl.Sq:]))
    want = -lse.double().numpy().reshape(BH, wl.Sq) * np.log2(np.e)
    assert np.all(np.abs(nlse2[:, :wl.Sq] - want) <= 1e-6 * (1 + np.abs(want)))
