"""Pins for the fp64 oracle, each independent of the oracle's own code.

* central finite differences of L = sum(dO * O) (backward vs forward);
* torch's scaled_dot_product_attention in float64 (a library routine) with the
  sink appended as an extra key column of value zero, forward and autograd;
* closed forms and invariants: a single visible key, sink = -inf, an all-ones
  block mask, block-mask expansion to a token mask, sum_j dV_j, the shift
  invariance that ties dSink to the row sums of dS, empty rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import MASK_BLOCK, MASK_CAUSAL, MASK_NONE, MASK_SLIDING, MASK_TOKEN


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _problem(kind, B=1, Hq=2, Hkv=1, Sq=13, Skv=13, D=8, sink=None, window=4,
             bx=3, by=5, rng=None, block_mask=None, token_mask=None):
    pb = oracle.Problem(B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Skv=Skv, D=D,
                        scale=1.0 / math.sqrt(D), mask_kind=kind, window=window,
                        bx=bx, by=by, sink=sink)
    if kind == MASK_BLOCK:
        if block_mask is None:
            nqb, nkb = -(-Sq // bx), -(-Skv // by)
            block_mask = (rng.random((B, Hq, nqb, nkb)) < 0.6).astype(np.uint8)
            block_mask[..., 0] = 1  # no empty row
        pb.block_mask = block_mask
    if kind == MASK_TOKEN:
        if token_mask is None:
            token_mask = (rng.random((B, Hq, Sq, Skv)) < 0.5).astype(np.uint8)
            token_mask[..., 0] = 1
        pb.token_mask = token_mask
    return pb


def _token_mask_of(pb):
    """Dense boolean visibility [B,Hq,Sq,Skv], written directly from the mask rules."""
    i = np.arange(pb.Sq)[:, None]
    j = np.arange(pb.Skv)[None, :]
    if pb.mask_kind == MASK_NONE:
        m = np.ones((pb.Sq, pb.Skv), bool)
    elif pb.mask_kind == MASK_CAUSAL:
        m = j <= i
    elif pb.mask_kind == MASK_SLIDING:
        m = (j <= i) & (i - j < pb.window)
    elif pb.mask_kind == MASK_BLOCK:
        bm = np.asarray(pb.block_mask).astype(bool)
        big = np.repeat(np.repeat(bm, pb.bx, axis=2), pb.by, axis=3)
        return big[:, :, :pb.Sq, :pb.Skv]
    else:
        return np.asarray(pb.token_mask).astype(bool)
    return np.broadcast_to(m, (pb.B, pb.Hq, pb.Sq, pb.Skv))


def _loss(pb, q, k, v, dO):
    O, _ = oracle.forward(pb, q, k, v)
    return float(np.sum(O * dO))


ALL_KINDS = [MASK_NONE, MASK_CAUSAL, MASK_SLIDING, MASK_BLOCK, MASK_TOKEN]


@pytest.mark.parametrize("kind", ALL_KINDS)
@pytest.mark.parametrize("with_sink", [False, True])
@pytest.mark.parametrize("dims", [(1, 2, 1, 13, 13), (2, 4, 2, 9, 11)])
def test_finite_differences(kind, with_sink, dims):
    B, Hq, Hkv, Sq, Skv = dims
    if kind in (MASK_CAUSAL, MASK_SLIDING) and Sq != Skv:
        Skv = Sq
    rng = np.random.default_rng(100 + kind + 7 * with_sink + Sq)
    D = 8
    sink = _rand(rng, Hq) if with_sink else None
    pb = _problem(kind, B, Hq, Hkv, Sq, Skv, D, sink=sink, rng=rng)
    q, k, v = _rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Skv, D), _rand(rng, B, Hkv, Skv, D)
    dO = _rand(rng, B, Hq, Sq, D)
    g = oracle.backward_exact(pb, q, k, v, dO)
    h = 1e-6

    def fd(x, setter):
        out = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            out[idx] = (setter(xp) - setter(xm)) / (2 * h)
        return out

    num_dq = fd(q, lambda x: _loss(pb, x, k, v, dO))
    num_dk = fd(k, lambda x: _loss(pb, q, x, v, dO))
    num_dv = fd(v, lambda x: _loss(pb, q, k, x, dO))
    for name, num in (("dq", num_dq), ("dk", num_dk), ("dv", num_dv)):
        ana = g[name]
        err = np.max(np.abs(num - ana))
        assert err <= 1e-6 * max(1.0, np.max(np.abs(ana))), (name, err)
    if with_sink:
        def lsink(s):
            pb2 = _problem(kind, B, Hq, Hkv, Sq, Skv, D, sink=s,
                           block_mask=pb.block_mask, token_mask=pb.token_mask, rng=rng)
            return _loss(pb2, q, k, v, dO)
        num_ds = fd(sink, lsink)
        err = np.max(np.abs(num_ds - g["dsink"]))
        assert err <= 1e-6 * max(1.0, np.max(np.abs(g["dsink"]))), err


def _sdpa_reference(pb, q, k, v, dO):
    """torch fp64 SDPA with the sink as an extra zero-value key; autograd backward."""
    g = pb.Hq // pb.Hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    kk = tk.repeat_interleave(g, dim=1)
    vv = tv.repeat_interleave(g, dim=1)
    vis = torch.tensor(np.ascontiguousarray(_token_mask_of(pb)))
    bias = torch.zeros(vis.shape, dtype=torch.float64).masked_fill(~vis, float("-inf"))
    ts = None
    if pb.sink is not None:
        ts = torch.tensor(pb.sink, requires_grad=True)
        zk = torch.zeros(pb.B, pb.Hq, 1, pb.D, dtype=torch.float64)
        kk = torch.cat([kk, zk], dim=2)
        vv = torch.cat([vv, zk], dim=2)
        sb = ts.view(1, pb.Hq, 1, 1).expand(pb.B, pb.Hq, pb.Sq, 1)
        bias = torch.cat([bias, sb], dim=3)
    O = torch.nn.functional.scaled_dot_product_attention(
        tq, kk, vv, attn_mask=bias, scale=pb.scale)
    logits = torch.einsum("bhid,bhjd->bhij", tq, kk) * pb.scale + bias
    lse = torch.logsumexp(logits, dim=-1)
    (O * torch.tensor(dO)).sum().backward()
    out = {"o": O.detach().numpy(), "lse": lse.detach().numpy(),
           "dq": tq.grad.numpy(), "dk": tk.grad.numpy(), "dv": tv.grad.numpy()}
    if ts is not None:
        out["dsink"] = ts.grad.numpy()
    return out


@pytest.mark.parametrize("kind", ALL_KINDS)
@pytest.mark.parametrize("with_sink", [False, True])
def test_against_torch_sdpa(kind, with_sink):
    rng = np.random.default_rng(7 + kind + 11 * with_sink)
    B, Hq, Hkv, S, D = 2, 4, 2, 37, 16
    sink = _rand(rng, Hq) if with_sink else None
    pb = _problem(kind, B, Hq, Hkv, S, S, D, sink=sink, window=9, bx=6, by=7, rng=rng)
    q, k, v = _rand(rng, B, Hq, S, D), _rand(rng, B, Hkv, S, D), _rand(rng, B, Hkv, S, D)
    dO = _rand(rng, B, Hq, S, D)
    ours = oracle.backward_exact(pb, q, k, v, dO)
    ref = _sdpa_reference(pb, q, k, v, dO)
    # torch's fp64 attention on the CPU reaches its result in a different
    # order from run to run (seen: 2e-10 relative on LSE within a full test
    # session); 1e-8 relative still fails any wrong term, sign or index
    for name in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(ours[name], ref[name], rtol=1e-8, atol=1e-9, err_msg=name)
    if with_sink:
        np.testing.assert_allclose(ours["dsink"], ref["dsink"], rtol=1e-8, atol=1e-9)
    else:
        assert np.all(ours["dsink"] == 0)


def test_single_visible_key_closed_form():
    # causal row 0 sees only key 0: O_0 = v_0 * sigma(s00 - sink), LSE = log(e^s00 + e^sink)
    rng = np.random.default_rng(3)
    D = 8
    q, k, v = _rand(rng, 1, 1, 5, D), _rand(rng, 1, 1, 5, D), _rand(rng, 1, 1, 5, D)
    dO = _rand(rng, 1, 1, 5, D)
    s00 = float(q[0, 0, 0] @ k[0, 0, 0]) / math.sqrt(D)
    pb = _problem(MASK_CAUSAL, 1, 1, 1, 5, 5, D, rng=rng)
    out = oracle.backward_exact(pb, q, k, v, dO)
    np.testing.assert_allclose(out["o"][0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-15)
    assert abs(out["lse"][0, 0, 0] - s00) < 1e-14
    np.testing.assert_allclose(out["dq"][0, 0, 0], 0, atol=1e-14)  # dS row 0 = 0
    sink = np.array([0.7])
    pb = _problem(MASK_CAUSAL, 1, 1, 1, 5, 5, D, sink=sink, rng=rng)
    out = oracle.backward_exact(pb, q, k, v, dO)
    sig = 1.0 / (1.0 + math.exp(-(s00 - 0.7)))
    np.testing.assert_allclose(out["o"][0, 0, 0], sig * v[0, 0, 0], rtol=1e-13)
    assert abs(out["lse"][0, 0, 0] - math.log(math.exp(s00) + math.exp(0.7))) < 1e-13


def test_sink_minus_inf_is_no_sink():
    rng = np.random.default_rng(4)
    B, Hq, Hkv, S, D = 1, 4, 2, 21, 8
    q, k, v = _rand(rng, B, Hq, S, D), _rand(rng, B, Hkv, S, D), _rand(rng, B, Hkv, S, D)
    dO = _rand(rng, B, Hq, S, D)
    for kind in (MASK_NONE, MASK_CAUSAL, MASK_SLIDING):
        a = oracle.backward_exact(_problem(kind, B, Hq, Hkv, S, S, D, rng=rng), q, k, v, dO)
        b = oracle.backward_exact(
            _problem(kind, B, Hq, Hkv, S, S, D, sink=np.full(Hq, -np.inf), rng=rng), q, k, v, dO)
        for name in ("o", "lse", "dq", "dk", "dv"):
            assert np.array_equal(a[name], b[name]), name
        assert np.all(b["dsink"] == 0)


def test_all_ones_block_mask_equals_dense():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, Sq, Skv, D = 2, 2, 1, 17, 23, 8
    q, k, v = _rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Skv, D), _rand(rng, B, Hkv, Skv, D)
    dO = _rand(rng, B, Hq, Sq, D)
    sink = _rand(rng, Hq)
    dense = oracle.backward_exact(_problem(MASK_NONE, B, Hq, Hkv, Sq, Skv, D, sink=sink), q, k, v, dO)
    ones = np.ones((B, Hq, -(-Sq // 4), -(-Skv // 6)), np.uint8)
    blk = oracle.backward_exact(_problem(MASK_BLOCK, B, Hq, Hkv, Sq, Skv, D, sink=sink, bx=4,
                                         by=6, block_mask=ones), q, k, v, dO)
    for name in ("o", "lse", "dq", "dk", "dv", "dsink"):
        assert np.array_equal(dense[name], blk[name]), name


def test_block_expansion_equals_token_mask():
    rng = np.random.default_rng(6)
    B, Hq, Hkv, Sq, Skv, D, bx, by = 1, 2, 2, 19, 26, 8, 4, 7
    q, k, v = _rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Skv, D), _rand(rng, B, Hkv, Skv, D)
    dO = _rand(rng, B, Hq, Sq, D)
    pb = _problem(MASK_BLOCK, B, Hq, Hkv, Sq, Skv, D, bx=bx, by=by, rng=rng)
    tok = np.repeat(np.repeat(pb.block_mask, bx, axis=2), by, axis=3)[:, :, :Sq, :Skv]
    pt = _problem(MASK_TOKEN, B, Hq, Hkv, Sq, Skv, D, token_mask=np.ascontiguousarray(tok))
    a = oracle.backward_exact(pb, q, k, v, dO)
    b = oracle.backward_exact(pt, q, k, v, dO)
    for name in ("o", "lse", "dq", "dk", "dv", "dsink"):
        assert np.array_equal(a[name], b[name]), name


@pytest.mark.parametrize("with_sink", [False, True])
def test_dv_column_sum(with_sink):
    # sum_j dV_j = sum_{h in group} sum_i (1 - psink_i) dO_i ; without a sink: sum dO
    rng = np.random.default_rng(8)
    B, Hq, Hkv, S, D = 2, 4, 2, 29, 8
    sink = _rand(rng, Hq) if with_sink else None
    q, k, v = _rand(rng, B, Hq, S, D), _rand(rng, B, Hkv, S, D), _rand(rng, B, Hkv, S, D)
    dO = _rand(rng, B, Hq, S, D)
    for kind in (MASK_NONE, MASK_CAUSAL, MASK_SLIDING):
        pb = _problem(kind, B, Hq, Hkv, S, S, D, sink=sink, window=5, rng=rng)
        out = oracle.backward_exact(pb, q, k, v, dO)
        w = np.ones((B, Hq, S)) if sink is None else 1 - np.exp(sink[None, :, None] - out["lse"])
        want = (w[..., None] * dO).reshape(B, Hkv, Hq // Hkv, S, D).sum(axis=(2, 3))
        np.testing.assert_allclose(out["dv"].sum(axis=2), want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("with_sink", [False, True])
def test_shift_invariance_ties_dsink_to_ds(with_sink):
    # Give every key a constant coordinate k_j[0] = 1: dQ_i[0] / scale = sum_j dS_ij.
    # Softmax over logits + sink is invariant to a common shift, so
    # sum_j dS_ij = -dsink contribution of row i, and sum_i over a head gives -dSink_h.
    # Without a sink, sum_j dS_ij = 0 and hence sum_j dK_j = 0 for every kv head.
    rng = np.random.default_rng(9)
    B, Hq, Hkv, S, D = 2, 4, 2, 25, 8
    sink = _rand(rng, Hq) if with_sink else None
    q, k, v = _rand(rng, B, Hq, S, D), _rand(rng, B, Hkv, S, D), _rand(rng, B, Hkv, S, D)
    k[..., 0] = 1.0
    dO = _rand(rng, B, Hq, S, D)
    pb = _problem(MASK_SLIDING, B, Hq, Hkv, S, S, D, sink=sink, window=7, rng=rng)
    out = oracle.backward_exact(pb, q, k, v, dO)
    rowsum_ds = out["dq"][..., 0] / pb.scale
    np.testing.assert_allclose(rowsum_ds.sum(axis=(0, 2)), -out["dsink"], rtol=1e-10, atol=1e-12)
    if not with_sink:
        np.testing.assert_allclose(rowsum_ds, 0, atol=1e-12)
        np.testing.assert_allclose(out["dk"].sum(axis=2), 0, atol=1e-11)


def test_empty_rows_give_zeros():
    rng = np.random.default_rng(10)
    B, Hq, Hkv, Sq, Skv, D, bx, by = 1, 2, 1, 12, 12, 8, 4, 4
    bm = np.ones((B, Hq, 3, 3), np.uint8)
    bm[0, 1, 1, :] = 0  # rows 4..7 of head 1 see nothing
    q, k, v = _rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Skv, D), _rand(rng, B, Hkv, Skv, D)
    dO = _rand(rng, B, Hq, Sq, D)
    pb = _problem(MASK_BLOCK, B, Hq, Hkv, Sq, Skv, D, bx=bx, by=by, block_mask=bm)
    out = oracle.backward_exact(pb, q, k, v, dO)
    assert np.all(np.isinf(out["lse"][0, 1, 4:8])) and np.all(out["lse"][0, 1, 4:8] > 0)
    assert np.all(out["o"][0, 1, 4:8] == 0)
    assert np.all(out["dq"][0, 1, 4:8] == 0)
    for name in ("o", "dq", "dk", "dv"):
        assert np.all(np.isfinite(out[name])), name
    # with a sink the empty rows attend only to the sink: O = 0, LSE = sink
    sink = np.array([0.3, -0.4])
    pb.sink = sink
    out = oracle.backward_exact(pb, q, k, v, dO)
    np.testing.assert_allclose(out["lse"][0, 1, 4:8], -0.4, rtol=0, atol=1e-15)
    assert np.all(out["o"][0, 1, 4:8] == 0)


def test_visible_count_closed_forms():
    S, W = 37, 5
    for kind, want in ((MASK_NONE, S * S), (MASK_CAUSAL, S * (S + 1) // 2),
                       (MASK_SLIDING, sum(min(i + 1, W) for i in range(S)))):
        pb = _problem(kind, 2, 3, 1, S, S, 8, window=W)
        assert oracle.count_visible(pb) == 2 * 3 * want


def test_parity_mode_matches_exact_mode_when_fed_its_own_stats():
    rng = np.random.default_rng(12)
    B, Hq, Hkv, S, D = 1, 2, 1, 15, 8
    q, k, v = _rand(rng, B, Hq, S, D), _rand(rng, B, Hkv, S, D), _rand(rng, B, Hkv, S, D)
    dO = _rand(rng, B, Hq, S, D)
    pb = _problem(MASK_CAUSAL, B, Hq, Hkv, S, S, D, sink=_rand(rng, Hq))
    ex = oracle.backward_exact(pb, q, k, v, dO)
    # sampled rows / columns agree with the full pass
    rows = np.array([0, 3, 14, 15 + 7], np.int64)
    lse = ex["lse"]
    dq = oracle.dq_rows(pb, q, k, v, dO, lse, ex["delta"], rows)
    np.testing.assert_array_equal(dq, ex["dq"].reshape(-1, D)[rows])
    cols = np.array([0, 5, 14], np.int64)
    dk, dv = oracle.dkdv_cols(pb, q, k, v, dO, lse, ex["delta"], cols)
    np.testing.assert_array_equal(dk, ex["dk"].reshape(-1, D)[cols])
    np.testing.assert_array_equal(dv, ex["dv"].reshape(-1, D)[cols])


@pytest.mark.parametrize("kind", [MASK_NONE, MASK_CAUSAL, MASK_SLIDING, MASK_BLOCK])
def test_varlen_matches_truncated_sequences(kind):
    # per-batch lengths: batch b is the problem cut to its first Lq[b] rows and
    # Lk[b] keys (torch fp64 SDPA on the cut problem, sink as an extra key);
    # rows and keys past the lengths get zeros and LSE = +inf
    rng = np.random.default_rng(21 + kind)
    B, Hq, Hkv, S, D = 4, 4, 2, 37, 16
    Lq = np.array([0, 1, 17, 37])
    Lk = Lq.copy() if kind in (MASK_CAUSAL, MASK_SLIDING) else np.array([5, 9, 30, 37])
    sink = _rand(rng, Hq)
    pb = _problem(kind, B, Hq, Hkv, S, S, D, sink=sink, window=9, bx=6, by=7, rng=rng)
    pb.seqlen_q, pb.seqlen_k = Lq, Lk
    q, k, v = _rand(rng, B, Hq, S, D), _rand(rng, B, Hkv, S, D), _rand(rng, B, Hkv, S, D)
    dO = _rand(rng, B, Hq, S, D)
    ours = oracle.backward_exact(pb, q, k, v, dO)
    dsink = np.zeros(Hq)
    for b in range(B):
        lq, lk = int(Lq[b]), int(Lk[b])
        assert np.all(ours["o"][b, :, lq:] == 0) and np.all(np.isposinf(ours["lse"][b, :, lq:]))
        assert np.all(ours["dq"][b, :, lq:] == 0)
        assert np.all(ours["dk"][b, :, lk:] == 0) and np.all(ours["dv"][b, :, lk:] == 0)
        if lq == 0:
            assert np.all(ours["dk"][b] == 0) and np.all(ours["dv"][b] == 0)
            continue
        cut = _problem(kind, 1, Hq, Hkv, lq, lk, D, sink=sink, window=9, bx=6, by=7, rng=rng,
                       block_mask=(pb.block_mask[b:b + 1, :, :-(-lq // 6), :-(-lk // 7)]
                                   if kind == MASK_BLOCK else None))
        ref = _sdpa_reference(cut, q[b:b + 1, :, :lq], k[b:b + 1, :, :lk], v[b:b + 1, :, :lk],
                              dO[b:b + 1, :, :lq])
        for name, got in (("o", ours["o"][b:b + 1, :, :lq]), ("lse", ours["lse"][b:b + 1, :, :lq]),
                          ("dq", ours["dq"][b:b + 1, :, :lq]), ("dk", ours["dk"][b:b + 1, :, :lk]),
                          ("dv", ours["dv"][b:b + 1, :, :lk])):
            np.testing.assert_allclose(got, ref[name], rtol=1e-8, atol=1e-9, err_msg=f"{name} b={b}")
        dsink += ref["dsink"]
    np.testing.assert_allclose(ours["dsink"], dsink, rtol=1e-8, atol=1e-9)


def test_varlen_backward_ignores_rows_past_the_length():
    # O, dO and LSE of rows outside the problem may hold anything
    rng = np.random.default_rng(33)
    B, Hq, Hkv, S, D = 2, 2, 1, 29, 8
    pb = _problem(MASK_CAUSAL, B, Hq, Hkv, S, S, D, sink=_rand(rng, Hq), rng=rng)
    pb.seqlen_q = pb.seqlen_k = np.array([11, 20])
    q, k, v = _rand(rng, B, Hq, S, D), _rand(rng, B, Hkv, S, D), _rand(rng, B, Hkv, S, D)
    dO = _rand(rng, B, Hq, S, D)
    O, lse = oracle.forward(pb, q, k, v)
    clean = oracle.backward(pb, q, k, v, O, dO, lse)
    O2, dO2, lse2 = O.copy(), dO.copy(), lse.copy()
    for b, l in enumerate((11, 20)):
        O2[b, :, l:] = _rand(rng, Hq, S - l, D)
        dO2[b, :, l:] = _rand(rng, Hq, S - l, D)
        lse2[b, :, l:] = -_rand(rng, Hq, S - l) ** 2 - 5.0
    dirty = oracle.backward(pb, q, k, v, O2, dO2, lse2)
    for name in ("dq", "dk", "dv", "dsink"):
        np.testing.assert_array_equal(dirty[name], clean[name], err_msg=name)
