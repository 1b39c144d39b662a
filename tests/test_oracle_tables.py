"""Pins for the oracle's block-mask tables (transpose and select tables).

The select tables are checked against a brute force that expands the block
mask to tokens and asks whether any token pair of a tile pair is visible, and
against the divisible-case mapping the BlockSparseAttentionGrad runbook prints
(cannbot-knowledge PR #174, optimisation 2: a query tile of BMK rows maps to
mask block qt // (bx // BMK)).
"""
import numpy as np
import pytest

import oracle


def _brute(mask, Sq, Skv, bx, by, tq, tk):
    B, H = mask.shape[:2]
    tok = np.repeat(np.repeat(mask.astype(bool), bx, axis=2), by, axis=3)[:, :, :Sq, :Skv]
    nqt, nkt = -(-Sq // tq), -(-Skv // tk)
    act = np.zeros((B, H, nqt, nkt), bool)
    for r in range(nqt):
        for t in range(nkt):
            act[:, :, r, t] = tok[:, :, r * tq:(r + 1) * tq, t * tk:(t + 1) * tk].any(axis=(2, 3))
    return act


@pytest.mark.parametrize("Sq,Skv,bx,by,tq,tk", [
    (130, 200, 16, 16, 64, 128),
    (250, 330, 48, 80, 64, 128),
    (5000 // 8, 7000 // 8, 48, 80, 128, 64),
    (97, 97, 128, 128, 64, 64),
    (300, 260, 7, 13, 32, 16),
    # blocks that start on the last row / key of a tile (63 = 64 - 1, 127 = 128 - 1)
    (300, 400, 63, 127, 64, 128),
])
def test_select_tables_brute_force(Sq, Skv, bx, by, tq, tk):
    rng = np.random.default_rng(Sq + Skv)
    nqb, nkb = -(-Sq // bx), -(-Skv // by)
    mask = (rng.random((2, 3, nqb, nkb)) < 0.2).astype(np.uint8)
    sel_k, cnt_k, sel_q, cnt_q = oracle.select_tables(mask, Sq, Skv, bx, by, tq, tk, tk, tq)
    act = _brute(mask, Sq, Skv, bx, by, tq, tk)          # [B,H,nqt,nkt]
    B, H, nqt, nkt = act.shape
    for b in range(B):
        for h in range(H):
            for t in range(nkt):
                want = np.nonzero(act[b, h, :, t])[0]
                assert cnt_k[b, h, t] == want.size
                assert np.array_equal(sel_k[b, h, t, :want.size], want)
                assert np.all(sel_k[b, h, t, want.size:] == -1)
    act_q = _brute(mask, Sq, Skv, bx, by, tk, tq)        # query tiles of size tk
    for b in range(B):
        for h in range(H):
            for r in range(act_q.shape[2]):
                want = np.nonzero(act_q[b, h, r, :])[0]
                assert cnt_q[b, h, r] == want.size
                assert np.array_equal(sel_q[b, h, r, :want.size], want)
                assert np.all(sel_q[b, h, r, want.size:] == -1)


def test_divisible_mapping_from_runbook():
    # bx = 128 with 64-row query tiles: tile qt reads mask block qt // (128 // 64)
    rng = np.random.default_rng(1)
    Sq = Skv = 1024
    bx = by = 128
    tq, tk = 64, 128
    mask = (rng.random((1, 2, 8, 8)) < 0.4).astype(np.uint8)
    maskT = oracle.mask_transpose(mask)
    sel_k, cnt_k, _, _ = oracle.select_tables(mask, Sq, Skv, bx, by, tq, tk, tk, tq)
    for h in range(2):
        for kt in range(Skv // tk):
            qts = np.arange(Sq // tq)
            mqs = qts // (bx // tq)
            keep = maskT[0, h, kt, mqs] != 0
            want = qts[keep]
            assert cnt_k[0, h, kt] == want.size
            assert np.array_equal(sel_k[0, h, kt, :want.size], want)


def test_mask_transpose_is_permute():
    rng = np.random.default_rng(2)
    mask = rng.integers(0, 2, size=(2, 3, 105, 88), dtype=np.uint8)
    assert np.array_equal(oracle.mask_transpose(mask), mask.transpose(0, 1, 3, 2))
