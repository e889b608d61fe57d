"""Pins for the oracle's router (logits, top-k, weights) and dispatch index.

Checked against exact rational arithmetic, brute force over all k-subsets,
the closed-form softmax identity and plain loops.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats as F
from oracle import moe as M


def _fl32_of_fraction(s: Fraction) -> np.float32:
    """Correctly rounded binary32 of an exact rational (ties to even), by bisection on neighbours."""
    f = np.float32(float(s))                      # within one fp32 ulp of s
    for _ in range(3):
        up = np.nextafter(f, np.float32(np.inf))
        dn = np.nextafter(f, np.float32(-np.inf))
        best = min((abs(Fraction(float(c)) - s), int(c.view(np.uint32)) & 1, c) for c in (dn, f, up))
        f = best[2]
    return np.float32(f)


def _bf16_bits_random(rng, shape):
    return np.asarray(
        (np.float32(rng.standard_normal(shape)).view(np.uint32) >> 16), dtype=np.uint16)


def test_logits_are_correctly_rounded_fp32():
    rng = np.random.default_rng(5)
    T, E, H = 4, 8, 96
    x = _bf16_bits_random(rng, (T, H))
    W = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    l32, _ = M.router_logits(x, W)
    X = F.bf16_to_f64(x)
    for t in range(T):
        for e in range(E):
            s = sum(Fraction(float(X[t, h])) * Fraction(float(W[e, h])) for h in range(H))
            assert l32[t, e] == _fl32_of_fraction(s)


def test_logits_exact_midpoint_cases():
    # dot products landing exactly on, and just beside, an fp32 rounding midpoint
    one = np.float32(1.0)
    half_ulp = 2.0 ** -24
    H = 4
    cases = [
        ([1.0, half_ulp, 0.0, 0.0], one),                          # exactly 1 + 2^-24: tie -> even (1.0)
        ([1.0, half_ulp, 2.0 ** -60, 0.0], np.nextafter(one, np.float32(2))),   # just above the tie
        ([1.0, half_ulp, -2.0 ** -60, 0.0], one),                  # just below the tie
        ([1.0 + 2.0 ** -23, half_ulp, 0.0, 0.0], np.float32(1.0 + 2.0 ** -22)),  # tie from odd -> up
    ]
    for terms, expect in cases:
        Wr = np.array([terms], dtype=np.float64)
        assert np.all(Wr.astype(np.float32).astype(np.float64) == Wr)
        x = np.full((1, H), 0x3F80, dtype=np.uint16)               # bf16 1.0
        l32, near = M.router_logits(x, Wr.astype(np.float32))
        assert l32[0, 0] == expect, (terms, l32[0, 0], expect)


def test_logit_bias_is_fp32_add_after_rounding():
    rng = np.random.default_rng(6)
    x = _bf16_bits_random(rng, (3, 64))
    W = (rng.standard_normal((5, 64)) * 0.02).astype(np.float32)
    b = rng.standard_normal(5).astype(np.float32)
    l0, _ = M.router_logits(x, W)
    lb, _ = M.router_logits(x, W, b)
    assert np.array_equal(lb, (l0 + b[None, :]).astype(np.float32))


def _brute_topk(row, k):
    best = None
    for sub in itertools.combinations(range(len(row)), k):
        key = sorted(((-float(row[e]), e) for e in sub))
        if best is None or key < best:
            best = key
    return [e for _, e in best]


@pytest.mark.parametrize("E,k", [(6, 1), (8, 2), (10, 3), (12, 4)])
def test_topk_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    for trial in range(40):
        # few distinct values -> many exact ties
        row = rng.integers(-3, 3, size=E).astype(np.float32) * np.float32(0.5)
        if trial % 4 == 0:
            row = rng.standard_normal(E).astype(np.float32)
        got = M.topk(row[None, :], k)[0]
        assert list(got) == _brute_topk(row, k)


def test_topk_order_descending_then_id():
    row = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]], dtype=np.float32)
    assert list(M.topk(row, 4)[0]) == [1, 2, 4, 3]


def test_weights_identity_and_sum():
    rng = np.random.default_rng(7)
    l32 = (rng.standard_normal((50, 64)) * 2).astype(np.float32)
    idx = M.topk(l32, 8)
    w = M.topk_weights(l32, idx)
    w_full = M.topk_weights_full_softmax(l32, idx)
    assert np.allclose(w.astype(np.float64), w_full, rtol=2 ** -23, atol=0)
    assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) <= 8 * 2 ** -24)
    assert np.all(np.diff(w, axis=1) <= 0)                         # ordered like the logits
    assert np.all(M.topk_weights(l32, M.topk(l32, 1)) == 1.0)      # k = 1 -> weight 1


def test_dispatch_matches_plain_loop():
    rng = np.random.default_rng(8)
    T, k, E = 37, 5, 23
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    cnt, off, pair = M.dispatch(idx, E)
    ref_lists = [[] for _ in range(E)]
    for t in range(T):
        for j in range(k):
            ref_lists[idx[t, j]].append(t * k + j)
    assert list(cnt) == [len(l) for l in ref_lists]
    assert off[0] == 0 and off[-1] == T * k
    for e in range(E):
        assert list(pair[off[e]:off[e + 1]]) == ref_lists[e]
    assert sorted(pair.tolist()) == list(range(T * k))


def test_dispatch_empty_experts_and_single_token():
    idx = np.array([[3, 0]], dtype=np.int32)
    cnt, off, pair = M.dispatch(idx, 6)
    assert list(cnt) == [1, 0, 0, 1, 0, 0]
    assert list(off) == [0, 1, 1, 1, 2, 2, 2]
    assert list(pair) == [1, 0]


# ------------------------------------------------------ near-midpoint mask ----

def _midpoint_case(delta: float, scale: float = 1.0):
    """One logit whose exact dot product is scale * (1 + 2^-24 + delta): the FP32
    midpoint between scale and scale * (1 + 2^-23), moved by scale * delta."""
    terms = np.array([[1.0, 2.0 ** -24, delta, 0.0]]) * scale
    Wr = terms.astype(np.float32)
    assert np.all(Wr.astype(np.float64) == terms)
    x = np.full((1, 4), 0x3F80, dtype=np.uint16)                   # bf16 1.0
    return M.router_logits(x, Wr)


@pytest.mark.parametrize("scale", [1.0, 2.0 ** 10, 2.0 ** -20])
def test_near_midpoint_mask_flags_only_the_window(scale):
    # on the midpoint, and 2^-42 away on either side: flagged (inside 2^-40 relative)
    for delta in (0.0, 2.0 ** -42, -2.0 ** -42):
        _, near = _midpoint_case(delta, scale)
        assert near[0, 0], (delta, scale)
    # 2^-30 away on either side: not flagged
    for delta in (2.0 ** -30, -2.0 ** -30):
        _, near = _midpoint_case(delta, scale)
        assert not near[0, 0], (delta, scale)


def test_near_midpoint_mask_empty_at_the_decode_seeds():
    # the decode workloads' router matrices and token batches, seeds 0-3: no logit lies within
    # 2^-40 of an FP32 midpoint (about 2^-15 expected per logit), so the GPU logits must all be exact
    import synth
    for name in ("tiny_nvfp4", "decode_nvfp4", "decode_mxfp4", "decode_int4"):
        cfg = synth.CONFIGS[name]
        Wr = synth.normal_f32(synth.stream_key(0, synth.configs.KIND_ROUTER, 0, 0), cfg.E * cfg.H,
                              synth.configs.WEIGHT_SIGMA).reshape(cfg.E, cfg.H)
        for seed in range(4):
            for T in cfg.batches:
                x = synth.make_tokens(cfg, T, seed=seed, batch=T)
                _, near = M.router_logits(x, Wr)
                assert not near.any(), (name, seed, T, int(near.sum()))


def test_near_midpoint_fraction_matches_its_width():
    # random logits: the flagged fraction is about the window's share of an FP32 ulp (2 * 2^-40 / 2^-24
    # on average); a mask 2^10 wider or narrower is far outside [1/8, 8] times that
    rng = np.random.default_rng(11)
    x = _bf16_bits_random(rng, (64, 256))
    W = (rng.standard_normal((2048, 256)) * 0.02).astype(np.float32)
    _, near = M.router_logits(x, W)
    assert int(near.sum()) <= 32                                   # 131072 logits, about 4 expected


# ------------------------------------------------- bias for selection only ----

@pytest.mark.parametrize("E,k", [(8, 2), (12, 4)])
def test_bias_select_routes_by_biased_and_weighs_by_unbiased(E, k):
    # selection: brute force over every k-subset of the biased FP32 logits; weights: a softmax over all
    # unbiased logits renormalised over the selected experts (the shared denominator cancels)
    rng = np.random.default_rng(40 + E)
    x = _bf16_bits_random(rng, (6, 64))
    W = (rng.standard_normal((E, 64)) * 0.05).astype(np.float32)
    b = (rng.standard_normal(E) * 0.5).astype(np.float32)
    lsel, _, idx, w = M.route(x, W, b, k, bias_select=True)
    l0, _ = M.router_logits(x, W)
    assert np.array_equal(lsel, (l0 + b[None, :]).astype(np.float32))
    for t in range(x.shape[0]):
        assert list(idx[t]) == _brute_topk(lsel[t], k)
    p = np.exp(l0.astype(np.float64) - l0.max(axis=1, keepdims=True))
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    assert np.allclose(w.astype(np.float64), sel / sel.sum(axis=1, keepdims=True), rtol=2 ** -23, atol=0)
    # the default mode weighs by the biased logits: a different result whenever the bias is not constant
    _, _, idx_d, w_d = M.route(x, W, b, k)
    assert np.array_equal(idx_d, idx) and not np.allclose(w_d, w)
