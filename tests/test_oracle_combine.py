"""Pins for the oracle's combine: bf16 rounding against torch's conversion and
exact rationals, fmaf against exact rounding, brute force on tiny inputs, and
the identity-expert invariant (dispatch -> identity expert -> combine returns
x scaled by the sum of the token's top-k weights).  CPU only."""
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
import workloads as W


def _f32(bits):
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def test_bf16_rounding_matches_torch_and_exact():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    # add exact ties (low half = 0x8000) and their neighbours
    ties = (rng.integers(0, 2**16, size=3000).astype(np.uint32) << 16) | 0x8000
    bits = np.concatenate([bits, ties, ties + 1, ties - 1])
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) < 3e38)]
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = np.array([oracle.f32_to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(mine, ref)
    for v in vals[:400]:
        assert oracle.f32_to_bf16(float(v)) == brute.round_to_bf16_bits(float(v))


def test_bf16_decode():
    for b in [0x0000, 0x8000, 0x3F80, 0xBF80, 0x7F7F, 0x0001, 0x4049]:
        assert oracle.bf16_to_f32(b) == _f32(b << 16)


def test_fmaf_is_rounded_once():
    rng = np.random.default_rng(1)
    a = rng.standard_normal(3000).astype(np.float32)
    b = rng.standard_normal(3000).astype(np.float32)
    c = (rng.standard_normal(3000) * 4).astype(np.float32)
    for x, y, z in zip(a, b, c):
        got = oracle.fmaf(float(x), float(y), float(z))
        assert got == brute.fma_f32(float(x), float(y), float(z))
    # a case where a separate multiply and add would differ from one rounding
    x = 1.0 + 2.0**-12
    exact = Fraction(x) * Fraction(x) - Fraction(1.0)
    assert oracle.fmaf(x, x, -1.0) == float(exact)


def _tiny():
    w = W.get("tiny")
    idx, wt = W.make_routing(w)
    lay = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, 8)
    return w, idx, wt, lay


def test_combine_brute_force_on_tiny():
    w, idx, wt, lay = _tiny()
    rng = np.random.default_rng(3)
    eo = W.bf16_bits_from_f32(rng.standard_normal((lay["n_recv"], w.hidden), dtype=np.float32))
    got = oracle.combine(lay, idx, wt, w.experts_per_rank, eo)
    assert np.array_equal(got, brute.combine(lay, idx, wt, w.experts_per_rank, eo))


def test_combine_with_empty_picks_brute_force():
    rng = np.random.default_rng(4)
    R, Tpr, E, K, H = 3, 5, 9, 3, 24
    idx = np.stack([rng.permutation(E)[:K] for _ in range(R * Tpr)]).astype(np.int32)
    idx[rng.random(idx.shape) < 0.25] = -1
    wt = rng.random((R * Tpr, K)).astype(np.float32)
    lay = oracle.layout(R, Tpr, E, idx, 1)
    eo = W.bf16_bits_from_f32(rng.standard_normal((max(lay["n_recv"], 1), H), dtype=np.float32))
    got = oracle.combine(lay, idx, wt, E // R, eo)
    assert np.array_equal(got, brute.combine(lay, idx, wt, E // R, eo))
    # a token with no picks at all combines to +0
    idx[0, :] = -1
    lay = oracle.layout(R, Tpr, E, idx, 1)
    got = oracle.combine(lay, idx, wt, E // R, eo[:max(lay["n_recv"], 1)])
    assert np.all(got[0] == 0)


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_identity_expert_returns_weighted_x(name):
    w = W.get(name)
    idx, wt = W.make_routing(w)
    G = oracle.default_rows_per_msg(w.hidden)
    lay = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, G)
    x = W.make_x(w)
    recv = oracle.dispatch(lay, x)
    T = min(w.num_tokens, 2048)
    out = oracle.combine(lay, idx, wt, w.experts_per_rank, recv, 0, T)
    xf = _bf16_to_f64(x[:T])
    sw = wt[:T].astype(np.float64).sum(axis=1, keepdims=True)
    ref = xf * sw
    got = _bf16_to_f64(out)
    # one bf16 rounding (half an ulp of 2^-8 relative) plus the fp32 chain's
    # reassociation error (K roundings of 2^-24 relative to sum |w x|)
    K = w.topk
    bound = np.abs(ref) * 2.0**-8 + K * 2.0**-23 * np.abs(xf) * sw + 1e-30
    assert np.all(np.abs(got - ref) <= bound)


def test_top1_unit_weight_returns_x_exactly():
    rng = np.random.default_rng(5)
    R, Tpr, E, H = 4, 6, 8, 40
    idx = rng.integers(0, E, size=(R * Tpr, 1)).astype(np.int32)
    wt = np.ones((R * Tpr, 1), np.float32)
    lay = oracle.layout(R, Tpr, E, idx, 1)
    x = W.bf16_bits_from_f32(rng.standard_normal((R * Tpr, H), dtype=np.float32))
    out = oracle.combine(lay, idx, wt, E // R, oracle.dispatch(lay, x))
    assert np.array_equal(out, x)


def test_single_rank_equal_weights_is_mean():
    # R = 1, all K picks on the one rank, w = 1/K with K a power of two: each
    # product is exact and so is the sum of K equal terms, so out = x exactly.
    rng = np.random.default_rng(6)
    T, E, K, H = 16, 8, 4, 32
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    wt = np.full((T, K), 1.0 / K, np.float32)
    lay = oracle.layout(1, T, E, idx, 1)
    x = W.bf16_bits_from_f32(rng.standard_normal((T, H), dtype=np.float32))
    out = oracle.combine(lay, idx, wt, E, oracle.dispatch(lay, x))
    assert np.array_equal(out, x)


def test_combine_rejects_rows_outside_expert_out():
    w, idx, wt, lay = _tiny()
    eo = np.zeros((lay["n_recv"] - 1, w.hidden), np.uint16)
    with pytest.raises(oracle.OracleError):
        oracle.combine(lay, idx, wt, w.experts_per_rank, eo)


def test_worked_example(golden):
    """A combine worked out by hand (tests/golden/combine_worked_example.txt):
    ties to even both ways, a negative tie, an exact cancellation to +0, a
    round up, and two picks on one rank reading the same row."""
    g = golden("combine_worked_example.txt")
    R, Tpr, E, K, H = g["R"][0], g["tokens_per_rank"][0], g["E"][0], g["K"][0], g["H"][0]
    idx = np.array(g["topk_idx"], np.int32).reshape(R * Tpr, K)
    wts = np.array(g["topk_weight_bits"], np.uint32).view(np.float32).reshape(R * Tpr, K)
    lay = oracle.layout(R, Tpr, E, idx, oracle.default_rows_per_msg(H))
    assert lay["token_slot"].ravel().tolist() == g["token_slot"]
    assert lay["recv_base"].tolist() == g["recv_base"]
    eo = np.array(g["expert_out_bits"], np.uint16)
    want = np.array(g["out_bits"], np.uint16)
    assert np.array_equal(oracle.combine(lay, idx, wts, E // R, eo), want)
    assert np.array_equal(brute.combine(lay, idx, wts, E // R, eo), want)

