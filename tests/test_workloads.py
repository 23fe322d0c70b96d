"""The seeded input generators: deterministic, the right shapes, distinct picks
per token, softmax weights, and first picks that follow the stated laws
(uniform, Zipf with s = 1.2) within sampling noise."""
import numpy as np
import pytest

import workloads as W


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_routing_shapes_and_determinism(name):
    w = W.get(name)
    a_idx, a_w = W.make_routing(w)
    b_idx, b_w = W.make_routing(w)
    assert a_idx.shape == (w.num_tokens, w.topk) and a_idx.dtype == np.int32
    assert a_w.shape == (w.num_tokens, w.topk) and a_w.dtype == np.float32
    assert np.array_equal(a_idx, b_idx) and np.array_equal(a_w, b_w)
    assert a_idx.min() >= 0 and a_idx.max() < w.num_experts
    s = np.sort(a_idx, axis=1)
    assert np.all(s[:, 1:] != s[:, :-1])                     # without replacement
    assert np.allclose(a_w.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)
    assert np.all(a_w > 0)


def test_seed_changes_routing():
    w = W.get("tiny")
    assert not np.array_equal(W.make_routing(w, seed=1)[0], W.make_routing(w, seed=2)[0])


def test_uniform_is_roughly_uniform():
    w = W.get("ll")
    idx, _ = W.make_routing(w)
    cnt = np.bincount(idx.ravel(), minlength=w.num_experts)
    mean = idx.size / w.num_experts
    assert cnt.max() < 1.5 * mean and cnt.min() > 0.5 * mean


def test_zipf_is_skewed():
    w = W.get("skew")
    idx, _ = W.make_routing(w)
    cnt = np.bincount(idx.ravel(), minlength=w.num_experts)
    per_rank = cnt.reshape(w.num_ranks, -1).sum(axis=1)
    assert per_rank.max() > 5 * per_rank.min()


def test_x_is_standard_normal_bf16():
    w = W.get("tiny")
    x = W.make_x(w)
    assert x.shape == (w.num_tokens, w.hidden) and x.dtype == np.uint16
    f = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(float(f.mean())) < 0.05 and abs(float(f.std()) - 1) < 0.05
    assert np.array_equal(x, W.make_x(w))


def _max_z(freq, p, n):
    return float(np.max(np.abs(freq - p) / np.sqrt(p * (1 - p) / n)))


def test_zipf_first_pick_follows_the_law():
    # keys are log p_e plus Gumbel noise and picks come in decreasing key
    # order, so the first pick is a Gumbel-max draw: P(first = e) = p_e exactly.
    # Compared rank by rank (the expert permutation is the generator's own).
    w = W.get("skew")
    idx, _ = W.make_routing(w)
    E, n = w.num_experts, idx.shape[0]
    p = np.arange(1, E + 1, dtype=np.float64) ** (-w.zipf_s)
    p /= p.sum()
    freq = np.sort(np.bincount(idx[:, 0], minlength=E) / n)[::-1]
    assert _max_z(freq, p, n) < 5


def test_uniform_first_pick_is_uniform():
    w = W.get("ll")
    idx, _ = W.make_routing(w)
    E, n = w.num_experts, idx.shape[0]
    freq = np.bincount(idx[:, 0], minlength=E) / n
    assert _max_z(freq, np.full(E, 1.0 / E), n) < 5


@pytest.mark.parametrize("name", ["tiny", "ll", "skew", "small"])
def test_weights_are_a_softmax_over_the_picks(name):
    w = W.get(name)
    idx, wt = W.make_routing(w)
    assert wt.dtype == np.float32 and wt.shape == idx.shape
    assert (wt > 0).all() and np.abs(wt.sum(axis=1, dtype=np.float64) - 1).max() < 1e-6
    # picks of one token are distinct (drawn without replacement)
    s = np.sort(idx, axis=1)
    assert (s[:, 1:] != s[:, :-1]).all()
