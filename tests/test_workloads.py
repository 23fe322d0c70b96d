"""The seeded input generators: deterministic, the right shapes, distinct picks
per token, softmax weights, and a skewed workload that is actually skewed."""
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
