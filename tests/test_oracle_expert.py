"""Pins for the oracle's expert-major receive metadata: the hand-worked
example, brute force (search and sort) on tiny inputs, and invariants that
follow from the definitions: every receive row belongs to exactly one
(token, rank) and carries exactly that token's picks on that rank; every pick
appears exactly once among the expert rows; per-expert counts are the
histogram summed over source ranks; the weights a token sends out add up to
its own weights.  CPU only."""
import numpy as np
import pytest

import oracle
from oracle import brute
import workloads as W

KEYS = ["recv_topk_idx", "recv_topk_weights", "recv_src_token", "expert_rows", "expert_count"]


def test_worked_example(golden):
    g = golden("layout_worked_example.txt")
    R, Tpr, E, K = g["R"][0], g["tokens_per_rank"][0], g["E"][0], g["K"][0]
    idx = np.array(g["topk_idx"], np.int32).reshape(R * Tpr, K)
    wt = np.array(g["topk_weights"], np.float32).reshape(R * Tpr, K)
    lay = oracle.layout(R, Tpr, E, idx, 1)
    x = oracle.expert_layout(lay, idx, wt, E)
    assert x["recv_src_token"].tolist() == g["recv_src_token"]
    assert x["recv_topk_idx"].ravel().tolist() == g["recv_topk_idx"]
    assert x["recv_topk_weights"].ravel().tolist() == [float(v) for v in g["recv_topk_weights"]]
    assert x["expert_rows"].tolist() == g["expert_rows"]
    assert x["expert_count"].tolist() == g["expert_count"]


def _random_tiny(rng, allow_none=True):
    R = int(rng.integers(1, 5))
    Tpr = int(rng.integers(1, 9))
    Er = int(rng.integers(1, 4))
    E = R * Er
    K = int(rng.integers(1, min(4, E) + 1))
    T = R * Tpr
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    if allow_none:
        idx[rng.random((T, K)) < 0.15] = -1
    wt = rng.random((T, K)).astype(np.float32)
    return R, Tpr, E, K, idx, wt


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_agrees(seed):
    rng = np.random.default_rng(1000 + seed)
    R, Tpr, E, K, idx, wt = _random_tiny(rng)
    lay = oracle.layout(R, Tpr, E, idx, 1)
    a = oracle.expert_layout(lay, idx, wt, E)
    b = brute.expert_layout(brute.layout(R, Tpr, E, idx, 1), idx, wt, E)
    for k in KEYS:
        assert a[k].shape == b[k].shape, k
        assert np.array_equal(a[k].view(np.uint32) if a[k].dtype == np.float32 else a[k],
                              b[k].view(np.uint32) if b[k].dtype == np.float32 else b[k]), k


def check_invariants(lay, idx, wt, E, x):
    T, K = idx.shape
    R = lay["recv_base"].shape[0]
    Er = E // R
    N = lay["n_recv"]
    src = x["recv_src_token"]
    # each receive row belongs to exactly one (token, rank): the inverse of the slot map
    t_of = np.full(N, -1, np.int64)
    d_of = np.full(N, -1, np.int64)
    tt, dd = np.nonzero(lay["token_slot"] >= 0)
    rows = lay["recv_base"][dd] + lay["token_slot"][tt, dd]
    t_of[rows], d_of[rows] = tt, dd
    assert np.array_equal(np.sort(rows), np.arange(N))
    assert np.array_equal(src, t_of)
    # the row's picks are the token's picks on the row's rank, as local ids
    tok_picks = idx[src]
    on_rank = (tok_picks >= 0) & (tok_picks // Er == d_of[:, None])
    assert np.array_equal(x["recv_topk_idx"], np.where(on_rank, tok_picks - d_of[:, None] * Er, -1))
    assert np.array_equal(x["recv_topk_weights"], np.where(on_rank, wt[src], np.float32(0)))
    assert (on_rank.sum(axis=1) >= 1).all()          # a row exists only for a rank with a pick
    # every pick appears exactly once among the expert rows
    cnt = x["expert_count"]
    assert np.array_equal(cnt, np.bincount(idx[idx >= 0], minlength=E))
    assert np.array_equal(cnt, lay["num_tokens_per_expert"].sum(axis=0))
    er = x["expert_rows"]
    assert er.shape[0] == int((idx >= 0).sum())
    off = lay["expert_off"]
    seen = set()
    for e in range(E):
        seg = er[off[e]:off[e] + cnt[e]]
        assert (np.diff(seg) > 0).all()              # increasing receive rows
        for r in seg:
            assert e - (e // Er) * Er in x["recv_topk_idx"][r] and d_of[r] == e // Er
            seen.add((int(src[r]), e))
    assert seen == {(t, int(e)) for t in range(T) for e in idx[t] if e >= 0}
    # weight mass: a token's rows carry exactly its weights, once each
    mass = np.zeros(T, np.float64)
    np.add.at(mass, src, x["recv_topk_weights"].astype(np.float64).sum(axis=1))
    assert np.array_equal(mass, np.where(idx >= 0, wt, 0).astype(np.float64).sum(axis=1))


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_invariants_on_workloads(name):
    w = W.get(name)
    if name == "small":
        w = w.replace(tokens_per_rank=64)
    idx, wt = W.make_routing(w)
    lay = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, 1)
    x = oracle.expert_layout(lay, idx, wt, w.num_experts)
    check_invariants(lay, idx, wt, w.num_experts, x)


@pytest.mark.parametrize("seed", range(10))
def test_invariants_random_with_empty_picks(seed):
    rng = np.random.default_rng(2000 + seed)
    R, Tpr, E, K, idx, wt = _random_tiny(rng)
    lay = oracle.layout(R, Tpr, E, idx, 1)
    check_invariants(lay, idx, wt, E, oracle.expert_layout(lay, idx, wt, E))


def test_one_rank_is_the_identity_grouping():
    # R = 1: receive row n is token n; expert rows are the tokens of each expert in order
    rng = np.random.default_rng(7)
    T, E, K = 20, 6, 2
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    wt = rng.random((T, K)).astype(np.float32)
    lay = oracle.layout(1, T, E, idx, 1)
    x = oracle.expert_layout(lay, idx, wt, E)
    assert np.array_equal(x["recv_src_token"], np.arange(T))
    assert np.array_equal(x["recv_topk_idx"], idx)
    want = np.concatenate([np.nonzero((idx == e).any(axis=1))[0] for e in range(E)])
    assert np.array_equal(x["expert_rows"], want)


def test_all_picks_to_one_expert():
    R, Tpr, E = 4, 8, 8
    idx = np.full((R * Tpr, 1), 5, np.int32)
    wt = np.ones((R * Tpr, 1), np.float32)
    lay = oracle.layout(R, Tpr, E, idx, 1)
    x = oracle.expert_layout(lay, idx, wt, E)
    assert x["expert_count"].tolist() == [0, 0, 0, 0, 0, R * Tpr, 0, 0]
    assert np.array_equal(x["expert_rows"], np.arange(R * Tpr))   # rank 2's window, in token order
    assert (x["recv_topk_idx"] == 1).all()


def test_duplicate_pick_is_rejected():
    idx = np.array([[0, 1], [2, 2]], np.int32)
    wt = np.ones((2, 2), np.float32)
    lay = oracle.layout(2, 1, 4, idx, 1)        # the layout itself counts duplicates
    with pytest.raises(oracle.OracleError):
        oracle.expert_layout(lay, idx, wt, 4)
