"""Pins for the oracle's layout: a hand-worked example, brute force on tiny
inputs, textbook routines (bincount, cumsum) and the invariants the EP
articles fix (counts sum to tokens x top-k; the dispatch map is a bijection
onto receive slots).  CPU only."""
import numpy as np
import pytest

import oracle
from oracle import brute
import workloads as W

KEYS = ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "token_slot",
        "recv_off", "send_off", "msg_count", "recv_count", "recv_base", "expert_off"]


def test_worked_example(golden):
    g = golden("layout_worked_example.txt")
    R, Tpr, E, K = g["R"][0], g["tokens_per_rank"][0], g["E"][0], g["K"][0]
    idx = np.array(g["topk_idx"], np.int32).reshape(R * Tpr, K)
    for G, key in [(1, "msg_count_G1"), (2, "msg_count_G2")]:
        lay = oracle.layout(R, Tpr, E, idx, G)
        assert lay["num_tokens_per_expert"].ravel().tolist() == g["num_tokens_per_expert"]
        assert lay["num_tokens_per_rank"].ravel().tolist() == g["num_tokens_per_rank"]
        assert lay["is_token_in_rank"].ravel().tolist() == g["is_token_in_rank"]
        assert lay["token_slot"].ravel().tolist() == g["token_slot"]
        assert lay["recv_count"].tolist() == g["recv_count"]
        assert lay["recv_base"].tolist() == g["recv_base"]
        assert lay["n_recv"] == g["n_recv"][0]
        assert lay["recv_off"].ravel().tolist() == g["recv_off"]
        assert lay["send_off"].ravel().tolist() == g["send_off"]
        assert lay["expert_off"].tolist() == g["expert_off"]
        assert lay["msg_count"].ravel().tolist() == g[key]


def _random_tiny(rng, allow_none=True):
    R = int(rng.integers(1, 5))
    Tpr = int(rng.integers(1, 9))
    Er = int(rng.integers(1, 4))
    E = R * Er
    K = int(rng.integers(1, min(3, E) + 1))
    T = R * Tpr
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    if allow_none:
        drop = rng.random((T, K)) < 0.15
        idx[drop] = -1
    G = int(rng.choice([1, 2, 3, 8]))
    return R, Tpr, E, K, G, idx


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_agrees(seed):
    rng = np.random.default_rng(seed)
    R, Tpr, E, K, G, idx = _random_tiny(rng)
    a = oracle.layout(R, Tpr, E, idx, G)
    b = brute.layout(R, Tpr, E, idx, G)
    for k in KEYS:
        assert np.array_equal(a[k], b[k]), k
    assert a["n_recv"] == b["n_recv"]


def _check_invariants(R, Tpr, E, idx, G, lay):
    T, K = idx.shape
    Er = E // R
    valid = idx >= 0
    # counts sum to tokens x top-k (less the empty picks)
    assert lay["num_tokens_per_expert"].sum() == int(valid.sum())
    # per-expert histogram = bincount of the picks of each source rank
    for s in range(R):
        picks = idx[s * Tpr:(s + 1) * Tpr][valid[s * Tpr:(s + 1) * Tpr]]
        assert np.array_equal(lay["num_tokens_per_expert"][s], np.bincount(picks, minlength=E))
    # membership = any pick on that rank
    member = np.zeros((T, R), bool)
    for k in range(K):
        ok = valid[:, k]
        member[np.nonzero(ok)[0], idx[ok, k] // Er] = True
    assert np.array_equal(lay["is_token_in_rank"].astype(bool), member)
    cnt = member.reshape(R, Tpr, R).sum(axis=1)
    assert np.array_equal(lay["num_tokens_per_rank"], cnt)
    # dedup: a rank counts a token at most once, never more than its picks there
    for s in range(R):
        for d in range(R):
            assert cnt[s, d] <= lay["num_tokens_per_expert"][s, d * Er:(d + 1) * Er].sum()
    N = int(member.sum())
    assert lay["n_recv"] == N == int(cnt.sum())
    # scans = shifted cumulative sums
    rc = cnt.sum(axis=0)
    assert np.array_equal(lay["recv_count"], rc)
    assert np.array_equal(lay["recv_base"], np.concatenate([[0], np.cumsum(rc)[:-1]]))
    assert np.array_equal(lay["recv_off"], np.vstack([np.zeros((1, R), int), np.cumsum(cnt, axis=0)[:-1]]))
    flat = cnt.ravel()
    assert np.array_equal(lay["send_off"].ravel(), np.concatenate([[0], np.cumsum(flat)[:-1]]))
    assert np.array_equal(lay["msg_count"], -(-cnt // G))
    tot_e = lay["num_tokens_per_expert"].sum(axis=0)
    assert np.array_equal(lay["expert_off"], np.concatenate([[0], np.cumsum(tot_e)[:-1]]))
    # slots: within column d, the members in token order get 0, 1, 2, ...
    ts = lay["token_slot"]
    for d in range(R):
        col = ts[:, d]
        assert np.array_equal(col[member[:, d]], np.arange(member[:, d].sum()))
        assert np.all(col[~member[:, d]] == -1)
    # bijection: (t, d) -> recv_base[d] + slot hits every row of [0, N) once
    rows = (lay["recv_base"][None, :] + ts)[member]
    assert np.array_equal(np.sort(rows), np.arange(N))


@pytest.mark.parametrize("name", ["tiny", "ll", "small", "skew", "ht"])
def test_invariants_on_workloads(name):
    w = W.get(name)
    idx, _ = W.make_routing(w)
    G = oracle.default_rows_per_msg(w.hidden)
    lay = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, G)
    _check_invariants(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, G, lay)


@pytest.mark.parametrize("seed", range(10))
def test_invariants_random(seed):
    rng = np.random.default_rng(1000 + seed)
    R = int(rng.integers(1, 9))
    Tpr = int(rng.integers(1, 70))
    Er = int(rng.integers(1, 5))
    E = R * Er
    K = int(rng.integers(1, min(6, E) + 1))
    idx = np.stack([rng.permutation(E)[:K] for _ in range(R * Tpr)]).astype(np.int32)
    idx[rng.random(idx.shape) < 0.1] = -1
    G = int(rng.integers(1, 10))
    _check_invariants(R, Tpr, E, idx, G, oracle.layout(R, Tpr, E, idx, G))


def test_expected_receive_rows_uniform():
    # Uniform K-of-E picks: P(token reaches rank d) = 1 - C(E-Er, K) / C(E, K).
    from math import comb
    for name in ["ll", "ht", "small"]:
        w = W.get(name)
        idx, _ = W.make_routing(w)
        lay = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, 1)
        p = 1 - comb(w.num_experts - w.experts_per_rank, w.topk) / comb(w.num_experts, w.topk)
        expect = w.num_tokens * w.num_ranks * p
        assert abs(lay["n_recv"] - expect) < 0.01 * expect


def test_single_rank_is_identity():
    rng = np.random.default_rng(7)
    T, E, K = 50, 6, 3
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    lay = oracle.layout(1, T, E, idx, 1)
    assert np.array_equal(lay["token_slot"][:, 0], np.arange(T))
    assert lay["n_recv"] == T


def test_top1_has_no_dedup():
    rng = np.random.default_rng(8)
    R, Tpr, E = 4, 10, 8
    idx = rng.integers(0, E, size=(R * Tpr, 1)).astype(np.int32)
    lay = oracle.layout(R, Tpr, E, idx, 1)
    assert lay["n_recv"] == R * Tpr
    assert np.array_equal(lay["num_tokens_per_rank"].sum(axis=1), np.full(R, Tpr))


def test_all_tokens_to_one_expert():
    R, Tpr, E, K = 4, 8, 8, 2
    idx = np.tile(np.array([[5, 4]], np.int32), (R * Tpr, 1))  # both on rank 2
    lay = oracle.layout(R, Tpr, E, idx, 8)
    assert lay["n_recv"] == R * Tpr
    assert lay["recv_count"].tolist() == [0, 0, R * Tpr, 0]
    assert np.array_equal(lay["token_slot"][:, 2], np.arange(R * Tpr))
    assert lay["num_tokens_per_expert"][:, 5].tolist() == [Tpr] * R


def test_all_picks_empty():
    idx = np.full((12, 3), -1, np.int32)
    lay = oracle.layout(3, 4, 6, idx, 8)
    assert lay["n_recv"] == 0 and np.all(lay["token_slot"] == -1)
    assert lay["msg_count"].sum() == 0


@pytest.mark.parametrize("bad", [-2, 16, 99])
def test_out_of_range_pick_is_rejected(bad):
    idx = np.zeros((8, 2), np.int32)
    idx[:, 1] = 1
    idx[5, 1] = bad
    with pytest.raises(oracle.OracleError):
        oracle.layout(2, 4, 16, idx, 1)


def test_rows_per_msg_rule(golden):
    g = golden("tuning_table.txt")
    thr = g["PACK_THRESHOLD_BYTES"][0]
    assert oracle.PACK_THRESHOLD_BYTES == thr and oracle.PACK_ROWS == g["PACK_ROWS"][0]
    # the five workloads: tiny 512 B, small 2 KB (the workload names 8 rows),
    # skew 4 KB rows -> packed; the DeepSeek-V3 shapes (14 KB rows) are not.
    assert oracle.default_rows_per_msg(256) == 8
    assert oracle.default_rows_per_msg(1024) == 8 == W.get("small").rows_per_msg
    assert oracle.default_rows_per_msg(2048) == 8
    assert oracle.default_rows_per_msg(7168) == 1
    assert oracle.default_rows_per_msg(3584) == 1   # exactly 7 KB is not "under 7 KB"
    assert oracle.default_rows_per_msg(3576) == 8
