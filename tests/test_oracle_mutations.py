"""The oracle's pins catch plausible mistakes: each test plants one mistake in
a copy of an oracle result (on the CPU) -- a dropped count, an off-by-one
slot, a swapped pair, a wrong rank, a misplaced weight, a reversed order --
and checks that the invariant checker the pins use rejects it.  A pin that
let such a mistake through would not be a pin."""
import copy

import numpy as np
import pytest

import oracle
import workloads as W
from test_oracle_expert import check_invariants as check_expert
from test_oracle_layout import _check_invariants as check_layout


def _layout_case():
    w = W.get("tiny")
    idx, wt = W.make_routing(w)
    lay = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, 8)
    return w, idx, wt, lay


def _mutants_of_layout(lay):
    R = lay["recv_base"].shape[0]
    out = []
    m = copy.deepcopy(lay); m["num_tokens_per_expert"][0, 3] += 1; out.append(("histogram +1", m))
    m = copy.deepcopy(lay)
    t = int(np.argmax(m["token_slot"][:, 1] >= 0)); m["token_slot"][t, 1] += 1; out.append(("slot off by one", m))
    m = copy.deepcopy(lay); m["recv_base"] = np.roll(m["recv_base"], 1); out.append(("scan shifted", m))
    m = copy.deepcopy(lay); m["recv_off"] = m["recv_off"].T.copy(); out.append(("recv_off transposed", m))
    m = copy.deepcopy(lay); m["send_off"] = m["send_off"].T.copy(); out.append(("send order column-major", m))
    m = copy.deepcopy(lay); m["msg_count"] = m["num_tokens_per_rank"] // 8; out.append(("floor, not ceil", m))
    m = copy.deepcopy(lay); m["is_token_in_rank"][0, (np.argmax(lay["is_token_in_rank"][0]) + 1) % R] ^= 1
    out.append(("membership flipped", m))
    m = copy.deepcopy(lay); e = m["expert_off"]; e[1:] = e[1:] - 1; out.append(("expert_off short", m))
    return out


@pytest.mark.parametrize("i", range(8))
def test_layout_mutants_are_caught(i):
    w, idx, wt, lay = _layout_case()
    check_layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, 8, lay)     # the real one passes
    name, bad = _mutants_of_layout(lay)[i]
    with pytest.raises(AssertionError):
        check_layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, 8, bad)


def _mutants_of_expert(x, Er):
    out = []
    m = copy.deepcopy(x)
    seg = np.nonzero(m["expert_count"] >= 2)[0][0]
    off = int(np.concatenate([[0], np.cumsum(m["expert_count"])[:-1]])[seg])
    m["expert_rows"][[off, off + 1]] = m["expert_rows"][[off + 1, off]]
    out.append(("segment order reversed", m))
    m = copy.deepcopy(x); r, k = np.argwhere(m["recv_topk_idx"] >= 0)[0]
    m["recv_topk_idx"][r, k] = (m["recv_topk_idx"][r, k] + 1) % Er; out.append(("local id off by one", m))
    m = copy.deepcopy(x); r, k = np.argwhere(m["recv_topk_idx"] >= 0)[0]
    kk = (k + 1) % m["recv_topk_weights"].shape[1]
    m["recv_topk_weights"][r, [k, kk]] = m["recv_topk_weights"][r, [kk, k]]; out.append(("weight in wrong column", m))
    m = copy.deepcopy(x); m["recv_src_token"][[0, 1]] = m["recv_src_token"][[1, 0]]; out.append(("rows swapped", m))
    m = copy.deepcopy(x); m["expert_count"][0] += 1; m["expert_count"][1] -= 1; out.append(("counts moved", m))
    return out


@pytest.mark.parametrize("i", range(5))
def test_expert_mutants_are_caught(i):
    w, idx, wt, lay = _layout_case()
    x = oracle.expert_layout(lay, idx, wt, w.num_experts)
    check_expert(lay, idx, wt, w.num_experts, x)                                # the real one passes
    name, bad = _mutants_of_expert(x, w.experts_per_rank)[i]
    with pytest.raises(AssertionError):
        check_expert(lay, idx, wt, w.num_experts, bad)


def _ulps(a, b):
    """largest bf16 ulp distance between two bit arrays (sign-magnitude order)"""
    def key(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u)
    return int(np.abs(key(a) - key(b)).max())


def test_combine_mutants_are_caught():
    # the combine parity bar is 1 bf16 ulp against the brute-force combine;
    # a dropped pick, weights swapped between picks and two tokens' receive
    # slots exchanged each move some output by far more than that
    from oracle import brute
    w = W.get("tiny")
    idx, wt = W.make_routing(w)
    lay = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, 8)
    eo = W.make_x(w.replace(tokens_per_rank=(lay["n_recv"] + w.num_ranks - 1) // w.num_ranks))[:lay["n_recv"]]
    Er = w.experts_per_rank
    ref = brute.combine(lay, idx, wt, Er, eo)
    assert _ulps(oracle.combine(lay, idx, wt, Er, eo), ref) <= 1
    dropped = np.where(np.arange(idx.shape[1]) == 1, -1, idx).astype(np.int32)
    assert _ulps(oracle.combine(lay, dropped, wt, Er, eo), ref) > 1
    swapped = wt.copy()
    swapped[:, [0, 1]] = swapped[:, [1, 0]]
    assert _ulps(oracle.combine(lay, idx, swapped, Er, eo), ref) > 1
    exchanged = copy.deepcopy(lay)
    col = exchanged["token_slot"][:, 0]
    a, b = np.nonzero(col >= 0)[0][:2]
    col[[a, b]] = col[[b, a]]
    assert _ulps(oracle.combine(exchanged, idx, wt, Er, eo), ref) > 1
