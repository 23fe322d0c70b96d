"""Pins for the oracle's dispatch and TransferCmd descriptors: receive rows
equal the source rows bit for bit, descriptor byte totals equal the payload,
destination ranges tile each window, replaying the logged commands on a
logical send buffer rebuilds the receive buffer, brute force agrees, and the
hand-worked example's descriptors.  CPU only."""
import numpy as np
import pytest

import oracle
from oracle import brute
import workloads as W


def _setup(name, G=None):
    w = W.get(name)
    idx, wt = W.make_routing(w)
    G = oracle.default_rows_per_msg(w.hidden) if G is None else G
    lay = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, G)
    return w, idx, wt, G, lay


def test_dispatch_rows_are_source_rows():
    w, idx, wt, G, lay = _setup("tiny")
    x = W.make_x(w)
    recv = oracle.dispatch(lay, x)
    T, R = lay["token_slot"].shape
    for t in range(T):
        for d in range(R):
            s = lay["token_slot"][t, d]
            if s >= 0:
                assert np.array_equal(recv[lay["recv_base"][d] + s], x[t])
    assert np.array_equal(recv, brute.dispatch(lay, x))


def test_dispatch_partial_range_matches_full():
    w, idx, wt, G, lay = _setup("small")
    x = W.make_x(w)
    full = oracle.dispatch(lay, x)
    part = np.zeros_like(full)
    oracle.dispatch(lay, x, 100, 3000, recv=part)
    rows = (lay["recv_base"][None, :] + lay["token_slot"][100:3000])[lay["token_slot"][100:3000] >= 0]
    assert np.array_equal(part[rows], full[rows])


def test_rows_per_msg_does_not_change_recv():
    w = W.get("tiny")
    idx, _ = W.make_routing(w)
    x = W.make_x(w)
    a = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, 1)
    b = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, 8)
    assert np.array_equal(oracle.dispatch(a, x), oracle.dispatch(b, x))


def test_worked_example_descriptors(golden):
    g = golden("layout_worked_example.txt")
    R, Tpr, E, K = g["R"][0], g["tokens_per_rank"][0], g["E"][0], g["K"][0]
    idx = np.array(g["topk_idx"], np.int32).reshape(R * Tpr, K)
    lay = oracle.layout(R, Tpr, E, idx, 2)
    cmds, per = oracle.descriptors(lay, 2, 2, 16)
    assert per.tolist() == g["channel_counts"]
    got = [[int(c["dst_rank"]), int(c["size"]), int(c["src_offset"]), int(c["dst_offset"])] for c in cmds]
    assert got == g["cmd"]
    assert np.all(cmds["type"] == 0) and np.all(cmds["reserved"] == 0)


def _replay(lay, x, cmds, B):
    """Build the logical send buffer (rows ordered source, destination, row)
    and apply every command; return the receive buffer it produces."""
    T, R = lay["token_slot"].shape
    Tpr = T // R
    send_rows = []
    for s in range(R):
        for d in range(R):
            toks = [t for t in range(s * Tpr, (s + 1) * Tpr) if lay["token_slot"][t, d] >= 0]
            send_rows.extend(toks)
    send = x[np.array(send_rows, dtype=np.int64)] if send_rows else np.zeros((0,) + x.shape[1:], x.dtype)
    sb = send.view(np.uint8).reshape(-1)
    recv = np.zeros((lay["n_recv"],) + x.shape[1:], x.dtype)
    rb = recv.view(np.uint8).reshape(-1)
    covered = np.zeros(rb.shape[0], np.int32)
    for c in cmds:
        d = int(c["dst_rank"])
        base = int(lay["recv_base"][d]) * B
        dst = base + int(c["dst_offset"])
        n = int(c["size"])
        rb[dst:dst + n] = sb[int(c["src_offset"]):int(c["src_offset"]) + n]
        covered[dst:dst + n] += 1
    return recv, covered


@pytest.mark.parametrize("name,G", [("tiny", 8), ("tiny", 1), ("tiny", 3), ("small", 8)])
def test_descriptor_invariants_and_replay(name, G):
    w, idx, wt, _, lay = _setup(name, G)
    B = 2 * w.hidden
    C = w.channels or oracle.HT_CHANNELS
    cmds, per = oracle.descriptors(lay, C, G, B)
    N = lay["n_recv"]
    assert int(cmds["size"].astype(np.int64).sum()) == N * B        # bytes = payload
    assert len(cmds) == int(lay["msg_count"].sum()) == int(per.sum())
    assert np.all(cmds["size"] <= G * B) and np.all(cmds["size"] % B == 0)
    # channel = dst_rank mod C, channel-major order
    chan = np.repeat(np.arange(C), per)
    assert np.array_equal(cmds["dst_rank"] % C, chan)
    # dst ranges are disjoint and tile each window [0, recv_count[d]*B)
    for d in range(w.num_ranks):
        m = cmds[cmds["dst_rank"] == d]
        order = np.argsort(m["dst_offset"])
        starts = m["dst_offset"][order].astype(np.int64)
        ends = starts + m["size"][order]
        assert (len(m) == 0 and lay["recv_count"][d] == 0) or (
            starts[0] == 0 and np.all(starts[1:] == ends[:-1]) and ends[-1] == lay["recv_count"][d] * B)
    # src ranges tile the logical send buffer
    order = np.argsort(cmds["src_offset"])
    s0 = cmds["src_offset"][order].astype(np.int64)
    e0 = s0 + cmds["size"][order]
    assert s0[0] == 0 and np.all(s0[1:] == e0[:-1]) and e0[-1] == N * B
    if name == "tiny":
        x = W.make_x(w)
        recv, covered = _replay(lay, x, cmds, B)
        assert np.all(covered == 1)
        assert np.array_equal(recv, oracle.dispatch(lay, x))
        # brute force: the same records per channel
        bc = brute.descriptors(lay, C, G, B)
        for c in range(C):
            mine = cmds[chan == c]
            got = sorted((int(r["dst_rank"]), int(r["size"]), int(r["src_offset"]), int(r["dst_offset"]))
                         for r in mine)
            assert got == sorted(bc[c])


def test_small_workload_rings_wrap():
    # the packing workload is meant to exercise ring wraparound: ~4k messages
    # per channel against a depth of 1024
    w, idx, wt, G, lay = _setup("small")
    per = oracle.channel_counts(lay, w.channels)
    assert G == 8 and np.all(per > 3 * w.ring_depth)


# ------------------------------------------------------------------ signals

@pytest.mark.parametrize("seed", range(12))
def test_signal_counts_are_messages_per_destination(seed):
    # one increment per message: the count of TransferCmds addressed to d,
    # taken here from the brute-force descriptor list (built message by message)
    rng = np.random.default_rng(3000 + seed)
    R = int(rng.integers(1, 6))
    Tpr = int(rng.integers(1, 10))
    Er = int(rng.integers(1, 3))
    E, K = R * Er, int(rng.integers(1, min(3, R * Er) + 1))
    idx = np.stack([rng.permutation(E)[:K] for _ in range(R * Tpr)]).astype(np.int32)
    G = int(rng.choice([1, 2, 8]))
    lay = oracle.layout(R, Tpr, E, idx, G)
    sig = oracle.signal_counts(lay)
    chans = brute.descriptors(lay, 3, G, 16)
    per_d = np.zeros(R, np.uint64)
    for ch in chans:
        for (d, _, _, _) in ch:
            per_d[d] += 1
    assert np.array_equal(sig, per_d)


def test_signal_counts_worked_example(golden):
    g = golden("layout_worked_example.txt")
    R, Tpr, E, K = g["R"][0], g["tokens_per_rank"][0], g["E"][0], g["K"][0]
    idx = np.array(g["topk_idx"], np.int32).reshape(R * Tpr, K)
    # G=2: messages to rank 0: (s0,d0) 1 + (s1,d0) 1; to rank 1: (s0,d1) 1 + (s1,d1) 2
    assert oracle.signal_counts(oracle.layout(R, Tpr, E, idx, 2)).tolist() == [2, 3]
    # G=1: one message per row: the receive counts 4 and 5
    assert oracle.signal_counts(oracle.layout(R, Tpr, E, idx, 1)).tolist() == g["recv_count"]
