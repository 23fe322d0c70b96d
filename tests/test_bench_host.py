"""Host-side logic of bench.py (no GPU): the message-size sweep's range, the
algorithmic byte counts on a layer small enough to count by hand, the CPU
baseline's sample shares, and the DRAM-traffic lookup's source check."""
import os

import numpy as np

import bench
import oracle
import workloads as W


def test_sweep_spans_1kb_to_16mb_messages_and_1kb_to_1mb_rows():
    pts = bench.sweep_points()
    msg = sorted(b * g for b, g in pts)
    rows = sorted({b for b, _ in pts})
    assert msg[0] == 1024 and msg[-1] >= 16 * 2**20 - 8192
    assert rows[0] == 1024 and rows[-1] == 2**20
    # 2, 4, 8 and 16 MB messages are all timed
    for mb in (2, 4, 8, 16):
        assert any(abs(b * g - mb * 2**20) <= 8192 for b, g in pts), mb
    # G never exceeds what a ring slot's 11-bit row field holds
    assert max(g for _, g in pts) <= 2047
    # the packing study: 4 KB and 7 KB rows at one and at eight rows a message
    for b in (4096, 7168):
        assert (b, 1) in pts and (b, 8) in pts


def test_algorithmic_bytes_of_a_hand_counted_layer():
    # 2 ranks x 2 tokens, H = 4 (8-byte rows), 2 experts, K = 1; tokens 0, 1
    # on rank 0 pick experts 0 and 1; tokens 2, 3 on rank 1 pick 1 and 1.
    idx = np.array([[0], [1], [1], [1]], np.int32)
    lay = oracle.layout(2, 2, 2, idx, 8)
    N = lay["n_recv"]
    assert N == 4
    n_msgs = int(lay["msg_count"].sum())
    n_sent = int((lay["is_token_in_rank"].sum(axis=1) > 0).sum())
    ab = bench.algorithmic_bytes(2, 4, 4, 2, 1, N, n_msgs, n_sent)
    B = 8
    # dispatch: read each sent token once, write each receive row, read the
    # token_slot table, write one 32-byte record per message
    assert ab["dispatch"] == 4 * B + 4 * B + 4 * 2 * 4 + n_msgs * 32
    # combine: read each receive row, write each token, read the picks and
    # weights and the token_slot table
    assert ab["combine"] == 4 * B + 4 * B + 4 * 1 * 8 + 4 * 2 * 4
    assert n_msgs == 3   # pairs (0,0), (0,1), (1,1) with G = 8


def test_cpu_sample_shares_cover_every_workload():
    assert set(bench.CPU_FRACTION) == {"tiny", "ll", "ht", "skew", "small"}
    for name, frac in bench.CPU_FRACTION.items():
        w = W.get(name)
        s_end = max(1, round(frac * w.num_ranks))
        assert 0 < s_end <= w.num_ranks


def test_traffic_is_reported_only_for_the_current_source(tmp_path, monkeypatch):
    sha = bench.kernel_src_sha("dispatch")
    assert sha is not None and len(sha) == 16
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic.txt").write_text(
        "# comment\n"
        f"kernel=dispatch workload=ht src_sha={sha} dram_bytes_per_launch=123\n"
        "kernel=combine workload=ht src_sha=0000000000000000 dram_bytes_per_launch=456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the sha is computed from the sources under ROOT: point those at the repo
    csrc_real = os.path.join(os.path.dirname(os.path.abspath(bench.__file__)), "combine_ep_layout_04_gb300")
    os.symlink(csrc_real, tmp_path / "combine_ep_layout_04_gb300")
    assert bench.read_traffic("dispatch", "ht") == 123
    assert bench.read_traffic("combine", "ht") is None     # taken on other code
    assert bench.read_traffic("dispatch", "ll") is None    # no line for it
