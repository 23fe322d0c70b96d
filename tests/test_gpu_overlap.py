"""Pieces of a layer for overlap: ep_dispatch_ranks over source-rank pieces
and ep_combine_tokens over token pieces must together give exactly what the
whole-layer calls give (receive rows, the TransferCmd multiset, the arrival
signals, the combined output), each piece touching only its own rows; and an
SM budget (ep_config.num_sms) must not change any result."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _helpers import (bf16_tensor_to_bits, bf16_ulp_distance, check_combine_all, check_dispatch_rows,
                      compare_descriptors, compare_layout, oracle_combine_sample, workload_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import combine_ep_layout_04_gb300  # noqa: F401  (fails loudly without libep.so)


def make_layer(w, **kw):
    from combine_ep_layout_04_gb300 import EpLayer
    opts = dict(channels=w.channels, ring_depth=w.ring_depth, max_inflight=w.max_inflight,
                rows_per_msg=w.rows_per_msg)
    opts.update(kw)
    return EpLayer(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk, **opts)


def piece_bounds(n, cuts):
    b = [0] + sorted(cuts) + [n]
    return list(zip(b[:-1], b[1:]))


@pytest.mark.parametrize("name,cuts", [("tiny", [1, 1, 3]), ("small", [5, 16, 17]), ("ll", [8, 24]),
                                       ("skew", [3, 11])])
def test_dispatch_pieces_equal_whole(name, cuts):
    w = W.get(name)
    idx, wt, x = workload_inputs(w, x_on_device=True)
    layer = make_layer(w)
    try:
        topk = torch.from_numpy(idx).cuda()
        lay = layer.layout(topk)
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
        compare_layout(lay.numpy(), lay_o)
        N, R, Tpr = lay.n_recv, w.num_ranks, w.tokens_per_rank
        recv = torch.full((N, w.hidden), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        # receive row -> source rank, from the oracle's layout
        ts = lay_o["token_slot"]
        t_idx, d_idx = np.nonzero(ts >= 0)
        row_src = np.empty(N, np.int64)
        row_src[lay_o["recv_base"][d_idx].astype(np.int64) + ts[t_idx, d_idx]] = t_idx // Tpr
        logs = [[] for _ in range(layer.cfg.channels)]
        sig_want = np.zeros(R, np.uint64)
        for (a, b) in piece_bounds(R, cuts):
            layer.dispatch(x, lay, recv, src_ranks=(a, b))
            torch.cuda.synchronize()
            assert layer.device_status() == 0
            for c, lg in enumerate(layer.cmd_log()):
                logs[c].append(lg)
            # only rows of the sources dispatched so far are written
            untouched = (recv.view(torch.int16) == -1).all(dim=1).cpu().numpy()
            assert np.array_equal(untouched, row_src >= b), (a, b)
            sig_want += lay_o["msg_count"][a:b].sum(axis=0).astype(np.uint64)
            assert np.array_equal(layer.signals(), sig_want)
        check_dispatch_rows(recv, x, lay_o)
        compare_descriptors([np.concatenate(l) for l in logs], lay_o, layer.cfg.channels, layer.G, 2 * w.hidden)
        assert np.array_equal(layer.signals(), oracle.signal_counts(lay_o))
    finally:
        layer.close()


@pytest.mark.parametrize("name", ["small", "ll"])
def test_combine_pieces_equal_whole(name):
    w = W.get(name)
    idx, wt, x = workload_inputs(w, x_on_device=True)
    layer = make_layer(w)
    try:
        topk = torch.from_numpy(idx).cuda()
        wts = torch.from_numpy(wt).cuda()
        lay = layer.layout(topk)
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
        eo = W.make_expert_out_torch(lay.n_recv, w.hidden, "cuda", w.seed)
        whole = layer.combine(eo, wts, topk, lay)
        T = w.num_tokens
        out = torch.full_like(whole.view(torch.int16), -1).view(torch.bfloat16)
        for (a, b) in piece_bounds(T, [0, 37, T // 2, T // 2, T - 1]):
            layer.combine(eo, wts, topk, lay, out=out, tokens=(a, b))
            torch.cuda.synchronize()
            written = ~(out.view(torch.int16) == -1).all(dim=1).cpu().numpy()
            assert written[:b].all() and not written[b:].any()
        assert layer.device_status() == 0
        assert torch.equal(out.view(torch.int16), whole.view(torch.int16))
        rng = np.random.default_rng(3)
        tokens = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 128, replace=False)]))
        ref = oracle_combine_sample(lay_o, idx, wt, w.experts_per_rank, eo, tokens)
        got = bf16_tensor_to_bits(out[torch.from_numpy(tokens).cuda()])
        assert bf16_ulp_distance(got, ref).max(initial=0) <= 1
    finally:
        layer.close()


@pytest.mark.parametrize("num_sms", [9, 40, 100])
def test_sm_budget_keeps_results(num_sms):
    w = W.get("small")
    idx, wt, x = workload_inputs(w, x_on_device=True)
    layer = make_layer(w, num_sms=num_sms)
    try:
        assert layer.info["dispatch_grid"] == num_sms
        topk = torch.from_numpy(idx).cuda()
        wts = torch.from_numpy(wt).cuda()
        lay = layer.layout(topk)
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
        recv = layer.dispatch(x, lay)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        check_dispatch_rows(recv, x, lay_o)
        compare_descriptors(layer.cmd_log(), lay_o, layer.cfg.channels, layer.G, 2 * w.hidden)
        out = layer.combine(recv, wts, topk, lay)
        torch.cuda.synchronize()
        T = w.num_tokens
        tokens = np.arange(0, T, 97)
        ref = oracle_combine_sample(lay_o, idx, wt, w.experts_per_rank, recv, tokens)
        got = bf16_tensor_to_bits(out[torch.from_numpy(tokens).cuda()])
        assert bf16_ulp_distance(got, ref).max(initial=0) <= 1
    finally:
        layer.close()


def test_bad_pieces_are_rejected_on_the_host():
    from combine_ep_layout_04_gb300 import _ep
    w = W.get("tiny")
    idx, wt, x = workload_inputs(w, x_on_device=True)
    layer = make_layer(w)
    try:
        topk = torch.from_numpy(idx).cuda()
        wts = torch.from_numpy(wt).cuda()
        lay = layer.layout(topk)
        recv = torch.empty((lay.n_recv, w.hidden), dtype=torch.bfloat16, device="cuda")
        for rng_ in [(-1, 2), (3, 2), (0, w.num_ranks + 1)]:
            with pytest.raises(_ep.EpError):
                layer.dispatch(x, lay, recv, src_ranks=rng_)
        for rng_ in [(-1, 2), (5, 4), (0, w.num_tokens + 1)]:
            with pytest.raises(_ep.EpError):
                layer.combine(recv, wts, topk, lay, tokens=rng_)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
    finally:
        layer.close()


def expected_chunk_tokens(T, grid, C):
    ct = 32
    while ct > 4 and T < 4 * (grid - C) * ct:
        ct //= 2
    return ct


@pytest.mark.parametrize("name,num_sms", [("ll", None), ("ht", None), ("small", None), ("ll", 40), ("tiny", 9)])
def test_dispatch_plan_follows_the_grid(name, num_sms):
    # small layers get smaller chunks so that every copy CTA has work; the
    # rule uses the grid actually launched (all SMs, or the SM budget)
    w = W.get(name)
    layer = make_layer(w, num_sms=num_sms)
    try:
        info = layer.info
        grid = info["sm_count"] if not num_sms else num_sms
        assert info["dispatch_grid"] == grid
        assert info["dispatch_chunk_tokens"] == expected_chunk_tokens(w.num_tokens, grid, layer.cfg.channels)
        if name == "ll" and num_sms is None:
            assert info["dispatch_chunk_tokens"] == 4
        if name == "ht":
            assert info["dispatch_chunk_tokens"] == 32
    finally:
        layer.close()


@pytest.mark.parametrize("compute_sms", [8, 64, 120])
def test_sm_split_partitions_are_disjoint(compute_sms):
    from combine_ep_layout_04_gb300 import SmSplit
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    with SmSplit(compute_sms) as sp:
        assert sp.compute_sms >= compute_sms and sp.comm_sms >= 1
        assert sp.comm_sms + sp.compute_sms <= n_sm
        a, b = sp.sm_ids(sp.comm), sp.sm_ids(sp.compute)
        assert not (a & b), "the partitions share SMs"
        assert len(a) <= sp.comm_sms and len(b) <= sp.compute_sms
        # 4096 blocks of 2 us reach every SM of a partition
        assert len(a) == sp.comm_sms and len(b) == sp.compute_sms
        everywhere = sp.sm_ids(torch.cuda.current_stream())
        assert len(everywhere) == n_sm


def test_sm_split_rejects_a_split_without_comm_sms():
    from combine_ep_layout_04_gb300 import SmSplit, _ep
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    for bad in (0, n_sm, n_sm + 8):
        with pytest.raises(_ep.EpError):
            SmSplit(bad)


@pytest.mark.parametrize("name", ["small", "ll"])
def test_layer_on_the_comm_partition_beside_a_gemm(name):
    # layout, dispatch and combine on the communication partition (grid =
    # its SM count) while a GEMM loop runs on the compute partition: the
    # results are the oracle's, and the GEMM's those of the same GEMM on the
    # whole GPU
    from combine_ep_layout_04_gb300 import SmSplit
    w = W.get(name)
    idx, wt, x = workload_inputs(w, x_on_device=True)
    A = torch.randn((8192, 4096), device="cuda").to(torch.bfloat16)
    B = (torch.randn((4096, 1024), device="cuda") * 0.02).to(torch.bfloat16)
    ref_y = A @ B
    with SmSplit(64) as sp:
        layer = make_layer(w, num_sms=sp.comm_sms)
        try:
            assert layer.info["dispatch_grid"] == sp.comm_sms
            topk = torch.from_numpy(idx).cuda()
            wts = torch.from_numpy(wt).cuda()
            torch.cuda.synchronize()
            ys = []
            with torch.cuda.stream(sp.compute):
                for _ in range(20):
                    ys.append(A @ B)
            with torch.cuda.stream(sp.comm):
                lay = layer.layout(topk)
                recv = layer.dispatch(x, lay)
                out = layer.combine(recv, wts, topk, lay)
            torch.cuda.synchronize()
            assert layer.device_status() == 0
            lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
            compare_layout(lay.numpy(), lay_o)
            check_dispatch_rows(recv, x, lay_o)
            compare_descriptors(layer.cmd_log(), lay_o, layer.cfg.channels, layer.G, 2 * w.hidden)
            worst = check_combine_all(out, lay_o, idx, wt, w.experts_per_rank, recv, max_ulp=1)
            assert worst <= 1
            for y in ys:
                assert torch.allclose(y.float(), ref_y.float(), rtol=1e-2, atol=1e-2)
        finally:
            layer.close()

