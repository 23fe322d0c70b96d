"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the five
workloads and on edge cases.  Layout, receive rows and TransferCmd records
must be bit-exact; combine within 1 bf16 ulp per element (the stated
tolerance; the kernel uses the oracle's fmaf order, so it is expected to be
exact)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _helpers import (bf16_tensor_to_bits, bf16_ulp_distance, check_combine_all, check_dispatch_rows,
                      check_identity_all, check_ring_invariants, compare_descriptors, compare_layout,
                      oracle_combine_sample, workload_inputs)

pytestmark = pytest.mark.gpu

COMBINE_ULP = 1


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


def run_and_check(w, *, x_on_device=False, identity_check=True, **kw):
    idx, wt, x = workload_inputs(w, x_on_device=x_on_device)
    layer = make_layer(w, **kw)
    try:
        G = layer.G
        if "rows_per_msg" not in kw and w.rows_per_msg is None:
            assert G == oracle.default_rows_per_msg(w.hidden)
        topk = torch.from_numpy(idx).cuda()
        wts = torch.from_numpy(wt).cuda()
        lay = layer.layout(topk)
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, G)
        compare_layout(lay.numpy(), lay_o)
        before = layer.ring_stats()
        recv = layer.dispatch(x, lay)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        check_dispatch_rows(recv, x, lay_o)
        logs = layer.cmd_log()
        compare_descriptors(logs, lay_o, layer.cfg.channels, G, 2 * w.hidden)
        check_ring_invariants(layer, logs, lay_o, before)

        N = lay_o["n_recv"]
        eo = W.make_expert_out_torch(N, w.hidden, "cuda", w.seed)
        out = layer.combine(eo, wts, topk, lay)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        # every token and every element against the oracle
        worst = check_combine_all(out, lay_o, idx, wt, w.experts_per_rank, eo, COMBINE_ULP)
        print(f"combine {w.name}: {w.num_tokens} tokens x {w.hidden}, max ulp {worst}")
        del eo, out

        if identity_check:
            # dispatch -> identity expert -> combine == x * sum_k w, every token
            out_id = layer.combine(recv, wts, topk, lay)
            torch.cuda.synchronize()
            check_identity_all(out_id, x, wt, w.topk)
        return layer, lay_o
    finally:
        layer.close()


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_workload_full(name):
    run_and_check(W.get(name))


def test_workload_ll():
    run_and_check(W.get("ll"))


def test_workload_skew():
    run_and_check(W.get("skew"), x_on_device=True)


def test_workload_ht():
    run_and_check(W.get("ht"), x_on_device=True)


# ------------------------------------------------------------------ edge cases

def _w(**kw):
    base = W.Workload("edge", 4, 16, 256, 16, 2, seed=11)
    return base.replace(**kw)


@pytest.mark.parametrize("kw", [
    dict(num_ranks=1, tokens_per_rank=70, num_experts=4, topk=2),             # one rank: identity
    dict(num_ranks=5, tokens_per_rank=45, num_experts=15, topk=3),            # ragged tokens, R % C != 0
    dict(num_ranks=12, tokens_per_rank=33, num_experts=24, topk=1),           # top-1: no dedup
    dict(num_ranks=8, tokens_per_rank=40, hidden=8, num_experts=16, topk=4),  # 16-byte rows
    dict(num_ranks=6, tokens_per_rank=37, hidden=72, num_experts=12, topk=3),
    dict(num_ranks=4, tokens_per_rank=20, hidden=12288, num_experts=8, topk=3),  # 24 KB rows: 2 pieces
    dict(num_ranks=3, tokens_per_rank=17, hidden=9000, num_experts=9, topk=2),   # 18 KB rows, odd pieces
    dict(num_ranks=64, tokens_per_rank=40, hidden=64, num_experts=128, topk=8),  # the most ranks
    dict(num_ranks=33, tokens_per_rank=9, hidden=32, num_experts=66, topk=5),    # two column groups
    dict(num_ranks=4, tokens_per_rank=300, hidden=128, num_experts=64, topk=32),  # the largest top-k
    dict(num_ranks=64, tokens_per_rank=24, hidden=2048, num_experts=256, topk=8),  # 4 KB rows, 64 ranks
    dict(num_ranks=16, tokens_per_rank=1, hidden=1024, num_experts=32, topk=4),    # one token per rank
    dict(num_ranks=8, tokens_per_rank=97, hidden=2056, num_experts=32, topk=6),    # 4112-byte rows: TMA path
    dict(num_ranks=6, tokens_per_rank=40, hidden=14336, num_experts=12, topk=3),   # 28 KB rows: 2 pieces
    dict(num_ranks=4, tokens_per_rank=24, hidden=28672, num_experts=8, topk=2),    # 56 KB rows: 4 pieces
    dict(num_ranks=2, tokens_per_rank=12, hidden=524288, num_experts=2, topk=2),   # 1 MB rows: 64 pieces
])
def test_edge_shapes(kw):
    run_and_check(_w(**kw))


def test_one_16mb_message():
    # one rank, 2047 rows of 8 KB in one message (the most a message holds):
    # a 16 MB TransferCmd
    w = _w(num_ranks=1, tokens_per_rank=2047, hidden=4096, num_experts=1, topk=1)
    layer, lay_o = run_and_check(w, rows_per_msg=2047)
    ref, per = oracle.descriptors(lay_o, 8, 2047, 2 * 4096)
    assert len(ref) == 1 and int(ref["size"][0]) == 2047 * 8192


@pytest.mark.parametrize("opts", [
    dict(rows_per_msg=1), dict(rows_per_msg=3), dict(rows_per_msg=64), dict(batch=1), dict(channels=1),
    dict(channels=3), dict(ring_depth=16, max_inflight=8), dict(ring_depth=64, max_inflight=64, batch=5),
    dict(drain_batch=64), dict(ring_depth=8192, max_inflight=8192), dict(rows_per_msg=2047),
    dict(drain_batch=512, max_inflight=512), dict(rows_per_msg=3, debug_flags=2),
    dict(rows_per_msg=64, debug_flags=2), dict(rows_per_msg=5, channels=1, debug_flags=2),
])
def test_ring_options(opts):
    w = _w(num_ranks=8, tokens_per_rank=100, hidden=512, num_experts=32, topk=4)
    run_and_check(w, **opts)


@pytest.mark.parametrize("dev_counters", [False, True])
def test_multi_row_messages_twice(dev_counters):
    # messages of 4 rows spanning chunks, posted by whichever chunk lands last;
    # a second call on the same handle finds every counter back at zero
    from combine_ep_layout_04_gb300 import _ep
    w = W.get("small")
    idx, wt, x = workload_inputs(w)
    with make_layer(w, rows_per_msg=4, debug_flags=_ep.EP_DEBUG_DEVICE_COUNTERS if dev_counters else 0) as layer:
        topk = torch.from_numpy(idx).cuda()
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, 4)
        for _ in range(2):
            lay = layer.layout(topk)
            recv = layer.dispatch(x, lay)
            torch.cuda.synchronize()
            assert layer.device_status() == 0
            check_dispatch_rows(recv, x, lay_o)
            compare_descriptors(layer.cmd_log(), lay_o, layer.cfg.channels, 4, 2 * w.hidden)


def test_many_destinations_per_channel():
    # 64 ranks on one ring: the posters' per-destination ranges then take so
    # much shared memory that fewer poster warps run
    w = _w(num_ranks=64, tokens_per_rank=9, hidden=2056, num_experts=448, topk=8)
    run_and_check(w, channels=1, ring_depth=256, max_inflight=8, batch=2, rows_per_msg=3)


def test_small_rings_wrap_many_times():
    w = W.get("small")
    run_and_check(w, ring_depth=32, max_inflight=16, identity_check=False)


def test_all_tokens_to_one_expert():
    w = _w(num_ranks=8, tokens_per_rank=64, hidden=256, num_experts=16, topk=2)
    from combine_ep_layout_04_gb300 import EpLayer
    idx = np.tile(np.array([[5, 4]], np.int32), (w.num_tokens, 1))      # both on rank 2
    wt = np.full((w.num_tokens, 2), 0.5, np.float32)
    x = torch.randn(w.num_tokens, w.hidden, device="cuda").to(torch.bfloat16)
    with EpLayer(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk) as layer:
        topk = torch.from_numpy(idx).cuda()
        lay = layer.layout(topk)
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
        compare_layout(lay.numpy(), lay_o)
        recv = layer.dispatch(x, lay)
        check_dispatch_rows(recv, x, lay_o)
        compare_descriptors(layer.cmd_log(), lay_o, layer.cfg.channels, layer.G, 2 * w.hidden)
        out = layer.combine(recv, torch.from_numpy(wt).cuda(), topk, lay)
        # two picks of weight 1/2 on the same row: exactly x
        assert torch.equal(out.view(torch.int16), x.view(torch.int16))


def test_all_picks_empty():
    w = _w(num_ranks=4, tokens_per_rank=50, hidden=64, num_experts=8, topk=3)
    from combine_ep_layout_04_gb300 import EpLayer
    idx = np.full((w.num_tokens, 3), -1, np.int32)
    with EpLayer(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk) as layer:
        topk = torch.from_numpy(idx).cuda()
        lay = layer.layout(topk)
        assert lay.n_recv == 0
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
        compare_layout(lay.numpy(), lay_o)
        x = torch.randn(w.num_tokens, w.hidden, device="cuda").to(torch.bfloat16)
        recv = torch.empty((8, w.hidden), dtype=torch.bfloat16, device="cuda")
        layer.dispatch(x, lay, recv)
        assert all(len(l) == 0 for l in layer.cmd_log())
        out = layer.combine(recv, torch.ones((w.num_tokens, 3), device="cuda"), topk, lay)
        assert layer.device_status() == 0
        assert torch.equal(out.float(), torch.zeros_like(out.float()))


def test_some_picks_empty():
    w = _w(num_ranks=6, tokens_per_rank=41, hidden=96, num_experts=18, topk=4)
    from combine_ep_layout_04_gb300 import EpLayer
    idx, wt = W.make_routing(w)
    rng = np.random.default_rng(3)
    idx[rng.random(idx.shape) < 0.3] = -1
    with EpLayer(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk) as layer:
        topk = torch.from_numpy(idx).cuda()
        lay = layer.layout(topk)
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
        compare_layout(lay.numpy(), lay_o)
        x = torch.randn(w.num_tokens, w.hidden, device="cuda").to(torch.bfloat16)
        recv = layer.dispatch(x, lay)
        check_dispatch_rows(recv, x, lay_o)
        compare_descriptors(layer.cmd_log(), lay_o, layer.cfg.channels, layer.G, 2 * w.hidden)
        eo = W.make_expert_out_torch(lay_o["n_recv"], w.hidden, "cuda", 5)
        out = layer.combine(eo, torch.from_numpy(wt).cuda(), topk, lay)
        ref = oracle_combine_sample(lay_o, idx, wt, w.experts_per_rank, eo, np.arange(w.num_tokens))
        assert bf16_ulp_distance(bf16_tensor_to_bits(out), ref).max() <= COMBINE_ULP


def test_repeated_calls_on_one_handle():
    # the layout scan and the rings keep state across calls (tickets, epochs,
    # monotonic head/tail); five different routings in a row must all match
    w = _w(num_ranks=8, tokens_per_rank=300, hidden=256, num_experts=32, topk=4)
    from combine_ep_layout_04_gb300 import EpLayer
    with EpLayer(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk) as layer:
        x = torch.randn(w.num_tokens, w.hidden, device="cuda").to(torch.bfloat16)
        for seed in range(5):
            idx, wt = W.make_routing(w, seed=100 + seed)
            topk = torch.from_numpy(idx).cuda()
            lay = layer.layout(topk)
            lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
            compare_layout(lay.numpy(), lay_o)
            before = layer.ring_stats()
            recv = layer.dispatch(x, lay)
            check_dispatch_rows(recv, x, lay_o)
            logs = layer.cmd_log()
            compare_descriptors(logs, lay_o, layer.cfg.channels, layer.G, 2 * w.hidden)
            check_ring_invariants(layer, logs, lay_o, before)
