"""Arrival signals of ep_dispatch (GIN-style SignalInc per message, bounded
waitSignal) against the oracle's per-destination message counts: exact after
one and two dispatches, zero after a reset, satisfied and run-out waits
reported through the status word, and the same under CUDA-graph replay."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _helpers import workload_inputs

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


@pytest.mark.parametrize("name", ["tiny", "small", "ll", "skew", "ht"])
def test_signals_count_messages(name):
    w = W.get(name)
    idx, wt, x = workload_inputs(w, x_on_device=True)
    layer = make_layer(w)
    try:
        topk = torch.from_numpy(idx).cuda()
        lay = layer.layout(topk)
        want = oracle.signal_counts(oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G))
        assert (layer.signals() == 0).all()
        recv = layer.dispatch(x, lay)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        assert np.array_equal(layer.signals(), want)
        layer.dispatch(x, lay, recv)                 # signals accumulate until reset
        torch.cuda.synchronize()
        assert np.array_equal(layer.signals(), 2 * want)
        layer.reset_signals()
        torch.cuda.synchronize()
        assert (layer.signals() == 0).all()
        assert np.array_equal(layer.signal_tensor().cpu().numpy(), np.zeros(w.num_ranks, np.uint64))
    finally:
        layer.close()


def test_wait_signal_is_met_or_runs_out():
    from combine_ep_layout_04_gb300 import _ep
    w = W.get("small").replace(tokens_per_rank=256)
    idx, wt, x = workload_inputs(w, x_on_device=True)
    layer = make_layer(w)
    try:
        topk = torch.from_numpy(idx).cuda()
        lay = layer.layout(topk)
        layer.dispatch(x, lay)
        want = oracle.signal_counts(oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G))
        status = torch.full((w.num_ranks,), -1, dtype=torch.int32, device="cuda")
        for d in range(w.num_ranks):                 # ordered after the dispatch on the stream: met at once
            layer.wait_signal(d, int(want[d]), 1_000_000_000, status[d:d + 1])
        torch.cuda.synchronize()
        assert (status == _ep.EP_OK).all()
        # a value nothing will reach: the wait runs out after ~2 ms and says so
        late = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        t0 = time.time()
        layer.wait_signal(3, int(want[3]) + 1, 2_000_000, late)
        torch.cuda.synchronize()
        assert time.time() - t0 < 2.0
        assert int(late.item()) == _ep.EP_ERR_NOT_READY
        assert layer.device_status() == 0             # the handle's error word is not touched
        with pytest.raises(_ep.EpError):
            layer.wait_signal(w.num_ranks, 0, 0, late)
        with pytest.raises(_ep.EpError):
            layer.wait_signal(0, 0, 11_000_000_000, late)
    finally:
        layer.close()


def test_signals_under_graph_replay():
    from combine_ep_layout_04_gb300 import _ep
    w = W.get("small").replace(tokens_per_rank=512)
    idx, wt, x = workload_inputs(w, x_on_device=True)
    layer = make_layer(w)
    try:
        topk = torch.from_numpy(idx).cuda()
        lay = layer.layout(topk)
        recv = layer.dispatch(x, lay)
        torch.cuda.synchronize()
        want = oracle.signal_counts(oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                layer.reset_signals()
                layer.layout(topk, out=lay, sync=False)
                layer.dispatch(x, lay, recv)
                layer.wait_signal(5, int(want[5]), 1_000_000_000, status)
        for _ in range(3):
            status.fill_(-1)
            g.replay()
            torch.cuda.synchronize()
            assert layer.device_status() == 0
            assert int(status.item()) == _ep.EP_OK
            assert np.array_equal(layer.signals(), want)
    finally:
        layer.close()
