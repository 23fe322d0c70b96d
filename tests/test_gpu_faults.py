"""Device-side error paths (none traps or hangs the GPU): a pick outside
[-1, E), a receive buffer smaller than N, and ring producers whose bounded
flow-control wait runs out because the consumers were switched off by a flag.
Each sets the sticky device error word; ep_reset clears it and the handle
works again.  Also: the three calls captured once in a CUDA graph and replayed
(the layout scan and the rings keep no host-side per-call state)."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _helpers import (bf16_tensor_to_bits, bf16_ulp_distance, check_dispatch_rows, check_ring_invariants,
                      compare_descriptors, compare_layout, oracle_combine_sample)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _w():
    return W.Workload("fault", 8, 64, 256, 32, 4, seed=21)


def _layer(w, **kw):
    from combine_ep_layout_04_gb300 import EpLayer
    return EpLayer(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk, **kw)


def _good_round(layer, w):
    idx, wt = W.make_routing(w)
    topk = torch.from_numpy(idx).cuda()
    lay = layer.layout(topk)
    lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
    compare_layout(lay.numpy(), lay_o)
    x = torch.randn(w.num_tokens, w.hidden, device="cuda").to(torch.bfloat16)
    recv = layer.dispatch(x, lay)
    check_dispatch_rows(recv, x, lay_o)
    compare_descriptors(layer.cmd_log(), lay_o, layer.cfg.channels, layer.G, 2 * w.hidden)
    assert layer.device_status() == 0


def test_pick_out_of_range_sets_invalid_arg():
    from combine_ep_layout_04_gb300 import _ep
    w = _w()
    with _layer(w) as layer:
        idx, _ = W.make_routing(w)
        idx[17, 2] = w.num_experts          # out of range
        layer.layout(torch.from_numpy(idx).cuda())
        assert layer.device_status() == _ep.EP_ERR_INVALID_ARG
        layer.reset()
        assert layer.device_status() == 0
        _good_round(layer, w)


def test_receive_buffer_too_small_sets_capacity():
    from combine_ep_layout_04_gb300 import _ep
    w = _w()
    with _layer(w) as layer:
        idx, _ = W.make_routing(w)
        lay = layer.layout(torch.from_numpy(idx).cuda())
        x = torch.randn(w.num_tokens, w.hidden, device="cuda").to(torch.bfloat16)
        recv = torch.full((lay.n_recv - 1, w.hidden), 7.0, dtype=torch.bfloat16, device="cuda")
        layer.dispatch(x, lay, recv)
        assert layer.device_status() == _ep.EP_ERR_CAPACITY
        assert bool((recv == 7.0).all())     # nothing was written
        layer.reset()
        _good_round(layer, w)


def test_consumers_off_producers_time_out():
    from combine_ep_layout_04_gb300 import _ep
    w = _w()
    timeout_ns = 50_000_000
    with _layer(w, ring_depth=16, max_inflight=8, timeout_ns=timeout_ns,
                debug_flags=_ep.EP_DEBUG_DISABLE_CONSUMER) as layer:
        idx, _ = W.make_routing(w)
        lay = layer.layout(torch.from_numpy(idx).cuda())
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
        assert oracle.channel_counts(lay_o, layer.cfg.channels).max() > 4 * 8   # the rings must fill
        x = torch.randn(w.num_tokens, w.hidden, device="cuda").to(torch.bfloat16)
        t0 = time.time()
        layer.dispatch(x, lay)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
        assert layer.device_status() == _ep.EP_ERR_TIMEOUT
        assert elapsed < 5.0
        # the context is still usable
        y = torch.ones(16, device="cuda") * 2
        assert float(y.sum()) == 32.0
        stats = layer.ring_stats()
        assert all(s["max_inflight"] <= 8 for s in stats)
    with _layer(w) as layer:
        _good_round(layer, w)


def test_host_argument_checks():
    from combine_ep_layout_04_gb300 import _ep
    w = _w()
    with _layer(w) as layer:
        idx, _ = W.make_routing(w)
        lay = layer.layout(torch.from_numpy(idx).cuda())
        x = torch.randn(w.num_tokens, w.hidden, device="cuda").to(torch.bfloat16)
        recv = torch.empty((lay.n_recv + 1, w.hidden), dtype=torch.bfloat16, device="cuda")
        st = _ep.lib.ep_dispatch(layer.handle, x.data_ptr() + 2, lay.struct(), recv.data_ptr(), lay.n_recv,
                                 torch.cuda.current_stream().cuda_stream)
        assert st == _ep.EP_ERR_INVALID_ARG                  # misaligned x
        st = _ep.lib.ep_dispatch(layer.handle, x.data_ptr(), None, recv.data_ptr(), lay.n_recv, None)
        assert st == _ep.EP_ERR_INVALID_ARG                  # no layout
        assert layer.device_status() == 0


def test_pointer_kinds_checked_on_the_host():
    """The C ABI refuses pageable host memory before any launch and accepts
    page-locked host memory, which the kernels read through its device
    mapping; the binding refuses tensors on the wrong device or of the wrong
    shape before calling the library."""
    from combine_ep_layout_04_gb300 import _ep
    w = _w()
    stream = torch.cuda.current_stream().cuda_stream
    with _layer(w) as layer:
        idx, wt = W.make_routing(w)
        ref = layer.layout(torch.from_numpy(idx).cuda()).numpy()
        lay = layer.alloc_layout()
        pageable = np.ascontiguousarray(idx)
        assert _ep.lib.ep_layout(layer.handle, pageable.ctypes.data, lay.struct(), None, stream) == \
            _ep.EP_ERR_INVALID_ARG
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        pinned = torch.from_numpy(idx).pin_memory()
        n = _ep.ep_layout(layer.handle, pinned.data_ptr(), lay.struct(), stream, want_n=True)
        assert n == ref["n_recv"]
        got = lay.numpy()
        for k in ref:
            if k != "n_recv":
                assert np.array_equal(got[k], ref[k]), k
        with pytest.raises(ValueError):
            layer.layout(torch.from_numpy(idx))                      # host tensor
        with pytest.raises(TypeError):
            layer.layout(torch.from_numpy(idx).cuda().long())         # int64 picks
        x = torch.randn(w.num_tokens, w.hidden, device="cuda").to(torch.bfloat16)
        lay2 = layer.layout(torch.from_numpy(idx).cuda())
        recv = layer.dispatch(x, lay2)
        wts = torch.from_numpy(wt).cuda()
        topk = torch.from_numpy(idx).cuda()
        with pytest.raises(ValueError):
            layer.combine(recv, wts, topk, lay2, out=torch.empty((w.num_tokens - 1, w.hidden), dtype=torch.bfloat16,
                                                                    device="cuda"))
        bad = layer.alloc_layout()
        bad.token_slot = bad.token_slot[:-1]
        with pytest.raises(ValueError):
            layer.layout(topk, out=bad)
        assert layer.device_status() == 0


def test_cuda_graph_replay():
    w = W.get("small")
    idx, wt = W.make_routing(w)
    with _layer(w, channels=w.channels, ring_depth=w.ring_depth, max_inflight=w.max_inflight,
                rows_per_msg=w.rows_per_msg) as layer:
        topk = torch.from_numpy(idx).cuda()
        wts = torch.from_numpy(wt).cuda()
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
        N = lay_o["n_recv"]
        x = torch.randn(w.num_tokens, w.hidden, device="cuda").to(torch.bfloat16)
        lay = layer.alloc_layout()
        recv = torch.empty((N, w.hidden), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((w.num_tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            layer.layout(topk, out=lay, sync=False)
            layer.dispatch(x, lay, recv)
            layer.combine(recv, wts, topk, lay, out)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer.layout(topk, out=lay, sync=False)
            layer.dispatch(x, lay, recv)
            layer.combine(recv, wts, topk, lay, out)
        tokens = np.arange(0, w.num_tokens, 97)
        for rep in range(3):
            for t in (lay.token_slot, lay.recv_base):
                t.fill_(-7)
            recv.fill_(0)
            before = layer.ring_stats()
            g.replay()
            torch.cuda.synchronize()
            assert layer.device_status() == 0
            compare_layout(lay.numpy(), lay_o)
            check_dispatch_rows(recv, x, lay_o)
            logs = layer.cmd_log()
            compare_descriptors(logs, lay_o, layer.cfg.channels, layer.G, 2 * w.hidden)
            check_ring_invariants(layer, logs, lay_o, before)
            ref = oracle_combine_sample(lay_o, idx, wt, w.experts_per_rank, recv, tokens)
            got = bf16_tensor_to_bits(out[torch.from_numpy(tokens).cuda()])
            assert bf16_ulp_distance(got, ref).max() <= 1
