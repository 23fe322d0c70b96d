"""The allocation-free layout (ep_layout_static), for callers that cannot
call cudaMalloc -- a serving loop that must not let an allocation stall the
device, or a framework whose allocator owns all device memory.  It must give
exactly the oracle's layout, call after call, although every call reuses one
fixed scratch array inside the library; and it must take no device memory.

This file sorts last so that a run stopping at its first failure has already
run every other test."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _helpers import compare_layout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _alloc_outputs(R, T, E):
    from combine_ep_layout_04_gb300.layer import Layout
    i32 = dict(dtype=torch.int32, device="cuda")
    return Layout(torch.empty((R, E), **i32), torch.empty((R, R), **i32),
                  torch.empty((T, R), dtype=torch.uint8, device="cuda"), torch.empty((T, R), **i32),
                  torch.empty((R, R), **i32), torch.empty((R, R), **i32), torch.empty((R, R), **i32),
                  torch.empty((R,), **i32), torch.empty((R,), **i32), torch.empty((E,), **i32))


def _cfg(w):
    from combine_ep_layout_04_gb300 import _ep
    cfg = _ep.ep_config_init(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk)
    if w.rows_per_msg:
        cfg.rows_per_msg = w.rows_per_msg
    return cfg


def _static(cfg, topk, out, want_n=True):
    """ep_layout_static through the C ABI into caller-owned outputs; returns
    (status, N or None)."""
    import ctypes

    from combine_ep_layout_04_gb300 import _ep
    n = ctypes.c_int64(-1)
    st = _ep.lib.ep_layout_static(ctypes.byref(cfg), topk.data_ptr(), ctypes.byref(out.struct()),
                                  ctypes.byref(n) if want_n else None, torch.cuda.current_stream().cuda_stream)
    out.n_recv = int(n.value) if (want_n and st == 0) else None
    return st, out.n_recv


def _oracle(w, idx):
    G = w.rows_per_msg or oracle.default_rows_per_msg(w.hidden)
    return oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, G)


SHAPES = {
    "tiny": W.get("tiny"),
    "ll": W.get("ll"),
    "skew": W.get("skew"),
    "small": W.get("small"),
    # the array's limits: 262144 tokens, 64 ranks, 1024 experts
    "limit": W.Workload("limit", 64, 4096, 64, 1024, 8, seed=919),
    # a 256-token tile spans 8 ranks x 1024 experts > 4096 shared bins: the
    # histogram goes through warp-aggregated global atomics on the array
    "global_hist": W.Workload("global_hist", 64, 32, 64, 1024, 6, seed=929),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_static_layout_matches_oracle_twice(name):
    from combine_ep_layout_04_gb300 import _ep
    w = SHAPES[name]
    cfg = _cfg(w)
    # two calls in a row, each with its own routing: the shared scratch keeps
    # the first call's contents when the second starts
    for seed in (w.seed, w.seed + 1):
        idx, _ = W.make_routing(w, seed=seed)
        topk = torch.from_numpy(idx).cuda()
        out = _alloc_outputs(w.num_ranks, w.num_tokens, w.num_experts)
        st, n = _static(cfg, topk, out)
        assert st == _ep.EP_OK, _ep.status_str(st)
        compare_layout(out.numpy(), _oracle(w, idx))


def test_static_layout_matches_the_handle_layout():
    from combine_ep_layout_04_gb300 import EpLayer
    w = W.get("ll")
    idx, _ = W.make_routing(w, seed=7)
    topk = torch.from_numpy(idx).cuda()
    with EpLayer(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk) as layer:
        ref = layer.layout(topk).numpy()
    out = _alloc_outputs(w.num_ranks, w.num_tokens, w.num_experts)
    _static(_cfg(w), topk, out)
    compare_layout(out.numpy(), ref)


def test_static_layout_without_waiting_for_n():
    # n_recv_host = NULL: the call returns at once; after a stream sync the
    # outputs are the oracle's
    from combine_ep_layout_04_gb300 import _ep
    w = W.get("small")
    cfg = _cfg(w)
    for seed in (1, 2):
        idx, _ = W.make_routing(w, seed=seed)
        topk = torch.from_numpy(idx).cuda()
        out = _alloc_outputs(w.num_ranks, w.num_tokens, w.num_experts)
        st, n = _static(cfg, topk, out, want_n=False)
        assert st == _ep.EP_OK and n is None
        torch.cuda.current_stream().synchronize()
        lay_o = _oracle(w, idx)
        got = out.numpy()
        got["n_recv"] = None
        compare_layout(got, lay_o)


def test_static_layout_reports_a_bad_pick_then_recovers():
    from combine_ep_layout_04_gb300 import _ep
    w = W.get("tiny")
    cfg = _cfg(w)
    idx, _ = W.make_routing(w)
    bad = idx.copy()
    bad[5, 1] = w.num_experts            # outside [-1, E)
    out = _alloc_outputs(w.num_ranks, w.num_tokens, w.num_experts)
    st, _ = _static(cfg, torch.from_numpy(bad).cuda(), out)
    assert st == _ep.EP_ERR_INVALID_ARG
    # the next clean call starts from a cleared error word and is exact
    st, _ = _static(cfg, torch.from_numpy(idx).cuda(), out)
    assert st == _ep.EP_OK
    compare_layout(out.numpy(), _oracle(w, idx))


def test_static_layout_allocates_no_device_memory():
    w = W.get("skew")
    cfg = _cfg(w)
    idx, _ = W.make_routing(w)
    topk = torch.from_numpy(idx).cuda()
    out = _alloc_outputs(w.num_ranks, w.num_tokens, w.num_experts)
    _static(cfg, topk, out)            # first call: looks up the array's address
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for i in range(50):
        _static(cfg, topk, out, want_n=(i % 2 == 0))
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert torch.cuda.memory_reserved() == reserved0
    compare_layout(out.numpy(), _oracle(w, idx))


def test_static_layout_rejects_sizes_beyond_its_array():
    from combine_ep_layout_04_gb300 import _ep
    out = _ep.ep_layout_out()
    for f, _ in _ep.ep_layout_out._fields_:
        setattr(out, f, 16)                               # never dereferenced: rejected first
    for shape in [(32, 16384, 1024, 256, 8),              # 524288 tokens > 262144
                  (4, 16, 256, 2048, 2)]:                 # 2048 experts > 1024
        cfg = _ep.ep_config_init(*shape)
        st = _ep.lib.ep_layout_static(cfg, 16, out, None, None)
        assert st == _ep.EP_ERR_CAPACITY
