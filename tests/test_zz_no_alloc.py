"""The allocation-free layout (ep_layout_static), for callers that cannot
call cudaMalloc -- a serving loop that must not let an allocation stall the
device, or a framework whose allocator owns all device memory.  It must give
exactly what the handle-based ep_layout gives, call after call, although every
call reuses one fixed scratch array inside the library.

This file sorts last so that a run stopping at its first failure has already
run every other test."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _static_layout(layer, topk):
    """ep_layout_static through the C ABI, into fresh torch outputs."""
    from combine_ep_layout_04_gb300 import _ep
    out = layer.alloc_layout()
    n = _ep.ep_layout_static(layer.cfg, topk.data_ptr(), out.struct(), torch.cuda.current_stream().cuda_stream)
    out.n_recv = n
    return out


FIELDS = ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "token_slot", "recv_off",
          "send_off", "msg_count", "recv_count", "recv_base", "expert_off"]


def _same(a, b):
    da, db = a.numpy(), b.numpy()
    for f in FIELDS:
        assert np.array_equal(da[f], db[f]), f
    assert a.n_recv == b.n_recv


@pytest.mark.parametrize("name", ["tiny", "ll", "skew"])
def test_static_layout_matches_handle_layout_twice(name):
    from combine_ep_layout_04_gb300 import EpLayer
    w = W.get(name)
    with EpLayer(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk,
                 rows_per_msg=w.rows_per_msg) as layer:
        # two calls in a row, each with its own routing: the shared scratch
        # keeps the first call's contents when the second starts
        for seed in (w.seed, w.seed + 1):
            idx, _ = W.make_routing(w, seed=seed)
            topk = torch.from_numpy(idx).cuda()
            ref = layer.layout(topk)
            got = _static_layout(layer, topk)
            torch.cuda.synchronize()
            _same(got, ref)


def test_static_layout_rejects_sizes_beyond_its_array():
    from combine_ep_layout_04_gb300 import _ep
    cfg = _ep.ep_config_init(32, 16384, 1024, 256, 8)    # 524288 tokens > 262144
    out = _ep.ep_layout_out()
    for f, _ in _ep.ep_layout_out._fields_:
        setattr(out, f, 16)                               # never dereferenced: rejected first
    st = _ep.lib.ep_layout_static(cfg, 16, out, None, None)
    assert st == _ep.EP_ERR_CAPACITY
