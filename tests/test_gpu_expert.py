"""Parity of ep_expert_layout (through the C ABI) with the CPU oracle: every
output bit-exact (int32 arrays and fp32 weight bits) on the five workloads at
full size, on edge shapes, with empty picks, after repeated calls and under
CUDA-graph replay; bad input and short buffers are reported on the device
without writing out of bounds."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _helpers import compare_layout

pytestmark = pytest.mark.gpu

KEYS = ("recv_topk_idx", "recv_topk_weights", "recv_src_token", "expert_rows", "expert_count")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import combine_ep_layout_04_gb300  # noqa: F401  (fails loudly without libep.so)


def make_layer(w, **kw):
    from combine_ep_layout_04_gb300 import EpLayer
    return EpLayer(w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk, **kw)


def as_bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a


def compare_expert(xl, want: dict) -> None:
    M = want["expert_rows"].shape[0]
    got = {k: getattr(xl, k).cpu().numpy() for k in KEYS}
    got["expert_rows"] = got["expert_rows"][:M]
    for k in KEYS:
        assert got[k].shape == want[k].shape, k
        bad = np.nonzero(as_bits(got[k]).ravel() != as_bits(want[k]).ravel())[0]
        assert bad.size == 0, f"{k}: {bad.size} mismatches, first at {bad[:5]}"


def run_case(w, idx=None, wt=None, repeats=1):
    if idx is None:
        idx, wt = W.make_routing(w)
    layer = make_layer(w)
    try:
        topk = torch.from_numpy(idx).cuda()
        wts = torch.from_numpy(wt).cuda()
        lay = layer.layout(topk)
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
        compare_layout(lay.numpy(), lay_o)
        want = oracle.expert_layout(lay_o, idx, wt, w.num_experts)
        xl = None
        for _ in range(repeats):
            xl = layer.expert_layout(topk, wts, lay, out=xl)
            torch.cuda.synchronize()
            assert layer.device_status() == 0
            compare_expert(xl, want)
    finally:
        layer.close()


@pytest.mark.parametrize("name", ["tiny", "small", "ll", "skew", "ht"])
def test_workloads(name):
    run_case(W.get(name), repeats=2 if name in ("tiny", "ll") else 1)


EDGE = [
    dict(num_ranks=1, tokens_per_rank=300, num_experts=8, topk=2),             # one rank
    dict(num_ranks=5, tokens_per_rank=77, num_experts=20, topk=3),             # ragged tiles, odd K
    dict(num_ranks=12, tokens_per_rank=33, num_experts=24, topk=1),            # top-1
    dict(num_ranks=64, tokens_per_rank=9, num_experts=128, topk=8),            # many ranks, < 1 tile each
    dict(num_ranks=33, tokens_per_rank=40, num_experts=66, topk=4),            # R not a power of 2
    dict(num_ranks=4, tokens_per_rank=130, num_experts=64, topk=32),           # K = 32
    dict(num_ranks=8, tokens_per_rank=64, num_experts=4096, topk=8),           # E = 4096 (80 KB smem)
    dict(num_ranks=2, tokens_per_rank=1, num_experts=2, topk=1),               # two tokens
]


@pytest.mark.parametrize("kw", EDGE, ids=lambda d: "R{num_ranks}_T{tokens_per_rank}_E{num_experts}_K{topk}".format(**d))
def test_edge_shapes(kw):
    w = W.Workload("edge", kw["num_ranks"], kw["tokens_per_rank"], 256, kw["num_experts"], kw["topk"], seed=31)
    run_case(w)


def test_empty_picks_and_tokens_without_picks():
    w = W.Workload("holes", 6, 100, 256, 24, 4, seed=41)
    idx, wt = W.make_routing(w)
    rng = np.random.default_rng(5)
    idx = idx.copy()
    idx[rng.random(idx.shape) < 0.3] = -1
    idx[::7] = -1                                   # every 7th token picks nothing
    run_case(w, idx, wt, repeats=3)


def test_all_picks_to_one_expert():
    w = W.Workload("one", 8, 200, 256, 32, 1, seed=51)
    idx = np.full((w.num_tokens, 1), 17, np.int32)
    wt = np.ones((w.num_tokens, 1), np.float32)
    run_case(w, idx, wt)


def test_interleaved_with_layout_calls():
    # the expert scan's epoch is its own; layouts in between do not disturb it
    w = W.get("small").replace(tokens_per_rank=256)
    idx, wt = W.make_routing(w)
    idx2, wt2 = W.make_routing(w, seed=w.seed + 9)
    layer = make_layer(w)
    try:
        for a, b in [(idx, wt), (idx2, wt2), (idx, wt)]:
            topk = torch.from_numpy(a).cuda()
            lay = layer.layout(topk)
            xl = layer.expert_layout(topk, torch.from_numpy(b).cuda(), lay)
            torch.cuda.synchronize()
            assert layer.device_status() == 0
            lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, a, layer.G)
            compare_expert(xl, oracle.expert_layout(lay_o, a, b, w.num_experts))
    finally:
        layer.close()


def test_duplicate_pick_sets_invalid_arg():
    from combine_ep_layout_04_gb300 import _ep
    w = W.Workload("dup", 4, 64, 256, 16, 2, seed=61)
    idx, wt = W.make_routing(w)
    idx = idx.copy()
    idx[10, 1] = idx[10, 0]
    layer = make_layer(w)
    try:
        topk = torch.from_numpy(idx).cuda()
        lay = layer.layout(topk)           # the layout itself accepts it (counts the pick twice)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        layer.expert_layout(topk, torch.from_numpy(wt).cuda(), lay)
        torch.cuda.synchronize()
        assert layer.device_status() == _ep.EP_ERR_INVALID_ARG
        layer.reset()
        assert layer.device_status() == 0
    finally:
        layer.close()


def test_short_buffers_set_capacity_and_stay_in_bounds():
    from combine_ep_layout_04_gb300 import ExpertLayout, _ep
    w = W.get("tiny")
    idx, wt = W.make_routing(w)
    layer = make_layer(w)
    try:
        topk = torch.from_numpy(idx).cuda()
        lay = layer.layout(topk)
        N, K, M = lay.n_recv, w.topk, int((idx >= 0).sum())
        guard = 64
        for rows, cap in [(N - 3, M), (N, M - 5)]:
            i32 = dict(dtype=torch.int32, device="cuda")
            big = ExpertLayout(torch.full((N + guard, K), -7, **i32),
                               torch.full((N + guard, K), -7.0, dtype=torch.float32, device="cuda"),
                               torch.full((N + guard,), -7, **i32), torch.full((M + guard,), -7, **i32),
                               torch.full((w.num_experts,), -7, **i32))
            _ep.ep_expert_layout(layer.handle, topk.data_ptr(), torch.from_numpy(wt).cuda().data_ptr(),
                                 lay.struct(), big.struct(), rows, cap,
                                 torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            assert layer.device_status() == _ep.EP_ERR_CAPACITY
            assert (big.recv_src_token[rows:] == -7).all()
            assert (big.recv_topk_idx[rows:] == -7).all()
            assert (big.recv_topk_weights[rows:] == -7.0).all()
            assert (big.expert_rows[cap:] == -7).all()
            layer.reset()
    finally:
        layer.close()


def test_cuda_graph_replay():
    w = W.get("small").replace(tokens_per_rank=512)
    idx, wt = W.make_routing(w)
    layer = make_layer(w)
    try:
        topk = torch.from_numpy(idx).cuda()
        wts = torch.from_numpy(wt).cuda()
        lay = layer.layout(topk)
        xl = layer.expert_layout(topk, wts, lay)          # allocates outside the capture
        torch.cuda.synchronize()
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
        want = oracle.expert_layout(lay_o, idx, wt, w.num_experts)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                layer.layout(topk, out=lay, sync=False)
                layer.expert_layout(topk, wts, lay, out=xl)
        for _ in range(3):
            for k in KEYS:
                getattr(xl, k).fill_(-1)
            g.replay()
            torch.cuda.synchronize()
            assert layer.device_status() == 0
            compare_expert(xl, want)
    finally:
        layer.close()


def test_runs_beside_dispatch_on_another_stream():
    # the metadata needs only the layout, so it may overlap the data movement
    from _helpers import check_dispatch_rows
    w = W.get("ll")
    idx, wt = W.make_routing(w)
    layer = make_layer(w)
    try:
        topk = torch.from_numpy(idx).cuda()
        wts = torch.from_numpy(wt).cuda()
        x = W.make_x_torch(w, "cuda")
        lay = layer.layout(topk)
        recv = torch.empty((lay.n_recv, w.hidden), dtype=torch.bfloat16, device="cuda")
        side = torch.cuda.Stream()
        ev = torch.cuda.Event()
        ev.record()
        side.wait_event(ev)
        with torch.cuda.stream(side):
            xl = layer.expert_layout(topk, wts, lay)
        layer.dispatch(x, lay, recv)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        lay_o = oracle.layout(w.num_ranks, w.tokens_per_rank, w.num_experts, idx, layer.G)
        compare_expert(xl, oracle.expert_layout(lay_o, idx, wt, w.num_experts))
        check_dispatch_rows(recv, x, lay_o)
    finally:
        layer.close()
