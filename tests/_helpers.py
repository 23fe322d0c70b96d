"""Helpers shared by the GPU tests: run the CUDA path on a workload and compare
it with the oracle.  Expected values come only from the oracle (or from the
inputs themselves); nothing expected is computed by the CUDA path."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

LAYOUT_KEYS = ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "token_slot",
               "recv_off", "send_off", "msg_count", "recv_count", "recv_base", "expert_off"]


def bits_to_bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_tensor_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """|a - b| in bf16 ulps on the monotone integer map (+0 == -0)."""
    def key(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u)
    return np.abs(key(a_bits) - key(b_bits))


def compare_layout(lay_gpu: dict, lay_o: dict) -> None:
    for k in LAYOUT_KEYS:
        a, b = np.asarray(lay_gpu[k]), np.asarray(lay_o[k])
        assert a.shape == b.shape, (k, a.shape, b.shape)
        if not np.array_equal(a, b):
            bad = np.argwhere(a != b)
            raise AssertionError(f"layout field {k} differs at {len(bad)} places, first {bad[:5].tolist()}: "
                                 f"gpu {a[tuple(bad[0])]} oracle {b[tuple(bad[0])]}")
    assert lay_gpu["n_recv"] is None or lay_gpu["n_recv"] == lay_o["n_recv"]


def compare_descriptors(logs: list, lay_o: dict, channels: int, G: int, B: int) -> None:
    """Per channel, the logged records sorted by (dst_rank, dst_offset) must be
    byte-identical to the oracle's canonical list sorted the same way."""
    ref, per = oracle.descriptors(lay_o, channels, G, B)
    start = np.concatenate([[0], np.cumsum(per)])
    assert len(logs) == channels
    for c in range(channels):
        got = np.asarray(logs[c])
        exp = ref[start[c]:start[c + 1]]
        assert len(got) == len(exp), (c, len(got), len(exp))
        if len(exp) == 0:
            continue
        go = np.lexsort((got["dst_offset"], got["dst_rank"]))
        eo = np.lexsort((exp["dst_offset"], exp["dst_rank"]))
        assert got[go].tobytes() == exp[eo].tobytes(), f"channel {c} records differ"


def check_dispatch_rows(recv: torch.Tensor, x: torch.Tensor, lay_o: dict, chunk_rows: int = 65536) -> None:
    """recv[recv_base[d] + token_slot[t][d]] == x[t] for every (t, d), with the
    indices taken from the oracle's layout; compared on the device, bitwise."""
    ts = lay_o["token_slot"]
    t_idx, d_idx = np.nonzero(ts >= 0)
    rows = lay_o["recv_base"][d_idx].astype(np.int64) + ts[t_idx, d_idx]
    assert len(rows) == lay_o["n_recv"]
    xi = x.view(torch.int16)
    ri = recv.view(torch.int16)
    for i in range(0, len(rows), chunk_rows):
        r = torch.from_numpy(rows[i:i + chunk_rows]).to(recv.device)
        t = torch.from_numpy(t_idx[i:i + chunk_rows].astype(np.int64)).to(recv.device)
        if not torch.equal(ri.index_select(0, r), xi.index_select(0, t)):
            bad = (ri.index_select(0, r) != xi.index_select(0, t)).any(dim=1).nonzero()
            j = int(bad[0])
            raise AssertionError(f"recv row {int(rows[i + j])} != x[{int(t_idx[i + j])}]")


def oracle_combine_sample(lay_o: dict, idx: np.ndarray, wt: np.ndarray, Er: int, expert_out: torch.Tensor,
                          tokens: np.ndarray) -> np.ndarray:
    """Oracle combine for a sample of tokens, fetching only the expert_out rows
    those tokens read (the receive rows are renumbered into a compact array;
    row(t, k) is unchanged in meaning)."""
    R = lay_o["recv_base"].shape[0]
    need = []
    for t in tokens:
        for d in range(R):
            if lay_o["token_slot"][t, d] >= 0:
                need.append(int(lay_o["recv_base"][d]) + int(lay_o["token_slot"][t, d]))
    uniq = np.array(sorted(set(need)), dtype=np.int64)
    eo = bf16_tensor_to_bits(expert_out.index_select(0, torch.from_numpy(uniq).to(expert_out.device))) \
        if len(uniq) else np.zeros((1, expert_out.shape[1]), np.uint16)
    pos = {int(r): i for i, r in enumerate(uniq)}
    sub_slot = np.full((len(tokens), R), -1, np.int32)
    for i, t in enumerate(tokens):
        for d in range(R):
            if lay_o["token_slot"][t, d] >= 0:
                sub_slot[i, d] = pos[int(lay_o["recv_base"][d]) + int(lay_o["token_slot"][t, d])]
    sub_lay = {"token_slot": sub_slot, "recv_base": np.zeros(R, np.int32)}
    return oracle.combine(sub_lay, idx[tokens], wt[tokens], Er, eo)


def check_ring_invariants(layer, logs, lay_o, before=None) -> None:
    stats = layer.ring_stats()
    per = oracle.channel_counts(lay_o, layer.cfg.channels)
    for c, s in enumerate(stats):
        assert s["head"] == s["tail"], (c, s)
        assert s["last_count"] == per[c] == len(logs[c]), (c, s, per[c])
        if before is not None:
            assert s["head"] - before[c]["head"] == per[c]
        assert s["max_batch"] <= layer.cfg.batch
        assert s["max_inflight"] <= layer.cfg.max_inflight
        if per[c] > 0:
            assert layer.check_completion(c, s["tail"] - 1)
        assert not layer.check_completion(c, s["tail"] + 5)


def workload_inputs(w: W.Workload, device="cuda", x_on_device: bool = False):
    idx, wt = W.make_routing(w)
    if x_on_device:
        x = W.make_x_torch(w, device)
    else:
        x = bits_to_bf16_tensor(W.make_x(w), device)
    return idx, wt, x
