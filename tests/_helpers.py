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
    """Oracle combine for a set of tokens, fetching only the expert_out rows
    those tokens read (the receive rows are renumbered into a compact array;
    row(t, k) is unchanged in meaning)."""
    tokens = np.asarray(tokens, dtype=np.int64)
    R = lay_o["recv_base"].shape[0]
    ts = lay_o["token_slot"][tokens]
    mask = ts >= 0
    rows = lay_o["recv_base"].astype(np.int64)[None, :] + ts
    uniq = np.unique(rows[mask])
    eo = bf16_tensor_to_bits(expert_out.index_select(0, torch.from_numpy(uniq).to(expert_out.device))) \
        if len(uniq) else np.zeros((1, expert_out.shape[1]), np.uint16)
    sub_slot = np.where(mask, np.searchsorted(uniq, rows), -1).astype(np.int32)
    sub_lay = {"token_slot": np.ascontiguousarray(sub_slot), "recv_base": np.zeros(R, np.int32)}
    return oracle.combine(sub_lay, idx[tokens], wt[tokens], Er, eo)


def check_combine_all(out: torch.Tensor, lay_o: dict, idx: np.ndarray, wt: np.ndarray, Er: int,
                      expert_out: torch.Tensor, max_ulp: int, chunk: int = 8192, workers: int = 0) -> int:
    """Every element of `out` against the oracle's combine, token chunk by
    token chunk so that host memory stays bounded; the oracle runs on a pool
    of host threads (it is single-threaded C called through ctypes, which
    releases the GIL).  Raises on the first element more than max_ulp bf16
    ulps away; returns the largest distance seen."""
    import concurrent.futures as cf
    import os
    T = idx.shape[0]
    workers = workers or max(1, min(8, (os.cpu_count() or 2) - 1))
    worst = 0

    def finish(fut):
        nonlocal worst
        t0, got, ref = fut.result()
        ulp = bf16_ulp_distance(got, ref)
        m = int(ulp.max(initial=0))
        if m > max_ulp:
            bad = np.argwhere(ulp > max_ulp)[:5]
            raise AssertionError(f"combine: max ulp {m}; first elements (token, column) "
                                 f"{[(int(t0 + b[0]), int(b[1])) for b in bad]}")
        worst = max(worst, m)

    def job(t0, tokens, got, rows):
        return t0, got, oracle_combine_sample(lay_o, idx, wt, Er, rows, tokens)

    # expert_out rows are gathered on the device in the main thread (torch
    # calls stay on one thread); only the oracle runs in the pool, with at
    # most 2 * workers chunks held on the host
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        pending = []
        for t0 in range(0, T, chunk):
            t1 = min(T, t0 + chunk)
            tokens = np.arange(t0, t1)
            ts = lay_o["token_slot"][t0:t1]
            mask = ts >= 0
            rows = lay_o["recv_base"].astype(np.int64)[None, :] + ts
            uniq = np.unique(rows[mask])
            got = bf16_tensor_to_bits(out[t0:t1])
            pending.append(ex.submit(job, t0, tokens, got, _HostRows(expert_out, uniq)))
            while len(pending) >= 2 * workers:
                finish(pending.pop(0))
        for f in pending:
            finish(f)
    return worst


class _HostRows:
    """The rows `uniq` of a device tensor, copied to the host once, served to
    oracle_combine_sample's index_select (which asks for exactly those rows,
    in the same sorted order)."""

    def __init__(self, t: torch.Tensor, uniq: np.ndarray):
        self.shape = t.shape
        self.device = "cpu"
        self._uniq = uniq
        self._rows = t.index_select(0, torch.from_numpy(uniq).to(t.device)).cpu() if len(uniq) else None

    def index_select(self, dim, index):
        assert dim == 0 and np.array_equal(index.cpu().numpy(), self._uniq)
        return self._rows


def check_identity_all(out_id: torch.Tensor, x: torch.Tensor, wt: np.ndarray, topk: int,
                       chunk: int = 8192) -> None:
    """dispatch -> identity expert -> combine == x * sum_k w on every token,
    within one bf16 rounding plus the fp32 chain's reassociation error
    (tokens with no picks combine to zero)."""
    T = x.shape[0]
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        xf = x[t0:t1].double()
        sw = torch.from_numpy(wt[t0:t1].astype(np.float64)).to(x.device).sum(dim=1, keepdim=True)
        ref = xf * sw
        err = (out_id[t0:t1].double() - ref).abs()
        bound = ref.abs() * 2.0**-8 + topk * 2.0**-23 * xf.abs() * sw + 1e-30
        if not bool((err <= bound).all()):
            bad = (err > bound).nonzero()[:5].tolist()
            raise AssertionError(f"identity-expert combine off at (token, column) "
                                 f"{[(t0 + b[0], b[1]) for b in bad]}")


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
