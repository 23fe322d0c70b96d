"""Second oracle for tiny inputs: brute force by counting, in pure Python.

TEST INFRASTRUCTURE ONLY (see the package docstring).  It is written
differently from ``ep_oracle.c`` on purpose, so that a slip in one is caught by
the other:

- every receive slot is recounted from scratch (no running counters, no
  scans), every offset is a direct sum over the definition's index set;
- combine works in exact rationals: each fused multiply-add is the exact value
  a*b + c rounded once to the nearest binary32 (ties to even), and the final
  value is rounded to the nearest bf16 (ties to even) by comparing exact
  distances to the neighbouring representable values.

Definitions: the token layout, dispatch, TransferCmd and combine of one EP
layer, as the UCCL-EP article (sections 1, 2.3, 4.1, 4.2, 6) describes them,
with the readings listed in ``ep_oracle.c``.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction

import numpy as np


def _rank_of(e: int, Er: int) -> int:
    return e // Er


def layout(R: int, Tpr: int, E: int, topk_idx, G: int) -> dict:
    T = R * Tpr
    K = len(topk_idx[0]) if T else 0
    Er = E // R
    picks = [[int(v) for v in row] for row in topk_idx]

    def in_rank(t: int, d: int) -> bool:
        return any(e != -1 and _rank_of(e, Er) == d for e in picks[t])

    def src(t: int) -> int:
        return t // Tpr

    ntpe = [[sum(1 for t in range(T) if src(t) == s for k in range(K) if picks[t][k] == e)
             for e in range(E)] for s in range(R)]
    cnt = [[sum(1 for t in range(T) if src(t) == s and in_rank(t, d)) for d in range(R)]
           for s in range(R)]
    slot = [[(sum(1 for u in range(t) if in_rank(u, d)) if in_rank(t, d) else -1)
             for d in range(R)] for t in range(T)]
    recv_count = [sum(cnt[s][d] for s in range(R)) for d in range(R)]
    recv_base = [sum(recv_count[:d]) for d in range(R)]
    recv_off = [[sum(cnt[u][d] for u in range(s)) for d in range(R)] for s in range(R)]
    send_off = [[sum(cnt[u][v] for u in range(R) for v in range(R) if (u, v) < (s, d))
                 for d in range(R)] for s in range(R)]
    msg_count = [[-(-cnt[s][d] // G) for d in range(R)] for s in range(R)]
    expert_off = [sum(ntpe[s][f] for s in range(R) for f in range(e)) for e in range(E)]
    return {
        "num_tokens_per_expert": np.array(ntpe, np.int32).reshape(R, E),
        "num_tokens_per_rank": np.array(cnt, np.int32).reshape(R, R),
        "is_token_in_rank": np.array([[int(in_rank(t, d)) for d in range(R)] for t in range(T)],
                                     np.uint8).reshape(T, R),
        "token_slot": np.array(slot, np.int32).reshape(T, R),
        "recv_off": np.array(recv_off, np.int32).reshape(R, R),
        "send_off": np.array(send_off, np.int32).reshape(R, R),
        "msg_count": np.array(msg_count, np.int32).reshape(R, R),
        "recv_count": np.array(recv_count, np.int32),
        "recv_base": np.array(recv_base, np.int32),
        "expert_off": np.array(expert_off, np.int32),
        "n_recv": sum(recv_count),
    }


def dispatch(lay: dict, x) -> np.ndarray:
    """Find, for every receive row, the (token, rank) it belongs to."""
    T, R = lay["token_slot"].shape
    n = lay["n_recv"]
    x = np.asarray(x)
    recv = np.zeros((n,) + x.shape[1:], dtype=x.dtype)
    for row in range(n):
        owners = [(t, d) for t in range(T) for d in range(R)
                  if lay["token_slot"][t][d] >= 0 and lay["recv_base"][d] + lay["token_slot"][t][d] == row]
        assert len(owners) == 1, owners
        recv[row] = x[owners[0][0]]
    return recv


def descriptors(lay: dict, C: int, G: int, B: int) -> list[list[tuple]]:
    """Per channel, the set of (dst_rank, size, src_offset, dst_offset) records,
    built from message numbers directly."""
    R = lay["recv_base"].shape[0]
    cnt = lay["num_tokens_per_rank"]
    chans: list[list[tuple]] = [[] for _ in range(C)]
    for s in range(R):
        for d in range(R):
            nmsg = -(-int(cnt[s][d]) // G)
            for g in range(nmsg):
                rows = [j for j in range(int(cnt[s][d])) if j // G == g]
                chans[d % C].append((d, len(rows) * B,
                                     (int(lay["send_off"][s][d]) + rows[0]) * B,
                                     (int(lay["recv_off"][s][d]) + rows[0]) * B))
    return chans


def expert_layout(lay: dict, topk_idx, topk_weights, E: int) -> dict:
    """Expert-major receive metadata by search and sort: each receive row is
    matched to its (token, rank) by scanning all pairs; each expert's rows
    come from sorting all picks by (expert, token, k) with Python's sort."""
    T, R = lay["token_slot"].shape
    Er = E // R
    n = lay["n_recv"]
    picks = [[int(v) for v in row] for row in topk_idx]
    K = len(picks[0]) if T else 0

    def row_of(t, d):
        return int(lay["recv_base"][d]) + int(lay["token_slot"][t][d])

    src = np.zeros((n,), np.int32)
    ridx = np.zeros((n, K), np.int32)
    rw = np.zeros((n, K), np.float32)
    for row in range(n):
        owners = [(t, d) for t in range(T) for d in range(R)
                  if lay["token_slot"][t][d] >= 0 and row_of(t, d) == row]
        assert len(owners) == 1, owners
        t, d = owners[0]
        src[row] = t
        for k, e in enumerate(picks[t]):
            on_d = e != -1 and e // Er == d
            ridx[row, k] = e - d * Er if on_d else -1
            rw[row, k] = topk_weights[t][k] if on_d else 0.0
    triples = sorted((e, t, k) for t in range(T) for k, e in enumerate(picks[t]) if e != -1)
    rows = [row_of(t, e // Er) for (e, t, k) in triples]
    count = [sum(1 for (f, _, _) in triples if f == e) for e in range(E)]
    return {"recv_topk_idx": ridx, "recv_topk_weights": rw, "recv_src_token": src,
            "expert_rows": np.array(rows, np.int32), "expert_count": np.array(count, np.int32)}


# ------------------------------------------------------ exact rounding helpers


def _f32_neighbours(v: float):
    f = np.float32(v)
    return [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]


def _f32_bits(f) -> int:
    return struct.unpack("<I", struct.pack("<f", float(f)))[0]


def round_to_f32(q: Fraction) -> float:
    """Nearest binary32 to the exact rational q, ties to even mantissa."""
    best = None
    for c in _f32_neighbours(float(q)):
        if not math.isfinite(float(c)):
            continue
        dist = abs(Fraction(float(c)) - q)
        key = (dist, _f32_bits(c) & 1)
        if best is None or key < best[0]:
            best = (key, float(c))
    return best[1]


def fma_f32(a: float, b: float, c: float) -> float:
    return round_to_f32(Fraction(a) * Fraction(b) + Fraction(c))


def bf16_value(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (bits & 0xFFFF) << 16))[0]


def round_to_bf16_bits(v: float) -> int:
    """Nearest bf16 to the binary32 value v, ties to even; by exact distance
    to the two bf16 values that bracket v."""
    q = Fraction(v)
    hi = _f32_bits(v) >> 16
    cands = [hi, (hi + 1) & 0xFFFF, (hi - 1) & 0xFFFF]
    best = None
    for c in cands:
        cv = bf16_value(c)
        if not math.isfinite(cv):
            continue
        key = (abs(Fraction(cv) - q), c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    bits = best[1]
    if v == 0.0:  # keep the sign of zero
        bits = 0x8000 if math.copysign(1.0, v) < 0 else 0
    return bits


def combine(lay: dict, topk_idx, topk_weights, Er: int, expert_out_bits,
            tokens=None) -> np.ndarray:
    """out rows for `tokens` (default: all), in the order given."""
    T, R = lay["token_slot"].shape
    eo = np.asarray(expert_out_bits)
    H = eo.shape[1]
    tokens = list(range(T)) if tokens is None else list(tokens)
    out = np.zeros((len(tokens), H), np.uint16)
    for i, t in enumerate(tokens):
        for h in range(H):
            acc = 0.0
            for k in range(len(topk_idx[t])):
                e = int(topk_idx[t][k])
                if e == -1:
                    continue
                d = e // Er
                row = int(lay["recv_base"][d]) + int(lay["token_slot"][t][d])
                acc = fma_f32(float(np.float32(topk_weights[t][k])), bf16_value(int(eo[row][h])), acc)
            out[i][h] = round_to_bf16_bits(acc)
    return out
