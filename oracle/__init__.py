"""CPU oracle for the EP layer's layout, dispatch, TransferCmd descriptors and
combine.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg are the only code that may import this package.  The
product path (``combine_ep_layout_04_gb300``) never imports it, and this
package never imports the product.  The arithmetic lives in ``ep_oracle.c``
(plain single-threaded C, built with gcc and no fast-math or FMA contraction);
this module only marshals numpy arrays into it.  ``brute.py`` is a second,
differently written oracle for tiny inputs (pure Python, exact rationals).

Every function cites the article passage it follows (see ``ep_oracle.c``).
Parity pins: see ``tests/test_oracle_*.py``; every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

# Tuning table of the UCCL-EP article (section 5.2 "performance tuning
# parameters") and its batch limit (section 2.2: batches of up to 8 commands).
FIFO_DEPTH = 1024
MAX_INFLIGHT = 256
HT_CHANNELS = 8
DRAIN_BATCH_SIZE = 32
MAX_BATCH = 8
# UCCL-EP section 4.1: tokens under 7 KB are packed into one message; section
# 5.3 gives the packing batch size 8.
PACK_THRESHOLD_BYTES = 7 * 1024
PACK_ROWS = 8

CMD_DTYPE = np.dtype([("dst_rank", "<u4"), ("size", "<u4"), ("src_offset", "<u8"),
                      ("dst_offset", "<u8"), ("type", "<u4"), ("reserved", "<u4")])
assert CMD_DTYPE.itemsize == 32


def default_rows_per_msg(hidden: int) -> int:
    """Rows per message G: 8 when a bf16 row (2*hidden bytes) is under the
    7 KB packing threshold (UCCL-EP s4.1, batch size 8 from s5.3), else 1."""
    return PACK_ROWS if 2 * hidden < PACK_THRESHOLD_BYTES else 1


def build(force: bool = False) -> str:
    """Compile ep_oracle.c into liboracle.so next to it (gcc -O3, no FMA
    contraction and no fast-math, so every fused multiply-add is the explicit
    fmaf and every other operation is rounded as written; no -march=native,
    so the x86 and Arm builds give the same results)."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O3", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                        "-fno-fast-math", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_layout.argtypes = [i32, i32, i32, i32, i32, p] + [p] * 10 + [p]
        lib.oracle_layout.restype = i32
        lib.oracle_dispatch.argtypes = [i32, i64, i64, i64, p, p, p, p]
        lib.oracle_dispatch.restype = None
        lib.oracle_channel_counts.argtypes = [i32, i32, p, p]
        lib.oracle_channel_counts.restype = None
        lib.oracle_descriptors.argtypes = [i32, i32, i32, i64, p, p, p, p]
        lib.oracle_descriptors.restype = None
        lib.oracle_combine.argtypes = [i32, i32, i32, i64, i64, i64, p, p, p, p, p, i64, p]
        lib.oracle_combine.restype = i32
        lib.oracle_expert_layout.argtypes = [i32, i32, i32, i32, p, p, p, p, p, i64, p, p, p, p, p]
        lib.oracle_expert_layout.restype = i32
        lib.oracle_signal_counts.argtypes = [i32, p, p]
        lib.oracle_signal_counts.restype = None
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_fmaf.argtypes = [ctypes.c_float] * 3
        lib.oracle_fmaf.restype = ctypes.c_float
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags.c_contiguous
    return ctypes.c_void_p(a.ctypes.data)


class OracleError(RuntimeError):
    pass


def layout(num_ranks: int, tokens_per_rank: int, num_experts: int, topk_idx: np.ndarray,
           rows_per_msg: int) -> dict:
    """Layout of one EP layer (UCCL-EP s1); definitions in ep_oracle.c."""
    lib = _load()
    R, Tpr, E = num_ranks, tokens_per_rank, num_experts
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, K = topk_idx.shape
    assert T == R * Tpr
    out = {
        "num_tokens_per_expert": np.zeros((R, E), np.int32),
        "num_tokens_per_rank": np.zeros((R, R), np.int32),
        "is_token_in_rank": np.zeros((T, R), np.uint8),
        "token_slot": np.zeros((T, R), np.int32),
        "recv_off": np.zeros((R, R), np.int32),
        "send_off": np.zeros((R, R), np.int32),
        "msg_count": np.zeros((R, R), np.int32),
        "recv_count": np.zeros((R,), np.int32),
        "recv_base": np.zeros((R,), np.int32),
        "expert_off": np.zeros((E,), np.int32),
    }
    n = np.zeros((1,), np.int64)
    order = ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "token_slot",
             "recv_off", "send_off", "msg_count", "recv_count", "recv_base", "expert_off"]
    rc = lib.oracle_layout(R, Tpr, E, K, rows_per_msg, _ptr(topk_idx),
                           *[_ptr(out[k]) for k in order], _ptr(n))
    if rc != 0:
        raise OracleError(f"oracle_layout: code {rc}")
    out["n_recv"] = int(n[0])
    return out


def dispatch(lay: dict, x_bits: np.ndarray, t_begin: int = 0, t_end: int | None = None,
             recv: np.ndarray | None = None, x_first_token: int = 0) -> np.ndarray:
    """recv rows recv_base[d] + token_slot[t][d] <- x[t] (UCCL-EP s6 "Dispatch").
    x_bits: uint16 [rows, H] (bf16 bits) holding tokens x_first_token onward.
    Returns recv uint16 [n_recv, H]."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits)
    rows, H = x_bits.shape
    R = lay["recv_base"].shape[0]
    if recv is None:
        recv = np.zeros((lay["n_recv"], H), dtype=x_bits.dtype)
    t_end = x_first_token + rows if t_end is None else t_end
    assert x_first_token <= t_begin <= t_end <= x_first_token + rows
    row_bytes = H * x_bits.itemsize
    # the C routine addresses x by absolute token index
    x_base = ctypes.c_void_p(x_bits.ctypes.data - x_first_token * row_bytes)
    lib.oracle_dispatch(R, t_begin, t_end, row_bytes, _ptr(lay["token_slot"]),
                        _ptr(lay["recv_base"]), x_base, _ptr(recv))
    return recv


def channel_counts(lay: dict, channels: int) -> np.ndarray:
    lib = _load()
    R = lay["recv_base"].shape[0]
    per = np.zeros((channels,), np.int64)
    lib.oracle_channel_counts(R, channels, _ptr(lay["msg_count"]), _ptr(per))
    return per


def descriptors(lay: dict, channels: int, rows_per_msg: int, row_bytes: int):
    """Canonical TransferCmd list (UCCL-EP s2.3 fields, s4.1 packing, s4.2
    channels).  Returns (records[CMD_DTYPE], per-channel counts)."""
    lib = _load()
    R = lay["recv_base"].shape[0]
    per = channel_counts(lay, channels)
    out = np.zeros((int(per.sum()),), dtype=CMD_DTYPE)
    lib.oracle_descriptors(R, channels, rows_per_msg, row_bytes, _ptr(lay["num_tokens_per_rank"]),
                           _ptr(lay["recv_off"]), _ptr(lay["send_off"]), _ptr(out))
    return out, per


def combine(lay: dict, topk_idx: np.ndarray, topk_weights: np.ndarray, experts_per_rank: int,
            expert_out_bits: np.ndarray, t_begin: int = 0, t_end: int | None = None) -> np.ndarray:
    """Top-k weighted fp32 fmaf chain back to token order, bf16 RNE
    (UCCL-EP s6 "Combine").  Returns out bits uint16 [t_end - t_begin, H]."""
    lib = _load()
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    expert_out_bits = np.ascontiguousarray(expert_out_bits, dtype=np.uint16)
    T, K = topk_idx.shape
    n_rows, H = expert_out_bits.shape
    R = lay["recv_base"].shape[0]
    t_end = T if t_end is None else t_end
    out = np.zeros((t_end - t_begin, H), dtype=np.uint16)
    rc = lib.oracle_combine(R, experts_per_rank, K, H, t_begin, t_end, _ptr(topk_idx),
                            _ptr(topk_weights), _ptr(lay["token_slot"]), _ptr(lay["recv_base"]),
                            _ptr(expert_out_bits), n_rows, _ptr(out))
    if rc != 0:
        raise OracleError(f"oracle_combine: code {rc}")
    return out


def expert_layout(lay: dict, topk_idx: np.ndarray, topk_weights: np.ndarray, num_experts: int) -> dict:
    """Expert-major receive metadata (UCCL-EP s1 token-level routing to the
    experts of each pick): per receive row its source token and its local
    picks and weights; per expert the receive rows of its picks in pick order.
    Definitions in ep_oracle.c.  Returns recv_topk_idx int32 [N, K],
    recv_topk_weights float32 [N, K], recv_src_token int32 [N], expert_rows
    int32 [picks], expert_count int32 [E]."""
    lib = _load()
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    T, K = topk_idx.shape
    R = lay["recv_base"].shape[0]
    E = num_experts
    N = lay["n_recv"]
    out = {
        "recv_topk_idx": np.zeros((N, K), np.int32),
        "recv_topk_weights": np.zeros((N, K), np.float32),
        "recv_src_token": np.zeros((N,), np.int32),
        "expert_rows": np.zeros((int((topk_idx >= 0).sum()),), np.int32),
        "expert_count": np.zeros((E,), np.int32),
    }
    rc = lib.oracle_expert_layout(R, T // R, E, K, _ptr(topk_idx), _ptr(topk_weights), _ptr(lay["token_slot"]),
                                  _ptr(lay["recv_base"]), _ptr(lay["expert_off"]), N,
                                  *[_ptr(out[k]) for k in ("recv_topk_idx", "recv_topk_weights",
                                                           "recv_src_token", "expert_rows", "expert_count")])
    if rc != 0:
        raise OracleError(f"oracle_expert_layout: code {rc}")
    return out


def signal_counts(lay: dict) -> np.ndarray:
    """Per destination rank, the signal value one dispatch leaves: one
    increment per message landing there (NCCL GIN s2.2.2 signals, s2.1.2
    put with SignalInc).  Returns uint64 [R]."""
    msg = np.ascontiguousarray(lay["msg_count"], dtype=np.int32)
    R = msg.shape[0]
    out = np.zeros((R,), np.uint64)
    _load().oracle_signal_counts(R, _ptr(msg), _ptr(out))
    return out


def f32_to_bf16(f: float) -> int:
    return int(_load().oracle_f32_to_bf16(f))


def bf16_to_f32(b: int) -> float:
    return float(_load().oracle_bf16_to_f32(b))


def fmaf(a: float, b: float, c: float) -> float:
    return float(_load().oracle_fmaf(a, b, c))
