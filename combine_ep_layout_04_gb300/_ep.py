"""ctypes binding of libep.so: the C ABI of include/ep.h, same names, argument
marshalling only.  Every step of the layer runs in the library's CUDA kernels;
there is no other code path.  If libep.so is missing, importing this module
raises."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libep.so")

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_CAPACITY = 2
EP_ERR_TIMEOUT = 3
EP_ERR_CUDA = 4
EP_ERR_NOT_READY = 5
EP_DEBUG_DISABLE_CONSUMER = 0x1
EP_DEBUG_DEVICE_COUNTERS = 0x2

_STATUS_NAMES = {0: "EP_OK", 1: "EP_ERR_INVALID_ARG", 2: "EP_ERR_CAPACITY", 3: "EP_ERR_TIMEOUT",
                 4: "EP_ERR_CUDA", 5: "EP_ERR_NOT_READY"}


class ep_config(ctypes.Structure):
    _fields_ = [("num_ranks", ctypes.c_int32), ("tokens_per_rank", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("channels", ctypes.c_int32), ("ring_depth", ctypes.c_int32),
                ("max_inflight", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("rows_per_msg", ctypes.c_int32), ("drain_batch", ctypes.c_int32),
                ("debug_flags", ctypes.c_int32), ("num_sms", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("timeout_ns", ctypes.c_uint64)]


class ep_transfer_cmd(ctypes.Structure):
    _fields_ = [("dst_rank", ctypes.c_uint32), ("size", ctypes.c_uint32), ("src_offset", ctypes.c_uint64),
                ("dst_offset", ctypes.c_uint64), ("type", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class ep_layout_out(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "token_slot", "recv_off",
        "send_off", "msg_count", "recv_count", "recv_base", "expert_off")]


class ep_expert_layout_out(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "recv_topk_idx", "recv_topk_weights", "recv_src_token", "expert_rows", "expert_count")]


class ep_cmd_log(ctypes.Structure):
    _fields_ = [("cmds", ctypes.c_void_p), ("count", ctypes.c_void_p),
                ("capacity_per_channel", ctypes.c_int64), ("channels", ctypes.c_int32)]


class ep_ring_stats(ctypes.Structure):
    _fields_ = [("head", ctypes.c_uint64), ("tail", ctypes.c_uint64), ("batches", ctypes.c_uint64),
                ("stall_polls", ctypes.c_uint64), ("max_batch", ctypes.c_uint32),
                ("max_inflight", ctypes.c_uint32), ("last_count", ctypes.c_int64)]


class ep_info(ctypes.Structure):
    _fields_ = [("rows_per_msg", ctypes.c_int32), ("sm_count", ctypes.c_int32),
                ("dispatch_grid", ctypes.c_int32), ("dispatch_stages", ctypes.c_int32),
                ("dispatch_stage_bytes", ctypes.c_int32), ("combine_grid", ctypes.c_int32),
                ("layout_tiles", ctypes.c_int32), ("dispatch_chunk_tokens", ctypes.c_int32),
                ("log_capacity_per_channel", ctypes.c_int64), ("scratch_bytes", ctypes.c_int64)]


assert ctypes.sizeof(ep_transfer_cmd) == 32
assert ctypes.sizeof(ep_config) == 64

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libep.so is not built ({LIB_PATH}); run "
                      "`python -m combine_ep_layout_04_gb300.build` (needs nvcc)")
lib = ctypes.CDLL(LIB_PATH)

_h = ctypes.c_void_p
_p = ctypes.c_void_p
_sigs = {
    "ep_config_init": ([ctypes.POINTER(ep_config)] + [ctypes.c_int32] * 5, ctypes.c_int),
    "ep_config_check": ([ctypes.POINTER(ep_config)], ctypes.c_int),
    "ep_create": ([ctypes.POINTER(ep_config), ctypes.POINTER(_h)], ctypes.c_int),
    "ep_destroy": ([_h], ctypes.c_int),
    "ep_status_str": ([ctypes.c_int], ctypes.c_char_p),
    "ep_last_device_status": ([_h, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
    "ep_reset": ([_h], ctypes.c_int),
    "ep_layout": ([_h, _p, ctypes.POINTER(ep_layout_out), ctypes.POINTER(ctypes.c_int64), _p], ctypes.c_int),
    "ep_dispatch": ([_h, _p, ctypes.POINTER(ep_layout_out), _p, ctypes.c_int64, _p], ctypes.c_int),
    "ep_combine": ([_h, _p, ctypes.c_int64, _p, _p, ctypes.POINTER(ep_layout_out), _p, _p], ctypes.c_int),
    "ep_dispatch_ranks": ([_h, _p, ctypes.POINTER(ep_layout_out), _p, ctypes.c_int64, ctypes.c_int32,
                           ctypes.c_int32, _p], ctypes.c_int),
    "ep_combine_tokens": ([_h, _p, ctypes.c_int64, _p, _p, ctypes.POINTER(ep_layout_out), _p, ctypes.c_int64,
                           ctypes.c_int64, _p], ctypes.c_int),
    "ep_expert_layout": ([_h, _p, _p, ctypes.POINTER(ep_layout_out), ctypes.POINTER(ep_expert_layout_out),
                          ctypes.c_int64, ctypes.c_int64, _p], ctypes.c_int),
    "ep_signal_ptr": ([_h, ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
    "ep_signal_get": ([_h, ctypes.POINTER(ctypes.c_uint64), ctypes.c_int32], ctypes.c_int),
    "ep_signal_reset": ([_h, _p], ctypes.c_int),
    "ep_wait_signal": ([_h, ctypes.c_int32, ctypes.c_uint64, ctypes.c_uint64, _p, _p], ctypes.c_int),
    "ep_cmd_log_get": ([_h, ctypes.POINTER(ep_cmd_log)], ctypes.c_int),
    "ep_ring_stats_get": ([_h, ctypes.POINTER(ep_ring_stats), ctypes.c_int32], ctypes.c_int),
    "ep_check_completion": ([_h, ctypes.c_int32, ctypes.c_uint64], ctypes.c_int),
    "ep_get_info": ([_h, ctypes.POINTER(ep_info)], ctypes.c_int),
    "ep_layout_static": ([ctypes.POINTER(ep_config), _p, ctypes.POINTER(ep_layout_out),
                          ctypes.POINTER(ctypes.c_int64), _p], ctypes.c_int),
    "ep_sm_split_create": ([ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(_h)], ctypes.c_int),
    "ep_sm_split_get": ([_h, ctypes.POINTER(_p), ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(_p),
                         ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
    "ep_sm_split_destroy": ([_h], ctypes.c_int),
    "ep_sm_ids": ([_p, ctypes.c_int32, _p], ctypes.c_int),
}
for _name, (_args, _res) in _sigs.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_sigs)


class EpError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_str(status)}" if what else status_str(status))


def status_str(status: int) -> str:
    return lib.ep_status_str(status).decode()


def check(status: int, what: str = "") -> None:
    if status != EP_OK:
        raise EpError(status, what)


# ----------------------------------------------------------------- the calls

def ep_config_init(num_ranks, tokens_per_rank, hidden, num_experts, topk) -> ep_config:
    cfg = ep_config()
    check(lib.ep_config_init(ctypes.byref(cfg), num_ranks, tokens_per_rank, hidden, num_experts, topk),
          "ep_config_init")
    return cfg


def ep_config_check(cfg: ep_config) -> int:
    return lib.ep_config_check(ctypes.byref(cfg))


def ep_create(cfg: ep_config) -> ctypes.c_void_p:
    h = _h()
    check(lib.ep_create(ctypes.byref(cfg), ctypes.byref(h)), "ep_create")
    return h


def ep_destroy(h) -> None:
    check(lib.ep_destroy(h), "ep_destroy")


def ep_last_device_status(h) -> int:
    code = ctypes.c_int32(0)
    check(lib.ep_last_device_status(h, ctypes.byref(code)), "ep_last_device_status")
    return int(code.value)


def ep_reset(h) -> None:
    check(lib.ep_reset(h), "ep_reset")


def ep_layout(h, topk_idx_ptr: int, out: ep_layout_out, stream: int, want_n: bool = True):
    n = ctypes.c_int64(-1)
    check(lib.ep_layout(h, topk_idx_ptr, ctypes.byref(out), ctypes.byref(n) if want_n else None, stream),
          "ep_layout")
    return int(n.value) if want_n else None


def ep_dispatch(h, x_ptr: int, layout: ep_layout_out, recv_ptr: int, capacity_rows: int, stream: int) -> None:
    check(lib.ep_dispatch(h, x_ptr, ctypes.byref(layout), recv_ptr, capacity_rows, stream), "ep_dispatch")


def ep_combine(h, expert_out_ptr: int, expert_out_rows: int, weights_ptr: int, topk_idx_ptr: int,
               layout: ep_layout_out, out_ptr: int, stream: int) -> None:
    check(lib.ep_combine(h, expert_out_ptr, expert_out_rows, weights_ptr, topk_idx_ptr, ctypes.byref(layout),
                         out_ptr, stream), "ep_combine")


def ep_dispatch_ranks(h, x_ptr: int, layout: ep_layout_out, recv_ptr: int, capacity_rows: int, src_begin: int,
                      src_end: int, stream: int) -> None:
    check(lib.ep_dispatch_ranks(h, x_ptr, ctypes.byref(layout), recv_ptr, capacity_rows, src_begin, src_end,
                                stream), "ep_dispatch_ranks")


def ep_combine_tokens(h, expert_out_ptr: int, expert_out_rows: int, weights_ptr: int, topk_idx_ptr: int,
                      layout: ep_layout_out, out_ptr: int, t_begin: int, t_end: int, stream: int) -> None:
    check(lib.ep_combine_tokens(h, expert_out_ptr, expert_out_rows, weights_ptr, topk_idx_ptr, ctypes.byref(layout),
                                out_ptr, t_begin, t_end, stream), "ep_combine_tokens")


def ep_expert_layout(h, topk_idx_ptr: int, weights_ptr: int, layout: ep_layout_out, out: ep_expert_layout_out,
                     recv_rows: int, rows_cap: int, stream: int) -> None:
    check(lib.ep_expert_layout(h, topk_idx_ptr, weights_ptr, ctypes.byref(layout), ctypes.byref(out), recv_rows,
                               rows_cap, stream), "ep_expert_layout")


def ep_signal_ptr(h) -> int:
    p = ctypes.c_void_p()
    check(lib.ep_signal_ptr(h, ctypes.byref(p)), "ep_signal_ptr")
    return int(p.value)


def ep_signal_get(h, n: int) -> list:
    arr = (ctypes.c_uint64 * n)()
    check(lib.ep_signal_get(h, arr, n), "ep_signal_get")
    return [int(v) for v in arr]


def ep_signal_reset(h, stream: int) -> None:
    check(lib.ep_signal_reset(h, stream), "ep_signal_reset")


def ep_wait_signal(h, dst_rank: int, expected: int, timeout_ns: int, status_ptr: int, stream: int) -> None:
    check(lib.ep_wait_signal(h, dst_rank, expected, timeout_ns, status_ptr, stream), "ep_wait_signal")


def ep_cmd_log_get(h) -> ep_cmd_log:
    log = ep_cmd_log()
    check(lib.ep_cmd_log_get(h, ctypes.byref(log)), "ep_cmd_log_get")
    return log


def ep_ring_stats_get(h, n: int) -> list:
    arr = (ep_ring_stats * n)()
    check(lib.ep_ring_stats_get(h, arr, n), "ep_ring_stats_get")
    return [{f: getattr(a, f) for f, _ in ep_ring_stats._fields_} for a in arr]


def ep_check_completion(h, channel: int, cmd_idx: int) -> int:
    return lib.ep_check_completion(h, channel, cmd_idx)


def ep_layout_static(cfg: ep_config, topk_idx_ptr: int, out: ep_layout_out, stream: int, want_n: bool = True):
    """The allocation-free layout (no handle; fixed scratch in the library)."""
    n = ctypes.c_int64(-1)
    check(lib.ep_layout_static(ctypes.byref(cfg), topk_idx_ptr, ctypes.byref(out),
                               ctypes.byref(n) if want_n else None, stream), "ep_layout_static")
    return int(n.value) if want_n else None


def ep_get_info(h) -> dict:
    info = ep_info()
    check(lib.ep_get_info(h, ctypes.byref(info)), "ep_get_info")
    return {f: getattr(info, f) for f, _ in ep_info._fields_}


def ep_sm_split_create(device: int, compute_sms: int):
    s = ctypes.c_void_p()
    check(lib.ep_sm_split_create(device, compute_sms, ctypes.byref(s)), "ep_sm_split_create")
    return s


def ep_sm_split_get(s) -> tuple:
    """(comm_stream, comm_sms, compute_stream, compute_sms)"""
    cs, ks = ctypes.c_void_p(), ctypes.c_void_p()
    cn, kn = ctypes.c_int32(), ctypes.c_int32()
    check(lib.ep_sm_split_get(s, ctypes.byref(cs), ctypes.byref(cn), ctypes.byref(ks), ctypes.byref(kn)),
          "ep_sm_split_get")
    return int(cs.value), int(cn.value), int(ks.value), int(kn.value)


def ep_sm_split_destroy(s) -> None:
    check(lib.ep_sm_split_destroy(s), "ep_sm_split_destroy")


def ep_sm_ids(stream: int, blocks: int, out_ptr: int) -> None:
    check(lib.ep_sm_ids(stream, blocks, out_ptr), "ep_sm_ids")
