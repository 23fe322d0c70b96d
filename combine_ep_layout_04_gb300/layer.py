"""Torch-facing wrapper of the C ABI: allocates the caller-owned outputs with
torch on the handle's device and passes raw device pointers and the current
CUDA stream to libep.  Marshalling only; all arithmetic is in the library's
kernels (layout, dispatch with its TransferCmd rings, combine)."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import _ep

CMD_DTYPE = np.dtype([("dst_rank", "<u4"), ("size", "<u4"), ("src_offset", "<u8"),
                      ("dst_offset", "<u8"), ("type", "<u4"), ("reserved", "<u4")])

_LAYOUT_FIELDS = ("num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "token_slot",
                  "recv_off", "send_off", "msg_count", "recv_count", "recv_base", "expert_off")


@dataclasses.dataclass
class Layout:
    """Device outputs of ep_layout (shapes in include/ep.h)."""
    num_tokens_per_expert: torch.Tensor
    num_tokens_per_rank: torch.Tensor
    is_token_in_rank: torch.Tensor
    token_slot: torch.Tensor
    recv_off: torch.Tensor
    send_off: torch.Tensor
    msg_count: torch.Tensor
    recv_count: torch.Tensor
    recv_base: torch.Tensor
    expert_off: torch.Tensor
    n_recv: int | None = None

    def struct(self) -> _ep.ep_layout_out:
        s = _ep.ep_layout_out()
        for f in _LAYOUT_FIELDS:
            setattr(s, f, getattr(self, f).data_ptr())
        return s

    def numpy(self) -> dict:
        d = {f: getattr(self, f).cpu().numpy() for f in _LAYOUT_FIELDS}
        d["n_recv"] = self.n_recv
        return d


_EXPERT_FIELDS = ("recv_topk_idx", "recv_topk_weights", "recv_src_token", "expert_rows", "expert_count")


@dataclasses.dataclass
class ExpertLayout:
    """Device outputs of ep_expert_layout (shapes in include/ep.h).
    expert_rows holds T*K entries; the first sum(expert_count) are written."""
    recv_topk_idx: torch.Tensor
    recv_topk_weights: torch.Tensor
    recv_src_token: torch.Tensor
    expert_rows: torch.Tensor
    expert_count: torch.Tensor

    def struct(self) -> _ep.ep_expert_layout_out:
        s = _ep.ep_expert_layout_out()
        for f in _EXPERT_FIELDS:
            setattr(s, f, getattr(self, f).data_ptr())
        return s


class _DevArray:
    """Exposes a library-owned device buffer to torch (zero copy)."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3}


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


class EpLayer:
    """One EP layer: R simulated ranks in this GPU's memory."""

    def __init__(self, num_ranks: int, tokens_per_rank: int, hidden: int, num_experts: int, topk: int, *,
                 channels=None, ring_depth=None, max_inflight=None, batch=None, rows_per_msg=None,
                 drain_batch=None, timeout_ns=None, num_sms=None, debug_flags: int = 0, device=None):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        cfg = _ep.ep_config_init(num_ranks, tokens_per_rank, hidden, num_experts, topk)
        for name, val in (("channels", channels), ("ring_depth", ring_depth), ("max_inflight", max_inflight),
                          ("batch", batch), ("rows_per_msg", rows_per_msg), ("drain_batch", drain_batch),
                          ("timeout_ns", timeout_ns), ("num_sms", num_sms)):
            if val is not None:
                setattr(cfg, name, val)
        cfg.debug_flags = debug_flags
        self.cfg = cfg
        with torch.cuda.device(self.device):
            self.handle = _ep.ep_create(cfg)
        self.info = _ep.ep_get_info(self.handle)
        self.R, self.Tpr, self.H, self.E, self.K = num_ranks, tokens_per_rank, hidden, num_experts, topk
        self.T = num_ranks * tokens_per_rank
        self.G = self.info["rows_per_msg"]

    # -- lifetime
    def close(self) -> None:
        if getattr(self, "handle", None) is not None:
            with torch.cuda.device(self.device):
                _ep.ep_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- the three calls
    def alloc_layout(self) -> Layout:
        R, T, E = self.R, self.T, self.E
        i32 = dict(dtype=torch.int32, device=self.device)
        return Layout(torch.empty((R, E), **i32), torch.empty((R, R), **i32),
                      torch.empty((T, R), dtype=torch.uint8, device=self.device), torch.empty((T, R), **i32),
                      torch.empty((R, R), **i32), torch.empty((R, R), **i32), torch.empty((R, R), **i32),
                      torch.empty((R,), **i32), torch.empty((R,), **i32), torch.empty((E,), **i32))

    def layout(self, topk_idx: torch.Tensor, out: Layout | None = None, sync: bool = True) -> Layout:
        """ep_layout.  topk_idx: int32 [T, K] on the device.  With sync=True the
        call waits for N (n_recv) so that the caller can size recv."""
        assert topk_idx.dtype == torch.int32 and topk_idx.is_contiguous() and topk_idx.shape == (self.T, self.K)
        out = self.alloc_layout() if out is None else out
        out.n_recv = _ep.ep_layout(self.handle, topk_idx.data_ptr(), out.struct(), _stream(self.device), want_n=sync)
        return out

    def dispatch(self, x: torch.Tensor, lay: Layout, recv: torch.Tensor | None = None,
                 src_ranks: tuple[int, int] | None = None) -> torch.Tensor:
        """ep_dispatch (ep_dispatch_ranks for src_ranks=(begin, end)).
        x: bf16 [T, H].  Returns recv bf16 [capacity, H]."""
        assert x.dtype == torch.bfloat16 and x.is_contiguous() and x.shape == (self.T, self.H)
        if recv is None:
            if lay.n_recv is None:
                raise ValueError("dispatch needs recv or a layout computed with sync=True")
            recv = torch.empty((lay.n_recv, self.H), dtype=torch.bfloat16, device=self.device)
        assert recv.dtype == torch.bfloat16 and recv.is_contiguous() and recv.shape[1] == self.H
        if src_ranks is None:
            _ep.ep_dispatch(self.handle, x.data_ptr(), lay.struct(), recv.data_ptr(), recv.shape[0],
                            _stream(self.device))
        else:
            _ep.ep_dispatch_ranks(self.handle, x.data_ptr(), lay.struct(), recv.data_ptr(), recv.shape[0],
                                  src_ranks[0], src_ranks[1], _stream(self.device))
        return recv

    def combine(self, expert_out: torch.Tensor, topk_weights: torch.Tensor, topk_idx: torch.Tensor, lay: Layout,
                out: torch.Tensor | None = None, tokens: tuple[int, int] | None = None) -> torch.Tensor:
        """ep_combine (ep_combine_tokens for tokens=(begin, end)).
        expert_out: bf16 [rows, H]; topk_weights fp32 [T, K]."""
        assert expert_out.dtype == torch.bfloat16 and expert_out.is_contiguous() and expert_out.shape[1] == self.H
        assert topk_weights.dtype == torch.float32 and topk_weights.is_contiguous()
        assert topk_idx.dtype == torch.int32 and topk_idx.is_contiguous()
        if out is None:
            out = torch.empty((self.T, self.H), dtype=torch.bfloat16, device=self.device)
        if tokens is None:
            _ep.ep_combine(self.handle, expert_out.data_ptr(), expert_out.shape[0], topk_weights.data_ptr(),
                           topk_idx.data_ptr(), lay.struct(), out.data_ptr(), _stream(self.device))
        else:
            _ep.ep_combine_tokens(self.handle, expert_out.data_ptr(), expert_out.shape[0], topk_weights.data_ptr(),
                                  topk_idx.data_ptr(), lay.struct(), out.data_ptr(), tokens[0], tokens[1],
                                  _stream(self.device))
        return out

    def expert_layout(self, topk_idx: torch.Tensor, topk_weights: torch.Tensor, lay: Layout,
                      out: ExpertLayout | None = None) -> ExpertLayout:
        """ep_expert_layout: per receive row its source token and local picks
        and weights; per expert its receive rows.  Needs N (a layout computed
        with sync=True) unless `out` is given."""
        assert topk_idx.dtype == torch.int32 and topk_idx.is_contiguous() and topk_idx.shape == (self.T, self.K)
        assert topk_weights.dtype == torch.float32 and topk_weights.is_contiguous()
        assert topk_weights.shape == (self.T, self.K)
        if out is None:
            if lay.n_recv is None:
                raise ValueError("expert_layout needs `out` or a layout computed with sync=True")
            N, K = lay.n_recv, self.K
            i32 = dict(dtype=torch.int32, device=self.device)
            out = ExpertLayout(torch.empty((N, K), **i32), torch.empty((N, K), dtype=torch.float32, device=self.device),
                               torch.empty((N,), **i32), torch.empty((self.T * K,), **i32),
                               torch.empty((self.E,), **i32))
        _ep.ep_expert_layout(self.handle, topk_idx.data_ptr(), topk_weights.data_ptr(), lay.struct(), out.struct(),
                             out.recv_src_token.shape[0], out.expert_rows.shape[0], _stream(self.device))
        return out

    # -- arrival signals
    def signals(self) -> np.ndarray:
        """signal[R] on the host (synchronises the device)."""
        return np.array(_ep.ep_signal_get(self.handle, self.R), dtype=np.uint64)

    def signal_tensor(self) -> torch.Tensor:
        """The library-owned signal[R] as a uint64 device tensor (zero copy)."""
        return torch.as_tensor(_DevArray(_ep.ep_signal_ptr(self.handle), (self.R,), "<u8"), device=self.device)

    def reset_signals(self) -> None:
        _ep.ep_signal_reset(self.handle, _stream(self.device))

    def wait_signal(self, dst_rank: int, expected: int, timeout_ns: int, status: torch.Tensor) -> torch.Tensor:
        """ep_wait_signal: enqueue a bounded wait; `status` (device int32 [1])
        receives EP_OK or EP_ERR_NOT_READY."""
        assert status.dtype == torch.int32 and status.device == self.device
        _ep.ep_wait_signal(self.handle, dst_rank, expected, timeout_ns, status.data_ptr(), _stream(self.device))
        return status

    # -- rings, status
    def cmd_log(self):
        """Per-channel TransferCmd logs of the last dispatch, as numpy records
        (copies to the host after synchronising the device)."""
        log = _ep.ep_cmd_log_get(self.handle)
        C, cap = log.channels, log.capacity_per_channel
        torch.cuda.synchronize(self.device)
        counts = torch.as_tensor(_DevArray(log.count, (C,), "<i8"), device=self.device).cpu().numpy()
        raw = torch.as_tensor(_DevArray(log.cmds, (C, cap * 32), "|u1"), device=self.device)
        out = []
        for c in range(C):
            n = int(counts[c])
            out.append(raw[c, :n * 32].cpu().numpy().view(CMD_DTYPE))
        return out

    def ring_stats(self) -> list:
        return _ep.ep_ring_stats_get(self.handle, self.cfg.channels)

    def device_status(self) -> int:
        return _ep.ep_last_device_status(self.handle)

    def check_completion(self, channel: int, cmd_idx: int) -> bool:
        st = _ep.ep_check_completion(self.handle, channel, cmd_idx)
        if st not in (_ep.EP_OK, _ep.EP_ERR_NOT_READY):
            raise _ep.EpError(st, "ep_check_completion")
        return st == _ep.EP_OK

    def reset(self) -> None:
        _ep.ep_reset(self.handle)
