"""Torch-facing wrapper of the C ABI: allocates the caller-owned outputs with
torch on the handle's device and passes raw device pointers and the current
CUDA stream to libep.  Marshalling only; all arithmetic is in the library's
kernels (layout, dispatch with its TransferCmd rings, combine)."""
from __future__ import annotations

import dataclasses
import weakref

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


def check_tensor(t, name: str, dtype: torch.dtype, device: torch.device, shape=None) -> None:
    """Raise unless t is a contiguous `dtype` tensor on `device` whose shape
    matches `shape` (None entries match any size).  The kernels index these
    buffers by the layer's sizes, so a wrong one must not reach them."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, the layer is on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and (t.dim() != len(shape) or
                              any(want is not None and got != want for got, want in zip(t.shape, shape))):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple('*' if v is None else v for v in shape)}")


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
    def _layout_shapes(self) -> dict:
        R, T, E = self.R, self.T, self.E
        return {"num_tokens_per_expert": (R, E), "num_tokens_per_rank": (R, R), "is_token_in_rank": (T, R),
                "token_slot": (T, R), "recv_off": (R, R), "send_off": (R, R), "msg_count": (R, R),
                "recv_count": (R,), "recv_base": (R,), "expert_off": (E,)}

    def _check_layout(self, lay: Layout) -> None:
        """Shapes, dtypes and device of a Layout's tensors, checked once per
        Layout object (a Layout that passed is marked with this layer)."""
        if not isinstance(lay, Layout):
            raise TypeError(f"expected a Layout, got {type(lay).__name__}")
        ref = getattr(lay, "_checked_by", None)
        if ref is not None and ref() is self:
            return
        for f, shape in self._layout_shapes().items():
            check_tensor(getattr(lay, f), f, torch.uint8 if f == "is_token_in_rank" else torch.int32,
                         self.device, shape)
        lay._checked_by = weakref.ref(self)   # no strong reference: the layer may go first

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
        check_tensor(topk_idx, "topk_idx", torch.int32, self.device, (self.T, self.K))
        out = self.alloc_layout() if out is None else out
        self._check_layout(out)
        out.n_recv = _ep.ep_layout(self.handle, topk_idx.data_ptr(), out.struct(), _stream(self.device), want_n=sync)
        return out

    def dispatch(self, x: torch.Tensor, lay: Layout, recv: torch.Tensor | None = None,
                 src_ranks: tuple[int, int] | None = None) -> torch.Tensor:
        """ep_dispatch (ep_dispatch_ranks for src_ranks=(begin, end)).
        x: bf16 [T, H].  Returns recv bf16 [capacity, H]."""
        check_tensor(x, "x", torch.bfloat16, self.device, (self.T, self.H))
        self._check_layout(lay)
        if recv is None:
            if lay.n_recv is None:
                raise ValueError("dispatch needs recv or a layout computed with sync=True")
            recv = torch.empty((lay.n_recv, self.H), dtype=torch.bfloat16, device=self.device)
        check_tensor(recv, "recv", torch.bfloat16, self.device, (None, self.H))
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
        check_tensor(expert_out, "expert_out", torch.bfloat16, self.device, (None, self.H))
        check_tensor(topk_weights, "topk_weights", torch.float32, self.device, (self.T, self.K))
        check_tensor(topk_idx, "topk_idx", torch.int32, self.device, (self.T, self.K))
        self._check_layout(lay)
        if out is None:
            out = torch.empty((self.T, self.H), dtype=torch.bfloat16, device=self.device)
        check_tensor(out, "out", torch.bfloat16, self.device, (self.T, self.H))
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
        check_tensor(topk_idx, "topk_idx", torch.int32, self.device, (self.T, self.K))
        check_tensor(topk_weights, "topk_weights", torch.float32, self.device, (self.T, self.K))
        self._check_layout(lay)
        if out is None:
            if lay.n_recv is None:
                raise ValueError("expert_layout needs `out` or a layout computed with sync=True")
            N, K = lay.n_recv, self.K
            i32 = dict(dtype=torch.int32, device=self.device)
            out = ExpertLayout(torch.empty((N, K), **i32), torch.empty((N, K), dtype=torch.float32, device=self.device),
                               torch.empty((N,), **i32), torch.empty((self.T * K,), **i32),
                               torch.empty((self.E,), **i32))
        if not isinstance(out, ExpertLayout):
            raise TypeError(f"out: expected an ExpertLayout, got {type(out).__name__}")
        n = out.recv_src_token.shape[0] if isinstance(out.recv_src_token, torch.Tensor) else None
        check_tensor(out.recv_src_token, "recv_src_token", torch.int32, self.device, (None,))
        check_tensor(out.recv_topk_idx, "recv_topk_idx", torch.int32, self.device, (n, self.K))
        check_tensor(out.recv_topk_weights, "recv_topk_weights", torch.float32, self.device, (n, self.K))
        check_tensor(out.expert_rows, "expert_rows", torch.int32, self.device, (None,))
        check_tensor(out.expert_count, "expert_count", torch.int32, self.device, (self.E,))
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
        check_tensor(status, "status", torch.int32, self.device, (None,))
        if status.numel() < 1:
            raise ValueError("status: needs at least one element")
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


class SmSplit:
    """Two disjoint SM partitions of one GPU (ep_sm_split_create): `comm`, a
    torch stream for layout/dispatch/combine (use an EpLayer made with
    num_sms=comm_sms), and `compute`, a torch stream for the caller's
    computation.  Order work between them with events only."""

    def __init__(self, compute_sms: int, device=None):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self._s = _ep.ep_sm_split_create(self.device.index, int(compute_sms))
        cs, self.comm_sms, ks, self.compute_sms = _ep.ep_sm_split_get(self._s)
        self.comm = torch.cuda.ExternalStream(cs, device=self.device)
        self.compute = torch.cuda.ExternalStream(ks, device=self.device)

    def sm_ids(self, stream, blocks: int = 4096) -> set:
        """SM ids that `blocks` short blocks enqueued on `stream` ran on."""
        out = torch.full((blocks,), -1, dtype=torch.int32, device=self.device)
        _ep.ep_sm_ids(stream.cuda_stream, blocks, out.data_ptr())
        stream.synchronize()
        return set(out.cpu().tolist())

    def close(self) -> None:
        if self._s is not None:
            _ep.ep_sm_split_destroy(self._s)
            self._s = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
