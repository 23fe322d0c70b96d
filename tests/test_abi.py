"""The C-ABI library without a GPU: it builds, loads, exports every function
include/ep.h declares, and its host-only calls (defaults, argument checks,
status strings) behave.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ep():
    from combine_ep_layout_04_gb300 import build
    build.build()
    from combine_ep_layout_04_gb300 import _ep
    return _ep


def declared_functions():
    names = []
    for path in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not path.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", path)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(ep_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(ep):
    names = declared_functions()
    assert len(names) >= 14
    lib = ctypes.CDLL(ep.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ep.EXPORTED)


def test_defaults_are_the_tuning_table(ep, golden):
    g = golden("tuning_table.txt")
    cfg = ep.ep_config_init(32, 4096, 7168, 256, 8)
    assert cfg.channels == g["HT_CHANNELS"][0]
    assert cfg.ring_depth == g["FIFO_DEPTH"][0]
    assert cfg.max_inflight == g["MAX_INFLIGHT"][0]
    assert cfg.drain_batch == g["DRAIN_BATCH_SIZE"][0]
    assert cfg.batch == g["MAX_BATCH"][0]
    assert cfg.rows_per_msg == 0 and cfg.debug_flags == 0
    assert ep.ep_config_check(cfg) == ep.EP_OK
    # slot of a command index: idx % depth (the ring's completion check)
    for idx, slot in g["SLOT_OF"]:
        assert idx & (cfg.ring_depth - 1) == slot


@pytest.mark.parametrize("field,value", [
    ("num_ranks", 0), ("num_ranks", 65), ("tokens_per_rank", 0), ("hidden", 100), ("hidden", 0),
    ("num_experts", 250), ("topk", 0), ("topk", 33), ("channels", 0), ("channels", 65),
    ("ring_depth", 1000), ("ring_depth", 4), ("ring_depth", 16384), ("max_inflight", 2048), ("max_inflight", 4), ("batch", 9),
    ("batch", 0), ("rows_per_msg", -1), ("drain_batch", 48), ("drain_batch", 1024), ("debug_flags", 4),
    ("num_sms", -1), ("num_sms", 5), ("reserved", 1),
])
def test_invalid_configs_are_rejected_on_the_host(ep, field, value):
    cfg = ep.ep_config_init(32, 128, 7168, 256, 8)
    setattr(cfg, field, value)
    assert ep.ep_config_check(cfg) == ep.EP_ERR_INVALID_ARG
    h = ep._h()
    # rejected before any CUDA call, so this works without a GPU
    assert ep.lib.ep_create(ctypes.byref(cfg), ctypes.byref(h)) == ep.EP_ERR_INVALID_ARG
    assert not h.value


def test_topk_larger_than_experts_is_rejected(ep):
    cfg = ep.ep_config_init(4, 8, 64, 4, 5)
    assert ep.ep_config_check(cfg) == ep.EP_ERR_INVALID_ARG


def test_status_strings(ep):
    assert [ep.status_str(i) for i in range(6)] == [
        "EP_OK", "EP_ERR_INVALID_ARG", "EP_ERR_CAPACITY", "EP_ERR_TIMEOUT", "EP_ERR_CUDA", "EP_ERR_NOT_READY"]


def test_null_handles_are_rejected(ep):
    assert ep.lib.ep_destroy(None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_reset(None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_layout(None, None, None, None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_dispatch(None, None, None, None, 0, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_combine(None, None, 0, None, None, None, None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_get_info(None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_cmd_log_get(None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_check_completion(None, 0, 0) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_expert_layout(None, None, None, None, None, 0, 0, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_dispatch_ranks(None, None, None, None, 0, 0, 0, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_combine_tokens(None, None, 0, None, None, None, None, 0, 0, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_signal_ptr(None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_signal_get(None, None, 0) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_signal_reset(None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_wait_signal(None, 0, 0, 0, None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_sm_split_get(None, None, None, None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_sm_split_destroy(None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_sm_ids(None, 1, None) == ep.EP_ERR_INVALID_ARG


def test_sm_split_arguments_are_checked_before_the_device(ep):
    import ctypes
    s = ctypes.c_void_p()
    assert ep.lib.ep_sm_split_create(0, 0, ctypes.byref(s)) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_sm_split_create(-1, 8, ctypes.byref(s)) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_sm_split_create(0, 8, None) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_sm_ids(None, 0, None) == ep.EP_ERR_INVALID_ARG


def test_struct_sizes_match_the_header(ep):
    assert ctypes.sizeof(ep.ep_transfer_cmd) == 32
    assert ctypes.sizeof(ep.ep_config) == 64
    assert ctypes.sizeof(ep.ep_layout_out) == 80
    assert ctypes.sizeof(ep.ep_ring_stats) == 48
    assert ctypes.sizeof(ep.ep_expert_layout_out) == 40
