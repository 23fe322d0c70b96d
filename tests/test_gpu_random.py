"""Seeded random configurations of the whole path against the oracle: layout,
receive rows and TransferCmd records bit-exact, combine within 1 bf16 ulp,
ring invariants, and the arrival signals -- across ranks, tokens, row sizes
on both store paths (TMA bulk stores above 4 KB, store warps at or below),
top-k, channels, ring depth, admission limit, batch, rows per message and SM
budget."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from test_gpu_parity import run_and_check

pytestmark = pytest.mark.gpu

HIDDEN = (8, 64, 256, 520, 1024, 2048, 2056, 4096, 7168)


def random_case(seed: int):
    rng = np.random.default_rng(9000 + seed)
    R = int(rng.choice([1, 2, 3, 5, 8, 16, 32, 64]))
    Er = int(rng.integers(1, 9))
    E = R * Er
    K = int(rng.integers(1, min(8, E) + 1)) if rng.random() < 0.85 else int(min(E, 32))
    H = int(rng.choice(HIDDEN))
    Tpr = int(rng.integers(1, 4096 // max(1, R // 4) // max(1, H // 2048) + 2))
    C = int(rng.integers(1, 9))
    D = int(rng.choice([16, 64, 256, 1024]))
    opts = dict(channels=C, ring_depth=D, max_inflight=int(rng.choice([8, D // 2, D])) if D >= 16 else 8,
                batch=int(rng.integers(1, 9)), rows_per_msg=int(rng.choice([0, 1, 3, 8])))
    if rng.random() < 0.3:
        opts["num_sms"] = int(rng.integers(C + 1, C + 60))
    w = W.Workload(f"random{seed}", R, Tpr, H, E, K, seed=9100 + seed)
    return w, opts


@pytest.mark.parametrize("seed", range(32))
def test_random_configuration(seed):
    w, opts = random_case(seed)
    run_and_check(w, **opts)
