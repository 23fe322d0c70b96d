"""The binding's argument checks (CPU): every tensor the kernels index by the
layer's sizes is checked for type, dtype, device, contiguity and shape before
the library is called."""
import pytest
import torch

CPU = torch.device("cpu")


@pytest.fixture(scope="module")
def check_tensor():
    from combine_ep_layout_04_gb300 import build
    build.build()                      # the binding loads libep.so on import
    from combine_ep_layout_04_gb300.layer import check_tensor
    return check_tensor


def test_a_matching_tensor_passes(check_tensor):
    check_tensor(torch.zeros(4, 3, dtype=torch.int32), "t", torch.int32, CPU, (4, 3))
    check_tensor(torch.zeros(7, 3, dtype=torch.int32), "t", torch.int32, CPU, (None, 3))


@pytest.mark.parametrize("t, exc", [
    (torch.zeros(4, 3, dtype=torch.int64), TypeError),             # dtype
    (torch.zeros(3, 4, dtype=torch.int32).t(), ValueError),        # not contiguous
    (torch.zeros(4, 2, dtype=torch.int32), ValueError),            # shape
    (torch.zeros(12, dtype=torch.int32), ValueError),              # rank
    (torch.zeros(4, 3, 1, dtype=torch.int32), ValueError),         # rank
    ([[0] * 3] * 4, TypeError),                                    # not a tensor
])
def test_a_wrong_tensor_is_refused(check_tensor, t, exc):
    with pytest.raises(exc):
        check_tensor(t, "t", torch.int32, CPU, (4, 3))


def test_a_tensor_on_another_device_is_refused(check_tensor):
    with pytest.raises(ValueError, match="on cpu"):
        check_tensor(torch.zeros(4, 3, dtype=torch.int32), "t", torch.int32, torch.device("cuda", 0), (4, 3))
