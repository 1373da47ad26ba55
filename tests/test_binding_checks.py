"""CPU tests of the Python binding's argument checks (no device is touched: the
tensors and streams below are stand-ins carrying only what the checks read)."""
import types

import pytest
import torch

from gated_delta_rule_40_gb300 import kda


class _Fake:
    def __init__(self, device, dtype=torch.bfloat16, shape=(2, 3), contiguous=True):
        self.device, self.dtype, self.shape, self._c = device, dtype, shape, contiguous

    def is_contiguous(self):
        return self._c


@pytest.fixture
def on_device_1(monkeypatch):
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)


def test_check_accepts_a_tensor_on_the_current_device(on_device_1):
    kda._check(_Fake(torch.device("cuda", 1)), "q", torch.bfloat16, (2, 3))


def test_check_rejects_a_tensor_on_another_device(on_device_1):
    with pytest.raises(ValueError, match="current CUDA device"):
        kda._check(_Fake(torch.device("cuda", 0)), "q", torch.bfloat16, (2, 3))


def test_check_rejects_dtype_shape_layout_and_host_tensors(on_device_1):
    dev = torch.device("cuda", 1)
    with pytest.raises(TypeError):
        kda._check(_Fake(dev, dtype=torch.float16), "q", torch.bfloat16)
    with pytest.raises(ValueError, match="shape"):
        kda._check(_Fake(dev, shape=(3, 2)), "q", torch.bfloat16, (2, 3))
    with pytest.raises(ValueError, match="contiguous"):
        kda._check(_Fake(dev, contiguous=False), "q", torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        kda._check(_Fake(torch.device("cpu")), "q", torch.bfloat16)
    with pytest.raises(ValueError, match="required"):
        kda._check(None, "q", torch.bfloat16)
    kda._check(None, "initial_state", torch.float32, optional=True)
    kda._check(_Fake(torch.device("cpu")), "q", torch.bfloat16, device="cpu")   # host-buffer entry point


def test_stream_on_another_device_is_rejected(on_device_1):
    other = types.SimpleNamespace(device=torch.device("cuda", 0), cuda_stream=0)
    with pytest.raises(ValueError, match="current CUDA device"):
        kda._stream(other)
    same = types.SimpleNamespace(device=torch.device("cuda", 1), cuda_stream=1234)
    assert kda._stream(same).value == 1234
