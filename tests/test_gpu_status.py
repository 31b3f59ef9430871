"""Failure reporting on the GPU, tested without faulting or hanging it: a kernel's bounded
wait on a barrier that nothing completes must give up and surface as
MQ_ERR_DEVICE_TIMEOUT, after which the context keeps working."""
import numpy as np
import pytest

from quantized_q8_activation_quantize_gb300 import binding as B
from quantized_q8_activation_quantize_gb300 import inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def test_clean_status_after_normal_work():
    x = inputs.activations(np.random.default_rng(0), 4, 256)
    G.gpu_plane(x)
    assert B.mq_device_status() == B.MQ_OK


def test_forced_wait_timeout_is_reported_then_cleared():
    import torch
    B.mq_debug_forced_timeout(20000)              # 20 ms bound
    with pytest.raises(B.MQError) as e:
        B.mq_device_status()
    assert e.value.status == B.MQ_ERR_DEVICE_TIMEOUT
    assert "forced-test-wait" in str(e.value)
    assert B.mq_device_status() == B.MQ_OK          # cleared
    # the context is intact: a normal call still matches the oracle
    x = inputs.activations(np.random.default_rng(1), 3, 512)
    _, got = G.gpu_plane(x)
    G.assert_plane_equal(got, G.oracle_plane(x))
    torch.cuda.synchronize()


def test_empty_calls_launch_nothing():
    import torch
    y = torch.zeros(1, device="cuda")
    assert B.mq_gemm_q4k(16, 0, 256, 256, 4, y) == B.MQ_OK
    assert B.mq_gemv_q6k(16, 8, 256, 256, 0, y) == B.MQ_OK
    assert B.mq_quantize_q8(16, 0, 256, None, 0.0, 256) == B.MQ_OK
