"""Failure detection without a fault: a device-side wait that nothing completes
runs out of its bound, the device reports it through the status word, and the
context stays usable (the same bounded wait and report as every mbarrier wait
in the kernels)."""
import time

import pytest
import torch

import oracle
import rwkv_linear_attention_gb300 as wkv7
from rwkv_linear_attention_gb300 import _lib, inputs
from tests.gpu_util import NAMES, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from rwkv_linear_attention_gb300 import build
    build.build()
    return torch.device("cuda:0")


def test_expired_wait_is_reported_and_the_context_survives(dev):
    wkv7.check_device_status()  # start clean
    t0 = time.perf_counter()
    wkv7.diag_bounded_wait(20000)  # 20 ms
    with pytest.raises(wkv7.WKV7Error) as e:
        wkv7.check_device_status()
    elapsed = time.perf_counter() - t0
    assert e.value.status == _lib.ERR_TIMEOUT
    assert 0.015 <= elapsed < 5.0, elapsed
    wkv7.check_device_status()  # the report was read and cleared

    # the next call on the same context runs and is right
    B, H, N = 2, 4, 64
    x = inputs.decode_inputs(B, H, N, steps=1, seed=77, device=dev)
    x = {n: t[0].contiguous() for n, t in x.items()}
    s0 = inputs.initial_state(B, H, N, seed=77, device=dev)
    state = s0.clone()
    o = wkv7.step(x["r"], x["w"], x["k"], x["v"], x["kk"], x["a"], state)
    wkv7.check_device_status()
    o_ref, s_ref = oracle.step(*(x[n].cpu() for n in NAMES), state=s0.double().cpu())
    assert rel_err(o, o_ref) <= 1e-5 and rel_err(state, s_ref) <= 1e-5


def test_rejects_out_of_range_bound(dev):
    for bad in (0, 2000001):
        with pytest.raises(wkv7.WKV7Error) as e:
            wkv7.diag_bounded_wait(bad)
        assert e.value.status == _lib.ERR_INVALID_ARG
