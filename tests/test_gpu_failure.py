"""Failure reporting on the GPU, without a fault: a bounded wait on a barrier that
nothing arrives on gives up, records GDR_ERR_DEVICE_TIMEOUT in the device error
word, and leaves the context usable for the next call."""

import pytest

import oracle
from gated_deltanet_scan_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_stays_usable():
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    assert gdr.gdr_device_error() == 0
    gdr.gdr_selftest_wait_timeout(2_000_000)  # about 1 ms of SM clocks
    assert gdr.gdr_device_error() == gdr.GDR_ERR_DEVICE_TIMEOUT
    assert gdr.gdr_device_error() == 0  # the read cleared it
    # the next call runs normally and matches the oracle
    w = synth.make_workload("after_timeout", [200], 16, 32, 128, 64, "bf16", seed=77, state_std=0.02)
    x = gu.dev_inputs(w)
    o = gu.out_like(x["v"], "f32")
    gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"])
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    o_ref, S_ref = oracle.run_workload(w)
    gu.check_outputs(gu.to_np(o), o_ref)
    gu.check_state(gu.to_np(x["state"]), S_ref)
