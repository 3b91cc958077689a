"""gdr_prefill_chunked_static: the prefill with the library's fixed scratch array.

Checked against gdr_prefill_chunked (caller workspace) on the same inputs, two
calls in a row each (the second continues from the first's state), and its
size limit checked on the host."""

import ctypes

import numpy as np
import pytest

import gated_deltanet_scan_gb300 as gdr
from gated_deltanet_scan_gb300 import synth
from tests import gpu_util as gu


def test_static_entry_rejects_oversize_before_launch():
    L = gdr.lib()
    cap = L.gdr_prefill_static_workspace_capacity()
    assert cap == 64 << 20
    d = gdr.gdr_dims(h_qk=16, h_v=32, d_k=128, d_v=128, chunk=64, in_dtype=gdr.GDR_BF16,
                     out_dtype=gdr.GDR_F32, scale=1.0)
    A = 0x100000  # aligned stand-in addresses: nothing is dereferenced on this path
    # one chunk position of 32 V heads and 16 QK heads takes 32 * 17152 + 16 * 16384
    # bytes: the 64 MiB array holds 82 positions, i.e. one sequence of up to 81
    # chunks (5184 tokens; one position is the per-sequence spare)
    assert L.gdr_prefill_workspace_bytes(ctypes.byref(d), 1, 5184) <= cap
    assert L.gdr_prefill_workspace_bytes(ctypes.byref(d), 1, 5185) > cap
    assert L.gdr_prefill_workspace_bytes(ctypes.byref(d), 2, 5120) <= cap
    assert L.gdr_prefill_workspace_bytes(ctypes.byref(d), 2, 5121) > cap
    for n, t in ((1, 5185), (2, 5121), (1, 1 << 20)):
        st = L.gdr_prefill_chunked_static(ctypes.byref(d), n, A, t, A, A, A, A, A, A, A, None)
        assert st == gdr.GDR_ERR_UNSUPPORTED, (n, t, st)


@pytest.mark.gpu
def test_static_entry_matches_workspace_entry_twice():
    torch = gu.require_gpu()
    w = synth.make_workload("no_alloc", [300, 77, 0, 129], 16, 32, 128, 64, "bf16", seed=71, state_std=0.02)
    x = gu.dev_inputs(w)
    s_ws, s_st = x["state"].clone(), x["state"].clone()
    for _ in range(2):  # two calls in a row: the second starts from the first's state
        o_ws, o_st = gu.out_like(x["v"], "f32"), gu.out_like(x["v"], "f32")
        gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], s_ws, o_ws, x["cu_seqlens"])
        gdr.gdr_prefill_chunked_static(x["q"], x["k"], x["v"], x["g"], x["beta"], s_st, o_st, x["cu_seqlens"])
        torch.cuda.synchronize()
        assert np.array_equal(gu.to_np(o_ws), gu.to_np(o_st))
        assert np.array_equal(gu.to_np(s_ws), gu.to_np(s_st))
    assert gdr.gdr_device_error(device=x["q"].device) == 0


@pytest.mark.gpu
def test_static_entry_at_its_largest_single_sequence():
    """One Qwen3.5-9B sequence of 5184 tokens fills the fixed array to its last
    chunk position.  At this length gdr_prefill_chunked splits the prefill into
    four launches (the static entry keeps two), which regroups a few products,
    so the two agree to rounding: both are checked against the oracle, and
    against each other within the tensor-core path's own spread."""
    import oracle

    torch = gu.require_gpu()
    w = synth.make_workload("no_alloc_max", [5184], 16, 32, 128, 64, "bf16", seed=72, state_std=0.02)
    x = gu.dev_inputs(w)
    s_ws, s_st = x["state"].clone(), x["state"].clone()
    o_ws, o_st = gu.out_like(x["v"], "f32"), gu.out_like(x["v"], "f32")
    gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], s_ws, o_ws, x["cu_seqlens"])
    gdr.gdr_prefill_chunked_static(x["q"], x["k"], x["v"], x["g"], x["beta"], s_st, o_st, x["cu_seqlens"])
    torch.cuda.synchronize()
    assert gdr.gdr_device_error(device=x["q"].device) == 0
    o_ref, s_ref = oracle.run_workload(w)
    for o, s in ((o_ws, s_ws), (o_st, s_st)):
        gu.check_outputs(gu.to_np(o), o_ref)
        gu.check_state(gu.to_np(s), s_ref)
    assert gu.o_error(gu.to_np(o_st), gu.to_np(o_ws)) < gu.TC_O_TOL
    assert gu.state_error(gu.to_np(s_st), gu.to_np(s_ws)) < gu.TC_S_TOL
