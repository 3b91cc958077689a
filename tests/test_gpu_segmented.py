"""Two-level (segment-parallel) prefill on the GPU against the fp64 oracle and
against the ordinary one-chain prefill."""

import numpy as np
import pytest

import oracle
from gated_deltanet_scan_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

SLOW = (-0.05, -0.001)  # the start state survives whole segments: the combine matters


def run_segmented(w, P, out_dtype="f32"):
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    x = gu.dev_inputs(w)
    o = gu.out_like(x["v"], out_dtype)
    gdr.gdr_prefill_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"], P)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    return gu.to_np(o), gu.to_np(x["state"])


def run_plain(w):
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    x = gu.dev_inputs(w)
    o = gu.out_like(x["v"], "f32")
    gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"])
    torch.cuda.synchronize()
    return gu.to_np(o), gu.to_np(x["state"])


@pytest.mark.parametrize("T,P,regime", [
    (1000, 2, "slow"), (4096, 4, "slow"), (5000, 5, "uniform"), (3000, 3, "fixed"), (4033, 8, "slow"),
])
def test_segmented_matches_oracle(T, P, regime):
    """Few heads (4 V heads, 2 QK heads), one long sequence with a ragged last
    chunk, cut into P segments; slow decay carries the start state across whole
    segments, so the transitions, the combine and the fix-up all count."""
    kw = dict(g_fixed=-6.72) if regime == "fixed" else dict(g_range=SLOW) if regime == "slow" else {}
    w = synth.make_workload(f"seg_{regime}", [T], 2, 4, 128, 64, "bf16", seed=T + P, state_std=0.02, **kw)
    o, S = run_segmented(w, P)
    o_ref, S_ref = oracle.run_workload(w)
    gu.check_outputs(o, o_ref)
    gu.check_state(S, S_ref)
    o1, S1 = run_plain(w)
    assert gu.o_error(o, o1) < gu.TC_O_TOL
    assert gu.state_error(S, S1) < gu.TC_S_TOL


def test_segmented_qwen_heads_and_bf16_output():
    """Qwen3.5-9B heads (16 QK / 32 V): two segments over 2000 tokens, bf16 output."""
    w = synth.make_workload("seg_9b", [2000], 16, 32, 128, 64, "bf16", seed=81, state_std=0.02, g_range=SLOW)
    o, S = run_segmented(w, 2, out_dtype="bf16")
    o_ref, S_ref = oracle.run_workload(w)
    gu.check_outputs(o, o_ref, "bf16")
    gu.check_state(S, S_ref)


def test_segmented_packed_sequences_of_unequal_length():
    """Segments are cut on chunk positions of the longest possible sequence: a
    short sequence lies in the first segments only, an empty one is untouched,
    and every state and output comes out as the oracle's."""
    lens = [3000, 700, 0, 1500]
    w = synth.make_workload("seg_pack", lens, 2, 4, 128, 64, "bf16", seed=82, state_std=0.02, g_range=SLOW)
    o, S = run_segmented(w, 3)
    o_ref, S_ref = oracle.run_workload(w)
    gu.check_outputs(o, o_ref)
    gu.check_state(S, S_ref)


def test_more_segments_than_chunks_and_one_segment():
    """P larger than the chunk count means one segment per chunk; P = 1 is the
    ordinary prefill."""
    for T, P in ((130, 8), (100, 1)):
        w = synth.make_workload("seg_small", [T], 2, 4, 128, 64, "bf16", seed=83 + T, state_std=0.02, g_range=SLOW)
        o, S = run_segmented(w, P)
        o_ref, S_ref = oracle.run_workload(w)
        gu.check_outputs(o, o_ref)
        gu.check_state(S, S_ref)


def test_segments_hint_on_this_gpu():
    """The hint puts every run of the scan launch on the GPU at once: 4 V heads of
    one 16K-token sequence get (2P - 1) * 16 CTAs <= SMs; 32 V heads get one chain."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    q = torch.empty((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    v4 = torch.empty((1, 4, 128), dtype=torch.bfloat16, device="cuda")
    o4 = torch.empty((1, 4, 128), dtype=torch.float32, device="cuda")
    P = gdr.gdr_prefill_segments_hint(q, v4, o4, 1, 16384)
    assert P == min(8, ((sms // 16) + 1) // 2)
    q32 = torch.empty((1, 16, 128), dtype=torch.bfloat16, device="cuda")
    v32 = torch.empty((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    o32 = torch.empty((1, 32, 128), dtype=torch.float32, device="cuda")
    assert gdr.gdr_prefill_segments_hint(q32, v32, o32, 1, 16384) == 1
