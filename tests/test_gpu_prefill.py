"""Chunked prefill on the GPU against the fp64 oracle."""

import numpy as np
import pytest

import oracle
from gated_deltanet_scan_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def run_prefill(w, chunk=None, out_dtype="f32", state=None):
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    x = gu.dev_inputs(w)
    if state is not None:
        x["state"] = state
    o = gu.out_like(x["v"], out_dtype)
    gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o,
                            x["cu_seqlens"], chunk=chunk or w.chunk)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    return gu.to_np(o), gu.to_np(x["state"])


def check(w, chunk=None, out_dtype="f32", s_tol=gu.S_TOL):
    o, S = run_prefill(w, chunk, out_dtype)
    o_ref, S_ref = oracle.run_workload(w)
    eo = gu.check_outputs(o, o_ref, out_dtype)
    es = gu.check_state(S, S_ref, s_tol)
    return eo, es


def test_tiny_fp32():
    """B=1, T=64, H 2/4, d=32, fp32, chunk 16, seed 0."""
    check(synth.tiny(), s_tol=1e-5)


def test_qwen35_9b_layer_prefill_T1024():
    """B=1, T=1024, H 16/32, d=128, bf16 q/k/v, zero state, chunk 64."""
    check(synth.prefill_9b(1024))


@pytest.mark.parametrize("run", ["A", "B"])
def test_long_prefill_T16384(run):
    """T=16384 from a N(0,0.02) state; A: log alpha ~ U[-8,-0.01]; B: log alpha = -6.72."""
    check(synth.long_prefill(run, 16384))


@pytest.mark.parametrize("chunk", [16, 64])
@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 128, 192, 256, 320, 449, 1000])
def test_lengths_around_chunk_boundaries(T, chunk):
    """Also 1 to 16 chunks of 64: the tensor-core scan's four-slot operand ring
    (two tiles per chunk, none for X after the last chunk) wraps every two chunks,
    and its two full barriers per tile kind alternate by chunk parity."""
    w = synth.make_workload("len", [T], 16, 32, 128, chunk, "bf16", seed=T, state_std=0.02)
    check(w)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_shapes_and_dtypes_batch3(d, io):
    w = synth.make_workload("shape", [70, 1, 130], 2, 4, d, 64, io, seed=d, state_std=0.02)
    check(w, s_tol=1e-5 if io == "f32" else gu.S_TOL)


def test_bf16_output():
    check(synth.prefill_9b(256), out_dtype="bf16")


def test_varlen_with_empty_sequences():
    lens = [0, 65, 0, 1, 200, 64, 0]
    w = synth.make_workload("varlen_empty", lens, 16, 32, 128, 64, "bf16", seed=5, state_std=0.02)
    check(w)


def test_strong_decay_is_finite_and_exact():
    """log alpha = -6.72 everywhere: the log-space mask keeps every exponent <= 0."""
    w = synth.make_workload("strong", [300], 16, 32, 128, 64, "bf16", seed=6, g_fixed=-6.72, state_std=0.02)
    check(w)


def test_chunk_size_does_not_change_the_result():
    w = synth.make_workload("chunks", [333], 16, 32, 128, 64, "bf16", seed=7, state_std=0.02)
    o64, s64 = run_prefill(w, chunk=64)
    o16, s16 = run_prefill(w, chunk=16)
    # chunk 64 runs on the tensor cores (fp16 factor operands), chunk 16 on CUDA cores in fp32
    assert gu.o_error(o64, o16) < gu.TC_O_TOL
    assert gu.state_error(s64, s16) < gu.TC_S_TOL


def test_prefill_then_decode_handoff():
    """prefill(T1) then T2 decode steps equals prefill(T1 + T2)."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    T1, T2 = 150, 5
    w = synth.make_workload("handoff", [T1 + T2], 16, 32, 128, 64, "bf16", seed=8, state_std=0.02)
    x = gu.dev_inputs(w)
    state = x["state"].clone()
    o = gu.out_like(x["v"], "f32")
    cu1 = torch.tensor([0, T1], dtype=torch.int32, device="cuda")
    gdr.gdr_prefill_chunked(x["q"][:T1], x["k"][:T1], x["v"][:T1], x["g"][:T1], x["beta"][:T1],
                            state, o[:T1], cu1)
    for t in range(T1, T1 + T2):
        sl = slice(t, t + 1)
        gdr.gdr_decode_step(x["q"][sl], x["k"][sl], x["v"][sl], x["g"][sl], x["beta"][sl], state, o[sl])
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.run_workload(w)
    gu.check_outputs(gu.to_np(o), o_ref)
    gu.check_state(gu.to_np(state), S_ref)


def test_packing_equals_separate_calls():
    lens = [40, 129, 64]
    w = synth.make_workload("pack", lens, 16, 32, 128, 64, "bf16", seed=9, state_std=0.02)
    o_all, s_all = run_prefill(w)
    for i, L in enumerate(lens):
        a, b = int(w.cu_seqlens[i]), int(w.cu_seqlens[i + 1])
        wi = synth.make_workload("pack", lens, 16, 32, 128, 64, "bf16", seed=9, state_std=0.02)
        wi.cu_seqlens = np.array([0, L], dtype=np.int32)
        for name in ("q", "k", "v", "g", "beta", "q_bits", "k_bits", "v_bits"):
            setattr(wi, name, np.ascontiguousarray(getattr(w, name)[a:b]))
        wi.state0 = np.ascontiguousarray(w.state0[i:i + 1])
        oi, si = run_prefill(wi)
        assert gu.o_error(oi, o_all[a:b]) < 1e-5
        assert gu.state_error(si[0], s_all[i]) < 1e-6


@pytest.mark.parametrize("h_qk,h_v", [(4, 4), (2, 8)])
def test_tensor_core_head_ratios(h_qk, h_v):
    """One V head per QK head, and four: the factor kernel's X tiles (written by the
    first one or two V heads of a QK head's group) reach every V head."""
    w = synth.make_workload("ratio", [200, 64, 131], h_qk, h_v, 128, 64, "bf16", seed=60 + h_v, state_std=0.02)
    check(w)


@pytest.mark.parametrize("lens", [[1500, 4000], [0, 5000]])
def test_split_prefill_over_two_sequences(lens):
    """16 V heads (8 QK heads) and two sequences: the chunk scan runs 128 CTAs and
    the factors need over two waves, so on a 152-SM GB300 the call splits at a
    chunk (50 of 86 for [1500, 4000], 46 of 79 for [0, 5000]): a sequence that ends
    before the split chunk, one that is cut by it, and an empty one all come out as
    the oracle's."""
    w = synth.make_workload("split2", lens, 8, 16, 128, 64, "bf16", seed=51 + lens[0], state_std=0.02)
    check(w)


@pytest.mark.parametrize("e", [16, 12, -10, -16, -20])
def test_scaled_values_keep_their_relative_accuracy(e):
    """v and the initial state scaled by 2^e (exact in bf16 and fp32).  The
    tensor-core path's fp16 operands R and D~ scale with them; each scan CTA picks
    a power-of-two operand scale from its first V tile and its initial state, so
    that they stay in the middle of fp16's range: at 2^16 (R and D~ up to ~2^21,
    past the fp16 maximum without the scale) and at 2^-16 and 2^-20 (values' RMS
    ~1.5e-5 and ~1e-6, in fp16's subnormals without it) the result keeps the
    unscaled run's relative accuracy and is 2^e times it up to rounding."""
    import dataclasses
    from gated_deltanet_scan_gb300 import synth as sy
    w = synth.make_workload("scaled", [700], 16, 32, 128, 64, "bf16", seed=11, state_std=0.02)
    f = np.float32(2.0 ** e)
    v = w.v * f
    ws = dataclasses.replace(w, name=f"scaled_2^{e}", v=v, v_bits=sy.bf16_bits(v), state0=w.state0 * f)
    assert np.array_equal(sy.bf16_values(ws.v_bits), v)  # the scaling is exact
    check(ws)
    o1, s1 = run_prefill(w)
    o2, s2 = run_prefill(ws)
    assert gu.o_error(o2 / float(f), o1) < 2e-3
    assert gu.state_error(s2 / float(f), s1) < 2e-4
