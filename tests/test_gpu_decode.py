"""Decode step on the GPU against the fp64 oracle."""

import numpy as np
import pytest

import oracle
from gated_deltanet_scan_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _step_inputs(w, s, b, dev):
    torch = gu.torch_mod()
    rows = slice(s * b, (s + 1) * b)

    def io(vals, bits):
        if w.io == "bf16":
            return torch.from_numpy(bits[rows].view(np.int16).copy()).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(vals[rows], dtype=np.float32)).to(dev)

    return (io(w.q, w.q_bits), io(w.k, w.k_bits), io(w.v, w.v_bits),
            torch.from_numpy(np.ascontiguousarray(w.g[rows])).to(dev),
            torch.from_numpy(np.ascontiguousarray(w.beta[rows])).to(dev))


def _run_decode(w, b, steps, out_dtype="f32"):
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    state = torch.from_numpy(np.ascontiguousarray(w.state0)).cuda()
    outs = []
    for s in range(steps):
        q, k, v, g, beta = _step_inputs(w, s, b, "cuda")
        o = gu.out_like(v, out_dtype)
        gdr.gdr_decode_step(q, k, v, g, beta, state, o)
        outs.append(o)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    return np.concatenate([gu.to_np(o) for o in outs]), gu.to_np(state)


def _oracle_decode(w, b, steps):
    # step-major rows: token s*b + i belongs to sequence i
    T = b * steps
    order = np.arange(T).reshape(steps, b).T.reshape(-1)  # sequence-major token order
    cu = np.arange(0, T + 1, steps)
    o, S = oracle.gdr_sequential(cu, w.q[order], w.k[order], w.v[order], w.g[order], w.beta[order], w.state0)
    o_step = np.empty_like(o)
    o_step[order] = o
    return o_step[:T], S


def test_decode_qwen35_9b_batch64_256_steps():
    """B=64 sequences x 256 consecutive steps, H 16/32, d=128, bf16 q/k/v, state ~ N(0, 0.02)."""
    w = synth.decode_batch(64, 256)
    o, S = _run_decode(w, 64, 256)
    o_ref, S_ref = _oracle_decode(w, 64, 256)
    gu.check_outputs(o, o_ref)
    gu.check_state(S, S_ref)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("io,out", [("f32", "f32"), ("bf16", "f32"), ("bf16", "bf16")])
def test_decode_small_shapes(d, io, out):
    b, steps = 3, 5
    w = synth.make_workload("dec_small", [1] * (b * steps), 2, 4, d, 16, io, seed=21 + d,
                            state_std=0.05, n_states=b)
    o, S = _run_decode(w, b, steps, out)
    o_ref, S_ref = _oracle_decode(w, b, steps)
    gu.check_outputs(o, o_ref, out)
    gu.check_state(S, S_ref, 1e-5 if io == "f32" else gu.S_TOL)


def test_decode_equals_one_token_prefill():
    """A decode step and a one-token prefill from the same state agree (same math, two kernels;
    the prefill's tensor-core operands are fp16)."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    w = synth.make_workload("dec1", [1] * 4, 16, 32, 128, 64, "bf16", seed=33, state_std=0.02)
    x = gu.dev_inputs(w)
    s1, s2 = x["state"].clone(), x["state"].clone()
    o1, o2 = gu.out_like(x["v"], "f32"), gu.out_like(x["v"], "f32")
    gdr.gdr_decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], s1, o1)
    gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], s2, o2, x["cu_seqlens"], chunk=64)
    torch.cuda.synchronize()
    assert gu.o_error(gu.to_np(o1), gu.to_np(o2)) < gu.TC_O_TOL
    assert gu.state_error(gu.to_np(s1), gu.to_np(s2)) < gu.TC_S_TOL


def test_decode_overlapped_beside_a_prefill():
    """A decode step queued right after a long prefill as a programmatic dependent
    launch runs beside the prefill's last chunk-scan launch; both give the
    oracle's results, three times in a row on one stream."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    pre = synth.make_workload("ovl_pre", [2048], 16, 32, 128, 64, "bf16", seed=41, state_std=0.02)
    dec = synth.decode_batch(8, 3, seed=42)
    x = gu.dev_inputs(pre)
    o_pre = gu.out_like(x["v"], "f32")
    dstate = torch.from_numpy(np.ascontiguousarray(dec.state0)).cuda()
    outs = []
    for s in range(3):
        x["state"].copy_(torch.from_numpy(np.ascontiguousarray(pre.state0)))
        gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o_pre, x["cu_seqlens"],
                                chunk=64)
        q, k, v, g, beta = _step_inputs(dec, s, 8, "cuda")
        o = gu.out_like(v, "f32")
        gdr.gdr_decode_step_overlapped(q, k, v, g, beta, dstate, o)
        outs.append(o)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    o_ref, s_ref = oracle.run_workload(pre)
    gu.check_outputs(gu.to_np(o_pre), o_ref)
    gu.check_state(gu.to_np(x["state"]), s_ref)
    od_ref, sd_ref = _oracle_decode(dec, 8, 3)
    gu.check_outputs(np.concatenate([gu.to_np(o) for o in outs]), od_ref)
    gu.check_state(gu.to_np(dstate), sd_ref)
