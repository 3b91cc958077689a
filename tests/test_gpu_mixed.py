"""A prefill and a decode step of another batch in one chunk-scan launch
(gdr_prefill_with_decode, continuous batching): both parts equal the separate
calls bit for bit (gdr_prefill_chunked, gdr_decode_step), and match the oracle."""

import numpy as np
import pytest

import oracle
from gated_deltanet_scan_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _decode_inputs(b, seed, **kw):
    w = synth.make_workload("mix_dec", [1] * b, 16, 32, 128, 64, "bf16", seed=seed, state_std=0.02, **kw)
    return w, gu.dev_inputs(w)


def _mixed_vs_separate(pre_w, dec_b, seed, qk_l2norm=False, beta_logits=False):
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    kw = dict(qk_raw_scale=(0.5, 4.0), beta_logits=True) if qk_l2norm else {}
    dw, dx = _decode_inputs(dec_b, seed, **kw)
    px = gu.dev_inputs(pre_w)
    flags = dict(qk_l2norm=qk_l2norm, beta_logits=beta_logits)
    # separate calls
    s_pre, s_dec = px["state"].clone(), dx["state"].clone()
    o_pre, o_dec = gu.out_like(px["v"], "f32"), gu.out_like(dx["v"], "f32")
    gdr.gdr_prefill_chunked(px["q"], px["k"], px["v"], px["g"], px["beta"], s_pre, o_pre, px["cu_seqlens"],
                            t_total=pre_w.q.shape[0], **flags)
    gdr.gdr_decode_step(dx["q"], dx["k"], dx["v"], dx["g"], dx["beta"], s_dec, o_dec, **flags)
    # one mixed call
    m_pre, m_dec = px["state"].clone(), dx["state"].clone()
    mo_pre, mo_dec = gu.out_like(px["v"], "f32"), gu.out_like(dx["v"], "f32")
    gdr.gdr_prefill_with_decode(px["q"], px["k"], px["v"], px["g"], px["beta"], m_pre, mo_pre, px["cu_seqlens"],
                                dx["q"], dx["k"], dx["v"], dx["g"], dx["beta"], m_dec, mo_dec,
                                t_total=pre_w.q.shape[0], **flags)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    for a, b in ((o_pre, mo_pre), (s_pre, m_pre), (o_dec, mo_dec), (s_dec, m_dec)):
        assert torch.equal(a, b)
    return dw, gu.to_np(mo_dec), gu.to_np(m_dec), gu.to_np(mo_pre), gu.to_np(m_pre)


def _check_decode(dw, o, s, qk_l2norm=False):
    if qk_l2norm:
        o_ref, s_ref = oracle.gdr_fused(dw.cu_seqlens, dw.q, dw.k, dw.v, dw.g, dw.beta, dw.state0, qk_l2norm=True,
                                        beta_logits=True)
    else:
        o_ref, s_ref = oracle.run_workload(dw)
    gu.check_outputs(o, o_ref)
    gu.check_state(s, s_ref)


def test_long_prefill_with_decode_batch64():
    """The bench's step: prefill B=1, T=16384 (split into two scan launches; the
    decode blocks ride the second) and a B=64 decode step."""
    pw = synth.long_prefill("A", 16384)
    dw, o, s, _, _ = _mixed_vs_separate(pw, 64, seed=81)
    _check_decode(dw, o, s)


@pytest.mark.parametrize("lens,dec_b", [([300], 5), ([200, 0, 700], 3), ([1], 1)])
def test_short_prefills_with_decode(lens, dec_b):
    """One scan launch (no split); a packed prefill with an empty sequence."""
    pw = synth.make_workload("mix_pre", lens, 16, 32, 128, 64, "bf16", seed=82 + len(lens), state_std=0.02)
    dw, o, s, op, sp = _mixed_vs_separate(pw, dec_b, seed=83 + dec_b)
    _check_decode(dw, o, s)
    o_ref, s_ref = oracle.run_workload(pw)
    gu.check_outputs(op, o_ref)
    gu.check_state(sp, s_ref)


def test_packed_prefill_leaving_no_free_sm():
    """8 sequences keep every SM busy with scan CTAs: the one decode block runs
    after them, still in the same launch."""
    pw = synth.make_workload("mix_packed", [700, 333, 64, 129, 1000, 65, 512, 255], 16, 32, 128, 64, "bf16",
                             seed=84, state_std=0.02)
    dw, o, s, _, _ = _mixed_vs_separate(pw, 4, seed=85)
    _check_decode(dw, o, s)


def test_mixed_with_fused_qk_norm_and_beta_logits():
    pw = synth.make_workload("mix_fused", [500], 16, 32, 128, 64, "bf16", seed=86, state_std=0.02,
                             qk_raw_scale=(0.5, 4.0), beta_logits=True)
    dw, o, s, _, _ = _mixed_vs_separate(pw, 6, seed=87, qk_l2norm=True, beta_logits=True)
    _check_decode(dw, o, s, qk_l2norm=True)


def test_empty_prefill_is_a_decode_step():
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    dw, dx = _decode_inputs(3, seed=88)
    pw = synth.make_workload("mix_empty", [0], 16, 32, 128, 64, "bf16", seed=89, state_std=0.02)
    px = gu.dev_inputs(pw)
    o = gu.out_like(dx["v"], "f32")
    gdr.gdr_prefill_with_decode(px["q"], px["k"], px["v"], px["g"], px["beta"], px["state"],
                                gu.out_like(px["v"], "f32"), px["cu_seqlens"], dx["q"], dx["k"], dx["v"], dx["g"],
                                dx["beta"], dx["state"], o, t_total=0)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    _check_decode(dw, gu.to_np(o), gu.to_np(dx["state"]))
