"""Packed variable-length prefill, then a 16-token verify block per sequence from
a state snapshot, accepting a random prefix and re-feeding it (the prompt-lookup
decoding loop of the Qwen3.5-9B NPU model card, "New in v2"), against the
oracle's sequential result; and the same prefix committed from the block's cached
corrections (gdr_verify_commit) instead of re-fed."""

import numpy as np
import pytest

import oracle
from gated_deltanet_scan_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _verify_flow(w, n_verify=16):
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    vb = w.extra["verify"]
    acc = np.asarray(w.extra["accepted"], dtype=np.int64)
    n = w.n_seqs

    x = gu.dev_inputs(w)
    o = gu.out_like(x["v"], "f32")
    gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"])
    state = x["state"]

    y = gu.dev_inputs(vb)
    snap = torch.empty_like(state)
    ov = gu.out_like(y["v"], "f32")
    deltas = torch.full(y["v"].shape, float("nan"), dtype=torch.float32, device="cuda")
    gdr.gdr_verify_block(y["q"], y["k"], y["v"], y["g"], y["beta"], state, snap, ov, n_verify, deltas=deltas)
    state_after_block = state.clone()

    # commit the accepted prefix from the cached corrections (no re-feed)
    state_commit = torch.full_like(state, float("nan"))
    acc_dev = torch.from_numpy(acc.astype(np.int32)).cuda()
    gdr.gdr_verify_commit(y["k"], y["g"], deltas, snap, state_commit, acc_dev, n_verify)

    # accept a_s tokens per sequence: restore the snapshot, re-feed the accepted prefix
    gdr.gdr_state_restore(snap, state)
    rows = np.concatenate([np.arange(s * n_verify, s * n_verify + acc[s]) for s in range(n)]).astype(np.int64)
    cu = np.zeros(n + 1, dtype=np.int32)
    cu[1:] = np.cumsum(acc)
    idx = torch.from_numpy(rows).cuda()
    pick = {k: y[k].index_select(0, idx).contiguous() for k in ("q", "k", "v", "g", "beta")}
    o_re = gu.out_like(pick["v"], "f32")
    gdr.gdr_prefill_chunked(pick["q"], pick["k"], pick["v"], pick["g"], pick["beta"], state, o_re,
                            torch.from_numpy(cu).cuda(), t_total=int(cu[-1]))
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    return (gu.to_np(o), gu.to_np(ov), gu.to_np(snap), gu.to_np(state_after_block),
            gu.to_np(o_re), gu.to_np(state), rows, acc, gu.to_np(state_commit))


def _oracle_flow(w, n_verify=16):
    vb = w.extra["verify"]
    acc = np.asarray(w.extra["accepted"], dtype=np.int64)
    o_pre, S_pre = oracle.run_workload(w)
    # the whole 16-token block from the prefill state
    o_blk, S_blk = oracle.gdr_sequential(vb.cu_seqlens, vb.q, vb.k, vb.v, vb.g, vb.beta, S_pre)
    # the accepted prefix only
    rows = np.concatenate([np.arange(s * n_verify, s * n_verify + acc[s]) for s in range(w.n_seqs)])
    cu = np.zeros(w.n_seqs + 1, dtype=np.int64)
    cu[1:] = np.cumsum(acc)
    o_acc, S_acc = oracle.gdr_sequential(cu, vb.q[rows], vb.k[rows], vb.v[rows], vb.g[rows], vb.beta[rows], S_pre)
    return o_pre, S_pre, o_blk, S_blk, o_acc, S_acc


def test_varlen_prefill_then_verify_and_refeed():
    """8 sequences, lengths ~ U{512..8192}, H 16/32, d=128, bf16; verify 16 tokens
    from the snapshot, accept a ~ U{0..16}, re-feed the accepted tokens."""
    w = synth.varlen_verify()
    o, ov, snap, s_blk, o_re, s_final, rows, acc, s_commit = _verify_flow(w)
    o_pre, S_pre, o_blk, S_blk, o_acc, S_acc = _oracle_flow(w)
    gu.check_outputs(o, o_pre)
    gu.check_state(snap, S_pre)  # snapshot holds the state before the block
    gu.check_outputs(ov, o_blk)
    gu.check_state(s_blk, S_blk)
    if len(rows):
        gu.check_outputs(o_re, o_acc)
        # re-fed outputs equal the verify block's outputs for the accepted tokens
        assert gu.o_error(o_re, ov[rows]) < gu.TC_O_TOL
    gu.check_state(s_final, S_acc)
    # committing from the cached corrections reaches the same state as the re-feed
    gu.check_state(s_commit, S_acc)
    assert gu.state_error(s_commit, s_final) < gu.TC_S_TOL


@pytest.mark.parametrize("n_tok", [0, 1, 7, 16])
def test_verify_block_lengths(n_tok):
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    n = 3
    w = synth.make_workload("vb", [n_tok] * n, 16, 32, 128, 16, "bf16", seed=40 + n_tok, state_std=0.02)
    x = gu.dev_inputs(w)
    snap = torch.empty_like(x["state"])
    o = gu.out_like(x["v"], "f32")
    deltas = torch.zeros(x["v"].shape, dtype=torch.float32, device="cuda")
    gdr.gdr_verify_block(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], snap, o, n_tok, deltas=deltas)
    acc = np.array([0, n_tok // 2, n_tok], dtype=np.int32)
    committed = torch.full_like(x["state"], float("nan"))
    gdr.gdr_verify_commit(x["k"], x["g"], deltas, snap, committed, torch.from_numpy(acc).cuda(), n_tok)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    o_ref, S_ref = oracle.run_workload(w)
    np.testing.assert_array_equal(gu.to_np(snap), w.state0.astype(np.float64))
    if n_tok:
        gu.check_outputs(gu.to_np(o), o_ref)
    gu.check_state(gu.to_np(x["state"]), S_ref)
    # the accepted prefixes 0, n_tok / 2 and n_tok of the three sequences
    rows = np.concatenate([np.arange(s * n_tok, s * n_tok + acc[s]) for s in range(n)]).astype(np.int64)
    cu = np.zeros(n + 1, dtype=np.int64)
    cu[1:] = np.cumsum(acc)
    _, S_acc = oracle.gdr_sequential(cu, w.q[rows], w.k[rows], w.v[rows], w.g[rows], w.beta[rows], w.state0)
    c = gu.to_np(committed)
    np.testing.assert_array_equal(c[0], w.state0[0].astype(np.float64))  # a = 0: the snapshot itself
    gu.check_state(c, S_acc)


def test_verify_commit_rejects_out_of_range_count_on_the_device():
    """An accepted count above n_tok is reported through the device error word and
    leaves that sequence's state as it was; the other sequences commit normally."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    n_tok = 4
    w = synth.make_workload("vbad", [n_tok] * 2, 16, 32, 128, 16, "bf16", seed=77, state_std=0.02)
    x = gu.dev_inputs(w)
    snap = torch.empty_like(x["state"])
    o = gu.out_like(x["v"], "f32")
    deltas = torch.zeros(x["v"].shape, dtype=torch.float32, device="cuda")
    gdr.gdr_verify_block(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], snap, o, n_tok, deltas=deltas)
    target = torch.full_like(x["state"], 7.0)
    gdr.gdr_verify_commit(x["k"], x["g"], deltas, snap, target, torch.tensor([2, n_tok + 1], dtype=torch.int32,
                                                                             device="cuda"), n_tok)
    assert gdr.gdr_device_error() == gdr.GDR_ERR_INVALID_ARG
    assert bool(torch.all(target[1] == 7.0))
    assert gdr.gdr_device_error() == 0  # read and cleared


def test_snapshot_restore_roundtrip():
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    s = torch.randn(5, 32, 128, 128, device="cuda")
    snap = torch.empty_like(s)
    gdr.gdr_state_snapshot(s, snap)
    s2 = torch.zeros_like(s)
    gdr.gdr_state_restore(snap, s2)
    torch.cuda.synchronize()
    assert torch.equal(snap, s) and torch.equal(s2, s)


@pytest.mark.parametrize("d,io,out,n_tok,heads", [
    (128, "bf16", "f32", 16, (16, 32)),
    (128, "bf16", "bf16", 11, (16, 32)),
    (64, "bf16", "f32", 16, (2, 4)),
    (32, "bf16", "f32", 9, (4, 4)),
    (32, "f32", "f32", 16, (2, 4)),
    (128, "f32", "f32", 3, (1, 4)),
])
def test_verify_block_shapes(d, io, out, n_tok, heads):
    """Every head size and input type of the verify block (bf16 inputs on the
    tensor-core verify kernel, fp32 inputs on the CUDA-core chunk kernel) from a
    random state, against the oracle: outputs, the state after the block, the
    snapshot (bit-exact) and the corrections (through a full commit)."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    n = 2
    w = synth.make_workload("vs", [n_tok] * n, heads[0], heads[1], d, 16, io, seed=90 + d + n_tok, state_std=0.05)
    x = gu.dev_inputs(w)
    snap = torch.empty_like(x["state"])
    o = gu.out_like(x["v"], out)
    deltas = torch.full(x["v"].shape, float("nan"), dtype=torch.float32, device="cuda")
    gdr.gdr_verify_block(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], snap, o, n_tok, deltas=deltas)
    committed = torch.full_like(x["state"], float("nan"))
    gdr.gdr_verify_commit(x["k"], x["g"], deltas, snap, committed,
                          torch.full((n,), n_tok, dtype=torch.int32, device="cuda"), n_tok)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    o_ref, S_ref = oracle.run_workload(w)
    np.testing.assert_array_equal(gu.to_np(snap), w.state0.astype(np.float64))
    # both kernels keep fp32-level precision (the tensor-core one splits the state
    # into bf16 hi and lo halves): far inside the tolerances of the tensor-core prefill
    gu.check_outputs(gu.to_np(o), o_ref, out, tol=1e-3 if out == "f32" else gu.O_TOL)
    gu.check_state(gu.to_np(x["state"]), S_ref, tol=1e-4)
    gu.check_state(gu.to_np(committed), S_ref, tol=1e-4)
