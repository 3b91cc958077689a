"""A seeded random sweep over the entry points, shapes, dtypes and options, each
case checked against the oracle on the same inputs: packed prefills (every entry:
with a workspace, without an allocation, two-level), verify block + commit,
decode, and the prefill + decode launch.  The cases are drawn once from a fixed
seed, so the sweep is the same on every run; each stays small enough for the
oracle to finish in about a second."""

import numpy as np
import pytest

import oracle
from gated_deltanet_scan_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

HEADS = [(16, 32), (2, 4), (4, 4), (1, 4), (8, 16)]


def _cases(n=16, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        h_qk, h_v = HEADS[rng.integers(len(HEADS))]
        n_seqs = int(rng.integers(1, 5))
        lens = [int(x) for x in rng.integers(0, 700, n_seqs)]
        if sum(lens) == 0:
            lens[0] = 65
        out.append(dict(
            idx=i, h_qk=h_qk, h_v=h_v, lens=lens,
            d=int(rng.choice([128, 128, 64, 32])),
            io=str(rng.choice(["bf16", "bf16", "f32"])),
            out=str(rng.choice(["f32", "bf16"])),
            fused=bool(rng.integers(2)),
            entry=str(rng.choice(["chunked", "static", "segmented"])),
            g_fixed=(None if rng.integers(3) else -6.72),
        ))
    return out


CASES = _cases()


def _workload(c, seed):
    kw = dict(qk_raw_scale=(0.3, 3.0), beta_logits=True) if c["fused"] else {}
    if c["g_fixed"] is not None:
        kw["g_fixed"] = c["g_fixed"]
    return synth.make_workload(f"sweep{c['idx']}", c["lens"], c["h_qk"], c["h_v"], c["d"], 64, c["io"],
                               seed=seed, state_std=0.02, **kw)


def _oracle(w, fused):
    if fused:
        return oracle.gdr_fused(w.cu_seqlens, w.q, w.k, w.v, w.g, w.beta, w.state0, qk_l2norm=True,
                                beta_logits=True)
    return oracle.run_workload(w)


def _tensor_core(c):
    return c["d"] == 128 and c["io"] == "bf16"


@pytest.mark.parametrize("c", CASES, ids=[f"case{c['idx']}" for c in CASES])
def test_prefill_sweep(c):
    """One prefill per case through the drawn entry point (the static and
    two-level entries exist for the tensor-core shapes; other shapes use the
    workspace entry), against the oracle."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    w = _workload(c, 300 + c["idx"])
    x = gu.dev_inputs(w)
    o = gu.out_like(x["v"], c["out"])
    flags = dict(qk_l2norm=c["fused"], beta_logits=c["fused"])
    T = int(w.cu_seqlens[-1])
    entry = c["entry"] if _tensor_core(c) else "chunked"
    if entry == "chunked":
        gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"],
                                t_total=T, **flags)
    elif entry == "static":
        gdr.gdr_prefill_chunked_static(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"],
                                       t_total=T, **flags)
    else:
        gdr.gdr_prefill_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"],
                                  3, t_total=T, **flags)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    o_ref, s_ref = _oracle(w, c["fused"])
    gu.check_outputs(gu.to_np(o), o_ref, c["out"])
    gu.check_state(gu.to_np(x["state"]), s_ref)


@pytest.mark.parametrize("c", CASES[:8], ids=[f"case{c['idx']}" for c in CASES[:8]])
def test_verify_commit_decode_sweep(c):
    """A verify block of n_tok tokens (drawn) and the commit of a random prefix per
    sequence, then one decode step of the same sequences from the committed
    states, each against the oracle."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    rng = np.random.default_rng(500 + c["idx"])
    n = len(c["lens"])
    n_tok = int(rng.integers(1, 17))
    kw = dict(qk_raw_scale=(0.3, 3.0), beta_logits=True) if c["fused"] else {}
    vb = synth.make_workload(f"sweepv{c['idx']}", [n_tok] * n, c["h_qk"], c["h_v"], c["d"], 16, c["io"],
                             seed=600 + c["idx"], state_std=0.05, **kw)
    flags = dict(qk_l2norm=c["fused"], beta_logits=c["fused"])
    x = gu.dev_inputs(vb)
    snap = torch.empty_like(x["state"])
    o = gu.out_like(x["v"], c["out"])
    deltas = torch.zeros(x["v"].shape, dtype=torch.float32, device="cuda")
    gdr.gdr_verify_block(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], snap, o, n_tok, deltas=deltas,
                         **flags)
    acc = rng.integers(0, n_tok + 1, n).astype(np.int32)
    committed = torch.empty_like(x["state"])
    gdr.gdr_verify_commit(x["k"], x["g"], deltas, snap, committed, torch.from_numpy(acc).cuda(), n_tok,
                          qk_l2norm=c["fused"])
    # one decode token per sequence from the committed state
    dw = synth.make_workload(f"sweepd{c['idx']}", [1] * n, c["h_qk"], c["h_v"], c["d"], 16, c["io"],
                             seed=700 + c["idx"], state_std=0.0, **kw)
    dx = gu.dev_inputs(dw)
    od = gu.out_like(dx["v"], c["out"])
    dstate = committed.clone()
    gdr.gdr_decode_step(dx["q"], dx["k"], dx["v"], dx["g"], dx["beta"], dstate, od, **flags)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    o_ref, s_ref = _oracle(vb, c["fused"])
    gu.check_outputs(gu.to_np(o), o_ref, c["out"])
    gu.check_state(gu.to_np(x["state"]), s_ref)
    rows = np.concatenate([np.arange(s * n_tok, s * n_tok + acc[s]) for s in range(n)]).astype(np.int64)
    cu = np.zeros(n + 1, dtype=np.int64)
    cu[1:] = np.cumsum(acc)
    sub = dict(q=vb.q[rows], k=vb.k[rows], v=vb.v[rows], g=vb.g[rows], beta=vb.beta[rows])
    if c["fused"]:
        _, s_acc = oracle.gdr_fused(cu, sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], vb.state0,
                                    qk_l2norm=True, beta_logits=True)
    else:
        _, s_acc = oracle.gdr_sequential(cu, sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], vb.state0)
    gu.check_state(gu.to_np(committed), s_acc)
    if c["fused"]:
        od_ref, ds_ref = oracle.gdr_fused(dw.cu_seqlens, dw.q, dw.k, dw.v, dw.g, dw.beta, s_acc, qk_l2norm=True,
                                          beta_logits=True)
    else:
        od_ref, ds_ref = oracle.gdr_sequential(dw.cu_seqlens, dw.q, dw.k, dw.v, dw.g, dw.beta, s_acc)
    gu.check_outputs(gu.to_np(od), od_ref, c["out"])
    gu.check_state(gu.to_np(dstate), ds_ref)


@pytest.mark.parametrize("c", [c for c in CASES if _tensor_core(c)][:4],
                         ids=[f"case{c['idx']}" for c in CASES if _tensor_core(c)][:4])
def test_prefill_with_decode_sweep(c):
    """The prefill + decode launch on the drawn prefill and a decode batch of the same
    heads: both parts against the oracle."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    w = _workload(c, 800 + c["idx"])
    kw = dict(qk_raw_scale=(0.3, 3.0), beta_logits=True) if c["fused"] else {}
    dw = synth.make_workload(f"sweepm{c['idx']}", [1] * 3, c["h_qk"], c["h_v"], c["d"], 64, c["io"],
                             seed=900 + c["idx"], state_std=0.02, **kw)
    x, dx = gu.dev_inputs(w), gu.dev_inputs(dw)
    o, od = gu.out_like(x["v"], c["out"]), gu.out_like(dx["v"], c["out"])
    gdr.gdr_prefill_with_decode(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"],
                                dx["q"], dx["k"], dx["v"], dx["g"], dx["beta"], dx["state"], od,
                                t_total=int(w.cu_seqlens[-1]), qk_l2norm=c["fused"], beta_logits=c["fused"])
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    o_ref, s_ref = _oracle(w, c["fused"])
    gu.check_outputs(gu.to_np(o), o_ref, c["out"])
    gu.check_state(gu.to_np(x["state"]), s_ref)
    od_ref, ds_ref = _oracle(dw, c["fused"])
    gu.check_outputs(gu.to_np(od), od_ref, c["out"])
    gu.check_state(gu.to_np(dx["state"]), ds_ref)


@pytest.mark.parametrize("entry", ["chunked", "segmented"])
def test_many_short_sequences(entry):
    """64 packed sequences of 0..200 tokens (Qwen3.5-9B heads): the factor kernel's
    search over cu_seqlens, one spare chunk position per sequence, and the
    two-level prefill's segments over packed sequences."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    rng = np.random.default_rng(4242)
    lens = [int(x) for x in rng.integers(0, 201, 64)]
    w = synth.make_workload("many_short", lens, 16, 32, 128, 64, "bf16", seed=4243, state_std=0.02)
    x = gu.dev_inputs(w)
    o = gu.out_like(x["v"], "f32")
    if entry == "chunked":
        gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"])
    else:
        gdr.gdr_prefill_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"], 2)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    o_ref, s_ref = oracle.run_workload(w)
    gu.check_outputs(gu.to_np(o), o_ref)
    gu.check_state(gu.to_np(x["state"]), s_ref)


@pytest.mark.parametrize("n,ties", [(2, True), (32, False), (32, True), (33, False)])
def test_packed_sequence_order(n, ties):
    """The chunk scan takes 2..32 packed sequences longest first (ranked by every warp
    with shuffles; equal lengths by index) and more in order: 2 and 32 sequences with
    and without equal lengths, 33 sequences (natural order), against the oracle."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    rng = np.random.default_rng(900 + n + (1000 if ties else 0))
    lens = [int(x) for x in rng.integers(0, 160, n)]
    if ties:
        lens = [lens[0]] * n if n == 2 else [int(x) for x in rng.choice([0, 64, 65, 130], n)]
    lens[-1] = max(lens[-1], 1)
    w = synth.make_workload(f"order{n}", lens, 4, 8, 128, 64, "bf16", seed=901 + n, state_std=0.02)
    x = gu.dev_inputs(w)
    o = gu.out_like(x["v"], "f32")
    gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"])
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    o_ref, s_ref = oracle.run_workload(w)
    gu.check_outputs(gu.to_np(o), o_ref)
    gu.check_state(gu.to_np(x["state"]), s_ref)
