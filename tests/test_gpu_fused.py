"""The steps on either side of the rule, fused into the kernels (GDR_FLAG_QK_L2NORM,
GDR_FLAG_BETA_LOGITS, the gated RMSNorm), against the oracle run with the same
steps around the plain recurrence."""

import numpy as np
import pytest

import oracle
from gated_deltanet_scan_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

RAW = (0.05, 20.0)  # per-row factors of the raw q and k rows


def check_gated(y, y_ref, z, wt, out_dtype):
    """The gated norm's output against the oracle's, in the units of the normalised
    output o / rms(o): the gate and the weight, w silu(z) (exact fp32 products in
    the kernel), scale each element by up to ~10x the row's typical size, and the
    rule's own error is measured against the output's RMS before that scaling.
    Elements where |w silu(z)| < 1e-3 carry no information and are skipped."""
    c = wt * (z / (1.0 + np.exp(-z)))
    keep = np.abs(c) >= 1e-3
    gu.check_outputs(np.where(keep, y / np.where(keep, c, 1.0), 0.0),
                     np.where(keep, y_ref / np.where(keep, c, 1.0), 0.0), out_dtype)


def fused_ref(w, z=None, wt=None):
    return oracle.gdr_fused(w.cu_seqlens, w.q, w.k, w.v, w.g, w.beta, w.state0, qk_l2norm=True,
                            beta_logits=True, z=z, norm_weight=wt)


def run(w, fn="chunked", chunk=None, P=None):
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    x = gu.dev_inputs(w)
    o = gu.out_like(x["v"], "f32")
    kw = dict(qk_l2norm=True, beta_logits=True)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"])
    if fn == "chunked":
        gdr.gdr_prefill_chunked(*args, chunk=chunk or w.chunk, **kw)
    elif fn == "static":
        gdr.gdr_prefill_chunked_static(*args, **kw)
    else:
        gdr.gdr_prefill_segmented(*args, P, **kw)
    torch.cuda.synchronize()
    assert gdr.gdr_device_error() == 0
    return gu.to_np(o), gu.to_np(x["state"])


@pytest.mark.parametrize("lens,chunk", [([1024], 64), ([300, 77, 0, 129], 64), ([200, 33], 16)])
def test_prefill_with_raw_qk_and_beta_logits(lens, chunk):
    """Tensor-core prefill (chunk 64: row scales from the factor kernel's slot) and
    the CUDA-core chunk kernel (chunk 16: rows normalised in shared memory)."""
    w = synth.make_workload("fused_pre", lens, 16, 32, 128, chunk, "bf16", seed=91 + len(lens), state_std=0.02,
                            qk_raw_scale=RAW, beta_logits=True)
    o, S = run(w)
    o_ref, S_ref = fused_ref(w)
    gu.check_outputs(o, o_ref)
    gu.check_state(S, S_ref)


def test_long_prefill_split_with_fused_norm():
    """A prefill long enough to split into four launches, strong decay."""
    w = synth.make_workload("fused_long", [6000], 16, 32, 128, 64, "bf16", seed=93, state_std=0.02, g_fixed=-6.72,
                            qk_raw_scale=RAW, beta_logits=True)
    o, S = run(w)
    o_ref, S_ref = fused_ref(w)
    gu.check_outputs(o, o_ref)
    gu.check_state(S, S_ref)


def test_segmented_and_static_entries_with_fused_norm():
    w = synth.make_workload("fused_seg", [2000], 2, 4, 128, 64, "bf16", seed=94, state_std=0.02,
                            g_range=(-0.05, -0.001), qk_raw_scale=RAW, beta_logits=True)
    o_ref, S_ref = fused_ref(w)
    for fn, P in (("segmented", 3), ("static", None)):
        o, S = run(w, fn=fn, P=P)
        gu.check_outputs(o, o_ref)
        gu.check_state(S, S_ref)


@pytest.mark.parametrize("d", [32, 128])
def test_decode_verify_commit_with_fused_norm(d):
    """Decode step, 16-token verify block and the commit of an accepted prefix,
    all with raw q/k and beta logits."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    hq, hv = (2, 4) if d == 32 else (16, 32)
    dec = synth.make_workload("fused_dec", [1] * 8, hq, hv, d, 64, "bf16", seed=95, state_std=0.02,
                              qk_raw_scale=RAW, beta_logits=True)
    x = gu.dev_inputs(dec)
    o = gu.out_like(x["v"], "f32")
    gdr.gdr_decode_step(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, qk_l2norm=True, beta_logits=True)
    torch.cuda.synchronize()
    o_ref, S_ref = fused_ref(dec)
    gu.check_outputs(gu.to_np(o), o_ref)
    gu.check_state(gu.to_np(x["state"]), S_ref)
    # verify block of 16 from the decoded states, then commit 5 / 11 / 0 / 16 ... tokens
    vb = synth.make_workload("fused_vb", [16] * 8, hq, hv, d, 16, "bf16", seed=96, qk_raw_scale=RAW, beta_logits=True)
    y = gu.dev_inputs(vb)
    snap = torch.empty_like(x["state"])
    ov = gu.out_like(y["v"], "f32")
    deltas = torch.empty(y["v"].shape, dtype=torch.float32, device="cuda")
    gdr.gdr_verify_block(y["q"], y["k"], y["v"], y["g"], y["beta"], x["state"], snap, ov, 16, deltas=deltas,
                         qk_l2norm=True, beta_logits=True)
    torch.cuda.synchronize()
    ov_ref, S16_ref = oracle.gdr_fused(vb.cu_seqlens, vb.q, vb.k, vb.v, vb.g, vb.beta, S_ref, qk_l2norm=True,
                                       beta_logits=True)
    gu.check_outputs(gu.to_np(ov), ov_ref)
    gu.check_state(gu.to_np(x["state"]), S16_ref)
    acc = np.array([5, 11, 0, 16, 1, 7, 15, 3], dtype=np.int32)
    gdr.gdr_verify_commit(y["k"], y["g"], deltas, snap, x["state"], torch.from_numpy(acc).cuda(), 16,
                          qk_l2norm=True)
    torch.cuda.synchronize()
    rows = np.concatenate([np.arange(s * 16, s * 16 + acc[s]) for s in range(8)])
    cu = np.concatenate([[0], np.cumsum(acc)])
    _, Sa_ref = oracle.gdr_fused(cu, vb.q[rows], vb.k[rows], vb.v[rows], vb.g[rows], vb.beta[rows], S_ref,
                                 qk_l2norm=True, beta_logits=True)
    gu.check_state(gu.to_np(x["state"]), Sa_ref)
    assert gdr.gdr_device_error() == 0


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_gated_rmsnorm_standalone_and_fused_in_decode(out_dtype):
    """y = w o / sqrt(mean(o^2) + 1e-6) silu(z): one pass over a prefill's outputs,
    and fused into the decode step (whose block holds whole output rows)."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    w = synth.make_workload("gnorm", [500, 64], 16, 32, 128, 64, "bf16", seed=97, state_std=0.02,
                            qk_raw_scale=RAW, beta_logits=True)
    zst = synth.make_workload("gnorm_z", [564], 16, 32, 128, 64, "bf16", seed=98)
    z = zst.v  # bf16 values shaped like v
    wt = (0.5 + synth.Stream(98, "norm_w").uniform(128)).astype(np.float32)
    x = gu.dev_inputs(w)
    zdev = gu.dev_inputs(zst)["v"]
    wdev = torch.from_numpy(wt).cuda()
    o = gu.out_like(x["v"], out_dtype)
    gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state"], o, x["cu_seqlens"],
                            qk_l2norm=True, beta_logits=True)
    yv = torch.empty_like(o)
    gdr.gdr_gated_rmsnorm(o, zdev, wdev, yv)
    torch.cuda.synchronize()
    # the norm itself, against the oracle's on the very outputs the kernel normalised
    y_of_o = oracle.gated_rmsnorm(gu.to_np(o), z, wt)
    got = gu.to_np(yv)
    bound = 1e-5 * np.abs(y_of_o) + 1e-6 * np.sqrt(np.mean(y_of_o ** 2))
    if out_dtype == "bf16":
        bound = bound + 2.0 ** -8 * np.abs(y_of_o)
    assert np.all(np.abs(got - y_of_o) <= bound)
    # and the whole path against the oracle
    y_ref, _ = fused_ref(w, z=z, wt=wt)
    check_gated(got, y_ref, z, wt, out_dtype)
    # decode with the norm fused
    dec = synth.make_workload("gnorm_dec", [1] * 16, 16, 32, 128, 64, "bf16", seed=99, state_std=0.02,
                              qk_raw_scale=RAW, beta_logits=True)
    zd = synth.make_workload("gnorm_dz", [16], 16, 32, 128, 64, "bf16", seed=100).v
    d = gu.dev_inputs(dec)
    zdd = torch.from_numpy(synth.bf16_bits(zd).view(np.int16).copy()).view(torch.bfloat16).cuda()
    yd = gu.out_like(d["v"], out_dtype)
    gdr.gdr_decode_step_gated(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"], zdd, wdev, yd,
                              qk_l2norm=True, beta_logits=True)
    torch.cuda.synchronize()
    yd_ref, Sd_ref = fused_ref(dec, z=zd, wt=wt)
    check_gated(gu.to_np(yd), yd_ref, zd, wt, out_dtype)
    gu.check_state(gu.to_np(d["state"]), Sd_ref)
    assert gdr.gdr_device_error() == 0


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("o_dtype,z_dtype", [("f32", "bf16"), ("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32")])
def test_gated_rmsnorm_shapes_and_dtypes(d, o_dtype, z_dtype):
    """The one-pass norm for every head size (a lane holds d / 32 values: vector and
    scalar accesses) and every dtype pairing, over row counts that leave the last
    step of the two-rows-per-warp loop with one row or none (1, 7, 1001, and more
    rows than the grid has warps), against the oracle's norm of the same values."""
    import gated_deltanet_scan_gb300 as gdr
    torch = gu.require_gpu()
    st = synth.Stream(4242 + d, f"norm_{o_dtype}_{z_dtype}")
    wt = (0.5 + st.uniform(d)).astype(np.float32)
    wdev = torch.from_numpy(wt).cuda()
    for rows in (1, 7, 1001, 50001):
        o = st.normal(rows * d).reshape(rows, d).astype(np.float32) * np.float32(0.3)
        z = st.normal(rows * d).reshape(rows, d).astype(np.float32) * np.float32(2.0)

        def dev(a, dt):
            if dt == "bf16":
                return torch.from_numpy(synth.bf16_bits(a).view(np.int16).copy()).view(torch.bfloat16).cuda()
            return torch.from_numpy(np.ascontiguousarray(a)).cuda()

        odev, zdev = dev(o, o_dtype), dev(z, z_dtype)
        y = torch.empty_like(odev)
        gdr.gdr_gated_rmsnorm(odev, zdev, wdev, y)
        torch.cuda.synchronize()
        ref = oracle.gated_rmsnorm(gu.to_np(odev), gu.to_np(zdev), wt)  # the values the kernel read
        got = gu.to_np(y)
        bound = 1e-5 * np.abs(ref) + 1e-6 * np.sqrt(np.mean(ref ** 2))
        if o_dtype == "bf16":
            bound = bound + 2.0 ** -8 * np.abs(ref)
        assert np.all(np.abs(got - ref) <= bound), (d, o_dtype, z_dtype, rows)
    assert gdr.gdr_device_error() == 0
