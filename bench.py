"""Benchmark of the gated delta rule hot path on GB300.

One step = one pass of the whole path over one batch of synthetic Qwen3.5-9B
linear-attention inputs (16 QK heads, 32 V heads, d = 128, bf16 q/k/v, fp32
gates and state, fp32 output):

  1. gdr_prefill_chunked   B = 1, T = 16384, from a N(0, 0.02) state (two launches:
                           the per-chunk factors of all chunks, then the chunk scan)
  2. gdr_verify_block      16 draft tokens on that sequence (snapshot taken, each
                           token's correction kept)
     gdr_verify_commit     the state after the accepted prefix (7 tokens), formed
                           from the snapshot and the kept corrections
  3. gdr_decode_step_overlapped
                           B = 64 independent sequences, one token each; it shares
                           nothing with steps 1-2, so it is queued right after the
                           prefill as a programmatic dependent launch and runs on
                           the SMs the prefill's last chunk-scan launch leaves free
                           (24 of 152)

tokens/s counts the 16384 prefill, 16 verify and 64 decode tokens of a step
(the committed prefix is not counted again).  Inputs are resident in
HBM before the timed region; per step they exceed L2 (q, k, v, o and the decode
state are > 600 MB), so no flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica of the step (the path has
no cross-GPU exchange); rank 0 prints one JSON line.  ``--impl reference``
times the fp64 CPU oracle (the only other implementation of this path) on a
bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "gated-delta-rule tokens/s (prefill T=16K, decode B=64) and % of roofline, 1 GB300"
H_QK, H_V, D = 16, 32, 128
T_PREFILL, B_DECODE, N_VERIFY, N_ACCEPT = 16384, 64, 16, 7
TOKENS_PER_STEP = T_PREFILL + N_VERIFY + B_DECODE

# algorithmic bytes: q, k (bf16, per QK head), v (bf16), o (fp32), g, beta (fp32)
PREFILL_BYTES_PER_TOKEN = H_QK * D * 2 * 2 + H_V * D * 2 + H_V * D * 4 + H_V * 4 * 2
# the same count with o in bf16 like v (24,832 B/token): the unit the survey's roofline uses
SURVEY_BYTES_PER_TOKEN = H_QK * D * 2 * 2 + H_V * D * 2 + H_V * D * 2 + H_V * 4 * 2
STATE_BYTES = H_V * D * D * 4
# algorithmic FLOPs per token and V head of the chunk form at C = 64 (triangles once)
PREFILL_FLOP_PER_TOKEN = 4.25e6
DECODE_BYTES_PER_SEQ = 2 * STATE_BYTES + H_QK * D * 2 * 2 + H_V * D * 2 + H_V * D * 4 + H_V * 8

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def max_over_ranks(values, device):
    """Each of `values` maximised over the ranks of the default process group
    (the job's time is the slowest rank's)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_tokens_per_s(world, ms_per_step):
    """Tokens/s of the whole job: every rank runs one replica step, so the job
    moves world x TOKENS_PER_STEP tokens per slowest-rank step."""
    return world * TOKENS_PER_STEP / (ms_per_step * 1e-3)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---------------------------------------------------------------------------------
# inputs


def host_inputs(seed_base=100):
    """The step's synthetic inputs on the host (bf16 bits for q/k/v)."""
    from gated_deltanet_scan_gb300 import synth

    pre = synth.make_workload("bench_prefill", [T_PREFILL], H_QK, H_V, D, 64, "bf16",
                              seed=seed_base, state_std=0.02)
    ver = synth.make_workload("bench_verify", [N_VERIFY], H_QK, H_V, D, 16, "bf16", seed=seed_base + 1)
    dec = synth.make_workload("bench_decode", [1] * B_DECODE, H_QK, H_V, D, 64, "bf16",
                              seed=seed_base + 2, state_std=0.02)
    return pre, ver, dec


def _bf(torch, bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)


def _pinned(torch, w):
    def io(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).pin_memory()

    return dict(q=io(w.q_bits), k=io(w.k_bits), v=io(w.v_bits),
                g=torch.from_numpy(np.ascontiguousarray(w.g)).pin_memory(),
                beta=torch.from_numpy(np.ascontiguousarray(w.beta)).pin_memory())


# ---------------------------------------------------------------------------------
# clocks


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------------
# our arm


PREFILL_SOURCES = ("gdr_factor.cu", "gdr_prefill_tc.cu", "gdr_factor_layout.h", "tc_ptx.cuh", "gdr_common.cuh",
                   "gdr_internal.h")


def prefill_source_digest():
    h = hashlib.sha256()
    for name in PREFILL_SOURCES:
        with open(os.path.join(ROOT, "gated_deltanet_scan_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record():
    """DRAM bytes of one T = 16384 prefill (both launches) from the committed ncu
    summary, if the kernel sources are unchanged since it was measured (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        digest = prefill_source_digest()
    except (OSError, ValueError):
        return None
    r = rec.get("prefill_T16384")
    if not r or r.get("source_sha256_16") != digest:
        return None
    return r.get("dram_bytes_per_launch")


def run_ours(args):
    import torch
    import gated_deltanet_scan_gb300 as gdr

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)

    pre, ver, dec = host_inputs()
    hp, hv, hd = _pinned(torch, pre), _pinned(torch, ver), _pinned(torch, dec)

    def device_set():
        # one set of device inputs and outputs of a step (the end-to-end run keeps two)
        return dict(p={k: t.to(dev) for k, t in hp.items()}, v={k: t.to(dev) for k, t in hv.items()},
                    d={k: t.to(dev) for k, t in hd.items()},
                    o_pre=torch.empty((T_PREFILL, H_V, D), dtype=torch.float32, device=dev),
                    o_ver=torch.empty((N_VERIFY, H_V, D), dtype=torch.float32, device=dev),
                    o_dec=torch.empty((B_DECODE, H_V, D), dtype=torch.float32, device=dev))

    main_set = device_set()
    dp, dv, dd = main_set["p"], main_set["v"], main_set["d"]
    state0 = torch.from_numpy(np.ascontiguousarray(pre.state0)).to(dev)
    state = state0.clone()
    snap = torch.empty_like(state)
    dstate = torch.from_numpy(np.ascontiguousarray(dec.state0)).to(dev)
    o_pre, o_ver, o_dec = main_set["o_pre"], main_set["o_ver"], main_set["o_dec"]
    deltas = torch.empty((N_VERIFY, H_V, D), dtype=torch.float32, device=dev)
    cu_pre = torch.tensor([0, T_PREFILL], dtype=torch.int32, device=dev)
    accepted = torch.tensor([N_ACCEPT], dtype=torch.int32, device=dev)
    # the prefill's factor workspace, allocated once
    ws_bytes = gdr.gdr_prefill_workspace_bytes(dp["q"], dp["v"], o_pre, 1, T_PREFILL)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    only = args.only

    def step(timers=None, bufs=None):
        dp, dv, dd = (main_set if bufs is None else bufs)["p"], (main_set if bufs is None else bufs)["v"], \
            (main_set if bufs is None else bufs)["d"]
        o_pre, o_ver, o_dec = [(main_set if bufs is None else bufs)[n] for n in ("o_pre", "o_ver", "o_dec")]
        if timers is not None:
            timers[0].record(stream)
        if only == "all" and args.decode_in_scan:
            # one launch carries the prefill's last chunk scan and the decode step
            gdr.gdr_prefill_with_decode(dp["q"], dp["k"], dp["v"], dp["g"], dp["beta"], state, o_pre, cu_pre,
                                        dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dstate, o_dec,
                                        workspace=ws, stream=stream)
        else:
            if only in ("all", "prefill"):
                gdr.gdr_prefill_chunked(dp["q"], dp["k"], dp["v"], dp["g"], dp["beta"], state, o_pre, cu_pre,
                                        chunk=64, workspace=ws, stream=stream)
            if only == "all":
                # beside the prefill's last chunk-scan launch (no event between them:
                # a stream operation there would end the overlap)
                gdr.gdr_decode_step_overlapped(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dstate, o_dec,
                                               stream=stream)
        if timers is not None:
            timers[1].record(stream)
        if only in ("all", "verify"):
            gdr.gdr_verify_block(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], state, snap, o_ver,
                                 N_VERIFY, deltas=deltas, stream=stream)
            gdr.gdr_verify_commit(dv["k"], dv["g"], deltas, snap, state, accepted, N_VERIFY, stream=stream)
        if timers is not None:
            timers[2].record(stream)
        if only == "decode":
            gdr.gdr_decode_step(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dstate, o_dec, stream=stream)
        if timers is not None:
            timers[3].record(stream)

    # prefill: factor + chunk-scan launches, twice when the library splits a long
    # prefill so that the later chunks' factors run beside the scan of the earlier
    # ones (its rule: chunks x V heads >= 8 x SMs, and at least 16 SMs left free
    # by the scan's 4 CTAs per V head); verify: the block and the commit
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    split = (T_PREFILL + 63) // 64 * H_V >= 8 * sms and sms - 4 * H_V >= 16
    pre_launches = 4 if split else 2
    launches_per_step = {"all": 3 + pre_launches, "prefill": pre_launches, "verify": 2, "decode": 1}[only]
    if only == "all" and args.decode_in_scan:
        launches_per_step -= 1  # the decode step rides the last chunk-scan launch

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        step()
    barrier()
    timers = [[ev() for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = ev(), ev()
    barrier()
    t_start.record(stream)
    for i in range(args.steps):
        step(timers[i])
    t_end.record(stream)
    barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    clk = clocks.stop()
    assert gdr.gdr_device_error(stream=stream) == 0, "a device-side wait timed out"

    prefill_ms = statistics.median(t[0].elapsed_time(t[1]) for t in timers)
    verify_ms = statistics.median(t[1].elapsed_time(t[2]) for t in timers)
    if only == "all":
        # inside the timed steps the decode ran beside the prefill (prefill_ms
        # spans both); its own speed is timed alone right after
        dts = []
        for _ in range(20):
            d0, d1 = ev(), ev()
            d0.record(stream)
            gdr.gdr_decode_step(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dstate, o_dec, stream=stream)
            d1.record(stream)
            dts.append((d0, d1))
        barrier()
        decode_ms = statistics.median(a.elapsed_time(b) for a, b in dts[5:])
    else:
        decode_ms = statistics.median(t[2].elapsed_time(t[3]) for t in timers)
    verify_alone_ms = None
    if only in ("all", "verify"):
        # verify block + commit alone, replayed from a CUDA graph of 20 pairs: the
        # pair's own time with graph launch gaps and its inputs in L2 (inside the
        # step they follow the prefill, cold, after eager launches)
        def pair():
            gdr.gdr_verify_block(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], state, snap, o_ver,
                                 N_VERIFY, deltas=deltas, stream=stream)
            gdr.gdr_verify_commit(dv["k"], dv["g"], deltas, snap, state, accepted, N_VERIFY, stream=stream)
        for _ in range(3):
            pair()
        barrier()
        vg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(vg, stream=stream):
            for _ in range(20):
                pair()
        barrier()
        vts = []
        for _ in range(5):
            v0, v1 = ev(), ev()
            v0.record(stream)
            vg.replay()
            v1.record(stream)
            vts.append((v0, v1))
        barrier()
        verify_alone_ms = statistics.median(a.elapsed_time(b) for a, b in vts) / 20
        del vg

    # The other configured workloads, timed alone after the steps (informational):
    # the Qwen3.5-9B layer prefill at T = 1024 and the packed prefill of 8
    # sequences with lengths ~ U{512..8192}.
    other = {}
    if only == "all" and not args.no_other_configs:
        from gated_deltanet_scan_gb300 import synth

        l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size

        def time_prefill(w, reps=10, segments=None, flags=None):
            """Median of `reps` prefills, each on the next of several copies of the
            inputs, outputs, states and workspace whose total is over twice the L2
            size (so no call finds its operands in L2 from the call before), launched
            eagerly and replayed as CUDA graphs (one per copy); a workload that alone
            exceeds L2 runs on one copy."""
            n = len(w.cu_seqlens) - 1
            tokens = int(w.cu_seqlens[-1])

            def one_set():
                x = dict(q=_bf(torch, w.q_bits).to(dev), k=_bf(torch, w.k_bits).to(dev),
                         v=_bf(torch, w.v_bits).to(dev), g=torch.from_numpy(np.ascontiguousarray(w.g)).to(dev),
                         beta=torch.from_numpy(np.ascontiguousarray(w.beta)).to(dev))
                x["st"] = torch.zeros((n, H_V, D, D), dtype=torch.float32, device=dev)
                x["cu"] = torch.from_numpy(w.cu_seqlens.astype(np.int32)).to(dev)
                x["o"] = torch.empty((tokens, H_V, D), dtype=torch.float32, device=dev)
                need = (gdr.gdr_prefill_workspace_bytes(x["q"], x["v"], x["o"], n, tokens) if segments is None else
                        gdr.gdr_prefill_segmented_workspace_bytes(x["q"], x["v"], x["o"], n, tokens, segments))
                x["ws"] = torch.empty(need, dtype=torch.uint8, device=dev)
                return x

            sets = [one_set()]
            set_bytes = sum(t.numel() * t.element_size() for t in sets[0].values())
            while len(sets) * set_bytes < 2 * l2_bytes:
                sets.append(one_set())

            def call(x):
                if segments is None:
                    gdr.gdr_prefill_chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["st"], x["o"], x["cu"],
                                            chunk=64, workspace=x["ws"], stream=stream, **(flags or {}))
                else:
                    gdr.gdr_prefill_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["st"], x["o"], x["cu"],
                                              segments, chunk=64, workspace=x["ws"], stream=stream)

            def timed(launch):
                ts = []
                for r in range(reps + 3):
                    a0, a1 = ev(), ev()
                    a0.record(stream)
                    launch(r % len(sets))
                    a1.record(stream)
                    ts.append((a0, a1))
                barrier()
                return statistics.median(a.elapsed_time(b) for a, b in ts[3:])

            ms = timed(lambda i: call(sets[i]))
            graphs = []
            for x in sets:
                call(x)  # loads the kernels and sets their attributes before capture
                barrier()
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=stream):
                    call(x)
                graphs.append(gr)
            ms_graph = timed(lambda i: graphs[i].replay())
            del graphs
            hv = w.h_v / H_V  # byte counts below are for 32 V heads and 16 QK heads
            alg = hv * (tokens * PREFILL_BYTES_PER_TOKEN + 2 * n * STATE_BYTES)
            alg_survey = hv * (tokens * SURVEY_BYTES_PER_TOKEN + 2 * n * STATE_BYTES)
            hbm = load_peaks()[0]["hbm_gbs"]
            gbs = alg / (ms * 1e-3) / 1e9
            return {"ms": ms, "ms_graph": ms_graph, "tokens": tokens, "tokens_per_s": tokens / (ms * 1e-3),
                    "tokens_per_s_graph": tokens / (ms_graph * 1e-3), "hbm_gbs": gbs, "frac_hbm": gbs / hbm,
                    "frac_hbm_survey_bytes": alg_survey / (ms * 1e-3) / 1e9 / hbm,
                    "buffer_sets": len(sets), "bytes_per_set": set_bytes,
                    "l2": (f"rotated over {len(sets)} copies of every buffer ({len(sets) * set_bytes / 1e6:.0f} MB, "
                           f"L2 {l2_bytes / 1e6:.0f} MB)") if len(sets) > 1 else "inputs larger than L2"}

        other["prefill_T1024"] = time_prefill(synth.prefill_9b(1024))
        other["packed_prefill_8_seqs"] = time_prefill(synth.varlen_verify())
        # few heads, one long sequence (e.g. a layer split 8 ways by heads: 2 QK, 4 V):
        # one chain per head, against the two-level scan with the library's segment count
        few = synth.make_workload("few_heads_T16384", [16384], 2, 4, D, 64, "bf16", seed=105, state_std=0.02)
        q_, v_, o_ = (torch.empty((1, nh, D), dtype=dt, device=dev)
                      for nh, dt in ((2, torch.bfloat16), (4, torch.bfloat16), (4, torch.float32)))
        P = gdr.gdr_prefill_segments_hint(q_, v_, o_, 1, 16384)
        plain = time_prefill(few)
        seg = time_prefill(few, segments=P)
        other["few_heads_T16384_hqk2_hv4"] = {"one_chain": plain, "segmented": dict(seg, segments=P),
                                              "speedup": plain["ms"] / seg["ms"]}
        del few, plain, seg

        # The steps on either side of the rule, on the same shapes with the options on:
        # raw q/k normalised inside the kernels and beta from logits (the T = 16384
        # prefill; the B = 64 decode step, also with the gated RMSNorm fused in), and
        # the one-pass gated RMSNorm over the prefill's output.
        fw = synth.make_workload("fused_T16384", [T_PREFILL], H_QK, H_V, D, 64, "bf16", seed=106, state_std=0.02,
                                 qk_raw_scale=(0.3, 3.0), beta_logits=True)
        fused = {"prefill_T16384_plain_alone": time_prefill(pre),
                 "prefill_T16384_qk_l2norm_beta_logits": time_prefill(fw, flags=dict(qk_l2norm=True, beta_logits=True))}
        del fw
        hbm_peak = load_peaks()[0]["hbm_gbs"]

        def time_calls(fn, reps=20):
            ts = []
            for _ in range(reps + 5):
                a0, a1 = ev(), ev()
                a0.record(stream)
                fn()
                a1.record(stream)
                ts.append((a0, a1))
            barrier()
            return statistics.median(a.elapsed_time(b) for a, b in ts[5:])

        def bw(nbytes, ms):
            gbs = nbytes / (ms * 1e-3) / 1e9
            return {"ms": ms, "bytes": nbytes, "hbm_gbs": gbs, "frac_hbm": gbs / hbm_peak}

        st2 = dstate.clone()
        w_norm = torch.ones(D, dtype=torch.float32, device=dev)
        ms = time_calls(lambda: gdr.gdr_decode_step(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], st2, o_dec,
                                                    qk_l2norm=True, beta_logits=True, stream=stream))
        fused["decode_B64_qk_l2norm_beta_logits"] = dict(bw(B_DECODE * DECODE_BYTES_PER_SEQ, ms),
                                                         plain_decode_ms=decode_ms)
        # z is the v rows (any bf16 values serve for the timing); y replaces o
        ms = time_calls(lambda: gdr.gdr_decode_step_gated(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], st2,
                                                          dd["v"], w_norm, o_dec, stream=stream))
        fused["decode_B64_gated_rmsnorm"] = dict(bw(B_DECODE * (DECODE_BYTES_PER_SEQ + H_V * D * 2), ms),
                                                 plain_decode_ms=decode_ms)
        del st2
        # over the prefill's fp32 output rows, z = the prefill's bf16 v rows, y fp32
        y_norm = torch.empty_like(o_pre)
        ms = time_calls(lambda: gdr.gdr_gated_rmsnorm(o_pre, dp["v"], w_norm, y_norm, stream=stream), reps=10)
        fused["gated_rmsnorm_T16384"] = dict(bw(T_PREFILL * H_V * D * (4 + 2 + 4), ms),
                                             rows=T_PREFILL * H_V, io="o fp32, z bf16, y fp32")
        del y_norm
        other["fused_steps"] = fused

    # End to end through the same public API: every step uploads its inputs from
    # pinned host memory and reads its outputs back.  Like a serving pipeline, the
    # uploads run on one copy stream and the read-backs on another, with two sets
    # of device buffers, so step i's kernels overlap step i+1's upload and step
    # i-1's read-back; the timed region spans every copy of every step.
    outs_host = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in (o_pre, o_ver, o_dec)]
    h2d = sum(t.numel() * t.element_size() for d in (hp, hv, hd) for t in d.values())
    d2h = sum(t.numel() * t.element_size() for t in outs_host)
    e2e_steps = max(3, min(args.steps, 20)) if only == "all" else 0

    e2e_ms = float("nan")
    if e2e_steps:
        sets = [main_set, device_set()]
        # copy streams per direction (each large copy is cut into NCOPY parts); more
        # than one measured slower on GB300: the copies share one link
        NCOPY = 1
        ups = [torch.cuda.Stream(dev) for _ in range(NCOPY)]
        downs = [torch.cuda.Stream(dev) for _ in range(NCOPY)]
        done = [torch.cuda.Event() for _ in sets]   # a set's kernels have finished
        for e in done:
            e.record(stream)
        read = [[torch.cuda.Event() for _ in downs] for _ in sets]  # its outputs have been read back
        for es in read:
            for e in es:
                e.record(stream)
        loaded = [[torch.cuda.Event() for _ in ups] for _ in sets]

        def parts(t):
            flat = t.view(-1)
            n = flat.numel()
            cut = [n * j // NCOPY for j in range(NCOPY + 1)]
            return [flat[cut[j]:cut[j + 1]] for j in range(NCOPY)]

        def e2e_step(i):
            b = i % 2
            bufs = sets[b]
            for j, u in enumerate(ups):
                u.wait_event(done[b])  # the set's previous step no longer reads its inputs
                with torch.cuda.stream(u):
                    for src, key in ((hp, "p"), (hv, "v"), (hd, "d")):
                        for k in src:
                            parts(bufs[key][k])[j].copy_(parts(src[k])[j], non_blocking=True)
                loaded[b][j].record(u)
                stream.wait_event(loaded[b][j])
                stream.wait_event(read[b][j])  # its previous outputs have been read back
            step(bufs=bufs)
            done[b].record(stream)
            for j, dn in enumerate(downs):
                dn.wait_event(done[b])
                with torch.cuda.stream(dn):
                    for n, h in zip(("o_pre", "o_ver", "o_dec"), outs_host):
                        parts(h)[j].copy_(parts(bufs[n])[j], non_blocking=True)
                read[b][j].record(dn)

        for i in range(2):
            e2e_step(i)
        barrier()
        e0, e1 = ev(), ev()
        e0.record(stream)
        for c in ups + downs:
            c.wait_event(e0)
        for i in range(e2e_steps):
            e2e_step(i)
        for c in ups + downs:
            stream.wait_stream(c)
        e1.record(stream)
        barrier()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps

    ms_step = elapsed_ms / args.steps
    if world > 1:
        ms_step, e2e_ms = max_over_ranks([ms_step, e2e_ms], dev)
    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    bf16 = peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"])
    pre_bytes = T_PREFILL * PREFILL_BYTES_PER_TOKEN + 2 * STATE_BYTES
    pre_gbs = pre_bytes / (prefill_ms * 1e-3) / 1e9
    # the same time against 24,832 B/token (o counted in bf16, like v)
    pre_bytes_survey = T_PREFILL * SURVEY_BYTES_PER_TOKEN + 2 * STATE_BYTES
    pre_gbs_survey = pre_bytes_survey / (prefill_ms * 1e-3) / 1e9
    pre_tflops = PREFILL_FLOP_PER_TOKEN * T_PREFILL / (prefill_ms * 1e-3) / 1e12
    dec_bytes = B_DECODE * DECODE_BYTES_PER_SEQ
    dec_gbs = dec_bytes / (decode_ms * 1e-3) / 1e9
    traffic = traffic_record() if T_PREFILL == 16384 else None  # counters are for T = 16384
    value = whole_job_tokens_per_s(world, ms_step)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "precision": "prefill tensor-core operands: bf16 hi/lo splits for the state products, fp16 for the "
                     "products with the chunk factors; fp32 accumulation, state and outputs; decode and "
                     "verify in fp32 on CUDA cores",
        "data": "synthetic (seeded SplitMix64; Qwen3.5-9B linear-attention shapes)",
        "config": {
            "workload": "gated delta rule, Qwen3.5-9B layer: prefill B=1 T=16384 + 16-token verify "
                        "with snapshot and commit of 7 accepted tokens + decode step B=64",
            "h_qk": H_QK, "h_v": H_V, "d_k": D, "d_v": D, "chunk": 64,
            "io": "q/k/v bf16, g/beta fp32, state fp32, o fp32",
            "tokens_per_step": TOKENS_PER_STEP,
            "l2": "inputs larger than L2 (no flush)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "overlap": "decode step queued after the prefill as a programmatic dependent launch (beside its last chunk-scan launch)",
        },
        "components": {
            "prefill_T16384": {"ms": prefill_ms, "tokens_per_s": T_PREFILL / (prefill_ms * 1e-3),
                               "hbm_gbs": pre_gbs, "frac_hbm": pre_gbs / hbm,
                               "frac_hbm_survey_bytes": pre_gbs_survey / hbm,
                               "alg_tflops": pre_tflops, "frac_bf16": pre_tflops / bf16},
            "verify16_commit7": {"ms": verify_ms, "ms_alone_graph": verify_alone_ms},
            "decode_B64": {"ms": decode_ms, "tokens_per_s": B_DECODE / (decode_ms * 1e-3),
                           "hbm_gbs": dec_gbs, "frac_hbm": dec_gbs / hbm},
        },
        "roofline": {
            "kernel": "prefill: the factor_kernel + prefill_tc_kernel launches of one gdr_prefill_chunked call "
                      "(timed span also covers the decode step running beside it)",
            "bound": "hbm",
            "achieved": pre_gbs,
            "peak": hbm,
            "unit": "GB/s",
            "frac": pre_gbs / hbm,
            "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
            "traffic": traffic,
            "algorithmic_bytes_per_launch": pre_bytes,
            "algorithmic_bytes_note": "33,024 B/token (o in fp32, as stored) + 2 x 2 MiB of state",
            "frac_survey_bytes": pre_gbs_survey / hbm,
            "survey_bytes_per_launch": pre_bytes_survey,
            "survey_bytes_note": "24,832 B/token (o counted in bf16) + 2 x 2 MiB of state",
        },
        "e2e": {"value": whole_job_tokens_per_s(world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "other_configs": other or None,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if only != "all":
        line["partial_step"] = only  # a profiling run of one component, not a bench line
        line["prefill_tokens"] = T_PREFILL
        line.pop("e2e")
        line.pop("other_configs")
        keep = {"prefill": "prefill_T16384", "verify": "verify16_commit7", "decode": "decode_B64"}[only]
        comp = line["components"][keep]
        if only == "prefill":  # named for the prefill length actually timed (--prefill-tokens)
            keep = f"prefill_T{T_PREFILL}"
        line["components"] = {keep: comp}
        if only != "prefill":
            line.pop("roofline")
    elif not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(pre, ver, dec)
    return line


def run_segmented_profile(args):
    """A profiling run (no bench line): the two-level prefill of one sequence of
    T = 16384 with 2 QK / 4 V heads (the `other_configs` few-head case), W
    warm-up and K timed calls on one buffer set, CUDA events around each."""
    import torch
    import gated_deltanet_scan_gb300 as gdr
    from gated_deltanet_scan_gb300 import synth

    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    w = synth.make_workload("few_heads_T16384", [16384], 2, 4, D, 64, "bf16", seed=105, state_std=0.02)
    x = dict(q=_bf(torch, w.q_bits).to(dev), k=_bf(torch, w.k_bits).to(dev), v=_bf(torch, w.v_bits).to(dev),
             g=torch.from_numpy(np.ascontiguousarray(w.g)).to(dev),
             beta=torch.from_numpy(np.ascontiguousarray(w.beta)).to(dev),
             cu=torch.from_numpy(w.cu_seqlens.astype(np.int32)).to(dev))
    st = torch.zeros((1, 4, D, D), dtype=torch.float32, device=dev)
    o = torch.empty((16384, 4, D), dtype=torch.float32, device=dev)
    P = gdr.gdr_prefill_segments_hint(x["q"], x["v"], o, 1, 16384)
    ws = torch.empty(gdr.gdr_prefill_segmented_workspace_bytes(x["q"], x["v"], o, 1, 16384, P), dtype=torch.uint8,
                     device=dev)

    def call():
        gdr.gdr_prefill_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], st, o, x["cu"], P, chunk=64,
                                  workspace=ws, stream=stream)

    for _ in range(args.warmup):
        call()
    ts = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize(dev)
    assert gdr.gdr_device_error(stream=stream) == 0, "a device-side wait timed out"
    ms = statistics.median(a.elapsed_time(b) for a, b in ts) if ts else float("nan")
    return {"partial_step": "segmented", "workload": "one sequence T=16384, 2 QK / 4 V heads, two-level prefill",
            "segments": P, "steps": args.steps, "warmup": args.warmup, "ms": ms}


# ---------------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)


def oracle_step_sample(pre, ver, dec, threads, prefill_tokens=None):
    """The oracle over one step's work on all 32 V heads: the prefill (its first
    ``prefill_tokens`` tokens when given, else all of them), the 16-token verify
    block, the accepted prefix and the B = 64 decode step.  Returns (seconds,
    tokens processed)."""
    import oracle

    T = pre.q.shape[0] if prefill_tokens is None else int(prefill_tokens)
    t0 = time.perf_counter()
    _, s_pre = oracle.gdr_sequential([0, T], pre.q[:T], pre.k[:T], pre.v[:T], pre.g[:T], pre.beta[:T],
                                     pre.state0, threads=threads)
    oracle.gdr_sequential(ver.cu_seqlens, ver.q, ver.k, ver.v, ver.g, ver.beta, s_pre, threads=threads)
    acc = slice(0, N_ACCEPT)
    oracle.gdr_sequential([0, N_ACCEPT], ver.q[acc], ver.k[acc], ver.v[acc], ver.g[acc], ver.beta[acc], s_pre,
                          threads=threads)
    oracle.gdr_sequential(dec.cu_seqlens, dec.q, dec.k, dec.v, dec.g, dec.beta, dec.state0, threads=threads)
    return time.perf_counter() - t0, T + N_VERIFY + B_DECODE


SINGLE_THREAD_PREFILL = 2048  # prefill tokens of the one-thread sample (a few seconds of work)


def single_thread_sample(pre, ver, dec):
    """The oracle on one host thread over a shortened step (the first 2048
    prefill tokens, then the verify block, the accepted prefix and the decode
    step; all 32 V heads)."""
    secs, tokens = oracle_step_sample(pre, ver, dec, 1, SINGLE_THREAD_PREFILL)
    return {"value": tokens / secs, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"1 thread: first {SINGLE_THREAD_PREFILL} prefill tokens + verify 16 + accepted prefix 7 + "
                      f"decode B=64, all 32 V heads ({tokens} tokens, {secs:.1f} s)"}


def cpu_baseline_sample(pre, ver, dec, min_seconds=10.0, max_seconds=30.0):
    """The oracle, as it stands, over whole steps (all 32 heads) on every host
    thread until about 10 s of CPU work has accumulated, and on one thread over
    a shortened step."""
    import oracle

    threads = oracle.default_threads()
    secs, n, tokens = 0.0, 0, 0
    while secs < min_seconds and (n == 0 or secs + secs / n <= max_seconds):
        s, tok = oracle_step_sample(pre, ver, dec, threads)
        secs += s
        tokens += tok
        n += 1
    return {"value": tokens / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} full step(s) (prefill T=16384 + verify 16 + accepted prefix 7 + decode B=64, all 32 V "
                      f"heads), {secs:.1f} s of fp64 CPU work on {threads} threads",
            "single_thread": single_thread_sample(pre, ver, dec)}


REF_BUDGET_S = 150.0  # the reference arm's whole run (warm-up + timed steps) stays near this


def run_reference(args):
    """The oracle timed as the reference arm: every step is the oracle over one
    step of the workload on all 32 V heads and every host thread; when whole
    steps would make the run much longer than REF_BUDGET_S, each step's prefill
    is cut to its first tokens (a bounded sample of the same workload: tokens/s
    counts only the tokens processed, nothing is extrapolated)."""
    import oracle

    rank, world, _ = dist_env()
    if rank != 0:
        return None
    pre, ver, dec = host_inputs()
    threads = oracle.default_threads()
    n_runs = args.warmup + args.steps
    first, _ = oracle_step_sample(pre, ver, dec, threads)  # the first warm-up step, whole
    prefill_tokens = None
    if first * (n_runs - 1) > REF_BUDGET_S:
        frac = REF_BUDGET_S / (first * (n_runs - 1))
        prefill_tokens = max(256, int(T_PREFILL * frac) // 64 * 64)
    times, tokens = [], 0
    for i in range(1, n_runs):
        secs, tok = oracle_step_sample(pre, ver, dec, threads, prefill_tokens)
        if i >= args.warmup:
            times.append(secs)
            tokens += tok
    if not times:  # --steps 0: nothing timed
        times, tokens = [first], TOKENS_PER_STEP
    value = tokens / sum(times)
    ms = 1e3 * statistics.mean(times)
    what = (f"whole steps (prefill T=16384 + verify 16 + accepted prefix 7 + decode B=64)" if prefill_tokens is None
            else f"steps with the prefill cut to its first {prefill_tokens} of {T_PREFILL} tokens (+ verify 16 + "
                 f"accepted prefix 7 + decode B=64), to keep the run within ~{REF_BUDGET_S:.0f} s")
    sample = f"each step: the fp64 oracle over {what}, all 32 V heads, {threads} threads"
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same inputs as the GPU arm)",
        "config": {"workload": "gated delta rule, Qwen3.5-9B layer: prefill B=1 T=16384 + 16-token verify "
                               "with snapshot and commit of 7 accepted tokens + decode step B=64",
                   "h_qk": H_QK, "h_v": H_V, "d_k": D, "d_v": D},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample,
                         "single_thread": single_thread_sample(pre, ver, dec)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-in-scan", action="store_true",
                    help="run the decode step inside the prefill's last chunk-scan launch (gdr_prefill_with_decode) "
                         "instead of as a programmatic dependent launch beside it")
    ap.add_argument("--only", choices=["all", "prefill", "verify", "decode", "segmented"], default="all",
                    help="run one component of the step (for profiling; 'segmented': the two-level prefill of "
                         "one 16K-token sequence of 2 QK / 4 V heads); the default runs the full step")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the informational timing of the T=1024 and packed prefill workloads")
    ap.add_argument("--prefill-tokens", type=int, default=T_PREFILL,
                    help="prefill length of a profiling run (with --only prefill); not a bench line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.prefill_tokens != T_PREFILL:
        if args.only != "prefill" or args.prefill_tokens <= 0:
            ap.error("--prefill-tokens is for profiling runs with --only prefill")
        globals()["T_PREFILL"] = args.prefill_tokens
    if args.impl == "ours" and args.only == "segmented":
        line = run_segmented_profile(args)
    else:
        line = run_ours(args) if args.impl == "ours" else run_reference(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
