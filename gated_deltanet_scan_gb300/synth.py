"""Seeded synthetic inputs for the gated delta rule.

This module only draws numbers: it holds none of the recurrence's arithmetic,
so both the CUDA path and the fp64 checker can be fed from it without sharing
any of the method's code.

Generator: one counter-based SplitMix64 stream per tensor (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014).  Output
``i`` of a stream is ``mix64(base + (i + 1) * 0x9E3779B97F4A7C15)`` where
``base`` is derived from the workload seed and the tensor's name.  Uniforms are
the top 53 bits scaled by 2**-53; normals come from the Box-Muller transform
(one normal per pair of uniforms).

Shapes and distributions follow the workloads the pages describe for
Qwen3.5-9B's linear-attention layers (16 QK heads, 32 V heads, head dim 128:
"Qwen3.5-9B: Giai ma kien truc Gated DeltaNet", section "Gated DeltaNet"), and
the strong-decay case log(alpha) = -6.72 from the Candle pull request's
"Float32 overflow fix" paragraph.

Layouts (token-major, packed over sequences):
    q, k : [T_total, H_qk, d_k]     v : [T_total, H_v, d_v]
    g    : [T_total, H_v] fp32 (log alpha)   beta : [T_total, H_v] fp32
    state: [n_seqs, H_v, d_k, d_v] fp32
For bf16 workloads the tensors carry both the bf16 bit patterns (``*_bits``,
uint16) and the exact values they encode (float32).
"""

from __future__ import annotations

import concurrent.futures
import dataclasses
import os
import zlib
from typing import Dict, List, Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BLOCK = 1 << 18


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _scalar_mix64(x: int) -> int:
    m = (1 << 64) - 1
    x &= m
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & m
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & m
    return x ^ (x >> 31)


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
    return _POOL


_POOL = None


def _for_blocks(n: int, fn) -> None:
    """Run fn(lo, hi) over [0, n) in blocks; numpy releases the GIL, so blocks run
    in parallel.  Each block depends only on its own counters, so the result does
    not depend on the scheduling."""
    spans = [(lo, min(n, lo + _BLOCK)) for lo in range(0, n, _BLOCK)]
    if len(spans) <= 1:
        for lo, hi in spans:
            fn(lo, hi)
        return
    for f in [_pool().submit(fn, lo, hi) for lo, hi in spans]:
        f.result()


class Stream:
    """One counter-based SplitMix64 stream, keyed by (seed, name)."""

    def __init__(self, seed: int, name: str):
        key = (int(seed) * 0x100000001B3) ^ zlib.crc32(name.encode())
        self.base = _scalar_mix64(key + 0x632BE59BD9B4E019)
        self.pos = 0

    def _raw_into(self, out: np.ndarray, first: int) -> None:
        """out[i] = mix64(base + (first + i + 1) * gamma), in place."""
        with np.errstate(over="ignore"):
            np.add(np.arange(first + 1, first + 1 + out.shape[0], dtype=np.uint64), 0, out=out)
            np.multiply(out, _GAMMA, out=out)
            np.add(out, np.uint64(self.base), out=out)
            t = out >> np.uint64(30)
            np.bitwise_xor(out, t, out=out)
            np.multiply(out, _M1, out=out)
            np.right_shift(out, np.uint64(27), out=t)
            np.bitwise_xor(out, t, out=out)
            np.multiply(out, _M2, out=out)
            np.right_shift(out, np.uint64(31), out=t)
            np.bitwise_xor(out, t, out=out)

    def raw(self, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.uint64)
        first = self.pos
        _for_blocks(n, lambda lo, hi: self._raw_into(out[lo:hi], first + lo))
        self.pos += n
        return out

    def uniform(self, n: int) -> np.ndarray:
        """n doubles in [0, 1)."""
        out = np.empty(n, dtype=np.float64)
        first = self.pos

        def blk(lo, hi):
            r = np.empty(hi - lo, dtype=np.uint64)
            self._raw_into(r, first + lo)
            np.right_shift(r, np.uint64(11), out=r)
            np.multiply(r.astype(np.float64), 2.0 ** -53, out=out[lo:hi])

        _for_blocks(n, blk)
        self.pos += n
        return out

    def normal(self, n: int) -> np.ndarray:
        """n standard normals (Box-Muller, cosine branch; normal i uses uniforms 2i, 2i+1)."""
        out = np.empty(n, dtype=np.float64)
        first = self.pos

        def blk(lo, hi):
            r = np.empty(2 * (hi - lo), dtype=np.uint64)
            self._raw_into(r, first + 2 * lo)
            np.right_shift(r, np.uint64(11), out=r)
            u = r.astype(np.float64).reshape(-1, 2)
            u *= 2.0 ** -53
            rad = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
            np.multiply(rad, np.cos(2.0 * np.pi * u[:, 1]), out=out[lo:hi])

        _for_blocks(n, blk)
        self.pos += 2 * n
        return out

    def integers(self, n: int, lo: int, hi: int) -> np.ndarray:
        """n integers uniform on [lo, hi] inclusive."""
        span = hi - lo + 1
        return lo + np.floor(self.uniform(n) * span).astype(np.int64)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float values to bfloat16 (nearest, ties to even); return uint16 bits."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    fb, ob = f.reshape(-1), out.reshape(-1)

    def blk(lo, hi):
        b = fb[lo:hi].view(np.uint32)
        r = (b >> np.uint32(16)) & np.uint32(1)
        r += b
        r += np.uint32(0x7FFF)
        r >>= np.uint32(16)
        r[np.isnan(fb[lo:hi])] = 0x7FC0
        ob[lo:hi] = r

    _for_blocks(fb.shape[0], blk)
    return out


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """The float32 values that bf16 bit patterns encode (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Workload:
    """One batch of synthetic inputs, with the exact values both sides consume."""

    name: str
    h_qk: int
    h_v: int
    d_k: int
    d_v: int
    chunk: int
    io: str  # "f32" or "bf16"
    cu_seqlens: np.ndarray  # int32 [n+1]
    q: np.ndarray  # float32 exact values [T, H_qk, d_k]
    k: np.ndarray
    v: np.ndarray  # [T, H_v, d_v]
    g: np.ndarray  # float32 [T, H_v]
    beta: np.ndarray  # float32 [T, H_v]
    state0: np.ndarray  # float32 [n, H_v, d_k, d_v]
    q_bits: Optional[np.ndarray] = None  # uint16 when io == "bf16"
    k_bits: Optional[np.ndarray] = None
    v_bits: Optional[np.ndarray] = None
    extra: Dict[str, object] = dataclasses.field(default_factory=dict)

    @property
    def n_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def t_total(self) -> int:
        return int(self.cu_seqlens[-1])


def _unit_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, 1e-300)


def _draw_qkv(st: Dict[str, Stream], t: int, h_qk: int, h_v: int, d_k: int, d_v: int, io: str,
              qk_raw_scale=None):
    if qk_raw_scale is None:
        q = _unit_rows(st["q"].normal(t * h_qk * d_k).reshape(t, h_qk, d_k))
        k = _unit_rows(st["k"].normal(t * h_qk * d_k).reshape(t, h_qk, d_k))
    else:
        # raw rows for the fused normalisation: N(0, 1) times a per-row factor drawn
        # log-uniformly in [lo, hi]
        lo, hi = np.log(qk_raw_scale[0]), np.log(qk_raw_scale[1])
        fq = np.exp(lo + (hi - lo) * st["qscale"].uniform(t * h_qk)).reshape(t, h_qk, 1)
        fk = np.exp(lo + (hi - lo) * st["kscale"].uniform(t * h_qk)).reshape(t, h_qk, 1)
        q = st["q"].normal(t * h_qk * d_k).reshape(t, h_qk, d_k) * fq
        k = st["k"].normal(t * h_qk * d_k).reshape(t, h_qk, d_k) * fk
    v = st["v"].normal(t * h_v * d_v).reshape(t, h_v, d_v)
    out = {}
    for name, x in (("q", q), ("k", k), ("v", v)):
        if io == "bf16":
            bits = bf16_bits(x)
            out[name + "_bits"] = bits
            out[name] = bf16_values(bits)
        else:
            out[name] = x.astype(np.float32)
    return out


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def make_workload(
    name: str,
    seqlens: List[int],
    h_qk: int,
    h_v: int,
    d: int,
    chunk: int,
    io: str,
    seed: int,
    g_range=(-8.0, -0.01),
    g_fixed: Optional[float] = None,
    state_std: float = 0.0,
    tag: str = "",
    n_states: Optional[int] = None,
    qk_raw_scale=None,
    beta_logits: bool = False,
) -> Workload:
    """Draw one packed batch.

    q, k ~ N(0, 1) then L2-normalised per (token, head) in fp64 before rounding
    to the io type; v ~ N(0, 1); log alpha ~ U[g_range] (or fixed);
    beta = sigmoid(N(0, 1)); initial state ~ N(0, state_std) (std, not variance).
    With ``qk_raw_scale = (lo, hi)`` q and k are left unnormalised, each row
    scaled by a factor log-uniform in [lo, hi] (inputs for the fused
    normalisation); with ``beta_logits`` the beta array holds the N(0, 1) logits
    themselves.
    """
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(seqlens, dtype=np.int64))
    t = int(cu[-1])
    st = {n: Stream(seed, tag + n) for n in ("q", "k", "v", "g", "beta", "state", "qscale", "kscale")}
    qkv = _draw_qkv(st, t, h_qk, h_v, d, d, io, qk_raw_scale)
    if g_fixed is not None:
        g = np.full((t, h_v), g_fixed, dtype=np.float32)
    else:
        lo, hi = g_range
        g = (lo + (hi - lo) * st["g"].uniform(t * h_v)).astype(np.float32).reshape(t, h_v)
    logits = st["beta"].normal(t * h_v)
    beta = (logits if beta_logits else _sigmoid(logits)).astype(np.float32).reshape(t, h_v)
    n = len(seqlens) if n_states is None else n_states
    if state_std > 0.0:
        s0 = (state_std * st["state"].normal(n * h_v * d * d)).astype(np.float32)
    else:
        s0 = np.zeros(n * h_v * d * d, dtype=np.float32)
    return Workload(
        name=name, h_qk=h_qk, h_v=h_v, d_k=d, d_v=d, chunk=chunk, io=io, cu_seqlens=cu,
        q=qkv["q"], k=qkv["k"], v=qkv["v"], g=g, beta=beta,
        state0=s0.reshape(n, h_v, d, d),
        q_bits=qkv.get("q_bits"), k_bits=qkv.get("k_bits"), v_bits=qkv.get("v_bits"),
    )


# --- the five workloads -------------------------------------------------------

QWEN35_9B = dict(h_qk=16, h_v=32, d=128)


def tiny(seed: int = 0) -> Workload:
    """B=1, T=64, H_qk=2, H_v=4, d=32, fp32, log alpha ~ U[-2,-0.01], zero state, chunk 16."""
    return make_workload("tiny", [64], 2, 4, 32, 16, "f32", seed, g_range=(-2.0, -0.01))


def prefill_9b(t: int = 1024, seed: int = 1) -> Workload:
    """One Qwen3.5-9B linear-attention layer prefill, B=1, bf16 q/k/v, zero state, chunk 64."""
    return make_workload(f"prefill_T{t}", [t], io="bf16", chunk=64, seed=seed, **QWEN35_9B)


def long_prefill(run: str, t: int = 16384, seed: int = 2) -> Workload:
    """T=16384 prefill from a N(0, 0.02) state; run 'A' draws log alpha ~ U[-8,-0.01],
    run 'B' fixes log alpha = -6.72 for every token and head."""
    kw = dict(io="bf16", chunk=64, seed=seed, state_std=0.02, **QWEN35_9B)
    if run == "A":
        return make_workload(f"long_T{t}_A", [t], tag="A", **kw)
    if run == "B":
        return make_workload(f"long_T{t}_B", [t], tag="B", g_fixed=-6.72, **kw)
    raise ValueError(run)


def decode_batch(b: int = 64, steps: int = 256, seed: int = 3) -> Workload:
    """B independent sequences, ``steps`` decode steps each (fresh inputs per step).

    Tokens are stored step-major: row ``s * b + i`` is step s of sequence i, so
    step s is the contiguous slice [s*b, (s+1)*b)."""
    w = make_workload(f"decode_B{b}", [1] * (b * steps), io="bf16", chunk=64, seed=seed,
                      state_std=0.02, n_states=b, **QWEN35_9B)
    w.cu_seqlens = np.arange(b + 1, dtype=np.int32)  # per-step view: b sequences of length 1
    w.extra.update(batch=b, steps=steps)
    return w


def varlen_verify(n: int = 8, lo: int = 512, hi: int = 8192, seed: int = 4, n_verify: int = 16) -> Workload:
    """n sequences with lengths ~ U{lo..hi} packed by cu_seqlens (zero state), plus a
    16-token verify block per sequence and an accepted prefix length ~ U{0..16}."""
    lens = Stream(seed, "lengths").integers(n, lo, hi).tolist()
    w = make_workload(f"varlen_{n}", lens, io="bf16", chunk=64, seed=seed, **QWEN35_9B)
    vb = make_workload("verify", [n_verify] * n, io="bf16", chunk=16, seed=seed, tag="verify", **QWEN35_9B)
    acc = Stream(seed, "accept").integers(n, 0, n_verify).astype(np.int32)
    w.extra.update(verify=vb, accepted=acc)
    return w
