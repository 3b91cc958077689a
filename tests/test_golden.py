"""Fixtures under tests/golden: the pages' own constants, and a regression
record of the oracle on the tiny workload (written by make_oracle_samples.py,
which calls only the oracle)."""

import json
import os

import numpy as np

import oracle
from gated_deltanet_scan_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_workload_shapes_follow_the_pages():
    c = _load("pages_constants.json")
    heads = c["qwen35_9b_linear_attention_heads"]
    assert synth.QWEN35_9B == dict(h_qk=heads["h_qk"], h_v=heads["h_v"], d=heads["head_dim"])
    shape = c["state_shape_per_layer"]
    assert (shape["rows"], shape["cols"]) == (heads["head_dim"], heads["head_dim"])
    w = synth.long_prefill("B", t=128)
    assert np.all(w.g == np.float32(c["strong_decay_log_alpha"]["value"]))
    assert synth.prefill_9b(t=64).chunk == c["chunk_sizes"]["prefill"]
    assert synth.tiny().chunk == c["chunk_sizes"]["small_block"]


def test_overflow_reading_of_the_strong_decay():
    """At log alpha = -6.72 per token, exp of the unmasked exponent G_t - G_j for
    t < j passes fp32's largest finite value from a distance of 14 tokens
    (the Candle PR's overflow paragraph; its printed 'exp(~275) ... t >= 15' is
    garbled, this is the reading taken)."""
    a = np.float32(-6.72)
    with np.errstate(over="ignore"):
        assert np.isfinite(np.exp(np.float32(-13) * a))
        assert not np.isfinite(np.exp(np.float32(-14) * a))


def test_oracle_regression_samples():
    ref = _load("tiny_oracle_samples.json")
    w = synth.tiny()
    chk = ref["inputs_checksum"]
    assert float(np.sum(w.q, dtype=np.float64)) == chk["q_sum"]
    assert float(np.sum(w.v, dtype=np.float64)) == chk["v_sum"]
    assert float(np.sum(w.g, dtype=np.float64)) == chk["g_sum"]
    assert float(np.sum(w.beta, dtype=np.float64)) == chk["beta_sum"]
    o, S = oracle.run_workload(w, threads=1)
    for t, h, j, val in ref["o_samples"]:
        assert abs(o[t, h, j] - val) <= 1e-13 * max(1.0, abs(val))
    assert abs(np.sqrt(np.mean(o * o)) - ref["o_rms"]) <= 1e-13
    for h, fro in enumerate(ref["state_fro"]):
        assert abs(np.linalg.norm(S[0, h]) - fro) <= 1e-12 * fro


def test_synth_streams_are_deterministic_and_distinct():
    a = synth.Stream(1, "q").raw(1000)
    b = synth.Stream(1, "q").raw(1000)
    c = synth.Stream(1, "k").raw(1000)
    d = synth.Stream(2, "q").raw(1000)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)
    # counter-based: drawing in two pieces equals one draw
    s = synth.Stream(7, "v")
    x = np.concatenate([s.raw(300), s.raw(700)])
    assert np.array_equal(x, synth.Stream(7, "v").raw(1000))
    u = synth.Stream(3, "u").uniform(200000)
    assert 0.0 <= u.min() and u.max() < 1.0 and abs(u.mean() - 0.5) < 0.005
    z = synth.Stream(3, "z").normal(200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 3.0e38, 1e-40], dtype=np.float32)
    bits = synth.bf16_bits(x)
    vals = synth.bf16_values(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties to even gives 1
    assert vals[0] == 1.0 and vals[1] == 1.0
    assert vals[2] == np.float32(1.0 + 2 ** -7)
    assert vals[3] == -2.5
    assert np.isfinite(vals[4])
