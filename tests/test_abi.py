"""The C-ABI library on the CPU: it loads, exports every entry point that
include/gdr.h declares, and rejects bad arguments on the host before any launch.
No call here reaches a kernel (no GPU is needed)."""

import ctypes
import os
import re

import pytest

import gated_deltanet_scan_gb300 as gdr
from gated_deltanet_scan_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr.h")

A = 0x100000  # a 16-byte aligned stand-in address: validation never dereferences it
B = 0x200000
MISALIGNED = 0x100004


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return gdr.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdr_[a-z_]+)\s*\(", text)))


def dims(**kw):
    d = dict(h_qk=16, h_v=32, d_k=128, d_v=128, chunk=64, in_dtype=gdr.GDR_BF16,
             out_dtype=gdr.GDR_F32, scale=1.0)
    d.update(kw)
    return gdr.gdr_dims(**d)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"gdr_prefill_chunked", "gdr_decode_step", "gdr_verify_block", "gdr_verify_commit",
            "gdr_state_snapshot", "gdr_state_restore"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in gdr.h but not exported"


def test_abi_version_matches_header(L):
    m = re.search(r"#define GDR_ABI_VERSION (\d+)", open(HEADER).read())
    assert L.gdr_abi_version() == int(m.group(1))


def test_status_strings(L):
    for code in range(5):
        s = L.gdr_status_string(code).decode()
        assert s.startswith("GDR_")
    assert L.gdr_status_string(99).decode() == "unknown gdr_status"


def _prefill(L, d, n=1, cu=A, t=10, q=A, k=A, v=A, g=A, beta=A, state=A, o=B, ws=A, ws_bytes=1 << 40):
    return L.gdr_prefill_chunked(ctypes.byref(d) if d is not None else None, n, cu, t,
                                 q, k, v, g, beta, state, o, ws, ws_bytes, None)


@pytest.mark.parametrize("bad,code", [
    (dict(h_v=33), gdr.GDR_ERR_INVALID_ARG),
    (dict(h_qk=0), gdr.GDR_ERR_INVALID_ARG),
    (dict(in_dtype=7), gdr.GDR_ERR_INVALID_ARG),
    (dict(out_dtype=-1), gdr.GDR_ERR_INVALID_ARG),
    (dict(d_k=96, d_v=96), gdr.GDR_ERR_UNSUPPORTED),
    (dict(d_v=64), gdr.GDR_ERR_UNSUPPORTED),
    (dict(chunk=32), gdr.GDR_ERR_UNSUPPORTED),
])
def test_prefill_rejects_bad_dims(L, bad, code):
    assert _prefill(L, dims(**bad)) == code


def test_prefill_rejects_bad_pointers_and_counts(L):
    d = dims()
    assert _prefill(L, None) == gdr.GDR_ERR_INVALID_ARG
    assert _prefill(L, d, q=None) == gdr.GDR_ERR_INVALID_ARG
    assert _prefill(L, d, v=MISALIGNED) == gdr.GDR_ERR_INVALID_ARG
    assert _prefill(L, d, cu=None) == gdr.GDR_ERR_INVALID_ARG
    assert _prefill(L, d, state=None) == gdr.GDR_ERR_INVALID_ARG
    assert _prefill(L, d, n=-1) == gdr.GDR_ERR_INVALID_ARG
    assert _prefill(L, d, t=-5) == gdr.GDR_ERR_INVALID_ARG
    assert _prefill(L, d, n=0, t=5) == gdr.GDR_ERR_INVALID_ARG
    assert _prefill(L, d, n=0, t=0) == gdr.GDR_OK  # nothing to do, nothing launched


def test_prefill_workspace_size_and_checks(L):
    d = dims()
    # one 17,152-byte slot per (chunk position, V head), positions = ceil(T / 64) + n_seqs,
    # then from the next 1 KiB boundary one 16 KiB X tile per (position, QK head)
    need = L.gdr_prefill_workspace_bytes(ctypes.byref(d), 3, 1000)
    slots = (1000 + 63) // 64 + 3
    x_off = (slots * 32 * 17152 + 1023) // 1024 * 1024
    assert need == (x_off + slots * 16 * 16384 + 255) // 256 * 256
    assert L.gdr_prefill_workspace_bytes(ctypes.byref(d), 0, 0) == 0
    assert L.gdr_prefill_workspace_bytes(ctypes.byref(dims(in_dtype=gdr.GDR_F32)), 3, 1000) == 0
    assert L.gdr_prefill_workspace_bytes(ctypes.byref(dims(chunk=16)), 3, 1000) == 0
    assert L.gdr_prefill_workspace_bytes(None, 3, 1000) == 0
    need10 = L.gdr_prefill_workspace_bytes(ctypes.byref(d), 1, 10)
    assert _prefill(L, d, ws=None) == gdr.GDR_ERR_INVALID_ARG
    assert _prefill(L, d, ws=MISALIGNED) == gdr.GDR_ERR_INVALID_ARG
    assert _prefill(L, d, ws_bytes=need10 - 1) == gdr.GDR_ERR_INVALID_ARG


def test_decode_and_verify_reject_bad_arguments(L):
    d = dims()
    for dec in (L.gdr_decode_step, L.gdr_decode_step_overlapped):
        assert dec(ctypes.byref(d), -1, A, A, A, A, A, A, B, None) == gdr.GDR_ERR_INVALID_ARG
        assert dec(ctypes.byref(d), 4, A, A, None, A, A, A, B, None) == gdr.GDR_ERR_INVALID_ARG
        assert dec(ctypes.byref(d), 4, A, A, A, A, A, A, MISALIGNED, None) == gdr.GDR_ERR_INVALID_ARG
        assert dec(ctypes.byref(d), 0, None, None, None, None, None, None, None, None) == gdr.GDR_OK
    ver = L.gdr_verify_block
    assert ver(ctypes.byref(d), 2, 17, A, A, A, A, A, A, B, B, None, None) == gdr.GDR_ERR_INVALID_ARG
    assert ver(ctypes.byref(d), 2, 16, A, A, A, A, A, A, A, B, None, None) == gdr.GDR_ERR_INVALID_ARG
    assert ver(ctypes.byref(d), 2, 16, A, A, A, A, A, A, None, B, None, None) == gdr.GDR_ERR_INVALID_ARG
    assert ver(ctypes.byref(d), -2, 16, A, A, A, A, A, A, B, B, None, None) == gdr.GDR_ERR_INVALID_ARG
    assert ver(ctypes.byref(d), 2, 16, A, A, A, A, A, A, B, B, MISALIGNED, None) == gdr.GDR_ERR_INVALID_ARG


def test_verify_commit_rejects_bad_arguments(L):
    d = dims(chunk=16)
    com = L.gdr_verify_commit
    # (dims, n_seqs, n_tok, accepted, k, g, deltas, snapshot, state, stream)
    assert com(ctypes.byref(d), 2, 17, A, A, A, A, A, B, None) == gdr.GDR_ERR_INVALID_ARG
    assert com(ctypes.byref(d), -1, 16, A, A, A, A, A, B, None) == gdr.GDR_ERR_INVALID_ARG
    assert com(ctypes.byref(d), 2, 16, None, A, A, A, A, B, None) == gdr.GDR_ERR_INVALID_ARG
    assert com(ctypes.byref(d), 2, 16, A, A, A, A, A, A, None) == gdr.GDR_ERR_INVALID_ARG  # snapshot == state
    assert com(ctypes.byref(d), 2, 16, A, A, A, None, A, B, None) == gdr.GDR_ERR_INVALID_ARG
    assert com(ctypes.byref(d), 2, 16, A, A, A, MISALIGNED, A, B, None) == gdr.GDR_ERR_INVALID_ARG
    assert com(ctypes.byref(d), 2, 16, A, A, A, A, MISALIGNED, B, None) == gdr.GDR_ERR_INVALID_ARG
    assert com(ctypes.byref(gdr.gdr_dims(h_qk=16, h_v=32, d_k=96, d_v=96, chunk=16, in_dtype=gdr.GDR_BF16,
                                         out_dtype=gdr.GDR_F32, scale=1.0)),
               2, 16, A, A, A, A, A, B, None) != gdr.GDR_OK
    assert com(ctypes.byref(d), 0, 16, None, None, None, None, None, None, None) == gdr.GDR_OK


def test_snapshot_restore_reject_bad_arguments(L):
    d = dims()
    assert L.gdr_state_snapshot(ctypes.byref(d), 2, A, A, None) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_state_restore(ctypes.byref(d), 2, None, A, None) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_state_restore(ctypes.byref(d), 2, MISALIGNED, A, None) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_state_snapshot(ctypes.byref(d), 0, A, B, None) == gdr.GDR_OK
    assert L.gdr_device_error(None, None) == gdr.GDR_ERR_INVALID_ARG


def test_selftest_wait_timeout_rejects_bad_limits(L):
    # checked on the host before any launch (no GPU here)
    for bad in (0, -5, (1 << 31) + 1):
        assert L.gdr_selftest_wait_timeout(bad, None) == gdr.GDR_ERR_INVALID_ARG


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(gdr, "_lib", None)
    monkeypatch.setattr(gdr, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        gdr.lib()


def test_product_package_never_imports_the_oracle():
    pkg = os.path.dirname(gdr.__file__)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "gdr_oracle" not in text and "liboracle" not in text, f


def test_segmented_workspace_size_and_checks(L):
    """Sizes and host-side rejections of the two-level prefill (no launch)."""
    d = dims()
    base = L.gdr_prefill_workspace_bytes(ctypes.byref(d), 1, 16384)
    assert L.gdr_prefill_segmented_workspace_bytes(ctypes.byref(d), 1, 16384, 1) == base
    # four state-sized blocks per (segment after the first, V head): Phi, B and the
    # start state in fp32, the start state's bf16 hi/lo operand tiles; two fp32 arrays like o
    st, rows = 32 * 128 * 128 * 4, 16384 * 32 * 128 * 4
    for P in (2, 4, 8):
        got = L.gdr_prefill_segmented_workspace_bytes(ctypes.byref(d), 1, 16384, P)
        assert got == ((base + 255) // 256 * 256) + 4 * (P - 1) * st + 2 * rows, P
    # more segments than chunk positions: one per chunk (2 chunks here)
    two = L.gdr_prefill_segmented_workspace_bytes(ctypes.byref(d), 1, 100, 2)
    assert L.gdr_prefill_segmented_workspace_bytes(ctypes.byref(d), 1, 100, 8) == two
    assert L.gdr_prefill_segmented_workspace_bytes(ctypes.byref(d), 1, 64, 8) == \
        L.gdr_prefill_workspace_bytes(ctypes.byref(d), 1, 64)
    ws = L.gdr_prefill_segmented_workspace_bytes(ctypes.byref(d), 1, 4096, 4)
    args = lambda P, dd=d, w=ws, wp=A: (ctypes.byref(dd), 1, A, 4096, A, A, A, A, A, A, A, P, wp, w, None)
    for P in (0, 9, -1):
        assert L.gdr_prefill_segmented(*args(P)) == gdr.GDR_ERR_INVALID_ARG, P
    assert L.gdr_prefill_segmented(*args(4, w=ws - 1)) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_prefill_segmented(*args(4, wp=MISALIGNED)) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_prefill_segmented(*args(4, dd=dims(in_dtype=gdr.GDR_F32))) == gdr.GDR_ERR_UNSUPPORTED
    assert L.gdr_prefill_segmented(*args(4, dd=dims(chunk=16))) == gdr.GDR_ERR_UNSUPPORTED
    assert L.gdr_prefill_segmented(*args(4, dd=dims(h_v=30))) == gdr.GDR_ERR_INVALID_ARG
    # more (sequence, V head) pairs than one grid dimension indexes
    many = (ctypes.byref(d), 2048, A, 4096, A, A, A, A, A, A, A, 4, A, 1 << 40, None)
    assert L.gdr_prefill_segmented(*many) == gdr.GDR_ERR_UNSUPPORTED
    bad_ptr = (ctypes.byref(d), 1, A, 4096, A, MISALIGNED, A, A, A, A, A, 4, A, ws, None)
    assert L.gdr_prefill_segmented(*bad_ptr) == gdr.GDR_ERR_INVALID_ARG
    # without a GPU the hint is 1 (no SMs to spread segments over); invalid dims: 1
    assert L.gdr_prefill_segments_hint(None, 1, 16384) == 1
    assert L.gdr_prefill_segments_hint(ctypes.byref(dims(chunk=16)), 1, 16384) == 1


def test_flags_and_gated_rmsnorm_checks(L):
    """Unknown flag bits and bad norm arguments are rejected on the host."""
    assert L.gdr_decode_step(ctypes.byref(dims(flags=4)), 1, A, A, A, A, A, A, A, None) == gdr.GDR_ERR_INVALID_ARG
    ok = dims(flags=gdr.GDR_FLAG_QK_L2NORM | gdr.GDR_FLAG_BETA_LOGITS)
    assert L.gdr_prefill_workspace_bytes(ctypes.byref(ok), 1, 1000) == L.gdr_prefill_workspace_bytes(
        ctypes.byref(dims()), 1, 1000)  # flags change no size
    nrm = L.gdr_gated_rmsnorm
    assert nrm(ctypes.byref(dims()), 0, A, A, A, 1e-6, A, None) == gdr.GDR_OK
    assert nrm(ctypes.byref(dims()), -1, A, A, A, 1e-6, A, None) == gdr.GDR_ERR_INVALID_ARG
    assert nrm(ctypes.byref(dims()), 5, A, A, A, -1.0, A, None) == gdr.GDR_ERR_INVALID_ARG
    assert nrm(ctypes.byref(dims()), 5, MISALIGNED, A, A, 1e-6, A, None) == gdr.GDR_ERR_INVALID_ARG
    assert nrm(ctypes.byref(dims()), 5, A, None, A, 1e-6, A, None) == gdr.GDR_ERR_INVALID_ARG
    gated = L.gdr_decode_step_gated
    assert gated(ctypes.byref(dims()), 1, A, A, A, A, A, A, None, A, 1e-6, A, None) == gdr.GDR_ERR_INVALID_ARG
    assert gated(ctypes.byref(dims()), 1, A, A, A, A, A, A, A, MISALIGNED, 1e-6, A, None) == gdr.GDR_ERR_INVALID_ARG


def test_prefill_with_decode_checks(L):
    """Host-side rejections of the mixed prefill + decode launch (nothing launched)."""
    d = dims()

    def args(dd=d, nd=4, dq=A, dstate=B):
        # dims, n_seqs, cu, T, q, k, v, g, beta, state, o, ws, ws_bytes, dec_batch, dq, dk, dv, dg, dbeta, dstate, do
        return (ctypes.byref(dd), 1, A, 4096, A, A, A, A, A, A, A, A, 1 << 30, nd, dq, A, A, A, A, dstate, A, None)
    assert L.gdr_prefill_with_decode(*args(dd=dims(in_dtype=gdr.GDR_F32))) == gdr.GDR_ERR_UNSUPPORTED
    assert L.gdr_prefill_with_decode(*args(dd=dims(chunk=16))) == gdr.GDR_ERR_UNSUPPORTED
    assert L.gdr_prefill_with_decode(*args(dd=dims(h_v=30))) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_prefill_with_decode(*args(nd=-1)) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_prefill_with_decode(*args(dq=None)) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_prefill_with_decode(*args(dq=MISALIGNED)) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_prefill_with_decode(*args(dstate=A)) == gdr.GDR_ERR_INVALID_ARG  # the prefill's own state
