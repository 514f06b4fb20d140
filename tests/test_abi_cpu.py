"""The C-ABI library builds, loads and exports every symbol the header declares; host-side
argument checks return their error codes without touching a GPU (CPU only)."""
import ctypes
import glob
import os
import re

import pytest

from speculative_decoding_verification_34_gb300 import build
from speculative_decoding_verification_34_gb300 import specverify as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return sv.load_library(path)


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(spec_\w+)\s*\(", text))
    return sorted(names)


def test_header_symbols_exported(lib):
    names = declared_functions()
    assert {"spec_verify_greedy", "spec_verify_sample", "spec_commit_kv_lengths",
            "spec_last_error"} <= set(names)
    raw = ctypes.CDLL(build.LIB)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in include/ but not exported"


FAKE = 0x10000  # never dereferenced: every call below fails its checks before any CUDA call


def greedy(lib, target=FAKE, dtype=0, toks=FAKE, B=4, gmax=3, V=100, out=FAKE, macc=FAKE):
    return lib.spec_verify_greedy(target, dtype, toks, None, B, gmax, V, out, macc, None, FAKE, 1 << 30, None)


def sample(lib, target=FAKE, draft=FAKE, dtype=0, temp=FAKE, ua=FAKE, us=FAKE, B=4, gmax=3, V=100):
    return lib.spec_verify_sample(target, draft, dtype, FAKE, None, temp, ua, us, B, gmax, V,
                                  FAKE, FAKE, None, None, FAKE, 1 << 30, None)


def test_host_argument_checks(lib):
    n0 = lib.spec_launch_count()
    assert greedy(lib, dtype=7) == 2 and b"dtype" in lib.spec_last_error()
    assert greedy(lib, B=-1) == 1
    assert greedy(lib, V=0) == 1
    assert greedy(lib, V=(1 << 30) + 1) == 1
    assert greedy(lib, gmax=-1) == 1
    assert greedy(lib, gmax=33) == 3
    assert greedy(lib, target=None) == 1
    assert greedy(lib, toks=None) == 1
    assert greedy(lib, out=None) == 1 and greedy(lib, macc=None) == 1
    assert greedy(lib, B=0) == 0 and lib.spec_last_error() == b""
    assert greedy(lib, toks=None, gmax=0, B=0) == 0
    assert sample(lib, draft=None) == 1 and sample(lib, temp=None) == 1
    assert sample(lib, ua=None) == 1 and sample(lib, us=None) == 1
    assert sample(lib, B=0) == 0
    assert sample(lib, draft=None, ua=None, gmax=0, B=0) == 0
    c = lib.spec_commit_kv_lengths
    assert c(FAKE, 4, FAKE, None, 1, FAKE, 3, None, None, 10, None, None) == 1   # partial history args
    assert c(FAKE, 4, FAKE, None, 1, FAKE, 3, FAKE, FAKE, 0, None, None) == 1    # cap < 1
    assert c(None, 4, FAKE, None, 1, None, 3, None, None, 0, None, None) == 1
    assert c(FAKE, 4, FAKE, None, 1, None, 64, None, None, 0, None, None) == 3
    assert c(FAKE, 0, FAKE, None, 1, None, 3, None, None, 0, None, None) == 0
    assert c(None, 0, None, None, 1, None, 3, None, None, 0, None, None) == 0
    s = lib.spec_apply_stops
    assert s(None, FAKE, 4, 3, 0, None, None, None) == 1 and s(FAKE, None, 4, 3, 0, None, None, None) == 1
    assert s(FAKE, FAKE, -1, 3, 0, None, None, None) == 1 and s(FAKE, FAKE, 4, 64, 0, None, None, None) == 3
    assert s(None, None, 0, 3, 0, None, None, None) == 0
    assert greedy(lib, target=None, toks=None, out=None, macc=None, B=0) == 0
    assert sample(lib, target=None, draft=None, temp=None, ua=None, us=None, B=0) == 0
    assert lib.spec_launch_count() == n0      # nothing was launched


def test_split_layout_argument_checks(lib):
    """The split-layout calls check their two target arrays on the host: the saved row is
    always required, the block rows only when there are drafts."""
    n0 = lib.spec_launch_count()
    g = lambda saved=FAKE, block=FAKE, B=4, gmax=3: lib.spec_verify_greedy_split(
        saved, block, 0, FAKE, None, B, gmax, 100, FAKE, FAKE, None, FAKE, 8, None)
    s = lambda saved=FAKE, block=FAKE, B=4, gmax=3: lib.spec_verify_sample_split(
        saved, block, FAKE, 0, FAKE, None, FAKE, FAKE, FAKE, B, gmax, 100, FAKE, FAKE, None, None, FAKE, 8, None)
    assert g(saved=None) == 1 and s(saved=None) == 1
    assert g(block=None) == 1 and b"block_logits" in lib.spec_last_error()
    assert s(block=None) == 1
    # block may be null without drafts; the 8-byte workspace is then what is refused
    assert g(block=None, gmax=0) == 3 and b"workspace" in lib.spec_last_error()
    assert g(saved=None, block=None, B=0) == 0 and s(saved=None, block=None, B=0) == 0
    assert lib.spec_launch_count() == n0


def test_tree_argument_checks(lib):
    n0 = lib.spec_launch_count()
    t = lambda tgt=FAKE, toks=FAKE, par=FAKE, B=4, nmax=7, V=100, dtype=0: lib.spec_verify_tree_greedy(
        tgt, dtype, toks, par, None, B, nmax, V, FAKE, FAKE, None, None, FAKE, 8, None)
    assert t(dtype=5) == 2
    assert t(B=-1) == 1 and t(nmax=-1) == 1 and t(V=0) == 1
    assert t(nmax=64) == 3 and b"SPEC_MAX_TREE_NODES" in lib.spec_last_error()
    assert t(tgt=None) == 1 and t(toks=None) == 1 and t(par=None) == 1
    assert t(toks=None, par=None, nmax=0) == 3 and b"workspace" in lib.spec_last_error()
    assert t(tgt=None, toks=None, par=None, B=0) == 0
    assert lib.spec_launch_count() == n0
    assert sv.spec_verify_workspace_bytes(4, 63, 100) > 0 and sv.spec_verify_workspace_bytes(4, 64, 100) == 0


def test_truncated_argument_checks(lib):
    n0 = lib.spec_launch_count()
    t = lambda dtype=0, draft=FAKE, temp=FAKE, B=4, V=100: lib.spec_verify_sample_truncated(
        FAKE, draft, dtype, FAKE, None, temp, None, None, FAKE, FAKE, B, 3, V, FAKE, FAKE, None, None, FAKE, 8, None)
    assert t(dtype=1) == 2 and b"bf16" in lib.spec_last_error()
    assert t(draft=None) == 1 and t(temp=None) == 1
    assert t(V=(1 << 21) + 8) == 3
    assert t() == 3 and b"workspace" in lib.spec_last_error()
    assert t(draft=None, temp=None, B=0) == 0
    # the split layout: the saved row always, the block rows when there are drafts
    ts = lambda saved=FAKE, block=FAKE, dtype=0, B=4, gmax=3: lib.spec_verify_sample_truncated_split(
        saved, block, FAKE, dtype, FAKE, None, FAKE, None, None, FAKE, FAKE, B, gmax, 100, FAKE, FAKE, None, None,
        FAKE, 8, None)
    assert ts(saved=None) == 1
    assert ts(block=None) == 1 and b"block_logits" in lib.spec_last_error()
    assert ts(dtype=1) == 2
    assert ts(block=None, gmax=0) == 3 and b"workspace" in lib.spec_last_error()
    assert ts(saved=None, block=None, B=0) == 0
    assert lib.spec_launch_count() == n0


def test_plan_splits_vocabulary(lib):
    for V in [1, 3, 1024, 4096, 4097, 32000, 50000, 128256, 151936, 1 << 20]:
        cl, chunk = sv.spec_verify_plan(V)
        assert 1 <= cl <= 64 and chunk % 8 == 0
        assert cl * chunk >= V and (cl - 1) * chunk < V, (V, cl, chunk)
    assert sv.spec_verify_plan(128256) == (2, 64128)
    assert sv.spec_verify_plan(151936) == (3, 50648)


def test_workspace_size(lib):
    n = sv.spec_verify_workspace_bytes(128, 4, 128256)
    cl, _ = sv.spec_verify_plan(128256)
    # per-(row, chunk) partials, draft logits and per-warp draw masses are handed over in it
    assert n >= 128 * (9 * cl * 8 + 9 * 8)
    assert n < 1 << 20
    assert sv.spec_verify_workspace_bytes(128, 4, 128256) == sv.spec_verify_workspace_bytes(128, 4, 128256, 1)
    assert sv.spec_verify_workspace_bytes(-1, 4, 100) == 0
    assert sv.spec_verify_workspace_bytes(4, 64, 100) == 0   # beyond a tree call's 63 nodes
    # too small a workspace is refused on the host, before any CUDA call
    assert lib.spec_verify_greedy(FAKE, 0, FAKE, None, 4, 3, 100, FAKE, FAKE, None, FAKE, 8, None) == 3
    assert b"workspace" in lib.spec_last_error()
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_plan(0)


def test_static_workspace_limits_in_header():
    """The largest batches the static workspace takes, as include/specverify.h states them."""
    text = open(os.path.join(ROOT, "include", "specverify.h"), encoding="utf-8").read()
    cap = 1 << 20
    for B, V in ((1110, 128256), (910, 151936)):
        assert f"B = {B} at" in text and f"V = {V}" in text
        assert sv.spec_verify_workspace_bytes(B, 4, V) <= cap < sv.spec_verify_workspace_bytes(B + 1, 4, V)


def test_binding_arity_matches_header(lib):
    """The ctypes argument lists of the binding match the parameter lists in include/."""
    text = ""
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text += re.sub(r"/\*.*?\*/", "", open(h, encoding="utf-8").read(), flags=re.S)
    for name in ("spec_verify_greedy", "spec_verify_sample", "spec_commit_kv_lengths",
                 "spec_verify_workspace_bytes", "spec_verify_plan", "spec_verify_sample_static",
                 "spec_apply_stops", "spec_verify_greedy_split", "spec_verify_sample_split",
                 "spec_verify_tree_greedy", "spec_verify_sample_truncated",
                 "spec_verify_sample_truncated_split", "spec_verify_greedy_commit",
                 "spec_verify_sample_truncated_commit", "spec_verify_tree_greedy_commit",
                 "spec_verify_sample_commit"):
        m = re.search(r"\b" + name + r"\s*\(([^)]*)\)", text)
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(getattr(lib, name).argtypes) == len(params), name
    # the prepared call marshals the same argument list
    import inspect
    src = inspect.getsource(sv.prepare_verify_sample)
    assert "wsp, wsn" in src


def test_static_workspace_refuses_oversized_calls(lib):
    """The static-workspace entry refuses, on the host, a batch whose counters alone exceed
    the array (B = 100000 at gmax = 4, V = 128256: 6.4 MB of draw-chunk states)."""
    n0 = lib.spec_launch_count()
    rc = lib.spec_verify_sample_static(FAKE, FAKE, 0, FAKE, None, FAKE, FAKE, FAKE, 100000, 4, 128256,
                                       FAKE, FAKE, None, None, None)
    assert rc == 3 and b"static workspace" in lib.spec_last_error()
    assert lib.spec_launch_count() == n0
    assert lib.spec_verify_sample_static(FAKE, FAKE, 0, FAKE, None, FAKE, FAKE, FAKE, 0, 4, 128256,
                                         FAKE, FAKE, None, None, None) == 0


def test_fused_commit_argument_checks(lib):
    """The fused verify-and-commit calls refuse bad commit arguments on the host, before any
    CUDA call, the way spec_commit_kv_lengths does."""
    n0 = lib.spec_launch_count()
    g = lambda t=FAKE, h=None, c=None, cap=0: lib.spec_verify_greedy_commit(
        FAKE, 0, FAKE, None, 4, 3, 100, FAKE, FAKE, None, FAKE, 8, t, None, 1, h, c, cap, None)
    assert g(t=None) == 1 and b"target_kv_len" in lib.spec_last_error()
    assert g(h=FAKE) == 1 and g(c=FAKE) == 1
    assert g(h=FAKE, c=FAKE, cap=0) == 1 and b"capacity" in lib.spec_last_error()
    s = lambda t=FAKE, h=None, c=None, cap=0, B=4: lib.spec_verify_sample_commit(
        FAKE, FAKE, 0, FAKE, None, FAKE, FAKE, FAKE, B, 3, 100, FAKE, FAKE, None, None, FAKE, 8,
        t, None, 1, h, c, cap, None)
    assert s(t=None) == 1 and s(h=FAKE) == 1
    assert s(t=None, B=0) == 0          # empty batch: nothing to check, nothing enqueued
    tr = lambda t=FAKE, h=None, c=None, cap=0, B=4, dtype=0: lib.spec_verify_sample_truncated_commit(
        FAKE, FAKE, dtype, FAKE, None, FAKE, None, None, FAKE, FAKE, B, 3, 100, FAKE, FAKE, None, None, FAKE, 8,
        t, None, 1, h, c, cap, None)
    assert tr(t=None) == 1 and tr(h=FAKE) == 1 and tr(h=FAKE, c=FAKE, cap=0) == 1
    assert tr(t=None, B=0) == 0
    assert tr(dtype=1) == 2 and b"bf16" in lib.spec_last_error()
    tc = lambda t=FAKE, h=None, c=None, cap=0, B=4: lib.spec_verify_tree_greedy_commit(
        FAKE, 0, FAKE, FAKE, None, B, 3, 100, FAKE, FAKE, None, None, FAKE, 8, t, None, 1, h, c, cap, None)
    assert tc(t=None) == 1 and tc(h=FAKE) == 1 and tc(h=FAKE, c=FAKE, cap=0) == 1
    assert tc(t=None, B=0) == 0
    # valid commit arguments reach the workspace check (8 bytes: refused) and stop there
    assert tc() == 3 and b"workspace" in lib.spec_last_error()
    assert g() == 3 and s() == 3 and b"workspace" in lib.spec_last_error()
    assert tr() == 3 and b"workspace" in lib.spec_last_error()
    assert lib.spec_launch_count() == n0
