"""Helpers for GPU-vs-oracle parity tests: upload a workload, run the C-ABI through the
binding, compare with the float64 oracle sequence by sequence."""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

from oracle import specverify_oracle as O
from speculative_decoding_verification_34_gb300 import specverify as sv

CANARY = 64
SENT_I = -123456789
PROB_TOL = 1e-5
MARGIN_TOL = 1e-5


def dev(a: np.ndarray, dtype: str = None) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays become bfloat16 (bit pattern preserved)."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def padded(shape, dtype, fill):
    """A CUDA buffer with CANARY sentinel elements after the returned view."""
    n = int(np.prod(shape))
    buf = torch.full((n + CANARY,), fill, dtype=dtype, device="cuda")
    return buf, buf[:n].view(*shape)


def canary_ok(buf, n, fill) -> bool:
    tail = buf[n:].cpu()
    if tail.dtype.is_floating_point and math.isnan(fill):
        return bool(torch.isnan(tail).all())
    return bool((tail == fill).all())


_WS = {}


def workspace(B, g, V, code):
    """A zero-filled workspace reused across calls (each call must return its counters to 0)."""
    n = sv.spec_verify_workspace_bytes(B, g, V, code)
    key = torch.cuda.current_device()
    if key not in _WS or _WS[key].numel() < n:
        _WS[key] = torch.zeros(max(n, 64), dtype=torch.uint8, device="cuda")
    return _WS[key]


def workspace_is_clean() -> bool:
    """The whole workspace (counters and hand-over words) is zero again after a call."""
    return all(bool((w == 0).all()) for w in _WS.values())


def run_gpu(wl, mode: str = "auto", target=None, draft=None, check_canary=True):
    """Run one verify call on a Workload.  mode: 'greedy' (spec_verify_greedy) or 'sample'."""
    if mode == "auto":
        mode = "greedy" if wl.greedy_only else "sample"
    B, g = wl.B, wl.gmax
    tgt = dev(wl.target) if target is None else target
    toks = dev(wl.draft_tokens)
    nd = dev(wl.num_draft)
    ob, out = padded((B, g + 1), torch.int32, SENT_I)
    mb, macc = padded((B,), torch.int32, SENT_I)
    sb, st = padded((B,), torch.int32, SENT_I)
    db, dg = padded((B, 2 * g + 1), torch.float32, float("nan"))
    code = sv.SPEC_BF16 if wl.dtype == "bf16" else sv.SPEC_F32
    ws = workspace(B, g, wl.V, code)
    if mode == "greedy":
        sv.spec_verify_greedy(tgt, toks, nd, out, macc, st, workspace=ws)
    else:
        drf = dev(wl.draft) if draft is None else draft
        sv.spec_verify_sample(tgt, drf, toks, nd, dev(wl.temperature), dev(wl.u_accept),
                              dev(wl.u_sample), out, macc, dg, st, workspace=ws)
    torch.cuda.synchronize()
    if check_canary:
        assert workspace_is_clean(), "the call did not return the workspace counters to zero"
    if check_canary:
        assert canary_ok(ob, B * (g + 1), SENT_I), "out_tokens overrun"
        assert canary_ok(mb, B, SENT_I), "num_accepted overrun"
        assert canary_ok(sb, B, SENT_I), "status overrun"
        if mode == "sample":
            assert canary_ok(db, B * (2 * g + 1), float("nan")), "diag overrun"
    return {"out": out.cpu().numpy(), "m": macc.cpu().numpy(), "status": st.cpu().numpy(),
            "diag": dg.cpu().numpy() if mode == "sample" else None}


def oracle_results(wl, seqs=None, mode="auto"):
    if mode == "auto":
        mode = "greedy" if wl.greedy_only else "sample"
    temp = None if mode == "greedy" else wl.temperature
    return O.verify_batch(wl.target, wl.draft, wl.dtype, wl.draft_tokens, wl.num_draft, temp,
                          wl.u_accept, wl.u_sample, seqs=seqs)


def draft_probs(wl, b, g):
    """p_i(d_i), q_i(d_i) for every i < g from the oracle's softmax (NaN for bad ids)."""
    T = float(wl.temperature[b])
    pd, qd = [], []
    for i in range(g):
        d = int(wl.draft_tokens[b, i])
        if 0 <= d < wl.V:
            p = O.softmax_at_temperature(O.widen(wl.target[b, i], wl.dtype), T)
            q = O.softmax_at_temperature(O.widen(wl.draft[b, i], wl.dtype), T)
            pd.append(p[d])
            qd.append(q[d])
        else:
            pd.append(math.nan)
            qd.append(math.nan)
    return pd, qd


def compare(wl, gpu, results, seqs=None, check_probs=True):
    """Element-by-element comparison.  Returns (n_checked, flagged, differ): flagged are the
    sequences with an oracle decision margin < MARGIN_TOL, differ those of them whose GPU
    result is not the oracle's.  Raises on any mismatch in an unflagged sequence."""
    seqs = list(range(wl.B)) if seqs is None else list(seqs)
    flagged, differ = [], []
    g_all = wl.gmax
    for b, r in zip(seqs, results):
        out, m, st = gpu["out"][b], int(gpu["m"][b]), int(gpu["status"][b])
        want = np.full(g_all + 1, -1)
        want[: len(r.tokens)] = r.tokens
        same = m == r.m and list(out) == list(want) and st == r.status
        if r.status & O.ST_BAD_ROW:
            # no distribution on one of the rows: the mark, and a well-formed step
            flagged.append(b)
            if not same:
                differ.append(b)
            assert st & O.ST_BAD_ROW, f"seq {b}: status gpu={st}, oracle marks a row without a distribution"
            assert 0 <= m <= r.gamma and 0 <= out[m] < wl.V, (b, out, m)
            assert list(out[:m]) == list(wl.draft_tokens[b, :m]), (b, out)
            assert all(x == -1 for x in out[m + 1:]), (b, out)
            continue
        assert not st & O.ST_BAD_ROW, f"seq {b}: gpu marks a bad row the oracle does not see"
        if r.flagged(MARGIN_TOL):
            flagged.append(b)
            if not same:
                differ.append(b)
            # several answers are correct here: check that this one is a valid step
            assert 0 <= m <= r.gamma and out[m] >= 0 and out[m] < wl.V, (b, out, m)
            assert list(out[:m]) == list(wl.draft_tokens[b, :m]), (b, out)
            assert all(x == -1 for x in out[m + 1:]), (b, out)
        else:
            assert m == r.m, f"seq {b}: m gpu={m} oracle={r.m}"
            assert list(out) == list(want), f"seq {b}: tokens gpu={list(out)} oracle={list(want)}"
            assert st == r.status, f"seq {b}: status gpu={st} oracle={r.status}"
        if gpu["diag"] is None:
            continue
        dg = gpu["diag"][b]
        if r.greedy:
            assert np.isnan(dg).all(), (b, dg)
            continue
        if check_probs:
            # p_i(d_i), q_i(d_i) do not depend on any decision: checked for every sequence
            pd, qd = draft_probs(wl, b, r.gamma)
            for i in range(g_all):
                gp, gq = dg[2 * i], dg[2 * i + 1]
                if i < r.gamma and not math.isnan(pd[i]):
                    assert abs(gp - pd[i]) <= PROB_TOL and abs(gq - qd[i]) <= PROB_TOL, \
                        f"seq {b} row {i}: p {gp} vs {pd[i]}, q {gq} vs {qd[i]}"
                else:
                    assert math.isnan(gp) and math.isnan(gq), (b, i, gp, gq)
        if same:
            assert abs(dg[2 * g_all] - r.mass) <= PROB_TOL, f"seq {b}: mass {dg[2 * g_all]} vs {r.mass}"
    return len(seqs), flagged, differ


def record(name, n, flagged, differ, **extra):
    """Append {workload, checked, flagged, differ} as one JSON line to the file named by the
    SPEC_PARITY_RECORD environment variable (nothing when it is unset), so that a test run
    leaves the count of sequences exempted from the bit-exact check."""
    path = os.environ.get("SPEC_PARITY_RECORD")
    if not path:
        return
    rec = {"workload": name, "checked": n, "flagged": len(flagged), "differ": len(differ),
           "flagged_seqs": list(map(int, flagged[:20])), "differ_seqs": list(map(int, differ[:20]))}
    rec.update(extra)
    with open(path, "a", encoding="utf-8") as f:
        f.write(json.dumps(rec) + "\n")
