"""spec_verify_sample_static (the library's per-device static workspace, no allocation) gives
bit-identical results to spec_verify_sample with a caller-owned workspace, on two calls of
different sizes in a row.  Collected last, so it runs both after the other GPU tests and, on
its own, in a fresh process."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_34_gb300 import specverify as sv
from speculative_decoding_verification_34_gb300 import workloads as W
from tests.parity import dev

pytestmark = pytest.mark.gpu


def _outputs(wl):
    B, g = wl.B, wl.gmax
    return (torch.full((B, g + 1), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, 2 * g + 1), 1234.5, dtype=torch.float32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"))


def _run(wl, static):
    tgt, drf = dev(wl.target), dev(wl.draft)
    args = (tgt, drf, dev(wl.draft_tokens), dev(wl.num_draft), dev(wl.temperature),
            dev(wl.u_accept), dev(wl.u_sample))
    out, m, diag, st = _outputs(wl)
    if static:
        sv.spec_verify_sample_static(*args, out, m, diag=diag, status=st)
    else:
        ws = torch.zeros(sv.spec_verify_workspace_bytes(wl.B, wl.gmax, wl.V,
                                                        0 if wl.dtype == "bf16" else 1),
                         dtype=torch.uint8, device="cuda")
        sv.spec_verify_sample(*args, out, m, diag=diag, status=st, workspace=ws)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (out, m, diag.view(torch.int32), st)]


def test_static_workspace_matches_caller_workspace_two_calls():
    a = W.sampling_workload("static-a", cfg=31, seed=0, B=40, gmax=4, V=128256, dtype="bf16",
                            target_sigma=3.0, draft_scale=1.0, draft_sigma=1.0, temperature=0.8,
                            greedy_mask=(np.arange(40) % 5) == 0, equal_mask=(np.arange(40) % 7) == 3)
    b = W.sampling_workload("static-b", cfg=32, seed=1, B=9, gmax=3, V=50000, dtype="f32",
                            target_sigma=2.0, draft_scale=0.9, draft_sigma=0.5, temperature=1.2,
                            num_draft=np.array([3, 0, 2, 3, 1, 3, 3, 2, 3], np.int32))
    n0 = sv.spec_launch_count()
    for wl in (a, b):
        want = _run(wl, static=False)
        got = _run(wl, static=True)
        for name, x, y in zip(("out_tokens", "num_accepted", "diag", "status"), want, got):
            assert np.array_equal(x, y), (wl.name, name)
        assert (got[1] >= 0).all()
    assert sv.spec_launch_count() > n0
