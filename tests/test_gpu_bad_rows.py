"""Rows that define no distribution on the GPU: the sequence is marked SPEC_ST_BAD_ROW and its
step is well formed (drafts 0..m-1, then one id in [0, V)); every other sequence of the batch
stays equal to the oracle.  Untruncated: a row whose max is not finite (all -inf, a +inf) or
which holds a NaN.  Truncated entry point: a NaN logit is an id never kept (its key search counts
no NaN key), so only a row whose max over the other logits is not finite is marked.  Rows past
num_draft and greedy sequences are not marked."""
import numpy as np
import pytest
import torch

from oracle import specverify_oracle as O
from speculative_decoding_verification_34_gb300 import specverify as sv
from speculative_decoding_verification_34_gb300 import workloads as W
from tests import parity
from tests.test_gpu_truncated import run_truncated

pytestmark = pytest.mark.gpu

NEG_INF = int(W.f32_to_bf16_bits(np.array([-np.inf], np.float32))[0])
POS_INF = int(W.f32_to_bf16_bits(np.array([np.inf], np.float32))[0])
NAN = 0x7FC0


def planted():
    B, g = 10, 4
    wl = W.sampling_workload("bad-rows", cfg=81, seed=3, B=B, gmax=g, V=6000, dtype="bf16",
                             target_sigma=3.0, draft_scale=1.0, draft_sigma=0.8, temperature=0.9)
    wl.target[0, 1, :] = NEG_INF              # a target row, every logit -inf
    wl.draft[1, 0, :] = NEG_INF               # a draft row
    wl.target[2, 2, 1234] = NAN               # one NaN among finite logits
    wl.target[3, 0, 77] = POS_INF             # one +inf
    wl.target[4, g, :] = NEG_INF              # the bonus row
    wl.target[5, 0, :5000] = NEG_INF          # a NaN in a thread whose other ids are all -inf; max finite
    wl.target[5, 0, 17] = NAN
    wl.draft[8, 1, :] = NAN                   # a draft row of NaN only
    wl.draft[8, 1, 3] = NEG_INF
    wl.num_draft[6] = 2                       # a row past num_draft: not read
    wl.target[6, 3, :] = NEG_INF
    wl.temperature[7] = 0.0                   # greedy: an all -inf row keeps argmax id 0
    wl.target[7, 2, :] = NEG_INF
    return wl, {0, 1, 2, 3, 4, 5, 8}, {0, 1, 3, 4, 8}


def check_batch(wl, gpu, res, bad):
    n, flagged, differ = parity.compare(wl, gpu, res)
    marked = {b for b in range(wl.B) if int(gpu["status"][b]) & sv.ST_BAD_ROW}
    assert marked == bad, (marked, bad)
    assert {b for b, r in enumerate(res) if r.status & O.ST_BAD_ROW} == bad
    assert set(differ) <= bad, differ
    return n, flagged, differ


def test_untruncated_marks_rows_without_a_distribution():
    wl, bad, _ = planted()
    gpu = parity.run_gpu(wl)
    res = parity.oracle_results(wl)
    n, flagged, differ = check_batch(wl, gpu, res, bad)
    parity.record(wl.name, n, flagged, differ, entry="sample")


@pytest.mark.parametrize("top_k,top_p", [(None, None), (50, 0.9)])
def test_truncated_marks_rows_without_a_distribution(top_k, top_p):
    wl, _, bad = planted()
    B = wl.B
    tk = None if top_k is None else [top_k] * B
    tp = None if top_p is None else [top_p] * B
    gpu = run_truncated(wl, tk, tp)
    res = O.verify_batch(wl.target, wl.draft, wl.dtype, wl.draft_tokens, wl.num_draft, wl.temperature,
                         wl.u_accept, wl.u_sample, top_k=None if tk is None else np.asarray(tk),
                         top_p=None if tp is None else np.asarray(tp), nan_masked=True)
    gpu["diag"] = None   # p'(d), q'(d) are checked by the truncated tests
    n, flagged, differ = check_batch(wl, gpu, res, bad)
    parity.record(wl.name, n, flagged, differ, entry="sample_truncated")
