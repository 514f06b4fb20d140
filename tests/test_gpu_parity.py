"""CUDA path vs the float64 oracle, through the C ABI (needs a GPU).

Bar: tokens, accepted counts and status bit-exact except for sequences where some decision
the oracle took sits within 1e-5 of its threshold (counted and reported); p(d), q(d) and the
residual mass within 1e-5 absolute.  Greedy results are bit-exact always.
"""
import numpy as np
import pytest
import torch
from scipy import stats

from oracle import specverify_oracle as O
from speculative_decoding_verification_34_gb300 import specverify as sv
from speculative_decoding_verification_34_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    from speculative_decoding_verification_34_gb300 import build
    build.build()
    sv.load_library()


def _check(wl, seqs=None, mode="auto", max_differ_frac=0.01, **kw):
    """Flagged sequences (an oracle decision within 1e-5 of its threshold) are counted and
    reported; among them the GPU may legitimately take the other branch, which is bounded
    here as a sanity check on the fp32 arithmetic (it is normally 0)."""
    gpu = parity.run_gpu(wl, mode=mode, **kw)
    res = parity.oracle_results(wl, seqs=seqs, mode=mode)
    n, flagged, differ = parity.compare(wl, gpu, res, seqs=seqs)
    print(f"{wl.name}: {n} sequences checked, {len(flagged)} flagged within 1e-5 margin "
          f"{flagged[:10]}, {len(differ)} of them differ {differ[:10]}")
    parity.record(wl.name, n, flagged, differ, entry="greedy" if mode == "greedy" else "sample")
    assert len(differ) <= max(1, int(max_differ_frac * n))
    return gpu, res


def test_small_fp32_workload():
    _check(W.small_fp32(seed=0))
    _check(W.small_fp32(seed=1))


def test_three_token_trials():
    """The worked example, 1e5 seeded trials in one batch: parity with the oracle on every
    trial, and the GPU's first emitted tokens follow p = (0.5, 0.3, 0.2)."""
    wl = W.three_token_workload(100_000, seed=0)
    gpu, res = _check(wl)
    counts = np.bincount(gpu["out"][:, 0], minlength=3)
    assert stats.chisquare(counts, np.array([0.5, 0.3, 0.2]) * counts.sum()).pvalue > 1e-3, counts


def test_greedy_workload_both_entry_points():
    wl = W.greedy_32k(seed=0)
    gpu, res = _check(wl, mode="greedy", max_differ_frac=0.0)
    # the same sequences through spec_verify_sample with temperature 0 give the same result
    wl2 = W.greedy_32k(seed=0)
    wl2.greedy_only = False
    wl2.draft = np.zeros((wl.B, wl.gmax, wl.V), np.uint16)
    gpu2 = parity.run_gpu(wl2, mode="sample")
    assert np.array_equal(gpu["out"], gpu2["out"]) and np.array_equal(gpu["m"], gpu2["m"])


def test_sampling_128k_workload():
    _check(W.sampling_128k(seed=0))


def test_mixed_152k_workload():
    _check(W.mixed_152k(seed=0))


def test_large_batch_workload_every_sequence():
    """B=1024 at full size on the GPU, every sequence checked against the oracle."""
    wl = W.large_batch_128k(seed=0)
    gpu = parity.run_gpu(wl)
    res = parity.oracle_results(wl)
    n, flagged, differ = parity.compare(wl, gpu, res)
    print(f"{wl.name}: {n} sequences, {len(flagged)} flagged, {len(differ)} differ")
    parity.record(wl.name, n, flagged, differ, entry="sample")
    assert n == wl.B and len(differ) <= max(1, n // 100)
    eq = np.arange(wl.B) % 16 == 0
    # q == p: every draft kept (ratio exactly 1), the bonus drawn, no status bits
    assert (gpu["m"][eq] == 4).all() and (gpu["status"][eq] == 0).all()
    assert np.isfinite(gpu["diag"][eq]).all()


@pytest.mark.parametrize("V", [1, 2, 3, 31, 1025, 4097, 50000])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_edge_vocab_sizes(V, dtype):
    g = [0, 1, 3, 2, 3]
    wl = W.sampling_workload(f"edge-V{V}", cfg=100 + V, seed=1, B=5, gmax=3, V=V, dtype=dtype,
                             target_sigma=2.0, draft_scale=1.0, draft_sigma=0.7,
                             temperature=[0.9, 1.0, 0.0, 1.3, 0.6], num_draft=g,
                             greedy_mask=[0, 0, 1, 0, 0])
    _check(wl)
    cl, chunk = sv.spec_verify_plan(V, sv.SPEC_BF16 if dtype == "bf16" else sv.SPEC_F32)
    assert chunk % 8 == 0 and cl * chunk >= V and (cl - 1) * chunk < V


def test_misaligned_rows_take_scalar_path():
    """A target buffer starting 2 bytes past a 16-byte boundary gives the same results."""
    wl = W.sampling_workload("misaligned", cfg=7, seed=3, B=6, gmax=4, V=9000, dtype="bf16",
                             target_sigma=3.0, draft_scale=1.0, draft_sigma=1.0, temperature=0.8)
    base = parity.run_gpu(wl)
    flat = torch.from_numpy(np.concatenate([[0], wl.target.reshape(-1)]).astype(np.uint16).view(np.int16))
    t_off = flat.view(torch.bfloat16).cuda()[1:].view(wl.B, wl.gmax + 1, wl.V)
    assert t_off.data_ptr() % 16 == 2
    moved = parity.run_gpu(wl, target=t_off)
    for k in ("out", "m", "status"):
        assert np.array_equal(base[k], moved[k]), k
    assert np.allclose(base["diag"], moved["diag"], atol=1e-6, equal_nan=True)


def test_invalid_inputs_set_status():
    wl = W.sampling_workload("bad", cfg=8, seed=0, B=8, gmax=4, V=3000, dtype="bf16",
                             target_sigma=2.0, draft_scale=1.0, draft_sigma=0.3, temperature=1.0)
    wl.draft_tokens[0, 0] = -5
    wl.draft_tokens[1, 2] = 3000
    wl.draft_tokens[2, 1] = 10 ** 9
    wl.num_draft[3] = -1
    wl.num_draft[4] = 9
    wl.temperature[5] = np.nan
    wl.temperature[6] = -1.0
    gpu, res = _check(wl)
    assert gpu["status"][0] & sv.ST_BAD_DRAFT and gpu["m"][0] == 0
    assert gpu["status"][3] == sv.ST_CLAMPED_GAMMA and gpu["m"][3] == 0
    assert gpu["status"][4] & sv.ST_CLAMPED_GAMMA


def test_greedy_ties_resolve_to_lowest_id():
    V = 270000
    cl, chunk = sv.spec_verify_plan(V)
    assert cl > 3
    rng = np.random.default_rng(9)
    t32 = rng.normal(0, 1, (3, 4, V)).astype(np.float32)
    # equal maxima in different blocks, in different threads of one block, and in one vector
    t32[0, 0, [5 + 3 * chunk, 7 + chunk, 2 * chunk + 9]] = 20.0
    t32[0, 1, [chunk + 300, chunk + 44]] = 20.0
    t32[0, 2, [17, 18, 16]] = 20.0
    t32[1, :, :] = 1.0                       # a constant row: id 0
    t32[2, :, :] = -np.inf                   # all -inf: id 0
    t32[2, :, [V - 1]] = -np.inf
    tgt = W.f32_to_bf16_bits(t32)
    wl = W.Workload("ties", "bf16", 3, 3, V, tgt, None, np.zeros((3, 3), np.int32),
                    np.full(3, 3, np.int32), np.zeros(3, np.float32), np.zeros((3, 3), np.float32),
                    np.zeros(3, np.float32), np.zeros(3, np.int32), greedy_only=True)
    wl.draft_tokens[0] = [7 + chunk, chunk + 44, 16]
    gpu, _ = _check(wl, mode="greedy", max_differ_frac=0.0)
    assert list(gpu["out"][0]) == [7 + chunk, chunk + 44, 16, int(np.argmax(t32[0, 3]))]


def test_masked_logits_and_extreme_uniforms():
    wl = W.sampling_workload("masked", cfg=10, seed=2, B=12, gmax=4, V=20000, dtype="bf16",
                             target_sigma=3.0, draft_scale=1.0, draft_sigma=1.0, temperature=0.9)
    rng = np.random.default_rng(4)
    ninf = W.f32_to_bf16_bits(np.array([-np.inf], np.float32))[0]
    for b in range(wl.B):
        mask = rng.random(wl.V) < 0.5
        mask[wl.draft_tokens[b]] = False        # drafts stay possible under q
        wl.target[b, :, mask] = ninf
        wl.draft[b, :, mask & (rng.random(wl.V) < 0.5)] = ninf
    one_minus = np.nextafter(np.float32(1), np.float32(0))
    wl.u_accept[0:3] = 0.0
    wl.u_accept[3:6] = one_minus
    wl.u_sample[0:6:2] = 0.0
    wl.u_sample[1:6:2] = one_minus
    _check(wl)


def test_q_equals_p_and_forced_rejection():
    """q == p: every draft kept whatever u; a forced rejection (bad id) meets R == 0 and
    falls back to p_m without NaN."""
    wl = W.sampling_workload("qp", cfg=11, seed=0, B=6, gmax=4, V=128256, dtype="bf16",
                             target_sigma=3.0, draft_scale=1.0, draft_sigma=1.0, temperature=1.0,
                             equal_mask=[1] * 6)
    wl.u_accept[:] = np.nextafter(np.float32(1), np.float32(0))
    wl.draft_tokens[5, 1] = -1
    gpu, res = _check(wl)
    assert (gpu["m"][:5] == 4).all()
    assert gpu["m"][5] == 1 and gpu["status"][5] == sv.ST_BAD_DRAFT | sv.ST_R_ZERO
    assert gpu["diag"][5][-1] == 0.0 and not np.isnan(gpu["diag"][:, :2]).any()


def test_max_gamma_and_single_sequence():
    wl = W.sampling_workload("g32", cfg=12, seed=0, B=3, gmax=32, V=5000, dtype="bf16",
                             target_sigma=1.0, draft_scale=1.0, draft_sigma=0.05, temperature=1.0)
    _check(wl)
    wl1 = W.sampling_workload("b1", cfg=13, seed=0, B=1, gmax=4, V=128256, dtype="bf16",
                              target_sigma=3.0, draft_scale=0.7, draft_sigma=1.0, temperature=0.8)
    _check(wl1)


def test_zero_gamma_batch():
    wl = W.sampling_workload("g0", cfg=14, seed=0, B=4, gmax=0, V=7000, dtype="f32",
                             target_sigma=2.0, draft_scale=1.0, draft_sigma=1.0, temperature=0.7)
    _check(wl)


def test_deterministic_repeat():
    wl = W.sampling_128k(seed=1)
    a = parity.run_gpu(wl)
    b = parity.run_gpu(wl)
    for k in ("out", "m", "status"):
        assert np.array_equal(a[k], b[k])
    assert np.array_equal(a["diag"].view(np.uint32), b["diag"].view(np.uint32))


def test_empty_batch_is_noop():
    t = torch.zeros((0, 5, 100), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((0, 5), dtype=torch.int32, device="cuda")
    n = sv.spec_launch_count()
    sv.spec_verify_greedy(t, torch.zeros((0, 4), dtype=torch.int32, device="cuda"), None, out,
                          torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert sv.spec_launch_count() == n


def test_commit_kv_lengths_matches_oracle():
    rng = np.random.default_rng(3)
    B, g, cap = 300, 6, 40
    m = rng.integers(0, g + 1, B).astype(np.int32)
    m[0], m[1] = -3, 99                           # clamped into [0, g]
    out = rng.integers(0, 1000, (B, g + 1)).astype(np.int32)
    t = rng.integers(512, 8193, B).astype(np.int32)
    dkv = t.copy()
    clen = rng.integers(0, cap, B).astype(np.int32)
    clen[2] = -1
    hist = np.full((B, cap), -1, np.int32)
    for proc in (False, True):
        T_, D_, H_, C_, S_ = (dev(t), dev(dkv), dev(hist), dev(clen), dev(np.zeros(B, np.int32)))
        sv.spec_commit_kv_lengths(dev(m), T_, D_, proc, dev(out), H_, C_, S_)
        torch.cuda.synchronize()
        mc = np.clip(m, 0, g)
        kv, dk, hh, cc, st = O.commit_kv_lengths(t, mc, proc, draft_kv_len=dkv, out_tokens=out,
                                                 history=hist, committed_len=clen)
        assert np.array_equal(T_.cpu().numpy(), kv) and np.array_equal(D_.cpu().numpy(), dk)
        assert np.array_equal(H_.cpu().numpy(), hh) and np.array_equal(C_.cpu().numpy(), cc)
        assert np.array_equal(S_.cpu().numpy(), st)
    # lengths only
    T_ = dev(t)
    sv.spec_commit_kv_lengths(dev(m), T_, None, True, gmax=g)
    torch.cuda.synchronize()
    assert np.array_equal(T_.cpu().numpy(), t + np.clip(m, 0, g) + 1)


def test_binding_rejects_bad_tensors():
    wl = W.small_fp32(seed=0)
    with pytest.raises(ValueError):
        sv.spec_verify_greedy(torch.zeros((2, 3, 4)), torch.zeros((2, 2), dtype=torch.int32),
                              None, torch.zeros((2, 3), dtype=torch.int32), torch.zeros(2, dtype=torch.int32))
    with pytest.raises(TypeError):
        t = dev(wl.target).double()
        sv.spec_verify_greedy(t, dev(wl.draft_tokens), None,
                              torch.zeros((8, 5), dtype=torch.int32, device="cuda"),
                              torch.zeros(8, dtype=torch.int32, device="cuda"))


def dev(a):
    return parity.dev(a)


def test_workspace_reuse_across_sizes():
    """One zero-filled workspace serves calls of different sizes in any order."""
    big = W.sampling_workload("ws-big", cfg=15, seed=0, B=96, gmax=6, V=40000, dtype="bf16",
                              target_sigma=3.0, draft_scale=1.0, draft_sigma=1.0, temperature=0.9)
    small = W.sampling_workload("ws-small", cfg=16, seed=0, B=5, gmax=2, V=3000, dtype="bf16",
                                target_sigma=3.0, draft_scale=1.0, draft_sigma=1.0, temperature=1.1)
    mid = W.sampling_workload("ws-mid", cfg=17, seed=0, B=40, gmax=8, V=9000, dtype="bf16",
                              target_sigma=3.0, draft_scale=1.0, draft_sigma=1.0, temperature=0.7,
                              greedy_mask=(np.arange(40) % 3) == 0)
    n = max(sv.spec_verify_workspace_bytes(w.B, w.gmax, w.V) for w in (big, small, mid))
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    for wl in (small, big, mid, small, big):
        B, g = wl.B, wl.gmax
        out = torch.empty((B, g + 1), dtype=torch.int32, device="cuda")
        macc = torch.empty(B, dtype=torch.int32, device="cuda")
        st = torch.empty(B, dtype=torch.int32, device="cuda")
        dg = torch.empty((B, 2 * g + 1), dtype=torch.float32, device="cuda")
        sv.spec_verify_sample(dev(wl.target), dev(wl.draft), dev(wl.draft_tokens), dev(wl.num_draft),
                              dev(wl.temperature), dev(wl.u_accept), dev(wl.u_sample), out, macc, dg, st,
                              workspace=ws)
        torch.cuda.synchronize()
        assert bool((ws == 0).all())
        gpu = {"out": out.cpu().numpy(), "m": macc.cpu().numpy(), "status": st.cpu().numpy(),
               "diag": dg.cpu().numpy()}
        res = parity.oracle_results(wl)
        _, _, differ = parity.compare(wl, gpu, res)
        assert len(differ) <= 1


def test_batch_spanning_several_launches():
    """A batch larger than one grid runs as several launches over consecutive sequence ranges
    (at V = 64, gamma = 2: about 49,000 sampling sequences per launch on a 152-SM GPU, 65,535
    greedy ones).  Every sequence's step is well formed; the sequences at both ends of every
    launch and a sample elsewhere equal the oracle; the workspace returns to zero."""
    B = 70000
    wl = W.sampling_workload("multi-launch", cfg=91, seed=0, B=B, gmax=2, V=64, dtype="bf16",
                             target_sigma=2.0, draft_scale=1.0, draft_sigma=0.7, temperature=1.0,
                             greedy_mask=(np.arange(B) % 11) == 0)
    n0 = sv.spec_launch_count()
    gpu = parity.run_gpu(wl)
    assert sv.spec_launch_count() - n0 >= 2      # the batch did not fit one grid
    out, m = gpu["out"], gpu["m"]
    assert ((m >= 0) & (m <= 2)).all()
    for b in range(0, B, 997):
        assert list(out[b, :m[b]]) == list(wl.draft_tokens[b, :m[b]]) and 0 <= out[b, m[b]] < wl.V
    rng = np.random.default_rng(0)
    seqs = set(range(0, 40)) | set(range(48960, 49040)) | set(range(B - 40, B))
    seqs |= set(int(x) for x in rng.choice(B, 1200, replace=False))
    seqs = sorted(seqs)
    n, flagged, differ = parity.compare(wl, gpu, parity.oracle_results(wl, seqs), seqs)
    parity.record(wl.name, n, flagged, differ, entry="sample")
    assert len(differ) <= max(1, n // 100), differ
    # the greedy-only kernel: 65,535 sequences per launch
    g = W.greedy_planted_workload("multi-launch-g", cfg=92, seed=0, B=B, gmax=2, V=64, alpha=0.8)
    n0 = sv.spec_launch_count()
    gg = parity.run_gpu(g, mode="greedy")
    assert sv.spec_launch_count() - n0 >= 2
    seqs = sorted(set(range(0, 40)) | set(range(65500, 65570)) | set(range(B - 40, B)) |
                  set(int(x) for x in rng.choice(B, 1200, replace=False)))
    n, flagged, differ = parity.compare(g, gg, parity.oracle_results(g, seqs, mode="greedy"), seqs)
    parity.record(g.name, n, flagged, differ, entry="greedy")
    assert not differ
