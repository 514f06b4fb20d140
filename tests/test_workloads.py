"""Seeded synthetic input generator (CPU only)."""
import numpy as np

from speculative_decoding_verification_34_gb300 import workloads as W


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, 1.0078125 + 2 ** -10, -2.5, 3.0e38, np.inf],
                 dtype=np.float32)
    b = W.f32_to_bf16_bits(x)
    back = W.bf16_bits_to_f32(b)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to the even mantissa (1.0)
    assert back[0] == 1.0 and back[1] == 1.0
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties to even (1 + 2^-6)
    assert back[2] == 1.015625
    assert back[3] == 1.0078125 and back[4] == -2.5 and np.isinf(back[6])
    assert W.f32_to_bf16_bits(np.array([np.nan], np.float32))[0] == 0x7FC0
    # every bf16 value survives a round trip
    allb = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    f = W.bf16_bits_to_f32(allb)
    ok = ~np.isnan(f)
    assert np.array_equal(W.f32_to_bf16_bits(f)[ok], allb[ok])


def test_deterministic_and_shapes():
    a = W.small_fp32(seed=3)
    b = W.small_fp32(seed=3)
    c = W.small_fp32(seed=4)
    assert np.array_equal(a.target, b.target) and np.array_equal(a.u_sample, b.u_sample)
    assert not np.array_equal(a.target, c.target)
    assert a.target.shape == (8, 5, 1024) and a.draft.shape == (8, 4, 1024)
    assert a.target.dtype == np.float32 and a.draft_tokens.dtype == np.int32
    assert (a.u_accept >= 0).all() and (a.u_accept < 1).all()
    assert a.algorithmic_bytes() == 8 * 9 * 1024 * 4 and a.verified_rows() == 32


def test_greedy_planted_argmax_unique():
    wl = W.greedy_32k(seed=1)
    f = W.bf16_bits_to_f32(wl.target)
    top = f.max(axis=2)
    assert np.all(top == 19.0)
    assert np.all((f == 19.0).sum(axis=2) == 1)
    am = f.argmax(axis=2)[:, :5]
    rate = (am == wl.draft_tokens).mean()
    assert 0.7 < rate < 0.9


def test_ragged_padding_is_nan():
    wl = W.sampling_workload("t", cfg=9, seed=0, B=6, gmax=5, V=40, dtype="bf16",
                             target_sigma=3.0, draft_scale=1.0, draft_sigma=1.0,
                             temperature=0.7, num_draft=[0, 1, 5, 2, 3, 4],
                             greedy_mask=[1, 0, 0, 1, 0, 0], equal_mask=[0, 0, 1, 0, 0, 0])
    for b, g in enumerate(wl.num_draft):
        assert np.all(wl.target[b, g + 1:] == W.BF16_NAN)
        assert np.all(wl.draft[b, g:] == W.BF16_NAN)
        assert np.all(wl.draft_tokens[b, g:] == -1)
        assert np.all((wl.draft_tokens[b, :g] >= 0) & (wl.draft_tokens[b, :g] < 40))
    assert np.array_equal(wl.draft[2, :5], wl.target[2, :5])
    assert wl.temperature[0] == 0 and wl.temperature[3] == 0 and wl.temperature[1] > 0
    # greedy sequences draft the argmax of their own draft logits
    q = W.bf16_bits_to_f32(wl.draft[3, :2])
    assert list(wl.draft_tokens[3, :2]) == list(q.argmax(axis=1))
