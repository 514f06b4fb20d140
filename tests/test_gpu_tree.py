"""Greedy tree verification on the GPU (spec_verify_tree_greedy) against the float64 oracle:
bit-exact tokens, accepted counts, paths and status bits; chain trees against
spec_verify_greedy; the tutorial's §5.3 tree figure; invalid nodes; the scalar load path."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import specverify_oracle as O
from speculative_decoding_verification_34_gb300 import specverify as sv
from speculative_decoding_verification_34_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


def run_tree(wl, target=None, num_nodes="given"):
    B, n = wl.B, wl.nmax
    tgt = parity.dev(wl.target) if target is None else target
    nn = parity.dev(wl.num_nodes) if num_nodes == "given" else num_nodes
    ob, out = parity.padded((B, n + 1), torch.int32, parity.SENT_I)
    mb, m = parity.padded((B,), torch.int32, parity.SENT_I)
    pb, path = parity.padded((B, n), torch.int32, parity.SENT_I)
    sb, st = parity.padded((B,), torch.int32, parity.SENT_I)
    ws = torch.zeros(sv.spec_verify_workspace_bytes(B, n, wl.V, sv.SPEC_BF16 if wl.dtype == "bf16" else sv.SPEC_F32),
                     dtype=torch.uint8, device="cuda")
    sv.spec_verify_tree_greedy(tgt, parity.dev(wl.node_tokens), parity.dev(wl.node_parents), nn,
                               out, m, path, st, workspace=ws)
    torch.cuda.synchronize()
    assert bool((ws == 0).all()), "workspace not returned to zero"
    for buf, count in ((ob, B * (n + 1)), (mb, B), (pb, B * n), (sb, B)):
        assert parity.canary_ok(buf, count, parity.SENT_I), "output overrun"
    return out.cpu().numpy(), m.cpu().numpy(), path.cpu().numpy(), st.cpu().numpy()


def check_against_oracle(wl, gpu, num_nodes=None):
    out, m, path, st = gpu
    res = O.verify_tree_batch(wl.target, wl.dtype, wl.node_tokens, wl.node_parents,
                              wl.num_nodes if num_nodes is None else num_nodes)
    for b, r in enumerate(res):
        want_out = np.full(wl.nmax + 1, -1)
        want_out[: len(r.tokens)] = r.tokens
        want_path = np.full(wl.nmax, -1)
        want_path[: len(r.path)] = r.path
        assert int(m[b]) == r.m, (b, int(m[b]), r)
        assert list(out[b]) == list(want_out), (b, list(out[b]), r)
        assert list(path[b]) == list(want_path), (b, list(path[b]), r)
        assert int(st[b]) == r.status, (b, int(st[b]), r.status)
    return res


def test_random_trees_match_oracle():
    wl = W.tree_workload("tree-rand", cfg=61, seed=0, B=24, nmax=31, V=32000,
                         num_nodes=[31, 0, 1, 5, 31, 17, 31, 2, 30, 31, 12, 31, 31, 8, 31, 3,
                                    31, 31, 25, 31, 4, 31, 31, 31])
    res = check_against_oracle(wl, run_tree(wl))
    assert sum(r.m for r in res) > wl.B   # the planted trees do accept paths


def test_largest_trees_full_vocabulary():
    wl = W.tree_workload("tree-max", cfg=62, seed=1, B=4, nmax=63, V=128256, alpha=0.85, width=3)
    res = check_against_oracle(wl, run_tree(wl))
    assert max(r.m for r in res) >= 3


def test_chain_trees_equal_chain_verification():
    """A tree whose node j hangs below node j-1 is a chain: spec_verify_greedy's results."""
    g = W.greedy_planted_workload("tree-chain", cfg=63, seed=2, B=16, gmax=8, V=32000, alpha=0.8)
    chain = parity.run_gpu(g, mode="greedy")
    parents = np.tile(np.arange(g.gmax, dtype=np.int32), (g.B, 1))
    wl = W.TreeWorkload("chain-as-tree", "bf16", g.B, g.gmax, g.V, g.target, g.draft_tokens, parents,
                        g.num_draft.copy(), g.kv_len)
    out, m, path, st = run_tree(wl)
    assert np.array_equal(out, chain["out"]) and np.array_equal(m, chain["m"])
    assert np.array_equal(st, chain["status"])
    for b in range(g.B):
        assert list(path[b][: m[b]]) == list(range(1, m[b] + 1)) and (path[b][m[b]:] == -1).all()
    check_against_oracle(wl, (out, m, path, st))


def test_tree_figure_on_gpu():
    G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tree_figure.json"), encoding="utf-8"))
    names = G["nodes"]
    words = sorted(set(names) | {"<bonus>", "<other>", "root"})
    ids = {w: i for i, w in enumerate(words)}
    V, n = 64, len(names)
    cases = G["cases"]
    tgt = np.zeros((len(cases), n + 1, V), dtype=np.float32)
    for c, case in enumerate(cases):
        for after, nxt in case["target_greedy_after"].items():
            r = 0 if after == "root" else names.index(after) + 1
            tgt[c, r, ids[nxt]] = 1.0
    toks = np.tile(np.array([ids[w] for w in names], dtype=np.int32), (len(cases), 1))
    pars = np.tile(np.array(G["parents"], dtype=np.int32), (len(cases), 1))
    wl = W.TreeWorkload("figure", "f32", len(cases), n, V, tgt, toks, pars,
                        np.full(len(cases), n, dtype=np.int32), np.zeros(len(cases), np.int32))
    out, m, path, st = run_tree(wl)
    for c, case in enumerate(cases):
        assert [names[j - 1] for j in path[c][: m[c]]] == case["path"]
        assert list(out[c][: m[c] + 1]) == [ids[w] for w in case["emitted"]]
    check_against_oracle(wl, (out, m, path, st))


def test_invalid_nodes_and_counts():
    wl = W.tree_workload("tree-bad", cfg=64, seed=3, B=8, nmax=12, V=5000, alpha=0.9, width=2)
    wl.node_parents[0, 4] = 5          # node 5 names itself
    wl.node_parents[1, 2] = 7          # node 3 names a later node
    wl.node_parents[2, 0] = -1         # node 1 below nothing
    wl.node_tokens[3, :] = wl.V + 11   # every candidate outside the vocabulary
    wl.node_tokens[4, 0] = -3
    nn = wl.num_nodes.copy()
    nn[5], nn[6] = 40, -2              # clamped to 12 and 0
    check_against_oracle(wl, run_tree(wl, num_nodes=parity.dev(nn)), num_nodes=nn)


def test_misaligned_fp32_takes_scalar_path():
    wl = W.tree_workload("tree-f32", cfg=65, seed=4, B=6, nmax=20, V=3001, dtype="f32")
    base = run_tree(wl)
    flat = torch.from_numpy(np.concatenate([[0.0], wl.target.reshape(-1)]).astype(np.float32)).cuda()
    t_off = flat[1:].view(wl.B, wl.nmax + 1, wl.V)
    assert t_off.data_ptr() % 16 == 4
    moved = run_tree(wl, target=t_off)
    for x, y in zip(base, moved):
        assert np.array_equal(x, y)
    check_against_oracle(wl, moved)
