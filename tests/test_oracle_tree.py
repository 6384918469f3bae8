"""Pins of the greedy tree-verify oracle: the pages' printed trees, the row convention, ties, and
"greedy tree verify emits exactly what plain greedy decoding emits" (Module 16 lesson, section
'Verify the Tree -- and Why It's Exact')."""
import json
import os

import numpy as np
import pytest

from oracle import oracle as O
from speculative_decoding_verification_spec_gb300 import synth as S

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def cartesian_tree(head_topw):
    """Tokens and parents of a Cartesian candidate tree in BFS order (test-side fixture)."""
    tokens, parents = [], []
    level = [-1]
    for heads in head_topw:
        nxt = []
        for p in level:
            for t in heads:
                tokens.append(t)
                parents.append(p)
                nxt.append(len(tokens) - 1)
        level = nxt
    return np.array(tokens, np.int32), np.array(parents, np.int32)


def one_hot_rows(argmaxes, V):
    x = np.full((len(argmaxes), V), -1.0)
    x[np.arange(len(argmaxes)), argmaxes] = 1.0
    return x


def test_medusa_tree_layout():
    g = gold("trees.json")["medusa_tree"]
    tok, par = cartesian_tree(g["head_topw"])
    assert tok.tolist() == g["tokens"] and par.tolist() == g["parents"]
    assert S.medusa_tree_parents([2, 2]).tolist() == g["parents"]
    paths = []
    for leaf in range(len(tok)):
        if leaf in par:
            continue
        path, i = [], leaf
        while i >= 0:
            path.append(int(tok[i]))
            i = par[i]
        paths.append(path[::-1])
    assert sorted(paths) == sorted(g["paths"])


def test_greedy_tree_example():
    g = gold("trees.json")["greedy_tree_verify"]
    chain = {int(k): v for k, v in g["next_token_map"].items()}
    tok, par = cartesian_tree(g["head_topw"])
    V = 8
    amax = [g["root_next"]] + [chain[int(t)] for t in tok]  # row 0 frontier, row i+1 node i
    logits = one_hot_rows(amax, V)[None]
    out = O.tree_verify_greedy(logits, par[None], tok[None])
    A = out["accepted_len"][0]
    assert A == len(g["accepted"])
    assert out["out_tokens"][0, :A].tolist() == g["accepted"]
    assert out["out_tokens"][0, :A + 1].tolist() == g["emitted"]
    assert np.all(out["out_tokens"][0, A + 1:] == -1)


def test_row_convention():
    g = gold("trees.json")["row_convention"]
    par = np.array(g["parents"], np.int32)
    V = 10
    tok = np.array([1, 2, 3, 4], np.int32)  # A, B, C, D
    # frontier predicts A; row of A predicts B; row of B predicts D (so C is wrong); row of D -> 9
    amax = [1, 2, 4, 7, 9]
    out = O.tree_verify_greedy(one_hot_rows(amax, V)[None], par[None], tok[None])
    assert out["accepted_len"][0] == 3
    assert out["out_tokens"][0, :4].tolist() == [1, 2, 4, 9]
    assert out["out_nodes"][0, :3].tolist() == [0, 1, 3]


def greedy_decode(table, last, steps):
    out = []
    for _ in range(steps):
        last = int(table[last])
        out.append(last)
    return out


def test_tree_emits_plain_greedy_decode():
    """25 random next-token tables and tree shapes; the target's argmax after a prefix depends on
    the prefix's last token (a next-token map, as in the lesson's toy target)."""
    rng = np.random.default_rng(12)
    for trial in range(25):
        V = int(rng.integers(3, 12))
        table = rng.integers(0, V, V)
        N = int(rng.integers(1, 30))
        par = np.array([int(rng.integers(-1, i)) for i in range(N)], np.int32)
        last = int(rng.integers(0, V))
        # node tokens: the greedy next token of its prefix with prob 0.7, else random
        tok = np.empty(N, np.int32)
        for i in range(N):
            prev = last if par[i] < 0 else tok[par[i]]
            tok[i] = table[prev] if rng.random() < 0.7 else rng.integers(0, V)
        amax = [table[last]] + [table[t] for t in tok]
        logits = one_hot_rows(amax, V)[None]
        out = O.tree_verify_greedy(logits, par[None], tok[None])
        A = out["accepted_len"][0]
        assert out["out_tokens"][0, :A + 1].tolist() == greedy_decode(table, last, A + 1)


def test_tree_ties_and_duplicates():
    V = 6
    # argmax ties go to the lowest index
    row = np.array([0.5, 2.0, 2.0, -1.0, 2.0, 0.0])
    logits = np.stack([row, row, row])[None]
    par = np.array([[-1, 0]], np.int32)
    tok = np.array([[1, 1]], np.int32)
    out = O.tree_verify_greedy(logits, par, tok)
    assert out["amax"][0].tolist() == [1, 1, 1]
    assert out["out_tokens"][0].tolist() == [1, 1, 1]
    # duplicate sibling tokens: both valid at equal depth -> the lower node index wins
    par = np.array([[-1, -1, 1]], np.int32)
    tok = np.array([[1, 1, 3]], np.int32)
    logits = np.stack([one_hot_rows([1, 5, 3, 2], V)])
    out = O.tree_verify_greedy(logits, par, tok)
    assert out["accepted_len"][0] == 2 and out["out_nodes"][0, :2].tolist() == [1, 2]
    par = np.array([[-1, -1]], np.int32)
    out = O.tree_verify_greedy(one_hot_rows([1, 5, 3], V)[None], par, np.array([[1, 1]], np.int32))
    assert out["out_nodes"][0, 0] == 0 and out["out_tokens"][0, :2].tolist() == [1, 5]


def test_tree_statuses():
    V = 5
    lg = np.tile(one_hot_rows([0, 1, 2], V)[None], (5, 1, 1))
    par = np.tile(np.array([[-1, 0]], np.int32), (5, 1))
    tok = np.tile(np.array([[0, 1]], np.int32), (5, 1))
    lg[0, 2, 3] = np.nan
    lg[1, 1, :] = -np.inf
    par[2, 1] = 1      # a node cannot be its own parent
    tok[3, 0] = 5      # token out of range
    out = O.tree_verify_greedy(lg, par, tok, max_out=3)
    np.testing.assert_array_equal(out["row_status"], [1, 1, 5, 3, 0])
    assert out["accepted_len"][4] == 2 and out["out_tokens"][4].tolist() == [0, 1, 2]
    ov = O.tree_verify_greedy(lg[4:], par[4:], tok[4:], max_out=2)
    assert ov["row_status"][0] == O.ROW_OVERFLOW and ov["accepted_len"][0] == -1
    # no valid node: the output is the frontier argmax alone
    out = O.tree_verify_greedy(lg[4:], par[4:], np.array([[3, 3]], np.int32))
    assert out["accepted_len"][0] == 0 and out["out_tokens"][0].tolist() == [0, -1, -1]


def test_synthetic_tree_shape():
    par = S.medusa_tree_parents((4, 4, 2, 2), 64)
    assert len(par) == 64
    depth = np.zeros(64, int)
    for i, p in enumerate(par):
        assert -1 <= p < i
        depth[i] = 1 if p < 0 else depth[p] + 1
    assert np.bincount(depth).tolist() == [0, 4, 16, 32, 12]


def test_linear_greedy_is_greedy_decoding():
    """A chain verified greedily emits what greedy decoding does: the drafted prefix that agrees
    with the target's greedy next tokens, then the target's next token ([M16] "Verify the Tree";
    greedy is the p/q rule with one-hot p, M7.1)."""
    rng = np.random.default_rng(21)
    V, gamma = 12, 6
    nxt = rng.integers(0, V, V)  # a context-free next-token table: the target's greedy step
    for trial in range(200):
        start = int(rng.integers(0, V))
        greedy = [start]
        for _ in range(gamma + 1):
            greedy.append(int(nxt[greedy[-1]]))
        m = int(rng.integers(0, gamma + 1))          # the draft follows greedy decoding m steps
        draft = greedy[1:1 + m] + [int((greedy[1 + j] + 1 + rng.integers(0, V - 1)) % V)
                                   for j in range(m, gamma)]
        prefix = [start] + draft
        rows = one_hot_rows([nxt[t] for t in prefix], V)  # row i: the greedy step after token i
        o = O.spec_verify_greedy(rows[None], np.array([draft], np.int32))
        assert o["accepted_len"][0] == m
        assert list(o["out_tokens"][0, : m + 1]) == greedy[1:m + 2]
        assert np.all(o["out_tokens"][0, m + 1:] == -1)
