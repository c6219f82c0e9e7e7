"""Pins of the accept-step oracle (greedy tree walk + KV compaction) against
hand-derived cases and an independent brute-force characterisation."""
import itertools

import numpy as np
import pytest

from oracle import accept as acc

T = 16


def planted_logits(rng, choice, vocab=64):
    """Logits whose per-row maximum sits at choice[i] (all other values < 1 < 10)."""
    lg = rng.random((T, vocab), dtype=np.float64).astype(np.float32)
    for i, c in enumerate(choice):
        lg[i, c] = 10.0
    return lg


def test_chain_all_agree_accepts_everything():
    rng = np.random.default_rng(1)
    choice = rng.integers(0, 64, T)
    parent = [-1] + list(range(T - 1))
    tokens = [7] + [int(choice[i - 1]) for i in range(1, T)]
    path, bonus, g = acc.greedy_accept(planted_logits(rng, choice), tokens, parent)
    assert path == list(range(T))
    assert bonus == int(choice[T - 1])
    assert list(g) == [int(c) for c in choice]


def test_root_rejected_accepts_only_root():
    rng = np.random.default_rng(2)
    choice = np.full(T, 5)
    parent = [-1] + [0] * (T - 1)  # star
    tokens = [0] + [6] * (T - 1)   # no child carries the root's argmax (5)
    path, bonus, _ = acc.greedy_accept(planted_logits(rng, choice), tokens, parent)
    assert path == [0] and bonus == 5


def test_branching_follows_the_matching_child():
    # root -> {1, 2}; 1 -> {3, 4}; 2 -> {5}; 3 -> {6}
    parent = [-1, 0, 0, 1, 1, 2, 3] + [6] * (T - 7)
    choice = [11, 20, 30, 40, 0, 0, 50] + [0] * (T - 7)
    tokens = [0, 12, 11, 21, 20, 30, 40] + [99] * (T - 7)
    # argmax(root)=11 -> child 2 (token 11); argmax(2)=30 -> child 5; argmax(5)=0 -> none
    rng = np.random.default_rng(3)
    path, bonus, _ = acc.greedy_accept(planted_logits(rng, choice), tokens, parent)
    assert path == [0, 2, 5] and bonus == 0


def test_duplicate_siblings_take_the_smallest_index():
    # two children of the root carry the root's argmax; the later one has a longer
    # matching subtree, the walk still takes the earlier one
    parent = [-1, 0, 0, 2, 3] + [4] * (T - 5)
    choice = [9, 1, 4, 5, 6] + [0] * (T - 5)
    tokens = [0, 9, 9, 4, 5] + [63] * (T - 5)
    rng = np.random.default_rng(4)
    path, bonus, _ = acc.greedy_accept(planted_logits(rng, choice), tokens, parent)
    assert path == [0, 1] and bonus == 1


def test_argmax_ties_nan_and_signed_zero():
    lg = np.zeros((T, 12), np.float32) - 1.0
    lg[0, [3, 7]] = 2.0                  # equal maxima: first index
    lg[1, [5, 9]] = np.nan               # NaN beats every number, first NaN
    lg[1, 2] = np.inf
    lg[2, :] = -0.0
    lg[2, 4] = 0.0                       # -0.0 == +0.0: index 0 (first maximum)
    lg[3, :] = -np.inf
    lg[3, 11] = -1e30
    g = acc.target_argmax(lg)
    assert g[0] == 3 and g[1] == 5 and g[2] == 0 and g[3] == 11


def brute_force_path(lg, tokens, parent):
    """Independent characterisation: node v is accepted iff every edge p -> c on its
    root path has tokens[c] == choice(p) and no earlier sibling of c also does;
    choice(p) is the largest logit, smallest index (python max over (value, -index))."""
    V = lg.shape[1]
    choice = [max(range(V), key=lambda v: (float(lg[i, v]), -v)) for i in range(T)]

    def ok_edge(c):
        p = parent[c]
        if int(tokens[c]) != choice[p]:
            return False
        return not any(parent[s] == p and int(tokens[s]) == choice[p] for s in range(1, c))

    accepted = []
    for v in range(T):
        chain, x = [], v
        while x != 0:
            chain.append(x)
            x = parent[x]
        if all(ok_edge(c) for c in chain):
            accepted.append((len(chain), v))
    accepted.sort()
    depths = [d for d, _ in accepted]
    assert depths == list(range(len(depths)))  # one accepted node per depth: a chain
    return [v for _, v in accepted], choice[accepted[-1][1]]


@pytest.mark.parametrize("seed", range(40))
def test_walk_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    parent = [-1] + [int(rng.integers(0, i)) for i in range(1, T)]
    vocab = 3  # small vocabulary: frequent matches, duplicate siblings and ties
    lg = rng.integers(0, 3, (T, vocab)).astype(np.float32)
    tokens = [int(x) for x in rng.integers(0, vocab, T)]
    path, bonus, _ = acc.greedy_accept(lg, tokens, parent)
    bp, bb = brute_force_path(lg, tokens, parent)
    assert path == bp and bonus == bb


def test_compaction_moves_accepted_rows_only():
    rng = np.random.default_rng(5)
    hkv, ctx, hd, pos0 = 2, 40, 8, 20
    ks = [rng.integers(0, 2**16, (hkv, ctx, hd)).astype(np.uint16) for _ in range(3)]
    vs = [rng.integers(0, 2**16, (hkv, ctx, hd)).astype(np.uint16) for _ in range(3)]
    path = [0, 2, 5, 6, 11]
    nk, nv = acc.compact_kv(ks, vs, pos0, path)
    for l in range(3):
        for j, node in enumerate(path):
            assert np.array_equal(nk[l][:, pos0 + j], ks[l][:, pos0 + node])
            assert np.array_equal(nv[l][:, pos0 + j], vs[l][:, pos0 + node])
        untouched = [r for r in range(ctx) if not pos0 <= r < pos0 + len(path)]
        assert np.array_equal(nk[l][:, untouched], ks[l][:, untouched])
        assert np.array_equal(nv[l][:, untouched], vs[l][:, untouched])
    # an identity path (a chain accepted node by node) changes nothing
    ik, iv = acc.compact_kv(ks, vs, pos0, list(range(7)))
    assert all(np.array_equal(a, b) for a, b in itertools.chain(zip(ik, ks), zip(iv, vs)))


@pytest.mark.parametrize("seed", range(6))
def test_bench_accept_tokens_plant_the_requested_depth(seed):
    """bench.accept_tokens: the walk follows the first-child chain for `depth` nodes
    (or the whole chain when it is shorter) and stops there."""
    import bench
    rng = np.random.default_rng(500 + seed)
    parent = [-1] + [int(rng.integers(0, i)) for i in range(1, T)]
    choice = rng.integers(0, 50, T)
    lg = planted_logits(rng, choice, vocab=64)
    depth = int(rng.integers(0, 9))
    tokens, taken = bench.accept_tokens(choice, parent, depth)
    tokens = [t % 64 for t in tokens]
    path, _, _ = acc.greedy_accept(lg, tokens, parent)
    assert len(path) == taken + 1 and taken <= depth
    chain, cur = [0], 0
    for c in range(1, T):
        if parent[c] == cur:
            chain.append(c)
            cur = c
    assert path == chain[:taken + 1]
