"""CPU oracle for the accept step -- TEST INFRASTRUCTURE ONLY.

Only the test suite may import this module; the product (the CUDA library and
its binding) never loads it and shares no code with it.

What it computes (greedy acceptance of a verified draft tree, then KV-cache
compaction):

  * alphasignal.ai, "LMSYS Doubles Muse Spark Open Speed to 1,109 Tokens per
    Second", section "Draft and verify share one graph": the target model scores
    a 16-token tree in one pass; candidates it agrees with become output tokens,
    rejected branches are dropped; draft, verify and accept form one CUDA graph.
  * orcarouter.ai, "Muse Spark Open: 1,109 tokens/s is a kernel-level change",
    closing figure (the repository screenshot): decoding is greedy, at batch 1,
    and draft, verify and accept run as one CUDA graph per decode step.

Readings (the pages give no formula):
  * greedy = the target's choice after a tree node is the argmax of that node's
    logits; equal maxima resolve to the smallest vocabulary index and a NaN
    counts as larger than every number (numpy's argmax rule);
  * from the root, the walk moves to a child whose draft token equals the
    parent's argmax; among several such children the one with the smallest tree
    index; it stops at the first node with no such child;
  * the step emits the accepted children's tokens plus one "bonus" token, the
    argmax at the last accepted node;
  * tree token i's K/V rows sit at cache row pos0 + i during the verify step;
    compaction moves the j-th accepted node's rows to row pos0 + j in every
    layer, K and V, every KV head; no other row changes.
"""
from __future__ import annotations

import numpy as np

T = 16


def target_argmax(logits: np.ndarray) -> np.ndarray:
    """Per tree node, the vocabulary index of the largest logit (first of equal
    maxima; a NaN wins): numpy's argmax over each row."""
    lg = np.asarray(logits)
    return np.array([int(np.argmax(lg[i])) for i in range(lg.shape[0])], dtype=np.int64)


def greedy_accept(logits: np.ndarray, tokens, parent):
    """Greedy walk of the verified tree.

    logits: [16][vocab] target logits of the tree nodes; tokens: draft token of
    each node (tokens[0], the root, is not checked); parent: parent[0] == -1,
    0 <= parent[i] < i.  Returns (path, bonus, argmax): path = accepted node
    indices starting with the root, bonus = argmax at the last accepted node."""
    g = target_argmax(logits)
    path = [0]
    cur = 0
    while True:
        nxt = None
        for c in range(1, T):  # children in tree order: the smallest index wins
            if parent[c] == cur and int(tokens[c]) == int(g[cur]):
                nxt = c
                break
        if nxt is None:
            break
        path.append(nxt)
        cur = nxt
    return path, int(g[cur]), g


def compact_kv(k_caches, v_caches, pos0: int, path):
    """Copies of the per-layer caches ([n_kv_heads][max_ctx][head_dim]) with row
    pos0 + j replaced by the old row pos0 + path[j] for every accepted j."""
    out_k, out_v = [], []
    for kc, vc in zip(k_caches, v_caches):
        nk, nv = np.array(kc, copy=True), np.array(vc, copy=True)
        for j, node in enumerate(path):
            nk[:, pos0 + j, :] = kc[:, pos0 + node, :]
            nv[:, pos0 + j, :] = vc[:, pos0 + node, :]
        out_k.append(nk)
        out_v.append(nv)
    return out_k, out_v
