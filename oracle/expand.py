"""Draft-side tree growth: maximum-likelihood expansion and subtree selection.

SwiftSpec summary, §3.1.1 (the draft worker's iteration, Algorithm 1: Expand
the w most probable leaves d times while the target verifies, then Select
the most promising subtree of size bs) and §3.1.3 (maximum-likelihood
expansion: a node's value is the log-softmax probability of its token, its
weight the sum of the values from the root, and the leaves to expand come
from a priority queue); Figure 2 (bs = 4, d = 3, w = 2: six nodes t7..t12
grow during one verification, two per expansion).

Readings (the pages leave these open; each is restated where it is used):

* The root's weight is its input weight (0 for a fresh root: the last
  verified token).  The weight of a child is its parent's weight plus the
  child token's log-softmax value under the draft model run on the parent.
* A node that has been run through the draft model offers its k most
  probable tokens (ties: lower token id) as candidate children, in that
  order.  Its candidates are known once the caller passes its logits.
* One expansion step adds w nodes: w times, the candidate of largest weight
  over all nodes' next untaken candidates becomes a new node (appended with
  that parent, token and weight).  A node's candidates are taken in order
  (they have decreasing weights), so one node may give several children in
  a step.  Ties between nodes go to the lower node index.  Growth stops at
  the tree's capacity or when no candidate is left.  Figure 2's count (six
  nodes in d = 3 steps of w = 2) agrees.
* The w new nodes are the next draft queries (the non-square mask of
  Figure 3); their logits give their candidates at the next step.
* "Most promising subtree of size bs": the bs nodes of largest weight (ties:
  lower index), kept in index order with parents remapped.  Values are
  log-probabilities (<= 0), so a child never outweighs its parent, and a tie
  goes to the parent's smaller index: the set holds every selected node's
  parent, i.e. it is a subtree containing the root.  Among all subtrees of
  bs nodes containing the root it maximises the sum of exp(weight), the
  expected number of accepted nodes when a draft probability is read as an
  acceptance probability.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence, Tuple

import numpy as np


def draft_candidates(logits_row: np.ndarray, k: int) -> List[Tuple[int, float]]:
    """The k most probable tokens of one draft distribution with their
    log-softmax values, in decreasing order (ties: lower token id)."""
    x = np.asarray(logits_row, dtype=np.float64)
    m = float(x.max())
    lse = m + float(np.log(np.sum(np.exp(x - m))))
    order = np.lexsort((np.arange(x.size), -x))[:k]   # primary: larger logit; then lower token
    return [(int(v), float(x[v] - lse)) for v in order]


@dataclasses.dataclass
class DraftTree:
    """One request's draft tree with each node's candidate children."""
    parent: List[int]
    tokens: List[int]
    weight: List[float]
    cand: List[List[Tuple[int, float]]]   # per node: (token, log-prob) in decreasing order; [] = not run yet
    taken: List[int]                       # per node: candidates already turned into children

    @property
    def n(self) -> int:
        return len(self.parent)


def expand_step(tree: DraftTree, new_rows: Sequence[int], logits: np.ndarray, w: int, k: int,
                capacity: int) -> List[int]:
    """One expansion step, in place.  ``new_rows[r]`` is the node whose draft
    logits are ``logits[r]`` (-1: no row); those nodes get their candidates.
    Returns the nodes added (at most w), in the order they were added."""
    for r, u in enumerate(new_rows):
        if u < 0:
            continue
        tree.cand[u] = draft_candidates(logits[r], k)
        tree.taken[u] = 0
    added = []
    for _ in range(w):
        if tree.n >= capacity:
            break
        best, best_w = -1, -np.inf
        for u in range(tree.n):   # each node's next untaken candidate; ties: lower node index
            if tree.taken[u] < len(tree.cand[u]):
                cw = tree.weight[u] + tree.cand[u][tree.taken[u]][1]
                if cw > best_w:
                    best, best_w = u, cw
        if best < 0:
            break
        tok = tree.cand[best][tree.taken[best]][0]
        tree.taken[best] += 1
        tree.parent.append(best)
        tree.tokens.append(tok)
        tree.weight.append(best_w)
        tree.cand.append([])
        tree.taken.append(0)
        added.append(tree.n - 1)
    return added


@dataclasses.dataclass
class SelectResult:
    keep: List[int]          # old node indices, increasing
    parent: List[int]        # remapped parents (-1: hangs off the prefix tail)
    tokens: List[int]
    weight: List[float]


def select_subtree(parent: Sequence[int], tokens: Sequence[int], weight: Sequence[float], n: int,
                   bs: int) -> SelectResult:
    """The bs nodes of largest weight (ties: lower index), in index order."""
    order = sorted(range(n), key=lambda i: (-float(weight[i]), i))[:bs]
    keep = sorted(order)
    newidx = {old: j for j, old in enumerate(keep)}
    new_parent = []
    for i in keep:
        p = int(parent[i])
        assert p < 0 or p in newidx, "selected set is not closed under parent"
        new_parent.append(newidx[p] if p >= 0 else -1)
    return SelectResult(keep, new_parent, [int(tokens[i]) for i in keep], [float(weight[i]) for i in keep])
