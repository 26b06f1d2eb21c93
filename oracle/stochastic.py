"""Stochastic tree acceptance: speculative sampling at temperature T > 0,
generalised from a chain to a tree.

MineDraft summary (on a rejection, resample one token from
norm(max(0, p - q)); the default temperature is 1.0) and the NVIDIA
draft-length article (acceptance length AL in [1, 1 + D]); the tree form
follows the SwiftSpec summary, Figure 2 (the target picks one path of the
draft tree).

Readings (the pages give the chain's residual only):

* p_u = softmax(target_logits[u] / T) is the target's distribution after
  node u, q_u = softmax(draft_logits[u] / T) the draft's, from which u's
  children were drawn.
* At the current node u the children are tried in index order with a
  running target r (r = p_u first): child c (token t) is accepted iff
  U_acc[c] < r(t) / q_u(t), i.e. with probability min(1, r(t) / q_u(t));
  on a rejection r becomes norm(max(0, r - q_u)) and the next child is
  tried.  An accepted child becomes the current node (its r restarts at
  p_c).  When every child was rejected, or the node has none, one token is
  drawn from r by inverse transform with U_bonus[u]: the smallest v with
  r(0) + ... + r(v) > U_bonus[u].  Node 0 (the root, the last verified
  token) is always accepted.  Children drawn independently from q_u make
  the emitted token follow p_u exactly (recursive rejection sampling).
* If max(0, r - q_u) is all zero (r equals q_u in the arithmetic), r is
  kept: in exact arithmetic that case accepts every child.  A child whose
  draft probability is 0 in the arithmetic (underflow at a low temperature)
  is accepted iff its target probability is positive (an infinite ratio).
* The uniforms are inputs (the random numbers of the method), in [0, 1).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).
"""
from __future__ import annotations

import dataclasses
from typing import List

import numpy as np


def softmax_t(logits_row: np.ndarray, temperature: float) -> np.ndarray:
    z = np.asarray(logits_row, dtype=np.float64) / temperature
    e = np.exp(z - z.max())
    return e / e.sum()


def sample_inverse(r: np.ndarray, u: float) -> int:
    """Smallest v with r[0] + ... + r[v] > u * sum(r) (r need not be normalised)."""
    c = np.cumsum(np.asarray(r, dtype=np.float64))
    v = int(np.searchsorted(c, u * c[-1], side="right"))
    return min(v, len(c) - 1)


@dataclasses.dataclass
class StochasticResult:
    path: List[int]
    bonus: int

    @property
    def accept_len(self) -> int:
        return len(self.path)


def stochastic_accept(target_logits: np.ndarray, draft_logits: np.ndarray, tokens, parent, n: int,
                      temperature: float, u_acc, u_bonus) -> StochasticResult:
    """One request: target_logits / draft_logits [n][V] (row u = distributions
    after node u), u_acc / u_bonus [n] uniforms in [0, 1)."""
    children = [[] for _ in range(n)]
    for i in range(1, n):
        if int(parent[i]) >= 0:
            children[int(parent[i])].append(i)
    u, path = 0, [0]
    while True:
        r = softmax_t(target_logits[u], temperature)
        q = softmax_t(draft_logits[u], temperature)
        nxt = -1
        for c in children[u]:
            t = int(tokens[c])
            accept = (float(u_acc[c]) < r[t] / q[t]) if q[t] > 0 else r[t] > 0
            if accept:
                nxt = c
                break
            res = np.maximum(0.0, r - q)
            z = res.sum()
            if z > 0:
                r = res / z
        if nxt < 0:
            return StochasticResult(path, sample_inverse(r, float(u_bonus[u])))
        path.append(nxt)
        u = nxt
