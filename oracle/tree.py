"""Tree bookkeeping for speculative decoding, written as plain list walks.

Conventions (the pages leave these open; the readings are stated here):

* A draft tree of ``n`` nodes is a ``parent`` array: ``parent[i] = -1`` means
  node ``i`` hangs directly off the prefix tail, otherwise ``parent[i]`` is an
  earlier node (``parent[i] < i``): new leaves are appended after the nodes
  they extend (SwiftSpec summary, §3.1.3, Figure 3: t7..t10 follow t1..t6).
* The KV cache of a request holds ``P`` verified prefix rows followed by the
  ``n`` tree rows; tree node ``i`` lives in row ``P + i`` (SwiftSpec summary,
  §3.2, the prefix-cache / tree-cache invariant).
* Queries are the last ``n_query`` nodes of the tree.
"""
from __future__ import annotations

import dataclasses
from typing import List

import numpy as np


def check_tree(parent, n: int) -> None:
    for i in range(n):
        p = int(parent[i])
        assert -1 <= p < i, f"parent[{i}] = {p} violates -1 <= parent[i] < i"


def ancestors_or_self(parent, u: int) -> List[int]:
    """[u, parent[u], parent[parent[u]], ...] up to the prefix tail."""
    out = []
    while u >= 0:
        out.append(u)
        u = int(parent[u])
    return out


def depth(parent, u: int) -> int:
    return len(ancestors_or_self(parent, u)) - 1


def tree_mask(parent, prefix_len: int, n: int, n_query: int) -> np.ndarray:
    """Boolean [n_query][prefix_len + n] visibility matrix.

    SwiftSpec summary, §3.1.3, Figure 3: rows are the new leaves, columns are
    every key (prefix, existing tree and the new leaves themselves); a leaf
    sees the whole verified prefix and, inside the tree, exactly its
    ancestors and itself (t7 -> t1, t2, t4, t7).
    """
    check_tree(parent, n)
    assert 0 <= n_query <= n
    mask = np.zeros((n_query, prefix_len + n), dtype=bool)
    mask[:, :prefix_len] = True
    for r in range(n_query):
        u = n - n_query + r
        for a in ancestors_or_self(parent, u):
            mask[r, prefix_len + a] = True
    return mask


# ---------------------------------------------------------------------------
# greedy acceptance
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class AcceptResult:
    argmax: List[int]          # target argmax per node (lowest index on ties)
    path: List[int]            # accepted root path, node 0 first
    accept_len: int            # AL = len(path) = accepted drafts + 1
    bonus: int                 # target token after the last accepted node
    verified: List[int]        # tokens along the path, then the bonus (AL + 1 tokens)


def greedy_accept(logits: np.ndarray, tokens, parent, n: int) -> AcceptResult:
    """Greedy (temperature 0) verification of a draft tree.

    NVIDIA draft-length article, "Speculative Decoding 작동 원리" and the
    Acceptance Length definition: the target accepts draft tokens up to the
    first mismatch and adds one token of its own, so AL is in [1, 1 + D].
    SwiftSpec summary §3.1 / Figure 2: the target picks one path of the tree
    (target output (t1, t3, t6) = root, accepted t3, new token t6).

    Reading for trees: node 0 is the root (the last verified token, whose
    token is not checked); node i >= 1 is accepted iff its parent is accepted
    and token[i] equals the target argmax at its parent.  The result is the
    longest accepted root path; among equally long paths the one whose last
    node has the smallest index wins; argmax ties go to the lowest token id.
    An empty tree (n = 0) gives AL = 0 and bonus = -1.
    """
    check_tree(parent, n)
    if n == 0:
        return AcceptResult([], [], 0, -1, [])
    am = [int(np.argmax(logits[i])) for i in range(n)]   # first maximum on ties
    children = [[] for _ in range(n)]
    for i in range(1, n):
        if int(parent[i]) >= 0:
            children[int(parent[i])].append(i)
    accepted = {0}
    stack = [0]
    while stack:
        a = stack.pop()
        for c in children[a]:
            if int(tokens[c]) == am[a]:
                accepted.add(c)
                stack.append(c)
    best = min(accepted, key=lambda u: (-depth(parent, u), u))
    path = list(reversed(ancestors_or_self(parent, best)))
    bonus = am[best]
    return AcceptResult(am, path, len(path), bonus, [int(tokens[u]) for u in path] + [bonus])


# ---------------------------------------------------------------------------
# evolving tree cache: re-root and compaction
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class RerootResult:
    path: List[int]            # matched nodes, in walk order (promoted to the prefix)
    survivors: List[int]       # nodes kept as the new tree cache, increasing index
    src: List[int]             # path ++ survivors: old node feeding new row P + j
    new_prefix_len: int
    new_n_tree: int
    new_parent: List[int]
    new_tokens: List[int]


def reroot(parent, tokens, n: int, prefix_len: int, verified) -> RerootResult:
    """Walk the verified tokens down the tree and re-root.

    SwiftSpec summary, §3.2 (update procedure) and Figure 4: walk the tree
    along the verified tokens and re-root at the last one; if that token is a
    node of the tree, keep only its subtree (moved to sit right after the
    prefix), otherwise start a new tree.  Figure 2 / its walkthrough table:
    re-rooting at t6 reuses t6's subtree; a target token that is not in the
    tree (t16) reuses nothing.

    Steps: start at the prefix tail (cur = -1); for each verified token take
    the lowest-index child of cur carrying it; stop at the first token with no
    such child.  Matched nodes join the prefix in walk order.  If every
    verified token matched, the proper descendants of the last one survive
    (all nodes when nothing was verified); otherwise nothing survives.
    """
    check_tree(parent, n)
    cur = -1
    path: List[int] = []
    matched_all = True
    for tok in verified:
        cands = [c for c in range(n) if int(parent[c]) == cur and int(tokens[c]) == int(tok)]
        if not cands:
            matched_all = False
            break
        cur = min(cands)
        path.append(cur)
    if matched_all:
        survivors = [u for u in range(n) if u != cur and (cur == -1 or cur in ancestors_or_self(parent, u))]
    else:
        survivors = []
    new_index = {old: j for j, old in enumerate(survivors)}
    new_parent = [-1 if int(parent[old]) == cur else new_index[int(parent[old])] for old in survivors]
    new_tokens = [int(tokens[old]) for old in survivors]
    return RerootResult(path, survivors, path + survivors, prefix_len + len(path), len(survivors),
                        new_parent, new_tokens)


def compact_rows(rows: np.ndarray, prefix_len: int, src) -> np.ndarray:
    """Move tree rows so the kept ones sit right after the prefix (out of place).

    SwiftSpec summary, §3.2 and Figure 4: t12, t15 become prefix rows, t17,
    t18 move to the front of the tree cache, the rest are dropped.  ``rows``
    is one request's logical KV rows ``[rows][...]``; new row ``P + j`` takes
    old row ``P + src[j]``.  Rows below ``P`` are untouched; rows at or beyond
    ``P + len(src)`` keep whatever they held (their content is unspecified).
    """
    out = rows.copy()
    for j, s in enumerate(src):
        out[prefix_len + j] = rows[prefix_len + int(s)]
    return out
