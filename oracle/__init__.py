"""CPU oracle for the tree verify / expand step -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct definitions in fp64 (numpy) and Python lists:

* ``oracle.tree``       -- ancestor sets, the tree mask, greedy acceptance,
                           re-root + KV-row compaction.
* ``oracle.attention``  -- tree-masked GQA attention with an explicit mask.
* ``oracle.stochastic`` -- stochastic tree acceptance (speculative sampling
                           with the residual norm(max(0, p - q)), per child).
* ``oracle.expand``     -- draft-side maximum-likelihood expansion (candidate
                           children from log-softmax, priority picks) and the
                           selection of the most promising subtree.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and it
shares no code, table or helper with the CUDA library: the two meet only in
the seeded inputs produced by ``workloads.py``.

Every function cites the passage of the source pages it restates.  The pages
are three web summaries: "SwiftSpec 논문 요약 -- Disaggregated Speculative
Decoding" (cited as *SwiftSpec summary*), "MineDraft 정리" (*MineDraft
summary*) and "Speculative Decoding으로 더 빠른 LLM 추론을 위한 AI 모델 공동
설계" (*NVIDIA draft-length article*).

Parity status: every function here is pinned by tests under ``tests/`` that
check it against the pages' worked figures (Figures 2, 3, 4 of the SwiftSpec
summary), closed forms and brute force.  Absolute attention values on a real
model are not available anywhere and are not claimed.
"""
from . import attention, expand, stochastic, tree  # noqa: F401
