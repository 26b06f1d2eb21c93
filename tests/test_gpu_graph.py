"""The whole verify step (attention, greedy acceptance, KV compaction) captured
in one CUDA graph: replays equal eager runs bit for bit, and follow changes to
the device inputs made between replays (per-request lengths, trees and tokens
live on the device; only maxima are baked into the launches)."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():   # on a GPU machine a missing library is an error, not a skip
    import speculative_decoding_tree_forward_gb300 as ts
else:
    ts = None
from gpu_util import attn_inputs, i32_dev  # noqa: E402


class Step:
    """Attention of a 128-row (tcgen05) case, acceptance over its own tree and
    the re-root + row moves of that tree over two layers of KV."""

    def __init__(self):
        dev = torch.device("cuda")
        self.attn_case = W.random_attn_case(70, num_req=4, hq=32, hkv=8, d=128, n_tree_max=32,
                                            prefix_range=(100, 1500))
        c = self.attn_case
        self.d = attn_inputs(c)
        self.out = torch.empty_like(self.d["q"])
        self.lse = torch.empty((c.num_req, c.num_q_heads, c.n_query), dtype=torch.float32, device=dev)
        self.aa = ts.attn_args(self.d["q"], self.d["k_cache"], self.d["v_cache"], self.d["prefix_len"],
                               self.d["n_tree"], self.d["parent"], self.out, self.lse, None, c.softmax_scale)
        self.aws = ts.new_workspace(ts.tree_attn_workspace_size(self.aa))

        acc = W.random_accept_case(71, num_req=4, n_tree_max=32, vocab=5000, p_accept=0.8)
        self.logits = torch.from_numpy(acc.logits).to(dev)
        self.tok, self.par, self.ntree = i32_dev(acc.tokens), i32_dev(acc.parent), i32_dev(acc.n_tree)
        self.res = {k: torch.empty(s, dtype=torch.int32, device=dev) for k, s in [
            ("argmax", (4, 32)), ("path", (4, 32)), ("accept_len", (4,)), ("bonus", (4,)),
            ("verified", (4, 33)), ("verified_len", (4,))]}
        self.ca = ts.accept_args(self.logits, self.tok, self.par, self.ntree, **self.res)
        self.cws = ts.new_workspace(ts.tree_accept_workspace_size(self.ca))

        g = torch.Generator(device=dev)
        g.manual_seed(72)
        self.prefix = i32_dev(np.array([40, 0, 77, 5], np.int32))
        self.k0 = [torch.randn((4, 200, 2, 64), generator=g, device=dev).to(torch.bfloat16) for _ in range(2)]
        self.v0 = [torch.randn((4, 200, 2, 64), generator=g, device=dev).to(torch.bfloat16) for _ in range(2)]
        self.k = [t.clone() for t in self.k0]
        self.v = [t.clone() for t in self.v0]
        self.kp, self.vp = ts.layer_pointer_table(self.k), ts.layer_pointer_table(self.v)
        self.new = {k: torch.empty(s, dtype=torch.int32, device=dev) for k, s in [
            ("new_prefix_len", (4,)), ("new_n_tree", (4,)), ("new_parent", (4, 32)), ("new_tokens", (4, 32)),
            ("src_rows", (4, 32))]}
        self.xa = ts.compact_args(self.kp, self.vp, 2, 2, 64, self.prefix, self.ntree, self.par, self.tok,
                                  self.res["verified"], self.res["verified_len"], self.new["new_prefix_len"],
                                  self.new["new_n_tree"], self.new["new_parent"], self.new["new_tokens"],
                                  self.new["src_rows"], 200)
        self.xws = ts.new_workspace(ts.tree_compact_workspace_size(self.xa))

    def restore(self):
        for t, t0 in zip(self.k + self.v, self.k0 + self.v0):
            t.copy_(t0)

    def run(self):
        ts.tree_attn_forward_args(self.aa, self.aws)
        ts.tree_accept_greedy_args(self.ca, self.cws)
        ts.tree_cache_compact_args(self.xa, self.xws)

    def results(self):
        torch.cuda.synchronize()
        r = {"out": self.out.view(torch.int16).clone(), "lse": self.lse.clone()}
        r.update({k: v.clone() for k, v in self.res.items()})
        r.update({k: v.clone() for k, v in self.new.items()})
        for i, t in enumerate(self.k + self.v):
            r["kv%d" % i] = t.view(torch.int16).clone()
        return r


def _same(a, b):
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_verify_step_replays_from_a_cuda_graph():
    s = Step()
    s.restore()
    s.run()
    eager = s.results()
    assert int(eager["accept_len"].min()) >= 1

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        s.run()
    for _ in range(2):
        s.restore()
        graph.replay()
        _same(eager, s.results())

    # new per-request inputs written into the same device buffers
    rng = np.random.default_rng(73)
    s.d["prefix_len"].copy_(i32_dev(rng.integers(0, int(s.attn_case.prefix_len.max()) + 1, size=4).astype(np.int32)))
    s.d["q"].copy_(torch.randn(s.d["q"].shape, device="cuda").to(torch.bfloat16))
    s.logits.copy_(torch.randn(s.logits.shape, device="cuda"))
    s.prefix.copy_(i32_dev(np.array([3, 90, 0, 150], np.int32)))
    s.restore()
    s.run()
    eager2 = s.results()
    s.restore()
    graph.replay()
    replay2 = s.results()
    _same(eager2, replay2)
    assert not torch.equal(eager["out"], replay2["out"])   # the replay read the new inputs
