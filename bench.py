"""Benchmark of the tree verify step on one GB300 (or N independent replicas).

One step = one pass of the whole hot path over one batch of the long-context
verify workload (4 requests, 32 q / 8 kv heads, d 128, prefix 32768, 32-node
trees, vocab 152064, 64 layers):

  1. tree-masked GQA attention of one layer (tree_attn_forward),
  2. greedy acceptance over the vocab logits (tree_accept_greedy),
  3. target-side re-root + KV compaction over 64 layers (tree_cache_compact),
  4. draft-side re-root + KV compaction of the 64-node draft trees over the
     draft cache's 64 layers, in the same launch as 3 (tree_cache_compact_batch:
     the two caches are disjoint; --serial-compaction makes two calls).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.  With torchrun and N > 1 every
rank runs its own replica of the workload (no data exchange: requests are
independent), and the value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tree tokens/s and achieved HBM GB/s (fraction of ~8 TB/s) per attention layer"
UNIT = "tree tokens/s"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="longctx_verify_b4_p32k",
                    choices=["longctx_verify_b4_p32k", "verify_b8_tree16", "chain_verify_b16_paged",
                             "expand_w8_prefix2048", "tree16_prefix128"])
    ap.add_argument("--layers", type=int, default=64)
    ap.add_argument("--force-path", type=int, default=0)
    ap.add_argument("--temperature", type=float, default=0.0,
                    help="> 0: stochastic acceptance at this temperature instead of greedy")
    ap.add_argument("--rope-theta", type=float, default=0.0,
                    help="rotate the queries at their tree positions with this RoPE base (0: off)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay of the step")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the flushed attention calls of the verify-b8 and paged chain workloads")
    ap.add_argument("--oracle-child", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--serial-compaction", action="store_true",
                    help="compact the target- and draft-side caches with two calls instead of one batched launch")
    return ap.parse_args()


# ---------------------------------------------------------------------------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Largest value over the ranks (the slowest replica's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(tokens_per_step, world, ms_max):
    """Whole-job throughput: every rank runs its own replica of the step, so the
    job verifies world x tokens_per_step tokens in the slowest rank's step time."""
    return tokens_per_step * world / (ms_max / 1e3)


# ---------------------------------------------------------------------------
class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    def __init__(self, index: int):
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={q}", "--format=csv,noheader",
                                          "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1].split()[0]), float(parts[2].split()[0]), parts[5:9]))
                except ValueError:
                    continue
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
def attn_algorithmic_bytes(case) -> int:
    """K and V rows each read once per (request, KV head), Q read, O and lse written, metadata."""
    keys = sum(int(case.prefix_len[b]) + int(case.n_tree[b]) for b in range(case.num_req))
    kv = keys * case.num_kv_heads * case.head_dim * 2 * 2
    qo = 2 * case.num_req * case.n_query * case.num_q_heads * case.head_dim * 2
    lse = case.num_req * case.num_q_heads * case.n_query * 4
    meta = case.num_req * (case.n_tree_max + 2) * 4
    if case.paged:
        meta += case.block_table.size * 4
    return kv + qo + lse + meta


# the sources that decide what the attention kernels read and write
ATTN_SOURCES = ("api.cu", "attn_common.cuh", "attn_merge.cu", "attn_mma.cu", "attn_tc.cu", "common.cuh", "internal.h",
                "tcgen05.cuh")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_tree_forward_gb300", "csrc")
    for name in ATTN_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, path: str):
    """Per-launch DRAM bytes of the attention kernels from a committed ncu summary, if still current."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t.get(workload, {}).get(path)
        if e and e.get("source_hash") == kernel_source_hash():
            return e["dram_bytes_per_launch"]
    except (OSError, ValueError):
        pass
    return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
def build_step(args, torch, ts, W, device):
    """Allocate the workload on the device and return (step_fn, info)."""
    wl = getattr(W, args.workload)
    kw = {"num_layers": args.layers} if args.workload.startswith("longctx") else {}
    w = wl(**kw)
    attn_inputs, i32_dev = W.attn_inputs, W.i32_dev
    stream = torch.cuda.current_stream()
    calls = []        # (name, fn) run in order each step
    info = {"workload": w.name, "attn_cases": w.attn}
    tokens_per_step = 0
    attn_bytes = 0
    attn_calls = []
    for case in w.attn:
        d = attn_inputs(case)
        out = torch.empty_like(d["q"])
        lse = torch.empty((case.num_req, case.num_q_heads, case.n_query), dtype=torch.float32, device=device)
        a = ts.attn_args(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"], out, lse,
                         d.get("block_table"), case.softmax_scale, args.force_path, 0, args.rope_theta)
        ws = ts.new_workspace(ts.tree_attn_workspace_size(a), device)
        attn_calls.append((a, ws, d, out, lse))
        tokens_per_step += case.num_req * case.n_query
        attn_bytes += attn_algorithmic_bytes(case)
    info["attn_bytes"] = attn_bytes
    info["attn_inputs"] = attn_calls
    launches = 2 * len(attn_calls)

    # draft-side iteration (config 2): each attention call queries the w nodes
    # an expansion step just added to the tree it reads; a subtree is
    # selected at the end; the tree is reset to its initial state first
    draft = None
    if w.draft is not None:
        D = w.draft
        tree = ts.DraftTree(D.num_req, D.parent.shape[1], D.k, device)
        for name in ("parent", "tokens", "weight", "cand_tok", "cand_lp", "cand_taken"):
            getattr(tree, name).copy_(torch.from_numpy(getattr(D, name)).to(device))
        n0 = torch.full((D.num_req,), D.n0, dtype=torch.int32, device=device)
        taken0 = tree.cand_taken.clone()
        tree.n_tree.copy_(n0)
        dlogits = [torch.from_numpy(x).to(device) for x in D.logits]
        added = [torch.full((D.num_req, D.w), -1, dtype=torch.int32, device=device) for _ in attn_calls]
        rows0 = torch.full((D.num_req, D.w), -1, dtype=torch.int32, device=device)
        exp_args = [ts.expand_args(tree, dlogits[max(e - 1, 0)], added[e - 1] if e > 0 else rows0, added[e])
                    for e in range(len(attn_calls))]   # expansion 1 queries no row: its logits are not read
        ews = ts.new_workspace(max(ts.tree_expand_workspace_size(x) for x in exp_args), device)
        sel_out = {"keep": torch.empty((D.num_req, D.bs), dtype=torch.int32, device=device),
                   "new_parent": torch.empty((D.num_req, D.bs), dtype=torch.int32, device=device),
                   "new_tokens": torch.empty((D.num_req, D.bs), dtype=torch.int32, device=device),
                   "new_weight": torch.empty((D.num_req, D.bs), dtype=torch.float32, device=device),
                   "n_sel": torch.empty(D.num_req, dtype=torch.int32, device=device)}
        sel = ts.select_args(tree.n_tree, tree.parent, tree.tokens, tree.weight, D.bs, sel_out)
        sws = ts.new_workspace(256, device)
        for a, *_ in attn_calls:   # the attention calls read the tree the expansions grow
            a.parent, a.n_tree = tree.parent.data_ptr(), tree.n_tree.data_ptr()
        draft = dict(tree=tree, n0=n0, taken0=taken0, exp_args=exp_args, ews=ews, sel=sel, sws=sws,
                     sel_out=sel_out, logits=dlogits, added=added)
        launches += 2 * len(attn_calls) + 1
        info["expand_logit_bytes"] = sum(x.nbytes for x in D.logits)

    acc_state = None
    if w.accept is not None:
        A = w.accept
        logits = torch.from_numpy(A.logits).to(device)
        # When the step's inputs are not flushed from L2 between steps (K/V
        # larger than L2), the acceptance reads one of several copies of the
        # logits in turn, so that every step streams them from DRAM.
        n_rep = 1 if attn_bytes < 2 * L2_BYTES else min(8, -(-3 * L2_BYTES // A.logits.nbytes))
        if A.logits.nbytes >= (8 << 20):
            n_rep = max(n_rep, 2)   # the end-to-end leg copies large logits into two device copies in turn
        reps = [logits] + [logits.clone() for _ in range(n_rep - 1)]
        tok = i32_dev(A.tokens)
        res = {k: torch.empty(s, dtype=torch.int32, device=device) for k, s in [
            ("argmax", (A.num_req, A.n_tree_max)), ("path", (A.num_req, A.n_tree_max)),
            ("accept_len", (A.num_req,)), ("bonus", (A.num_req,)), ("verified", (A.num_req, A.n_tree_max + 1)),
            ("verified_len", (A.num_req,))]}
        par = attn_calls[0][2]["parent"] if attn_calls else i32_dev(A.parent)
        ntree = attn_calls[0][2]["n_tree"] if attn_calls else i32_dev(A.n_tree)
        if args.temperature > 0:
            # stochastic acceptance: a draft that differs from the target by
            # N(0, 0.5^2) per logit, and the walk's uniforms (seeded inputs)
            g = torch.Generator(device=device)
            g.manual_seed(7)
            dlog = logits + 0.5 * torch.randn(logits.shape, generator=g, device=device)
            u_acc = torch.rand(tok.shape, generator=g, device=device)
            u_bon = torch.rand(tok.shape, generator=g, device=device)
            dreps = [dlog] + [dlog.clone() for _ in range(n_rep - 1)]
            aas = [ts.sample_args(x, y, tok, par, ntree, u_acc, u_bon, args.temperature, res)
                   for x, y in zip(reps, dreps)]
            aws = ts.new_workspace(ts.tree_accept_sample_workspace_size(aas[0]), device)
            acc_state = (aas, aws, logits, tok, res, "sample", [dlog, u_acc, u_bon])
            info["logits_keep"] = reps + dreps   # the copies the argument structs point at stay alive
            info["logits_sets"] = [[x, y] for x, y in zip(reps, dreps)]   # copy k: what the k-th call reads
            info["accept_bytes"] = 2 * A.logits.nbytes
        else:
            aas = [ts.accept_args(x, tok, par, ntree, **res) for x in reps]
            aws = ts.new_workspace(ts.tree_accept_workspace_size(aas[0]), device)
            acc_state = (aas, aws, logits, tok, res, "greedy", [])
            info["logits_keep"] = reps   # the copies the argument structs point at stay alive
            info["logits_sets"] = [[x] for x in reps]
        info["logits_copies"] = n_rep
        launches += 2
        info.setdefault("accept_bytes", A.logits.nbytes)

    comp_states = []
    if w.compact is not None and acc_state is not None:
        res = acc_state[4]
        for side, C in (("target", w.compact), ("draft", w.compact_draft)):
            if C is None:
                continue
            layers = w.num_layers
            case0 = w.attn[0]
            max_kv = int(C.prefix_len.max()) + C.n_tree_max
            hkv, d = case0.num_kv_heads, case0.head_dim
            g = torch.Generator(device=device)
            g.manual_seed(1 + len(comp_states))
            shape = (C.num_req, max_kv, hkv, d)
            kl, vl = [], []
            for li in range(layers):
                if side == "target" and li == 0 and not case0.paged and case0.max_kv_len == max_kv:
                    kl.append(attn_calls[0][2]["k_cache"])
                    vl.append(attn_calls[0][2]["v_cache"])
                    continue
                kl.append(torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16))
                vl.append(torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16))
            kp, vp = ts.layer_pointer_table(kl, device), ts.layer_pointer_table(vl, device)
            outs = {k: torch.empty(s, dtype=torch.int32, device=device) for k, s in [
                ("new_prefix_len", (C.num_req,)), ("new_n_tree", (C.num_req,)),
                ("new_parent", (C.num_req, C.n_tree_max)), ("new_tokens", (C.num_req, C.n_tree_max)),
                ("src_rows", (C.num_req, C.n_tree_max))]}
            P, N, par, tok = i32_dev(C.prefix_len), i32_dev(C.n_tree), i32_dev(C.parent), i32_dev(C.tokens)
            ca = ts.compact_args(kp, vp, layers, hkv, d, P, N, par, tok, res["verified"], res["verified_len"],
                                 outs["new_prefix_len"], outs["new_n_tree"], outs["new_parent"], outs["new_tokens"],
                                 outs["src_rows"], max_kv)
            cws = ts.new_workspace(ts.tree_compact_workspace_size(ca), device)
            comp_states.append((ca, cws, kl, vl, kp, vp, P, N, par, tok, outs, side))
            launches += 1  # re-root and row moves are one kernel

    # the step as phases: ("attn" | "accept" | "other", [calls]); attention
    # phases are the ones the roofline times
    phases = []
    if draft is not None:
        dt = draft
        phases.append(("other", [lambda: (dt["tree"].n_tree.copy_(dt["n0"]), dt["tree"].cand_taken.copy_(dt["taken0"]))]))
        for e, (a, ws, *_) in enumerate(attn_calls):
            phases.append(("other", [lambda x=dt["exp_args"][e]: ts.tree_expand_args(x, dt["ews"])]))
            phases.append(("attn", [lambda a=a, ws=ws: ts.tree_attn_forward_args(a, ws)]))
        phases.append(("other", [lambda: ts.tree_select_subtree_args(dt["sel"], dt["sws"])]))
    else:
        phases.append(("attn", [lambda a=a, ws=ws: ts.tree_attn_forward_args(a, ws) for a, ws, *_ in attn_calls]))
    if acc_state is not None:
        accept_call = ts.tree_accept_sample_args if acc_state[5] == "sample" else ts.tree_accept_greedy_args
        turn = [0]

        def accept_next():   # the next copy of the logits, in turn
            a = acc_state[0][turn[0] % len(acc_state[0])]
            turn[0] += 1
            accept_call(a, acc_state[1])
        phases.append(("accept", [accept_next]))
        info["accept_first"] = lambda: accept_call(acc_state[0][0], acc_state[1])
        info["accept_copy"] = lambda k: accept_call(acc_state[0][k], acc_state[1])
    if len(comp_states) == 2 and not args.serial_compaction:
        # the target- and draft-side caches and their metadata are disjoint:
        # both compactions run as one launch (tree_cache_compact_batch)
        batch_args, batch_ws = [st[0] for st in comp_states], [st[1] for st in comp_states]
        launches -= 1   # one kernel for both
        phases.append(("other", [lambda: ts.tree_cache_compact_batch_args(batch_args, batch_ws)]))
    elif comp_states:
        phases.append(("other", [lambda st=st: ts.tree_cache_compact_args(st[0], st[1]) for st in comp_states]))

    def step():
        for _, calls in phases:
            for f in calls:
                f()

    info.update(tokens_per_step=tokens_per_step, launches=launches, acc_state=acc_state, comp_states=comp_states,
                workload_obj=w, phases=phases, draft=draft)
    return step, info


def phase_device_times(info, torch, peak):
    """Device time per call of each phase of the step, from a CUDA graph of that
    phase alone replayed back to back between one pair of events.

    An event pair around a single launch adds a few microseconds to it (the
    launch after a recorded event starts only after that event, with no
    overlap of its set-up), and Python-side launches can fall behind
    microsecond kernels; replaying a graph of several calls leaves the
    kernels' own time and their programmatic-dependent overlap.  These
    figures are supplementary: the step times and the roofline above are the
    event-timed ones.  Inputs larger than L2 are read from DRAM; the draft
    workload's logits and K/V (a few MB) stay in L2 across replays.
    """
    stream = torch.cuda.current_stream()

    def graph_of(fn):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        return g

    def per_replay_us(g, n):
        vals = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(n):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            vals.append(a.elapsed_time(b) * 1e3 / n)
        return sorted(vals)[len(vals) // 2]

    out = {"method": "CUDA graph of one phase alone, replayed back to back; device microseconds per call"}
    phases = info["phases"]
    if info["draft"] is not None:
        reset = phases[0][1][0]
        exps = [calls[0] for kind, calls in phases[1:-1] if kind == "other"]
        attns = [calls[0] for kind, calls in phases if kind == "attn"]

        def seq(k, with_attn):
            def f():
                reset()
                for i in range(k):
                    exps[i]()
                    if with_attn:
                        attns[i]()
            return f
        t0 = per_replay_us(graph_of(seq(0, False)), 20)
        te = per_replay_us(graph_of(seq(len(exps), False)), 20)
        ta = per_replay_us(graph_of(seq(len(exps), True)), 20)
        out["expansion_us"] = (te - t0) / len(exps)
        out["attention_us"] = (ta - te) / len(attns)
        out["note"] = "expansion = candidate pass + step kernel; logits and K/V L2-resident across replays"
        return out
    attn = [f for kind, calls in phases if kind == "attn" for f in calls]
    reps = max(4, -(-4 * L2_BYTES // max(info["attn_bytes"], 1)))   # chained calls read more than L2 between reuses
    t = per_replay_us(graph_of(lambda: [f() for _ in range(reps) for f in attn]), 5) / (reps * len(attn))
    out["attention_us"] = t
    out["attention_frac"] = info["attn_bytes"] / len(attn) / (t / 1e6) / 1e9 / peak
    accept = [f for kind, calls in phases if kind == "accept" for f in calls]
    if accept:
        n = info.get("logits_copies", 1)
        out["acceptance_us"] = per_replay_us(graph_of(lambda: [accept[0]() for _ in range(n)]), 10) / n
    comp = [f for kind, calls in phases if kind == "other" for f in calls]
    if comp:
        out["compaction_us"] = per_replay_us(graph_of(lambda: [f() for _ in range(4) for f in comp]), 10) / 4
    return out


def e2e_measure(args, torch, ts, info, steps, warmup):
    """Same step through the public API with host (pinned) inputs copied in and results copied out every step.

    All host->device copies of a step go on a side stream, the small inputs
    (queries, tree metadata, draft tokens) first and the vocab logits (the bulk
    of the bytes) after them: the copy engine takes host->device copies in the
    order they are issued, so a small copy issued after the logits would wait
    for all of them.  The side stream starts a step's copies once the previous
    step's work on the main stream has finished with its inputs.  The
    logits go to one of two device copies in turn: step k + 1's logits are
    copied while step k computes (after the acceptance that last read that
    copy), so the link carries one step's inputs per step without pauses.
    The attention, which does not read the logits, starts as soon as the
    small inputs are in; the acceptance waits for its logits.  The results go
    back on the main stream.  A step with no large input and small results
    copies everything on the main stream.
    """
    small_in = [d["q"] for a, ws, d, out, lse in info["attn_inputs"]]
    if info["draft"] is not None:
        small_in += info["draft"]["logits"]   # draft logits of the nodes the expansions query
    acc = info["acc_state"]
    big_in = []
    if acc is not None:
        small_in.append(acc[3])               # draft tokens
        small_in += acc[6][1:]                # uniforms (sampling)
        big_in = [acc[2]] + acc[6][:1]        # target logits (+ draft logits, sampling)
    for st in info["comp_states"]:
        small_in += [st[8], st[9]]          # parent, tokens (tree metadata)
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())
    small_host = [pin(t) for t in small_in]
    big_host = [pin(t) for t in big_in]
    attn_outs = [o for *_, o, l in info["attn_inputs"]] + [l for *_, l in info["attn_inputs"]]
    outs = []
    if acc is not None:
        outs += list(acc[4].values())
    for st in info["comp_states"]:
        outs += list(st[10].values())
    if info["draft"] is not None:
        outs += list(info["draft"]["sel_out"].values())
    host_outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    host_attn_outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in attn_outs]
    h2d = sum(t.numel() * t.element_size() for t in small_host + big_host)
    d2h = sum(t.numel() * t.element_size() for t in host_outs + host_attn_outs)
    side = torch.cuda.Stream()
    back = torch.cuda.Stream()   # device->host copies of the attention results
    main = torch.cuda.current_stream()
    done = torch.cuda.Event()   # the main stream has finished with the step's inputs
    done.record(main)

    # A side stream pays when there is something to overlap: the logits with
    # the attention, or a step's results going out (1 MB or more) with the
    # next step's inputs coming in.  Otherwise its events cost more than it saves.
    use_side = bool(big_in) or d2h >= (1 << 20)
    # The attention results go back early, on a stream of their own, only
    # while a long host->device copy is running: for a short step the extra
    # stream and events cost more than the overlap saves.
    use_back = sum(t.numel() * t.element_size() for t in big_host) >= (8 << 20)

    # With two device copies of the large inputs (the logits), step k + 1's
    # copy crosses the link while step k computes: the copy engine is never
    # idle, and the step's period is the link time of its inputs.  Every step
    # still copies all of its inputs in and its results out.
    sets = info.get("logits_sets") or []
    dbl = use_side and bool(big_in) and len(sets) >= 2
    big_ready = [torch.cuda.Event(), torch.cuda.Event()]
    acc_done = [torch.cuda.Event(), torch.cuda.Event()]
    for ev in acc_done:
        ev.record(main)
    turn = {"k": 0, "primed": False}

    def copy_big(k):
        # step k's large inputs into device copy k % 2, once the acceptance
        # that read that copy (step k - 2) is done
        side.wait_event(acc_done[k % 2])
        with torch.cuda.stream(side):
            for h, dv in zip(big_host, sets[k % 2]):
                dv.copy_(h, non_blocking=True)
            big_ready[k % 2].record(side)

    def step():
        if not use_side:   # copy on the main stream
            for h, dv in zip(small_host, small_in):
                dv.copy_(h, non_blocking=True)
            for _, calls in info["phases"]:
                for f in calls:
                    f()
            for dv, h in zip(attn_outs + outs, host_attn_outs + host_outs):
                h.copy_(dv, non_blocking=True)
            return
        k = turn["k"]
        if dbl and not turn["primed"]:
            copy_big(k)
            turn["primed"] = True
        side.wait_event(done)
        with torch.cuda.stream(side):
            for h, dv in zip(small_host, small_in):
                dv.copy_(h, non_blocking=True)
            small = torch.cuda.Event()
            small.record(side)
            if not dbl:
                for h, dv in zip(big_host, big_in):
                    dv.copy_(h, non_blocking=True)
                big = torch.cuda.Event()
                big.record(side)
        if dbl:
            copy_big(k + 1)   # the next step's logits cross while this step computes
        main.wait_event(small)
        attn_left = sum(1 for kind, _ in info["phases"] if kind == "attn")
        back_done = None
        for kind, calls in info["phases"]:
            if kind == "accept":
                if dbl:
                    main.wait_event(big_ready[k % 2])
                    calls = [lambda: info["accept_copy"](k % 2)]
                else:
                    main.wait_event(big)
                    calls = [info["accept_first"]]   # the copy the host writes into
            for f in calls:
                f()
            if kind == "accept" and dbl:
                acc_done[k % 2].record(main)
            if kind == "attn" and use_back:
                attn_left -= 1
                if attn_left == 0:
                    # the attention results are final: they go back on their own
                    # stream, over the link's other direction, while the logits
                    # are still coming in
                    ready = torch.cuda.Event()
                    ready.record(main)
                    back.wait_event(ready)
                    with torch.cuda.stream(back):
                        for dv, h in zip(attn_outs, host_attn_outs):
                            h.copy_(dv, non_blocking=True)
                        back_done = torch.cuda.Event()
                        back_done.record(back)
        if not dbl:
            main.wait_event(big)
        if back_done is not None:
            main.wait_event(back_done)   # the next step's attention rewrites those outputs
        done.record(main)
        for dv, h in zip(outs if use_back else attn_outs + outs, host_outs if use_back else host_attn_outs + host_outs):
            h.copy_(dv, non_blocking=True)
        turn["k"] = k + 1

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        step()
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    return ms, h2d, d2h


# ---------------------------------------------------------------------------
SIDE_WORKLOADS = ("verify_b8_tree16", "chain_verify_b16_paged")
ATTN_EVENT_EVERY = 4   # steps between those whose attention calls are bracketed by events


def side_workloads(args, torch, ts, W, device, calls: int):
    """The attention call of the verify-b8 (64 q / 8 kv heads, 8 requests, 16-node trees, R = 128) and
    paged chain verify (16 requests, chains of 5, paged K/V) workloads, in the bench's own process: each
    call after an L2 flush (258 MB write, then 258 MB read), event-timed on the launching stream."""
    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    flush_r = torch.ones(2 * L2_BYTES // 4, dtype=torch.int32, device=device)
    peak, peak_kind = peaks()
    out = {}
    for name in SIDE_WORKLOADS:
        case = getattr(W, name)().attn[0]
        d = W.attn_inputs(case)
        o = torch.empty_like(d["q"])
        lse = torch.empty((case.num_req, case.num_q_heads, case.n_query), dtype=torch.float32, device=device)
        a = ts.attn_args(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"], o, lse,
                         d.get("block_table"), case.softmax_scale, args.force_path, 0, args.rope_theta)
        ws = ts.new_workspace(ts.tree_attn_workspace_size(a), device)
        for _ in range(max(args.warmup, 3)):
            ts.tree_attn_forward_args(a, ws)
        torch.cuda.synchronize()
        assert ts.read_device_error(ws) == 0
        clocks = Clocks(torch.cuda.current_device())
        time.sleep(0.2)
        evs = []
        for _ in range(calls):
            flush.zero_()
            flush_r.max()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ts.tree_attn_forward_args(a, ws)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        ms = [x.elapsed_time(y) for x, y in evs]
        # the same call chained back to back over copies of the K/V cache that
        # together exceed L2 (each call reads the copy least recently read),
        # events only at the ends: the launch of each call overlaps the
        # previous one's tail, as between the layers of a model
        kv_bytes = d["k_cache"].nbytes + d["v_cache"].nbytes
        n_copies = max(2, -(-4 * L2_BYTES // kv_bytes))
        copies = [(d["k_cache"], d["v_cache"])] + [(d["k_cache"].clone(), d["v_cache"].clone())
                                                   for _ in range(n_copies - 1)]
        chain_args = [ts.attn_args(d["q"], kc, vc, d["prefix_len"], d["n_tree"], d["parent"], o, lse,
                                   d.get("block_table"), case.softmax_scale, args.force_path, 0, args.rope_theta)
                      for kc, vc in copies]
        for x in chain_args:
            ts.tree_attn_forward_args(x, ws)
        torch.cuda.synchronize()
        n_chain = max(4 * n_copies, calls)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n_chain):
            ts.tree_attn_forward_args(chain_args[i % n_copies], ws)
        e1.record(stream)
        torch.cuda.synchronize()
        ck = clocks.stop()
        chain_ms = e0.elapsed_time(e1) / n_chain
        assert ts.read_device_error(ws) == 0
        mean_ms = sum(ms) / len(ms)
        nbytes = attn_algorithmic_bytes(case)
        path = ts.tree_attn_selected_path(a)
        achieved = nbytes / (mean_ms / 1e3) / 1e9
        out[name] = {"launch_ms": mean_ms, "launch_ms_median": statistics.median(ms), "calls": calls,
                     "algorithmic_bytes_per_launch": nbytes, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": measured_traffic(name, path), "attention_path": path,
                     "tree_tokens_per_s": case.num_req * case.n_query / (mean_ms / 1e3),
                     "l2": "flushed before every call (258 MB write, then 258 MB read), outside the call times",
                     "chained": {"launch_ms": chain_ms, "calls": n_chain, "kv_copies": n_copies,
                                 "achieved": nbytes / (chain_ms / 1e3) / 1e9,
                                 "frac": nbytes / (chain_ms / 1e3) / 1e9 / peak,
                                 "l2": "%d copies of the K/V cache (%.0f MB in all) read in turn, no flush"
                                       % (n_copies, n_copies * kv_bytes / 1e6)},
                     "clocks": ck}
        del d, o, lse, ws, copies, chain_args
    return out


# ---------------------------------------------------------------------------
class OracleSample:
    """One request of the long-context workload, processed completely by the CPU oracle.

    The work of one request of a step: fp64 attention of all 32 query heads x
    32 tree queries against 32800 keys, greedy acceptance of its 32-node tree
    over 152064 logits, the target-side re-root (32-node tree) and the
    draft-side re-root (the 64-node tree grown from it), and the out-of-place
    row compaction of K and V over every layer for both sides.  The inputs are
    drawn with the workload's shapes and recipe (seeded)."""

    def __init__(self, layers: int):
        import numpy as np

        import workloads as W
        from oracle import attention as OA
        self.layers = layers
        case = W.random_attn_case(0, num_req=1, hq=32, hkv=8, d=128, n_tree_max=32, prefix_range=(32768, 32768))
        self.case = case
        keys = 32768 + 32
        # widening the bf16 inputs to fp64 is input preparation, done once
        self.q = OA.bf16_bits_to_f64(case.q[0])
        self.k = OA.bf16_bits_to_f64(case.k[0, :keys])
        self.v = OA.bf16_bits_to_f64(case.v[0, :keys])
        self.acc = W.random_accept_case(0, num_req=1, n_tree_max=32, vocab=152064, p_accept=0.8, ragged_tree=False)
        rs = np.random.default_rng(1)
        self.dparent = W.grow_parents(rs, self.acc.parent[0], 32)
        grown = W.draft_tokens(rs, self.dparent, self.acc.planted[0], 152064, 0.8, peak_rows=32)
        self.dtokens = np.concatenate([self.acc.tokens[0], grown[32:]]).astype(np.int32)
        self.rows_t = np.zeros((keys, 8, 128), np.uint16)
        self.rows_d = np.zeros((32768 + 64, 8, 128), np.uint16)

    def run(self) -> float:
        """Wall time (s) of the oracle on the sample."""
        from oracle import attention as OA
        from oracle import tree as OT
        t0 = time.perf_counter()
        OA.tree_attention(self.q, self.k, self.v, 32768, 32, self.case.parent[0], 32, self.case.scale)
        r = OT.greedy_accept(self.acc.logits[0], self.acc.tokens[0], self.acc.parent[0], 32)
        rt = OT.reroot(self.acc.parent[0], self.acc.tokens[0], 32, 32768, r.verified)
        rd = OT.reroot(self.dparent, self.dtokens, 64, 32768, r.verified)
        for _ in range(self.layers):
            for _kv in range(2):
                OT.compact_rows(self.rows_t, 32768, rt.src)
                OT.compact_rows(self.rows_d, 32768, rd.src)
        return time.perf_counter() - t0


SAMPLE_TEXT = ("one request of the workload processed completely (32 tree tokens): fp64 attention of 32 q heads x 32 "
               "queries x 32800 keys, greedy acceptance over 152064 logits, target- and draft-side re-roots, and the "
               "out-of-place compaction of K and V over %d layers for both sides; tree tokens/s = 32 / sample time")


def oracle_sample_child(threads: int, repeats: int, layers: int):
    """Runs in a fresh process whose BLAS thread count was fixed by the environment: prints the sample times."""
    s = OracleSample(layers)
    times = [s.run() for _ in range(repeats)]
    print(json.dumps({"times": times, "threads": threads}))


def oracle_sample_times(threads: int, repeats: int, layers: int):
    """Times the oracle sample `repeats` times in a child process with `threads` BLAS threads."""
    env = dict(os.environ)
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = str(threads)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", str(threads), "--layers",
                        str(layers), "--steps", str(repeats)], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])["times"]


def cpu_oracle_sample(args):
    """The oracle on the sample, single-threaded and on all host cores, median of 3 wall-clock runs each."""
    if not args.workload.startswith("longctx"):
        return None
    cores = os.cpu_count() or 1
    one = statistics.median(oracle_sample_times(1, 3, args.layers))
    allc = statistics.median(oracle_sample_times(cores, 3, args.layers))
    return {"value": 32.0 / allc, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": SAMPLE_TEXT % args.layers + "; median of 3 runs, all cores (BLAS threads = cores)",
            "single_thread": {"value": 32.0 / one, "median_s": one, "cores": 1},
            "all_cores": {"value": 32.0 / allc, "median_s": allc, "cores": cores}}


def reference_arm(args):
    world, rank, local = dist_setup(args)
    if rank != 0:
        return
    if not args.workload.startswith("longctx"):
        print(json.dumps({"impl": "reference", "unavailable": "the CPU oracle sample is defined for the "
                          "long-context workload only"}))
        return
    s = OracleSample(args.layers)
    for _ in range(args.warmup):
        s.run()
    times = [s.run() for _ in range(args.steps)]
    total = sum(times)
    v = 32.0 * args.steps / total
    cores = os.cpu_count() or 1
    sample = ("per step: " + SAMPLE_TEXT % args.layers + "; BLAS on the default thread count of the host (%d cores)"
              % cores)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "tree_tokens_per_step": 32},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ---------------------------------------------------------------------------
def main():
    args = parse()
    if args.oracle_child:
        oracle_sample_child(args.oracle_child, args.steps, args.layers)
        return
    if args.impl == "reference":
        reference_arm(args)
        return
    import torch
    world, rank, local = dist_setup(args)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    import speculative_decoding_tree_forward_gb300 as ts
    import workloads as W

    step, info = build_step(args, torch, ts, W, device)
    info["step"] = step
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    for _, ws, *_ in info["attn_inputs"]:
        code = ts.read_device_error(ws)
        assert code == 0, f"device error word {code:#x}"

    # attention launches timed on the launching stream inside the timed region
    n_attn = len(info["attn_inputs"])
    n_phases = sum(1 for kind, _ in info["phases"] if kind == "attn")
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_phases)]
          for _ in range(args.steps)]
    clocks = Clocks(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # workloads whose K/V would stay in L2 get L2 flushed before every timed
    # step: a write larger than L2, then a read of another buffer larger than
    # L2, so the dirty lines of the write are written back before the step
    # rather than inside it.  The flush itself is outside the step times.
    flush = flush_r = None
    if info["attn_bytes"] < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
        flush_r = torch.ones(2 * L2_BYTES // 4, dtype=torch.int32, device=device)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    # An event recorded between two launches removes their programmatic-
    # dependent overlap, so the attention calls are bracketed by events on
    # every ATTN_EVENT_EVERY-th step only (each of those steps still times
    # every attention call it makes); the other steps run as a user's would.
    # Steps are bracketed by events only when a flush between them has to be
    # left out of the step time.
    timed = [i for i in range(args.steps) if i % ATTN_EVENT_EVERY == ATTN_EVENT_EVERY - 1] or [args.steps - 1]
    for _ in range(3):   # the GPU idled while the clock sampler started: warm it again, untimed
        if flush is not None:
            flush.zero_()
            flush_r.max()
        step()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
            flush_r.max()
            step_ev[i][0].record(stream)
        j = 0
        for kind, calls in info["phases"]:
            if kind == "attn" and i in timed:
                ev[i][j][0].record(stream)
            for f in calls:
                f()
            if kind == "attn" and i in timed:
                ev[i][j][1].record(stream)
                j += 1
        if flush is not None:
            step_ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ck = clocks.stop() if clocks else None
    if flush is None:
        ms = t_start.elapsed_time(t_end) / args.steps
    else:
        ms = sum(a.elapsed_time(b) for a, b in step_ev) / args.steps
    attn_ms = sum(a.elapsed_time(b) for i in timed for a, b in ev[i]) / len(timed) / n_attn
    ms_max = max_over_ranks(ms, world)

    # the same step captured once as a CUDA graph and replayed (launch
    # latency off the host; the kernels and their dependencies are the same)
    graph = None
    if not args.no_graph:
        # one captured step per copy of the logits; one step when L2 is flushed
        # before every replay (a second step in the graph would find the first's
        # inputs in L2)
        per_graph = info.get("logits_copies", 1) if flush is None else 1
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(per_graph):
                step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        replays = max(1, -(-args.steps // per_graph))
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
        barrier(world)
        for i in range(replays):
            if flush is not None:
                flush.zero_()
                flush_r.max()
            gev[i][0].record(stream)
            g.replay()
            gev[i][1].record(stream)
        torch.cuda.synchronize()
        g_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in gev) / (replays * per_graph), world)
        graph = {"ms_per_step": g_ms, "value": replica_value(info["tokens_per_step"], world, g_ms), "unit": UNIT}
        del g

    tokens = info["tokens_per_step"] * world
    value = replica_value(info["tokens_per_step"], world, ms_max)
    peak, peak_kind = peaks()
    attn_bytes = info["attn_bytes"] / n_attn
    achieved = attn_bytes / (attn_ms / 1e3) / 1e9
    path = ts.tree_attn_selected_path(info["attn_inputs"][0][0])

    # (workloads flushed between steps fit in L2: chained replays would re-read them from L2,
    # except the draft iteration, whose figures say so)
    phases_graph = (phase_device_times(info, torch, peak)
                    if not args.no_graph and (flush is None or info["draft"] is not None) else None)

    side = None
    if not args.no_workloads and args.workload.startswith("longctx"):
        side = side_workloads(args, torch, ts, W, device, max(20, min(args.steps * 5, 200)))

    e2e = None
    if not args.no_e2e:
        e2e_steps = max(10, min(args.steps, 200))
        e_ms, h2d, d2h = e2e_measure(args, torch, ts, info, e2e_steps, 3)
        e_ms = max_over_ranks(e_ms, world)
        e2e = {"value": tokens / (e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_oracle_sample(args)
    traffic = measured_traffic(args.workload, path)
    # mean acceptance length of the last step (the inputs are the same every step)
    acceptance = None
    if info["acc_state"] is not None:
        al = info["acc_state"][4]["accept_len"].float()
        acceptance = {"mean_accept_len": float(al.mean()),
                      "emitted_tokens_per_s": float(al.sum()) * world / (ms_max / 1e3)}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": info["workload"], "requests": info["attn_cases"][0].num_req,
                   "q_heads": info["attn_cases"][0].num_q_heads, "kv_heads": info["attn_cases"][0].num_kv_heads,
                   "head_dim": info["attn_cases"][0].head_dim, "tree_nodes": info["attn_cases"][0].n_tree_max,
                   "layers_compacted": args.layers if info["comp_states"] else 0,
                   "compaction": ("one launch for both caches" if len(info["comp_states"]) == 2
                                  and not args.serial_compaction else "one launch per cache"),
                   "rope_theta": args.rope_theta,
                   "acceptance": "stochastic, T = %g" % args.temperature if args.temperature > 0 else "greedy", "draft_expansions": len(info["draft"]["exp_args"]) if info["draft"] else 0, "attention_path": path,
                   "logits_copies": info.get("logits_copies", 1),
                   "l2": ("inputs larger than L2: %.0f MB of K/V read per step vs 129 MB L2; the acceptance "
                          "reads %d copies of the logits in turn" % (attn_bytes / 1e6, info.get("logits_copies", 1))
                          if flush is None else
                          "L2 flushed (258 MB write, then 258 MB read) before every timed step, outside the step times: "
                          "%.0f MB of K/V per step" % (attn_bytes / 1e6)),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": f"tree_attn_forward ({path} kernel + LSE merge)",
                     "algorithmic_bytes_per_launch": attn_bytes, "launch_ms": attn_ms,
                     "timed_launches": len(timed) * n_attn,
                     "events": f"attention calls of every {ATTN_EVENT_EVERY}th timed step bracketed by CUDA events"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": info["launches"] * args.steps,
        "graph": graph,
        "phases_graph": phases_graph,
        "clocks": ck,
        "acceptance": acceptance,
        "workloads": side,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
