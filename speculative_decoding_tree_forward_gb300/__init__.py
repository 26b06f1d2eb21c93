"""Python binding of ``libtreespec.so`` (the tree verify / expand step, sm_103a).

Argument marshalling only: every function below fills the C structs declared
in ``include/treespec.h`` from torch tensors (device pointers, sizes) and calls
the C entry point of the same name on the current CUDA stream.  All
computation happens in the library's CUDA kernels.  Importing this package
fails loudly when the library has not been built
(``python speculative_decoding_tree_forward_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtreespec.so")

TS_OK, TS_ERR_INVALID_ARG, TS_ERR_UNSUPPORTED, TS_ERR_CUDA, TS_ERR_WORKSPACE = range(5)
TS_KV_CONTIGUOUS, TS_KV_PAGED = 0, 1
TS_DEVERR_BAD_PARENT, TS_DEVERR_BAD_LENGTH, TS_DEVERR_BAD_BLOCK, TS_DEVERR_TIMEOUT = 1, 2, 4, 8
TS_DEVERR_BAD_TOKEN = 16
TS_DEVERR_BAD_WORKSPACE = 32
TS_MAX_TREE = 128

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python speculative_decoding_tree_forward_gb300/build.py` (needs nvcc)")
_lib = ctypes.CDLL(LIB_PATH)

_i32 = ctypes.c_int
_vp = ctypes.c_void_p


class AttnArgs(ctypes.Structure):
    _fields_ = [("num_requests", _i32), ("num_q_heads", _i32), ("num_kv_heads", _i32), ("head_dim", _i32),
                ("n_tree_max", _i32), ("n_query", _i32), ("max_kv_len", _i32), ("kv_layout", _i32),
                ("page_size", _i32), ("max_blocks_per_req", _i32), ("num_blocks", _i32),
                ("prefix_len", _vp), ("n_tree", _vp), ("parent", _vp), ("q", _vp), ("k_cache", _vp),
                ("v_cache", _vp), ("block_table", _vp), ("out", _vp), ("lse", _vp),
                ("softmax_scale", ctypes.c_float), ("force_path", _i32), ("num_ctas", _i32),
                ("rope_theta", ctypes.c_float), ("wait_limit_ns", ctypes.c_uint)]


class AcceptArgs(ctypes.Structure):
    _fields_ = [("num_requests", _i32), ("n_tree_max", _i32), ("vocab", _i32), ("logits", _vp),
                ("tokens", _vp), ("parent", _vp), ("n_tree", _vp), ("argmax", _vp), ("path", _vp),
                ("accept_len", _vp), ("bonus", _vp), ("verified", _vp), ("verified_len", _vp)]


class CompactArgs(ctypes.Structure):
    _fields_ = [("num_requests", _i32), ("n_tree_max", _i32), ("m_max", _i32), ("num_layers", _i32),
                ("num_kv_heads", _i32), ("head_dim", _i32), ("elem_bytes", _i32), ("kv_layout", _i32),
                ("max_kv_len", _i32), ("page_size", _i32), ("max_blocks_per_req", _i32), ("num_blocks", _i32),
                ("k_layers", _vp), ("v_layers", _vp), ("block_table", _vp), ("prefix_len", _vp),
                ("n_tree", _vp), ("parent", _vp), ("tokens", _vp), ("verified", _vp), ("m", _vp),
                ("new_prefix_len", _vp), ("new_n_tree", _vp), ("new_parent", _vp), ("new_tokens", _vp),
                ("src_rows", _vp)]


class SampleArgs(ctypes.Structure):
    _fields_ = [("num_requests", _i32), ("n_tree_max", _i32), ("vocab", _i32), ("temperature", ctypes.c_float),
                ("target_logits", _vp), ("draft_logits", _vp), ("tokens", _vp), ("parent", _vp), ("n_tree", _vp),
                ("u_accept", _vp), ("u_bonus", _vp), ("path", _vp), ("accept_len", _vp), ("bonus", _vp),
                ("verified", _vp), ("verified_len", _vp), ("wait_limit_ns", ctypes.c_uint)]


class ExpandArgs(ctypes.Structure):
    _fields_ = [("num_requests", _i32), ("n_tree_max", _i32), ("vocab", _i32), ("w", _i32), ("k", _i32),
                ("logits", _vp), ("rows", _vp), ("n_tree", _vp), ("parent", _vp), ("tokens", _vp), ("weight", _vp),
                ("cand_tok", _vp), ("cand_lp", _vp), ("cand_taken", _vp), ("added", _vp)]


class SelectArgs(ctypes.Structure):
    _fields_ = [("num_requests", _i32), ("n_tree_max", _i32), ("bs", _i32), ("n_tree", _vp), ("parent", _vp),
                ("tokens", _vp), ("weight", _vp), ("keep", _vp), ("new_parent", _vp), ("new_tokens", _vp),
                ("new_weight", _vp), ("n_sel", _vp)]


def _sig(name, restype, argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = argtypes
    return f


_meta_ws = _sig("tree_meta_workspace_size", ctypes.c_size_t, [])
_build_mask = _sig("tree_build_mask", _i32, [_vp, _vp, _i32, _i32, _vp, _vp, _vp, ctypes.c_size_t, _vp])
_attn_ws = _sig("tree_attn_workspace_size", ctypes.c_size_t, [ctypes.POINTER(AttnArgs)])
_attn_path = _sig("tree_attn_selected_path", _i32, [ctypes.POINTER(AttnArgs)])
_attn = _sig("tree_attn_forward", _i32, [ctypes.POINTER(AttnArgs), _vp, ctypes.c_size_t, _vp])
_attn_noalloc = _sig("tree_attn_forward_noalloc", _i32, [ctypes.POINTER(AttnArgs), _vp])
_acc_ws = _sig("tree_accept_workspace_size", ctypes.c_size_t, [ctypes.POINTER(AcceptArgs)])
_acc = _sig("tree_accept_greedy", _i32, [ctypes.POINTER(AcceptArgs), _vp, ctypes.c_size_t, _vp])
_cmp_ws = _sig("tree_compact_workspace_size", ctypes.c_size_t, [ctypes.POINTER(CompactArgs)])
_cmp = _sig("tree_cache_compact", _i32, [ctypes.POINTER(CompactArgs), _vp, ctypes.c_size_t, _vp])
_cmp_batch = _sig("tree_cache_compact_batch", _i32, [ctypes.POINTER(CompactArgs), _i32, ctypes.POINTER(_vp),
                                                  ctypes.POINTER(ctypes.c_size_t), _vp])
_smp_ws = _sig("tree_accept_sample_workspace_size", ctypes.c_size_t, [ctypes.POINTER(SampleArgs)])
_smp = _sig("tree_accept_sample", _i32, [ctypes.POINTER(SampleArgs), _vp, ctypes.c_size_t, _vp])
_exp_ws = _sig("tree_expand_workspace_size", ctypes.c_size_t, [ctypes.POINTER(ExpandArgs)])
_exp = _sig("tree_expand", _i32, [ctypes.POINTER(ExpandArgs), _vp, ctypes.c_size_t, _vp])
_sel_ws = _sig("tree_select_workspace_size", ctypes.c_size_t, [ctypes.POINTER(SelectArgs)])
_sel = _sig("tree_select_subtree", _i32, [ctypes.POINTER(SelectArgs), _vp, ctypes.c_size_t, _vp])
_status_string = _sig("ts_status_string", ctypes.c_char_p, [_i32])
_read_err = _sig("ts_read_device_error", _i32, [_vp, ctypes.POINTER(_i32), _i32, _vp])
_version = _sig("ts_version", _i32, [])

EXPORTED = ["tree_meta_workspace_size", "tree_build_mask", "tree_attn_workspace_size", "tree_attn_selected_path",
            "tree_attn_forward", "tree_attn_forward_noalloc",
            "tree_accept_workspace_size", "tree_accept_greedy", "tree_compact_workspace_size",
            "tree_cache_compact", "tree_cache_compact_batch", "tree_accept_sample_workspace_size",
            "tree_accept_sample",
            "tree_expand_workspace_size", "tree_expand", "tree_select_workspace_size",
            "tree_select_subtree", "ts_status_string", "ts_read_device_error", "ts_version"]


class TreeSpecError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {_status_string(status).decode()}")
        self.status = status


def _check(status: int, where: str) -> None:
    if status != TS_OK:
        raise TreeSpecError(status, where)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled device workspace (the error word must start at zero)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def version() -> tuple:
    v = _version()
    return v >> 16, v & 0xFFFF


def read_device_error(workspace: torch.Tensor, clear: bool = True, stream=None) -> int:
    code = _i32(0)
    _check(_read_err(workspace.data_ptr(), ctypes.byref(code), int(clear), _stream(stream)), "ts_read_device_error")
    return code.value


# ---------------------------------------------------------------- metadata
def tree_build_mask(parent: torch.Tensor, n_tree: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                    stream=None):
    """Depth [B][n] and ancestor-or-self bitmask [B][n][4] (uint32 as int32) of every node."""
    B, n_max = parent.shape
    depth = torch.empty((B, n_max), dtype=torch.int32, device=parent.device)
    anc = torch.empty((B, n_max, 4), dtype=torch.int32, device=parent.device)
    ws = workspace if workspace is not None else new_workspace(_meta_ws(), parent.device)
    _check(_build_mask(parent.data_ptr(), n_tree.data_ptr(), B, n_max, depth.data_ptr(), anc.data_ptr(),
                       ws.data_ptr(), ws.numel(), _stream(stream)), "tree_build_mask")
    return depth, anc


# ---------------------------------------------------------------- attention
@dataclass
class AttnPlan:
    args: AttnArgs
    workspace_bytes: int


def attn_args(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, prefix_len: torch.Tensor,
              n_tree: torch.Tensor, parent: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor] = None,
              block_table: Optional[torch.Tensor] = None, softmax_scale: float = 0.0, force_path: int = 0,
              num_ctas: int = 0, rope_theta: float = 0.0, wait_limit_ns: int = 0) -> AttnArgs:
    """Fill ``ts_attn_args`` from tensors.

    q, out: bf16 [B][n_query][Hq][d].  Contiguous KV: bf16 [B][max_kv_len][Hkv][d];
    paged KV: bf16 pool [num_blocks][page][Hkv][d] plus int32 block_table [B][max_blocks].
    """
    B, nq, hq, d = q.shape
    a = AttnArgs()
    a.num_requests, a.num_q_heads, a.head_dim, a.n_query = B, hq, d, nq
    a.n_tree_max = parent.shape[1]
    if block_table is None:
        a.kv_layout = TS_KV_CONTIGUOUS
        a.max_kv_len, a.num_kv_heads = k_cache.shape[1], k_cache.shape[2]
    else:
        a.kv_layout = TS_KV_PAGED
        a.num_blocks, a.page_size, a.num_kv_heads = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
        a.max_blocks_per_req = block_table.shape[1]
        a.max_kv_len = a.max_blocks_per_req * a.page_size
        a.block_table = block_table.data_ptr()
    a.prefix_len, a.n_tree, a.parent = prefix_len.data_ptr(), n_tree.data_ptr(), parent.data_ptr()
    a.q, a.k_cache, a.v_cache, a.out = q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr()
    a.lse = _ptr(lse)
    a.softmax_scale, a.force_path, a.num_ctas = softmax_scale, force_path, num_ctas
    a.rope_theta = rope_theta
    a.wait_limit_ns = wait_limit_ns
    return a


def tree_attn_workspace_size(args: AttnArgs) -> int:
    n = _attn_ws(ctypes.byref(args))
    if n == 0:
        raise TreeSpecError(TS_ERR_INVALID_ARG, "tree_attn_workspace_size")
    return n


def tree_attn_selected_path(args: AttnArgs) -> str:
    """'mma' or 'tcgen05': the attention kernel the library picks for these arguments."""
    r = _attn_path(ctypes.byref(args))
    if r < 0:
        raise TreeSpecError(-r, "tree_attn_selected_path")
    return "tcgen05" if r == 2 else "mma"


def tree_attn_forward_args(args: AttnArgs, workspace: torch.Tensor, stream=None) -> None:
    _check(_attn(ctypes.byref(args), workspace.data_ptr(), workspace.numel(), _stream(stream)), "tree_attn_forward")


def tree_attn_forward(q, k_cache, v_cache, prefix_len, n_tree, parent, out=None, lse=None, block_table=None,
                      softmax_scale: float = 0.0, workspace=None, stream=None, force_path: int = 0,
                      num_ctas: int = 0, want_lse: bool = True, rope_theta: float = 0.0, wait_limit_ns: int = 0):
    """Tree-masked GQA attention; returns (out, lse).  rope_theta > 0 rotates
    the queries at their tree positions (prefix length + depth) first;
    wait_limit_ns > 0 bounds each pipeline wait in the kernels (testing)."""
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=q.device)
    a = attn_args(q, k_cache, v_cache, prefix_len, n_tree, parent, out, lse, block_table, softmax_scale,
                  force_path, num_ctas, rope_theta, wait_limit_ns)
    if workspace is None:
        workspace = new_workspace(tree_attn_workspace_size(a), q.device)
    tree_attn_forward_args(a, workspace, stream)
    return out, lse


def tree_attn_forward_noalloc(q, k_cache, v_cache, prefix_len, n_tree, parent, out, lse=None, block_table=None,
                              softmax_scale: float = 0.0, stream=None, force_path: int = 0, num_ctas: int = 0,
                              rope_theta: float = 0.0):
    """tree_attn_forward for callers that cannot allocate device memory.

    The library keeps the split-KV scratch in its own 16 MiB device array, so
    the caller passes only inputs and preallocated outputs (``out`` and
    optionally ``lse``).  Calls that overlap on the GPU race on that array.
    """
    a = attn_args(q, k_cache, v_cache, prefix_len, n_tree, parent, out, lse, block_table, softmax_scale,
                  force_path, num_ctas, rope_theta)
    _check(_attn_noalloc(ctypes.byref(a), _stream(stream)), "tree_attn_forward_noalloc")
    return out, lse


# ---------------------------------------------------------------- acceptance
def accept_args(logits, tokens, parent, n_tree, argmax, path, accept_len, bonus, verified=None,
                verified_len=None) -> AcceptArgs:
    B, n_max, V = logits.shape
    a = AcceptArgs()
    a.num_requests, a.n_tree_max, a.vocab = B, n_max, V
    a.logits, a.tokens, a.parent, a.n_tree = logits.data_ptr(), tokens.data_ptr(), parent.data_ptr(), n_tree.data_ptr()
    a.argmax, a.path, a.accept_len, a.bonus = argmax.data_ptr(), path.data_ptr(), accept_len.data_ptr(), bonus.data_ptr()
    a.verified, a.verified_len = _ptr(verified), _ptr(verified_len)
    return a


def tree_accept_workspace_size(args: AcceptArgs) -> int:
    return _acc_ws(ctypes.byref(args))


def tree_accept_greedy_args(args: AcceptArgs, workspace: torch.Tensor, stream=None) -> None:
    _check(_acc(ctypes.byref(args), workspace.data_ptr(), workspace.numel(), _stream(stream)), "tree_accept_greedy")


def tree_accept_greedy(logits, tokens, parent, n_tree, workspace=None, stream=None) -> dict:
    """Greedy acceptance; returns dict of argmax, path, accept_len, bonus, verified, verified_len."""
    B, n_max, _ = logits.shape
    dev = logits.device
    out = {
        "argmax": torch.empty((B, n_max), dtype=torch.int32, device=dev),
        "path": torch.empty((B, n_max), dtype=torch.int32, device=dev),
        "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
        "bonus": torch.empty(B, dtype=torch.int32, device=dev),
        "verified": torch.empty((B, n_max + 1), dtype=torch.int32, device=dev),
        "verified_len": torch.empty(B, dtype=torch.int32, device=dev),
    }
    a = accept_args(logits, tokens, parent, n_tree, **out)
    if workspace is None:
        workspace = new_workspace(tree_accept_workspace_size(a), dev)
    tree_accept_greedy_args(a, workspace, stream)
    return out


# ---------------------------------------------------------------- compaction
def layer_pointer_table(layers: Sequence[torch.Tensor], device=None) -> torch.Tensor:
    """Device array of the layers' data pointers (int64), as ``k_layers``/``v_layers`` expect."""
    return torch.tensor([t.data_ptr() for t in layers], dtype=torch.int64, device=device or layers[0].device)


def compact_args(k_ptrs: torch.Tensor, v_ptrs: torch.Tensor, num_layers: int, num_kv_heads: int, head_dim: int,
                 prefix_len, n_tree, parent, tokens, verified, m, new_prefix_len, new_n_tree, new_parent,
                 new_tokens, src_rows=None, max_kv_len: int = 0, block_table=None, page_size: int = 0,
                 num_blocks: int = 0, elem_bytes: int = 2) -> CompactArgs:
    a = CompactArgs()
    B, n_max = parent.shape
    a.num_requests, a.n_tree_max, a.m_max = B, n_max, verified.shape[1]
    a.num_layers, a.num_kv_heads, a.head_dim, a.elem_bytes = num_layers, num_kv_heads, head_dim, elem_bytes
    if block_table is None:
        a.kv_layout, a.max_kv_len = TS_KV_CONTIGUOUS, max_kv_len
    else:
        a.kv_layout, a.page_size, a.num_blocks = TS_KV_PAGED, page_size, num_blocks
        a.max_blocks_per_req = block_table.shape[1]
        a.max_kv_len = a.max_blocks_per_req * page_size
        a.block_table = block_table.data_ptr()
    a.k_layers, a.v_layers = k_ptrs.data_ptr(), v_ptrs.data_ptr()
    a.prefix_len, a.n_tree, a.parent, a.tokens = prefix_len.data_ptr(), n_tree.data_ptr(), parent.data_ptr(), tokens.data_ptr()
    a.verified, a.m = verified.data_ptr(), m.data_ptr()
    a.new_prefix_len, a.new_n_tree = new_prefix_len.data_ptr(), new_n_tree.data_ptr()
    a.new_parent, a.new_tokens, a.src_rows = new_parent.data_ptr(), new_tokens.data_ptr(), _ptr(src_rows)
    return a


def tree_compact_workspace_size(args: CompactArgs) -> int:
    return _cmp_ws(ctypes.byref(args))


def tree_cache_compact_args(args: CompactArgs, workspace: torch.Tensor, stream=None) -> None:
    _check(_cmp(ctypes.byref(args), workspace.data_ptr(), workspace.numel(), _stream(stream)), "tree_cache_compact")


def tree_cache_compact_batch_args(args: Sequence[CompactArgs], workspaces: Sequence[torch.Tensor], stream=None) -> None:
    """Several independent compactions (e.g. the target- and draft-side caches) in one launch; each call keeps
    the workspace it would take alone."""
    n = len(args)
    if n != len(workspaces):
        raise ValueError("one workspace per compaction")
    arr = (CompactArgs * n)(*args)
    ptrs = (_vp * n)(*[w.data_ptr() for w in workspaces])
    sizes = (ctypes.c_size_t * n)(*[w.numel() for w in workspaces])
    _check(_cmp_batch(arr, n, ptrs, sizes, _stream(stream)), "tree_cache_compact_batch")


def tree_cache_compact(k_layers: Sequence[torch.Tensor], v_layers: Sequence[torch.Tensor], prefix_len, n_tree,
                       parent, tokens, verified, m, block_table=None, workspace=None, stream=None,
                       in_place_metadata: bool = False) -> dict:
    """Re-root + in-place KV compaction over every layer; returns the new metadata."""
    k0 = k_layers[0]
    B, n_max = parent.shape
    dev = parent.device
    if block_table is None:
        max_kv_len, hkv, d = k0.shape[1], k0.shape[2], k0.shape[3]
        page, nblk = 0, 0
    else:
        nblk, page, hkv, d = k0.shape[0], k0.shape[1], k0.shape[2], k0.shape[3]
        max_kv_len = 0
    out = {
        "new_prefix_len": torch.empty(B, dtype=torch.int32, device=dev),
        "new_n_tree": torch.empty(B, dtype=torch.int32, device=dev),
        "new_parent": parent if in_place_metadata else torch.empty_like(parent),
        "new_tokens": tokens if in_place_metadata else torch.empty_like(tokens),
        "src_rows": torch.empty_like(parent),
    }
    kp = layer_pointer_table(k_layers, dev)
    vp = layer_pointer_table(v_layers, dev)
    a = compact_args(kp, vp, len(k_layers), hkv, d, prefix_len, n_tree, parent, tokens, verified, m,
                     out["new_prefix_len"], out["new_n_tree"], out["new_parent"], out["new_tokens"],
                     out["src_rows"], max_kv_len, block_table, page, nblk, k0.element_size())
    if workspace is None:
        workspace = new_workspace(tree_compact_workspace_size(a), dev)
    tree_cache_compact_args(a, workspace, stream)
    out["_ptr_tables"] = (kp, vp)   # keep the pointer tables alive until the stream reaches the kernels
    return out


# ------------------------------------------------------------------ draft-side expansion and selection
TS_MAX_EXPAND = 16


class DraftTree:
    """Device state of a batch of draft trees for ``tree_expand`` (per node:
    parent, token, weight, and k candidate children with their log-probs and
    how many have been taken)."""

    def __init__(self, num_requests: int, n_tree_max: int, k: int, device=None):
        dev = device or "cuda"
        B, N = num_requests, n_tree_max
        self.k = k
        self.n_tree = torch.zeros(B, dtype=torch.int32, device=dev)
        self.parent = torch.full((B, N), -1, dtype=torch.int32, device=dev)
        self.tokens = torch.zeros((B, N), dtype=torch.int32, device=dev)
        self.weight = torch.zeros((B, N), dtype=torch.float32, device=dev)
        self.cand_tok = torch.full((B, N, k), -1, dtype=torch.int32, device=dev)
        self.cand_lp = torch.full((B, N, k), float("-inf"), dtype=torch.float32, device=dev)
        self.cand_taken = torch.full((B, N), k, dtype=torch.int32, device=dev)


def expand_args(tree: DraftTree, logits: torch.Tensor, rows: torch.Tensor, added: torch.Tensor) -> ExpandArgs:
    """logits fp32 [B][w][vocab] (16-byte aligned rows when vocab % 4 == 0), rows / added int32 [B][w]."""
    B, w, V = logits.shape
    a = ExpandArgs()
    a.num_requests, a.n_tree_max, a.vocab, a.w, a.k = B, tree.parent.shape[1], V, w, tree.k
    a.logits, a.rows = logits.data_ptr(), rows.data_ptr()
    a.n_tree, a.parent, a.tokens, a.weight = (tree.n_tree.data_ptr(), tree.parent.data_ptr(),
                                              tree.tokens.data_ptr(), tree.weight.data_ptr())
    a.cand_tok, a.cand_lp, a.cand_taken = tree.cand_tok.data_ptr(), tree.cand_lp.data_ptr(), tree.cand_taken.data_ptr()
    a.added = added.data_ptr()
    return a


def tree_expand_workspace_size(args: ExpandArgs) -> int:
    n = _exp_ws(ctypes.byref(args))
    if n == 0:
        raise TreeSpecError(TS_ERR_INVALID_ARG, "tree_expand_workspace_size")
    return n


def tree_expand_args(args: ExpandArgs, workspace: torch.Tensor, stream=None) -> None:
    _check(_exp(ctypes.byref(args), workspace.data_ptr(), workspace.numel(), _stream(stream)), "tree_expand")


def tree_expand(tree: DraftTree, logits: torch.Tensor, rows: torch.Tensor, workspace=None, stream=None) -> torch.Tensor:
    """One maximum-likelihood expansion step in place; returns the added nodes [B][w] (-1 past the last)."""
    added = torch.empty_like(rows)
    a = expand_args(tree, logits, rows, added)
    if workspace is None:
        workspace = new_workspace(tree_expand_workspace_size(a), logits.device)
    tree_expand_args(a, workspace, stream)
    return added


def select_args(n_tree, parent, tokens, weight, bs: int, out: dict) -> SelectArgs:
    B, N = parent.shape
    a = SelectArgs()
    a.num_requests, a.n_tree_max, a.bs = B, N, bs
    a.n_tree, a.parent, a.tokens, a.weight = n_tree.data_ptr(), parent.data_ptr(), tokens.data_ptr(), weight.data_ptr()
    a.keep, a.new_parent, a.new_tokens = out["keep"].data_ptr(), out["new_parent"].data_ptr(), out["new_tokens"].data_ptr()
    a.new_weight, a.n_sel = out["new_weight"].data_ptr(), out["n_sel"].data_ptr()
    return a


def tree_select_subtree_args(args: SelectArgs, workspace: torch.Tensor, stream=None) -> None:
    _check(_sel(ctypes.byref(args), workspace.data_ptr(), workspace.numel(), _stream(stream)), "tree_select_subtree")


def tree_select_subtree(n_tree, parent, tokens, weight, bs: int, workspace=None, stream=None) -> dict:
    """The bs heaviest nodes of each tree, in index order, with remapped parents."""
    B = parent.shape[0]
    dev = parent.device
    out = {"keep": torch.empty((B, bs), dtype=torch.int32, device=dev),
           "new_parent": torch.empty((B, bs), dtype=torch.int32, device=dev),
           "new_tokens": torch.empty((B, bs), dtype=torch.int32, device=dev),
           "new_weight": torch.empty((B, bs), dtype=torch.float32, device=dev),
           "n_sel": torch.empty(B, dtype=torch.int32, device=dev)}
    a = select_args(n_tree, parent, tokens, weight, bs, out)
    if workspace is None:
        workspace = new_workspace(int(_sel_ws(ctypes.byref(a))), dev)
    _check(_sel(ctypes.byref(a), workspace.data_ptr(), workspace.numel(), _stream(stream)), "tree_select_subtree")
    return out


# ------------------------------------------------------------------ stochastic acceptance
def sample_args(target_logits, draft_logits, tokens, parent, n_tree, u_accept, u_bonus, temperature: float,
                out: dict, wait_limit_ns: int = 0) -> SampleArgs:
    """target_logits / draft_logits fp32 [B][n_max][V]; u_accept / u_bonus fp32 [B][n_max] in [0, 1)."""
    B, n_max, V = target_logits.shape
    a = SampleArgs()
    a.num_requests, a.n_tree_max, a.vocab, a.temperature = B, n_max, V, temperature
    a.target_logits, a.draft_logits = target_logits.data_ptr(), draft_logits.data_ptr()
    a.tokens, a.parent, a.n_tree = tokens.data_ptr(), parent.data_ptr(), n_tree.data_ptr()
    a.u_accept, a.u_bonus = u_accept.data_ptr(), u_bonus.data_ptr()
    a.path, a.accept_len, a.bonus = out["path"].data_ptr(), out["accept_len"].data_ptr(), out["bonus"].data_ptr()
    a.verified, a.verified_len = out["verified"].data_ptr(), out["verified_len"].data_ptr()
    a.wait_limit_ns = wait_limit_ns
    return a


def tree_accept_sample_workspace_size(args: SampleArgs) -> int:
    n = _smp_ws(ctypes.byref(args))
    if n == 0:
        raise TreeSpecError(TS_ERR_INVALID_ARG, "tree_accept_sample_workspace_size")
    return n


def tree_accept_sample_args(args: SampleArgs, workspace: torch.Tensor, stream=None) -> None:
    _check(_smp(ctypes.byref(args), workspace.data_ptr(), workspace.numel(), _stream(stream)), "tree_accept_sample")


def tree_accept_sample(target_logits, draft_logits, tokens, parent, n_tree, u_accept, u_bonus, temperature: float,
                       workspace=None, stream=None, wait_limit_ns: int = 0) -> dict:
    """Stochastic tree acceptance; returns dict of path, accept_len, bonus, verified, verified_len.
    wait_limit_ns > 0 bounds each wait of the walk's hand-offs (testing)."""
    B, n_max, _ = target_logits.shape
    dev = target_logits.device
    out = {"path": torch.empty((B, n_max), dtype=torch.int32, device=dev),
           "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
           "bonus": torch.empty(B, dtype=torch.int32, device=dev),
           "verified": torch.empty((B, n_max + 1), dtype=torch.int32, device=dev),
           "verified_len": torch.empty(B, dtype=torch.int32, device=dev)}
    a = sample_args(target_logits, draft_logits, tokens, parent, n_tree, u_accept, u_bonus, temperature, out,
                    wait_limit_ns)
    if workspace is None:
        workspace = new_workspace(tree_accept_sample_workspace_size(a), dev)
    tree_accept_sample_args(a, workspace, stream)
    return out

