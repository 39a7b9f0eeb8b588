"""Torch-facing wrappers over libtpa. Tensors are only allocated here and
their pointers handed to the library; no arithmetic of the method runs in
Python."""
from __future__ import annotations

import ctypes as C
from typing import Sequence

import numpy as np
import torch

from ._abi import (BALANCE_FFD, BALANCE_KK, GRAD_BF16, GRAD_F32, LOGITS_COMPACT, LOGITS_PADDED, MASK_BITS,
                   MASK_U8, BlockMaskView, PackingMetrics, TreeInfo, TreeView, check, lib)


def _stream_ptr(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


class Tree:
    """Packed trees on the host (owns a library tree handle)."""

    def __init__(self, handle: C.c_void_p):
        self._h = handle
        info = TreeInfo()
        check("tpa_tree_get_info", lib().tpa_tree_get_info(self._h, C.byref(info)))
        self.info = info

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().tpa_tree_free(h)
            self._h = None

    @property
    def n_trees(self) -> int:
        return self.info.n_trees

    @property
    def t_pad(self) -> int:
        return self.info.t_pad

    @property
    def tree_token_ratio(self) -> float:
        return self.info.tree_token_ratio

    def host_view(self) -> TreeView:
        v = TreeView()
        base = lib().tpa_tree_host_blob(self._h)
        check("tpa_tree_make_view", lib().tpa_tree_make_view(self._h, base, C.byref(v)))
        return v

    def host_blob(self) -> np.ndarray:
        """A copy of the metadata blob (uint8)."""
        base = lib().tpa_tree_host_blob(self._h)
        return np.ctypeslib.as_array((C.c_uint8 * self.info.blob_bytes).from_address(base)).copy()

    def arrays(self) -> dict[str, np.ndarray]:
        """Copies of every metadata array, shaped per tree."""
        v = self.host_view()
        B, T, S, N, M = (self.info.n_trees, self.info.t_pad, self.info.n_seqs,
                         self.info.total_seq_tokens, self.info.max_nodes)

        def arr(ptr, ctype, n, shape):
            return np.ctypeslib.as_array((ctype * n).from_address(ptr)).reshape(shape).copy()

        return {
            "tokens": arr(v.tokens, C.c_int32, B * T, (B, T)),
            "subtree_end": arr(v.subtree_end, C.c_int32, B * T, (B, T)),
            "parent": arr(v.parent, C.c_int32, B * T, (B, T)),
            "depth": arr(v.depth, C.c_int32, B * T, (B, T)),
            "node_id": arr(v.node_id, C.c_int32, B * T, (B, T)),
            "child_off": arr(v.child_off, C.c_int32, B * (T + 1), (B, T + 1)),
            "child_pos": arr(v.child_pos, C.c_int32, B * T, (B, T)),
            "n_tokens": arr(v.n_tokens, C.c_int32, B, (B,)),
            "tok_base": arr(v.tok_base, C.c_int64, B + 1, (B + 1,)),
            "node_info": arr(v.node_info, C.c_int32, B * M * 4, (B, M, 4)),
            "n_nodes": arr(v.n_nodes, C.c_int32, B, (B,)),
            "seq_tree": arr(v.seq_tree, C.c_int32, S, (S,)),
            "seq_off": arr(v.seq_off, C.c_int64, S + 1, (S + 1,)),
            "seq_pos": arr(v.seq_pos, C.c_int32, N, (N,)),
        }

    def upload(self, device="cuda", stream=None, buffer: torch.Tensor | None = None) -> "DeviceTree":
        """Copy the metadata blob into device memory (a torch uint8 buffer)."""
        nbytes = int(self.info.blob_bytes)
        if buffer is None:
            buffer = torch.empty(nbytes, dtype=torch.uint8, device=device)
        check("tpa_tree_upload", lib().tpa_tree_upload(self._h, buffer.data_ptr(), buffer.numel(),
                                                       _stream_ptr(stream)))
        return DeviceTree(self, buffer)


class DeviceTree:
    """Packed-tree metadata resident on the device."""

    def __init__(self, tree: Tree, buf: torch.Tensor):
        self.tree = tree
        self.buf = buf
        self.view = TreeView()
        check("tpa_tree_make_view", lib().tpa_tree_make_view(tree._h, buf.data_ptr(), C.byref(self.view)))

    @property
    def info(self) -> TreeInfo:
        return self.tree.info

    @property
    def device(self) -> torch.device:
        return self.buf.device


class BlockMask:
    """128x128 tile classes and the two CSR lists, in one device buffer."""

    def __init__(self, n_trees: int, t_pad: int, device, buf: torch.Tensor | None = None):
        nbytes = int(lib().tpa_blockmask_bytes(n_trees, t_pad))
        if buf is None:
            buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.buf = buf
        self.view = BlockMaskView()
        check("tpa_blockmask_make_view",
              lib().tpa_blockmask_make_view(buf.data_ptr(), n_trees, t_pad, C.byref(self.view)))
        self.n_trees, self.t_pad, self.n_blk, self.cap = n_trees, t_pad, self.view.n_blk, self.view.cap

    def _slice(self, ptr: int, nbytes: int, dtype, shape):
        off = ptr - self.buf.data_ptr()
        return self.buf[off:off + nbytes].view(dtype).view(shape)

    def arrays(self) -> dict[str, torch.Tensor]:
        B, n, cap = self.n_trees, self.n_blk, self.cap
        v = self.view
        return {
            "cls": self._slice(v.cls, B * n * n, torch.uint8, (B, n, n)),
            "q_ptr": self._slice(v.q_ptr, 4 * B * (n + 1), torch.int32, (B, n + 1)),
            "q_idx": self._slice(v.q_idx, 4 * B * cap, torch.int32, (B, cap)),
            "k_ptr": self._slice(v.k_ptr, 4 * B * (n + 1), torch.int32, (B, n + 1)),
            "k_idx": self._slice(v.k_idx, 4 * B * cap, torch.int32, (B, cap)),
            "qmask": self._slice(v.qmask, 2048 * B * cap, torch.int32, (B, cap, 128, 4)),
            "sched": self._slice(v.sched, 4 * 16, torch.int32, (16,)),
        }


def tree_pack(seqs: Sequence[Sequence[int]] | None = None, max_tokens_per_mb: int = 8192, *,
              tokens: np.ndarray | None = None, offsets: np.ndarray | None = None) -> Tree:
    """Pack sequences (a list of token lists, or flat ``tokens`` + ``offsets``)."""
    if tokens is None:
        offsets = np.zeros(len(seqs) + 1, dtype=np.int64)
        offsets[1:] = np.cumsum([len(s) for s in seqs])
        tokens = np.fromiter((t for s in seqs for t in s), dtype=np.int32, count=int(offsets[-1]))
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    h = C.c_void_p()
    n = len(offsets) - 1
    tok_p = tokens.ctypes.data_as(C.POINTER(C.c_int32)) if tokens.size else \
        C.cast(C.pointer(C.c_int32(0)), C.POINTER(C.c_int32))
    check("tpa_tree_pack", lib().tpa_tree_pack(tok_p, offsets.ctypes.data_as(C.POINTER(C.c_int64)), n,
                                               int(max_tokens_per_mb), C.byref(h)))
    return Tree(h)


def _padded(input_ids, attention_mask):
    ids = np.ascontiguousarray(np.asarray(input_ids), dtype=np.int32)
    msk = np.ascontiguousarray(np.asarray(attention_mask) != 0, dtype=np.uint8)
    if ids.ndim != 2 or ids.shape != msk.shape:
        raise ValueError("input_ids and attention_mask must be 2-D arrays of one shape")
    return ids, msk


def extract_sequences(input_ids, attention_mask) -> tuple[np.ndarray, np.ndarray]:
    """Real tokens of a padded batch (tpa_extract_sequences): flat int32
    tokens and int64 offsets, the input format of ``tree_pack``."""
    ids, msk = _padded(input_ids, attention_mask)
    n, L = ids.shape
    tokens = np.empty(n * L, dtype=np.int32)
    offsets = np.empty(n + 1, dtype=np.int64)
    check("tpa_extract_sequences", lib().tpa_extract_sequences(
        ids.ctypes.data_as(C.POINTER(C.c_int32)), msk.ctypes.data_as(C.POINTER(C.c_uint8)), n, L,
        tokens.ctypes.data_as(C.POINTER(C.c_int32)), offsets.ctypes.data_as(C.POINTER(C.c_int64))))
    return tokens[:int(offsets[-1])], offsets


def tree_pack_padded(input_ids, attention_mask, max_tokens_per_mb: int = 8192) -> Tree:
    """Extract the real tokens of a padded batch and pack them (tpa_tree_pack_padded)."""
    ids, msk = _padded(input_ids, attention_mask)
    h = C.c_void_p()
    check("tpa_tree_pack_padded", lib().tpa_tree_pack_padded(
        ids.ctypes.data_as(C.POINTER(C.c_int32)), msk.ctypes.data_as(C.POINTER(C.c_uint8)), ids.shape[0],
        ids.shape[1], int(max_tokens_per_mb), C.byref(h)))
    return Tree(h)


def balance(weights: Sequence[int], capacity: int, min_groups: int = 1, groups_divisor: int = 1,
            algorithm: str = "ffd") -> tuple[np.ndarray, int, str]:
    """Split weighted items into groups (tpa_balance): returns (group of each
    item, number of groups, algorithm whose result it is)."""
    w = np.ascontiguousarray(np.asarray(weights, dtype=np.int64))
    if algorithm not in ("ffd", "kk"):
        raise ValueError(f"unknown balancing algorithm {algorithm!r}; choose 'ffd' or 'kk'")
    algo = BALANCE_FFD if algorithm == "ffd" else BALANCE_KK
    out = np.empty(len(w), dtype=np.int32)
    ng, used = C.c_int32(0), C.c_int32(0)
    check("tpa_balance", lib().tpa_balance(w.ctypes.data_as(C.POINTER(C.c_int64)), len(w), int(capacity),
                                           int(min_groups), int(groups_divisor), algo,
                                           out.ctypes.data_as(C.POINTER(C.c_int32)), C.byref(ng),
                                           C.byref(used)))
    return out, ng.value, "kk" if used.value == BALANCE_KK else "ffd"


def packing_metrics(weights: Sequence[int], group_of: Sequence[int], n_groups: int, capacity: int) -> dict:
    """The packing metrics of a grouping (tpa_packing_metrics) as a dict."""
    w = np.ascontiguousarray(np.asarray(weights, dtype=np.int64))
    g = np.ascontiguousarray(np.asarray(group_of, dtype=np.int32))
    m = PackingMetrics()
    check("tpa_packing_metrics", lib().tpa_packing_metrics(w.ctypes.data_as(C.POINTER(C.c_int64)), len(w),
                                                           g.ctypes.data_as(C.POINTER(C.c_int32)), int(n_groups),
                                                           int(capacity), C.byref(m)))
    return {f: getattr(m, f) for f, _ in PackingMetrics._fields_ if f != "pad_"}


def dense_mask(dtree: DeviceTree, fmt: str = "u8", invert: bool = False, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """Dense ancestor mask of every tree (tpa_dense_mask): uint8 [B, T, T]
    for fmt "u8", or int32 words [B, T, T/32] (bit j%32 of word j/32) for
    fmt "bits"; 1 marks a visible pair, or a removed pair with invert."""
    if fmt not in ("u8", "bits"):
        raise ValueError(f"unknown mask format {fmt!r}; choose 'u8' or 'bits'")
    B, T = dtree.info.n_trees, dtree.info.t_pad
    code = MASK_U8 if fmt == "u8" else MASK_BITS
    if out is None:
        out = (torch.empty((B, T, T), dtype=torch.uint8, device=dtree.device) if fmt == "u8" else
               torch.empty((B, T, T // 32), dtype=torch.int32, device=dtree.device))
    nbytes = out.numel() * out.element_size()
    check("tpa_dense_mask", lib().tpa_dense_mask(C.byref(dtree.view), out.data_ptr(), nbytes, code,
                                                 1 if invert else 0, _stream_ptr(stream)))
    return out


def block_classify(dtree: DeviceTree, stream=None, out: BlockMask | None = None) -> BlockMask:
    mask = out or BlockMask(dtree.info.n_trees, dtree.info.t_pad, dtree.device)
    check("tpa_block_classify", lib().tpa_block_classify(C.byref(dtree.view), C.byref(mask.view),
                                                         _stream_ptr(stream)))
    return mask


def _check_qkv(dtree: DeviceTree, q, k, v):
    B, T = dtree.info.n_trees, dtree.info.t_pad
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor [B, T_pad, H, d]")
        if t.shape[0] != B or t.shape[1] != T:
            raise ValueError(f"{name} has shape {tuple(t.shape)}; expected [{B}, {T}, H, d]")
    if k.shape != v.shape or q.shape[3] != k.shape[3]:
        raise ValueError("k and v must match, and share head_dim with q")
    return B, T, q.shape[2], k.shape[2], q.shape[3]


def tree_attn_fwd(dtree: DeviceTree, mask: BlockMask, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                  softmax_scale: float | None = None, out: torch.Tensor | None = None,
                  lse: torch.Tensor | None = None, stream=None):
    """Tree attention forward: returns O [B, T_pad, Hq, d] bf16 and LSE [B, Hq, T_pad] fp32."""
    B, T, Hq, Hkv, d = _check_qkv(dtree, q, k, v)
    o = out if out is not None else torch.empty_like(q)
    lse = lse if lse is not None else torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    check("tpa_tree_attn_fwd", lib().tpa_tree_attn_fwd(
        C.byref(dtree.view), C.byref(mask.view), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
        lse.data_ptr(), Hq, Hkv, d, float(softmax_scale or 0.0), _stream_ptr(stream)))
    return o, lse


_GRAD = {torch.float32: GRAD_F32, torch.bfloat16: GRAD_BF16}


def tree_attn_bwd_workspace_bytes(n_trees: int, t_pad: int, n_heads_q: int, n_heads_kv: int, head_dim: int,
                                  grad_dtype: torch.dtype = torch.float32) -> int:
    return int(lib().tpa_tree_attn_bwd_workspace_bytes(n_trees, t_pad, n_heads_q, n_heads_kv, head_dim,
                                                       _GRAD[grad_dtype]))


def tree_attn_bwd(dtree: DeviceTree, mask: BlockMask, q, k, v, o, lse, dout,
                  softmax_scale: float | None = None, workspace: torch.Tensor | None = None,
                  out: tuple | None = None, grad_dtype: torch.dtype = torch.float32, stream=None):
    """Tree attention backward: returns dQ, dK, dV shaped like q, k, v, in
    ``grad_dtype`` (fp32 by default, or bf16)."""
    B, T, Hq, Hkv, d = _check_qkv(dtree, q, k, v)
    if dout.shape != q.shape or dout.dtype != torch.bfloat16 or not dout.is_contiguous():
        raise ValueError("dout must be a contiguous bf16 tensor shaped like q")
    if grad_dtype not in _GRAD:
        raise ValueError("grad_dtype must be torch.float32 or torch.bfloat16")
    if workspace is None:
        nbytes = tree_attn_bwd_workspace_bytes(B, T, Hq, Hkv, d, grad_dtype)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if out is None:
        out = tuple(torch.empty(x.shape, dtype=grad_dtype, device=x.device) for x in (q, k, v))
    dq, dk, dv = out
    if not all(x.dtype == grad_dtype and x.is_contiguous() for x in out):
        raise ValueError("gradient buffers must be contiguous and of grad_dtype")
    check("tpa_tree_attn_bwd", lib().tpa_tree_attn_bwd(
        C.byref(dtree.view), C.byref(mask.view), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
        lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
        workspace.numel(), Hq, Hkv, d, float(softmax_scale or 0.0), _GRAD[grad_dtype], _stream_ptr(stream)))
    return dq, dk, dv


def tree_logprobs_entropy(dtree: DeviceTree, logits: torch.Tensor, layout: str = "compact",
                          out: tuple | None = None, stream=None):
    """Per-position (pos_logp, pos_entropy: [B, T_pad]) and per-sequence
    (seq_logp, seq_entropy: [total_seq_tokens]) fp32 results."""
    if logits.dtype != torch.bfloat16 or logits.dim() != 2 or logits.stride(1) != 1 or not logits.is_cuda:
        raise ValueError("logits must be a CUDA bf16 [rows, V] tensor with unit column stride")
    lay = {"compact": LOGITS_COMPACT, "padded": LOGITS_PADDED}[layout]
    B, T, N = dtree.info.n_trees, dtree.info.t_pad, dtree.info.total_seq_tokens
    dev = logits.device
    if out is None:
        out = (torch.empty((B, T), dtype=torch.float32, device=dev), torch.empty((B, T), dtype=torch.float32, device=dev),
               torch.empty(N, dtype=torch.float32, device=dev), torch.empty(N, dtype=torch.float32, device=dev))
    pl, pe, sl, se = out
    check("tpa_tree_logprobs_entropy", lib().tpa_tree_logprobs_entropy(
        C.byref(dtree.view), logits.data_ptr(), logits.stride(0), lay, logits.shape[1], pl.data_ptr(),
        pe.data_ptr(), sl.data_ptr(), se.data_ptr(), _stream_ptr(stream)))
    return pl, pe, sl, se


def lm_head_workspace_bytes(rows: int, vocab: int, n_trees: int, t_pad: int) -> int:
    return int(lib().tpa_lm_head_workspace_bytes(int(rows), int(vocab), int(n_trees), int(t_pad)))


def lm_head_logprobs_entropy(dtree: DeviceTree, hidden: torch.Tensor, weight: torch.Tensor,
                             out: tuple | None = None, workspace: torch.Tensor | None = None, stream=None):
    """The log-prob pass with the LM head fused in: ``hidden`` [tree tokens, H]
    (compact rows) and ``weight`` [V, H], both CUDA bf16; returns the four
    outputs of ``tree_logprobs_entropy`` without forming the logits."""
    for name, t in (("hidden", hidden), ("weight", weight)):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA bf16 matrix")
    if hidden.shape[1] != weight.shape[1]:
        raise ValueError("hidden and weight must have the same hidden size")
    B, T, N = dtree.info.n_trees, dtree.info.t_pad, dtree.info.total_seq_tokens
    rows, V, H = hidden.shape[0], weight.shape[0], hidden.shape[1]
    if rows != dtree.info.total_tree_tokens:
        raise ValueError("hidden must have one row per tree token (compact rows)")
    dev = hidden.device
    if out is None:
        out = (torch.empty((B, T), dtype=torch.float32, device=dev), torch.empty((B, T), dtype=torch.float32, device=dev),
               torch.empty(N, dtype=torch.float32, device=dev), torch.empty(N, dtype=torch.float32, device=dev))
    nbytes = lm_head_workspace_bytes(rows, V, B, T)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    pl, pe, sl, se = out
    check("tpa_lm_head_logprobs_entropy", lib().tpa_lm_head_logprobs_entropy(
        C.byref(dtree.view), hidden.data_ptr(), weight.data_ptr(), H, V, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), pl.data_ptr(), pe.data_ptr(), sl.data_ptr(), se.data_ptr(),
        _stream_ptr(stream)))
    return pl, pe, sl, se


def sync_status(stream=None) -> None:
    """Synchronise the stream and raise if any kernel reported a device-side failure."""
    check("tpa_sync_status", lib().tpa_sync_status(_stream_ptr(stream)))


def wait_probe(limit_ns: int, arrive: bool, stream=None) -> None:
    """Launch the bounded-wait diagnostic (tpa_wait_probe): with ``arrive``
    False its one wait runs out after about ``limit_ns`` and the next
    ``sync_status`` raises TPA_ERR_DEVICE_TIMEOUT."""
    check("tpa_wait_probe", lib().tpa_wait_probe(int(limit_ns), 1 if arrive else 0, _stream_ptr(stream)))


def device_check() -> None:
    check("tpa_device_check", lib().tpa_device_check())
