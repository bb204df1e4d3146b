"""ctypes binding of libpkv.so: same entry points as include/pkv.h, torch tensors in.

Argument marshalling only: every step runs in the library's CUDA kernels on the
current torch CUDA stream.  There is no CPU path; if the library is missing the
calls raise.  Buffers the library needs (workspaces, outputs) are allocated here
with torch when the caller does not pass them.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

PKV_OK = 0
PKV_DTYPE_BF16 = 0
PKV_DTYPE_F32 = 1
STATUS_NAMES = {0: "PKV_OK", -1: "PKV_ERR_NULL", -2: "PKV_ERR_SHAPE", -3: "PKV_ERR_UNSUPPORTED",
                -4: "PKV_ERR_WORKSPACE", -5: "PKV_ERR_BAD_BLOCK", -6: "PKV_ERR_CUDA",
                -7: "PKV_ERR_ALIGN", -8: "PKV_ERR_TIMEOUT", -9: "PKV_ERR_OUT_OF_BLOCKS"}
PKV_BLOCK_KEY_EMPTY = 0xFFFFFFFFFFFFFFFF

# every exported symbol of include/pkv.h
EXPORTED = ("pkv_abi_version", "paged_kv_append", "paged_attention_workspace_size",
            "paged_attention_workspace_init", "paged_attention_forward", "spec_accept_workspace_size",
            "spec_accept_greedy", "pkv_last_error_string", "pkv_device_status",
            "paged_attention_forward_noalloc", "paged_tree_attention_forward", "spec_accept_tree_greedy",
            "spec_accept_sampled", "paged_block_hashes", "pkv_qrecord_bytes", "paged_kv_append_quant",
            "paged_attention_forward_quant", "paged_attention_forward_gather", "pkv_debug_set_wait_limit",
            "paged_block_index_init", "paged_block_allocate_workspace_size", "paged_block_allocate",
            "pkv_set_attention_kernel")
PKV_KERNEL_MMA_SYNC = 0
PKV_KERNEL_TCGEN05 = 1


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class _Pool(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class _QPool(ctypes.Structure):
    _fields_ = [("records", ctypes.c_void_p), ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("bits", ctypes.c_int32)]


class _BlockIndexC(ctypes.Structure):
    _fields_ = [("keys", ctypes.c_void_p), ("block_ids", ctypes.c_void_p), ("refcounts", ctypes.c_void_p),
                ("capacity", ctypes.c_int32), ("free_ids", ctypes.c_void_p), ("free_count", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = False):
    """Load libpkv.so (raises if it is not built; no fallback exists)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(f"libpkv.so is not built ({path}); run __graft_entry__.build()")
                _build.build()
            L = ctypes.CDLL(path)
            P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            L.pkv_abi_version.argtypes = []
            L.pkv_abi_version.restype = ctypes.c_int
            L.paged_kv_append.argtypes = [ctypes.POINTER(_Pool), P, i32, P, P, P, P, i32, i32, P]
            L.paged_kv_append.restype = ctypes.c_int
            L.paged_attention_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
            L.paged_attention_workspace_size.restype = sz
            L.paged_attention_workspace_init.argtypes = [P, sz, P]
            L.paged_attention_workspace_init.restype = ctypes.c_int
            L.paged_attention_forward.argtypes = [ctypes.POINTER(_Pool), P, P, P, i32, P, i32, i32, i32,
                                                  i32, i32, P, P, i32, ctypes.c_float, P, i32, P, sz, P]
            L.paged_attention_forward.restype = ctypes.c_int
            L.paged_attention_forward_noalloc.argtypes = [ctypes.POINTER(_Pool), P, P, P, i32, P, i32, i32,
                                                          i32, i32, i32, P, P, i32, ctypes.c_float, P, i32, P]
            L.paged_attention_forward_noalloc.restype = ctypes.c_int
            L.paged_tree_attention_forward.argtypes = [ctypes.POINTER(_Pool), P, P, P, i32, P, i32, i32, i32,
                                                       i32, i32, P, P, P, ctypes.c_float, P, i32, P, sz, P]
            L.paged_tree_attention_forward.restype = ctypes.c_int
            L.spec_accept_tree_greedy.argtypes = [P, i32, P, P, P, i32, i32, P, P, P, P, P, sz, P]
            L.spec_accept_tree_greedy.restype = ctypes.c_int
            L.spec_accept_sampled.argtypes = [P, i32, P, P, P, P, ctypes.c_uint64, ctypes.c_float, i32,
                                              ctypes.c_float, ctypes.c_float, i32, i32, P, P, P, P, P, sz, P]
            L.spec_accept_sampled.restype = ctypes.c_int
            L.paged_block_hashes.argtypes = [P, P, i32, i32, i32, ctypes.c_uint64, P, P, i32, P]
            L.paged_block_hashes.restype = ctypes.c_int
            L.pkv_qrecord_bytes.argtypes = [i32, i32, i32]
            L.pkv_qrecord_bytes.restype = sz
            L.paged_kv_append_quant.argtypes = [ctypes.POINTER(_QPool), P, i32, P, P, P, P, i32, i32, P]
            L.paged_kv_append_quant.restype = ctypes.c_int
            L.paged_attention_forward_quant.argtypes = [ctypes.POINTER(_QPool), P, P, P, i32, P, i32, i32, i32,
                                                        i32, i32, P, P, i32, ctypes.c_float, P, i32, P, sz, P]
            L.paged_attention_forward_quant.restype = ctypes.c_int
            L.paged_attention_forward_gather.argtypes = [ctypes.POINTER(_Pool), P, P, P, i32, P, i32, i32, P, P,
                                                         i32, i32, P, P, ctypes.c_float, P, i32, P, sz, P]
            L.paged_attention_forward_gather.restype = ctypes.c_int
            L.spec_accept_workspace_size.argtypes = [i32, i32]
            L.spec_accept_workspace_size.restype = sz
            L.spec_accept_greedy.argtypes = [P, i32, P, P, i32, i32, P, P, P, P, sz, P]
            L.spec_accept_greedy.restype = ctypes.c_int
            L.pkv_last_error_string.argtypes = []
            L.pkv_last_error_string.restype = ctypes.c_char_p
            L.pkv_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
            L.paged_block_index_init.argtypes = [ctypes.POINTER(_BlockIndexC), i32, P]
            L.paged_block_index_init.restype = ctypes.c_int
            L.paged_block_allocate_workspace_size.argtypes = [i32, i32]
            L.paged_block_allocate_workspace_size.restype = sz
            L.paged_block_allocate.argtypes = [ctypes.POINTER(_BlockIndexC), P, P, P, i32, i32, i32, P, P, P, sz, P]
            L.paged_block_allocate.restype = ctypes.c_int
            L.pkv_set_attention_kernel.argtypes = [i32]
            L.pkv_set_attention_kernel.restype = ctypes.c_int
            L.pkv_debug_set_wait_limit.argtypes = [ctypes.c_longlong]
            L.pkv_debug_set_wait_limit.restype = ctypes.c_int
            L.pkv_device_status.restype = ctypes.c_int
            _lib = L
        return _lib


def _check(rc: int):
    if rc != PKV_OK:
        raise PkvError(rc, lib().pkv_last_error_string().decode(errors="replace"))


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
        raise ValueError("expected a contiguous CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _pool(k_pool: torch.Tensor, v_pool: torch.Tensor) -> _Pool:
    for t in (k_pool, v_pool):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
            raise ValueError("K / V pools must be contiguous CUDA tensors")
    if k_pool.dtype != torch.bfloat16 or v_pool.dtype != torch.bfloat16:
        raise TypeError("K / V pools must be bfloat16")
    if k_pool.shape != v_pool.shape or k_pool.dim() != 4:
        raise ValueError("K / V pools must share one shape [num_blocks, H_kv, block_size, head_dim]")
    nb, hkv, bs, d = k_pool.shape
    return _Pool(k_pool.data_ptr(), v_pool.data_ptr(), nb, bs, hkv, d)


def paged_kv_append(k_pool, v_pool, block_tables, context_lens_old, new_starts, k_new, v_new,
                    stream=None) -> None:
    """Scatter k_new/v_new [R_new, H_kv, D] into the pools (see include/pkv.h)."""
    pool = _pool(k_pool, v_pool)
    _check(lib().paged_kv_append(ctypes.byref(pool), _dptr(block_tables), block_tables.shape[1],
                                 _dptr(context_lens_old), _dptr(new_starts), _dptr(k_new), _dptr(v_new),
                                 block_tables.shape[0], k_new.shape[0], _stream(stream)))


def paged_attention_workspace_size(num_seqs, total_q_rows, num_q_heads, num_kv_heads, head_dim,
                                   max_context_len) -> int:
    return int(lib().paged_attention_workspace_size(num_seqs, total_q_rows, num_q_heads, num_kv_heads,
                                                    head_dim, max_context_len))


def new_attention_workspace(num_seqs, total_q_rows, num_q_heads, num_kv_heads, head_dim, max_context_len,
                            device=None) -> torch.Tensor:
    """A workspace of the right size, zeroed (the calls do not depend on its contents)."""
    n = paged_attention_workspace_size(num_seqs, total_q_rows, num_q_heads, num_kv_heads, head_dim,
                                       max_context_len)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def paged_attention_forward(k_pool, v_pool, q, q_starts, block_tables, context_lens, *,
                            max_context_len: int, max_q_rows_per_seq: int,
                            kv_head_of_q_head=None, sinks=None, causal: bool = False,
                            scale: float = 0.0, out: Optional[torch.Tensor] = None,
                            out_dtype=torch.bfloat16, workspace: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """Paged attention (see include/pkv.h).  q: bf16 [R, H_q, D]; returns out [R, H_q, D].

    kv_head_of_q_head is a host sequence of ints (or None); sinks a CUDA float32 [H_q] or None.
    """
    pool = _pool(k_pool, v_pool)
    R, Hq, D = q.shape
    S = block_tables.shape[0]
    if out is None:
        out = torch.empty((R, Hq, D), dtype=out_dtype, device=q.device)
    dt = PKV_DTYPE_F32 if out.dtype == torch.float32 else PKV_DTYPE_BF16
    if workspace is None:
        workspace = new_attention_workspace(S, R, Hq, pool.num_kv_heads, D, max_context_len, q.device)
    hmap = None
    if kv_head_of_q_head is not None:
        arr = (ctypes.c_int32 * Hq)(*[int(x) for x in kv_head_of_q_head])
        hmap = ctypes.cast(arr, ctypes.c_void_p)
    _check(lib().paged_attention_forward(
        ctypes.byref(pool), _dptr(q), _dptr(q_starts), _dptr(block_tables), block_tables.shape[1],
        _dptr(context_lens), S, R, int(max_context_len), int(max_q_rows_per_seq), Hq, hmap,
        _dptr(sinks), int(bool(causal)), float(scale), _dptr(out), dt, _dptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def paged_attention_forward_gather(k_pool, v_pool, q, q_starts, block_tables, context_lens, key_idx, key_counts, *,
                                   kv_head_of_q_head=None, sinks=None, scale: float = 0.0,
                                   out: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                                   workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Attention of each row over its own key list (see include/pkv.h).

    key_idx: CUDA int32 [R, max_keys]; key_counts: CUDA int32 [R]."""
    pool = _pool(k_pool, v_pool)
    R, Hq, D = q.shape
    S = block_tables.shape[0]
    max_keys = key_idx.shape[1]
    if out is None:
        out = torch.empty((R, Hq, D), dtype=out_dtype, device=q.device)
    dt = PKV_DTYPE_F32 if out.dtype == torch.float32 else PKV_DTYPE_BF16
    if workspace is None:
        workspace = new_attention_workspace(S, R, Hq, pool.num_kv_heads, D, max_keys, q.device)
    hmap = None
    if kv_head_of_q_head is not None:
        arr = (ctypes.c_int32 * Hq)(*[int(x) for x in kv_head_of_q_head])
        hmap = ctypes.cast(arr, ctypes.c_void_p)
    _check(lib().paged_attention_forward_gather(
        ctypes.byref(pool), _dptr(q), _dptr(q_starts), _dptr(block_tables), block_tables.shape[1],
        _dptr(context_lens), S, R, _dptr(key_idx), _dptr(key_counts), int(max_keys), Hq, hmap, _dptr(sinks),
        float(scale), _dptr(out), dt, _dptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return out


def qrecord_bytes(block_size: int, head_dim: int, bits: int) -> int:
    return int(lib().pkv_qrecord_bytes(int(block_size), int(head_dim), int(bits)))


def _qpool(records: torch.Tensor, block_size: int, head_dim: int, bits: int) -> _QPool:
    if not (isinstance(records, torch.Tensor) and records.is_cuda and records.is_contiguous()):
        raise ValueError("records must be a contiguous CUDA tensor")
    if records.dtype != torch.uint8 or records.dim() != 3:
        raise TypeError("records must be uint8 [num_blocks, H_kv, record_bytes]")
    nb, hkv, rb = records.shape
    if rb != qrecord_bytes(block_size, head_dim, bits):
        raise ValueError("record size does not match the codec")
    return _QPool(records.data_ptr(), nb, int(block_size), hkv, int(head_dim), int(bits))


def paged_kv_append_quant(records, block_size, head_dim, bits, block_tables, context_lens_old, new_starts,
                          k_new, v_new, stream=None) -> None:
    """Quantise k_new/v_new [R_new, H_kv, D] (bf16) into the record pool uint8 [nb, H_kv, R]."""
    pool = _qpool(records, block_size, head_dim, bits)
    _check(lib().paged_kv_append_quant(ctypes.byref(pool), _dptr(block_tables), block_tables.shape[1],
                                       _dptr(context_lens_old), _dptr(new_starts), _dptr(k_new), _dptr(v_new),
                                       block_tables.shape[0], k_new.shape[0], _stream(stream)))


def paged_attention_forward_quant(records, block_size, head_dim, bits, q, q_starts, block_tables, context_lens, *,
                                  max_context_len: int, max_q_rows_per_seq: int, kv_head_of_q_head=None,
                                  sinks=None, causal: bool = False, scale: float = 0.0,
                                  out: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                                  workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Paged attention over a quantised record pool (see include/pkv.h)."""
    pool = _qpool(records, block_size, head_dim, bits)
    R, Hq, D = q.shape
    S = block_tables.shape[0]
    if out is None:
        out = torch.empty((R, Hq, D), dtype=out_dtype, device=q.device)
    dt = PKV_DTYPE_F32 if out.dtype == torch.float32 else PKV_DTYPE_BF16
    if workspace is None:
        workspace = new_attention_workspace(S, R, Hq, pool.num_kv_heads, D, max_context_len, q.device)
    hmap = None
    if kv_head_of_q_head is not None:
        arr = (ctypes.c_int32 * Hq)(*[int(x) for x in kv_head_of_q_head])
        hmap = ctypes.cast(arr, ctypes.c_void_p)
    _check(lib().paged_attention_forward_quant(
        ctypes.byref(pool), _dptr(q), _dptr(q_starts), _dptr(block_tables), block_tables.shape[1],
        _dptr(context_lens), S, R, int(max_context_len), int(max_q_rows_per_seq), Hq, hmap,
        _dptr(sinks), int(bool(causal)), float(scale), _dptr(out), dt, _dptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def paged_tree_attention_forward(k_pool, v_pool, q, q_starts, block_tables, context_lens, tree_masks, *,
                                 max_context_len: int, max_q_rows_per_seq: int, kv_head_of_q_head=None,
                                 sinks=None, scale: float = 0.0, out: Optional[torch.Tensor] = None,
                                 out_dtype=torch.bfloat16, workspace: Optional[torch.Tensor] = None,
                                 stream=None) -> torch.Tensor:
    """Tree verify attention (see include/pkv.h); tree_masks: CUDA int32/uint32 [R]."""
    pool = _pool(k_pool, v_pool)
    R, Hq, D = q.shape
    S = block_tables.shape[0]
    if out is None:
        out = torch.empty((R, Hq, D), dtype=out_dtype, device=q.device)
    dt = PKV_DTYPE_F32 if out.dtype == torch.float32 else PKV_DTYPE_BF16
    if workspace is None:
        workspace = new_attention_workspace(S, R, Hq, pool.num_kv_heads, D, max_context_len, q.device)
    hmap = None
    if kv_head_of_q_head is not None:
        arr = (ctypes.c_int32 * Hq)(*[int(x) for x in kv_head_of_q_head])
        hmap = ctypes.cast(arr, ctypes.c_void_p)
    _check(lib().paged_tree_attention_forward(
        ctypes.byref(pool), _dptr(q), _dptr(q_starts), _dptr(block_tables), block_tables.shape[1],
        _dptr(context_lens), S, R, int(max_context_len), int(max_q_rows_per_seq), Hq, hmap, _dptr(sinks),
        _dptr(tree_masks), float(scale), _dptr(out), dt, _dptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def spec_accept_tree_greedy(logits, q_starts, draft_tokens, parents, *, argmax_out=None, accept_len=None,
                            out_tokens=None, accepted_rows=None, workspace=None, stream=None):
    """Greedy accept over draft trees (see include/pkv.h);
    returns (argmax [R], accept_len [S], out_tokens [R], accepted_rows [R])."""
    R, V = logits.shape
    S = q_starts.shape[0] - 1
    dev = logits.device
    mk = lambda n: torch.empty(n, dtype=torch.int32, device=dev)  # noqa: E731
    argmax_out = mk(R) if argmax_out is None else argmax_out
    accept_len = mk(S) if accept_len is None else accept_len
    out_tokens = mk(R) if out_tokens is None else out_tokens
    accepted_rows = mk(R) if accepted_rows is None else accepted_rows
    if workspace is None:
        workspace = torch.empty(max(spec_accept_workspace_size(R, V), 256), dtype=torch.uint8, device=dev)
    _check(lib().spec_accept_tree_greedy(_dptr(logits), V, _dptr(q_starts), _dptr(draft_tokens), _dptr(parents),
                                         S, R, _dptr(argmax_out), _dptr(accept_len), _dptr(out_tokens),
                                         _dptr(accepted_rows), _dptr(workspace), workspace.numel(),
                                         _stream(stream)))
    return argmax_out, accept_len, out_tokens, accepted_rows


def spec_accept_sampled(logits, q_starts, draft_tokens, positions, *, seed: int, temperature: float,
                        min_p: float = 0.0, top_k: int = 0, top_p: float = 1.0, parents=None, sampled_out=None,
                        accept_len=None, out_tokens=None, accepted_rows=None, workspace=None, stream=None):
    """Keyed sampled accept (see include/pkv.h);
    returns (sampled [R], accept_len [S], out_tokens [R], accepted_rows [R])."""
    R, V = logits.shape
    S = q_starts.shape[0] - 1
    dev = logits.device
    mk = lambda n: torch.empty(n, dtype=torch.int32, device=dev)  # noqa: E731
    sampled_out = mk(R) if sampled_out is None else sampled_out
    accept_len = mk(S) if accept_len is None else accept_len
    out_tokens = mk(R) if out_tokens is None else out_tokens
    accepted_rows = mk(R) if accepted_rows is None else accepted_rows
    if workspace is None:
        workspace = torch.empty(sampled_accept_workspace_size(R, V), dtype=torch.uint8, device=dev)
    _check(lib().spec_accept_sampled(_dptr(logits), V, _dptr(q_starts), _dptr(draft_tokens), _dptr(parents),
                                     _dptr(positions), int(seed), float(temperature), int(top_k), float(top_p),
                                     float(min_p), S, R,
                                     _dptr(sampled_out), _dptr(accept_len), _dptr(out_tokens),
                                     _dptr(accepted_rows), _dptr(workspace), workspace.numel(), _stream(stream)))
    return sampled_out, accept_len, out_tokens, accepted_rows


def spec_accept_workspace_size(total_rows, vocab) -> int:
    return int(lib().spec_accept_workspace_size(total_rows, vocab))


def sampled_accept_workspace_size(total_rows, vocab) -> int:
    """Workspace bytes spec_accept_sampled needs (see include/pkv.h)."""
    return 2 * spec_accept_workspace_size(total_rows, vocab) + (total_rows * 8 + 255) // 256 * 256


def spec_accept_greedy(logits, q_starts, draft_tokens, *, argmax_out=None, accept_len=None,
                       out_tokens=None, workspace=None, stream=None):
    """Greedy accept (see include/pkv.h); returns (argmax [R], accept_len [S], out_tokens [R])."""
    R, V = logits.shape
    S = q_starts.shape[0] - 1
    dev = logits.device
    if argmax_out is None:
        argmax_out = torch.empty(R, dtype=torch.int32, device=dev)
    if accept_len is None:
        accept_len = torch.empty(S, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(R, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(spec_accept_workspace_size(R, V), 256), dtype=torch.uint8, device=dev)
    _check(lib().spec_accept_greedy(_dptr(logits), V, _dptr(q_starts), _dptr(draft_tokens), S, R,
                                    _dptr(argmax_out), _dptr(accept_len), _dptr(out_tokens),
                                    _dptr(workspace), workspace.numel(), _stream(stream)))
    return argmax_out, accept_len, out_tokens


def paged_block_hashes(tokens, token_starts, block_size: int, seed: int, max_blocks_per_seq: int, *,
                       chain_in=None, out=None, stream=None):
    """Chained content keys of full blocks (see include/pkv.h).

    tokens int32 [T], token_starts int32 [S+1], chain_in int64 [S] or None (the uint64
    key bits); returns int64 [S, max_blocks_per_seq] holding the uint64 key bits."""
    S = token_starts.shape[0] - 1
    if out is None:
        out = torch.empty((S, max_blocks_per_seq), dtype=torch.int64, device=token_starts.device)
    _check(lib().paged_block_hashes(_dptr(tokens), _dptr(token_starts), S, tokens.numel(), int(block_size),
                                    int(seed) & 0xFFFFFFFFFFFFFFFF, _dptr(chain_in), _dptr(out),
                                    int(max_blocks_per_seq), _stream(stream)))
    return out


def device_status(stream=None):
    """Synchronise and read/clear the device status word; returns (status, bits)."""
    bits = ctypes.c_int32(0)
    rc = lib().pkv_device_status(_stream(stream), ctypes.byref(bits))
    return rc, bits.value


def debug_set_wait_limit(cycles: int):
    """Test hook: the SM-cycle limit of the attention pipeline's stage waits in later calls
    (0: give up at once, taking the kernels' timeout path; negative: the default)."""
    _check(lib().pkv_debug_set_wait_limit(int(cycles)))


class BlockIndex:
    """Device block index and free stack for paged_block_allocate (see include/pkv.h).

    keys int64 [capacity] (the uint64 keys' bits), block_ids / refcounts int32 [capacity],
    free_ids int32 [n], free_count int32 [1]; all CUDA tensors owned here."""

    def __init__(self, capacity: int, free_ids: torch.Tensor, device="cuda", stream=None):
        if capacity < 1 or capacity & (capacity - 1):
            raise ValueError("capacity must be a positive power of two")
        self.keys = torch.empty(capacity, dtype=torch.int64, device=device)
        self.block_ids = torch.empty(capacity, dtype=torch.int32, device=device)
        self.refcounts = torch.empty(capacity, dtype=torch.int32, device=device)
        self.free_ids = free_ids.to(device=device, dtype=torch.int32).contiguous()
        self.free_count = torch.empty(1, dtype=torch.int32, device=device)
        _check(lib().paged_block_index_init(ctypes.byref(self._c()), self.free_ids.numel(), _stream(stream)))

    def _c(self) -> _BlockIndexC:
        return _BlockIndexC(self.keys.data_ptr(), self.block_ids.data_ptr(), self.refcounts.data_ptr(),
                            self.keys.numel(), self.free_ids.data_ptr(), self.free_count.data_ptr())

    def entries(self):
        """The index as {key (uint64 int): (block id, refcount)} (host copy of the occupied slots)."""
        k = self.keys.cpu().numpy().view("uint64")
        i = self.block_ids.cpu().numpy()
        r = self.refcounts.cpu().numpy()
        return {int(a): (int(b) if b >= 0 else -1, int(c)) for a, b, c in zip(k, i, r)
                if int(a) != PKV_BLOCK_KEY_EMPTY}


def paged_block_allocate(index: BlockIndex, block_keys, context_lens, first_block, block_size: int, block_tables,
                         *, fresh: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """Fill block_tables [S, max_blocks] in place from the index (see include/pkv.h); returns
    fresh int32 [S, max_blocks] (1 where a block was allocated that the caller must fill)."""
    S, mb = block_tables.shape
    if block_keys.dtype not in (torch.int64, torch.uint64) or tuple(block_keys.shape) != (S, mb):
        raise ValueError("block_keys must be 64-bit [num_seqs, max_blocks_per_seq]")
    if fresh is None:
        fresh = torch.empty((S, mb), dtype=torch.int32, device=block_tables.device)
    if workspace is None:
        n = lib().paged_block_allocate_workspace_size(S, mb)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=block_tables.device)
    _check(lib().paged_block_allocate(ctypes.byref(index._c()), _dptr(block_keys), _dptr(context_lens),
                                      _dptr(first_block), S, int(block_size), mb, _dptr(block_tables), _dptr(fresh),
                                      _dptr(workspace), workspace.numel(), _stream(stream)))
    return fresh


def set_attention_kernel(which: int):
    """Choose the kernel of the bf16 attention calls (PKV_KERNEL_MMA_SYNC or PKV_KERNEL_TCGEN05)."""
    _check(lib().pkv_set_attention_kernel(int(which)))
