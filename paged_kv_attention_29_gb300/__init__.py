"""Paged GQA attention for GB300 (sm_103a): Python binding of libpkv.

The binding only marshals arguments: it checks tensor dtypes, devices and
shapes, passes raw device pointers and the current CUDA stream to the C ABI
(``include/pkv.h``), and turns a non-zero status into :class:`PkvError`.
Every step of the path runs in the library's CUDA kernels.  There is no CPU
fallback: if ``libpkv.so`` has not been built, :func:`load` raises.

Build the library with ``python -m paged_kv_attention_29_gb300.build``.

Functions carry the C names:

=========================  ================================================
``pkv_slot_mapping``       slot of each new token (block table lookup)
``pkv_store_kvcache``      scatter new K/V rows into the paged pools
``pkv_prefill_varlen``     varlen prefill attention with the offset causal mask
``pkv_decode``             single-token decode attention over block tables
``pkv_sample``             temperature sampling by exponential race
=========================  ================================================
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "PkvError", "load", "lib_path", "pkv_abi_version", "pkv_status_string", "pkv_slot_mapping",
    "pkv_store_kvcache", "pkv_prefill_workspace_size", "pkv_prefill_varlen", "pkv_prefill_plan",
    "pkv_prefill_varlen_planned",
    "pkv_decode_workspace_size", "pkv_decode", "pkv_sample", "pkv_get_device_error", "pkv_check_wait_timeout",
    "WAIT_CHECK_INFO",
    "decode_workspace", "pkv_decode_append", "pkv_decode_noalloc", "pkv_sample_dev", "pkv_rope_store_kvcache", "DecodeAppendCall", "DEVERR",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpkv.so")
_lib: Optional[ctypes.CDLL] = None

DEVERR = {0: "none", 1: "block id outside pool", 2: "slot outside pool", 3: "sequence lengths",
          4: "temperature", 5: "pipeline wait timed out", 6: "position past block table",
          7: "no prefill plan for these arguments in the workspace"}

_c_int32 = ctypes.c_int32
_c_int64 = ctypes.c_int64
_c_size = ctypes.c_size_t
_c_ptr = ctypes.c_void_p
_c_float = ctypes.c_float
_c_u64 = ctypes.c_uint64


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {pkv_status_string(status)} ({status})")


def lib_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libpkv.so (once).  Raises if it was not built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing; build it with `python -m paged_kv_attention_29_gb300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    sig = {
        "pkv_abi_version": (_c_int32, []),
        "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "pkv_slot_mapping": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_int32, _c_int32,
                                            _c_int32, _c_int32, _c_ptr, _c_ptr]),
        "pkv_store_kvcache": (ctypes.c_int, [_c_ptr, _c_ptr, _c_int64, _c_int64, _c_int64, _c_ptr, _c_ptr,
                                             _c_ptr, _c_int32, _c_int32, _c_int32, _c_int32, _c_ptr]),
        "pkv_rope_store_kvcache": (ctypes.c_int, [_c_ptr, _c_int64, _c_ptr, _c_int64, _c_ptr, _c_int64, _c_ptr,
                                                  _c_int64, _c_ptr, _c_int64, _c_int32, _c_int32, _c_int32,
                                                  ctypes.c_double, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_int32,
                                                  _c_ptr]),
        "pkv_prefill_workspace_size": (_c_size, [_c_int32] * 5),
        "pkv_prefill_varlen": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_int32,
                                              _c_int32, _c_int32, _c_int32, _c_int32, _c_int32, _c_int32,
                                              _c_int32, _c_int32, _c_float, _c_ptr, _c_ptr, _c_size, _c_ptr]),
        "pkv_prefill_plan": (ctypes.c_int, [_c_ptr, _c_ptr, _c_int32, _c_int32, _c_int32, _c_int32, _c_int32,
                                            _c_int32, _c_int32, _c_int32, _c_int32, _c_ptr, _c_size, _c_ptr]),
        "pkv_prefill_varlen_planned": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32,
                                                      _c_int32, _c_int32, _c_int32, _c_int32, _c_int32, _c_int32,
                                                      _c_int32, _c_int32, _c_int32, _c_float, _c_ptr, _c_ptr,
                                                      _c_size, _c_ptr]),
        "pkv_decode_workspace_size": (_c_size, [_c_int32] * 4),
        "pkv_decode": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_ptr, _c_int32, _c_int32,
                                      _c_int32, _c_int32, _c_int32, _c_int32, _c_int32, _c_float, _c_ptr,
                                      _c_ptr, _c_size, _c_ptr]),
        "pkv_decode_append": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_ptr,
                                             _c_int32, _c_int32, _c_int32, _c_int32, _c_int32, _c_int32,
                                             _c_int32, _c_float, _c_ptr, _c_ptr, _c_ptr, _c_size, _c_ptr]),
        "pkv_decode_noalloc": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int32, _c_ptr, _c_int32,
                                              _c_int32, _c_int32, _c_int32, _c_int32, _c_int32, _c_int32,
                                              _c_float, _c_ptr, _c_ptr]),
        "pkv_sample": (ctypes.c_int, [_c_ptr, _c_int32, _c_int32, _c_int64, _c_ptr, _c_u64, _c_u64, _c_ptr,
                                      _c_ptr]),
        "pkv_sample_dev": (ctypes.c_int, [_c_ptr, _c_int32, _c_int32, _c_int64, _c_ptr, _c_ptr, _c_ptr, _c_ptr]),
        "pkv_get_device_error": (ctypes.c_int, [ctypes.POINTER(_c_int32), ctypes.POINTER(_c_int32), _c_int32]),
        "pkv_check_wait_timeout": (ctypes.c_int, [ctypes.c_void_p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype, ndim=None, contiguous=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libpkv has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class _on_device:
    """Run a library call with the tensors' device current.

    The library launches on the current device and looks up per-device state
    (error word, kernel attributes, scratch) there, so every tensor of a call
    must sit on one device and that device must be current.  Makes it current
    for the duration of the call when it is not already; a stream given by the
    caller must belong to it."""

    __slots__ = ("dev", "prev")

    def __init__(self, *tensors, stream=None):
        dev = None
        for t in tensors:
            if t is None:
                continue
            if dev is None:
                dev = t.device
            elif t.device != dev:
                raise ValueError(f"all tensors of a call must be on one device (got {dev} and {t.device})")
        self.dev = dev.index if dev is not None else torch.cuda.current_device()
        if stream is not None and stream.device.index != self.dev:
            raise ValueError(f"stream is on cuda:{stream.device.index}, tensors on cuda:{self.dev}")
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.dev:
            self.prev = cur
            torch.cuda.set_device(self.dev)
        return self

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
        return False


def _row_stride(logits: torch.Tensor) -> int:
    """Elements between rows; a single row's stride is meaningless (it may be 0), so use its length."""
    return logits.stride(0) if logits.shape[0] > 1 else logits.shape[1]


def _raise(status: int, where: str):
    if status != 0:
        raise PkvError(status, where)


# ---------------------------------------------------------------------------
# API
# ---------------------------------------------------------------------------

def pkv_abi_version() -> int:
    return int(load().pkv_abi_version())


def pkv_status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def pkv_slot_mapping(block_tables: torch.Tensor, num_blocks: int, block_size: int,
                     slot_mapping: torch.Tensor, *, cu_seqlens_q: Optional[torch.Tensor] = None,
                     cu_seqlens_k: Optional[torch.Tensor] = None, context_lens: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """Fill ``slot_mapping`` (int32 [total_q]) with the slot of every new token."""
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(slot_mapping, "slot_mapping", torch.int32, 1)
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k), ("context_lens", context_lens)):
        if t is not None:
            _check(t, name, torch.int32, 1)
    num_seqs = block_tables.shape[0]
    with _on_device(block_tables, slot_mapping, cu_seqlens_q, cu_seqlens_k, context_lens, stream=stream):
        _raise(load().pkv_slot_mapping(_ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(context_lens), _ptr(block_tables),
                                   block_tables.shape[1], num_seqs, slot_mapping.shape[0], block_size, num_blocks,
                                   _ptr(slot_mapping), _stream(stream)), "pkv_slot_mapping")
    return slot_mapping


def _pool_shape(k_cache: torch.Tensor):
    _check(k_cache, "k_cache", torch.bfloat16, 4)
    nb, bs, hkv, d = k_cache.shape
    return nb, bs, hkv, d


def pkv_store_kvcache(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, stream=None) -> None:
    """k_cache[slot // bs, slot % bs] = k[i] (and v) for every row i; slot < 0 skips."""
    nb, bs, hkv, d = _pool_shape(k_cache)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    for name, t in (("k", k), ("v", v)):
        _check(t, name, torch.bfloat16, 3, contiguous=False)
        if tuple(t.shape[1:]) != (hkv, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{name} must be [n, {hkv}, {d}] with contiguous rows")
    _check(slot_mapping, "slot_mapping", torch.int32, 1)
    n = k.shape[0]
    if v.shape[0] != n or slot_mapping.shape[0] != n:
        raise ValueError("k, v and slot_mapping disagree on the token count")
    with _on_device(k, v, slot_mapping, k_cache, v_cache, stream=stream):
        _raise(load().pkv_store_kvcache(_ptr(k), _ptr(v), n, k.stride(0), v.stride(0), _ptr(slot_mapping),
                                        _ptr(k_cache), _ptr(v_cache), nb, bs, hkv, d, _stream(stream)),
               "pkv_store_kvcache")


def pkv_rope_store_kvcache(q: Optional[torch.Tensor], k: torch.Tensor, v: torch.Tensor, positions: torch.Tensor,
                           slot_mapping: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           rope_base: float, q_out: Optional[torch.Tensor] = None,
                           stream=None) -> Optional[torch.Tensor]:
    """Rotate q and k by `positions` (rotary embedding), write rotated k and plain v to the pool.

    Returns the rotated q (a new tensor, or `q_out`; pass ``q_out=q`` to rotate in place)."""
    nb, bs, hkv, d = _pool_shape(k_cache)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    for name, t in (("k", k), ("v", v)):
        _check(t, name, torch.bfloat16, 3, contiguous=False)
        if tuple(t.shape[1:]) != (hkv, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{name} must be [n, {hkv}, {d}] with contiguous rows")
    _check(positions, "positions", torch.int32, 1)
    _check(slot_mapping, "slot_mapping", torch.int32, 1)
    n = k.shape[0]
    if v.shape[0] != n or slot_mapping.shape[0] != n or positions.shape[0] != n:
        raise ValueError("k, v, positions and slot_mapping disagree on the token count")
    hq = 0
    if q is not None:
        _check(q, "q", torch.bfloat16, 3, contiguous=False)
        hq = q.shape[1]
        if q.shape[0] != n or q.shape[2] != d or q.stride(2) != 1 or q.stride(1) != d:
            raise ValueError(f"q must be [n, Hq, {d}] with contiguous rows")
        if q_out is None:
            q_out = torch.empty(n, hq, d, dtype=torch.bfloat16, device=q.device)
        _check(q_out, "q_out", torch.bfloat16, 3, contiguous=False)
        if tuple(q_out.shape) != tuple(q.shape) or q_out.stride(2) != 1 or q_out.stride(1) != d:
            raise ValueError("q_out must match q's shape with contiguous rows")
    elif q_out is not None:
        raise ValueError("q_out given without q")
    with _on_device(q, q_out, k, v, positions, slot_mapping, k_cache, v_cache, stream=stream):
        _raise(load().pkv_rope_store_kvcache(_ptr(q), q.stride(0) if q is not None else 0, _ptr(q_out),
                                             q_out.stride(0) if q_out is not None else 0, _ptr(k), k.stride(0),
                                             _ptr(v), v.stride(0), _ptr(positions), n, hq, hkv, d, float(rope_base),
                                             _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), nb, bs,
                                             _stream(stream)),
               "pkv_rope_store_kvcache")
    return q_out


def pkv_prefill_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                               max_seqlen_q: int) -> int:
    return int(load().pkv_prefill_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, max_seqlen_q))


def _prefill(entry: str, q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, max_seqlen_q, max_seqlen_k,
             softmax_scale, out, workspace, stream):
    nb, bs, hkv, d = _pool_shape(k_cache)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    _check(q, "q", torch.bfloat16, 3)
    _check(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _check(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    _check(block_tables, "block_tables", torch.int32, 2)
    total_q, hq, dq = q.shape
    if dq != d:
        raise ValueError("q head_dim differs from the pool's")
    num_seqs = cu_seqlens_q.shape[0] - 1
    if cu_seqlens_k.shape[0] != num_seqs + 1 or block_tables.shape[0] != num_seqs:
        raise ValueError("cu_seqlens_q, cu_seqlens_k and block_tables disagree on the sequence count")
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 3)
    if workspace is None:
        if entry == "pkv_prefill_varlen_planned":
            raise ValueError("a planned prefill needs the workspace its plan was written to")
        n = pkv_prefill_workspace_size(num_seqs, hq, hkv, d, int(max_seqlen_q))
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on_device(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, out, workspace, stream=stream):
        _raise(getattr(load(), entry)(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                      _ptr(block_tables), block_tables.shape[1], num_seqs, total_q, int(max_seqlen_q),
                                      int(max_seqlen_k), hq, hkv, d, bs, nb, float(softmax_scale), _ptr(out),
                                      _ptr(workspace), ws_bytes, _stream(stream)), entry)
    return out


def pkv_prefill_varlen(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, cu_seqlens_q: torch.Tensor,
                       cu_seqlens_k: torch.Tensor, block_tables: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int,
                       softmax_scale: float, out: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Varlen prefill attention over the paged cache (the new tokens' K/V already stored)."""
    return _prefill("pkv_prefill_varlen", q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables,
                    max_seqlen_q, max_seqlen_k, softmax_scale, out, workspace, stream)


def pkv_prefill_plan(cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, total_q: int, max_seqlen_q: int,
                     max_seqlen_k: int, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                     max_blocks_per_seq: int, workspace: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """Write the prefill work list for one batch into `workspace` (allocated if None) and return
    it; every layer's pkv_prefill_varlen_planned call on this batch then reuses it."""
    _check(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _check(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    num_seqs = cu_seqlens_q.shape[0] - 1
    if cu_seqlens_k.shape[0] != num_seqs + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k disagree on the sequence count")
    if workspace is None:
        n = pkv_prefill_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, int(max_seqlen_q))
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=cu_seqlens_q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on_device(cu_seqlens_q, cu_seqlens_k, workspace, stream=stream):
        _raise(load().pkv_prefill_plan(_ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(max_blocks_per_seq), num_seqs,
                                       int(total_q), int(max_seqlen_q), int(max_seqlen_k), int(num_heads),
                                       int(num_kv_heads), int(head_dim), int(block_size), _ptr(workspace), ws_bytes,
                                       _stream(stream)), "pkv_prefill_plan")
    return workspace


def pkv_prefill_varlen_planned(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, block_tables: torch.Tensor,
                               max_seqlen_q: int, max_seqlen_k: int, softmax_scale: float, workspace: torch.Tensor,
                               out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """pkv_prefill_varlen on the work list pkv_prefill_plan left in `workspace` (no planning launch)."""
    return _prefill("pkv_prefill_varlen_planned", q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables,
                    max_seqlen_q, max_seqlen_k, softmax_scale, out, workspace, stream)


def pkv_decode_workspace_size(batch: int, num_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(load().pkv_decode_workspace_size(batch, num_heads, num_kv_heads, head_dim))


def decode_workspace(batch: int, num_heads: int, num_kv_heads: int, head_dim: int, device=None) -> torch.Tensor:
    """A uint8 device buffer of the size pkv_decode needs (256-byte aligned by the allocator)."""
    n = pkv_decode_workspace_size(batch, num_heads, num_kv_heads, head_dim)
    if n == 0:
        raise PkvError(2, "pkv_decode_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def pkv_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
               context_lens: torch.Tensor, max_context_len: int, softmax_scale: float,
               out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """Decode attention: one query token per sequence over context_lens[b] cached keys."""
    nb, bs, hkv, d = _pool_shape(k_cache)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    _check(q, "q", torch.bfloat16, 3)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    batch, hq, dq = q.shape
    if dq != d or context_lens.shape[0] != batch or block_tables.shape[0] != batch:
        raise ValueError("q, context_lens and block_tables disagree")
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 3)
    if workspace is None:
        workspace = decode_workspace(batch, hq, hkv, d, q.device)
    _check(workspace, "workspace", torch.uint8, 1)
    with _on_device(q, k_cache, v_cache, block_tables, context_lens, out, workspace, stream=stream):
        _raise(load().pkv_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                                 _ptr(context_lens), batch, int(max_context_len), hq, hkv, d, bs, nb,
                                 float(softmax_scale), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)),
               "pkv_decode")
    return out


def pkv_decode_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                      max_context_len: int, softmax_scale: float, out: Optional[torch.Tensor] = None,
                      slot_mapping: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """Decode step with the KV write fused in: the new token's K/V go to position
    context_lens[b] - 1, then decode attention over context_lens[b] keys."""
    nb, bs, hkv, d = _pool_shape(k_cache)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    _check(q, "q", torch.bfloat16, 3)
    _check(k_new, "k_new", torch.bfloat16, 3)
    _check(v_new, "v_new", torch.bfloat16, 3)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    batch, hq, dq = q.shape
    if dq != d or context_lens.shape[0] != batch or block_tables.shape[0] != batch:
        raise ValueError("q, context_lens and block_tables disagree")
    if tuple(k_new.shape) != (batch, hkv, d) or tuple(v_new.shape) != (batch, hkv, d):
        raise ValueError(f"k_new / v_new must be [{batch}, {hkv}, {d}]")
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 3)
    if slot_mapping is not None:
        _check(slot_mapping, "slot_mapping", torch.int32, 1)
    if workspace is None:
        workspace = decode_workspace(batch, hq, hkv, d, q.device)
    _check(workspace, "workspace", torch.uint8, 1)
    with _on_device(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, slot_mapping, workspace,
                    stream=stream):
        _raise(load().pkv_decode_append(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), batch,
                                        int(max_context_len), hq, hkv, d, bs, nb, float(softmax_scale), _ptr(out),
                                        _ptr(slot_mapping), _ptr(workspace), workspace.numel(), _stream(stream)),
               "pkv_decode_append")
    return out


class DecodeAppendCall:
    """pkv_decode_append on a fixed set of buffers, checked and marshalled once.

    A serving loop calls the same step on the same buffers (inputs copied into
    them) every iteration; this object does the argument checks and the ctypes
    marshalling at construction, so each call is one C-ABI call.  The buffers
    must stay alive and keep their shapes; their contents may change freely."""

    def __init__(self, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, max_context_len,
                 softmax_scale, out, slot_mapping=None, workspace=None, stream=None):
        # one validating call through the checked path (it also runs the step once)
        pkv_decode_append(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, max_context_len,
                          softmax_scale, out=out, slot_mapping=slot_mapping, workspace=workspace, stream=stream)
        nb, bs, hkv, d = _pool_shape(k_cache)
        batch, hq, _ = q.shape
        if workspace is None:
            workspace = decode_workspace(batch, hq, hkv, d, q.device)
        self._keep = (q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, slot_mapping, workspace)
        self._fn = load().pkv_decode_append
        self._args = (_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                      block_tables.shape[1], _ptr(context_lens), batch, int(max_context_len), hq, hkv, d, bs, nb,
                      float(softmax_scale), _ptr(out), _ptr(slot_mapping), _ptr(workspace), workspace.numel())
        self._stream = None if stream is None else _stream(stream)   # None: the current stream per call
        self._dev = q.device.index
        self.out = out

    def __call__(self, stream=None) -> torch.Tensor:
        """Launch on `stream`, else on the stream given at construction, else on the current stream
        of the buffers' device (so a call made while a CUDA graph is being captured is captured)."""
        if stream is None and torch.cuda.current_device() == self._dev:
            s = self._stream if self._stream is not None else _stream()
            _raise(self._fn(*self._args, s), "pkv_decode_append")
            return self.out
        with _on_device(self.out, stream=stream):
            s = _stream(stream) if stream is not None else (self._stream if self._stream is not None else _stream())
            _raise(self._fn(*self._args, s), "pkv_decode_append")
        return self.out


def pkv_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                       context_lens: torch.Tensor, max_context_len: int, softmax_scale: float,
                       out: torch.Tensor, stream=None) -> torch.Tensor:
    """pkv_decode for callers that cannot allocate: the scratch lives inside the
    library (4 MiB per GPU, shared by all calls, so overlapping calls race) and
    ``out`` must be given.  A batch too large for that scratch raises PkvError."""
    nb, bs, hkv, d = _pool_shape(k_cache)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    _check(q, "q", torch.bfloat16, 3)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    _check(out, "out", torch.bfloat16, 3)
    batch, hq, dq = q.shape
    if dq != d or context_lens.shape[0] != batch or block_tables.shape[0] != batch or out.shape != q.shape:
        raise ValueError("q, out, context_lens and block_tables disagree")
    with _on_device(q, k_cache, v_cache, block_tables, context_lens, out, stream=stream):
        _raise(load().pkv_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                         block_tables.shape[1], _ptr(context_lens), batch, int(max_context_len), hq,
                                         hkv, d, bs, nb, float(softmax_scale), _ptr(out), _stream(stream)),
               "pkv_decode_noalloc")
    return out


def pkv_sample(logits: torch.Tensor, temperatures: torch.Tensor, seed: int, offset: int = 0,
               out_ids: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Exponential-race temperature sampling; returns int64 ids [batch]."""
    _check(logits, "logits", torch.float32, 2, contiguous=False)
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    _check(temperatures, "temperatures", torch.float32, 1)
    batch, vocab = logits.shape
    if out_ids is None:
        out_ids = torch.empty(batch, dtype=torch.int64, device=logits.device)
    _check(out_ids, "out_ids", torch.int64, 1)
    with _on_device(logits, temperatures, out_ids, stream=stream):
        _raise(load().pkv_sample(_ptr(logits), batch, vocab, _row_stride(logits), _ptr(temperatures),
                                 int(seed) & (2 ** 64 - 1), int(offset) & (2 ** 64 - 1), _ptr(out_ids),
                                 _stream(stream)), "pkv_sample")
    return out_ids


def pkv_sample_dev(logits: torch.Tensor, temperatures: torch.Tensor, seed_offset: torch.Tensor,
                   out_ids: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """pkv_sample with {seed, offset} read from a device int64 tensor of 2 elements
    (so a captured CUDA graph can advance the noise between replays)."""
    _check(logits, "logits", torch.float32, 2, contiguous=False)
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    _check(temperatures, "temperatures", torch.float32, 1)
    _check(seed_offset, "seed_offset", torch.int64, 1)
    if seed_offset.numel() != 2:
        raise ValueError("seed_offset holds {seed, offset}")
    batch, vocab = logits.shape
    if out_ids is None:
        out_ids = torch.empty(batch, dtype=torch.int64, device=logits.device)
    _check(out_ids, "out_ids", torch.int64, 1)
    with _on_device(logits, temperatures, seed_offset, out_ids, stream=stream):
        _raise(load().pkv_sample_dev(_ptr(logits), batch, vocab, _row_stride(logits), _ptr(temperatures),
                                     _ptr(seed_offset),
                                     _ptr(out_ids), _stream(stream)), "pkv_sample_dev")
    return out_ids


WAIT_CHECK_INFO = 0x5741


def pkv_check_wait_timeout(stream=None) -> None:
    """Run the failure-path check: one wait that nothing completes gives up after its limit
    (about 2 s) and records (DEVERR timeout, WAIT_CHECK_INFO); read it with pkv_get_device_error."""
    with _on_device(stream=stream):
        _raise(load().pkv_check_wait_timeout(_stream(stream)), "pkv_check_wait_timeout")


def pkv_get_device_error(clear: bool = True):
    """(code, info) of the current device's error word; synchronises the device."""
    code = _c_int32(0)
    info = _c_int32(0)
    _raise(load().pkv_get_device_error(ctypes.byref(code), ctypes.byref(info), 1 if clear else 0),
           "pkv_get_device_error")
    return int(code.value), int(info.value)
