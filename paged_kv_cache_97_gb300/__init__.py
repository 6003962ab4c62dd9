"""paged_kv_cache_97_gb300 -- decode-phase paged attention on one GB300 GPU.

A thin ctypes binding over ``libpagedkv.so`` (C ABI in ``include/pagedkv.h``):
argument marshalling only.  Every step runs in the library's CUDA kernels;
PyTorch provides device memory and streams.  There is no CPU fallback: if the
library is not built, the first call raises.

    import paged_kv_cache_97_gb300 as pkv
    pkv.slot_mapping(block_tables, seq_lens, num_blocks, block_size, out=slots)
    pkv.reshape_and_cache(k, v, k_cache, v_cache, slots)
    pkv.paged_attention_decode(out, q, k_cache, v_cache, block_tables, seq_lens,
                               max_seq_len, scale, workspace=ws)
"""
from __future__ import annotations

import ctypes
import os

from . import _build

LIB_PATH = _build.LIB_PATH

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_OUT_OF_BLOCKS, KV_ERR_CUDA, KV_ERR_DEVICE_INDEX, \
    KV_ERR_NOT_IMPLEMENTED = range(6)
DTYPE_BF16, DTYPE_INT8, DTYPE_FP8_E4M3 = 0, 1, 2
FLAG_BAD_SLOT, FLAG_BAD_BLOCK, FLAG_BAD_SEQ_LEN, FLAG_WAIT_TIMEOUT = 0x1, 0x2, 0x4, 0x8

# Every symbol include/pagedkv.h declares, with its ctypes signature.
_P, _I, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "kv_pool_create": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_P)]),
    "kv_pool_destroy": (None, [_P]),
    "kv_pool_block_bytes": (_SZ, [_P]),
    "kv_pool_alloc": (_I, [_P, _I, _P]),
    "kv_pool_free": (_I, [_P, _P, _I]),
    "kv_pool_stats": (_I, [_P, _P, _P]),
    "kv_pool_fork": (_I, [_P, _P, _I]),
    "kv_pool_refcount": (_I, [_P, ctypes.c_int32]),
    "kv_pool_prepare_append": (_I, [_P, _P, _I, _P, _I, _P, _P]),
    "pagedkv_copy_blocks": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pagedkv_check_block_pairs": (_I, [_P, _I, _I]),
    "pagedkv_multi_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "pagedkv_block_hash": (ctypes.c_uint64, [ctypes.c_uint64, _P, _I, ctypes.c_uint64]),
    "kv_pool_match_prefix": (_I, [_P, _P, _I, ctypes.c_uint64, _P, _P]),
    "kv_pool_register_prefix": (_I, [_P, _P, _P, _I, ctypes.c_uint64]),
    "kv_pool_cached_blocks": (_I, [_P]),
    "paged_attention_multi": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I,
                                   _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "pagedkv_multi_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I,
                                _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "pagedkv_pool_tensor_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "pagedkv_slot_mapping": (_I, [_P, _I, _P, _I, _I, _I, _P, _P]),
    "pagedkv_token_slot_mapping": (_I, [_P, _I, _P, _P, _I, _I, _I, _P, _P]),
    "reshape_and_cache": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pagedkv_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "paged_attention_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I,
                                    _I, _F, _I, _P, _SZ, _P]),
    "paged_attention_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I,
                                            _I, _I, _I, _F, _I, _P]),
    "pagedkv_noalloc_scratch_bytes": (_SZ, []),
    "pagedkv_get_status": (_I, [_P, ctypes.POINTER(ctypes.c_uint)]),
    "pagedkv_last_error": (ctypes.c_char_p, []),
    "pagedkv_partition_tokens": (_I, [_I, _I, _I, _I]),
    "pagedkv_multi_partition_tokens": (_I, [_I, _I, _I, _I, _I, _I]),
    "pagedkv_decode_step_prefix": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I,
                                        _I, _I, _I, _F, _I, _P, _I, _P, _SZ, _P]),
    "pagedkv_prefix_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "pagedkv_decode_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I,
                                 _I, _I, _F, _I, _P, _SZ, _P]),
}

_lib = None


class KVError(RuntimeError):
    """A libpagedkv call returned a status other than KV_OK."""

    def __init__(self, status: int, message: str):
        super().__init__(f"libpagedkv status {status}: {message}")
        self.status = status


def load(path: str = LIB_PATH):
    """Load libpagedkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


def _check(st: int):
    if st != KV_OK:
        raise KVError(st, load().pagedkv_last_error().decode(errors="replace"))


_raw_stream = None          # torch's raw current-stream query, resolved once


def _stream(stream):
    """The cudaStream_t to launch on: `stream` (a torch stream or a raw
    handle), else torch's current stream on the current device.  Pointer
    arguments go to ctypes as plain ints (the signatures convert them)."""
    global _raw_stream
    import torch
    if stream is None:
        if _raw_stream is None:
            # the raw query skips torch.cuda.current_stream's device-argument
            # handling (a third of a small step's host time); same stream
            _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", False)
        if _raw_stream:
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t, dtype, name, ndim=None):
    import torch
    if type(t) is not torch.Tensor and not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {tuple(t.shape)}")


def _pool_dtype(k_cache):
    import torch
    if k_cache.dtype == torch.bfloat16:
        return DTYPE_BF16
    if k_cache.dtype == torch.int8:
        return DTYPE_INT8
    if k_cache.dtype == torch.float8_e4m3fn:
        return DTYPE_FP8_E4M3
    raise TypeError("pools must be torch.bfloat16, torch.int8 or torch.float8_e4m3fn")


# --------------------------------------------------------------------------
# Block pool
# --------------------------------------------------------------------------

class KVPool:
    """Host bookkeeping of a block pool: FIFO free list, all-or-nothing
    allocation, a reference count per block and copy-on-write before a
    decode append."""

    def __init__(self, num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                 dtype: int = DTYPE_BF16):
        self._lib = load()
        h = ctypes.c_void_p()
        _check(self._lib.kv_pool_create(num_blocks, block_size, num_kv_heads, head_dim, dtype,
                                        ctypes.byref(h)))
        self._h = h
        self.block_size_ = block_size

    def close(self):
        if self._h:
            self._lib.kv_pool_destroy(self._h)
            self._h = None

    __del__ = close

    def block_bytes(self) -> int:
        return self._lib.kv_pool_block_bytes(self._h)

    def alloc(self, n: int) -> list:
        ids = (ctypes.c_int32 * max(n, 1))()
        _check(self._lib.kv_pool_alloc(self._h, n, ids))
        return list(ids[:n])

    def free(self, ids) -> None:
        ids = list(ids)
        arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _check(self._lib.kv_pool_free(self._h, arr, len(ids)))

    def stats(self):
        used, free = ctypes.c_int(), ctypes.c_int()
        _check(self._lib.kv_pool_stats(self._h, ctypes.byref(used), ctypes.byref(free)))
        return used.value, free.value

    def fork(self, ids) -> None:
        """One more reference on each block (a forked sequence maps them)."""
        ids = list(ids)
        arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _check(self._lib.kv_pool_fork(self._h, arr, len(ids)))

    def refcount(self, block_id: int) -> int:
        return self._lib.kv_pool_refcount(self._h, block_id)

    def match_prefix(self, tokens, extra_key: int = 0) -> list:
        """Ids of the cached blocks that hold the prompt's leading full
        blocks (each gains a reference)."""
        import numpy as np
        tk = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.zeros(max(len(tk) // self.block_size_, 1), np.int32)
        n = ctypes.c_int()
        _check(self._lib.kv_pool_match_prefix(self._h, tk.ctypes.data, len(tk), extra_key,
                                              out.ctypes.data, ctypes.byref(n)))
        return out[:n.value].tolist()

    def register_prefix(self, block_ids, tokens, extra_key: int = 0) -> None:
        """Register the sequence's full blocks for later prefix matches."""
        import numpy as np
        tk = np.ascontiguousarray(tokens, dtype=np.int32)
        ids = np.ascontiguousarray(block_ids, dtype=np.int32)
        if len(ids) < len(tk) // self.block_size_:
            raise ValueError("one block id per full block of tokens is needed")
        _check(self._lib.kv_pool_register_prefix(self._h, ids.ctypes.data if len(ids) else None,
                                                 tk.ctypes.data if len(tk) else None, len(tk),
                                                 extra_key))

    def cached_blocks(self) -> int:
        return self._lib.kv_pool_cached_blocks(self._h)

    def prepare_append(self, block_tables, seq_lens):
        """Blocks for this step's appends (host int32 numpy arrays; the table
        is updated in place).  Returns the (src, dst) copy pairs as an int32
        array [n, 2] for copy_blocks."""
        import numpy as np
        bt, sl = block_tables, np.ascontiguousarray(seq_lens, dtype=np.int32)
        if bt.dtype != np.int32 or not bt.flags.c_contiguous or bt.ndim != 2:
            raise TypeError("block_tables must be a C-contiguous int32 [batch, max_blocks] array")
        if sl.shape != (bt.shape[0],):
            raise ValueError("seq_lens must have one entry per table row")
        pairs = np.zeros((max(bt.shape[0], 1), 2), np.int32)
        n = ctypes.c_int()
        _check(self._lib.kv_pool_prepare_append(self._h, bt.ctypes.data, bt.shape[1], sl.ctypes.data,
                                                bt.shape[0], pairs.ctypes.data, ctypes.byref(n)))
        return pairs[:n.value].copy()


def block_hash(parent_hash: int, tokens, extra_key: int = 0) -> int:
    """The prefix cache's hash of one full block (FNV-1a 64 over parent,
    key and token ids)."""
    import numpy as np
    tk = np.ascontiguousarray(tokens, dtype=np.int32)
    return load().pagedkv_block_hash(parent_hash, tk.ctypes.data, len(tk), extra_key)


def pool_tensor_bytes(num_blocks, block_size, num_kv_heads, head_dim, dtype=DTYPE_BF16) -> int:
    return load().pagedkv_pool_tensor_bytes(num_blocks, block_size, num_kv_heads, head_dim, dtype)


# --------------------------------------------------------------------------
# Kernels
# --------------------------------------------------------------------------

def slot_mapping(block_tables, seq_lens, num_blocks, block_size, out, stream=None):
    """Slots of each sequence's new token (position seq_lens[b] - 1) into ``out``."""
    import torch
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(out, torch.int64, "out", 1)
    B = seq_lens.shape[0]
    if block_tables.shape[0] != B or out.shape[0] != B:
        raise ValueError("block_tables, seq_lens and out disagree on the batch size")
    _check(load().pagedkv_slot_mapping(_ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B,
                                       block_size, num_blocks, _ptr(out), _stream(stream)))
    return out


def token_slot_mapping(block_tables, positions, num_blocks, block_size, out, seq_idx=None,
                       stream=None):
    """Slots of tokens (seq_idx[i], positions[i]) into ``out``."""
    import torch
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(positions, torch.int32, "positions", 1)
    _need(out, torch.int64, "out", 1)
    n = positions.shape[0]
    if seq_idx is not None:
        _need(seq_idx, torch.int32, "seq_idx", 1)
        if seq_idx.shape[0] != n:
            raise ValueError("seq_idx and positions disagree")
    if out.shape[0] != n:
        raise ValueError("out and positions disagree")
    _check(load().pagedkv_token_slot_mapping(_ptr(block_tables), block_tables.shape[1], _ptr(seq_idx),
                                             _ptr(positions), n, block_size, num_blocks, _ptr(out),
                                             _stream(stream)))
    return out


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, k_scale=None, v_scale=None,
                      stream=None):
    """Append bf16 k, v [n, Hkv, d] into pools [NB, bs, Hkv, d] at the slots."""
    import torch
    _need(k, torch.bfloat16, "k", 3)
    _need(v, torch.bfloat16, "v", 3)
    dt = _pool_dtype(k_cache)
    _need(k_cache, k_cache.dtype, "k_cache", 4)
    _need(v_cache, k_cache.dtype, "v_cache", 4)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    nb, bs, hkv, d = k_cache.shape
    if v_cache.shape != k_cache.shape or k.shape != v.shape or k.shape[1:] != (hkv, d):
        raise ValueError("k, v and the pools disagree on (num_kv_heads, head_dim)")
    if slot_mapping.shape[0] != k.shape[0]:
        raise ValueError("slot_mapping must have one entry per token")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t is not None:
            _need(t, torch.float32, name, 2)
    _check(load().reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                    _ptr(v_scale), _ptr(slot_mapping), k.shape[0], nb, bs, hkv, d, dt,
                                    _stream(stream)))


def copy_blocks(k_cache, v_cache, block_pairs, k_scale=None, v_scale=None, stream=None):
    """Copy whole blocks src -> dst of both pools (and 8-bit scales), for
    the device int32 pairs [n, 2]."""
    import torch
    dt = _pool_dtype(k_cache)
    _need(k_cache, k_cache.dtype, "k_cache", 4)
    _need(v_cache, k_cache.dtype, "v_cache", 4)
    _need(block_pairs, torch.int32, "block_pairs", 2)
    if v_cache.shape != k_cache.shape or block_pairs.shape[1] != 2:
        raise ValueError("pools must match and block_pairs must be [n, 2]")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t is not None:
            _need(t, torch.float32, name, 2)
    nb, bs, hkv, d = k_cache.shape
    _check(load().pagedkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                      _ptr(block_pairs), block_pairs.shape[0], nb, bs, hkv, d, dt,
                                      _stream(stream)))


def check_block_pairs(block_pairs, num_blocks):
    """Host check of a copy list for copy_blocks (a host int32 array [n, 2] of
    (src, dst)): every id in range, destinations distinct and none of them a
    source.  Raises KVError otherwise."""
    import numpy as np
    pairs = np.ascontiguousarray(block_pairs, np.int32).reshape(-1, 2)
    _check(load().pagedkv_check_block_pairs(pairs.ctypes.data if len(pairs) else None, len(pairs),
                                            int(num_blocks)))


def multi_workspace_bytes(num_tokens, num_q_heads, head_dim, max_seq_len, block_size) -> int:
    return load().pagedkv_multi_workspace_bytes(num_tokens, num_q_heads, head_dim, max_seq_len,
                                                block_size)


def paged_attention_multi(out, q, k_cache, v_cache, block_tables, seq_lens, query_start,
                          max_seq_len, max_query_len, scale, workspace=None, k_scale=None,
                          v_scale=None, stream=None):
    """Causal attention of several query tokens per sequence (the last
    query_start[b+1] - query_start[b] tokens of sequence b, already
    appended): q, out bf16 [T, Hq, d]."""
    import torch
    dt = _pool_dtype(k_cache)
    _need(out, torch.bfloat16, "out", 3)
    _need(q, torch.bfloat16, "q", 3)
    _need(k_cache, k_cache.dtype, "k_cache", 4)
    _need(v_cache, k_cache.dtype, "v_cache", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(query_start, torch.int32, "query_start", 1)
    nb, bs, hkv, d = k_cache.shape
    T, hq, d2 = q.shape
    B = seq_lens.shape[0]
    if out.shape != q.shape or d2 != d or query_start.shape[0] != B + 1 or block_tables.shape[0] != B:
        raise ValueError("shapes of out, q, the pools, the table, seq_lens and query_start disagree")
    ws_ptr, ws_n = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel() * workspace.element_size())
    _check(load().paged_attention_multi(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                        _ptr(v_scale), _ptr(block_tables), block_tables.shape[1],
                                        _ptr(seq_lens), _ptr(query_start), B, T, int(max_query_len),
                                        hq, hkv, d, nb, bs, int(max_seq_len), float(scale), dt,
                                        ws_ptr, ws_n,
                                        _stream(stream)))


def multi_step(out, q, new_k, new_v, k_cache, v_cache, block_tables, seq_lens, query_start,
               max_seq_len, max_query_len, scale, workspace=None, k_scale=None, v_scale=None,
               stream=None):
    """One multi-token step: the step's new K/V rows (bf16 [T, Hkv, d], row
    query_start[b] + i at position seq_lens[b] - n_b + i) appended to the
    pool, then paged_attention_multi over the query tokens."""
    import torch
    dt = _pool_dtype(k_cache)
    _need(out, torch.bfloat16, "out", 3)
    _need(q, torch.bfloat16, "q", 3)
    _need(new_k, torch.bfloat16, "new_k", 3)
    _need(new_v, torch.bfloat16, "new_v", 3)
    _need(k_cache, k_cache.dtype, "k_cache", 4)
    _need(v_cache, k_cache.dtype, "v_cache", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(query_start, torch.int32, "query_start", 1)
    nb, bs, hkv, d = k_cache.shape
    T, hq, d2 = q.shape
    B = seq_lens.shape[0]
    if (out.shape != q.shape or d2 != d or query_start.shape[0] != B + 1 or
            block_tables.shape[0] != B or tuple(new_k.shape) != (T, hkv, d) or
            new_v.shape != new_k.shape):
        raise ValueError("shapes of out, q, new_k, new_v, the pools, the table, seq_lens and "
                         "query_start disagree")
    ws_ptr, ws_n = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel() * workspace.element_size())
    _check(load().pagedkv_multi_step(_ptr(out), _ptr(q), _ptr(new_k), _ptr(new_v), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                     _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                     _ptr(query_start), B, T, int(max_query_len), hq, hkv, d, nb,
                                     bs, int(max_seq_len), float(scale), dt, ws_ptr, ws_n,
                                     _stream(stream)))


def workspace_bytes(batch, num_q_heads, head_dim, max_seq_len, block_size) -> int:
    return load().pagedkv_workspace_bytes(batch, num_q_heads, head_dim, max_seq_len, block_size)


def partition_tokens(batch, num_kv_heads, max_seq_len, block_size) -> int:
    """Token partition size the decode kernel uses for this shape."""
    return load().pagedkv_partition_tokens(batch, num_kv_heads, max_seq_len, block_size)


def multi_partition_tokens(batch, num_tokens, max_query_len, num_q_heads, num_kv_heads,
                           max_seq_len) -> int:
    """Token partition size paged_attention_multi uses for this call."""
    return load().pagedkv_multi_partition_tokens(batch, num_tokens, max_query_len, num_q_heads,
                                                 num_kv_heads, max_seq_len)


def _check_decode(out, q, k_cache, v_cache, block_tables, seq_lens, k_scale, v_scale, workspace):
    import torch
    _need(out, torch.bfloat16, "out", 3)
    _need(q, torch.bfloat16, "q", 3)
    _pool_dtype(k_cache)
    _need(k_cache, k_cache.dtype, "k_cache", 4)
    _need(v_cache, k_cache.dtype, "v_cache", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, hq, d = q.shape
    if out.shape != q.shape or k_cache.shape[3] != d or v_cache.shape != k_cache.shape:
        raise ValueError("q, out and the pools disagree")
    if block_tables.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_tables / seq_lens must have one row per sequence")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t is not None:
            _need(t, torch.float32, name, 2)
    if workspace is None:
        return 0
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return workspace.numel() * workspace.element_size()


def decode_step(out, q, k, v, k_cache, v_cache, block_tables, seq_lens, max_seq_len, scale,
                workspace, k_scale=None, v_scale=None, stream=None):
    """Append k[b], v[b] (bf16 [B, Hkv, d]) at position seq_lens[b] - 1 and
    attend, in two launches (the append runs inside the attention kernel)."""
    import torch
    wbytes = _check_decode(out, q, k_cache, v_cache, block_tables, seq_lens, k_scale, v_scale,
                           workspace)
    _need(k, torch.bfloat16, "k", 3)
    _need(v, torch.bfloat16, "v", 3)
    B, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    if k.shape != (B, hkv, d) or v.shape != k.shape:
        raise ValueError("k, v must be [batch, num_kv_heads, head_dim]")
    _check(load().pagedkv_decode_step(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache),
                                      _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                      _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B,
                                      hq, hkv, d, nb, bs, int(max_seq_len), float(scale),
                                      _pool_dtype(k_cache), _ptr(workspace), wbytes,
                                      _stream(stream)))
    return out


_raw_lib = None


def _raw():
    """A second handle on the library whose functions take ctypes objects
    as they are (no per-call argument conversion): for prepared calls."""
    global _raw_lib
    if _raw_lib is None:
        load()
        _raw_lib = ctypes.CDLL(LIB_PATH)
        _raw_lib.pagedkv_decode_step.restype = ctypes.c_int
    return _raw_lib


class DecodeStepPlan:
    """pagedkv_decode_step with its arguments checked and marshalled once.

    Arguments as ``decode_step``.  The plan holds the tensors (their memory
    stays valid while it lives); they must keep their shapes and storage,
    while their contents may change between calls -- the usual serving loop
    writes the next step's q, k, v, tables and lengths in place.  Each call
    runs one step on the current stream (or ``stream``) and returns ``out``;
    only the stream is looked up per call, which keeps a small step's host
    time near the C call itself."""

    def __init__(self, out, q, k, v, k_cache, v_cache, block_tables, seq_lens, max_seq_len, scale,
                 workspace, k_scale=None, v_scale=None):
        import torch
        wbytes = _check_decode(out, q, k_cache, v_cache, block_tables, seq_lens, k_scale, v_scale,
                               workspace)
        _need(k, torch.bfloat16, "k", 3)
        _need(v, torch.bfloat16, "v", 3)
        B, hq, d = q.shape
        nb, bs, hkv, _ = k_cache.shape
        if k.shape != (B, hkv, d) or v.shape != k.shape:
            raise ValueError("k, v must be [batch, num_kv_heads, head_dim]")
        self.out = out
        self._keep = (q, k, v, k_cache, v_cache, block_tables, seq_lens, workspace, k_scale, v_scale)
        P, I = ctypes.c_void_p, ctypes.c_int
        self._fn = _raw().pagedkv_decode_step
        self._args = (P(_ptr(out)), P(_ptr(q)), P(_ptr(k)), P(_ptr(v)), P(_ptr(k_cache)),
                      P(_ptr(v_cache)), P(_ptr(k_scale)), P(_ptr(v_scale)), P(_ptr(block_tables)),
                      I(block_tables.shape[1]), P(_ptr(seq_lens)), I(B), I(hq), I(hkv), I(d), I(nb),
                      I(bs), I(int(max_seq_len)), ctypes.c_float(float(scale)),
                      I(_pool_dtype(k_cache)), P(_ptr(workspace)), ctypes.c_size_t(wbytes))

    def __call__(self, stream=None):
        st = self._fn(*self._args, ctypes.c_void_p(_stream(stream)))
        if st != KV_OK:
            _check(st)
        return self.out


def prefix_workspace_bytes(batch, num_q_heads, head_dim, max_seq_len, block_size,
                           num_prefix_blocks) -> int:
    return load().pagedkv_prefix_workspace_bytes(batch, num_q_heads, head_dim, max_seq_len,
                                                 block_size, num_prefix_blocks)


def decode_step_prefix(out, q, k, v, k_cache, v_cache, block_tables, seq_lens, max_seq_len, scale,
                       prefix_blocks, workspace, k_scale=None, v_scale=None, stream=None):
    """decode_step for a batch whose sequences all start with the physical
    blocks ``prefix_blocks`` (int32 [P]): the prefix is attended once per KV
    head for all query rows.  k, v may both be None (attend only)."""
    import torch
    wbytes = _check_decode(out, q, k_cache, v_cache, block_tables, seq_lens, k_scale, v_scale,
                           workspace)
    _need(prefix_blocks, torch.int32, "prefix_blocks", 1)
    B, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    if k is not None:
        _need(k, torch.bfloat16, "k", 3)
        _need(v, torch.bfloat16, "v", 3)
        if k.shape != (B, hkv, d) or v.shape != k.shape:
            raise ValueError("k, v must be [batch, num_kv_heads, head_dim]")
    _check(load().pagedkv_decode_step_prefix(
        _ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B, hq, hkv, d,
        nb, bs, int(max_seq_len), float(scale), _pool_dtype(k_cache), _ptr(prefix_blocks),
        prefix_blocks.shape[0], _ptr(workspace), wbytes, _stream(stream)))
    return out


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, scale,
                           workspace=None, k_scale=None, v_scale=None, stream=None):
    """out[b, h] = softmax(scale q[b, h] . K) V over sequence b's paged tokens."""
    wbytes = _check_decode(out, q, k_cache, v_cache, block_tables, seq_lens, k_scale, v_scale,
                           workspace)
    B, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    dt = _pool_dtype(k_cache)
    _check(load().paged_attention_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
                                         block_tables.shape[1], _ptr(seq_lens), B, hq, hkv, d, nb, bs,
                                         int(max_seq_len), float(scale), dt, _ptr(workspace), wbytes,
                                         _stream(stream)))
    return out


def noalloc_scratch_bytes() -> int:
    """Size of the fixed device scratch paged_attention_decode_noalloc uses,
    as compiled into the library."""
    return load().pagedkv_noalloc_scratch_bytes()


def paged_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, seq_lens, max_seq_len,
                                   scale, k_scale=None, v_scale=None, stream=None):
    """paged_attention_decode for callers that cannot allocate device memory:
    the split-K partials go to the library's fixed device scratch
    (``noalloc_scratch_bytes()``, 32 MiB) instead of a caller workspace.  Calls that overlap on the GPU race on
    that scratch; the first call on a device should come before any stream
    capture."""
    import torch
    _need(out, torch.bfloat16, "out", 3)
    _need(q, torch.bfloat16, "q", 3)
    dt = _pool_dtype(k_cache)
    _need(k_cache, k_cache.dtype, "k_cache", 4)
    _need(v_cache, k_cache.dtype, "v_cache", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if out.shape != q.shape or d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("q, out and the pools disagree")
    if block_tables.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_tables / seq_lens must have one row per sequence")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t is not None:
            _need(t, torch.float32, name, 2)
    _check(load().paged_attention_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                                 _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
                                                 block_tables.shape[1], _ptr(seq_lens), B, hq, hkv, d,
                                                 nb, bs, int(max_seq_len), float(scale), dt,
                                                 _stream(stream)))
    return out


def get_status(stream=None):
    """(status, flags): waits for the stream, then reads and clears the
    device status word (FLAG_* bits)."""
    flags = ctypes.c_uint()
    st = load().pagedkv_get_status(_stream(stream), ctypes.byref(flags))
    return st, flags.value
