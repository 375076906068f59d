"""Python binding of the C interface in include/gqa.h (argument marshalling only).

Every function here checks tensor dtypes/shapes/devices, allocates outputs
with torch when the caller did not pass them, and forwards raw device
pointers to ``libgqa_b300.so``. All arithmetic happens in the CUDA kernels;
there is no fallback: if the native library is missing, importing the
functions raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libgqa_b300.so")

GQA_OK = 0
GQA_ERR_NULL = 1
GQA_ERR_SHAPE = 2
GQA_ERR_ALIGN = 3
GQA_ERR_WORKSPACE = 4
GQA_ERR_CACHE_FULL = 5
GQA_ERR_CUDA = 6
GQA_ERR_TIMEOUT = 7
GQA_ERR_BAD_LENGTH = 8
GQA_ERR_SCRATCH_LIMIT = 9
GQA_ERR_BAD_PAGE = 10
GQA_OUT_F32 = 0
GQA_OUT_BF16 = 1

_lib = None


class GQAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


def load_library() -> ctypes.CDLL:
    """Load the native library once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"native GQA library not found at {LIB_PATH}; build it with "
            "`python -m grouped_query_attention_10_b300.build_native`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.gqa_status_string.argtypes = [i32]
    lib.gqa_status_string.restype = ctypes.c_char_p
    lib.gqa_version.argtypes = []
    lib.gqa_version.restype = i32
    lib.gqa_prefill_fwd.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f32,
                                    i32, vp, vp]
    lib.gqa_prefill_fwd.restype = i32
    lib.gqa_prefill_fwd_ex.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f32,
                                       i32, i32, vp, vp, vp]
    lib.gqa_prefill_fwd_ex.restype = i32
    lib.gqa_prefill_kvcache_fwd.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                            i32, i32, f32, i32, vp, vp, vp]
    lib.gqa_prefill_kvcache_fwd.restype = i32
    lib.gqa_decode_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f32,
                                      i32, vp, vp, sz, vp, vp]
    lib.gqa_decode_fwd_ex.restype = i32
    lib.gqa_decode_paged_workspace_bytes.argtypes = [i32] * 6
    lib.gqa_decode_paged_workspace_bytes.restype = sz
    lib.gqa_decode_paged_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                         i32, i32, i32, f32, i32, vp, vp, sz, vp, vp]
    lib.gqa_decode_paged_fwd.restype = i32
    lib.kv_cache_append_paged.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                          i32, vp, vp]
    lib.kv_cache_append_paged.restype = i32
    lib.gqa_selftest_bounded_wait.argtypes = [vp, i32, vp]
    lib.gqa_selftest_bounded_wait.restype = i32
    lib.kv_cache_append_rope.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                         i32, i32, i32, vp, vp]
    lib.kv_cache_append_rope.restype = i32
    lib.kv_cache_append_paged_rope.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                               i32, i32, i32, i32, i32, i32, i32, vp, vp]
    lib.kv_cache_append_paged_rope.restype = i32
    lib.gqa_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.gqa_decode_workspace_bytes.restype = sz
    lib.gqa_decode_fwd.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f32,
                                   vp, sz, vp, vp]
    lib.gqa_decode_fwd.restype = i32
    lib.kv_cache_append.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]
    lib.kv_cache_append.restype = i32
    lib.gqa_decode_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32,
                                           f32, vp, vp]
    lib.gqa_decode_fwd_noalloc.restype = i32
    lib.gqa_decode_noalloc_scratch_bytes.argtypes = []
    lib.gqa_decode_noalloc_scratch_bytes.restype = sz
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().gqa_status_string(int(code)).decode()


def gqa_status_string(code: int) -> str:
    return status_string(code)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream, device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _out_code(dtype) -> int:
    if dtype == torch.float32:
        return GQA_OUT_F32
    if dtype == torch.bfloat16:
        return GQA_OUT_BF16
    raise TypeError("output dtype must be float32 or bfloat16")


def _check_slopes(alibi_slopes, h_q):
    if alibi_slopes is not None:
        _check(alibi_slopes, "alibi_slopes", torch.float32, (h_q,))


def gqa_prefill_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, causal: bool,
                    scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                    out_dtype=torch.float32, lse: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None, stream=None, window: int = 0,
                    alibi_slopes: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Prefill attention. q [B,L,h_q,d], k/v [B,L,g,d] bf16 -> out [B,L,h_q,d].

    ``window`` > 0 (causal only) keeps the last ``window`` keys of every row;
    ``alibi_slopes`` (fp32 [h_q]) subtracts ``slope_h * |i - j|``."""
    lib = load_library()
    B, L, h_q, d = q.shape
    g = k.shape[2]
    _check(q, "q", torch.bfloat16)
    _check(k, "k", torch.bfloat16, (B, L, g, d))
    _check(v, "v", torch.bfloat16, (B, L, g, d))
    if out is None:
        out = torch.empty((B, L, h_q, d), dtype=out_dtype, device=q.device)
    _check(out, "out", out.dtype, (B, L, h_q, d))
    if lse is not None:
        _check(lse, "lse", torch.float32, (B, h_q, L))
    if status is not None:
        _check(status, "status", torch.int32)
    _check_slopes(alibi_slopes, h_q)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    if window == 0 and alibi_slopes is None:
        rc = lib.gqa_prefill_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _out_code(out.dtype),
                                 _ptr(lse), B, L, h_q, g, d, float(scale), int(bool(causal)),
                                 _ptr(status), _stream_ptr(stream, q.device))
    else:
        rc = lib.gqa_prefill_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _out_code(out.dtype),
                                    _ptr(lse), B, L, h_q, g, d, float(scale),
                                    int(bool(causal)), int(window), _ptr(alibi_slopes),
                                    _ptr(status), _stream_ptr(stream, q.device))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_fwd")
    return out


def gqa_prefill_kvcache_fwd(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            seq_lens: torch.Tensor, *, scale: Optional[float] = None,
                            out: Optional[torch.Tensor] = None, out_dtype=torch.float32,
                            lse: Optional[torch.Tensor] = None, window: int = 0,
                            alibi_slopes: Optional[torch.Tensor] = None,
                            status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Chunked prefill: q [B,T,h_q,d] (the T newest tokens) over a [B,g,S_max,d]
    cache that already holds them; seq_lens [B] device int32, each >= T."""
    lib = load_library()
    B, T, h_q, d = q.shape
    g, S_max = k_cache.shape[1], k_cache.shape[2]
    _check(q, "q", torch.bfloat16)
    _check(k_cache, "k_cache", torch.bfloat16, (B, g, S_max, d))
    _check(v_cache, "v_cache", torch.bfloat16, (B, g, S_max, d))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, T, h_q, d), dtype=out_dtype, device=q.device)
    _check(out, "out", out.dtype, (B, T, h_q, d))
    if lse is not None:
        _check(lse, "lse", torch.float32, (B, h_q, T))
    if status is not None:
        _check(status, "status", torch.int32)
    _check_slopes(alibi_slopes, h_q)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    rc = lib.gqa_prefill_kvcache_fwd(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
                                     _ptr(out), _out_code(out.dtype), _ptr(lse), B, T, h_q, g,
                                     d, S_max, float(scale), int(window), _ptr(alibi_slopes),
                                     _ptr(status), _stream_ptr(stream, q.device))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_kvcache_fwd")
    return out


def gqa_decode_workspace_bytes(B: int, h_q: int, g: int, d: int, S_max: int) -> int:
    return int(load_library().gqa_decode_workspace_bytes(B, h_q, g, d, S_max))


def gqa_decode_fwd(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   seq_lens: torch.Tensor, *, scale: Optional[float] = None,
                   out: Optional[torch.Tensor] = None, out_dtype=torch.float32,
                   lse: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None, stream=None, window: int = 0,
                   alibi_slopes: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Decode one token per sequence over a [B,g,S_max,d] cache -> out [B,h_q,d].

    ``window`` > 0 keeps the last ``window`` rows; ``alibi_slopes`` (fp32 [h_q])
    subtracts ``slope_h * (seq_lens[b] - 1 - j)``."""
    lib = load_library()
    B, h_q, d = q.shape
    g, S_max = k_cache.shape[1], k_cache.shape[2]
    _check(q, "q", torch.bfloat16)
    _check(k_cache, "k_cache", torch.bfloat16, (B, g, S_max, d))
    _check(v_cache, "v_cache", torch.bfloat16, (B, g, S_max, d))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, h_q, d), dtype=out_dtype, device=q.device)
    _check(out, "out", out.dtype, (B, h_q, d))
    if lse is not None:
        _check(lse, "lse", torch.float32, (B, h_q))
    if status is not None:
        _check(status, "status", torch.int32)
    need = gqa_decode_workspace_bytes(B, h_q, g, d, S_max)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    _check_slopes(alibi_slopes, h_q)
    if window == 0 and alibi_slopes is None:
        rc = lib.gqa_decode_fwd(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
                                _ptr(out), _out_code(out.dtype), _ptr(lse), B, h_q, g, d, S_max,
                                float(scale), _ptr(workspace), workspace.numel(), _ptr(status),
                                _stream_ptr(stream, q.device))
    else:
        rc = lib.gqa_decode_fwd_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
                                   _ptr(out), _out_code(out.dtype), _ptr(lse), B, h_q, g, d,
                                   S_max, float(scale), int(window), _ptr(alibi_slopes),
                                   _ptr(workspace), workspace.numel(), _ptr(status),
                                   _stream_ptr(stream, q.device))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_decode_fwd")
    return out


def gqa_decode_fwd_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           seq_lens: torch.Tensor, *, out: torch.Tensor,
                           scale: Optional[float] = None, lse: Optional[torch.Tensor] = None,
                           status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode without a workspace: the library's built-in scratch array holds
    the split partials. ``out`` must be given (this call allocates nothing)."""
    lib = load_library()
    B, h_q, d = q.shape
    g, S_max = k_cache.shape[1], k_cache.shape[2]
    _check(q, "q", torch.bfloat16)
    _check(k_cache, "k_cache", torch.bfloat16, (B, g, S_max, d))
    _check(v_cache, "v_cache", torch.bfloat16, (B, g, S_max, d))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    _check(out, "out", out.dtype, (B, h_q, d))
    if lse is not None:
        _check(lse, "lse", torch.float32, (B, h_q))
    if status is not None:
        _check(status, "status", torch.int32)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    rc = lib.gqa_decode_fwd_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
                                    _ptr(out), _out_code(out.dtype), _ptr(lse), B, h_q, g, d,
                                    S_max, float(scale), _ptr(status),
                                    _stream_ptr(stream, q.device))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_decode_fwd_noalloc")
    return out


def kv_cache_append(k_cache: torch.Tensor, v_cache: torch.Tensor, seq_lens: torch.Tensor,
                    k_new: torch.Tensor, v_new: torch.Tensor, *,
                    status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Append k_new/v_new [B,T,g,d] behind each sequence's rows; advances seq_lens."""
    lib = load_library()
    B, g, S_max, d = k_cache.shape
    T = k_new.shape[1]
    _check(k_cache, "k_cache", torch.bfloat16)
    _check(v_cache, "v_cache", torch.bfloat16, (B, g, S_max, d))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    _check(k_new, "k_new", torch.bfloat16, (B, T, g, d))
    _check(v_new, "v_new", torch.bfloat16, (B, T, g, d))
    if status is not None:
        _check(status, "status", torch.int32)
    rc = lib.kv_cache_append(_ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), _ptr(k_new),
                             _ptr(v_new), B, g, d, S_max, T, _ptr(status),
                             _stream_ptr(stream, k_cache.device))
    if rc != GQA_OK:
        raise GQAError(rc, "kv_cache_append")


def gqa_decode_paged_workspace_bytes(B: int, h_q: int, g: int, d: int, page_size: int,
                                     max_blocks: int) -> int:
    return int(load_library().gqa_decode_paged_workspace_bytes(B, h_q, g, d, page_size,
                                                               max_blocks))


def gqa_decode_paged_fwd(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                         block_table: torch.Tensor, seq_lens: torch.Tensor, *,
                         scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                         out_dtype=torch.float32, lse: Optional[torch.Tensor] = None,
                         window: int = 0, alibi_slopes: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None,
                         status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode over a paged cache: pools [num_pages, g, page_size, d], block_table
    [B, max_blocks] int32 (physical page of each logical block) -> out [B, h_q, d]."""
    lib = load_library()
    B, h_q, d = q.shape
    num_pages, g, page_size = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    max_blocks = block_table.shape[1]
    _check(q, "q", torch.bfloat16)
    _check(k_pool, "k_pool", torch.bfloat16, (num_pages, g, page_size, d))
    _check(v_pool, "v_pool", torch.bfloat16, (num_pages, g, page_size, d))
    _check(block_table, "block_table", torch.int32, (B, max_blocks))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, h_q, d), dtype=out_dtype, device=q.device)
    _check(out, "out", out.dtype, (B, h_q, d))
    if lse is not None:
        _check(lse, "lse", torch.float32, (B, h_q))
    if status is not None:
        _check(status, "status", torch.int32)
    _check_slopes(alibi_slopes, h_q)
    need = gqa_decode_paged_workspace_bytes(B, h_q, g, d, page_size, max_blocks)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    rc = lib.gqa_decode_paged_fwd(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                  _ptr(seq_lens), _ptr(out), _out_code(out.dtype), _ptr(lse), B,
                                  h_q, g, d, page_size, num_pages, max_blocks, float(scale),
                                  int(window), _ptr(alibi_slopes), _ptr(workspace),
                                  workspace.numel(), _ptr(status),
                                  _stream_ptr(stream, q.device))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_decode_paged_fwd")
    return out


def kv_cache_append_paged(k_pool: torch.Tensor, v_pool: torch.Tensor,
                          block_table: torch.Tensor, seq_lens: torch.Tensor,
                          k_new: torch.Tensor, v_new: torch.Tensor, *,
                          status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Append k_new/v_new [B,T,g,d] through the block table; advances seq_lens."""
    lib = load_library()
    num_pages, g, page_size, d = k_pool.shape
    B, max_blocks = block_table.shape
    T = k_new.shape[1]
    _check(k_pool, "k_pool", torch.bfloat16)
    _check(v_pool, "v_pool", torch.bfloat16, (num_pages, g, page_size, d))
    _check(block_table, "block_table", torch.int32, (B, max_blocks))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    _check(k_new, "k_new", torch.bfloat16, (B, T, g, d))
    _check(v_new, "v_new", torch.bfloat16, (B, T, g, d))
    if status is not None:
        _check(status, "status", torch.int32)
    rc = lib.kv_cache_append_paged(_ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                   _ptr(seq_lens), _ptr(k_new), _ptr(v_new), B, g, d, page_size,
                                   num_pages, max_blocks, T, _ptr(status),
                                   _stream_ptr(stream, k_pool.device))
    if rc != GQA_OK:
        raise GQAError(rc, "kv_cache_append_paged")


def _rope_operands(q, q_out, rope_cos, rope_sin, B, T, d):
    _check(rope_cos, "rope_cos", torch.float32)
    n_pos = rope_cos.shape[0]
    _check(rope_cos, "rope_cos", torch.float32, (n_pos, d // 2))
    _check(rope_sin, "rope_sin", torch.float32, (n_pos, d // 2))
    h_q = 0
    if q is not None:
        h_q = q.shape[2]
        _check(q, "q", torch.bfloat16, (B, T, h_q, d))
        if q_out is None:
            q_out = q
        _check(q_out, "q_out", torch.bfloat16, (B, T, h_q, d))
    elif q_out is not None:
        raise ValueError("q_out given without q")
    return q_out, n_pos, h_q


def kv_cache_append_rope(k_cache: torch.Tensor, v_cache: torch.Tensor, seq_lens: torch.Tensor,
                         k_new: torch.Tensor, v_new: torch.Tensor, rope_cos: torch.Tensor,
                         rope_sin: torch.Tensor, *, q: Optional[torch.Tensor] = None,
                         q_out: Optional[torch.Tensor] = None,
                         status: Optional[torch.Tensor] = None, stream=None):
    """kv_cache_append with RoPE: keys rotated into the cache at their rows,
    values copied, and (if q is given) the same tokens' queries rotated into
    q_out (default: in place). Returns q_out (or None)."""
    lib = load_library()
    B, g, S_max, d = k_cache.shape
    T = k_new.shape[1]
    _check(k_cache, "k_cache", torch.bfloat16)
    _check(v_cache, "v_cache", torch.bfloat16, (B, g, S_max, d))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    _check(k_new, "k_new", torch.bfloat16, (B, T, g, d))
    _check(v_new, "v_new", torch.bfloat16, (B, T, g, d))
    q_out, n_pos, h_q = _rope_operands(q, q_out, rope_cos, rope_sin, B, T, d)
    if status is not None:
        _check(status, "status", torch.int32)
    rc = lib.kv_cache_append_rope(_ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), _ptr(k_new),
                                  _ptr(v_new), _ptr(q), _ptr(q_out), _ptr(rope_cos),
                                  _ptr(rope_sin), n_pos, B, h_q, g, d, S_max, T, _ptr(status),
                                  _stream_ptr(stream, k_cache.device))
    if rc != GQA_OK:
        raise GQAError(rc, "kv_cache_append_rope")
    return q_out


def kv_cache_append_paged_rope(k_pool: torch.Tensor, v_pool: torch.Tensor,
                               block_table: torch.Tensor, seq_lens: torch.Tensor,
                               k_new: torch.Tensor, v_new: torch.Tensor, rope_cos: torch.Tensor,
                               rope_sin: torch.Tensor, *, q: Optional[torch.Tensor] = None,
                               q_out: Optional[torch.Tensor] = None,
                               status: Optional[torch.Tensor] = None, stream=None):
    """kv_cache_append_rope into a paged pool through the block table."""
    lib = load_library()
    num_pages, g, page_size, d = k_pool.shape
    B, max_blocks = block_table.shape
    T = k_new.shape[1]
    _check(k_pool, "k_pool", torch.bfloat16)
    _check(v_pool, "v_pool", torch.bfloat16, (num_pages, g, page_size, d))
    _check(block_table, "block_table", torch.int32, (B, max_blocks))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    _check(k_new, "k_new", torch.bfloat16, (B, T, g, d))
    _check(v_new, "v_new", torch.bfloat16, (B, T, g, d))
    q_out, n_pos, h_q = _rope_operands(q, q_out, rope_cos, rope_sin, B, T, d)
    if status is not None:
        _check(status, "status", torch.int32)
    rc = lib.kv_cache_append_paged_rope(_ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                        _ptr(seq_lens), _ptr(k_new), _ptr(v_new), _ptr(q),
                                        _ptr(q_out), _ptr(rope_cos), _ptr(rope_sin), n_pos, B,
                                        h_q, g, d, page_size, num_pages, max_blocks, T,
                                        _ptr(status), _stream_ptr(stream, k_pool.device))
    if rc != GQA_OK:
        raise GQAError(rc, "kv_cache_append_paged_rope")
    return q_out


def gqa_selftest_bounded_wait(status: torch.Tensor, limit_us: int = 1000, stream=None) -> None:
    """Run the kernels' bounded wait against a barrier that never completes;
    ``status`` (device int32) then holds GQA_ERR_TIMEOUT."""
    lib = load_library()
    _check(status, "status", torch.int32)
    rc = lib.gqa_selftest_bounded_wait(_ptr(status), int(limit_us),
                                       _stream_ptr(stream, status.device))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_selftest_bounded_wait")
