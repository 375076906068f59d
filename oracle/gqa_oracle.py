"""Plain fp64 CPU oracle for the grouped-query attention (GQA) forward pass.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this module:
the tests, the smoke check and the benchmark's CPU-baseline leg are its only
callers. It shares no code, tables or helpers with the CUDA library.

What it computes, and where the pages define it
-----------------------------------------------
* Scaled dot-product attention ``softmax(Q K^T / sqrt(d_k)) V``:
  "Modern LLM architecture (1): GQA and RMSNorm" (zeeklog.com), section 2.1,
  the Attention formula.
* GQA: ``h_q`` query heads, ``g`` key/value heads, ``group_size = h_q // g``.
  Every K/V head is duplicated ``group_size`` times along the head axis
  (``repeat_interleave(group_size, dim=1)``) so that query head ``i`` reads
  K/V head ``i // group_size``; scores are scaled by ``1/sqrt(head_dim)``,
  masked entries set to ``-inf`` before the softmax, then multiplied by V:
  same page, section 2.3, the GroupedQueryAttention code.  The index map is
  stated again as ``kv_head_id = query_head_id // group_size`` in the
  "Qwen, DeepSeek and LLaMA3 attention survey" (jsqmd.com), section 2.2.
* KV cache: two tensors ``[batch, g, seq_len, d_head]`` that grow by
  concatenation along the sequence axis, and a decode step in which one new
  query token attends over every cached K/V row: "What is Grouped-Query
  Attention" explainer (ijyty.com), section 2.1 and section 2.2 (second step),
  section 3.2 (cache concat).

* Score-bias variants named by the pages: the sliding-window attention of
  Mistral (the model table of the zeeklog.com page, section 2.4) and ALiBi,
  a per-head linear distance penalty ``-slope_h * |i - j|`` added to the
  scores (the jsqmd.com survey, section 3.2).
* Chunked prefill against a KV cache: new query tokens attend to the cached
  rows and, causally, to each other (the cache concatenation of the ijyty.com
  explainer, section 3.2, applied to more than one new token).
* Paged KV cache with group-aligned pages (the jsqmd.com survey, section 4.3,
  on PagedAttention: a page holds page_size tokens of one K/V group, and the
  pages of the g groups of one block sit next to each other): a pool
  ``[num_pages, g, page_size, d]`` and a per-sequence block table whose entry
  ``i`` is the physical page of logical rows ``i*page_size .. (i+1)*page_size-1``.

* Rotary position embedding (RoPE) of queries and keys: the pair
  ``(x[2i], x[2i+1])`` of a row at position ``p`` is turned by the angle whose
  cosine and sine are ``cos[p, i]`` and ``sin[p, i]``; the turned even parts
  form the first half of the output row and the turned odd parts the second
  half (the RoPE code of the jsqmd.com survey, chapter 1, whose cos/sin
  tables of shape ``[seq_len, head_dim // 2]`` are inputs). Applied to the new
  tokens' Q and K rows on their way into the cache, at the positions they
  take there (the survey's fused-RoPE build option, chapter 5).

Readings where the pages are silent (each listed in the design notes):
* causal mask: key ``j`` is visible to query ``i`` iff ``j <= i + q_offset``
  (``q_offset = 0`` when queries and keys cover the same positions; a chunk
  of T new tokens over L cached keys has ``q_offset = L - T``);
* sliding window of size W (causal only): key ``j`` is also required to
  satisfy ``j > i + q_offset - W``;
* ALiBi: ``slope_h * |i + q_offset - j|`` (natural-log units, one slope per
  query head, supplied by the caller) is subtracted from the scaled score;
* a decode query sits at position ``seq_len - 1`` of its sequence;
* dropout is the identity (inference);
* a decode row with zero valid cache rows returns zeros and ``lse = -inf``;
* ``append`` drops rows that would land past ``S_max`` and reports it;
* RoPE precision: the survey's code multiplies bf16 rows by fp32 tables, so
  the rotation is evaluated in binary32 (each product and the sum or
  difference rounded to binary32, no fused multiply-add) and the result is
  rounded to bf16 when it is stored; a new token ``t`` of sequence ``b`` sits
  at position ``seq_lens[b] + t`` (the cache row it is written to), and query
  rows of tokens dropped for lack of room are left unwritten.

Everything here is the definition written out: one K/V duplication, one
score matrix per (batch, head), one softmax, one product with V. No tiling,
no online softmax, no fusion.

Parity pins (tests/test_oracle_pins.py): PyTorch's library SDPA with
``enable_gqa`` in fp64, brute-force loops on tiny inputs, the MHA (g = h_q)
and MQA (g = 1, broadcast ``expand`` form) special cases, hand-derived
closed-form fixtures under tests/golden/, and the invariants listed there.
"""

from __future__ import annotations

import numpy as np

# Status values reported by ``append``; they mirror the numbering the C
# interface documents, written out here independently.
APPEND_OK = 0
APPEND_CACHE_FULL = 5


# ---------------------------------------------------------------------------
# bf16 <-> fp64 (exact definitions of the storage format)
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 numbers given as their raw uint16 bit patterns.

    bf16 is the upper half of an IEEE-754 binary32, so widening is a shift.
    """
    u32 = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 (round to nearest, ties to even).

    Used only to state what a bf16 output must equal; NaN is not expected.
    """
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return rounded.astype(np.uint16)


# ---------------------------------------------------------------------------
# Building blocks of the definition
# ---------------------------------------------------------------------------

def head_map(h_q: int, g: int) -> np.ndarray:
    """K/V head read by each query head: ``i // (h_q // g)``."""
    if g <= 0 or h_q % g != 0:
        raise ValueError("h_q must be a positive multiple of g")
    group_size = h_q // g
    return np.array([i // group_size for i in range(h_q)], dtype=np.int64)


def _expand_kv(x: np.ndarray, group_size: int, axis: int) -> np.ndarray:
    """Duplicate every K/V head ``group_size`` times, consecutively.

    Same result as ``repeat_interleave(group_size, dim=head_axis)``: head
    ``j`` becomes heads ``j*group_size .. j*group_size + group_size - 1``.
    """
    return np.repeat(x, group_size, axis=axis)


def _visible(i: int, j: int, q_offset: int, window: int = 0) -> bool:
    """Causal visibility of key ``j`` to query row ``i`` (and the window)."""
    if j > i + q_offset:
        return False
    return window <= 0 or j > i + q_offset - window


def _alibi_bias(n_q: int, n_k: int, slope: float, q_offset: int) -> np.ndarray:
    """ALiBi penalty ``-slope * |i + q_offset - j|`` for every (query, key)."""
    i = np.arange(n_q)[:, None] + q_offset
    j = np.arange(n_k)[None, :]
    return -slope * np.abs(i - j).astype(np.float64)


def _softmax_rows(scores: np.ndarray):
    """Row softmax; returns (P, row max, row sum of exp(s - max)).

    Rows that are entirely ``-inf`` give P = 0 and sum 0.
    """
    m = np.max(scores, axis=-1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(scores - m_safe)
    s = np.sum(e, axis=-1, keepdims=True)
    p = np.divide(e, s, out=np.zeros_like(e), where=s > 0)
    return p, m, s


def _lse(m: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Natural-log sum-exp of a row from its max and its shifted sum."""
    with np.errstate(divide="ignore"):
        return np.where(s > 0, m + np.log(np.where(s > 0, s, 1.0)), -np.inf)


# ---------------------------------------------------------------------------
# Prefill
# ---------------------------------------------------------------------------

def attention_probs(q, k, causal: bool, scale: float, q_offset: int = 0):
    """Attention weights P[b, h, i, j] (tiny inputs; used by invariant tests).

    q: [B, Lq, h_q, d]; k: [B, Lk, g, d].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    B, Lq, h_q, _ = q.shape
    Lk, g = k.shape[1], k.shape[2]
    group_size = h_q // g
    out = np.zeros((B, h_q, Lq, Lk))
    for b in range(B):
        k_rep = _expand_kv(k[b], group_size, axis=1)  # [Lk, h_q, d]
        for h in range(h_q):
            s = (q[b, :, h, :] @ k_rep[:, h, :].T) * scale
            if causal:
                for i in range(Lq):
                    for j in range(Lk):
                        if not _visible(i, j, q_offset):
                            s[i, j] = -np.inf
            out[b, h], _, _ = _softmax_rows(s)
    return out


def prefill(q, k, v, causal: bool, scale: float, q_offset: int = 0, window: int = 0,
            alibi_slopes=None):
    """GQA prefill: ``O = softmax(Q K_rep^T * scale + bias + mask) V_rep``.

    q: [B, Lq, h_q, d]; k, v: [B, Lk, g, d] (the projection output layout
    ``view(B, L, heads, d_head)``).  Returns (O [B, Lq, h_q, d] fp64,
    lse [B, h_q, Lq] fp64, natural log).  Query row ``i`` sits at key
    position ``i + q_offset``; ``causal`` hides later keys, ``window`` > 0
    (causal only) also hides keys ``window`` or more positions back, and
    ``alibi_slopes`` ([h_q], or None) subtracts ``slope_h * distance``.
    A row that sees no key returns zeros and lse = -inf.
    """
    if window > 0 and not causal:
        raise ValueError("a sliding window needs causal attention")
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Lq, h_q, d = q.shape
    Lk, g = k.shape[1], k.shape[2]
    if h_q % g != 0:
        raise ValueError("h_q must be a multiple of g")
    group_size = h_q // g
    if causal:
        mask = np.zeros((Lq, Lk), dtype=bool)
        for i in range(Lq):
            for j in range(Lk):
                mask[i, j] = not _visible(i, j, q_offset, window)
    out = np.empty((B, Lq, h_q, d))
    lse = np.empty((B, h_q, Lq))
    for b in range(B):
        # explicit per-head duplication of K and V, one batch element at a time
        k_rep = _expand_kv(k[b], group_size, axis=1)  # [Lk, h_q, d]
        v_rep = _expand_kv(v[b], group_size, axis=1)
        for h in range(h_q):
            s = (q[b, :, h, :] @ k_rep[:, h, :].T) * scale
            if alibi_slopes is not None:
                s = s + _alibi_bias(Lq, Lk, float(alibi_slopes[h]), q_offset)
            if causal:
                s[mask] = -np.inf
            p, m, ssum = _softmax_rows(s)
            out[b, :, h, :] = p @ v_rep[:, h, :]
            lse[b, h, :] = _lse(m, ssum)[:, 0]
    return out, lse


def prefill_cached(q, k_cache, v_cache, seq_lens, scale: float, window: int = 0,
                   alibi_slopes=None):
    """Chunked prefill over a KV cache (bottom-right causal alignment).

    q: [B, T, h_q, d], the T newest tokens of each sequence; k_cache,
    v_cache: [B, g, S_max, d] already holding those tokens' K/V at the end of
    each sequence; seq_lens: [B] rows per sequence, each >= T. Token ``t`` of
    sequence ``b`` sits at position ``seq_lens[b] - T + t`` and sees every
    cached row up to its own position. Returns (O [B, T, h_q, d],
    lse [B, h_q, T]).
    """
    q = np.asarray(q, dtype=np.float64)
    B, T = q.shape[0], q.shape[1]
    outs, lses = [], []
    for b in range(B):
        n = int(seq_lens[b])
        if n < T:
            raise ValueError("every sequence must hold at least the T new tokens")
        # the cache rows of this sequence in the projection layout [1, n, g, d]
        kb = np.asarray(k_cache[b:b + 1, :, :n, :], dtype=np.float64).transpose(0, 2, 1, 3)
        vb = np.asarray(v_cache[b:b + 1, :, :n, :], dtype=np.float64).transpose(0, 2, 1, 3)
        o, l = prefill(q[b:b + 1], kb, vb, True, scale, q_offset=n - T, window=window,
                       alibi_slopes=alibi_slopes)
        outs.append(o)
        lses.append(l)
    return np.concatenate(outs, axis=0), np.concatenate(lses, axis=0)


# ---------------------------------------------------------------------------
# Decode over a [B, g, S_max, d] KV cache
# ---------------------------------------------------------------------------

def decode(q, k_cache, v_cache, seq_lens, scale: float, window: int = 0, alibi_slopes=None):
    """One-token GQA decode over the cache.

    q: [B, h_q, d]; k_cache, v_cache: [B, g, S_max, d]; seq_lens: [B] valid
    rows per sequence. The query sits at position ``seq_lens[b] - 1``; row
    ``j`` of sequence ``b`` is visible iff ``j < seq_lens[b]`` (and, with a
    window, ``j >= seq_lens[b] - window``); ``alibi_slopes`` subtracts
    ``slope_h * (seq_lens[b] - 1 - j)``. Returns (O [B, h_q, d], lse [B, h_q]).
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    B, h_q, d = q.shape
    g = k_cache.shape[1]
    group_size = h_q // g
    out = np.zeros((B, h_q, d))
    lse = np.full((B, h_q), -np.inf)
    for b in range(B):
        n = int(seq_lens[b])
        if n <= 0:
            continue
        k_rep = _expand_kv(k_cache[b, :, :n, :], group_size, axis=0)  # [h_q, n, d]
        v_rep = _expand_kv(v_cache[b, :, :n, :], group_size, axis=0)
        for h in range(h_q):
            s = (k_rep[h] @ q[b, h]) * scale  # [n]
            if alibi_slopes is not None:
                s = s + _alibi_bias(1, n, float(alibi_slopes[h]), n - 1)[0]
            if window > 0:
                s = np.where(np.arange(n) >= n - window, s, -np.inf)
            p, m, ssum = _softmax_rows(s[None, :])
            out[b, h] = (p @ v_rep[h])[0]
            lse[b, h] = _lse(m, ssum)[0, 0]
    return out, lse


# ---------------------------------------------------------------------------
# KV cache append
# ---------------------------------------------------------------------------

def append(k_cache, v_cache, seq_lens, k_new, v_new):
    """Write T new tokens per sequence at the end of its valid rows.

    k_cache, v_cache: [B, g, S_max, d] (any dtype; copied, not converted);
    seq_lens: [B]; k_new, v_new: [B, T, g, d] (projection layout).
    Token ``t`` of sequence ``b`` goes to cache row ``seq_lens[b] + t`` of
    every K/V head -- the concatenation along the sequence axis.  Rows that
    would land at or past ``S_max`` are dropped and the status becomes
    APPEND_CACHE_FULL; the new length is ``min(seq_lens[b] + T, S_max)``.
    Returns (k_cache', v_cache', seq_lens', status).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    lens = np.array(seq_lens, copy=True).astype(np.int64)
    B, g, S_max, _ = kc.shape
    T = k_new.shape[1]
    status = APPEND_OK
    new_lens = lens.copy()
    for b in range(B):
        for t in range(T):
            pos = int(lens[b]) + t
            if pos >= S_max:
                status = APPEND_CACHE_FULL
                continue
            for h in range(g):
                kc[b, h, pos, :] = k_new[b, t, h, :]
                vc[b, h, pos, :] = v_new[b, t, h, :]
        new_lens[b] = min(int(lens[b]) + T, S_max)
    return kc, vc, new_lens, status


# ---------------------------------------------------------------------------
# Paged KV cache
# ---------------------------------------------------------------------------

def gather_paged(pool, block_table, seq_lens, page_size: int):
    """Contiguous ``[B, g, S, d]`` copy of a paged cache, S = blocks * page_size.

    Logical row ``j`` of sequence ``b`` is row ``j % page_size`` of physical
    page ``block_table[b][j // page_size]`` (of every K/V head). Rows at or
    past ``seq_lens[b]`` are filled with zeros (they are never visible).
    """
    pool = np.asarray(pool)
    table = np.asarray(block_table)
    B, n_blocks = table.shape
    g, d = pool.shape[1], pool.shape[3]
    out = np.zeros((B, g, n_blocks * page_size, d), dtype=pool.dtype)
    for b in range(B):
        for j in range(int(seq_lens[b])):
            page = int(table[b, j // page_size])
            out[b, :, j, :] = pool[page, :, j % page_size, :]
    return out


def decode_paged(q, k_pool, v_pool, block_table, seq_lens, page_size: int, scale: float,
                 window: int = 0, alibi_slopes=None):
    """One-token GQA decode over a paged cache: the decode of the gathered rows."""
    kc = gather_paged(k_pool, block_table, seq_lens, page_size)
    vc = gather_paged(v_pool, block_table, seq_lens, page_size)
    return decode(q, kc, vc, seq_lens, scale, window=window, alibi_slopes=alibi_slopes)


def append_paged(k_pool, v_pool, block_table, seq_lens, k_new, v_new, page_size: int):
    """``append`` for a paged cache: token ``t`` of sequence ``b`` goes to logical
    row ``seq_lens[b] + t``, i.e. row ``(seq_lens[b] + t) % page_size`` of page
    ``block_table[b][(seq_lens[b] + t) // page_size]``; rows past the table's
    capacity are dropped and reported as APPEND_CACHE_FULL.
    Returns (k_pool', v_pool', seq_lens', status).
    """
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool, copy=True)
    table = np.asarray(block_table)
    lens = np.array(seq_lens, copy=True).astype(np.int64)
    B, n_blocks = table.shape
    cap = n_blocks * page_size
    g = kp.shape[1]
    T = k_new.shape[1]
    status = APPEND_OK
    new_lens = lens.copy()
    for b in range(B):
        for t in range(T):
            pos = int(lens[b]) + t
            if pos >= cap:
                status = APPEND_CACHE_FULL
                continue
            page = int(table[b, pos // page_size])
            for h in range(g):
                kp[page, h, pos % page_size, :] = k_new[b, t, h, :]
                vp[page, h, pos % page_size, :] = v_new[b, t, h, :]
        new_lens[b] = min(int(lens[b]) + T, cap)
    return kp, vp, new_lens, status


# ---------------------------------------------------------------------------
# Rotary position embedding on the way into the cache
# ---------------------------------------------------------------------------

def rope(x, cos, sin, positions):
    """The survey's rotary embedding in fp64 (jsqmd.com, chapter 1).

    x: [..., n, d] rows; positions: [n] (or broadcastable) table rows;
    cos, sin: [n_pos, d // 2]. Returns the rows with
    ``out[..., i] = x[2i] cos - x[2i+1] sin`` and
    ``out[..., d/2 + i] = x[2i] sin + x[2i+1] cos``.
    """
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(cos, dtype=np.float64)[np.asarray(positions)]
    s = np.asarray(sin, dtype=np.float64)[np.asarray(positions)]
    even = x[..., 0::2]
    odd = x[..., 1::2]
    return np.concatenate([even * c - odd * s, even * s + odd * c], axis=-1)


def rope_f32(x, cos, sin, positions):
    """``rope`` as the survey's code evaluates it for bf16 rows and fp32
    tables: every product, sum and difference rounded to binary32."""
    x = np.asarray(x, dtype=np.float32)
    c = np.asarray(cos, dtype=np.float32)[np.asarray(positions)]
    s = np.asarray(sin, dtype=np.float32)[np.asarray(positions)]
    even = x[..., 0::2]
    odd = x[..., 1::2]
    first = (even * c).astype(np.float32) - (odd * s).astype(np.float32)
    second = (even * s).astype(np.float32) + (odd * c).astype(np.float32)
    return np.concatenate([first, second], axis=-1).astype(np.float32)


def _rope_new_rows(x_bits, cos, sin, seq_lens, capacity):
    """Rotate rows ``[B, T, H, d]`` (bf16 bit patterns) of new tokens at their
    cache positions ``seq_lens[b] + t``; rows at or past ``capacity`` (dropped)
    are returned as given. Result: bf16 bit patterns."""
    x_bits = np.asarray(x_bits).view(np.uint16)
    out = x_bits.copy()
    B, T = x_bits.shape[:2]
    for b in range(B):
        for t in range(T):
            pos = int(seq_lens[b]) + t
            if pos >= capacity:
                continue
            row = bf16_bits_to_f64(x_bits[b, t])  # [H, d], exact
            out[b, t] = f32_to_bf16_bits(rope_f32(row, cos, sin, pos))
    return out


def append_rope(k_cache, v_cache, seq_lens, k_new, v_new, cos, sin, q=None, q_out=None):
    """``append`` of RoPE-rotated keys, and the new tokens' queries rotated at
    the same positions.

    k_cache, v_cache, k_new, v_new, q, q_out: bf16 bit patterns (uint16 or
    int16 views); q, q_out: [B, T, h_q, d]. Returns
    (k_cache', v_cache', seq_lens', status, q_out') where q_out' is q_out
    (a copy of q if q_out is None) with the rows of stored tokens replaced by
    their rotated queries. V rows are copied unchanged.
    """
    S_max = np.asarray(k_cache).shape[2]
    k_rot = _rope_new_rows(k_new, cos, sin, seq_lens, S_max)
    kc, vc, lens, status = append(np.asarray(k_cache).view(np.uint16),
                                  np.asarray(v_cache).view(np.uint16), seq_lens, k_rot,
                                  np.asarray(v_new).view(np.uint16))
    q_res = None
    if q is not None:
        q_res = _merge_rotated_queries(q, q_out, cos, sin, seq_lens, S_max)
    return kc, vc, lens, status, q_res


def append_paged_rope(k_pool, v_pool, block_table, seq_lens, k_new, v_new, page_size: int,
                      cos, sin, q=None, q_out=None):
    """``append_rope`` into a paged cache (positions are logical rows)."""
    cap = np.asarray(block_table).shape[1] * page_size
    k_rot = _rope_new_rows(k_new, cos, sin, seq_lens, cap)
    kp, vp, lens, status = append_paged(np.asarray(k_pool).view(np.uint16),
                                        np.asarray(v_pool).view(np.uint16), block_table,
                                        seq_lens, k_rot, np.asarray(v_new).view(np.uint16),
                                        page_size)
    q_res = None
    if q is not None:
        q_res = _merge_rotated_queries(q, q_out, cos, sin, seq_lens, cap)
    return kp, vp, lens, status, q_res


def _merge_rotated_queries(q, q_out, cos, sin, seq_lens, capacity):
    q_bits = np.asarray(q).view(np.uint16)
    res = (q_bits if q_out is None else np.asarray(q_out).view(np.uint16)).copy()
    rot = _rope_new_rows(q_bits, cos, sin, seq_lens, capacity)
    B, T = q_bits.shape[:2]
    for b in range(B):
        for t in range(T):
            if int(seq_lens[b]) + t < capacity:
                res[b, t] = rot[b, t]
    return res
