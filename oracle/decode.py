"""fp64 CPU oracle for one autoregressive decode step of grouped-query attention.

TEST INFRASTRUCTURE. This module is the reference the CUDA path is checked
against. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import it; the library itself never does,
and nothing here calls the CUDA library.

Everything is float64 on values that were first rounded to the cache dtype.
No blocking, fusion or split: each function is the plain definition, so it
can be checked against the pages by eye.

Sources (page title, then section / equation):
  * "KV Cache" explainer (lensaml.com), Langkah 3 "Menyimpan Key dan Value di
    Cache": the cache of a layer is a pair [batch, kv_heads, tokens, head_dim];
    each decode step writes one slice on the token axis; each key is rotated
    (RoPE) by its position once and stored rotated; only the newest token is
    projected.
  * "Grouped-query attention: berbagi KV head di antara grup query"
    (nalar.dev), section "Jumlah head menentukan batas grup": G = H_q / H_kv,
    g(h) = floor(h / G), A_h = softmax(Q_h K_g(h)^T / sqrt(d)), O_h = A_h V_g(h).
  * same page, "GQA berada di antara MHA dan MQA": H_kv = H_q is MHA,
    H_kv = 1 is MQA.
  * "KV Cache 최적화 심층 분석: GQA·MLA·MHA" (youngju.dev), class PagedKVCache:
    block index = position // block_size, offset = position % block_size,
    gathering a sequence walks its block table in order.
  * "Arsitektur Inferensi LLM ..." (tveniu.com) section 4 PagedAttention:
    logical block i of a request maps to a physical block through the page
    table, 16 tokens per block.
  * "KV Cache" explainer, Langkah 1 and FAQ: the causal mask is what makes the
    cache valid; cached and uncached computation give the same result in exact
    arithmetic.

Readings where the pages are silent (the pages give no RoPE formula):
  * RoPE rotates adjacent pairs (x[2i], x[2i+1]) by angle pos * theta_i with
    theta_i = base^(-2i/d), i in [0, d/2): (x cos - y sin, x sin + y cos).
  * The position is the 0-based cache index of the token; q and k of the new
    token use the same position; q is rotated and never stored.
  * The decode query attends to every cached position including its own.
  * Scale 1/sqrt(d). Stored keys and values are rounded to the cache dtype
    (round to nearest, ties to even); the attention reads the stored values.

Parity pins (tests/test_oracle_pins.py): every function below is pinned by at
least one test against something other than itself.
"""

from __future__ import annotations

import numpy as np

F64 = np.float64
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


# ---------------------------------------------------------------- rounding
def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), kept as float64.

    bfloat16 has 8 significant bits and fp32's exponent range: the quantum of a
    value with binary exponent e (x = m 2^e, 0.5 <= |m| < 1) is 2^(e-8), never
    below the subnormal quantum 2^-133.
    """
    x = np.asarray(x, dtype=F64)
    _, e = np.frexp(x)
    q_exp = np.maximum(e.astype(np.int64) - 8, -133)
    r = np.ldexp(np.round(np.ldexp(x, -q_exp)), q_exp)  # np.round: half to even
    big = np.isfinite(x) & (np.abs(r) > BF16_MAX)
    return np.where(big, np.copysign(np.inf, x), r)


def round_to(x, dtype: str) -> np.ndarray:
    """Round to the storage dtype: "bf16", "f32", or "f64" (exact)."""
    x = np.asarray(x, dtype=F64)
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "f32":
        return x.astype(np.float32).astype(F64)
    if dtype == "f64":
        return x.copy()
    raise ValueError(dtype)


# --------------------------------------------------------- uint8 KV cache
def quantize_u8(x):
    """Asymmetric uint8 quantisation of each row of the last axis, the pages'
    QuantizedKVCache ("KV Cache 최적화 심층 분석", youngju.dev):
    scale = (max - min) / 255, zero_point = round(-min / scale) clamped to
    [0, 255], code = round(x / scale + zero_point) clamped to [0, 255] (round
    half to even, as torch.round). Reading: the arithmetic is float32, in that
    operation order, and a constant row (max == min) takes scale 1.
    Returns (codes uint8 [..., d], scale float32 [...], zero_point float32 [...])."""
    x = np.asarray(x, dtype=np.float32)
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    scale = ((mx - mn) / np.float32(255.0)).astype(np.float32)
    scale = np.where(scale == 0, np.float32(1.0), scale).astype(np.float32)
    zp = np.clip(np.rint((-mn) / scale), 0, 255).astype(np.float32)
    codes = np.clip(np.rint(x / scale[..., None] + zp[..., None]), 0, 255).astype(np.uint8)
    return codes, scale, zp


def dequantize_u8(codes, scale, zp):
    """(code - zero_point) * scale, exactly (float64)."""
    return (np.asarray(codes, F64) - np.asarray(zp, F64)[..., None]) * np.asarray(scale, F64)[..., None]


# ------------------------------------------------------ fp8 (e5m2) KV cache
E5M2_MAX = 57344.0  # 1.75 * 2^15, the largest finite e5m2 value


def quantize_e5m2(x):
    """fp8 e5m2 codes of float64 values: the KV-cache format of the serving
    flag `--kv-cache-dtype fp8_e5m2` in the vLLM examples ("KV Cache 최적화
    심층 분석", youngju.dev, the deployment section; "Arsitektur Inferensi
    LLM", tveniu.com, the vLLM configuration). e5m2 is 1 sign bit, 5 exponent
    bits (bias 15) and 2 mantissa bits: (1 + m/4) 2^(E-15) for E in 1..30,
    (m/4) 2^-14 for E = 0, E = 31 infinities and NaN.
    Readings (the pages name the flag only): round to nearest, ties to even,
    on the float64 value itself; magnitudes beyond the largest finite value
    saturate to it; NaN maps to a NaN code. Returns uint8 codes."""
    x = np.asarray(x, F64)
    ax = np.abs(x)
    _, e = np.frexp(ax)                                    # ax = m 2^e, 0.5 <= m < 1
    q_exp = np.maximum(e.astype(np.int64) - 3, -16)        # quantum: 2 bits below the leading one, >= 2^-16
    r = np.minimum(np.ldexp(np.rint(np.ldexp(ax, -q_exp)), q_exp), E5M2_MAX)  # np.rint: half to even
    mr, er = np.frexp(r)
    binade = er.astype(np.int64) - 1
    normal = (r > 0) & (binade >= -14)
    field = np.where(normal, binade + 15, 0)
    mant = np.where(normal, np.ldexp(r, -binade) * 4 - 4, np.ldexp(r, 16))
    codes = (field * 4 + np.rint(mant)).astype(np.int64)
    codes = np.where(np.isnan(x), 0x7F, codes)
    codes = np.where(np.signbit(x), codes | 0x80, codes)
    return codes.astype(np.uint8)


def dequantize_e5m2(codes):
    """Value of each e5m2 code (float64), from the format's definition."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    field = (c >> 2) & 31
    m = (c & 3).astype(F64)
    val = np.where(field == 0, np.ldexp(m, -16), np.ldexp(1.0 + m / 4.0, field - 15))
    val = np.where(field == 31, np.where(m == 0, np.inf, np.nan), val)
    return sign * val


# -------------------------------------------------------------------- RoPE
def rope_inv_freq(head_dim: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/d), i = 0 .. d/2-1 (reading; the pages give no formula)."""
    i = np.arange(head_dim // 2, dtype=F64)
    return np.power(F64(base), -2.0 * i / head_dim)


def rope_rotate(x, pos: int, base: float) -> np.ndarray:
    """Rotate every adjacent pair of the last axis of ``x`` by pos * theta_i.

    "KV Cache" explainer, Langkah 3: position information is applied before
    storing -- each key is rotated by its position once and stored rotated.
    """
    x = np.asarray(x, dtype=F64)
    ang = F64(pos) * rope_inv_freq(x.shape[-1], base)
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


# ------------------------------------------------------------ cache layout
def page_slot(table_row, pos: int, page_size: int) -> tuple[int, int]:
    """(physical page, offset) of token ``pos``: PagedKVCache block index
    pos // block_size looked up in the block table, offset pos % block_size."""
    return int(table_row[pos // page_size]), pos % page_size


def append_contiguous(k_cache, v_cache, b: int, pos: int, k_stored, v_stored) -> None:
    """Write one token slice at index ``pos`` of the token axis of sequence ``b``
    ([batch, kv_heads, tokens, head_dim] cache, "KV Cache" explainer Langkah 3)."""
    k_cache[b, :, pos, :] = k_stored
    v_cache[b, :, pos, :] = v_stored


def append_paged(k_pool, v_pool, table_row, page_size: int, pos: int, k_stored, v_stored) -> None:
    """Write one token slice into its page: pool[page, :, offset, :]."""
    page, off = page_slot(table_row, pos, page_size)
    k_pool[page, :, off, :] = k_stored
    v_pool[page, :, off, :] = v_stored


def gather_paged(pool, table_row, length: int, page_size: int) -> np.ndarray:
    """Assemble tokens [0, length) of one sequence as [kv_heads, length, d],
    walking the block table in logical order (PagedKVCache.get_kv)."""
    rows = []
    for t in range(length):
        page, off = page_slot(table_row, t, page_size)
        rows.append(pool[page, :, off, :])
    return np.stack(rows, axis=1).astype(F64)


# --------------------------------------------------------------- attention
def gqa_attention(q_rot, K, V, scale: float, return_weights: bool = False):
    """O_h = softmax(Q_h K_g(h)^T * scale) V_g(h), g(h) = floor(h / G), G = H_q / H_kv.

    q_rot [H_q, d]; K, V [H_kv, L, d]. Returns out [H_q, d] and the natural-log
    normaliser lse [H_q] = log sum_t exp(score_t) (and the weights [H_q, L]).
    Source: nalar.dev GQA page, equations for G, g(h), A_h and O_h.
    """
    q_rot = np.asarray(q_rot, dtype=F64)
    K = np.asarray(K, dtype=F64)
    V = np.asarray(V, dtype=F64)
    h_q, d = q_rot.shape
    h_kv, length, _ = K.shape
    G = h_q // h_kv
    out = np.empty((h_q, d), dtype=F64)
    lse = np.empty(h_q, dtype=F64)
    weights = np.empty((h_q, length), dtype=F64)
    for h in range(h_q):
        j = h // G
        s = (K[j] @ q_rot[h]) * scale
        m = s.max()
        w = np.exp(s - m)
        total = w.sum()
        weights[h] = w / total
        out[h] = (w @ V[j]) / total
        lse[h] = m + np.log(total)
    if return_weights:
        return out, lse, weights
    return out, lse


def mha_attention(q_rot, K, V, scale: float) -> np.ndarray:
    """Multi-head attention: head h reads its own K[h], V[h] (H_kv = H_q)."""
    s = np.einsum("hd,hld->hl", np.asarray(q_rot, F64), np.asarray(K, F64)) * scale
    s = s - s.max(axis=1, keepdims=True)
    w = np.exp(s)
    w = w / w.sum(axis=1, keepdims=True)
    return np.einsum("hl,hld->hd", w, np.asarray(V, F64))


def mqa_attention(q_rot, K1, V1, scale: float) -> np.ndarray:
    """Multi-query attention: every query head reads the one shared K1, V1 [L, d]."""
    s = (np.asarray(q_rot, F64) @ np.asarray(K1, F64).T) * scale
    s = s - s.max(axis=1, keepdims=True)
    w = np.exp(s)
    w = w / w.sum(axis=1, keepdims=True)
    return w @ np.asarray(V1, F64)


def window_start(length: int, window: int) -> int:
    """First token a query at position length-1 attends to: 0 for full
    attention (window 0), else max(0, length - window) -- the last `window`
    cached tokens, its own included ("KV Cache 최적화 심층 분석",
    SlidingWindowAttention: after the concatenation the cache keeps only its
    last window_size tokens)."""
    return 0 if window <= 0 else max(0, length - window)


def attention_partial(q_rot, K, V, scale: float, t0: int, t1: int):
    """Attention restricted to tokens [t0, t1): normalised partial output and its
    log-sum-exp; an empty range gives output 0 and lse = -inf."""
    h_q, d = np.asarray(q_rot).shape
    if t1 <= t0:
        return np.zeros((h_q, d), F64), np.full(h_q, -np.inf)
    return gqa_attention(q_rot, np.asarray(K)[:, t0:t1], np.asarray(V)[:, t0:t1], scale)


def lse_combine(o_parts, lse_parts):
    """Merge partial results over disjoint token ranges (flash-decoding combine).

    With O_s the normalised output over range s and lse_s its log-sum-exp:
    LSE = log sum_s exp(lse_s) and O = sum_s exp(lse_s - LSE) O_s.
    o_parts [S, ..., d], lse_parts [S, ...].
    """
    o_parts = np.asarray(o_parts, F64)
    lse_parts = np.asarray(lse_parts, F64)
    m = lse_parts.max(axis=0)
    w = np.exp(lse_parts - m)
    total = w.sum(axis=0)
    lse = m + np.log(total)
    out = (w[..., None] * o_parts).sum(axis=0) / total[..., None]
    return out, lse


def causal_attention(Q, K, V, scale: float) -> np.ndarray:
    """Full causal attention over n positions, every row: Q [H_q, n, d],
    K, V [H_kv, n, d]. Query heads are mapped to KV heads by repeating each KV
    head G times in order (the repeat_interleave / expand form of g(h)). Row i
    sees keys j <= i (mask = strictly upper triangle)."""
    Q = np.asarray(Q, F64)
    G = Q.shape[0] // K.shape[0]
    Kr = np.repeat(np.asarray(K, F64), G, axis=0)
    Vr = np.repeat(np.asarray(V, F64), G, axis=0)
    n = Q.shape[1]
    s = np.einsum("hid,hjd->hij", Q, Kr) * scale
    mask = np.triu(np.ones((n, n), dtype=bool), k=1)
    s = np.where(mask[None], -np.inf, s)
    s = s - s.max(axis=2, keepdims=True)
    w = np.exp(s)
    w = w / w.sum(axis=2, keepdims=True)
    return np.einsum("hij,hjd->hid", w, Vr)


# ------------------------------------------------------------- decode step
def _f64(t) -> np.ndarray:
    """Exact widening of a torch tensor or array to float64 numpy."""
    if hasattr(t, "detach"):
        t = t.detach().cpu()
        import torch  # local: torch is only needed to read bf16 tensors

        t = t.to(torch.float64).numpy()
    return np.asarray(t, dtype=F64)


def decode_step_contiguous(k_cache, v_cache, q_new, k_new, v_new, seq_lens, rope_base: float,
                           scale: float, cache_dtype: str, window: int = 0):
    """One decode step over a contiguous cache [B, H_kv, capacity, d].

    For each sequence b with length L_b (after append), p = L_b - 1:
    rotate q_new[b] and k_new[b] by p, store round(k_rot) and v_new[b] at
    token p, then attend over tokens [0, L_b) of the updated cache.
    Returns dict(out [B,H_q,d], lse [B,H_q], q_rot [B,H_q,d], k_cache, v_cache)
    with the caches as updated copies.
    """
    K = _f64(k_cache).copy()
    V = _f64(v_cache).copy()
    q_new, k_new, v_new = _f64(q_new), _f64(k_new), _f64(v_new)
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, h_q, d = q_new.shape
    out = np.empty((B, h_q, d), F64)
    lse = np.empty((B, h_q), F64)
    q_rot = np.empty((B, h_q, d), F64)
    for b in range(B):
        L = int(lens[b])
        p = L - 1
        q_rot[b] = rope_rotate(q_new[b], p, rope_base)
        k_stored = round_to(rope_rotate(k_new[b], p, rope_base), cache_dtype)
        append_contiguous(K, V, b, p, k_stored, v_new[b])
        t0 = window_start(L, window)
        out[b], lse[b] = gqa_attention(q_rot[b], K[b, :, t0:L], V[b, :, t0:L], scale)
    return {"out": out, "lse": lse, "q_rot": q_rot, "k_cache": K, "v_cache": V}


def decode_step_paged(k_pool, v_pool, block_table, q_new, k_new, v_new, seq_lens, page_size: int,
                      rope_base: float, scale: float, cache_dtype: str, window: int = 0):
    """One decode step over a paged pool [num_pages, H_kv, page_size, d] with a
    block table [B, max_pages]; same steps as the contiguous form, with the slot
    of token p at (table[b][p // page_size], p % page_size)."""
    K = _f64(k_pool).copy()
    V = _f64(v_pool).copy()
    table = np.asarray(_f64(block_table), dtype=np.int64)
    q_new, k_new, v_new = _f64(q_new), _f64(k_new), _f64(v_new)
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, h_q, d = q_new.shape
    out = np.empty((B, h_q, d), F64)
    lse = np.empty((B, h_q), F64)
    q_rot = np.empty((B, h_q, d), F64)
    for b in range(B):
        L = int(lens[b])
        p = L - 1
        q_rot[b] = rope_rotate(q_new[b], p, rope_base)
        k_stored = round_to(rope_rotate(k_new[b], p, rope_base), cache_dtype)
        append_paged(K, V, table[b], page_size, p, k_stored, v_new[b])
        t0 = window_start(L, window)
        Kb = gather_paged(K, table[b], L, page_size)[:, t0:]
        Vb = gather_paged(V, table[b], L, page_size)[:, t0:]
        out[b], lse[b] = gqa_attention(q_rot[b], Kb, Vb, scale)
    return {"out": out, "lse": lse, "q_rot": q_rot, "k_pool": K, "v_pool": V}


def decode_step_u8(k_codes, k_sz, v_codes, v_sz, q_new, k_new, v_new, seq_lens, rope_base: float, scale: float,
                   block_table=None, page_size: int = 0, window: int = 0):
    """One decode step over a uint8 cache (contiguous [B, H_kv, capacity, d]
    codes with (scale, zero_point) pairs [B, H_kv, capacity, 2], or paged
    [num_pages, H_kv, page_size, d] with a block table). The new token's key
    is rotated in fp64, rounded to fp32 and quantised; its value (bf16 input)
    is quantised; the attention reads the dequantised cache.
    Returns dict(out, lse, q_rot, k_codes, k_sz, v_codes, v_sz) with updated copies."""
    Kc, Vc = np.array(k_codes, copy=True), np.array(v_codes, copy=True)
    Ks, Vs = np.array(k_sz, dtype=np.float32, copy=True), np.array(v_sz, dtype=np.float32, copy=True)
    q_new, k_new, v_new = _f64(q_new), _f64(k_new), _f64(v_new)
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    table = None if block_table is None else np.asarray(_f64(block_table), dtype=np.int64)
    B, h_q, d = q_new.shape
    out = np.empty((B, h_q, d), F64)
    lse = np.empty((B, h_q), F64)
    q_rot = np.empty((B, h_q, d), F64)
    for b in range(B):
        L = int(lens[b])
        p = L - 1
        q_rot[b] = rope_rotate(q_new[b], p, rope_base)
        kq, ks, kz = quantize_u8(rope_rotate(k_new[b], p, rope_base))
        vq, vs, vz = quantize_u8(v_new[b])
        if table is None:
            Kc[b, :, p], Vc[b, :, p] = kq, vq
            Ks[b, :, p] = np.stack([ks, kz], -1)
            Vs[b, :, p] = np.stack([vs, vz], -1)
            Kd = dequantize_u8(Kc[b, :, :L], Ks[b, :, :L, 0], Ks[b, :, :L, 1])
            Vd = dequantize_u8(Vc[b, :, :L], Vs[b, :, :L, 0], Vs[b, :, :L, 1])
        else:
            page, off = page_slot(table[b], p, page_size)
            Kc[page, :, off], Vc[page, :, off] = kq, vq
            Ks[page, :, off] = np.stack([ks, kz], -1)
            Vs[page, :, off] = np.stack([vs, vz], -1)
            kcode = gather_paged(Kc, table[b], L, page_size)
            vcode = gather_paged(Vc, table[b], L, page_size)
            ksz = gather_paged(Ks, table[b], L, page_size)
            vsz = gather_paged(Vs, table[b], L, page_size)
            Kd = dequantize_u8(kcode, ksz[..., 0], ksz[..., 1])
            Vd = dequantize_u8(vcode, vsz[..., 0], vsz[..., 1])
        t0 = window_start(L, window)
        out[b], lse[b] = gqa_attention(q_rot[b], Kd[:, t0:], Vd[:, t0:], scale)
    return {"out": out, "lse": lse, "q_rot": q_rot, "k_codes": Kc, "k_sz": Ks, "v_codes": Vc, "v_sz": Vs}


def decode_step_e5m2(k_codes, v_codes, q_new, k_new, v_new, seq_lens, rope_base: float, scale: float,
                     block_table=None, page_size: int = 0, window: int = 0):
    """One decode step over an fp8 e5m2 cache (codes, contiguous [B, H_kv,
    capacity, d] or paged [num_pages, H_kv, page_size, d] with a block table).
    The new token's key is rotated in fp64 and rounded once to e5m2; its value
    (bf16 input) is rounded to e5m2; the attention reads the decoded cache.
    Returns dict(out, lse, q_rot, k_codes, v_codes) with updated copies."""
    Kc, Vc = np.array(k_codes, dtype=np.uint8, copy=True), np.array(v_codes, dtype=np.uint8, copy=True)
    q_new, k_new, v_new = _f64(q_new), _f64(k_new), _f64(v_new)
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    table = None if block_table is None else np.asarray(_f64(block_table), dtype=np.int64)
    B, h_q, d = q_new.shape
    out = np.empty((B, h_q, d), F64)
    lse = np.empty((B, h_q), F64)
    q_rot = np.empty((B, h_q, d), F64)
    for b in range(B):
        L = int(lens[b])
        p = L - 1
        q_rot[b] = rope_rotate(q_new[b], p, rope_base)
        kq = quantize_e5m2(rope_rotate(k_new[b], p, rope_base))
        vq = quantize_e5m2(v_new[b])
        if table is None:
            Kc[b, :, p], Vc[b, :, p] = kq, vq
            Kd = dequantize_e5m2(Kc[b, :, :L])
            Vd = dequantize_e5m2(Vc[b, :, :L])
        else:
            page, off = page_slot(table[b], p, page_size)
            Kc[page, :, off], Vc[page, :, off] = kq, vq
            Kd = dequantize_e5m2(gather_paged(Kc, table[b], L, page_size))
            Vd = dequantize_e5m2(gather_paged(Vc, table[b], L, page_size))
        t0 = window_start(L, window)
        out[b], lse[b] = gqa_attention(q_rot[b], Kd[:, t0:], Vd[:, t0:], scale)
    return {"out": out, "lse": lse, "q_rot": q_rot, "k_codes": Kc, "v_codes": Vc}


def decode_step_multi(k_cache, v_cache, q_new, k_new, v_new, seq_lens, rope_base: float, scale: float,
                      cache_dtype: str, block_table=None, page_size: int = 0, window: int = 0):
    """n new tokens per sequence in one pass: the target-model verification of
    speculative decoding ("Arsitektur Inferensi LLM", section 7), where the
    drafted tokens are checked in parallel and the result must equal decoding
    them one at a time.

    q_new [B, n, H_q, d], k_new / v_new [B, n, H_kv, d]; seq_lens = L_b after
    the append, so new token i of sequence b sits at position p = L_b - n + i.
    Each new token's q and k are rotated by p, its k (rounded to the cache
    dtype) and v stored at p (contiguous cache [B, H_kv, capacity, d], or a
    paged pool through block_table); query i then attends to the tokens
    [window_start(p + 1, W), p + 1) of the updated cache: causal within the
    new tokens.
    Returns dict(out [B,n,H_q,d], lse [B,n,H_q], q_rot [B,n,H_q,d], k_cache,
    v_cache) with the caches as updated copies.
    """
    K = _f64(k_cache).copy()
    V = _f64(v_cache).copy()
    q_new, k_new, v_new = _f64(q_new), _f64(k_new), _f64(v_new)
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    table = None if block_table is None else np.asarray(_f64(block_table), dtype=np.int64)
    B, n, h_q, d = q_new.shape
    out = np.empty((B, n, h_q, d), F64)
    lse = np.empty((B, n, h_q), F64)
    q_rot = np.empty((B, n, h_q, d), F64)
    for b in range(B):
        L = int(lens[b])
        for i in range(n):
            p = L - n + i
            q_rot[b, i] = rope_rotate(q_new[b, i], p, rope_base)
            k_stored = round_to(rope_rotate(k_new[b, i], p, rope_base), cache_dtype)
            if table is None:
                append_contiguous(K, V, b, p, k_stored, v_new[b, i])
            else:
                append_paged(K, V, table[b], page_size, p, k_stored, v_new[b, i])
        if table is None:
            Kb, Vb = K[b, :, :L], V[b, :, :L]
        else:
            Kb, Vb = gather_paged(K, table[b], L, page_size), gather_paged(V, table[b], L, page_size)
        for i in range(n):
            p = L - n + i
            t0 = window_start(p + 1, window)
            out[b, i], lse[b, i] = gqa_attention(q_rot[b, i], Kb[:, t0:p + 1], Vb[:, t0:p + 1], scale)
    res = {"out": out, "lse": lse, "q_rot": q_rot}
    res.update({"k_cache": K, "v_cache": V} if table is None else {"k_pool": K, "v_pool": V})
    return res


def decode_step_multi_e5m2(k_codes, v_codes, q_new, k_new, v_new, seq_lens, rope_base: float, scale: float,
                           block_table=None, page_size: int = 0, window: int = 0):
    """n new tokens per sequence in one pass (the verification of drafted
    tokens, "Arsitektur Inferensi LLM", section 7) over an fp8 e5m2 cache:
    decode_step_multi's steps with decode_step_e5m2's storage. New token i of
    sequence b sits at p = L_b - n + i; its q and k are rotated by p in fp64,
    its key is rounded once to e5m2 and its value (bf16 input) likewise, both
    stored at p; query i then attends to [window_start(p + 1, W), p + 1) of
    the decoded cache.
    Returns dict(out [B,n,H_q,d], lse [B,n,H_q], q_rot [B,n,H_q,d], k_codes,
    v_codes) with the codes as updated copies."""
    Kc, Vc = np.array(k_codes, dtype=np.uint8, copy=True), np.array(v_codes, dtype=np.uint8, copy=True)
    q_new, k_new, v_new = _f64(q_new), _f64(k_new), _f64(v_new)
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    table = None if block_table is None else np.asarray(_f64(block_table), dtype=np.int64)
    B, n, h_q, d = q_new.shape
    out = np.empty((B, n, h_q, d), F64)
    lse = np.empty((B, n, h_q), F64)
    q_rot = np.empty((B, n, h_q, d), F64)
    for b in range(B):
        L = int(lens[b])
        for i in range(n):
            p = L - n + i
            q_rot[b, i] = rope_rotate(q_new[b, i], p, rope_base)
            kq = quantize_e5m2(rope_rotate(k_new[b, i], p, rope_base))
            vq = quantize_e5m2(v_new[b, i])
            if table is None:
                Kc[b, :, p], Vc[b, :, p] = kq, vq
            else:
                page, off = page_slot(table[b], p, page_size)
                Kc[page, :, off], Vc[page, :, off] = kq, vq
        if table is None:
            Kd, Vd = dequantize_e5m2(Kc[b, :, :L]), dequantize_e5m2(Vc[b, :, :L])
        else:
            Kd = dequantize_e5m2(gather_paged(Kc, table[b], L, page_size))
            Vd = dequantize_e5m2(gather_paged(Vc, table[b], L, page_size))
        for i in range(n):
            p = L - n + i
            t0 = window_start(p + 1, window)
            out[b, i], lse[b, i] = gqa_attention(q_rot[b, i], Kd[:, t0:p + 1], Vd[:, t0:p + 1], scale)
    return {"out": out, "lse": lse, "q_rot": q_rot, "k_codes": Kc, "v_codes": Vc}


def decode_step_multi_u8(k_codes, k_sz, v_codes, v_sz, q_new, k_new, v_new, seq_lens, rope_base: float,
                         scale: float, block_table=None, page_size: int = 0, window: int = 0):
    """n new tokens per sequence in one pass (the verification of drafted
    tokens, "Arsitektur Inferensi LLM", section 7) over a uint8 cache (the
    QuantizedKVCache of "KV Cache 최적화 심층 분석"): decode_step_multi's steps
    with decode_step_u8's storage. New token i of sequence b sits at
    p = L_b - n + i; its q and k are rotated by p in fp64, its key (rounded to
    fp32) and its value (bf16 input) are quantised row by row and stored at p
    with their (scale, zero point); query i then attends to
    [window_start(p + 1, W), p + 1) of the dequantised cache.
    Returns dict(out [B,n,H_q,d], lse [B,n,H_q], q_rot [B,n,H_q,d], k_codes,
    k_sz, v_codes, v_sz) with the cache as updated copies."""
    Kc, Vc = np.array(k_codes, copy=True), np.array(v_codes, copy=True)
    Ks, Vs = np.array(k_sz, dtype=np.float32, copy=True), np.array(v_sz, dtype=np.float32, copy=True)
    q_new, k_new, v_new = _f64(q_new), _f64(k_new), _f64(v_new)
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    table = None if block_table is None else np.asarray(_f64(block_table), dtype=np.int64)
    B, n, h_q, d = q_new.shape
    out = np.empty((B, n, h_q, d), F64)
    lse = np.empty((B, n, h_q), F64)
    q_rot = np.empty((B, n, h_q, d), F64)
    for b in range(B):
        L = int(lens[b])
        for i in range(n):
            p = L - n + i
            q_rot[b, i] = rope_rotate(q_new[b, i], p, rope_base)
            kq, ks, kz = quantize_u8(rope_rotate(k_new[b, i], p, rope_base))
            vq, vs, vz = quantize_u8(v_new[b, i])
            if table is None:
                Kc[b, :, p], Vc[b, :, p] = kq, vq
                Ks[b, :, p] = np.stack([ks, kz], -1)
                Vs[b, :, p] = np.stack([vs, vz], -1)
            else:
                page, off = page_slot(table[b], p, page_size)
                Kc[page, :, off], Vc[page, :, off] = kq, vq
                Ks[page, :, off] = np.stack([ks, kz], -1)
                Vs[page, :, off] = np.stack([vs, vz], -1)
        if table is None:
            Kd = dequantize_u8(Kc[b, :, :L], Ks[b, :, :L, 0], Ks[b, :, :L, 1])
            Vd = dequantize_u8(Vc[b, :, :L], Vs[b, :, :L, 0], Vs[b, :, :L, 1])
        else:
            ksz = gather_paged(Ks, table[b], L, page_size)
            vsz = gather_paged(Vs, table[b], L, page_size)
            Kd = dequantize_u8(gather_paged(Kc, table[b], L, page_size), ksz[..., 0], ksz[..., 1])
            Vd = dequantize_u8(gather_paged(Vc, table[b], L, page_size), vsz[..., 0], vsz[..., 1])
        for i in range(n):
            p = L - n + i
            t0 = window_start(p + 1, window)
            out[b, i], lse[b, i] = gqa_attention(q_rot[b, i], Kd[:, t0:p + 1], Vd[:, t0:p + 1], scale)
    return {"out": out, "lse": lse, "q_rot": q_rot, "k_codes": Kc, "k_sz": Ks, "v_codes": Vc, "v_sz": Vs}


def decode_unit(q_group, k_row, v_row, K_unit, V_unit, seq_len: int, rope_base: float, scale: float,
                cache_dtype: str, window: int = 0):
    """The decode step for ONE (sequence, KV head) unit, for sampled checks at
    full size: q_group [G, d] are the query heads of the group, k_row / v_row
    [d] the new token's key / value for this KV head, K_unit / V_unit [>= L, d]
    the unit's cached tokens before the append. Returns (out [G,d], lse [G],
    k_stored [d])."""
    L = int(seq_len)
    p = L - 1
    q_rot = rope_rotate(_f64(q_group), p, rope_base)
    k_stored = round_to(rope_rotate(_f64(k_row), p, rope_base), cache_dtype)
    K = _f64(K_unit)[:L].copy()
    V = _f64(V_unit)[:L].copy()
    K[p] = k_stored
    V[p] = _f64(v_row)
    t0 = window_start(L, window)
    out, lse = gqa_attention(q_rot, K[None, t0:], V[None, t0:], scale)
    return out, lse, k_stored


# ---------------------------------------------- whole short sequence, pins
def run_cached_sequence(q, k, v, prompt_len: int, evals: int, rope_base: float, scale: float,
                        cache_dtype: str):
    """Generate with a KV cache ("KV Cache" explainer, Langkah 2-3).

    q, k, v: raw per-position vectors [n, B, H, d] with n = P + T - 1. Every
    position's key/value is projected (here: taken from the inputs) exactly
    once, rotated by its position, rounded and appended. Attention is
    evaluated for the query at positions P-1 .. P+T-2 (T evaluations; the
    first uses the prompt). Returns (outputs [T, B, H_q, d], lse [T, B, H_q],
    projections, written) where ``projections`` counts K/V slices computed
    and ``written`` marks every cache scalar that was stored.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, B, h_kv, d = k.shape
    h_q = q.shape[2]
    K = np.zeros((B, h_kv, n, d), F64)
    V = np.zeros((B, h_kv, n, d), F64)
    written = np.zeros((2, B, h_kv, n, d), dtype=bool)
    outs, lses = [], []
    projections = 0
    for p in range(prompt_len + evals - 1):
        projections += 1  # only the newest token is projected
        for b in range(B):
            k_stored = round_to(rope_rotate(k[p, b], p, rope_base), cache_dtype)
            append_contiguous(K, V, b, p, k_stored, round_to(v[p, b], cache_dtype))
            written[:, b, :, p, :] = True
        if p >= prompt_len - 1:
            o = np.empty((B, h_q, d), F64)
            ls = np.empty((B, h_q), F64)
            for b in range(B):
                o[b], ls[b] = gqa_attention(rope_rotate(q[p, b], p, rope_base), K[b, :, :p + 1],
                                            V[b, :, :p + 1], scale)
            outs.append(o)
            lses.append(ls)
    return np.stack(outs), np.stack(lses), projections, written


def run_uncached_sequence(q, k, v, prompt_len: int, evals: int, rope_base: float, scale: float):
    """Generate WITHOUT a cache: step s recomputes the keys and values of all
    P + s - 1 positions of its context and runs full causal attention over
    every row ("KV Cache" explainer, Langkah 2). Returns (outputs [T, B, H_q, d]
    -- the last row of each step --, every row of the final step
    [B, H_q, n, d], projections)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B = k.shape[1]
    outs = []
    projections = 0
    last_all_rows = None
    for s in range(1, evals + 1):
        n = prompt_len + s - 1
        projections += n
        rows = []
        for b in range(B):
            Q = np.stack([rope_rotate(q[t, b], t, rope_base) for t in range(n)], axis=1)
            Kb = np.stack([rope_rotate(k[t, b], t, rope_base) for t in range(n)], axis=1)
            Vb = np.stack([v[t, b] for t in range(n)], axis=1)
            rows.append(causal_attention(Q, Kb, Vb, scale))
        all_rows = np.stack(rows)  # [B, H_q, n, d]
        outs.append(all_rows[:, :, n - 1, :])
        last_all_rows = all_rows
    return np.stack(outs), last_all_rows, projections
