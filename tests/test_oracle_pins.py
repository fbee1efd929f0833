"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each check takes the implementation under test as an argument, so the
mutation tests at the bottom can run the same checks on deliberately broken
copies of oracle functions (planted here on the CPU) and show that each
plausible mistake is caught.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle
from oracle import decode as od
from synthetic import make_tiny_sequence, workload

RNG = np.random.default_rng(12345)


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ rounding
def check_round_bf16(fn):
    # fp32-representable values: RNE fp64->bf16 equals torch's fp32->bf16 RNE
    x32 = torch.randn(20000, dtype=torch.float32) * torch.exp(torch.randn(20000) * 8)
    ref = x32.to(torch.bfloat16).to(torch.float64).numpy()
    got = fn(x32.to(torch.float64).numpy())
    assert np.array_equal(got, ref)
    # exact ties go to the even neighbour; one fp64 ulp past a tie goes away from zero
    one_plus_half = 1.0 + 2.0 ** -8  # halfway between 1 and 1 + 2^-7
    assert fn(np.array([one_plus_half]))[0] == 1.0
    three_half = 1.0 + 3 * 2.0 ** -8  # halfway between 1+2^-7 (odd) and 1+2^-6 (even)
    assert fn(np.array([three_half]))[0] == 1.0 + 2.0 ** -6
    assert fn(np.array([np.nextafter(one_plus_half, 2.0)]))[0] == 1.0 + 2.0 ** -7
    assert fn(np.array([-np.nextafter(one_plus_half, 2.0)]))[0] == -(1.0 + 2.0 ** -7)
    # values that fp32 rounding would tie but fp64 does not (no double rounding)
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert fn(np.array([v]))[0] == 1.0 + 2.0 ** -7
    assert fn(np.array([0.0]))[0] == 0.0
    assert np.isinf(fn(np.array([3.5e38]))[0])


def test_round_bf16():
    check_round_bf16(oracle.round_bf16)


def test_round_to_f32_matches_numpy_cast():
    x = RNG.standard_normal(1000)
    assert np.array_equal(oracle.round_to(x, "f32"), x.astype(np.float32).astype(np.float64))
    assert np.array_equal(oracle.round_to(x, "f64"), x)


# ---------------------------------------------------------------------- RoPE
def check_rope(rotate_fn, inv_freq_fn):
    d, base = 64, 10000.0
    theta = inv_freq_fn(d, base)
    assert theta.shape == (d // 2,)
    assert theta[0] == 1.0
    # geometric progression with ratio base^(-2/d), last term base^(-(d-2)/d)
    ratio = theta[1:] / theta[:-1]
    assert np.allclose(ratio, math.exp(-2.0 / d * math.log(base)), rtol=1e-13, atol=0)
    assert math.isclose(theta[-1], math.exp(-(d - 2) / d * math.log(base)), rel_tol=1e-13)
    x = RNG.standard_normal((3, d))
    # position 0 is the identity
    assert np.array_equal(rotate_fn(x, 0, base), x)
    for pos in (1, 7, 4095, 131071):
        y = rotate_fn(x, pos, base)
        # complex form: (x0 + i x1) * exp(i pos theta) for each adjacent pair
        z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * pos * theta)
        assert np.allclose(y[:, 0::2], z.real, rtol=0, atol=1e-12)
        assert np.allclose(y[:, 1::2], z.imag, rtol=0, atol=1e-12)
        # every pair keeps its norm
        assert np.allclose(np.hypot(y[:, 0::2], y[:, 1::2]), np.hypot(x[:, 0::2], x[:, 1::2]), atol=1e-12)
    # scores depend only on the position difference
    q, k = RNG.standard_normal(d), RNG.standard_normal(d)
    for m, n, shift in ((5, 2, 100), (17, 17, 3), (1000, 3, 7)):
        a = rotate_fn(q, m, base) @ rotate_fn(k, n, base)
        b = rotate_fn(q, m + shift, base) @ rotate_fn(k, n + shift, base)
        assert abs(a - b) < 1e-11
    # rotations compose: R(a) R(b) = R(a + b)
    assert np.allclose(rotate_fn(rotate_fn(x, 3, base), 5, base), rotate_fn(x, 8, base), atol=1e-12)
    # direction: position 1 turns (1, 0) of pair 0 to (cos 1, sin 1)
    e = np.zeros(d)
    e[0] = 1.0
    r = rotate_fn(e, 1, base)
    assert math.isclose(r[0], math.cos(1.0), abs_tol=1e-15) and math.isclose(r[1], math.sin(1.0), abs_tol=1e-15)


def test_rope():
    check_rope(oracle.rope_rotate, oracle.rope_inv_freq)


# ----------------------------------------------------------------- attention
def _sdpa(q_rot, K, V, scale):
    """torch scaled_dot_product_attention, fp64 on CPU, GQA enabled (library routine)."""
    q = torch.from_numpy(q_rot)[None, :, None, :]
    k = torch.from_numpy(K)[None]
    v = torch.from_numpy(V)[None]
    return F.scaled_dot_product_attention(q, k, v, scale=scale, enable_gqa=True)[0, :, 0, :].numpy()


def check_gqa(attn_fn):
    for h_q, h_kv, L, d in ((8, 2, 37, 64), (4, 4, 5, 32), (32, 1, 64, 128), (6, 3, 1, 16), (12, 4, 100, 64)):
        q = RNG.standard_normal((h_q, d))
        K = RNG.standard_normal((h_kv, L, d))
        V = RNG.standard_normal((h_kv, L, d))
        scale = 1.0 / math.sqrt(d)
        out, lse = attn_fn(q, K, V, scale)
        assert np.allclose(out, _sdpa(q, K, V, scale), rtol=0, atol=1e-12)
        G = h_q // h_kv
        for h in range(h_q):
            s = K[h // G] @ q[h] * scale
            assert abs(lse[h] - logsumexp(s)) < 1e-12


def test_gqa_matches_library_sdpa():
    check_gqa(oracle.gqa_attention)


def test_gqa_special_cases():
    d = 64
    # L = 1: the single value is the output, exactly
    q = RNG.standard_normal((4, d))
    K = RNG.standard_normal((2, 1, d))
    V = RNG.standard_normal((2, 1, d))
    out, lse = oracle.gqa_attention(q, K, V, 0.125)
    assert np.array_equal(out, np.repeat(V[:, 0], 2, axis=0))
    # q = 0: uniform weights, output is the mean of V
    K = RNG.standard_normal((2, 50, d))
    V = RNG.standard_normal((2, 50, d))
    out, lse = oracle.gqa_attention(np.zeros((4, d)), K, V, 0.125)
    assert np.allclose(out, np.repeat(V.mean(axis=1), 2, axis=0), atol=1e-14)
    assert np.allclose(lse, math.log(50), atol=1e-14)
    # rows of the attention matrix sum to 1
    q = RNG.standard_normal((8, d))
    _, _, w = oracle.gqa_attention(q, K, V, 0.125, return_weights=True)
    assert np.all(w >= 0) and np.max(np.abs(w.sum(axis=1) - 1.0)) <= 1e-12
    # heads sharing a KV head but with different queries give different outputs
    out, _ = oracle.gqa_attention(q, K, V, 0.125)
    assert not np.allclose(out[0], out[1])


def test_gqa_reduces_to_mha_and_mqa():
    d, L = 64, 33
    q = RNG.standard_normal((8, d))
    K = RNG.standard_normal((8, L, d))
    V = RNG.standard_normal((8, L, d))
    assert np.allclose(oracle.gqa_attention(q, K, V, 0.125)[0], oracle.mha_attention(q, K, V, 0.125), atol=1e-13)
    assert np.allclose(oracle.gqa_attention(q, K[:1], V[:1], 0.125)[0], oracle.mqa_attention(q, K[0], V[0], 0.125),
                       atol=1e-13)
    # the MHA / MQA routines themselves against the library
    assert np.allclose(oracle.mha_attention(q, K, V, 0.125), _sdpa(q, K, V, 0.125), atol=1e-12)
    assert np.allclose(oracle.mqa_attention(q, K[0], V[0], 0.125), _sdpa(q, K[:1], V[:1], 0.125), atol=1e-12)


def test_causal_attention_matches_library():
    h_q, h_kv, n, d = 8, 2, 23, 32
    Q = RNG.standard_normal((h_q, n, d))
    K = RNG.standard_normal((h_kv, n, d))
    V = RNG.standard_normal((h_kv, n, d))
    ref = F.scaled_dot_product_attention(torch.from_numpy(Q)[None], torch.from_numpy(K)[None],
                                         torch.from_numpy(V)[None], is_causal=True, scale=0.3,
                                         enable_gqa=True)[0].numpy()
    assert np.allclose(oracle.causal_attention(Q, K, V, 0.3), ref, atol=1e-12)


def check_split_combine(partial_fn, combine_fn):
    h_q, h_kv, L, d = 8, 2, 300, 64
    q = RNG.standard_normal((h_q, d))
    K = RNG.standard_normal((h_kv, L, d))
    V = RNG.standard_normal((h_kv, L, d))
    full, full_lse = oracle.gqa_attention(q, K, V, 0.125)
    for bounds in ([0, 300], [0, 64, 300], [0, 1, 2, 299, 300], [0, 100, 100, 250, 300, 300]):
        parts = [partial_fn(q, K, V, 0.125, a, b) for a, b in zip(bounds[:-1], bounds[1:])]
        out, lse = combine_fn(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        assert np.allclose(out, full, atol=1e-13)
        assert np.allclose(lse, full_lse, atol=1e-13)


def test_split_combine_is_exact():
    check_split_combine(oracle.attention_partial, oracle.lse_combine)


def test_empty_partial():
    o, lse = oracle.attention_partial(np.ones((2, 8)), np.ones((1, 4, 8)), np.ones((1, 4, 8)), 1.0, 3, 3)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


# ------------------------------------------------------------- paged layout
def test_page_slots_match_printed_example(golden_dir):
    ex = _load(golden_dir, "paged_example.json")
    for t, page, off in ex["slots"]:
        assert oracle.page_slot(ex["block_table"], t, ex["page_size"]) == (page, off)
    n_blocks = -(-ex["length"] // ex["page_size"])
    assert n_blocks == len(ex["block_table"])
    assert ex["length"] - (n_blocks - 1) * ex["page_size"] == ex["last_block_filled"]
    assert n_blocks * ex["page_size"] - ex["length"] <= ex["max_waste_tokens"]


def _contiguous_to_paged(K, lens, page_size, rng):
    """Scatter a contiguous cache into a shuffled pool through a block table."""
    B, h_kv, cap, d = K.shape
    npages = [-(-int(L) // page_size) for L in lens]
    total = sum(npages) + 3
    perm = rng.permutation(total)
    table = -np.ones((B, max(npages) + 2), dtype=np.int64)
    pool = rng.standard_normal((total, h_kv, page_size, d))  # junk in unused rows
    off = 0
    for b in range(B):
        for i in range(npages[b]):
            page = perm[off + i]
            table[b, i] = page
            lo, hi = i * page_size, min((i + 1) * page_size, cap)
            pool[page, :, : hi - lo, :] = K[b, :, lo:hi, :]
        off += npages[b]
    return pool, table


def test_paged_equals_contiguous():
    rng = np.random.default_rng(7)
    B, h_q, h_kv, d, ps = 3, 8, 2, 64, 16
    lens = np.array([1, 40, 64])
    cap = 64
    Kc = oracle.round_bf16(rng.standard_normal((B, h_kv, cap, d)))
    Vc = oracle.round_bf16(rng.standard_normal((B, h_kv, cap, d)))
    q = oracle.round_bf16(rng.standard_normal((B, h_q, d)))
    k = oracle.round_bf16(rng.standard_normal((B, h_kv, d)))
    v = oracle.round_bf16(rng.standard_normal((B, h_kv, d)))
    rc = oracle.decode_step_contiguous(Kc, Vc, q, k, v, lens, 10000.0, 0.125, "bf16")
    pk, table = _contiguous_to_paged(Kc, lens, ps, np.random.default_rng(1))
    pv, _ = _contiguous_to_paged(Vc, lens, ps, np.random.default_rng(1))
    rp = oracle.decode_step_paged(pk, pv, table, q, k, v, lens, ps, 10000.0, 0.125, "bf16")
    assert np.array_equal(rp["out"], rc["out"])
    assert np.array_equal(rp["lse"], rc["lse"])
    for b in range(B):
        L = int(lens[b])
        assert np.array_equal(oracle.gather_paged(rp["k_pool"], table[b], L, ps), rc["k_cache"][b, :, :L])
        assert np.array_equal(oracle.gather_paged(rp["v_pool"], table[b], L, ps), rc["v_cache"][b, :, :L])


def test_append_writes_only_the_new_slot():
    rng = np.random.default_rng(3)
    B, h_q, h_kv, d, cap = 2, 4, 2, 32, 10
    Kc = rng.standard_normal((B, h_kv, cap, d))
    Vc = rng.standard_normal((B, h_kv, cap, d))
    q, k, v = rng.standard_normal((B, h_q, d)), rng.standard_normal((B, h_kv, d)), rng.standard_normal((B, h_kv, d))
    lens = np.array([4, 10])
    r = oracle.decode_step_contiguous(Kc, Vc, q, k, v, lens, 10000.0, 0.2, "f64")
    changed = np.argwhere(np.any(r["v_cache"] != Vc, axis=-1))
    assert sorted(map(tuple, changed)) == [(b, h, int(lens[b]) - 1) for b in range(B) for h in range(h_kv)]
    assert np.array_equal(np.any(r["k_cache"] != Kc, axis=-1), np.any(r["v_cache"] != Vc, axis=-1))
    assert np.array_equal(r["v_cache"][0, :, 3], v[0])


def test_decode_unit_equals_full_step():
    rng = np.random.default_rng(11)
    B, h_q, h_kv, d, cap = 2, 8, 2, 64, 70
    Kc = oracle.round_bf16(rng.standard_normal((B, h_kv, cap, d)))
    Vc = oracle.round_bf16(rng.standard_normal((B, h_kv, cap, d)))
    q = oracle.round_bf16(rng.standard_normal((B, h_q, d)))
    k = oracle.round_bf16(rng.standard_normal((B, h_kv, d)))
    v = oracle.round_bf16(rng.standard_normal((B, h_kv, d)))
    lens = np.array([70, 33])
    r = oracle.decode_step_contiguous(Kc, Vc, q, k, v, lens, 10000.0, 0.125, "bf16")
    G = h_q // h_kv
    for b in range(B):
        for j in range(h_kv):
            out, lse, ks = oracle.decode_unit(q[b, j * G:(j + 1) * G], k[b, j], v[b, j], Kc[b, j], Vc[b, j],
                                              lens[b], 10000.0, 0.125, "bf16")
            assert np.array_equal(out, r["out"][b, j * G:(j + 1) * G])
            assert np.array_equal(ks, r["k_cache"][b, j, lens[b] - 1])


# ---------------------------------------------- cached == uncached, counts
@pytest.mark.parametrize("evals", [16, 64])
def test_cached_equals_recomputation_and_projection_counts(golden_dir, evals):
    gold = {c["evals"]: c for c in _load(golden_dir, "projection_counts.json")["cases"]}[evals]
    w = workload("tiny")
    seq = make_tiny_sequence(w, prompt_len=gold["prompt_len"], decode_evals=evals)
    scale = 1.0 / math.sqrt(w.head_dim)
    outs, lses, n_cached, written = oracle.run_cached_sequence(seq.q, seq.k, seq.v, seq.prompt_len, evals,
                                                               w.rope_base, scale, "f64")
    ref, last_rows, n_uncached = oracle.run_uncached_sequence(seq.q, seq.k, seq.v, seq.prompt_len, evals,
                                                              w.rope_base, scale)
    # the pages' printed counts, and the closed form printed beside them
    assert (n_uncached, n_cached) == (gold["no_cache"], gold["with_cache"])
    assert oracle.projection_counts_closed_form(gold["prompt_len"], evals) == (gold["no_cache"], gold["with_cache"])
    if "ratio" in gold:
        assert round(n_uncached / n_cached, 1) == gold["ratio"]
    else:
        assert round(n_uncached / n_cached) == gold["ratio_approx"]
    # cached decode equals brute-force recomputation under the causal mask
    assert np.max(np.abs(outs - ref)) <= 1e-12
    # ... and every earlier cached output equals the matching row of the final causal pass
    n = seq.prompt_len + evals - 1
    for i, p in enumerate(range(seq.prompt_len - 1, n)):
        assert np.max(np.abs(outs[i] - last_rows[:, :, p, :])) <= 1e-12
    # the cache holds 2 * T * H_kv * d scalars per layer (T = stored positions)
    assert int(written.sum()) // w.batch == oracle.layer_cache_scalars(n, w.h_kv, w.head_dim)


def test_decode_step_matches_recomputation():
    """One decode step over a cache built from the first n-1 positions equals
    the last row of full causal recomputation over all n positions."""
    w = workload("tiny")
    seq = make_tiny_sequence(w)
    scale = 1.0 / math.sqrt(w.head_dim)
    n = seq.prompt_len + seq.decode_evals - 1
    q = seq.q.double().numpy()
    k = seq.k.double().numpy()
    v = seq.v.double().numpy()
    K = np.zeros((w.batch, w.h_kv, n, w.head_dim))
    V = np.zeros_like(K)
    for p in range(n - 1):
        K[:, :, p] = np.stack([oracle.rope_rotate(k[p, b], p, w.rope_base) for b in range(w.batch)])
        V[:, :, p] = v[p]
    r = oracle.decode_step_contiguous(K, V, q[n - 1], k[n - 1], v[n - 1], np.full(w.batch, n), w.rope_base, scale,
                                      "f64")
    _, last_rows, _ = oracle.run_uncached_sequence(seq.q, seq.k, seq.v, seq.prompt_len, seq.decode_evals,
                                                   w.rope_base, scale)
    assert np.max(np.abs(r["out"] - last_rows[:, :, n - 1, :])) <= 1e-12


# ------------------------------------------------------------ byte figures
UNITS = {"GB": 1e9, "TB": 1e12, "MiB": 2.0 ** 20, "GiB": 2.0 ** 30, "KiB": 2.0 ** 10}


def test_kv_bytes_match_printed_figures(golden_dir):
    g = _load(golden_dir, "kv_bytes.json")
    for c in g["per_token"]:
        got = oracle.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], c["bytes"])
        if "exact" in c:
            assert got == c["exact"], c["source"]
        else:
            assert round(got / UNITS[c["unit"]], c["decimals"]) == c["rounded"], c["source"]
    for c in g["totals"]:
        got = oracle.kv_cache_bytes(c["layers"], c["kv_heads"], c["head_dim"], c["bytes"], c["seq_len"], c["batch"])
        assert round(got / UNITS[c["unit"]], c["decimals"]) == c["rounded"], c["source"]
    for c in g["bounds"]:
        got = oracle.kv_cache_bytes(c["layers"], c["kv_heads"], c["head_dim"], c["bytes"], c["seq_len"], c["batch"])
        if "greater_than" in c:
            assert got > c["greater_than"], c["source"]
        else:
            assert abs(got / c["about"] - 1) <= c["rel_tol"], c["source"]


def test_layer_scalars_grow_with_kv_heads():
    # halving H_kv halves the stored scalars at fixed T and d
    assert oracle.layer_cache_scalars(100, 8, 128) == 2 * oracle.layer_cache_scalars(100, 4, 128)
    assert oracle.layer_cache_scalars(100, 8, 128) * 2 == oracle.kv_bytes_per_token(1, 8, 128, 2) * 100


# -------------------------------------------- planted mistakes are caught
def _fails(check, *impls):
    try:
        check(*impls)
    except AssertionError:
        return True
    return False


def test_planted_mistakes_are_caught():
    def rope_sign_flipped(x, pos, base):
        return od.rope_rotate(x, -pos, base)

    def rope_half_split(x, pos, base):
        x = np.asarray(x, dtype=np.float64)
        d = x.shape[-1]
        ang = pos * od.rope_inv_freq(d, base)
        c, s = np.cos(ang), np.sin(ang)
        a, b = x[..., : d // 2], x[..., d // 2:]
        return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)

    def inv_freq_wrong_exponent(d, base):
        return np.power(base, -np.arange(d // 2) / d)

    assert _fails(check_rope, rope_sign_flipped, od.rope_inv_freq)
    assert _fails(check_rope, rope_half_split, od.rope_inv_freq)
    assert _fails(check_rope, od.rope_rotate, inv_freq_wrong_exponent)

    def gqa_modulo_group(q, K, V, scale):
        h_q, h_kv = q.shape[0], K.shape[0]
        out = np.empty_like(q)
        lse = np.empty(h_q)
        for h in range(h_q):
            o, l = od.gqa_attention(q[h:h + 1], K[h % h_kv][None], V[h % h_kv][None], scale)
            out[h], lse[h] = o[0], l[0]
        return out, lse

    def gqa_no_scale(q, K, V, scale):
        return od.gqa_attention(q, K, V, 1.0)

    def gqa_k_for_v(q, K, V, scale):
        return od.gqa_attention(q, K, K, scale)

    assert _fails(check_gqa, gqa_modulo_group)
    assert _fails(check_gqa, gqa_no_scale)
    assert _fails(check_gqa, gqa_k_for_v)

    def combine_unweighted(o, lse):
        return o.mean(axis=0), lse.max(axis=0)

    def partial_off_by_one(q, K, V, scale, t0, t1):
        return od.attention_partial(q, K, V, scale, t0, max(t0, t1 - 1)) if t1 - t0 > 1 else \
            od.attention_partial(q, K, V, scale, t0, t1)

    assert _fails(check_split_combine, od.attention_partial, combine_unweighted)
    assert _fails(check_split_combine, partial_off_by_one, od.lse_combine)

    def round_truncating(x):
        x = np.asarray(x, np.float64)
        _, e = np.frexp(x)
        q = np.maximum(e.astype(np.int64) - 8, -133)
        return np.ldexp(np.trunc(np.ldexp(x, -q)), q)

    def round_half_up(x):
        x = np.asarray(x, np.float64)
        _, e = np.frexp(x)
        q = np.maximum(e.astype(np.int64) - 8, -133)
        return np.ldexp(np.floor(np.ldexp(x, -q) + 0.5), q)

    assert _fails(check_round_bf16, round_truncating)
    assert _fails(check_round_bf16, round_half_up)


# ------------------------------------------------------- sliding window
def test_sliding_window_decode_pins():
    """Sliding-window decode (youngju.dev SlidingWindowAttention: the cache keeps
    its last window_size tokens): window 1 attends to the new token alone, a
    window >= L is full attention, and every step of a sequence equals the last
    row of causal attention under a band mask (keys j with i - W < j <= i),
    computed by the library routine SDPA with an explicit boolean mask."""
    rng = np.random.default_rng(21)
    B, h_q, h_kv, d, cap = 2, 8, 2, 32, 50
    K = rng.standard_normal((B, h_kv, cap, d))
    V = rng.standard_normal((B, h_kv, cap, d))
    q, k, v = rng.standard_normal((B, h_q, d)), rng.standard_normal((B, h_kv, d)), rng.standard_normal((B, h_kv, d))
    lens = np.array([50, 7])
    one = oracle.decode_step_contiguous(K, V, q, k, v, lens, 10000.0, 0.2, "f64", window=1)
    assert np.array_equal(one["out"], np.repeat(v, h_q // h_kv, axis=1))
    full = oracle.decode_step_contiguous(K, V, q, k, v, lens, 10000.0, 0.2, "f64")
    wide = oracle.decode_step_contiguous(K, V, q, k, v, lens, 10000.0, 0.2, "f64", window=64)
    assert np.array_equal(full["out"], wide["out"])
    assert oracle.window_start(10, 0) == 0 and oracle.window_start(10, 4) == 6 and oracle.window_start(3, 4) == 0

    # band-masked causal attention over a whole sequence, every row
    n, W = 23, 5
    Qs = rng.standard_normal((h_q, n, d))
    Ks = rng.standard_normal((h_kv, n, d))
    Vs = rng.standard_normal((h_kv, n, d))
    i = np.arange(n)[:, None]
    jj = np.arange(n)[None, :]
    band = torch.from_numpy((jj <= i) & (jj > i - W))
    ref = F.scaled_dot_product_attention(torch.from_numpy(Qs)[None], torch.from_numpy(Ks)[None],
                                         torch.from_numpy(Vs)[None], attn_mask=band, scale=0.3,
                                         enable_gqa=True)[0].numpy()
    for row in range(n):
        t0 = oracle.window_start(row + 1, W)
        o, _ = oracle.gqa_attention(Qs[:, row], Ks[:, t0:row + 1], Vs[:, t0:row + 1], 0.3)
        assert np.allclose(o, ref[:, row], atol=1e-12)

    # paged with a window equals contiguous with the same window
    Kc = oracle.round_bf16(rng.standard_normal((B, h_kv, 64, d)))
    Vc = oracle.round_bf16(rng.standard_normal((B, h_kv, 64, d)))
    lens = np.array([64, 40])
    rc = oracle.decode_step_contiguous(Kc, Vc, q, k, v, lens, 10000.0, 0.2, "bf16", window=19)
    pk, table = _contiguous_to_paged(Kc, lens, 16, np.random.default_rng(5))
    pv, _ = _contiguous_to_paged(Vc, lens, 16, np.random.default_rng(5))
    rp = oracle.decode_step_paged(pk, pv, table, q, k, v, lens, 16, 10000.0, 0.2, "bf16", window=19)
    assert np.array_equal(rp["out"], rc["out"])


# ---------------------------------------------------------- uint8 cache
def listing_quantize_torch(x):
    """QuantizedKVCache.quantize ("KV Cache 최적화 심층 분석", youngju.dev) run as the
    listing states it, in torch float32: the row's min and max over the last
    axis, scale = (max - min) / 255, zero point = round(-min / scale) clamped to
    [0, 255], code = round(x / scale + zero point) clamped and cast to uint8;
    torch.round rounds half to even. The one reading added is the constant
    row, whose scale the listing leaves at 0 (a division by zero): scale 1.
    This route shares nothing with the oracle's numpy code."""
    t = torch.as_tensor(np.asarray(x, np.float32))
    lo = t.min(dim=-1, keepdim=True)[0]
    hi = t.max(dim=-1, keepdim=True)[0]
    step = (hi - lo) / 255.0
    step = torch.where(step == 0, torch.ones_like(step), step)
    zero = (-lo / step).round().clamp(0, 255)
    codes = ((t / step) + zero).round().clamp(0, 255).to(torch.uint8)
    return codes.numpy(), step[..., 0].numpy(), zero[..., 0].numpy()


def _u8_rows(rng):
    """Rows that separate the plausible readings of the listing: N(0,1) rows of
    mixed scales; rows with a positive minimum (zero point clamped to 0) and a
    negative maximum (clamped to 255); rows whose -min / scale is far from an
    integer (the order of the offset matters); and tie rows, where
    x / scale + zero point lands exactly on c + 1/2."""
    rows = [rng.standard_normal((40, 128)).astype(np.float32) * rng.uniform(0.05, 20, (40, 1)).astype(np.float32)]
    rows.append(rng.uniform(1.0, 3.0, (8, 128)).astype(np.float32))
    rows.append(rng.uniform(-5.0, -0.5, (8, 128)).astype(np.float32))
    # min = -100.4 s, max = 154.6 s: scale ~s, -min / scale ~100.4 -> zero point 100; values
    # (c - 99.7) s: x / scale + 100 ~ c + 0.3 (code c), (x - min) / scale ~ c + 0.7 (code c + 1)
    s = np.float32(2.0 ** -6)
    off = np.tile(np.arange(255, dtype=np.float32) - np.float32(99.7), (4, 1))
    off[:, 0], off[:, 1] = np.float32(-100.4), np.float32(154.6)
    rows.append(off * s)
    return rows


def check_u8_quantise(fn):
    rng = np.random.default_rng(31)
    for x in _u8_rows(rng):
        codes, scale, zp = fn(x)
        rc, rs, rz = listing_quantize_torch(x)
        assert codes.dtype == np.uint8 and scale.dtype == np.float32
        assert np.array_equal(scale, rs) and np.array_equal(zp, rz) and np.array_equal(codes, rc)
        back = (codes.astype(np.float64) - zp.astype(np.float64)[:, None]) * scale.astype(np.float64)[:, None]
        inside = (x >= -zp[:, None] * scale[:, None]) & (x <= (255 - zp[:, None]) * scale[:, None])
        assert np.all(np.abs(back - x)[inside] <= (scale[:, None] * (0.5 + 1e-5) + 1e-7)[np.nonzero(inside)[0], 0])
    # ties: scale 2^-5 exactly (min -100 s, max 155 s), x = (c - 100 + 1/2) s gives
    # x / scale + zp = c + 1/2 exactly: half to even picks c for even c, c + 1 for odd
    s = np.float32(2.0 ** -5)
    c = np.arange(0, 255)
    row = np.concatenate([[-100.0, 155.0], c - 100 + 0.5]).astype(np.float32) * s
    codes, scale, zp = fn(row[None])
    assert scale[0] == s and zp[0] == 100
    assert np.array_equal(codes[0, 2:].astype(np.int64), c + (c % 2))
    assert codes[0, 0] == 0 and codes[0, 1] == 255
    # the zero point itself on a tie: -min / scale = 100.5 -> 100, 101.5 -> 102
    for lo, want in ((-100.5, 100), (-101.5, 102)):
        r = np.array([[lo, lo + 255.0]], np.float32) * s
        _, sc, z = fn(r)
        assert sc[0] == s and z[0] == want
    # clamped zero points: a positive minimum gives 0, a negative maximum 255
    _, _, z = fn(np.array([[1.0, 2.0, 3.0], [-3.0, -2.0, -1.0]], np.float32))
    assert z[0] == 0 and z[1] == 255
    # a constant row takes scale 1 and dequantises to 0 (its value is lost, as the listing's formula would lose it)
    c3, s3, z3 = fn(np.full((1, 8), 0.5, np.float32))
    assert s3[0] == 1.0 and np.all(c3.astype(np.float64) - z3[0] == 0.0)


def test_u8_quantisation_pins():
    """QuantizedKVCache (youngju.dev): the oracle's quantiser equals the listing
    run in torch float32 (codes, scales and zero points identical) on rows that
    separate the readings, rounds exact ties to even, clamps the zero point,
    and round-trips within half a step. Values already on the grid come back
    exactly; the row min and max land on codes 0 and 255."""
    check_u8_quantise(oracle.quantize_u8)
    rng = np.random.default_rng(33)
    s = np.float32(0.03125)
    grid = ((rng.integers(0, 256, (4, 64)) - 100) * s).astype(np.float32)
    grid[:, 0] = -100 * s
    grid[:, 1] = 155 * s
    c2, s2, z2 = oracle.quantize_u8(grid)
    assert np.all(s2 == s) and np.all(z2 == 100)
    assert np.array_equal(oracle.dequantize_u8(c2, s2, z2), grid.astype(np.float64))
    assert np.all(c2[:, 0] == 0) and np.all(c2[:, 1] == 255)


def test_u8_planted_mistakes_are_caught():
    """Plausible misreadings of the quantiser each fail a pin: rounding half up,
    offsetting before the division ((x - min) / scale, no rounded zero point),
    and an unclamped zero point."""
    def quantise(x, rnd=np.rint, offset_first=False, clamp_zp=True):
        x = np.asarray(x, np.float32)
        mn, mx = x.min(axis=-1), x.max(axis=-1)
        scale = ((mx - mn) / np.float32(255.0)).astype(np.float32)
        scale = np.where(scale == 0, np.float32(1.0), scale).astype(np.float32)
        zp = rnd((-mn) / scale)
        zp = (np.clip(zp, 0, 255) if clamp_zp else zp).astype(np.float32)
        if offset_first:
            v = (x - mn[..., None]) / scale[..., None]
        else:
            v = x / scale[..., None] + zp[..., None]
        return np.clip(rnd(v), 0, 255).astype(np.uint8), scale, zp

    def half_up(v):
        return np.floor(np.asarray(v) + np.float32(0.5))

    assert not _fails(check_u8_quantise, quantise)  # the restatement itself passes
    assert _fails(check_u8_quantise, lambda x: quantise(x, rnd=half_up))
    assert _fails(check_u8_quantise, lambda x: quantise(x, offset_first=True))
    assert _fails(check_u8_quantise, lambda x: quantise(x, clamp_zp=False))


def test_u8_step_matches_listing_and_library():
    """The uint8 decode step against a route that shares nothing with the oracle:
    RoPE in complex form (torch), the new key rounded to float32 and quantised
    by the listing in torch float32, the value likewise, the cache dequantised
    as the listing's dequantize does ((code - zero point) * scale, here in
    float64), and torch's fp64 scaled_dot_product_attention over it."""
    rng = np.random.default_rng(34)
    B, h_q, h_kv, d, cap, base, sc = 2, 8, 2, 64, 40, 10000.0, 0.125
    kc = rng.integers(0, 256, (B, h_kv, cap, d)).astype(np.uint8)
    vc = rng.integers(0, 256, (B, h_kv, cap, d)).astype(np.uint8)
    ks = np.stack([rng.uniform(0.01, 0.03, (B, h_kv, cap)), rng.integers(100, 156, (B, h_kv, cap))], -1)
    vs = np.stack([rng.uniform(0.01, 0.03, (B, h_kv, cap)), rng.integers(100, 156, (B, h_kv, cap))], -1)
    ks, vs = ks.astype(np.float32), vs.astype(np.float32)
    q = oracle.round_bf16(rng.standard_normal((B, h_q, d)))
    k = oracle.round_bf16(rng.standard_normal((B, h_kv, d)))
    v = oracle.round_bf16(rng.standard_normal((B, h_kv, d)))
    lens = np.array([40, 13])
    r = oracle.decode_step_u8(kc, ks, vc, vs, q, k, v, lens, base, sc)
    theta = torch.pow(torch.tensor(base, dtype=torch.float64), -torch.arange(0, d, 2, dtype=torch.float64) / d)

    def turn(x, pos):
        z = torch.view_as_complex(torch.from_numpy(np.ascontiguousarray(x)).reshape(*x.shape[:-1], d // 2, 2))
        return torch.view_as_real(z * torch.polar(torch.ones_like(theta), pos * theta)).reshape(x.shape).numpy()

    for b in range(B):
        L = int(lens[b])
        kq, kss, kz = listing_quantize_torch(turn(k[b], L - 1).astype(np.float32))
        vq, vss, vz = listing_quantize_torch(v[b].astype(np.float32))
        assert np.array_equal(r["k_codes"][b, :, L - 1], kq) and np.array_equal(r["v_codes"][b, :, L - 1], vq)
        assert np.array_equal(r["k_sz"][b, :, L - 1], np.stack([kss, kz], -1))
        assert np.array_equal(r["v_sz"][b, :, L - 1], np.stack([vss, vz], -1))
        Kc, Vc = kc[b, :, :L].copy(), vc[b, :, :L].copy()
        Ks, Vs = ks[b, :, :L].copy(), vs[b, :, :L].copy()
        Kc[:, L - 1], Vc[:, L - 1] = kq, vq
        Ks[:, L - 1], Vs[:, L - 1] = np.stack([kss, kz], -1), np.stack([vss, vz], -1)
        Kd = (torch.from_numpy(Kc).double() - torch.from_numpy(Ks[..., 1:]).double()) * torch.from_numpy(Ks[..., :1]).double()
        Vd = (torch.from_numpy(Vc).double() - torch.from_numpy(Vs[..., 1:]).double()) * torch.from_numpy(Vs[..., :1]).double()
        qr = torch.from_numpy(turn(q[b], L - 1))
        ref = F.scaled_dot_product_attention(qr[None, :, None], Kd[None], Vd[None], scale=sc,
                                             enable_gqa=True)[0, :, 0].numpy()
        assert np.allclose(r["out"][b], ref, rtol=0, atol=1e-12)


def test_u8_decode_step_pins():
    """The uint8 step equals the bf16-free definition: attention over the
    dequantised cache, with the new token quantised by quantize_u8; paged
    equals contiguous on the same logical data."""
    rng = np.random.default_rng(32)
    B, h_q, h_kv, d, cap = 2, 8, 2, 64, 48
    kc = rng.integers(0, 256, (B, h_kv, cap, d)).astype(np.uint8)
    vc = rng.integers(0, 256, (B, h_kv, cap, d)).astype(np.uint8)
    ks = np.stack([rng.uniform(0.01, 0.03, (B, h_kv, cap)), rng.integers(100, 156, (B, h_kv, cap))], -1)
    vs = np.stack([rng.uniform(0.01, 0.03, (B, h_kv, cap)), rng.integers(100, 156, (B, h_kv, cap))], -1)
    ks, vs = ks.astype(np.float32), vs.astype(np.float32)
    q = oracle.round_bf16(rng.standard_normal((B, h_q, d)))
    k = oracle.round_bf16(rng.standard_normal((B, h_kv, d)))
    v = oracle.round_bf16(rng.standard_normal((B, h_kv, d)))
    lens = np.array([48, 20])
    r = oracle.decode_step_u8(kc, ks, vc, vs, q, k, v, lens, 10000.0, 0.125)
    for b in range(B):
        L = int(lens[b])
        Kd = oracle.dequantize_u8(r["k_codes"][b, :, :L], r["k_sz"][b, :, :L, 0], r["k_sz"][b, :, :L, 1])
        Vd = oracle.dequantize_u8(r["v_codes"][b, :, :L], r["v_sz"][b, :, :L, 0], r["v_sz"][b, :, :L, 1])
        out, _ = oracle.gqa_attention(oracle.rope_rotate(q[b], L - 1, 10000.0), Kd, Vd, 0.125)
        assert np.array_equal(out, r["out"][b])
        kq, kss, kz = oracle.quantize_u8(oracle.rope_rotate(k[b], L - 1, 10000.0))
        assert np.array_equal(r["k_codes"][b, :, L - 1], kq)
        # only the new slot changed
        assert np.array_equal(np.delete(r["k_codes"][b], L - 1, axis=1), np.delete(kc[b], L - 1, axis=1))
    # paged == contiguous
    pk, table = _contiguous_to_paged(kc, lens, 16, np.random.default_rng(2))
    pv, _ = _contiguous_to_paged(vc, lens, 16, np.random.default_rng(2))
    pks, _ = _contiguous_to_paged(ks, lens, 16, np.random.default_rng(2))
    pvs, _ = _contiguous_to_paged(vs, lens, 16, np.random.default_rng(2))
    rp = oracle.decode_step_u8(pk.astype(np.uint8), pks, pv.astype(np.uint8), pvs, q, k, v, lens, 10000.0, 0.125,
                               block_table=table, page_size=16)
    assert np.array_equal(rp["out"], r["out"])


# ------------------------------------------------------ fp8 e5m2 cache
def test_e5m2_format_pins():
    """e5m2 is the high byte of an IEEE half: every code decodes to the
    float16 whose bit pattern is code << 8 (numpy's float16, an independent
    route); every finite code encodes back to itself; hand-worked roundings
    (ties to even, subnormals, saturation, signed zero)."""
    c = np.arange(256, dtype=np.uint8)
    v = oracle.dequantize_e5m2(c)
    half = (c.astype(np.uint16) << 8).view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(v), np.isnan(half))
    assert np.array_equal(v[~np.isnan(v)], half[~np.isnan(half)])
    fin = np.isfinite(v)
    assert np.array_equal(oracle.quantize_e5m2(v[fin]), c[fin])
    cases = [
        (1.0, 0x3C), (1.25, 0x3D), (1.2, 0x3D), (1.125, 0x3C),  # 1.125: tie between 1.0 (even) and 1.25
        (1.375, 0x3E),                                          # tie between 1.25 and 1.5 (even)
        (-0.5, 0xB8), (57344.0, 0x7B), (61440.0, 0x7B), (1e9, 0x7B), (-1e9, 0xFB),  # saturation
        (2.0 ** -14, 0x04), (2.0 ** -16, 0x01), (2.0 ** -17, 0x00), (3 * 2.0 ** -17, 0x02),  # subnormals, ties
        (0.0, 0x00), (-0.0, 0x80),
    ]
    got = oracle.quantize_e5m2(np.array([x for x, _ in cases]))
    assert [int(x) for x in got] == [c for _, c in cases]
    # the rounding error stays within half a quantum (2 mantissa bits)
    rng = np.random.default_rng(41)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-8, 8, 20000))
    x = x[np.abs(x) < 57344]
    back = oracle.dequantize_e5m2(oracle.quantize_e5m2(x))
    quantum = np.ldexp(1.0, np.maximum(np.floor(np.log2(np.abs(x))).astype(int) - 2, -16))
    assert np.all(np.abs(back - x) <= quantum / 2)


def test_e5m2_decode_step_pins():
    """The e5m2 step is attention over the decoded cache, with the new token
    rotated in fp64 and rounded once to e5m2; only the new slot changes;
    paged equals contiguous on the same logical data."""
    rng = np.random.default_rng(42)
    B, h_q, h_kv, d, cap = 2, 8, 2, 64, 48
    kc = oracle.quantize_e5m2(rng.standard_normal((B, h_kv, cap, d)))
    vc = oracle.quantize_e5m2(rng.standard_normal((B, h_kv, cap, d)))
    q = oracle.round_bf16(rng.standard_normal((B, h_q, d)))
    k = oracle.round_bf16(rng.standard_normal((B, h_kv, d)))
    v = oracle.round_bf16(rng.standard_normal((B, h_kv, d)))
    lens = np.array([48, 20])
    r = oracle.decode_step_e5m2(kc, vc, q, k, v, lens, 10000.0, 0.125)
    for b in range(B):
        L = int(lens[b])
        Kd = oracle.dequantize_e5m2(r["k_codes"][b, :, :L])
        Vd = oracle.dequantize_e5m2(r["v_codes"][b, :, :L])
        out, _ = oracle.gqa_attention(oracle.rope_rotate(q[b], L - 1, 10000.0), Kd, Vd, 0.125)
        assert np.array_equal(out, r["out"][b])
        assert np.array_equal(r["k_codes"][b, :, L - 1], oracle.quantize_e5m2(oracle.rope_rotate(k[b], L - 1, 10000.0)))
        assert np.array_equal(r["v_codes"][b, :, L - 1], oracle.quantize_e5m2(v[b]))
        assert np.array_equal(np.delete(r["k_codes"][b], L - 1, axis=1), np.delete(kc[b], L - 1, axis=1))
        assert np.array_equal(np.delete(r["v_codes"][b], L - 1, axis=1), np.delete(vc[b], L - 1, axis=1))
    pk, table = _contiguous_to_paged(kc, lens, 16, np.random.default_rng(2))
    pv, _ = _contiguous_to_paged(vc, lens, 16, np.random.default_rng(2))
    rp = oracle.decode_step_e5m2(pk.astype(np.uint8), pv.astype(np.uint8), q, k, v, lens, 10000.0, 0.125,
                                 block_table=table, page_size=16)
    assert np.array_equal(rp["out"], r["out"])


# ------------------------------------------- multi-token (verify) decode
def _multi_variant(K, V, q, k, v, lens, base, scale, dtype, rot_of, end_of):
    """A restatement of the multi-token step with the RoPE position of new
    token i and the end of its key range as parameters, to plant mistakes in.
    New token i is stored at slot L - n + i."""
    K, V = np.array(K, np.float64), np.array(V, np.float64)
    B, n, h_q, d = q.shape
    out = np.empty((B, n, h_q, d))
    lse = np.empty((B, n, h_q))
    qr = np.empty((B, n, h_q, d))
    for b in range(B):
        L = int(lens[b])
        for i in range(n):
            r = rot_of(L, n, i)
            qr[b, i] = oracle.rope_rotate(q[b, i], r, base)
            K[b, :, L - n + i] = oracle.round_to(oracle.rope_rotate(k[b, i], r, base), dtype)
            V[b, :, L - n + i] = v[b, i]
        for i in range(n):
            e = end_of(L, n, i)
            out[b, i], lse[b, i] = oracle.gqa_attention(qr[b, i], K[b, :, :e], V[b, :, :e], scale)
    return {"out": out, "lse": lse, "q_rot": qr, "k_cache": K, "v_cache": V}


def check_multi_step(fn):
    """n new tokens in one pass equal n single-token steps taken in order (the
    verification of drafted tokens is lossless, tveniu.com section 7), for the
    outputs, the log-sum-exps, q_rot and the updated caches, with and without a
    sliding window."""
    rng = np.random.default_rng(41)
    B, h_q, h_kv, d, cap, n = 2, 8, 2, 32, 40, 5
    K0 = oracle.round_bf16(rng.standard_normal((B, h_kv, cap, d)))
    V0 = oracle.round_bf16(rng.standard_normal((B, h_kv, cap, d)))
    q = oracle.round_bf16(rng.standard_normal((B, n, h_q, d)))
    k = oracle.round_bf16(rng.standard_normal((B, n, h_kv, d)))
    v = oracle.round_bf16(rng.standard_normal((B, n, h_kv, d)))
    lens = np.array([40, 7])
    for window in (0, 3):
        r = fn(K0, V0, q, k, v, lens, 10000.0, 0.17, "bf16", window=window)
        K, V = K0.copy(), V0.copy()
        for i in range(n):
            s = oracle.decode_step_contiguous(K, V, q[:, i], k[:, i], v[:, i], lens - n + i + 1, 10000.0, 0.17,
                                              "bf16", window=window)
            K, V = s["k_cache"], s["v_cache"]
            assert np.max(np.abs(s["out"] - r["out"][:, i])) <= 1e-12
            assert np.max(np.abs(s["lse"] - r["lse"][:, i])) <= 1e-12
            assert np.array_equal(s["q_rot"], r["q_rot"][:, i])
        assert np.array_equal(K, r["k_cache"]) and np.array_equal(V, r["v_cache"])


def check_multi_e5m2(fn):
    """n new tokens over an e5m2 cache in one pass equal n single-token e5m2
    steps in order (each sees the codes the earlier ones stored), with and
    without a window; the stored codes are identical; a paged pool holding the
    same logical cache gives the same result."""
    rng = np.random.default_rng(61)
    B, h_q, h_kv, d, cap, n = 2, 8, 2, 32, 40, 4
    Kc = oracle.quantize_e5m2(rng.standard_normal((B, h_kv, cap, d)))
    Vc = oracle.quantize_e5m2(rng.standard_normal((B, h_kv, cap, d)))
    q = oracle.round_bf16(rng.standard_normal((B, n, h_q, d)))
    k = oracle.round_bf16(rng.standard_normal((B, n, h_kv, d)))
    v = oracle.round_bf16(rng.standard_normal((B, n, h_kv, d)))
    lens = np.array([40, 9])
    for window in (0, 5):
        r = fn(Kc, Vc, q, k, v, lens, 10000.0, 0.2, window=window)
        kc, vc = Kc.copy(), Vc.copy()
        for i in range(n):
            one = oracle.decode_step_e5m2(kc, vc, q[:, i], k[:, i], v[:, i], lens - n + i + 1, 10000.0, 0.2,
                                          window=window)
            kc, vc = one["k_codes"], one["v_codes"]
            assert np.allclose(r["out"][:, i], one["out"], rtol=0, atol=1e-12)
            assert np.allclose(r["lse"][:, i], one["lse"], rtol=0, atol=1e-12)
        assert np.array_equal(r["k_codes"], kc) and np.array_equal(r["v_codes"], vc)
    # paged: the same logical cache dealt into permuted 8-token pages
    ps = 8
    npg = cap // ps
    perm = rng.permutation(B * npg)
    table = perm.reshape(B, npg)
    Kp = np.zeros((B * npg, h_kv, ps, d), np.uint8)
    Vp = np.zeros_like(Kp)
    for b in range(B):
        for lp in range(npg):
            Kp[table[b, lp]] = Kc[b, :, lp * ps:(lp + 1) * ps]
            Vp[table[b, lp]] = Vc[b, :, lp * ps:(lp + 1) * ps]
    r = fn(Kc, Vc, q, k, v, lens, 10000.0, 0.2)
    rp = fn(Kp, Vp, q, k, v, lens, 10000.0, 0.2, block_table=table, page_size=ps)
    assert np.allclose(rp["out"], r["out"], rtol=0, atol=1e-12)
    for b in range(B):
        for lp in range(npg):
            assert np.array_equal(rp["k_codes"][table[b, lp]], r["k_codes"][b, :, lp * ps:(lp + 1) * ps])


def check_multi_u8(fn):
    """n new tokens over a uint8 cache in one pass equal n single-token uint8
    steps in order (each sees the codes, scales and zero points the earlier
    ones stored), with and without a window; a paged pool holding the same
    logical cache gives the same result."""
    rng = np.random.default_rng(67)
    B, h_q, h_kv, d, cap, n = 2, 8, 2, 32, 40, 4
    Kc, Ks, Kz = oracle.quantize_u8(rng.standard_normal((B, h_kv, cap, d)))
    Vc, Vs, Vz = oracle.quantize_u8(rng.standard_normal((B, h_kv, cap, d)))
    Ksz = np.stack([Ks, Kz], -1).astype(np.float32)
    Vsz = np.stack([Vs, Vz], -1).astype(np.float32)
    q = oracle.round_bf16(rng.standard_normal((B, n, h_q, d)))
    k = oracle.round_bf16(rng.standard_normal((B, n, h_kv, d)))
    v = oracle.round_bf16(rng.standard_normal((B, n, h_kv, d)))
    lens = np.array([40, 9])
    for window in (0, 5):
        r = fn(Kc, Ksz, Vc, Vsz, q, k, v, lens, 10000.0, 0.2, window=window)
        kc, ksz, vc, vsz = Kc.copy(), Ksz.copy(), Vc.copy(), Vsz.copy()
        for i in range(n):
            one = oracle.decode_step_u8(kc, ksz, vc, vsz, q[:, i], k[:, i], v[:, i], lens - n + i + 1, 10000.0, 0.2,
                                        window=window)
            kc, ksz, vc, vsz = one["k_codes"], one["k_sz"], one["v_codes"], one["v_sz"]
            assert np.allclose(r["out"][:, i], one["out"], rtol=0, atol=1e-12)
            assert np.allclose(r["lse"][:, i], one["lse"], rtol=0, atol=1e-12)
        for key, ref in (("k_codes", kc), ("k_sz", ksz), ("v_codes", vc), ("v_sz", vsz)):
            assert np.array_equal(r[key], ref), key
    ps = 8
    npg = cap // ps
    table = rng.permutation(B * npg).reshape(B, npg)
    pools = []
    for a in (Kc, Ksz, Vc, Vsz):
        pool = np.zeros((B * npg, h_kv, ps) + a.shape[3:], a.dtype)
        for b in range(B):
            for lp in range(npg):
                pool[table[b, lp]] = a[b, :, lp * ps:(lp + 1) * ps]
        pools.append(pool)
    r = fn(Kc, Ksz, Vc, Vsz, q, k, v, lens, 10000.0, 0.2)
    rp = fn(*pools, q, k, v, lens, 10000.0, 0.2, block_table=table, page_size=ps)
    assert np.allclose(rp["out"], r["out"], rtol=0, atol=1e-12)
    for b in range(B):
        for lp in range(npg):
            assert np.array_equal(rp["k_codes"][table[b, lp]], r["k_codes"][b, :, lp * ps:(lp + 1) * ps])
            assert np.array_equal(rp["v_sz"][table[b, lp]], r["v_sz"][b, :, lp * ps:(lp + 1) * ps])


def test_multi_token_u8_pins():
    check_multi_u8(oracle.decode_step_multi_u8)


def test_multi_token_u8_planted_mistake_is_caught():
    """Quantising the key before it is rotated (rotating the dequantised
    codes) fails the pin."""
    def quantise_first(k_codes, k_sz, v_codes, v_sz, q_new, k_new, v_new, seq_lens, rope_base, scale,
                       block_table=None, page_size=0, window=0):
        kc, ks, kz = oracle.quantize_u8(np.asarray(k_new, np.float64))
        k_pre = oracle.dequantize_u8(kc, ks, kz)
        return oracle.decode_step_multi_u8(k_codes, k_sz, v_codes, v_sz, q_new, k_pre, v_new, seq_lens, rope_base,
                                           scale, block_table=block_table, page_size=page_size, window=window)
    with pytest.raises(AssertionError):
        check_multi_u8(quantise_first)


def test_multi_token_e5m2_pins():
    check_multi_e5m2(oracle.decode_step_multi_e5m2)


def test_multi_token_e5m2_planted_mistake_is_caught():
    """Without the causal mask among the new tokens (every query sees all n
    new rows) the pin fails."""
    def no_causal(k_codes, v_codes, q_new, k_new, v_new, seq_lens, rope_base, scale, window=0):
        r = oracle.decode_step_multi_e5m2(k_codes, v_codes, q_new, k_new, v_new, seq_lens, rope_base, scale,
                                          window=window)
        n = q_new.shape[1]
        for b, L in enumerate(np.asarray(seq_lens)):
            Kd = oracle.dequantize_e5m2(r["k_codes"][b, :, :L])
            Vd = oracle.dequantize_e5m2(r["v_codes"][b, :, :L])
            for i in range(n):
                t0 = oracle.window_start(L, window)
                r["out"][b, i], r["lse"][b, i] = oracle.gqa_attention(r["q_rot"][b, i], Kd[:, t0:], Vd[:, t0:], scale)
        return r

    assert _fails(check_multi_e5m2, no_causal)


def test_multi_token_decode_pins(golden_dir):
    check_multi_step(oracle.decode_step_multi)
    # n = 1 is the single-token step
    rng = np.random.default_rng(43)
    K0 = oracle.round_bf16(rng.standard_normal((2, 2, 30, 16)))
    V0 = oracle.round_bf16(rng.standard_normal((2, 2, 30, 16)))
    q = oracle.round_bf16(rng.standard_normal((2, 1, 4, 16)))
    k = oracle.round_bf16(rng.standard_normal((2, 1, 2, 16)))
    v = oracle.round_bf16(rng.standard_normal((2, 1, 2, 16)))
    lens = np.array([30, 9])
    r1 = oracle.decode_step_multi(K0, V0, q, k, v, lens, 500.0, 0.25, "bf16")
    s1 = oracle.decode_step_contiguous(K0, V0, q[:, 0], k[:, 0], v[:, 0], lens, 500.0, 0.25, "bf16")
    assert np.array_equal(r1["out"][:, 0], s1["out"]) and np.array_equal(r1["k_cache"], s1["k_cache"])
    # the n new tokens of one pass equal the last n rows of full causal recomputation
    w = workload("tiny")
    seq = make_tiny_sequence(w)
    scale = 1.0 / math.sqrt(w.head_dim)
    N = seq.prompt_len + seq.decode_evals - 1
    n = 6
    qa, ka, va = (t.double().numpy() for t in (seq.q, seq.k, seq.v))
    K = np.zeros((w.batch, w.h_kv, N, w.head_dim))
    V = np.zeros_like(K)
    for p in range(N - n):
        K[:, :, p] = np.stack([oracle.rope_rotate(ka[p, b], p, w.rope_base) for b in range(w.batch)])
        V[:, :, p] = va[p]
    tail = lambda x: np.transpose(x[N - n:N], (1, 0, 2, 3))  # [n, B, ...] -> [B, n, ...]
    r = oracle.decode_step_multi(K, V, tail(qa), tail(ka), tail(va), np.full(w.batch, N), w.rope_base, scale, "f64")
    _, last_rows, _ = oracle.run_uncached_sequence(seq.q, seq.k, seq.v, seq.prompt_len, seq.decode_evals,
                                                   w.rope_base, scale)
    for i in range(n):
        assert np.max(np.abs(r["out"][:, i] - last_rows[:, :, N - n + i, :])) <= 1e-12
    # paged equals contiguous on the same logical data
    rng = np.random.default_rng(44)
    B, h_kv, cap, d, n = 3, 2, 50, 16, 4
    Kc = oracle.round_bf16(rng.standard_normal((B, h_kv, cap, d)))
    Vc = oracle.round_bf16(rng.standard_normal((B, h_kv, cap, d)))
    q = oracle.round_bf16(rng.standard_normal((B, n, 8, d)))
    k = oracle.round_bf16(rng.standard_normal((B, n, h_kv, d)))
    v = oracle.round_bf16(rng.standard_normal((B, n, h_kv, d)))
    lens = np.array([50, 4, 17])
    rc = oracle.decode_step_multi(Kc, Vc, q, k, v, lens, 10000.0, 0.25, "bf16")
    pk, table = _contiguous_to_paged(Kc, lens, 16, np.random.default_rng(5))
    pv, _ = _contiguous_to_paged(Vc, lens, 16, np.random.default_rng(5))
    rp = oracle.decode_step_multi(pk, pv, q, k, v, lens, 10000.0, 0.25, "bf16", block_table=table, page_size=16)
    assert np.array_equal(rp["out"], rc["out"]) and np.array_equal(rp["lse"], rc["lse"])
    # the pages' expected tokens per verification pass
    g = _load(golden_dir, "speculative.json")
    for c in g["cases"]:
        got = oracle.expected_tokens_per_verify(c["alpha"], c["gamma"])
        assert round(got, c["digits"]) == c["value"]
        # brute force over accept / reject patterns: the pass yields the accepted
        # prefix of the drafts plus one token from the target model
        a, gam = c["alpha"], c["gamma"]
        expect = 0.0
        for pattern in range(2 ** gam):
            accepts = [(pattern >> t) & 1 for t in range(gam)]
            prob = np.prod([a if x else 1 - a for x in accepts])
            prefix = next((t for t, x in enumerate(accepts) if not x), gam)
            expect += prob * (prefix + 1)
        assert abs(expect - got) <= 1e-12
    assert oracle.expected_tokens_per_verify(1.0, 5) == 6.0
    assert abs(oracle.expected_tokens_per_verify(0.0, 5) - 1.0) <= 1e-15


def test_multi_token_planted_mistakes_are_caught():
    def planted(rot_of, end_of):
        def fn(K, V, q, k, v, lens, base, scale, dtype, window=0):
            if window:  # the variants carry no window: the windowed half of the check uses the oracle
                return oracle.decode_step_multi(K, V, q, k, v, lens, base, scale, dtype, window=window)
            return _multi_variant(K, V, q, k, v, lens, base, scale, dtype, rot_of, end_of)
        return fn

    pos = lambda L, n, i: L - n + i
    end = lambda L, n, i: L - n + i + 1
    assert not _fails(check_multi_step, planted(pos, end))  # the restatement itself passes
    assert _fails(check_multi_step, planted(pos, lambda L, n, i: L))  # no causal mask among the new tokens
    assert _fails(check_multi_step, planted(pos, lambda L, n, i: min(L, L - n + i + 2)))  # sees the next draft
    assert _fails(check_multi_step, planted(lambda L, n, i: L - 1, end))  # every new token rotated by L - 1
    assert _fails(check_multi_step, planted(lambda L, n, i: L - n + i + 1, end))  # rotation one position late
