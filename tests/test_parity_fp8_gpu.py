"""GPU parity of the fp8 e5m2 KV cache (MQA_FP8_E5M2) against the fp64 oracle.

The oracle rounds the new token's fp64-rotated key and its bf16 value once to
e5m2 and attends over the decoded cache in fp64. The append is byte work and
must match exactly: the appended codes, and nothing else in the caches
changes. Outputs are bf16, max |err| <= 2e-2 like the bf16 cache path; the
fp32 lse is held to 1e-4 of the log-sum-exp over the scores the kernels form
(tests/lse_model.py): an fp16 query operand on the one-token kernels, e4m3 hi +
lo on the tcgen05 kernel that serves several new tokens.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from lse_model import assert_lse, paged_keys
from synthetic import make_contiguous_case, make_e5m2_cache, make_paged_case, normal, workload

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
DEV = "cuda"


@pytest.fixture(scope="module")
def m(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mqa_decode_attention_gb300 as mod

    mod.library()
    return mod


def _np(t):
    return t.detach().cpu().to(torch.float64).numpy()


def _codes(t):
    return t.detach().cpu().view(torch.uint8).numpy()


def run_f8(m, w, case, kc8, vc8, paged, splits=0, window=0, table=None, max_len=None):
    kc, vc = kc8.to(DEV), vc8.to(DEV)
    if paged:
        bt = (case.block_table if table is None else table).to(DEV)
        lay = m.layout_paged(kc, vc, bt, w.h_q, window=window)
    else:
        lay = m.layout_contiguous(kc, vc, w.h_q, window=window)
    max_len = int(case.seq_lens.max()) if max_len is None else max_len
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=splits, device=DEV)
    m.decode_step(lay, case.q_new.to(DEV), case.k_new.to(DEV), case.v_new.to(DEV), case.pos.to(DEV),
                  case.seq_lens.to(DEV), max_len, bufs, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                  num_splits=splits)
    torch.cuda.synchronize()
    return dict(out=_np(bufs.out), lse=_np(bufs.lse), q_rot=_np(bufs.q_rot), err=int(bufs.err.item()),
                k_codes=_codes(kc), v_codes=_codes(vc))


def _oracle(w, case, kc8, vc8, paged, window=0):
    kw = dict(block_table=case.block_table, page_size=case.page_size) if paged else {}
    return oracle.decode_step_e5m2(_codes(kc8), _codes(vc8), case.q_new, case.k_new, case.v_new, case.seq_lens,
                                   w.rope_base, 1.0 / math.sqrt(w.head_dim), window=window, **kw)


def _keys(ref, case, paged):
    """The logical keys after the append, decoded from the oracle's codes."""
    k = oracle.dequantize_e5m2(ref["k_codes"])
    return paged_keys(k, case.block_table, case.seq_lens, case.page_size) if paged else k


def q_fmt(case, paged=False):
    """The query operand of the kernel that serves a one-token step over an
    e5m2 cache: the warp-MMA kernels, fp16 (the tcgen05 kernel's fp8 form,
    e4m3 hi + lo, serves only several new tokens)."""
    return "f16"


def check(got, ref, case, paged=False, window=0):
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= BF16_TOL
    assert_lse(got["lse"], ref["q_rot"], _keys(ref, case, paged), case.seq_lens, 1.0 / math.sqrt(case.q_new.shape[-1]),
               q_fmt(case, paged), window=window)
    assert np.max(np.abs(got["q_rot"] - ref["q_rot"])) <= 1e-5 * (1 + np.max(np.abs(ref["q_rot"])))
    for key in ("k_codes", "v_codes"):  # the appended rows bit for bit, every other row untouched
        bad = np.argwhere(got[key] != ref[key])
        assert bad.size == 0, (key, bad[:5])


SHAPES = [
    # B, h_q, h_kv, d, lens, capacity
    (2, 32, 8, 128, [1000, 257], 1000),      # G=4, ragged tail
    (3, 8, 8, 128, [64, 1, 129], 130),       # MHA
    (1, 16, 1, 128, [777], 778),             # MQA, G=16
    (2, 64, 2, 128, [300, 45], 300),         # G=32: two head blocks in one CTA
    (1, 96, 1, 64, [200], 200),              # G=96, d=64
    (2, 12, 3, 64, [513, 64], 514),          # d=64, G=4
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s[0]}q{s[1]}kv{s[2]}d{s[3]}")
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_e5m2_contiguous_matches_oracle(m, shape, splits):
    B, hq, hkv, d, lens, cap = shape
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, head_dim=d, seed=400 + hq + d)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=cap)
    kc8, vc8 = make_e5m2_cache((B, hkv, cap), d, seed=11 + d)
    check(run_f8(m, w, c, kc8, vc8, paged=False, splits=splits), _oracle(w, c, kc8, vc8, paged=False), c)


@pytest.mark.parametrize("page_size", [16, 32, 64])
@pytest.mark.parametrize("heads", [(16, 2, 128), (32, 8, 128), (12, 3, 128), (64, 2, 128), (16, 4, 64)],
                         ids=lambda h: f"q{h[0]}kv{h[1]}d{h[2]}")
def test_e5m2_paged_matches_oracle(m, page_size, heads):
    """16- and 32-token pages with G <= 16 and an even kv head count take the
    head-group kernel, the rest the token-slice kernel."""
    w = workload("paged").with_(batch=5, h_q=heads[0], h_kv=heads[1], head_dim=heads[2], page_size=page_size,
                                len_lo=1, len_hi=700, seed=29)
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor([1, 16, 17, 700, 333], dtype=torch.int32), spare_pages=2)
    kc8, vc8 = make_e5m2_cache((pc.num_pages, w.h_kv, pc.page_size), w.head_dim, seed=31)
    ref = _oracle(w, pc, kc8, vc8, paged=True)
    for splits in (1, 3, 0):
        check(run_f8(m, w, pc, kc8, vc8, paged=True, splits=splits), ref, pc, paged=True)


@pytest.mark.parametrize("window", [1, 17, 100, 1000])
def test_e5m2_sliding_window(m, window):
    w = workload("gqa4k").with_(batch=3, h_q=16, h_kv=4, seed=81)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor([700, 65, 3], dtype=torch.int32), capacity=704)
    kc8, vc8 = make_e5m2_cache((3, 4, 704), 128, seed=12)
    ref = _oracle(w, c, kc8, vc8, paged=False, window=window)
    for splits in (1, 0):
        got = run_f8(m, w, c, kc8, vc8, paged=False, splits=splits, window=window, max_len=700)
        assert got["err"] == 0
        assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL, (splits, window)
        assert_lse(got["lse"], ref["q_rot"], _keys(ref, c, False), c.seq_lens, 1.0 / math.sqrt(128), q_fmt(c),
                   window=window, what=splits)


def test_e5m2_nan_codes_past_the_sequence(m):
    """Rows at or past L hold NaN / infinity codes: the masked keys and values
    contribute nothing (their V codes are cleared before the P V product)."""
    w = workload("gqa4k").with_(batch=3, h_q=32, h_kv=8, seed=82)
    lens = [100, 37, 64]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=200)
    kc8, vc8 = make_e5m2_cache((3, 8, 200), 128, seed=13)
    for b, L in enumerate(lens):
        kc8.view(torch.uint8)[b, :, L:] = 0x7F  # NaN
        vc8.view(torch.uint8)[b, :, L:] = 0xFC  # -inf
    ref = oracle.decode_step_e5m2(_codes(kc8)[:, :, :100], _codes(vc8)[:, :, :100], c.q_new, c.k_new, c.v_new,
                                  c.seq_lens, w.rope_base, 1.0 / math.sqrt(128))
    for splits in (1, 2):
        got = run_f8(m, w, c, kc8, vc8, paged=False, splits=splits, max_len=100)
        assert got["err"] == 0
        assert np.all(np.isfinite(got["out"]))
        assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL


def _new_tokens(w, n, seed):
    q = normal((w.batch, n, w.h_q, w.head_dim), seed, 21)
    k = normal((w.batch, n, w.h_kv, w.head_dim), seed, 22)
    v = normal((w.batch, n, w.h_kv, w.head_dim), seed, 23)
    return q, k, v


def _check_multi(got_out, got_lse, kc8, vc8, ref, lens, w, n, window=0, what=None):
    assert np.max(np.abs(got_out.reshape(ref["out"].shape) - ref["out"])) <= BF16_TOL, what
    assert np.max(np.abs(got_lse.reshape(ref["lse"].shape) - ref["lse"])) <= BF16_TOL, what
    assert_lse(got_lse.reshape(ref["lse"].shape), ref["q_rot"], oracle.dequantize_e5m2(ref["k_codes"]), lens,
               1.0 / math.sqrt(w.head_dim), "e4m3x2", window=window, what=what)
    assert np.array_equal(_codes(kc8), ref["k_codes"]) and np.array_equal(_codes(vc8), ref["v_codes"]), what


MULTI = [
    # B, h_q, h_kv, lens, capacity, n: 32 or more query rows (G x n) per kv head
    (2, 32, 8, [1000, 257], 1000, 8),    # G = 4 x 8 tokens
    (2, 32, 1, [700, 2], 704, 2),        # MQA, G = 32 x 2
    (3, 16, 2, [300, 129, 4], 300, 4),   # G = 8 x 4
    (1, 32, 1, [260], 260, 5),           # 160 rows: two row blocks
]


@pytest.mark.parametrize("shape", MULTI, ids=lambda s: f"B{s[0]}q{s[1]}kv{s[2]}n{s[5]}")
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_e5m2_multi_token_matches_oracle(m, shape, splits):
    """Several new tokens per sequence (the verification pass) over an e5m2
    cache, on the tcgen05 kernel's fp8 form: the appended codes bit for bit,
    outputs and lse against the oracle's decode_step_multi_e5m2."""
    B, hq, hkv, lens, cap, n = shape
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, seed=470 + hq + n)
    kc8, vc8 = make_e5m2_cache((B, hkv, cap), 128, seed=19 + n)
    q, k, v = _new_tokens(w, n, w.seed)
    ref = oracle.decode_step_multi_e5m2(_codes(kc8), _codes(vc8), q, k, v, lens, w.rope_base,
                                        1.0 / math.sqrt(w.head_dim))
    kd, vd = kc8.to(DEV), vc8.to(DEV)
    lay = m.layout_contiguous(kd, vd, hq)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    bufs = m.DecodeBuffers.allocate(lay, max(lens), num_splits=splits, device=DEV, n_new=n)
    m.decode_step_multi(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), lens_d - n, lens_d, max(lens), bufs, w.rope_base,
                        1.0 / math.sqrt(w.head_dim), num_splits=splits)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    _check_multi(_np(bufs.out), _np(bufs.lse), kd, vd, ref, lens, w, n, what=splits)


@pytest.mark.parametrize("window", [1, 100])
def test_e5m2_multi_token_window(m, window):
    n, lens = 3, [900, 50]
    w = workload("gqa4k").with_(batch=2, h_q=32, h_kv=1, seed=481)
    kc8, vc8 = make_e5m2_cache((2, 1, 900), 128, seed=23)
    q, k, v = _new_tokens(w, n, w.seed)
    ref = oracle.decode_step_multi_e5m2(_codes(kc8), _codes(vc8), q, k, v, lens, w.rope_base,
                                        1.0 / math.sqrt(128), window=window)
    kd, vd = kc8.to(DEV), vc8.to(DEV)
    lay = m.layout_contiguous(kd, vd, 32, window=window)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    for splits in (1, 4, 0):
        bufs = m.DecodeBuffers.allocate(lay, 900, num_splits=splits, device=DEV, n_new=n)
        kd.copy_(kc8.to(DEV))
        vd.copy_(vc8.to(DEV))
        m.decode_step_multi(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), lens_d - n, lens_d, 900, bufs, w.rope_base,
                            1.0 / math.sqrt(128), num_splits=splits)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0
        _check_multi(_np(bufs.out), _np(bufs.lse), kd, vd, ref, lens, w, n, window=window, what=(window, splits))


PREFILL = [
    # B, h_q, h_kv, n (prompt), prefix, capacity
    (2, 8, 2, 5, 0, 8),
    (2, 8, 2, 129, 0, 140),
    (2, 8, 2, 200, 57, 260),
    (1, 16, 1, 140, 10, 150),
    (2, 12, 4, 129, 0, 140),   # G = 3: query rows by plain loads
]


@pytest.mark.parametrize("case", PREFILL, ids=lambda c: f"B{c[0]}q{c[1]}kv{c[2]}n{c[3]}pre{c[4]}")
def test_e5m2_prefill_matches_oracle(m, case):
    """A prompt appended and attended causally in one pass over an e5m2 cache
    (with and without a cached prefix): prefill is the multi-token step with n
    = prompt length."""
    B, hq, hkv, n, pre, cap = case
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, seed=560 + n + pre)
    lens = [pre + n] * B
    kc8, vc8 = make_e5m2_cache((B, hkv, cap), 128, seed=29 + n)
    q, k, v = _new_tokens(w, n, w.seed)
    ref = oracle.decode_step_multi_e5m2(_codes(kc8), _codes(vc8), q, k, v, lens, w.rope_base,
                                        1.0 / math.sqrt(128))
    kd, vd = kc8.to(DEV), vc8.to(DEV)
    lay = m.layout_contiguous(kd, vd, hq)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    bufs = m.DecodeBuffers.allocate(lay, max(lens), num_splits=1, device=DEV, n_new=n)
    m.prefill_step(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), lens_d - n, lens_d, max(lens), bufs, w.rope_base,
                   1.0 / math.sqrt(128))
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    _check_multi(_np(bufs.out), _np(bufs.lse), kd, vd, ref, lens, w, n)


def test_e5m2_full_size_sampled(m):
    """The 4096-token GQA workload (batch 32, 32 query / 8 kv heads) over an
    e5m2 cache: three (sequence, kv head) units against the oracle."""
    w = workload("gqa4k")
    L = w.seq_len
    c = make_contiguous_case(w, DEV)
    kc8, vc8 = make_e5m2_cache((w.batch, w.h_kv, L), w.head_dim, 15, device=DEV)
    units = [(0, 0), (w.batch - 1, w.h_kv - 1), (13, 5)]
    saved = {(b, j): (_codes(kc8[b, j]), _codes(vc8[b, j])) for b, j in units}
    lay = m.layout_contiguous(kc8, vc8, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, L, num_splits=0, device=DEV)
    m.decode_step(lay, c.q_new, c.k_new, c.v_new, c.pos, c.seq_lens, L, bufs, w.rope_base,
                  1.0 / math.sqrt(w.head_dim), num_splits=0)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    G = w.group
    for b, j in units:
        kc, vc = saved[(b, j)]
        ref = oracle.decode_step_e5m2(kc[None, None], vc[None, None], c.q_new[b:b + 1, j * G:(j + 1) * G].cpu(),
                                      c.k_new[b:b + 1, j:j + 1].cpu(), c.v_new[b:b + 1, j:j + 1].cpu(), [L],
                                      w.rope_base, 1.0 / math.sqrt(w.head_dim))
        assert np.max(np.abs(_np(bufs.out[b, j * G:(j + 1) * G]) - ref["out"][0])) <= BF16_TOL, (b, j)
        assert np.array_equal(_codes(kc8[b, j, L - 1]), ref["k_codes"][0, 0, L - 1])


MANY_HEADS = [
    # B, h_q, h_kv, lens, capacity: 32 or more query heads per kv head (two or more 16-head blocks)
    (3, 32, 1, [1000, 129, 1], 1000),   # MQA: 32 rows, 4 parts
    (2, 64, 1, [700, 300], 704),        # 64 rows, 2 parts
    (1, 128, 1, [300], 300),            # 128 rows, 1 part
    (2, 64, 2, [513, 64], 514),         # two kv heads
]


@pytest.mark.parametrize("shape", MANY_HEADS, ids=lambda s: f"B{s[0]}q{s[1]}kv{s[2]}")
@pytest.mark.parametrize("splits", [1, 2, 3, 0])
def test_e5m2_many_heads_matches_oracle(m, shape, splits):
    B, hq, hkv, lens, cap = shape
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, seed=420 + hq + hkv)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=cap)
    kc8, vc8 = make_e5m2_cache((B, hkv, cap), 128, seed=16 + hq)
    check(run_f8(m, w, c, kc8, vc8, paged=False, splits=splits), _oracle(w, c, kc8, vc8, paged=False), c)


@pytest.mark.parametrize("window", [1, 100, 1000])
def test_e5m2_mqa_window_and_nan_tail(m, window):
    """MQA over e5m2 with a window, and NaN / infinity codes in the rows past
    each sequence (their codes are cleared before the P V product)."""
    w = workload("gqa4k").with_(batch=3, h_q=32, h_kv=1, seed=431)
    lens = [900, 200, 37]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=1024)
    kc8, vc8 = make_e5m2_cache((3, 1, 1024), 128, seed=17)
    for b, L in enumerate(lens):
        kc8.view(torch.uint8)[b, :, L:] = 0x7F
        vc8.view(torch.uint8)[b, :, L:] = 0xFC
    ref = oracle.decode_step_e5m2(_codes(kc8)[:, :, :900], _codes(vc8)[:, :, :900], c.q_new, c.k_new, c.v_new,
                                  c.seq_lens, w.rope_base, 1.0 / math.sqrt(128), window=window)
    for splits in (1, 2, 0):
        got = run_f8(m, w, c, kc8, vc8, paged=False, splits=splits, window=window, max_len=900)
        assert got["err"] == 0
        assert np.all(np.isfinite(got["out"]))
        assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL, (splits, window)
        assert_lse(got["lse"], ref["q_rot"], _keys(ref, c, False), c.seq_lens, 1.0 / math.sqrt(128), q_fmt(c),
                   window=window, what=splits)


def test_e5m2_mqa_full_size_sampled(m):
    """The MQA workload (64 sequences of 8192 tokens, 32 query heads on one kv
    head) over an e5m2 cache: three sequences against the oracle."""
    w = workload("mqa8k")
    L = w.seq_len
    c = make_contiguous_case(w, DEV)
    kc8, vc8 = make_e5m2_cache((w.batch, 1, L), 128, 18, device=DEV)
    seqs = [0, 31, 63]
    saved = {b: (_codes(kc8[b, 0]), _codes(vc8[b, 0])) for b in seqs}
    lay = m.layout_contiguous(kc8, vc8, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, L, num_splits=0, device=DEV)
    m.decode_step(lay, c.q_new, c.k_new, c.v_new, c.pos, c.seq_lens, L, bufs, w.rope_base, 1.0 / math.sqrt(128))
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    for b in seqs:
        kc, vc = saved[b]
        ref = oracle.decode_step_e5m2(kc[None, None], vc[None, None], c.q_new[b:b + 1].cpu(), c.k_new[b:b + 1].cpu(),
                                      c.v_new[b:b + 1].cpu(), [L], w.rope_base, 1.0 / math.sqrt(128))
        assert np.max(np.abs(_np(bufs.out[b]) - ref["out"][0])) <= BF16_TOL, b


SMALL_MULTI = [
    # B, h_q, h_kv, lens, capacity, n: fewer than 32 (token, head) rows per kv
    # head, on the warp-MMA one-byte kernel (fp16 query operand)
    (2, 8, 2, [300, 64], 300, 2),     # G = 4 x 2
    (2, 32, 8, [1000, 9], 1000, 4),   # G = 4 x 4
    (1, 16, 2, [129], 129, 3),        # G = 8 x 3
]


@pytest.mark.parametrize("shape", SMALL_MULTI, ids=lambda s: f"B{s[0]}q{s[1]}kv{s[2]}n{s[5]}")
@pytest.mark.parametrize("splits", [1, 3])
def test_e5m2_multi_token_small_groups(m, shape, splits):
    """Several new tokens with fewer than 32 rows per kv head over an e5m2
    cache (the one-byte warp-MMA kernel's multi-token form) against
    decode_step_multi_e5m2."""
    B, hq, hkv, lens, cap, n = shape
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, seed=590 + hq + n)
    kc8, vc8 = make_e5m2_cache((B, hkv, cap), 128, seed=31 + n)
    q, k, v = _new_tokens(w, n, w.seed)
    ref = oracle.decode_step_multi_e5m2(_codes(kc8), _codes(vc8), q, k, v, lens, w.rope_base,
                                        1.0 / math.sqrt(w.head_dim))
    kd, vd = kc8.to(DEV), vc8.to(DEV)
    lay = m.layout_contiguous(kd, vd, hq)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    bufs = m.DecodeBuffers.allocate(lay, max(lens), num_splits=splits, device=DEV, n_new=n)
    m.decode_step_multi(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), lens_d - n, lens_d, max(lens), bufs, w.rope_base,
                        1.0 / math.sqrt(w.head_dim), num_splits=splits)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    got_out, got_lse = _np(bufs.out), _np(bufs.lse)
    assert np.max(np.abs(got_out.reshape(ref["out"].shape) - ref["out"])) <= BF16_TOL
    assert np.max(np.abs(got_lse.reshape(ref["lse"].shape) - ref["lse"])) <= BF16_TOL
    assert_lse(got_lse.reshape(ref["lse"].shape), ref["q_rot"], oracle.dequantize_e5m2(ref["k_codes"]), lens,
               1.0 / math.sqrt(w.head_dim), "f16")
    assert np.array_equal(_codes(kd), ref["k_codes"]) and np.array_equal(_codes(vd), ref["v_codes"])


@pytest.mark.parametrize("page_size", [16, 64])
def test_e5m2_multi_token_paged(m, page_size):
    """Several new tokens over a paged e5m2 pool (the one-byte warp-MMA kernel
    for every row count: the tcgen05 fp8 form reads contiguous caches only)."""
    n = 8
    w = workload("paged").with_(batch=3, h_q=32, h_kv=8, page_size=page_size, seed=600 + page_size)
    lens = [700, n, 130]
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=2)
    kc8, vc8 = make_e5m2_cache((pc.num_pages, w.h_kv, page_size), 128, seed=37)
    q, k, v = _new_tokens(w, n, w.seed)
    ref = oracle.decode_step_multi_e5m2(_codes(kc8), _codes(vc8), q, k, v, lens, w.rope_base,
                                        1.0 / math.sqrt(w.head_dim), block_table=pc.block_table,
                                        page_size=page_size)
    for splits in (1, 3):
        kd, vd = kc8.to(DEV), vc8.to(DEV)
        bt = pc.block_table.to(DEV)
        lay = m.layout_paged(kd, vd, bt, w.h_q)
        lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
        bufs = m.DecodeBuffers.allocate(lay, max(lens), num_splits=splits, device=DEV, n_new=n)
        m.decode_step_multi(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), lens_d - n, lens_d, max(lens), bufs,
                            w.rope_base, 1.0 / math.sqrt(w.head_dim), num_splits=splits)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0, splits
        got_out, got_lse = _np(bufs.out), _np(bufs.lse)
        assert np.max(np.abs(got_out.reshape(ref["out"].shape) - ref["out"])) <= BF16_TOL, splits
        keys = paged_keys(oracle.dequantize_e5m2(ref["k_codes"]), pc.block_table, lens, page_size)
        assert_lse(got_lse.reshape(ref["lse"].shape), ref["q_rot"], keys, lens, 1.0 / math.sqrt(w.head_dim), "f16",
                   what=splits)
        assert np.array_equal(_codes(kd), ref["k_codes"]) and np.array_equal(_codes(vd), ref["v_codes"])
