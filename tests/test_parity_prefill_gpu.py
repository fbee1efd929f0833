"""GPU parity of prefill (the prompt's tokens appended and attended causally
in one pass, on the tcgen05 tensor cores) against the fp64 oracle's
``decode_step_multi`` -- prefill is the multi-token step with n = prompt
length.

Tolerances: bf16 outputs and lse max |err| <= 2e-2, fp32 outputs <= 2e-2
(the scores and P pass through bf16 on the tensor cores), lse <= 1e-4 of the
log-sum-exp over the scores the kernel forms (its bf16 query operand,
tests/lse_model.py); the appended cache rows are placement-exact (V byte
copies, K within one bf16 ulp).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from lse_model import assert_lse, paged_keys
from synthetic import make_contiguous_case, make_paged_case, normal, workload

pytestmark = pytest.mark.gpu

TOL = 2e-2
DEV = "cuda"
S_QM, S_KM, S_VM = 21, 22, 23


@pytest.fixture(scope="module")
def m(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mqa_decode_attention_gb300 as mod

    mod.library()
    return mod


def _np(t):
    return t.detach().cpu().to(torch.float64).numpy()


def new_tokens(w, n, device="cpu"):
    q = normal((w.batch, n, w.h_q, w.head_dim), w.seed, S_QM, w.dtype, device)
    k = normal((w.batch, n, w.h_kv, w.head_dim), w.seed, S_KM, w.dtype, device)
    v = normal((w.batch, n, w.h_kv, w.head_dim), w.seed, S_VM, w.dtype, device)
    return q, k, v


def ulp_bf16(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def run_prefill(m, w, n, case, q, k, v, lens, window=0, out_dtype=None):
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q, window=window)
    lens_d = torch.as_tensor(lens, dtype=torch.int32).to(DEV)
    max_len = int(max(lens))
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=1, device=DEV, n_new=n, out_dtype=out_dtype)
    pos = (lens_d - n).to(torch.int32)
    m.prefill_step(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), pos, lens_d, max_len, bufs, w.rope_base,
                   1.0 / math.sqrt(w.head_dim))
    torch.cuda.synchronize()
    B, hq = w.batch, w.h_q  # single-token buffers are [B, H_q, ...]: view them as [B, 1, H_q, ...]
    return dict(out=_np(bufs.out).reshape(B, n, hq, -1), lse=_np(bufs.lse).reshape(B, n, hq), k=kc.cpu(),
                v=vc.cpu(), err=int(bufs.err.item()))


CASES = [
    # B, h_q, h_kv, n (prompt), prefix, capacity
    (2, 8, 2, 1, 0, 8),
    (2, 8, 2, 5, 0, 8),
    (2, 8, 2, 127, 0, 130),
    (1, 8, 2, 128, 0, 128),
    (2, 8, 2, 129, 0, 140),
    (2, 8, 2, 300, 0, 300),
    (2, 8, 2, 200, 57, 260),   # cached prefix of 57 tokens
    (1, 4, 4, 150, 300, 450),  # MHA, prefix longer than the prompt
    (1, 16, 1, 140, 10, 150),  # MQA
    (2, 12, 4, 150, 20, 180),  # G = 3: a block's rows are not whole tokens (query rows by plain loads)
    (1, 6, 1, 100, 0, 100),    # G = 6
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}q{c[1]}kv{c[2]}n{c[3]}pre{c[4]}")
def test_prefill_matches_oracle(m, case):
    B, hq, hkv, n, pre, cap = case
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, seed=500 + n + pre + hq)
    lens = [pre + n] * B
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=cap)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16")
    got = run_prefill(m, w, n, c, q, k, v, lens)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= TOL
    assert_lse(got["lse"], ref["q_rot"], ref["k_cache"], lens, 1.0 / math.sqrt(w.head_dim), "bf16")
    # appended rows: V byte copies, K within one bf16 ulp, nothing else touched
    bk, ak = _np(c.k_cache), _np(got["k"])
    assert np.array_equal(np.any(ak != bk, axis=-1), np.any(ref["k_cache"] != bk, axis=-1))
    assert np.all(np.abs(ak - ref["k_cache"]) <= ulp_bf16(ref["k_cache"]) + 1e-30)
    assert np.array_equal(_np(got["v"]), ref["v_cache"])


@pytest.mark.parametrize("window", [1, 64, 200])
def test_prefill_sliding_window(m, window):
    w = workload("gqa4k").with_(batch=2, h_q=8, h_kv=2, seed=611)
    n, pre = 300, 40
    lens = [pre + n] * 2
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=340)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16", window=window)
    got = run_prefill(m, w, n, c, q, k, v, lens, window=window)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= TOL, window
    assert_lse(got["lse"], ref["q_rot"], ref["k_cache"], lens, 1.0 / math.sqrt(w.head_dim), "bf16", window=window)


def test_prefill_f32_output_and_unequal_rows(m):
    """fp32 output; two sequences of different lengths (the prefix differs)."""
    w = workload("gqa4k").with_(batch=2, h_q=8, h_kv=2, seed=612)
    n = 130
    lens = [n + 3, n + 200]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=340)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16")
    got = run_prefill(m, w, n, c, q, k, v, lens, out_dtype=torch.float32)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= TOL


def test_prefill_errors_and_refusals(m):
    w = workload("gqa4k").with_(batch=2, h_q=8, h_kv=2, seed=613)
    n = 64
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor([64, 64], dtype=torch.int32), capacity=64)
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    q_rot = torch.zeros(2, n, 8, 128, device=DEV)
    out = torch.empty(2, n, 8, 128, dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.gqa_prefill_attention(lay, n, q_rot, torch.tensor([64, 10], dtype=torch.int32, device=DEV), 64, 0.1, out,
                            err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & m.MQA_DEVERR_SEQ_LEN
    wp = workload("paged").with_(batch=1, h_q=8, h_kv=2, seed=614)
    pc = make_paged_case(wp, "cpu", seq_lens=torch.tensor([64], dtype=torch.int32))
    bt = pc.block_table.to(DEV)
    lay_f32 = m.layout_paged(pc.k_pool.float().to(DEV), pc.v_pool.float().to(DEV), bt, 8)
    with pytest.raises(m.MqaError):  # an fp32 (debug) cache has no prefill
        m.gqa_prefill_attention(lay_f32, n, q_rot[:1], torch.tensor([64], dtype=torch.int32, device=DEV), 64, 0.1,
                                out[:1], err=err)


def test_prefill_full_size_sampled(m):
    """4 sequences of 2048 prompt tokens, 32 query / 8 kv heads: two
    (sequence, kv head) units against the oracle, every row of their groups."""
    w = workload("gqa4k").with_(batch=4, seed=615)
    n = 2048
    lens = [n] * w.batch
    c = make_contiguous_case(w, DEV, seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=n)
    q, k, v = new_tokens(w, n, DEV)
    lay = m.layout_contiguous(c.k_cache, c.v_cache, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, n, num_splits=1, device=DEV, n_new=n)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    m.prefill_step(lay, n, q, k, v, lens_d - n, lens_d, n, bufs, w.rope_base)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    G = w.group
    for b, j in [(0, 0), (3, 5)]:
        Kz = torch.zeros(1, 1, n, w.head_dim, dtype=torch.bfloat16)
        ref = oracle.decode_step_multi(Kz, Kz, q[b:b + 1, :, j * G:(j + 1) * G].cpu(), k[b:b + 1, :, j:j + 1].cpu(),
                                       v[b:b + 1, :, j:j + 1].cpu(), [n], w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                       "bf16")
        got = _np(bufs.out[b, :, j * G:(j + 1) * G])
        assert np.max(np.abs(got - ref["out"][0])) <= TOL, (b, j)


def test_prefill_ignores_garbage_past_the_sequence(m):
    """Cache rows at or past L hold NaN: the masked keys contribute nothing."""
    w = workload("gqa4k").with_(batch=2, h_q=8, h_kv=2, seed=616)
    n = 100
    lens = [n, n]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=256)
    c.k_cache[:, :, n:] = float("nan")
    c.v_cache[:, :, n:] = float("nan")
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(c.k_cache[:, :, :n], c.v_cache[:, :, :n], q, k, v, lens, w.rope_base,
                                   1.0 / math.sqrt(w.head_dim), "bf16")
    got = run_prefill(m, w, n, c, q, k, v, lens)
    assert got["err"] == 0
    assert np.all(np.isfinite(got["out"]))
    assert np.max(np.abs(got["out"] - ref["out"])) <= TOL


def run_prefill_paged(m, w, n, pc, q, k, v, lens, window=0, table=None):
    kp, vp = pc.k_pool.to(DEV), pc.v_pool.to(DEV)
    bt = (pc.block_table if table is None else table).to(DEV)
    lay = m.layout_paged(kp, vp, bt, w.h_q, window=window)
    lens_d = torch.as_tensor(lens, dtype=torch.int32).to(DEV)
    max_len = int(max(lens))
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=1, device=DEV, n_new=n)
    m.prefill_step(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), (lens_d - n).to(torch.int32), lens_d, max_len, bufs,
                   w.rope_base, 1.0 / math.sqrt(w.head_dim))
    torch.cuda.synchronize()
    B, hq = w.batch, w.h_q
    return dict(out=_np(bufs.out).reshape(B, n, hq, -1), lse=_np(bufs.lse).reshape(B, n, hq), k=kp.cpu(),
                v=vp.cpu(), err=int(bufs.err.item()))


PAGED_CASES = [
    # B, h_q, h_kv, n (prompt), prefixes, page_size
    (2, 8, 2, 5, [0, 0], 16),
    (2, 8, 2, 129, [0, 3], 16),
    (2, 8, 2, 200, [57, 0], 32),
    (2, 8, 2, 300, [0, 64], 64),
    (1, 8, 2, 250, [100], 128),
    (2, 16, 1, 140, [10, 300], 256),   # MQA, prefix longer than a page
    (1, 4, 4, 190, [70], 64),          # MHA
    (2, 12, 4, 130, [0, 17], 32),      # G = 3 (query rows by plain loads)
]


@pytest.mark.parametrize("case", PAGED_CASES, ids=lambda c: f"B{c[0]}q{c[1]}kv{c[2]}n{c[3]}ps{c[5]}")
def test_prefill_paged_matches_oracle(m, case):
    """Prefill over a paged pool (PagedAttention, "Arsitektur Inferensi LLM",
    section 4): the prompt's rows land in the pages the block table names and
    the key tiles are gathered page by page."""
    B, hq, hkv, n, pre, ps = case
    w = workload("paged").with_(batch=B, h_q=hq, h_kv=hkv, page_size=ps, seed=700 + n + ps + hq)
    lens = [p_ + n for p_ in pre]
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=2)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(pc.k_pool, pc.v_pool, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16", block_table=pc.block_table, page_size=ps)
    got = run_prefill_paged(m, w, n, pc, q, k, v, lens)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= TOL
    keys = paged_keys(ref["k_pool"], pc.block_table, lens, ps)
    assert_lse(got["lse"], ref["q_rot"], keys, lens, 1.0 / math.sqrt(w.head_dim), "bf16")
    bk, ak = _np(pc.k_pool), _np(got["k"])
    assert np.array_equal(np.any(ak != bk, axis=-1), np.any(ref["k_pool"] != bk, axis=-1))
    assert np.all(np.abs(ak - ref["k_pool"]) <= ulp_bf16(ref["k_pool"]) + 1e-30)
    assert np.array_equal(_np(got["v"]), ref["v_pool"])


@pytest.mark.parametrize("window, ps", [(1, 16), (64, 16), (200, 64), (100, 256)])
def test_prefill_paged_window_released_pages(m, window, ps):
    """A sliding window over a paged pool: the pages wholly before the first
    prompt token's window are released (table entry -1) and never read."""
    w = workload("paged").with_(batch=2, h_q=8, h_kv=2, page_size=ps, seed=720 + window)
    n, pre = 300, 600
    lens = [pre + n, pre + n - 50]
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=1)
    table = pc.block_table.clone()
    for b, L in enumerate(lens):
        first = max(0, L - n + 1 - window)  # the first key the first prompt token attends
        table[b, :first // ps] = -1
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(pc.k_pool, pc.v_pool, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16", block_table=pc.block_table, page_size=ps, window=window)
    got = run_prefill_paged(m, w, n, pc, q, k, v, lens, window=window, table=table)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= TOL
    keys = paged_keys(ref["k_pool"], pc.block_table, lens, ps)
    assert_lse(got["lse"], ref["q_rot"], keys, lens, 1.0 / math.sqrt(w.head_dim), "bf16", window=window)


def test_prefill_paged_bad_page_is_reported(m):
    """A table entry outside the pool, for a page the prompt attends: the call
    reports MQA_DEVERR_PAGE_RANGE (the page reads as zeros) and the other
    sequence's rows are unaffected."""
    w = workload("paged").with_(batch=2, h_q=8, h_kv=2, page_size=16, seed=731)
    n, lens = 40, [40 + 80, 40 + 80]
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=1)
    table = pc.block_table.clone()
    table[0, 1] = pc.num_pages + 7  # a cached prefix page of sequence 0
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(pc.k_pool, pc.v_pool, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16", block_table=pc.block_table, page_size=16)
    got = run_prefill_paged(m, w, n, pc, q, k, v, lens, table=table)
    assert got["err"] & m.MQA_DEVERR_PAGE_RANGE
    assert np.max(np.abs(got["out"][1] - ref["out"][1])) <= TOL


# ------------------------------------------------------- one-byte caches
@pytest.mark.parametrize("paged, pre", [(False, 0), (False, 70), (True, 0), (True, 45)],
                         ids=["contiguous", "contiguous_prefix", "paged", "paged_prefix"])
def test_prefill_u8_matches_oracle(m, paged, pre):
    """Prefill over a uint8 cache (the one-byte warp-MMA kernel's multi-token
    form over the whole prompt) against decode_step_multi_u8: the prompt's
    codes, scales and zero points bit for bit, outputs within 2e-2."""
    from synthetic import make_u8_cache
    n, B, hq, hkv = 150, 2, 8, 2
    lens = [pre + n, n]
    w = workload("paged" if paged else "gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, page_size=32, seed=760 + pre)
    q, k, v = new_tokens(w, n)
    scale = 1.0 / math.sqrt(128)
    if paged:
        pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=1)
        u = make_u8_cache((pc.num_pages, hkv, 32), 128, 77)
        ref = oracle.decode_step_multi_u8(u.k_codes, u.k_sz, u.v_codes, u.v_sz, q, k, v, lens, w.rope_base, scale,
                                          block_table=pc.block_table, page_size=32)
        bt = pc.block_table.to(DEV)
    else:
        u = make_u8_cache((B, hkv, pre + n), 128, 77)
        ref = oracle.decode_step_multi_u8(u.k_codes, u.k_sz, u.v_codes, u.v_sz, q, k, v, lens, w.rope_base, scale)
    kc, vc, ks, vs = u.k_codes.to(DEV), u.v_codes.to(DEV), u.k_sz.to(DEV), u.v_sz.to(DEV)
    lay = (m.layout_paged(kc, vc, bt, hq, k_scale_zero=ks, v_scale_zero=vs) if paged else
           m.layout_contiguous(kc, vc, hq, k_scale_zero=ks, v_scale_zero=vs))
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    bufs = m.DecodeBuffers.allocate(lay, max(lens), num_splits=1, device=DEV, n_new=n)
    m.prefill_step(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), lens_d - n, lens_d, max(lens), bufs, w.rope_base, scale)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    out = _np(bufs.out).reshape(ref["out"].shape)
    assert np.max(np.abs(out - ref["out"])) <= TOL
    assert np.max(np.abs(_np(bufs.lse).reshape(ref["lse"].shape) - ref["lse"])) <= TOL
    assert np.array_equal(kc.cpu().numpy(), ref["k_codes"]) and np.array_equal(vc.cpu().numpy(), ref["v_codes"])
    for got, want in ((ks, ref["k_sz"]), (vs, ref["v_sz"])):
        assert np.array_equal(got.cpu().numpy().view(np.uint32), np.asarray(want, np.float32).view(np.uint32))


@pytest.mark.parametrize("pre", [0, 40])
def test_prefill_e5m2_paged_matches_oracle(m, pre):
    """Prefill over a paged e5m2 pool (the one-byte warp-MMA kernel) against
    decode_step_multi_e5m2."""
    from synthetic import make_e5m2_cache
    n, B, hq, hkv = 140, 2, 16, 2
    lens = [pre + n, n + 5]
    w = workload("paged").with_(batch=B, h_q=hq, h_kv=hkv, page_size=16, seed=780 + pre)
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=1)
    kc8, vc8 = make_e5m2_cache((pc.num_pages, hkv, 16), 128, seed=79)
    q, k, v = new_tokens(w, n)
    scale = 1.0 / math.sqrt(128)
    codes = lambda t: t.detach().cpu().view(torch.uint8).numpy()
    ref = oracle.decode_step_multi_e5m2(codes(kc8), codes(vc8), q, k, v, lens, w.rope_base, scale,
                                        block_table=pc.block_table, page_size=16)
    kd, vd, bt = kc8.to(DEV), vc8.to(DEV), pc.block_table.to(DEV)
    lay = m.layout_paged(kd, vd, bt, hq)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    bufs = m.DecodeBuffers.allocate(lay, max(lens), num_splits=1, device=DEV, n_new=n)
    m.prefill_step(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), lens_d - n, lens_d, max(lens), bufs, w.rope_base, scale)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    assert np.max(np.abs(_np(bufs.out).reshape(ref["out"].shape) - ref["out"])) <= TOL
    assert np.array_equal(codes(kd), ref["k_codes"]) and np.array_equal(codes(vd), ref["v_codes"])
