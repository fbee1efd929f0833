"""GPU parity of multi-token decode (the verification pass of speculative
decoding: n new tokens per sequence, causal among them) against the fp64
oracle's ``decode_step_multi``.

Tolerances as for single-token decode: bf16 outputs and lse max |err| <= 2e-2,
and lse <= 1e-4 of the log-sum-exp over the scores the kernel forms (its bf16
query operand, tests/lse_model.py);
the append is placement-exact (only the n target slots of each sequence
change, V slices are byte copies, K within one bf16 ulp of the fp64 RoPE).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from lse_model import assert_lse, paged_keys
from synthetic import make_contiguous_case, make_paged_case, normal, workload

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
DEV = "cuda"
S_QM, S_KM, S_VM = 21, 22, 23  # seeded streams of the new tokens' q, k, v


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


def check_cache(before, after, ref, v_cache: bool):
    """Rows the GPU changed are exactly the rows the oracle changed; there V is
    a byte copy and K within one bf16 ulp of the oracle's rounded fp64 RoPE."""
    b, a = _np(before), _np(after)
    rows_ref = np.any(ref != b, axis=-1)
    rows_gpu = np.any(a != b, axis=-1)
    assert np.array_equal(rows_ref, rows_gpu)
    if v_cache:
        assert np.array_equal(a, ref)
    else:
        assert np.all(np.abs(a - ref) <= ulp_bf16(ref) + 1e-30)


def run_multi(m, w, n, kc, vc, q, k, v, lens, splits=0, window=0, table=None, page_size=0, max_len=None,
              variant=0):
    kc, vc = kc.to(DEV), vc.to(DEV)
    bt = None if table is None else table.to(DEV)  # held: the layout keeps only its address
    if bt is None:
        lay = m.layout_contiguous(kc, vc, w.h_q, window=window)
    else:
        lay = m.layout_paged(kc, vc, bt, w.h_q, window=window)
    lens_d = torch.as_tensor(lens, dtype=torch.int32).to(DEV)
    max_len = int(max(lens)) if max_len is None else max_len
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=splits, variant=variant, device=DEV, n_new=n)
    pos = (lens_d - n).to(torch.int32)
    m.decode_step_multi(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), pos, lens_d, max_len, bufs, w.rope_base,
                        1.0 / math.sqrt(w.head_dim), num_splits=splits, variant=variant)
    torch.cuda.synchronize()
    return dict(out=_np(bufs.out), lse=_np(bufs.lse), q_rot=_np(bufs.q_rot), k=kc.cpu(), v=vc.cpu(),
                err=int(bufs.err.item()))


SHAPES = [
    # B, h_q, h_kv, d, lens, capacity, n
    (2, 32, 8, 128, [1000, 257], 1000, 4),   # G=4 x 4 tokens = one 16-row tile
    (2, 32, 8, 128, [300, 6], 300, 6),       # G=4 x 6 = 24 rows (two head blocks in one block), L = n
    (3, 16, 2, 128, [129, 64, 65], 130, 2),  # G=8 x 2
    (2, 8, 8, 128, [77, 5], 80, 5),          # MHA x 5
    (1, 16, 1, 128, [500], 500, 3),          # MQA G=16 x 3 = 48 rows: two blocks of 32
    (2, 12, 3, 64, [200, 33], 200, 8),       # d=64, G=4 x 8
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s[0]}q{s[1]}kv{s[2]}d{s[3]}n{s[6]}")
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_multi_contiguous_matches_oracle(m, shape, splits):
    B, hq, hkv, d, lens, cap, n = shape
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, head_dim=d, seed=400 + hq + d + n)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=cap)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(d), "bf16")
    got = run_multi(m, w, n, c.k_cache, c.v_cache, q, k, v, lens, splits=splits)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= BF16_TOL
    assert_lse(got["lse"], ref["q_rot"], ref["k_cache"], lens, 1.0 / math.sqrt(d), "bf16")
    assert np.max(np.abs(got["q_rot"] - ref["q_rot"])) <= 1e-5 * (1 + np.max(np.abs(ref["q_rot"])))
    check_cache(c.k_cache, got["k"], ref["k_cache"], v_cache=False)
    check_cache(c.v_cache, got["v"], ref["v_cache"], v_cache=True)


@pytest.mark.parametrize("page_size", [16, 64])
@pytest.mark.parametrize("n", [2, 5])
def test_multi_paged_matches_oracle(m, page_size, n):
    w = workload("paged").with_(batch=4, h_q=16, h_kv=4, page_size=page_size, seed=31 + n)
    lens = [700, n, 17, 64]
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=2)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(pc.k_pool, pc.v_pool, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16", block_table=pc.block_table, page_size=page_size)
    keys = paged_keys(ref["k_pool"], pc.block_table, lens, page_size)
    for splits in (1, 3, 0):
        got = run_multi(m, w, n, pc.k_pool, pc.v_pool, q, k, v, lens, splits=splits, table=pc.block_table,
                        page_size=page_size)
        assert got["err"] == 0
        assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL, splits
        assert np.max(np.abs(got["lse"] - ref["lse"])) <= BF16_TOL, splits
        assert_lse(got["lse"], ref["q_rot"], keys, lens, 1.0 / math.sqrt(w.head_dim), "bf16", what=splits)
        check_cache(pc.k_pool, got["k"], ref["k_pool"], v_cache=False)
        check_cache(pc.v_pool, got["v"], ref["v_pool"], v_cache=True)


@pytest.mark.parametrize("page_size", [16, 32, 128, 256])
@pytest.mark.parametrize("shape", [(32, 8, 8), (32, 1, 2), (64, 8, 16), (32, 8, 32), (64, 8, 32)],
                         ids=lambda s: f"q{s[0]}kv{s[1]}n{s[2]}")
def test_multi_paged_tc05_matches_oracle(m, page_size, shape):
    """32 or more (token, head) rows per kv head over a paged pool: the
    tcgen05 kernel gathering each key tile page by page -- with the append
    inside the launch (n <= 16, one row block) or after the append launch (n =
    32; 256 rows: two row blocks)."""
    hq, hkv, n = shape
    w = workload("paged").with_(batch=4, h_q=hq, h_kv=hkv, page_size=page_size, seed=41 + n + hq + page_size)
    lens = [700, n, 129 + n, 300]
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=2)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(pc.k_pool, pc.v_pool, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16", block_table=pc.block_table, page_size=page_size)
    keys = paged_keys(ref["k_pool"], pc.block_table, lens, page_size)
    for splits in (1, 2, 3, 0):
        got = run_multi(m, w, n, pc.k_pool, pc.v_pool, q, k, v, lens, splits=splits, table=pc.block_table,
                        page_size=page_size)
        assert got["err"] == 0
        assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL, splits
        assert np.max(np.abs(got["lse"] - ref["lse"])) <= BF16_TOL, splits
        assert_lse(got["lse"], ref["q_rot"], keys, lens, 1.0 / math.sqrt(w.head_dim), "bf16", what=splits)
        check_cache(pc.k_pool, got["k"], ref["k_pool"], v_cache=False)
        check_cache(pc.v_pool, got["v"], ref["v_pool"], v_cache=True)


@pytest.mark.parametrize("window", [1, 50, 300])
def test_multi_paged_tc05_window_released_pages(m, window):
    """Sliding window over a paged pool on the tcgen05 kernel: pages wholly
    before the first new token's window are released (-1) and never read."""
    n, ps = 8, 16
    w = workload("paged").with_(batch=3, h_q=32, h_kv=8, page_size=ps, seed=51 + window)
    lens = [900, 400, n]
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=1)
    table = pc.block_table.clone()
    for b, L in enumerate(lens):
        table[b, :max(0, L - n + 1 - window) // ps] = -1
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(pc.k_pool, pc.v_pool, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16", block_table=pc.block_table, page_size=ps, window=window)
    keys = paged_keys(ref["k_pool"], pc.block_table, lens, ps)
    for splits in (1, 3, 0):
        got = run_multi(m, w, n, pc.k_pool, pc.v_pool, q, k, v, lens, splits=splits, table=table, page_size=ps,
                        window=window)
        assert got["err"] == 0, (window, splits)
        assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL, (window, splits)
        assert_lse(got["lse"], ref["q_rot"], keys, lens, 1.0 / math.sqrt(w.head_dim), "bf16", window=window,
                   what=splits)


def test_multi_paged_tc05_bad_page_is_reported(m):
    """A table entry outside the pool for a page the new tokens attend, and
    one for the page a new token is appended to: both reported as
    MQA_DEVERR_PAGE_RANGE; the other sequences match the oracle."""
    n, ps = 8, 16
    w = workload("paged").with_(batch=3, h_q=32, h_kv=8, page_size=ps, seed=61)
    lens = [300, 200, 100]
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=1)
    table = pc.block_table.clone()
    table[0, 3] = pc.num_pages  # attended, cached page of sequence 0
    table[1, (lens[1] - 1) // ps] = -5  # the page sequence 1's last new token goes to
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(pc.k_pool, pc.v_pool, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16", block_table=pc.block_table, page_size=ps)
    for splits in (1, 3):
        got = run_multi(m, w, n, pc.k_pool, pc.v_pool, q, k, v, lens, splits=splits, table=table, page_size=ps)
        assert got["err"] & m.MQA_DEVERR_PAGE_RANGE, splits
        out = got["out"].reshape(ref["out"].shape)
        assert np.max(np.abs(out[2] - ref["out"][2])) <= BF16_TOL, splits


@pytest.mark.parametrize("window", [1, 3, 17, 100])
def test_multi_sliding_window(m, window):
    """Query token i sees the last W tokens up to its own position."""
    n = 5
    w = workload("gqa4k").with_(batch=3, h_q=16, h_kv=4, seed=81)
    lens = [700, 70, 5]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=704)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16", window=window)
    for splits in (1, 3, 0):
        got = run_multi(m, w, n, c.k_cache, c.v_cache, q, k, v, lens, splits=splits, window=window)
        assert got["err"] == 0
        assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL, (splits, window)
        assert np.max(np.abs(got["lse"] - ref["lse"])) <= BF16_TOL
        assert_lse(got["lse"], ref["q_rot"], ref["k_cache"], lens, 1.0 / math.sqrt(w.head_dim), "bf16",
                   window=window, what=splits)


def test_multi_with_one_token_is_the_single_token_step(m):
    w = workload("gqa4k").with_(batch=2, h_q=32, h_kv=8, seed=82)
    lens = [500, 64]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=500)
    q, k, v = new_tokens(w, 1)
    got = run_multi(m, w, 1, c.k_cache, c.v_cache, q, k, v, lens, splits=1, variant=2)
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, 500, num_splits=1, variant=2, device=DEV)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    m.decode_step(lay, q[:, 0].to(DEV), k[:, 0].to(DEV), v[:, 0].to(DEV), lens_d - 1, lens_d, 500, bufs, w.rope_base,
                  1.0 / math.sqrt(w.head_dim), num_splits=1, variant=2)
    torch.cuda.synchronize()
    assert np.max(np.abs(got["out"] - _np(bufs.out))) <= 1e-2
    assert torch.equal(got["k"], kc.cpu()) and torch.equal(got["v"], vc.cpu())


def test_multi_short_sequence_sets_error(m):
    n = 4
    w = workload("gqa4k").with_(batch=2, h_q=8, h_kv=2, seed=83)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor([50, 50], dtype=torch.int32), capacity=50)
    q, k, v = new_tokens(w, n)
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, 50, num_splits=1, device=DEV, n_new=n)
    m.kv_append_rope_multi(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), torch.tensor([46, 46], dtype=torch.int32,
                           device=DEV), w.rope_base, bufs.q_rot, bufs.err)
    m.gqa_decode_attention_multi(lay, n, bufs.q_rot, torch.tensor([50, 2], dtype=torch.int32, device=DEV), 50,
                                 0.1, 1, bufs.out, bufs.lse, bufs.workspace, 0, bufs.err)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) & m.MQA_DEVERR_SEQ_LEN


def test_multi_unsupported_paths_are_refused(m):
    n = 3
    w = workload("gqa4k").with_(batch=1, h_q=8, h_kv=2, seed=84)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor([40], dtype=torch.int32), capacity=40)
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, 40, num_splits=1, variant=2, device=DEV, n_new=n)
    with pytest.raises(m.MqaError):  # CUDA-core kernel: single token only
        m.gqa_decode_attention_multi(lay, n, bufs.q_rot, torch.tensor([40], dtype=torch.int32, device=DEV), 40, 0.1,
                                     1, bufs.out, bufs.lse, None, 1, bufs.err)
    with pytest.raises(m.MqaError):  # more new tokens than the bound allows
        m.gqa_decode_attention_multi(lay, 33, bufs.q_rot, torch.tensor([40], dtype=torch.int32, device=DEV), 40,
                                     0.1, 1, bufs.out, bufs.lse, None, 0, bufs.err)


def test_multi_full_size_sampled(m):
    """The GQA 4K batch (32 sequences, 32 query / 8 kv heads, 4096 tokens after
    the append) verifying 6 tokens per sequence (5 drafts + 1), sampled units
    against the oracle."""
    n = 6
    w = workload("gqa4k")
    L = w.seq_len
    c = make_contiguous_case(w, DEV)
    q, k, v = new_tokens(w, n, DEV)
    units = [(0, 0), (w.batch - 1, w.h_kv - 1), (17, 3)]
    saved = {(b, j): (c.k_cache[b, j].cpu(), c.v_cache[b, j].cpu()) for b, j in units}
    lay = m.layout_contiguous(c.k_cache, c.v_cache, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, L, num_splits=0, device=DEV, n_new=n)
    m.decode_step_multi(lay, n, q, k, v, (c.seq_lens - n).to(torch.int32), c.seq_lens, L, bufs, w.rope_base,
                        1.0 / math.sqrt(w.head_dim))
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    G = w.group
    for b, j in units:
        K, V = saved[(b, j)]
        ref = oracle.decode_step_multi(K[None, None], V[None, None], q[b:b + 1, :, j * G:(j + 1) * G].cpu(),
                                       k[b:b + 1, :, j:j + 1].cpu(), v[b:b + 1, :, j:j + 1].cpu(), [L], w.rope_base,
                                       1.0 / math.sqrt(w.head_dim), "bf16")
        got = _np(bufs.out[b, :, j * G:(j + 1) * G])
        assert np.max(np.abs(got - ref["out"][0])) <= BF16_TOL, (b, j)
