"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances: bf16 outputs max |err| <= 2e-2, fp32 (debug) outputs <= 1e-4.
The fp32 lse outputs: <= 1e-4 of the oracle's log-sum-exp over the scores the
kernel forms (its query rounded to the MMA operand type, tests/lse_model.py),
and <= 2e-2 of the oracle's exact lse.
Cache-append placement is bit-exact (the set of changed elements is exactly
the oracle's target slots, V slices are byte copies); an appended K element
may differ from round-to-nearest of the fp64 RoPE by at most one bf16 ulp.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from lse_model import assert_lse, paged_keys
from synthetic import (make_contiguous_case, make_paged_case, make_tiny_sequence, workload)

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
F32_TOL = 1e-4
VARIANTS = {"tc": 2, "cc": 1}
Q_FMT = {"tc": "bf16", "cc": "f32", 2: "bf16", 1: "f32", 0: "bf16"}  # the query operand of each bf16-cache path


@pytest.fixture(scope="module")
def m(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mqa_decode_attention_gb300 as mod

    mod.library()
    return mod


DEV = "cuda"


def _np(t):
    return t.detach().cpu().to(torch.float64).numpy()


def ulp_bf16(x):
    """Spacing of bfloat16 numbers at |x| (normal range)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def run_contiguous(m, c, w, splits=0, variant=0, out_dtype=None, max_len=None):
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    max_len = int(c.seq_lens.max()) if max_len is None else max_len
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=splits, variant=variant, out_dtype=out_dtype, device=DEV)
    m.decode_step(lay, c.q_new.to(DEV), c.k_new.to(DEV), c.v_new.to(DEV), c.pos.to(DEV), c.seq_lens.to(DEV),
                  max_len, bufs, w.rope_base, 1.0 / math.sqrt(w.head_dim), num_splits=splits, variant=variant)
    torch.cuda.synchronize()
    return dict(out=_np(bufs.out), lse=_np(bufs.lse), q_rot=_np(bufs.q_rot), k=kc.cpu(), v=vc.cpu(),
                err=int(bufs.err.item()))


def run_paged(m, pc, w, splits=0, variant=0, out_dtype=None):
    kp, vp, bt = pc.k_pool.to(DEV), pc.v_pool.to(DEV), pc.block_table.to(DEV)
    lay = m.layout_paged(kp, vp, bt, w.h_q)
    max_len = int(pc.seq_lens.max())
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=splits, variant=variant, out_dtype=out_dtype, device=DEV)
    m.decode_step(lay, pc.q_new.to(DEV), pc.k_new.to(DEV), pc.v_new.to(DEV), pc.pos.to(DEV), pc.seq_lens.to(DEV),
                  max_len, bufs, w.rope_base, 1.0 / math.sqrt(w.head_dim), num_splits=splits, variant=variant)
    torch.cuda.synchronize()
    return dict(out=_np(bufs.out), lse=_np(bufs.lse), q_rot=_np(bufs.q_rot), k=kp.cpu(), v=vp.cpu(),
                err=int(bufs.err.item()))


def check_append(before_k, before_v, after_k, after_v, ref_k, ref_v, cache_dtype):
    """Only the target slots changed; V there is a byte copy; K within 1 ulp of the oracle."""
    bk, bv = _np(before_k), _np(before_v)
    ak, av = _np(after_k), _np(after_v)
    changed_ref = (ref_k != bk) | (ref_v != bv)
    changed_gpu = (ak != bk) | (av != bv)
    # rows (all but the last axis) the oracle writes must be the only rows the GPU writes
    rows_ref = np.any(changed_ref, axis=-1)
    rows_gpu = np.any(changed_gpu, axis=-1)
    assert not np.any(rows_gpu & ~rows_ref), "GPU wrote outside the target slots"
    assert np.array_equal(av, ref_v), "V slot is not a byte copy of v_new"
    diff = np.abs(ak - ref_k)
    tol = ulp_bf16(ref_k) if cache_dtype == "bf16" else np.abs(ref_k) * 2.0 ** -23
    assert np.all(diff <= tol), f"K slot off by more than 1 ulp: {np.max(diff / np.maximum(tol, 1e-300))}"


# --------------------------------------------------------------- small cases
SHAPES = [
    # (batch, h_q, h_kv, head_dim, lens, capacity)
    (3, 8, 2, 128, [200, 65, 1], 256),       # GQA G=4, ragged tails, L=1
    (2, 4, 4, 64, [63, 64], 64),             # MHA, d=64, L at capacity
    (2, 32, 1, 128, [300, 129], 320),        # MQA G=32 (two head blocks of 16)
    (1, 12, 4, 128, [1000], 1024),           # G=3 (padded head rows)
    (2, 16, 2, 128, [130, 7], 130),          # G=8
    (1, 96, 1, 64, [77], 80),                # G=96: several head super-blocks
]


@pytest.mark.parametrize("variant", ["tc", "cc"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s[0]}q{s[1]}kv{s[2]}d{s[3]}")
@pytest.mark.parametrize("splits", [1, 2, 7, 0])
def test_contiguous_matches_oracle(m, variant, shape, splits):
    B, hq, hkv, d, lens, cap = shape
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, head_dim=d, seed=100 + B + hq + d)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=cap)
    ref = oracle.decode_step_contiguous(c.k_cache, c.v_cache, c.q_new, c.k_new, c.v_new, c.seq_lens, w.rope_base,
                                        1.0 / math.sqrt(d), "bf16")
    got = run_contiguous(m, c, w, splits=splits, variant=VARIANTS[variant])
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= BF16_TOL
    assert_lse(got["lse"], ref["q_rot"], ref["k_cache"], c.seq_lens, 1.0 / math.sqrt(d), Q_FMT[variant])
    assert np.max(np.abs(got["q_rot"] - ref["q_rot"])) <= 1e-5 * (1 + np.max(np.abs(ref["q_rot"])))
    check_append(c.k_cache, c.v_cache, got["k"], got["v"], ref["k_cache"], ref["v_cache"], "bf16")


@pytest.mark.parametrize("variant", ["tc", "cc"])
@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("heads", [(16, 2), (32, 8), (12, 3), (64, 2)], ids=lambda h: f"q{h[0]}kv{h[1]}")
def test_paged_matches_oracle(m, variant, page_size, heads):
    """Covers the head-group paged kernel (16-token pages, kv heads in groups of
    2 or 4, G <= 16) and the per-head kernel (other page sizes, odd kv head
    counts, G > 16)."""
    if heads != (16, 2) and page_size not in (16, 64):
        pytest.skip("page-size sweep runs on the first head layout")
    w = workload("paged").with_(batch=5, h_q=heads[0], h_kv=heads[1], page_size=page_size, len_lo=1, len_hi=700,
                                seed=9)
    lens = torch.tensor([1, 16, 17, 700, 333], dtype=torch.int32)
    pc = make_paged_case(w, "cpu", seq_lens=lens, spare_pages=3)
    ref = oracle.decode_step_paged(pc.k_pool, pc.v_pool, pc.block_table, pc.q_new, pc.k_new, pc.v_new,
                                   pc.seq_lens, pc.page_size, w.rope_base, 1.0 / math.sqrt(w.head_dim), "bf16")
    keys = paged_keys(ref["k_pool"], pc.block_table, pc.seq_lens, pc.page_size)
    for splits in (1, 3, 0):
        got = run_paged(m, pc, w, splits=splits, variant=VARIANTS[variant])
        assert got["err"] == 0
        assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL
        assert np.max(np.abs(got["lse"] - ref["lse"])) <= BF16_TOL
        assert_lse(got["lse"], ref["q_rot"], keys, pc.seq_lens, 1.0 / math.sqrt(w.head_dim), Q_FMT[variant],
                   what=splits)
        check_append(pc.k_pool, pc.v_pool, got["k"], got["v"], ref["k_pool"], ref["v_pool"], "bf16")


def test_shared_pages_read_path(m):
    """Two sequences whose tables point at the same physical pages (copy-on-write
    prefix sharing) read the same data; appends go to private last pages."""
    w = workload("paged").with_(batch=2, h_q=8, h_kv=2, seed=21)
    lens = torch.tensor([40, 40], dtype=torch.int32)
    pc = make_paged_case(w, "cpu", seq_lens=lens, spare_pages=0)
    table = pc.block_table.clone()
    table[1, :2] = table[0, :2]  # shared prefix pages 0..31 tokens
    pc.block_table = table
    ref = oracle.decode_step_paged(pc.k_pool, pc.v_pool, table, pc.q_new, pc.k_new, pc.v_new, pc.seq_lens,
                                   pc.page_size, w.rope_base, 1.0 / math.sqrt(w.head_dim), "bf16")
    got = run_paged(m, pc, w, splits=1, variant=2)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL


def test_fp32_output_mode_tight(m):
    """bf16 cache with fp32 output on CUDA cores: only fp32 rounding remains."""
    w = workload("gqa4k").with_(batch=2, h_q=8, h_kv=2, seed=5)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor([129, 64], dtype=torch.int32), capacity=130)
    ref = oracle.decode_step_contiguous(c.k_cache, c.v_cache, c.q_new, c.k_new, c.v_new, c.seq_lens, w.rope_base,
                                        1.0 / math.sqrt(w.head_dim), "bf16")
    got = run_contiguous(m, c, w, splits=2, variant=1, out_dtype=torch.float32)
    assert np.max(np.abs(got["out"] - ref["out"])) <= F32_TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= F32_TOL


# ----------------------------------------------------- fp32 debug sequence
def test_tiny_fp32_sequence_matches_oracle_and_recomputation(m):
    """The tiny workload token by token: prompt P=5 then decoding until T=16
    attention evaluations (queries at positions 4..19), fp32 cache and output,
    CUDA-core path."""
    w = workload("tiny")
    seq = make_tiny_sequence(w)
    scale = 1.0 / math.sqrt(w.head_dim)
    n = seq.prompt_len + seq.decode_evals - 1
    ref_out, ref_lse, n_proj, _ = oracle.run_cached_sequence(seq.q, seq.k, seq.v, seq.prompt_len, seq.decode_evals,
                                                             w.rope_base, scale, "f32")
    brute, _, _ = oracle.run_uncached_sequence(seq.q, seq.k, seq.v, seq.prompt_len, seq.decode_evals, w.rope_base,
                                               scale)
    kc = torch.zeros(w.batch, w.h_kv, n, w.head_dim, dtype=torch.float32, device=DEV)
    vc = torch.zeros_like(kc)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, n, num_splits=1, variant=1, device=DEV)
    outs = []
    for p in range(n):
        lens = torch.full((w.batch,), p + 1, dtype=torch.int32, device=DEV)
        m.decode_step(lay, seq.q[p].to(DEV), seq.k[p].to(DEV), seq.v[p].to(DEV), lens - 1, lens, p + 1, bufs,
                      w.rope_base, scale, num_splits=1, variant=1)
        if p >= seq.prompt_len - 1:
            outs.append(_np(bufs.out))
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    got = np.stack(outs)
    assert got.shape == ref_out.shape
    assert np.max(np.abs(got - ref_out)) <= F32_TOL
    assert np.max(np.abs(got - brute)) <= F32_TOL
    assert n_proj == 20  # one K/V projection per position with the cache


# ----------------------------------------------------------- combine, splits
def test_splitkv_combine_matches_oracle(m):
    rng = np.random.default_rng(4)
    B, hq, d, S = 3, 8, 128, 9
    o = rng.standard_normal((B, hq, S, d)).astype(np.float32)
    lse = (rng.standard_normal((B, hq, S)) * 3).astype(np.float32)
    lse[0, 0, :4] = -np.inf  # empty splits
    lse[1, 2, 5] = -np.inf
    out = torch.empty(B, hq, d, dtype=torch.float32, device=DEV)
    lse_out = torch.empty(B, hq, dtype=torch.float32, device=DEV)
    m.splitkv_combine(torch.from_numpy(o).to(DEV), torch.from_numpy(lse).to(DEV), out, lse_out)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.lse_combine(np.moveaxis(o.astype(np.float64), 2, 0), np.moveaxis(lse.astype(np.float64), 2, 0))
    assert np.max(np.abs(_np(out) - ref_o)) <= 1e-5
    assert np.max(np.abs(_np(lse_out) - ref_l)) <= 1e-5


def test_split_counts_agree(m):
    w = workload("gqa4k").with_(batch=2, h_q=8, h_kv=2, seed=33)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor([4096, 1500], dtype=torch.int32), capacity=4096)
    outs = [run_contiguous(m, c, w, splits=s, variant=2, out_dtype=torch.float32)["out"] for s in (1, 2, 7, 64)]
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= 1e-3


# ------------------------------------------------------------- error words
def test_append_position_out_of_range_sets_error_and_skips(m):
    w = workload("gqa4k").with_(batch=2, h_q=8, h_kv=2, seed=3)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor([64, 64], dtype=torch.int32), capacity=64)
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    k0, v0 = kc.clone(), vc.clone()
    lay = m.layout_contiguous(kc, vc, w.h_q)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    q_rot = torch.empty(2, 8, 128, dtype=torch.float32, device=DEV)
    pos = torch.tensor([64, -1], dtype=torch.int32, device=DEV)  # both outside [0, capacity)
    m.kv_append_rope(lay, c.q_new.to(DEV), c.k_new.to(DEV), c.v_new.to(DEV), pos, 10000.0, q_rot, err)
    torch.cuda.synchronize()
    assert int(err.item()) & m.MQA_DEVERR_POS_RANGE
    assert torch.equal(kc, k0) and torch.equal(vc, v0)


def test_bad_block_table_entries_set_error(m):
    w = workload("paged").with_(batch=2, h_q=8, h_kv=2, seed=8)
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor([100, 40], dtype=torch.int32))
    bt = pc.block_table.clone()
    bt[0, 6] = pc.num_pages + 5  # page of the appended token (pos 99 -> logical page 6)
    bt[1, 0] = -7                # a page the attention reads
    kp, vp, btd = pc.k_pool.to(DEV), pc.v_pool.to(DEV), bt.to(DEV)
    k0 = kp.clone()
    lay = m.layout_paged(kp, vp, btd, w.h_q)
    for variant in (1, 2):
        bufs = m.DecodeBuffers.allocate(lay, 100, num_splits=1, variant=variant, device=DEV)
        m.decode_step(lay, pc.q_new.to(DEV), pc.k_new.to(DEV), pc.v_new.to(DEV), pc.pos.to(DEV),
                      pc.seq_lens.to(DEV), 100, bufs, num_splits=1, variant=variant)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) & m.MQA_DEVERR_PAGE_RANGE
    # sequence 0's append was skipped; sequence 1's append landed in its own page
    changed = (kp != k0).any(dim=-1).nonzero().tolist()
    assert all(int(bt[1, 39 // 16]) == row[0] for row in changed)


def test_bad_lengths_set_error(m):
    w = workload("gqa4k").with_(batch=2, h_q=8, h_kv=2, seed=2)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor([64, 64], dtype=torch.int32), capacity=64)
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    for variant in (1, 2):
        bufs = m.DecodeBuffers.allocate(lay, 64, num_splits=1, variant=variant, device=DEV)
        bufs.q_rot.zero_()
        lens = torch.tensor([0, 70], dtype=torch.int32, device=DEV)  # empty and beyond max_seq_len
        m.gqa_decode_attention(lay, bufs.q_rot, lens, 64, 0.1, 1, bufs.out, bufs.lse, None, variant, bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) & m.MQA_DEVERR_SEQ_LEN
        assert torch.isfinite(bufs.out.float()).all()


def test_host_status_is_raised(m):
    w = workload("gqa4k").with_(batch=1, h_q=8, h_kv=2)
    kc = torch.zeros(1, 2, 256, 128, dtype=torch.bfloat16, device=DEV)
    lay = m.layout_contiguous(kc, kc.clone(), 8)
    out = torch.empty(1, 8, 128, dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    q = torch.zeros(1, 8, 128, device=DEV)
    lens = torch.ones(1, dtype=torch.int32, device=DEV)
    with pytest.raises(m.MqaError):
        m.gqa_decode_attention(lay, q, lens, 256, 0.1, 4, out, None, None, 0, err)  # split without workspace


# ------------------------------------------------- full-size workloads
def _full_contiguous(m, name, n_samples=6):
    w = workload(name)
    gen = torch.Generator().manual_seed(w.seed)
    c = make_contiguous_case(w, DEV)
    L = w.seq_len
    G = w.group
    samples = sorted({(int(torch.randint(0, w.batch, (1,), generator=gen)), int(torch.randint(0, w.h_kv, (1,),
                                                                                                generator=gen)))
                      for _ in range(n_samples)} | {(w.batch - 1, w.h_kv - 1), (0, 0)})
    saved = {(b, j): (c.k_cache[b, j, :L].cpu(), c.v_cache[b, j, :L].cpu()) for b, j in samples}
    lay = m.layout_contiguous(c.k_cache, c.v_cache, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, L, num_splits=w.num_splits, device=DEV)
    m.decode_step(lay, c.q_new, c.k_new, c.v_new, c.pos, c.seq_lens, L, bufs, w.rope_base,
                  1.0 / math.sqrt(w.head_dim), num_splits=w.num_splits)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    out = bufs.out.float()
    assert torch.isfinite(out).all()
    q_new, k_new, v_new = c.q_new.cpu(), c.k_new.cpu(), c.v_new.cpu()
    for (b, j), (Ku, Vu) in saved.items():
        ro, rl, ks = oracle.decode_unit(q_new[b, j * G:(j + 1) * G], k_new[b, j], v_new[b, j], Ku, Vu, L, w.rope_base,
                                        1.0 / math.sqrt(w.head_dim), "bf16")
        assert np.max(np.abs(_np(bufs.out[b, j * G:(j + 1) * G]) - ro)) <= BF16_TOL, (b, j)
        assert np.max(np.abs(_np(bufs.lse[b, j * G:(j + 1) * G]) - rl)) <= BF16_TOL, (b, j)
        keys = _np(Ku)[None, None].copy()
        keys[0, 0, L - 1] = ks
        assert_lse(_np(bufs.lse[b, j * G:(j + 1) * G])[None],
                   oracle.rope_rotate(_np(q_new[b, j * G:(j + 1) * G]), L - 1, w.rope_base)[None], keys, [L],
                   1.0 / math.sqrt(w.head_dim), "bf16", what=(b, j))
        got_k = _np(c.k_cache[b, j, L - 1])
        assert np.all(np.abs(got_k - ks) <= ulp_bf16(ks))
        assert torch.equal(c.v_cache[b, j, L - 1].cpu(), v_new[b, j])
    # any size: each output is a convex combination of the values it read
    vmax = c.v_cache[:, :, :L].abs().amax(dim=2).float()  # [B, H_kv, d]
    bound = vmax.repeat_interleave(G, dim=1)
    assert (out.abs() <= bound * (1 + 2 ** -7) + 1e-6).all()


@pytest.mark.parametrize("name", ["gqa4k", "mqa8k", "long"])
def test_full_size_contiguous_sampled(m, name):
    _full_contiguous(m, name)


def test_full_size_paged_sampled(m):
    w = workload("paged")
    pc = make_paged_case(w, DEV)
    lens = pc.seq_lens.cpu()
    G = w.group
    gen = torch.Generator().manual_seed(w.seed)
    samples = {(int(torch.argmax(lens)), 3), (int(torch.argmin(lens)), 0)}
    samples |= {(int(torch.randint(0, w.batch, (1,), generator=gen)), int(torch.randint(0, w.h_kv, (1,),
                                                                                         generator=gen)))
                for _ in range(4)}
    table = pc.block_table.cpu()
    saved = {}
    for b, j in samples:
        n = (int(lens[b]) + w.page_size - 1) // w.page_size
        pages = table[b, :n]
        saved[(b, j)] = (pages, pc.k_pool[pages.to(DEV).long(), j].cpu(), pc.v_pool[pages.to(DEV).long(), j].cpu())
    lay = m.layout_paged(pc.k_pool, pc.v_pool, pc.block_table, w.h_q)
    max_len = int(lens.max())
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=w.num_splits, device=DEV)
    m.decode_step(lay, pc.q_new, pc.k_new, pc.v_new, pc.pos, pc.seq_lens, max_len, bufs, w.rope_base,
                  1.0 / math.sqrt(w.head_dim), num_splits=w.num_splits)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    assert torch.isfinite(bufs.out.float()).all()
    q_new, k_new, v_new = pc.q_new.cpu(), pc.k_new.cpu(), pc.v_new.cpu()
    for (b, j), (pages, kpg, vpg) in saved.items():
        # a small pool holding this unit's pages in physical order, table remapped to it
        order = torch.argsort(pages)
        small_k = kpg[order][:, None]  # [n, 1, ps, d]
        small_v = vpg[order][:, None]
        rank = torch.empty_like(order)
        rank[order] = torch.arange(len(order))
        r = oracle.decode_step_paged(small_k, small_v, rank[None], q_new[b:b + 1, j * G:(j + 1) * G],
                                     k_new[b:b + 1, j:j + 1], v_new[b:b + 1, j:j + 1], lens[b:b + 1], w.page_size,
                                     w.rope_base, 1.0 / math.sqrt(w.head_dim), "bf16")
        assert np.max(np.abs(_np(bufs.out[b, j * G:(j + 1) * G]) - r["out"][0])) <= BF16_TOL, (b, j)
        assert np.max(np.abs(_np(bufs.lse[b, j * G:(j + 1) * G]) - r["lse"][0])) <= BF16_TOL, (b, j)
        assert_lse(_np(bufs.lse[b, j * G:(j + 1) * G])[None], r["q_rot"],
                   paged_keys(r["k_pool"], rank[None], lens[b:b + 1], w.page_size), lens[b:b + 1],
                   1.0 / math.sqrt(w.head_dim), "bf16", what=(b, j))
        p = int(lens[b]) - 1
        page = int(table[b, p // w.page_size])
        got_k = _np(pc.k_pool[page, j, p % w.page_size])
        want_k = r["k_pool"][int(rank[p // w.page_size]), 0, p % w.page_size]
        assert np.all(np.abs(got_k - want_k) <= ulp_bf16(want_k))


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("paged", [False, True])
def test_fused_step_equals_separate_calls(m, variant, paged):
    """mqa_decode_step (append, then attention started early) gives exactly the
    result of kv_append_rope followed by gqa_decode_attention."""
    w = workload("paged" if paged else "gqa4k").with_(batch=3, h_q=16, h_kv=4, seed=44)
    lens = torch.tensor([700, 1, 129], dtype=torch.int32)
    outs = []
    for fused in (True, False):
        if paged:
            c = make_paged_case(w, "cpu", seq_lens=lens)
            kc, vc, bt = c.k_pool.to(DEV), c.v_pool.to(DEV), c.block_table.to(DEV)
            lay = m.layout_paged(kc, vc, bt, w.h_q)
        else:
            c = make_contiguous_case(w, "cpu", seq_lens=lens, capacity=704)
            kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
            lay = m.layout_contiguous(kc, vc, w.h_q)
        bufs = m.DecodeBuffers.allocate(lay, 700, num_splits=3, variant=variant, device=DEV)
        args = (c.q_new.to(DEV), c.k_new.to(DEV), c.v_new.to(DEV), c.pos.to(DEV), c.seq_lens.to(DEV))
        if fused:
            m.decode_step(lay, *args, 700, bufs, w.rope_base, 0.1, num_splits=3, variant=variant)
        else:
            m.kv_append_rope(lay, args[0], args[1], args[2], args[3], w.rope_base, bufs.q_rot, bufs.err)
            m.gqa_decode_attention(lay, bufs.q_rot, args[4], 700, 0.1, 3, bufs.out, bufs.lse, bufs.workspace,
                                   variant, bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0
        outs.append((bufs.out.clone(), bufs.lse.clone(), kc.clone(), vc.clone(), bufs.q_rot.clone()))
    # the fused step appends and rotates q inside the tensor-core kernel (same
    # formulas as the append kernel): the cache is bit-identical, q_rot and the
    # outputs agree to fp32 / bf16 rounding
    assert (outs[0][0].float() - outs[1][0].float()).abs().max().item() <= 1e-2
    assert (outs[0][1] - outs[1][1]).abs().max().item() <= 1e-3
    assert torch.equal(outs[0][2], outs[1][2]) and torch.equal(outs[0][3], outs[1][3])
    assert (outs[0][4] - outs[1][4]).abs().max().item() <= 1e-5 * (1 + outs[1][4].abs().max().item())


# ---------------------------------------------------------- sliding window
@pytest.mark.parametrize("variant", [2, 1])
@pytest.mark.parametrize("window", [1, 7, 16, 17, 100, 1000])
def test_sliding_window_contiguous(m, variant, window):
    w = workload("gqa4k").with_(batch=3, h_q=16, h_kv=4, seed=61)
    lens = torch.tensor([700, 65, 3], dtype=torch.int32)
    c = make_contiguous_case(w, "cpu", seq_lens=lens, capacity=704)
    ref = oracle.decode_step_contiguous(c.k_cache, c.v_cache, c.q_new, c.k_new, c.v_new, c.seq_lens, w.rope_base,
                                        1.0 / math.sqrt(w.head_dim), "bf16", window=window)
    for splits in (1, 3, 0):
        kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
        lay = m.layout_contiguous(kc, vc, w.h_q, window=window)
        bufs = m.DecodeBuffers.allocate(lay, 700, num_splits=splits, variant=variant, device=DEV)
        m.decode_step(lay, c.q_new.to(DEV), c.k_new.to(DEV), c.v_new.to(DEV), c.pos.to(DEV), c.seq_lens.to(DEV),
                      700, bufs, w.rope_base, 1.0 / math.sqrt(w.head_dim), num_splits=splits, variant=variant)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0
        assert np.max(np.abs(_np(bufs.out) - ref["out"])) <= BF16_TOL, (splits, window)
        assert np.max(np.abs(_np(bufs.lse) - ref["lse"])) <= BF16_TOL
        assert_lse(_np(bufs.lse), ref["q_rot"], ref["k_cache"], c.seq_lens, 1.0 / math.sqrt(w.head_dim),
                   Q_FMT[variant], window=window, what=splits)


@pytest.mark.parametrize("variant", [2, 1])
@pytest.mark.parametrize("h_kv", [4, 3])
@pytest.mark.parametrize("window", [1, 15, 16, 33, 300])
def test_sliding_window_paged_with_released_pages(m, variant, h_kv, window):
    """Pages wholly before the window are released (table entry -1): no error,
    and the result equals the oracle's windowed attention."""
    w = workload("paged").with_(batch=4, h_q=4 * h_kv, h_kv=h_kv, seed=62)
    lens = torch.tensor([700, 64, 17, 1], dtype=torch.int32)
    pc = make_paged_case(w, "cpu", seq_lens=lens)
    ref = oracle.decode_step_paged(pc.k_pool, pc.v_pool, pc.block_table, pc.q_new, pc.k_new, pc.v_new, pc.seq_lens,
                                   pc.page_size, w.rope_base, 1.0 / math.sqrt(w.head_dim), "bf16", window=window)
    keys = paged_keys(ref["k_pool"], pc.block_table, pc.seq_lens, pc.page_size)
    table = pc.block_table.clone()
    for b in range(w.batch):
        t_lo = max(0, int(lens[b]) - window)
        table[b, :t_lo // pc.page_size] = -1
    for splits in (1, 3, 0):
        kp, vp, bt = pc.k_pool.to(DEV), pc.v_pool.to(DEV), table.to(DEV)
        lay = m.layout_paged(kp, vp, bt, w.h_q, window=window)
        bufs = m.DecodeBuffers.allocate(lay, 700, num_splits=splits, variant=variant, device=DEV)
        m.decode_step(lay, pc.q_new.to(DEV), pc.k_new.to(DEV), pc.v_new.to(DEV), pc.pos.to(DEV),
                      pc.seq_lens.to(DEV), 700, bufs, w.rope_base, 1.0 / math.sqrt(w.head_dim), num_splits=splits,
                      variant=variant)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0, (splits, int(bufs.err.item()))
        assert np.max(np.abs(_np(bufs.out) - ref["out"])) <= BF16_TOL, (splits, window)
        assert_lse(_np(bufs.lse), ref["q_rot"], keys, pc.seq_lens, 1.0 / math.sqrt(w.head_dim), Q_FMT[variant],
                   window=window, what=splits)


def test_sliding_window_full_size_long(m):
    """131072-token sequences with a 4096-token window (Mistral's W): sampled
    units against the oracle."""
    w = workload("long")
    W = 4096
    c = make_contiguous_case(w, DEV)
    L = w.seq_len
    G = w.group
    units = [(0, 0), (3, 7), (2, 4)]
    saved = {(b, j): (c.k_cache[b, j, L - W:L].cpu(), c.v_cache[b, j, L - W:L].cpu()) for b, j in units}
    lay = m.layout_contiguous(c.k_cache, c.v_cache, w.h_q, window=W)
    bufs = m.DecodeBuffers.allocate(lay, L, num_splits=0, device=DEV)
    m.decode_step(lay, c.q_new, c.k_new, c.v_new, c.pos, c.seq_lens, L, bufs, w.rope_base,
                  1.0 / math.sqrt(w.head_dim), num_splits=0)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    q_new, k_new, v_new = c.q_new.cpu(), c.k_new.cpu(), c.v_new.cpu()
    for (b, j), (Ku, Vu) in saved.items():
        # the unit seen from the window's start: positions keep their absolute values
        ro, rl, _ = oracle.decode_unit(q_new[b, j * G:(j + 1) * G], k_new[b, j], v_new[b, j],
                                       torch.cat([torch.zeros(L - W, w.head_dim, dtype=Ku.dtype), Ku]),
                                       torch.cat([torch.zeros(L - W, w.head_dim, dtype=Vu.dtype), Vu]), L,
                                       w.rope_base, 1.0 / math.sqrt(w.head_dim), "bf16", window=W)
        assert np.max(np.abs(_np(bufs.out[b, j * G:(j + 1) * G]) - ro)) <= BF16_TOL
