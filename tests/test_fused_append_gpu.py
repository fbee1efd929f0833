"""GPU: the new token's key row written by the fused decode step is bit for bit
the row the standalone append kernel writes.

The fused kernels turn each key pair in fp32 and redo it in fp64 only when the
fp32 result could round to another bf16 than the fp64 rotation
(rope_k_bf16). These tests feed them many rows whose values cover the cases
that decide between the two: ordinary N(0,1) values, values scaled over most
of the bf16 exponent range, zeros of both signs, bf16 subnormals, pairs with
y = +-x or y = 0, infinities and NaN. Each comparison is against
kv_append_rope, which rotates in fp64 throughout; both must also stay within
one bf16 ulp of the oracle's rounding wherever the oracle's value is finite.
One-byte caches (uint8 codes with per-row scale and zero point, fp8 e5m2):
the fused step of the warp-MMA kernel quantises the new rows itself and must
write the same bytes as the append kernel.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from lse_model import assert_lse
from synthetic import make_contiguous_case, make_e5m2_cache, make_paged_case, make_u8_cache, workload

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def m(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mqa_decode_attention_gb300 as mod

    mod.library()
    return mod


def hard_keys(shape, seed):
    """bf16 key values mixing ordinary, scaled, zero, subnormal and special cases."""
    gen = torch.Generator().manual_seed(seed)
    k = torch.randn(shape, generator=gen, dtype=torch.float64)
    flat = k.view(-1)
    n = flat.numel()
    kind = torch.randint(0, 100, (n,), generator=gen)
    expo = torch.randint(-120, 121, (n,), generator=gen).to(torch.float64)
    flat[:] = torch.where((kind >= 60) & (kind < 72), flat * torch.pow(2.0, expo), flat)
    sub = torch.randint(-127, 128, (n,), generator=gen).to(torch.float64) * 2.0 ** -133  # bf16 subnormals
    flat[:] = torch.where((kind >= 72) & (kind < 77), sub, flat)
    flat[:] = torch.where(kind == 77, torch.zeros_like(flat), flat)
    flat[:] = torch.where(kind == 78, -torch.zeros_like(flat), flat)
    flat[:] = torch.where(kind == 79, torch.full_like(flat, math.inf), flat)
    flat[:] = torch.where(kind == 80, torch.full_like(flat, -math.inf), flat)
    flat[:] = torch.where(kind == 81, torch.full_like(flat, math.nan), flat)
    kb = k.to(torch.bfloat16)
    # pairs (x, y) = (x, +-x) and (x, 0) for some rotation pairs
    pairs = kb.view(-1, 2)
    pk = torch.randint(0, 10, (pairs.shape[0],), generator=gen)
    pairs[pk == 0, 1] = pairs[pk == 0, 0]
    pairs[pk == 1, 1] = -pairs[pk == 1, 0]
    pairs[pk == 2, 1] = 0
    return kb


def bits(t):
    return t.contiguous().view(torch.int16)


def check_against_oracle(k_new, got_rows, pos, base):
    """Each appended element whose oracle value is finite lies within one bf16
    ulp of it (k_new, got_rows: [B, H_kv, d]; pos: [B])."""
    for b in range(k_new.shape[0]):
        with np.errstate(invalid="ignore", over="ignore"):
            want = oracle.rope_rotate(k_new[b].to(torch.float64).numpy(), int(pos[b]), base)
        got = got_rows[b].to(torch.float64).numpy()
        fin = np.isfinite(want) & (np.abs(want) < 3.0e38)
        e = np.floor(np.log2(np.maximum(np.abs(want[fin]), 2.0 ** -126)))
        assert np.all(np.abs(got[fin] - want[fin]) <= 2.0 ** (e - 7)), b


@pytest.mark.parametrize("base", [10000.0, 500000.0])
def test_fused_append_warp_mma_contiguous(m, base):
    w = workload("gqa4k").with_(batch=64, h_q=32, h_kv=8, seed=91)
    lens = torch.randint(1, 2049, (w.batch,), generator=torch.Generator().manual_seed(92), dtype=torch.int32)
    c = make_contiguous_case(w, "cpu", seq_lens=lens, capacity=2048)
    k_new = hard_keys(c.k_new.shape, 93)
    caches = []
    for fused in (True, False):
        kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
        lay = m.layout_contiguous(kc, vc, w.h_q)
        bufs = m.DecodeBuffers.allocate(lay, 2048, num_splits=1, variant=2, device=DEV)
        args = (c.q_new.to(DEV), k_new.to(DEV), c.v_new.to(DEV), c.pos.to(DEV), c.seq_lens.to(DEV))
        if fused:
            m.decode_step(lay, *args, 2048, bufs, base, 0.1, num_splits=1, variant=2)
        else:
            m.kv_append_rope(lay, args[0], args[1], args[2], args[3], base, bufs.q_rot, bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0
        caches.append((kc.cpu(), vc.cpu()))
    assert torch.equal(bits(caches[0][0]), bits(caches[1][0]))
    assert torch.equal(bits(caches[0][1]), bits(caches[1][1]))
    b_idx = torch.arange(w.batch)
    rows = caches[0][0][b_idx, :, c.pos.long()]  # [B, H_kv, d]
    check_against_oracle(k_new, rows, c.pos, base)


def test_fused_append_paged_head_group(m):
    w = workload("paged").with_(batch=48, seed=94)
    lens = torch.randint(1, 1500, (w.batch,), generator=torch.Generator().manual_seed(95), dtype=torch.int32)
    pc = make_paged_case(w, "cpu", seq_lens=lens)
    k_new = hard_keys(pc.k_new.shape, 96)
    pools = []
    for fused in (True, False):
        kp, vp, bt = pc.k_pool.to(DEV), pc.v_pool.to(DEV), pc.block_table.to(DEV)
        lay = m.layout_paged(kp, vp, bt, w.h_q)
        L = int(lens.max())
        bufs = m.DecodeBuffers.allocate(lay, L, num_splits=0, variant=2, device=DEV)
        args = (pc.q_new.to(DEV), k_new.to(DEV), pc.v_new.to(DEV), pc.pos.to(DEV), pc.seq_lens.to(DEV))
        if fused:
            m.decode_step(lay, *args, L, bufs, w.rope_base, 0.1, num_splits=0, variant=2)
        else:
            m.kv_append_rope(lay, args[0], args[1], args[2], args[3], w.rope_base, bufs.q_rot, bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0
        pools.append((kp.cpu(), vp.cpu()))
    assert torch.equal(bits(pools[0][0]), bits(pools[1][0]))
    assert torch.equal(bits(pools[0][1]), bits(pools[1][1]))


def test_fused_append_tc05_mqa(m):
    w = workload("mqa8k").with_(batch=256, seed=97)
    lens = torch.randint(1, 1025, (w.batch,), generator=torch.Generator().manual_seed(98), dtype=torch.int32)
    c = make_contiguous_case(w, "cpu", seq_lens=lens, capacity=1024)
    k_new = hard_keys(c.k_new.shape, 99)
    caches = []
    for fused in (True, False):
        kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
        lay = m.layout_contiguous(kc, vc, w.h_q)
        bufs = m.DecodeBuffers.allocate(lay, 1024, num_splits=0, variant=2, device=DEV)
        args = (c.q_new.to(DEV), k_new.to(DEV), c.v_new.to(DEV), c.pos.to(DEV), c.seq_lens.to(DEV))
        if fused:
            m.decode_step(lay, *args, 1024, bufs, w.rope_base, 0.1, num_splits=0, variant=2)
        else:
            m.kv_append_rope(lay, args[0], args[1], args[2], args[3], w.rope_base, bufs.q_rot, bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0
        caches.append((kc.cpu(), vc.cpu()))
    assert torch.equal(bits(caches[0][0]), bits(caches[1][0]))
    assert torch.equal(bits(caches[0][1]), bits(caches[1][1]))


@pytest.mark.parametrize("cache, h_kv", [("u8", 8), ("fp8", 8), ("u8", 1), ("fp8", 1)])
def test_fused_append_byte_cache(m, cache, h_kv):
    """G = 4 (warp-MMA kernel) and G = 32 (the MQA tcgen05 kernels)."""
    w = workload("gqa4k").with_(batch=48 if h_kv > 1 else 192, h_q=32, h_kv=h_kv, seed=101)
    cap = 1024
    lens = torch.randint(1, cap + 1, (w.batch,), generator=torch.Generator().manual_seed(102), dtype=torch.int32)
    c = make_contiguous_case(w, "cpu", seq_lens=lens, capacity=cap)
    k_new = hard_keys(c.k_new.shape, 103)
    if cache == "u8":
        # finite keys over a wide range (a row's scale comes from its min and max)
        k_new = torch.where(torch.isfinite(k_new.float()), k_new, torch.zeros_like(k_new))
        u = make_u8_cache((w.batch, w.h_kv, cap), w.head_dim, 104)
        tensors = (u.k_codes, u.v_codes, u.k_sz, u.v_sz)
    else:
        kc8, vc8 = make_e5m2_cache((w.batch, w.h_kv, cap), w.head_dim, seed=105)
        tensors = (kc8, vc8)
    results = []
    for fused in (True, False):
        t = [x.clone().to(DEV) for x in tensors]
        if cache == "u8":
            lay = m.layout_contiguous(t[0], t[1], w.h_q, k_scale_zero=t[2], v_scale_zero=t[3])
        else:
            lay = m.layout_contiguous(t[0], t[1], w.h_q)
        bufs = m.DecodeBuffers.allocate(lay, cap, num_splits=1, variant=2, device=DEV)
        args = (c.q_new.to(DEV), k_new.to(DEV), c.v_new.to(DEV), c.pos.to(DEV), c.seq_lens.to(DEV))
        if fused:
            m.decode_step(lay, *args, cap, bufs, w.rope_base, 0.1, num_splits=1, variant=2)
        else:
            m.kv_append_rope(lay, args[0], args[1], args[2], args[3], w.rope_base, bufs.q_rot, bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) & ~int(m.MQA_DEVERR_U8_SCALE) == 0
        results.append(([x.cpu() for x in t], bufs.q_rot.cpu()))
    for a, b in zip(results[0][0], results[1][0]):
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))
    qa, qb = results[0][1], results[1][1]
    assert (qa - qb).abs().max().item() <= 1e-5 * (1 + qb.abs().max().item())


@pytest.mark.parametrize("cache", ["u8", "fp8"])
def test_fused_append_byte_cache_paged(m, cache):
    """Paged one-byte pools (16-token pages, G = 8: the head-group kernel,
    whose producer warp appends the group's rows)."""
    w = workload("paged").with_(batch=40, seed=111)
    lens = torch.randint(1, 1500, (w.batch,), generator=torch.Generator().manual_seed(112), dtype=torch.int32)
    pc = make_paged_case(w, "cpu", seq_lens=lens)
    k_new = hard_keys(pc.k_new.shape, 113)
    rows = (pc.num_pages, w.h_kv, pc.page_size)
    if cache == "u8":
        k_new = torch.where(torch.isfinite(k_new.float()), k_new, torch.zeros_like(k_new))
        u = make_u8_cache(rows, w.head_dim, 114)
        tensors = (u.k_codes, u.v_codes, u.k_sz, u.v_sz)
    else:
        tensors = make_e5m2_cache(rows, w.head_dim, seed=115)
    L = int(lens.max())
    results = []
    for fused in (True, False):
        t = [x.clone().to(DEV) for x in tensors]
        bt = pc.block_table.to(DEV)
        if cache == "u8":
            lay = m.layout_paged(t[0], t[1], bt, w.h_q, k_scale_zero=t[2], v_scale_zero=t[3])
        else:
            lay = m.layout_paged(t[0], t[1], bt, w.h_q)
        bufs = m.DecodeBuffers.allocate(lay, L, num_splits=0, variant=2, device=DEV)
        args = (pc.q_new.to(DEV), k_new.to(DEV), pc.v_new.to(DEV), pc.pos.to(DEV), pc.seq_lens.to(DEV))
        if fused:
            m.decode_step(lay, *args, L, bufs, w.rope_base, 0.1, num_splits=0, variant=2)
        else:
            m.kv_append_rope(lay, args[0], args[1], args[2], args[3], w.rope_base, bufs.q_rot, bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) & ~int(m.MQA_DEVERR_U8_SCALE) == 0
        results.append(([x.cpu() for x in t], bufs.q_rot.cpu()))
    for a, b in zip(results[0][0], results[1][0]):
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))
    qa, qb = results[0][1], results[1][1]
    assert (qa - qb).abs().max().item() <= 1e-5 * (1 + qb.abs().max().item())


def fused_multi_case(m, h_q, h_kv, n, splits, seed):
    """The fused multi-token step against the separate append (cache bits,
    q_rot) and then against the oracle. Sequences whose new rows straddle a
    split boundary (lengths 705.., 1409..) are written by two blocks."""
    w = workload("gqa4k").with_(batch=12, h_q=h_q, h_kv=h_kv, seed=seed)
    cap = 2048
    lens = torch.tensor([705, 706, 707, 1409, 1410, 2048, n, 64 + n - 1, 1000, 129, 700, 1500], dtype=torch.int32)
    c = make_contiguous_case(w, "cpu", seq_lens=lens, capacity=cap)
    gen = torch.Generator().manual_seed(seed + 1)
    q = torch.randn((w.batch, n, w.h_q, w.head_dim), generator=gen).to(torch.bfloat16)
    k = hard_keys((w.batch, n, w.h_kv, w.head_dim), seed + 2)
    v = torch.randn((w.batch, n, w.h_kv, w.head_dim), generator=gen).to(torch.bfloat16)
    pos = (lens - n).to(torch.int32)
    results = []
    for fused in (True, False):
        kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
        lay = m.layout_contiguous(kc, vc, w.h_q)
        bufs = m.DecodeBuffers.allocate(lay, cap, num_splits=splits, variant=2, device=DEV, n_new=n)
        args = (q.to(DEV), k.to(DEV), v.to(DEV), pos.to(DEV))
        if fused:
            m.decode_step_multi(lay, n, *args, lens.to(DEV), cap, bufs, w.rope_base, 0.1, num_splits=splits, variant=2)
        else:
            m.kv_append_rope_multi(lay, n, *args, w.rope_base, bufs.q_rot, bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0
        results.append((kc.cpu(), vc.cpu(), bufs.q_rot.cpu()))
    assert torch.equal(bits(results[0][0]), bits(results[1][0]))
    assert torch.equal(bits(results[0][1]), bits(results[1][1]))
    qa, qb = results[0][2], results[1][2]
    assert (qa - qb).abs().max().item() <= 1e-5 * (1 + qb.abs().max().item())
    # the attention of the fused launch on these boundary cases, with ordinary
    # keys, against the oracle: a block must see the rows that another block
    # appended inside its own token range before it reads them
    k = torch.randn((w.batch, n, w.h_kv, w.head_dim), generator=gen).to(torch.bfloat16)
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, cap, num_splits=splits, variant=2, device=DEV, n_new=n)
    m.decode_step_multi(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), pos.to(DEV), lens.to(DEV), cap, bufs, w.rope_base,
                        1.0 / math.sqrt(w.head_dim), num_splits=splits, variant=2)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16")
    out = bufs.out.double().cpu().numpy().reshape(ref["out"].shape)
    lse = bufs.lse.double().cpu().numpy().reshape(ref["lse"].shape)
    assert np.max(np.abs(out - ref["out"])) <= 2e-2
    assert np.max(np.abs(lse - ref["lse"])) <= 2e-2
    assert_lse(lse, ref["q_rot"], ref["k_cache"], lens, 1.0 / math.sqrt(w.head_dim), "bf16")


@pytest.mark.parametrize("n", [2, 4, 7])
@pytest.mark.parametrize("splits", [1, 3])
def test_fused_append_multi_token(m, n, splits):
    """Several new tokens per sequence on the warp-MMA kernel (G n < 32)."""
    fused_multi_case(m, 32, 8, n, splits, 121 + n)


@pytest.mark.parametrize("h_q, h_kv, n", [(32, 8, 8), (32, 8, 16), (64, 8, 16), (32, 1, 2), (32, 1, 4)],
                         ids=lambda v: str(v))
@pytest.mark.parametrize("splits", [1, 2, 3])
def test_fused_append_multi_token_tc05(m, h_q, h_kv, n, splits):
    """Several new tokens per sequence on the tcgen05 kernel (32 <= G n <=
    128, n <= 16: one launch, the kernel's append warp writing the rows of its
    split; G n <= 64 at two splits merges them in a two-block cluster)."""
    fused_multi_case(m, h_q, h_kv, n, splits, 131 + n + h_q)


@pytest.mark.parametrize("page_size, n, splits", [(16, 8, 1), (16, 8, 3), (32, 16, 2), (256, 4, 3), (64, 2, 2)])
def test_fused_append_multi_token_tc05_paged(m, page_size, n, splits):
    """The fused multi-token step over a paged pool (tcgen05 kernel): every
    pool byte equals what kv_append_rope_multi writes, new rows crossing page
    and split boundaries alike."""
    h_q, h_kv = (32, 1) if n <= 4 else (32, 8)
    w = workload("paged").with_(batch=6, h_q=h_q, h_kv=h_kv, page_size=page_size, seed=141 + n + page_size)
    lens = torch.tensor([705, 706, 1409, n, 64 + n - 1, 1000], dtype=torch.int32)
    pc = make_paged_case(w, "cpu", seq_lens=lens, spare_pages=2)
    gen = torch.Generator().manual_seed(142 + n)
    q = torch.randn((w.batch, n, w.h_q, w.head_dim), generator=gen).to(torch.bfloat16)
    k = hard_keys((w.batch, n, w.h_kv, w.head_dim), 143 + n)
    v = torch.randn((w.batch, n, w.h_kv, w.head_dim), generator=gen).to(torch.bfloat16)
    pos = (lens - n).to(torch.int32)
    bt = pc.block_table.to(DEV)
    cap = int(lens.max())
    results = []
    for fused in (True, False):
        kp, vp = pc.k_pool.to(DEV), pc.v_pool.to(DEV)
        lay = m.layout_paged(kp, vp, bt, w.h_q)
        if fused:
            assert m.step_launches(lay, cap, splits, 2, n)[1], "the step should append inside the attention launch"
        bufs = m.DecodeBuffers.allocate(lay, cap, num_splits=splits, variant=2, device=DEV, n_new=n)
        args = (q.to(DEV), k.to(DEV), v.to(DEV), pos.to(DEV))
        if fused:
            m.decode_step_multi(lay, n, *args, lens.to(DEV), cap, bufs, w.rope_base, 0.1, num_splits=splits, variant=2)
        else:
            m.kv_append_rope_multi(lay, n, *args, w.rope_base, bufs.q_rot, bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0
        results.append((kp.cpu(), vp.cpu()))
    assert torch.equal(bits(results[0][0]), bits(results[1][0]))
    assert torch.equal(bits(results[0][1]), bits(results[1][1]))
