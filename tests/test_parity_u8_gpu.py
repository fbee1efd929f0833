"""GPU parity of the uint8 KV cache (MQA_U8) against the fp64 oracle.

The oracle quantises the new token's rotated key and its value in float32 (the
pages' QuantizedKVCache) and attends over the dequantised cache in fp64. The
append is integer / byte work and must match exactly: codes, scale and zero
point of the appended rows, and nothing else in the caches changes. Outputs
are bf16, max |err| <= 2e-2 like the bf16 cache path. The fp32 lse is held to
the log-sum-exp over the scores the kernels form (their fp16 query operand)
within 1e-4 plus a bound on the zero-point cancellation of the warp-MMA
kernel's score form (tests/lse_model.py).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from lse_model import assert_lse, paged_keys
from synthetic import make_contiguous_case, make_paged_case, make_u8_cache, workload

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


def _contiguous(w, lens, cap, seed):
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=cap)
    u = make_u8_cache((w.batch, w.h_kv, cap), w.head_dim, seed)
    return c, u


def _paged(w, lens, seed):
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=2)
    u = make_u8_cache((pc.num_pages, w.h_kv, pc.page_size), w.head_dim, seed)
    return pc, u


def run_u8(m, w, case, u, paged, splits=0, window=0, table=None, max_len=None):
    kc, vc = u.k_codes.to(DEV), u.v_codes.to(DEV)
    ks, vs = u.k_sz.to(DEV), u.v_sz.to(DEV)
    if paged:
        bt = (case.block_table if table is None else table).to(DEV)
        lay = m.layout_paged(kc, vc, bt, w.h_q, window=window, k_scale_zero=ks, v_scale_zero=vs)
    else:
        lay = m.layout_contiguous(kc, vc, w.h_q, window=window, k_scale_zero=ks, v_scale_zero=vs)
    max_len = int(case.seq_lens.max()) if max_len is None else max_len
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=splits, device=DEV)
    m.decode_step(lay, case.q_new.to(DEV), case.k_new.to(DEV), case.v_new.to(DEV), case.pos.to(DEV),
                  case.seq_lens.to(DEV), max_len, bufs, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                  num_splits=splits)
    torch.cuda.synchronize()
    return dict(out=_np(bufs.out), lse=_np(bufs.lse), q_rot=_np(bufs.q_rot), err=int(bufs.err.item()),
                k_codes=kc.cpu().numpy(), v_codes=vc.cpu().numpy(), k_sz=ks.cpu().numpy(), v_sz=vs.cpu().numpy())


def _oracle(w, case, u, paged, window=0):
    if paged:
        return oracle.decode_step_u8(u.k_codes, u.k_sz, u.v_codes, u.v_sz, case.q_new, case.k_new, case.v_new,
                                     case.seq_lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                     block_table=case.block_table,
                                     page_size=case.page_size, window=window)
    return oracle.decode_step_u8(u.k_codes, u.k_sz, u.v_codes, u.v_sz, case.q_new, case.k_new, case.v_new,
                                 case.seq_lens, w.rope_base, 1.0 / math.sqrt(w.head_dim), window=window)


def check_u8_lse(got, ref, case, paged=False, window=0, what=None):
    """lse against the model over the dequantised keys the kernel reads."""
    kd = oracle.dequantize_u8(ref["k_codes"], ref["k_sz"][..., 0], ref["k_sz"][..., 1])
    ks = np.asarray(ref["k_sz"][..., :1], np.float64)
    if paged:
        kd = paged_keys(kd, case.block_table, case.seq_lens, case.page_size)
        ks = paged_keys(ks, case.block_table, case.seq_lens, case.page_size)
    d = case.q_new.shape[-1]
    assert_lse(got["lse"], ref["q_rot"], kd, case.seq_lens, 1.0 / math.sqrt(d), "f16", window=window, what=what,
               key_scales=ks[..., 0])


def check_u8_append(got, ref):
    """Codes and (scale, zero) pairs equal the oracle's everywhere: the appended
    rows bit for bit, every other row untouched."""
    for key in ("k_codes", "v_codes"):
        bad = np.argwhere(got[key] != ref[key])
        assert bad.size == 0, (key, bad[:5])
    for key in ("k_sz", "v_sz"):
        assert np.array_equal(got[key].view(np.uint32), np.asarray(ref[key], np.float32).view(np.uint32)), key


SHAPES = [
    # B, h_q, h_kv, d, lens, capacity
    (2, 32, 8, 128, [1000, 257], 1000),      # G=4, ragged tail
    (3, 8, 8, 128, [64, 1, 129], 130),       # MHA
    (1, 16, 1, 128, [777], 778),             # MQA, G=16
    (2, 64, 2, 128, [300, 45], 300),         # G=32: two head blocks in one CTA
    (1, 96, 1, 64, [200], 200),              # G=96: several head super-blocks, d=64
    (2, 12, 3, 64, [513, 64], 514),          # d=64, G=4
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s[0]}q{s[1]}kv{s[2]}d{s[3]}")
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_u8_contiguous_matches_oracle(m, shape, splits):
    B, hq, hkv, d, lens, cap = shape
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, head_dim=d, seed=300 + hq + d)
    c, u = _contiguous(w, lens, cap, seed=7 + d)
    ref = _oracle(w, c, u, paged=False)
    got = run_u8(m, w, c, u, paged=False, splits=splits)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= BF16_TOL
    check_u8_lse(got, ref, c)
    assert np.max(np.abs(got["q_rot"] - ref["q_rot"])) <= 1e-5 * (1 + np.max(np.abs(ref["q_rot"])))
    check_u8_append(got, ref)


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("heads", [(16, 2, 128), (32, 8, 128), (12, 3, 128), (64, 2, 128), (16, 4, 64)],
                         ids=lambda h: f"q{h[0]}kv{h[1]}d{h[2]}")
def test_u8_paged_matches_oracle(m, page_size, heads):
    """16- and 32-token pages with G <= 16 and an even kv head count run the
    head-group kernel (groups of 4 or 2 kv heads per block); the rest the
    token-slice kernel."""
    w = workload("paged").with_(batch=5, h_q=heads[0], h_kv=heads[1], head_dim=heads[2], page_size=page_size,
                                len_lo=1, len_hi=700, seed=19)
    pc, u = _paged(w, [1, 16, 17, 700, 333], seed=23)
    ref = _oracle(w, pc, u, paged=True)
    for splits in (1, 3, 0):
        got = run_u8(m, w, pc, u, paged=True, splits=splits)
        assert got["err"] == 0
        assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL, splits
        assert np.max(np.abs(got["lse"] - ref["lse"])) <= BF16_TOL
        check_u8_lse(got, ref, pc, paged=True, what=splits)
        check_u8_append(got, ref)


@pytest.mark.parametrize("window", [1, 16, 17, 100, 1000])
def test_u8_sliding_window(m, window):
    w = workload("gqa4k").with_(batch=3, h_q=16, h_kv=4, seed=71)
    c, u = _contiguous(w, [700, 65, 3], 704, seed=5)
    ref = _oracle(w, c, u, paged=False, window=window)
    for splits in (1, 0):
        got = run_u8(m, w, c, u, paged=False, splits=splits, window=window, max_len=700)
        assert got["err"] == 0
        assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL, (splits, window)
    wp = workload("paged").with_(batch=4, h_q=16, h_kv=4, seed=72)
    pc, up = _paged(wp, [700, 64, 17, 1], seed=6)
    refp = _oracle(wp, pc, up, paged=True, window=window)
    table = pc.block_table.clone()
    for b, L in enumerate([700, 64, 17, 1]):
        table[b, :max(0, L - window) // pc.page_size] = -1  # released pages before the window
    got = run_u8(m, wp, pc, up, paged=True, splits=0, window=window, table=table, max_len=700)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - refp["out"])) <= BF16_TOL, window


def test_u8_quantised_values_match_dequantised_input(m):
    """A cache built by quantising N(0,1) rows with the oracle's quantiser:
    the GPU result equals attention over the dequantised values."""
    w = workload("gqa4k").with_(batch=2, h_q=8, h_kv=2, seed=73)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor([500, 77], dtype=torch.int32), capacity=500)
    kq, ks, kz = oracle.quantize_u8(c.k_cache.float().numpy())
    vq, vs, vz = oracle.quantize_u8(c.v_cache.float().numpy())

    class U:
        k_codes = torch.from_numpy(kq)
        v_codes = torch.from_numpy(vq)
        k_sz = torch.from_numpy(np.stack([ks, kz], -1).astype(np.float32))
        v_sz = torch.from_numpy(np.stack([vs, vz], -1).astype(np.float32))

    ref = _oracle(w, c, U, paged=False)
    got = run_u8(m, w, c, U, paged=False)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL
    check_u8_append(got, ref)


def test_u8_large_v_scale_sets_error(m):
    """A V scale beyond what the kernel's fp16 P' holds is reported, not
    silently wrong."""
    w = workload("gqa4k").with_(batch=1, h_q=8, h_kv=2, seed=74)
    c, u = _contiguous(w, [100], 100, seed=8)
    u.v_sz[0, 1, 10, 0] = 2000.0
    got = run_u8(m, w, c, u, paged=False, splits=1)
    assert got["err"] & m.MQA_DEVERR_U8_SCALE


def test_u8_full_size_sampled(m):
    """The 4096-token GQA workload (batch 32, 32 query / 8 kv heads) over a
    uint8 cache: three (sequence, kv head) units against the oracle."""
    w = workload("gqa4k")
    L = w.seq_len
    c = make_contiguous_case(w, DEV)
    u = make_u8_cache((w.batch, w.h_kv, L), w.head_dim, 9, device=DEV)
    units = [(0, 0), (w.batch - 1, w.h_kv - 1), (13, 5)]
    saved = {(b, j): (u.k_codes[b, j].cpu(), u.k_sz[b, j].cpu(), u.v_codes[b, j].cpu(), u.v_sz[b, j].cpu())
             for b, j in units}
    lay = m.layout_contiguous(u.k_codes, u.v_codes, w.h_q, k_scale_zero=u.k_sz, v_scale_zero=u.v_sz)
    bufs = m.DecodeBuffers.allocate(lay, L, num_splits=0, device=DEV)
    m.decode_step(lay, c.q_new, c.k_new, c.v_new, c.pos, c.seq_lens, L, bufs, w.rope_base,
                  1.0 / math.sqrt(w.head_dim), num_splits=0)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    G = w.group
    for b, j in units:
        kc, ks, vc, vs = saved[(b, j)]
        sub = workload("gqa4k").with_(batch=1, h_q=G, h_kv=1)

        class Case:
            q_new = c.q_new[b:b + 1, j * G:(j + 1) * G].cpu()
            k_new = c.k_new[b:b + 1, j:j + 1].cpu()
            v_new = c.v_new[b:b + 1, j:j + 1].cpu()
            seq_lens = torch.tensor([L], dtype=torch.int32)

        class Unit:
            k_codes, k_sz, v_codes, v_sz = kc[None, None], ks[None, None], vc[None, None], vs[None, None]

        ref = _oracle(sub, Case, Unit, paged=False)
        got = _np(bufs.out[b, j * G:(j + 1) * G])
        assert np.max(np.abs(got - ref["out"][0])) <= BF16_TOL, (b, j)
        assert np.array_equal(u.k_codes[b, j, L - 1].cpu().numpy(), ref["k_codes"][0, 0, L - 1])


# One new token with 32 query heads per kv head (MQA) runs on the tcgen05
# kernel that puts the keys on the MMA rows: codes widened to exact fp16
# (c - z), K scale on the scores, V scale folded into P.
MQA_SHAPES = [
    # B, h_q, h_kv, lens, capacity
    (9, 32, 1, [1, 2, 127, 128, 129, 255, 256, 257, 1000], 1000),  # tile edges, a single key
    (2, 64, 2, [700, 77], 704),                                    # two kv heads
]


@pytest.mark.parametrize("shape", MQA_SHAPES, ids=lambda s: f"B{s[0]}q{s[1]}kv{s[2]}")
@pytest.mark.parametrize("splits", [1, 2, 5, 0])
def test_u8_mqa_matches_oracle(m, shape, splits):
    B, hq, hkv, lens, cap = shape
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, seed=360 + hq)
    c, u = _contiguous(w, lens, cap, seed=31)
    ref = _oracle(w, c, u, paged=False)
    got = run_u8(m, w, c, u, paged=False, splits=splits)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= BF16_TOL
    check_u8_lse(got, ref, c)
    check_u8_append(got, ref)


@pytest.mark.parametrize("window", [1, 63, 64, 100, 1000])
def test_u8_mqa_window_and_nan_rows_past_the_sequence(m, window):
    """MQA over uint8 with a window; the rows past each sequence hold NaN
    scales and zero points (their V rows are zeroed and their P is 0)."""
    lens = [900, 200, 37]
    w = workload("gqa4k").with_(batch=3, h_q=32, h_kv=1, seed=362)
    c, u = _contiguous(w, lens, 1024, seed=32)
    ref = _oracle(w, c, u, paged=False, window=window)
    for b, L in enumerate(lens):
        u.k_sz[b, :, L:] = float("nan")
        u.v_sz[b, :, L:] = float("nan")
    for splits in (1, 3, 0):
        got = run_u8(m, w, c, u, paged=False, splits=splits, window=window, max_len=900)
        assert got["err"] == 0
        assert np.all(np.isfinite(got["out"]))
        assert np.max(np.abs(got["out"] - ref["out"])) <= BF16_TOL, (window, splits)


def test_u8_mqa_large_v_scale_sets_error(m):
    """MQA: a V scale above 1023 is reported (P' = p s^v / 4 would leave fp16)."""
    w = workload("gqa4k").with_(batch=1, h_q=32, h_kv=1, seed=363)
    c, u = _contiguous(w, [300], 300, seed=33)
    u.v_sz[0, 0, 10, 0] = 2000.0
    got = run_u8(m, w, c, u, paged=False, splits=1)
    assert got["err"] & m.MQA_DEVERR_U8_SCALE


def test_u8_mqa_full_size_sampled(m):
    """The MQA workload (64 sequences of 8192 tokens, 32 query heads on one kv
    head) over a uint8 cache: three sequences against the oracle."""
    w = workload("mqa8k")
    L = w.seq_len
    c = make_contiguous_case(w, DEV)
    u = make_u8_cache((w.batch, 1, L), w.head_dim, 34, device=DEV)
    seqs = [0, 31, 63]
    saved = {b: (u.k_codes[b, 0].cpu(), u.k_sz[b, 0].cpu(), u.v_codes[b, 0].cpu(), u.v_sz[b, 0].cpu()) for b in seqs}
    lay = m.layout_contiguous(u.k_codes, u.v_codes, w.h_q, k_scale_zero=u.k_sz, v_scale_zero=u.v_sz)
    bufs = m.DecodeBuffers.allocate(lay, L, num_splits=0, device=DEV)
    m.decode_step(lay, c.q_new, c.k_new, c.v_new, c.pos, c.seq_lens, L, bufs, w.rope_base,
                  1.0 / math.sqrt(w.head_dim), num_splits=0)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    for b in seqs:
        kc, ks, vc, vs = saved[b]
        sub = workload("gqa4k").with_(batch=1, h_q=32, h_kv=1)

        class Case:
            q_new = c.q_new[b:b + 1].cpu()
            k_new = c.k_new[b:b + 1].cpu()
            v_new = c.v_new[b:b + 1].cpu()
            seq_lens = torch.tensor([L], dtype=torch.int32)

        class Unit:
            k_codes, k_sz, v_codes, v_sz = kc[None, None], ks[None, None], vc[None, None], vs[None, None]

        ref = _oracle(sub, Case, Unit, paged=False)
        assert np.max(np.abs(_np(bufs.out[b]) - ref["out"][0])) <= BF16_TOL, b


# ------------------------------------------------------------ several new tokens
def run_u8_multi(m, w, n, u, q, k, v, lens, splits=0, window=0, table=None, page_size=0):
    kc, vc = u.k_codes.to(DEV), u.v_codes.to(DEV)
    ks, vs = u.k_sz.to(DEV), u.v_sz.to(DEV)
    if table is not None:
        bt = table.to(DEV)
        lay = m.layout_paged(kc, vc, bt, w.h_q, window=window, k_scale_zero=ks, v_scale_zero=vs)
    else:
        lay = m.layout_contiguous(kc, vc, w.h_q, window=window, k_scale_zero=ks, v_scale_zero=vs)
    lens_d = torch.as_tensor(lens, dtype=torch.int32).to(DEV)
    max_len = int(max(lens))
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=splits, device=DEV, n_new=n)
    m.decode_step_multi(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), (lens_d - n).to(torch.int32), lens_d, max_len,
                        bufs, w.rope_base, 1.0 / math.sqrt(w.head_dim), num_splits=splits)
    torch.cuda.synchronize()
    return dict(out=_np(bufs.out), lse=_np(bufs.lse), q_rot=_np(bufs.q_rot), err=int(bufs.err.item()),
                k_codes=kc.cpu().numpy(), v_codes=vc.cpu().numpy(), k_sz=ks.cpu().numpy(), v_sz=vs.cpu().numpy())


def _new_tokens(w, n, seed):
    from synthetic import normal
    return (normal((w.batch, n, w.h_q, w.head_dim), seed, 21), normal((w.batch, n, w.h_kv, w.head_dim), seed, 22),
            normal((w.batch, n, w.h_kv, w.head_dim), seed, 23))


def check_multi(got, ref, lens, w, paged_table=None, page_size=0, window=0, what=None):
    assert got["err"] == 0, what
    assert np.max(np.abs(got["out"].reshape(ref["out"].shape) - ref["out"])) <= BF16_TOL, what
    assert np.max(np.abs(got["lse"].reshape(ref["lse"].shape) - ref["lse"])) <= BF16_TOL, what
    check_u8_append(got, ref)
    kd = oracle.dequantize_u8(ref["k_codes"], ref["k_sz"][..., 0], ref["k_sz"][..., 1])
    ks = np.asarray(ref["k_sz"][..., :1], np.float64)
    if paged_table is not None:
        kd = paged_keys(kd, paged_table, lens, page_size)
        ks = paged_keys(ks, paged_table, lens, page_size)
    assert_lse(got["lse"].reshape(ref["lse"].shape), ref["q_rot"], kd, lens, 1.0 / math.sqrt(w.head_dim), "f16",
               window=window, what=what, key_scales=ks[..., 0])


MULTI = [
    # B, h_q, h_kv, d, lens, capacity, n
    (2, 32, 8, 128, [1000, 257], 1000, 4),   # G = 4 x 4 tokens: one 16-row block
    (2, 32, 8, 128, [300, 6], 300, 6),       # 24 rows, L = n
    (3, 16, 2, 128, [129, 64, 65], 130, 2),  # G = 8 x 2
    (1, 32, 1, 128, [500], 500, 3),          # MQA: 96 rows, three CTAs of 32
    (2, 12, 3, 64, [200, 33], 200, 8),       # d = 64, G = 4 x 8
]


@pytest.mark.parametrize("shape", MULTI, ids=lambda s: f"B{s[0]}q{s[1]}kv{s[2]}d{s[3]}n{s[6]}")
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_u8_multi_token_matches_oracle(m, shape, splits):
    """Several new tokens per sequence over a uint8 cache (the warp-MMA uint8
    kernel, rows = (token, head) pairs with per-row key limits) against the
    oracle's decode_step_multi_u8: the appended rows (codes, scales, zero
    points) bit for bit, outputs within 2e-2, lse against the model."""
    B, hq, hkv, d, lens, cap, n = shape
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, head_dim=d, seed=820 + hq + d + n)
    u = make_u8_cache((B, hkv, cap), d, 83 + n)
    q, k, v = _new_tokens(w, n, w.seed)
    ref = oracle.decode_step_multi_u8(u.k_codes, u.k_sz, u.v_codes, u.v_sz, q, k, v, lens, w.rope_base,
                                      1.0 / math.sqrt(d))
    got = run_u8_multi(m, w, n, u, q, k, v, lens, splits=splits)
    check_multi(got, ref, lens, w, what=splits)


@pytest.mark.parametrize("page_size", [16, 32, 64])
def test_u8_multi_token_paged(m, page_size):
    n = 5
    w = workload("paged").with_(batch=4, h_q=16, h_kv=4, page_size=page_size, seed=840 + page_size)
    lens = [700, n, 17, 64]
    pc, u = _paged(w, lens, 85)
    q, k, v = _new_tokens(w, n, w.seed)
    ref = oracle.decode_step_multi_u8(u.k_codes, u.k_sz, u.v_codes, u.v_sz, q, k, v, lens, w.rope_base,
                                      1.0 / math.sqrt(w.head_dim), block_table=pc.block_table, page_size=page_size)
    for splits in (1, 3, 0):
        got = run_u8_multi(m, w, n, u, q, k, v, lens, splits=splits, table=pc.block_table, page_size=page_size)
        check_multi(got, ref, lens, w, paged_table=pc.block_table, page_size=page_size, what=splits)


@pytest.mark.parametrize("window", [1, 3, 100])
def test_u8_multi_token_window(m, window):
    n = 5
    w = workload("gqa4k").with_(batch=3, h_q=16, h_kv=4, seed=851)
    lens = [700, 70, 5]
    u = make_u8_cache((3, 4, 704), 128, 86)
    q, k, v = _new_tokens(w, n, w.seed)
    ref = oracle.decode_step_multi_u8(u.k_codes, u.k_sz, u.v_codes, u.v_sz, q, k, v, lens, w.rope_base,
                                      1.0 / math.sqrt(128), window=window)
    for splits in (1, 3, 0):
        got = run_u8_multi(m, w, n, u, q, k, v, lens, splits=splits, window=window)
        check_multi(got, ref, lens, w, window=window, what=(window, splits))
