"""GPU parity of decode steps that run on the tensor-memory (tcgen05) kernel:
32 or more query rows per kv head (MQA's G = 32; several new tokens per
sequence), contiguous bf16 cache, head_dim 128. Checked against the fp64
oracle like every other decode path: outputs and lse <= 2e-2, and lse <= 1e-4
of the log-sum-exp over the scores the kernel forms (its bf16 query operand,
tests/lse_model.py).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from lse_model import assert_lse
from synthetic import make_contiguous_case, normal, workload

pytestmark = pytest.mark.gpu

TOL = 2e-2
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


def new_tokens(w, n):
    q = normal((w.batch, n, w.h_q, w.head_dim), w.seed, 21, w.dtype)
    k = normal((w.batch, n, w.h_kv, w.head_dim), w.seed, 22, w.dtype)
    v = normal((w.batch, n, w.h_kv, w.head_dim), w.seed, 23, w.dtype)
    return q, k, v


def run(m, w, n, c, q, k, v, lens, splits, window=0):
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q, window=window)
    lens_d = torch.as_tensor(lens, dtype=torch.int32).to(DEV)
    max_len = int(max(lens))
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=splits, device=DEV, n_new=n)
    if n == 1:
        m.decode_step(lay, q[:, 0].to(DEV), k[:, 0].to(DEV), v[:, 0].to(DEV), lens_d - 1, lens_d, max_len, bufs,
                      w.rope_base, 1.0 / math.sqrt(w.head_dim), num_splits=splits)
    else:
        m.decode_step_multi(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), lens_d - n, lens_d, max_len, bufs, w.rope_base,
                            1.0 / math.sqrt(w.head_dim), num_splits=splits)
    torch.cuda.synchronize()
    B, hq = w.batch, w.h_q
    return dict(out=_np(bufs.out).reshape(B, n, hq, -1), lse=_np(bufs.lse).reshape(B, n, hq),
                q_rot=_np(bufs.q_rot).reshape(B, n, hq, -1), k=kc.cpu(), v=vc.cpu(), err=int(bufs.err.item()))


def ulp_bf16(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def check_step(got, ref, lens):
    """Outputs within the bf16 tolerance, lse within fp32 rounding of the
    scores the kernel forms, q_rot within fp32 rounding, the appended rows
    placement-exact (V bytes, K within one bf16 ulp)."""
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= TOL
    assert_lse(got["lse"], ref["q_rot"], ref["k_cache"], lens, 1.0 / math.sqrt(128), "bf16")
    assert np.max(np.abs(got["q_rot"] - ref["q_rot"])) <= 1e-5 * (1 + np.max(np.abs(ref["q_rot"])))
    assert np.array_equal(_np(got["v"]), ref["v_cache"])
    k = _np(got["k"])
    assert np.all(np.abs(k - ref["k_cache"]) <= ulp_bf16(ref["k_cache"]) + 1e-30)


CASES = [
    # B, h_q, h_kv, n, lens, capacity
    (3, 32, 1, 1, [1000, 129, 1], 1000),    # MQA, G = 32: one 128-row block, 96 padding rows
    (2, 64, 1, 1, [700, 300], 704),         # G = 64
    (2, 32, 4, 4, [400, 33], 400),          # G = 8 x 4 tokens = 32 rows
    (2, 32, 8, 8, [300, 8], 300),           # G = 4 x 8 tokens, L = n
    (1, 32, 1, 5, [260], 260),              # G = 32 x 5 = 160 rows: two row blocks
    (2, 32, 8, 32, [300, 40], 300),         # G = 4 x 32 = 128 rows: query rows as two TMA boxes
    (1, 10, 2, 32, [250], 250),             # G = 5 x 32 = 160 rows: a group that does not divide 64 (plain loads)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}q{c[1]}kv{c[2]}n{c[3]}")
@pytest.mark.parametrize("splits", [1, 2, 3, 0])
def test_tc05_decode_matches_oracle(m, case, splits):
    B, hq, hkv, n, lens, cap = case
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, seed=700 + hq + n)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=cap)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16")
    got = run(m, w, n, c, q, k, v, lens, splits)
    check_step(got, ref, lens)


@pytest.mark.parametrize("window", [1, 100, 1000])
def test_tc05_decode_sliding_window(m, window):
    w = workload("gqa4k").with_(batch=2, h_q=32, h_kv=1, seed=711)
    n, lens = 3, [900, 50]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=900)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16", window=window)
    for splits in (1, 4, 0):
        got = run(m, w, n, c, q, k, v, lens, splits, window=window)
        assert got["err"] == 0
        assert np.max(np.abs(got["out"] - ref["out"])) <= TOL, (splits, window)
        assert_lse(got["lse"], ref["q_rot"], ref["k_cache"], lens, 1.0 / math.sqrt(128), "bf16", window=window,
                   what=splits)


def test_tc05_mqa_full_size_sampled(m):
    """The MQA batch (64 sequences of 8192 tokens, 32 query heads on one kv
    head): three sequences against the oracle."""
    w = workload("mqa8k")
    L = w.seq_len
    c = make_contiguous_case(w, DEV)
    seqs = [0, 31, 63]
    saved = {b: (c.k_cache[b, 0].cpu(), c.v_cache[b, 0].cpu()) for b in seqs}
    lay = m.layout_contiguous(c.k_cache, c.v_cache, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, L, num_splits=0, device=DEV)
    m.decode_step(lay, c.q_new, c.k_new, c.v_new, c.pos, c.seq_lens, L, bufs, w.rope_base,
                  1.0 / math.sqrt(w.head_dim))
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    for b in seqs:
        K, V = saved[b]
        o, _, _ = oracle.decode_unit(c.q_new[b].cpu(), c.k_new[b, 0].cpu(), c.v_new[b, 0].cpu(), K, V, L,
                                     w.rope_base, 1.0 / math.sqrt(w.head_dim), "bf16")
        assert np.max(np.abs(_np(bufs.out[b]) - o)) <= TOL, b


@pytest.mark.parametrize("standalone", [False, True])
def test_tc05_splits_with_garbage_workspace(m, standalone):
    """The split scratch starts as garbage, and three standalone calls after
    the step give the same result: nothing carries over between calls."""
    w = workload("gqa4k").with_(batch=3, h_q=32, h_kv=1, seed=741)
    n, lens = 2, [700, 300, 65]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=704)
    q, k, v = new_tokens(w, n)
    scale = 1.0 / math.sqrt(w.head_dim)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, scale, "bf16")
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    lens_d = torch.as_tensor(lens, dtype=torch.int32).to(DEV)
    bufs = m.DecodeBuffers.allocate(lay, 700, num_splits=4, device=DEV, n_new=n)
    bufs.workspace.fill_(0x5A)
    m.decode_step_multi(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), lens_d - n, lens_d, 700, bufs, w.rope_base, scale,
                        num_splits=4)
    for _ in range(3):
        if standalone:
            bufs.out.zero_()
            m.gqa_decode_attention_multi(lay, n, bufs.q_rot, lens_d, 700, scale, 4, bufs.out, bufs.lse,
                                         bufs.workspace, err=bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0
        got = _np(bufs.out).reshape(3, n, 32, -1)
        assert np.max(np.abs(got - ref["out"])) <= TOL
        assert np.max(np.abs(_np(bufs.lse).reshape(3, n, 32) - ref["lse"])) <= TOL
        assert_lse(_np(bufs.lse).reshape(3, n, 32), ref["q_rot"], ref["k_cache"], lens, scale, "bf16")


@pytest.mark.parametrize("n, hq", [(1, 32), (1, 64), (2, 32)])
def test_tc05_two_split_cluster_merge(m, n, hq):
    """Two splits with at most 64 rows per kv head: the two blocks of a
    (sequence, kv head) are one cluster and merge their results in shared
    memory (no combine). Split 1 is empty for the short sequences (only split
    0 holds keys), the fused step and the standalone call agree with the
    oracle, in bf16 and fp32 output, on three calls in a row."""
    w = workload("gqa4k").with_(batch=4, h_q=hq, h_kv=1, seed=760 + hq + n)
    lens = [1000, 513, 512, max(n, 1)]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=1000)
    q, k, v = new_tokens(w, n)
    scale = 1.0 / math.sqrt(w.head_dim)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, scale, "bf16")
    check_step(run(m, w, n, c, q, k, v, lens, 2), ref, lens)
    # standalone attention over the appended cache, fp32 output
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    lens_d = torch.as_tensor(lens, dtype=torch.int32).to(DEV)
    bufs = m.DecodeBuffers.allocate(lay, 1000, num_splits=2, device=DEV, n_new=n, out_dtype=torch.float32)
    bufs.workspace.fill_(0x7F)
    m.kv_append_rope_multi(lay, n, q.to(DEV), k.to(DEV), v.to(DEV), lens_d - n, w.rope_base, bufs.q_rot, bufs.err)
    for _ in range(3):
        bufs.out.fill_(float("nan"))
        m.gqa_decode_attention_multi(lay, n, bufs.q_rot, lens_d, 1000, scale, 2, bufs.out, bufs.lse,
                                     bufs.workspace, err=bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0
        got = _np(bufs.out).reshape(4, n, hq, -1)
        # (fp32 output of a tensor-core path: Q and P are bf16 MMA operands)
        assert np.max(np.abs(got - ref["out"])) <= TOL
        assert np.max(np.abs(_np(bufs.lse).reshape(4, n, hq) - ref["lse"])) <= TOL
        assert_lse(_np(bufs.lse).reshape(4, n, hq), ref["q_rot"], ref["k_cache"], lens, scale, "bf16")


def test_tc05_many_short_splits(m):
    """128 rows per kv head and 204 splits of 64 tokens (250 requested): one
    128-key tile per split reaching into the next split's keys."""
    w = workload("gqa4k").with_(batch=1, h_q=32, h_kv=1, seed=742)
    n, lens = 4, [13000]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=13000)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16")
    got = run(m, w, n, c, q, k, v, lens, 250)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= TOL
    assert_lse(got["lse"], ref["q_rot"], ref["k_cache"], lens, 1.0 / math.sqrt(128), "bf16")


def test_tc05_fused_step_new_slot_holds_nan(m):
    """One-token step on the tcgen05 kernel is a single launch: the block whose
    split holds the new position writes its k / v row. Splits of 192 tokens
    (L = 400, 3 splits) let split 1's last 128-key tile reach the new row at
    399 while split 2 writes it; the slot holds NaN before the step."""
    w = workload("gqa4k").with_(batch=2, h_q=32, h_kv=1, seed=751)
    lens = [400, 400]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=400)
    c.k_cache[:, :, 399] = float("nan")
    c.v_cache[:, :, 399] = float("nan")
    q, k, v = new_tokens(w, 1)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16")
    for splits in (3, 1, 0):
        got = run(m, w, 1, c, q, k, v, lens, splits)
        assert np.all(np.isfinite(got["out"]))
        check_step(got, ref, lens)


def test_tc05_fused_step_position_out_of_range(m):
    """pos past the cache: MQA_DEVERR_POS_RANGE, the cache untouched, q_rot
    still written."""
    w = workload("gqa4k").with_(batch=2, h_q=32, h_kv=1, seed=752)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor([128, 128], dtype=torch.int32), capacity=128)
    q, k, v = new_tokens(w, 1)
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    k0 = kc.clone()
    lay = m.layout_contiguous(kc, vc, w.h_q)
    lens_d = torch.tensor([128, 128], dtype=torch.int32, device=DEV)
    pos = torch.tensor([127, 128], dtype=torch.int32, device=DEV)  # sequence 1: one past the cache
    bufs = m.DecodeBuffers.allocate(lay, 128, num_splits=1, device=DEV)
    m.decode_step(lay, q[:, 0].to(DEV), k[:, 0].to(DEV), v[:, 0].to(DEV), pos, lens_d, 128, bufs, w.rope_base,
                  num_splits=1)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) & m.MQA_DEVERR_POS_RANGE
    assert torch.equal(kc[1], k0[1])       # nothing written for sequence 1
    assert not torch.equal(kc[0], k0[0])   # sequence 0's row landed
    ref = oracle.decode_step_multi(c.k_cache[:1], c.v_cache[:1], q[:1], k[:1], v[:1], [128], w.rope_base,
                                   1.0 / math.sqrt(w.head_dim), "bf16")
    assert np.max(np.abs(_np(bufs.q_rot[1]) - oracle_q_rot(q[1:2], 128, w.rope_base))) <= 1e-4
    assert np.max(np.abs(_np(bufs.out[0]) - ref["out"][0, 0])) <= TOL


def oracle_q_rot(q, pos, rope_base):
    """RoPE of one sequence's new query at `pos` through the oracle (a
    zero-length cache suffices: only q_rot is used)."""
    kz = torch.zeros(1, 1, pos + 1, q.shape[-1], dtype=torch.bfloat16)
    hkv = 1
    kn = torch.zeros(1, 1, hkv, q.shape[-1], dtype=torch.bfloat16)
    r = oracle.decode_step_multi(kz, kz, q, kn, kn, [pos + 1], rope_base, 1.0, "bf16")
    return r["q_rot"][0, 0]
