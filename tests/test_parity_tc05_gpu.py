"""GPU parity of decode steps that run on the tensor-memory (tcgen05) kernel:
32 or more query rows per kv head (MQA's G = 32; several new tokens per
sequence), contiguous bf16 cache, head_dim 128. Checked against the fp64
oracle like every other decode path: outputs and lse <= 2e-2.
"""

import math

import numpy as np
import pytest
import torch

import oracle
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
    return dict(out=_np(bufs.out).reshape(B, n, hq, -1), lse=_np(bufs.lse).reshape(B, n, hq), k=kc.cpu(),
                v=vc.cpu(), err=int(bufs.err.item()))


CASES = [
    # B, h_q, h_kv, n, lens, capacity
    (3, 32, 1, 1, [1000, 129, 1], 1000),    # MQA, G = 32: one 128-row block, 96 padding rows
    (2, 64, 1, 1, [700, 300], 704),         # G = 64
    (2, 32, 4, 4, [400, 33], 400),          # G = 8 x 4 tokens = 32 rows
    (2, 32, 8, 8, [300, 8], 300),           # G = 4 x 8 tokens, L = n
    (1, 32, 1, 5, [260], 260),              # G = 32 x 5 = 160 rows: two row blocks
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}q{c[1]}kv{c[2]}n{c[3]}")
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_tc05_decode_matches_oracle(m, case, splits):
    B, hq, hkv, n, lens, cap = case
    w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, seed=700 + hq + n)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=cap)
    q, k, v = new_tokens(w, n)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16")
    got = run(m, w, n, c, q, k, v, lens, splits)
    assert got["err"] == 0
    assert np.max(np.abs(got["out"] - ref["out"])) <= TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= TOL
    assert np.array_equal(_np(got["v"]), ref["v_cache"])


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
