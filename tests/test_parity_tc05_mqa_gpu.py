"""GPU parity of the one-token decode step with 32 query heads per kv head
(MQA) over a bf16 cache, on the tcgen05 kernel (the 32 query rows replicated
over the MMA's 128 rows, each copy a quarter of every key tile). Checked
against the fp64 oracle: outputs and lse <= 2e-2, lse <= 1e-4 of the
log-sum-exp over the scores the kernel forms (its bf16 query operand,
tests/lse_model.py), the appended rows placement-exact.

Cases: lengths at the 128-key tile edges and below one tile, sliding windows
(a block's first tile starts up to 63 keys before the window), several kv
heads, the standalone attention call on a given q_rot with fp32 output, and
scores whose per-head maxima grow by more than 2^8 after the first tiles, so
that the reference maxima move and O is rescaled mid-sequence.
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


def new_token(w):
    q = normal((w.batch, 1, w.h_q, w.head_dim), w.seed, 21, w.dtype)
    k = normal((w.batch, 1, w.h_kv, w.head_dim), w.seed, 22, w.dtype)
    v = normal((w.batch, 1, w.h_kv, w.head_dim), w.seed, 23, w.dtype)
    return q, k, v


def ulp_bf16(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def step(m, w, c, q, k, v, lens, splits, window=0):
    """The fused one-launch step (RoPE, append, attention) through decode_step."""
    kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q, window=window)
    lens_d = torch.as_tensor(lens, dtype=torch.int32).to(DEV)
    max_len = int(max(lens))
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=splits, device=DEV)
    m.decode_step(lay, q[:, 0].to(DEV), k[:, 0].to(DEV), v[:, 0].to(DEV), lens_d - 1, lens_d, max_len, bufs,
                  w.rope_base, 1.0 / math.sqrt(w.head_dim), num_splits=splits)
    torch.cuda.synchronize()
    B, hq = w.batch, w.h_q
    return dict(out=_np(bufs.out).reshape(B, 1, hq, -1), lse=_np(bufs.lse).reshape(B, 1, hq),
                q_rot=_np(bufs.q_rot).reshape(B, 1, hq, -1), k=_np(kc), v=_np(vc), err=int(bufs.err.item()))


def check(got, ref, what, lens, window=0):
    assert got["err"] == 0, what
    assert np.max(np.abs(got["out"] - ref["out"])) <= TOL, what
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= TOL, what
    assert_lse(got["lse"], ref["q_rot"], ref["k_cache"], lens, 1.0 / math.sqrt(128), "bf16", window=window,
               what=what)
    assert np.max(np.abs(got["q_rot"] - ref["q_rot"])) <= 1e-5 * (1 + np.max(np.abs(ref["q_rot"]))), what
    assert np.array_equal(got["v"], ref["v_cache"]), what
    assert np.all(np.abs(got["k"] - ref["k_cache"]) <= ulp_bf16(ref["k_cache"]) + 1e-30), what


@pytest.mark.parametrize("splits", [1, 2, 5, 0])
def test_keys_kernel_tile_edges(m, splits):
    """Lengths 1, 2, 127, 128, 129, 255, 256, 257 and 1000 in one batch: whole
    tiles, one key past a tile, a single key."""
    lens = [1, 2, 127, 128, 129, 255, 256, 257, 1000]
    w = workload("gqa4k").with_(batch=len(lens), h_q=32, h_kv=1, seed=801)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=1000)
    q, k, v = new_token(w)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16")
    check(step(m, w, c, q, k, v, lens, splits), ref, splits, lens)


@pytest.mark.parametrize("window", [1, 63, 64, 100, 129, 1000])
def test_keys_kernel_sliding_window(m, window):
    lens = [900, 50, 300]
    w = workload("gqa4k").with_(batch=3, h_q=32, h_kv=1, seed=802)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=900)
    q, k, v = new_token(w)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16", window=window)
    for splits in (1, 3, 0):
        check(step(m, w, c, q, k, v, lens, splits, window=window), ref, (window, splits), lens, window)


def test_keys_kernel_two_kv_heads(m):
    """h_q = 64 on h_kv = 2: the group of 32 query heads of each kv head."""
    lens = [600, 77]
    w = workload("gqa4k").with_(batch=2, h_q=64, h_kv=2, seed=803)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=640)
    q, k, v = new_token(w)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16")
    for splits in (1, 4, 0):
        check(step(m, w, c, q, k, v, lens, splits), ref, splits, lens)


@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_keys_kernel_standalone_attention(m, out_dtype):
    """gqa_decode_attention on the oracle's q_rot and appended cache (no
    RoPE, no append in the launch)."""
    lens = [700, 129, 64]
    w = workload("gqa4k").with_(batch=3, h_q=32, h_kv=1, seed=804)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=704)
    q, k, v = new_token(w)
    scale = 1.0 / math.sqrt(w.head_dim)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, scale, "bf16")
    kc = torch.from_numpy(ref["k_cache"]).to(torch.bfloat16).to(DEV)
    vc = torch.from_numpy(ref["v_cache"]).to(torch.bfloat16).to(DEV)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    q_rot = torch.from_numpy(ref["q_rot"][:, 0]).to(torch.float32).to(DEV).contiguous()
    lens_d = torch.as_tensor(lens, dtype=torch.int32).to(DEV)
    dt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    for splits in (1, 3, 0):
        bufs = m.DecodeBuffers.allocate(lay, 700, num_splits=splits, device=DEV)
        out = torch.full((3, w.h_q, w.head_dim), float("nan"), dtype=dt, device=DEV)
        lse = torch.full((3, w.h_q), float("nan"), dtype=torch.float32, device=DEV)
        m.gqa_decode_attention(lay, q_rot, lens_d, 700, scale, splits, out, lse, bufs.workspace, err=bufs.err)
        torch.cuda.synchronize()
        assert int(bufs.err.item()) == 0
        assert np.max(np.abs(_np(out) - ref["out"][:, 0])) <= TOL, splits
        assert np.max(np.abs(_np(lse) - ref["lse"][:, 0])) <= TOL, splits
        assert_lse(_np(lse), ref["q_rot"][:, 0], ref["k_cache"], lens, scale, "bf16", what=splits)


def test_keys_kernel_growing_scores_rescale(m):
    """K rows scaled by 0.05 over the first three tiles and by 2.2 after: at
    tile 3 nearly every head's maximum score grows by more than 2^8, so the
    reference maxima move after the first tile and O is rescaled,
    while the first tiles still carry 2-8% of the output (a missing or wrong
    rescale would weigh them ~2^9 times too much). Scores stay near 12 (log2):
    much larger ones would test bf16 rounding of q instead, whose error grows
    with the score (ideal bf16-operand arithmetic is ~5e-3 off here)."""
    lens = [1280, 1100]
    w = workload("gqa4k").with_(batch=2, h_q=32, h_kv=1, seed=805)
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=1280)
    f = torch.tensor([0.05 if t < 384 else 2.2 for t in range(1280)], dtype=torch.float32)
    c.k_cache.copy_((c.k_cache.float() * f[None, None, :, None]).to(torch.bfloat16))
    q, k, v = new_token(w)
    ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, 1.0 / math.sqrt(w.head_dim),
                                   "bf16")
    # the case does what it claims (sequence 0, log2 units)
    qr = torch.from_numpy(ref["q_rot"][0, 0])
    kf = torch.from_numpy(ref["k_cache"][0, 0]).to(torch.float64)
    s = (qr @ kf[:1280].T) / math.sqrt(w.head_dim) / math.log(2)
    assert int(((s[:, 384:].amax(1) - s[:, :384].amax(1)) > 8).sum()) >= 16
    for splits in (1, 3, 0):
        check(step(m, w, c, q, k, v, lens, splits), ref, splits, lens)
