"""A decode step whose new-token inputs (q, k, v, positions, lengths) and
output live in pinned host memory: the kernels read and write them across the
CPU-GPU link. Same results as with device buffers, checked against the fp64
oracle (bf16 outputs <= 2e-2)."""

import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import make_contiguous_case, make_paged_case, workload

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def m(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mqa_decode_attention_gb300 as mod

    mod.library()
    return mod


def _pinned(t):
    return t.detach().cpu().contiguous().pin_memory()


@pytest.mark.parametrize("hq,hkv,splits", [(32, 8, 1), (32, 1, 2), (16, 2, 3)], ids=["gqa", "mqa", "split3"])
def test_host_io_contiguous(m, hq, hkv, splits):
    w = workload("gqa4k").with_(batch=3, h_q=hq, h_kv=hkv, seed=900 + hq + hkv)
    lens = [700, 129, 1]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=700)
    scale = 1.0 / math.sqrt(w.head_dim)
    ref = oracle.decode_step_contiguous(c.k_cache, c.v_cache, c.q_new, c.k_new, c.v_new, c.seq_lens, w.rope_base,
                                        scale, "bf16")
    kc, vc = c.k_cache.cuda(), c.v_cache.cuda()
    lay = m.layout_contiguous(kc, vc, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, 700, num_splits=splits, device="cuda")
    bufs.out = _pinned(torch.zeros(bufs.out.shape, dtype=bufs.out.dtype))
    m.decode_step(lay, _pinned(c.q_new), _pinned(c.k_new), _pinned(c.v_new), _pinned(c.pos), _pinned(c.seq_lens), 700,
                  bufs, w.rope_base, scale, num_splits=splits)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    assert np.max(np.abs(bufs.out.to(torch.float64).numpy() - ref["out"])) <= TOL
    assert np.array_equal(vc.cpu().to(torch.float64).numpy(), ref["v_cache"])


def test_host_io_paged(m):
    w = workload("paged").with_(batch=4, h_q=16, h_kv=2, seed=905)
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor([300, 17, 1, 64], dtype=torch.int32))
    scale = 1.0 / math.sqrt(w.head_dim)
    ref = oracle.decode_step_paged(pc.k_pool, pc.v_pool, pc.block_table, pc.q_new, pc.k_new, pc.v_new, pc.seq_lens,
                                   pc.page_size, w.rope_base, scale, "bf16")
    kp, vp, bt = pc.k_pool.cuda(), pc.v_pool.cuda(), pc.block_table.cuda()
    lay = m.layout_paged(kp, vp, bt, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, 300, num_splits=2, device="cuda")
    bufs.out = _pinned(torch.zeros(bufs.out.shape, dtype=bufs.out.dtype))
    m.decode_step(lay, _pinned(pc.q_new), _pinned(pc.k_new), _pinned(pc.v_new), _pinned(pc.pos), _pinned(pc.seq_lens),
                  300, bufs, w.rope_base, scale, num_splits=2)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    assert np.max(np.abs(bufs.out.to(torch.float64).numpy() - ref["out"])) <= TOL
