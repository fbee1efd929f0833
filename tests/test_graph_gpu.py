"""A decode step captured into a CUDA graph (the launches, with their
programmatic dependencies, recorded once and replayed): the replay gives the
eager result exactly, and both match the fp64 oracle (bf16 <= 2e-2)."""

import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import make_contiguous_case, make_paged_case, normal, workload

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


def _capture_and_replay(step):
    """Eager call (also the warm-up), then the same call captured and replayed."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = step.result()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    return eager, step.result()


class Step:
    def __init__(self, fn, bufs):
        self.fn, self.bufs = fn, bufs

    def __call__(self):
        self.fn()

    def result(self):
        return self.bufs.out.detach().clone().cpu(), int(self.bufs.err.item())


@pytest.mark.parametrize("hq,hkv,splits", [(32, 8, 1), (32, 1, 2), (16, 2, 3)], ids=["gqa_fused", "mqa_tc05", "split3"])
def test_contiguous_step_graph(m, hq, hkv, splits):
    w = workload("gqa4k").with_(batch=3, h_q=hq, h_kv=hkv, seed=950 + hq)
    lens = [600, 129, 2]
    c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=600)
    scale = 1.0 / math.sqrt(w.head_dim)
    ref = oracle.decode_step_contiguous(c.k_cache, c.v_cache, c.q_new, c.k_new, c.v_new, c.seq_lens, w.rope_base,
                                        scale, "bf16")
    lay = m.layout_contiguous(c.k_cache.to(DEV), c.v_cache.to(DEV), w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, 600, num_splits=splits, device=DEV)
    args = [x.to(DEV) for x in (c.q_new, c.k_new, c.v_new, c.pos, c.seq_lens)]
    step = Step(lambda: m.decode_step(lay, *args, 600, bufs, w.rope_base, scale, num_splits=splits), bufs)
    (eo, ee), (go, ge) = _capture_and_replay(step)
    assert ee == 0 and ge == 0
    assert torch.equal(eo, go)
    assert np.max(np.abs(go.double().numpy() - ref["out"])) <= TOL


def test_paged_step_graph(m):
    w = workload("paged").with_(batch=4, h_q=16, h_kv=2, seed=960)
    pc = make_paged_case(w, "cpu", seq_lens=torch.tensor([300, 17, 1, 64], dtype=torch.int32))
    scale = 1.0 / math.sqrt(w.head_dim)
    ref = oracle.decode_step_paged(pc.k_pool, pc.v_pool, pc.block_table, pc.q_new, pc.k_new, pc.v_new, pc.seq_lens,
                                   pc.page_size, w.rope_base, scale, "bf16")
    lay = m.layout_paged(pc.k_pool.to(DEV), pc.v_pool.to(DEV), pc.block_table.to(DEV), w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, 300, num_splits=2, device=DEV)
    args = [x.to(DEV) for x in (pc.q_new, pc.k_new, pc.v_new, pc.pos, pc.seq_lens)]
    step = Step(lambda: m.decode_step(lay, *args, 300, bufs, w.rope_base, scale, num_splits=2), bufs)
    (eo, ee), (go, ge) = _capture_and_replay(step)
    assert ee == 0 and ge == 0
    assert torch.equal(eo, go)
    assert np.max(np.abs(go.double().numpy() - ref["out"])) <= TOL


@pytest.mark.parametrize("hq,hkv,n,paged", [(32, 4, 4, False), (32, 8, 32, False), (32, 8, 8, True)],
                         ids=["tc05_fused", "tc05_append_launch", "tc05_paged_fused"])
def test_multi_token_step_graph(m, hq, hkv, n, paged):
    """Several new tokens per sequence on the tcgen05 kernel: one launch (the
    kernel appends), or the append launch and the attention launch that
    starts while it runs; contiguous and paged."""
    w = workload("paged" if paged else "gqa4k").with_(batch=2, h_q=hq, h_kv=hkv, page_size=32, seed=970 + n)
    lens = [400, n + 33]
    q = normal((2, n, hq, 128), w.seed, 21, "bf16")
    k = normal((2, n, hkv, 128), w.seed, 22, "bf16")
    v = normal((2, n, hkv, 128), w.seed, 23, "bf16")
    scale = 1.0 / math.sqrt(128)
    if paged:
        pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=1)
        ref = oracle.decode_step_multi(pc.k_pool, pc.v_pool, q, k, v, lens, w.rope_base, scale, "bf16",
                                       block_table=pc.block_table, page_size=32)
        bt = pc.block_table.to(DEV)
        lay = m.layout_paged(pc.k_pool.to(DEV), pc.v_pool.to(DEV), bt, hq)
    else:
        c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=400)
        ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, scale, "bf16")
        lay = m.layout_contiguous(c.k_cache.to(DEV), c.v_cache.to(DEV), hq)
    bufs = m.DecodeBuffers.allocate(lay, 400, num_splits=0, device=DEV, n_new=n)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    step = Step(lambda: m.decode_step_multi(lay, n, qd, kd, vd, lens_d - n, lens_d, 400, bufs, w.rope_base, scale),
                bufs)
    (eo, ee), (go, ge) = _capture_and_replay(step)
    assert ee == 0 and ge == 0
    assert torch.equal(eo, go)
    assert np.max(np.abs(go.double().numpy().reshape(2, n, hq, 128) - ref["out"])) <= TOL


@pytest.mark.parametrize("paged", [False, True])
def test_prefill_step_graph(m, paged):
    """The prefill step (append launch + the two-query-tile prefill kernel)."""
    n, pre = 300, 20
    w = workload("paged" if paged else "gqa4k").with_(batch=2, h_q=8, h_kv=2, page_size=64, seed=980)
    lens = [pre + n, n]
    q = normal((2, n, 8, 128), w.seed, 21, "bf16")
    k = normal((2, n, 2, 128), w.seed, 22, "bf16")
    v = normal((2, n, 2, 128), w.seed, 23, "bf16")
    scale = 1.0 / math.sqrt(128)
    if paged:
        pc = make_paged_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), spare_pages=1)
        ref = oracle.decode_step_multi(pc.k_pool, pc.v_pool, q, k, v, lens, w.rope_base, scale, "bf16",
                                       block_table=pc.block_table, page_size=64)
        bt = pc.block_table.to(DEV)
        lay = m.layout_paged(pc.k_pool.to(DEV), pc.v_pool.to(DEV), bt, 8)
    else:
        c = make_contiguous_case(w, "cpu", seq_lens=torch.tensor(lens, dtype=torch.int32), capacity=pre + n)
        ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, w.rope_base, scale, "bf16")
        lay = m.layout_contiguous(c.k_cache.to(DEV), c.v_cache.to(DEV), 8)
    bufs = m.DecodeBuffers.allocate(lay, pre + n, num_splits=1, device=DEV, n_new=n)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    step = Step(lambda: m.prefill_step(lay, n, qd, kd, vd, lens_d - n, lens_d, pre + n, bufs, w.rope_base, scale),
                bufs)
    (eo, ee), (go, ge) = _capture_and_replay(step)
    assert ee == 0 and ge == 0
    assert torch.equal(eo, go)
    assert np.max(np.abs(go.double().numpy().reshape(2, n, 8, 128) - ref["out"])) <= TOL
