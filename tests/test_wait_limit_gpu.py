"""GPU: the bounded-wait failure path.

Every wait of an attention kernel for another warp's progress gives up after
the layout's wait_limit_ns; the kernel then sets MQA_DEVERR_TIMEOUT, lets its
own copies and tensor-core products in flight complete, and returns. With a
limit of 1 ns every wait that is not satisfied at once runs out (a tile takes
at least a memory round trip to land), so each launch below takes the timeout
path, at whichever waits it happens to hit first. The call must come back
(the stream synchronises), report the timeout, and leave the stream and the
library usable: the same step with the default limit right after it, on the
same stream, matches the oracle.

Kernels covered: the warp-MMA kernel (fused one-launch step; split with the
combine), the paged head-group kernel, the tcgen05 MQA kernel (one split and
a two-block cluster), the CUDA-core kernel, the uint8 warp-MMA kernel and the
prefill kernel (contiguous and paged).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import make_contiguous_case, make_paged_case, make_u8_cache, workload

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = 2e-2


@pytest.fixture(scope="module")
def m(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mqa_decode_attention_gb300 as mod

    mod.library()
    return mod


def _np(t):
    return t.detach().cpu().to(torch.float64).numpy()


CASES = {
    # name: (workload, batch, h_q, h_kv, lens, splits, variant, cache)
    "warp_mma_fused": ("gqa4k", 2, 32, 8, [1000, 300], 1, 2, "bf16"),
    "warp_mma_split_combine": ("gqa4k", 2, 32, 8, [1000, 300], 3, 2, "bf16"),
    "paged_head_group": ("paged", 3, 16, 4, [700, 64, 17], 1, 2, "bf16"),
    "tc05_mqa": ("gqa4k", 2, 32, 1, [1000, 700], 1, 2, "bf16"),
    "tc05_mqa_cluster": ("gqa4k", 2, 32, 1, [1000, 700], 2, 2, "bf16"),
    "cuda_core": ("gqa4k", 2, 8, 2, [1000, 300], 2, 1, "bf16"),
    "u8_warp_mma": ("gqa4k", 2, 32, 8, [1000, 300], 1, 2, "u8"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_timeout_then_normal_call(m, name):
    wl, B, hq, hkv, lens, splits, variant, cache = CASES[name]
    w = workload(wl).with_(batch=B, h_q=hq, h_kv=hkv, seed=900 + len(name))
    L = torch.tensor(lens, dtype=torch.int32)
    max_len = int(L.max())
    scale = 1.0 / math.sqrt(w.head_dim)
    if w.paged:
        c = make_paged_case(w, "cpu", seq_lens=L)
        kc, vc, bt = c.k_pool.to(DEV), c.v_pool.to(DEV), c.block_table.to(DEV)
        lay = m.layout_paged(kc, vc, bt, hq)
        ref = oracle.decode_step_paged(c.k_pool, c.v_pool, c.block_table, c.q_new, c.k_new, c.v_new, L,
                                       c.page_size, w.rope_base, scale, "bf16")
    elif cache == "u8":
        c = make_contiguous_case(w, "cpu", seq_lens=L, capacity=1024)
        u = make_u8_cache((B, hkv, 1024), w.head_dim, 41)
        kc, vc, ks, vs = u.k_codes.to(DEV), u.v_codes.to(DEV), u.k_sz.to(DEV), u.v_sz.to(DEV)
        lay = m.layout_contiguous(kc, vc, hq, k_scale_zero=ks, v_scale_zero=vs)
        ref = oracle.decode_step_u8(u.k_codes, u.k_sz, u.v_codes, u.v_sz, c.q_new, c.k_new, c.v_new, L, w.rope_base,
                                    scale)
    else:
        c = make_contiguous_case(w, "cpu", seq_lens=L, capacity=1024)
        kc, vc = c.k_cache.to(DEV), c.v_cache.to(DEV)
        lay = m.layout_contiguous(kc, vc, hq)
        ref = oracle.decode_step_contiguous(c.k_cache, c.v_cache, c.q_new, c.k_new, c.v_new, L, w.rope_base, scale,
                                            "bf16")
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=splits, variant=variant, device=DEV)
    args = (c.q_new.to(DEV), c.k_new.to(DEV), c.v_new.to(DEV), c.pos.to(DEV), L.to(DEV))

    # a limit no wait can meet: the launch takes the timeout path and comes back
    lay.wait_limit_ns = 1
    bufs.err.zero_()
    m.decode_step(lay, *args, max_len, bufs, w.rope_base, scale, num_splits=splits, variant=variant)
    torch.cuda.synchronize()
    err = int(bufs.err.item())
    assert err & m.MQA_DEVERR_TIMEOUT, (name, hex(err))

    # the default limit, same stream, same inputs (the timed-out launch wrote
    # the same new rows this one writes): the oracle's result
    lay.wait_limit_ns = 0
    bufs.err.zero_()
    bufs.out.fill_(float("nan"))
    m.decode_step(lay, *args, max_len, bufs, w.rope_base, scale, num_splits=splits, variant=variant)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0, name
    assert np.max(np.abs(_np(bufs.out) - ref["out"])) <= TOL, name
    assert np.max(np.abs(_np(bufs.lse) - ref["lse"])) <= TOL, name


@pytest.mark.parametrize("paged", [False, True])
def test_prefill_timeout_then_normal_call(m, paged):
    """The prefill kernel (two query tiles per block, contiguous and paged)
    takes the same timeout path."""
    n, B, hq, hkv = 300, 2, 8, 2
    lens = [n + 40, n]
    L = torch.tensor(lens, dtype=torch.int32)
    scale = 1.0 / math.sqrt(128)
    gen = torch.Generator().manual_seed(911)
    q = torch.randn((B, n, hq, 128), generator=gen).to(torch.bfloat16)
    k = torch.randn((B, n, hkv, 128), generator=gen).to(torch.bfloat16)
    v = torch.randn((B, n, hkv, 128), generator=gen).to(torch.bfloat16)
    if paged:
        w = workload("paged").with_(batch=B, h_q=hq, h_kv=hkv, page_size=32, seed=912)
        c = make_paged_case(w, "cpu", seq_lens=L, spare_pages=1)
        pools = (c.k_pool.to(DEV), c.v_pool.to(DEV))
        bt = c.block_table.to(DEV)
        lay = m.layout_paged(pools[0], pools[1], bt, hq)
        ref = oracle.decode_step_multi(c.k_pool, c.v_pool, q, k, v, lens, 10000.0, scale, "bf16",
                                       block_table=c.block_table, page_size=32)
    else:
        w = workload("gqa4k").with_(batch=B, h_q=hq, h_kv=hkv, seed=912)
        c = make_contiguous_case(w, "cpu", seq_lens=L, capacity=n + 40)
        caches = (c.k_cache.to(DEV), c.v_cache.to(DEV))
        lay = m.layout_contiguous(caches[0], caches[1], hq)
        ref = oracle.decode_step_multi(c.k_cache, c.v_cache, q, k, v, lens, 10000.0, scale, "bf16")
    bufs = m.DecodeBuffers.allocate(lay, max(lens), num_splits=1, device=DEV, n_new=n)
    Ld = L.to(DEV)
    args = (q.to(DEV), k.to(DEV), v.to(DEV), (Ld - n).to(torch.int32), Ld, max(lens), bufs, 10000.0, scale)

    lay.wait_limit_ns = 1
    bufs.err.zero_()
    m.prefill_step(lay, n, *args)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) & m.MQA_DEVERR_TIMEOUT, hex(int(bufs.err.item()))

    # the default limit, same inputs (the append wrote the same rows): the oracle
    lay.wait_limit_ns = 0
    bufs.err.zero_()
    bufs.out.fill_(float("nan"))
    m.prefill_step(lay, n, *args)
    torch.cuda.synchronize()
    assert int(bufs.err.item()) == 0
    out = _np(bufs.out).reshape(ref["out"].shape)
    assert np.max(np.abs(out - ref["out"])) <= TOL
