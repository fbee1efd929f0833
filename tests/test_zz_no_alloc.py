"""gqa_decode_attention_noalloc: the attention call that allocates nothing.

Some callers cannot allocate device memory (a plugin inside a process whose
framework already holds the device memory, or a loop that must not take
cudaMalloc's device synchronisation); this entry point keeps its split
scratch in a fixed array inside the library. The test calls it through the
C ABI twice in a row and checks each result against gqa_decode_attention
with a caller-allocated workspace, and the first one also directly against
the fp64 oracle (outputs <= 2e-2, lse <= 1e-4 of the log-sum-exp over the
scores the kernel forms). This file is collected last.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from lse_model import assert_lse, paged_keys
from mqa_decode_attention_gb300 import _abi
from synthetic import make_contiguous_case, make_paged_case, workload

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def lib(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _abi.load()
    fn = lib.gqa_decode_attention_noalloc
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(_abi.KVLayout), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                   ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                   ctypes.c_void_p]
    return lib


def _case(paged: bool, seed: int):
    import mqa_decode_attention_gb300 as m

    dev = "cuda"
    if paged:
        w = workload("paged").with_(batch=4, h_q=16, h_kv=2, seed=seed)
        c = make_paged_case(w, dev, seq_lens=torch.tensor([1000, 17, 1, 640], dtype=torch.int32))
        lay = m.layout_paged(c.k_pool, c.v_pool, c.block_table, w.h_q)
    else:
        w = workload("gqa4k").with_(batch=3, h_q=32, h_kv=8, seed=seed)
        c = make_contiguous_case(w, dev, seq_lens=torch.tensor([1000, 333, 64], dtype=torch.int32), capacity=1024)
        lay = m.layout_contiguous(c.k_cache, c.v_cache, w.h_q)
    q_rot = torch.randn(w.batch, w.h_q, w.head_dim, device=dev, generator=torch.Generator(dev).manual_seed(seed))
    return w, c, lay, q_rot


def _oracle(w, c, paged, q_rot, scale):
    """Attention of the given q_rot over each sequence's logical cache (fp64)."""
    lens = c.seq_lens.cpu().numpy()
    if paged:
        keys = paged_keys(c.k_pool.cpu().double().numpy(), c.block_table.cpu(), lens, c.page_size)
        vals = paged_keys(c.v_pool.cpu().double().numpy(), c.block_table.cpu(), lens, c.page_size)
    else:
        keys, vals = c.k_cache.cpu().double().numpy(), c.v_cache.cpu().double().numpy()
    q = q_rot.cpu().double().numpy()
    out = np.empty(q.shape)
    lse = np.empty(q.shape[:2])
    for b, L in enumerate(lens):
        out[b], lse[b] = oracle.gqa_attention(q[b], keys[b, :, :L], vals[b, :, :L], scale)
    return out, lse, keys


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("variant", [1, 2])
def test_noalloc_matches_workspace_call(lib, paged, variant):
    w, c, lay, q_rot = _case(paged, 7 + variant)
    stream = torch.cuda.current_stream().cuda_stream
    scale = 1.0 / math.sqrt(w.head_dim)
    splits = 5
    ws_bytes = lib.mqa_workspace_size(ctypes.byref(lay), 1000, splits, variant)
    assert ws_bytes > 0
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for call in range(2):
        ref = torch.empty(w.batch, w.h_q, w.head_dim, dtype=torch.bfloat16, device="cuda")
        got = torch.full_like(ref, float("nan"))
        ref_lse = torch.empty(w.batch, w.h_q, device="cuda")
        got_lse = torch.full_like(ref_lse, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        qr = q_rot * (1.0 + call)  # a different query on the second call
        st = lib.gqa_decode_attention(ctypes.byref(lay), qr.data_ptr(), c.seq_lens.data_ptr(), 1000, scale, splits,
                                      ref.data_ptr(), _abi.MQA_BF16, ref_lse.data_ptr(), ws.data_ptr(), ws_bytes,
                                      variant, err.data_ptr(), stream)
        assert st == 0
        st = lib.gqa_decode_attention_noalloc(ctypes.byref(lay), qr.data_ptr(), c.seq_lens.data_ptr(), 1000, scale,
                                              splits, got.data_ptr(), _abi.MQA_BF16, got_lse.data_ptr(), variant,
                                              err.data_ptr(), stream)
        assert st == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.isfinite(got.float()).all()
        assert (got.float() - ref.float()).abs().max().item() <= TOL
        assert (got_lse - ref_lse).abs().max().item() <= TOL
        if call == 0:
            o, l, keys = _oracle(w, c, paged, qr, scale)
            assert np.max(np.abs(got.double().cpu().numpy() - o)) <= TOL
            assert np.max(np.abs(got_lse.double().cpu().numpy() - l)) <= TOL
            assert_lse(got_lse.double().cpu().numpy(), qr.double().cpu().numpy(), keys, c.seq_lens.cpu().numpy(),
                       scale, "bf16" if variant == 2 else "f32")


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    """A split whose partial results exceed the 32 MiB scratch is refused
    before anything is launched (the cache is real, so even a launch would
    stay in bounds)."""
    import mqa_decode_attention_gb300 as m

    B, hq, hkv, L = 256, 64, 8, 1024
    big = torch.zeros(B, hkv, L, 128, dtype=torch.bfloat16, device="cuda")
    lay = m.layout_contiguous(big, big, hq)
    need = lib.mqa_workspace_size(ctypes.byref(lay), L, 16, 2)  # 16384 rows x 16 splits x 129 floats
    assert need > 32 << 20
    out = torch.empty(B, hq, 128, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(B, hq, 128, device="cuda")
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = lib.gqa_decode_attention_noalloc(ctypes.byref(lay), q.data_ptr(), lens.data_ptr(), L, 0.1, 16,
                                          out.data_ptr(), _abi.MQA_BF16, None, 2, err.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
    assert st == _abi.MQA_ERR_WORKSPACE
