"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function the header declares, and rejects bad arguments before it
touches CUDA."""

import ctypes

import pytest

from mqa_decode_attention_gb300 import _abi

FAKE = 0x10000  # 16-byte-aligned stand-in pointer; never dereferenced (calls fail validation first)


@pytest.fixture(scope="module")
def lib(built_lib):
    return _abi.load()


def _layout(**kw):
    base = dict(cache_dtype=_abi.MQA_BF16, batch=2, h_q=8, h_kv=2, head_dim=128, paged=0, k_cache=FAKE,
                v_cache=FAKE + 4096, capacity=256, page_size=0, num_pages=0, max_pages_per_seq=0, window=0,
                block_table=None)
    base.update(kw)
    return _abi.KVLayout(**base)


def test_exports_every_declared_function(lib):
    names = _abi.header_functions()
    assert {"kv_append_rope", "gqa_decode_attention", "splitkv_combine"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(5):
        assert lib.mqa_status_string(code)
    assert lib.mqa_status_string(0) == b"ok"


def _append(lib, lay, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, pos=FAKE, base=10000.0, q_rot=FAKE, err=FAKE)
    args.update(kw)
    return lib.kv_append_rope(ctypes.byref(lay) if lay is not None else None, args["q"], args["k"], args["v"],
                              args["pos"], args["base"], args["q_rot"], args["err"], None)


def test_append_rejects_bad_arguments(lib):
    assert _append(lib, None) == _abi.MQA_ERR_INVALID_ARG
    assert _append(lib, _layout(h_q=6, h_kv=4)) == _abi.MQA_ERR_INVALID_ARG  # h_q % h_kv != 0
    assert _append(lib, _layout(head_dim=96)) == _abi.MQA_ERR_UNSUPPORTED
    assert _append(lib, _layout(cache_dtype=7)) == _abi.MQA_ERR_UNSUPPORTED
    assert _append(lib, _layout(k_cache=None)) == _abi.MQA_ERR_INVALID_ARG
    assert _append(lib, _layout(k_cache=FAKE + 8)) == _abi.MQA_ERR_INVALID_ARG  # misaligned
    assert _append(lib, _layout(capacity=0)) == _abi.MQA_ERR_INVALID_ARG
    assert _append(lib, _layout(), pos=None) == _abi.MQA_ERR_INVALID_ARG
    assert _append(lib, _layout(), base=-1.0) == _abi.MQA_ERR_INVALID_ARG
    assert _append(lib, _layout(), base=float("nan")) == _abi.MQA_ERR_INVALID_ARG
    # paged: page size must be a power of two in [16, 256], table present
    assert _append(lib, _layout(paged=1, page_size=24, num_pages=4, max_pages_per_seq=2, block_table=FAKE)) == \
        _abi.MQA_ERR_UNSUPPORTED
    assert _append(lib, _layout(paged=1, page_size=16, num_pages=4, max_pages_per_seq=2, block_table=None)) == \
        _abi.MQA_ERR_INVALID_ARG


def _attn(lib, lay, **kw):
    a = dict(q_rot=FAKE, lens=FAKE, max_len=100, scale=0.1, splits=1, out=FAKE, out_dtype=_abi.MQA_BF16,
             lse=None, ws=None, ws_bytes=0, variant=0, err=FAKE)
    a.update(kw)
    return lib.gqa_decode_attention(ctypes.byref(lay), a["q_rot"], a["lens"], a["max_len"], a["scale"], a["splits"],
                                    a["out"], a["out_dtype"], a["lse"], a["ws"], a["ws_bytes"], a["variant"],
                                    a["err"], None)


def test_attention_rejects_bad_arguments(lib):
    lay = _layout()
    assert _attn(lib, lay, max_len=0) == _abi.MQA_ERR_INVALID_ARG
    assert _attn(lib, lay, max_len=257) == _abi.MQA_ERR_INVALID_ARG  # beyond capacity
    assert _attn(lib, lay, scale=float("inf")) == _abi.MQA_ERR_INVALID_ARG
    assert _attn(lib, lay, splits=-1) == _abi.MQA_ERR_INVALID_ARG
    assert _attn(lib, lay, out_dtype=5) == _abi.MQA_ERR_UNSUPPORTED
    assert _attn(lib, lay, variant=9) == _abi.MQA_ERR_INVALID_ARG
    assert _attn(lib, lay, out=None) == _abi.MQA_ERR_INVALID_ARG
    assert _attn(lib, _layout(window=-1)) == _abi.MQA_ERR_INVALID_ARG
    assert _attn(lib, lay, err=None) == _abi.MQA_ERR_INVALID_ARG
    # tensor cores read bf16 or uint8 caches, CUDA cores bf16 or fp32
    assert _attn(lib, _layout(cache_dtype=_abi.MQA_F32), variant=_abi.MQA_VARIANT_TENSOR_CORE) == \
        _abi.MQA_ERR_UNSUPPORTED
    # a split run needs its workspace
    assert _attn(lib, lay, splits=4) == _abi.MQA_ERR_WORKSPACE
    assert _attn(lib, lay, splits=4, ws=FAKE, ws_bytes=16) == _abi.MQA_ERR_WORKSPACE


def test_u8_layout_checks(lib):
    """A uint8 cache needs its (scale, zero) arrays, 16-byte aligned, an even
    capacity (the pairs of a kv head are copied with 16-byte strides), and the
    tensor-core kernel."""
    ok = dict(cache_dtype=_abi.MQA_U8, k_scale_zero=FAKE + 8192, v_scale_zero=FAKE + 12288)
    assert _append(lib, _layout(cache_dtype=_abi.MQA_U8)) == _abi.MQA_ERR_INVALID_ARG
    assert _append(lib, _layout(**dict(ok, k_scale_zero=FAKE + 8))) == _abi.MQA_ERR_INVALID_ARG
    assert _append(lib, _layout(**dict(ok, capacity=255))) == _abi.MQA_ERR_UNSUPPORTED
    assert _attn(lib, _layout(**dict(ok, v_scale_zero=None))) == _abi.MQA_ERR_INVALID_ARG
    assert _attn(lib, _layout(**ok), variant=_abi.MQA_VARIANT_CUDA_CORE) == _abi.MQA_ERR_UNSUPPORTED
    # paged pools have no capacity constraint
    assert _attn(lib, _layout(**dict(ok, paged=1, capacity=0, page_size=16, num_pages=4, max_pages_per_seq=2,
                                     block_table=FAKE)), max_len=32, variant=_abi.MQA_VARIANT_CUDA_CORE) == \
        _abi.MQA_ERR_UNSUPPORTED


def test_e5m2_layout_checks(lib):
    """An fp8 e5m2 cache needs no scale arrays and no capacity rule; it is
    read on tensor cores only, one new token per sequence."""
    ok = dict(cache_dtype=_abi.MQA_FP8_E5M2)
    assert _attn(lib, _layout(**ok), variant=_abi.MQA_VARIANT_CUDA_CORE) == _abi.MQA_ERR_UNSUPPORTED
    assert _attn(lib, _layout(**dict(ok, capacity=255)), variant=_abi.MQA_VARIANT_CUDA_CORE) == \
        _abi.MQA_ERR_UNSUPPORTED
    assert _attn(lib, _layout(cache_dtype=4)) == _abi.MQA_ERR_UNSUPPORTED  # no such dtype


def test_combine_rejects_bad_arguments(lib):
    assert lib.splitkv_combine(None, FAKE, 1, 1, 1, 128, FAKE, 0, None, None) == _abi.MQA_ERR_INVALID_ARG
    assert lib.splitkv_combine(FAKE, FAKE, 0, 1, 1, 128, FAKE, 0, None, None) == _abi.MQA_ERR_INVALID_ARG
    assert lib.splitkv_combine(FAKE, FAKE, 1, 1, 1, 96, FAKE, 0, None, None) == _abi.MQA_ERR_UNSUPPORTED
    assert lib.splitkv_combine(FAKE, FAKE, 1, 1, 1, 128, FAKE, 3, None, None) == _abi.MQA_ERR_UNSUPPORTED


@pytest.mark.parametrize("B,hq,d,max_len,splits,expect_splits", [
    (2, 8, 128, 256, 1, 1), (2, 8, 128, 256, 4, 4), (4, 32, 128, 131072, 64, 64), (1, 4, 64, 300, 7, 5),
    (3, 8, 64, 65, 2, 2), (3, 8, 64, 64, 2, 1),
])
def test_workspace_size_matches_split_plan(lib, B, hq, d, max_len, splits, expect_splits):
    """Explicit split counts are rounded to 64-token chunks: chunk =
    ceil(ceil(L/S)/64)*64, effective splits = ceil(L/chunk); the workspace holds
    fp32 partial outputs [B, H_q, S, d] (padded to 256 bytes) and fp32 lse [B, H_q, S]."""
    lay = _layout(batch=B, h_q=hq, h_kv=hq // 4 or 1, head_dim=d, capacity=max(max_len, 1))
    got = lib.mqa_workspace_size(ctypes.byref(lay), max_len, splits, 0)
    if expect_splits == 1:
        assert got == 0
    else:
        o = (B * hq * expect_splits * d * 4 + 255) // 256 * 256
        assert got == o + B * hq * expect_splits * 4


def test_invalid_layout_queries(lib):
    assert lib.mqa_choose_splits(None, 10, 0) == -1
    assert lib.mqa_choose_splits(ctypes.byref(_layout(h_kv=3)), 10, 0) == -1
    assert lib.mqa_workspace_size(ctypes.byref(_layout()), 0, 1, 0) == 0


@pytest.mark.parametrize("hq,hkv,n,splits,expect,fused", [
    (32, 8, 1, 1, 1, True),     # G = 4, one token: warp-MMA, append inside
    (32, 8, 1, 3, 2, True),     # ... plus the combine
    (32, 1, 1, 2, 1, True),     # MQA on tcgen05: two splits merged in a cluster
    (32, 1, 1, 3, 2, True),
    (32, 8, 8, 1, 1, True),     # 32 (token, head) rows: tcgen05, append inside
    (32, 8, 8, 2, 1, True),     # ... two splits merged
    (32, 8, 8, 4, 2, True),
    (32, 8, 16, 2, 1, True),    # 64 rows, two splits merged
    (32, 8, 32, 1, 2, False),   # 128 rows, but 32 tokens: the append launch is faster
    (64, 8, 32, 1, 2, False),   # 256 rows: two row blocks, separate append
    (64, 8, 32, 3, 3, False),
    (32, 8, 2, 1, 1, True),     # 8 rows: warp-MMA fused multi-token
    (32, 8, 16, 1, 1, True),
    (64, 8, 16, 1, 1, True),    # 128 rows, 16 tokens
])
def test_step_launches(lib, hq, hkv, n, splits, expect, fused):
    """The launch count of one step follows the routing the header states."""
    lay = _layout(batch=2, h_q=hq, h_kv=hkv, capacity=4096)
    f = ctypes.c_int32(-1)
    assert lib.mqa_step_launches(ctypes.byref(lay), n, 4096, splits, 2, ctypes.byref(f)) == expect
    assert bool(f.value) == fused


def test_step_launches_refused(lib):
    f = ctypes.c_int32(0)
    assert lib.mqa_step_launches(None, 1, 10, 1, 2, ctypes.byref(f)) == -1
    assert lib.mqa_step_launches(ctypes.byref(_layout()), 33, 4096, 1, 2, None) == -1
    assert lib.mqa_step_launches(ctypes.byref(_layout(capacity=4096)), 2, 4096, 1, 1, None) == -1  # CUDA cores, n > 1
    u8 = _layout(cache_dtype=_abi.MQA_U8, k_scale_zero=FAKE, v_scale_zero=FAKE, capacity=4096)
    assert lib.mqa_step_launches(ctypes.byref(u8), 2, 4096, 1, 2, None) == 2  # uint8: append launch + attention
