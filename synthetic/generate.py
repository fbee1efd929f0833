"""Seeded tensors for the decode workloads.

Values are N(0, 1) drawn by torch's seeded generator in fp32 and rounded
(round-to-nearest-even, torch's conversion) to the cache dtype. Every role
(q, k, v, cached K, cached V, lengths, page permutation) has its own stream,
so changing one shape never shifts another role's values. Generation on a
CUDA device gives different (equally valid) values than on the CPU for the
same seed; callers that compare against the oracle copy the inputs they
generated, they never regenerate them on the other device.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from .workloads import Workload

# stream ids: one per tensor role
S_Q, S_K, S_V, S_KC, S_VC, S_LEN, S_PERM = 1, 2, 3, 4, 5, 6, 7


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _generator(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + stream)
    return g


def normal(shape, seed: int, stream: int, dtype: str = "bf16", device="cpu") -> torch.Tensor:
    """N(0,1) samples of ``shape`` rounded to ``dtype`` ("bf16" or "f32")."""
    g = _generator(seed, stream, device)
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    return x.to(torch_dtype(dtype))


def paged_lengths(w: Workload) -> torch.Tensor:
    """Sequence lengths (after append) uniform on the integers [len_lo, len_hi]."""
    g = _generator(w.seed, S_LEN, "cpu")
    return torch.randint(w.len_lo, w.len_hi + 1, (w.batch,), generator=g, dtype=torch.int64).to(torch.int32)


@dataclass
class ContiguousCase:
    k_cache: torch.Tensor  # [B, H_kv, capacity, d]
    v_cache: torch.Tensor
    q_new: torch.Tensor  # [B, H_q, d]
    k_new: torch.Tensor  # [B, H_kv, d]
    v_new: torch.Tensor
    seq_lens: torch.Tensor  # [B] int32, length after append
    pos: torch.Tensor  # [B] int32 = seq_lens - 1
    capacity: int


@dataclass
class PagedCase:
    k_pool: torch.Tensor  # [num_pages, H_kv, page_size, d]
    v_pool: torch.Tensor
    block_table: torch.Tensor  # [B, max_pages] int32, unused entries -1
    q_new: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    seq_lens: torch.Tensor
    pos: torch.Tensor
    page_size: int
    num_pages: int
    max_pages: int


def _new_token(w: Workload, device):
    q = normal((w.batch, w.h_q, w.head_dim), w.seed, S_Q, w.dtype, device)
    k = normal((w.batch, w.h_kv, w.head_dim), w.seed, S_K, w.dtype, device)
    v = normal((w.batch, w.h_kv, w.head_dim), w.seed, S_V, w.dtype, device)
    return q, k, v


def make_contiguous_case(w: Workload, device="cpu", seq_lens=None, capacity: int | None = None) -> ContiguousCase:
    """Contiguous cache prefilled with N(0,1) values (taken as already rotated)."""
    if seq_lens is None:
        seq_lens = torch.full((w.batch,), w.seq_len, dtype=torch.int32)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32).cpu()
    cap = int(capacity if capacity is not None else int(seq_lens.max()))
    shape = (w.batch, w.h_kv, cap, w.head_dim)
    kc = normal(shape, w.seed, S_KC, w.dtype, device)
    vc = normal(shape, w.seed, S_VC, w.dtype, device)
    q, k, v = _new_token(w, device)
    sl = seq_lens.to(device)
    return ContiguousCase(kc, vc, q, k, v, sl, (sl - 1).to(torch.int32), cap)


def make_paged_case(w: Workload, device="cpu", seq_lens=None, spare_pages: int = 0) -> PagedCase:
    """Paged pool whose pages are dealt to the sequences by a seeded permutation.

    Sequence b owns ceil(L_b / page_size) pages; its logical block i maps to
    physical page ``perm[offset_b + i]``. Unused table entries are -1.
    """
    if seq_lens is None:
        seq_lens = paged_lengths(w)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32).cpu()
    ps = w.page_size
    npages_seq = (seq_lens.to(torch.int64) + ps - 1) // ps
    total = int(npages_seq.sum()) + spare_pages
    max_pages = int(max(int(npages_seq.max()), (max(w.len_hi, int(seq_lens.max())) + ps - 1) // ps))
    g = _generator(w.seed, S_PERM, "cpu")
    perm = torch.randperm(total, generator=g).to(torch.int32)
    table = torch.full((w.batch, max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(w.batch):
        n = int(npages_seq[b])
        table[b, :n] = perm[off:off + n]
        off += n
    shape = (total, w.h_kv, ps, w.head_dim)
    kp = normal(shape, w.seed, S_KC, w.dtype, device)
    vp = normal(shape, w.seed, S_VC, w.dtype, device)
    q, k, v = _new_token(w, device)
    sl = seq_lens.to(device)
    return PagedCase(kp, vp, table.to(device), q, k, v, sl, (sl - 1).to(torch.int32), ps, total, max_pages)


@dataclass
class TinySequence:
    """Raw (un-rotated) per-position q, k, v of one short sequence batch."""

    q: torch.Tensor  # [T_total, B, H_q, d]
    k: torch.Tensor  # [T_total, B, H_kv, d]
    v: torch.Tensor
    prompt_len: int
    decode_evals: int


def make_tiny_sequence(w: Workload, prompt_len: int | None = None, decode_evals: int | None = None) -> TinySequence:
    p = w.prompt_len if prompt_len is None else prompt_len
    t = w.decode_evals if decode_evals is None else decode_evals
    n = p + t - 1  # positions that ever receive a K/V slice
    q = normal((n, w.batch, w.h_q, w.head_dim), w.seed, S_Q, w.dtype)
    k = normal((n, w.batch, w.h_kv, w.head_dim), w.seed, S_K, w.dtype)
    v = normal((n, w.batch, w.h_kv, w.head_dim), w.seed, S_V, w.dtype)
    return TinySequence(q, k, v, p, t)


@dataclass
class U8Cache:
    """A uint8 cache drawn directly: codes uniform on [0, 255], scale and
    zero point as a quantised N(0,1) row would have them (scale about
    6 / 255, zero point about 128), one pair per (token, kv head)."""

    k_codes: torch.Tensor
    k_sz: torch.Tensor  # float32 [..., 2] (scale, zero_point)
    v_codes: torch.Tensor
    v_sz: torch.Tensor


S_KQ, S_VQ, S_KS, S_VS = 8, 9, 10, 11


def make_u8_cache(shape_rows, head_dim: int, seed: int, device="cpu") -> U8Cache:
    """shape_rows: the leading shape of the cache rows ([B, H_kv, capacity] or
    [num_pages, H_kv, page_size])."""
    out = []
    for sc, ss in ((S_KQ, S_KS), (S_VQ, S_VS)):
        g = _generator(seed, sc, device)
        codes = torch.randint(0, 256, tuple(shape_rows) + (head_dim,), generator=g, device=device,
                              dtype=torch.int32).to(torch.uint8)
        g2 = _generator(seed, ss, device)
        scale = (5.0 + 2.0 * torch.rand(tuple(shape_rows), generator=g2, device=device)) / 255.0
        zp = torch.randint(100, 156, tuple(shape_rows), generator=g2, device=device).to(torch.float32)
        out += [codes, torch.stack([scale.to(torch.float32), zp], dim=-1).contiguous()]
    return U8Cache(*out)


# fp8 e5m2 caches: streams of their own
S_K8, S_V8 = 12, 13


def make_e5m2_cache(shape_rows, head_dim: int, seed: int, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """K and V caches in torch.float8_e5m2: N(0, 1) values rounded by torch's
    conversion. shape_rows: [B, H_kv, capacity] or [num_pages, H_kv, page_size]."""
    out = []
    for st in (S_K8, S_V8):
        g = _generator(seed, st, device)
        x = torch.randn(tuple(shape_rows) + (head_dim,), generator=g, device=device, dtype=torch.float32)
        out.append(x.to(torch.float8_e5m2))
    return out[0], out[1]
