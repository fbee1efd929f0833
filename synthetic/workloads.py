"""The five decode workloads: shapes, cache dtype, length mix and seed.

Each is named for what it is. The shapes follow the Llama-style GQA, MQA,
paged and long-context decode batches the pages discuss (Llama 3 uses 8 KV
heads for 32 query heads; PagedAttention blocks of 16 tokens; contexts up to
128K tokens). Lengths are the sequence length AFTER the new token is
appended, so the new token sits at position ``seq_len - 1``.
"""

from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    h_q: int
    h_kv: int
    head_dim: int
    dtype: str  # cache / q / k / v / output dtype: "bf16" or "f32"
    seq_len: int = 0  # contiguous: every sequence has this length after append
    paged: bool = False
    page_size: int = 16
    len_lo: int = 0  # paged: lengths uniform on the integers [len_lo, len_hi]
    len_hi: int = 0
    num_splits: int = 0  # 0 = let the library choose
    rope_base: float = 10000.0
    seed: int = 0
    prompt_len: int = 0  # tiny sequence workload: prompt length P
    decode_evals: int = 0  # tiny sequence workload: attention evaluations T

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    @property
    def esize(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    # fp32 debug sequence: P=5 prompt tokens, then decoding until 16 attention
    # evaluations have run (queries at positions 4..19), one token at a time.
    "tiny": Workload(
        "tiny", batch=1, h_q=4, h_kv=2, head_dim=64, dtype="f32",
        seq_len=20, prompt_len=5, decode_evals=16, seed=1001,
    ),
    "gqa4k": Workload(
        "gqa4k", batch=32, h_q=32, h_kv=8, head_dim=128, dtype="bf16",
        seq_len=4096, seed=1002,
    ),
    "mqa8k": Workload(
        "mqa8k", batch=64, h_q=32, h_kv=1, head_dim=128, dtype="bf16",
        seq_len=8192, seed=1003,
    ),
    "paged": Workload(
        "paged", batch=128, h_q=64, h_kv=8, head_dim=128, dtype="bf16",
        paged=True, page_size=16, len_lo=128, len_hi=16384, seed=1004,
    ),
    "long": Workload(
        "long", batch=4, h_q=32, h_kv=8, head_dim=128, dtype="bf16",
        seq_len=131072, num_splits=64, seed=1005,
    ),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]
