"""KV-cache size accounting, as the pages state it.

TEST INFRASTRUCTURE (see oracle/decode.py): used by the oracle's pins only.

  * "Grouped-query attention: berbagi KV head ..." (nalar.dev), section
    "Ukuran KV cache mengikuti jumlah KV head": one layer stores
    2 x T x H_kv x d scalars (key and value for every stored position).
  * "Arsitektur Inferensi LLM ..." (tveniu.com), section 2 "Kalkulus Memori
    KV-Cache": bytes per token = 2 x n_layers x n_kv_heads x d_head x
    bytes_per_element; total = bytes per token x seq_len x batch.
  * "KV Cache" explainer (lensaml.com), Langkah 5 and FAQ: the same product,
    cache per token = 2 x layers x kv_heads x head_dim x bytes.
  * "Arsitektur Inferensi LLM ..." (tveniu.com), section 7 (speculative
    decoding): with per-draft acceptance rate alpha and gamma drafted
    tokens, one verification pass yields (1 - alpha^(gamma+1)) / (1 - alpha)
    tokens in expectation (3.69 for alpha = 0.8, gamma = 5).
  * fahmindra.github.io bab 2.5.1: the formula's factors l (layers),
    u (batch), n (heads), b (head size), z (sequence length), a first 2 for
    K and V and a second 2 for 16-bit bytes (the formula itself was lost in
    extraction; this is the product of the factors the page lists).
"""

from __future__ import annotations


def layer_cache_scalars(tokens: int, h_kv: int, head_dim: int) -> int:
    """Scalars one layer's cache holds: 2 * T * H_kv * d."""
    return 2 * tokens * h_kv * head_dim


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    """2 * layers * kv_heads * head_dim * bytes."""
    return 2 * n_layers * n_kv_heads * head_dim * bytes_per_elem


def kv_cache_bytes(n_layers: int, n_kv_heads: int, head_dim: int, bytes_per_elem: int, seq_len: int,
                   batch: int) -> int:
    """Bytes per token x tokens x sequences."""
    return kv_bytes_per_token(n_layers, n_kv_heads, head_dim, bytes_per_elem) * seq_len * batch


def projection_counts_closed_form(prompt_len: int, evals: int) -> tuple[int, int]:
    """K/V projections per layer without and with the cache ("KV Cache"
    explainer, Langkah 2): T*P + T(T-1)/2 versus P + T - 1."""
    p, t = prompt_len, evals
    return t * p + t * (t - 1) // 2, p + t - 1


def expected_tokens_per_verify(alpha: float, gamma: int) -> float:
    """Expected tokens one verification pass yields ("Arsitektur Inferensi
    LLM", section 7): the accepted prefix of the gamma drafts plus the one
    token the target model supplies, each draft accepted with probability
    alpha while all before it were: sum_{k=0..gamma} alpha^k
    = (1 - alpha^(gamma+1)) / (1 - alpha)."""
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)
