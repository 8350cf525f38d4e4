"""Algorithmic work of the hot path: the bytes and flops a step must move or
compute, independent of how a kernel does it. Used for roofline fractions.

[vLLM-wiki "배경: LLM 서빙은 메모리 문제다"] states the KV footprint of one token
as 2 (K and V) x hidden width x layers x bytes per element (OPT-13B: 800 KB per
token); with GQA the width is num_kv_heads x head_dim.
"""
from typing import Iterable, Sequence

import numpy as np


def kv_bytes_per_token(num_kv_heads: int, head_dim: int, elt_bytes: int,
                       num_layers: int = 1) -> int:
    """Bytes of K plus V stored for one token."""
    return 2 * num_kv_heads * head_dim * elt_bytes * num_layers


def decode_kv_bytes(seq_lens: Iterable[int], num_kv_heads: int, head_dim: int,
                    elt_bytes: int) -> int:
    """Logical KV bytes a decode step reads: every visible key and value once
    per request (each (request, kv head) pair streams its context once)."""
    return int(sum(int(s) for s in seq_lens)) * kv_bytes_per_token(num_kv_heads, head_dim,
                                                                   elt_bytes)


def unique_kv_bytes(tables: np.ndarray, seq_lens: Sequence[int], block_size: int,
                    num_kv_heads: int, head_dim: int, elt_bytes: int) -> int:
    """KV bytes of the distinct physical blocks that hold visible tokens
    (shared prefix blocks counted once); partial last blocks count their
    used slots only."""
    used = {}
    for r, s in enumerate(seq_lens):
        s = int(s)
        for i in range(-(-s // block_size)):
            b = int(tables[r][i])
            used[b] = max(used.get(b, 0), min(block_size, s - i * block_size))
    return sum(used.values()) * kv_bytes_per_token(num_kv_heads, head_dim, elt_bytes)


def causal_pairs(q_len: int, seq_len: int) -> int:
    """Visible (query, key) pairs of a causal chunk of q_len queries at the end
    of a seq_len-token context: query j (0-based) at position P + j sees
    P + j + 1 keys, P = seq_len - q_len."""
    P = seq_len - q_len
    return q_len * P + q_len * (q_len + 1) // 2


def attention_flops(pairs: int, num_q_heads: int, head_dim: int) -> int:
    """2 flops per multiply-add for q.k and for p.v: 4 * D per pair per head."""
    return 4 * head_dim * num_q_heads * int(pairs)
