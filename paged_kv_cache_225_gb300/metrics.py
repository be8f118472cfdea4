"""Byte accounting for the decode-attention roofline.

The KV-cache size per token follows the "Inference optimization" lesson, section
"Caches de KV" (memory formula): 2 (K and V) x layers x KV heads x head_dim x
bytes per element.  The algorithmic bytes of one decode launch count only the
valid tokens of each sequence, so they are the minimum any kernel must move.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from .workloads import ELEM_BYTES, Workload


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """K and V bytes one token occupies across ``num_layers`` layers."""
    return 2 * num_layers * num_kv_heads * head_dim * elem_bytes


def algorithmic_bytes(w: Workload, seq_lens: Optional[np.ndarray] = None,
                      out_elem_bytes: int = 4) -> dict:
    """Minimum HBM bytes of one decode launch over ``seq_lens`` (valid tokens only).

    kv: K and V rows of every valid token; q: the query rows; out: the output
    rows; table: the block-table entries that are read plus the lengths.
    """
    cfg = w.cfg
    L = np.asarray(w.seq_lens if seq_lens is None else seq_lens, dtype=np.int64)
    tok = int(L.sum())
    row = cfg.num_kv_heads * 2 * cfg.head_dim * ELEM_BYTES[cfg.kv_dtype]
    kv = tok * row
    pages = int(((L + cfg.block_size - 1) // cfg.block_size).sum())
    q = cfg.num_seqs * cfg.num_q_heads * cfg.head_dim * ELEM_BYTES[cfg.q_dtype]
    out = cfg.num_seqs * cfg.num_q_heads * cfg.head_dim * out_elem_bytes
    table = pages * 4 + cfg.num_seqs * 4
    return {"tokens": tok, "kv": kv, "q": q, "out": out, "table": table,
            "total": kv + q + out + table, "kv_page_rounded": pages * cfg.block_size * row}
