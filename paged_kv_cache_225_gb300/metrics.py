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


def prefill_algorithmic(w, out_elem_bytes: int = 4) -> dict:
    """Minimum HBM bytes and the flops of one several-queries attention launch.

    Every (sequence, KV head) must read the K/V rows of its valid tokens once,
    whatever its number of queries; q and out are read / written once; the
    table entries and lengths are read once.  Flops count the multiply-adds of
    q.k and p.v over each query's visible rows (causal), two flops each.
    """
    base = w.cfg.base
    L = np.asarray(w.seq_lens, dtype=np.int64)
    n = np.diff(np.asarray(w.q_start, dtype=np.int64))
    row = base.num_kv_heads * 2 * base.head_dim * ELEM_BYTES[base.kv_dtype]
    kv = int(L.sum()) * row
    pages = int(((L + base.block_size - 1) // base.block_size).sum())
    T = int(n.sum())
    q = T * base.num_q_heads * base.head_dim * ELEM_BYTES[base.q_dtype]
    out = T * base.num_q_heads * base.head_dim * out_elem_bytes
    table = pages * 4 + (2 * L.size + 1) * 4
    # Query i of a sequence sees L - n + i + 1 rows.
    visible = int(((L - n) * n + n * (n + 1) // 2).sum())
    flops = 4 * base.head_dim * base.num_q_heads * visible
    return {"tokens": int(L.sum()), "queries": T, "kv": kv, "q": q, "out": out, "table": table,
            "total": kv + q + out + table, "flops": flops, "visible_rows": visible}
