"""Pins of the oracle's several-queries-per-sequence (causal) paged attention.

Chunked prefill and speculative verification attend several new query tokens
of one sequence at once; each sees the cached rows up to its own position.
The pins tie that oracle to facts outside it: the dense masked attention of
the "Inference optimization" lesson (Step 2, scaled_dot_product_attention
with its triu mask of offset seq_len_k - seq_len_q + 1 and -1e9 fill) in
numpy, the already pinned single-query oracle run on shortened sequences,
and closed forms (the first prompt token sees only itself).
"""
import numpy as np
import pytest

import oracle
from paged_kv_cache_225_gb300 import workloads as W

F32, BF16, FP8 = W.F32, W.BF16, W.FP8_E5M2


def _problem(kv_dtype, q_dtype, lens, nq, Hq=4, Hkv=2, D=16, B=16, seed=0, kv_scale=1.0):
    rng = np.random.default_rng(seed)
    S = len(lens)
    nb = [(L + B - 1) // B for L in lens]
    N = sum(nb) + 3
    ids = rng.permutation(N).astype(np.int32)
    tables = np.full((S, max(nb) + 1), -1, dtype=np.int32)
    c = 0
    for s in range(S):
        tables[s, :nb[s]] = ids[c:c + nb[s]]
        c += nb[s]
    q_start = np.zeros(S + 1, dtype=np.int32)
    q_start[1:] = np.cumsum(nq)
    T = int(q_start[-1])
    k = W.round_to_storage(rng.standard_normal((N, Hkv, D, B)).astype(np.float32), kv_dtype)
    v = W.round_to_storage(rng.standard_normal((N, Hkv, D, B)).astype(np.float32), kv_dtype)
    q = W.round_to_storage(rng.standard_normal((T, Hq, D)).astype(np.float32), q_dtype)
    return dict(q=q, q_dtype=q_dtype, q_start=q_start, k_cache=k, v_cache=v,
                kv_dtype=kv_dtype, block_tables=tables, seq_lens=np.array(lens, np.int32),
                scale=1.0 / np.sqrt(D), k_scale=kv_scale, v_scale=kv_scale)


def _prefill(p, **kw):
    return oracle.paged_prefill(p["q"], p["q_dtype"], p["q_start"], p["k_cache"], p["v_cache"],
                                p["kv_dtype"], p["block_tables"], p["seq_lens"], p["scale"],
                                k_scale=p["k_scale"], v_scale=p["v_scale"], **kw)


def _dense(p, s):
    """Logical K, V [Hkv, L, D] of sequence s by numpy fancy indexing (float64)."""
    k = W.storage_to_float32(p["k_cache"], p["kv_dtype"]).astype(np.float64)
    v = W.storage_to_float32(p["v_cache"], p["kv_dtype"]).astype(np.float64)
    if p["kv_dtype"] in W.SCALED:
        k, v = k * p["k_scale"], v * p["v_scale"]
    L = int(p["seq_lens"][s])
    B = k.shape[3]
    nb = (L + B - 1) // B
    blocks = p["block_tables"][s, :nb]
    ks = k[blocks].transpose(1, 0, 3, 2).reshape(k.shape[1], nb * B, k.shape[2])[:, :L]
    vs = v[blocks].transpose(1, 0, 3, 2).reshape(v.shape[1], nb * B, v.shape[2])[:, :L]
    return ks, vs


def _masked_sdpa(query, keys, values, scale):
    """The lesson's dense attention for a block of queries: additive -1e9 on the
    keys above the shifted diagonal, max subtraction, normalised weights."""
    scores = (query @ keys.T) * scale
    lq, lk = scores.shape
    if lq > 1:
        mask = np.triu(np.ones((lq, lk)), k=lk - lq + 1)
        scores = scores + mask * (-1e9)
    e = np.exp(scores - scores.max(axis=-1, keepdims=True))
    return (e / e.sum(axis=-1, keepdims=True)) @ values


@pytest.mark.parametrize("kv_dtype,q_dtype,kv_scale",
                         [(F32, F32, 1.0), (BF16, BF16, 1.0), (FP8, BF16, 0.5),
                          (W.FP8_E4M3, BF16, 0.25), (W.INT4, BF16, 0.5)])
def test_prefill_equals_dense_masked_sdpa(kv_dtype, q_dtype, kv_scale):
    lens, nq = (1, 17, 40, 33), (1, 5, 40, 16)
    p = _problem(kv_dtype, q_dtype, lens, nq, kv_scale=kv_scale, seed=1)
    got = _prefill(p)
    qd = W.storage_to_float32(p["q"], q_dtype).astype(np.float64)
    G = qd.shape[1] // p["k_cache"].shape[1]
    for s in range(len(lens)):
        ks, vs = _dense(p, s)
        r0, r1 = p["q_start"][s], p["q_start"][s + 1]
        for h in range(qd.shape[1]):
            ref = _masked_sdpa(qd[r0:r1, h], ks[h // G], vs[h // G], p["scale"])
            np.testing.assert_allclose(got[r0:r1, h], ref, rtol=0, atol=1e-12)


def test_each_query_equals_decode_of_its_prefix():
    lens, nq = (23, 48, 9), (7, 20, 9)
    p = _problem(BF16, BF16, lens, nq, seed=2)
    got = _prefill(p)
    for s, (L, n) in enumerate(zip(lens, nq)):
        for i in range(n):
            row = p["q_start"][s] + i
            lens_i = np.array(lens, np.int32)
            lens_i[s] = L - n + i + 1
            q1 = np.repeat(p["q"][row:row + 1], len(lens), axis=0)
            ref = oracle.paged_decode(q1, BF16, p["k_cache"], p["v_cache"], BF16,
                                      p["block_tables"], lens_i, p["scale"])
            assert np.array_equal(got[row], ref[s])


def test_one_query_per_sequence_is_decode():
    lens = (1, 30, 64, 5)
    p = _problem(BF16, BF16, lens, (1, 1, 1, 1), seed=3)
    ref = oracle.paged_decode(p["q"], BF16, p["k_cache"], p["v_cache"], BF16,
                              p["block_tables"], p["seq_lens"], p["scale"])
    assert np.array_equal(_prefill(p), ref)


def test_first_prompt_token_sees_only_itself():
    lens = (12, 35)
    p = _problem(F32, F32, lens, lens, seed=4)
    got = _prefill(p)
    for s in range(2):
        ks, vs = _dense(p, s)
        G = got.shape[1] // vs.shape[0]
        for h in range(got.shape[1]):
            assert np.array_equal(got[p["q_start"][s], h], vs[h // G, 0])


@pytest.mark.parametrize("part", [16, 32, 48])
def test_prefill_split_merge_equals_single_softmax(part):
    p = _problem(BF16, BF16, (70, 129, 16), (70, 9, 3), seed=5)
    np.testing.assert_allclose(_prefill(p, partition_tokens=part), _prefill(p),
                               rtol=0, atol=1e-13)


def test_sequences_without_queries_write_nothing():
    p = _problem(BF16, BF16, (20, 31, 7), (0, 4, 0), seed=6)
    got = _prefill(p)
    assert got.shape[0] == 4 and np.all(np.isfinite(got))
    ks, vs = _dense(p, 1)
    G = got.shape[1] // vs.shape[0]
    qd = W.storage_to_float32(p["q"], BF16).astype(np.float64)
    for h in range(got.shape[1]):
        ref = _masked_sdpa(qd[0:4, h], ks[h // G], vs[h // G], p["scale"])
        np.testing.assert_allclose(got[0:4, h], ref, rtol=0, atol=1e-12)


def test_more_queries_than_tokens_is_rejected():
    p = _problem(BF16, BF16, (5, 8), (6, 1), seed=7)
    with pytest.raises(ValueError):
        _prefill(p)
