"""GPU parity of causal paged attention with several queries per sequence.

The CUDA path (pkv_paged_attn_prefill, through the C ABI) against the fp64
oracle element by element, for both kernels (mma.sync and tcgen05): the
small mixed case under every split setting,
the speculative-verification and chunked-prefill layers at full size, edge
shapes (whole-prompt prefill, one-token sequences, sequences without queries,
row counts that fill one to four warp tiles and several row blocks, long
contexts forced through the split path), both output dtypes, and the
device-side error reports.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_225_gb300 as pkv
from paged_kv_cache_225_gb300 import workloads as W

from gpu_util import TOL, max_abs, to_torch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
_IMPL = {"flags": 0}


@pytest.fixture(params=["mma", "tc"], autouse=True)
def impl(request):
    _IMPL["flags"] = pkv.IMPL[request.param]
    yield request.param


def _device(w: W.PrefillWorkload) -> dict:
    base = w.cfg.base
    return {
        "q": to_torch(w.q, base.q_dtype).to(DEV),
        "q_start": torch.from_numpy(w.q_start).to(DEV),
        "k_cache": to_torch(w.k_cache, base.kv_dtype).to(DEV),
        "v_cache": to_torch(w.v_cache, base.kv_dtype).to(DEV),
        "block_tables": torch.from_numpy(w.block_tables).to(DEV),
        "seq_lens": torch.from_numpy(w.seq_lens).to(DEV),
    }


def _gpu(w, d, *, partition_tokens=0, out_dtype=torch.float32, flags=0, max_q_len=None):
    out = torch.full(d["q"].shape, float("nan"), dtype=out_dtype, device=DEV)
    ws = torch.empty(pkv.prefill_workspace_size(
        w.seq_lens.size, w.num_tokens, w.q.shape[1], w.k_cache.shape[1], w.q.shape[2],
        max_q_len or w.max_q_len, int(w.seq_lens.max()), partition_tokens),
        dtype=torch.uint8, device=DEV)
    pkv.paged_attn_prefill(d["q"], d["q_start"], d["k_cache"], d["v_cache"], d["block_tables"],
                           d["seq_lens"], w.scale, out, max_q_len=max_q_len or w.max_q_len,
                           max_seq_len=int(w.seq_lens.max()), partition_tokens=partition_tokens,
                           workspace=ws, flags=flags | _IMPL["flags"])
    torch.cuda.synchronize()
    status = pkv.read_status(ws)
    return out.float().cpu().numpy().astype(np.float64), status


def _oracle(w):
    base = w.cfg.base
    return oracle.paged_prefill(w.q, base.q_dtype, w.q_start, w.k_cache, w.v_cache,
                                base.kv_dtype, w.block_tables, w.seq_lens, w.scale)


@functools.lru_cache(maxsize=2)
def _config(name):
    w = W.make_prefill_workload(name)
    return w, _oracle(w)


@pytest.mark.parametrize("part", [0, -1, 16, 48, 64, 4096])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_tiny_parity(part, out_dtype):
    w, ref = _config("prefill_tiny")
    d = _device(w)
    out, status = _gpu(w, d, partition_tokens=part, out_dtype=out_dtype)
    assert status == 0
    if out_dtype == torch.bfloat16:
        ref = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        tol = TOL[W.BF16] + 2.0 ** -7 * np.abs(ref).max()
    else:
        tol = TOL[W.BF16]
    assert max_abs(out, ref) <= tol


@pytest.mark.parametrize("name", ["spec_verify_70b", "chunked_prefill_8b"])
@pytest.mark.parametrize("part", [0, -1, 512])
def test_layer_parity(name, part):
    w, ref = _config(name)
    d = _device(w)
    out, status = _gpu(w, d, partition_tokens=part)
    assert status == 0
    err = max_abs(out, ref)
    assert err <= TOL[W.BF16], f"{name} part={part}: max-abs {err}"


def _edge(seq_lens, q_lens, seed, Hq=8, Hkv=2, D=64):
    base = W.DecodeConfig(name="edge", num_seqs=len(seq_lens), num_q_heads=Hq,
                          num_kv_heads=Hkv, head_dim=D, block_size=16, q_dtype=W.BF16,
                          kv_dtype=W.BF16, len_dist="const", len_lo=1, len_hi=1,
                          garbage="nan", new_tokens=False)
    cfg = W.PrefillConfig(name="edge", base=base)
    return W.make_prefill_workload(cfg, seed=seed, seq_lens=np.array(seq_lens),
                                   q_lens=np.array(q_lens))


@pytest.mark.parametrize("case", [
    # (seq_lens, q_lens, Hq, Hkv, D)
    ([1, 16, 17, 32, 33], [1, 16, 17, 1, 33], 8, 2, 64),        # whole prompts, page edges
    ([40, 200, 5], [0, 70, 0], 8, 2, 64),                        # sequences without queries
    ([300, 64], [300, 64], 16, 1, 128),                          # G=16: 4800 rows
    ([129, 77], [12, 77], 24, 8, 128),                           # G=3: rows straddle tiles
    ([512, 513, 1000], [5, 9, 3], 64, 8, 128),                   # 70B grouping
])
@pytest.mark.parametrize("part", [0, 16, 96])
def test_edge_shapes(case, part):
    lens, qlens, Hq, Hkv, D = case
    w = _edge(lens, qlens, seed=sum(lens), Hq=Hq, Hkv=Hkv, D=D)
    d = _device(w)
    out, status = _gpu(w, d, partition_tokens=part)
    assert status == 0
    ref = _oracle(w)
    assert max_abs(out, ref) <= TOL[W.BF16]


@pytest.mark.parametrize("lens,qlens,Hq,Hkv,D", [
    ([300, 64, 17, 129], [8, 5, 1, 3], 64, 8, 128),       # G=8: 64 rows, the 64-row tile full
    ([200, 31, 16, 90], [16, 2, 9, 13], 32, 8, 64),       # G=4: 64 rows, page-edge lengths
    ([700, 21], [21, 7], 12, 4, 128),                     # G=3: 63 rows
])
@pytest.mark.parametrize("part", [0, 16, 96])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_items_of_at_most_64_rows(lens, qlens, Hq, Hkv, D, part, out_dtype):
    # Every sequence's rows fit 64: the tcgen05 kernel takes its M = 64 form.
    w = _edge(lens, qlens, seed=sum(lens) + D, Hq=Hq, Hkv=Hkv, D=D)
    d = _device(w)
    out, status = _gpu(w, d, partition_tokens=part, out_dtype=out_dtype)
    assert status == 0
    ref = _oracle(w)
    if out_dtype == torch.bfloat16:
        ref = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        tol = TOL[W.BF16] + 2.0 ** -7 * np.abs(ref).max()
    else:
        tol = TOL[W.BF16]
    assert max_abs(out, ref) <= tol


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 64), (16, 8, 128), (40, 8, 128), (96, 8, 128),
                                       (24, 2, 64)])
def test_head_groups(Hq, Hkv, D):
    # G = 1, 2, 5, 12, 12: row counts that are not multiples of 8 or 16, and
    # (16 queries x 12 heads = 192 rows) more than one 128-row block.
    w = _edge([70, 300, 16, 129], [3, 7, 16, 1], seed=Hq + D, Hq=Hq, Hkv=Hkv, D=D)
    d = _device(w)
    for part in (0, 64):
        out, status = _gpu(w, d, partition_tokens=part)
        assert status == 0
        assert max_abs(out, _oracle(w)) <= TOL[W.BF16]


def test_long_context_split_path():
    # Few sequences with long contexts: the automatic plan splits them.
    w = _edge([32768, 20000], [5, 3], seed=5, Hq=64, Hkv=8, D=128)
    assert pkv.prefill_partition_tokens(2, w.num_tokens, 64, 8, 128, w.max_q_len, 32768) > 0
    d = _device(w)
    out, status = _gpu(w, d)
    assert status == 0
    ref = _oracle(w)
    assert max_abs(out, ref) <= TOL[W.BF16]


def test_one_query_per_sequence_matches_decode():
    w = _edge([100, 37, 1, 64], [1, 1, 1, 1], seed=9, Hq=32, Hkv=8, D=128)
    d = _device(w)
    out, status = _gpu(w, d)
    assert status == 0
    dec = torch.empty(d["q"].shape, dtype=torch.float32, device=DEV)
    pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["seq_lens"],
                          w.scale, dec, max_seq_len=100)
    torch.cuda.synchronize()
    assert max_abs(out, dec.double().cpu().numpy()) <= 2 * TOL[W.BF16]
    assert max_abs(out, _oracle(w)) <= TOL[W.BF16]


def test_more_queries_than_tokens_is_reported():
    w = _edge([20, 30], [4, 6], seed=11)
    d = _device(w)
    lens = d["seq_lens"].clone()
    lens[1] = 3                       # 6 queries but only 3 tokens
    d["seq_lens"] = lens
    out, status = _gpu(w, d)
    assert status == 4  # PKV_ERR_OUT_OF_RANGE
    ref = _oracle(w)
    # Sequence 0 is still computed correctly.
    assert max_abs(out[:4], ref[:4]) <= TOL[W.BF16]


def test_out_of_pool_page_is_reported_and_skipped():
    w = _edge([40, 90, 33], [3, 5, 2], seed=13, Hq=16, Hkv=2, D=128)
    d = _device(w)
    tables = d["block_tables"].clone()
    tables[1, 2] = w.k_cache.shape[0] + 7            # a page of sequence 1 outside the pool
    d["block_tables"] = tables
    out, status = _gpu(w, d)
    assert status == 4  # PKV_ERR_OUT_OF_RANGE
    ref = _oracle(w)
    rows = np.r_[0:3, 8:10]                           # sequences 0 and 2
    assert max_abs(out[rows], ref[rows]) <= TOL[W.BF16]


def test_bounded_wait_reports_timeout_and_recovers():
    w = _edge([64, 80], [8, 8], seed=12)
    d = _device(w)
    _, status = _gpu(w, d, flags=pkv.FLAG_TEST_DROP_FIRST_COPY)
    assert status == 5
    out, status = _gpu(w, d)
    assert status == 0
    assert max_abs(out, _oracle(w)) <= TOL[W.BF16]
