"""GPU parity of causal paged attention with several queries per sequence over
fp8 (e5m2, e4m3) and INT4 caches.

These caches run on the mma.sync kernel (its fragments widen the codes to
f16 in registers, as the decode kernels do); the tcgen05 kernel is bf16 only
and refuses them.  The fp64 oracle reads the same codes with its own
decoders and scales.  Cases: the small mixed batch under every split
setting with each dtype and a non-unit scale, edge shapes, the
speculative-verification layer over an fp8-e5m2 cache at full size, and one
query per sequence against the decode kernel.
"""
import dataclasses
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
COMPACT = [(W.FP8_E5M2, 1.0), (W.FP8_E5M2, 0.5), (W.FP8_E4M3, 0.125), (W.INT4, 0.5)]


def _device(w):
    base = w.cfg.base
    return {"q": to_torch(w.q, base.q_dtype).to(DEV),
            "q_start": torch.from_numpy(w.q_start).to(DEV),
            "k_cache": to_torch(w.k_cache, base.kv_dtype).to(DEV),
            "v_cache": to_torch(w.v_cache, base.kv_dtype).to(DEV),
            "block_tables": torch.from_numpy(w.block_tables).to(DEV),
            "seq_lens": torch.from_numpy(w.seq_lens).to(DEV)}


def _gpu(w, d, *, partition_tokens=0, flags=0, out_dtype=torch.float32):
    base = w.cfg.base
    out = torch.full(d["q"].shape, float("nan"), dtype=out_dtype, device=DEV)
    ws = torch.empty(pkv.prefill_workspace_size(
        w.seq_lens.size, w.num_tokens, w.q.shape[1], w.k_cache.shape[1], w.q.shape[2],
        w.max_q_len, int(w.seq_lens.max()), partition_tokens), dtype=torch.uint8, device=DEV)
    pkv.paged_attn_prefill(d["q"], d["q_start"], d["k_cache"], d["v_cache"], d["block_tables"],
                           d["seq_lens"], w.scale, out, max_q_len=w.max_q_len,
                           max_seq_len=int(w.seq_lens.max()), partition_tokens=partition_tokens,
                           workspace=ws, flags=flags, k_scale=base.kv_scale,
                           v_scale=base.kv_scale)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), pkv.read_status(ws)


def _oracle(w):
    base = w.cfg.base
    return oracle.paged_prefill(w.q, base.q_dtype, w.q_start, w.k_cache, w.v_cache,
                                base.kv_dtype, w.block_tables, w.seq_lens, w.scale,
                                k_scale=base.kv_scale, v_scale=base.kv_scale)


@functools.lru_cache(maxsize=4)
def _tiny(kv_dtype, kv_scale):
    cfg = W.PREFILL_CONFIGS["prefill_tiny"]
    base = dataclasses.replace(cfg.base, kv_dtype=kv_dtype, kv_scale=kv_scale)
    w = W.make_prefill_workload(dataclasses.replace(cfg, base=base),
                                seed=W.PREFILL_SEED["prefill_tiny"])
    return w, _oracle(w)


@pytest.mark.parametrize("kv_dtype,kv_scale", COMPACT)
@pytest.mark.parametrize("part", [0, -1, 16, 48, 4096])
@pytest.mark.parametrize("impl", ["auto", "mma"])
def test_tiny_parity(kv_dtype, kv_scale, part, impl):
    w, ref = _tiny(kv_dtype, kv_scale)
    out, status = _gpu(w, _device(w), partition_tokens=part, flags=pkv.IMPL[impl])
    assert status == 0
    # Outputs scale with the V factor: the stated bound times max(1, scale).
    assert max_abs(out, ref) <= TOL[kv_dtype] * max(1.0, kv_scale)


@pytest.mark.parametrize("kv_dtype,kv_scale", COMPACT[1:])
def test_bf16_output(kv_dtype, kv_scale):
    w, ref = _tiny(kv_dtype, kv_scale)
    out32, st32 = _gpu(w, _device(w))
    out16, st16 = _gpu(w, _device(w), out_dtype=torch.bfloat16)
    assert st32 == 0 and st16 == 0
    rounded = torch.from_numpy(out32.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(out16, rounded)


def test_tcgen05_kernel_refuses_compact_caches():
    w, _ = _tiny(W.FP8_E5M2, 1.0)
    with pytest.raises(pkv.PkvError):
        _gpu(w, _device(w), flags=pkv.IMPL["tc"])


def _edge(seq_lens, q_lens, kv_dtype, kv_scale, seed, Hq=8, Hkv=2, D=64):
    base = W.DecodeConfig(name="edge", num_seqs=len(seq_lens), num_q_heads=Hq,
                          num_kv_heads=Hkv, head_dim=D, block_size=16, q_dtype=W.BF16,
                          kv_dtype=kv_dtype, kv_scale=kv_scale, len_dist="const", len_lo=1,
                          len_hi=1, garbage="nan", new_tokens=False)
    return W.make_prefill_workload(W.PrefillConfig(name="edge", base=base), seed=seed,
                                   seq_lens=np.array(seq_lens), q_lens=np.array(q_lens))


@pytest.mark.parametrize("kv_dtype,kv_scale", COMPACT[1:])
@pytest.mark.parametrize("case", [
    ([1, 16, 17, 32, 33], [1, 16, 17, 1, 33], 8, 2, 64),     # whole prompts, page edges
    ([40, 200, 5], [0, 70, 0], 8, 2, 64),                     # sequences without queries
    ([300, 64], [300, 64], 16, 1, 128),                       # G = 16: two N tiles
    ([129, 77], [12, 77], 24, 8, 128),                        # G = 3: rows straddle tiles
    ([512, 513, 1000], [5, 9, 3], 64, 8, 128),                # 70B grouping
])
@pytest.mark.parametrize("part", [0, 96])
def test_edge_shapes(kv_dtype, kv_scale, case, part):
    lens, qlens, Hq, Hkv, D = case
    w = _edge(lens, qlens, kv_dtype, kv_scale, seed=sum(lens) + kv_dtype, Hq=Hq, Hkv=Hkv, D=D)
    out, status = _gpu(w, _device(w), partition_tokens=part)
    assert status == 0
    assert max_abs(out, _oracle(w)) <= TOL[kv_dtype] * max(1.0, kv_scale)


@pytest.mark.parametrize("part", [0, 512])
def test_speculative_verification_layer_over_fp8(part):
    w = W.make_prefill_workload("spec_verify_70b_fp8")
    ref = _oracle(w)
    out, status = _gpu(w, _device(w), partition_tokens=part)
    assert status == 0
    assert max_abs(out, ref) <= TOL[W.FP8_E5M2]


@pytest.mark.parametrize("kv_dtype,kv_scale", COMPACT[1:])
def test_one_query_per_sequence_matches_decode(kv_dtype, kv_scale):
    w = _edge([100, 37, 1, 64], [1, 1, 1, 1], kv_dtype, kv_scale, seed=9, Hq=32, Hkv=8, D=128)
    d = _device(w)
    out, status = _gpu(w, d)
    assert status == 0
    dec = torch.empty(d["q"].shape, dtype=torch.float32, device=DEV)
    pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["seq_lens"],
                          w.scale, dec, max_seq_len=100, k_scale=kv_scale, v_scale=kv_scale)
    torch.cuda.synchronize()
    tol = TOL[kv_dtype] * max(1.0, kv_scale)
    assert max_abs(out, dec.double().cpu().numpy()) <= 2 * tol
    assert max_abs(out, _oracle(w)) <= tol
