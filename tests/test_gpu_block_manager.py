"""GPU parity of copy-on-write page copies and of a block-manager-driven decode.

pkv_copy_blocks against a numpy copy of the same pages (bit-exact, every KV
dtype), its out-of-pool report, and a shared-prompt batch built by the
library's block manager (fork, then appends that copy the shared last page)
whose caches and decode output are compared with the oracle replaying the
same steps on host copies.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_225_gb300 as pkv
from paged_kv_cache_225_gb300 import workloads as W

from gpu_util import TOL, bits, max_abs, to_torch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
B = 16


def _pool(rng, N, Hkv, D, dtype):
    k = W.round_to_storage(rng.standard_normal((N, Hkv, D, B)).astype(np.float32), dtype)
    v = W.round_to_storage(rng.standard_normal((N, Hkv, D, B)).astype(np.float32), dtype)
    return k, v


@pytest.mark.parametrize("dtype,Hkv,D", [(W.BF16, 8, 128), (W.FP8_E5M2, 8, 128),
                                         (W.F32, 2, 64), (W.BF16, 1, 64)])
@pytest.mark.parametrize("npairs", [1, 7, 300])
def test_copy_blocks_is_bit_exact(dtype, Hkv, D, npairs):
    rng = np.random.default_rng(npairs + D)
    N = 2 * npairs + 5
    k, v = _pool(rng, N, Hkv, D, dtype)
    ids = rng.permutation(N)[:2 * npairs]
    pairs = ids.reshape(npairs, 2).astype(np.int32)
    kd, vd = to_torch(k, dtype).to(DEV), to_torch(v, dtype).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.copy_blocks(kd, vd, torch.from_numpy(pairs).to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    k[pairs[:, 1]] = k[pairs[:, 0]]
    v[pairs[:, 1]] = v[pairs[:, 0]]
    assert np.array_equal(bits(kd), k.view(np.uint8).reshape(-1))
    assert np.array_equal(bits(vd), v.view(np.uint8).reshape(-1))


def test_copy_blocks_reports_and_skips_out_of_pool_pairs():
    rng = np.random.default_rng(3)
    k, v = _pool(rng, 6, 2, 64, W.BF16)
    pairs = np.array([[0, 1], [2, 9], [-1, 3], [4, 5]], dtype=np.int32)
    kd, vd = to_torch(k, W.BF16).to(DEV), to_torch(v, W.BF16).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.copy_blocks(kd, vd, torch.from_numpy(pairs).to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 4
    k[[1, 5]] = k[[0, 4]]
    assert np.array_equal(bits(kd), k.view(np.uint8).reshape(-1))


def test_shared_prompt_batch_through_the_block_manager():
    rng = np.random.default_rng(11)
    N, Hq, Hkv, D, max_blocks = 96, 16, 2, 128, 12
    kv_dtype = q_dtype = W.BF16
    k_h, v_h = _pool(rng, N, Hkv, D, kv_dtype)       # garbage everywhere at first
    kd, vd = to_torch(k_h, kv_dtype).to(DEV), to_torch(v_h, kv_dtype).to(DEV)
    bm = pkv.BlockManager(N, B, max_blocks)

    def write(slots):
        n = len(slots)
        nk = W.round_to_storage(rng.standard_normal((n, Hkv, D)).astype(np.float32), q_dtype)
        nv = W.round_to_storage(rng.standard_normal((n, Hkv, D)).astype(np.float32), q_dtype)
        pkv.reshape_and_cache(to_torch(nk, q_dtype).to(DEV), to_torch(nv, q_dtype).to(DEV),
                              torch.from_numpy(np.asarray(slots, np.int64)).to(DEV), kd, vd)
        assert oracle.reshape_and_cache(nk, nv, q_dtype, np.asarray(slots, np.int64), k_h, v_h,
                                        kv_dtype) == 0

    # A 75-token system prompt (last page partly filled), shared by 6 requests.
    write(bm.add(0, 75))
    children = list(range(1, 7))
    for c in children:
        bm.fork(0, c)
    bm.free(0)
    for step in range(30):
        slots, pairs = bm.append(children)
        if len(pairs):
            pkv.copy_blocks(kd, vd, torch.from_numpy(np.ascontiguousarray(pairs)).to(DEV))
            k_h[pairs[:, 1]] = k_h[pairs[:, 0]]
            v_h[pairs[:, 1]] = v_h[pairs[:, 0]]
        write(slots)
    assert bm.num_free() == N - (4 + 6 * 3)            # 4 shared pages + 3 private each
    tables, lens = bm.tables(children, max_blocks)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kd), k_h.view(np.uint8).reshape(-1))
    assert np.array_equal(bits(vd), v_h.view(np.uint8).reshape(-1))

    q = W.round_to_storage(rng.standard_normal((len(children), Hq, D)).astype(np.float32),
                           q_dtype)
    out = torch.empty((len(children), Hq, D), dtype=torch.float32, device=DEV)
    pkv.paged_attn_decode(to_torch(q, q_dtype).to(DEV), kd, vd, torch.from_numpy(tables).to(DEV),
                          torch.from_numpy(lens).to(DEV), 1 / np.sqrt(D), out,
                          max_seq_len=int(lens.max()))
    torch.cuda.synchronize()
    ref = oracle.paged_decode(q, q_dtype, k_h, v_h, kv_dtype, tables, lens, 1 / np.sqrt(D))
    assert max_abs(out.double().cpu().numpy(), ref) <= TOL[kv_dtype]
