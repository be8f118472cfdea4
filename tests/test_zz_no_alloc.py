"""The allocation-free decode entry point, checked against the regular one.

pkv_paged_attn_decode_noalloc serves callers that cannot allocate device
memory (a plugin inside a runtime that owns all device memory, or a loop
where cudaMalloc's implicit synchronisation is not allowed): it takes its
scratch from a fixed array inside the library instead of a caller workspace.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import paged_kv_cache_225_gb300 as pkv
from paged_kv_cache_225_gb300 import workloads as W

from gpu_util import TOL, device_workload, max_abs

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024   # PKV_NOALLOC_SCRATCH_BYTES in include/pkv.h
PKV_ERR_WORKSPACE = 6


def _noalloc():
    f = pkv.lib().pkv_paged_attn_decode_noalloc
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, i, vp, vp, i, fl, fl, vp, vp, i, i, i, i, i, i, i, i, fl, vp, i, i, i, vp]
    f.restype = i
    return f


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    dev = torch.device("cuda", 0)
    cfg = dataclasses.replace(W.CONFIGS["llama3_8b"], name="noalloc", num_seqs=16)
    w = W.make_workload(cfg, seed=77)
    d = device_workload(w, dev)
    S, Hq, D = w.q.shape
    N, Hkv, _, B = w.k_cache.shape
    max_len = int(w.seq_lens.max())
    f = _noalloc()
    stream = torch.cuda.current_stream(dev).cuda_stream
    # Both schedules that keep partial results in scratch memory: the
    # automatic (stream-K) one and fixed 256-token partitions.
    for part in (0, 256):
        assert pkv.partition_tokens(S, Hq, Hkv, D, max_len, part) != 0
        assert 256 < pkv.workspace_size(S, Hq, Hkv, D, max_len, part) <= NOALLOC_SCRATCH_BYTES

        ref = torch.empty((S, Hq, D), dtype=torch.float32, device=dev)
        pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                              d["seq_lens"], w.scale, ref, max_seq_len=max_len,
                              partition_tokens=part)
        torch.cuda.synchronize()
        assert pkv.read_status(device=dev) == 0
        ref_np = ref.cpu().numpy()

        for _ in range(2):
            out = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device=dev)
            rc = f(d["q"].data_ptr(), pkv.BF16, d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
                   pkv.BF16, 1.0, 1.0, d["block_tables"].data_ptr(), d["seq_lens"].data_ptr(), S,
                   Hq, Hkv, D, B, N, w.max_blocks_per_seq, max_len, w.scale, out.data_ptr(),
                   pkv.F32, part, 0, stream)
            assert rc == 0
            torch.cuda.synchronize()
            assert max_abs(out.cpu().numpy(), ref_np) <= TOL[W.BF16]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    f = _noalloc()
    # 128 sequences x 64 heads x 512 partitions of 64 tokens needs ~2 GB of partials.
    need = pkv.workspace_size(128, 64, 8, 128, 32768, 64)
    assert need > NOALLOC_SCRATCH_BYTES
    rc = f(0x1000, pkv.BF16, 0x2000, 0x3000, pkv.BF16, 1.0, 1.0, 0x4000, 0x5000, 128, 64, 8, 128,
           16, 100, 2048, 32768, 0.1, 0x6000, pkv.F32, 64, 0, None)
    assert rc == PKV_ERR_WORKSPACE
