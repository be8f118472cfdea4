"""Helpers shared by the GPU parity tests: moving a host workload to the GPU,
running one decode step through the library, and the oracle's answer for the
same step."""
import numpy as np
import torch

import oracle
import paged_kv_cache_225_gb300 as pkv
from paged_kv_cache_225_gb300 import workloads as W

# Max-abs tolerances against the fp64 oracle on identically rounded inputs.
TOL = {W.F32: 1e-5, W.BF16: 4e-3, W.FP8_E5M2: 3e-2, W.FP8_E4M3: 3e-2, W.INT4: 4e-3}


def to_torch(a: np.ndarray, dtype: int) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if dtype == W.F32:
        return torch.from_numpy(a)
    if dtype == W.BF16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    if dtype == W.FP8_E5M2:
        return torch.from_numpy(a).view(torch.float8_e5m2)
    if dtype == W.FP8_E4M3:
        return torch.from_numpy(a).view(torch.float8_e4m3fn)
    if dtype == W.INT4:
        return torch.from_numpy(a)                   # packed nibbles as uint8
    raise ValueError(dtype)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bytes of a tensor as a numpy uint8 array (for bit-exact compares)."""
    t = t.detach().contiguous().cpu()
    return t.view(torch.uint8).numpy().reshape(-1)


def device_workload(w: W.Workload, dev: torch.device) -> dict:
    cfg = w.cfg
    d = {
        "q": to_torch(w.q, cfg.q_dtype).to(dev),
        "k_cache": to_torch(w.k_cache, cfg.kv_dtype).to(dev),
        "v_cache": to_torch(w.v_cache, cfg.kv_dtype).to(dev),
        "block_tables": torch.from_numpy(w.block_tables).to(dev),
        "seq_lens": torch.from_numpy(w.seq_lens).to(dev),
    }
    if w.new_k is not None:
        d["new_k"] = to_torch(w.new_k, cfg.q_dtype).to(dev)
        d["new_v"] = to_torch(w.new_v, cfg.q_dtype).to(dev)
        d["slot_mapping"] = torch.from_numpy(w.slot_mapping).to(dev)
    return d


def gpu_step(w: W.Workload, d: dict, *, impl="auto", partition_tokens=0, out_dtype=torch.float32,
             append=True, kv_scale=None, flags=0):
    """One decode step on the GPU: write the new tokens, attend over L+1 tokens."""
    cfg = w.cfg
    ks = vs = cfg.kv_scale if kv_scale is None else kv_scale
    lens = w.seq_lens.copy()
    if append:
        pkv.reshape_and_cache(d["new_k"], d["new_v"], d["slot_mapping"], d["k_cache"],
                              d["v_cache"], k_scale=ks, v_scale=vs)
        lens = lens + 1
    lens_dev = torch.from_numpy(lens.astype(np.int32)).to(d["q"].device)
    out = torch.empty(d["q"].shape, dtype=out_dtype, device=d["q"].device)
    pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], lens_dev,
                          w.scale, out, k_scale=ks, v_scale=vs, max_seq_len=int(lens.max()),
                          partition_tokens=partition_tokens, impl=impl, flags=flags)
    torch.cuda.synchronize()
    status = pkv.read_status(device=d["q"].device)
    return out.float().cpu().numpy().astype(np.float64), status, lens


def oracle_step(w: W.Workload, append=True, kv_scale=None):
    """The oracle's caches after the write and its output for the same step."""
    cfg = w.cfg
    ks = vs = cfg.kv_scale if kv_scale is None else kv_scale
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    lens = w.seq_lens.copy()
    if append:
        rc = oracle.reshape_and_cache(w.new_k, w.new_v, cfg.q_dtype, w.slot_mapping, kc, vc,
                                      cfg.kv_dtype, ks, vs)
        assert rc == 0
        lens = lens + 1
    ref = oracle.paged_decode(w.q, cfg.q_dtype, kc, vc, cfg.kv_dtype, w.block_tables, lens,
                              w.scale, k_scale=ks, v_scale=vs)
    return ref, kc, vc


def max_abs(a, b) -> float:
    d = np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))
    return float(np.nanmax(d)) if not np.isnan(d).any() else float("inf")


def gpu_step_fused(w: W.Workload, d: dict, *, impl="auto", partition_tokens=0,
                   out_dtype=torch.float32, kv_scale=None, flags=0):
    """The same decode step in one launch: cache write fused into the decode."""
    cfg = w.cfg
    ks = vs = cfg.kv_scale if kv_scale is None else kv_scale
    lens = w.seq_lens + 1
    lens_dev = torch.from_numpy(lens.astype(np.int32)).to(d["q"].device)
    out = torch.empty(d["q"].shape, dtype=out_dtype, device=d["q"].device)
    pkv.paged_attn_decode_append(d["q"], d["new_k"], d["new_v"], d["k_cache"], d["v_cache"],
                                 d["block_tables"], lens_dev, w.scale, out, k_scale=ks,
                                 v_scale=vs, max_seq_len=int(lens.max()),
                                 partition_tokens=partition_tokens, impl=impl, flags=flags)
    torch.cuda.synchronize()
    status = pkv.read_status(device=d["q"].device)
    return out.float().cpu().numpy().astype(np.float64), status, lens

