"""CPU oracle for paged decode attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never links or calls it,
and it shares no code with the CUDA path: it is a plain C implementation in
double precision (``pkv_oracle.c``) of the definitions on the pages, compiled
with gcc and reached through ctypes.

Every function here takes the exact stored bit patterns the GPU reads
(float32 / bf16 bits / fp8-e5m2 codes) and widens them with the oracle's own
decoders.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, FP8_E5M2, FP8_E4M3, INT4 = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE arithmetic, no FMA contraction, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, ip, i32p, i64p, dp = (ctypes.c_void_p, ctypes.c_int,
                                      ctypes.POINTER(ctypes.c_int32),
                                      ctypes.POINTER(ctypes.c_int64),
                                      ctypes.POINTER(ctypes.c_double))
            lib.pkvo_decode_values.argtypes = [vp, ip, ctypes.c_size_t, dp]
            lib.pkvo_decode_values.restype = None
            lib.pkvo_encode_values.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_size_t,
                                               ip, ctypes.c_float, vp]
            lib.pkvo_encode_values.restype = ip
            common = [vp, ip, vp, vp, ip, ctypes.c_double, ctypes.c_double, i32p, i32p,
                      ip, ip, ip, ip, ip, ip, ip, ctypes.c_double]
            lib.pkvo_paged_decode.argtypes = common + [ip, dp, ip]
            lib.pkvo_paged_decode.restype = ip
            fp = ctypes.POINTER(ctypes.c_float)
            lib.pkvo_paged_decode_head_scaled.argtypes = (common[:7] + [fp, fp] + common[7:]
                                                          + [ip, dp, ip])
            lib.pkvo_paged_decode_head_scaled.restype = ip
            lib.pkvo_reshape_and_cache_head_scaled.argtypes = [
                vp, vp, ip, i64p, ip, ip, ip, ip, ip, vp, vp, ip, ctypes.c_float, ctypes.c_float,
                fp, fp]
            lib.pkvo_reshape_and_cache_head_scaled.restype = ip
            lib.pkvo_paged_decode_seqs.argtypes = common + [i32p, ip, dp, ip]
            lib.pkvo_paged_decode_seqs.restype = ip
            lib.pkvo_paged_prefill.argtypes = [vp, ip, i32p] + common[2:] + [ip, dp, ip]
            lib.pkvo_paged_prefill.restype = ip
            lib.pkvo_reshape_and_cache.argtypes = [vp, vp, ip, i64p, ip, ip, ip, ip, ip, vp, vp,
                                                   ip, ctypes.c_float, ctypes.c_float]
            lib.pkvo_reshape_and_cache.restype = ip
            lib.pkvo_max_threads.argtypes = []
            lib.pkvo_max_threads.restype = ip
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype=None):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    if ctype is None:
        return ctypes.c_void_p(a.ctypes.data)
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def max_threads() -> int:
    return int(_load().pkvo_max_threads())


def decode_values(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Widen stored elements to float64 with the oracle's own decoders.

    INT4 storage holds two elements per byte: the result has twice the last
    dimension.
    """
    bits = np.ascontiguousarray(bits)
    n = bits.size * (2 if dtype == INT4 else 1)
    out = np.empty(n, dtype=np.float64)
    _load().pkvo_decode_values(_ptr(bits), dtype, n, _ptr(out, ctypes.c_double))
    shape = bits.shape[:-1] + (bits.shape[-1] * 2,) if dtype == INT4 else bits.shape
    return out.reshape(shape)


def encode_values(x: np.ndarray, dtype: int, scale: float = 1.0) -> np.ndarray:
    """Encode float32 values to a stored dtype with the oracle's own encoders."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    storage = {F32: np.float32, BF16: np.uint16, FP8_E5M2: np.uint8,
               FP8_E4M3: np.uint8, INT4: np.uint8}[dtype]
    if dtype == INT4:
        assert x.shape[-1] % 2 == 0, "INT4 packs pairs along the last axis"
        out = np.zeros(x.shape[:-1] + (x.shape[-1] // 2,), dtype=storage)
    else:
        out = np.empty(x.shape, dtype=storage)
    rc = _load().pkvo_encode_values(_ptr(x, ctypes.c_float), x.size, dtype, scale, _ptr(out))
    if rc:
        raise ValueError(f"encode_values failed ({rc})")
    return out


def _pool_dims(cache, kv_dtype):
    """(N, Hkv, D, block_size) of a cache array (INT4 holds two tokens per byte)."""
    N, Hkv, D, B = cache.shape
    return N, Hkv, D, (2 * B if kv_dtype == INT4 else B)


def _attn_args(q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, seq_lens, scale,
               k_scale, v_scale):
    S, Hq, D = q.shape
    N, Hkv, D2, B = _pool_dims(k_cache, kv_dtype)
    assert D2 == D and v_cache.shape == k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    q = np.ascontiguousarray(q)
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    keep = (q, k_cache, v_cache, bt, sl)
    args = [_ptr(q), q_dtype, _ptr(k_cache), _ptr(v_cache), kv_dtype, float(k_scale),
            float(v_scale), _ptr(bt, ctypes.c_int32), _ptr(sl, ctypes.c_int32), S, Hq, Hkv, D, B,
            N, bt.shape[1], float(scale)]
    return args, keep, (S, Hq, D)


def paged_decode(q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, seq_lens, scale,
                 k_scale=1.0, v_scale=1.0, partition_tokens=0, num_threads=0,
                 k_head_scales=None, v_head_scales=None) -> np.ndarray:
    """Paged decode attention of the whole batch in float64: out [S, Hq, D].

    ``partition_tokens > 0`` evaluates the split-sequence form with the
    log-sum-exp merge instead of one softmax per sequence.  For fp8 caches,
    ``k_head_scales`` / ``v_head_scales`` ([Hkv] float32) multiply the
    dequant scale of each KV head.
    """
    args, keep, shape = _attn_args(q, q_dtype, k_cache, v_cache, kv_dtype, block_tables,
                                   seq_lens, scale, k_scale, v_scale)
    out = np.zeros(shape, dtype=np.float64)
    if k_head_scales is None and v_head_scales is None:
        rc = _load().pkvo_paged_decode(*args, int(partition_tokens), _ptr(out, ctypes.c_double),
                                       int(num_threads))
    else:
        Hkv = k_cache.shape[1]
        ones = np.ones(Hkv, np.float32)
        ksh = np.ascontiguousarray(ones if k_head_scales is None else k_head_scales, np.float32)
        vsh = np.ascontiguousarray(ones if v_head_scales is None else v_head_scales, np.float32)
        assert ksh.shape == (Hkv,) and vsh.shape == (Hkv,)
        rc = _load().pkvo_paged_decode_head_scaled(
            *args[:7], _ptr(ksh, ctypes.c_float), _ptr(vsh, ctypes.c_float), *args[7:],
            int(partition_tokens), _ptr(out, ctypes.c_double), int(num_threads))
    del keep
    if rc:
        raise ValueError(f"oracle paged_decode failed ({rc})")
    return out


def paged_decode_seqs(q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, seq_lens, scale,
                      seqs, k_scale=1.0, v_scale=1.0, num_threads=0) -> np.ndarray:
    """Like ``paged_decode`` but only for the listed sequences: returns [len(seqs), Hq, D]
    (row i is sequence ``seqs[i]``; nothing is computed or allocated for the others)."""
    args, keep, shape = _attn_args(q, q_dtype, k_cache, v_cache, kv_dtype, block_tables,
                                   seq_lens, scale, k_scale, v_scale)
    seqs = np.ascontiguousarray(seqs, dtype=np.int32)
    out = np.empty((seqs.size,) + shape[1:], dtype=np.float64)
    rc = _load().pkvo_paged_decode_seqs(*args, _ptr(seqs, ctypes.c_int32), seqs.size,
                                        _ptr(out, ctypes.c_double), int(num_threads))
    del keep
    if rc:
        raise ValueError(f"oracle paged_decode_seqs failed ({rc})")
    return out


def paged_prefill(q, q_dtype, q_start, k_cache, v_cache, kv_dtype, block_tables, seq_lens,
                  scale, k_scale=1.0, v_scale=1.0, partition_tokens=0,
                  num_threads=0) -> np.ndarray:
    """Paged attention of several causal query tokens per sequence: out [T, Hq, D].

    ``q`` is [T, Hq, D]; the queries of sequence s are rows
    ``q_start[s] .. q_start[s+1]-1``, the last positions of its
    ``seq_lens[s]`` cached tokens.
    """
    T, Hq, D = q.shape
    N, Hkv, D2, B = _pool_dims(k_cache, kv_dtype)
    assert D2 == D and v_cache.shape == k_cache.shape
    qs = np.ascontiguousarray(q_start, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    S = sl.size
    assert qs.size == S + 1 and qs[0] == 0 and qs[-1] == T
    q = np.ascontiguousarray(q)
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    rc = _load().pkvo_paged_prefill(
        _ptr(q), q_dtype, _ptr(qs, ctypes.c_int32), _ptr(k_cache), _ptr(v_cache), kv_dtype,
        float(k_scale), float(v_scale), _ptr(bt, ctypes.c_int32), _ptr(sl, ctypes.c_int32), S,
        Hq, Hkv, D, B, N, bt.shape[1], float(scale), int(partition_tokens),
        _ptr(out, ctypes.c_double), int(num_threads))
    if rc:
        raise ValueError(f"oracle paged_prefill failed ({rc})")
    return out


def reshape_and_cache(k, v, in_dtype, slot_mapping, k_cache, v_cache, kv_dtype,
                      k_scale=1.0, v_scale=1.0, k_head_scales=None, v_head_scales=None) -> int:
    """Scatter new K/V rows into host cache copies in place; returns the status code.

    For fp8 caches ``k_head_scales`` / ``v_head_scales`` ([Hkv] float32)
    multiply the quantisation scale of each KV head.
    """
    T, Hkv, D = k.shape
    N, Hkv2, D2, B = _pool_dims(k_cache, kv_dtype)
    assert Hkv2 == Hkv and D2 == D and v.shape == k.shape
    assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    if k_head_scales is None and v_head_scales is None:
        return int(_load().pkvo_reshape_and_cache(_ptr(k), _ptr(v), in_dtype,
                                                  _ptr(sm, ctypes.c_int64), T, Hkv, D, B, N,
                                                  _ptr(k_cache), _ptr(v_cache), kv_dtype,
                                                  float(k_scale), float(v_scale)))
    ones = np.ones(Hkv, np.float32)
    ksh = np.ascontiguousarray(ones if k_head_scales is None else k_head_scales, np.float32)
    vsh = np.ascontiguousarray(ones if v_head_scales is None else v_head_scales, np.float32)
    return int(_load().pkvo_reshape_and_cache_head_scaled(
        _ptr(k), _ptr(v), in_dtype, _ptr(sm, ctypes.c_int64), T, Hkv, D, B, N, _ptr(k_cache),
        _ptr(v_cache), kv_dtype, float(k_scale), float(v_scale), _ptr(ksh, ctypes.c_float),
        _ptr(vsh, ctypes.c_float)))
