"""GB300 (sm_103a) paged KV-cache decode attention.

Thin Python binding over the C ABI of ``_build/libpkv.so`` (include/pkv.h):
argument marshalling only.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and the calls
raise if the library is missing.  PyTorch provides device memory, the
current stream and the workspace allocation.

    paged_attn_decode(q, k_cache, v_cache, block_tables, seq_lens, scale, out)
    paged_attn_decode_append(q, new_k, new_v, k_cache, v_cache, ..., out)
    paged_attn_prefill(q, q_start, k_cache, v_cache, block_tables, seq_lens, scale, out)
    reshape_and_cache(k, v, slot_mapping, k_cache, v_cache)
    copy_blocks(k_cache, v_cache, pairs)
    BlockManager(num_blocks)   (host-side page pool: add / fork / append / free / tables)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

__all__ = ["paged_attn_decode", "paged_attn_decode_append", "paged_attn_prefill",
           "paged_attn_decode_head_scaled", "reshape_and_cache_head_scaled",
           "reshape_and_cache", "workspace_size", "partition_tokens",
           "prefill_workspace_size", "prefill_partition_tokens", "copy_blocks",
           "BlockManager",
           "read_status", "PkvError", "lib", "F32", "BF16", "FP8_E5M2", "FP8_E4M3",
           "INT4"]

F32, BF16, FP8_E5M2, FP8_E4M3, INT4 = 0, 1, 2, 3, 4
IMPL = {"auto": 0x0, "simt": 0x1, "mma": 0x2, "tc": 0x3}  # "tc": several-queries kernel only
FLAG_SEPARATE_MERGE = 0x4
FLAG_TEST_DROP_FIRST_COPY = 0x100
STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_CUDA",
          4: "PKV_ERR_OUT_OF_RANGE", 5: "PKV_ERR_TIMEOUT", 6: "PKV_ERR_WORKSPACE",
          7: "PKV_ERR_NO_BLOCKS"}

_lock = threading.Lock()
_lib = None
_workspaces: dict = {}


class PkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = _lib.pkv_status_string(code).decode() if _lib is not None else STATUS.get(code, "?")
        super().__init__(f"{what}: {msg}")


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """The loaded C library (compiled on first use if ``build_if_missing``)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing:
                path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"paged KV-cache CUDA library not built: {path}")
            L = ctypes.CDLL(path)
            vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.pkv_paged_attn_workspace_size.argtypes = [i, i, i, i, i, i, i]
            L.pkv_paged_attn_workspace_size.restype = sz
            L.pkv_paged_attn_partition_tokens.argtypes = [i, i, i, i, i, i, i]
            L.pkv_paged_attn_partition_tokens.restype = i
            L.pkv_paged_attn_decode.argtypes = [vp, i, vp, vp, i, f, f, vp, vp, i, i, i, i, i, i,
                                                i, i, f, vp, i, vp, sz, i, i, vp]
            L.pkv_paged_attn_decode.restype = i
            L.pkv_paged_attn_decode_append.argtypes = [vp, i, vp, vp, i, vp, vp, i, f, f, vp, vp,
                                                       i, i, i, i, i, i, i, i, f, vp, i, vp, sz, i,
                                                       i, vp]
            L.pkv_paged_attn_decode_append.restype = i
            L.pkv_paged_attn_layers_workspace_size.argtypes = [i] * 8
            L.pkv_paged_attn_layers_workspace_size.restype = sz
            L.pkv_paged_attn_layers_partition_tokens.argtypes = [i] * 8
            L.pkv_paged_attn_layers_partition_tokens.restype = i
            L.pkv_paged_attn_decode_layers.argtypes = [vp, i, i, i, i, f, f, vp, vp, i, i, i, i,
                                                       i, i, i, i, f, i, vp, sz, i, i, vp]
            L.pkv_paged_attn_decode_layers.restype = i
            L.pkv_paged_attn_prefill_workspace_size.argtypes = [i] * 9
            L.pkv_paged_attn_prefill_workspace_size.restype = sz
            L.pkv_paged_attn_prefill_partition_tokens.argtypes = [i] * 9
            L.pkv_paged_attn_prefill_partition_tokens.restype = i
            L.pkv_paged_attn_prefill.argtypes = [vp, i, vp, vp, vp, i, f, f, vp, vp, i, i, i, i,
                                                 i, i, i, i, i, i, f, vp, i, vp, sz, i, i, vp]
            L.pkv_paged_attn_prefill.restype = i
            L.pkv_paged_attn_decode_head_scaled.argtypes = [vp, i, vp, vp, i, vp, vp, vp, vp, i,
                                                            i, i, i, i, i, i, i, f, vp, i, vp,
                                                            sz, i, i, vp]
            L.pkv_paged_attn_decode_head_scaled.restype = i
            L.pkv_reshape_and_cache_head_scaled.argtypes = [vp, vp, i, vp, i, i, i, i, i, vp, vp,
                                                            i, vp, vp, vp, vp]
            L.pkv_reshape_and_cache_head_scaled.restype = i
            L.pkv_copy_blocks.argtypes = [vp, vp, i, i, i, i, i, vp, i, vp, vp]
            L.pkv_copy_blocks.restype = i
            ip, i32p, i64p = (ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int32),
                              ctypes.POINTER(ctypes.c_int64))
            L.pkv_bm_create.argtypes = [i, i, i, ctypes.POINTER(vp)]
            L.pkv_bm_create.restype = i
            L.pkv_bm_destroy.argtypes = [vp]
            L.pkv_bm_destroy.restype = None
            L.pkv_bm_add.argtypes = [vp, i, i, i64p]
            L.pkv_bm_add.restype = i
            L.pkv_bm_fork.argtypes = [vp, i, i]
            L.pkv_bm_fork.restype = i
            L.pkv_bm_append.argtypes = [vp, i32p, i, i64p, i32p, ip]
            L.pkv_bm_append.restype = i
            L.pkv_bm_free.argtypes = [vp, i]
            L.pkv_bm_free.restype = i
            L.pkv_bm_tables.argtypes = [vp, i32p, i, i, i32p, i32p]
            L.pkv_bm_tables.restype = i
            L.pkv_bm_num_free.argtypes = [vp]
            L.pkv_bm_num_free.restype = i
            L.pkv_bm_ref_count.argtypes = [vp, i]
            L.pkv_bm_ref_count.restype = i
            L.pkv_reshape_and_cache.argtypes = [vp, vp, i, vp, i, i, i, i, i, vp, vp, i, f, f, vp,
                                                vp]
            L.pkv_reshape_and_cache.restype = i
            L.pkv_read_status.argtypes = [vp, i, ctypes.POINTER(ctypes.c_int32), vp]
            L.pkv_read_status.restype = i
            L.pkv_status_string.argtypes = [i]
            L.pkv_status_string.restype = ctypes.c_char_p
            L.pkv_version.argtypes = []
            L.pkv_version.restype = i
            _lib = L
    return _lib


def _dtype_code(t: torch.Tensor, what: str) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float8_e5m2:
        return FP8_E5M2
    if t.dtype == torch.float8_e4m3fn:
        return FP8_E4M3
    if t.dtype == torch.uint8:
        return INT4          # packed signed nibbles, two tokens per byte
    raise TypeError(f"{what}: unsupported dtype {t.dtype}")


def _check(t: torch.Tensor, what: str, ndim: int, device: torch.device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{what} must be a CUDA tensor (the library has no CPU path)")
    if t.device != device:
        raise ValueError(f"{what} is on {t.device}, expected {device}")
    if t.dim() != ndim:
        raise ValueError(f"{what} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")


def _pool_dims(cache: torch.Tensor):
    """(N, Hkv, D, block_size) of a cache tensor; INT4 caches (uint8) hold two
    tokens per byte in the last dimension."""
    N, Hkv, D, B = cache.shape
    return N, Hkv, D, (2 * B if cache.dtype == torch.uint8 else B)


def _stream(device: torch.device, stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   max_seq_len: int, partition_tokens: int = 0, block_size: int = 16) -> int:
    n = lib().pkv_paged_attn_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                            block_size, max_seq_len, partition_tokens)
    if n == 0:
        raise ValueError("invalid sizes for the decode workspace")
    return int(n)


SCHEDULE_STREAMK = -2


def partition_tokens(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                     max_seq_len: int, partition_tokens: int = 0, block_size: int = 16) -> int:
    """Schedule of the decode call: tokens per fixed partition (> 0), 0 for one
    pass per (sequence, KV head), SCHEDULE_STREAMK for equal page ranges per CTA."""
    return int(lib().pkv_paged_attn_partition_tokens(num_seqs, num_q_heads, num_kv_heads,
                                                     head_dim, block_size, max_seq_len,
                                                     partition_tokens))


def get_workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    """A cached device workspace of at least ``nbytes`` (grown on demand)."""
    key = (device.type, device.index)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def paged_attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                      out: torch.Tensor, *, k_scale: float = 1.0, v_scale: float = 1.0,
                      max_seq_len: Optional[int] = None, partition_tokens: int = 0,
                      impl: str = "auto", workspace: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None, flags: int = 0) -> torch.Tensor:
    """PagedAttention decode: out[s, h] = softmax(scale q[s,h] K_s^T) V_s.

    q [S, Hq, D] (f32/bf16); k_cache, v_cache [N, Hkv, D, 16] (f32/bf16/
    float8_e5m2/float8_e4m3fn); block_tables int32 [S, max_blocks]; seq_lens int32 [S];
    out [S, Hq, D] (f32/bf16).  ``max_seq_len`` bounds seq_lens (default:
    max_blocks * 16, no device sync).  Returns ``out``.
    """
    dev = q.device
    _check(q, "q", 3, dev)
    _check(k_cache, "k_cache", 4, dev)
    _check(v_cache, "v_cache", 4, dev)
    _check(block_tables, "block_tables", 2, dev)
    _check(seq_lens, "seq_lens", 1, dev)
    _check(out, "out", 3, dev)
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must have the same shape and dtype")
    S, Hq, D = q.shape
    N, Hkv, D2, B = _pool_dims(k_cache)
    if D2 != D or out.shape != q.shape or block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("inconsistent shapes")
    max_blocks = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = max_blocks * B
    L = lib()
    need = L.pkv_paged_attn_workspace_size(S, Hq, Hkv, D, B, max_seq_len, partition_tokens)
    if need == 0:
        raise ValueError("invalid sizes or partition_tokens")
    if workspace is None:
        workspace = get_workspace(need, dev)
    flags |= IMPL[impl]
    rc = L.pkv_paged_attn_decode(
        q.data_ptr(), _dtype_code(q, "q"), k_cache.data_ptr(), v_cache.data_ptr(),
        _dtype_code(k_cache, "k_cache"), float(k_scale), float(v_scale), block_tables.data_ptr(),
        seq_lens.data_ptr(), S, Hq, Hkv, D, B, N, max_blocks, int(max_seq_len), float(scale),
        out.data_ptr(), _dtype_code(out, "out"), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), int(partition_tokens), int(flags),
        _stream(dev, stream))
    if rc != 0:
        raise PkvError(rc, "pkv_paged_attn_decode")
    return out


def paged_attn_decode_head_scaled(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  k_head_scales: torch.Tensor, v_head_scales: torch.Tensor,
                                  block_tables: torch.Tensor, seq_lens: torch.Tensor,
                                  scale: float, out: torch.Tensor, *,
                                  max_seq_len: Optional[int] = None, partition_tokens: int = 0,
                                  impl: str = "auto", workspace: Optional[torch.Tensor] = None,
                                  stream: Optional[torch.cuda.Stream] = None,
                                  flags: int = 0) -> torch.Tensor:
    """Decode over an fp8 cache with one dequant scale per KV head
    (k_head_scales, v_head_scales: float32 [Hkv] on the device)."""
    dev = q.device
    for t, name, nd in ((q, "q", 3), (k_cache, "k_cache", 4), (v_cache, "v_cache", 4),
                        (k_head_scales, "k_head_scales", 1), (v_head_scales, "v_head_scales", 1),
                        (block_tables, "block_tables", 2), (seq_lens, "seq_lens", 1),
                        (out, "out", 3)):
        _check(t, name, nd, dev)
    if k_head_scales.dtype != torch.float32 or v_head_scales.dtype != torch.float32:
        raise TypeError("per-head scales must be float32")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    S, Hq, D = q.shape
    N, Hkv, D2, B = _pool_dims(k_cache)
    if (D2 != D or out.shape != q.shape or k_cache.shape != v_cache.shape
            or k_head_scales.shape[0] != Hkv or v_head_scales.shape[0] != Hkv):
        raise ValueError("inconsistent shapes")
    max_blocks = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = max_blocks * B
    L = lib()
    need = L.pkv_paged_attn_workspace_size(S, Hq, Hkv, D, B, max_seq_len, partition_tokens)
    if need == 0:
        raise ValueError("invalid sizes or partition_tokens")
    if workspace is None:
        workspace = get_workspace(need, dev)
    rc = L.pkv_paged_attn_decode_head_scaled(
        q.data_ptr(), _dtype_code(q, "q"), k_cache.data_ptr(), v_cache.data_ptr(),
        _dtype_code(k_cache, "k_cache"), k_head_scales.data_ptr(), v_head_scales.data_ptr(),
        block_tables.data_ptr(), seq_lens.data_ptr(), S, Hq, Hkv, D, B, N, max_blocks,
        int(max_seq_len), float(scale), out.data_ptr(), _dtype_code(out, "out"),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        int(partition_tokens), int(flags) | IMPL[impl], _stream(dev, stream))
    if rc != 0:
        raise PkvError(rc, "pkv_paged_attn_decode_head_scaled")
    return out


def reshape_and_cache_head_scaled(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                                  k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  k_head_scales: torch.Tensor, v_head_scales: torch.Tensor, *,
                                  status: Optional[torch.Tensor] = None,
                                  stream: Optional[torch.cuda.Stream] = None) -> None:
    """The cache write into an fp8 cache with one quantisation scale per KV head."""
    dev = k.device
    for t, name, nd in ((k, "k", 3), (v, "v", 3), (slot_mapping, "slot_mapping", 1),
                        (k_cache, "k_cache", 4), (v_cache, "v_cache", 4),
                        (k_head_scales, "k_head_scales", 1), (v_head_scales, "v_head_scales", 1)):
        _check(t, name, nd, dev)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    if k_head_scales.dtype != torch.float32 or v_head_scales.dtype != torch.float32:
        raise TypeError("per-head scales must be float32")
    T, Hkv, D = k.shape
    N, Hkv2, D2, B = _pool_dims(k_cache)
    if (v.shape != k.shape or Hkv2 != Hkv or D2 != D or v_cache.shape != k_cache.shape
            or slot_mapping.shape[0] != T or k_head_scales.shape[0] != Hkv
            or v_head_scales.shape[0] != Hkv):
        raise ValueError("inconsistent shapes")
    st_ptr = None
    if status is not None:
        _check(status, "status", 1, dev)
        st_ptr = status.data_ptr()
    rc = lib().pkv_reshape_and_cache_head_scaled(
        k.data_ptr(), v.data_ptr(), _dtype_code(k, "k"), slot_mapping.data_ptr(), T, Hkv, D, B,
        N, k_cache.data_ptr(), v_cache.data_ptr(), _dtype_code(k_cache, "k_cache"),
        k_head_scales.data_ptr(), v_head_scales.data_ptr(), st_ptr, _stream(dev, stream))
    if rc != 0:
        raise PkvError(rc, "pkv_reshape_and_cache_head_scaled")


def paged_attn_decode_append(q: torch.Tensor, new_k: torch.Tensor, new_v: torch.Tensor,
                             k_cache: torch.Tensor, v_cache: torch.Tensor,
                             block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                             out: torch.Tensor, *, k_scale: float = 1.0, v_scale: float = 1.0,
                             max_seq_len: Optional[int] = None, partition_tokens: int = 0,
                             impl: str = "auto", workspace: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None,
                             flags: int = 0) -> torch.Tensor:
    """One decode step with the cache write fused in.

    new_k, new_v [S, Hkv, D] (f32/bf16) are the K/V rows of each sequence's
    new token, logical position seq_lens[s] - 1 (seq_lens include it); they
    are written into the cache and attended in the same launch.  Other
    arguments as for ``paged_attn_decode``.  Returns ``out``.
    """
    dev = q.device
    for t, name, nd in ((q, "q", 3), (new_k, "new_k", 3), (new_v, "new_v", 3),
                        (k_cache, "k_cache", 4), (v_cache, "v_cache", 4),
                        (block_tables, "block_tables", 2), (seq_lens, "seq_lens", 1),
                        (out, "out", 3)):
        _check(t, name, nd, dev)
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must have the same shape and dtype")
    S, Hq, D = q.shape
    N, Hkv, D2, B = _pool_dims(k_cache)
    if (D2 != D or out.shape != q.shape or block_tables.shape[0] != S
            or seq_lens.shape[0] != S or new_k.shape != (S, Hkv, D)
            or new_v.shape != new_k.shape or new_v.dtype != new_k.dtype):
        raise ValueError("inconsistent shapes")
    max_blocks = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = max_blocks * B
    L = lib()
    need = L.pkv_paged_attn_workspace_size(S, Hq, Hkv, D, B, max_seq_len, partition_tokens)
    if need == 0:
        raise ValueError("invalid sizes or partition_tokens")
    if workspace is None:
        workspace = get_workspace(need, dev)
    flags |= IMPL[impl]
    rc = L.pkv_paged_attn_decode_append(
        q.data_ptr(), _dtype_code(q, "q"), new_k.data_ptr(), new_v.data_ptr(),
        _dtype_code(new_k, "new_k"), k_cache.data_ptr(), v_cache.data_ptr(),
        _dtype_code(k_cache, "k_cache"), float(k_scale), float(v_scale), block_tables.data_ptr(),
        seq_lens.data_ptr(), S, Hq, Hkv, D, B, N, max_blocks, int(max_seq_len), float(scale),
        out.data_ptr(), _dtype_code(out, "out"), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), int(partition_tokens), int(flags),
        _stream(dev, stream))
    if rc != 0:
        raise PkvError(rc, "pkv_paged_attn_decode_append")
    return out


def layers_workspace_size(num_layers: int, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                          head_dim: int, max_seq_len: int, partition_tokens: int = 0) -> int:
    """Workspace bytes of ``paged_attn_decode_layers`` (pkv_paged_attn_layers_workspace_size)."""
    n = lib().pkv_paged_attn_layers_workspace_size(num_layers, num_seqs, num_q_heads,
                                                   num_kv_heads, head_dim, 16, max_seq_len,
                                                   partition_tokens)
    if n == 0:
        raise ValueError("invalid sizes or partition_tokens")
    return int(n)


def layers_partition_tokens(num_layers: int, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                            head_dim: int, max_seq_len: int, partition_tokens: int = 0) -> int:
    """The schedule ``paged_attn_decode_layers`` uses (as ``partition_tokens``)."""
    return int(lib().pkv_paged_attn_layers_partition_tokens(
        num_layers, num_seqs, num_q_heads, num_kv_heads, head_dim, 16, max_seq_len,
        partition_tokens))


# Field order of one pkv_layer entry.
LAYER_FIELDS = ("q", "new_k", "new_v", "k_cache", "v_cache", "out")


def layer_table(layers, device: Optional[torch.device] = None) -> torch.Tensor:
    """The device table of pkv_layer entries (int64 [L, 6]) for ``layers``, a list
    of dicts with keys LAYER_FIELDS (new_k / new_v may be None or absent)."""
    rows = [[(lay[k].data_ptr() if lay.get(k) is not None else 0) for k in LAYER_FIELDS]
            for lay in layers]
    dev = device if device is not None else layers[0]["q"].device
    return torch.tensor(rows, dtype=torch.int64).to(dev)


def paged_attn_decode_layers(layers, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                             scale: float, *, k_scale: float = 1.0, v_scale: float = 1.0,
                             max_seq_len: Optional[int] = None, partition_tokens: int = 0,
                             impl: str = "auto", workspace: Optional[torch.Tensor] = None,
                             table: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None, flags: int = 0):
    """Decode of several layers in one launch (pkv_paged_attn_decode_layers).

    ``layers``: list of dicts with keys LAYER_FIELDS: per layer q [S, Hq, D],
    optional new_k / new_v [S, Hkv, D] (the fused cache write of
    ``paged_attn_decode_append``; seq_lens then include the new token),
    k_cache / v_cache [N, Hkv, D, 16] and out [S, Hq, D].  All layers share
    block_tables and seq_lens, and the dtypes and shapes of the first layer.
    ``table`` is a prebuilt ``layer_table(layers)`` (needed under CUDA-graph
    capture; otherwise built here).  Returns the list of outputs.
    """
    dev = layers[0]["q"].device
    first = layers[0]
    for lay in layers:
        for name, nd in (("q", 3), ("k_cache", 4), ("v_cache", 4), ("out", 3)):
            _check(lay[name], name, nd, dev)
            if lay[name].shape != first[name].shape or lay[name].dtype != first[name].dtype:
                raise ValueError(f"layer {name} differs from the first layer's")
        for name in ("new_k", "new_v"):
            if lay.get(name) is not None:
                _check(lay[name], name, 3, dev)
    _check(block_tables, "block_tables", 2, dev)
    _check(seq_lens, "seq_lens", 1, dev)
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    q, kc = first["q"], first["k_cache"]
    S, Hq, D = q.shape
    N, Hkv, D2, B = _pool_dims(kc)
    if D2 != D or first["out"].shape != q.shape or block_tables.shape[0] != S \
            or seq_lens.shape[0] != S:
        raise ValueError("inconsistent shapes")
    new_dtype = F32
    for lay in layers:
        nk, nv = lay.get("new_k"), lay.get("new_v")
        if (nk is None) != (nv is None):
            raise ValueError("new_k and new_v must both be given or both be None")
        if nk is not None:
            if nk.shape != (S, Hkv, D) or nv.shape != nk.shape or nv.dtype != nk.dtype:
                raise ValueError("inconsistent new row shapes")
            new_dtype = _dtype_code(nk, "new_k")
    max_blocks = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = max_blocks * B
    NL = len(layers)
    L = lib()
    need = L.pkv_paged_attn_layers_workspace_size(NL, S, Hq, Hkv, D, B, max_seq_len,
                                                  partition_tokens)
    if need == 0:
        raise ValueError("invalid sizes or partition_tokens")
    if workspace is None:
        workspace = get_workspace(need, dev)
    if table is None:
        table = layer_table(layers, dev)
    if table.dtype != torch.int64 or tuple(table.shape) != (NL, len(LAYER_FIELDS)) \
            or table.device != dev or not table.is_contiguous():
        raise ValueError("table must be a contiguous int64 [num_layers, 6] tensor on q's device")
    flags |= IMPL[impl]
    rc = L.pkv_paged_attn_decode_layers(
        table.data_ptr(), NL, _dtype_code(q, "q"), new_dtype, _dtype_code(kc, "k_cache"),
        float(k_scale), float(v_scale), block_tables.data_ptr(), seq_lens.data_ptr(), S, Hq,
        Hkv, D, B, N, max_blocks, int(max_seq_len), float(scale),
        _dtype_code(first["out"], "out"), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), int(partition_tokens), int(flags),
        _stream(dev, stream))
    if rc != 0:
        raise PkvError(rc, "pkv_paged_attn_decode_layers")
    return [lay["out"] for lay in layers]


def prefill_workspace_size(num_seqs: int, num_tokens: int, num_q_heads: int, num_kv_heads: int,
                           head_dim: int, max_q_len: int, max_seq_len: int,
                           partition_tokens: int = 0, block_size: int = 16) -> int:
    n = lib().pkv_paged_attn_prefill_workspace_size(num_seqs, num_tokens, num_q_heads,
                                                    num_kv_heads, head_dim, block_size,
                                                    max_q_len, max_seq_len, partition_tokens)
    if n == 0:
        raise ValueError("invalid sizes for the prefill workspace")
    return int(n)


def prefill_partition_tokens(num_seqs: int, num_tokens: int, num_q_heads: int,
                             num_kv_heads: int, head_dim: int, max_q_len: int, max_seq_len: int,
                             partition_tokens: int = 0, block_size: int = 16) -> int:
    """Partition of the several-queries call: 0 none, > 0 tokens per partition."""
    return int(lib().pkv_paged_attn_prefill_partition_tokens(
        num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size, max_q_len,
        max_seq_len, partition_tokens))


def paged_attn_prefill(q: torch.Tensor, q_start: torch.Tensor, k_cache: torch.Tensor,
                       v_cache: torch.Tensor, block_tables: torch.Tensor,
                       seq_lens: torch.Tensor, scale: float, out: torch.Tensor, *,
                       max_q_len: Optional[int] = None, max_seq_len: Optional[int] = None,
                       partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None, flags: int = 0,
                       k_scale: float = 1.0, v_scale: float = 1.0) -> torch.Tensor:
    """Causal paged attention of several query tokens per sequence.

    q [T, Hq, D] bf16; q_start int32 [S+1] (queries of sequence s are rows
    q_start[s]..q_start[s+1]-1, its last positions); k_cache, v_cache
    [N, Hkv, D, 16] bf16 / fp8 (e5m2, e4m3) / INT4 (uint8, [N, Hkv, D, 8])
    already holding the queries' K/V, with dequant scales k_scale, v_scale;
    block_tables int32 [S, max_blocks]; seq_lens int32 [S] (queries
    included); out [T, Hq, D] f32/bf16.  ``max_q_len`` defaults to T,
    ``max_seq_len`` to max_blocks*16.  ``flags``: ``IMPL["auto"]`` runs the
    tcgen05 kernel on bf16 caches and the mma.sync one on the others;
    ``IMPL["tc"]`` (bf16 only) / ``IMPL["mma"]`` choose (same results within
    the tolerance).  Returns ``out``.
    """
    dev = q.device
    for t, name, nd in ((q, "q", 3), (q_start, "q_start", 1), (k_cache, "k_cache", 4),
                        (v_cache, "v_cache", 4), (block_tables, "block_tables", 2),
                        (seq_lens, "seq_lens", 1), (out, "out", 3)):
        _check(t, name, nd, dev)
    if (block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32
            or q_start.dtype != torch.int32):
        raise TypeError("q_start, block_tables and seq_lens must be int32")
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must have the same shape and dtype")
    T, Hq, D = q.shape
    N, Hkv, D2, B = _pool_dims(k_cache)
    S = seq_lens.shape[0]
    if (D2 != D or out.shape != q.shape or block_tables.shape[0] != S
            or q_start.shape[0] != S + 1):
        raise ValueError("inconsistent shapes")
    max_blocks = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = max_blocks * B
    if max_q_len is None:
        max_q_len = T
    L = lib()
    need = L.pkv_paged_attn_prefill_workspace_size(S, T, Hq, Hkv, D, B, int(max_q_len),
                                                   int(max_seq_len), int(partition_tokens))
    if need == 0:
        raise ValueError("invalid sizes or partition_tokens")
    if workspace is None:
        workspace = get_workspace(need, dev)
    rc = L.pkv_paged_attn_prefill(
        q.data_ptr(), _dtype_code(q, "q"), q_start.data_ptr(), k_cache.data_ptr(),
        v_cache.data_ptr(), _dtype_code(k_cache, "k_cache"), float(k_scale), float(v_scale),
        block_tables.data_ptr(),
        seq_lens.data_ptr(), S, T, Hq, Hkv, D, B, N, max_blocks, int(max_q_len),
        int(max_seq_len), float(scale), out.data_ptr(), _dtype_code(out, "out"),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        int(partition_tokens), int(flags), _stream(dev, stream))
    if rc != 0:
        raise PkvError(rc, "pkv_paged_attn_prefill")
    return out


def reshape_and_cache(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                      k_cache: torch.Tensor, v_cache: torch.Tensor, *, k_scale: float = 1.0,
                      v_scale: float = 1.0, status: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> None:
    """Writes k, v [T, Hkv, D] into their slots (block*16+offset; <0 = skip)."""
    dev = k.device
    _check(k, "k", 3, dev)
    _check(v, "v", 3, dev)
    _check(slot_mapping, "slot_mapping", 1, dev)
    _check(k_cache, "k_cache", 4, dev)
    _check(v_cache, "v_cache", 4, dev)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    T, Hkv, D = k.shape
    N, Hkv2, D2, B = _pool_dims(k_cache)
    if v.shape != k.shape or Hkv2 != Hkv or D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent shapes")
    if slot_mapping.shape[0] != T:
        raise ValueError("slot_mapping must have one entry per token")
    st_ptr = None
    if status is not None:
        _check(status, "status", 1, dev)
        st_ptr = status.data_ptr()
    rc = lib().pkv_reshape_and_cache(
        k.data_ptr(), v.data_ptr(), _dtype_code(k, "k"), slot_mapping.data_ptr(), T, Hkv, D, B,
        N, k_cache.data_ptr(), v_cache.data_ptr(), _dtype_code(k_cache, "k_cache"),
        float(k_scale), float(v_scale), st_ptr, _stream(dev, stream))
    if rc != 0:
        raise PkvError(rc, "pkv_reshape_and_cache")


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, pairs: torch.Tensor, *,
                status: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy-on-write page copies: block pairs[i, 1] of both caches becomes a copy
    of block pairs[i, 0] (pairs: int32 [n, 2] on the caches' device)."""
    dev = k_cache.device
    _check(k_cache, "k_cache", 4, dev)
    _check(v_cache, "v_cache", 4, dev)
    _check(pairs, "pairs", 2, dev)
    if pairs.dtype != torch.int32 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int32 [n, 2]")
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must have the same shape and dtype")
    N, Hkv, D, B = _pool_dims(k_cache)
    st_ptr = None
    if status is not None:
        _check(status, "status", 1, dev)
        st_ptr = status.data_ptr()
    rc = lib().pkv_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(),
                               _dtype_code(k_cache, "k_cache"), Hkv, D, B, N, pairs.data_ptr(),
                               pairs.shape[0], st_ptr, _stream(dev, stream))
    if rc != 0:
        raise PkvError(rc, "pkv_copy_blocks")


class BlockManager:
    """Host-side page pool of one paged cache (the C library's pkv_bm_* calls).

    ``add`` a sequence with its prompt, ``fork`` a sequence that shares every
    page of another, ``append`` one token to each listed sequence (returns the
    slots and the copy-on-write page pairs to copy first), ``free`` a
    sequence, and ``tables`` for the dense block tables attention reads.
    """

    def __init__(self, num_blocks: int, block_size: int = 16, max_blocks_per_seq: int = 1 << 20):
        self._lib = lib()
        h = ctypes.c_void_p()
        rc = self._lib.pkv_bm_create(num_blocks, block_size, max_blocks_per_seq, ctypes.byref(h))
        if rc != 0:
            raise PkvError(rc, "pkv_bm_create")
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.max_blocks_per_seq = max_blocks_per_seq

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.pkv_bm_destroy(h)
            self._h = None

    @staticmethod
    def _p(a, ct):
        return a.ctypes.data_as(ctypes.POINTER(ct))

    def add(self, seq_id: int, num_tokens: int):
        import numpy as np
        slots = np.empty(max(num_tokens, 1), dtype=np.int64)
        rc = self._lib.pkv_bm_add(self._h, seq_id, num_tokens, self._p(slots, ctypes.c_int64))
        if rc != 0:
            raise PkvError(rc, "pkv_bm_add")
        return slots[:num_tokens]

    def fork(self, parent_id: int, child_id: int) -> None:
        rc = self._lib.pkv_bm_fork(self._h, parent_id, child_id)
        if rc != 0:
            raise PkvError(rc, "pkv_bm_fork")

    def append(self, seq_ids):
        """One token for each sequence; returns (slots int64 [n], pairs int32 [c, 2])."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        n = ids.size
        slots = np.empty(max(n, 1), dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int32)
        nc = ctypes.c_int(0)
        rc = self._lib.pkv_bm_append(self._h, self._p(ids, ctypes.c_int32), n,
                                     self._p(slots, ctypes.c_int64),
                                     self._p(pairs, ctypes.c_int32), ctypes.byref(nc))
        if rc != 0:
            raise PkvError(rc, "pkv_bm_append")
        return slots[:n], pairs[:nc.value]

    def free(self, seq_id: int) -> None:
        rc = self._lib.pkv_bm_free(self._h, seq_id)
        if rc != 0:
            raise PkvError(rc, "pkv_bm_free")

    def tables(self, seq_ids, max_blocks_per_seq: int):
        """Dense block tables int32 [n, max_blocks_per_seq] (-1 padded) and lengths."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        tab = np.empty((max(ids.size, 1), max_blocks_per_seq), dtype=np.int32)
        lens = np.empty(max(ids.size, 1), dtype=np.int32)
        rc = self._lib.pkv_bm_tables(self._h, self._p(ids, ctypes.c_int32), ids.size,
                                     max_blocks_per_seq, self._p(tab, ctypes.c_int32),
                                     self._p(lens, ctypes.c_int32))
        if rc != 0:
            raise PkvError(rc, "pkv_bm_tables")
        return tab[:ids.size], lens[:ids.size]

    def num_free(self) -> int:
        return int(self._lib.pkv_bm_num_free(self._h))

    def ref_count(self, block: int) -> int:
        return int(self._lib.pkv_bm_ref_count(self._h, block))


def read_status(workspace: Optional[torch.Tensor] = None, clear: bool = True,
                device: Optional[torch.device] = None) -> int:
    """Status word of a decode workspace (default: the cached one of ``device``)."""
    if workspace is None:
        dev = device or torch.device("cuda", torch.cuda.current_device())
        workspace = _workspaces[(dev.type, dev.index)]
    out = ctypes.c_int32(0)
    rc = lib().pkv_read_status(workspace.data_ptr(), int(clear), ctypes.byref(out),
                               _stream(workspace.device, None))
    if rc != 0:
        raise PkvError(rc, "pkv_read_status")
    return int(out.value)
