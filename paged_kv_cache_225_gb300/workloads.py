"""Seeded synthetic decode-step workloads for paged decode attention.

This module only draws random numbers and lays them out as a paged KV pool
(block tables, sequence lengths, slot mappings).  It holds none of the
attention arithmetic: both the CUDA path and the CPU oracle consume what it
produces, and neither depends on the other.

Every array is a host numpy array holding the exact bit patterns the kernels
read: float32 values as ``np.float32``, bf16 as ``np.uint16`` bit patterns and
fp8-e5m2 as ``np.uint8`` codes.  Rounding of the drawn float32 normals to the
stored dtype is done by PyTorch's round-to-nearest-even casts.

Shapes follow the pages' workloads (vLLM PagedAttention pseudocode page:
``K_cache [num_blocks, num_heads, head_dim, block_size]``, 16-token blocks;
"Inference optimization" lesson, Step 6 model table: Llama-3 8B/70B with 8 KV
heads of dim 128; 128 concurrent sequences, 32K context, 256-in/256-out chat,
a shared system prompt).

New-token convention (the pages never define a slot mapping): slot =
physical_block * block_size + offset.  The new token of sequence s is its next
logical position ``seq_lens[s]``; if that position starts a new block, a free
block of the pool is appended to the sequence's block table.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

F32, BF16, FP8_E5M2, FP8_E4M3, INT4 = 0, 1, 2, 3, 4
DTYPE_NAMES = {F32: "f32", BF16: "bf16", FP8_E5M2: "fp8_e5m2", FP8_E4M3: "fp8_e4m3",
               INT4: "int4"}
ELEM_BYTES = {F32: 4, BF16: 2, FP8_E5M2: 1, FP8_E4M3: 1, INT4: 0.5}
NP_STORAGE = {F32: np.float32, BF16: np.uint16, FP8_E5M2: np.uint8, FP8_E4M3: np.uint8,
              INT4: np.uint8}
FP8 = (FP8_E5M2, FP8_E4M3)
SCALED = (FP8_E5M2, FP8_E4M3, INT4)   # stored codes times a dequant scale


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    """Shape and distribution recipe of one synthetic decode-attention layer."""

    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    q_dtype: int
    kv_dtype: int
    len_dist: str               # "uniform" | "lognormal" | "const"
    len_lo: int = 1
    len_hi: int = 1
    len_median: float = 0.0
    len_sigma: float = 0.0
    pool_blocks: int = 0        # fixed pool size; 0 = needed blocks + slack
    pool_slack: float = 0.10
    garbage: str = "normal"     # content of slots no sequence owns: "normal" | "nan"
    heavy_key_frac: float = 0.0  # fraction of (token, kv_head) key rows scaled x8
    shared_prefix_group: int = 0   # sequences per shared-prefix group
    shared_prefix_blocks: int = 0  # leading table columns shared inside a group
    kv_scale: float = 1.0
    new_tokens: bool = True     # draw one new token per sequence (cache write)


# The five decode layers the benchmark and the parity suite run.
CONFIGS = {
    "tiny_fp32": DecodeConfig(
        name="tiny_fp32", num_seqs=4, num_q_heads=4, num_kv_heads=4, head_dim=64,
        block_size=16, q_dtype=F32, kv_dtype=F32, len_dist="uniform", len_lo=1,
        len_hi=64, pool_blocks=32, garbage="nan"),
    "llama3_8b": DecodeConfig(
        name="llama3_8b", num_seqs=64, num_q_heads=32, num_kv_heads=8, head_dim=128,
        block_size=16, q_dtype=BF16, kv_dtype=BF16, len_dist="uniform", len_lo=512,
        len_hi=4096),
    "llama3_70b": DecodeConfig(
        name="llama3_70b", num_seqs=128, num_q_heads=64, num_kv_heads=8, head_dim=128,
        block_size=16, q_dtype=BF16, kv_dtype=BF16, len_dist="lognormal",
        len_median=2048.0, len_sigma=0.8, len_lo=16, len_hi=32768),
    "long_split": DecodeConfig(
        name="long_split", num_seqs=8, num_q_heads=64, num_kv_heads=8, head_dim=128,
        block_size=16, q_dtype=BF16, kv_dtype=BF16, len_dist="const", len_lo=32768,
        len_hi=32768, heavy_key_frac=0.01),
    "fp8_chat": DecodeConfig(
        name="fp8_chat", num_seqs=128, num_q_heads=64, num_kv_heads=8, head_dim=128,
        block_size=16, q_dtype=BF16, kv_dtype=FP8_E5M2, len_dist="uniform", len_lo=256,
        len_hi=512, shared_prefix_group=8, shared_prefix_blocks=8),
    # The 70B layer with an fp8-e4m3 cache and a per-tensor scale of 1/8
    # (values stored as x * 8 before rounding, so N(0,1) data uses the
    # format's finer upper range).
    "e4m3_70b": DecodeConfig(
        name="e4m3_70b", num_seqs=128, num_q_heads=64, num_kv_heads=8, head_dim=128,
        block_size=16, q_dtype=BF16, kv_dtype=FP8_E4M3, len_dist="lognormal",
        len_median=2048.0, len_sigma=0.8, len_lo=16, len_hi=32768, kv_scale=0.125),
    # The 70B layer with an INT4 cache (scale 1/2: N(0,1) data spans the
    # codes -8..7 at +-3.5 sigma).
    "int4_70b": DecodeConfig(
        name="int4_70b", num_seqs=128, num_q_heads=64, num_kv_heads=8, head_dim=128,
        block_size=16, q_dtype=BF16, kv_dtype=INT4, len_dist="lognormal",
        len_median=2048.0, len_sigma=0.8, len_lo=16, len_hi=32768, kv_scale=0.5),
}
CONFIG_ORDER = ["tiny_fp32", "llama3_8b", "llama3_70b", "long_split", "fp8_chat", "e4m3_70b",
                "int4_70b"]
CONFIG_SEED = {name: i for i, name in enumerate(CONFIG_ORDER)}


@dataclasses.dataclass
class Workload:
    """One decode step's inputs, all on the host, as stored bit patterns."""

    cfg: DecodeConfig
    q: np.ndarray             # [S, Hq, D]
    k_cache: np.ndarray       # [N, Hkv, D, B]
    v_cache: np.ndarray       # [N, Hkv, D, B]
    block_tables: np.ndarray  # int32 [S, max_blocks]; -1 past each sequence's blocks
    seq_lens: np.ndarray      # int32 [S]  (context before the new token)
    new_k: Optional[np.ndarray]  # [S, Hkv, D] in q's dtype (f32 or bf16)
    new_v: Optional[np.ndarray]
    slot_mapping: Optional[np.ndarray]  # int64 [S]
    scale: float

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


def round_to_storage(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float32 values to the stored dtype (RNE, by PyTorch) and return bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F32:
        return x
    t = torch.from_numpy(x)
    if dtype == BF16:
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if dtype == FP8_E5M2:
        return t.clamp(-57344.0, 57344.0).to(torch.float8_e5m2).view(torch.uint8).numpy()
    if dtype == FP8_E4M3:
        # Clamp first: saturating to the largest finite value (448).
        return t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    if dtype == INT4:
        # Round half to even, clamp to -8..7 (NaN -> 0), pack pairs along the
        # last axis: even element in the low nibble.
        qv = np.clip(np.rint(np.nan_to_num(x, nan=0.0, posinf=7.0, neginf=-8.0)), -8, 7)
        nib = (qv.astype(np.int8).astype(np.uint8) & 0xF)
        return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    raise ValueError(f"unknown dtype {dtype}")


def storage_to_float32(x: np.ndarray, dtype: int) -> np.ndarray:
    """Widen stored bit patterns to float32 (exact for all three dtypes), by PyTorch."""
    if dtype == F32:
        return np.asarray(x, dtype=np.float32)
    if dtype == BF16:
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
        return t.float().numpy()
    if dtype == FP8_E5M2:
        t = torch.from_numpy(np.ascontiguousarray(x)).view(torch.float8_e5m2)
        return t.float().numpy()
    if dtype == FP8_E4M3:
        t = torch.from_numpy(np.ascontiguousarray(x)).view(torch.float8_e4m3fn)
        return t.float().numpy()
    if dtype == INT4:
        b = np.ascontiguousarray(x, dtype=np.uint8)
        lo = (b & 0xF).astype(np.int16)
        hi = (b >> 4).astype(np.int16)
        out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.float32)
        out[..., 0::2] = np.where(lo >= 8, lo - 16, lo)
        out[..., 1::2] = np.where(hi >= 8, hi - 16, hi)
        return out
    raise ValueError(f"unknown dtype {dtype}")


def _draw_lengths(cfg: DecodeConfig, rng: np.random.Generator) -> np.ndarray:
    S = cfg.num_seqs
    if cfg.len_dist == "uniform":
        L = rng.integers(cfg.len_lo, cfg.len_hi, size=S, endpoint=True)
    elif cfg.len_dist == "lognormal":
        z = rng.standard_normal(S)
        L = np.clip(np.round(cfg.len_median * np.exp(cfg.len_sigma * z)), cfg.len_lo, cfg.len_hi)
    elif cfg.len_dist == "const":
        L = np.full(S, cfg.len_lo)
    else:
        raise ValueError(cfg.len_dist)
    return L.astype(np.int32)


def _normal_pool(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """Draw a float32 N(0,1) array chunk by chunk (bounded temporary memory)."""
    out = np.empty(int(np.prod(shape)), dtype=np.float32)
    for lo in range(0, out.size, chunk):
        hi = min(out.size, lo + chunk)
        out[lo:hi] = rng.standard_normal(hi - lo, dtype=np.float32)
    return out.reshape(shape)


def _pool_to_storage(pool_f32: np.ndarray, dtype: int, chunk: int = 1 << 24) -> np.ndarray:
    flat = pool_f32.reshape(-1)
    per = 2 if dtype == INT4 else 1          # elements per stored byte
    out = np.empty(flat.size // per, dtype=NP_STORAGE[dtype])
    for lo in range(0, flat.size, chunk):    # chunk is even: INT4 pairs stay together
        hi = min(flat.size, lo + chunk)
        out[lo // per:hi // per] = round_to_storage(flat[lo:hi], dtype)
    shape = pool_f32.shape[:-1] + (pool_f32.shape[-1] // per,)
    return out.reshape(shape)


def make_workload(cfg: DecodeConfig | str, seed: Optional[int] = None,
                  seq_lens: Optional[np.ndarray] = None) -> Workload:
    """Build the seeded workload of ``cfg``.

    Draw order from ``numpy.random.default_rng(seed)``: sequence lengths,
    block permutation, q, K pool, V pool, heavy-key mask, new K, new V.
    ``seq_lens`` overrides the drawn lengths (edge-case tests).
    """
    if isinstance(cfg, str):
        if seed is None:
            seed = CONFIG_SEED[cfg]
        cfg = CONFIGS[cfg]
    if seed is None:
        seed = 0
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, D, B = cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size

    L = _draw_lengths(cfg, rng)
    if seq_lens is not None:
        L = np.asarray(seq_lens, dtype=np.int32).copy()
        assert L.shape == (S,)
    nb = (L.astype(np.int64) + B - 1) // B            # blocks holding the context
    app = (L % B == 0) & cfg.new_tokens                # new token opens a block
    nb_total = nb + app.astype(np.int64)

    # Physical pool: a seeded permutation hands out block ids; shared prefixes
    # point several table rows at the same blocks.
    share_g, share_b = cfg.shared_prefix_group, cfg.shared_prefix_blocks
    if share_g:
        assert S % share_g == 0 and np.all(nb >= share_b) and np.all(L > share_b * B)
        private = nb_total - share_b
        needed = int(private.sum()) + (S // share_g) * share_b
    else:
        needed = int(nb_total.sum())
    if cfg.pool_blocks:
        N = cfg.pool_blocks
        assert N >= needed, (N, needed)
    else:
        N = int(math.ceil(needed * (1.0 + cfg.pool_slack)))
    perm = rng.permutation(N).astype(np.int32)

    max_blocks = int(nb_total.max()) if S else 1
    max_blocks = max(max_blocks, 1)
    tables = np.full((S, max_blocks), -1, dtype=np.int32)
    cursor = 0
    if share_g:
        for g0 in range(0, S, share_g):
            shared = perm[cursor:cursor + share_b]
            cursor += share_b
            for s in range(g0, g0 + share_g):
                tables[s, :share_b] = shared
                n_priv = int(nb[s]) - share_b
                tables[s, share_b:share_b + n_priv] = perm[cursor:cursor + n_priv]
                cursor += n_priv
    else:
        for s in range(S):
            n = int(nb[s])
            tables[s, :n] = perm[cursor:cursor + n]
            cursor += n
    # Blocks opened by the new tokens come after every context block.
    for s in range(S):
        if app[s]:
            tables[s, nb[s]] = perm[cursor]
            cursor += 1

    q, k_cache, v_cache, new_k, new_v = _draw_values(cfg, rng, N, tables, L, nb)
    slots = None
    if cfg.new_tokens:
        slots = np.empty(S, dtype=np.int64)
        for s in range(S):
            pos = int(L[s])
            slots[s] = int(tables[s, pos // B]) * B + pos % B

    return Workload(cfg=cfg, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=tables,
                    seq_lens=L, new_k=new_k, new_v=new_v, slot_mapping=slots,
                    scale=1.0 / math.sqrt(D))


def _draw_values(cfg: DecodeConfig, rng: np.random.Generator, N: int, tables: np.ndarray,
                 L: np.ndarray, nb: np.ndarray):
    """q, the K and V pools and the new rows of one layer, in that draw order."""
    S, Hq, Hkv, D, B = cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size
    q = round_to_storage(rng.standard_normal((S, Hq, D), dtype=np.float32), cfg.q_dtype)
    k_pool = _normal_pool(rng, (N, Hkv, D, B))
    v_pool = _normal_pool(rng, (N, Hkv, D, B))
    if cfg.heavy_key_frac > 0:
        heavy = rng.random((N, Hkv, B)) < cfg.heavy_key_frac
        k_pool *= np.where(heavy, np.float32(8.0), np.float32(1.0))[:, :, None, :]
    if cfg.garbage == "nan":
        owned = np.zeros((N, B), dtype=bool)
        for s in range(S):
            for j in range(int(nb[s])):
                valid = min(B, int(L[s]) - j * B)
                owned[tables[s, j], :valid] = True
        k_pool[np.broadcast_to(~owned[:, None, None, :], k_pool.shape)] = np.nan
        v_pool[np.broadcast_to(~owned[:, None, None, :], v_pool.shape)] = np.nan
    if cfg.kv_dtype in SCALED and cfg.kv_scale != 1.0:
        k_pool /= np.float32(cfg.kv_scale)
        v_pool /= np.float32(cfg.kv_scale)
    k_cache = _pool_to_storage(k_pool, cfg.kv_dtype)
    del k_pool
    v_cache = _pool_to_storage(v_pool, cfg.kv_dtype)
    del v_pool

    new_k = new_v = None
    if cfg.new_tokens:
        new_k = round_to_storage(rng.standard_normal((S, Hkv, D), dtype=np.float32), cfg.q_dtype)
        new_v = round_to_storage(rng.standard_normal((S, Hkv, D), dtype=np.float32), cfg.q_dtype)
    return q, k_cache, v_cache, new_k, new_v


def make_layers(cfg: DecodeConfig | str, num_layers: int, seed: Optional[int] = None,
                seq_lens: Optional[np.ndarray] = None) -> list:
    """num_layers workloads of one decoder stack over the same batch: layer 0 is
    ``make_workload(cfg, seed)``; every other layer shares its block tables,
    lengths and slots and draws its own q, K/V pools and new rows (same
    recipe) from ``default_rng((seed, layer))``."""
    if isinstance(cfg, str):
        if seed is None:
            seed = CONFIG_SEED[cfg]
        cfg = CONFIGS[cfg]
    if seed is None:
        seed = 0
    w0 = make_workload(cfg, seed=seed, seq_lens=seq_lens)
    B = cfg.block_size
    nb = (w0.seq_lens.astype(np.int64) + B - 1) // B
    out = [w0]
    for layer in range(1, num_layers):
        rng = np.random.default_rng((seed, layer))
        q, kc, vc, nk, nv = _draw_values(cfg, rng, w0.num_blocks, w0.block_tables, w0.seq_lens,
                                         nb)
        out.append(dataclasses.replace(w0, q=q, k_cache=kc, v_cache=vc, new_k=nk, new_v=nv))
    return out


# ------------------------------------------------------------------ several queries per sequence

@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    """Recipe of one batch with several causal query tokens per sequence.

    ``base`` fixes head shapes, dtypes and the context-length recipe; here a
    sequence's length counts its queries, whose K/V are already in the cache.
    Every sequence gets ``q_len`` queries (0 = all of its tokens), capped at
    its length, unless ``q_lens`` lists them; the first ``chunk_seqs``
    sequences instead run a prefill chunk of ``chunk_len`` queries at a
    length drawn from U{chunk_ctx_lo..chunk_ctx_hi} (vLLM's chunked prefill
    mixes such chunks with decoding sequences in one step).
    """

    name: str
    base: DecodeConfig
    q_len: int = 1
    q_lens: tuple = ()
    chunk_seqs: int = 0
    chunk_len: int = 0
    chunk_ctx_lo: int = 0
    chunk_ctx_hi: int = 0


PREFILL_CONFIGS = {
    # Small mixed case the oracle finishes in well under a second: ragged
    # lengths, a whole-prompt prefill, row counts that need one to four warp
    # tiles and several row blocks, NaN in every slot no sequence owns.
    "prefill_tiny": PrefillConfig(
        name="prefill_tiny",
        base=DecodeConfig(name="prefill_tiny", num_seqs=7, num_q_heads=8, num_kv_heads=2,
                          head_dim=64, block_size=16, q_dtype=BF16, kv_dtype=BF16,
                          len_dist="uniform", len_lo=1, len_hi=200, garbage="nan",
                          new_tokens=False),
        q_lens=(1, 3, 16, 33, 0, 10, 2)),
    # Speculative verification on the Llama-3-70B layer: five draft tokens
    # per sequence checked in one pass ("Inference optimization" lesson,
    # speculative decoding: the target model scores the ~5 guesses at once).
    "spec_verify_70b": PrefillConfig(
        name="spec_verify_70b",
        base=DecodeConfig(name="spec_verify_70b", num_seqs=128, num_q_heads=64,
                          num_kv_heads=8, head_dim=128, block_size=16, q_dtype=BF16,
                          kv_dtype=BF16, len_dist="lognormal", len_median=2048.0,
                          len_sigma=0.8, len_lo=16, len_hi=32768, new_tokens=False),
        q_len=5),
    # Chunked prefill on the Llama-3-8B layer: four 256-token prompt chunks
    # scheduled with 60 decoding sequences.
    "chunked_prefill_8b": PrefillConfig(
        name="chunked_prefill_8b",
        base=DecodeConfig(name="chunked_prefill_8b", num_seqs=64, num_q_heads=32,
                          num_kv_heads=8, head_dim=128, block_size=16, q_dtype=BF16,
                          kv_dtype=BF16, len_dist="uniform", len_lo=512, len_hi=4096,
                          new_tokens=False),
        q_len=1, chunk_seqs=4, chunk_len=256, chunk_ctx_lo=1024, chunk_ctx_hi=4096),
    # The speculative-verification layer over an fp8-e5m2 cache (scale 1),
    # the KV dtype of the pages' vLLM serving setup.
    "spec_verify_70b_fp8": PrefillConfig(
        name="spec_verify_70b_fp8",
        base=DecodeConfig(name="spec_verify_70b_fp8", num_seqs=128, num_q_heads=64,
                          num_kv_heads=8, head_dim=128, block_size=16, q_dtype=BF16,
                          kv_dtype=FP8_E5M2, len_dist="lognormal", len_median=2048.0,
                          len_sigma=0.8, len_lo=16, len_hi=32768, new_tokens=False),
        q_len=5),
}
PREFILL_SEED = {name: 100 + i for i, name in enumerate(PREFILL_CONFIGS)}


@dataclasses.dataclass
class PrefillWorkload:
    cfg: PrefillConfig
    q: np.ndarray             # [T, Hq, D]
    q_start: np.ndarray       # int32 [S + 1]
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_tables: np.ndarray
    seq_lens: np.ndarray      # int32 [S], queries included
    scale: float

    @property
    def num_tokens(self) -> int:
        return int(self.q_start[-1])

    @property
    def max_q_len(self) -> int:
        return int(np.max(np.diff(self.q_start))) if self.seq_lens.size else 0


def make_prefill_workload(cfg: PrefillConfig | str, seed: Optional[int] = None,
                          seq_lens: Optional[np.ndarray] = None,
                          q_lens: Optional[np.ndarray] = None) -> PrefillWorkload:
    """Build the seeded several-queries workload of ``cfg``.

    Draw order from ``default_rng(seed)``: lengths, chunk lengths, then the
    cache (``make_workload`` of the base recipe with seed + 1), then q.
    ``seq_lens`` / ``q_lens`` override the drawn values (edge-case tests).
    """
    if isinstance(cfg, str):
        if seed is None:
            seed = PREFILL_SEED[cfg]
        cfg = PREFILL_CONFIGS[cfg]
    if seed is None:
        seed = 0
    rng = np.random.default_rng(seed)
    base = cfg.base
    S = base.num_seqs
    L = _draw_lengths(base, rng)
    if cfg.chunk_seqs:
        L[:cfg.chunk_seqs] = rng.integers(cfg.chunk_ctx_lo, cfg.chunk_ctx_hi,
                                          size=cfg.chunk_seqs, endpoint=True)
    if seq_lens is not None:
        L = np.asarray(seq_lens, dtype=np.int32).copy()
    if q_lens is not None:
        n = np.asarray(q_lens, dtype=np.int64).copy()
    elif cfg.q_lens:
        n = np.asarray(cfg.q_lens, dtype=np.int64)
        n = np.where(n == 0, L, n)
    else:
        n = np.full(S, cfg.q_len if cfg.q_len > 0 else 0, dtype=np.int64)
        n = np.where(n == 0, L, n)
        if cfg.chunk_seqs:
            n[:cfg.chunk_seqs] = cfg.chunk_len
    n = np.minimum(n, L).astype(np.int32)
    w = make_workload(base, seed=seed + 1, seq_lens=L)
    q_start = np.zeros(S + 1, dtype=np.int32)
    q_start[1:] = np.cumsum(n)
    T = int(q_start[-1])
    q = round_to_storage(rng.standard_normal((T, base.num_q_heads, base.head_dim),
                                             dtype=np.float32), base.q_dtype)
    return PrefillWorkload(cfg=cfg, q=q, q_start=q_start, k_cache=w.k_cache,
                           v_cache=w.v_cache, block_tables=w.block_tables, seq_lens=w.seq_lens,
                           scale=w.scale)
