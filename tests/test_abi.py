"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/pkv.h declares, plans workspaces, and rejects bad arguments
before it touches CUDA."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_225_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]

OK, INVALID, UNSUPPORTED, CUDA, OOR, TIMEOUT, WORKSPACE = range(7)
F32, BF16, FP8 = pkv.F32, pkv.BF16, pkv.FP8_E5M2


def declared_functions():
    names = []
    for h in HEADERS:
        txt = open(h).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        txt = re.sub(r"//[^\n]*", "", txt)
        names += re.findall(r"\b(pkv_\w+)\s*\(", txt)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pkv_paged_attn_decode", "pkv_reshape_and_cache",
                     "pkv_paged_attn_workspace_size", "pkv_read_status", "pkv_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol():
    L = pkv.lib()
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in include/*.h but not exported"


def test_status_strings_and_version():
    L = pkv.lib()
    for code in range(8):
        assert L.pkv_status_string(code).decode().startswith(pkv.STATUS[code])
    assert L.pkv_version() >= 100


def test_partition_plan():
    P = pkv.partition_tokens
    assert P(4, 4, 4, 64, 65, -1) == 0
    assert P(4, 4, 4, 64, 65, 48) == 48
    assert P(4, 4, 4, 64, 65, 40) == -1           # not a multiple of the block size
    # Automatic: many (sequence, KV head) units -> one pass (short contexts) or
    # 4096-token items; few units -> stream-K.
    assert P(128, 64, 8, 128, 514, 0) == 0              # fp8 chat mix: 1024 units
    assert P(128, 64, 8, 128, 14626, 0) == 4096         # 70B-shaped layer: 1024 units
    assert P(64, 32, 8, 128, 4097, 0) == pkv.SCHEDULE_STREAMK    # 8B-shaped: 512 units
    assert P(8, 64, 8, 128, 32769, 0) == pkv.SCHEDULE_STREAMK    # long context: 64 units
    assert P(1, 8, 8, 128, 512, 0) == pkv.SCHEDULE_STREAMK
    assert P(128, 64, 8, 128, 14626, -2) == pkv.SCHEDULE_STREAMK   # asked for explicitly


def test_workspace_size():
    W = pkv.workspace_size
    assert W(4, 4, 4, 64, 65, -1) == 256
    S, Hq, D, P, L = 8, 64, 128, 512, 32769
    parts = -(-L // P)
    rows = S * Hq * parts

    def a(x):
        return (x + 255) // 256 * 256
    # header | arrival counters [S*Hkv] | partial outputs | partial (m, l)
    assert W(S, Hq, 8, D, L, P) == 256 + a(S * 8 * 4) + a(rows * D * 4) + a(rows * 8)
    # Stream-K: two partial slots of G rows for each of up to 1024 CTAs,
    # independent of the lengths.
    G = Hq // 8
    rows = 2 * 1024 * G
    sk = 256 + a(S * 8 * 4) + a(rows * D * 4) + a(rows * 8)
    assert W(S, Hq, 8, D, L, 0) == sk == W(S, Hq, 8, D, 16, 0)
    with pytest.raises(ValueError):
        W(4, 6, 4, 64, 65, 0)                       # heads do not divide


def _decode(**kw):
    args = dict(q=0x1000, q_dtype=BF16, k=0x2000, v=0x3000, kv_dtype=BF16, ks=1.0, vs=1.0,
                bt=0x4000, sl=0x5000, S=2, Hq=8, Hkv=2, D=128, B=16, N=10, maxb=4, maxl=64,
                scale=0.1, out=0x6000, out_dtype=F32, ws=0x7000, wsb=1 << 26, part=0, flags=0)
    args.update(kw)
    return pkv.lib().pkv_paged_attn_decode(
        args["q"], args["q_dtype"], args["k"], args["v"], args["kv_dtype"], args["ks"], args["vs"],
        args["bt"], args["sl"], args["S"], args["Hq"], args["Hkv"], args["D"], args["B"], args["N"],
        args["maxb"], args["maxl"], args["scale"], args["out"], args["out_dtype"], args["ws"],
        args["wsb"], args["part"], args["flags"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=6, Hkv=4), INVALID),
    (dict(D=96), UNSUPPORTED),
    (dict(B=32), UNSUPPORTED),
    (dict(Hq=34, Hkv=2), UNSUPPORTED),            # 17 query heads per KV head
    (dict(q_dtype=FP8), UNSUPPORTED),
    (dict(out_dtype=FP8), UNSUPPORTED),
    (dict(kv_dtype=7), UNSUPPORTED),
    (dict(maxl=65), INVALID),                     # longer than the table allows
    (dict(ws=0), WORKSPACE),
    (dict(ws=0x7010), WORKSPACE),                 # not 256-byte aligned
    (dict(wsb=100), WORKSPACE),
    (dict(q=0), INVALID),
    (dict(k=0x2008), INVALID),                    # misaligned cache
    (dict(bt=0x4002), INVALID),
    (dict(part=40), INVALID),
    (dict(flags=0x3), INVALID),                   # the tcgen05 kernel is several-queries only
    (dict(flags=0x40), INVALID),
    (dict(flags=0x8), INVALID),
    (dict(flags=0x2, kv_dtype=F32), UNSUPPORTED),  # tensor cores need bf16/fp8 KV
    (dict(flags=0x2, q_dtype=F32), UNSUPPORTED),
    (dict(scale=float("nan")), INVALID),
    (dict(S=0), OK),                              # nothing to do, nothing enqueued
])
def test_decode_argument_errors(kw, code):
    assert _decode(**kw) == code


def _cache(**kw):
    args = dict(k=0x1000, v=0x2000, in_dtype=BF16, slots=0x3000, T=4, Hkv=2, D=128, B=16, N=8,
                kc=0x4000, vc=0x5000, kv_dtype=BF16, ks=1.0, vs=1.0, status=None)
    args.update(kw)
    return pkv.lib().pkv_reshape_and_cache(
        args["k"], args["v"], args["in_dtype"], args["slots"], args["T"], args["Hkv"], args["D"],
        args["B"], args["N"], args["kc"], args["vc"], args["kv_dtype"], args["ks"], args["vs"],
        args["status"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(in_dtype=FP8), UNSUPPORTED),
    (dict(kv_dtype=9), UNSUPPORTED),
    (dict(B=8), UNSUPPORTED),
    (dict(k=0), INVALID),
    (dict(slots=0x3004), INVALID),
    (dict(kc=0x4004), INVALID),
    (dict(kv_dtype=FP8, ks=0.0), INVALID),
    (dict(T=-1), INVALID),
    (dict(T=0), OK),
])
def test_reshape_argument_errors(kw, code):
    assert _cache(**kw) == code


def test_binding_rejects_cpu_tensors_without_fallback():
    import torch
    q = torch.zeros(1, 1, 64)
    kc = torch.zeros(1, 1, 64, 16)
    with pytest.raises((ValueError, RuntimeError, TypeError)):
        pkv.paged_attn_decode(q, kc, kc, torch.zeros(1, 1, dtype=torch.int32),
                              torch.ones(1, dtype=torch.int32), 0.125, torch.empty_like(q))


# ------------------------------------------------- several queries per sequence

def test_prefill_partition_plan():
    P = pkv.prefill_partition_tokens
    assert P(4, 20, 8, 2, 64, 8, 200, -1) == 0
    assert P(4, 20, 8, 2, 64, 8, 200, 48) == 48
    assert P(4, 20, 8, 2, 64, 8, 200, 40) == -1          # not a multiple of the block size
    # Enough (KV head, 64-row block) items: no split for short contexts,
    # 4096-token partitions for long ones.
    assert P(128, 640, 64, 8, 128, 5, 2000, 0) == 0
    assert P(128, 640, 64, 8, 128, 5, 14563, 0) == 4096
    # One wave of items (304..607 estimated): no split, no merge.
    assert P(64, 4 * 256 + 60, 32, 8, 128, 256, 4352, 0) == 0    # chunked prefill: 544
    # Few items: split so that about four items per resident CTA exist.
    assert P(2, 8, 64, 8, 128, 5, 32768, 0) == 1024       # 16 items -> 38 parts
    assert P(2, 8, 64, 8, 128, 5, 300, 0) == 256
    assert P(2, 8, 64, 8, 128, 5, 256, 0) == 0           # one partition covers it


def test_prefill_workspace_size():
    W = pkv.prefill_workspace_size
    assert W(4, 20, 8, 2, 64, 8, 200, -1) == 256
    T, Hq, D, P, L = 40, 64, 128, 512, 2049
    parts = -(-L // P)
    rows = T * Hq * parts

    def a(x):
        return (x + 255) // 256 * 256
    assert W(8, T, Hq, 8, D, 5, L, P) == 256 + a(rows * D * 4) + a(rows * 8)
    with pytest.raises(ValueError):
        W(4, 20, 6, 4, 64, 8, 200, 0)                     # heads do not divide


def test_prefill_workspace_of_a_mixed_batch_holds_the_routed_decode():
    """A batch that mixes one-query sequences with longer ones (fewer query
    rows than num_seqs * max_q_len) sends the one-query sequences to the
    decode kernels: the workspace adds that decode plan's counters and
    partials after the several-queries partials."""
    W, WD = pkv.prefill_workspace_size, pkv.workspace_size

    def a(x):
        return (x + 255) // 256 * 256
    S, Hq, Hkv, D, L, P = 64, 32, 8, 128, 4096, 512
    T = 4 * 256 + 60                                   # chunked prefill: 4 chunks + 60 decodes
    parts = -(-L // P)
    rows = T * Hq * parts
    own = 256 + a(rows * D * 4) + a(rows * 8)
    assert W(S, T, Hq, Hkv, D, 256, L, P) == a(own) + WD(S, Hq, Hkv, D, L, P) - 256
    # Uniform batches (every sequence has max_q_len queries) route nothing.
    assert W(S, S * 5, Hq, Hkv, D, 5, L, P) == 256 + a(S * 5 * Hq * parts * D * 4) + \
        a(S * 5 * Hq * parts * 8)
    # All one-query: the decode plan only (after the 256-byte header).
    assert W(S, S, Hq, Hkv, D, 1, L, -1) == 256
    # Automatic plan of the chunked-prefill mix (64 x 8 = 512 units, one wave
    # of decode CTAs or more): the prompt chunks unsplit (about 544 items),
    # the one-query sequences on 4096-token decode items, not stream-K.
    L2 = 4096 + 256
    assert pkv.prefill_partition_tokens(S, T, Hq, Hkv, D, 256, L2, 0) == 0
    assert W(S, T, Hq, Hkv, D, 256, L2, 0) == WD(S, Hq, Hkv, D, L2, 4096)
    assert WD(S, Hq, Hkv, D, L2, 4096) != WD(S, Hq, Hkv, D, L2, pkv.SCHEDULE_STREAMK)


def _prefill(**kw):
    args = dict(q=0x1000, q_dtype=BF16, qs=0x1800, k=0x2000, v=0x3000, kv_dtype=BF16, bt=0x4000,
                sl=0x5000, S=2, T=6, Hq=8, Hkv=2, D=128, B=16, N=10, maxb=4, maxq=4, maxl=64,
                scale=0.1, out=0x6000, out_dtype=F32, ws=0x7000, wsb=1 << 26, part=0, flags=0,
                ks=1.0, vs=1.0)
    args.update(kw)
    return pkv.lib().pkv_paged_attn_prefill(
        args["q"], args["q_dtype"], args["qs"], args["k"], args["v"], args["kv_dtype"],
        args["ks"], args["vs"],
        args["bt"], args["sl"], args["S"], args["T"], args["Hq"], args["Hkv"], args["D"],
        args["B"], args["N"], args["maxb"], args["maxq"], args["maxl"], args["scale"],
        args["out"], args["out_dtype"], args["ws"], args["wsb"], args["part"], args["flags"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=6, Hkv=4), INVALID),
    (dict(D=96), UNSUPPORTED),
    (dict(B=32), UNSUPPORTED),
    (dict(Hq=34, Hkv=2), UNSUPPORTED),
    (dict(q_dtype=F32), UNSUPPORTED),             # tensor-core paths: bf16 q
    (dict(kv_dtype=F32), UNSUPPORTED),
    (dict(kv_dtype=FP8, ws=0), WORKSPACE),        # fp8 / INT4 caches accepted (mma.sync)
    (dict(kv_dtype=pkv.FP8_E4M3, ws=0), WORKSPACE),
    (dict(kv_dtype=pkv.INT4, ws=0), WORKSPACE),
    (dict(kv_dtype=FP8, flags=0x2, ws=0), WORKSPACE),
    (dict(kv_dtype=FP8, flags=0x3), UNSUPPORTED),  # the tcgen05 kernel is bf16 only
    (dict(kv_dtype=pkv.INT4, ks=0.0), INVALID),
    (dict(kv_dtype=FP8, vs=float("nan")), INVALID),
    (dict(kv_dtype=BF16, ks=0.0, ws=0), WORKSPACE),  # scales ignored for bf16
    (dict(out_dtype=FP8), UNSUPPORTED),
    (dict(maxl=65), INVALID),
    (dict(T=-1), INVALID),
    (dict(maxq=-1), INVALID),
    (dict(ws=0), WORKSPACE),
    (dict(ws=0x7010), WORKSPACE),
    (dict(wsb=100, part=16), WORKSPACE),
    (dict(q=0), INVALID),
    (dict(qs=0), INVALID),
    (dict(qs=0x1802), INVALID),                   # misaligned q_start
    (dict(k=0x2008), INVALID),
    (dict(part=40), INVALID),
    (dict(flags=0x1), INVALID),                   # no CUDA-core variant
    (dict(flags=0x4), INVALID),
    (dict(flags=0x2, ws=0), WORKSPACE),           # mma.sync kernel accepted
    (dict(flags=0x3, ws=0), WORKSPACE),           # tcgen05 kernel accepted
    (dict(flags=0x103, ws=0), WORKSPACE),         # with the test hook
    (dict(flags=0x3, S=0), OK),
    (dict(scale=float("inf")), INVALID),
    (dict(S=0), OK),
    (dict(T=0), OK),
])
def test_prefill_argument_errors(kw, code):
    assert _prefill(**kw) == code


def _copy(**kw):
    args = dict(k=0x1000, v=0x2000, kv_dtype=BF16, Hkv=8, D=128, B=16, N=10, pairs=0x3000, n=4,
                status=None)
    args.update(kw)
    return pkv.lib().pkv_copy_blocks(args["k"], args["v"], args["kv_dtype"], args["Hkv"], args["D"],
                                     args["B"], args["N"], args["pairs"], args["n"], args["status"],
                                     None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=32), UNSUPPORTED),
    (dict(kv_dtype=9), UNSUPPORTED),
    (dict(Hkv=0), INVALID),
    (dict(N=0), INVALID),
    (dict(n=-1), INVALID),
    (dict(pairs=0), INVALID),
    (dict(pairs=0x3002), INVALID),
    (dict(k=0x1008), INVALID),
    (dict(n=0), OK),
])
def test_copy_blocks_argument_errors(kw, code):
    assert _copy(**kw) == code


def test_head_scaled_entries_reject_non_fp8_and_missing_scales():
    L = pkv.lib()
    args = [0x1000, BF16, 0x2000, 0x3000, BF16, 0x4000, 0x4100, 0x5000, 0x6000, 2, 8, 2, 128, 16,
            10, 4, 64, 0.1, 0x7000, F32, 0x8000, 1 << 26, 0, 0, None]
    assert L.pkv_paged_attn_decode_head_scaled(*args) == UNSUPPORTED
    args[4] = FP8
    args[5] = None
    assert L.pkv_paged_attn_decode_head_scaled(*args) == INVALID
    args[5] = 0x4002                                  # misaligned scales
    assert L.pkv_paged_attn_decode_head_scaled(*args) == INVALID
    r = [0x1000, 0x2000, BF16, 0x3000, 4, 2, 128, 16, 8, 0x4000, 0x5000, BF16, 0x6000, 0x6100,
         None, None]
    assert L.pkv_reshape_and_cache_head_scaled(*r) == UNSUPPORTED
    r[11] = FP8
    r[12] = None
    assert L.pkv_reshape_and_cache_head_scaled(*r) == INVALID


# ------------------------------------------------ several layers in one launch

def test_layers_plan_counts_every_layers_units():
    P, PL = pkv.partition_tokens, pkv.layers_partition_tokens
    for args in ((128, 64, 8, 128, 514, 0), (64, 32, 8, 128, 4097, 0), (8, 64, 8, 128, 32769, 0),
                 (4, 4, 4, 64, 65, -1), (4, 4, 4, 64, 65, 48), (128, 64, 8, 128, 14626, -2)):
        assert PL(1, *args) == P(*args)
    # 512 (sequence, KV head) units per layer: stream-K alone, whole units with two layers.
    assert P(64, 32, 8, 128, 4097, 0) == pkv.SCHEDULE_STREAMK
    assert PL(2, 64, 32, 8, 128, 4097, 0) == 4096
    assert PL(8, 4, 4, 4, 64, 65, 0) == pkv.SCHEDULE_STREAMK      # tiny: 128 units
    assert PL(0, 4, 4, 4, 64, 65, 0) == -1


def test_layers_workspace_size():
    W1, WL = pkv.workspace_size, pkv.layers_workspace_size

    def a(x):
        return (x + 255) // 256 * 256
    S, Hq, Hkv, D, L, P = 8, 64, 8, 128, 32769, 512
    parts = -(-L // P)
    for NL in (1, 3):
        rows = NL * S * Hq * parts
        assert WL(NL, S, Hq, Hkv, D, L, P) == 256 + a(NL * S * Hkv * 4) + a(rows * D * 4) + \
            a(rows * 8)
    assert WL(1, S, Hq, Hkv, D, L, P) == W1(S, Hq, Hkv, D, L, P)
    # Stream-K: partial slots per CTA, arrival counters per (layer, sequence, KV head).
    G = Hq // Hkv
    rows = 2 * 1024 * G
    assert WL(4, S, Hq, Hkv, D, L, -2) == 256 + a(4 * S * Hkv * 4) + a(rows * D * 4) + a(rows * 8)
    assert WL(3, 4, 4, 4, 64, 65, -1) == 256


def _layers(**kw):
    args = dict(table=0x1000, NL=2, q_dtype=BF16, new_dtype=BF16, kv_dtype=BF16, ks=1.0, vs=1.0,
                bt=0x4000, sl=0x5000, S=2, Hq=8, Hkv=2, D=128, B=16, N=10, maxb=4, maxl=64,
                scale=0.1, out_dtype=F32, ws=0x7000, wsb=1 << 26, part=0, flags=0)
    args.update(kw)
    return pkv.lib().pkv_paged_attn_decode_layers(
        args["table"], args["NL"], args["q_dtype"], args["new_dtype"], args["kv_dtype"],
        args["ks"], args["vs"], args["bt"], args["sl"], args["S"], args["Hq"], args["Hkv"],
        args["D"], args["B"], args["N"], args["maxb"], args["maxl"], args["scale"],
        args["out_dtype"], args["ws"], args["wsb"], args["part"], args["flags"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(table=0), INVALID),
    (dict(table=0x1004), INVALID),                # entries hold pointers: 8-byte aligned
    (dict(NL=0), INVALID),
    (dict(NL=-1), INVALID),
    (dict(new_dtype=FP8), UNSUPPORTED),
    (dict(kv_dtype=FP8, ks=0.0), INVALID),
    (dict(Hq=6, Hkv=4), INVALID),
    (dict(D=96), UNSUPPORTED),
    (dict(ws=0), WORKSPACE),
    (dict(wsb=100), WORKSPACE),
    (dict(bt=0x4002), INVALID),
    (dict(part=40), INVALID),
    (dict(S=0), OK),
])
def test_layers_argument_errors(kw, code):
    assert _layers(**kw) == code
