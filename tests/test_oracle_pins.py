"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test ties one part of the oracle to something independent: another
library's decoder or rounding, the dense attention of the "Inference
optimization" lesson (Step 2, scaled_dot_product_attention) computed by numpy,
closed forms (seq_len = 1, q = 0, constant V), invariants the pages state
(pages can sit anywhere in memory: "PagedAttention" section of the lesson, and
section 3 of "Continuous Batching e PagedAttention no vLLM"), and a
40-digit decimal brute force on tiny shapes.
"""
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_225_gb300 import workloads as W

F32, BF16, FP8, E4M3, INT4 = W.F32, W.BF16, W.FP8_E5M2, W.FP8_E4M3, W.INT4


# ----------------------------------------------------------------- decoders

def test_e5m2_decode_all_codes_match_float16_high_byte_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_values(codes, FP8)
    # e5m2 shares binary16's sign, 5-bit exponent and bias: a code is the high
    # byte of the binary16 with the same value.
    via_f16 = (codes.astype(np.uint16) << 8).view(np.float16).astype(np.float64)
    via_torch = torch.from_numpy(codes).view(torch.float8_e5m2).double().numpy()
    for ref in (via_f16, via_torch):
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7b] == 57344.0 and got[0x01] == 2.0 ** -16 and got[0x7c] == np.inf


def test_e4m3_decode_all_codes_match_closed_form_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_values(codes, E4M3)
    # From the format: sign | 4 exponent bits (bias 7) | 3 mantissa bits;
    # exponent 0 is subnormal, the all-ones code is NaN, no infinities.
    sign = np.where(codes >> 7, -1.0, 1.0)
    e = (codes >> 3) & 15
    m = (codes & 7).astype(np.float64)
    closed = sign * np.where(e == 0, m / 8 * 2.0 ** -6, (1 + m / 8) * 2.0 ** (e.astype(float) - 7))
    closed[(e == 15) & (m == 7)] = np.nan
    via_torch = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    for ref in (closed, via_torch):
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7e] == 448.0 and got[0x01] == 2.0 ** -9 and np.isnan(got[0x7f])
    assert np.isnan(got).sum() == 2


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=200_000, dtype=np.uint64).astype(np.uint16)
    got = oracle.decode_values(bits, BF16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f32_decode_is_identity():
    x = np.random.default_rng(2).standard_normal(1000).astype(np.float32)
    assert np.array_equal(oracle.decode_values(x, F32), x.astype(np.float64))


# ----------------------------------------------------------------- encoders

def _bf16_edge_values():
    rng = np.random.default_rng(3)
    vals = [rng.standard_normal(100_000) * 10.0 ** rng.integers(-40, 38, 100_000)]
    # Exact ties between neighbouring bf16 values, both parities.
    hi = rng.integers(0, 1 << 15, size=20_000, dtype=np.uint64).astype(np.uint32)
    vals.append(((hi << 16) | 0x8000).view(np.float32))
    vals.append(np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 3.4028235e38, 1e-45,
                          -1e-45, 1.1754944e-38], dtype=np.float32))
    return np.concatenate([v.astype(np.float32) for v in vals])


def test_bf16_encode_matches_torch_rne():
    x = _bf16_edge_values()
    got = oracle.encode_values(x, BF16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert nan.sum() > 0 and np.array_equal(got[~nan], ref[~nan])
    # NaN payloads are not part of the contract: any NaN maps to a bf16 NaN.
    assert np.all(np.isnan(oracle.decode_values(got[nan], BF16)))


def test_e5m2_encode_matches_torch_rne_in_range_and_saturates():
    rng = np.random.default_rng(4)
    finite = oracle.decode_values(np.arange(256, dtype=np.uint8), FP8)
    finite = np.unique(finite[np.isfinite(finite)])
    mids = ((finite[1:] + finite[:-1]) / 2).astype(np.float32)       # exact ties
    x = np.concatenate([
        (rng.standard_normal(200_000) * 2.0 ** rng.integers(-18, 16, 200_000)).astype(np.float32),
        mids, -mids, finite.astype(np.float32),
        np.array([57344.0, 60000.0, 61440.0, 65535.0, 1e9, np.inf, -np.inf, -70000.0],
                 dtype=np.float32)])
    got = oracle.encode_values(x, FP8)
    # Saturation to the largest finite value is the same as clamping first.
    ref = torch.from_numpy(np.clip(x, -57344.0, 57344.0)).to(torch.float8_e5m2)
    ref = ref.view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    assert got[-3] == 0x7b and got[-2] == 0xfb and got[-1] == 0xfb


def test_e4m3_encode_matches_torch_rne_in_range_and_saturates():
    rng = np.random.default_rng(40)
    finite = oracle.decode_values(np.arange(256, dtype=np.uint8), E4M3)
    finite = np.unique(finite[np.isfinite(finite)])
    mids = ((finite[1:] + finite[:-1]) / 2).astype(np.float32)       # exact ties
    x = np.concatenate([
        (rng.standard_normal(200_000) * 2.0 ** rng.integers(-12, 9, 200_000)).astype(np.float32),
        mids, -mids, finite.astype(np.float32),
        np.array([448.0, 460.0, 464.0, 470.0, 1e9, np.inf, -np.inf, -1000.0],
                 dtype=np.float32)])
    got = oracle.encode_values(x, E4M3)
    ref = torch.from_numpy(np.clip(x, -448.0, 448.0)).to(torch.float8_e4m3fn)
    assert np.array_equal(got, ref.view(torch.uint8).numpy())
    assert got[-3] == 0x7e and got[-2] == 0xfe and got[-1] == 0xfe


def test_e4m3_round_trip_and_scale():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode_values(codes, E4M3)
    finite = np.isfinite(vals)
    back = oracle.encode_values(vals[finite].astype(np.float32), E4M3)
    # +0 and -0 both come back; every finite code maps to itself.
    assert np.array_equal(back, codes[finite])
    x = np.random.default_rng(41).standard_normal(50_000).astype(np.float32) * 3
    for scale in (2.0, 0.37):
        got = oracle.encode_values(x, E4M3, scale=scale)
        xs = (x / np.float32(scale)).astype(np.float32)
        ref = torch.from_numpy(np.clip(xs, -448, 448)).to(torch.float8_e4m3fn)
        assert np.array_equal(got, ref.view(torch.uint8).numpy())


def test_e5m2_round_trip_of_every_finite_code():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode_values(codes, FP8)
    finite = np.isfinite(vals)
    back = oracle.encode_values(vals[finite].astype(np.float32), FP8)
    assert np.array_equal(back, codes[finite])
    assert oracle.encode_values(np.array([np.nan], np.float32), FP8)[0] == 0x7f


def test_e5m2_encode_divides_by_scale_in_float32():
    x = np.random.default_rng(5).standard_normal(50_000).astype(np.float32) * 3
    for scale in (2.0, 0.5, 3.0, 0.37):
        got = oracle.encode_values(x, FP8, scale=scale)
        xs = (x / np.float32(scale)).astype(np.float32)
        ref = torch.from_numpy(np.clip(xs, -57344, 57344)).to(torch.float8_e5m2)
        assert np.array_equal(got, ref.view(torch.uint8).numpy())


# ------------------------------------------------------------ attention pins

def _tiny_problem(kv_dtype, q_dtype, S=3, Hq=4, Hkv=2, D=16, B=16, lens=(1, 17, 40),
                  seed=0, identity=False, kv_scale=1.0):
    rng = np.random.default_rng(seed)
    nb = [(L + B - 1) // B for L in lens]
    N = sum(nb) + 3
    ids = np.arange(N, dtype=np.int32) if identity else rng.permutation(N).astype(np.int32)
    tables = np.full((S, max(nb) + 1), -1, dtype=np.int32)
    c = 0
    for s in range(S):
        tables[s, :nb[s]] = ids[c:c + nb[s]]
        c += nb[s]
    kf = rng.standard_normal((N, Hkv, D, B)).astype(np.float32)
    vf = rng.standard_normal((N, Hkv, D, B)).astype(np.float32)
    qf = rng.standard_normal((S, Hq, D)).astype(np.float32)
    k = W.round_to_storage(kf, kv_dtype)
    v = W.round_to_storage(vf, kv_dtype)
    q = W.round_to_storage(qf, q_dtype)
    return dict(q=q, q_dtype=q_dtype, k_cache=k, v_cache=v, kv_dtype=kv_dtype,
                block_tables=tables, seq_lens=np.array(lens, dtype=np.int32),
                scale=1.0 / np.sqrt(D), k_scale=kv_scale, v_scale=kv_scale)


def _dense_kv(p):
    """Contiguous per-sequence K/V [Hkv, L, D] by numpy indexing, in float64."""
    k = W.storage_to_float32(p["k_cache"], p["kv_dtype"]).astype(np.float64)
    v = W.storage_to_float32(p["v_cache"], p["kv_dtype"]).astype(np.float64)
    if p["kv_dtype"] in (FP8, E4M3, INT4):
        k, v = k * p["k_scale"], v * p["v_scale"]
    out = []
    B = k.shape[3]
    for s, L in enumerate(p["seq_lens"]):
        nb = (L + B - 1) // B
        blocks = p["block_tables"][s, :nb]
        ks = k[blocks].transpose(1, 0, 3, 2).reshape(k.shape[1], nb * B, k.shape[2])[:, :L]
        vs = v[blocks].transpose(1, 0, 3, 2).reshape(v.shape[1], nb * B, v.shape[2])[:, :L]
        out.append((ks, vs))
    return out


def _numpy_sdpa(q, keys, values, scale):
    """Dense single-query attention with max subtraction (lesson, Step 2)."""
    scores = (q @ keys.T) * scale
    e = np.exp(scores - scores.max())
    return (e / e.sum()) @ values


def _run(p, **kw):
    return oracle.paged_decode(p["q"], p["q_dtype"], p["k_cache"], p["v_cache"], p["kv_dtype"],
                               p["block_tables"], p["seq_lens"], p["scale"],
                               k_scale=p["k_scale"], v_scale=p["v_scale"], **kw)


@pytest.mark.parametrize("kv_dtype,q_dtype,kv_scale",
                         [(F32, F32, 1.0), (BF16, BF16, 1.0), (FP8, BF16, 1.0), (FP8, BF16, 0.5),
                          (E4M3, BF16, 1.0), (E4M3, BF16, 0.25)])
@pytest.mark.parametrize("identity", [True, False])
def test_paged_equals_dense_sdpa(kv_dtype, q_dtype, kv_scale, identity):
    p = _tiny_problem(kv_dtype, q_dtype, identity=identity, kv_scale=kv_scale)
    got = _run(p)
    qd = W.storage_to_float32(p["q"], q_dtype).astype(np.float64)
    G = qd.shape[1] // p["k_cache"].shape[1]
    for s, (ks, vs) in enumerate(_dense_kv(p)):
        for h in range(qd.shape[1]):
            ref = _numpy_sdpa(qd[s, h], ks[h // G], vs[h // G], p["scale"])
            np.testing.assert_allclose(got[s, h], ref, rtol=0, atol=1e-12)


def test_physical_permutation_is_bit_exact():
    p = _tiny_problem(BF16, BF16, lens=(5, 33, 48), seed=7)
    base = _run(p)
    N = p["k_cache"].shape[0]
    perm = np.random.default_rng(8).permutation(N)
    q = dict(p)
    q["k_cache"] = np.empty_like(p["k_cache"])
    q["v_cache"] = np.empty_like(p["v_cache"])
    q["k_cache"][perm] = p["k_cache"]
    q["v_cache"][perm] = p["v_cache"]
    t = p["block_tables"].copy()
    t[t >= 0] = perm[t[t >= 0]]
    q["block_tables"] = t
    assert np.array_equal(_run(q), base)


def test_seq_len_one_returns_that_value_row():
    p = _tiny_problem(F32, F32, lens=(1, 1, 1))
    got = _run(p)
    for s, (ks, vs) in enumerate(_dense_kv(p)):
        G = got.shape[1] // vs.shape[0]
        for h in range(got.shape[1]):
            assert np.array_equal(got[s, h], vs[h // G, 0])


def test_zero_query_gives_mean_of_values():
    p = _tiny_problem(BF16, BF16, lens=(7, 16, 45))
    p["q"] = np.zeros_like(p["q"])
    got = _run(p)
    for s, (ks, vs) in enumerate(_dense_kv(p)):
        G = got.shape[1] // vs.shape[0]
        for h in range(got.shape[1]):
            np.testing.assert_allclose(got[s, h], vs[h // G].mean(axis=0), rtol=0, atol=1e-13)


def test_constant_values_give_that_constant_and_hull_holds():
    p = _tiny_problem(F32, F32, lens=(3, 29, 64))
    got = _run(p)
    for s, (ks, vs) in enumerate(_dense_kv(p)):
        G = got.shape[1] // vs.shape[0]
        for h in range(got.shape[1]):
            lo, hi = vs[h // G].min(axis=0), vs[h // G].max(axis=0)
            assert np.all(got[s, h] >= lo - 1e-12) and np.all(got[s, h] <= hi + 1e-12)
    c = np.float32(0.8125)
    p["v_cache"] = np.full_like(p["v_cache"], c)
    np.testing.assert_allclose(_run(p), float(c), rtol=0, atol=1e-14)


def test_decimal_brute_force_tiny():
    getcontext().prec = 40
    p = _tiny_problem(BF16, BF16, S=2, Hq=2, Hkv=1, D=4, lens=(9, 23), seed=11)
    got = _run(p)
    k = W.storage_to_float32(p["k_cache"], BF16)
    v = W.storage_to_float32(p["v_cache"], BF16)
    q = W.storage_to_float32(p["q"], BF16)
    scale = Decimal(1) / Decimal(4).sqrt()
    B = 16
    for s in range(2):
        L = int(p["seq_lens"][s])
        for h in range(2):
            z = []
            for t in range(L):
                blk = int(p["block_tables"][s, t // B])
                acc = Decimal(0)
                for d in range(4):
                    acc += Decimal(float(q[s, h, d])) * Decimal(float(k[blk, 0, d, t % B]))
                z.append(acc * scale)
            m = max(z)
            w = [(zi - m).exp() for zi in z]
            tot = sum(w)
            for d in range(4):
                num = Decimal(0)
                for t in range(L):
                    blk = int(p["block_tables"][s, t // B])
                    num += w[t] * Decimal(float(v[blk, 0, d, t % B]))
                assert abs(float(num / tot) - got[s, h, d]) < 1e-14


@pytest.mark.parametrize("part", [16, 48, 100, 1])
def test_split_merge_equals_single_softmax(part):
    p = _tiny_problem(BF16, BF16, lens=(1, 70, 129), seed=12)
    np.testing.assert_allclose(_run(p, partition_tokens=part), _run(p), rtol=0, atol=1e-13)


def test_shared_prefix_equals_duplicated_blocks():
    p = _tiny_problem(BF16, BF16, lens=(40, 40, 40), seed=13)
    shared = p["block_tables"].copy()
    shared[1:, :2] = shared[0, :2]           # rows 1, 2 reuse row 0's first two blocks
    p["block_tables"] = shared
    a = _run(p)
    # Same thing with the shared blocks copied to fresh physical blocks.
    N = p["k_cache"].shape[0]
    extra = 4
    dup = dict(p)
    dup["k_cache"] = np.concatenate([p["k_cache"], p["k_cache"][np.r_[shared[0, :2], shared[0, :2]]]])
    dup["v_cache"] = np.concatenate([p["v_cache"], p["v_cache"][np.r_[shared[0, :2], shared[0, :2]]]])
    t = shared.copy()
    t[1, :2] = [N, N + 1]
    t[2, :2] = [N + 2, N + 3]
    dup["block_tables"] = t
    assert dup["k_cache"].shape[0] == N + extra
    assert np.array_equal(_run(dup), a)


def test_unowned_slots_and_table_padding_are_never_read():
    p = _tiny_problem(F32, F32, lens=(5, 17, 33), seed=14)
    base = _run(p)
    k, v = p["k_cache"].copy(), p["v_cache"].copy()
    owned = np.zeros(k.shape[0:1] + k.shape[3:], bool)
    for s, L in enumerate(p["seq_lens"]):
        for t in range(L):
            owned[p["block_tables"][s, t // 16], t % 16] = True
    k[np.broadcast_to(~owned[:, None, None, :], k.shape)] = np.nan
    v[np.broadcast_to(~owned[:, None, None, :], v.shape)] = np.inf
    p2 = dict(p, k_cache=k, v_cache=v)
    t = p["block_tables"].copy()
    t[t < 0] = 10 ** 6                      # padding entries past the used blocks
    for s, L in enumerate(p["seq_lens"]):
        t[s, (L + 15) // 16:] = 10 ** 6
    p2["block_tables"] = t
    assert np.array_equal(_run(p2), base)


def test_seq_len_zero_gives_zero_row():
    p = _tiny_problem(BF16, BF16, lens=(0, 5, 0))
    got = _run(p)
    assert np.all(got[0] == 0) and np.all(got[2] == 0) and np.all(np.isfinite(got[1]))


def test_decode_seqs_matches_full():
    p = _tiny_problem(BF16, BF16, lens=(5, 40, 33), seed=15)
    full = _run(p)
    part = oracle.paged_decode_seqs(p["q"], BF16, p["k_cache"], p["v_cache"], BF16,
                                    p["block_tables"], p["seq_lens"], p["scale"], seqs=[2, 0])
    assert np.array_equal(part, full[[2, 0]])


# ---------------------------------------------------------------- cache write

@pytest.mark.parametrize("in_dtype,kv_dtype,scale", [(F32, F32, 1.0), (F32, BF16, 1.0),
                                                     (BF16, BF16, 1.0), (BF16, FP8, 1.0),
                                                     (F32, FP8, 0.25), (BF16, E4M3, 1.0),
                                                     (F32, E4M3, 0.5)])
def test_reshape_and_cache_matches_numpy_scatter(in_dtype, kv_dtype, scale):
    rng = np.random.default_rng(21)
    N, Hkv, D, B, T = 9, 3, 16, 16, 7
    k_cache = W.round_to_storage(rng.standard_normal((N, Hkv, D, B)).astype(np.float32), kv_dtype)
    v_cache = W.round_to_storage(rng.standard_normal((N, Hkv, D, B)).astype(np.float32), kv_dtype)
    kin = W.round_to_storage(rng.standard_normal((T, Hkv, D)).astype(np.float32), in_dtype)
    vin = W.round_to_storage(rng.standard_normal((T, Hkv, D)).astype(np.float32), in_dtype)
    slots = rng.choice(N * B, size=T, replace=False).astype(np.int64)
    slots[3] = -1                                   # padding token: skipped
    kc, vc = k_cache.copy(), v_cache.copy()
    assert oracle.reshape_and_cache(kin, vin, in_dtype, slots, kc, vc, kv_dtype, scale, scale) == 0
    # Independent scatter: numpy fancy indexing + torch's casts.
    ek, ev = k_cache.copy(), v_cache.copy()
    for i, slot in enumerate(slots):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), B)
        for src, dst in ((kin, ek), (vin, ev)):
            x = W.storage_to_float32(src[i], in_dtype)
            if kv_dtype in (FP8, E4M3):
                x = (x / np.float32(scale)).astype(np.float32)
            dst[blk, :, :, off] = W.round_to_storage(x, kv_dtype)   # clamps fp8 to its range
    assert np.array_equal(kc.view(np.uint8), ek.view(np.uint8))
    assert np.array_equal(vc.view(np.uint8), ev.view(np.uint8))


def test_reshape_and_cache_reports_out_of_pool_slot():
    kc = np.zeros((2, 1, 4, 16), np.float32)
    vc = kc.copy()
    k = np.ones((1, 1, 4), np.float32)
    assert oracle.reshape_and_cache(k, k, F32, np.array([32]), kc, vc, F32) == 1
    assert not kc.any()


# ------------------------------------------------------------ byte accounting

def _golden(name):
    vals = {}
    with open(f"{__file__.rsplit('/', 1)[0]}/golden/{name}") as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if len(line) == 2:
                vals[line[0]] = float(line[1])
    return vals


def test_kv_bytes_per_token_matches_page_worked_example():
    from paged_kv_cache_225_gb300.metrics import kv_bytes_per_token
    g = _golden("kv_cache_size_llama3_70b.txt")
    per_tok = kv_bytes_per_token(int(g["num_layers"]), int(g["num_kv_heads"]),
                                 int(g["head_dim"]), int(g["bytes_per_elem"]))
    assert per_tok == g["per_token_bytes"] and per_tok / 1024 == g["per_token_kib"]
    assert round(per_tok * g["tokens_a"] / 1024 / 1024 / 1000, 2) == g["total_a_printed_gb"]
    assert per_tok * g["tokens_b"] / 2 ** 30 == g["total_b_printed_gib"]
    mha = kv_bytes_per_token(int(g["num_layers"]), int(g["num_q_heads"]), int(g["head_dim"]),
                             int(g["bytes_per_elem"]))
    assert mha / per_tok == g["gqa_reduction"]


# ------------------------------------------------------ per-head fp8 scales

@pytest.mark.parametrize("kv_dtype", [FP8, E4M3])
def test_per_head_scales_reduce_to_per_tensor_runs(kv_dtype):
    p = _tiny_problem(kv_dtype, BF16, S=3, Hq=6, Hkv=3, lens=(9, 40, 23), seed=30)
    ks, vs = np.array([0.5, 2.0, 0.25], np.float32), np.array([3.0, 0.125, 1.0], np.float32)
    got = _run(dict(p, k_scale=1.0, v_scale=1.0), k_head_scales=ks, v_head_scales=vs)
    G = 2
    for h in range(3):
        ref = _run(dict(p, k_scale=float(ks[h]), v_scale=float(vs[h])))
        assert np.array_equal(got[:, h * G:(h + 1) * G], ref[:, h * G:(h + 1) * G])
    # Equal factors are the per-tensor scale; the tensor scale multiplies in.
    same = _run(dict(p, k_scale=1.0, v_scale=1.0), k_head_scales=np.full(3, 0.5, np.float32),
                v_head_scales=np.full(3, 0.5, np.float32))
    assert np.array_equal(same, _run(dict(p, k_scale=0.5, v_scale=0.5)))
    two = _run(dict(p, k_scale=2.0, v_scale=1.0), k_head_scales=np.full(3, 0.25, np.float32))
    assert np.array_equal(two, _run(dict(p, k_scale=0.5, v_scale=1.0)))


def test_per_head_v_scale_scales_only_that_heads_rows():
    p = _tiny_problem(E4M3, BF16, S=2, Hq=4, Hkv=2, lens=(17, 33), seed=31)
    base = _run(p)
    got = _run(p, v_head_scales=np.array([1.0, 4.0], np.float32))
    np.testing.assert_array_equal(got[:, :2], base[:, :2])
    np.testing.assert_allclose(got[:, 2:], 4.0 * base[:, 2:], rtol=1e-14, atol=0)


@pytest.mark.parametrize("kv_dtype", [FP8, E4M3])
def test_reshape_with_per_head_scales_matches_numpy(kv_dtype):
    rng = np.random.default_rng(32)
    N, Hkv, D, B, T = 6, 3, 16, 16, 5
    kc = np.zeros((N, Hkv, D, B), np.uint8)
    vc = np.zeros_like(kc)
    kin = rng.standard_normal((T, Hkv, D)).astype(np.float32) * 4
    vin = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    slots = rng.choice(N * B, size=T, replace=False).astype(np.int64)
    ks, vs = np.array([0.5, 2.0, 0.1], np.float32), np.array([0.25, 1.0, 8.0], np.float32)
    assert oracle.reshape_and_cache(kin, vin, F32, slots, kc, vc, kv_dtype, 2.0, 1.0,
                                    k_head_scales=ks, v_head_scales=vs) == 0
    ek, ev = np.zeros_like(kc), np.zeros_like(vc)
    for i, slot in enumerate(slots):
        blk, off = divmod(int(slot), B)
        for h in range(Hkv):
            kd = np.float32(2.0) * ks[h]
            vd = np.float32(1.0) * vs[h]
            ek[blk, h, :, off] = W.round_to_storage((kin[i, h] / kd).astype(np.float32), kv_dtype)
            ev[blk, h, :, off] = W.round_to_storage((vin[i, h] / vd).astype(np.float32), kv_dtype)
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


# ------------------------------------------------------------------ INT4 KV

def test_int4_codes_decode_to_signed_nibbles():
    b = np.arange(256, dtype=np.uint8)
    got = oracle.decode_values(b, INT4)
    assert got.shape == (512,)
    lo, hi = got[0::2], got[1::2]
    assert np.array_equal(lo, [((x & 15) ^ 8) - 8 for x in range(256)])
    assert np.array_equal(hi, [((x >> 4) ^ 8) - 8 for x in range(256)])
    assert np.array_equal(got, W.storage_to_float32(b, INT4).astype(np.float64))


def test_int4_encode_rounds_half_even_and_clamps():
    x = np.array([0.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 6.49, 6.5, 7.5, 100.0, -7.5, -8.5,
                  -100.0, np.nan, 3.25], dtype=np.float32)
    got = oracle.encode_values(x, INT4)
    ref = np.array([0, 0, 2, 2, 0, -2, -2, 6, 6, 7, 7, -8, -8, -8, 0, 3], np.float64)
    assert np.array_equal(oracle.decode_values(got, INT4), ref)
    assert np.array_equal(got, W.round_to_storage(x, INT4))
    # The scale divides first (float32); every code round-trips.
    y = np.random.default_rng(50).standard_normal(4096).astype(np.float32) * 3
    for s in (0.5, 0.37):
        got = oracle.encode_values(y, INT4, scale=s)
        assert np.array_equal(got, W.round_to_storage((y / np.float32(s)).astype(np.float32),
                                                      INT4))
    codes = np.arange(256, dtype=np.uint8)
    assert np.array_equal(oracle.encode_values(oracle.decode_values(codes, INT4)
                                               .astype(np.float32), INT4), codes)


@pytest.mark.parametrize("identity", [True, False])
def test_int4_paged_equals_dense_sdpa(identity):
    p = _tiny_problem(INT4, BF16, identity=identity, kv_scale=0.5)
    got = _run(p)
    qd = W.storage_to_float32(p["q"], BF16).astype(np.float64)
    G = qd.shape[1] // p["k_cache"].shape[1]
    for s, (ks, vs) in enumerate(_dense_kv(p)):
        for h in range(qd.shape[1]):
            ref = _numpy_sdpa(qd[s, h], ks[h // G], vs[h // G], p["scale"])
            np.testing.assert_allclose(got[s, h], ref, rtol=0, atol=1e-12)


def test_int4_cache_write_matches_numpy_scatter():
    rng = np.random.default_rng(51)
    N, Hkv, D, B, T = 9, 3, 16, 16, 11
    kc = W.round_to_storage(rng.standard_normal((N, Hkv, D, B)).astype(np.float32) * 3, INT4)
    vc = W.round_to_storage(rng.standard_normal((N, Hkv, D, B)).astype(np.float32) * 3, INT4)
    kin = rng.standard_normal((T, Hkv, D)).astype(np.float32) * 2
    vin = rng.standard_normal((T, Hkv, D)).astype(np.float32) * 2
    slots = rng.choice(N * B, size=T, replace=False).astype(np.int64)
    k2, v2 = kc.copy(), vc.copy()
    assert oracle.reshape_and_cache(kin, vin, F32, slots, k2, v2, INT4, 0.5, 0.25) == 0
    ek = W.storage_to_float32(kc, INT4)
    ev = W.storage_to_float32(vc, INT4)
    for i, slot in enumerate(slots):
        blk, off = divmod(int(slot), B)
        ek[blk, :, :, off] = np.clip(np.rint(kin[i] / np.float32(0.5)), -8, 7)
        ev[blk, :, :, off] = np.clip(np.rint(vin[i] / np.float32(0.25)), -8, 7)
    assert np.array_equal(k2, W.round_to_storage(ek, INT4))
    assert np.array_equal(v2, W.round_to_storage(ev, INT4))
