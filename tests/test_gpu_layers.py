"""GPU parity of the several-layers decode launch (pkv_paged_attn_decode_layers).

Every layer of one launch is checked against the fp64 oracle run on that
layer alone (cache write of the new token, then attention over the grown
sequences), its cache writes bit for bit; with the item schedules each layer
also equals the single-layer fused launch bit for bit.  Layers without new
rows, a bad table entry (skipped and reported) and the separate merge kernel
are covered as well.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_225_gb300 as pkv
from paged_kv_cache_225_gb300 import workloads as W

from gpu_util import TOL, bits, max_abs, to_torch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
INVALID_ARG = 1


@functools.lru_cache(maxsize=2)
def _stack(name, num_layers):
    """Host layers and, per layer, the oracle's caches and output for the step."""
    ws = W.make_layers(name, num_layers)
    refs = []
    for w in ws:
        cfg = w.cfg
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        assert oracle.reshape_and_cache(w.new_k, w.new_v, cfg.q_dtype, w.slot_mapping, kc, vc,
                                        cfg.kv_dtype, cfg.kv_scale, cfg.kv_scale) == 0
        ref = oracle.paged_decode(w.q, cfg.q_dtype, kc, vc, cfg.kv_dtype, w.block_tables,
                                  w.seq_lens + 1, w.scale, k_scale=cfg.kv_scale,
                                  v_scale=cfg.kv_scale)
        refs.append((ref, kc, vc))
    return ws, refs


def _device_layers(ws, write=None):
    """Device tensors of every layer (write[l] False: no new rows in layer l)."""
    out = []
    for l, w in enumerate(ws):
        cfg = w.cfg
        lay = {"q": to_torch(w.q, cfg.q_dtype).to(DEV),
               "k_cache": to_torch(w.k_cache, cfg.kv_dtype).to(DEV),
               "v_cache": to_torch(w.v_cache, cfg.kv_dtype).to(DEV),
               "out": torch.full(w.q.shape, 7.0, dtype=torch.float32, device=DEV)}
        if write is None or write[l]:
            lay["new_k"] = to_torch(w.new_k, cfg.q_dtype).to(DEV)
            lay["new_v"] = to_torch(w.new_v, cfg.q_dtype).to(DEV)
        out.append(lay)
    return out


def _run(ws, layers, part, flags=0, table=None):
    w = ws[0]
    lens = torch.from_numpy((w.seq_lens + 1).astype(np.int32)).to(DEV)
    ks = w.cfg.kv_scale
    nbytes = pkv.layers_workspace_size(len(layers), w.cfg.num_seqs, w.cfg.num_q_heads,
                                       w.cfg.num_kv_heads, w.cfg.head_dim,
                                       int(w.seq_lens.max()) + 1, part)
    wsp = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    pkv.paged_attn_decode_layers(layers, torch.from_numpy(w.block_tables).to(DEV), lens, w.scale,
                                 k_scale=ks, v_scale=ks, max_seq_len=int(w.seq_lens.max()) + 1,
                                 partition_tokens=part, workspace=wsp, table=table, flags=flags)
    torch.cuda.synchronize()
    return pkv.read_status(wsp)


@pytest.mark.parametrize("name,num_layers", [("tiny_fp32", 4), ("fp8_chat", 3),
                                             ("llama3_8b", 2)])
@pytest.mark.parametrize("part", [0, -1, -2, 64])
def test_every_layer_matches_the_oracle(name, num_layers, part):
    ws, refs = _stack(name, num_layers)
    layers = _device_layers(ws)
    assert _run(ws, layers, part) == 0
    tol = TOL[ws[0].cfg.kv_dtype]
    for lay, (ref, kc, vc) in zip(layers, refs):
        assert np.array_equal(bits(lay["k_cache"]), kc.view(np.uint8).reshape(-1))
        assert np.array_equal(bits(lay["v_cache"]), vc.view(np.uint8).reshape(-1))
        assert max_abs(lay["out"].double().cpu().numpy(), ref) <= tol


@pytest.mark.parametrize("name,num_layers", [("tiny_fp32", 3), ("fp8_chat", 2)])
@pytest.mark.parametrize("part", [-1, 64, 0])
def test_item_schedules_equal_single_layer_launches_bitwise(name, num_layers, part):
    ws, _ = _stack(name, num_layers)
    cfg = ws[0].cfg
    max_len = int(ws[0].seq_lens.max()) + 1
    plan = pkv.layers_partition_tokens(num_layers, cfg.num_seqs, cfg.num_q_heads,
                                       cfg.num_kv_heads, cfg.head_dim, max_len, part)
    if plan == pkv.SCHEDULE_STREAMK:
        pytest.skip("stream-K ranges depend on the launch's total work")
    layers = _device_layers(ws)
    assert _run(ws, layers, part) == 0
    single = _device_layers(ws)
    lens = torch.from_numpy((ws[0].seq_lens + 1).astype(np.int32)).to(DEV)
    tables = torch.from_numpy(ws[0].block_tables).to(DEV)
    for lay in single:
        pkv.paged_attn_decode_append(lay["q"], lay["new_k"], lay["new_v"], lay["k_cache"],
                                     lay["v_cache"], tables, lens, ws[0].scale, lay["out"],
                                     k_scale=cfg.kv_scale, v_scale=cfg.kv_scale,
                                     max_seq_len=max_len, partition_tokens=plan if plan else -1)
    torch.cuda.synchronize()
    assert pkv.read_status(device=DEV) == 0
    for a, b in zip(layers, single):
        assert torch.equal(a["out"], b["out"])
        assert torch.equal(a["k_cache"].view(torch.uint8), b["k_cache"].view(torch.uint8))


@pytest.mark.parametrize("part", [-1, -2, 64])
def test_layer_without_new_rows_and_a_bad_entry(part):
    """Layer 0 writes its new token; layer 1 has no new rows and attends its
    cache as it is over the same lengths (its cache already holds the token,
    written beforehand); layer 2's entry holds a misaligned q: it is skipped
    (out untouched, nothing written) and reported."""
    ws, refs = _stack("tiny_fp32", 3)
    layers = _device_layers(ws, write=[True, False, True])
    layers[1]["k_cache"] = to_torch(refs[1][1], W.F32).to(DEV)
    layers[1]["v_cache"] = to_torch(refs[1][2], W.F32).to(DEV)
    table = pkv.layer_table(layers)
    table[2, 0] += 4                                    # q of layer 2: not 16-byte aligned
    k2 = layers[2]["k_cache"].clone()
    assert _run(ws, layers, part, table=table) == INVALID_ARG
    assert max_abs(layers[0]["out"].double().cpu().numpy(), refs[0][0]) <= TOL[W.F32]
    assert max_abs(layers[1]["out"].double().cpu().numpy(), refs[1][0]) <= TOL[W.F32]
    assert np.array_equal(bits(layers[1]["k_cache"]), refs[1][1].view(np.uint8).reshape(-1))
    assert torch.all(layers[2]["out"] == 7.0)
    assert np.array_equal(bits(layers[2]["k_cache"]), bits(k2))   # NaN-filled slots: bytes


def test_separate_merge_kernel_equals_in_kernel_merge():
    ws, _ = _stack("fp8_chat", 2)
    a = _device_layers(ws)
    b = _device_layers(ws)
    assert _run(ws, a, 64) == 0
    assert _run(ws, b, 64, flags=pkv.FLAG_SEPARATE_MERGE) == 0
    for x, y in zip(a, b):
        assert torch.equal(x["out"], y["out"])
