"""GPU: KV_DECODE_OUT_F16, the attention result stored as float16 (the output of the
cached decode step in "大模型推理加速——KV Cache篇" §3.1 is cast back to the query's type).

The kernels merge in float32 and round only the final store, so a float16 call must
return exactly the float32 call's result rounded to nearest even (torch's float32 ->
float16 conversion), on every path that writes the output: a single-partition item on
the CUDA cores (one head, head pairs, head quads), the tensor-core grouped-query
consumer, and the one- and two-level split-context merges.  Each float16 result is also
held to the float64 oracle: the float32 tolerance plus half a float16 ulp of the value.
"""

import math

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import max_abs, poison, prefill, tables_for, tol_for
from oracle import attention as OA
from oracle import fp8 as OF
from paged_kv_cache_169_gb300 import abi
from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

pytestmark = pytest.mark.gpu

FP8_SCALE = np.float32(0.011)


def _cache(dtype, L, nb, B, H, d):
    cache = PagedKVCache(L, nb, B, H, d, dtype)
    poison(cache)
    if dtype == "fp8":
        for t in cache.k_scale + cache.v_scale:
            t.fill_(float(FP8_SCALE))
    return cache


def _dequant(dtype, xs):
    if dtype != "fp8":
        return xs
    return [OF.decode(OF.quantize(x, FP8_SCALE)) * float(FP8_SCALE) for x in xs]


def _held_to_oracle(out16, want, dtype):
    """float16 result against the float64 oracle: the float32 path's tolerance plus the
    rounding of the final store (at most half an ulp: 2^-11 of the value)."""
    got = out16.float().cpu().numpy().astype(np.float64)
    bound = tol_for(dtype) + np.abs(want) * 2.0 ** -11
    assert np.all(np.abs(got - want) <= bound), float(np.max(np.abs(got - want) - bound))


@pytest.mark.parametrize("dtype,d,B,H,G", [
    ("f16", 128, 16, 2, 1),      # one head per item, CUDA cores
    ("f16", 128, 8, 2, 1),       # head pairs
    ("fp8", 128, 16, 2, 1),      # FP8 head pairs
    ("fp8", 128, 8, 4, 1),       # FP8 head quads
    ("f16", 64, 16, 2, 1),
    ("f32", 64, 16, 2, 1),
    ("f16", 128, 16, 2, 8),      # grouped queries on the tensor cores
    ("fp8", 128, 16, 2, 4),      # FP8 grouped queries on the tensor cores
    ("f16", 64, 32, 2, 4),       # grouped queries on the CUDA cores
])
def test_f16_output_is_the_f32_result_rounded(dtype, d, B, H, G):
    lens = [0, 1, 17, 300, 1025, 3000]
    nb = sum(-(-n // B) for n in lens) + 4
    w = W.Workload("out_f16", 130 + d + B + G, 1, H, d, B, "f16", len(lens), lens, nb, 1 / math.sqrt(d),
                   num_q_heads=G * H)
    cache = _cache(dtype, 1, nb, B, H, d)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    if dtype == "f32":
        ks = [k.astype(np.float32) for k in ks]
        vs = [v.astype(np.float32) for v in vs]
    prefill(cache, alloc, seqs, ks, vs)
    bt, cl, _ = tables_for(alloc, seqs, max(-(-n // B) for n in lens))
    qh = W.host_queries(w)
    if dtype == "f32":
        qh = qh.astype(np.float32)
    q = torch.from_numpy(qh).cuda()
    kd, vd = _dequant(dtype, ks), _dequant(dtype, vs)
    want = OA.decode_attention_gqa(qh, kd, vd, w.scale)
    for P in (0, 32, 256):           # 32: contexts of 3000 merge in two levels
        o32 = cache.attention_ex(0, q, bt, cl, max(lens), w.scale, partition_tokens=P)
        o16 = cache.attention_ex(0, q, bt, cl, max(lens), w.scale, partition_tokens=P,
                                 out_dtype=torch.float16)
        assert o16.dtype == torch.float16
        assert torch.equal(o16, o32.half()), (P, float((o16.float() - o32.half().float()).abs().max()))
        assert torch.all(o16[0] == 0)
        _held_to_oracle(o16, want, dtype)
    assert cache.device_error() == 0
    cache.close()
    alloc.close()


@pytest.mark.parametrize("dtype,B,H,G", [("fp8", 8, 4, 1), ("f16", 16, 2, 8), ("f16", 16, 4, 1)])
def test_f16_output_with_fused_append_window_and_launch_flags(dtype, B, H, G):
    """The benchmark's call (fused append, zeroed workspace, PDL, early tables and K/V
    tiles) with a sliding window, float16 result: equal to the float32 call's, rounded,
    and to the oracle over the window."""
    d, window = 128, 256
    lens = [1, 9, 255, 257, 700, 2049]
    nb = sum(-(-n // B) for n in lens) + 4
    w = W.Workload("out_f16_fused", 150 + B + G, 1, H, d, B, "f16", len(lens), lens, nb, 1 / math.sqrt(d),
                   num_q_heads=G * H)
    cache = _cache(dtype, 1, nb, B, H, d)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    prefill(cache, alloc, seqs, [k[:-1] for k in ks], [v[:-1] for v in vs])
    for sid in seqs:                 # the newest token's slot, written by the fused call
        alloc.append_slots(sid, 1)
    bt, cl, _ = tables_for(alloc, seqs, max(-(-n // B) for n in lens))
    qh = W.host_queries(w)
    q = torch.from_numpy(qh).cuda()
    k_new = torch.from_numpy(np.stack([k[-1] for k in ks])).cuda()
    v_new = torch.from_numpy(np.stack([v[-1] for v in vs])).cuda()
    flags = (abi.KV_DECODE_WORKSPACE_ZEROED | abi.KV_DECODE_PDL | abi.KV_DECODE_EARLY_TABLES |
             abi.KV_DECODE_EARLY_POOL)
    ws = cache.zeroed_workspace(len(lens), max(lens), num_q_heads=G * H, window=window)
    kw = dict(window=window, k_new=k_new, v_new=v_new, workspace=ws, flags=flags)
    o32 = cache.attention_ex(0, q, bt, cl, max(lens), w.scale, **kw)
    o16 = cache.attention_ex(0, q, bt, cl, max(lens), w.scale, out_dtype=torch.float16, **kw)
    assert torch.equal(o16, o32.half())
    kd, vd = _dequant(dtype, ks), _dequant(dtype, vs)
    want = OA.decode_attention_gqa(qh, [k[-window:] for k in kd], [v[-window:] for v in vd], w.scale)
    _held_to_oracle(o16, want, dtype)
    assert cache.device_error() == 0
    cache.close()
    alloc.close()


def test_f16_output_flag_needs_a_float16_buffer():
    """The binding refuses KV_DECODE_OUT_F16 on a float32 tensor and any other dtype."""
    B, H, d = 16, 2, 64
    cache = _cache("f16", 1, 8, B, H, d)
    q = torch.zeros((1, H, d), dtype=torch.float16, device="cuda")
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    cl = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        cache.attention_ex(0, q, bt, cl, 1, 0.125, flags=abi.KV_DECODE_OUT_F16)
    with pytest.raises(ValueError):
        cache.attention_ex(0, q, bt, cl, 1, 0.125, out_dtype=torch.bfloat16)
    o16 = cache.attention_ex(0, q, bt, cl, 1, 0.125, out_dtype=torch.float16)
    assert o16.shape == (1, H, d) and cache.device_error() == 0
    cache.close()
