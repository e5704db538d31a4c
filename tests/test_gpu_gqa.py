"""GPU: grouped-query / multi-query decode attention (paged_decode_attention_gqa) through
the C ABI, against the float64 oracle's grouped-query attention.  Max-abs tolerance 2e-3
(fp16 and FP8-dequantised K/V, fp32 accumulation); FP8 pools are compared with the
oracle run on the values it quantises itself."""

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


def _setup(G, Hkv, d, B, dtype, seed, lens):
    nb = sum(-(-n // B) for n in lens) + 4
    w = W.Workload("gqa_small", seed, 1, Hkv, d, B, "f16", len(lens), lens, nb, 1 / math.sqrt(d),
                   num_q_heads=G * Hkv)
    cache = PagedKVCache(1, nb, B, Hkv, d, dtype)
    poison(cache)
    if dtype == "fp8":
        for t in cache.k_scale + cache.v_scale:
            t.fill_(0.011)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    return w, cache, alloc, seqs, ks, vs


def _oracle_values(dtype, ks, vs):
    if dtype != "fp8":
        return ks, vs
    s = np.float32(0.011)
    deq = lambda x: OF.decode(OF.quantize(x, s)) * float(s)
    return [deq(k) for k in ks], [deq(v) for v in vs]


@pytest.mark.parametrize("G", [2, 4, 8])
@pytest.mark.parametrize("dtype,d,B", [("f16", 128, 16), ("f16", 128, 8), ("f16", 128, 32), ("f16", 64, 8),
                                       ("fp8", 128, 16), ("fp8", 128, 8), ("fp8", 128, 32), ("fp8", 64, 32)])
def test_gqa_against_oracle(G, dtype, d, B):
    lens = [0, 1, 15, 16, 17, 100, 513, 1400, 2200]
    w, cache, alloc, seqs, ks, vs = _setup(G, 2, d, B, dtype, 80 + G, lens)
    # fp16 pools of head_dim 128 take the tensor-core path (tensor-map tiles)
    want_tc = abi.KV_FEATURE_TENSOR_MAPS if (dtype in ("f16", "fp8") and d == 128) else 0
    assert abi.kv_pool_features(cache.handle) == want_tc
    prefill(cache, alloc, seqs, ks, vs)
    bt, cl, _ = tables_for(alloc, seqs, max(-(-n // B) for n in lens))
    q = W.host_queries(w)
    kd, vd = _oracle_values(dtype, ks, vs)
    want = OA.decode_attention_gqa(q, kd, vd, w.scale)
    for P in (0, 64):
        out = cache.attention_gqa(0, torch.from_numpy(q).cuda(), bt, cl, max(lens), w.scale,
                                  partition_tokens=P).cpu().numpy()
        assert max_abs(out, want) <= tol_for("f16"), (P, max_abs(out, want))
        assert np.all(out[0] == 0.0)
    assert cache.device_error() == 0


@pytest.mark.parametrize("G", [2, 8])
@pytest.mark.parametrize("dtype", ["f16", "fp8"])
def test_gqa_odd_kv_head_count(G, dtype):
    """Three K/V heads: FP8 pools cannot pair heads per stage here (pairs need an even
    count), so this runs the one-head-per-stage tensor-core shape that even counts skip."""
    lens = [0, 1, 17, 513, 1400]
    w, cache, alloc, seqs, ks, vs = _setup(G, 3, 128, 16, dtype, 90 + G, lens)
    prefill(cache, alloc, seqs, ks, vs)
    bt, cl, _ = tables_for(alloc, seqs, max(-(-n // 16) for n in lens))
    q = W.host_queries(w)
    kd, vd = _oracle_values(dtype, ks, vs)
    want = OA.decode_attention_gqa(q, kd, vd, w.scale)
    for P in (0, 64):
        out = cache.attention_gqa(0, torch.from_numpy(q).cuda(), bt, cl, max(lens), w.scale,
                                  partition_tokens=P).cpu().numpy()
        assert max_abs(out, want) <= tol_for("f16"), (P, max_abs(out, want))
    assert cache.device_error() == 0


@pytest.mark.parametrize("G,dtype", [(4, "f16"), (8, "fp8"), (2, "f16")])
def test_gqa_fused_append_equals_append_then_attention(G, dtype):
    lens = [1, 33, 300, 1025]
    d, B, Hkv = 128, 16, 4
    w, c1, alloc, seqs, ks, vs = _setup(G, Hkv, d, B, dtype, 90 + G, lens)
    c2 = PagedKVCache(1, c1.num_blocks, B, Hkv, d, dtype)
    poison(c2)
    if dtype == "fp8":
        for t in c2.k_scale + c2.v_scale:
            t.fill_(0.011)
    slots_last = []
    for s, sid in enumerate(seqs):
        n = lens[s]
        slots, _ = alloc.append_slots(sid, n)
        for c in (c1, c2):
            if n > 1:
                c.append(0, torch.from_numpy(ks[s][:n - 1]).cuda(), torch.from_numpy(vs[s][:n - 1]).cuda(),
                         torch.tensor(slots[:n - 1], dtype=torch.int64, device="cuda"))
        slots_last.append(slots[-1])
    bt, cl, _ = tables_for(alloc, seqs, max(-(-n // B) for n in lens))
    q = torch.from_numpy(W.host_queries(w)).cuda()
    k_new = torch.from_numpy(np.stack([k[-1] for k in ks])).cuda()
    v_new = torch.from_numpy(np.stack([v[-1] for v in vs])).cuda()
    c1.append(0, k_new, v_new, torch.tensor(slots_last, dtype=torch.int64, device="cuda"))
    ref = c1.attention_gqa(0, q, bt, cl, max(lens), w.scale)
    got = c2.attention_gqa(0, q, bt, cl, max(lens), w.scale, k_new=k_new, v_new=v_new)
    assert torch.equal(c1.k[0].view(torch.uint8), c2.k[0].view(torch.uint8))
    assert torch.equal(c1.v[0].view(torch.uint8), c2.v[0].view(torch.uint8))
    assert torch.equal(ref, got)
    kd, vd = _oracle_values(dtype, ks, vs)
    assert max_abs(got.cpu().numpy(), OA.decode_attention_gqa(q.cpu().numpy(), kd, vd, w.scale)) <= tol_for("f16")
    for c in (c1, c2):
        assert c.device_error() == 0


def test_group_of_one_equals_mha_entry_and_bad_groups_are_refused():
    lens = [7, 300, 900]
    w, cache, alloc, seqs, ks, vs = _setup(1, 4, 128, 16, "f16", 95, lens)
    prefill(cache, alloc, seqs, ks, vs)
    bt, cl, _ = tables_for(alloc, seqs, max(-(-n // 16) for n in lens))
    q = torch.from_numpy(W.host_queries(w)).cuda()
    a = cache.attention(0, q, bt, cl, max(lens), w.scale)
    b = cache.attention_gqa(0, q, bt, cl, max(lens), w.scale)
    assert torch.equal(a, b)
    q3 = torch.zeros((3, 12, 128), dtype=torch.float16, device="cuda")        # G = 3
    with pytest.raises(abi.KvError):
        cache.attention_gqa(0, q3, bt, cl, max(lens), w.scale)
    q16 = torch.zeros((3, 64, 128), dtype=torch.float16, device="cuda")       # G = 16
    with pytest.raises(abi.KvError):
        cache.attention_gqa(0, q16, bt, cl, max(lens), w.scale)
    f32 = PagedKVCache(1, 8, 16, 2, 64, "f32")
    with pytest.raises(abi.KvError):                                          # fp32 pools: G = 1 only
        f32.attention_gqa(0, torch.zeros((1, 4, 64), device="cuda"),
                          torch.zeros((1, 1), dtype=torch.int32, device="cuda"),
                          torch.ones(1, dtype=torch.int32, device="cuda"), 1, 0.125)


def test_gqa70b_full_size_layer_sampled():
    """The LLaMA-2-70B-shaped layer (64 query / 8 KV heads, batch 32, context 4096) in the
    launch configuration the benchmark times, with the fused append; sampled heads."""
    w = W.gqa70b(num_layers=2)
    B, H, Hq, d = w.block_size, w.num_heads, w.q_heads, w.head_dim
    cache = PagedKVCache(w.num_layers, w.num_blocks, B, H, d, "f16")
    for l in range(w.num_layers):
        W.device_fill_normal(cache.k[l], w.seed * 1000 + 2 * l)
        W.device_fill_normal(cache.v[l], w.seed * 1000 + 2 * l + 1)
    nbs = [n // B for n in w.lens]
    tables = W.shuffled_tables(w, nbs)
    bt = torch.from_numpy(tables).cuda()
    cl = torch.tensor(w.lens, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(97)
    samples = [(int(rng.integers(w.batch)), int(rng.integers(Hq))) for _ in range(12)] + [(31, 63), (0, 0)]
    l = 1
    snap = {}
    for s, j in samples:
        idx = torch.tensor(tables[s, :nbs[s]], dtype=torch.int64, device="cuda")
        snap[(s, j)] = tuple(p.index_select(0, idx)[:, j // 8].reshape(-1, d).cpu().numpy()
                             for p in (cache.k[l], cache.v[l]))
    q = W.host_queries(w, 0, l)
    k_new, v_new = W.host_step_tokens(w, 0, l, "k"), W.host_step_tokens(w, 0, l, "v")
    # the benchmark's call: every option in one argument block, a workspace zero-filled
    # once, programmatic dependent launch, early tables and early K/V tiles
    ws = cache.zeroed_workspace(w.batch, max(w.lens), num_q_heads=Hq)
    out = cache.attention_ex(l, torch.from_numpy(q).cuda(), bt, cl, max(w.lens), w.scale,
                             k_new=torch.from_numpy(k_new).cuda(), v_new=torch.from_numpy(v_new).cuda(),
                             workspace=ws, flags=abi.KV_DECODE_WORKSPACE_ZEROED | abi.KV_DECODE_PDL |
                             abi.KV_DECODE_EARLY_TABLES | abi.KV_DECODE_EARLY_POOL)
    out = out.cpu().numpy()
    worst = 0.0
    for (s, j) in samples:
        K, V = (a.copy() for a in snap[(s, j)])
        n = w.lens[s]
        K[n - 1], V[n - 1] = k_new[s, j // 8], v_new[s, j // 8]
        worst = max(worst, max_abs(out[s, j], OA.decode_attention_one(q[s, j], K[:n], V[:n], w.scale)))
    assert worst <= tol_for("f16"), worst
    assert cache.device_error() == 0
