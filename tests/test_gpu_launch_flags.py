"""GPU: the launch flags of paged_decode_attention_ex through the C ABI.

* KV_DECODE_WORKSPACE_ZEROED: the call trusts that the workspace's counters are zero and
  does not clear them.  Every launch leaves its work, exit and arrival counters zero when
  it completes, so a zero-filled workspace stays valid over any number of decode calls.
  Checked by reading the counter region back after each call (it must be all zero) and
  by comparing every call's output with the float64 oracle, over contexts split into one-
  and two-level merges (MHA on the CUDA cores, grouped queries on the tensor cores, FP8).
* KV_DECODE_PDL: programmatic dependent launch.  Back-to-back fused decode steps on one
  stream, eagerly and replayed from a CUDA graph, each step's output against the oracle.
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

ZEROED, PDL, EARLY = abi.KV_DECODE_WORKSPACE_ZEROED, abi.KV_DECODE_PDL, abi.KV_DECODE_EARLY_TABLES
EARLY_POOL = abi.KV_DECODE_EARLY_POOL
COUNTER_BYTES = 512          # work and exit counters at the start of every workspace
MERGE_FAN = 16               # partitions folded per group in a two-level merge


def _counter_bytes(batch: int, heads: int, max_context: int, P: int) -> int:
    """Bytes of the workspace's counter region for an explicit partition size P: the
    work/exit counters, then per (sequence, K/V head) arrival counters and, for contexts
    split into more than 16 partitions, the per-group arrival counters (each 256-aligned)."""
    parts = -(-max_context // P)
    if parts <= 1:
        return COUNTER_BYTES
    units = batch * heads
    groups = -(-parts // MERGE_FAN) if parts > MERGE_FAN else 0
    a256 = lambda n: (n + 255) & ~255
    return COUNTER_BYTES + a256(units * 4) + a256(units * groups * 4)


def _setup(dtype, G, seed):
    B, Hkv, d = 16, 2, 128
    lens = [0, 1, 15 * 32, 16 * 32 + 1, 33 * 32 - 5, 257 * 32, 9000]
    nb = sum(-(-n // B) for n in lens) + 4
    w = W.Workload("launch_flags", seed, 1, Hkv, d, B, "f16", len(lens), lens, nb, 1 / math.sqrt(d),
                   num_q_heads=G * Hkv)
    cache = PagedKVCache(1, nb, B, Hkv, d, dtype)
    poison(cache)
    sc = np.float32(0.01)
    if dtype == "fp8":
        for t in cache.k_scale + cache.v_scale:
            t.fill_(float(sc))
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    prefill(cache, alloc, seqs, ks, vs)
    if dtype == "fp8":
        ks = [OF.decode(OF.quantize(k, sc)) * float(sc) for k in ks]
        vs = [OF.decode(OF.quantize(v, sc)) * float(sc) for v in vs]
    bt, cl, _ = tables_for(alloc, seqs, max(-(-n // B) for n in lens))
    return w, cache, alloc, ks, vs, bt, cl


@pytest.mark.parametrize("dtype,G", [("f16", 1), ("f16", 8), ("fp8", 1), ("fp8", 4)])
@pytest.mark.parametrize("P", [32, 256])
def test_zeroed_workspace_over_repeated_calls(dtype, G, P):
    w, cache, alloc, ks, vs, bt, cl = _setup(dtype, G, 300 + G)
    max_ctx = max(w.lens)
    ws = cache.zeroed_workspace(w.batch, max_ctx, P, num_q_heads=w.q_heads)
    nbytes = _counter_bytes(w.batch, w.num_heads, max_ctx, P)
    assert ws.numel() >= nbytes
    oracle = OA.decode_attention_gqa if G > 1 else OA.decode_attention
    for call in range(3):
        q = W.host_queries(w, call)
        out = cache.attention_ex(0, torch.from_numpy(q).cuda(), bt, cl, max_ctx, w.scale,
                                 partition_tokens=P, workspace=ws, flags=ZEROED)
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        err = max_abs(got, oracle(q, ks, vs, w.scale))
        assert err <= tol_for("f16"), (call, err)
        # the launch left every counter zero for the next call
        assert int(torch.count_nonzero(ws[:nbytes])) == 0, call
    # the same call with the clearing copy gives the same output
    ref = cache.attention_ex(0, torch.from_numpy(q).cuda(), bt, cl, max_ctx, w.scale, partition_tokens=P)
    assert max_abs(ref.cpu().numpy(), got) <= tol_for("f16")
    assert cache.device_error() == 0
    cache.close()
    alloc.close()


def _decode_loop_case(G):
    """8 sequences of the LLaMA-7B length mix, 2 K/V heads, 12 fused decode steps."""
    w0 = W.llama7b()
    B, Hkv, d, steps = 16, 2, 128, 12
    init = [n - 1 for n in w0.lens]
    total = [n + steps for n in init]
    nb = sum(-(-n // B) for n in total) + 8
    w = W.Workload("pdl_loop", 410 + G, 1, Hkv, d, B, "f16", len(init), total, nb, 1 / math.sqrt(d),
                   num_q_heads=G * Hkv)
    cache = PagedKVCache(1, nb, B, Hkv, d, "f16")
    poison(cache)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in init]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(total)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(total)]
    prefill(cache, alloc, seqs, [k[:n] for k, n in zip(ks, init)], [v[:n] for v, n in zip(vs, init)])
    max_blocks = -(-max(total) // B)
    tabs, lens, qs, kn, vn = [], [], [], [], []
    for step in range(steps):
        pos = [n + step for n in init]
        for sid in seqs:
            alloc.append_slots(sid, 1)
        bt, cl, got = tables_for(alloc, seqs, max_blocks)
        assert got == [p + 1 for p in pos]
        tabs.append(bt)
        lens.append(cl)
        qs.append(torch.from_numpy(W.host_queries(w, step)).cuda())
        kn.append(torch.from_numpy(np.stack([k[p] for k, p in zip(ks, pos)])).cuda())
        vn.append(torch.from_numpy(np.stack([v[p] for v, p in zip(vs, pos)])).cuda())
    want = []
    for step in range(steps):
        pos = [n + step for n in init]
        q = qs[step].cpu().numpy()
        f = OA.decode_attention_gqa if G > 1 else OA.decode_attention
        want.append(f(q, [k[:p + 1] for k, p in zip(ks, pos)], [v[:p + 1] for v, p in zip(vs, pos)], w.scale))
    return w, cache, alloc, max(total), tabs, lens, qs, kn, vn, want


@pytest.mark.parametrize("G", [1, 8])
@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("early", [0, EARLY, EARLY | EARLY_POOL])
def test_pdl_back_to_back_fused_steps(G, graph, early):
    """early: KV_DECODE_EARLY_TABLES as well (every step's tables and lengths are written
    before the loop, so each launch may read them before the previous launch ends), and
    KV_DECODE_EARLY_POOL (each launch fetches its first K/V tiles while the previous step,
    which appended row context_len - 2 of every sequence of this same layer, finishes)."""
    w, cache, alloc, max_ctx, tabs, lens, qs, kn, vn, want = _decode_loop_case(G)
    steps = len(qs)
    P = 128     # several partitions per sequence: merges run in every launch
    ws = cache.zeroed_workspace(w.batch, max_ctx, P, num_q_heads=w.q_heads)
    outs = [torch.empty((w.batch, w.q_heads, w.head_dim), dtype=torch.float32, device="cuda")
            for _ in range(steps)]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())

    def loop():
        for i in range(steps):
            cache.attention_ex(0, qs[i], tabs[i], lens[i], max_ctx, w.scale, k_new=kn[i], v_new=vn[i],
                               out=outs[i], partition_tokens=P, workspace=ws, stream=stream,
                               flags=ZEROED | PDL | early)

    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            loop()
        with torch.cuda.stream(stream):
            g.replay()
    else:
        with torch.cuda.stream(stream):
            loop()
    stream.synchronize()
    for i in range(steps):
        err = max_abs(outs[i].cpu().numpy(), want[i])
        assert err <= tol_for("f16"), (i, err)
    assert int(torch.count_nonzero(ws[:_counter_bytes(w.batch, w.num_heads, max_ctx, P)])) == 0
    assert cache.device_error() == 0
    cache.close()
    alloc.close()


def test_unknown_flags_are_refused():
    w, cache, alloc, ks, vs, bt, cl = _setup("f16", 1, 320)
    q = torch.from_numpy(W.host_queries(w)).cuda()
    with pytest.raises(abi.KvError):
        cache.attention_ex(0, q, bt, cl, max(w.lens), w.scale, flags=32)
    cache.close()
    alloc.close()


def test_flags_over_several_launches_with_head_pairs_and_fp8():
    """2100 sequences (three launches of at most 1024), FP8 pool with B 16 and 2 heads
    (head-pair items), fused append, 32-token partitions (a few long sequences merge in
    two levels), KV_DECODE_WORKSPACE_ZEROED | KV_DECODE_PDL, three calls in a row on one
    zeroed workspace (the later ones with early tables, then early K/V tiles too): every
    launch's counters start and end at zero."""
    B, H, d = 16, 2, 128
    rng = np.random.default_rng(21)
    lens = rng.integers(0, 70, 2100).tolist()
    lens[5], lens[1024 + 5], lens[2048 + 5] = 900, 1000, 700
    nb = sum(-(-n // B) for n in lens) + 1
    w = W.Workload("bigbatch_fp8", 92, 1, H, d, B, "f16", len(lens), lens, nb, 1 / math.sqrt(d))
    cache = PagedKVCache(1, nb, B, H, d, "fp8")
    poison(cache)
    sc = np.float32(0.01)
    for t in cache.k_scale + cache.v_scale:
        t.fill_(float(sc))
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    # everything but each sequence's newest token is prefilled; the call appends it
    prefill(cache, alloc, seqs, [k[:-1] if len(k) else k for k in ks], [v[:-1] if len(v) else v for v in vs])
    for s, sid in enumerate(seqs):
        if lens[s]:
            alloc.append_slots(sid, 1)
    bt, cl, got = tables_for(alloc, seqs, max(1, max(-(-n // B) for n in lens)))
    assert got == lens
    kn = torch.from_numpy(np.stack([k[-1] if len(k) else np.zeros((H, d), np.float16) for k in ks])).cuda()
    vn = torch.from_numpy(np.stack([v[-1] if len(v) else np.zeros((H, d), np.float16) for v in vs])).cuda()
    ksd = [OF.decode(OF.quantize(k, sc)) * float(sc) for k in ks]
    vsd = [OF.decode(OF.quantize(v, sc)) * float(sc) for v in vs]
    P = 32
    ws = cache.zeroed_workspace(w.batch, max(lens), P)
    for call, extra in enumerate((0, EARLY, EARLY | EARLY_POOL)):
        q = W.host_queries(w, call)
        # later calls append the same token again into the same slot (same bytes)
        out = cache.attention_ex(0, torch.from_numpy(q).cuda(), bt, cl, max(lens), w.scale, k_new=kn, v_new=vn,
                                 partition_tokens=P, workspace=ws, flags=ZEROED | PDL | extra)
        err = max_abs(out.cpu().numpy(), OA.decode_attention(q, ksd, vsd, w.scale))
        assert err <= tol_for("f16"), (call, err)
    assert cache.device_error() == 0
    cache.close()
    alloc.close()
