"""GPU: paged_decode_attention_append (append of each sequence's newest token fused into
the attention launch) through the C ABI.

* Against the unfused path (kv_append, then paged_decode_attention) on identical pools:
  the pool bytes and the outputs must be bit-identical (the same bytes reach the same
  arithmetic).
* Against the float64 oracle over the 64 decode steps of the LLaMA-7B layer and the
  128 steps of parallel sampling with copy-on-write (max abs 2e-3, fp16 K/V).
"""

import math

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import max_abs, poison, prefill, tables_for, tol_for
from oracle import attention as OA
from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

pytestmark = pytest.mark.gpu


def _bits(t):
    a = t.cpu().numpy()
    return a.view({4: np.uint32, 2: np.uint16, 1: np.uint8}[a.itemsize])


@pytest.mark.parametrize("dtype,B,d,P,H", [("f16", 16, 128, 0, 6), ("f16", 8, 128, 64, 6), ("f16", 32, 64, 0, 6),
                                           ("f32", 16, 64, 32, 6), ("fp8", 16, 128, 0, 6), ("fp8", 8, 64, 64, 6),
                                           ("fp8", 8, 128, 0, 8), ("fp8", 8, 128, 32, 6)])
def test_fused_equals_append_then_attention(dtype, B, d, P, H):
    """Head groups: FP8 with B 8 and 8 heads takes four heads per work item, with 6 heads
    two; FP8 with B 16 and fp16 with B 8 two."""
    rng = np.random.default_rng(61)
    lens = [0, 1, B, B + 1, 31, 32, 33, 300, 777, 1500]
    nb = sum(-(-n // B) for n in lens) + 5
    w = W.Workload("fused", 61, 1, H, d, B, "f32" if dtype == "f32" else "f16", len(lens), lens, nb,
                   1 / math.sqrt(d))
    caches = [PagedKVCache(1, nb, B, H, d, dtype) for _ in range(2)]
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    # prefill all but the newest token, identically in both pools (FP8: random block scales)
    sc = rng.uniform(0.004, 0.02, (2, (nb + 3) // 4 * 4)).astype(np.float32)
    for c in caches:
        poison(c)
        if dtype == "fp8":
            c.k_scale[0].copy_(torch.from_numpy(sc[0]))
            c.v_scale[0].copy_(torch.from_numpy(sc[1]))
    for s, sid in enumerate(seqs):
        n = lens[s]
        if n == 0:
            continue
        slots, _ = alloc.append_slots(sid, n)
        if n > 1:
            for c in caches:
                c.append(0, torch.from_numpy(ks[s][:n - 1]).cuda(), torch.from_numpy(vs[s][:n - 1]).cuda(),
                         torch.tensor(slots[:n - 1], dtype=torch.int64, device="cuda"))
    max_blocks = max(-(-n // B) for n in lens)
    bt, cl, _ = tables_for(alloc, seqs, max_blocks)
    q = torch.from_numpy(W.host_queries(w)).cuda()
    tdt = torch.float32 if dtype == "f32" else torch.float16
    k_new = torch.zeros((len(lens), H, d), dtype=tdt)
    v_new = torch.zeros((len(lens), H, d), dtype=tdt)
    last_slots = []
    for s, n in enumerate(lens):
        if n:
            k_new[s] = torch.from_numpy(ks[s][n - 1])
            v_new[s] = torch.from_numpy(vs[s][n - 1])
            last_slots.append(alloc.table(seqs[s])[(n - 1) // B] * B + (n - 1) % B)
        else:
            last_slots.append(-1)
    k_new, v_new = k_new.cuda(), v_new.cuda()
    # unfused: append, then attend
    caches[0].append(0, k_new, v_new, torch.tensor(last_slots, dtype=torch.int64, device="cuda"))
    ref = caches[0].attention(0, q, bt, cl, max(lens), w.scale, partition_tokens=P)
    # fused
    got = caches[1].attention_append(0, q, k_new, v_new, bt, cl, max(lens), w.scale, partition_tokens=P)
    assert np.array_equal(_bits(caches[0].k[0]), _bits(caches[1].k[0]))
    assert np.array_equal(_bits(caches[0].v[0]), _bits(caches[1].v[0]))
    assert np.array_equal(ref.cpu().numpy(), got.cpu().numpy())
    assert np.all(got[0].cpu().numpy() == 0.0)                 # empty sequence: nothing appended
    for c in caches:
        assert c.device_error() == 0
        c.close()


def test_fused_llama7b_64_steps_against_oracle():
    w = W.llama7b()
    init = [n - 1 for n in w.lens]
    total = [n + w.steps for n in init]
    cache = PagedKVCache(1, w.num_blocks, w.block_size, w.num_heads, w.head_dim, "f16")
    poison(cache)
    alloc = BlockAllocator(w.num_blocks, w.block_size, W.free_order(w))
    seqs = [alloc.new_seq() for _ in range(w.batch)]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(total)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(total)]
    prefill(cache, alloc, seqs, [k[:n] for k, n in zip(ks, init)], [v[:n] for v, n in zip(vs, init)])
    max_blocks = -(-max(total) // w.block_size)
    worst = 0.0
    for step in range(w.steps):
        pos = [n + step for n in init]
        for sid in seqs:
            _, cow = alloc.append_slots(sid, 1)      # host bookkeeping only; the kernel writes
            assert cow is None
        bt, cl, lens = tables_for(alloc, seqs, max_blocks)
        q = W.host_queries(w, step)
        k_new = torch.from_numpy(np.stack([k[p] for k, p in zip(ks, pos)])).cuda()
        v_new = torch.from_numpy(np.stack([v[p] for v, p in zip(vs, pos)])).cuda()
        out = cache.attention_append(0, torch.from_numpy(q).cuda(), k_new, v_new, bt, cl, max(total), w.scale)
        want = OA.decode_attention(q, [k[:p + 1] for k, p in zip(ks, pos)],
                                   [v[:p + 1] for v, p in zip(vs, pos)], w.scale)
        worst = max(worst, max_abs(out.cpu().numpy(), want))
    assert worst <= tol_for("f16"), worst
    # the pool now holds every token: read sequence 3 back through its table
    table = alloc.table(seqs[3])
    got = torch.stack([cache.k[0][table[t // 16], :, t % 16] for t in range(total[3])]).cpu().numpy()
    assert np.array_equal(got.view(np.uint16), ks[3].view(np.uint16))
    assert cache.device_error() == 0


def test_fused_parallel_sampling_after_cow():
    w = W.parallel_sampling()
    P0, NCAND = W.PROMPT_LEN_PARALLEL, W.CANDIDATES_PARALLEL
    cache = PagedKVCache(1, w.num_blocks, w.block_size, w.num_heads, w.head_dim, "f16")
    poison(cache)
    alloc = BlockAllocator(w.num_blocks, w.block_size, W.free_order(w))
    root = alloc.new_seq()
    pk, pv = W.host_tokens(w, 0, P0, "k"), W.host_tokens(w, 0, P0, "v")
    prefill(cache, alloc, [root], [pk], [pv])
    cands = [root] + [alloc.fork(root) for _ in range(NCAND - 1)]
    gk = [W.host_tokens(w, 100 + c, 8, "k") for c in range(NCAND)]
    gv = [W.host_tokens(w, 100 + c, 8, "v") for c in range(NCAND)]
    max_blocks = -(-(P0 + 8) // 16)
    worst = 0.0
    for step in range(8):
        cows = []
        for sid in cands:
            _, cow = alloc.append_slots(sid, 1)
            if cow:
                cows.append(cow)
        if cows:                                   # copy-on-write before the fused write
            cache.copy_blocks(torch.tensor(cows, dtype=torch.int32, device="cuda"))
        assert len(cows) == (NCAND - 1 if step == 0 else 0)
        bt, cl, lens = tables_for(alloc, cands, max_blocks)
        q = W.host_queries(w, step)
        out = cache.attention_append(0, torch.from_numpy(q).cuda(),
                                     torch.from_numpy(np.stack([g[step] for g in gk])).cuda(),
                                     torch.from_numpy(np.stack([g[step] for g in gv])).cuda(),
                                     bt, cl, P0 + 8, w.scale)
        kk = [np.concatenate([pk, g[:step + 1]]) for g in gk]
        vv = [np.concatenate([pv, g[:step + 1]]) for g in gv]
        worst = max(worst, max_abs(out.cpu().numpy(), OA.decode_attention(q, kk, vv, w.scale)))
    assert worst <= tol_for("f16"), worst
    assert cache.device_error() == 0
