"""GPU: decode attention with shared prompt prefixes (kv_decode_args.prefix_groups).

Parallel sampling forks several candidates from one prompt; until they write into them
the candidates hold the prompt's physical blocks ([PagedAttention] §5.1).  A prefix group
tells the call so, and each shared (block, head) tile is read once for all candidates'
query rows.  The result must still be plain decode attention of every (sequence, head)
over its own context: every output is compared with the float64 oracle (max abs 2e-3),
which sees only each sequence's own token list (host arrays, never the pool).

* the parallel-sampling workload (8 candidates, a 1030-token prompt, 128 steps of the
  fused call with the benchmark's launch flags, copy-on-write at the first step);
* groups of 2 to 8 members mixed with single sequences, fp16 and FP8 pools, B 8/16/32,
  with and without the fused append, shared prefixes of 0 to 2000 tokens (several
  partitions), members with no tokens of their own, float16 output;
* groups that break the rules are attended without sharing and flagged; calls the
  feature does not support are refused.
"""

import math

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import max_abs, poison, tables_for, tol_for
from oracle import fp8 as OF
from oracle_batch import gather_seqs, oracle_sequences
from paged_kv_cache_169_gb300 import abi
from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

pytestmark = pytest.mark.gpu

FLAGS = abi.KV_DECODE_WORKSPACE_ZEROED | abi.KV_DECODE_PDL | abi.KV_DECODE_EARLY_TABLES


def _heads_major(x):
    """[n, H, d] token-major host array -> [H, n, d] (the oracle helper's layout)."""
    return np.ascontiguousarray(np.asarray(x).transpose(1, 0, 2))


def _groups(rows):
    return torch.tensor(rows, dtype=torch.int32, device="cuda").reshape(-1, 3)


def test_parallel_sampling_prefix_groups_every_step():
    w = W.parallel_sampling()
    P0, NC, S, B = W.PROMPT_LEN_PARALLEL, W.CANDIDATES_PARALLEL, w.steps, w.block_size
    cache = PagedKVCache(1, w.num_blocks, B, w.num_heads, w.head_dim, "f16")
    poison(cache)
    alloc = BlockAllocator(w.num_blocks, B, W.free_order(w))
    root = alloc.new_seq()
    prompt_k, prompt_v = W.host_tokens(w, 0, P0, "k"), W.host_tokens(w, 0, P0, "v")
    slots, _ = alloc.append_slots(root, P0)
    cache.append(0, torch.from_numpy(prompt_k).cuda(), torch.from_numpy(prompt_v).cuda(),
                 torch.tensor(slots, dtype=torch.int64, device="cuda"))
    cands = [root] + [alloc.fork(root) for _ in range(NC - 1)]
    gen_k = [W.host_tokens(w, 100 + c, S, "k") for c in range(NC)]
    gen_v = [W.host_tokens(w, 100 + c, S, "v") for c in range(NC)]
    max_blocks = -(-(P0 + S) // B)
    shared = (P0 // B) * B                               # 64 whole blocks stay shared
    groups = _groups([0, NC, shared])
    ws = cache.zeroed_workspace(NC, P0 + S, prefix_groups=True)
    n_cow, worst = 0, 0.0
    for step in range(S):
        cows = []
        for sid in cands:
            _, cow = alloc.append_slots(sid, 1)          # the fused call writes the slot
            if cow:
                cows.append(cow)
        n_cow += len(cows)
        if cows:
            cache.copy_blocks(torch.tensor(cows, dtype=torch.int32, device="cuda"))
        bt, cl, lens = tables_for(alloc, cands, max_blocks)
        assert lens == [P0 + step + 1] * NC
        q = W.host_queries(w, step)
        kn = np.stack([g[step] for g in gen_k])
        vn = np.stack([g[step] for g in gen_v])
        out = cache.attention_ex(0, torch.from_numpy(q).cuda(), bt, cl, P0 + S, w.scale,
                                 k_new=torch.from_numpy(kn).cuda(), v_new=torch.from_numpy(vn).cuda(),
                                 workspace=ws, flags=FLAGS, prefix_groups=groups).cpu().numpy()
        kk = [_heads_major(np.concatenate([prompt_k, g[:step + 1]])) for g in gen_k]
        vv = [_heads_major(np.concatenate([prompt_v, g[:step + 1]])) for g in gen_v]
        worst = max(worst, max_abs(out, oracle_sequences(q, kk, vv, w.scale)))
    print(f"[parity] parallel sampling with prefix groups: 128 steps x 8 x 40 outputs, "
          f"worst max-abs {worst:.3e} (bound 2e-03)", flush=True)
    assert worst <= tol_for("f16"), worst
    assert n_cow == NC - 1
    st = alloc.stats()
    assert st.num_blocks - st.free_blocks == 136            # 64 shared + 8 x 9 private
    # every candidate's cache, read back through its table, is its own token list
    for c, sid in enumerate(cands):
        tab = alloc.table(sid)
        idx = torch.tensor(tab, dtype=torch.int64, device="cuda")
        got = cache.k[0].index_select(0, idx).permute(0, 2, 1, 3).reshape(-1, w.num_heads, w.head_dim)
        want = np.concatenate([prompt_k, gen_k[c]])
        assert np.array_equal(got[:P0 + S].cpu().numpy().view(np.int16), want.view(np.int16))
    assert cache.device_error() == 0


def _build_batch(dtype, B, fused, seed, H=4, d=128):
    """A batch of single sequences and prefix groups built through the allocator: a group's
    root is prefilled, forked, and every member appends tokens of its own (copy-on-write of
    a partly filled shared block included).  With the fused call, each sequence's newest
    token is left for the call to write (its slot reserved here).  Returns everything the
    call and the oracle need; for FP8 pools the host keeps its own copy of the per-block
    scales (a block copy carries its source's scales)."""
    rng = np.random.default_rng(seed)
    # (prompt length, members, own tokens per member); members 1 = a single sequence
    plan = [(int(rng.integers(1, 400)), 1, [int(rng.integers(1, 30))]),
            (2000, 8, [int(x) for x in rng.integers(1, 200, 8)]),
            (int(rng.integers(1, 700)), 1, [int(rng.integers(1, 30))]),
            (37, 3, [1, 60, 5]),
            (5, 2, [3, 9]),                                   # prompt shorter than a block
            (4 * B, 3, [1, 1, 1] if fused else [0, 0, 0]),    # no own token before this call
            (int(rng.integers(100, 900)), 5, [int(x) for x in rng.integers(1, 40, 5)]),
            (int(rng.integers(1, 300)), 1, [int(rng.integers(1, 30))])]
    total = sum(p + m * max(o) for p, m, o in plan)
    nb = 2 * (-(-total // B)) + 64
    w = W.Workload("prefix", seed, 1, H, d, B, "f16", 0, [], nb, 1 / math.sqrt(d))
    cache = PagedKVCache(1, nb, B, H, d, dtype)
    poison(cache)
    sk = sv = None
    if dtype == "fp8":
        sk = (0.02 + 0.001 * (np.arange(cache.k_scale[0].numel()) % 11)).astype(np.float32)
        sv = (0.025 + 0.001 * (np.arange(cache.v_scale[0].numel()) % 7)).astype(np.float32)
        cache.k_scale[0].copy_(torch.from_numpy(sk))
        cache.v_scale[0].copy_(torch.from_numpy(sv))
    alloc = BlockAllocator(nb, B, W.free_order(w))

    def reserve(sid, n):
        slots, cow = alloc.append_slots(sid, n)
        if cow:
            cache.copy_blocks(torch.tensor([cow], dtype=torch.int32, device="cuda"))
            if dtype == "fp8":
                sk[cow[1]], sv[cow[1]] = sk[cow[0]], sv[cow[0]]
        return torch.tensor(slots, dtype=torch.int64, device="cuda")

    seqs, toks_k, toks_v, groups = [], [], [], []
    for key, (prompt, members, own) in enumerate(plan):
        wk = W.Workload("prefix", seed * 100 + key, 1, H, d, B, "f16", 0)
        root = alloc.new_seq()
        pk, pv = W.host_tokens(wk, 0, prompt, "k"), W.host_tokens(wk, 0, prompt, "v")
        cache.append(0, torch.from_numpy(pk).cuda(), torch.from_numpy(pv).cuda(), reserve(root, prompt))
        mem = [root] + [alloc.fork(root) for _ in range(members - 1)]
        if members > 1:
            groups.append([len(seqs), members, (prompt // B) * B])
        for m, sid in enumerate(mem):
            ok, ov = W.host_tokens(wk, 1 + m, own[m], "k"), W.host_tokens(wk, 1 + m, own[m], "v")
            before = own[m] - (1 if fused else 0)         # the fused call writes the last one
            if before > 0:
                cache.append(0, torch.from_numpy(ok[:before]).cuda(), torch.from_numpy(ov[:before]).cuda(),
                             reserve(sid, before))
            seqs.append(sid)
            toks_k.append(np.concatenate([pk, ok]))
            toks_v.append(np.concatenate([pv, ov]))
    n = len(seqs)
    kn = np.stack([t[-1] for t in toks_k])
    vn = np.stack([t[-1] for t in toks_v])
    if fused:
        for sid in seqs:
            reserve(sid, 1)                               # the slot of the call's new token
    lens_want = [t.shape[0] for t in toks_k]
    max_blocks = max(-(-x // B) for x in lens_want)
    bt, cl, lens = tables_for(alloc, seqs, max_blocks)
    assert lens == lens_want
    q = W.host_queries(W.Workload("prefix", seed, 1, H, d, B, "f16", n))
    if dtype == "fp8":
        # the values the host's own quantisation stores, with each token's block scale
        qk, qv = [], []
        for s, sid in enumerate(seqs):
            tab = alloc.table(sid)
            phys = np.array([tab[t // B] for t in range(lens[s])], dtype=np.int64)
            ksc, vsc = sk[phys].reshape(-1, 1, 1), sv[phys].reshape(-1, 1, 1)
            qk.append(OF.decode(OF.quantize(toks_k[s], ksc)) * ksc.astype(np.float64))
            qv.append(OF.decode(OF.quantize(toks_v[s], vsc)) * vsc.astype(np.float64))
        toks_k, toks_v = qk, qv
    want = oracle_sequences(q, [_heads_major(t) for t in toks_k], [_heads_major(t) for t in toks_v], w.scale)
    return dict(cache=cache, alloc=alloc, q=q, bt=bt, cl=cl, lens=lens, groups=groups, want=want,
                kn=kn, vn=vn, scale=w.scale, B=B)


def _pmin(max_ctx):
    """The smallest explicit partition a call with groups accepts."""
    return max(32, (-(-max_ctx // 31) + 31) // 32 * 32)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("dtype", ["f16", "fp8"])
def test_prefix_groups_against_oracle(dtype, B, fused):
    c = _build_batch(dtype, B, fused, seed=600 + B + (7 if fused else 0) + (50 if dtype == "fp8" else 0))
    cache, lens = c["cache"], c["lens"]
    grp = _groups(c["groups"])
    max_ctx = max(lens)
    q = torch.from_numpy(c["q"]).cuda()
    kw = {}
    if fused:
        kw = dict(k_new=torch.from_numpy(c["kn"]).cuda(), v_new=torch.from_numpy(c["vn"]).cuda())
    worst = 0.0
    for P in (0, _pmin(max_ctx), 1024):
        out = cache.attention_ex(0, q, c["bt"], c["cl"], max_ctx, c["scale"], partition_tokens=P,
                                 prefix_groups=grp, **kw)
        worst = max(worst, max_abs(out.cpu().numpy(), c["want"]))
        # the same call again gives the same bits, whichever warps finish last and merge
        again = cache.attention_ex(0, q, c["bt"], c["cl"], max_ctx, c["scale"], partition_tokens=P,
                                   prefix_groups=grp, **kw)
        assert torch.equal(again, out)
        # float16 output: the float32 result rounded to nearest even
        o16 = cache.attention_ex(0, q, c["bt"], c["cl"], max_ctx, c["scale"], partition_tokens=P,
                                 prefix_groups=grp, out_dtype=torch.float16, **kw)
        assert torch.equal(o16, out.half())
    assert worst <= tol_for("f16"), worst
    # the same batch without groups agrees with the oracle as well
    out = cache.attention_ex(0, q, c["bt"], c["cl"], max_ctx, c["scale"], **kw)
    assert max_abs(out.cpu().numpy(), c["want"]) <= tol_for("f16")
    assert cache.device_error() == 0


@pytest.mark.parametrize("dtype", ["f16", "fp8"])
def test_prefix_groups_odd_head_count(dtype):
    """Three heads: the head-pair stages need an even count, so this runs the one-head-per-
    stage shape of the shared-prefix launch."""
    c = _build_batch(dtype, 16, False, seed=680, H=3)
    grp = _groups(c["groups"])
    out = c["cache"].attention_ex(0, torch.from_numpy(c["q"]).cuda(), c["bt"], c["cl"], max(c["lens"]),
                                  c["scale"], prefix_groups=grp)
    assert max_abs(out.cpu().numpy(), c["want"]) <= tol_for("f16")
    assert c["cache"].device_error() == 0


def _simple_batch(lens_prompt=64, members=6, own=(3, 20, 1, 7, 40, 2), B=16, H=2, seed=700):
    d = 128
    nb = 64
    w = W.Workload("prefix_rules", seed, 1, H, d, B, "f16", 0, [], nb, 1 / math.sqrt(d))
    cache = PagedKVCache(1, nb, B, H, d, "f16")
    poison(cache)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    root = alloc.new_seq()
    pk, pv = W.host_tokens(w, 0, lens_prompt, "k"), W.host_tokens(w, 0, lens_prompt, "v")
    sl, _ = alloc.append_slots(root, lens_prompt)
    cache.append(0, torch.from_numpy(pk).cuda(), torch.from_numpy(pv).cuda(), torch.tensor(sl, device="cuda"))
    mem = [root] + [alloc.fork(root) for _ in range(members - 1)]
    ks, vs = [], []
    for m, sid in enumerate(mem):
        ok, ov = W.host_tokens(w, 1 + m, own[m], "k"), W.host_tokens(w, 1 + m, own[m], "v")
        sl, cow = alloc.append_slots(sid, own[m])
        assert cow is None
        cache.append(0, torch.from_numpy(ok).cuda(), torch.from_numpy(ov).cuda(), torch.tensor(sl, device="cuda"))
        ks.append(np.concatenate([pk, ok]))
        vs.append(np.concatenate([pv, ov]))
    bt, cl, lens = tables_for(alloc, mem, 8)
    q = W.host_queries(W.Workload("prefix_rules", seed, 1, H, d, B, "f16", members))
    want = oracle_sequences(q, [_heads_major(x) for x in ks], [_heads_major(x) for x in vs], w.scale)
    return cache, alloc, torch.from_numpy(q).cuda(), bt, cl, lens, want, w.scale


@pytest.mark.parametrize("rows", [
    [[0, 4, 64], [2, 4, 64]],          # overlapping: the second is dropped
    [[3, 3, 64], [0, 2, 64]],          # not sorted: the second is dropped
    [[0, 9, 64]],                      # more than 8 members (and beyond the batch)
    [[0, 1, 64]],                      # fewer than 2
    [[0, 6, 40]],                      # not whole blocks
    [[0, 6, 80]],                      # longer than a member's context (65)
    [[0, 5, 64], [5, 2, 64]],          # the second group runs past the batch
])
def test_prefix_groups_breaking_the_rules_are_flagged(rows):
    cache, alloc, q, bt, cl, lens, want, scale = _simple_batch()
    out = cache.attention_ex(0, q, bt, cl, max(lens), scale, prefix_groups=_groups(rows))
    assert max_abs(out.cpu().numpy(), want) <= tol_for("f16")
    assert cache.device_error() & abi.KV_DEVERR_PREFIX
    # a valid group on the same batch sets nothing
    out = cache.attention_ex(0, q, bt, cl, max(lens), scale, prefix_groups=_groups([[0, 6, 64]]))
    assert max_abs(out.cpu().numpy(), want) <= tol_for("f16")
    assert cache.device_error() == 0


def test_prefix_group_with_fused_append_needs_an_own_token():
    """With the fused append every member must keep at least its newest token outside the
    shared prefix: a member whose whole context is shared breaks the rule."""
    cache, alloc, q, bt, cl, lens, want, scale = _simple_batch(own=(3, 20, 1, 7, 40, 2))
    kn = torch.zeros((6, 2, 128), dtype=torch.float16, device="cuda")
    ok = _groups([[0, 6, 64]])                            # every member has 65 tokens or more
    cache.attention_ex(0, q, bt, cl, max(lens), scale, k_new=kn, v_new=kn, prefix_groups=ok)
    assert cache.device_error() == 0
    cl2 = cl.clone()
    cl2[2] = 64                                           # member 2: all 64 tokens shared
    cache.attention_ex(0, q, bt, cl2, max(lens), scale, prefix_groups=ok)
    assert cache.device_error() == 0                      # fine without an append
    # the same lengths with the append: member 2's new token would land in the prefix
    cache.attention_ex(0, q, bt, cl2, max(lens), scale, k_new=kn, v_new=kn, prefix_groups=ok)
    assert cache.device_error() & abi.KV_DEVERR_PREFIX


def test_prefix_group_crossing_a_launch_of_1024_sequences():
    """Calls of more than 1024 sequences run as several launches; a group may not span two."""
    B, H, d, n = 16, 2, 128, 1030
    lens = [20] * n
    nb = n * 2 + 8
    w = W.Workload("prefix_span", 710, 1, H, d, B, "f16", n, lens, nb, 1 / math.sqrt(d))
    cache = PagedKVCache(1, nb, B, H, d, "f16")
    W.device_fill_normal(cache.k[0], 7101)
    W.device_fill_normal(cache.v[0], 7102)
    tables = W.shuffled_tables(w, [2] * n)
    tables[1000:1004, 0] = tables[1000, 0]                # 4 sequences share their first block
    tables[1020:1028, 0] = tables[1020, 0]                # 8 more, across sequence 1024
    k0, v0 = cache.k[0].clone(), cache.v[0].clone()       # the oracle's inputs
    bt = torch.from_numpy(tables).cuda()
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    q = W.host_queries(w)
    out = cache.attention_ex(0, torch.from_numpy(q).cuda(), bt, cl, 20, w.scale,
                             prefix_groups=_groups([[1000, 4, 16], [1020, 8, 16]])).cpu().numpy()
    assert cache.device_error() & abi.KV_DEVERR_PREFIX       # the second spans two launches
    want = oracle_sequences(q, gather_seqs(k0, tables, lens, B), gather_seqs(v0, tables, lens, B), w.scale)
    assert max_abs(out, want) <= tol_for("f16")


def test_prefix_groups_refused_where_unsupported():
    B, H, d = 16, 2, 128
    z = torch.zeros((2, H, d), dtype=torch.float16, device="cuda")
    bt = torch.zeros((2, 1), dtype=torch.int32, device="cuda")
    cl = torch.ones(2, dtype=torch.int32, device="cuda")
    g = _groups([[0, 2, 0]])
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    f16 = PagedKVCache(1, 4, B, H, d, "f16")
    with pytest.raises(abi.KvError) as e:             # grouped-query heads
        f16.attention_ex(0, torch.zeros((2, 2 * H, d), dtype=torch.float16, device="cuda"), bt, cl, 1, 0.1,
                         workspace=ws, prefix_groups=g)
    assert e.value.status == abi.KV_ERR_UNSUPPORTED
    with pytest.raises(abi.KvError) as e:             # sliding window
        f16.attention_ex(0, z, bt, cl, 1, 0.1, window=8, workspace=ws, prefix_groups=g)
    assert e.value.status == abi.KV_ERR_UNSUPPORTED
    with pytest.raises(abi.KvError) as e:             # a partition too small for one merge step
        f16.attention_ex(0, z, bt, cl, 4096, 0.1, partition_tokens=64, workspace=ws, prefix_groups=g)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
    for dt, dd in (("f32", 128), ("f16", 64)):        # no tensor maps
        p = PagedKVCache(1, 4, B, H, dd, dt)
        qq = torch.zeros((2, H, dd), dtype=torch.float32 if dt == "f32" else torch.float16, device="cuda")
        with pytest.raises(abi.KvError) as e:
            p.attention_ex(0, qq, bt, cl, 1, 0.1, workspace=ws, prefix_groups=g)
        assert e.value.status == abi.KV_ERR_UNSUPPORTED
    # a group count without a pointer, or more groups than sequences
    a = abi.kv_decode_args()
    out = torch.zeros((2, H, d), device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    a.layer, a.q, a.out, a.block_tables, a.max_blocks_per_seq = 0, z.data_ptr(), out.data_ptr(), bt.data_ptr(), 1
    a.context_lens, a.batch, a.max_context, a.scale = cl.data_ptr(), 2, 1, 0.1
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    a.stream = torch.cuda.current_stream().cuda_stream
    a.num_prefix_groups = 1
    with pytest.raises(abi.KvError) as e:
        abi.paged_decode_attention_ex(f16.handle, a)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
    a.prefix_groups, a.num_prefix_groups = g.data_ptr(), 3
    with pytest.raises(abi.KvError) as e:
        abi.paged_decode_attention_ex(f16.handle, a)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
