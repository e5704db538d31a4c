"""GPU: full-size workloads in the launch configuration the benchmark times, checked on
sampled (layer, sequence, head) outputs that the float64 oracle computes one by one.

Pools are filled with seeded N(0,1) values by torch's device generator (inputs, not
kernel output); the oracle reads the sampled tiles back before the decode append and
adds the new token itself.  The benchmark's call: one paged_decode_attention_ex per
layer that appends each sequence's new token and attends, library-chosen partitioning,
a workspace zero-filled once and kept over all calls (KV_DECODE_WORKSPACE_ZEROED),
programmatic dependent launch (KV_DECODE_PDL), tables read before the previous launch
ends (KV_DECODE_EARLY_TABLES: they are written before the layer loop) and the first K/V
tiles fetched before it ends (KV_DECODE_EARLY_POOL: the previous launch wrote another
layer's pool).  The 13B step also runs as kv_append followed by paged_decode_attention.
"""

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import max_abs, tol_for
from oracle import attention as OA
from oracle import fp8 as OF
from paged_kv_cache_169_gb300 import abi
from paged_kv_cache_169_gb300.cache import PagedKVCache

pytestmark = pytest.mark.gpu

BENCH_FLAGS = (abi.KV_DECODE_WORKSPACE_ZEROED | abi.KV_DECODE_PDL | abi.KV_DECODE_EARLY_TABLES |
               abi.KV_DECODE_EARLY_POOL)


def _snapshot(pool: torch.Tensor, table_row, n_blocks: int, h: int) -> np.ndarray:
    """[n_blocks*B, d] tokens of one head, read from the pool through a table row."""
    idx = torch.tensor(table_row[:n_blocks], dtype=torch.int64, device=pool.device)
    t = pool.index_select(0, idx)[:, h]                  # [n_blocks, B, d]
    return t.reshape(-1, t.shape[-1]).cpu().numpy()


@pytest.mark.parametrize("path", ["fused_flags", "unfused"])
def test_llama13b_full_step_sampled(path):
    w = W.llama13b()
    B, H, d = w.block_size, w.num_heads, w.head_dim
    cache = PagedKVCache(w.num_layers, w.num_blocks, B, H, d, "f16")
    for l in range(w.num_layers):
        W.device_fill_normal(cache.k[l], w.seed * 1000 + 2 * l)
        W.device_fill_normal(cache.v[l], w.seed * 1000 + 2 * l + 1)
    nbs = [n // B for n in w.lens]                                   # 128 blocks each
    tables = W.shuffled_tables(w, nbs)
    bt = torch.from_numpy(tables).cuda()
    cl = torch.tensor(w.lens, dtype=torch.int32, device="cuda")
    slots = torch.tensor([int(tables[s, (n - 1) // B]) * B + (n - 1) % B for s, n in enumerate(w.lens)],
                         dtype=torch.int64, device="cuda")
    rng = np.random.default_rng(31)
    samples = [(l, int(rng.integers(w.batch)), int(rng.integers(H))) for l in (0, 13, 27, 39) for _ in range(6)]
    samples += [(39, w.batch - 1, H - 1), (0, 0, 0)]
    snap = {}
    for (l, s, h) in samples:
        snap[(l, s, h)] = (_snapshot(cache.k[l], tables[s], nbs[s], h), _snapshot(cache.v[l], tables[s], nbs[s], h))
    outs = {}
    fused = path == "fused_flags"
    ws = cache.zeroed_workspace(w.batch, max(w.lens)) if fused else cache.workspace(w.batch, max(w.lens))
    for l in range(w.num_layers):
        k_new = W.host_step_tokens(w, 0, l, "k")
        v_new = W.host_step_tokens(w, 0, l, "v")
        q = W.host_queries(w, 0, l)
        if fused:
            out = cache.attention_ex(l, torch.from_numpy(q).cuda(), bt, cl, max(w.lens), w.scale,
                                     k_new=torch.from_numpy(k_new).cuda(), v_new=torch.from_numpy(v_new).cuda(),
                                     workspace=ws, flags=BENCH_FLAGS)
        else:
            cache.append(l, torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda(), slots)
            out = cache.attention(l, torch.from_numpy(q).cuda(), bt, cl, max(w.lens), w.scale, workspace=ws)
        if any(x[0] == l for x in samples):
            outs[l] = (out.cpu().numpy(), q, k_new, v_new)
    worst = 0.0
    for (l, s, h) in samples:
        out, q, k_new, v_new = outs[l]
        K, V = snap[(l, s, h)]
        K, V = K.copy(), V.copy()
        n = w.lens[s]
        K[n - 1], V[n - 1] = k_new[s, h], v_new[s, h]                # the oracle's own append
        want = OA.decode_attention_one(q[s, h], K[:n], V[:n], w.scale)
        worst = max(worst, max_abs(out[s, h], want))
    assert worst <= tol_for("f16"), worst
    assert cache.device_error() == 0
    del cache
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("dtype", ["f16", "fp8"])
def test_ragged_full_size_sampled(B, dtype):
    w = W.ragged(B)
    H, d = w.num_heads, w.head_dim
    cache = PagedKVCache(1, w.num_blocks, B, H, d, dtype)
    nbs = [-(-n // B) for n in w.lens]
    tables = W.shuffled_tables(w, nbs)
    if dtype == "f16":
        W.device_fill_normal(cache.k[0], w.seed * 1000 + B)
        W.device_fill_normal(cache.v[0], w.seed * 1000 + B + 1)
    else:
        # FP8 content: N(0,1) fp16 values stored with a per-block scale amax/448
        # (input preparation with torch's own float8 cast), block by block
        for pool, sc, key in ((cache.k[0], cache.k_scale[0], 1), (cache.v[0], cache.v_scale[0], 2)):
            g = torch.Generator(device="cuda")
            g.manual_seed(w.seed * 1000 + B * 10 + key)
            step = 4096
            for b0 in range(0, w.num_blocks, step):
                nb = min(step, w.num_blocks - b0)
                x = torch.randn((nb, H, B, d), generator=g, device="cuda").half().float()
                amax = x.abs().amax(dim=(1, 2, 3)).clamp_min(2.0 ** -20 * 448)
                s = (amax / 448.0).float()
                codes = (x / s.view(-1, 1, 1, 1)).clamp(-448, 448).to(torch.float8_e4m3fn)
                pool[b0:b0 + nb].copy_(codes.view(torch.uint8))
                sc[b0:b0 + nb].copy_(s)
    bt = torch.from_numpy(tables).cuda()
    cl = torch.tensor(w.lens, dtype=torch.int32, device="cuda")
    slots = torch.tensor([int(tables[s, (n - 1) // B]) * B + (n - 1) % B for s, n in enumerate(w.lens)],
                         dtype=torch.int64, device="cuda")
    rng = np.random.default_rng(40 + B)
    order = np.argsort(w.lens)
    picks = [int(order[0]), int(order[1]), int(order[-1]), int(order[-2])] + rng.integers(0, w.batch, 12).tolist()
    samples = [(s, int(rng.integers(H))) for s in picks]
    snap = {(s, h): (_snapshot(cache.k[0], tables[s], nbs[s], h), _snapshot(cache.v[0], tables[s], nbs[s], h))
            for (s, h) in samples}
    ksc = cache.k_scale[0].cpu().numpy() if dtype == "fp8" else None
    vsc = cache.v_scale[0].cpu().numpy() if dtype == "fp8" else None
    k_new = W.host_step_tokens(w, 0, 0, "k")
    v_new = W.host_step_tokens(w, 0, 0, "v")
    q = W.host_queries(w)
    assert slots.numel() == w.batch                     # the slots the fused call writes
    ws = cache.zeroed_workspace(w.batch, max(w.lens))
    out = cache.attention_ex(0, torch.from_numpy(q).cuda(), bt, cl, max(w.lens), w.scale,
                             k_new=torch.from_numpy(k_new).cuda(), v_new=torch.from_numpy(v_new).cuda(),
                             workspace=ws, flags=BENCH_FLAGS).cpu().numpy()
    worst = 0.0
    for (s, h) in samples:
        n = w.lens[s]
        K, V = (a.copy() for a in snap[(s, h)])
        if dtype == "fp8":
            phys = np.array([tables[s, t // B] for t in range(nbs[s] * B)])
            last = int(tables[s, (n - 1) // B])
            # the oracle's own FP8 append of the new token, then dequantisation
            K[n - 1] = OF.quantize(k_new[s, h], ksc[last])
            V[n - 1] = OF.quantize(v_new[s, h], vsc[last])
            # bit-exact check of the slot the kernel wrote
            dev = cache.k[0][last, h, (n - 1) % B].cpu().numpy()
            assert np.array_equal(dev, K[n - 1])
            K = OF.decode(K) * ksc[phys].astype(np.float64)[:, None]
            V = OF.decode(V) * vsc[phys].astype(np.float64)[:, None]
        else:
            K[n - 1], V[n - 1] = k_new[s, h], v_new[s, h]
        want = OA.decode_attention_one(q[s, h], K[:n], V[:n], w.scale)
        worst = max(worst, max_abs(out[s, h], want))
    assert worst <= tol_for("f16"), worst
    assert np.all(np.isfinite(out))
    assert cache.device_error() == 0
    del cache
    torch.cuda.empty_cache()


def test_finer_partitions_for_the_sequences_handed_out_last():
    """A long launch of long items (library partitioning picks 576 tokens here: 128
    sequences of 12k-16k tokens, 4 heads) gives the sequences handed out last half-size
    partitions.  The plan shows it (a larger split count, hence a larger workspace than an
    explicit 576-token partition).  Outputs agree with the explicit partitioning to within
    rounding (1e-4: the softmax weights enter the V products as fp16, each rounded
    relative to its partition's running maximum, so two partitionings round them
    differently; 1.3e-5 measured), and with the float64 oracle on sampled (sequence, head)
    pairs, the last sequences included."""
    B, H, d, batch = 16, 4, 128, 128
    rng = np.random.default_rng(77)
    lens = rng.integers(12000, 16385, batch).tolist()
    lens[-1] = 16384
    nbs = [-(-n // B) for n in lens]
    w = W.Workload("fine_tail", 77, 1, H, d, B, "f16", batch, lens, sum(nbs), 1 / np.sqrt(d))
    cache = PagedKVCache(1, w.num_blocks, B, H, d, "f16")
    W.device_fill_normal(cache.k[0], 7701)
    W.device_fill_normal(cache.v[0], 7702)
    tables = W.shuffled_tables(w, nbs)
    bt = torch.from_numpy(tables).cuda()
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    max_ctx = max(lens)
    assert cache.workspace_bytes(batch, max_ctx, 0) > cache.workspace_bytes(batch, max_ctx, 576)
    q = W.host_queries(w)
    qt = torch.from_numpy(q).cuda()
    auto = cache.attention(0, qt, bt, cl, max_ctx, w.scale, partition_tokens=0).cpu().numpy()
    fixed = cache.attention(0, qt, bt, cl, max_ctx, w.scale, partition_tokens=576).cpu().numpy()
    assert max_abs(auto, fixed) <= 1e-4
    samples = [(int(rng.integers(batch)), int(rng.integers(H))) for _ in range(6)]
    samples += [(batch - 1, H - 1), (batch - 2, 0), (batch - 5, 1), (0, 0)]
    worst = 0.0
    for s, h in samples:
        K = _snapshot(cache.k[0], tables[s], nbs[s], h)[:lens[s]]
        V = _snapshot(cache.v[0], tables[s], nbs[s], h)[:lens[s]]
        worst = max(worst, max_abs(auto[s, h], OA.decode_attention_one(q[s, h], K, V, w.scale)))
    assert worst <= tol_for("f16"), worst
    assert cache.device_error() == 0
    del cache
    torch.cuda.empty_cache()
