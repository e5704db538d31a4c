"""GPU: full-size workloads in the launch configuration the benchmark times, checked on
EVERY output against the float64 oracle, and every pool byte checked after the step.

Pools are filled with seeded N(0,1) values by torch's device generator (inputs, not
kernel output).  After the call the test rebuilds each layer's pool as it was before the
step (the same seeded fill again, or a device copy taken before the call), writes each
sequence's new token into its slot itself (the oracle's own append; FP8: the oracle's
own quantisation), and then
  * checks that the pool the kernel left is bit-identical to that rebuilt pool (every
    appended slot exact, nothing else touched), and
  * gathers every sequence's cache from the rebuilt pool through its block table and
    runs the oracle on every (sequence, head): tests/oracle_batch.py spreads the units
    over the host cores.
The benchmark's call: one paged_decode_attention_ex per layer that appends each
sequence's new token and attends, library-chosen partitioning, a workspace zero-filled
once and kept over all calls (KV_DECODE_WORKSPACE_ZEROED), programmatic dependent launch
(KV_DECODE_PDL), tables read before the previous launch ends (KV_DECODE_EARLY_TABLES:
they are written before the layer loop) and the first K/V tiles fetched before it ends
(KV_DECODE_EARLY_POOL: the previous launch wrote another layer's pool).  The 13B step
also runs as kv_append followed by paged_decode_attention.

Each test prints its worst max-abs error against the bound ("[parity] ..." lines, shown
with pytest -s).
"""

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import max_abs, tol_for
from oracle import fp8 as OF
from oracle_batch import gather_seqs, oracle_sequences
from paged_kv_cache_169_gb300 import abi
from paged_kv_cache_169_gb300.cache import PagedKVCache

pytestmark = pytest.mark.gpu

BENCH_FLAGS = (abi.KV_DECODE_WORKSPACE_ZEROED | abi.KV_DECODE_PDL | abi.KV_DECODE_EARLY_TABLES |
               abi.KV_DECODE_EARLY_POOL)


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.uint8)


def _append_rows(pool: torch.Tensor, tables, lens, B: int, rows: torch.Tensor) -> None:
    """The test's own append into a copy of the pool: token n-1 of every sequence (every
    head) takes its new value.  rows: device [S, H, d] in the pool's dtype."""
    dev = pool.device
    blk = torch.tensor([int(tables[s, (n - 1) // B]) for s, n in enumerate(lens)], dtype=torch.int64, device=dev)
    off = torch.tensor([(n - 1) % B for n in lens], dtype=torch.int64, device=dev)
    pool[blk, :, off, :] = rows


def _report(name: str, worst: float, units: int, bound: float) -> None:
    print(f"[parity] {name}: {units} outputs, worst max-abs {worst:.3e} (bound {bound:.0e})", flush=True)


@pytest.mark.parametrize("path", ["fused_flags", "unfused"])
def test_llama13b_full_step_every_output(path):
    w = W.llama13b()
    B, H, d = w.block_size, w.num_heads, w.head_dim
    cache = PagedKVCache(w.num_layers, w.num_blocks, B, H, d, "f16")
    seed = {"k": lambda l: w.seed * 1000 + 2 * l, "v": lambda l: w.seed * 1000 + 2 * l + 1}
    for l in range(w.num_layers):
        W.device_fill_normal(cache.k[l], seed["k"](l))
        W.device_fill_normal(cache.v[l], seed["v"](l))
    nbs = [n // B for n in w.lens]                                   # 128 blocks each
    tables = W.shuffled_tables(w, nbs)
    bt = torch.from_numpy(tables).cuda()
    cl = torch.tensor(w.lens, dtype=torch.int32, device="cuda")
    slots = torch.tensor([int(tables[s, (n - 1) // B]) * B + (n - 1) % B for s, n in enumerate(w.lens)],
                         dtype=torch.int64, device="cuda")
    fused = path == "fused_flags"
    ws = cache.zeroed_workspace(w.batch, max(w.lens)) if fused else cache.workspace(w.batch, max(w.lens))
    outs, ins = [], []
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
        outs.append(out.cpu().numpy())
        ins.append((q, k_new, v_new))
    assert cache.device_error() == 0
    worst = 0.0
    before = {kind: torch.empty_like(cache.k[0]) for kind in ("k", "v")}
    for l in range(w.num_layers):
        q, k_new, v_new = ins[l]
        seqs = {}
        for kind, new, pool in (("k", k_new, cache.k[l]), ("v", v_new, cache.v[l])):
            ref = before[kind]
            W.device_fill_normal(ref, seed[kind](l))                 # the layer before the step
            _append_rows(ref, tables, w.lens, B, torch.from_numpy(new).cuda())
            assert torch.equal(_bits(pool), _bits(ref)), (l, kind)   # every pool byte
            seqs[kind] = gather_seqs(ref, tables, w.lens, B)
        want = oracle_sequences(q, seqs["k"], seqs["v"], w.scale)
        worst = max(worst, max_abs(outs[l], want))
        assert np.all(np.isfinite(outs[l]))
    _report(f"llama13b {path} (40 layers x 48 sequences x 40 heads)", worst, 40 * 48 * 40, tol_for("f16"))
    assert worst <= tol_for("f16"), worst
    del cache, before
    torch.cuda.empty_cache()


def _fill_fp8(pool: torch.Tensor, sc: torch.Tensor, seed: int) -> None:
    """FP8 content: N(0,1) fp16 values stored with a per-block scale amax/448 (input
    preparation with torch's own float8 cast), block by block."""
    H, B, d = pool.shape[1:]
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    step = 4096
    for b0 in range(0, pool.shape[0], step):
        nb = min(step, pool.shape[0] - b0)
        x = torch.randn((nb, H, B, d), generator=g, device="cuda").half().float()
        amax = x.abs().amax(dim=(1, 2, 3)).clamp_min(2.0 ** -20 * 448)
        s = (amax / 448.0).float()
        codes = (x / s.view(-1, 1, 1, 1)).clamp(-448, 448).to(torch.float8_e4m3fn)
        pool[b0:b0 + nb].copy_(codes.view(torch.uint8))
        sc[b0:b0 + nb].copy_(s)


@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("dtype", ["f16", "fp8"])
def test_ragged_full_size_every_output(B, dtype):
    w = W.ragged(B)
    H, d = w.num_heads, w.head_dim
    cache = PagedKVCache(1, w.num_blocks, B, H, d, dtype)
    nbs = [-(-n // B) for n in w.lens]
    tables = W.shuffled_tables(w, nbs)
    if dtype == "f16":
        W.device_fill_normal(cache.k[0], w.seed * 1000 + B)
        W.device_fill_normal(cache.v[0], w.seed * 1000 + B + 1)
    else:
        _fill_fp8(cache.k[0], cache.k_scale[0], w.seed * 1000 + B * 10 + 1)
        _fill_fp8(cache.v[0], cache.v_scale[0], w.seed * 1000 + B * 10 + 2)
    k_before, v_before = cache.k[0].clone(), cache.v[0].clone()     # the pool before the step
    ksc = cache.k_scale[0].cpu().numpy() if dtype == "fp8" else None
    vsc = cache.v_scale[0].cpu().numpy() if dtype == "fp8" else None
    bt = torch.from_numpy(tables).cuda()
    cl = torch.tensor(w.lens, dtype=torch.int32, device="cuda")
    k_new = W.host_step_tokens(w, 0, 0, "k")
    v_new = W.host_step_tokens(w, 0, 0, "v")
    q = W.host_queries(w)
    ws = cache.zeroed_workspace(w.batch, max(w.lens))
    out = cache.attention_ex(0, torch.from_numpy(q).cuda(), bt, cl, max(w.lens), w.scale,
                             k_new=torch.from_numpy(k_new).cuda(), v_new=torch.from_numpy(v_new).cuda(),
                             workspace=ws, flags=BENCH_FLAGS).cpu().numpy()
    assert cache.device_error() == 0
    assert np.all(np.isfinite(out))
    if dtype == "fp8":
        # the oracle's own FP8 append: each new row quantised with its block's scale
        last = [int(tables[s, (n - 1) // B]) for s, n in enumerate(w.lens)]
        k_rows = np.stack([OF.quantize(k_new[s], ksc[last[s]]) for s in range(w.batch)])
        v_rows = np.stack([OF.quantize(v_new[s], vsc[last[s]]) for s in range(w.batch)])
    else:
        k_rows, v_rows = k_new, v_new
    _append_rows(k_before, tables, w.lens, B, torch.from_numpy(k_rows).cuda())
    _append_rows(v_before, tables, w.lens, B, torch.from_numpy(v_rows).cuda())
    assert torch.equal(_bits(cache.k[0]), _bits(k_before))          # every pool byte
    assert torch.equal(_bits(cache.v[0]), _bits(v_before))
    worst = 0.0
    chunk = 32                                                      # bounded host memory
    for s0 in range(0, w.batch, chunk):
        seqs = list(range(s0, min(w.batch, s0 + chunk)))
        if dtype == "fp8":
            ks, kts = gather_seqs(k_before, tables, w.lens, B, seqs, tok_scale=ksc)
            vs, vts = gather_seqs(v_before, tables, w.lens, B, seqs, tok_scale=vsc)
            want = oracle_sequences(q[seqs], ks, vs, w.scale, k_tok_scale=kts, v_tok_scale=vts)
        else:
            ks = gather_seqs(k_before, tables, w.lens, B, seqs)
            vs = gather_seqs(v_before, tables, w.lens, B, seqs)
            want = oracle_sequences(q[seqs], ks, vs, w.scale)
        worst = max(worst, max_abs(out[seqs], want))
    _report(f"ragged {dtype} B {B} (256 sequences x 32 heads)", worst, w.batch * H, tol_for("f16"))
    assert worst <= tol_for("f16"), worst
    del cache, k_before, v_before
    torch.cuda.empty_cache()


def test_gqa70b_full_size_layer_every_output():
    """The LLaMA-2-70B-shaped layer (64 query / 8 KV heads, batch 32, context 4096) in the
    launch configuration the benchmark times, with the fused append (layer 1 of a 2-layer
    pool, so the layer index is exercised); every (sequence, query head)."""
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
    l = 1
    k_before, v_before = cache.k[l].clone(), cache.v[l].clone()
    q = W.host_queries(w, 0, l)
    k_new, v_new = W.host_step_tokens(w, 0, l, "k"), W.host_step_tokens(w, 0, l, "v")
    ws = cache.zeroed_workspace(w.batch, max(w.lens), num_q_heads=Hq)
    out = cache.attention_ex(l, torch.from_numpy(q).cuda(), bt, cl, max(w.lens), w.scale,
                             k_new=torch.from_numpy(k_new).cuda(), v_new=torch.from_numpy(v_new).cuda(),
                             workspace=ws, flags=BENCH_FLAGS).cpu().numpy()
    assert cache.device_error() == 0
    _append_rows(k_before, tables, w.lens, B, torch.from_numpy(k_new).cuda())
    _append_rows(v_before, tables, w.lens, B, torch.from_numpy(v_new).cuda())
    assert torch.equal(_bits(cache.k[l]), _bits(k_before))
    assert torch.equal(_bits(cache.v[l]), _bits(v_before))
    want = oracle_sequences(q, gather_seqs(k_before, tables, w.lens, B), gather_seqs(v_before, tables, w.lens, B),
                            w.scale, group=Hq // H)
    worst = max_abs(out, want)
    _report("gqa70b layer (32 sequences x 64 query heads)", worst, w.batch * Hq, tol_for("f16"))
    assert worst <= tol_for("f16"), worst
    del cache, k_before, v_before
    torch.cuda.empty_cache()


def test_finer_partitions_for_the_sequences_handed_out_last():
    """A long launch of long items (library partitioning picks 576 tokens here: 128
    sequences of 12k-16k tokens, 4 heads) gives the sequences handed out last half-size
    partitions.  The plan shows it (a larger split count, hence a larger workspace than an
    explicit 576-token partition).  Outputs agree with the explicit partitioning to within
    rounding (1e-4: the softmax weights enter the V products as fp16, each rounded
    relative to its partition's running maximum, so two partitionings round them
    differently; 1.3e-5 measured), and with the float64 oracle on every (sequence, head)."""
    B, H, d, batch = 16, 4, 128, 128
    rng = np.random.default_rng(77)
    lens = rng.integers(12000, 16385, batch).tolist()
    lens[-1] = 16384
    nbs = [-(-n // B) for n in lens]
    w = W.Workload("fine_tail", 77, 1, H, d, B, "f16", batch, lens, sum(nbs), 1 / np.sqrt(d))
    cache = PagedKVCache(1, w.num_blocks, B, H, d, "f16")
    W.device_fill_normal(cache.k[0], 7701)
    W.device_fill_normal(cache.v[0], 7702)
    k_before, v_before = cache.k[0].clone(), cache.v[0].clone()     # the oracle's inputs
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
    worst = 0.0
    for s0 in range(0, batch, 32):
        seqs = list(range(s0, min(batch, s0 + 32)))
        want = oracle_sequences(q[seqs], gather_seqs(k_before, tables, lens, B, seqs),
                                gather_seqs(v_before, tables, lens, B, seqs), w.scale)
        worst = max(worst, max_abs(auto[seqs], want))
    _report("fine tail partitions (128 sequences x 4 heads, 12k-16k tokens)", worst, batch * H, tol_for("f16"))
    assert worst <= tol_for("f16"), worst
    assert cache.device_error() == 0
    assert torch.equal(cache.k[0], k_before) and torch.equal(cache.v[0], v_before)
    del cache, k_before, v_before
    torch.cuda.empty_cache()
