"""GPU: sliding-window decode (paged_decode_attention_ex with window > 0) through the C ABI
against the oracle's sliding-window attention (max abs 2e-3, fp16 / FP8-dequantised K/V).

Blocks that fall wholly before the window are trimmed from the tables (entries -1), given
to another sequence and overwritten with NaN: the kernel must never read them (a read of
a -1 entry would also raise the device's block-id error bit)."""

import math

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import max_abs, poison, prefill, tables_for, tol_for
from oracle import attention as OA
from oracle import fp8 as OF
from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

pytestmark = pytest.mark.gpu


def _case(dtype, B, G, window, seed, fused):
    lens = [0, 1, 5, B, B + 3, 40, 77, 300, 1000, 2500]
    Hkv, d = 2, 128
    nb = 2 * sum(-(-n // B) for n in lens) + 8
    w = W.Workload("window", seed, 1, Hkv, d, B, "f16", len(lens), lens, nb, 1 / math.sqrt(d),
                   num_q_heads=G * Hkv)
    cache = PagedKVCache(1, nb, B, Hkv, d, dtype)
    poison(cache)
    sc = np.float32(0.011)
    if dtype == "fp8":
        for t in cache.k_scale + cache.v_scale:
            t.fill_(float(sc))
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    # prefill everything except (when fused) the newest token
    prefill(cache, alloc, seqs, [k[:-1] if fused and len(k) else k for k in ks],
            [v[:-1] if fused and len(v) else v for v in vs])
    if fused:
        for s, sid in enumerate(seqs):
            if lens[s]:
                alloc.append_slots(sid, 1)
    # the window leaves blocks behind: release them and let another sequence scribble on them
    released = 0
    for s, sid in enumerate(seqs):
        released += alloc.trim(sid, max(0, lens[s] - window))
    other = alloc.new_seq()
    if released:
        slots, _ = alloc.append_slots(other, released * B)
        junk = torch.full((released * B, Hkv, d), float("nan"), dtype=torch.float16, device="cuda")
        cache.append(0, junk, junk, torch.tensor(slots, dtype=torch.int64, device="cuda"))
    bt, cl, got_lens = tables_for(alloc, seqs, max(1, max(-(-n // B) for n in lens)))
    assert got_lens == lens
    q = W.host_queries(w)
    kn = vn = None
    if fused:
        kn = torch.from_numpy(np.stack([k[-1] if len(k) else np.zeros((Hkv, d), np.float16) for k in ks])).cuda()
        vn = torch.from_numpy(np.stack([v[-1] if len(v) else np.zeros((Hkv, d), np.float16) for v in vs])).cuda()
    kd, vd = ks, vs
    if dtype == "fp8":
        kd = [OF.decode(OF.quantize(k, sc)) * float(sc) for k in ks]
        vd = [OF.decode(OF.quantize(v, sc)) * float(sc) for v in vs]
    want = OA.decode_attention_window(q, kd, vd, w.scale, window)
    return cache, q, bt, cl, kn, vn, want, released, w


@pytest.mark.parametrize("dtype,B,G", [("f16", 16, 1), ("f16", 8, 4), ("f16", 32, 1), ("fp8", 16, 2),
                                       ("fp8", 32, 8)])
@pytest.mark.parametrize("window", [1, 7, 40, 256])
def test_window_against_oracle_with_trimmed_blocks(dtype, B, G, window):
    cache, q, bt, cl, _, _, want, released, w = _case(dtype, B, G, window, 120 + window, fused=False)
    assert window > 300 or released > 0
    for P in (0, 32):
        out = cache.attention_ex(0, torch.from_numpy(q).cuda(), bt, cl, max(w.lens), w.scale,
                                 window=window, partition_tokens=P).cpu().numpy()
        assert np.all(np.isfinite(out))
        assert max_abs(out, want) <= tol_for("f16"), (P, max_abs(out, want))
    assert cache.device_error() == 0


@pytest.mark.parametrize("dtype,B,G", [("f16", 16, 1), ("fp8", 8, 4)])
def test_window_with_fused_append(dtype, B, G):
    cache, q, bt, cl, kn, vn, want, _, w = _case(dtype, B, G, 100, 131, fused=True)
    out = cache.attention_ex(0, torch.from_numpy(q).cuda(), bt, cl, max(w.lens), w.scale, window=100,
                             k_new=kn, v_new=vn).cpu().numpy()
    assert max_abs(out, want) <= tol_for("f16")
    assert cache.device_error() == 0


@pytest.mark.parametrize("dtype,B,G", [("f16", 16, 1), ("fp8", 16, 1), ("fp8", 16, 8), ("f16", 8, 4)])
def test_window_with_fused_append_and_all_launch_flags(dtype, B, G):
    """The window, the fused append and the four launch flags together, twice in a row
    on one zero-filled workspace (the second call rewrites the same slots)."""
    from paged_kv_cache_169_gb300 import abi
    cache, q, bt, cl, kn, vn, want, _, w = _case(dtype, B, G, 100, 151 + G, fused=True)
    flags = (abi.KV_DECODE_WORKSPACE_ZEROED | abi.KV_DECODE_PDL | abi.KV_DECODE_EARLY_TABLES |
             abi.KV_DECODE_EARLY_POOL)
    ws = cache.zeroed_workspace(w.batch, max(w.lens), 0, num_q_heads=w.q_heads, window=100)
    for _ in range(2):
        out = cache.attention_ex(0, torch.from_numpy(q).cuda(), bt, cl, max(w.lens), w.scale, window=100,
                                 k_new=kn, v_new=vn, workspace=ws, flags=flags).cpu().numpy()
        assert max_abs(out, want) <= tol_for("f16")
    assert cache.device_error() == 0


def test_no_window_equals_plain_entry():
    cache, q, bt, cl, _, _, _, _, w = _case("f16", 16, 1, 10 ** 6, 140, fused=False)
    qt = torch.from_numpy(q).cuda()
    a = cache.attention(0, qt, bt, cl, max(w.lens), w.scale)
    b = cache.attention_ex(0, qt, bt, cl, max(w.lens), w.scale, window=0)
    c = cache.attention_ex(0, qt, bt, cl, max(w.lens), w.scale, window=10 ** 6)
    assert torch.equal(a, b) and torch.equal(a, c)
