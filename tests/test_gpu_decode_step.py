"""GPU: kv_decode_step, one decode step of a batch in one C call (slot reservation with
copy-on-write, tables and lengths, host-to-device copies, block copies, the fused append +
attention, the copy of the result back).

The same steps are also driven call by call through the C ABI (kv_alloc_decode_step,
kv_alloc_build_tables, kv_copy_blocks, paged_decode_attention_ex) on a second, identical
cache and allocator: every step's output, the final pools and the final tables must be
bit-identical, and the outputs must match the float64 oracle.  The batch is parallel
sampling's shape in small: candidates forked from one prompt whose last block is shared,
so the first step plans copies ([PagedAttention] §3.3, §5.1).
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import max_abs, poison, tol_for
from oracle import attention as OA
from paged_kv_cache_169_gb300 import abi, build
from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

pytestmark = pytest.mark.gpu

H, D, B = 4, 128, 16
PROMPT, CANDS, STEPS = 70, 4, 20          # 70 tokens: the prompt's last block is partly filled


def _setup(seed):
    nb = 64
    w = W.Workload("decode_step", seed, 1, H, D, B, "f16", CANDS, [PROMPT] * CANDS, nb, 1 / math.sqrt(D))
    cache = PagedKVCache(1, nb, B, H, D, "f16")
    poison(cache)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    root = alloc.new_seq()
    pk, pv = W.host_tokens(w, 0, PROMPT, "k"), W.host_tokens(w, 0, PROMPT, "v")
    slots, _ = alloc.append_slots(root, PROMPT)
    cache.append(0, torch.from_numpy(pk).cuda(), torch.from_numpy(pv).cuda(), torch.tensor(slots, device="cuda"))
    seqs = [root] + [alloc.fork(root) for _ in range(CANDS - 1)]
    g = np.random.default_rng(seed + 1)
    qkv = g.standard_normal((STEPS, 3, CANDS, H, D)).astype(np.float16)
    return w, cache, alloc, seqs, pk, pv, qkv


def _args(cache, ws, d_meta, d_qkv, d_out, n, max_blocks, max_ctx, scale, stream):
    a = abi.kv_decode_args()
    a.layer, a.q, a.num_q_heads = 0, d_qkv[0].data_ptr(), 0
    a.k_new, a.v_new, a.in_dtype = d_qkv[1].data_ptr(), d_qkv[2].data_ptr(), abi.KV_F16
    a.out, a.block_tables, a.max_blocks_per_seq = d_out.data_ptr(), d_meta.data_ptr(), max_blocks
    a.context_lens, a.batch, a.max_context = d_meta.data_ptr() + 4 * n * max_blocks, n, max_ctx
    a.scale, a.partition_tokens = float(scale), 0
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    a.stream = stream.cuda_stream
    a.flags = abi.KV_DECODE_WORKSPACE_ZEROED | abi.KV_DECODE_PDL
    return a


def _run(one_call: bool, seed: int, merged: bool = False):
    """The STEPS decode steps, through kv_decode_step or call by call.  merged: the inputs
    follow the staging data in one pinned row and one device buffer (a single copy)."""
    w, cache, alloc, seqs, pk, pv, qkv = _setup(seed)
    n, max_blocks = CANDS, -(-(PROMPT + STEPS) // B)
    max_ctx = PROMPT + STEPS
    width = n * max_blocks + 3 * n
    stream = torch.cuda.Stream()
    pin_meta = torch.empty((STEPS, width), dtype=torch.int32).pin_memory()
    pin_qkv = torch.from_numpy(qkv).pin_memory()
    pin_out = torch.empty((STEPS, n, H, D), dtype=torch.float32).pin_memory()
    d_meta = torch.empty(width, dtype=torch.int32, device="cuda")
    d_qkv = torch.empty((3, n, H, D), dtype=torch.float16, device="cuda")
    off = (width * 4 + 255) // 256 * 256
    qkv_bytes = 3 * n * H * D * 2
    if merged:
        rows = torch.empty((STEPS, off + qkv_bytes), dtype=torch.uint8).pin_memory()
        for i in range(STEPS):
            rows[i, off:].view(torch.float16).view(3, n, H, D).copy_(pin_qkv[i])
        d_row = torch.empty(off + qkv_bytes, dtype=torch.uint8, device="cuda")
        d_meta = d_row[:width * 4].view(torch.int32)
        d_qkv = d_row[off:].view(torch.float16).view(3, n, H, D)
    d_out = torch.empty((n, H, D), dtype=torch.float32, device="cuda")
    ws = cache.zeroed_workspace(n, max_ctx)
    a = _args(cache, ws, d_meta, d_qkv, d_out, n, max_blocks, max_ctx, w.scale, stream)
    seq_arr = (ctypes.c_int32 * n)(*seqs)
    copies = 0
    with torch.cuda.stream(stream):
        for i in range(STEPS):
            row = pin_meta[i]
            base = row.data_ptr()
            if one_call and merged:
                r = rows[i].data_ptr()
                copies += abi.kv_decode_step(alloc.handle, cache.handle, seq_arr, n, max_blocks, r,
                                             d_row.data_ptr(), r + off, d_row.data_ptr() + off, qkv_bytes,
                                             pin_out[i].data_ptr(), d_out.numel() * 4, a)
            elif one_call:
                copies += abi.kv_decode_step(alloc.handle, cache.handle, seq_arr, n, max_blocks, base,
                                             d_meta.data_ptr(), pin_qkv[i].data_ptr(), d_qkv.data_ptr(), qkv_bytes,
                                             pin_out[i].data_ptr(), d_out.numel() * 4, a)
            else:
                slots = (ctypes.c_int64 * n)()
                n_cow = abi.kv_alloc_decode_step(alloc.handle, seq_arr, n, slots, base + 4 * (n * max_blocks + n))
                abi.kv_alloc_build_tables_into(alloc.handle, seq_arr, n, base, max_blocks, base + 4 * n * max_blocks)
                d_meta.copy_(row, non_blocking=True)
                d_qkv.copy_(pin_qkv[i], non_blocking=True)
                if n_cow:
                    abi.kv_copy_blocks(cache.handle, d_meta.data_ptr() + 4 * (n * max_blocks + n), n_cow, 0, 1,
                                       a.stream)
                    copies += n_cow
                abi.paged_decode_attention_ex(cache.handle, a)
                pin_out[i].copy_(d_out, non_blocking=True)
    stream.synchronize()
    tabs, lens = alloc.build_tables(seqs, max_blocks)
    res = dict(out=pin_out.clone().numpy(), k=cache.k[0].clone(), v=cache.v[0].clone(), tabs=tabs, lens=lens,
               copies=copies, err=cache.device_error(), w=w, pk=pk, pv=pv, qkv=qkv)
    cache.close()
    alloc.close()
    return res


@pytest.mark.parametrize("merged", [False, True])
def test_decode_step_matches_the_call_by_call_path_and_the_oracle(merged):
    build.build()
    one = _run(True, 801, merged)
    ref = _run(False, 801)
    assert one["err"] == 0 and ref["err"] == 0
    assert one["copies"] == ref["copies"] == CANDS - 1        # all but the last sharer copy
    assert np.array_equal(one["out"], ref["out"])              # every step, bit for bit
    assert torch.equal(one["k"].view(torch.int16), ref["k"].view(torch.int16))
    assert torch.equal(one["v"].view(torch.int16), ref["v"].view(torch.int16))
    assert one["tabs"] == ref["tabs"] and one["lens"] == ref["lens"]
    # against the oracle: candidate c at step i attends the prompt and its own tokens 0..i
    qkv, w = one["qkv"], one["w"]
    worst = 0.0
    for i in range(STEPS):
        ks = [np.concatenate([one["pk"], qkv[: i + 1, 1, c]]) for c in range(CANDS)]
        vs = [np.concatenate([one["pv"], qkv[: i + 1, 2, c]]) for c in range(CANDS)]
        want = OA.decode_attention(qkv[i, 0], ks, vs, w.scale)
        worst = max(worst, max_abs(one["out"][i], want))
    assert worst <= tol_for("f16"), worst


def test_decode_step_refuses_before_reserving():
    build.build()
    w, cache, alloc, seqs, pk, pv, qkv = _setup(803)
    n = CANDS
    max_blocks = PROMPT // B                                   # 4 blocks: no room for 71 tokens
    width = n * (max_blocks + 1) + 3 * n
    stream = torch.cuda.Stream()
    pin = torch.empty(width, dtype=torch.int32).pin_memory()
    d_meta = torch.empty(width, dtype=torch.int32, device="cuda")
    d_qkv = torch.zeros((3, n, H, D), dtype=torch.float16, device="cuda")
    d_out = torch.zeros((n, H, D), dtype=torch.float32, device="cuda")
    ws = cache.zeroed_workspace(n, PROMPT + 1)
    seq_arr = (ctypes.c_int32 * n)(*seqs)
    before = alloc.build_tables(seqs, max_blocks + 1)
    a = _args(cache, ws, d_meta, d_qkv, d_out, n, max_blocks, PROMPT + 1, w.scale, stream)
    with pytest.raises(abi.KvError) as e:                      # a table would not fit
        abi.kv_decode_step(alloc.handle, cache.handle, seq_arr, n, max_blocks, pin.data_ptr(), d_meta.data_ptr(),
                           0, 0, 0, 0, 0, a)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
    a = _args(cache, ws, d_meta, d_qkv, d_out, n, max_blocks + 1, PROMPT + 1, w.scale, stream)
    a.batch = n - 1                                            # args describe another batch
    with pytest.raises(abi.KvError) as e:
        abi.kv_decode_step(alloc.handle, cache.handle, seq_arr, n, max_blocks + 1, pin.data_ptr(),
                           d_meta.data_ptr(), 0, 0, 0, 0, 0, a)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
    a.batch = n
    a.flags |= abi.KV_DECODE_EARLY_TABLES                       # tables are copied just before
    with pytest.raises(abi.KvError) as e:
        abi.kv_decode_step(alloc.handle, cache.handle, seq_arr, n, max_blocks + 1, pin.data_ptr(),
                           d_meta.data_ptr(), 0, 0, 0, 0, 0, a)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
    assert alloc.build_tables(seqs, max_blocks + 1) == before  # nothing was reserved
    torch.cuda.synchronize()
    assert float(d_out.abs().sum()) == 0.0                     # nothing was launched
    cache.close()
    alloc.close()
