"""Pins for the oracle's paged pool model and block manager (CPU only)."""

import math
import os

import numpy as np
import pytest

import workloads as W
from oracle import cache as C

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms_kv_sizes.txt")


def _closed_forms():
    out = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = int(v)
    return out


def test_kv_size_closed_forms_match_workload_shapes():
    cf = _closed_forms()
    # bytes per token over all layers: layers * 2 (K,V) * heads * dim * 2 bytes
    assert 32 * 2 * 32 * 128 * 2 == cf["llama7b_bytes_per_token"]
    w = W.llama13b()
    per_seq = w.num_layers * 2 * w.num_heads * 2048 * w.head_dim * w.elem_bytes
    assert per_seq == cf["llama13b_bytes_per_seq_2048"]
    # the 13B pool holds exactly batch * 2048 tokens per layer
    assert w.num_blocks * w.block_size == w.batch * 2048
    assert cf["blocks_for_1024_at_b16"] == 1024 // 16
    assert cf["max_waste_tokens_b16"] == 16 - 1


def test_parallel_sampling_counts_match_page_arithmetic():
    """Prompt 1024 + 8 x 128 generated: shared blocks hold 2048 token slots, unshared 9216."""
    cf = _closed_forms()
    B = 16
    m = C.BlockManager(num_blocks=200, block_size=B)
    root = m.new_seq()
    m.append_slots(root, 1024)
    kids = [root] + [m.fork(root) for _ in range(7)]
    for _ in range(128):
        for s in kids:
            m.append_slot(s)
    assert m.used_blocks() * B == cf["parallel_shared_token_slots"]
    assert sum(-(-m.lens[s] // B) for s in kids) * B == cf["parallel_unshared_token_slots"]


def test_parallel_sampling_1030_prompt_cow_count():
    """1030-token prompt (last block 6/16 full) shared by 8: the first append of the
    first 7 candidates copies the partial block; the last writes in place."""
    B = 16
    m = C.BlockManager(num_blocks=200, block_size=B)
    root = m.new_seq()
    m.append_slots(root, 1030)
    cands = [root] + [m.fork(root) for _ in range(7)]
    assert all(m.ref[b] == 8 for b in m.table(root))
    cows = []
    for s in cands:
        slot, cow = m.append_slot(s)
        cows.append(cow)
    assert sum(c is not None for c in cows) == 7 and cows[-1] is None
    last = m.table(root)[-1]
    for s, cow in zip(cands[:-1], cows[:-1]):
        assert cow[0] == m.table(cands[-1])[-1]          # all copied from the original
    for _ in range(127):
        for s in cands:
            m.append_slot(s)
    assert all(m.lens[s] == 1158 for s in cands)
    assert all(len(m.table(s)) == 73 for s in cands)
    assert m.used_blocks() == 64 + 8 * 9 == 136
    assert 8 * 73 == 584
    for s in cands:
        m.free_seq(s)
    assert m.used_blocks() == 0 and all(r == 0 for r in m.ref)
    del last


def test_table_length_is_ceil_len_over_b():
    rng = np.random.default_rng(1)
    for B in (8, 16, 32):
        m = C.BlockManager(num_blocks=400, block_size=B)
        seqs = [m.new_seq() for _ in range(6)]
        for _ in range(300):
            s = seqs[int(rng.integers(len(seqs)))]
            m.append_slots(s, int(rng.integers(1, 9)))
        for s in seqs:
            assert len(m.table(s)) == -(-m.lens[s] // B)
        assert m.used_blocks() == sum(-(-m.lens[s] // B) for s in seqs)


def test_out_of_blocks_leaves_state_unchanged():
    m = C.BlockManager(num_blocks=4, block_size=8)
    s = m.new_seq()
    m.append_slots(s, 30)
    before = (list(m.free), list(m.ref), m.table(s), m.lens[s])
    with pytest.raises(C.OutOfBlocks):
        m.append_slots(s, 3)
    assert (list(m.free), list(m.ref), m.table(s), m.lens[s]) == before


def test_random_ops_keep_every_sequence_readable():
    """Semantic model: a sequence is the list of token ids appended to it (forks copy
    the list).  Writing token ids through the block manager's slots into a pool,
    applying every planned copy first, must read back each sequence's own list."""
    rng = np.random.default_rng(2)
    B, nb = 4, 300
    m = C.BlockManager(nb, B, free_order=rng.permutation(nb))
    pool = np.full((nb, 1, B, 1), -1, dtype=np.int64)
    model = {}
    tok = 0
    live = [m.new_seq()]
    model[live[0]] = []
    for _ in range(1500):
        op = rng.integers(10)
        if op < 7 and live:
            s = live[int(rng.integers(len(live)))]
            n = int(rng.integers(1, 6))
            if m.blocks_needed(s, n) > len(m.free):
                continue
            slots, cows = m.append_slots(s, n)
            C.copy_blocks([pool], np.array(cows, dtype=np.int64).reshape(-1, 2))
            ids = np.arange(tok, tok + n).reshape(n, 1, 1)
            C.append(pool, pool.copy(), ids, ids, slots, B)   # K pool only is checked
            model[s] += list(range(tok, tok + n))
            tok += n
        elif op < 8 and live:
            p = live[int(rng.integers(len(live)))]
            c = m.fork(p)
            model[c] = list(model[p])
            live.append(c)
        elif op < 9 and len(live) > 1:
            s = live.pop(int(rng.integers(len(live))))
            m.free_seq(s)
            del model[s]
        else:
            s = m.new_seq()
            model[s] = []
            live.append(s)
        for s in live:
            table, n = m.table(s), m.lens[s]
            got = [int(pool[table[t // B], 0, t % B, 0]) for t in range(n)]
            assert got == model[s]
        # every block in use has exactly as many references as tables holding it
        counts = np.zeros(nb, dtype=np.int64)
        for s in live:
            for b in m.table(s):
                counts[b] += 1
        assert counts.tolist() == m.ref
        assert sorted(m.free + [b for b in range(nb) if m.ref[b] > 0]) == list(range(nb))


def test_append_and_copy_preserve_bits():
    rng = np.random.default_rng(3)
    B, H, d, nb = 16, 2, 8, 6
    kp = np.full((nb, H, B, d), np.nan, dtype=np.float16)
    vp = np.full((nb, H, B, d), np.nan, dtype=np.float16)
    k = rng.standard_normal((5, H, d)).astype(np.float16)
    v = rng.standard_normal((5, H, d)).astype(np.float16)
    slots = np.array([3 * B + 0, -1, 3 * B + 15, 0, 5 * B + 7], dtype=np.int64)
    C.append(kp, vp, k, v, slots, B)
    assert np.array_equal(kp[3, :, 0].view(np.uint16), k[0].view(np.uint16))
    assert np.array_equal(vp[5, :, 7].view(np.uint16), v[4].view(np.uint16))
    assert np.isnan(kp[1]).all()                         # the -1 slot wrote nowhere
    C.copy_blocks([kp, vp], np.array([[3, 1], [5, 2]]))
    assert np.array_equal(kp[1].view(np.uint16), kp[3].view(np.uint16))   # NaN slots too
    assert np.array_equal(vp[2].view(np.uint16), vp[5].view(np.uint16))


def test_fp8_append_uses_the_block_scale():
    from oracle import fp8
    rng = np.random.default_rng(4)
    B, H, d, nb = 8, 2, 16, 4
    kc = np.zeros((nb, H, B, d), dtype=np.uint8)
    vc = np.zeros((nb, H, B, d), dtype=np.uint8)
    ks = np.array([1.0, 0.01, 0.5, 2.0], dtype=np.float32)
    vs = np.array([0.25, 1.0, 4.0, 0.1], dtype=np.float32)
    k = rng.standard_normal((2, H, d)).astype(np.float16)
    v = rng.standard_normal((2, H, d)).astype(np.float16)
    C.append_fp8(kc, vc, k, v, np.array([1 * B + 2, 3 * B + 7]), B, ks, vs, fp8.quantize)
    assert np.array_equal(kc[1, :, 2], fp8.quantize(k[0], ks[1]))
    assert np.array_equal(vc[3, :, 7], fp8.quantize(v[1], vs[3]))
    assert math.isclose(float(fp8.decode(kc[1, 0, 2, 0])) * 0.01, float(k[0, 0, 0]), rel_tol=0.07)


def test_trim_releases_only_blocks_wholly_before_the_window():
    m = C.BlockManager(num_blocks=20, block_size=8)
    s = m.new_seq()
    m.append_slots(s, 45)                    # 6 blocks, the last with 5 tokens
    t = m.table(s)
    released = m.trim(s, 45 - 20)            # keep tokens 25..44: blocks 0..2 (tokens 0..23) go
    assert released == t[:3] and m.table(s)[:3] == [-1, -1, -1] and m.table(s)[3:] == t[3:]
    assert m.used_blocks() == 3 and m.lens[s] == 45
    assert m.trim(s, 25) == []               # idempotent
    c = m.fork(s)                            # a fork shares only the live blocks
    assert all(m.ref[b] == 2 for b in t[3:])
    m.free_seq(s)
    m.free_seq(c)
    assert m.used_blocks() == 0 and all(r == 0 for r in m.ref)


def test_swap_round_trip_and_layout():
    rng = np.random.default_rng(6)
    L, nb, H, B, d = 3, 7, 2, 4, 8
    kp = [rng.standard_normal((nb, H, B, d)).astype(np.float16) for _ in range(L)]
    vp = [rng.standard_normal((nb, H, B, d)).astype(np.float16) for _ in range(L)]
    ks = [rng.uniform(0.1, 1, nb).astype(np.float32) for _ in range(L)]
    vs = [rng.uniform(0.1, 1, nb).astype(np.float32) for _ in range(L)]
    blocks = [5, 0, 3]
    img = C.swap_out(kp, vp, blocks, ks, vs)
    blk = H * B * d * 2
    assert img.size == len(blocks) * L * 2 * blk + len(blocks) * L * 2 * 4
    # block 0 of the list, layer 1, V part sits at (0*L + 1)*2 + 1 block slots
    off = ((0 * L + 1) * 2 + 1) * blk
    assert np.array_equal(img[off:off + blk].view(np.float16).reshape(H, B, d), vp[1][5])
    # scales: list block 2 (physical 3), layer 2, K then V
    sc = img[len(blocks) * L * 2 * blk:].view(np.float32)
    assert sc[(2 * L + 2) * 2] == ks[2][3] and sc[(2 * L + 2) * 2 + 1] == vs[2][3]
    # round trip into other blocks, nothing else touched
    before = [p.copy() for p in kp + vp]
    C.swap_in(kp, vp, [1, 2, 6], img, ks, vs)
    for l in range(L):
        for src, dst in zip(blocks, [1, 2, 6]):
            assert np.array_equal(kp[l][dst].view(np.uint16), before[l][src].view(np.uint16))
            assert np.array_equal(vp[l][dst].view(np.uint16), before[L + l][src].view(np.uint16))
            assert ks[l][dst] == ks[l][src] and vs[l][dst] == vs[l][src]
        assert np.array_equal(kp[l][4], before[l][4])
