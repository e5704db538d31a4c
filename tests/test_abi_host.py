"""C-ABI library: builds, loads, exports every declared symbol; host-only entry points
(the block allocator, argument validation) checked on the CPU.

The allocator is compared with the oracle's block manager on the same inputs (same
initial free list, same operation sequence): block ids, slots, copy pairs, reference
counts and free lists must be identical (integer work: bit-exact).
"""

import copy
import ctypes as C
import os
import re

import numpy as np
import pytest

from oracle import cache as OC
from paged_kv_cache_169_gb300 import abi, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kvpaged.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    return re.findall(r"^KV_API\s+[\w\s\*]+?\b(\w+)\(", text, flags=re.M)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(abi._SIGS), "binding and header must list the same entry points"


def test_header_constants_match_the_binding():
    """Every #define KV_* with an integer value in the header equals the binding's constant
    of the same name (the flags and status codes cross the ABI as plain integers)."""
    text = open(HEADER, encoding="utf-8").read()
    defs = dict(re.findall(r"^#define\s+(KV_[A-Z0-9_]+)\s+\(?(-?\d+)u?\)?\s*$", text, flags=re.M))
    assert {"KV_DECODE_WORKSPACE_ZEROED", "KV_DECODE_PDL", "KV_DECODE_EARLY_TABLES",
            "KV_DECODE_OUT_F16", "KV_DECODE_EARLY_POOL"} <= set(defs)
    for name, value in defs.items():
        if hasattr(abi, name):
            assert getattr(abi, name) == int(value), name
    flags = [int(defs[n]) for n in defs if n.startswith("KV_DECODE_")]
    assert sum(flags) == 31 and all(f & (f - 1) == 0 for f in flags)   # distinct bits


def test_status_strings(lib):
    assert abi.kv_status_str(0) == "ok"
    assert abi.kv_status_str(abi.KV_ERR_NO_BLOCKS) == "no free blocks"
    assert abi.kv_status_str(12345) == "unknown status"
    assert abi.kv_version() >= 100


def test_selftest_entry_validates_before_any_device_call(lib):
    with pytest.raises(abi.KvError) as e:
        abi.kv_selftest_wait_timeout(0, 1000)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
    assert abi.KV_FEATURE_TENSOR_MAPS == 1
    with pytest.raises(abi.KvError):
        abi.kv_pool_features(0)


def test_pool_create_rejects_bad_descriptors_without_a_gpu(lib):
    bad = [dict(head_dim=96), dict(block_size=12), dict(num_heads=0), dict(num_layers=0),
           dict(num_blocks=0), dict(dtype=7)]
    base = dict(num_layers=1, num_blocks=4, block_size=16, num_heads=2, head_dim=64, dtype=abi.KV_F16)
    for b in bad:
        d = {**base, **b}
        with pytest.raises(abi.KvError) as e:
            abi.kv_pool_create(d["num_layers"], d["num_blocks"], d["block_size"], d["num_heads"],
                               d["head_dim"], d["dtype"], [256] * max(d["num_layers"], 1),
                               [256] * max(d["num_layers"], 1))
        assert e.value.status == abi.KV_ERR_INVALID_ARG
    # misaligned pointer, and FP8 without scales, are refused before any device call
    with pytest.raises(abi.KvError):
        abi.kv_pool_create(1, 4, 16, 2, 64, abi.KV_F16, [258], [256])
    with pytest.raises(abi.KvError):
        abi.kv_pool_create(1, 4, 16, 2, 64, abi.KV_FP8_E4M3, [256], [256])
    with pytest.raises(abi.KvError):
        abi.kv_pool_create(1, 4, 16, 2, 64, abi.KV_F16, [256], [256], [512], [512])


def _run_both(num_blocks, B, order, ops):
    """Apply the same operations to the C allocator and the oracle model."""
    a = abi.kv_alloc_create(num_blocks, B, order)
    m = OC.BlockManager(num_blocks, B, free_order=order)
    ids = {}
    try:
        for op in ops:
            kind = op[0]
            if kind == "new":
                ids[op[1]] = (abi.kv_alloc_seq_new(a), m.new_seq())
            elif kind == "fork":
                ids[op[2]] = (abi.kv_alloc_seq_fork(a, ids[op[1]][0]), m.fork(ids[op[1]][1]))
            elif kind == "append":
                ca, cm = ids[op[1]]
                try:
                    slots_m, cows_m = m.append_slots(cm, op[2])
                    ok_m = True
                except OC.OutOfBlocks:
                    ok_m = False
                try:
                    slots_a, cow_a = abi.kv_alloc_append_slots(a, ca, op[2])
                    ok_a = True
                except abi.KvError as e:
                    assert e.status == abi.KV_ERR_NO_BLOCKS
                    ok_a = False
                assert ok_a == ok_m
                if ok_a:
                    assert slots_a == slots_m
                    assert ([cow_a] if cow_a else []) == [tuple(c) for c in cows_m]
            elif kind == "step":                     # one slot for each listed sequence
                names = op[1]
                snap = copy.deepcopy(m)
                slots_m, cows_m, ok_m = [], [], True
                try:
                    for nm in names:
                        sl, cw = m.append_slots(ids[nm][1], 1)
                        slots_m += sl
                        cows_m += [tuple(c) for c in cw]
                except OC.OutOfBlocks:
                    ok_m = False
                    m = snap                         # the batch call changes nothing on failure
                n = len(names)
                seq_arr = (C.c_int32 * max(n, 1))(*[ids[nm][0] for nm in names])
                slots = (C.c_int64 * max(n, 1))()
                pairs = (C.c_int32 * max(2 * n, 2))()
                try:
                    n_cow = abi.kv_alloc_decode_step(a, seq_arr, n, slots, pairs)
                    ok_a = True
                except abi.KvError as e:
                    assert e.status == abi.KV_ERR_NO_BLOCKS
                    ok_a = False
                assert ok_a == ok_m
                if ok_a:
                    assert list(slots)[:n] == slots_m
                    assert [(pairs[2 * i], pairs[2 * i + 1]) for i in range(n_cow)] == cows_m
            elif kind == "free":
                ca, cm = ids.pop(op[1])
                abi.kv_alloc_seq_free(a, ca)
                m.free_seq(cm)
            elif kind == "trim":                     # keep the last op[2] tokens
                ca, cm = ids[op[1]]
                keep_from = max(0, m.lens[cm] - op[2])
                n = abi.kv_alloc_seq_trim(a, ca, keep_from)
                assert n == len(m.trim(cm, keep_from))
            # state comparison after every operation
            assert abi.kv_alloc_free_list(a, num_blocks) == m.free
            assert [abi.kv_alloc_ref_count(a, b) for b in range(num_blocks)] == m.ref
            for name, (ca, cm) in ids.items():
                assert abi.kv_alloc_block_table(a, ca) == m.table(cm)
                assert abi.kv_alloc_seq_info(a, ca) == (m.lens[cm], len(m.table(cm)))
        st = abi.kv_alloc_stats(a)
        assert st.free_blocks == len(m.free) and st.shared_blocks == m.shared_blocks()
        assert st.num_seqs == len(ids)
        assert st.used_slots == sum(m.lens[cm] - m.table(cm).count(-1) * B for _, cm in ids.values())
        assert st.wasted_slots == sum(len(m.table(cm)) * B - m.lens[cm] for _, cm in ids.values())
    finally:
        abi.kv_alloc_destroy(a)


@pytest.mark.parametrize("batched", [False, True])
def test_allocator_matches_oracle_parallel_sampling(lib, batched):
    """128 decode steps of 8 candidates forked from a 1030-token prompt, one slot per
    candidate per step: per sequence, or with one kv_alloc_decode_step call per step."""
    ops = [("new", "p"), ("append", "p", 1030)]
    ops += [("fork", "p", f"c{i}") for i in range(1, 8)]
    names = ["p"] + [f"c{i}" for i in range(1, 8)]
    for _ in range(128):
        ops += [("step", names)] if batched else [("append", n, 1) for n in names]
    ops += [("free", n) for n in names]
    _run_both(200, 16, np.random.default_rng(4).permutation(200).tolist(), ops)


def test_allocator_matches_oracle_random_ops(lib):
    rng = np.random.default_rng(11)
    for B in (8, 16, 32):
        nb = 120
        ops, live, k = [("new", 0)], [0], 1
        for _ in range(400):
            r = rng.integers(10)
            if r < 6:
                ops.append(("append", live[int(rng.integers(len(live)))], int(rng.integers(1, 40))))
            elif r < 7:
                ops.append(("fork", live[int(rng.integers(len(live)))], k))
                live.append(k)
                k += 1
            elif r < 8 and len(live) > 1 and rng.integers(2):
                ops.append(("free", live.pop(int(rng.integers(len(live))))))
            elif r < 9:
                ops.append(("trim", live[int(rng.integers(len(live)))], int(rng.integers(1, 60))))
            elif rng.integers(2):                    # a decode step over some live sequences
                pick = rng.permutation(len(live))[:int(rng.integers(1, len(live) + 1))]
                ops.append(("step", [live[int(i)] for i in pick]))
            else:
                ops.append(("new", k))
                live.append(k)
                k += 1
        _run_both(nb, B, rng.permutation(nb).tolist(), ops)


def test_allocator_errors(lib):
    a = abi.kv_alloc_create(4, 8)
    try:
        s = abi.kv_alloc_seq_new(a)
        abi.kv_alloc_append_slots(a, s, 32)
        with pytest.raises(abi.KvError) as e:
            abi.kv_alloc_append_slots(a, s, 1)
        assert e.value.status == abi.KV_ERR_NO_BLOCKS
        assert abi.kv_alloc_seq_info(a, s) == (32, 4)        # unchanged
        with pytest.raises(abi.KvError) as e:
            abi.kv_alloc_seq_free(a, 999)
        assert e.value.status == abi.KV_ERR_STATE
        with pytest.raises(abi.KvError):
            abi.kv_alloc_append_slots(a, s, 0)
        with pytest.raises(abi.KvError):
            abi.kv_alloc_seq_trim(a, s, 33)                   # beyond the length
        with pytest.raises(abi.KvError):
            abi.kv_alloc_build_tables(a, [s], 3)              # table longer than max_blocks
        tabs, lens = abi.kv_alloc_build_tables(a, [s], 6)
        assert lens == [32] and tabs[0][4:] == [-1, -1]
        # a decode step with an unknown sequence changes nothing
        before = abi.kv_alloc_free_list(a, 4)
        with pytest.raises(abi.KvError) as e:
            abi.kv_alloc_decode_step(a, (C.c_int32 * 2)(s, 999), 2, (C.c_int64 * 2)(), (C.c_int32 * 4)())
        assert e.value.status == abi.KV_ERR_STATE
        assert abi.kv_alloc_seq_info(a, s) == (32, 4) and abi.kv_alloc_free_list(a, 4) == before
        abi.kv_alloc_seq_free(a, s)
        assert sorted(abi.kv_alloc_free_list(a, 4)) == [0, 1, 2, 3]
        with pytest.raises(abi.KvError) as e:
            abi.kv_alloc_seq_free(a, s)                       # double free
        assert e.value.status == abi.KV_ERR_STATE
    finally:
        abi.kv_alloc_destroy(a)
    with pytest.raises(abi.KvError):
        abi.kv_alloc_create(4, 8, [0, 1, 1, 2])               # not a permutation


def test_decode_step_is_all_or_nothing(lib):
    """A decode step whose blocks do not all fit changes nothing; one sharer of a block
    copies and the last sharer writes in place, within one step as across steps."""
    a = abi.kv_alloc_create(5, 8)
    try:
        s0 = abi.kv_alloc_seq_new(a)
        abi.kv_alloc_append_slots(a, s0, 12)                 # blocks: 2 (the second half full)
        s1 = abi.kv_alloc_seq_fork(a, s0)                    # shares both
        s2 = abi.kv_alloc_seq_new(a)
        abi.kv_alloc_append_slots(a, s2, 16)                 # 2 more blocks, 1 free left
        free = abi.kv_alloc_free_list(a, 5)
        seqs = (C.c_int32 * 3)(s0, s1, s2)
        slots, pairs = (C.c_int64 * 3)(), (C.c_int32 * 6)()
        # s0 copies the shared half block (1), s1 then writes in place, s2 needs a new
        # block (1): 2 blocks, 1 free
        with pytest.raises(abi.KvError) as e:
            abi.kv_alloc_decode_step(a, seqs, 3, slots, pairs)
        assert e.value.status == abi.KV_ERR_NO_BLOCKS
        assert abi.kv_alloc_free_list(a, 5) == free
        assert [abi.kv_alloc_seq_info(a, s) for s in (s0, s1, s2)] == [(12, 2), (12, 2), (16, 2)]
        # without s2 it fits: one copy planned, for s0
        n = abi.kv_alloc_decode_step(a, seqs, 2, slots, pairs)
        assert n == 1 and pairs[1] == free[0]
        shared_last = abi.kv_alloc_block_table(a, s1)[-1]
        assert pairs[0] == shared_last and abi.kv_alloc_ref_count(a, shared_last) == 1
        assert slots[0] == pairs[1] * 8 + 4 and slots[1] == shared_last * 8 + 4
    finally:
        abi.kv_alloc_destroy(a)


def test_decode_step_entry_refuses_missing_arguments(lib):
    """kv_decode_step checks its pointers before touching the allocator or the device: with
    no pool (or no argument block) it returns KV_ERR_INVALID_ARG and reserves nothing."""
    a = abi.kv_alloc_create(4, 8)
    try:
        s0 = abi.kv_alloc_seq_new(a)
        abi.kv_alloc_append_slots(a, s0, 3)
        seqs = (C.c_int32 * 1)(s0)
        staging = (C.c_int32 * 8)()
        args = abi.kv_decode_args()
        f = lib.kv_decode_step
        assert f(a, None, seqs, 1, 2, C.addressof(staging), 1 << 20, None, None, 0, None, 0,
                 C.byref(args)) == abi.KV_ERR_INVALID_ARG
        assert f(a, None, seqs, 1, 2, C.addressof(staging), 1 << 20, None, None, 0, None, 0,
                 None) == abi.KV_ERR_INVALID_ARG                     # no argument block
        assert f(None, None, seqs, 1, 2, None, None, None, None, 0, None, 0,
                 C.byref(args)) == abi.KV_ERR_INVALID_ARG            # no allocator, no staging
        assert abi.kv_alloc_seq_info(a, s0) == (3, 1)                 # nothing reserved
    finally:
        abi.kv_alloc_destroy(a)
