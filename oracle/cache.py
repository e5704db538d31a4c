"""Oracle: the paged KV pool and its block manager as plain arrays and lists.

Test infrastructure only (see package doc).

Pool layout (one layer): ``pool[num_blocks, H, B, d]`` — a physical block holds B
token slots for every head.  Slot id ``= physical_block * B + offset``.

[PagedAttention] §2.1: a sequence's logical blocks map to non-contiguous
physical blocks through its block table; blocks are fixed-size allocation
units; different sequences can share physical blocks.
[PagedAttention] §3.1: a global physical-block pool, per-sequence block
tables, and first-fit allocation (for fixed-size blocks first fit is "take the
first block on the free list").
[PagedAttention] §3.3: every physical block has a reference count,
``ref_count > 1`` means shared; a write into a shared block first allocates a new
block, copies the whole block, decrements the old block's count and points the
sequence's table at the copy; then it writes.
[KV Cache篇] §3.1: the new token's K/V is written into the cache at position
``start_pos`` before attention reads ``[:start_pos + 1]``.
"""

from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# slot-mapped append and block copy: plain array copies
# --------------------------------------------------------------------------

def append(k_pool, v_pool, k, v, slot_mapping, block_size: int) -> None:
    """Write token i's K/V (``k[i, h, :]``) into slot ``slot_mapping[i]`` of every head.

    Slots < 0 are padding and skipped.  The copy keeps the bit pattern (same dtype).
    """
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        k_pool[blk, :, off, :] = k[i]
        v_pool[blk, :, off, :] = v[i]


def append_fp8(k_codes, v_codes, k, v, slot_mapping, block_size: int,
               k_block_scale, v_block_scale, quantize) -> None:
    """FP8 append: the slot receives ``quantize(x, scale[block])`` (see ``fp8.quantize``)."""
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        k_codes[blk, :, off, :] = quantize(k[i], k_block_scale[blk])
        v_codes[blk, :, off, :] = quantize(v[i], v_block_scale[blk])


def copy_blocks(pools, pairs, scales=()) -> None:
    """For each ``(src, dst)``: ``pool[dst] = pool[src]`` for every array given.

    ``pools`` is a list of [num_blocks, ...] arrays (K and V of every layer);
    ``scales`` a list of [num_blocks] arrays copied the same way.  Whole blocks,
    all B slots ([PagedAttention] §3.3 ``copy_block``).
    """
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        for p in pools:
            p[dst] = p[src]
        for sc in scales:
            sc[dst] = sc[src]


# --------------------------------------------------------------------------
# block manager
# --------------------------------------------------------------------------

class OutOfBlocks(Exception):
    pass


class BlockManager:
    """Free list + reference counts + per-sequence block tables.

    ``free_order``: the initial free list, head first.  Allocation takes the head
    (first fit); a block whose count drops to zero goes back to the head.
    """

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self.B = block_size
        self.num_blocks = num_blocks
        order = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        assert sorted(order) == list(range(num_blocks))
        self.free = order                   # head = index 0
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        self._next_seq = 0

    # -- helpers
    def _alloc(self) -> int:
        if not self.free:
            raise OutOfBlocks()
        blk = self.free.pop(0)
        self.ref[blk] = 1
        return blk

    def _release(self, blk: int) -> None:
        self.ref[blk] -= 1
        assert self.ref[blk] >= 0
        if self.ref[blk] == 0:
            self.free.insert(0, blk)

    # -- sequence operations
    def new_seq(self) -> int:
        sid = self._next_seq
        self._next_seq += 1
        self.tables[sid] = []
        self.lens[sid] = 0
        return sid

    def fork(self, parent: int) -> int:
        """A child that shares every block of ``parent`` (each count + 1)."""
        sid = self.new_seq()
        self.tables[sid] = list(self.tables[parent])
        self.lens[sid] = self.lens[parent]
        for blk in self.tables[sid]:
            if blk >= 0:
                self.ref[blk] += 1
        return sid

    def append_slot(self, sid: int):
        """Reserve the slot for the sequence's next token.

        Returns ``(slot, cow)`` where ``cow`` is ``(src, dst)`` when the write would
        land in a shared block and a copy was planned, else ``None``.
        """
        n = self.lens[sid]
        table = self.tables[sid]
        cow = None
        if n % self.B == 0:
            # the next token opens a new logical block
            table.append(self._alloc())
        else:
            last = table[-1]
            if self.ref[last] > 1:
                new = self._alloc()
                self.ref[last] -= 1          # still > 0: other sharers keep it
                table[-1] = new
                cow = (last, new)
        slot = table[n // self.B] * self.B + n % self.B
        self.lens[sid] = n + 1
        return slot, cow

    def append_slots(self, sid: int, count: int):
        """``count`` consecutive append_slot calls; fails up front if blocks run short."""
        need = self.blocks_needed(sid, count)
        if need > len(self.free):
            raise OutOfBlocks()
        slots, cows = [], []
        for _ in range(count):
            slot, cow = self.append_slot(sid)
            slots.append(slot)
            if cow is not None:
                cows.append(cow)
        return slots, cows

    def blocks_needed(self, sid: int, count: int) -> int:
        n = self.lens[sid]
        if count <= 0:
            return 0
        new_blocks = -(-(n + count) // self.B) - (-(-n // self.B))
        cow = 1 if (n % self.B != 0 and self.ref[self.tables[sid][-1]] > 1) else 0
        return new_blocks + cow

    def trim(self, sid: int, keep_from: int) -> list:
        """Sliding window: release every block that lies wholly before token ``keep_from``
        (its table entry becomes -1; later entries keep their logical positions).
        Returns the released block ids."""
        assert 0 <= keep_from <= self.lens[sid]      # the block for the next token stays
        table = self.tables[sid]
        released = []
        for j in range(min(keep_from // self.B, len(table))):
            if table[j] >= 0:
                released.append(table[j])
                self._release(table[j])
                table[j] = -1
        return released

    def free_seq(self, sid: int) -> None:
        for blk in self.tables.pop(sid):
            if blk >= 0:
                self._release(blk)
        del self.lens[sid]

    # -- views
    def table(self, sid: int) -> list[int]:
        return list(self.tables[sid])

    def used_blocks(self) -> int:
        return self.num_blocks - len(self.free)

    def shared_blocks(self) -> int:
        return sum(1 for r in self.ref if r > 1)


# --------------------------------------------------------------------------
# block swap to / from host memory
# --------------------------------------------------------------------------

def swap_out(k_pools, v_pools, blocks, k_scales=(), v_scales=()) -> np.ndarray:
    """Host image of physical blocks ([KV缓存机制解析] §6.1: blocks of a long context kept in
    CPU memory; [PagedAttention] §7.2: cold blocks swapped to CPU memory).

    Layout (bytes): for each listed block i, for each layer l: the whole K block, then the
    whole V block (raw bytes of [H, B, d]); after all blocks, for FP8 pools, per block and
    layer the K scale then the V scale (float32).
    """
    parts = []
    for b in np.asarray(blocks).tolist():
        for kp, vp in zip(k_pools, v_pools):
            parts.append(np.ascontiguousarray(kp[b]).view(np.uint8).reshape(-1))
            parts.append(np.ascontiguousarray(vp[b]).view(np.uint8).reshape(-1))
    if len(k_scales):
        sc = [np.float32(s[b]) for b in np.asarray(blocks).tolist() for ks, vs in zip(k_scales, v_scales)
              for s in (ks, vs)]
        parts.append(np.array(sc, dtype=np.float32).view(np.uint8))
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.uint8)


def swap_in(k_pools, v_pools, blocks, image, k_scales=(), v_scales=()) -> None:
    """Write a host image made by ``swap_out`` back into the listed physical blocks."""
    image = np.asarray(image, dtype=np.uint8)
    pos = 0
    for b in np.asarray(blocks).tolist():
        for kp, vp in zip(k_pools, v_pools):
            for p in (kp, vp):
                n = p[b].nbytes
                p[b] = image[pos:pos + n].view(p.dtype).reshape(p[b].shape)
                pos += n
    if len(k_scales):
        sc = image[pos:].view(np.float32)
        i = 0
        for b in np.asarray(blocks).tolist():
            for ks, vs in zip(k_scales, v_scales):
                ks[b] = sc[i]
                vs[b] = sc[i + 1]
                i += 2
