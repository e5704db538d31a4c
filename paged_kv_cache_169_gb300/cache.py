"""Tensor-owning convenience layer over the C ABI (PyTorch supplies device memory and streams).

No arithmetic happens here: every step of append, copy and attention runs in the
library's CUDA kernels.  These classes only allocate torch tensors, pass their
addresses, and keep the handles alive.
"""

from __future__ import annotations

import torch

from . import abi

_TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "fp8": torch.uint8}
_KV_DTYPE = {"f32": abi.KV_F32, "f16": abi.KV_F16, "fp8": abi.KV_FP8_E4M3}
_IN_DTYPE = {torch.float32: abi.KV_F32, torch.float16: abi.KV_F16}


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _dev_ptr(t: torch.Tensor, what: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


class PagedKVCache:
    """A paged K/V pool for ``num_layers`` layers, laid out [num_blocks, H, B, d] per layer.

    ``dtype``: "f32", "f16" or "fp8" (E4M3 codes + per-block float32 scales).
    """

    def __init__(self, num_layers: int, num_blocks: int, block_size: int, num_heads: int,
                 head_dim: int, dtype: str = "f16", device="cuda"):
        if dtype not in _TORCH_DTYPE:
            raise ValueError(f"dtype must be one of {list(_TORCH_DTYPE)}")
        self.num_layers, self.num_blocks, self.block_size = num_layers, num_blocks, block_size
        self.num_heads, self.head_dim, self.dtype = num_heads, head_dim, dtype
        shape = (num_blocks, num_heads, block_size, head_dim)
        td = _TORCH_DTYPE[dtype]
        self.k = [torch.empty(shape, dtype=td, device=device) for _ in range(num_layers)]
        self.v = [torch.empty(shape, dtype=td, device=device) for _ in range(num_layers)]
        self.k_scale = self.v_scale = None
        if dtype == "fp8":
            cap = (num_blocks + 3) // 4 * 4
            self.k_scale = [torch.ones(cap, dtype=torch.float32, device=device) for _ in range(num_layers)]
            self.v_scale = [torch.ones(cap, dtype=torch.float32, device=device) for _ in range(num_layers)]
        self.handle = abi.kv_pool_create(
            num_layers, num_blocks, block_size, num_heads, head_dim, _KV_DTYPE[dtype],
            [t.data_ptr() for t in self.k], [t.data_ptr() for t in self.v],
            [t.data_ptr() for t in self.k_scale] if self.k_scale else None,
            [t.data_ptr() for t in self.v_scale] if self.v_scale else None)
        self._ws = None

    # -------------------------------------------------------------- device ops
    def append(self, layer: int, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
               stream=None) -> None:
        """k, v: [n, H, d] (pool dtype; f16/f32 for FP8 pools); slot_mapping: int64 [n]."""
        if slot_mapping.dtype != torch.int64:
            raise ValueError("slot_mapping must be int64")
        n = slot_mapping.numel()
        if k.shape != (n, self.num_heads, self.head_dim) or v.shape != k.shape or k.dtype != v.dtype:
            raise ValueError("k and v must be [num_tokens, H, d] of one dtype")
        abi.kv_append(self.handle, layer, _dev_ptr(k, "k"), _dev_ptr(v, "v"), _IN_DTYPE[k.dtype],
                      _dev_ptr(slot_mapping, "slot_mapping"), n, _stream(stream))

    def copy_blocks(self, pairs: torch.Tensor, layer_begin: int = 0, layer_end: int | None = None,
                    stream=None) -> None:
        """pairs: device int32 [n, 2] of (src, dst) physical blocks."""
        if pairs.dtype != torch.int32 or pairs.dim() != 2 or pairs.shape[1] != 2:
            raise ValueError("pairs must be int32 [n, 2]")
        le = self.num_layers if layer_end is None else layer_end
        abi.kv_copy_blocks(self.handle, _dev_ptr(pairs, "pairs") if pairs.numel() else 0,
                           pairs.shape[0], layer_begin, le, _stream(stream))

    def swap_out(self, blocks: torch.Tensor, host: torch.Tensor | None = None, layer_begin: int = 0,
                 layer_end: int | None = None, stream=None) -> torch.Tensor:
        """Copy physical blocks (device int32 [n]) of the layers to a pinned host image
        (uint8, allocated if not given).  Asynchronous on the stream."""
        le = self.num_layers if layer_end is None else layer_end
        n = abi.kv_swap_bytes(self.handle, blocks.numel(), layer_begin, le)
        if host is None:
            host = torch.empty(n, dtype=torch.uint8).pin_memory()
        if host.numel() < n or host.is_cuda:
            raise ValueError("host image must be a pinned CPU tensor of kv_swap_bytes bytes")
        abi.kv_swap_out(self.handle, _dev_ptr(blocks, "blocks"), blocks.numel(), layer_begin, le,
                        host.data_ptr(), _stream(stream))
        return host

    def swap_in(self, host: torch.Tensor, blocks: torch.Tensor, layer_begin: int = 0,
                layer_end: int | None = None, stream=None) -> None:
        le = self.num_layers if layer_end is None else layer_end
        abi.kv_swap_in(self.handle, host.data_ptr(), _dev_ptr(blocks, "blocks"), blocks.numel(),
                       layer_begin, le, _stream(stream))

    def workspace_bytes(self, batch: int, max_context: int, partition_tokens: int = 0) -> int:
        return abi.paged_decode_workspace_size(self.handle, batch, max_context, partition_tokens)

    def workspace(self, batch: int, max_context: int, partition_tokens: int = 0) -> torch.Tensor:
        n = self.workspace_bytes(batch, max_context, partition_tokens)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(n, dtype=torch.uint8, device=self.k[0].device)
        return self._ws

    def attention(self, layer: int, q: torch.Tensor, block_tables: torch.Tensor,
                  context_lens: torch.Tensor, max_context: int, scale: float,
                  out: torch.Tensor | None = None, partition_tokens: int = 0,
                  workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """q: [batch, H, d]; block_tables: int32 [batch, max_blocks]; context_lens: int32 [batch].
        Returns out float32 [batch, H, d]."""
        batch = q.shape[0]
        if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
            raise ValueError("block_tables and context_lens must be int32")
        if out is None:
            out = torch.empty((batch, self.num_heads, self.head_dim), dtype=torch.float32, device=q.device)
        ws = workspace if workspace is not None else self.workspace(batch, max_context, partition_tokens)
        abi.paged_decode_attention(
            self.handle, layer, _dev_ptr(q, "q"), _dev_ptr(out, "out"),
            _dev_ptr(block_tables, "block_tables"), block_tables.shape[1],
            _dev_ptr(context_lens, "context_lens"), batch, max_context, float(scale),
            partition_tokens, _dev_ptr(ws, "workspace"), ws.numel(), _stream(stream))
        return out

    def attention_append(self, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                         block_tables: torch.Tensor, context_lens: torch.Tensor, max_context: int,
                         scale: float, out: torch.Tensor | None = None, partition_tokens: int = 0,
                         workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Fused decode step: store each sequence's newest token (k_new, v_new [batch, H, d])
        at position context_lens[s]-1 through its table, then attend.  Returns out."""
        batch = q.shape[0]
        if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
            raise ValueError("block_tables and context_lens must be int32")
        if k_new.shape != (batch, self.num_heads, self.head_dim) or v_new.shape != k_new.shape \
                or k_new.dtype != v_new.dtype:
            raise ValueError("k_new and v_new must be [batch, H, d] of one dtype")
        if out is None:
            out = torch.empty((batch, self.num_heads, self.head_dim), dtype=torch.float32, device=q.device)
        ws = workspace if workspace is not None else self.workspace(batch, max_context, partition_tokens)
        abi.paged_decode_attention_append(
            self.handle, layer, _dev_ptr(q, "q"), _dev_ptr(k_new, "k_new"), _dev_ptr(v_new, "v_new"),
            _IN_DTYPE[k_new.dtype], _dev_ptr(out, "out"), _dev_ptr(block_tables, "block_tables"),
            block_tables.shape[1], _dev_ptr(context_lens, "context_lens"), batch, max_context,
            float(scale), partition_tokens, _dev_ptr(ws, "workspace"), ws.numel(), _stream(stream))
        return out

    def attention_gqa(self, layer: int, q: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, max_context: int, scale: float,
                      k_new: torch.Tensor | None = None, v_new: torch.Tensor | None = None,
                      out: torch.Tensor | None = None, partition_tokens: int = 0,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Grouped-query decode attention: q [batch, Hq, d] with Hq a multiple (1, 2, 4, 8) of
        the pool's KV heads; optional fused append of k_new/v_new [batch, H, d]."""
        batch, hq = q.shape[0], q.shape[1]
        if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
            raise ValueError("block_tables and context_lens must be int32")
        if out is None:
            out = torch.empty((batch, hq, self.head_dim), dtype=torch.float32, device=q.device)
        if workspace is None:
            n = abi.paged_decode_workspace_size_gqa(self.handle, batch, hq, max_context, partition_tokens)
            if self._ws is None or self._ws.numel() < n:
                self._ws = torch.empty(n, dtype=torch.uint8, device=self.k[0].device)
            workspace = self._ws
        kp = _dev_ptr(k_new, "k_new") if k_new is not None else 0
        vp = _dev_ptr(v_new, "v_new") if v_new is not None else 0
        dt = _IN_DTYPE[k_new.dtype] if k_new is not None else 0
        abi.paged_decode_attention_gqa(
            self.handle, layer, _dev_ptr(q, "q"), hq, kp, vp, dt, _dev_ptr(out, "out"),
            _dev_ptr(block_tables, "block_tables"), block_tables.shape[1],
            _dev_ptr(context_lens, "context_lens"), batch, max_context, float(scale), partition_tokens,
            _dev_ptr(workspace, "workspace"), workspace.numel(), _stream(stream))
        return out

    def attention_ex(self, layer: int, q: torch.Tensor, block_tables: torch.Tensor,
                     context_lens: torch.Tensor, max_context: int, scale: float, window: int = 0,
                     k_new: torch.Tensor | None = None, v_new: torch.Tensor | None = None,
                     out: torch.Tensor | None = None, partition_tokens: int = 0,
                     workspace: torch.Tensor | None = None, stream=None, flags: int = 0,
                     out_dtype: torch.dtype = torch.float32,
                     prefix_groups: torch.Tensor | None = None) -> torch.Tensor:
        """Every decode option in one call (paged_decode_attention_ex): grouped-query heads
        (q [batch, Hq, d]), optional fused append, and a sliding window of ``window`` tokens.
        ``flags``: abi.KV_DECODE_WORKSPACE_ZEROED (the workspace's counters are zero: a
        zero-filled workspace used only by decode calls since), abi.KV_DECODE_PDL,
        abi.KV_DECODE_EARLY_TABLES.  A float16 ``out`` (or ``out_dtype``) adds
        abi.KV_DECODE_OUT_F16: the result is stored rounded to float16.
        ``prefix_groups``: int32 CUDA tensor [n, 3] of (first sequence, member count, shared
        tokens): sequences forked from one prompt read its shared blocks once per group."""
        batch, hq = q.shape[0], q.shape[1]
        if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
            raise ValueError("block_tables and context_lens must be int32")
        if out is None:
            out = torch.empty((batch, hq, self.head_dim), dtype=out_dtype, device=q.device)
        if out.dtype == torch.float16:
            flags |= abi.KV_DECODE_OUT_F16
        elif out.dtype != torch.float32 or flags & abi.KV_DECODE_OUT_F16:
            raise ValueError("out must be float32, or float16 (KV_DECODE_OUT_F16)")
        a = abi.kv_decode_args()
        a.layer, a.q, a.num_q_heads = layer, _dev_ptr(q, "q"), hq
        a.k_new = _dev_ptr(k_new, "k_new") if k_new is not None else None
        a.v_new = _dev_ptr(v_new, "v_new") if v_new is not None else None
        a.in_dtype = _IN_DTYPE[k_new.dtype] if k_new is not None else 0
        a.out = _dev_ptr(out, "out")
        a.block_tables, a.max_blocks_per_seq = _dev_ptr(block_tables, "block_tables"), block_tables.shape[1]
        a.context_lens, a.batch, a.max_context = _dev_ptr(context_lens, "context_lens"), batch, max_context
        a.window, a.scale, a.partition_tokens = window, float(scale), partition_tokens
        if prefix_groups is not None:
            if prefix_groups.dtype != torch.int32 or prefix_groups.dim() != 2 or prefix_groups.shape[1] != 3:
                raise ValueError("prefix_groups must be an int32 [n, 3] tensor")
            if prefix_groups.shape[0] > 0:
                a.prefix_groups = _dev_ptr(prefix_groups, "prefix_groups")
                a.num_prefix_groups = prefix_groups.shape[0]
        if workspace is None:
            n = abi.paged_decode_workspace_size_ex(self.handle, a)
            if self._ws is None or self._ws.numel() < n:
                self._ws = torch.empty(n, dtype=torch.uint8, device=self.k[0].device)
            workspace = self._ws
        a.workspace, a.workspace_bytes = _dev_ptr(workspace, "workspace"), workspace.numel()
        a.stream = _stream(stream)
        a.flags = flags
        abi.paged_decode_attention_ex(self.handle, a)
        return out

    def zeroed_workspace(self, batch: int, max_context: int, partition_tokens: int = 0,
                         num_q_heads: int = 0, window: int = 0, prefix_groups: bool = False) -> torch.Tensor:
        """A new zero-filled workspace for attention_ex(..., flags=KV_DECODE_WORKSPACE_ZEROED),
        valid for calls of this one shape (batch, query heads, max_context, partition, window,
        with or without prefix groups)."""
        a = abi.kv_decode_args()
        a.num_q_heads, a.batch, a.max_context = num_q_heads, batch, max_context
        a.window, a.partition_tokens = window, partition_tokens
        a.num_prefix_groups = 1 if prefix_groups else 0
        n = abi.paged_decode_workspace_size_ex(self.handle, a)
        return torch.zeros(n, dtype=torch.uint8, device=self.k[0].device)

    def device_error(self, clear: bool = True, stream=None) -> int:
        return abi.kv_get_device_error(self.handle, _stream(stream), clear)

    def close(self) -> None:
        if self.handle:
            abi.kv_pool_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BlockAllocator:
    """Host block allocator (free list, reference counts, fork, copy-on-write planning)."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self.num_blocks, self.block_size = num_blocks, block_size
        self.handle = abi.kv_alloc_create(num_blocks, block_size, free_order)

    def new_seq(self) -> int:
        return abi.kv_alloc_seq_new(self.handle)

    def fork(self, parent: int) -> int:
        return abi.kv_alloc_seq_fork(self.handle, parent)

    def append_slots(self, seq: int, count: int = 1):
        return abi.kv_alloc_append_slots(self.handle, seq, count)

    def free_seq(self, seq: int) -> None:
        abi.kv_alloc_seq_free(self.handle, seq)

    def trim(self, seq: int, keep_from: int) -> int:
        return abi.kv_alloc_seq_trim(self.handle, seq, keep_from)

    def seq_info(self, seq: int):
        return abi.kv_alloc_seq_info(self.handle, seq)

    def table(self, seq: int):
        return abi.kv_alloc_block_table(self.handle, seq)

    def build_tables(self, seqs, max_blocks: int):
        return abi.kv_alloc_build_tables(self.handle, list(seqs), max_blocks)

    def ref_count(self, block: int) -> int:
        return abi.kv_alloc_ref_count(self.handle, block)

    def free_list(self):
        return abi.kv_alloc_free_list(self.handle, self.num_blocks)

    def stats(self):
        return abi.kv_alloc_stats(self.handle)

    def close(self) -> None:
        if self.handle:
            abi.kv_alloc_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
