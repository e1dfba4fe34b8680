"""One decode step through libpagedkv: slot mapping, append into the slot, then attention.

``DecodeStep`` owns the per-step device buffers (slot mapping, output, lse, split-KV
workspace).  By default one ``pkv_decode_step`` call does the whole step (the attention kernel
appends the new token as it reads the sequence's last block); ``fused=False`` issues the
separate library calls instead:

1. ``pkv_slot_mapping``  -- the new token's slot from its block table and context length;
2. ``pkv_append``         -- its K/V written into that slot of the paged pools;
3. attention, in the mode ``plan_attention`` picks:
   ``single``   -- ``pkv_decode_attn`` (one CTA per sequence and KV head, no workspace);
   ``split``    -- ``pkv_decode_attn_splitk`` (fixed partitions of the block table, merge).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as B


@dataclass
class AttentionPlan:
    mode: str                      # "single" | "split" (| "prefix": PrefixDecodeStep)
    partition_blocks: int = 0      # split only
    max_partitions: int = 1        # split only

    @property
    def split(self) -> bool:
        return self.mode != "single"

    def describe(self) -> str:
        if self.mode == "prefix":
            return f"shared-prefix pass + {self.partition_blocks}-block suffix partitions, merged"
        if self.mode == "split":
            return f"split-KV, {self.partition_blocks}-block partitions (max {self.max_partitions})"
        return "single-pass"


class PackedInputs:
    """One host->device copy per step for a step's inputs.

    The given device tensors (a step's ``inputs()``) are moved into one device buffer (each
    segment 256-byte aligned, contents kept) and the step's attributes are re-pointed at those
    views; a pinned host buffer mirrors the layout.  Per step the caller writes the new inputs
    into ``host`` (views with the same shapes and dtypes) and calls ``upload(stream)``: a single
    cudaMemcpyAsync instead of one per tensor.
    """

    ALIGN = 256

    def __init__(self, step, names=("q", "k_new", "v_new", "block_tables", "context_lens")):
        tensors = [getattr(step, n) for n in names]
        dev = tensors[0].device
        offsets, off = [], 0
        for t in tensors:
            offsets.append(off)
            off += -(-t.numel() * t.element_size() // self.ALIGN) * self.ALIGN
        self.nbytes = off
        self.device_buf = torch.empty(off, dtype=torch.uint8, device=dev)
        self.host_buf = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.host = {}
        for n, t, o in zip(names, tensors, offsets):
            size = t.numel() * t.element_size()
            dview = self.device_buf[o:o + size].view(t.dtype).view(t.shape)
            dview.copy_(t)
            hview = self.host_buf[o:o + size].view(t.dtype).view(t.shape)
            hview.copy_(t.cpu())
            setattr(step, n, dview)
            self.host[n] = hview

    def upload(self, stream=None) -> None:
        stream = stream or torch.cuda.current_stream(self.device_buf.device)
        with torch.cuda.stream(stream):
            self.device_buf.copy_(self.host_buf, non_blocking=True)

    def bytes_per_step(self) -> int:
        return sum(v.numel() * v.element_size() for v in self.host.values())


LONG_PARTITION_BLOCKS = 128


def plan_attention(num_seqs: int, num_kv_heads: int, max_blocks_per_seq: int, num_sms: int,
                   partition_blocks: int | None = None, mode: str | None = None,
                   taper: bool = True) -> AttentionPlan:
    """Partitions sized by how well the (sequence, KV head) units cover the SMs.

    Measured on GB300 (Llama-3-8B / Llama-2-13B / long-context shapes):
      * with at least one unit per SM, one CTA per unit keeps HBM busy until the short sequences
        finish; then the longest ones stream alone, one CTA each at about 30 GB/s.  Tables longer
        than 128 blocks therefore get 128-block partitions (2K tokens): a sequence that fits in
        one partition is still a single pass (the split kernel writes it out directly and merges
        longer ones in the same launch), and the long ones are spread over more SMs -- 185 vs
        188 us on the ragged Llama-3-8B batch of 64, equal on uniform 1K-token batches;
      * with fewer units than SMs, partitions sized so the grid holds about 512 partition CTAs
        when every sequence is as long as the table allows (at least 8 blocks each) are fastest:
        256 blocks for two sequences of 128K/32K tokens, 128 for 16 sequences of up to 7.4K.
    With at least one unit per SM the grid runs in several waves; ``taper`` then leaves room for
    one more partition, so the split entry points taper (partition 0, launched last, covers half a
    partition and the final wave is short: bf16 180.2 -> 178.1 us, e4m3 118.8 -> 114.7 on the
    batch of 64).  The tcgen05 column kernel of several new tokens does not taper
    (``taper=False``); the mma.sync one does.
    """
    if mode == "single":
        return AttentionPlan("single", max_blocks_per_seq, 1)
    units = num_seqs * num_kv_heads
    if partition_blocks is None:
        if units >= num_sms and mode is None:
            if max_blocks_per_seq <= LONG_PARTITION_BLOCKS:
                return AttentionPlan("single", max_blocks_per_seq, 1)
            partition_blocks = LONG_PARTITION_BLOCKS
        else:
            want = -(-max_blocks_per_seq * units // 512)
            partition_blocks = 8
            while partition_blocks < want:
                partition_blocks *= 2
    count = B.tapered_partitions_for if taper and units >= num_sms else B.max_partitions_for
    return AttentionPlan("split", partition_blocks, count(max_blocks_per_seq, partition_blocks))


class DecodeStep:
    """State of one decode step over a paged cache: the pools and workspace on the GPU; q,
    k_new, v_new, block tables and context lengths on the GPU or in pinned host memory (then
    read in place by the kernel); out / lse / slot_mapping are allocated on the GPU and may be
    replaced by pinned host tensors.

    q [B, N, H] bf16; k_new/v_new [B, K, H] bf16; k_cache/v_cache [nb, 16, K, H] bf16;
    block_tables [B, max_blocks] int32; context_lens [B] int32 (including the new token).
    """

    def __init__(self, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale,
                 plan: AttentionPlan | None = None, err_flag=None, fused: bool = True):
        self.q, self.k_new, self.v_new = q, k_new, v_new
        self.k_cache, self.v_cache = k_cache, v_cache
        self.block_tables, self.context_lens = block_tables, context_lens
        self.scale = float(scale)
        dev = k_cache.device  # the pools' GPU (q and the other inputs may be pinned host memory)
        nseq = q.shape[0]
        self.num_blocks = k_cache.shape[0]
        if plan is None:
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            plan = plan_attention(nseq, k_cache.shape[2], block_tables.shape[1], sms)
        self.plan = plan
        self.slot_mapping = torch.empty(nseq, dtype=torch.int64, device=dev)
        self.out = torch.empty(tuple(q.shape), dtype=q.dtype, device=dev)
        self.lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=dev)
        self.err_flag = err_flag
        # fused: one pkv_decode_step call (single pass or fixed partitions) does it all
        self.fused = fused
        self.workspace = None
        if plan.mode == "split":
            nbytes = B.pkv_splitk_workspace_bytes(nseq, q.shape[1], q.shape[2], plan.max_partitions)
            self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)

    def slot_and_append(self, stream=None) -> None:
        B.check(B.pkv_slot_mapping(self.block_tables, self.context_lens, self.num_blocks,
                                   self.slot_mapping, self.err_flag, stream))
        B.check(B.pkv_append(self.k_new, self.v_new, self.slot_mapping, self.k_cache, self.v_cache,
                             self.err_flag, stream))

    def attention(self, stream=None) -> None:
        if self.plan.mode == "split":
            B.check(B.pkv_decode_attn_splitk(self.q, self.k_cache, self.v_cache, self.block_tables,
                                             self.context_lens, self.scale, self.out,
                                             self.plan.partition_blocks, self.plan.max_partitions,
                                             self.workspace, self.lse, self.err_flag, stream))
        else:
            B.check(B.pkv_decode_attn(self.q, self.k_cache, self.v_cache, self.block_tables,
                                      self.context_lens, self.scale, self.out, self.lse,
                                      self.err_flag, stream))

    def run(self, stream=None) -> None:
        if self.fused:
            split = self.plan.mode == "split"
            B.check(B.pkv_decode_step(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                                      self.block_tables, self.context_lens, self.scale, self.out,
                                      self.lse, self.slot_mapping,
                                      self.plan.partition_blocks if split else 0,
                                      self.plan.max_partitions if split else 0,
                                      self.workspace, self.err_flag, stream))
            return
        self.slot_and_append(stream)
        self.attention(stream)

    def launches_per_step(self) -> int:
        if self.plan.mode == "split":
            attn = B.split_attention_launches(self.q.shape[1], self.k_cache.shape[2], self.plan.max_partitions)
        else:
            attn = 1
        return attn if self.fused else 2 + attn

    def input_names(self):
        """The tensors a caller refreshes every step (the pools are state)."""
        return ("q", "k_new", "v_new", "block_tables", "context_lens")

    def inputs(self):
        return [getattr(self, n) for n in self.input_names()]


class DecodeStepFp8:
    """A decode step over e4m3 pools with per-KV-head scales [K] or per-(physical block, KV head)
    scales [num_blocks, K]: one ``pkv_decode_step_fp8`` call (single pass or fixed partitions, as
    ``plan_attention`` picks)."""

    def __init__(self, q, k_new, v_new, k_cache8, v_cache8, k_scale, v_scale, block_tables,
                 context_lens, scale, plan: AttentionPlan | None = None, err_flag=None):
        self.q, self.k_new, self.v_new = q, k_new, v_new
        self.k_cache, self.v_cache = k_cache8, v_cache8
        self.k_scale, self.v_scale = k_scale, v_scale
        self.block_tables, self.context_lens = block_tables, context_lens
        self.scale = float(scale)
        dev = k_cache8.device  # the pools' GPU (q and the other inputs may be pinned host memory)
        nseq = q.shape[0]
        if plan is None:
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            plan = plan_attention(nseq, k_cache8.shape[2], block_tables.shape[1], sms)
        self.plan = plan
        self.fused = True
        self.slot_mapping = torch.empty(nseq, dtype=torch.int64, device=dev)
        self.out = torch.empty(tuple(q.shape), dtype=q.dtype, device=dev)
        self.lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=dev)
        self.err_flag = err_flag
        self.workspace = None
        if plan.mode == "split":
            nbytes = B.pkv_splitk_workspace_bytes(nseq, q.shape[1], q.shape[2], plan.max_partitions)
            self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)

    def run(self, stream=None) -> None:
        split = self.plan.mode == "split"
        B.check(B.pkv_decode_step_fp8(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                                      self.k_scale, self.v_scale, self.block_tables, self.context_lens,
                                      self.scale, self.out, self.lse, self.slot_mapping,
                                      self.plan.partition_blocks if split else 0,
                                      self.plan.max_partitions if split else 0, self.workspace,
                                      self.err_flag, stream))

    def launches_per_step(self) -> int:
        if self.plan.mode == "split":
            return B.split_attention_launches(self.q.shape[1], self.k_cache.shape[2], self.plan.max_partitions)
        return 1

    def input_names(self):
        return ("q", "k_new", "v_new", "block_tables", "context_lens")

    def inputs(self):
        return [getattr(self, n) for n in self.input_names()]


class MultiTokenStep:
    """Verification of T new tokens per sequence (speculative decoding).  By default one
    ``pkv_decode_step_multi`` call does the whole step: the kernel writes the B*T new K/V rows into
    their slots as it loads their blocks and records the slots.  ``fused=False`` issues the separate
    calls: the slots of the last T positions (``pkv_slot_mapping_multi``), the append
    (``pkv_append``), then ``pkv_decode_attn_multi``.  Attention runs one pass when the (sequence,
    KV head, 32-row chunk) units cover the SMs, else fixed partitions sized like
    ``plan_attention``'s and a log-sum-exp merge (in the same launch for the mma.sync column
    kernel, a second one after the tcgen05 kernel).  The workspace is zeroed once here; each call
    leaves its merge counters at zero.

    q [B, T, N, H] bf16; k_new/v_new [B, T, K, H]; pools, tables and lengths as ``DecodeStep``
    (context_lens counts the T new tokens).
    """

    def __init__(self, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale,
                 partition_blocks: int | None = None, err_flag=None, fused: bool = True):
        self.q, self.k_new, self.v_new = q, k_new, v_new
        self.k_cache, self.v_cache = k_cache, v_cache
        self.block_tables, self.context_lens = block_tables, context_lens
        self.scale = float(scale)
        dev = k_cache.device  # the pools' GPU (q and the other inputs may be pinned host memory)
        nseq, T, N, H = q.shape
        K = k_cache.shape[2]
        self.T = T
        self.num_blocks = k_cache.shape[0]
        chunks = -(-T * (N // K) // 32)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        # the mma.sync column kernel tapers its partitions like the one-token kernel; the tcgen05
        # one keeps them uniform
        tc = bool(B.pkv_multi_uses_tcgen05(T, N, K, H))
        self.plan = plan_attention(nseq * chunks, K, block_tables.shape[1], sms,
                                   partition_blocks=partition_blocks, taper=not tc)
        self.fused = fused
        self.slot_mapping = torch.empty(nseq, T, dtype=torch.int64, device=dev)
        self.out = torch.empty(tuple(q.shape), dtype=q.dtype, device=dev)
        self.lse = torch.empty(nseq, T, N, dtype=torch.float32, device=dev)
        self.err_flag = err_flag
        self.workspace = None
        if self.plan.mode == "split":
            nbytes = B.pkv_splitk_workspace_bytes(nseq * T, N, H, self.plan.max_partitions)
            self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)

    def slot_and_append(self, stream=None) -> None:
        nseq, T = self.q.shape[0], self.T
        K, H = self.k_cache.shape[2], self.k_cache.shape[3]
        B.check(B.pkv_slot_mapping_multi(self.block_tables, self.context_lens, self.num_blocks,
                                         self.slot_mapping, self.err_flag, stream))
        B.check(B.pkv_append(self.k_new.view(nseq * T, K, H), self.v_new.view(nseq * T, K, H),
                             self.slot_mapping.view(-1), self.k_cache, self.v_cache, self.err_flag,
                             stream))

    def attention(self, stream=None) -> None:
        split = self.plan.mode == "split"
        B.check(B.pkv_decode_attn_multi(self.q, self.k_cache, self.v_cache, self.block_tables,
                                        self.context_lens, self.scale, self.out, self.lse,
                                        self.plan.partition_blocks if split else 0,
                                        self.plan.max_partitions if split else 0, self.workspace,
                                        self.err_flag, stream))

    def run(self, stream=None) -> None:
        if self.fused:
            split = self.plan.mode == "split"
            B.check(B.pkv_decode_step_multi(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                                            self.block_tables, self.context_lens, self.scale, self.out,
                                            self.lse, self.slot_mapping,
                                            self.plan.partition_blocks if split else 0,
                                            self.plan.max_partitions if split else 0, self.workspace,
                                            self.err_flag, stream))
            return
        self.slot_and_append(stream)
        self.attention(stream)

    def launches_per_step(self) -> int:
        attn = 1
        if self.plan.mode == "split":
            _, T, N, H = self.q.shape
            tc = bool(B.pkv_multi_uses_tcgen05(T, N, self.k_cache.shape[2], H))
            attn = B.multi_attention_launches(self.plan.max_partitions, tc)
        return attn if self.fused else 2 + attn

    def input_names(self):
        return ("q", "k_new", "v_new", "block_tables", "context_lens")

    def inputs(self):
        return [getattr(self, n) for n in self.input_names()]


def plan_prefix_decode(prefix_tokens: int, group_rows: int) -> int:
    """The shared-prefix cascade's prefix-pass partition size (blocks) when it is the better plan for
    a batch whose groups share ``prefix_tokens`` leading tokens and hold ``group_rows`` query rows
    (members x query heads per KV head), else 0 (the plain decode step).

    Measured on GB300 (20 sequences, 64 query / 8 KV heads, head_dim 128, suffixes of 16..512 tokens:
    160 rows a group; fused steps, µs per step in a CUDA graph, plain / cascade with its best prefix
    partitions): 1,000 shared tokens 29.0 / 30.0 (16 blocks), 2,008 33.5 / 32.7 (16), 4,008
    45.5 / 36.7 (32), 8,008 73.2 / 49.1 (32), 16,008 116.9 / 62.4 (64), 32,008 209.0 / 88.8 (128).
    The plain step reads the prefix once per sequence, mostly from L2, but each of its CTAs streams
    the whole prefix; the cascade spreads the prefix over partitions read once per KV head and
    128-row chunk (the tcgen05 column kernel, from 17 rows a group) and pays two more launches.  So
    the cascade from 3,000 shared tokens on, with partitions of 16 blocks up to 160 shared blocks,
    32 up to 600, 64 up to 1,200, then 128 (about 8 to 16 partitions).  Groups of 16 rows or fewer
    run the cascade on mma.sync, which does not save tile updates (1,000 tokens, 8-row chunks:
    41 vs 30 us): plain."""
    if group_rows <= 16 or prefix_tokens < 3000:
        return 0
    blocks = prefix_tokens // 16
    for limit, pb in ((160, 16), (600, 32), (1200, 64)):
        if blocks <= limit:
            return pb
    return 128


class PrefixDecodeStep:
    """A decode step of a batch whose sequences share leading blocks (copy-on-write prefix
    sharing): by default ``pkv_decode_step_prefix``, whose suffix pass appends each sequence's new
    token as it loads its block (``fused=False``: slot mapping and append of the new token, then
    ``pkv_decode_attn_prefix``, bit for bit the same results) -- each
    group's shared blocks attended once per KV head for all its members in partitions of
    ``prefix_partition_blocks`` (0: ``partition_blocks``), each sequence's own blocks in partitions
    of ``partition_blocks``, merged by log-sum-exp.  Every prefix partition leaves fp32 partials
    for a chunk of 32 query rows (128 when a group's rows outnumber 32 and the tcgen05 column
    kernel runs the prefix pass), so small prefix partitions cost more in partial traffic and
    merging than they gain in parallelism (measured on the 1000-token shared prompt with 32-row
    chunks: 1-block prefix partitions 126 us per step, 16-block 42 us).  ``plan_prefix_decode``
    says when the cascade beats the plain step and picks ``prefix_partition_blocks``.

    group_starts int32 [G+1] and prefix_blocks int32 [G] on the device; max_group_size and
    max_prefix_blocks are host-side bounds on them.
    """

    def __init__(self, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale,
                 group_starts, prefix_blocks, max_group_size: int, max_prefix_blocks: int,
                 partition_blocks: int | None = None, prefix_partition_blocks: int = 0, err_flag=None,
                 fused: bool = True):
        self.q, self.k_new, self.v_new = q, k_new, v_new
        self.k_cache, self.v_cache = k_cache, v_cache
        self.block_tables, self.context_lens = block_tables, context_lens
        self.group_starts, self.prefix_blocks = group_starts, prefix_blocks
        self.max_group_size, self.max_prefix_blocks = int(max_group_size), int(max_prefix_blocks)
        if partition_blocks is None:
            # The suffix pass's grid covers the table's width (the library cannot bound a suffix by
            # the prefix it follows), so its partitions grow with the table: at most 8 per sequence,
            # at least 16 blocks (a 32K-token shared prompt: 256-block partitions, 1,280 suffix CTAs
            # instead of 20,320 mostly empty ones at 16 blocks).
            partition_blocks = 16
            while partition_blocks * 8 < block_tables.shape[1]:
                partition_blocks *= 2
        self.partition_blocks = int(partition_blocks)
        self.prefix_partition_blocks = int(prefix_partition_blocks)
        self.scale = float(scale)
        dev = k_cache.device  # the pools' GPU (q and the other inputs may be pinned host memory)
        nseq, N, H = q.shape
        self.num_blocks = k_cache.shape[0]
        self.plan = AttentionPlan("prefix", self.partition_blocks, 0)
        self.fused = fused
        self.slot_mapping = torch.empty(nseq, dtype=torch.int64, device=dev)
        self.out = torch.empty(tuple(q.shape), dtype=q.dtype, device=dev)
        self.lse = torch.empty(nseq, N, dtype=torch.float32, device=dev)
        self.err_flag = err_flag
        nbytes = B.pkv_prefix_workspace_bytes(nseq, N, H, block_tables.shape[1], self.max_prefix_blocks,
                                              self.partition_blocks, self.prefix_partition_blocks)
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)

    def slot_and_append(self, stream=None) -> None:
        B.check(B.pkv_slot_mapping(self.block_tables, self.context_lens, self.num_blocks,
                                   self.slot_mapping, self.err_flag, stream))
        B.check(B.pkv_append(self.k_new, self.v_new, self.slot_mapping, self.k_cache, self.v_cache,
                             self.err_flag, stream))

    def attention(self, stream=None) -> None:
        B.check(B.pkv_decode_attn_prefix(self.q, self.k_cache, self.v_cache, self.block_tables,
                                         self.context_lens, self.scale, self.group_starts,
                                         self.prefix_blocks, self.max_group_size,
                                         self.max_prefix_blocks, self.out, self.lse,
                                         self.partition_blocks, self.workspace, self.err_flag, stream,
                                         prefix_partition_blocks=self.prefix_partition_blocks))

    def run(self, stream=None) -> None:
        if self.fused:
            B.check(B.pkv_decode_step_prefix(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                                             self.block_tables, self.context_lens, self.scale,
                                             self.group_starts, self.prefix_blocks, self.max_group_size,
                                             self.max_prefix_blocks, self.out, self.lse, self.slot_mapping,
                                             self.partition_blocks, self.workspace, self.err_flag, stream,
                                             prefix_partition_blocks=self.prefix_partition_blocks))
            return
        self.slot_and_append(stream)
        self.attention(stream)

    def launches_per_step(self) -> int:
        # the prefix and suffix passes (one launch, or the tcgen05 prefix pass and the mma.sync
        # suffix pass), the merge; unfused, slot mapping and append before them
        _, N, H = self.q.shape
        tc = B.pkv_multi_uses_tcgen05(self.max_group_size, N, self.k_cache.shape[2], H)
        attn = 3 if tc else 2
        return attn if self.fused else 2 + attn

    def input_names(self):
        return ("q", "k_new", "v_new", "block_tables", "context_lens", "group_starts", "prefix_blocks")

    def inputs(self):
        return [getattr(self, n) for n in self.input_names()]


class LayerStack:
    """One decode step of a model with several attention layers: the same sequences (block tables
    and context lengths) in every layer, each layer with its own pools and its own q, k_new and
    v_new.  ``run`` launches the layers' fused steps in order (one launch each, two with a
    separate merge); captured in a CUDA graph (``StepGraph``) the whole multi-layer step replays
    as one graph launch.  Attribute names ``"<name>.<layer>"`` (``"q.3"``) reach one layer's
    inputs, ``block_tables`` / ``context_lens`` are shared, ``out`` / ``lse`` are the last
    layer's; so ``PackedInputs(stack, stack.input_names())`` packs every layer's inputs into one
    host-to-device copy per step."""

    _SHARED = ("block_tables", "context_lens")

    def __init__(self, layers):
        layers = list(layers)
        if not layers or not all(getattr(l, "fused", False) for l in layers):
            raise ValueError("a layer stack needs fused decode steps")
        object.__setattr__(self, "layers", layers)
        object.__setattr__(self, "plan", layers[0].plan)
        object.__setattr__(self, "fused", True)

    def __getattr__(self, name):
        if "." in name:
            attr, idx = name.rsplit(".", 1)
            return getattr(self.layers[int(idx)], attr)
        if name in self._SHARED:
            return getattr(self.layers[0], name)
        if name in ("out", "lse", "slot_mapping"):
            return getattr(self.layers[-1], name)
        raise AttributeError(name)

    def __setattr__(self, name, value):
        if "." in name:
            attr, idx = name.rsplit(".", 1)
            setattr(self.layers[int(idx)], attr, value)
        elif name in self._SHARED:
            for layer in self.layers:
                setattr(layer, name, value)
        else:
            object.__setattr__(self, name, value)

    def run(self, stream=None) -> None:
        for layer in self.layers:
            layer.run(stream)

    def launches_per_step(self) -> int:
        return sum(layer.launches_per_step() for layer in self.layers)

    def input_names(self):
        return self._SHARED + tuple(f"{n}.{i}" for i in range(len(self.layers)) for n in ("q", "k_new", "v_new"))

    def inputs(self):
        return [getattr(self, n) for n in self.input_names()]


class StepGraph:
    """A step (or a LayerStack) captured once into a CUDA graph and replayed: the launches of all
    its kernels cost one graph launch.  The step is run once eagerly first (kernel attributes are
    set on first use, outside the capture); a decode step is idempotent for fixed inputs (the same
    rows land in the same slots), so that run changes nothing the replay would not."""

    def __init__(self, step, stream=None):
        dev = step.out.device
        self.step = step
        self.stream = stream or torch.cuda.Stream(dev)
        with torch.cuda.stream(self.stream):
            step.run(self.stream)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            step.run(self.stream)

    def replay(self) -> None:
        self.graph.replay()
