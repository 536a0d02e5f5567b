"""One continuous-batching step of the paged attention path.

A step writes the new tokens' K/V into the cache through the slot mapping
(``pa_cache_write``), then runs decode attention for the sequences that
generate one token (``pa_decode``) and causal chunked-prefill attention for
the sequences that bring a chunk of prompt tokens (``pa_prefill_chunk``) --
the unified continuous batch of the vllm.cpp engine ("C++20 Continuous
Batching Loop" in the "vllm.cpp ARCHITECTURE OVERVIEW" figure of "Building
and Deploying vllm.cpp ..."; chunked prefill in the Engine core bullet of the
vllm.cpp repository's "What's implemented").

This module only orders the library's calls on CUDA streams; every step of
the computation runs in the library's kernels.  Decode and prefill read
disjoint outputs and only read the cache, so after the write they may run
concurrently.  Three ways to issue them (``mode``):
  * "fused"  -- one launch of pa_mixed_attention: one persistent kernel whose
                CTAs take the prefill tiles and then the decode partitions
                from one work list (with both parts present and a descriptor
                it takes; "streams" otherwise).  A prefill of a few long
                chunks would leave most SMs idle there: given a prefill
                workspace, a step whose prefill has at most half as many
                (query tile, kv head) items as there are SMs, and which
                pa_prefill_chunk_balanced would run on its balanced kernel
                (pa_prefill_balanced_chosen), runs the decode and then that
                prefill instead (with more items the fused launch's decode
                fills the SMs the prefill leaves);
  * "streams" -- the decode on a second stream that waits for the write,
                beside the prefill on the caller's stream, so that the
                decode's CTAs take the SMs the prefill's last wave leaves idle;
  * "serial" -- the decode, then the prefill, on the caller's stream.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


class MixedStep:
    """Issues one step: the cache write, decode and prefill (as one launch
    where the library takes it, else as a cache write and the attention).

    Buffers that persist across steps (the caches, the decode workspace and
    the outputs) are given once; the per-step inputs are passed to
    ``__call__``.  Either part may be absent (``decode_out`` or
    ``prefill_out`` None).  With a ``prefill_workspace``
    (binding.prefill_workspace) the prefill runs as
    pa_prefill_chunk_balanced, its KV work spread evenly over the SMs;
    without one as pa_prefill_chunk.  With ``decode_append`` a step without a
    prefill part whose new rows are one token per decode sequence, in
    sequence order (k_new[s] at position context_lens[s] - 1), runs as one
    pa_decode_append launch instead of pa_cache_write and pa_decode; where
    the library does not take it (the CUDA-core decode kernel)
    the step falls back to the two calls.  With ``write_in_step`` the fused
    mode runs a step with both parts, cache write included, as one
    pa_mixed_attention_append launch: the caller's new rows are then the
    decode sequences' tokens in sequence order followed by the prefill
    chunks' tokens in query order, and every chunk starts at a block
    boundary."""

    MODES = ("fused", "streams", "serial")

    def __init__(self, desc: B.PaKvDesc, k_cache, v_cache, scale: float, *, decode_out=None, decode_lse=None,
                 workspace=None, max_context_len_decode: int = 0, prefill_out=None, prefill_lse=None,
                 max_q_len: int = 0, max_context_len_prefill: int = 0, mode: str = "fused",
                 prefill_workspace=None, decode_append: bool = False, write_in_step: bool = False):
        if mode not in self.MODES:
            raise ValueError(f"mode must be one of {self.MODES}")
        self.desc = desc
        self.k_cache, self.v_cache = k_cache, v_cache
        self.scale = float(scale)
        self.decode_out, self.decode_lse, self.workspace = decode_out, decode_lse, workspace
        self.max_context_len_decode = int(max_context_len_decode)
        self.prefill_out, self.prefill_lse = prefill_out, prefill_lse
        self.max_q_len, self.max_context_len_prefill = int(max_q_len), int(max_context_len_prefill)
        self.prefill_workspace = prefill_workspace
        self.decode_append = bool(decode_append) and decode_out is not None and prefill_out is None
        self.write_in_step = bool(write_in_step)
        self._balanced = {}  # (prefill sequences, table width) -> the balanced prefill runs
        both = decode_out is not None and prefill_out is not None
        fused_ok = (desc.kv_dtype in (B.PA_KV_BF16, B.PA_KV_F16) and desc.head_dim == 128
                    and desc.decode_impl in (B.PA_DECODE_AUTO, B.PA_DECODE_MMA)
                    and desc.prefill_impl in (B.PA_PREFILL_AUTO, B.PA_PREFILL_TCGEN05) and workspace is not None)
        if mode == "fused" and fused_ok and both:
            need = B.load().pa_mixed_workspace_size(B.ctypes.byref(desc), int(decode_out.shape[0]),
                                                    int(max_context_len_decode))
            if workspace.numel() < need:
                raise ValueError(f"the fused step needs a workspace of {need} bytes (binding.mixed_workspace)")
        # fused needs both parts and a descriptor pa_mixed_attention takes
        self.mode = "streams" if mode == "fused" and not (fused_ok and both) else mode
        self.overlap = self.mode == "streams" and both
        dev = k_cache.device
        self.side: Optional[torch.cuda.Stream] = torch.cuda.Stream(device=dev) if self.overlap else None
        self.ev_written = torch.cuda.Event()
        self.ev_decoded = torch.cuda.Event()

    def decode(self, q, block_tables, context_lens, stream=None):
        B.pa_decode(self.desc, self.decode_out, q, self.k_cache, self.v_cache, block_tables, context_lens,
                    self.max_context_len_decode, self.scale, self.workspace, lse=self.decode_lse, stream=stream)

    def prefill(self, q, query_start_loc, block_tables, context_lens, stream=None):
        if self.prefill_workspace is not None:
            B.pa_prefill_chunk_balanced(self.desc, self.prefill_out, q, query_start_loc, self.k_cache,
                                        self.v_cache, block_tables, context_lens, self.max_q_len,
                                        self.max_context_len_prefill, self.scale, self.prefill_workspace,
                                        lse=self.prefill_lse, stream=stream)
            return
        B.pa_prefill_chunk(self.desc, self.prefill_out, q, query_start_loc, self.k_cache, self.v_cache,
                           block_tables, context_lens, self.max_q_len, self.max_context_len_prefill, self.scale,
                           lse=self.prefill_lse, stream=stream)

    def prefill_balanced(self, pf_args) -> bool:
        """Whether this step's prefill runs pa_prefill_chunk_balanced's balanced
        kernel (a prefill workspace given and the library's choice)."""
        if self.prefill_workspace is None or pf_args is None or self.prefill_out is None:
            return False
        key = (int(pf_args[3].shape[0]), int(pf_args[2].shape[1]))
        if key not in self._balanced:
            # items as the prefill kernels count them: 256 (query, head) rows of one kv head
            g = self.desc.num_q_heads // self.desc.num_kv_heads
            qt = 256 // g
            items = key[0] * ((self.max_q_len + qt - 1) // qt) * self.desc.num_kv_heads
            sms = torch.cuda.get_device_properties(self.k_cache.device).multi_processor_count
            self._balanced[key] = (2 * items <= sms and
                                   B.pa_prefill_balanced_chosen(self.desc, key[0], self.max_q_len,
                                                                self.max_context_len_prefill, key[1]))
        return self._balanced[key]

    def _mixed_parts(self, dec_args, pf_args):
        """The dec and pf arguments of the mixed entry points."""
        dec = None
        if dec_args is not None and self.decode_out is not None:
            dec = (self.decode_out, *dec_args, self.max_context_len_decode, self.decode_lse)
        pf = None
        if pf_args is not None and self.prefill_out is not None:
            pf = (self.prefill_out, *pf_args, self.max_q_len, self.max_context_len_prefill, self.prefill_lse)
        return dec, pf

    def attend(self, dec_args, pf_args):
        """Decode and prefill after a cache write already issued on the current stream."""
        if self.mode == "fused" and self.prefill_balanced(pf_args):
            # a few long prefill chunks: the balanced kernel on every SM, after the decode
            if dec_args is not None and self.decode_out is not None:
                self.decode(*dec_args)
            self.prefill(*pf_args)
            return
        if self.mode == "fused":
            B.pa_mixed_attention(self.desc, self.k_cache, self.v_cache, self.scale, self.workspace,
                                 *self._mixed_parts(dec_args, pf_args))
            return
        if self.overlap:
            main = torch.cuda.current_stream()
            self.ev_written.record(main)
            self.side.wait_event(self.ev_written)
            with torch.cuda.stream(self.side):
                self.decode(*dec_args)
            self.ev_decoded.record(self.side)
            self.prefill(*pf_args)
            main.wait_event(self.ev_decoded)
            return
        if dec_args is not None and self.decode_out is not None:
            self.decode(*dec_args)
        if pf_args is not None and self.prefill_out is not None:
            self.prefill(*pf_args)

    def __call__(self, k_new, v_new, slot_mapping, dec_args=None, pf_args=None):
        """dec_args: (q, block_tables, context_lens); pf_args: (q, query_start_loc,
        block_tables, context_lens)."""
        if self.decode_append and dec_args is not None and k_new is not None and \
                k_new.shape[0] == dec_args[2].shape[0]:
            q, block_tables, context_lens = dec_args
            try:
                B.pa_decode_append(self.desc, self.decode_out, q, k_new, v_new, self.k_cache, self.v_cache,
                                   block_tables, context_lens, self.max_context_len_decode, self.scale,
                                   self.workspace, lse=self.decode_lse)
                return
            except B.PaError as e:
                if e.status != B.PA_ERR_UNSUPPORTED:
                    raise
                self.decode_append = False  # checked before anything was enqueued: the two calls below
        if (self.write_in_step and self.mode == "fused" and k_new is not None and dec_args is not None
                and pf_args is not None and not self.prefill_balanced(pf_args)):
            # the whole step in one launch, the cache write included
            B.pa_mixed_attention_append(self.desc, k_new, v_new, self.k_cache, self.v_cache, self.scale,
                                        self.workspace, *self._mixed_parts(dec_args, pf_args))
            return
        if slot_mapping is not None and slot_mapping.numel() > 0:
            B.pa_cache_write(self.desc, k_new, v_new, self.k_cache, self.v_cache, slot_mapping)
        self.attend(dec_args, pf_args)


class GraphedStep:
    """A whole step replayed from a CUDA graph.

    ``issue`` is a callable that enqueues one step on the current stream
    without allocating: typically the copy of the step's inputs from pinned
    host memory into device buffers, a MixedStep call on those buffers, and
    the copy of the outputs back into pinned host memory.  It is run a few
    times on a side stream (to settle every lazy set-up), then captured once;
    each call replays the graph on the current stream and waits for it.  The
    buffers ``issue`` names must stay alive and in place while the object is
    used: the graph holds their addresses."""

    def __init__(self, issue, warmup: int = 2):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                issue()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            issue()
        torch.cuda.synchronize()

    def __call__(self, wait: bool = True):
        self.graph.replay()
        if wait:
            torch.cuda.current_stream().synchronize()
