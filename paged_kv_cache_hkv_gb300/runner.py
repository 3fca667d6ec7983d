"""Device-resident copy of one step's inputs, run through the C ABI.

``DeviceStep`` uploads a host step (``synth.PagedStep``) once and runs the
hot path on it: slot mapping, cache write, attention. It is what the tests,
the smoke check and the benchmark drive.
"""

from __future__ import annotations

import numpy as np
import torch

from . import binding


def _bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def _i32(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bf16_to_numpy(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> host uint16 bit patterns."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def shared_prefix_of(step):
    """The shared-prefix hint of a step whose requests marked shares_prefix
    form one contiguous run of decodes: (prefix tokens, first request,
    requests), else None. This is what the caller's block manager knows
    (which leading blocks are referenced by several requests)."""
    idx = [i for i, s in enumerate(step.specs) if s.shares_prefix]
    if not idx or not step.prefix_tokens:
        return None
    first, num = idx[0], len(idx)
    if idx != list(range(first, first + num)):
        return None
    if any(step.specs[i].query_len != 1 for i in idx):
        return None
    return (int(step.prefix_tokens), first, num)


class DeviceStep:
    """One step's inputs on the GPU plus its output buffers."""

    def __init__(self, step, device="cuda", decode_splits=None, upload_pool=True,
                 shared_prefix=None, fused_write=False, write_in_attention=False):
        """shared_prefix: None, or (shared_prefix_len, shared_first_req,
        shared_num_reqs) for the attention call (see pagedkv.h); "auto" takes
        it from the step's shared prefix when its sharing requests form one
        contiguous run of decodes. fused_write: run() maps the slots and
        writes the rows in one launch (pkv_slot_mapping_and_write);
        write_in_attention: run() is the single call
        pkv_paged_attention_with_write."""
        self.step = step
        self.device = torch.device(device)
        dev = self.device
        self.kv_cache = _bf16(step.kv_cache, dev) if upload_pool else None
        self.q = _bf16(step.q, dev)
        self.k = _bf16(step.k, dev)
        self.v = _bf16(step.v, dev)
        self.block_table = _i32(step.block_table, dev)
        self.seq_lens = _i32(step.seq_lens, dev)
        self.query_start_loc = _i32(step.query_start_loc, dev)
        self.num_computed = _i32(step.num_computed, dev)
        T = step.num_tokens
        self.slot_mapping = torch.empty(T, dtype=torch.int64, device=dev)
        self.out = torch.zeros((T, step.num_q_heads, step.head_dim), dtype=torch.bfloat16,
                               device=dev)
        self.decode_splits = decode_splits
        self.fused_write = fused_write
        self.write_in_attention = write_in_attention
        if shared_prefix == "auto":
            shared_prefix = shared_prefix_of(step)
        self.shared_prefix = shared_prefix
        self.layout = binding.pkv_cache_layout(step.num_blocks, step.block_size,
                                               step.num_kv_heads, step.head_dim)
        nbytes = binding.pkv_attention_workspace_size(step.num_reqs, step.num_q_heads,
                                                      self.layout, decode_splits=decode_splits,
                                                      shared_prefix=shared_prefix)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self._calls = None
        self._calls_bufs = ()

    # -- the three calls of the hot path
    def slot_map(self, stream=None):
        s = self.step
        binding.pkv_slot_mapping(self.slot_mapping, self.block_table, self.query_start_loc,
                                 self.num_computed, s.num_blocks, s.block_size, stream=stream)

    def write(self, stream=None):
        binding.pkv_paged_kv_write(self.kv_cache, self.k, self.v, self.slot_mapping,
                                   stream=stream)

    def slot_map_and_write(self, stream=None):
        binding.pkv_slot_mapping_and_write(self.kv_cache, self.k, self.v, self.block_table,
                                           self.query_start_loc, self.num_computed,
                                           slot_mapping=self.slot_mapping, stream=stream)

    def attend_with_write(self, stream=None):
        s = self.step
        binding.pkv_paged_attention_with_write(
            self.out, self.q, self.kv_cache, self.k, self.v, self.block_table, self.seq_lens,
            self.query_start_loc, self.num_computed, max_query_len=s.max_query_len,
            max_seq_len=s.max_seq_len, scale=s.scale, workspace=self.workspace,
            slot_mapping=self.slot_mapping, decode_splits=self.decode_splits,
            shared_prefix=self.shared_prefix, stream=stream)

    def attend(self, stream=None):
        s = self.step
        binding.pkv_paged_attention(
            self.out, self.q, self.kv_cache, self.block_table, self.seq_lens,
            self.query_start_loc, self.num_computed, max_query_len=s.max_query_len,
            max_seq_len=s.max_seq_len, scale=s.scale, workspace=self.workspace,
            decode_splits=self.decode_splits, shared_prefix=self.shared_prefix, stream=stream)

    def run(self, stream=None):
        """The whole step: slot mapping, cache write (one launch with
        fused_write), attention. The calls' arguments are marshalled once and
        reused while the buffers stay the same objects (a test may swap a
        buffer between runs)."""
        self.calls().run(stream)

    def calls(self) -> "binding.StepCalls":
        """The step's three calls with their arguments marshalled (rebuilt
        when a buffer was replaced)."""
        bufs = (self.slot_mapping, self.block_table, self.query_start_loc, self.num_computed,
                self.kv_cache, self.k, self.v, self.out, self.q, self.seq_lens, self.workspace)
        if self._calls is None or any(a is not b for a, b in zip(bufs, self._calls_bufs)):
            s = self.step
            self._calls = binding.StepCalls(
                slot_mapping=self.slot_mapping, block_table=self.block_table,
                query_start_loc=self.query_start_loc, num_computed_tokens=self.num_computed,
                kv_cache=self.kv_cache, key=self.k, value=self.v, out=self.out, q=self.q,
                seq_lens=self.seq_lens, max_query_len=s.max_query_len,
                max_seq_len=s.max_seq_len, scale=s.scale, workspace=self.workspace,
                decode_splits=self.decode_splits, shared_prefix=self.shared_prefix,
                fused_write=self.fused_write, write_in_attention=self.write_in_attention)
            self._calls_bufs = bufs
        return self._calls

    # -- host copies
    def out_host(self) -> np.ndarray:
        return bf16_to_numpy(self.out)

    def pool_host(self) -> np.ndarray:
        return bf16_to_numpy(self.kv_cache).reshape(self.step.kv_cache.shape)

    def slots_host(self) -> np.ndarray:
        return self.slot_mapping.cpu().numpy()
