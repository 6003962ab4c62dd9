"""A seeded decode batch resident on the device, driven through the C ABI.

``DecodeBatch`` holds one workload's pools and step inputs in device memory
(filled by the library's own slot mapping and append from the generator's
token values) and runs the step's public calls on them: the fused decode step,
the shared-prefix step, the multi-token step, or the three separate calls.
It is how ``bench.py`` and the GPU tests drive the library; it adds no
arithmetic of its own.  ``wl`` is any object with the seeded workload's
attributes (``spec``, ``block_tables``, ``seq_lens``, ``q``, ``new_k``,
``new_v``, ``poisoned_pool()``, ``scales()``, ``fill_chunks()``, ...).
"""
import numpy as np
import torch

import paged_kv_cache_97_gb300 as pkv


def to_dev_bf16(bits: np.ndarray, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def bits_of(t: torch.Tensor) -> np.ndarray:
    """Raw bits of a device tensor (bf16 -> uint16, int8 -> int8, E4M3 ->
    uint8), the oracle's pool dtypes."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).cpu().numpy()
    return t.cpu().numpy()


def dev_pool(host: np.ndarray, dev="cuda") -> torch.Tensor:
    """A device pool from the oracle's host layout (uint16 bf16 bits, int8
    codes or uint8 E4M3 codes)."""
    if host.dtype == np.uint16:
        return to_dev_bf16(host, dev)
    if host.dtype == np.uint8:
        return torch.from_numpy(np.ascontiguousarray(host)).to(dev).view(torch.float8_e4m3fn)
    return torch.from_numpy(np.ascontiguousarray(host)).to(dev)


class DecodeBatch:
    """A workload's pools and step inputs on the device, filled by the
    library's own slot mapping and append."""

    def __init__(self, wl, dev="cuda", fill=True, seqs=None):
        s = wl.spec
        self.wl, self.dev = wl, dev
        self.q8 = s.kv_dtype != "bf16"
        poison = wl.poisoned_pool()
        if self.q8:
            self.k_cache = dev_pool(poison, dev)
            self.v_cache = self.k_cache.clone()
            ks, vs = wl.scales(seqs)
            self.k_scale = torch.from_numpy(ks).to(dev)
            self.v_scale = torch.from_numpy(vs).to(dev)
        else:
            self.k_cache = to_dev_bf16(poison, dev)
            self.v_cache = self.k_cache.clone()
            self.k_scale = self.v_scale = None
        del poison
        self.block_tables = torch.from_numpy(wl.block_tables).to(dev)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(dev)
        self.q = to_dev_bf16(wl.q, dev)
        self.new_k = to_dev_bf16(wl.new_k, dev)
        self.new_v = to_dev_bf16(wl.new_v, dev)
        B = s.batch
        self.slots = torch.empty(B, dtype=torch.int64, device=dev)
        self.out = torch.empty((B, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device=dev)
        self.max_seq_len = int(wl.seq_lens.max())
        ws = pkv.workspace_bytes(B, s.num_q_heads, s.head_dim, self.max_seq_len, s.block_size)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        if fill:
            self.fill(seqs)

    def fill(self, seqs=None):
        wl, s = self.wl, self.wl.spec
        for ch in wl.fill_chunks(seqs):
            n = ch.positions.shape[0]
            pos = torch.from_numpy(ch.positions).to(self.dev)
            sid = torch.from_numpy(ch.seq_idx).to(self.dev)
            slots = torch.empty(n, dtype=torch.int64, device=self.dev)
            pkv.token_slot_mapping(self.block_tables, pos, wl.num_blocks, s.block_size, slots, seq_idx=sid)
            pkv.reshape_and_cache(to_dev_bf16(ch.k, self.dev), to_dev_bf16(ch.v, self.dev),
                                  self.k_cache, self.v_cache, slots, self.k_scale, self.v_scale)
        torch.cuda.synchronize()

    def append(self):
        s = self.wl.spec
        pkv.slot_mapping(self.block_tables, self.seq_lens, self.wl.num_blocks, s.block_size, self.slots)
        pkv.reshape_and_cache(self.new_k, self.new_v, self.k_cache, self.v_cache, self.slots,
                              self.k_scale, self.v_scale)

    def attend(self, max_seq_len=None):
        s = self.wl.spec
        pkv.paged_attention_decode(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                   self.seq_lens, max_seq_len or self.max_seq_len, s.scale,
                                   workspace=self.workspace, k_scale=self.k_scale, v_scale=self.v_scale)
        return self.out

    def step(self):
        self.append()
        return self.attend()

    def prefix_step(self, append=True):
        """pagedkv_decode_step_prefix with the workload's shared prefix."""
        s = self.wl.spec
        P = s.shared_prefix_tokens // s.block_size
        if not hasattr(self, "prefix_blocks"):
            self.prefix_blocks = self.block_tables[0, :P].contiguous()
            ws = pkv.prefix_workspace_bytes(s.batch, s.num_q_heads, s.head_dim, self.max_seq_len,
                                            s.block_size, P)
            self.prefix_ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=self.dev)
        pkv.decode_step_prefix(self.out, self.q, self.new_k if append else None,
                               self.new_v if append else None, self.k_cache, self.v_cache,
                               self.block_tables, self.seq_lens, self.max_seq_len, s.scale,
                               self.prefix_blocks, self.prefix_ws, k_scale=self.k_scale,
                               v_scale=self.v_scale)
        return self.out

    def append_tokens(self):
        """Append every new token of the step (several per sequence for
        multi-token workloads) through the general slot mapping."""
        s = self.wl.spec
        seq, pos = self.wl.new_positions()
        if not hasattr(self, "tok_slots"):
            self.tok_seq = torch.from_numpy(seq).to(self.dev)
            self.tok_pos = torch.from_numpy(pos).to(self.dev)
            self.tok_slots = torch.empty(len(seq), dtype=torch.int64, device=self.dev)
        pkv.token_slot_mapping(self.block_tables, self.tok_pos, self.wl.num_blocks, s.block_size,
                               self.tok_slots, seq_idx=self.tok_seq)
        pkv.reshape_and_cache(self.new_k, self.new_v, self.k_cache, self.v_cache, self.tok_slots,
                              self.k_scale, self.v_scale)

    def _multi_buffers(self):
        s = self.wl.spec
        if not hasattr(self, "query_start"):
            self.query_start = torch.from_numpy(self.wl.query_start).to(self.dev)
            self.out_multi = torch.empty((self.wl.num_tokens, s.num_q_heads, s.head_dim),
                                         dtype=torch.bfloat16, device=self.dev)
            ws = pkv.multi_workspace_bytes(self.wl.num_tokens, s.num_q_heads, s.head_dim,
                                           self.max_seq_len, s.block_size)
            self.ws_multi = torch.empty(max(ws, 16), dtype=torch.uint8, device=self.dev)

    def attend_multi(self):
        """paged_attention_multi over the step's query tokens."""
        self._multi_buffers()
        pkv.paged_attention_multi(self.out_multi, self.q, self.k_cache, self.v_cache,
                                  self.block_tables, self.seq_lens, self.query_start,
                                  self.max_seq_len, max(int(self.wl.query_lens.max()), 1),
                                  self.wl.spec.scale, self.ws_multi, self.k_scale, self.v_scale)
        return self.out_multi

    def multi_step(self):
        """pagedkv_multi_step: the step's append and attention in one call."""
        self._multi_buffers()
        pkv.multi_step(self.out_multi, self.q, self.new_k, self.new_v, self.k_cache, self.v_cache,
                       self.block_tables, self.seq_lens, self.query_start, self.max_seq_len,
                       max(int(self.wl.query_lens.max()), 1), self.wl.spec.scale, self.ws_multi,
                       self.k_scale, self.v_scale)
        return self.out_multi

    def multi_step_unfused(self):
        """The same step as three calls: token slot mapping, reshape_and_cache,
        paged_attention_multi."""
        self.append_tokens()
        return self.attend_multi()

    def fused_step(self):
        """pagedkv_decode_step through a plan prepared once per set of
        buffers (the bench alternates two sets)."""
        key = tuple(id(t) for t in (self.out, self.q, self.new_k, self.new_v, self.k_cache,
                                    self.v_cache, self.block_tables, self.seq_lens,
                                    self.workspace))
        plans = self.__dict__.setdefault("_plans", {})
        plan = plans.get(key)
        if plan is None:
            if len(plans) >= 4:
                plans.clear()
            plan = plans[key] = pkv.DecodeStepPlan(
                self.out, self.q, self.new_k, self.new_v, self.k_cache, self.v_cache,
                self.block_tables, self.seq_lens, self.max_seq_len, self.wl.spec.scale,
                self.workspace, k_scale=self.k_scale, v_scale=self.v_scale)
        return plan()
