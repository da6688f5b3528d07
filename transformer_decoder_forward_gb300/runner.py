"""Drive the C ABI over one synthetic workload: device weights, block tables, buffers.

Used by the tests and the bench; a user would write the same few calls. Nothing
here computes any part of the forward pass.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

import workloads as wl
from . import Decoder, upload_weights


class WorkloadRun:
    def __init__(self, w: wl.Workload, host_weights: Optional[wl.Weights] = None, dev_w=None,
                 max_prefill_tokens: Optional[int] = None, batch: Optional[int] = None, extra_steps: int = 0,
                 lengths: Optional[np.ndarray] = None):
        import torch
        self.wl = w
        s = w.model
        self.shape = s
        all_lengths = np.asarray(lengths, dtype=np.int32) if lengths is not None else w.lengths()
        self.B = batch or len(all_lengths)
        self.lengths = all_lengths[: self.B]
        self.prompts = wl.draw_prompts(all_lengths, s.vocab)[: self.B]
        steps = w.decode_steps + extra_steps
        self.ctx = self.lengths + steps                         # slots each sequence will hold
        if w.contiguous_kv:
            self.mbps = wl.blocks_needed(int(self.ctx.max()))
            self.tables_np = wl.identity_tables(self.B, self.mbps)
            self.n_blocks = self.B * self.mbps
        else:
            self.mbps = wl.blocks_needed(int(self.ctx.max()))
            self.tables_np, self.n_blocks = wl.make_block_tables(self.ctx, self.mbps, shuffle=w.shuffle_tables)
        if dev_w is None:
            if host_weights is None:
                host_weights = wl.make_weights(s, scale=w.weight_scale)
            dev_w = upload_weights(host_weights)
        self.dev_w = dev_w
        mpt = max_prefill_tokens or max(int(self.lengths.max()), min(int(self.lengths.sum()), 16384))
        self.dec = Decoder(s, dev_w, max_batch=self.B, max_blocks_per_seq=self.mbps, num_kv_blocks=self.n_blocks,
                           max_prefill_tokens=mpt, contiguous_kv=w.contiguous_kv, kv_dtype=w.kv_dtype)
        dev = "cuda"
        self.tables = torch.from_numpy(self.tables_np).to(dev)
        self.tokens = torch.from_numpy(np.concatenate(self.prompts).astype(np.int32)).to(dev)
        self.next_ids = torch.zeros(self.B, dtype=torch.int32, device=dev)
        self.positions = torch.from_numpy(self.lengths.astype(np.int32)).to(dev)
        self.step_tokens = torch.zeros(self.B, dtype=torch.int32, device=dev)
        # positions of every decode step, built once: row i = lengths + i
        self.step_positions = (torch.from_numpy(self.lengths.astype(np.int32)).to(dev)[None, :]
                               + torch.arange(max(steps, 1), dtype=torch.int32, device=dev)[:, None]).contiguous()
        torch.cuda.synchronize()

    @property
    def stream(self):
        return self.dec.stream

    def prefill(self, logits=None):
        import torch
        with torch.cuda.stream(self.stream):
            self.dec.prefill(self.tokens, [int(x) for x in self.lengths], self.tables, self.next_ids, logits)

    def decode(self, tokens_dev, step: int, logits=None, next_ids=None):
        """Decode step `step` (0-based): each sequence feeds one token at position length + step."""
        import torch
        with torch.cuda.stream(self.stream):
            self.dec.decode_step(tokens_dev, self.step_positions[step], self.tables, next_ids if next_ids is not None else self.next_ids,
                                 logits)

    def decode_sample(self, tokens_dev, step: int, temperature: float, top_k: int, uniforms, logits=None,
                      next_ids=None):
        """Decode step `step` that samples the next token (temperature, top-k, the caller's uniforms)."""
        import torch
        with torch.cuda.stream(self.stream):
            self.dec.decode_step_sample(tokens_dev, self.step_positions[step], self.tables, temperature, top_k, uniforms,
                                        next_ids if next_ids is not None else self.next_ids, logits)

    def close(self):
        self.dec.close()
