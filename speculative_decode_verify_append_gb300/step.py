"""One verify step as a user runs it: append the window, attend, accept.

``VerifyStep`` owns the per-shape device buffers (attention output,
split-K workspace, accept outputs, status word) so that a serving loop, or
a CUDA graph capture, issues exactly the three library calls per step with
no allocation.  ``fill_context`` writes a lane's prompt K/V into the cache in
page-aligned chunks (the prefill side of the same append call).
"""
from __future__ import annotations

import math

import torch

from . import (KVCache, kv_append_quant, kv_append_quant_ragged, spec_accept, spec_accept_lazy, verify_attn,
               verify_attn_workspace_size, verify_step)


class VerifyStep:
    def __init__(self, num_lanes: int, window: int, num_q_heads: int, num_kv_heads: int, max_context: int,
                 vocab: int | None, device="cuda", sm_scale: float | None = None):
        self.num_lanes, self.window = num_lanes, window
        self.num_q_heads, self.num_kv_heads = num_q_heads, num_kv_heads
        self.max_context, self.vocab = max_context, vocab
        self.sm_scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(128.0)
        dev = torch.device(device)
        self.out = torch.empty((num_lanes, window, num_q_heads, 128), dtype=torch.bfloat16, device=dev)
        nbytes = verify_attn_workspace_size(num_lanes, window, num_q_heads, num_kv_heads, max_context)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self.accept_len = torch.zeros(num_lanes, dtype=torch.int32, device=dev)
        self.out_tokens = torch.zeros((num_lanes, window), dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def append(self, cache: KVCache, k_win, v_win, page_table, seq_lens, stream=None):
        kv_append_quant(cache, k_win, v_win, page_table, seq_lens, self.status, stream)

    def append_ragged(self, cache: KVCache, k_win, v_win, n_lane, page_table, seq_lens, stream=None):
        """Lane b appends only its first n_lane[b] window tokens (its own 1 + d_b)."""
        kv_append_quant_ragged(cache, k_win, v_win, n_lane, page_table, seq_lens, self.status, stream)

    def attend(self, cache: KVCache, q, page_table, seq_lens, stream=None):
        verify_attn(cache, q, page_table, seq_lens, self.max_context, self.sm_scale, self.out, self.workspace,
                    self.status, stream)

    def accept(self, logits, drafts, seq_lens_inout=None, stream=None):
        spec_accept(logits, drafts, self.accept_len, self.out_tokens, seq_lens_inout, self.status, stream)

    def accept_lazy(self, logits, drafts, num_drafts=None, seq_lens_inout=None, stream=None):
        """Acceptance reading each lane's rows only up to its first disagreement."""
        spec_accept_lazy(logits, drafts, self.accept_len, self.out_tokens, num_drafts, seq_lens_inout, self.status,
                         stream)

    def step(self, cache: KVCache, q, k_win, v_win, page_table, seq_lens, logits, drafts, commit: bool = True,
             stream=None):
        """The whole step in one library call (verify_step): the same results
        as run(), the three calls chained as programmatic dependent launches."""
        verify_step(cache, k_win, v_win, q, page_table, seq_lens, self.max_context, self.sm_scale, self.out,
                    self.workspace, logits, drafts, self.accept_len, self.out_tokens, commit, self.status, stream)

    def run(self, cache: KVCache, q, k_win, v_win, page_table, seq_lens, logits=None, drafts=None,
            commit: bool = True, stream=None):
        """append -> verify_attn -> spec_accept on one stream; seq_lens is
        advanced by 1 + accept_len when commit is true and logits are given."""
        self.append(cache, k_win, v_win, page_table, seq_lens, stream)
        self.attend(cache, q, page_table, seq_lens, stream)
        if logits is not None:
            self.accept(logits, drafts, seq_lens if commit else None, stream)


def fill_context(cache: KVCache, k: torch.Tensor, v: torch.Tensor, page_table_row: torch.Tensor, start: int = 0,
                 chunk: int = 4096, status: torch.Tensor | None = None, stream=None) -> None:
    """Append tokens [start, start + len(k)) of one lane.  k, v: bf16
    [n][Hkv][128] on the device; page_table_row: int32 [max_pages] (device)."""
    n = k.shape[0]
    dev = k.device
    row = page_table_row.reshape(1, -1)
    t = 0
    while t < n:
        c = min(chunk - ((start + t) % chunk), n - t)
        lens = torch.tensor([start + t], dtype=torch.int32, device=dev)
        kv_append_quant(cache, k[t:t + c].unsqueeze(0).contiguous(), v[t:t + c].unsqueeze(0).contiguous(), row,
                        lens, status, stream)
        t += c
