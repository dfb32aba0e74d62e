"""Cross-batch scheduling over a ragged pool (EXSPEC), host side.

"Correctness Forensics for Batch Speculative Decoding", §3.2: EXSPEC keeps
sequences ragged and forms batches of identical-length sequences, bypassing
realignment when lengths match; when grouping fails it falls back to
unpad-append-repad, and a sliding window of more than B sequences raises the
chance of a same-length group.  The pages give no algorithm (the appendix is a
bare heading), so the policy here is this library's:

  window   the first `window` active sequences in pool order;
  group    spec_group_by_length over the window: the largest same-length
           bucket (ties to the shorter length), members by pool index, the
           rest filled by nearest length;
  grouped  a full group of B equal lengths is verified in place on the pool
           and committed with spec_commit_ragged (no KV moves);
  fallback otherwise the B chosen sequences are repadded into a batch
           (spec_repad_gather), run as an ordinary round there (verify,
           spec_realign_kv, spec_rebuild_pos_mask) and unpadded back
           (spec_unpad_scatter).

Everything the round computes runs in the library's kernels; this module
only keeps the request bookkeeping and calls them.
"""
from __future__ import annotations

import numpy as np
import torch

from . import api


class ExspecScheduler:
    def __init__(self, pool_len: torch.Tensor, B: int, window: int):
        if window < 1 or B < 1:
            raise ValueError("B and window must be positive")
        self.pool_len = pool_len
        self.N = pool_len.shape[0]
        self.B, self.window = int(B), int(window)
        dev = pool_len.device
        self._mask_h = torch.zeros(self.N, dtype=torch.uint8).pin_memory()
        self._mask_d = torch.zeros(self.N, dtype=torch.uint8, device=dev)
        # the kernel's three outputs side by side: one copy brings them back
        self._out_d = torch.empty(self.B + 2, dtype=torch.int32, device=dev)
        self.idx = self._out_d[: self.B]
        self.count_equal = self._out_d[self.B:self.B + 1]
        self.group_len = self._out_d[self.B + 1:]
        self._out_h = torch.empty(self.B + 2, dtype=torch.int32).pin_memory()

    def select_async(self, active: np.ndarray, stream=None):
        """Enqueue the selection for the active mask (bool [N], host)."""
        win = np.flatnonzero(active)[: self.window]
        m = self._mask_h.numpy()
        m[:] = 0
        m[win] = 1
        self._mask_d.copy_(self._mask_h, non_blocking=True)
        api.spec_group_by_length(self.pool_len, self.B, active=self._mask_d, out_idx=self.idx,
                                 out_count_equal=self.count_equal, out_group_len=self.group_len, stream=stream)
        self._out_h.copy_(self._out_d, non_blocking=True)

    def selection(self):
        """After the stream reached select_async's copies: (pool indices of
        the chosen sequences, whether they form a full same-length group,
        that length)."""
        out = self._out_h.numpy()
        picks = out[: self.B]
        picks = picks[picks >= 0]
        full = int(out[self.B]) == self.B and len(picks) == self.B
        return picks.copy(), full, int(out[self.B + 1])
