"""A decode loop around the compression step.

The method's write-up (yeyulingfeng.com TriAttention article, section 主要方法,
pruning paragraph) runs the compression once every 128 generated tokens, when a
cache exceeds its budget, during online decoding.  DecodeLoop is the host side
of that loop on one cache: per token it appends the token's K/V to every unit
(tri_append_kv) and attends (tri_decode_attention); every `window` tokens it
calls tri_compress_step.  It only orders the calls and swaps buffers (the
sequence lengths and positions are double-buffered because each call writes
the next lengths or positions while its CTAs still read the current ones);
every step runs in libtri's kernels.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import tri as T


class DecodeLoop:
    def __init__(self, cache: T.KVCache, stats: T.Stats, theta: float, offsets: Sequence[int], budget: int,
                 pos: torch.Tensor, window: int = 128, compact: str = "ordered", pairing: str = "half",
                 scale: Optional[float] = None, stream=None):
        """cache: the KV cache (its seq_len is the current length of every
        sequence); pos [S] int32: the position of each sequence's next token."""
        self.cache, self.stats, self.theta = cache, stats, float(theta)
        self.offsets, self.budget, self.window = list(offsets), int(budget), int(window)
        self.compact, self.pairing, self.stream = compact, pairing, stream
        self.scale = scale
        self.Hq = stats.Hq
        self.len_bufs = [cache.seq_len, cache.seq_len.clone()]
        self.pos_bufs = [pos, pos.clone()]
        self.tokens = 0
        dev = cache.k.device
        self.idx = torch.empty((cache.L, cache.S, cache.Hkv, self.budget), dtype=torch.int32, device=dev)
        n = T.tri_decode_workspace_bytes(cache, self.Hq)
        self.dec_ws = None if n == 0 else torch.empty(n, dtype=torch.uint8, device=dev)
        self.cmp_ws = T.workspace(cache, stats, self._params())
        self.out = None

    @property
    def pos(self) -> torch.Tensor:
        return self.pos_bufs[0]

    def _params(self) -> T.Params:
        return T.Params(self.theta, self.pos_bufs[0], self.offsets, self.budget, pairing=self.pairing)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor) -> None:
        T.tri_append_kv(self.cache, k_new, v_new, self.pos_bufs[0], self.theta, self.len_bufs[1],
                        pos_out=self.pos_bufs[1], pairing=self.pairing, stream=self.stream)
        self.len_bufs.reverse()
        self.cache.seq_len = self.len_bufs[0]

    def attend(self, q: torch.Tensor) -> torch.Tensor:
        self.out = T.tri_decode_attention(self.cache, q, self.pos_bufs[0], self.theta, scale=self.scale,
                                          out=self.out, ws=self.dec_ws, pairing=self.pairing, stream=self.stream)
        return self.out

    def advance(self) -> bool:
        """Moves every sequence to its next position (written by the append);
        returns True when the token count reaches a multiple of the window
        (compress now)."""
        self.pos_bufs.reverse()
        self.tokens += 1
        return self.tokens % self.window == 0

    def compress(self) -> torch.Tensor:
        """tri_compress_step with t = the next query position; returns idx_out
        (the original slot of the row now at each kept slot)."""
        T.tri_compress_step(self.cache, self.stats, self._params(), idx_out=self.idx, new_len=self.len_bufs[1],
                            ws=self.cmp_ws, stream=self.stream, compact=self.compact)
        self.len_bufs.reverse()
        self.cache.seq_len = self.len_bufs[0]
        return self.idx

    def step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor) -> torch.Tensor:
        """One decoded token for every sequence: append, attend, advance, and
        compress at the window boundary.  Returns the attention output."""
        self.append(k_new, v_new)
        out = self.attend(q)
        if self.advance():
            self.compress()
        return out
