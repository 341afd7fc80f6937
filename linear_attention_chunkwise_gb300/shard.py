"""Splitting one packed batch across ranks (one process per GPU).

(sequence, head) units of the prefill never exchange data: each sequence's
recurrence starts from its own S0 and ends in its own S_final.  A batch is
therefore split across ranks by whole sequences, with no collective on the
data path: rank r runs kda_prefill (or its backward) on its slice of the
packed tensors, with its own cu_seqlens rebased to start at 0, and its
outputs are exactly that slice of the single-rank outputs.

The split is contiguous in sequence order (so every rank's tokens are one
slice of the packed [T, ...] tensors) and balances tokens: rank r takes the
sequences whose token midpoints fall in [r T / W, (r + 1) T / W).  Heads can
be split the same way (`split_heads`), since heads are independent too.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Shard:
    """Rank `rank`'s part of a packed batch: sequences [seq_begin, seq_end), tokens [tok_begin, tok_end)."""
    rank: int
    seq_begin: int
    seq_end: int
    tok_begin: int
    tok_end: int
    cu_seqlens: np.ndarray  # int32 [seq_end - seq_begin + 1], starts at 0

    @property
    def num_seqs(self) -> int:
        return self.seq_end - self.seq_begin

    @property
    def num_tokens(self) -> int:
        return self.tok_end - self.tok_begin

    def tokens(self, x):
        """The rank's rows of a packed [T, ...] tensor (a view)."""
        return x[self.tok_begin:self.tok_end]

    def seqs(self, x):
        """The rank's rows of a per-sequence [N, ...] tensor (S0, S_final, grad_S0), or None."""
        return None if x is None else x[self.seq_begin:self.seq_end]


def split_sequences(cu_seqlens, world: int) -> list[Shard]:
    """Contiguous, token-balanced split of a packed batch's sequences over `world` ranks.

    cu_seqlens: host array-like [N + 1], 0 = c_0 <= c_1 <= ... <= c_N = T.  Sequence n goes to the
    rank whose token range [r T / W, (r + 1) T / W) holds the midpoint of [c_n, c_{n+1}) (empty
    sequences: their start).  Every rank gets a Shard, possibly with no sequences.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64).reshape(-1)
    if world < 1:
        raise ValueError("world must be >= 1")
    if cu.size < 1 or cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0 and be non-decreasing")
    n, total = cu.size - 1, int(cu[-1])
    mid2 = cu[:-1] + cu[1:]  # twice the midpoints, exact in integers
    owner = np.minimum((mid2 * world) // max(2 * total, 1), world - 1) if total > 0 else np.zeros(n, np.int64)
    shards = []
    start = 0
    for r in range(world):
        end = start + int(np.count_nonzero(owner == r))
        local = (cu[start:end + 1] - cu[start]).astype(np.int32)
        shards.append(Shard(r, start, end, int(cu[start]), int(cu[end]), local))
        start = end
    assert start == n
    return shards


def split_heads(H: int, world: int) -> list[tuple[int, int]]:
    """Contiguous head ranges [h0, h1) per rank, sizes differing by at most one."""
    if world < 1 or H < 0:
        raise ValueError("world must be >= 1 and H >= 0")
    base, extra = divmod(H, world)
    out, h0 = [], 0
    for r in range(world):
        h1 = h0 + base + (1 if r < extra else 0)
        out.append((h0, h1))
        h0 = h1
    return out
