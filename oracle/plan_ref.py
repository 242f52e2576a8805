"""Reference split-KV plan (plain Python).  TEST INFRASTRUCTURE ONLY.

The pages describe splitting each request's cache into chunks for decode
attention (page 2, section 1.4 "Append Attention 优化",
FLAGS_cascade_attention_max_partition_size) and merging the chunks afterwards.
They do not fix a rule, so the plan used here is a plain balanced partition:

* Work units are (row block, request) pairs, ordered row-block-major:
  ``u = rb * B + b``.  A row block is 128 consecutive query rows of one
  request (rows are ``i * H + h`` for new token i and head h).
* A unit needs ``tiles_u = ceil(n_max / 64)`` KV pages, where ``n_max`` is the
  number of keys visible to the last row of the block
  (``seqlen - s_q + i_last + 1``, clipped to ``[0, max_pages*64]``).
* Its cost is ``tiles_u + overhead``.  The units of one row block are laid
  out back to back on a cost axis; unit u covers ``[pre[u], end[u])`` with
  ``end[u] = pre[u] + cost``.  Cluster c owns the cost range
  ``[c*W, (c+1)*W)``.
* With several row blocks (``n_rb > 1``) and at least ``n_rb`` clusters, each
  row block gets its own ``Gl = G // n_rb`` clusters: row block r starts at
  ``r * Gl * W`` with ``W = max_r ceil(total_r / Gl)``, so cluster
  ``r * Gl + g`` covers the same stretch of every request's pages for each
  r, and the row blocks of a request read each page at about the same time
  (the second read comes from L2).  Clusters past ``n_rb * Gl`` and the end
  of a row block's stretch stay idle.  Otherwise the row blocks follow each
  other and ``W = ceil(total / G)``.
* The pages of unit u sit at cost ``[pre[u] + overhead, end[u])``; a unit
  with no pages sits at ``pre[u]``.  A unit whose pages cross a cluster
  boundary is split; each piece writes a partial result into slot ``2c``
  (piece starts at ``c*W``) or ``2c+1`` (otherwise), and the combine step
  merges the pieces.
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence

PAGE = 64
ROWS_PER_BLOCK = 128
DEFAULT_OVERHEAD = 4  # the planner's cost per unit when the descriptor leaves it 0


@dataclasses.dataclass(frozen=True)
class Piece:
    unit: int
    b: int
    rb: int
    page_lo: int
    page_hi: int
    split: bool
    slot: int


@dataclasses.dataclass
class Plan:
    B: int
    s_q: int
    H: int
    G: int
    overhead: int
    n_rb: int
    tiles: List[int]
    pre: List[int]   # unit starts, then pre[U] = the end of the last unit
    W: int
    ends: List[int]  # end of each unit's cost range

    @property
    def rb_ends(self) -> List[int]:
        """End of each row block's stretch (the end of its last unit)."""
        return [self.ends[(r + 1) * self.B - 1] for r in range(self.n_rb)]

    @property
    def units(self) -> int:
        return len(self.tiles)

    def first_unit(self, c: int) -> int:
        """The unit containing cost point c*W (units if the range is past the end)."""
        x = c * self.W
        for u in range(self.units):
            if self.pre[u] <= x < self.ends[u]:
                return u
        return self.units

    def pieces(self, c: int) -> List[Piece]:
        """Segments cluster c processes, in order."""
        lo_c, hi_c = c * self.W, (c + 1) * self.W
        out = []
        for u in range(self.units):
            if self.ends[u] <= lo_c or self.pre[u] >= hi_c:
                continue
            b, rb = u % self.B, u // self.B
            if self.tiles[u] == 0:
                if lo_c <= self.pre[u] < hi_c:
                    out.append(Piece(u, b, rb, 0, 0, False, -1))
                continue
            a, e = self.pre[u] + self.overhead, self.ends[u]
            lo, hi = max(a, lo_c), min(e, hi_c)
            if lo >= hi:
                continue
            split = a < lo_c or e > hi_c
            slot = (2 * c if lo == lo_c else 2 * c + 1) if split else -1
            out.append(Piece(u, b, rb, lo - a, hi - a, split, slot))
        return out

    def piece_count(self, u: int) -> int:
        """Number of clusters unit u's pages fall in (0 for a unit with no pages)."""
        if self.tiles[u] == 0:
            return 0
        return len({c for c in range(self.G) for p in self.pieces(c) if p.unit == u})

    def combine_unit(self, c: int):
        """(unit, [(cluster, slot), ...]) the combine step of cluster c merges, or None."""
        lo_c, hi_c = c * self.W, (c + 1) * self.W
        x = hi_c - 1
        u = None
        for v in range(self.units):
            if self.pre[v] <= x < self.ends[v]:
                u = v
                break
        if u is None or self.tiles[u] == 0:
            return None
        a, e = self.pre[u] + self.overhead, self.ends[u]
        if not (lo_c <= a <= x and e > hi_c):
            return None
        last = (e - 1) // self.W
        pieces = []
        for cc in range(c, last + 1):
            slot = 2 * cc + 1 if (cc == c and a != lo_c) else 2 * cc
            pieces.append((cc, slot))
        return u, pieces


def unit_tiles(seqlen: int, s_q: int, H: int, rb: int, max_pages: int) -> int:
    R = s_q * H
    r_last = min(R, (rb + 1) * ROWS_PER_BLOCK) - 1
    i_last = r_last // H
    n = seqlen - s_q + i_last + 1
    n = max(0, min(n, max_pages * PAGE))
    return (n + PAGE - 1) // PAGE


def make_plan(seqlens: Sequence[int], s_q: int, H: int, max_pages: int, G: int, overhead: int) -> Plan:
    B = len(seqlens)
    R = s_q * H
    n_rb = (R + ROWS_PER_BLOCK - 1) // ROWS_PER_BLOCK
    tiles = []
    for rb in range(n_rb):
        for b in range(B):
            tiles.append(unit_tiles(int(seqlens[b]), s_q, H, rb, max_pages))
    totals = [sum(t + overhead for t in tiles[r * B:(r + 1) * B]) for r in range(n_rb)]
    if n_rb > 1 and G >= n_rb:
        gl = G // n_rb
        W = max(1, max((t + gl - 1) // gl for t in totals))
        base = [r * gl * W for r in range(n_rb)]
    else:
        W = max(1, (sum(totals) + G - 1) // G)
        base = [sum(totals[:r]) for r in range(n_rb)]
    pre, ends = [], []
    for r in range(n_rb):
        x = base[r]
        for b in range(B):
            pre.append(x)
            x += tiles[r * B + b] + overhead
            ends.append(x)
    pre.append(ends[-1])
    return Plan(B, s_q, H, G, overhead, n_rb, tiles, pre, W, ends)
