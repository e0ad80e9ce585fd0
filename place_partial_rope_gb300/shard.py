"""Data-parallel split of one workload's tokens across ranks.

One process per GPU, and nothing is exchanged: every row (b, s, n) of the
rotation needs only itself and its own cos/sin row, so rank r rotates the
rows of its own tokens with its own cos/sin rows.  This is the token-range
convention of "CANN ops-transformer aclnnMoeTokenUnpermuteWithEpGrad"
(section 一: each device handles only the tokens in [range[0], range[1])).

The split itself is the library's ``rope_partial_token_shard`` (host logic,
no CUDA call): rank r owns the tokens [t0, t1) of the flattened b * S + s
order, balanced to one token, as at most three runs that are each one
contiguous block of a BSND tensor (the end of a batch entered mid-way,
whole batches, the start of a batch).  This module turns a rank's share
into views: the run's block of the rank's own (t1 - t0, N, D) buffer and
the run's rows of a cos/sin (or positions) array, ready for one call of
the library per run.

Weak scaling grows the workload with the number of ranks (B * world
batches, each rank holding B of them); strong scaling splits the named
workload itself, so ranks may hold parts of a batch.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

from . import binding, synth


@dataclass(frozen=True)
class Run:
    """Batches [b0, b0 + nb) x positions [s0, s0 + ns); nb == 1 or ns == S."""
    b0: int
    s0: int
    nb: int
    ns: int

    @property
    def tokens(self) -> int:
        return self.nb * self.ns


@dataclass(frozen=True)
class Share:
    """A rank's tokens [t0, t1) of a (B, S) grid and their runs, in order."""
    B: int
    S: int
    t0: int
    t1: int
    runs: tuple

    @property
    def tokens(self) -> int:
        return self.t1 - self.t0

    def offset(self, run: Run) -> int:
        """Tokens between the share's first token and the run's."""
        return run.b0 * self.S + run.s0 - self.t0


def token_share(B: int, S: int, rank: int, world: int) -> Share:
    t0, t1, runs = binding.rope_partial_token_shard(B, S, rank, world)
    return Share(B, S, t0, t1, tuple(Run(*r) for r in runs))


def run_block(buf, share: Share, run: Run):
    """The run's (nb, ns, N, D) block of a rank's (t1 - t0, N, D) buffer (a
    view: numpy array or torch tensor)."""
    o = share.offset(run)
    blk = buf[o:o + run.tokens]
    shape = (run.nb, run.ns) + tuple(buf.shape[1:])
    return blk.reshape(shape) if isinstance(blk, np.ndarray) else blk.view(shape)


def run_rows(a, run: Run):
    """The run's rows of an array whose first two dims are (batch, position)
    or broadcast (size 1): cos/sin of shape (Br, Sr, Nr, L), or positions."""
    bs = slice(run.b0, run.b0 + run.nb) if a.shape[0] > 1 else slice(0, 1)
    ss = slice(run.s0, run.s0 + run.ns) if a.shape[1] > 1 else slice(0, 1)
    return a[bs, ss]


def weak_workload(w: synth.Workload, world: int) -> synth.Workload:
    """The workload of `world` ranks under weak scaling: B * world batches
    (cos/sin kept per batch where the named workload has them per batch),
    so each rank holds as many tokens as the named workload has."""
    if world == 1:
        return w
    B, S, N, D = w.shape
    Br = w.r_shape[0] * world if w.r_shape[0] > 1 else 1
    return dataclasses.replace(w, shape=(B * world, S, N, D), r_shape=(Br,) + tuple(w.r_shape[1:]))


@dataclass
class RankInputs:
    """A rank's host inputs: its tokens' rows of x and grad as (T, N, D)
    buffers (seeded N(0,1): the rank's own activations), and per run the
    cos/sin rows of its tokens (built from the global workload's positions,
    so a rank holding batch b uses batch b's position offset)."""
    workload: synth.Workload   # the global workload
    share: Share
    x: np.ndarray
    g: np.ndarray | None
    tables: list               # per run: (r1, r2) of shape (nb | 1, ns | 1, Nr, L)

    def algorithmic_bytes(self) -> int:
        """Slice bytes read + written plus the cos/sin bytes, of one launch
        per run (one direction)."""
        w = self.workload
        e = synth.ELEM_BYTES[w.dtype]
        N = w.shape[2]
        return sum(2 * run.tokens * N * w.L * e + 2 * r1.size * e
                   for run, (r1, _) in zip(self.share.runs, self.tables))


def rank_inputs(w: synth.Workload, rank: int, world: int, weak: bool = True) -> RankInputs:
    """Rank `rank`'s inputs for the named workload `w` on `world` ranks.  With
    one rank they are the named workload's own inputs (same values)."""
    wg = weak_workload(w, world) if weak else w
    B, S, N, D = wg.shape
    share = token_share(B, S, rank, world)
    x = synth.normal((share.tokens, N, D), w.dtype, w.seed + 1009 * rank)
    g = (synth.normal((share.tokens, N, D), w.dtype, w.seed + 500 + 1009 * rank)
         if "bwd" in w.directions else None)
    pos = synth.positions(wg)
    tables = [synth.rope_table(np.ascontiguousarray(run_rows(pos, run)), w.L, w.dtype)
              for run in share.runs]
    return RankInputs(wg, share, x, g, tables)
