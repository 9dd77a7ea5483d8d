"""Expert parallelism for the Switch layer: experts sharded over ranks, two all-to-alls.

The Switch Transformers card (ai-papers.xuzou.cn, section 方法适配) shards the experts over
the cores: each core routes its own tokens, an all-to-all sends every token to the core that
holds its expert, the experts run, and a second all-to-all brings the outputs back for the
combine.  Here a rank owns a contiguous range of experts and routes its own G routing
groups; the first all-to-all moves fixed-size chunks [El, R, d] of each rank's dispatched
buffer (R = its expert block rows, the pages' [E, C, d] per core), plus the valid row count
of every block; the receiver packs each local expert's rows source by source
(switch_ep_regroup), runs the expert FFN on them and unpacks the outputs into chunks for
the return all-to-all.  Routing, capacity and statistics stay per group and per rank, so
the result equals the single-rank layer over all ranks' groups.

Host logic (ExpertShards) is plain Python; the data plane (ExpertParallelSwitch) calls the
CUDA library for every step on the GPU and torch.distributed (NCCL) for the two exchanges.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional, Sequence

import numpy as np
import torch

from . import _lib
from ._lib import check
from .layer import SwitchMoE, _ptr, _stream


@dataclasses.dataclass(frozen=True)
class ExpertShards:
    """Ownership of E experts by `world` ranks: rank r holds experts begin(r) .. begin(r+1)-1,
    begin(r) = floor(r E / world) (contiguous ranges whose sizes differ by at most one)."""

    E: int
    world: int

    def __post_init__(self):
        if self.world < 1 or self.E < self.world:
            raise ValueError("need 1 <= world <= E (every rank owns at least one expert)")

    def begin(self, r: int) -> int:
        return (r * self.E) // self.world

    def local(self, r: int) -> int:
        """Experts owned by rank r."""
        return self.begin(r + 1) - self.begin(r)

    def owner(self, e: int) -> int:
        r = (e * self.world) // self.E
        while self.begin(r + 1) <= e:  # the floor split can put e one range later
            r += 1
        while self.begin(r) > e:
            r -= 1
        return r

    def send_rows(self, R: int) -> List[int]:
        """Rows of the dispatched buffer [E, R, d] sent to each rank (its experts' blocks)."""
        return [self.local(r) * R for r in range(self.world)]

    def recv_rows(self, rank: int, R: int) -> List[int]:
        """Rows this rank receives from each source: [El, R] blocks of every source."""
        return [self.local(rank) * R] * self.world

    @staticmethod
    def packed_offsets(counts: np.ndarray) -> tuple:
        """counts [W, El] (valid rows per source and local expert) -> (off [W, El], rows [El]):
        the first packed row of each (source, expert) block and the packed rows per expert."""
        counts = np.asarray(counts, dtype=np.int64)
        off = np.cumsum(counts, axis=0) - counts
        return off, counts.sum(axis=0)

    @staticmethod
    def packed_index(counts: np.ndarray, R: int) -> np.ndarray:
        """The return permutation, host side: for every packed row of every local expert (expert
        by expert, sources in rank order, rows in order), the flat row s*El*R + e*R + i of the
        chunk layout [W, El, R] it came from and goes back to."""
        counts = np.asarray(counts, dtype=np.int64)
        W, El = counts.shape
        idx = []
        for e in range(El):
            for s in range(W):
                base = (s * El + e) * R
                idx.extend(range(base, base + int(counts[s, e])))
        return np.asarray(idx, dtype=np.int64)


def all_to_all_rows(send: torch.Tensor, send_rows: Sequence[int], recv_rows: Sequence[int],
                    group=None, row_shape=()) -> torch.Tensor:
    """torch.distributed all-to-all of row blocks: rank r gets send rows [sum(send_rows[:r]),
    + send_rows[r]); the result holds the blocks of every source in rank order."""
    import torch.distributed as dist
    width = int(np.prod(row_shape)) if row_shape else 1
    flat = send.reshape(-1)
    out = torch.empty(sum(recv_rows) * width, dtype=send.dtype, device=send.device)
    dist.all_to_all_single(out, flat, [n * width for n in recv_rows], [n * width for n in send_rows], group=group)
    return out.view(sum(recv_rows), *row_shape) if row_shape else out


class ExpertParallelSwitch:
    """The Switch layer with its experts sharded over `world` ranks (one GPU each).

    Each rank routes its own G routing groups of T tokens with the replicated router and holds
    the weights of its experts only (W1 [El, d_ff, d], W2 [El, d, d_ff]).  forward() runs the
    stages below; `exchange` (default: torch.distributed all-to-all on `group`) moves the
    chunks.  The stages are public so that a caller can run the exchanges another way.
    """

    def __init__(self, G: int, T: int, d_model: int, d_ff: int, E: int, capacity_factor: float = 1.0, *,
                 rank: int, world: int, dtype: torch.dtype = torch.bfloat16, alpha: float = 0.01, device=None):
        self.shards = ExpertShards(E, world)
        self.rank, self.world = rank, world
        self.router = SwitchMoE(G, T, d_model, d_ff, E, capacity_factor, dtype=dtype, alpha=alpha, device=device)
        self.R = self.router.block_rows
        self.El = self.shards.local(rank)
        # the local experts' FFN over the rows received from every rank: world*G groups' worth
        # of blocks of the same capacity
        self.experts = SwitchMoE(world * G, T, d_model, d_ff, self.El, capacity_factor, dtype=dtype,
                                 capacity_override=self.router.C, device=device)
        assert self.experts.block_rows == world * self.R
        self.lib = self.router.lib
        self.d_model, self.dtype, self.device = d_model, dtype, self.router.device

    # ------------------------------------------------------------------ stages
    def route_and_dispatch(self, x, Wr, br=None, stream=None):
        """Local routing and dispatch: (route results, xe [E, R, d], expert_rows [E] int32)."""
        r = self.router.route(x, Wr, br, stream=stream)
        xe = self.router.dispatch(x, r, stream=stream)
        return r, xe, r.expert_rows

    def run_experts(self, recv_counts: torch.Tensor, recv_x: torch.Tensor, W1, b1, W2, b2, stream=None):
        """recv_counts [W, El] int32 and recv_x [W, El, R, d] as received -> the expert outputs
        as chunks [W, El, R, d] for the return exchange."""
        W, El, R, d = self.world, self.El, self.R, self.d_model
        es = recv_x.element_size()
        packed = torch.empty(El, W * R, d, dtype=self.dtype, device=self.device)
        rows = torch.empty(El, dtype=torch.int32, device=self.device)
        check(self.lib.switch_ep_regroup(_ptr(recv_x), _ptr(packed), _ptr(recv_counts), _ptr(rows), W, El, R, d * es, 0,
                                         _stream(stream)), "switch_ep_regroup")
        ye = self.experts.expert_ffn(packed, W1, b1, W2, b2, rows, stream=stream)
        back = torch.empty(W, El, R, d, dtype=self.dtype, device=self.device)
        check(self.lib.switch_ep_regroup(_ptr(ye), _ptr(back), _ptr(recv_counts), None, W, El, R, d * es, 1,
                                         _stream(stream)), "switch_ep_regroup")
        return back

    def combine(self, r, ye: torch.Tensor, x_residual=None, stream=None):
        return self.router.combine(ye, r, x_residual, stream=stream)

    # ------------------------------------------------------------------ the layer
    def forward(self, x, Wr, br, W1, b1, W2, b2, x_residual=None, group=None,
                exchange: Optional[Callable] = None, stream=None):
        """y [G*T, d] and this rank's route results; W1/b1/W2/b2 are this rank's experts."""
        ex = exchange or (lambda send, srows, rrows, shape: all_to_all_rows(send, srows, rrows, group, shape))
        S, W, El, R, d = self.shards, self.world, self.El, self.R, self.d_model
        r, xe, counts = self.route_and_dispatch(x, Wr, br, stream)
        recv_counts = ex(counts, [S.local(k) for k in range(W)], [El] * W, ()).view(W, El)
        recv_x = ex(xe.view(-1, d), S.send_rows(R), S.recv_rows(self.rank, R), (d,)).view(W, El, R, d)
        back = self.run_experts(recv_counts, recv_x, W1, b1, W2, b2, stream)
        ye = ex(back.view(-1, d), S.recv_rows(self.rank, R), S.send_rows(R), (d,)).view(self.shards.E, R, d)
        return self.combine(r, ye, x_residual, stream), r
