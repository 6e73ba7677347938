"""Context parallelism over the prompt pages (the Qwen path of the LongStraw
DeepRead summary, section Method: the prompt's KV pages are sharded over the
context-parallel ranks and partial results are merged globally by LSE; the
review, section 二: the query gradient is what crosses ranks).

Each rank owns a block-cyclic share of the logical prompt pages: page p
belongs to rank (p // block) % world.  It keeps them in its own pool, with a
local page table that lists them in ascending logical order.  Every rank
holds the whole response.  For one replay member:

  forward  : each rank computes the exact float32 partial (O, LSE) over its
             own pages; the response rank adds the causal response keys.
             The partials are all-gathered and merged by LSE on every rank,
             so every rank ends with the same O and LSE.
  backward : every rank takes the global LSE and D, computes its share of
             dQ over its keys, and the shares are summed by an all-reduce.
             The response dK/dV come from the response rank and are
             broadcast.

The arithmetic runs in the library (ls_replay_fwd_part, ls_lse_merge,
ls_replay_bwd_preprocess, ls_replay_bwd_part).  This module only chooses the
pages and moves the partials between ranks with torch.distributed.  The
operations are passed in as an object, so that the orchestration can be
exercised on CPU ranks with stand-ins.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist


def owned_pages(num_pages: int, world: int, rank: int, block: int = 1) -> list[int]:
    """Logical prompt pages of `rank` under block-cyclic ownership."""
    if world < 1 or not 0 <= rank < world or block < 1:
        raise ValueError("need world >= 1, 0 <= rank < world, block >= 1")
    return [p for p in range(num_pages) if (p // block) % world == rank]


def local_prompt_len(prompt_len: int, page_size: int, pages: list[int]) -> int:
    """Tokens held in `pages`: full pages except the partial last logical page.
    With `pages` ascending, a partial page can only be the last one."""
    n = 0
    for p in pages:
        n += max(0, min(page_size, prompt_len - p * page_size))
    return n


def local_page_table(page_table: torch.Tensor, pages: list[int]) -> torch.Tensor:
    """Slots of the owned pages, in ascending logical order (int32)."""
    idx = torch.tensor(pages, dtype=torch.long, device=page_table.device)
    return page_table.index_select(0, idx).to(torch.int32).contiguous()


class LibraryOps:
    """The library's entry points, as CPReplay calls them."""

    def __init__(self):
        from . import binding as ls

        self.ls = ls

    def fwd_part(self, desc, prompt, q, k, v, with_response, o_part, lse_part, ws):
        self.ls.ls_replay_fwd_part(desc, prompt, q, k, v, with_response, o_part, lse_part, ws)

    def lse_merge(self, o_parts, lse_parts, o, lse):
        self.ls.ls_lse_merge(o_parts, lse_parts, o, lse)

    def preprocess(self, desc, o, d_o, delta):
        self.ls.ls_replay_bwd_preprocess(desc, o, d_o, delta)

    def bwd_part(self, desc, prompt, q, k, v, d_o, lse, delta, with_response, dq_part, dk, dv, ws):
        self.ls.ls_replay_bwd_part(desc, prompt, q, k, v, d_o, lse, delta, with_response, dq_part,
                                   dk, dv, ws)


@dataclass
class CPReplay:
    """One rank of a context-parallel replay.  `prompt` is this rank's local
    prompt (its pages), `ws` a workspace sized for it."""
    desc: object
    prompt: object
    world: int
    rank: int
    group: object = None
    response_rank: int = 0
    ops: object = None

    def __post_init__(self):
        if self.ops is None:
            self.ops = LibraryOps()

    @property
    def has_response(self) -> bool:
        return self.rank == self.response_rank

    def forward(self, q, k, v, o, lse, ws):
        """o (element dtype) and lse (float32), identical on every rank."""
        R, hq, d = q.shape
        parts_o = torch.empty((self.world, R, hq, d), dtype=torch.float32, device=q.device)
        parts_l = torch.empty((self.world, R, hq), dtype=torch.float32, device=q.device)
        self.ops.fwd_part(self.desc, self.prompt, q, k, v, self.has_response, parts_o[self.rank],
                          parts_l[self.rank], ws)
        if self.world > 1:
            # in place: this rank's partial is already its slice of the output
            dist.all_gather_into_tensor(parts_o.view(self.world * R, hq, d), parts_o[self.rank],
                                        group=self.group)
            dist.all_gather_into_tensor(parts_l.view(self.world * R, hq), parts_l[self.rank],
                                        group=self.group)
        self.ops.lse_merge(parts_o.view(self.world, R * hq, d), parts_l.view(self.world, R * hq),
                           o, lse)

    def backward(self, q, k, v, d_o, o, lse, dq, dk, dv, ws):
        """dq float32 [R, Hq, d] (the global sum), dk/dv (element dtype) on
        every rank.  o and lse are the merged forward results."""
        R, hq, d = q.shape
        delta = torch.empty((R, hq), dtype=torch.float32, device=q.device)
        self.ops.preprocess(self.desc, o, d_o, delta)
        resp = self.has_response
        self.ops.bwd_part(self.desc, self.prompt, q, k, v, d_o, lse, delta, resp, dq,
                          dk if resp else None, dv if resp else None, ws)
        if self.world > 1:
            dist.all_reduce(dq, op=dist.ReduceOp.SUM, group=self.group)
            dist.broadcast(dk, src=self.response_rank, group=self.group)
            dist.broadcast(dv, src=self.response_rank, group=self.group)
