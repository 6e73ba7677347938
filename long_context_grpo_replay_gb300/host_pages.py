"""Prompt pages resident in host memory, streamed to the GPU in chunks.

The GLM path of the LongStraw DeepRead summary (section Method) keeps its
prompt state in CPU memory and stages it per layer.  Here that idea is
applied to the KV pages of the full-attention replay.  Pages live in pinned
host memory (on GB300 the Grace memory, reached over NVLink-C2C).  For each
pass the prompt is cut into chunks of whole logical pages.  Each chunk is
copied into one of two device staging pools on a copy stream while the
previous chunk computes; the copy is one library kernel per chunk
(ls_stage_pages) that reads the pinned pages directly over the CPU-GPU link
through a device copy of the page table.

Every chunk is an exact share of the keys, so the result is exact:

  forward  : ls_replay_fwd_part per chunk (the first chunk adds the causal
             response keys), then ls_lse_merge of the chunk partials;
  backward : ls_replay_bwd_part per chunk with the global LSE and D, then
             ls_sum_parts of the dQ shares; the response dK/dV come from the
             first chunk.

Device memory holds two chunks of pages plus one float32 partial per chunk,
however long the prompt.  Every step, the page copies included, runs in the
library.

A group can run chunk-major instead (forward_group, backward_group): each
pass stages every chunk once and runs all members' shares over it before
the next chunk, so the prompt crosses the CPU-GPU link once per pass for the
whole group rather than once per member.  The price is that every member's
chunk partials are live at once (float32 [chunks, R, Hq, d] per member)
instead of one member's.
"""
from __future__ import annotations

import torch

from . import binding as ls


def page_chunks(prompt_len: int, page_size: int, chunk_pages: int) -> list:
    """The prompt's logical pages cut into chunks of at most chunk_pages:
    (first page, end page, keys in the chunk) per chunk; none for an empty
    prompt.  The last chunk may end in a partial page."""
    if chunk_pages < 1:
        raise ValueError("chunk_pages must be >= 1")
    n_pages = -(-prompt_len // page_size)
    return [(c0, min(c0 + chunk_pages, n_pages),
             min(prompt_len, min(c0 + chunk_pages, n_pages) * page_size) - c0 * page_size)
            for c0 in range(0, n_pages, chunk_pages)]


class HostPagedReplay:
    """Replay over a prompt whose pages are in pinned host memory.

    k_pool_host, v_pool_host: pinned [pool_pages, Hkv, page_size, d] tensors;
    page_table: int32 [num_pages] (host), logical page -> pool slot;
    chunk_pages: pages per staged chunk."""

    def __init__(self, desc, k_pool_host, v_pool_host, page_table, prompt_len, chunk_pages, device):
        if not (k_pool_host.is_pinned() and v_pool_host.is_pinned()):
            raise ValueError("host pools must be pinned")
        if chunk_pages < 1:
            raise ValueError("chunk_pages must be >= 1")
        self.desc = desc
        self.kh, self.vh = k_pool_host, v_pool_host
        self.pt = page_table.cpu().to(torch.int64)
        self.P = int(prompt_len)
        self.page = k_pool_host.shape[2]
        n_pages = -(-self.P // self.page)
        if self.pt.shape[0] < n_pages:
            raise ValueError("page table shorter than the prompt")
        if n_pages and (int(self.pt[:n_pages].min()) < 0 or int(self.pt[:n_pages].max()) >= k_pool_host.shape[0]):
            raise ValueError("page table entry outside the host pool")
        self.chunks = [(c0, c1) for c0, c1, _ in page_chunks(self.P, self.page, chunk_pages)]
        shape = (chunk_pages,) + tuple(k_pool_host.shape[1:])
        self.kst = [torch.empty(shape, dtype=k_pool_host.dtype, device=device) for _ in range(2)]
        self.vst = [torch.empty(shape, dtype=v_pool_host.dtype, device=device) for _ in range(2)]
        self.local_pt = torch.arange(chunk_pages, dtype=torch.int32, device=device)
        self.pt_dev = self.pt.to(torch.int32).to(device)  # logical page -> host pool slot
        self.copy_stream = torch.cuda.Stream(device)
        self.device = device
        # passes alternate their chunk order, so that each pass starts on the
        # chunk the previous one left in a staging pool and never waits for
        # its first copy; held[b] is the chunk staging pool b holds
        self.reverse = False
        self.held = [None, None]

    def n_chunks(self) -> int:
        return max(1, len(self.chunks))

    def _prompt(self, b, c0, c1):
        n_tok = min(self.P, c1 * self.page) - c0 * self.page
        return ls.prompt_from(self.kst[b], self.vst[b], self.local_pt[: c1 - c0], n_tok)

    def workspace_bytes(self, max_resp_len) -> int:
        """Bytes of the one workspace every chunk's calls share."""
        if not self.chunks:
            return ls.ls_replay_workspace_size(self.desc, ls.prompt_from(None, None, None, 0),
                                               max_resp_len)
        return max(ls.ls_replay_workspace_size(self.desc, self._prompt(0, c0, c1), max_resp_len)
                   for c0, c1 in {self.chunks[0], self.chunks[-1]})

    def _stream_chunks(self, run_chunk, ws):
        """Stage every chunk (double-buffered) and call run_chunk(chunk index,
        prompt) for each; the order alternates between passes (see __init__)."""
        stream = torch.cuda.current_stream(self.device)
        if not self.chunks:
            run_chunk(0, ls.prompt_from(None, None, None, 0))
            return
        n = len(self.chunks)
        order = list(range(n - 1, -1, -1)) if self.reverse else list(range(n))
        self.reverse = not self.reverse
        b0 = self.held.index(order[0]) if order[0] in self.held else 0
        bufs = [b0 ^ (i & 1) for i in range(n)]
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        free = [torch.cuda.Event(), torch.cuda.Event()]
        for e in free:
            e.record(stream)
        need_copy = [True] * n
        need_copy[0] = self.held[b0] != order[0]

        def stage(i):
            b, ci = bufs[i], order[i]
            c0, c1 = self.chunks[ci]
            self.copy_stream.wait_event(free[b])
            ls.ls_stage_pages(self.desc, self.kh, self.vh, self.pt_dev, c0, c1 - c0, self.kst[b],
                              self.vst[b], ws, self.copy_stream)
            copied[b].record(self.copy_stream)
            self.held[b] = ci

        if need_copy[0]:
            stage(0)
        for i in range(n):
            b, ci = bufs[i], order[i]
            if i + 1 < n:
                stage(i + 1)
            if need_copy[i]:
                stream.wait_event(copied[b])
            c0, c1 = self.chunks[ci]
            run_chunk(ci, self._prompt(b, c0, c1))
            free[b].record(stream)

    def forward(self, q, k, v, o, lse, ws):
        R, hq, d = q.shape
        n = self.n_chunks()
        parts_o = torch.empty((n, R, hq, d), dtype=torch.float32, device=q.device)
        parts_l = torch.empty((n, R, hq), dtype=torch.float32, device=q.device)

        def run(i, prompt):
            ls.ls_replay_fwd_part(self.desc, prompt, q, k, v, i == 0, parts_o[i], parts_l[i], ws)

        self._stream_chunks(run, ws)
        ls.ls_lse_merge(parts_o.view(n, R * hq, d), parts_l.view(n, R * hq), o, lse)

    def backward(self, q, k, v, d_o, o, lse, dq, dk, dv, ws):
        """dq in its own dtype (the sum of the chunk shares)."""
        R, hq, d = q.shape
        n = self.n_chunks()
        delta = torch.empty((R, hq), dtype=torch.float32, device=q.device)
        ls.ls_replay_bwd_preprocess(self.desc, o, d_o, delta)
        dq_parts = torch.empty((n, R, hq, d), dtype=torch.float32, device=q.device)

        def run(i, prompt):
            first = i == 0
            ls.ls_replay_bwd_part(self.desc, prompt, q, k, v, d_o, lse, delta, first, dq_parts[i],
                                  dk if first else None, dv if first else None, ws)

        self._stream_chunks(run, ws)
        ls.ls_sum_parts(dq_parts, dq)

    def forward_group(self, members, ws):
        """Chunk-major forward of a group: members are dicts with q, k, v, o,
        lse (o and lse written)."""
        n = self.n_chunks()
        parts = []
        for m in members:
            R, hq, d = m["q"].shape
            parts.append((torch.empty((n, R, hq, d), dtype=torch.float32, device=m["q"].device),
                          torch.empty((n, R, hq), dtype=torch.float32, device=m["q"].device)))

        def run(i, prompt):
            for m, (po, pl) in zip(members, parts):
                ls.ls_replay_fwd_part(self.desc, prompt, m["q"], m["k"], m["v"], i == 0, po[i], pl[i], ws)

        self._stream_chunks(run, ws)
        for m, (po, pl) in zip(members, parts):
            R, hq, d = m["q"].shape
            ls.ls_lse_merge(po.view(n, R * hq, d), pl.view(n, R * hq), m["o"], m["lse"])

    def backward_group(self, members, ws):
        """Chunk-major backward of a group: members also carry d_o, and dq,
        dk, dv (written)."""
        n = self.n_chunks()
        state = []
        for m in members:
            R, hq, d = m["q"].shape
            delta = torch.empty((R, hq), dtype=torch.float32, device=m["q"].device)
            ls.ls_replay_bwd_preprocess(self.desc, m["o"], m["d_o"], delta)
            state.append((delta, torch.empty((n, R, hq, d), dtype=torch.float32, device=m["q"].device)))

        def run(i, prompt):
            first = i == 0
            for m, (delta, dqp) in zip(members, state):
                ls.ls_replay_bwd_part(self.desc, prompt, m["q"], m["k"], m["v"], m["d_o"], m["lse"], delta,
                                      first, dqp[i], m["dk"] if first else None,
                                      m["dv"] if first else None, ws)

        self._stream_chunks(run, ws)
        for m, (_, dqp) in zip(members, state):
            ls.ls_sum_parts(dqp, m["dq"])
