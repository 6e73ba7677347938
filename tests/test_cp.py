"""Context-parallel orchestration (long_context_grpo_replay_gb300/cp.py) on CPU
ranks (gloo, world size 2 and 3).

The pages are split block-cyclically over the ranks.  The library's part
entry points are replaced by float64 stand-ins: the definition, restricted
to a rank's keys and, in the backward, taking the global LSE and D.  The
merged forward (all-gather, then LSE merge) and the reduced backward
(all-reduce of dQ, broadcast of the response dK/dV) must reproduce the
oracle's single-rank replay on every rank.  The library side of the same
split (ls_replay_fwd_part / ls_replay_bwd_part on one GPU) is checked in
tests/test_gpu_cp.py.
"""
import os
import socket
from types import SimpleNamespace

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.ref as ref
from long_context_grpo_replay_gb300 import cp

HQ, HKV, D, PAGE, P, R = 4, 2, 16, 4, 37, 5  # P is not a multiple of the page


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    g = torch.Generator().manual_seed(5)
    n_pages = -(-P // PAGE)
    pool = 2 * n_pages
    k_pool = torch.randn(pool, HKV, PAGE, D, generator=g, dtype=torch.float64)
    v_pool = torch.randn(pool, HKV, PAGE, D, generator=g, dtype=torch.float64)
    pt = torch.randperm(pool, generator=g)[:n_pages].to(torch.int32)
    q = torch.randn(R, HQ, D, generator=g, dtype=torch.float64)
    k = torch.randn(R, HKV, D, generator=g, dtype=torch.float64)
    v = torch.randn(R, HKV, D, generator=g, dtype=torch.float64)
    d_o = torch.randn(R, HQ, D, generator=g, dtype=torch.float64)
    return k_pool, v_pool, pt, q, k, v, d_o


class _Stand:
    """float64 stand-ins of the library's part entry points."""

    def __init__(self, scale):
        self.scale = scale

    def _keys(self, prompt, k, v, kv, i, with_response):
        kp = ref.gather_prompt(prompt.k_pool, prompt.page_table, prompt.prompt_len, kv)
        vp = ref.gather_prompt(prompt.v_pool, prompt.page_table, prompt.prompt_len, kv)
        if with_response:
            kp = np.concatenate([kp, k[: i + 1, kv].numpy()])
            vp = np.concatenate([vp, v[: i + 1, kv].numpy()])
        return kp, vp

    def fwd_part(self, desc, prompt, q, k, v, with_response, o_part, lse_part, ws):
        gq = HQ // HKV
        for h in range(HQ):
            for i in range(R):
                kp, vp = self._keys(prompt, k, v, h // gq, i, with_response)
                if kp.shape[0] == 0:
                    o_part[i, h] = 0.0
                    lse_part[i, h] = -np.inf
                    continue
                s = self.scale * kp @ q[i, h].numpy()
                m = s.max()
                e = np.exp(s - m)
                o_part[i, h] = torch.from_numpy(e @ vp / e.sum())
                lse_part[i, h] = float(m + np.log(e.sum()))

    def lse_merge(self, o_parts, lse_parts, o, lse):
        mo, ml = ref.lse_merge(o_parts.double().numpy(), lse_parts.double().numpy())
        o.copy_(torch.from_numpy(mo).reshape(o.shape))
        lse.copy_(torch.from_numpy(ml).reshape(lse.shape))

    def preprocess(self, desc, o, d_o, delta):
        delta.copy_((o.double() * d_o.double()).sum(-1))

    def bwd_part(self, desc, prompt, q, k, v, d_o, lse, delta, with_response, dq, dk, dv, ws):
        gq = HQ // HKV
        dq.zero_()
        if with_response:
            dk.zero_()
            dv.zero_()
        for h in range(HQ):
            kv = h // gq
            for i in range(R):
                kp, vp = self._keys(prompt, k, v, kv, i, with_response)
                if kp.shape[0] == 0:
                    continue
                s = self.scale * kp @ q[i, h].numpy()
                p = np.exp(s - float(lse[i, h]))
                dp = vp @ d_o[i, h].numpy()
                ds = p * (dp - float(delta[i, h]))
                dq[i, h] += torch.from_numpy(self.scale * ds @ kp)
                if with_response:
                    nr = i + 1  # the response keys are the last i+1 rows of kp
                    dsr, pr = ds[-nr:], p[-nr:]
                    dk[:nr, kv] += torch.from_numpy(self.scale * np.outer(dsr, q[i, h].numpy()))
                    dv[:nr, kv] += torch.from_numpy(np.outer(pr, d_o[i, h].numpy()))


def _worker(rank, world, port, block, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    k_pool, v_pool, pt, q, k, v, d_o = _inputs()
    n_pages = pt.shape[0]
    pages = cp.owned_pages(n_pages, world, rank, block)
    prompt = SimpleNamespace(k_pool=k_pool, v_pool=v_pool, page_table=cp.local_page_table(pt, pages),
                             prompt_len=cp.local_prompt_len(P, PAGE, pages))
    scale = 1.0 / np.sqrt(D)
    run = cp.CPReplay(desc=None, prompt=prompt, world=world, rank=rank, response_rank=world - 1,
                      ops=_Stand(scale))
    o = torch.empty(R, HQ, D, dtype=torch.float64)
    lse = torch.empty(R, HQ, dtype=torch.float32)
    run.forward(q, k, v, o, lse, ws=None)
    dq = torch.empty(R, HQ, D, dtype=torch.float64)
    dk = torch.empty(R, HKV, D, dtype=torch.float64)
    dv = torch.empty(R, HKV, D, dtype=torch.float64)
    run.backward(q, k, v, d_o, o, lse, dq, dk, dv, ws=None)
    out[rank] = {x: t.clone() for x, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,block", [(2, 1), (3, 2)])
def test_cp_ranks_reproduce_the_single_rank_replay(world, block):
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, block, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(180)
            assert p.exitcode == 0
        res = dict(out)
    k_pool, v_pool, pt, q, k, v, d_o = _inputs()
    want = ref.replay_member(k_pool, v_pool, pt, P, q, k, v, d_o, scale=1.0 / np.sqrt(D))
    for r in range(world):
        got = res[r]
        # the partials travel as float32, so the comparison is at float32 level
        for key in ("o", "dq", "dk", "dv"):
            g = got[key].numpy()
            assert np.abs(g - want[key]).max() <= 1e-5 * max(1.0, np.abs(want[key]).max()), (r, key)
        assert np.abs(got["lse"].numpy() - want["lse"]).max() <= 1e-5, r


def test_block_cyclic_ownership_covers_every_page_once():
    for world, block, n in [(2, 1, 9), (3, 2, 10), (8, 4, 33)]:
        owned = [cp.owned_pages(n, world, r, block) for r in range(world)]
        flat = sorted(p for o in owned for p in o)
        assert flat == list(range(n))
        lens = [cp.local_prompt_len(n * PAGE - 3, PAGE, o) for o in owned]
        assert sum(lens) == n * PAGE - 3


def test_host_page_chunks_cover_the_prompt_once():
    """Host-resident pages are streamed in chunks of whole pages: together the
    chunks hold every key exactly once, in order, with a partial last page."""
    from long_context_grpo_replay_gb300.host_pages import page_chunks

    assert page_chunks(0, 256, 4) == []
    assert page_chunks(1, 256, 4) == [(0, 1, 1)]
    assert page_chunks(1000, 256, 3) == [(0, 3, 768), (3, 4, 232)]
    assert page_chunks(1024, 256, 8) == [(0, 4, 1024)]
    for P, S_p, n in [(20 * 16 - 5, 16, 3), (5000, 256, 1), (65536, 256, 64)]:
        ch = page_chunks(P, S_p, n)
        assert sum(k for _, _, k in ch) == P
        assert all(a[1] == b[0] for a, b in zip(ch, ch[1:]))
        assert all(c1 - c0 <= n for c0, c1, _ in ch)
    with pytest.raises(ValueError):
        page_chunks(10, 16, 0)
