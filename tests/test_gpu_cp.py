"""Context-parallel parts through the C ABI on one GPU.

The prompt pages are split block-cyclically into 2 or 3 virtual ranks that
share one pool through their own page tables.  Each rank runs
ls_replay_fwd_part / ls_replay_bwd_part; rank 0 adds the response keys.
A rank may own no page at all.  The partials are merged with
ls_lse_merge and the dQ shares are summed.  The result is checked against
the float64 oracle's single-rank replay at the parity tolerances, and
CPReplay with a single rank (no process group) runs the library's own
operations end to end.  The cross-rank collectives are covered on CPU ranks
in tests/test_cp.py.
"""
import numpy as np
import pytest
import torch

import long_context_grpo_replay_gb300.binding as ls
import oracle.ref as ref
from long_context_grpo_replay_gb300 import cp, inputs
from gpu_helpers import LSE_TOL, TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_grpo_replay_gb300 import build

    build.build()
    ls.lib()


def _check(w, pr, m, o, lse, dq, dk, dv):
    want = ref.replay_member(pr["k_pool"], pr["v_pool"], pr["page_table"], w.prompt_len, m["q"],
                             m["k"], m["v"], m["d_o"], scale=w.scale)
    tol = TOL[w.dtype]
    errs = {
        "o": rel_err(o.double().cpu().numpy(), want["o"]),
        "dq": rel_err(dq.double().cpu().numpy(), want["dq"]),
        "dk": rel_err(dk.double().cpu().numpy(), want["dk"]),
        "dv": rel_err(dv.double().cpu().numpy(), want["dv"]),
    }
    e_l = float(np.abs(lse.double().cpu().numpy() - want["lse"]).max())
    assert all(e <= tol for e in errs.values()) and e_l <= LSE_TOL, (w.name, errs, e_l)


@pytest.mark.parametrize("world,P", [(2, 5000), (3, 300)], ids=["2ranks_p5000", "3ranks_one_empty"])
def test_parts_merge_to_the_replay(cuda_device, world, P):
    dev = cuda_device
    w = inputs.Workload(f"cp{world}", 24, 4, 256, 256, P, (300,), "bf16", seed=21, pool_factor=2,
                        poison=True)
    pr = inputs.make_prompt(w, "cpu")
    m = inputs.make_member(w, 0, "cpu")
    kp, vp, pt = (pr[x].to(dev) for x in ("k_pool", "v_pool", "page_table"))
    q, k, v, d_o = (m[x].to(dev) for x in ("q", "k", "v", "d_o"))
    R, hq, d = q.shape
    desc = ls.desc_for(w.hq, w.hkv, w.head_dim, w.page_size, torch.bfloat16, w.scale)
    n_pages = pt.shape[0]
    prompts, tables = [], []  # the PromptKV structs hold raw pointers: keep the tables alive
    for r in range(world):
        pages = cp.owned_pages(n_pages, world, r)
        n = cp.local_prompt_len(P, w.page_size, pages)
        tables.append(cp.local_page_table(pt, pages) if pages else pt)
        prompts.append(ls.prompt_from(kp, vp, tables[-1], n))
    if world == 3:
        assert prompts[2].prompt_len == 0  # 2 pages over 3 ranks: rank 2 holds no key
    f32 = dict(device=dev, dtype=torch.float32)
    parts_o = torch.empty(world, R, hq, d, **f32)
    parts_l = torch.empty(world, R, hq, **f32)
    wss = []
    for r in range(world):
        ws = torch.empty(ls.ls_replay_workspace_size(desc, prompts[r], R), dtype=torch.uint8,
                         device=dev)
        ls.ls_clear_device_status(ws)
        wss.append(ws)
        ls.ls_replay_fwd_part(desc, prompts[r], q, k, v, r == 0, parts_o[r], parts_l[r], ws)
    if world == 3:  # no key on rank 2: O = 0, LSE = -inf
        assert torch.isinf(parts_l[2]).all() and (parts_l[2] < 0).all() and (parts_o[2] == 0).all()
    o = torch.empty_like(q)
    lse = torch.empty(R, hq, **f32)
    ls.ls_lse_merge(parts_o.view(world, R * hq, d), parts_l.view(world, R * hq), o, lse)
    delta = torch.empty(R, hq, **f32)
    ls.ls_replay_bwd_preprocess(desc, o, d_o, delta)
    dq_parts = torch.empty(world, R, hq, d, **f32)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    for r in range(world):
        first = r == 0
        ls.ls_replay_bwd_part(desc, prompts[r], q, k, v, d_o, lse, delta, first, dq_parts[r],
                              dk if first else None, dv if first else None, wss[r])
    for ws in wss:
        ls.ls_read_device_status(ws)
    _check(w, pr, m, o, lse, dq_parts.sum(0), dk, dv)


def test_single_rank_cpreplay_is_the_replay(cuda_device):
    dev = cuda_device
    w = inputs.Workload("cp1", 24, 4, 256, 256, 3000, (200,), "bf16", seed=22, pool_factor=2,
                        poison=True)
    pr = inputs.make_prompt(w, "cpu")
    m = inputs.make_member(w, 0, "cpu")
    kp, vp, pt = (pr[x].to(dev) for x in ("k_pool", "v_pool", "page_table"))
    q, k, v, d_o = (m[x].to(dev) for x in ("q", "k", "v", "d_o"))
    desc = ls.desc_for(w.hq, w.hkv, w.head_dim, w.page_size, torch.bfloat16, w.scale)
    prompt = ls.prompt_from(kp, vp, pt, w.prompt_len)
    ws = torch.empty(ls.ls_replay_workspace_size(desc, prompt, q.shape[0]), dtype=torch.uint8,
                     device=dev)
    ls.ls_clear_device_status(ws)
    run = cp.CPReplay(desc=desc, prompt=prompt, world=1, rank=0)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], w.hq, device=dev, dtype=torch.float32)
    run.forward(q, k, v, o, lse, ws)
    dq = torch.empty(q.shape, device=dev, dtype=torch.float32)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    run.backward(q, k, v, d_o, o, lse, dq, dk, dv, ws)
    ls.ls_read_device_status(ws)
    _check(w, pr, m, o, lse, dq, dk, dv)


def test_ranks_without_the_response_skip_its_part(cuda_device):
    """A rank called with with_response = 0 computes no causal response part:
    against the same call with the response, its workspace has exactly one
    partial fewer written (R*Hq*(d+1) float32 words in the forward, the
    partial O and LSE; R*Hq*d in the backward, the dQ share), and its merged
    share is unchanged."""
    dev = cuda_device
    w = inputs.Workload("cp_skip", 24, 4, 256, 256, 3000, (300,), "bf16", seed=23, pool_factor=2,
                        poison=True)
    pr = inputs.make_prompt(w, "cpu")
    m = inputs.make_member(w, 0, "cpu")
    kp, vp, pt = (pr[x].to(dev) for x in ("k_pool", "v_pool", "page_table"))
    q, k, v, d_o = (m[x].to(dev) for x in ("q", "k", "v", "d_o"))
    R, hq, d = q.shape
    desc = ls.desc_for(w.hq, w.hkv, w.head_dim, w.page_size, torch.bfloat16, w.scale)
    prompt = ls.prompt_from(kp, vp, pt, w.prompt_len)
    n = ls.ls_replay_workspace_size(desc, prompt, R)
    f32 = dict(device=dev, dtype=torch.float32)

    def fresh_ws():
        ws = torch.full((n,), 0xFF, dtype=torch.uint8, device=dev)  # NaN pattern everywhere
        ws[:256] = 0  # the status header starts clear
        return ws

    def written(ws):
        return int((ws[256:].view(torch.int32) != -1).sum())

    outs, counts = {}, {}
    for with_resp in (True, False):
        ws = fresh_ws()
        o_part = torch.empty(R, hq, d, **f32)
        l_part = torch.empty(R, hq, **f32)
        ls.ls_replay_fwd_part(desc, prompt, q, k, v, with_resp, o_part, l_part, ws)
        ls.ls_read_device_status(ws)
        counts[("fwd", with_resp)] = written(ws)
        outs[with_resp] = (o_part, l_part)
    assert counts[("fwd", True)] - counts[("fwd", False)] == R * hq * (d + 1), counts
    # the prompt-only share equals the oracle's replay over the prompt keys alone
    want = ref.replay_member(pr["k_pool"], pr["v_pool"], pr["page_table"], w.prompt_len,
                             m["q"], m["k"][:0], m["v"][:0], scale=w.scale)
    o_p, l_p = outs[False]
    assert rel_err(o_p.double().cpu().numpy(), want["o"]) <= TOL["bf16"]
    assert float(np.abs(l_p.double().cpu().numpy() - want["lse"]).max()) <= LSE_TOL

    o_full = torch.empty_like(q)
    lse = torch.empty(R, hq, **f32)
    ws = fresh_ws()
    ls.ls_replay_fwd(desc, prompt, q, k, v, o_full, lse, ws)
    delta = torch.empty(R, hq, **f32)
    ls.ls_replay_bwd_preprocess(desc, o_full, d_o, delta)
    for with_resp in (True, False):
        ws = fresh_ws()
        dq_part = torch.empty(R, hq, d, **f32)
        dk, dv = torch.empty_like(k), torch.empty_like(v)
        ls.ls_replay_bwd_part(desc, prompt, q, k, v, d_o, lse, delta, with_resp, dq_part,
                              dk if with_resp else None, dv if with_resp else None, ws)
        ls.ls_read_device_status(ws)
        counts[("bwd", with_resp)] = written(ws)
    assert counts[("bwd", True)] - counts[("bwd", False)] == R * hq * d, counts
