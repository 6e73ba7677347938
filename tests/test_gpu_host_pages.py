"""Prompt pages in pinned host memory, streamed in chunks (host_pages.py):
the chunked forward and backward through the C ABI against the float64
oracle's replay, at the parity tolerances.  Chunks of 3 pages over a prompt
of 20 pages with a partial last page; one chunk holding the whole prompt;
and no prompt at all."""
import numpy as np
import pytest
import torch

import long_context_grpo_replay_gb300.binding as ls
import oracle.ref as ref
from long_context_grpo_replay_gb300 import inputs
from long_context_grpo_replay_gb300.host_pages import HostPagedReplay
from gpu_helpers import LSE_TOL, TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_grpo_replay_gb300 import build

    build.build()
    ls.lib()


@pytest.mark.parametrize("P,chunk", [(5000, 3), (5000, 64), (0, 4)],
                         ids=["p5000_chunks3", "p5000_one_chunk", "no_prompt"])
def test_host_paged_replay_matches_the_oracle(cuda_device, P, chunk):
    dev = cuda_device
    w = inputs.Workload("hostpages", 24, 4, 256, 256, P, (300,), "bf16", seed=23, pool_factor=2,
                        poison=True)
    pr = inputs.make_prompt(w, "cpu")
    m = inputs.make_member(w, 0, "cpu")
    kh, vh = pr["k_pool"].pin_memory(), pr["v_pool"].pin_memory()
    desc = ls.desc_for(w.hq, w.hkv, w.head_dim, w.page_size, torch.bfloat16, w.scale)
    rep = HostPagedReplay(desc, kh, vh, pr["page_table"], P, chunk, dev)
    q, k, v, d_o = (m[x].to(dev) for x in ("q", "k", "v", "d_o"))
    R = q.shape[0]
    ws = torch.empty(rep.workspace_bytes(R), dtype=torch.uint8, device=dev)
    ls.ls_clear_device_status(ws)
    o = torch.empty_like(q)
    lse = torch.empty(R, w.hq, device=dev, dtype=torch.float32)
    rep.forward(q, k, v, o, lse, ws)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rep.backward(q, k, v, d_o, o, lse, dq, dk, dv, ws)
    ls.ls_read_device_status(ws)
    want = ref.replay_member(pr["k_pool"], pr["v_pool"], pr["page_table"], P, m["q"], m["k"],
                             m["v"], m["d_o"], scale=w.scale)
    tol = TOL["bf16"]
    errs = {key: rel_err(t.double().cpu().numpy(), want[key])
            for key, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv))}
    e_l = float(np.abs(lse.double().cpu().numpy() - want["lse"]).max())
    assert all(e <= tol for e in errs.values()) and e_l <= LSE_TOL, (P, chunk, errs, e_l)


def test_host_paged_group_chunk_major_matches_the_oracle(cuda_device):
    """Two members of different lengths, chunk-major (every chunk staged
    once for both): each member's O, LSE, dQ, dK, dV against the oracle."""
    dev = cuda_device
    P, chunk = 5000, 3
    w = inputs.Workload("hostgroup", 24, 4, 256, 256, P, (300, 77), "bf16", seed=29, pool_factor=2,
                        poison=True)
    pr = inputs.make_prompt(w, "cpu")
    kh, vh = pr["k_pool"].pin_memory(), pr["v_pool"].pin_memory()
    desc = ls.desc_for(w.hq, w.hkv, w.head_dim, w.page_size, torch.bfloat16, w.scale)
    rep = HostPagedReplay(desc, kh, vh, pr["page_table"], P, chunk, dev)
    cpu_members = [inputs.make_member(w, g, "cpu") for g in range(2)]
    members = []
    for m in cpu_members:
        q, k, v, d_o = (m[x].to(dev) for x in ("q", "k", "v", "d_o"))
        R = q.shape[0]
        members.append({"q": q, "k": k, "v": v, "d_o": d_o, "o": torch.empty_like(q),
                        "lse": torch.empty(R, w.hq, device=dev, dtype=torch.float32),
                        "dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v)})
    ws = torch.empty(rep.workspace_bytes(max(w.resp_lens)), dtype=torch.uint8, device=dev)
    ls.ls_clear_device_status(ws)
    rep.forward_group(members, ws)
    rep.backward_group(members, ws)
    ls.ls_read_device_status(ws)
    for m, mc in zip(members, cpu_members):
        want = ref.replay_member(pr["k_pool"], pr["v_pool"], pr["page_table"], P, mc["q"], mc["k"],
                                 mc["v"], mc["d_o"], scale=w.scale)
        errs = {key: rel_err(m[key].double().cpu().numpy(), want[key]) for key in ("o", "dq", "dk", "dv")}
        e_l = float(np.abs(m["lse"].double().cpu().numpy() - want["lse"]).max())
        assert all(e <= TOL["bf16"] for e in errs.values()) and e_l <= LSE_TOL, (errs, e_l)


def test_sum_parts(cuda_device):
    g = torch.Generator(device=cuda_device).manual_seed(3)
    parts = torch.randn(5, 1000, 4, device=cuda_device, generator=g)
    out = torch.empty(1000, 4, device=cuda_device)
    ls.ls_sum_parts(parts, out)
    want = parts.double().sum(0)
    assert float((out.double() - want).abs().max()) <= 1e-5
    outb = torch.empty(1000, 4, device=cuda_device, dtype=torch.bfloat16)
    ls.ls_sum_parts(parts, outb)
    assert float((outb.double() - want).abs().max() / want.abs().max()) <= 1e-2


@pytest.mark.parametrize("where", ["pinned_host", "device"])
def test_stage_pages_is_a_bit_exact_gather(cuda_device, where):
    """ls_stage_pages copies logical pages first..first+n-1 of a scattered pool
    into a compact staging pool in logical order, bit for bit, reading pinned
    host memory directly; an entry outside the pool zeroes its staging page
    and sets the status word."""
    w = inputs.Workload("stage", 24, 4, 256, 256, 256 * 40, (1,), "bf16", seed=9, pool_factor=2,
                        poison=True)
    pr = inputs.make_prompt(w, "cpu")
    desc = ls.desc_for(w.hq, w.hkv, w.head_dim, w.page_size, torch.bfloat16, w.scale)
    if where == "pinned_host":
        kp, vp = pr["k_pool"].pin_memory(), pr["v_pool"].pin_memory()
    else:
        kp, vp = pr["k_pool"].to(cuda_device), pr["v_pool"].to(cuda_device)
    pt = pr["page_table"].to(torch.int32)
    pt_dev = pt.to(cuda_device)
    first, n = 7, 20
    kd = torch.full((n,) + tuple(kp.shape[1:]), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    vd = kd.clone()
    ws = torch.zeros(256, dtype=torch.uint8, device=cuda_device)
    ls.ls_stage_pages(desc, kp, vp, pt_dev, first, n, kd, vd, ws)
    torch.cuda.synchronize()
    ls.ls_read_device_status(ws)
    sel = pt[first:first + n].long()
    want_k = pr["k_pool"][sel]
    want_v = pr["v_pool"][sel]
    assert torch.equal(kd.cpu().view(torch.int16), want_k.view(torch.int16))
    assert torch.equal(vd.cpu().view(torch.int16), want_v.view(torch.int16))
    # an out-of-pool entry: that staging page is zeroed and reported
    bad = pt.clone()
    bad[first + 3] = kp.shape[0] + 11
    ls.ls_stage_pages(desc, kp, vp, bad.to(cuda_device), first, n, kd, vd, ws)
    with pytest.raises(ls.LsError) as ei:
        ls.ls_read_device_status(ws)
    assert ei.value.status == 5
    assert not (kd[3].view(torch.int16) != 0).any() and not (vd[3].view(torch.int16) != 0).any()
    assert torch.equal(kd[4].cpu().view(torch.int16), want_k[4].view(torch.int16))
