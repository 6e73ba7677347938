"""Gated-DeltaNet state replay through the C ABI against the float64 oracle
(oracle/gdn.py) on the same seeded inputs: every output of the forward (o,
the final state) and of the backward (dq, dk, dv, dg, dbeta) element by
element at the float32 tolerance, for one member, a group, a single token,
a response that spans 17 of the backward's 8-token checkpoint segments (the
last one partial), and the empty response.  At the group size the benchmark times (8 members, 32
heads, 4096 tokens) two sampled (member, head) pairs are checked in full."""
import numpy as np
import pytest
import torch

import long_context_grpo_replay_gb300.binding as ls
from long_context_grpo_replay_gb300 import inputs
from oracle.gdn import gdn_replay
from gpu_helpers import TOL, rel_err

pytestmark = pytest.mark.gpu

TOL_F32 = TOL["f32"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_grpo_replay_gb300 import build

    build.build()
    ls.lib()


def _run(c):
    s0, q = c["s0"], c["q"]
    B, R, H, _ = q.shape
    o = torch.empty_like(c["v"])
    s_final = torch.empty((B,) + tuple(s0.shape), device=q.device, dtype=torch.float32)
    ls.ls_gdn_replay_fwd(s0, q, c["k"], c["v"], c["g"], c["beta"], o, s_final)  # exact path: no workspace
    grads = {n: torch.empty_like(c[x]) for n, x in
             (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta"))}
    ws = torch.empty(ls.ls_gdn_workspace_size(ls.GdnDesc(B, H, 128, 128), R), dtype=torch.uint8,
                     device=q.device)
    ls.ls_gdn_replay_bwd(s0, q, c["k"], c["v"], c["g"], c["beta"], c["d_o"], grads["dq"],
                         grads["dk"], grads["dv"], grads["dg"], grads["dbeta"], ws)
    torch.cuda.synchronize()
    return dict(o=o, s_final=s_final, **grads)


def _check(c, got, b, heads):
    """Member b, the listed heads, all tokens, every output."""
    hs = list(heads)
    a = {x: c[x].cpu() for x in ("s0", "q", "k", "v", "g", "beta", "d_o")}
    want = gdn_replay(a["s0"][hs], a["q"][b][:, hs], a["k"][b][:, hs], a["v"][b][:, hs],
                      a["g"][b][:, hs], a["beta"][b][:, hs], a["d_o"][b][:, hs])
    errs = {}
    for name in ("o", "dq", "dk", "dv", "dg", "dbeta"):
        errs[name] = rel_err(got[name][b][:, hs].double().cpu().numpy(), want[name])
    errs["s_final"] = rel_err(got["s_final"][b][hs].double().cpu().numpy(), want["s_final"])
    assert all(e <= TOL_F32 for e in errs.values()), (b, hs, errs)


@pytest.mark.parametrize("B,H,R", [(1, 4, 300), (2, 3, 1), (3, 2, 129)],
                         ids=["member_h4_r300", "group2_r1", "group3_r129"])
def test_gdn_replay_matches_the_oracle(cuda_device, B, H, R):
    c = inputs.make_gdn_group(B, H, R, seed=40 + R, device=cuda_device)
    got = _run(c)
    for b in range(B):
        _check(c, got, b, range(H))


def test_gdn_empty_response(cuda_device):
    c = inputs.make_gdn_group(2, 2, 0, seed=7, device=cuda_device)
    o = torch.empty_like(c["v"])
    s_final = torch.full((2, 2, 128, 128), float("nan"), device=cuda_device)
    ls.ls_gdn_replay_fwd(c["s0"], c["q"], c["k"], c["v"], c["g"], c["beta"], o, s_final)
    torch.cuda.synchronize()
    assert torch.equal(s_final, c["s0"].expand_as(s_final))


def test_gdn_group_at_bench_size_sampled(cuda_device):
    c = inputs.make_gdn_group(8, 32, 4096, seed=77, device=cuda_device)
    got = _run(c)
    for name, t in got.items():
        assert torch.isfinite(t).all(), name
    _check(c, got, 5, (0, 31))
