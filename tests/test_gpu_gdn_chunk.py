"""The tensor-core GDN path (precision LS_GDN_TENSOR_CORE: the chunkwise
forward and the chunk-parallel backward) against the float64 oracle at the
bf16 tolerance: its products take bf16 operands, which the CPU block
emulator puts near 4e-3 to 5e-3.  Cases: three chunks with a partial last
one, one exact chunk, a single token, the empty response, and two sampled
heads of the 8 x 32-head x 4096-token group; the workspace status word must
stay clear."""
import numpy as np
import pytest
import torch

import long_context_grpo_replay_gb300.binding as ls
from long_context_grpo_replay_gb300 import inputs
from oracle.gdn import gdn_replay
from gpu_helpers import TOL, rel_err

pytestmark = pytest.mark.gpu
TC = ls.LS_GDN_TENSOR_CORE


@pytest.fixture(autouse=True)
def _built():
    from long_context_grpo_replay_gb300 import build

    build.build()
    ls.lib()


def _fwd(c):
    B, R, H, _ = c["q"].shape
    o = torch.full_like(c["v"], float("nan"))
    s_final = torch.empty((B, H, 128, 128), device=c["q"].device)
    ws = torch.empty(max(1, ls.ls_gdn_workspace_size(ls.GdnDesc(B, H, 128, 128, TC), R)),
                     dtype=torch.uint8, device=c["q"].device)
    ls.ls_clear_device_status(ws)
    ls.ls_gdn_replay_fwd(c["s0"], c["q"], c["k"], c["v"], c["g"], c["beta"], o, s_final, ws,
                         precision=TC)
    torch.cuda.synchronize()
    ls.ls_read_device_status(ws)  # raises if a bounded device wait ran out
    return o, s_final


def _bwd(c):
    B, R, H, _ = c["q"].shape
    grads = {n: torch.empty_like(c[x]) for n, x in
             (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta"))}
    ws = torch.empty(ls.ls_gdn_workspace_size(ls.GdnDesc(B, H, 128, 128, TC), R),
                     dtype=torch.uint8, device=c["q"].device)
    ls.ls_clear_device_status(ws)
    ls.ls_gdn_replay_bwd(c["s0"], c["q"], c["k"], c["v"], c["g"], c["beta"], c["d_o"], grads["dq"],
                         grads["dk"], grads["dv"], grads["dg"], grads["dbeta"], ws, precision=TC)
    torch.cuda.synchronize()
    ls.ls_read_device_status(ws)  # raises if a bounded device wait ran out
    return grads


def _check(c, o, s_final, b, heads, grads=None):
    hs = list(heads)
    a = {x: c[x].cpu() for x in ("s0", "q", "k", "v", "g", "beta", "d_o")}
    want = gdn_replay(a["s0"][hs], a["q"][b][:, hs], a["k"][b][:, hs], a["v"][b][:, hs],
                      a["g"][b][:, hs], a["beta"][b][:, hs], a["d_o"][b][:, hs])
    errs = {"o": rel_err(o[b][:, hs].double().cpu().numpy(), want["o"]),
            "s_final": rel_err(s_final[b][hs].double().cpu().numpy(), want["s_final"])}
    for name, t in (grads or {}).items():
        errs[name] = rel_err(t[b][:, hs].double().cpu().numpy(), want[name])
    assert all(e <= TOL["bf16"] for e in errs.values()), (b, hs, errs)


@pytest.mark.parametrize("B,H,R", [(1, 4, 300), (2, 2, 128), (2, 3, 1)],
                         ids=["three_chunks_r300", "one_chunk_r128", "one_token"])
def test_chunk_path_matches_the_oracle(cuda_device, B, H, R):
    c = inputs.make_gdn_group(B, H, R, seed=60 + R, device=cuda_device)
    o, s_final = _fwd(c)
    grads = _bwd(c)
    for b in range(B):
        _check(c, o, s_final, b, range(H), grads)


def test_chunk_forward_empty_response(cuda_device):
    c = inputs.make_gdn_group(2, 2, 0, seed=8, device=cuda_device)
    _, s_final = _fwd(c)
    assert torch.equal(s_final, c["s0"].expand_as(s_final))


def test_chunk_path_at_bench_size_sampled(cuda_device):
    c = inputs.make_gdn_group(8, 32, 4096, seed=78, device=cuda_device)
    o, s_final = _fwd(c)
    grads = _bwd(c)
    assert torch.isfinite(o).all() and torch.isfinite(s_final).all()
    assert all(torch.isfinite(t).all() for t in grads.values())
    _check(c, o, s_final, 6, (1, 30), grads)


@pytest.mark.parametrize("B,H,R", [(2, 3, 300), (8, 32, 4096)], ids=["three_chunks", "bench_size"])
def test_backward_reusing_the_forward_is_bit_identical(cuda_device, B, H, R):
    """ls_gdn_replay_fwd, then ls_gdn_replay_bwd with LS_GDN_BWD_REUSES_FORWARD on
    the same workspace: the gradients equal, bit for bit, those of a backward
    that forms every term itself (the column sums of the output kernel are
    summed in a fixed order, so both runs are deterministic)."""
    c = inputs.make_gdn_group(B, H, R, seed=90 + R, device=cuda_device)
    want = _bwd(c)
    ws = torch.empty(ls.ls_gdn_workspace_size(ls.GdnDesc(B, H, 128, 128, TC), R), dtype=torch.uint8,
                     device=cuda_device)
    ls.ls_clear_device_status(ws)
    o = torch.empty_like(c["v"])
    s_final = torch.empty((B, H, 128, 128), device=cuda_device)
    ls.ls_gdn_replay_fwd(c["s0"], c["q"], c["k"], c["v"], c["g"], c["beta"], o, s_final, ws, precision=TC)
    got = {n: torch.empty_like(c[x]) for n, x in
           (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta"))}
    ls.ls_gdn_replay_bwd(c["s0"], c["q"], c["k"], c["v"], c["g"], c["beta"], c["d_o"], got["dq"], got["dk"],
                         got["dv"], got["dg"], got["dbeta"], ws, precision=TC, reuse_forward=True)
    torch.cuda.synchronize()
    ls.ls_read_device_status(ws)
    for name in want:
        assert torch.equal(got[name], want[name]), name
    if R <= 300:
        for b in range(B):
            _check(c, o, s_final, b, range(H), got)


def test_every_kernel_launch_is_counted(cuda_device):
    """ls_launch_count counts kernels, not calls: the forward runs three
    (prep, chain, output), the backward three when it reuses the forward's
    terms and four when it forms them itself."""
    B, H, R = 1, 2, 200
    c = inputs.make_gdn_group(B, H, R, seed=5, device=cuda_device)
    ws = torch.empty(ls.ls_gdn_workspace_size(ls.GdnDesc(B, H, 128, 128, TC), R), dtype=torch.uint8,
                     device=cuda_device)
    ls.ls_clear_device_status(ws)
    o = torch.empty_like(c["v"])
    s_final = torch.empty((B, H, 128, 128), device=cuda_device)
    grads = [torch.empty_like(c[x]) for x in ("q", "k", "v", "g", "beta")]
    n0 = ls.ls_launch_count()
    ls.ls_gdn_replay_fwd(c["s0"], c["q"], c["k"], c["v"], c["g"], c["beta"], o, s_final, ws, precision=TC)
    n1 = ls.ls_launch_count()
    ls.ls_gdn_replay_bwd(c["s0"], c["q"], c["k"], c["v"], c["g"], c["beta"], c["d_o"], *grads, ws,
                         precision=TC, reuse_forward=True)
    n2 = ls.ls_launch_count()
    ls.ls_gdn_replay_bwd(c["s0"], c["q"], c["k"], c["v"], c["g"], c["beta"], c["d_o"], *grads, ws,
                         precision=TC)
    n3 = ls.ls_launch_count()
    torch.cuda.synchronize()
    ls.ls_read_device_status(ws)
    assert (n1 - n0, n2 - n1, n3 - n2) == (3, 3, 4)
