"""The allocation-free replay forward (ls_replay_fwd_noalloc).

Callers that own every device allocation themselves (an embedding framework,
an allocator-free host) cannot hand the library a workspace; this entry point
uses the library's fixed device scratch instead.  Here it is called through
the C ABI twice in a row and checked against ls_replay_fwd with a
caller-owned workspace on the same inputs, within the bf16 tolerance of the
parity tests (2e-2 relative, LSE 1e-3 absolute).  The file is named so that
pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import long_context_grpo_replay_gb300.binding as ls
from long_context_grpo_replay_gb300 import inputs

pytestmark = pytest.mark.gpu


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def test_noalloc_forward_matches_workspace_forward(cuda_device):
    from long_context_grpo_replay_gb300 import build

    build.build()
    L = ls.lib()
    assert ls.ls_replay_fwd_noalloc_scratch_bytes() == 64 << 20
    w = inputs.Workload("noalloc", 24, 4, 256, 256, 5000, (300,), "bf16", seed=77, pool_factor=2,
                        poison=True)
    pr = inputs.make_prompt(w, "cpu")
    kp, vp, pt = (pr[k].to(cuda_device) for k in ("k_pool", "v_pool", "page_table"))
    desc = ls.desc_for(w.hq, w.hkv, w.head_dim, w.page_size, torch.bfloat16, w.scale)
    prompt = ls.prompt_from(kp, vp, pt, w.prompt_len)
    m = {k: v.to(cuda_device) for k, v in inputs.make_member(w, 0, "cpu").items()}
    R = m["q"].shape[0]
    f32 = dict(device=cuda_device, dtype=torch.float32)

    ws = torch.empty(ls.ls_replay_workspace_size(desc, prompt, R), dtype=torch.uint8,
                     device=cuda_device)
    ls.ls_clear_device_status(ws)
    o_ref = torch.empty_like(m["q"])
    lse_ref = torch.empty(R, w.hq, **f32)
    ls.ls_replay_fwd(desc, prompt, m["q"], m["k"], m["v"], o_ref, lse_ref, ws)
    ls.ls_read_device_status(ws)

    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        o = torch.full_like(m["q"], float("nan"))
        lse = torch.full((R, w.hq), float("nan"), **f32)
        st = L.ls_replay_fwd_noalloc(ctypes.byref(desc), ctypes.byref(prompt), m["q"].data_ptr(),
                                     m["k"].data_ptr(), m["v"].data_ptr(), R, o.data_ptr(),
                                     lse.data_ptr(), stream)
        assert st == 0, ls.ls_last_error()
        torch.cuda.synchronize()
        assert _rel(o, o_ref) <= 2e-2, (call, _rel(o, o_ref))
        assert float((lse - lse_ref).abs().max()) <= 1e-3, call


def test_noalloc_forward_rejects_calls_beyond_its_scratch(cuda_device):
    from long_context_grpo_replay_gb300 import build

    build.build()
    L = ls.lib()
    # a 2M-position prompt with 8192-token responses needs far more than 64 MiB
    # of partials; the call must be refused before any launch
    desc = ls.desc_for(24, 4, 256, 256, torch.bfloat16)
    fake = 1 << 24
    prompt = ls.PromptKV(fake, fake, 8192, fake, 8192, 2097152)
    st = L.ls_replay_fwd_noalloc(ctypes.byref(desc), ctypes.byref(prompt), fake, fake, fake, 8192,
                                 fake, fake, None)
    assert st == 3
    assert "64 MiB" in ls.ls_last_error()
