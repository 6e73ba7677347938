"""ls_prompt_prefill: the capture step (page write + causal self-attention of
the prompt) through the C ABI against the float64 oracle.

The pages written must equal the oracle's page write bit for bit (unused pool
slots keep their NaN poison); o and lse must match causal attention over the
prompt (the oracle's replay with an empty prompt and the prompt in the
response's place) within the parity tolerances (bf16 2e-2 relative, fp32
1e-5; |dLSE| <= 1e-3)."""
import numpy as np
import pytest
import torch

import long_context_grpo_replay_gb300.binding as ls
import oracle.ref as ref
from long_context_grpo_replay_gb300 import inputs
from gpu_helpers import LSE_TOL, TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_grpo_replay_gb300 import build

    build.build()
    ls.lib()


def _bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _run(w, dev, rows=None):
    N = w.prompt_len
    pr = inputs.make_prompt(w, "cpu")  # page table and poisoned pool layout
    m = inputs.make_member(w, 0, "cpu", resp_len=N)
    k_pool, v_pool = pr["k_pool"].to(dev), pr["v_pool"].to(dev)
    pt = pr["page_table"].to(dev)
    q, k, v = (m[x].to(dev) for x in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(N, w.hq, device=dev, dtype=torch.float32)
    desc = ls.desc_for(w.hq, w.hkv, w.head_dim, w.page_size, inputs.torch_dtype(w), w.scale)
    ws = torch.empty(ls.ls_prompt_prefill_workspace_size(desc, N), dtype=torch.uint8, device=dev)
    ls.ls_clear_device_status(ws)
    ls.ls_prompt_prefill(desc, q, k, v, o, lse, k_pool, v_pool, pt, ws)
    ls.ls_read_device_status(ws)

    # pages: the oracle's scatter on the same pool contents, bit for bit
    ek, ev = pr["k_pool"].clone(), pr["v_pool"].clone()
    ref.kv_page_write(ek, ev, pr["page_table"], w.page_size, 0, m["k"], m["v"])
    assert torch.equal(_bits(k_pool), _bits(ek)), "k pages differ"
    assert torch.equal(_bits(v_pool), _bits(ev)), "v pages differ"

    # attention: causal over the prompt itself
    r = ref.replay_member(pr["k_pool"], pr["v_pool"], pr["page_table"], 0, m["q"], m["k"], m["v"],
                          scale=w.scale, rows=rows)
    rr = r["rows"]
    tol = TOL[w.dtype]
    e_o = rel_err(o.double().cpu().numpy()[rr], r["o"])
    e_l = float(np.abs(lse.double().cpu().numpy()[rr] - r["lse"]).max())
    assert e_o <= tol and e_l <= LSE_TOL, (w.name, e_o, e_l)


CASES = [
    # name, hq, hkv, d, page, N, dtype
    ("prefill_tc_ragged", 24, 4, 256, 256, 1000, "bf16"),
    ("prefill_tc_exact", 24, 4, 256, 256, 1024, "bf16"),
    ("prefill_tc_one", 24, 4, 256, 256, 1, "bf16"),
    ("prefill_simt_f32", 4, 2, 64, 16, 300, "f32"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_small(cuda_device, case):
    name, hq, hkv, d, page, N, dt = case
    w = inputs.Workload(name, hq, hkv, d, page, N, (N,), dt, seed=11, pool_factor=2, poison=True)
    _run(w, cuda_device)


def test_prefill_32k_sampled(cuda_device):
    N = 32768
    w = inputs.Workload("prefill_32k", 24, 4, 256, 256, N, (N,), "bf16", seed=12, pool_factor=2,
                        poison=True)
    rng = np.random.default_rng(12)
    rows = np.unique(np.concatenate([rng.choice(N - 64, 64, replace=False), np.arange(N - 64, N)]))
    _run(w, cuda_device, rows=rows)


def test_prefill_workspace_too_small_is_refused(cuda_device):
    desc = ls.desc_for(24, 4, 256, 256, torch.bfloat16)
    need = ls.ls_prompt_prefill_workspace_size(desc, 4096)
    ws = torch.empty(need // 2, dtype=torch.uint8, device=cuda_device)
    q = torch.zeros(4096, 24, 256, dtype=torch.bfloat16, device=cuda_device)
    kv = torch.zeros(4096, 4, 256, dtype=torch.bfloat16, device=cuda_device)
    pool = torch.zeros(16, 4, 256, 256, dtype=torch.bfloat16, device=cuda_device)
    pt = torch.arange(16, dtype=torch.int32, device=cuda_device)
    lse = torch.empty(4096, 24, device=cuda_device)
    with pytest.raises(ls.LsError) as ei:
        ls.ls_prompt_prefill(desc, q, kv, kv, torch.empty_like(q), lse, pool, pool.clone(), pt, ws)
    assert ei.value.status == 3  # LS_ERR_WORKSPACE_TOO_SMALL
