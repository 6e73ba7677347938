"""Shared helpers of the GPU parity tests: run members through the C ABI and
compare them with the float64 oracle on the same seeded inputs."""
import numpy as np
import torch

import long_context_grpo_replay_gb300.binding as ls
import oracle.ref as ref
from long_context_grpo_replay_gb300 import inputs

TOL = {"f32": 1e-5, "bf16": 2e-2}
LSE_TOL = 1e-3


def rel_err(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    denom = np.abs(want).max()
    return float(np.abs(got - want).max() / (denom if denom > 0 else 1.0))


class DevicePrompt:
    """Prompt pools on the device plus the host copy the oracle reads."""

    def __init__(self, w, dev, gen_device=None):
        gen_device = gen_device or "cpu"
        pr = inputs.make_prompt(w, gen_device)
        self.w = w
        self.k_pool = pr["k_pool"].to(dev)
        self.v_pool = pr["v_pool"].to(dev)
        self.page_table = pr["page_table"].to(dev)
        self.host = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in pr.items()}
        self.desc = ls.desc_for(w.hq, w.hkv, w.head_dim, w.page_size, inputs.torch_dtype(w),
                                w.scale)
        self.prompt = ls.prompt_from(self.k_pool, self.v_pool, self.page_table, w.prompt_len)

    def workspace(self, max_r):
        n = ls.ls_replay_workspace_size(self.desc, self.prompt, max_r)
        ws = torch.empty(n, dtype=torch.uint8, device=self.k_pool.device)
        ls.ls_clear_device_status(ws)
        return ws


def alloc_member(m, hq):
    R = m["q"].shape[0]
    dev = m["q"].device
    out = dict(m)
    out.update(o=torch.empty_like(m["q"]), lse=torch.empty(R, hq, device=dev, dtype=torch.float32),
               delta=torch.empty(R, hq, device=dev, dtype=torch.float32), dq=torch.empty_like(m["q"]),
               dk=torch.empty_like(m["k"]), dv=torch.empty_like(m["v"]))
    return out


def run_group(dp, host_members, ws, dev):
    members = [alloc_member({k: v.to(dev) for k, v in m.items()}, dp.w.hq) for m in host_members]
    ls.ls_replay_group(dp.desc, dp.prompt, members, ws)
    ls.ls_read_device_status(ws)
    return members


def oracle_member(dp, m, rows=None):
    h = dp.host
    return ref.replay_member(h["k_pool"], h["v_pool"], h["page_table"], h["prompt_len"], m["q"],
                             m["k"], m["v"], m["d_o"], scale=dp.w.scale, rows=rows)


def check_member(dp, gpu, host_m, rows=None, label=""):
    """Compare one member with the oracle on `rows` (all rows when None)."""
    r = oracle_member(dp, host_m, rows)
    rr = r["rows"]
    tol = TOL[dp.w.dtype]
    errs = {}
    for key in ("o", "dq"):
        errs[key] = rel_err(gpu[key].double().cpu().numpy()[rr], r[key])
    errs["lse"] = float(np.abs(gpu["lse"].double().cpu().numpy()[rr] - r["lse"]).max())
    errs["delta"] = rel_err(gpu["delta"].double().cpu().numpy()[rr], r["delta"])
    j0 = r["dkv_exact_from"]
    for key in ("dk", "dv"):
        errs[key] = rel_err(gpu[key].double().cpu().numpy()[j0:], r[key][j0:])
    msg = f"{label} errors {errs}"
    for key in ("o", "dq", "dk", "dv", "delta"):
        assert errs[key] <= tol, msg
    assert errs["lse"] <= LSE_TOL, msg
    return errs


def sample_rows(R, seed, n_random=64, n_tail=64):
    """Seeded query rows: n_random uniform rows plus the last n_tail rows (the
    tail makes dK/dV exact for the last n_tail response keys)."""
    g = torch.Generator().manual_seed(seed)
    rnd = torch.randperm(R, generator=g)[: min(n_random, R)]
    tail = torch.arange(max(0, R - n_tail), R)
    return np.unique(np.concatenate([rnd.numpy(), tail.numpy()]))
