"""Float64 CPU oracle for the gated-DeltaNet state replay.

TEST INFRASTRUCTURE ONLY, like ``oracle.ref``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s oracle legs may import it.

What the pages fix: in the Qwen model, 48 of 64 layers are gated DeltaNet
(GDN) layers whose recurrent state has a fixed size however long the prompt
is.  LongStraw keeps that state for the prompt and replays each response from
it, with the prompt state detached (LongStraw DeepRead summary, section
Method, Qwen path; the review, sections 二 and 三).  The pages do not print
the recurrence.  The reading taken here is the published gated delta rule,
per head, with a state S of shape [dv, dk]:

    a_t = exp(g_t)                         (g_t <= 0: the decay gate)
    S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T
    o_t = S_t q_t

with S_0 the captured prompt state, b_t in (0, 1) the write strength, and q,
k given (the model normalises k; the recurrence does not).  Replay returns
o and the final state.  Its backward returns dq, dk, dv, dg and db for the
response tokens and no gradient for S_0 (the detached prompt state).

The forward below is the recurrence written out step by step.  The backward
is PyTorch autograd of that same float64 computation: the derivative of the
definition, checked by finite differences in the tests.
"""
from __future__ import annotations

import numpy as np
import torch


def _t64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64)
    return torch.as_tensor(np.asarray(x), dtype=torch.float64)


def gdn_replay(s0, q, k, v, g, beta, d_o=None):
    """s0 [H, dv, dk]; q, k [R, H, dk]; v [R, H, dv]; g, beta [R, H].

    Returns float64 numpy arrays: o [R, H, dv], s_final [H, dv, dk], and with
    d_o [R, H, dv] also dq, dk, dv, dg, dbeta (the gradient of sum(d_o * o))."""
    S0 = _t64(s0)
    ins = [_t64(x).requires_grad_(d_o is not None) for x in (q, k, v, g, beta)]
    q_, k_, v_, g_, b_ = ins
    R, H, _ = q_.shape
    outs = []
    finals = []
    for h in range(H):
        S = S0[h].clone()
        oh = []
        for t in range(R):
            a = torch.exp(g_[t, h])
            kt = k_[t, h]
            # S (I - b k k^T) = S - b (S k) k^T
            S = a * (S - b_[t, h] * torch.outer(S @ kt, kt)) + b_[t, h] * torch.outer(v_[t, h], kt)
            oh.append(S @ q_[t, h])
        outs.append(torch.stack(oh) if R else torch.zeros((0, S0.shape[1]), dtype=torch.float64))
        finals.append(S)
    o = torch.stack(outs, dim=1)
    res = {"o": o.detach().numpy(), "s_final": torch.stack(finals).detach().numpy()}
    if d_o is not None and R > 0:
        grads = torch.autograd.grad(o, ins, grad_outputs=_t64(d_o), allow_unused=True)
        for name, gr, x in zip(("dq", "dk", "dv", "dg", "dbeta"), grads, ins):
            res[name] = (torch.zeros_like(x) if gr is None else gr).detach().numpy()
    return res
