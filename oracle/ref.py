"""Float64 CPU oracle for exact response-replay attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The product path (the CUDA library and its Python binding) never
imports, calls or links anything here, and nothing here imports the product.

What it computes is the plain definition of the operator the LongStraw pages
describe, written out in float64 with numpy (library matmuls as the only
building block).  Sources, cited by page title and section:

* LongStraw DeepRead summary (page title "LongStraw: Long-Context RL Beyond 2M
  Tokens under a Fixed GPU Budget", kendrick-stein.github.io), section *Method*:
  the shared prompt is run once without gradients and only the state later
  tokens need is kept (the capture step); each short response is rebuilt under
  autograd one at a time (the serial replay step); the Qwen path keeps compact
  KV pages for its full-attention layers and merges partial results globally
  by LSE; the stored prompt state is stop-gradient.
* LongStraw review ("论文综述：LongStraw：固定GPU预算下突破200万Token的长上下文强化学习",
  paper.oopus.info), section 三 (models): full-attention layers are GQA with
  24 query heads, 4 KV heads, head dim 256; section 七 (mind map, node on the
  Qwen implementation): the forward is composed by a global LSE softmax
  recombination; mind map, node on equations 1-3: the term
  d(loss)/d(z_P) * d(z_P)/d(theta) is omitted (prompt state detached).
* LongStraw abstract (cortexa.online page): attention is composed exactly; one
  policy response at a time is rebuilt under autograd, backpropagated, and
  unwound to the prompt boundary; the claim is exactness of response-only
  execution, not equivalence with full-sequence gradients.

Readings taken where the pages are silent (each is listed in the design notes):
softmax scale is a parameter (default 1/sqrt(d)); GQA head h reads KV head
h // (Hq/Hkv); response row i sees response keys j <= i (inclusive diagonal)
and every prompt key; LSE is the natural log with the scale included; Q/K are
post-RoPE inputs; dK/dV of a KV head sum over its query heads; prompt K/V get
no gradient.

Layouts (identical to the library's):
  prompt pools  k_pool, v_pool : [pool_pages, Hkv, page_size, d]
  page_table                   : int32 [num_pages], logical page -> pool slot
  q, d_o, o, dq                : [R, Hq, d]
  k_resp, v_resp, dk, dv       : [R, Hkv, d]
  lse, delta                   : [R, Hq]

Every function here is pinned by ``tests/test_oracle.py`` against things other
than itself: a scalar-loop brute force, torch's SDPA and autograd, central
finite differences, closed forms and invariants.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "to_f64",
    "kv_page_write",
    "gather_prompt",
    "lse_merge",
    "bwd_preprocess",
    "replay_member",
    "paged_split_forward",
]


def to_f64(x) -> np.ndarray:
    """Exact conversion of a torch tensor (any float dtype, bf16 included) or a
    numpy array to a numpy float64 array.  bf16 -> f64 and f32 -> f64 are exact."""
    if isinstance(x, np.ndarray):
        return x.astype(np.float64, copy=False)
    import torch  # local: the oracle is usable on numpy input without torch

    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# A1: capture-side page write
# --------------------------------------------------------------------------
def kv_page_write(k_pool, v_pool, page_table, page_size, start_pos, k, v):
    """Scatter prompt rows into pool pages (DeepRead summary, *Method*: the
    no-grad prefill keeps compact KV pages for the full-attention layers).

    Token t of ``k``/``v`` ([n_tok, Hkv, d]) lands at
    ``pool[page_table[(start_pos + t) // page_size], :, (start_pos + t) % page_size, :]``.
    Works on torch tensors or numpy arrays; the copy is exact and in place.
    Returns the pools for convenience."""
    n_tok = k.shape[0]
    pos = np.arange(start_pos, start_pos + n_tok, dtype=np.int64)
    pt = np.asarray(page_table).astype(np.int64)
    slots = pt[pos // page_size]
    offs = pos % page_size
    # Plain per-token loop over the scatter: obviously correct, small cases only
    # need to be fast, and large ones use the vectorised form below.
    if n_tok <= 4096:
        for t in range(n_tok):
            k_pool[slots[t], :, offs[t], :] = k[t]
            v_pool[slots[t], :, offs[t], :] = v[t]
    else:
        k_pool[slots, :, offs, :] = k
        v_pool[slots, :, offs, :] = v
    return k_pool, v_pool


def gather_prompt(pool, page_table, prompt_len, kv) -> np.ndarray:
    """Logical prompt rows of KV head ``kv`` in token order, as float64 [P, d].

    Page p of the logical prompt lives in pool slot page_table[p] (the paged
    KV store of the DeepRead summary, *Method*, Qwen path).  Only the first
    ceil(P / page_size) table entries are read; the tail of the last page
    beyond ``prompt_len`` is not part of the prompt."""
    page_size = pool.shape[2]
    n_pages = -(-prompt_len // page_size) if prompt_len > 0 else 0
    pt = np.asarray(page_table).astype(np.int64)[:n_pages]
    if n_pages == 0:
        return np.zeros((0, pool.shape[3]), dtype=np.float64)
    rows = to_f64(pool[pt, kv])  # [n_pages, page_size, d]
    return rows.reshape(n_pages * page_size, -1)[:prompt_len]


# --------------------------------------------------------------------------
# A4: exact LSE / output merge of partial results
# --------------------------------------------------------------------------
def lse_merge(o_parts, lse_parts):
    """Exact recombination of partial softmax results (DeepRead summary,
    *Method*: the global LSE and output merge; review mind map: the global LSE
    softmax recombination).

    o_parts [n_parts, n_rows, d], lse_parts [n_parts, n_rows] (natural log).
    L = log sum_s exp(L_s);  O = sum_s exp(L_s - L) * O_s.
    A row whose parts are all -inf (no visible key) merges to O = 0, L = -inf."""
    o_parts = to_f64(o_parts)
    lse_parts = to_f64(lse_parts)
    m = lse_parts.max(axis=0)  # [n_rows]
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.exp(lse_parts - m_safe[None, :])  # exp(-inf) = 0 for empty parts
    tot = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, tot, 1.0)), -np.inf)
    coef = np.where(finite[None, :], w / np.where(finite, tot, 1.0)[None, :], 0.0)
    o = np.einsum("sn,snd->nd", coef, o_parts)
    return o, lse


# --------------------------------------------------------------------------
# A5: backward preprocess
# --------------------------------------------------------------------------
def bwd_preprocess(o, d_o) -> np.ndarray:
    """D = rowsum(dO * O) over the head dimension: [R, Hq, d] -> [R, Hq]."""
    return (to_f64(o) * to_f64(d_o)).sum(axis=-1)


# --------------------------------------------------------------------------
# A2-A7: the replayed member, by definition
# --------------------------------------------------------------------------
def _head_rows(qh, pos, kp, vp, kr, vr, doh, scale):
    """One query head, a set of response rows ``pos``.

    Softmax attention over the concatenation [prompt keys ; response keys],
    where row i sees every prompt key and the response keys j <= pos[i]
    (DeepRead summary, *Method*; abstract: exact attention composition).
    The backward holds the prompt K/V constant (stop-gradient prompt state,
    review mind map, node on equations 1-3), so only dQ and the response-key dK/dV
    exist.  Returns o, lse, delta, dq for the rows and this head's
    contributions to dK_resp and dV_resp from these rows."""
    n = qh.shape[0]
    P = kp.shape[0]
    R = kr.shape[0]
    s = scale * np.concatenate([qh @ kp.T, qh @ kr.T], axis=1)  # [n, P+R]
    causal = np.arange(R)[None, :] <= pos[:, None]
    s[:, P:][~causal] = -np.inf
    m = s.max(axis=1)
    lse = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
    p = np.exp(s - lse[:, None])  # masked entries give exactly 0
    del s
    o = p[:, :P] @ vp + p[:, P:] @ vr
    if doh is None:
        return o, lse, None, None, None, None
    delta = (doh * o).sum(axis=1)
    dp = np.concatenate([doh @ vp.T, doh @ vr.T], axis=1)
    ds = p * (dp - delta[:, None])
    del dp
    dq = scale * (ds[:, :P] @ kp + ds[:, P:] @ kr)
    dk_r = scale * (ds[:, P:].T @ qh)
    dv_r = p[:, P:].T @ doh
    assert n == o.shape[0]
    return o, lse, delta, dq, dk_r, dv_r


def replay_member(
    k_pool,
    v_pool,
    page_table,
    prompt_len,
    q,
    k_resp,
    v_resp,
    d_o=None,
    scale=None,
    rows=None,
    row_chunk=None,
):
    """One replayed group member (DeepRead summary, *Method*, the serial replay
    step): forward O and LSE and, when ``d_o`` is given, the backward with
    the prompt state detached.

    ``rows``: response positions to compute (default: all).  O, LSE, D and dQ
    are returned for those rows only, in the given order.  dK_resp/dV_resp are
    summed over the given rows only, so they are exact for every key j such
    that all rows i >= j are included: the returned ``dkv_exact_from`` is the
    smallest such j (0 when all rows are given).

    Returns a dict of float64 arrays:
      o [n, Hq, d], lse [n, Hq], and with d_o: delta [n, Hq], dq [n, Hq, d],
      dk [R, Hkv, d], dv [R, Hkv, d]; plus rows and dkv_exact_from."""
    q = to_f64(q)
    kr_all = to_f64(k_resp)
    vr_all = to_f64(v_resp)
    do_all = None if d_o is None else to_f64(d_o)
    R, Hq, d = q.shape
    Hkv = kr_all.shape[1]
    assert Hq % Hkv == 0, "GQA needs Hq to be a multiple of Hkv"
    gq = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rows = np.arange(R) if rows is None else np.asarray(rows, dtype=np.int64)
    n = rows.shape[0]
    if row_chunk is None:
        # keep the [rows, P+R] score matrix near 1 GiB
        row_chunk = max(1, int((1 << 27) // max(1, prompt_len + R)))
    o = np.zeros((n, Hq, d))
    lse = np.zeros((n, Hq))
    want_bwd = do_all is not None
    if want_bwd:
        delta = np.zeros((n, Hq))
        dq = np.zeros((n, Hq, d))
        dk = np.zeros((R, Hkv, d))
        dv = np.zeros((R, Hkv, d))
    for kv in range(Hkv):
        kp = gather_prompt(k_pool, page_table, prompt_len, kv)
        vp = gather_prompt(v_pool, page_table, prompt_len, kv)
        kr = kr_all[:, kv]
        vr = vr_all[:, kv]
        for h in range(kv * gq, (kv + 1) * gq):
            for c0 in range(0, n, row_chunk):
                sel = slice(c0, min(n, c0 + row_chunk))
                pos = rows[sel]
                res = _head_rows(
                    q[pos, h], pos, kp, vp, kr, vr,
                    None if not want_bwd else do_all[pos, h], scale,
                )
                o[sel, h] = res[0]
                lse[sel, h] = res[1]
                if want_bwd:
                    delta[sel, h] = res[2]
                    dq[sel, h] = res[3]
                    dk[:, kv] += res[4]
                    dv[:, kv] += res[5]
    out = {"o": o, "lse": lse, "rows": rows}
    if want_bwd:
        present = np.zeros(R + 1, dtype=bool)
        present[rows] = True
        # smallest j with every row i >= j present
        exact_from = R
        while exact_from > 0 and present[exact_from - 1]:
            exact_from -= 1
        out.update(delta=delta, dq=dq, dk=dk, dv=dv, dkv_exact_from=exact_from)
    return out


# --------------------------------------------------------------------------
# Self-check routine: paged partials merged by LSE (used only to pin the
# definition above; the method claims the two are equal exactly)
# --------------------------------------------------------------------------
def paged_split_forward(
    k_pool, v_pool, page_table, prompt_len, q, k_resp, v_resp, scale=None,
    pages_per_split=1, empty_splits=0,
):
    """Forward computed the paged way: one partial (O_s, LSE_s) per group of
    ``pages_per_split`` prompt pages, one more for the causal response keys,
    ``empty_splits`` partials with no keys at all (LSE = -inf, O = 0), then
    the exact LSE merge (review mind map: the forward is composed by a global
    LSE softmax recombination).  Returns o [R, Hq, d], lse [R, Hq]."""
    q = to_f64(q)
    kr_all = to_f64(k_resp)
    vr_all = to_f64(v_resp)
    R, Hq, d = q.shape
    Hkv = kr_all.shape[1]
    gq = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    page_size = k_pool.shape[2]
    n_pages = -(-prompt_len // page_size) if prompt_len > 0 else 0
    o_parts, lse_parts = [], []
    for _ in range(empty_splits):
        o_parts.append(np.zeros((R, Hq, d)))
        lse_parts.append(np.full((R, Hq), -np.inf))
    for kv in range(Hkv):
        kp = gather_prompt(k_pool, page_table, prompt_len, kv)
        vp = gather_prompt(v_pool, page_table, prompt_len, kv)
        split_bounds = [
            (p0 * page_size, min(prompt_len, (p0 + pages_per_split) * page_size))
            for p0 in range(0, n_pages, pages_per_split)
        ]
        if kv == 0:
            for _ in split_bounds:
                o_parts.append(np.zeros((R, Hq, d)))
                lse_parts.append(np.zeros((R, Hq)))
            o_parts.append(np.zeros((R, Hq, d)))  # response part
            lse_parts.append(np.zeros((R, Hq)))
        base = empty_splits
        for h in range(kv * gq, (kv + 1) * gq):
            qh = q[:, h]
            for si, (a, b) in enumerate(split_bounds):
                s = scale * (qh @ kp[a:b].T)
                m = s.max(axis=1)
                l = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
                o_parts[base + si][:, h] = np.exp(s - l[:, None]) @ vp[a:b]
                lse_parts[base + si][:, h] = l
            s = scale * (qh @ kr_all[:, kv].T)
            s[~(np.arange(R)[None, :] <= np.arange(R)[:, None])] = -np.inf
            m = s.max(axis=1)
            l = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
            o_parts[base + len(split_bounds)][:, h] = np.exp(s - l[:, None]) @ vr_all[:, kv]
            lse_parts[base + len(split_bounds)][:, h] = l
    o_parts = np.stack(o_parts).reshape(len(o_parts), R * Hq, d)
    lse_parts = np.stack(lse_parts).reshape(len(lse_parts), R * Hq)
    o, lse = lse_merge(o_parts, lse_parts)
    return o.reshape(R, Hq, d), lse.reshape(R, Hq)

