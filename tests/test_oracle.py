"""Pins for the float64 oracle, checked against things other than itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped scale, a
wrong GQA index, an exclusive causal diagonal, a transposed operand, a dropped
response or prompt term) fails at least one test; the last tests plant such
slips in a copy of the oracle and check that the pins catch them.
"""
import math

import numpy as np
import pytest
import torch

import oracle.ref as ref



@pytest.fixture(autouse=True)
def _float64_default():
    """float64 as torch's default dtype inside this module only."""
    old = torch.get_default_dtype()
    torch.set_default_dtype(torch.float64)
    yield
    torch.set_default_dtype(old)


def _case(P=40, R=7, Hq=4, Hkv=2, d=8, page=8, seed=0, pool_extra=3, scale_logits=1.0):
    g = torch.Generator().manual_seed(seed)
    n_pages = -(-P // page) if P else 0
    pool_pages = max(1, n_pages + pool_extra)
    pt = torch.randperm(pool_pages, generator=g)[:n_pages].to(torch.int32)
    kp = torch.randn(pool_pages, Hkv, page, d, generator=g) * scale_logits
    vp = torch.randn(pool_pages, Hkv, page, d, generator=g)
    q = torch.randn(R, Hq, d, generator=g)
    kr = torch.randn(R, Hkv, d, generator=g) * scale_logits
    vr = torch.randn(R, Hkv, d, generator=g)
    do = torch.randn(R, Hq, d, generator=g)
    return dict(k_pool=kp, v_pool=vp, page_table=pt, prompt_len=P, q=q, k_resp=kr,
                v_resp=vr, d_o=do)


def _logical(c):
    """Logical [P, Hkv, d] prompt K/V from pools, by direct indexing (torch)."""
    kp, vp, pt, P = c["k_pool"], c["v_pool"], c["page_table"].long(), c["prompt_len"]
    page = kp.shape[2]
    k = torch.cat([kp[pt[t // page], :, t % page][None] for t in range(P)]) if P else \
        kp.new_zeros(0, kp.shape[1], kp.shape[3])
    v = torch.cat([vp[pt[t // page], :, t % page][None] for t in range(P)]) if P else \
        vp.new_zeros(0, vp.shape[1], vp.shape[3])
    return k, v


def _run(c, scale=None, **kw):
    return ref.replay_member(c["k_pool"], c["v_pool"], c["page_table"], c["prompt_len"],
                             c["q"], c["k_resp"], c["v_resp"], c["d_o"], scale=scale, **kw)


def _sdpa_full_sequence(c, scale):
    """Detached full-sequence attention with torch's SDPA and autograd.

    All P+R positions are queries (prompt queries are random), the mask is
    plain causal over the whole sequence, prompt K/V are constants and dO is
    zero on prompt rows: the conventional full-sequence execution the review
    recommends as the parity target (review 七, the node on future research directions)."""
    P = c["prompt_len"]
    R, Hq, d = c["q"].shape
    Hkv = c["k_resp"].shape[1]
    kpl, vpl = _logical(c)
    g = torch.Generator().manual_seed(123)
    qp = torch.randn(P, Hq, d, generator=g)
    q = c["q"].clone().requires_grad_(True)
    kr = c["k_resp"].clone().requires_grad_(True)
    vr = c["v_resp"].clone().requires_grad_(True)
    qa = torch.cat([qp, q]).transpose(0, 1)[None]  # [1, Hq, L, d]
    ka = torch.cat([kpl, kr]).transpose(0, 1)[None]  # [1, Hkv, L, d]
    va = torch.cat([vpl, vr]).transpose(0, 1)[None]
    rep = Hq // Hkv
    ka = ka.repeat_interleave(rep, dim=1)
    va = va.repeat_interleave(rep, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(qa, ka, va, is_causal=True,
                                                           scale=scale)
    out = out[0].transpose(0, 1)  # [L, Hq, d]
    dO = torch.cat([torch.zeros(P, Hq, d), c["d_o"]])
    (out * dO).sum().backward()
    return out[P:].detach(), q.grad, kr.grad, vr.grad


# ---------------------------------------------------------------------------
# pin 1: library routine (SDPA + autograd) on the detached full sequence
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("P,R,Hq,Hkv,d,page", [(40, 7, 4, 2, 8, 8), (33, 5, 6, 1, 16, 16),
                                                (16, 9, 6, 3, 4, 4), (0, 6, 2, 1, 8, 4)])
def test_full_sequence_autograd_parity(P, R, Hq, Hkv, d, page):
    c = _case(P, R, Hq, Hkv, d, page, seed=P + R)
    scale = 0.7 / math.sqrt(d)
    o_t, dq_t, dk_t, dv_t = _sdpa_full_sequence(c, scale)
    r = _run(c, scale=scale)
    np.testing.assert_allclose(r["o"], o_t.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dq"], dq_t.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(r["dk"], dk_t.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(r["dv"], dv_t.numpy(), rtol=0, atol=1e-11)
    assert r["dkv_exact_from"] == 0


def test_lse_matches_library_logsumexp():
    c = _case(24, 5, 4, 2, 8, 8, seed=9)
    scale = 0.3
    r = _run(c, scale=scale)
    kpl, _ = _logical(c)
    R, Hq, d = c["q"].shape
    for h in range(Hq):
        kv = h // (Hq // c["k_resp"].shape[1])
        keys = torch.cat([kpl[:, kv], c["k_resp"][:, kv]])
        s = scale * c["q"][:, h] @ keys.T
        mask = torch.ones_like(s, dtype=torch.bool)
        mask[:, 24:] = torch.tril(torch.ones(R, R, dtype=torch.bool))
        s = s.masked_fill(~mask, float("-inf"))
        np.testing.assert_allclose(r["lse"][:, h], torch.logsumexp(s, dim=1).numpy(),
                                   rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# pin 2: central finite differences of loss = sum(dO * O)
# ---------------------------------------------------------------------------
def test_finite_differences():
    c = _case(P=20, R=5, Hq=4, Hkv=2, d=6, page=4, seed=3)
    scale = 0.9
    r = _run(c, scale=scale)
    do = c["d_o"].numpy()
    eps = 1e-6

    def loss(**over):
        cc = dict(c)
        cc.update(over)
        o = ref.replay_member(cc["k_pool"], cc["v_pool"], cc["page_table"], cc["prompt_len"],
                              cc["q"], cc["k_resp"], cc["v_resp"], None, scale=scale)["o"]
        return float((o * do).sum())

    for name, key in (("q", "dq"), ("k_resp", "dk"), ("v_resp", "dv")):
        x = c[name]
        fd = np.zeros(x.shape)
        for idx in np.ndindex(*x.shape):
            xp = x.clone()
            xm = x.clone()
            xp[idx] += eps
            xm[idx] -= eps
            fd[idx] = (loss(**{name: xp}) - loss(**{name: xm})) / (2 * eps)
        err = np.abs(fd - r[key]).max() / np.abs(r[key]).max()
        assert err < 1e-6, (name, err)


def test_prompt_gets_no_gradient_and_pool_is_untouched():
    c = _case(P=16, R=4, seed=5)
    k0, v0 = c["k_pool"].clone(), c["v_pool"].clone()
    r = _run(c)
    assert set(r) >= {"dq", "dk", "dv"}
    assert r["dk"].shape == tuple(c["k_resp"].shape)
    assert torch.equal(k0, c["k_pool"]) and torch.equal(v0, c["v_pool"])


# ---------------------------------------------------------------------------
# pin 3: paged partials + LSE merge equal the monolithic softmax
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("pps,empty", [(1, 0), (2, 1), (3, 2), (100, 0)])
def test_paged_merge_equals_monolithic(pps, empty):
    c = _case(P=45, R=6, Hq=4, Hkv=2, d=8, page=8, seed=11)  # partial last page
    scale = 0.8
    o_p, lse_p = ref.paged_split_forward(c["k_pool"], c["v_pool"], c["page_table"], 45,
                                         c["q"], c["k_resp"], c["v_resp"], scale=scale,
                                         pages_per_split=pps, empty_splits=empty)
    r = _run(c, scale=scale)
    np.testing.assert_allclose(o_p, r["o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse_p, r["lse"], rtol=0, atol=1e-13)


def test_lse_merge_edge_cases():
    rng = np.random.default_rng(0)
    o_parts = rng.standard_normal((3, 5, 4))
    lse_parts = rng.standard_normal((3, 5)) * 30
    lse_parts[1, 2] = -np.inf
    lse_parts[:, 4] = -np.inf  # row with no key at all
    o, lse = ref.lse_merge(o_parts, lse_parts)
    assert np.isneginf(lse[4]) and np.all(o[4] == 0) and not np.isnan(o).any()
    # weights by definition, computed with the library logsumexp
    for n in range(4):
        L = np.logaddexp.reduce(lse_parts[:, n])
        np.testing.assert_allclose(lse[n], L, rtol=0, atol=1e-12)
        w = np.exp(lse_parts[:, n] - L)
        np.testing.assert_allclose(o[n], (w[:, None] * o_parts[:, n]).sum(0), atol=1e-12)
    # merging a single part is the identity
    o1, l1 = ref.lse_merge(o_parts[:1], lse_parts[:1])
    np.testing.assert_array_equal(o1[:4], o_parts[0, :4])


# ---------------------------------------------------------------------------
# pin 4: page-table permutation invariance (bit-identical in float64)
# ---------------------------------------------------------------------------
def test_page_permutation_invariance():
    c = _case(P=64, R=6, Hq=4, Hkv=2, d=8, page=8, seed=13, pool_extra=5)
    r0 = _run(c)
    g = torch.Generator().manual_seed(1)
    perm = torch.randperm(c["k_pool"].shape[0], generator=g)  # new slot of old slot s
    k2 = torch.empty_like(c["k_pool"])
    v2 = torch.empty_like(c["v_pool"])
    k2[perm] = c["k_pool"]
    v2[perm] = c["v_pool"]
    c2 = dict(c, k_pool=k2, v_pool=v2, page_table=perm[c["page_table"].long()].to(torch.int32))
    r1 = _run(c2)
    for key in ("o", "lse", "dq", "dk", "dv"):
        assert np.array_equal(r0[key], r1[key]), key


# ---------------------------------------------------------------------------
# closed forms and special cases
# ---------------------------------------------------------------------------
def test_k_zero_closed_form():
    c = _case(P=24, R=5, Hq=4, Hkv=2, d=8, page=8, seed=17)
    c["k_pool"].zero_()
    c["k_resp"].zero_()
    r = _run(c)
    P = 24
    kv_logical = _logical(c)[1]
    for i in range(5):
        np.testing.assert_allclose(r["lse"][i], math.log(P + i + 1), atol=1e-14)
        for h in range(4):
            kv = h // 2
            vals = torch.cat([kv_logical[:, kv], c["v_resp"][: i + 1, kv]])
            np.testing.assert_allclose(r["o"][i, h], vals.mean(0).numpy(), atol=1e-14)
    assert np.abs(r["dq"]).max() < 1e-14


def test_k_constant_lse_closed_form():
    c = _case(P=16, R=4, Hq=2, Hkv=1, d=8, page=8, seed=19)
    kc = torch.randn(8, generator=torch.Generator().manual_seed(2))
    c["k_pool"][:] = kc
    c["k_resp"][:] = kc
    scale = 0.37
    r = _run(c, scale=scale)
    for i in range(4):
        for h in range(2):
            expect = scale * float(c["q"][i, h] @ kc) + math.log(16 + i + 1)
            np.testing.assert_allclose(r["lse"][i, h], expect, atol=1e-13)


def test_v_constant_closed_form():
    c = _case(P=24, R=5, seed=23)
    vc = torch.randn(c["v_pool"].shape[-1], generator=torch.Generator().manual_seed(4))
    c["v_pool"][:] = vc
    c["v_resp"][:] = vc
    r = _run(c)
    np.testing.assert_allclose(r["o"], np.broadcast_to(vc.numpy(), r["o"].shape), atol=1e-13)
    assert np.abs(r["dq"]).max() < 1e-12 and np.abs(r["dk"]).max() < 1e-12
    # dV_r[j] = sum over heads of the group and rows i >= j of P_ij dO_i: not zero
    assert np.abs(r["dv"]).max() > 1e-3


def test_prompt_free_is_causal_sdpa():
    c = _case(P=0, R=9, Hq=6, Hkv=2, d=8, page=4, seed=29)
    r = _run(c)
    q = c["q"].transpose(0, 1)[None]
    k = c["k_resp"].transpose(0, 1)[None].repeat_interleave(3, dim=1)
    v = c["v_resp"].transpose(0, 1)[None].repeat_interleave(3, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    np.testing.assert_allclose(r["o"], o[0].transpose(0, 1).numpy(), atol=1e-13)


def test_single_row_is_decode_attention():
    c = _case(P=30, R=1, Hq=4, Hkv=1, d=8, page=8, seed=31)
    r = _run(c)
    kpl, vpl = _logical(c)
    k = torch.cat([kpl, c["k_resp"]]).transpose(0, 1)[None].repeat_interleave(4, dim=1)
    v = torch.cat([vpl, c["v_resp"]]).transpose(0, 1)[None].repeat_interleave(4, dim=1)
    q = c["q"].transpose(0, 1)[None]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v)  # no mask: decode
    np.testing.assert_allclose(r["o"], o[0].transpose(0, 1).numpy(), atol=1e-13)


def test_brute_force_scalar_loops():
    """Pure-Python scalar loops on a tiny case (no numpy matmul, no masks)."""
    c = _case(P=6, R=3, Hq=2, Hkv=1, d=3, page=2, seed=37)
    scale = 0.6
    r = _run(c, scale=scale)
    kpl, vpl = _logical(c)
    q, kr, vr, do = (c[x].tolist() for x in ("q", "k_resp", "v_resp", "d_o"))
    kpl, vpl = kpl.tolist(), vpl.tolist()
    P, R, d = 6, 3, 3
    dq = [[[0.0] * d for _ in range(2)] for _ in range(R)]
    dk = [[0.0] * d for _ in range(R)]
    dv = [[0.0] * d for _ in range(R)]
    for h in range(2):
        for i in range(R):
            keys = [kpl[t][0] for t in range(P)] + [kr[j][0] for j in range(i + 1)]
            vals = [vpl[t][0] for t in range(P)] + [vr[j][0] for j in range(i + 1)]
            s = [scale * sum(q[i][h][x] * kk[x] for x in range(d)) for kk in keys]
            mx = max(s)
            den = sum(math.exp(a - mx) for a in s)
            lse = mx + math.log(den)
            p = [math.exp(a - lse) for a in s]
            o = [sum(p[j] * vals[j][x] for j in range(len(p))) for x in range(d)]
            assert abs(lse - r["lse"][i][h]) < 1e-13
            assert max(abs(o[x] - r["o"][i][h][x]) for x in range(d)) < 1e-13
            D = sum(do[i][h][x] * o[x] for x in range(d))
            for j in range(len(p)):
                dpj = sum(do[i][h][x] * vals[j][x] for x in range(d))
                ds = p[j] * (dpj - D)
                for x in range(d):
                    dq[i][h][x] += scale * ds * keys[j][x]
                    if j >= P:
                        dk[j - P][x] += scale * ds * q[i][h][x]
                        dv[j - P][x] += p[j] * do[i][h][x]
    np.testing.assert_allclose(r["dq"], np.array(dq), atol=1e-13)
    np.testing.assert_allclose(r["dk"][:, 0], np.array(dk), atol=1e-13)
    np.testing.assert_allclose(r["dv"][:, 0], np.array(dv), atol=1e-13)


def test_rows_subset_and_exactness_bound():
    c = _case(P=32, R=10, Hq=4, Hkv=2, d=8, page=8, seed=41)
    full = _run(c)
    rows = np.array([9, 2, 7, 8, 5])
    sub = _run(c, rows=rows, row_chunk=2)
    for key in ("o", "lse", "delta", "dq"):
        np.testing.assert_allclose(sub[key], full[key][rows], atol=1e-13)
    assert sub["dkv_exact_from"] == 7
    np.testing.assert_allclose(sub["dk"][7:], full["dk"][7:], atol=1e-13)
    np.testing.assert_allclose(sub["dv"][7:], full["dv"][7:], atol=1e-13)


def test_bwd_preprocess():
    g = torch.Generator().manual_seed(0)
    o = torch.randn(5, 3, 7, generator=g)
    do = torch.randn(5, 3, 7, generator=g)
    np.testing.assert_allclose(ref.bwd_preprocess(o, do),
                               torch.einsum("rhd,rhd->rh", o, do).numpy(), atol=1e-14)


@pytest.mark.parametrize("n_tok,start", [(37, 5), (5000, 3)])
def test_kv_page_write_roundtrip(n_tok, start):
    page, Hkv, d = 16, 2, 4
    n_pages = -(-(start + n_tok) // page)
    g = torch.Generator().manual_seed(n_tok)
    pt = torch.randperm(n_pages + 4, generator=g)[:n_pages].to(torch.int32)
    kp = torch.full((n_pages + 4, Hkv, page, d), float("nan"), dtype=torch.bfloat16)
    vp = kp.clone()
    k = torch.randn(n_tok, Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(n_tok, Hkv, d, generator=g).to(torch.bfloat16)
    ref.kv_page_write(kp, vp, pt, page, start, k, v)
    for t in (0, n_tok // 2, n_tok - 1):
        pos = start + t
        assert torch.equal(kp[pt[pos // page], :, pos % page], k[t])
        assert torch.equal(vp[pt[pos // page], :, pos % page], v[t])
    c = {"k_pool": kp, "v_pool": vp, "page_table": pt, "prompt_len": start + n_tok}
    kl = ref.gather_prompt(kp, pt, start + n_tok, 1)[start:]
    np.testing.assert_array_equal(kl, k[:, 1].double().numpy())
    written = kp[pt.long()].transpose(1, 2).reshape(-1, Hkv, d)[start:start + n_tok]
    assert not torch.isnan(written).any()
    del c


# ---------------------------------------------------------------------------
# the pins catch planted mistakes (each mistake lives in a patched copy of the
# oracle on the CPU; the oracle itself is untouched)
# ---------------------------------------------------------------------------
def _patched_head_rows(kind):
    orig = ref._head_rows

    def wrong(qh, pos, kp, vp, kr, vr, doh, scale):
        if kind == "exclusive_diagonal":
            return orig(qh, pos - 1, kp, vp, kr, vr, doh, scale)
        res = list(orig(qh, pos, kp, vp, kr, vr, doh, scale))
        if kind == "dq_without_scale" and res[3] is not None:
            res[3] = res[3] / scale
        if kind == "dv_transposed" and res[5] is not None:
            res[5] = res[5][::-1].copy()
        return tuple(res)
    return wrong


@pytest.mark.parametrize("kind", ["exclusive_diagonal", "dq_without_scale", "dv_transposed"])
def test_pins_catch_planted_mistakes(monkeypatch, kind):
    monkeypatch.setattr(ref, "_head_rows", _patched_head_rows(kind))
    with pytest.raises(AssertionError):
        test_full_sequence_autograd_parity(40, 7, 4, 2, 8, 8)


def test_pins_catch_wrong_gqa_mapping(monkeypatch):
    orig = ref.replay_member

    def wrong_gqa(k_pool, v_pool, page_table, prompt_len, q, k_resp, v_resp, d_o=None,
                  scale=None, rows=None, row_chunk=None):
        # heads interleaved across KV heads (h % Hkv) instead of contiguous groups
        Hq, Hkv = q.shape[1], k_resp.shape[1]
        gq = Hq // Hkv
        perm = torch.tensor([(h % Hkv) * gq + h // Hkv for h in range(Hq)])
        inv = torch.argsort(perm)
        r = orig(k_pool, v_pool, page_table, prompt_len, q[:, perm], k_resp, v_resp,
                 None if d_o is None else d_o[:, perm], scale, rows, row_chunk)
        r["o"] = r["o"][:, inv.numpy()]
        return r

    monkeypatch.setattr(ref, "replay_member", wrong_gqa)
    with pytest.raises(AssertionError):
        test_full_sequence_autograd_parity(40, 7, 4, 2, 8, 8)
