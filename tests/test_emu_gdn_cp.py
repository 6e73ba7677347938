"""The chunk-parallel GDN kernels (csrc/ls_gdn_cp.cu), their own source
compiled for the host and run on the CPU block emulator (tests/emu/), stage
by stage against the float64 chunk-parallel reference of
tests/test_oracle_gdn.py (itself pinned to the oracle), and the forward and
backward replays whole against the oracle, at the bf16 tolerance of their
tensor-core products."""
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest

from emu_support import check_run, compile_harness, rejected
from long_context_grpo_replay_gb300 import inputs
from test_oracle_gdn import _cp_prep

ROOT = Path(__file__).resolve().parents[1]
EMU = Path(__file__).resolve().parent / "emu"
CSRC = ROOT / "long_context_grpo_replay_gb300" / "csrc"
SRC = CSRC / "ls_gdn_cp.cu"
TOL_BF16 = 2e-2
# scratch per chunk: float32 [128 x 128] blocks E0, dU0, S_start, dU, GK;
# then bf16 tile images (32 KB, the swizzled shared-memory layout) ZK, ZW,
# -M, F hi, F lo, -M', F' hi, F' lo, T hi, T lo, K, Q, dO, S, G; then
# gamma_C, <G_end, S_start> and padding
FLOAT_BLOCKS, IMAGES = 5, 15
B_E0, B_DU0, B_SSTART, B_DU = range(4)
(I_ZK, I_ZW, I_M, I_FHI, I_FLO, I_MG, I_FGHI, I_FGLO, I_THI, I_TLO, I_K, I_Q, I_DO, I_S,
 I_G) = range(15)
SCR_FLOATS = FLOAT_BLOCKS * 128 * 128 + IMAGES * 8192 + 16
GAMMA_AT = FLOAT_BLOCKS * 128 * 128 + IMAGES * 8192
GS_AT = GAMMA_AT + 1


def block(chunk, i):
    """A float32 block decoded: element (r, c) at ((c // 4) * 128 + r) * 4 + c % 4."""
    return chunk[i * 16384:(i + 1) * 16384].reshape(32, 128, 4).transpose(1, 0, 2).reshape(128, 128)


def image(chunk, i):
    """A bf16 tile image decoded: element (r, c) sits in 64-column box c // 64,
    row r at 128 bytes per row, its 16-byte group XOR-ed with r mod 8."""
    raw = chunk[FLOAT_BLOCKS * 16384 + i * 8192:FLOAT_BLOCKS * 16384 + (i + 1) * 8192]
    u16 = raw.view(np.uint16)
    r = np.arange(128)[:, None]
    c = np.arange(128)[None, :]
    off = (c // 64) * 16384 + r * 128 + ((((c % 64) // 8) ^ (r % 8)) << 4) + (c % 8) * 2
    return (u16[off // 2].astype(np.uint32) << 16).view(np.float32)


def build(d, mutation=None):
    if shutil.which("g++") is None:
        pytest.skip("no host C++ compiler")
    src = SRC.read_text()
    if mutation:
        assert src.count(mutation[0]) == 1, mutation[0]
        src = src.replace(mutation[0], mutation[1])
    # the kernels, up to the end of their anonymous namespace; launchers stay out
    end = src.index("\n}  // namespace\n\nsize_t gdn_cp_workspace_bytes") + len("\n}  // namespace\n")
    text = src[:end] + "}  // namespace ls\n" + (EMU / "gdn_cp_run.inc").read_text()
    text = text.replace("extern __shared__", "extern")
    csrc = d / "x" / "csrc"
    csrc.mkdir(parents=True)
    (d / "include").mkdir()
    (csrc / "kernel.cu").write_text(text)
    shutil.copy(CSRC / "ls_internal.h", csrc / "ls_internal.h")
    shutil.copy(CSRC / "ls_gdn_tiles.cuh", csrc / "ls_gdn_tiles.cuh")
    shutil.copy(EMU / "ls_tc.cuh", csrc / "ls_tc.cuh")
    shutil.copy(ROOT / "include" / "ls.h", d / "include" / "ls.h")
    exe = d / "gdn_cp_emu"
    compile_harness("gdn_cp_main.cpp", csrc, exe)
    return exe


def run(exe, d, c, stage):
    B, R, H, _ = c["q"].shape
    with open(d / "in.bin", "wb") as f:
        np.array([B, H, R], dtype=np.int32).tofile(f)
        for x in ("s0", "q", "k", "v", "d_o", "g", "beta"):
            c[x].numpy().astype(np.float32).tofile(f)
    r = subprocess.run([str(exe), stage, str(d / "in.bin"), str(d / "out.bin")], capture_output=True,
                       text=True, timeout=900)
    check_run(r)
    nch = -(-R // 128)
    out = np.fromfile(d / "out.bin", dtype=np.float32, offset=4)
    n_scr = B * H * nch * SCR_FLOATS
    status = int(np.fromfile(d / "out.bin", dtype=np.uint32, count=1)[0])
    scr = out[:n_scr].reshape(B, H, nch, SCR_FLOATS)
    return status, scr, out[n_scr:]


@pytest.fixture(scope="module")
def emulator(tmp_path_factory):
    d = tmp_path_factory.mktemp("emu_gdn_cp")
    return build(d), d


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def _chain_terms(K, Q, dO, g, b, E0, ZK, dU0, ZW):
    """The chains' per-chunk terms from the chunk-local solves (float64):
    M = ZK^T W, F = E0^T W, M' = ZW^T diag(gamma b) K,
    F' = (gamma dO)^T Q - (gamma b dU0)^T K."""
    c = np.cumsum(g)
    gam = np.exp(c)
    W = np.exp(c[-1] - c)[:, None] * K
    return (ZK.T @ W, E0.T @ W, ZW.T @ ((gam * b)[:, None] * K),
            (gam[:, None] * dO).T @ Q - ((gam * b)[:, None] * dU0).T @ K)


def test_prep_solves_match_the_reference(emulator):
    exe, d = emulator
    B, H, R = 1, 2, 200  # two chunks, the second partial
    c = inputs.make_gdn_group(B, H, R, seed=31)
    status, scr, _ = run(exe, d, c, "prep")
    assert status == 0
    a = {x: t.numpy().astype(np.float64) for x, t in c.items()}
    errs = {}
    for h in range(H):
        for ch, (t0, t1) in enumerate([(0, 128), (128, 200)]):
            sl = slice(t0, t1)
            args = [a[x][0, sl, h] for x in ("k", "q", "v", "d_o", "g", "beta")]
            E0, ZK, dU0, ZW = _cp_prep(*args)
            M, F, Mg, Fg = _chain_terms(args[0], args[1], args[3], args[4], args[5], E0, ZK, dU0, ZW)
            n = t1 - t0
            sc = scr[0, h, ch]
            # T = (I + diag(b) GK)^-1, stored as its transpose's rows (row x = column x)
            n_ = t1 - t0
            kk, gg, bb = args[0], args[4], args[5]
            cc = np.cumsum(gg)
            A = bb[:, None] * np.tril(np.exp(cc[:, None] - cc[None, :]) * (kk @ kk.T), -1)
            Tn = np.linalg.inv(np.eye(n_) + A)
            Tt = image(sc, I_THI).astype(np.float64) + image(sc, I_TLO)
            errs["T"] = max(errs.get("T", 0.0), rel(Tt[:n_, :n_].T, Tn))
            got = {"E0": block(sc, B_E0), "dU0": block(sc, B_DU0), "ZK": image(sc, I_ZK),
                   "ZW": image(sc, I_ZW), "M": -image(sc, I_M),
                   "F": image(sc, I_FHI).astype(np.float64) + image(sc, I_FLO),
                   "Mg": -image(sc, I_MG),
                   "Fg": image(sc, I_FGHI).astype(np.float64) + image(sc, I_FGLO)}
            want = {"E0": E0, "dU0": dU0, "ZK": ZK, "ZW": ZW, "M": M, "F": F, "Mg": Mg, "Fg": Fg}
            for name, w in want.items():
                gv = got[name] if name in ("M", "F", "Mg", "Fg") else got[name][:n]
                errs[name] = max(errs.get(name, 0.0), rel(gv, w))
                if n < 128 and name in ("E0", "dU0", "ZK", "ZW"):
                    assert np.abs(got[name][n:]).max() == 0.0, name  # rows past the response
    print("prep max rel errs", errs)
    assert all(e <= TOL_BF16 for e in errs.values()), errs
    assert abs(scr[0, 0, 1, GAMMA_AT] - np.exp(a["g"][0, 128:200, 0].sum())) < 1e-5  # gamma_C, partial chunk


def _chains(s0, q, k, v, g, b, d_o):
    """float64 reference of the two chains over chunks of 128: S at each
    chunk's start, E, G at each chunk's end, dU, and the final state."""
    R = len(g)
    chunks = [(a, min(R, a + 128)) for a in range(0, R, 128)]
    pre = [_cp_prep(k[a:e], q[a:e], v[a:e], d_o[a:e], g[a:e], b[a:e]) for a, e in chunks]
    S, S_start, E = s0.copy(), [], []
    for (a, e), (E0, ZK, _, _) in zip(chunks, pre):
        S_start.append(S)
        c = np.cumsum(g[a:e])
        E.append(E0 - ZK @ S.T)
        S = np.exp(c[-1]) * S + E[-1].T @ (np.exp(c[-1] - c)[:, None] * k[a:e])
    G, G_end, dU = np.zeros_like(S), [None] * len(chunks), [None] * len(chunks)
    for ci in reversed(range(len(chunks))):
        a, e = chunks[ci]
        G_end[ci] = G
        c = np.cumsum(g[a:e])
        gam = np.exp(c)
        dU[ci] = pre[ci][2] + pre[ci][3] @ G.T
        G = np.exp(c[-1]) * G + (gam[:, None] * d_o[a:e]).T @ q[a:e] - \
            ((gam * b[a:e])[:, None] * dU[ci]).T @ k[a:e]
    return S_start, E, G_end, dU, S


def test_chains_match_the_reference(emulator):
    """S at each chunk's start (chain: fp32 and its bf16 image), G at its end
    (the bf16 image) and their inner product <G, S> (the backward chain), and
    dU (out), over three chunks, the last partial."""
    exe, d = emulator
    B, H, R = 2, 1, 300  # three chunks, the last partial; two members share s0
    c = inputs.make_gdn_group(B, H, R, seed=32)
    status, scr, _ = run(exe, d, c, "all")
    assert status == 0
    a = {x: t.numpy().astype(np.float64) for x, t in c.items()}
    errs = {}
    for m in range(B):
        S_start, E, G_end, dU, S_fin = _chains(a["s0"][0], a["q"][m, :, 0], a["k"][m, :, 0],
                                               a["v"][m, :, 0], a["g"][m, :, 0], a["beta"][m, :, 0],
                                               a["d_o"][m, :, 0])
        for ch in range(3):
            n = min(128, R - 128 * ch)
            sc = scr[m, 0, ch]
            for name, got, want in (("S_start", block(sc, B_SSTART), S_start[ch]),
                                    ("S image", image(sc, I_S), S_start[ch]),
                                    ("G image", image(sc, I_G), G_end[ch]),
                                    ("dU", block(sc, B_DU)[:n], dU[ch][:n])):
                if np.abs(want).max() == 0:
                    assert np.abs(got).max() == 0, name
                    continue
                errs[name] = max(errs.get(name, 0.0), rel(got, want))
            # <G, S>: against the product of the two norms (the sum cancels)
            gs = float((G_end[ch] * S_start[ch]).sum())
            scale = np.linalg.norm(G_end[ch]) * np.linalg.norm(S_start[ch])
            errs["<G,S>"] = max(errs.get("<G,S>", 0.0),
                                abs(float(sc[GS_AT]) - gs) / scale if scale else abs(float(sc[GS_AT])))
    print("chain max rel errs", errs)
    assert all(e <= TOL_BF16 for e in errs.values()), errs


def test_full_replay_matches_the_oracle(emulator):
    """prep, chain and out together: the forward (o, final state) and every
    gradient of a two-member group over three chunks, the last partial,
    against the float64 oracle."""
    from oracle.gdn import gdn_replay

    exe, d = emulator
    B, H, R = 2, 1, 300
    c = inputs.make_gdn_group(B, H, R, seed=33)
    status, _, rest = run(exe, d, c, "all")
    assert status == 0
    nt, ns, nsc = B * R * H * 128, B * H * 128 * 128, B * R * H
    got, i = {}, 0
    for name, n in (("o", nt), ("s_final", ns), ("dq", nt), ("dk", nt), ("dv", nt), ("dg", nsc),
                    ("dbeta", nsc)):
        got[name] = rest[i:i + n]
        i += n
    a = {x: t.numpy() for x, t in c.items()}
    errs = {}
    for m in range(B):
        want = gdn_replay(a["s0"], a["q"][m], a["k"][m], a["v"][m], a["g"][m], a["beta"][m],
                          a["d_o"][m])
        for name in got:
            gm = got[name].reshape((B,) + want[name].shape)[m]
            errs[name] = max(errs.get(name, 0.0), rel(gm, want[name]))
    print("full replay max rel errs", errs)
    assert all(e <= TOL_BF16 for e in errs.values()), errs


@pytest.mark.parametrize("B,H,R", [(1, 2, 1), (1, 1, 128), (1, 1, 129)],
                         ids=["one_token_two_heads", "one_exact_chunk", "one_token_past_a_chunk"])
def test_edge_lengths_match_the_oracle(emulator, B, H, R):
    from oracle.gdn import gdn_replay

    exe, d = emulator
    c = inputs.make_gdn_group(B, H, R, seed=40 + R)
    status, _, rest = run(exe, d, c, "all")
    assert status == 0
    nt, ns, nsc = B * R * H * 128, B * H * 128 * 128, B * R * H
    got, i = {}, 0
    for name, n in (("o", nt), ("s_final", ns), ("dq", nt), ("dk", nt), ("dv", nt), ("dg", nsc),
                    ("dbeta", nsc)):
        got[name] = rest[i:i + n]
        i += n
    a = {x: t.numpy() for x, t in c.items()}
    for m in range(B):
        want = gdn_replay(a["s0"], a["q"][m], a["k"][m], a["v"][m], a["g"][m], a["beta"][m],
                          a["d_o"][m])
        for name in got:
            gm = got[name].reshape((B,) + want[name].shape)[m]
            assert rel(gm, want[name]) <= TOL_BF16, (name, rel(gm, want[name]))


def test_bench_length_matches_the_oracle(emulator):
    """One head of one member at the benchmark's 4096 tokens (32 chunks):
    the chains' rounding does not grow over the chunks."""
    from oracle.gdn import gdn_replay

    exe, d = emulator
    B, H, R = 1, 1, 4096
    c = inputs.make_gdn_group(B, H, R, seed=77)
    status, _, rest = run(exe, d, c, "all")
    assert status == 0
    nt, ns, nsc = B * R * H * 128, B * H * 128 * 128, B * R * H
    got, i = {}, 0
    for name, n in (("o", nt), ("s_final", ns), ("dq", nt), ("dk", nt), ("dv", nt), ("dg", nsc),
                    ("dbeta", nsc)):
        got[name] = rest[i:i + n]
        i += n
    a = {x: t.numpy() for x, t in c.items()}
    want = gdn_replay(a["s0"], a["q"][0], a["k"][0], a["v"][0], a["g"][0], a["beta"][0], a["d_o"][0])
    errs = {n: rel(got[n].reshape(want[n].shape), want[n]) for n in got}
    assert all(e <= TOL_BF16 for e in errs.values()), errs


def _replay_outputs(rest, B, H, R):
    nt, ns, nsc = B * R * H * 128, B * H * 128 * 128, B * R * H
    got, i = {}, 0
    for name, n in (("o", nt), ("s_final", ns), ("dq", nt), ("dk", nt), ("dv", nt), ("dg", nsc),
                    ("dbeta", nsc)):
        got[name] = rest[i:i + n]
        i += n
    return got


def _forward_errors(exe, d, B, H, R, seed):
    from oracle.gdn import gdn_replay

    c = inputs.make_gdn_group(B, H, R, seed=seed)
    status, _, rest = run(exe, d, c, "fwd")
    assert status == 0
    got = _replay_outputs(rest, B, H, R)
    a = {x: t.numpy() for x, t in c.items()}
    errs = {}
    for m in range(B):
        want = gdn_replay(a["s0"], a["q"][m], a["k"][m], a["v"][m], a["g"][m], a["beta"][m],
                          a["d_o"][m])
        for name in ("o", "s_final"):
            gm = got[name].reshape((B,) + want[name].shape)[m]
            errs[name] = max(errs.get(name, 0.0), rel(gm, want[name]))
    return errs


@pytest.mark.parametrize("B,H,R", [(2, 1, 300), (1, 2, 1), (1, 1, 128), (1, 1, 129), (1, 1, 1024)],
                         ids=["three_chunks_two_members", "one_token_two_heads", "one_exact_chunk",
                              "one_token_past_a_chunk", "eight_chunks"])
def test_forward_matches_the_oracle(emulator, B, H, R):
    """The chunk-parallel forward (prep's forward share, the state chain, the
    forward output): o and the final state against the float64 oracle (the
    state chain over the bench's 32 chunks runs in the backward's
    bench-length case)."""
    exe, d = emulator
    errs = _forward_errors(exe, d, B, H, R, seed=50 + R)
    print("forward max rel errs", errs)
    assert all(e <= TOL_BF16 for e in errs.values()), errs


@pytest.mark.parametrize("mutation", [
    ("        f32[xx] = s <= t ? __expf(ct - sc[s]) * __uint_as_float(t32[xx]) : 0.f;\n      }\n"
     "#pragma unroll\n      for (int gg = 0; gg < 4; ++gg) st_shared_v4(F0",
     "        f32[xx] = s < t ? __expf(ct - sc[s]) * __uint_as_float(t32[xx]) : 0.f;\n      }\n"
     "#pragma unroll\n      for (int gg = 0; gg < 4; ++gg) st_shared_v4(F0"),
    ("mma_group_amn(tb + 0, sb + kPrepR3, sb + kPrepR2, true, false);    // M = ZK^T W",
     "mma_group(tb + 0, sb + kPrepR3, sb + kPrepR2, true, false);    // M = ZK^T W"),
    ("st[cb * 32 + xx] = fmaf(gc, st[cb * 32 + xx], __uint_as_float(t32[xx]));",
     "st[cb * 32 + xx] = fmaf(1.f, st[cb * 32 + xx], __uint_as_float(t32[xx]));"),
], ids=["P_without_its_diagonal", "M_with_ZK_read_K_major", "chain_without_the_decay"])
def test_emulator_rejects_planted_kernel_mistakes(tmp_path, mutation):
    """A mistake planted in a copy of the kernel source must fail the
    forward comparison."""
    exe = build(tmp_path, mutation)
    assert rejected(lambda: not all(e <= TOL_BF16 for e in
                                    _forward_errors(exe, tmp_path, 1, 1, 300, seed=61).values()))


def test_backward_reusing_the_forward_scratch_is_bit_identical(emulator):
    """The forward, then the backward with the forward's scratch (its terms
    and states not formed again), gives the gradients of the backward that
    forms everything itself, bit for bit."""
    exe, d = emulator
    B, H, R = 2, 1, 300
    c = inputs.make_gdn_group(B, H, R, seed=71)
    st1, _, full = run(exe, d, c, "all")
    st2, _, reuse = run(exe, d, c, "fwd_bwd")
    assert st1 == 0 and st2 == 0
    g1, g2 = _replay_outputs(full, B, H, R), _replay_outputs(reuse, B, H, R)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.array_equal(g1[name], g2[name]), name
    for name in ("o", "s_final"):  # the reusing run's o and s_final come from the forward
        assert np.array_equal(g1[name], g2[name]), name


def _backward_errors(exe, d, B, H, R, seed):
    from oracle.gdn import gdn_replay

    c = inputs.make_gdn_group(B, H, R, seed=seed)
    status, _, rest = run(exe, d, c, "fwd_bwd")
    assert status == 0
    got = _replay_outputs(rest, B, H, R)
    a = {x: t.numpy() for x, t in c.items()}
    errs = {}
    for m in range(B):
        want = gdn_replay(a["s0"], a["q"][m], a["k"][m], a["v"][m], a["g"][m], a["beta"][m],
                          a["d_o"][m])
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            gm = got[name].reshape((B,) + want[name].shape)[m]
            errs[name] = max(errs.get(name, 0.0), rel(gm, want[name]))
    return errs


def test_backward_reusing_the_forward_matches_the_oracle(emulator):
    exe, d = emulator
    errs = _backward_errors(exe, d, 2, 1, 300, seed=62)
    print("backward (reusing the forward) max rel errs", errs)
    assert all(e <= TOL_BF16 for e in errs.values()), errs


@pytest.mark.parametrize("mutation", [
    ("f32[xx] = s <= t ? __expf(ct - sc[s]) * dp : 0.f;",
     "f32[xx] = s < t ? __expf(ct - sc[s]) * dp : 0.f;"),
    ("mma_group(tb + 384, sb + kGr4, sb + kGr1, true, false);  // ZW = T^T (w K)",
     "mma_group_amn(tb + 384, sb + kGr4, sb + kGr1, true, false);  // ZW = T^T (w K)"),
    ("      for (int xx = 0; xx < 32; ++xx) f32[xx] += __uint_as_float(t32[xx]);",
     "      for (int xx = 0; xx < 32; ++xx) f32[xx] -= __uint_as_float(t32[xx]);"),
], ids=["LdP_without_its_diagonal", "ZW_with_T_read_M_major", "dU_with_ZW_G_subtracted"])
def test_emulator_rejects_planted_backward_mistakes(tmp_path, mutation):
    """A mistake planted in a copy of the backward kernels' source must fail
    the gradients' comparison."""
    exe = build(tmp_path, mutation)
    assert rejected(lambda: not all(e <= TOL_BF16 for e in
                                    _backward_errors(exe, tmp_path, 1, 1, 300, seed=63).values()))
