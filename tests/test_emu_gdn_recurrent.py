"""The recurrent GDN replay kernels (gdn_fwd_kernel, gdn_bwd_kernel in
csrc/ls_gdn.cu), their own source compiled for the host and run on the CPU
block emulator (tests/emu/), against the float64 oracle at the float32
tolerance: two members, a response that spans three of the backward's
8-token segments with a partial last one.  A mistake planted in a copy of
the source must fail.  This lets the recurrent kernels be changed and
checked without a GPU."""
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest

from emu_support import check_run, compile_harness
from long_context_grpo_replay_gb300 import inputs
from oracle.gdn import gdn_replay

ROOT = Path(__file__).resolve().parents[1]
EMU = Path(__file__).resolve().parent / "emu"
SRC = ROOT / "long_context_grpo_replay_gb300" / "csrc" / "ls_gdn.cu"
TOL_F32 = 1e-5


def build(d, mutation=None):
    if shutil.which("g++") is None:
        pytest.skip("no host C++ compiler")
    src = SRC.read_text()
    if mutation:
        assert mutation[0] in src, mutation[0]
        src = src.replace(mutation[0], mutation[1], 1)
    # the kernels and the workspace size; the launchers (<<<...>>>) stay out
    end = src.index("bool gdn_supported(")
    text = src[:end] + "}  // namespace ls\n"
    text = text.replace("extern __shared__ float red[];", "extern float red[];")
    (d / "kernel.cu").write_text(text)
    for name in ("ls_internal.h", "ls_tc.cuh"):
        shutil.copy(EMU / name, d / name)
    exe = d / "gdn_rec_emu"
    compile_harness("gdn_recurrent_main.cpp", d, exe)
    return exe


def run_case(exe, d, B=2, H=1, R=20, seed=13):
    c = inputs.make_gdn_group(B, H, R, seed=seed)
    with open(d / "in.bin", "wb") as f:
        np.array([B, H, R], dtype=np.int32).tofile(f)
        for x in ("s0", "q", "k", "v", "d_o", "g", "beta"):
            c[x].numpy().astype(np.float32).tofile(f)
    r = subprocess.run([str(exe), str(d / "in.bin"), str(d / "out.bin")], capture_output=True,
                       text=True, timeout=900)
    check_run(r)
    out = np.fromfile(d / "out.bin", dtype=np.float32)
    nt, ns, nsc = B * R * H * 128, B * H * 128 * 128, B * R * H
    sizes = [("o", nt), ("s_final", ns), ("dq", nt), ("dk", nt), ("dv", nt), ("dg", nsc),
             ("dbeta", nsc)]
    got, i = {}, 0
    for name, n in sizes:
        got[name] = out[i:i + n]
        i += n
    a = {x: t.numpy() for x, t in c.items()}
    errs = {}
    for b in range(B):
        want = gdn_replay(a["s0"], a["q"][b], a["k"][b], a["v"][b], a["g"][b], a["beta"][b],
                          a["d_o"][b])
        for name, _ in sizes:
            g_ = got[name].reshape((B,) + want[name].shape)[b]
            e = float(np.abs(g_ - want[name]).max() / np.abs(want[name]).max())
            errs[name] = max(errs.get(name, 0.0), e)
    return errs


def test_emulated_recurrent_kernels_match_the_oracle(tmp_path):
    errs = run_case(build(tmp_path), tmp_path)
    assert all(e <= TOL_F32 for e in errs.values()), errs


def test_emulator_rejects_a_planted_mistake(tmp_path):
    """dk without its decayed S^T dw term, planted in a copy of the source."""
    exe = build(tmp_path, ("r1[c] = b * gg[c] * w - a * sp[c] * dw;", "r1[c] = b * gg[c] * w;"))
    errs = run_case(exe, tmp_path)
    assert errs["dk"] > 100 * TOL_F32 and errs["o"] <= TOL_F32, errs
