"""The chunkwise tensor-core GDN forward (csrc/ls_gdn_chunk.cu), its own
source compiled for the host and run on the CPU block emulator
(tests/emu/): one std::thread per CUDA thread, shared and tensor memory as
host arrays, tcgen05.mma evaluated through the operand layouts the kernels
encode.  The result is compared with the float64 oracle at the bf16
tolerance, across three chunks with a partial last one, an exact chunk and a
single token.  This checks the kernel's indexing, phase order and barrier
protocol without a GPU; timing and hardware-only behaviour stay for the GPU
tests."""
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest

from emu_support import compile_harness
from long_context_grpo_replay_gb300 import inputs
from oracle.gdn import gdn_replay

ROOT = Path(__file__).resolve().parents[1]
EMU = Path(__file__).resolve().parent / "emu"
SRC = ROOT / "long_context_grpo_replay_gb300" / "csrc" / "ls_gdn_chunk.cu"
TOL_BF16 = 2e-2


def _build(d, mutation=None):
    """Compile the kernel's source (optionally with one text substitution) for
    the emulator, in directory d."""
    if shutil.which("g++") is None:
        pytest.skip("no host C++ compiler")
    src = SRC.read_text()
    if mutation:
        assert mutation[0] in src, mutation[0]
        src = src.replace(mutation[0], mutation[1], 1)
    start = src.index("gdn_chunk_fwd_kernel(")
    end = src.index("\n}  // namespace\n", start) + len("\n}  // namespace\n")
    src = src[:end].replace("extern __shared__", "extern")
    (d / "kernel.cu").write_text(src + "}  // namespace ls\n")
    for name in ("ls_internal.h", "ls_tc.cuh"):
        shutil.copy(EMU / name, d / name)
    exe = d / "gdn_chunk_emu"
    compile_harness("gdn_chunk_main.cpp", d, exe)
    return d, exe


@pytest.fixture(scope="module")
def emulator(tmp_path_factory):
    return _build(tmp_path_factory.mktemp("emu_gdn_chunk"))


def _run(emulator, c):
    d, exe = emulator
    B, R, H, _ = c["q"].shape
    with open(d / "in.bin", "wb") as f:
        np.array([B, H, R], dtype=np.int32).tofile(f)
        for x in ("s0", "q", "k", "v", "g", "beta"):
            c[x].numpy().astype(np.float32).tofile(f)
    r = subprocess.run([str(exe), str(d / "in.bin"), str(d / "out.bin")], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    out = np.fromfile(d / "out.bin", dtype=np.float32)
    n_o = B * R * H * 128
    return out[:n_o].reshape(B, R, H, 128), out[n_o:].reshape(B, H, 128, 128)


def _errors(emulator, B, H, R, seed):
    c = inputs.make_gdn_group(B, H, R, seed=seed)
    o, s_final = _run(emulator, c)
    a = {x: c[x].numpy() for x in c}
    errs = []
    for b in range(B):
        want = gdn_replay(a["s0"], a["q"][b], a["k"][b], a["v"][b], a["g"][b], a["beta"][b])
        errs.append((np.abs(o[b] - want["o"]).max() / np.abs(want["o"]).max(),
                     np.abs(s_final[b] - want["s_final"]).max() / np.abs(want["s_final"]).max()))
    return errs


@pytest.mark.parametrize("B,H,R", [(1, 2, 300), (1, 1, 128), (2, 1, 1), (2, 2, 129)],
                         ids=["three_chunks_r300", "one_chunk_r128", "one_token",
                              "one_token_past_a_chunk"])
def test_emulated_chunk_forward_matches_the_oracle(emulator, B, H, R):
    for e_o, e_s in _errors(emulator, B, H, R, seed=90 + R):
        assert e_o <= TOL_BF16 and e_s <= TOL_BF16, (e_o, e_s)


@pytest.mark.parametrize("mutation", [
    ("id_mn = idesc_bf16(128, 128, true)", "id_mn = idesc_bf16(128, 128, false)"),
    ("const float wj = expf(sc[kC - 1] - sc[j]);", "const float wj = 1.f;"),
    ("pv[xx] = s <= r ?", "pv[xx] = s < r ?"),
], ids=["W_read_K_major", "W_not_decayed", "P_without_diagonal"])
def test_emulator_rejects_planted_kernel_mistakes(tmp_path, mutation):
    """A wrong operand layout, a dropped decay or a dropped diagonal in a copy
    of the kernel source must fail the comparison."""
    emulator = _build(tmp_path, mutation)
    assert max(max(e) for e in _errors(emulator, 1, 1, 300, seed=91)) > 10 * TOL_BF16
