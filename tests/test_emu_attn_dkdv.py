"""The response dK/dV kernel (tc_dkdv_kernel in csrc/ls_tc_dkdv.cu), its own
source compiled for the host and run on the CPU block emulator (tests/emu/),
against the float64 oracle at the bf16 tolerance: a GQA 12/2 group with 200
response keys (a full and a partial 128-key tile; 64-row query steps with a
partial last one), and an empty prompt so that every query row's LSE and
delta come from the response keys alone."""
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle.ref as ref
from emu_support import check_run, compile_harness
from long_context_grpo_replay_gb300 import inputs

ROOT = Path(__file__).resolve().parents[1]
EMU = Path(__file__).resolve().parent / "emu"
SRC = ROOT / "long_context_grpo_replay_gb300" / "csrc" / "ls_tc_dkdv.cu"
TOL_BF16 = 2e-2


def build(d):
    if shutil.which("g++") is None:
        pytest.skip("no host C++ compiler")
    src = SRC.read_text()
    end = src.index("\n}  // namespace\n\ncudaError_t launch_tc_dkdv") + len("\n}  // namespace\n")
    text = src[:end] + "}  // namespace ls\n"
    text = text.replace("extern __shared__", "extern")
    ex2 = 'asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));'
    assert ex2 in text
    text = text.replace(ex2, "y = exp2f(x);")
    csrc = d / "x" / "csrc"
    csrc.mkdir(parents=True)
    (d / "include").mkdir()
    (csrc / "kernel.cu").write_text(text)
    shutil.copy(SRC.parent / "ls_internal.h", csrc / "ls_internal.h")
    shutil.copy(EMU / "ls_tc.cuh", csrc / "ls_tc.cuh")
    shutil.copy(ROOT / "include" / "ls.h", d / "include" / "ls.h")
    exe = d / "attn_dkdv_emu"
    compile_harness("attn_dkdv_main.cpp", csrc, exe)
    return exe


def _bf16_bytes(t):
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().tobytes()


def test_emulated_dkdv_matches_the_oracle(tmp_path):
    exe = build(tmp_path)
    R = 200
    w = inputs.Workload("emu", 12, 2, 256, 256, 256, (R,), "bf16", seed=8, pool_factor=2, poison=True)
    pr = inputs.make_prompt(w, "cpu")
    m = inputs.make_member(w, 0, "cpu")
    want = ref.replay_member(pr["k_pool"], pr["v_pool"], pr["page_table"], 0, m["q"], m["k"], m["v"],
                             m["d_o"], scale=w.scale)
    with open(tmp_path / "in.bin", "wb") as f:
        f.write(np.array([w.hq, w.hkv, R], dtype=np.int64).tobytes())
        f.write(np.array([w.scale], dtype=np.float32).tobytes())
        for x in ("q", "d_o", "k", "v"):
            f.write(_bf16_bytes(m[x]))
        f.write(want["lse"].astype(np.float32).tobytes())
        f.write(want["delta"].astype(np.float32).tobytes())
    r = subprocess.run([str(exe), str(tmp_path / "in.bin"), str(tmp_path / "out.bin")],
                       capture_output=True, text=True, timeout=900)
    check_run(r)
    status = np.fromfile(tmp_path / "out.bin", dtype=np.uint32, count=2)
    assert status[0] == 0, status
    raw = np.fromfile(tmp_path / "out.bin", dtype=np.uint16, offset=8)
    n = R * w.hkv * 256
    as_f = lambda u: torch.from_numpy(u.astype(np.int16)).view(torch.bfloat16).double().numpy()
    dk, dv = as_f(raw[:n]).reshape(R, w.hkv, 256), as_f(raw[n:]).reshape(R, w.hkv, 256)
    e_k = float(np.abs(dk - want["dk"]).max() / np.abs(want["dk"]).max())
    e_v = float(np.abs(dv - want["dv"]).max() / np.abs(want["dv"]).max())
    assert e_k <= TOL_BF16 and e_v <= TOL_BF16, (e_k, e_v)
