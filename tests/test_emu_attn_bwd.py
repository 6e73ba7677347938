"""The prompt-attention backward kernel (tc_bwd_dq_ring_kernel in
csrc/ls_tc_bwd.cu), its own source compiled for the host and run on the CPU
block emulator (tests/emu/): TMA copies and tcgen05 MMAs run asynchronously
on engine threads with random delays, so a missing wait or an early slot
reuse shows as wrong data or a timeout.  Three prompt parts over a scattered,
NaN-poisoned pool with a partial last page, plus the causal response part,
for a GQA 12/2 group; the parts' float32 dQ, summed and scaled, must match
the float64 oracle at the bf16 tolerance.  This checks the kernel's indexing
and its producer / MMA / softmax protocol without a GPU."""
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle.ref as ref
from emu_support import check_run, compile_harness, rejected
from long_context_grpo_replay_gb300 import inputs

ROOT = Path(__file__).resolve().parents[1]
EMU = Path(__file__).resolve().parent / "emu"
SRC = ROOT / "long_context_grpo_replay_gb300" / "csrc" / "ls_tc_bwd.cu"
TOL_BF16 = 2e-2


KERNELS = {  # kernel: (first line of its block, line after it)
    "ring": ("struct BwdRingLayout", "cudaError_t bwd_ring("),
}


def kernel_source(mutation=None, kernel="ring"):
    """A kernel's source, cut out of its file: the constants and parameter
    block, then the kernel; host launchers left out.  A mutation is applied
    inside the kernel's own block."""
    src = SRC.read_text()
    start, end = KERNELS[kernel]
    body = src[src.index(start):src.index(end)]
    if mutation:
        assert mutation[0] in body, mutation[0]
        i = body.rindex(mutation[0])
        body = body[:i] + mutation[1] + body[i + len(mutation[0]):]
    pre = src[:src.index("// ===========================================================================\n// Backward with 128-key tiles")]
    text = pre + body + "}  // namespace\n}  // namespace ls\n"
    text = text.replace("extern __shared__", "extern")
    ex2 = 'asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));'
    assert ex2 in text
    return text.replace(ex2, "y = exp2f(x);")


def build(d, mutation=None, kernel="ring"):
    if shutil.which("g++") is None:
        pytest.skip("no host C++ compiler")
    csrc = d / "x" / "csrc"
    csrc.mkdir(parents=True)
    (d / "include").mkdir()
    (csrc / "kernel.cu").write_text(kernel_source(mutation, kernel))
    shutil.copy(SRC.parent / "ls_internal.h", csrc / "ls_internal.h")
    shutil.copy(EMU / "ls_tc.cuh", csrc / "ls_tc.cuh")
    shutil.copy(ROOT / "include" / "ls.h", d / "include" / "ls.h")
    exe = d / "attn_bwd_emu"
    compile_harness("attn_bwd_main.cpp", csrc, exe)
    return exe


def _bf16_bytes(t):
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().tobytes()


def run_case(exe, d, P=600, R=64, seed=5, span=256):
    w = inputs.Workload("emu", 12, 2, 256, 256, P, (R,), "bf16", seed=seed, pool_factor=2,
                        poison=True)
    pr = inputs.make_prompt(w, "cpu")
    m = inputs.make_member(w, 0, "cpu")
    want = ref.replay_member(pr["k_pool"], pr["v_pool"], pr["page_table"], P, m["q"], m["k"], m["v"],
                             m["d_o"], scale=w.scale)
    ns = -(-P // span)
    kp, pt = pr["k_pool"], pr["page_table"]
    hdr = np.array([w.hq, w.hkv, R, P, w.page_size, kp.shape[0], pt.shape[0], ns, span],
                   dtype=np.int64)
    with open(d / "in.bin", "wb") as f:
        f.write(hdr.tobytes())
        f.write(np.array([w.scale], dtype=np.float32).tobytes())
        f.write(_bf16_bytes(kp))
        f.write(_bf16_bytes(pr["v_pool"]))
        f.write(pt.to(torch.int32).numpy().tobytes())
        for x in ("q", "d_o", "k", "v"):
            f.write(_bf16_bytes(m[x]))
        f.write(want["lse"].astype(np.float32).tobytes())
        f.write(want["delta"].astype(np.float32).tobytes())
    r = subprocess.run([str(exe), str(d / "in.bin"), str(d / "out.bin")], capture_output=True,
                       text=True, timeout=900)
    check_run(r)
    out = np.fromfile(d / "out.bin", dtype=np.uint32, count=2)
    parts = np.fromfile(d / "out.bin", dtype=np.float32, offset=8).reshape(ns + 1, R, w.hq, 256)
    dq = parts.astype(np.float64).sum(0) * w.scale
    return out, float(np.abs(dq - want["dq"]).max() / np.abs(want["dq"]).max())


@pytest.fixture(scope="module", params=["ring"])
def emulator(tmp_path_factory, request):
    d = tmp_path_factory.mktemp("emu_attn_bwd_" + request.param)
    return build(d, kernel=request.param), d


def test_emulated_backward_matches_the_oracle(emulator):
    exe, d = emulator
    status, err = run_case(exe, d)
    assert status[0] == 0, status  # no bad page, no wait that gave up
    assert err <= TOL_BF16, err


def test_emulated_backward_over_many_tiles(emulator):
    """One 1500-key part (12 tiles, 48 chunks: the ring's slot pattern runs
    through more than two periods) with a partial last tile."""
    exe, d = emulator
    status, err = run_case(exe, d, P=1500, R=40, seed=6, span=1536)
    assert status[0] == 0, status
    assert err <= TOL_BF16, err


@pytest.mark.parametrize("mutation", [
    ("constexpr uint32_t idesc_q = idesc_bf16(kBM, 128, true);",
     "constexpr uint32_t idesc_q = idesc_bf16(kBM, 128, false);"),
    ("        if (!mbar_wait(smem_u32(&bar_dsf), j & 1, abortp)) { fail(__LINE__); break; }\n", ""),
    ("(j > 0 || kk > 0) ? 1u : 0u);", "kk > 0 ? 1u : 0u);"),
    ("tbase + L::kTmemX + 32 * (kk >> 1) + 8 * (kk & 1)", "tbase + L::kTmemX + kk * 8"),
], ids=["K_read_K_major_in_dQ", "dQ_before_dS_is_written", "dQ_reset_every_tile",
        "dS_of_the_second_half_misplaced"])
def test_emulator_rejects_planted_kernel_mistakes(tmp_path, mutation):
    """A wrong operand layout, a missing wait, a lost accumulation and a
    misplaced operand, each planted in a copy of the ring kernel's source,
    must fail the comparison (or stop the emulated kernel on one of the
    emulator's checks, which a missing wait may do)."""
    exe = build(tmp_path, mutation)

    def wrong():
        status, err = run_case(exe, tmp_path)
        return not err <= TOL_BF16  # also true for NaN

    assert rejected(wrong)
