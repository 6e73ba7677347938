"""The prompt-attention forward kernel (tc_fwd_ring_kernel in
csrc/ls_tc_fwd.cu), its own source compiled for the host and run on the CPU
block emulator (tests/emu/), with asynchronous TMA and MMA engines.  Three
prompt parts over a scattered, NaN-poisoned pool with a partial last page,
plus the causal response part, for a GQA 12/2 group; the parts, merged by
log-sum-exp, must match the float64 oracle (bf16 tolerance on o, 1e-3 on the
LSE).  This checks the kernel's chunk ring, its producer / MMA / eight-warp
softmax protocol and its indexing without a GPU."""
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
SRC = ROOT / "long_context_grpo_replay_gb300" / "csrc" / "ls_tc_fwd.cu"
TOL_BF16, LSE_TOL = 2e-2, 1e-3


def kernel_source(mutation=None):
    """The default (chunk-ring) kernel's source cut out of its file: the
    constants and parameter block, then the ring kernel; launchers left out."""
    src = SRC.read_text()
    if mutation:  # applied to the last occurrence: the ring kernel comes last
        i = src.rindex(mutation[0])
        src = src[:i] + mutation[1] + src[i + len(mutation[0]):]
    pre = src[:src.index("// ===========================================================================\n// Chunk-ring forward")]
    body = src[src.index("struct FwdRingLayout"):src.index("cudaError_t fwd_ring(")]
    text = pre + body + "}  // namespace\n}  // namespace ls\n"
    text = text.replace("extern __shared__", "extern")
    for asm, host in [('asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));', "y = exp2f(x);"),
                      ('asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));',
                       "d = fmaxf(fmaxf(a, b), c);")]:
        assert asm in text
        text = text.replace(asm, host)
    return text


def build(d, mutation=None):
    if shutil.which("g++") is None:
        pytest.skip("no host C++ compiler")
    csrc = d / "x" / "csrc"
    csrc.mkdir(parents=True)
    (d / "include").mkdir()
    (csrc / "kernel.cu").write_text(kernel_source(mutation))
    shutil.copy(SRC.parent / "ls_internal.h", csrc / "ls_internal.h")
    shutil.copy(EMU / "ls_tc.cuh", csrc / "ls_tc.cuh")
    shutil.copy(ROOT / "include" / "ls.h", d / "include" / "ls.h")
    exe = d / "attn_fwd_emu"
    compile_harness("attn_fwd_main.cpp", csrc, exe)
    return exe


def _bf16_bytes(t):
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().tobytes()


def run_case(exe, d, P=600, R=64, seed=6, span=256):
    w = inputs.Workload("emu", 12, 2, 256, 256, P, (R,), "bf16", seed=seed, pool_factor=2,
                        poison=True)
    pr = inputs.make_prompt(w, "cpu")
    m = inputs.make_member(w, 0, "cpu")
    want = ref.replay_member(pr["k_pool"], pr["v_pool"], pr["page_table"], P, m["q"], m["k"], m["v"],
                             scale=w.scale)
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
        for x in ("q", "k", "v"):
            f.write(_bf16_bytes(m[x]))
    r = subprocess.run([str(exe), str(d / "in.bin"), str(d / "out.bin")], capture_output=True,
                       text=True, timeout=900)
    check_run(r)
    status = np.fromfile(d / "out.bin", dtype=np.uint32, count=2)
    n = (ns + 1) * R * w.hq
    vals = np.fromfile(d / "out.bin", dtype=np.float32, offset=8)
    o_parts = vals[:n * 256].reshape(ns + 1, R * w.hq, 256).astype(np.float64)
    l_parts = vals[n * 256:].reshape(ns + 1, R * w.hq).astype(np.float64)
    lse = np.logaddexp.reduce(l_parts, axis=0)
    o = (np.exp(l_parts - lse)[:, :, None] * np.nan_to_num(o_parts)).sum(0)
    e_o = float(np.abs(o.reshape(R, w.hq, 256) - want["o"]).max() / np.abs(want["o"]).max())
    e_l = float(np.abs(lse.reshape(R, w.hq) - want["lse"]).max())
    return status, e_o, e_l


@pytest.fixture(scope="module")
def emulator(tmp_path_factory):
    d = tmp_path_factory.mktemp("emu_attn_fwd")
    return build(d), d


def test_emulated_forward_matches_the_oracle(emulator):
    exe, d = emulator
    status, e_o, e_l = run_case(exe, d)
    assert status[0] == 0, status
    assert e_o <= TOL_BF16 and e_l <= LSE_TOL, (e_o, e_l)


def test_emulated_forward_over_many_tiles(emulator):
    """One 1500-key part: 12 tiles, 24 ring units, the slot releases wrap the
    five-chunk ring many times; partial last tile."""
    exe, d = emulator
    status, e_o, e_l = run_case(exe, d, P=1500, R=40, seed=7, span=1536)
    assert status[0] == 0, status
    assert e_o <= TOL_BF16 and e_l <= LSE_TOL, (e_o, e_l)


@pytest.mark.parametrize("mutation", [
    ("constexpr uint32_t idesc_pv = idesc_bf16(kBM, kD, true);",
     "constexpr uint32_t idesc_pv = idesc_bf16(kBM, kD, false);"),
    ("            if (!mbar_wait_warp(smem_u32(&bar_cd[v % NCD]), (v / NCD) & 1, abortp)) {",
     "            if (false) {"),
], ids=["V_read_K_major", "K_slot_reused_before_S_is_done"])
def test_emulator_rejects_planted_kernel_mistakes(tmp_path, mutation):
    """V read as a K-major operand in P V, or a K chunk's slot refilled
    before the S that reads it is complete, planted in a copy of the kernel
    source, must fail the comparison (or stop the emulated kernel on one of
    the emulator's checks, which a missing wait may do)."""
    exe = build(tmp_path, mutation)

    def wrong():
        status, e_o, e_l = run_case(exe, tmp_path, P=1500, R=40, seed=7, span=1536)
        return not (e_o <= TOL_BF16 and e_l <= LSE_TOL)

    assert rejected(wrong)
