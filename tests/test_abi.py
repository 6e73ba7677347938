"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every symbol include/ls.h declares, and rejects bad arguments
with a status before any launch."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def ls():
    from long_context_grpo_replay_gb300 import build

    build.build()
    import long_context_grpo_replay_gb300.binding as b

    b.lib()
    return b


def _declared_symbols():
    text = (ROOT / "include" / "ls.h").read_text()
    return sorted(set(re.findall(r"^LS_API\s+[\w\s\*]+?\b(ls_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for required in ("ls_kv_page_write", "ls_replay_fwd", "ls_lse_merge",
                     "ls_replay_bwd_preprocess", "ls_replay_bwd", "ls_replay_group",
                     "ls_replay_workspace_size", "ls_read_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(ls):
    L = ls.lib()
    for name in _declared_symbols():
        assert hasattr(L, name), name
    assert set(ls.EXPORTED_SYMBOLS) <= set(_declared_symbols())


def test_status_strings(ls):
    assert ls.ls_status_string(0) == "LS_OK"
    assert ls.ls_status_string(3) == "LS_ERR_WORKSPACE_TOO_SMALL"
    assert ls.ls_status_string(6) == "LS_ERR_DEVICE_TIMEOUT"
    assert ls.ls_num_kernel_ids() >= 8
    names = {ls.ls_kernel_name(k) for k in range(ls.ls_num_kernel_ids())}
    assert {"tc_fwd", "tc_bwd_dq", "lse_merge", "page_write"} <= names


def _desc(ls, **kw):
    d = dict(hq=24, hkv=4, head_dim=256, page_size=256, dtype=ls.LS_DTYPE_BF16)
    d.update(kw)
    return ls.desc_for(d["hq"], d["hkv"], d["head_dim"], d["page_size"], d["dtype"])


def _prompt(ls, P=4096, pool=16, pages=16):
    # fake, never-dereferenced but aligned device addresses: validation only
    return ls.PromptKV(1 << 20, 1 << 21, pool, 1 << 22, pages, P)


@pytest.mark.parametrize("bad,status", [
    (dict(hq=25), 1), (dict(hkv=0), 1), (dict(head_dim=96), 2), (dict(page_size=0), 1),
    (dict(dtype=7), 1),
])
def test_bad_desc_is_rejected(ls, bad, status):
    d = _desc(ls, **bad)
    n = ctypes.c_size_t(0)
    st = ls.lib().ls_replay_workspace_size(ctypes.byref(d), ctypes.byref(_prompt(ls)), 64,
                                           ctypes.byref(n))
    assert st == status
    assert ls.ls_last_error()


def test_bad_scale_is_rejected(ls):
    d = _desc(ls)
    d.softmax_scale = float("nan")
    n = ctypes.c_size_t(0)
    assert ls.lib().ls_replay_workspace_size(ctypes.byref(d), ctypes.byref(_prompt(ls)), 8,
                                             ctypes.byref(n)) == 1


def test_prompt_too_short_for_pages(ls):
    d = _desc(ls)
    p = _prompt(ls, P=5000, pages=16)  # 16 pages * 256 < 5000
    n = ctypes.c_size_t(0)
    assert ls.lib().ls_replay_workspace_size(ctypes.byref(d), ctypes.byref(p), 8,
                                             ctypes.byref(n)) == 1
    assert "prompt_len" in ls.ls_last_error()


def test_workspace_size_is_independent_of_group_and_monotone(ls):
    d = _desc(ls)
    p = _prompt(ls, P=2097152, pool=8192, pages=8192)
    sizes = [ls.ls_replay_workspace_size(d, p, R) for R in (1, 64, 512, 4096)]
    assert sizes == sorted(sizes)
    assert sizes[-1] >= 4096 * 24 * 256 * 4  # at least one float32 partial of O


def test_null_workspace_rejected_before_launch(ls):
    d = _desc(ls)
    p = _prompt(ls)
    L = ls.lib()
    fake = 1 << 24
    st = L.ls_replay_fwd(ctypes.byref(d), ctypes.byref(p), fake, fake, fake, 64, fake, fake,
                         None, 0, None)
    assert st == 1 and "workspace" in ls.ls_last_error()
    st = L.ls_replay_fwd(ctypes.byref(d), ctypes.byref(p), fake, fake, fake, 64, fake, fake,
                         fake, 16, None)
    assert st == 3  # too small


def test_misaligned_and_null_buffers_rejected(ls):
    d = _desc(ls)
    p = _prompt(ls)
    L = ls.lib()
    fake = 1 << 24
    assert L.ls_replay_fwd(ctypes.byref(d), ctypes.byref(p), fake + 2, fake, fake, 64, fake,
                           fake, fake, 1 << 30, None) == 1
    assert L.ls_replay_fwd(ctypes.byref(d), ctypes.byref(p), None, fake, fake, 64, fake, fake,
                           fake, 1 << 30, None) == 1
    assert L.ls_replay_bwd(ctypes.byref(d), ctypes.byref(p), fake, fake, fake, fake, fake, None,
                           64, fake, fake, fake, fake, 1 << 30, None) == 1
    assert L.ls_lse_merge(0, 10, 256, fake, fake, 1, fake, fake, None) == 1
    assert L.ls_lse_merge(2, 10, 6, fake, fake, 1, fake, fake, None) == 1


def test_zero_length_calls_are_noops(ls):
    d = _desc(ls)
    p = _prompt(ls)
    L = ls.lib()
    assert L.ls_replay_fwd(ctypes.byref(d), ctypes.byref(p), None, None, None, 0, None, None,
                           None, 0, None) == 0
    assert L.ls_replay_bwd_preprocess(ctypes.byref(d), None, None, 0, None, None) == 0
    assert L.ls_replay_group(ctypes.byref(d), ctypes.byref(p), 0, None, None, 0, None) == 0


def test_page_write_range_check(ls):
    d = _desc(ls)
    L = ls.lib()
    fake = 1 << 24
    # 4 pages of 256 hold 1024 tokens: writing 1000 tokens from position 100 overflows
    assert L.ls_kv_page_write(ctypes.byref(d), fake, fake, 8, fake, 4, 100, 1000, fake, fake,
                              None, 0, None) == 1


def test_product_path_does_not_import_the_oracle():
    pkg = ROOT / "long_context_grpo_replay_gb300"
    for f in pkg.rglob("*.py"):
        for line in f.read_text().splitlines():
            assert not re.match(r"\s*(import|from)\s+oracle\b", line), (f, line)
    for f in list(pkg.rglob("*.cu")) + list(pkg.rglob("*.h")) + list(pkg.rglob("*.cuh")):
        for line in f.read_text().splitlines():
            assert not (line.strip().startswith("#include") and "oracle" in line), (f, line)


def test_prefill_workspace_and_argument_checks(ls):
    """ls_prompt_prefill: host-side sizing and validation (no launch)."""
    d = _desc(ls)
    sizes = [ls.ls_prompt_prefill_workspace_size(d, n) for n in (1, 1000, 32768, 262144)]
    assert sizes == sorted(sizes)
    # one float32 partial of O and of LSE for n tokens after the 256-byte header
    n = 32768
    assert sizes[2] >= 256 + n * 24 * 256 * 4 + n * 24 * 4
    L = ls.lib()
    assert L.ls_prompt_prefill(ctypes.byref(d), None, None, None, 0, None, None, None, None, 0, None,
                               0, None, 0, None) == 0  # n_tok == 0: no-op
    st = L.ls_prompt_prefill(ctypes.byref(d), None, None, None, 16, None, None, None, None, 1, None,
                             1, None, 0, None)
    assert st == 1 and "workspace" in ls.ls_last_error()  # NULL workspace, before any launch
    out = ctypes.c_size_t(0)
    assert L.ls_prompt_prefill_workspace_size(ctypes.byref(d), -1, ctypes.byref(out)) == 1


def test_gdn_workspace_and_argument_checks(ls):
    """Gated-DeltaNet entry points: sizing and validation before any launch."""
    L = ls.lib()
    d = ls.GdnDesc(8, 32, 128, 128)
    assert d.precision == ls.LS_GDN_EXACT  # a zeroed desc selects the exact float32 path
    tc = ls.GdnDesc(8, 32, 128, 128, ls.LS_GDN_TENSOR_CORE)
    # the 256-byte status header, then the precision's own scratch: per (member,
    # head) the recurrent backward keeps one 128x128 float32 state per 8-token
    # checkpoint plus a segment of 8 states; the chunk-parallel one keeps, per
    # 128-token chunk, five 128x128 float32 blocks, fifteen 32 KB bf16 tiles
    # and 16 floats
    rec = [256 + 8 * 32 * (n + 8) * 128 * 128 * 4 for n in (1, 8, 9, 512)]
    cp = [256 + 8 * 32 * -(-R // 128) * (5 * 128 * 128 * 4 + 15 * 32768 + 64) for R in (1, 64, 65, 4096)]
    assert [ls.ls_gdn_workspace_size(d, r) for r in (1, 64, 65, 4096)] == rec
    assert [ls.ls_gdn_workspace_size(tc, r) for r in (1, 64, 65, 4096)] == cp
    out = ctypes.c_size_t(0)
    bad = ls.GdnDesc(8, 32, 64, 128)
    assert L.ls_gdn_workspace_size(ctypes.byref(bad), 10, ctypes.byref(out)) != 0
    assert "128" in ls.ls_last_error()
    badp = ls.GdnDesc(8, 32, 128, 128, 7)
    assert L.ls_gdn_workspace_size(ctypes.byref(badp), 10, ctypes.byref(out)) == 1
    assert "precision" in ls.ls_last_error()
    badf = ls.GdnDesc(8, 32, 128, 128, ls.LS_GDN_TENSOR_CORE, 2)
    assert L.ls_gdn_workspace_size(ctypes.byref(badf), 10, ctypes.byref(out)) == 1
    assert "flags" in ls.ls_last_error()
    assert L.ls_gdn_workspace_size(ctypes.byref(d), -1, ctypes.byref(out)) == 1
    args = [None] * 6
    assert L.ls_gdn_replay_fwd(ctypes.byref(d), *args, 0, None, None, None, 0, None) == 0  # no-op
    assert L.ls_gdn_replay_fwd(ctypes.byref(d), *args, 8, None, None, None, 0, None) == 1  # NULL buffers
    # the tensor-core forward needs the workspace, refused before any launch
    fw = [ctypes.c_void_p(256)] * 6
    st = L.ls_gdn_replay_fwd(ctypes.byref(tc), *fw, 8, ctypes.c_void_p(256), None, None, 0, None)
    assert st == 1 and "workspace" in ls.ls_last_error()
    st = L.ls_gdn_replay_fwd(ctypes.byref(tc), *fw, 8, ctypes.c_void_p(256), None, ctypes.c_void_p(256),
                             100, None)
    assert st == 3 and "workspace" in ls.ls_last_error()  # LS_ERR_WORKSPACE_TOO_SMALL
    bw = [ctypes.c_void_p(256)] * 7
    st = L.ls_gdn_replay_bwd(ctypes.byref(d), *bw, 8, *([ctypes.c_void_p(256)] * 5), None, 0, None)
    assert st == 1 and "workspace" in ls.ls_last_error()
    st = L.ls_gdn_replay_bwd(ctypes.byref(d), *bw, 8, *([ctypes.c_void_p(256)] * 5),
                             ctypes.c_void_p(256), 100, None)
    assert st != 0 and "workspace" in ls.ls_last_error()


def test_noalloc_forward_validates_before_touching_the_device(ls):
    """ls_replay_fwd_noalloc refuses a bad call before it looks up or clears
    its fixed scratch: these run without a GPU."""
    L = ls.lib()
    d = _desc(ls)
    prompt = _prompt(ls)
    A = ctypes.c_void_p(1 << 24)  # aligned, never dereferenced
    assert L.ls_replay_fwd_noalloc(None, ctypes.byref(prompt), A, A, A, 8, A, A, None) == 1
    assert L.ls_replay_fwd_noalloc(ctypes.byref(d), ctypes.byref(prompt), ctypes.c_void_p((1 << 24) + 2),
                                   A, A, 8, A, A, None) == 1
    assert "aligned" in ls.ls_last_error()
    assert L.ls_replay_fwd_noalloc(ctypes.byref(d), ctypes.byref(prompt), A, A, A, 0, A, A, None) == 0
    big = ls.PromptKV(1 << 24, 1 << 24, 8192, 1 << 24, 8192, 2097152)
    assert L.ls_replay_fwd_noalloc(ctypes.byref(d), ctypes.byref(big), A, A, A, 8192, A, A, None) == 3
    assert "64 MiB" in ls.ls_last_error()


def test_stage_pages_validates_before_any_launch(ls):
    """ls_stage_pages refuses NULL buffers, bad counts and memory the GPU
    cannot read (pageable host memory) with a status, launching nothing."""
    import numpy as np

    L = ls.lib()
    d = _desc(ls)
    A = ctypes.c_void_p(1 << 24)
    assert L.ls_stage_pages(ctypes.byref(d), A, A, 8, A, 0, 0, A, A, None, 0, None) == 0  # no-op
    assert L.ls_stage_pages(ctypes.byref(d), None, A, 8, A, 0, 4, A, A, None, 0, None) == 1
    assert L.ls_stage_pages(ctypes.byref(d), A, A, 8, A, 0, 70000, A, A, None, 0, None) == 1
    assert L.ls_stage_pages(ctypes.byref(d), A, A, 8, A, -1, 4, A, A, None, 0, None) == 1
    buf = np.zeros(1 << 16, dtype=np.uint8)  # pageable host memory
    p = ctypes.c_void_p((buf.ctypes.data + 15) // 16 * 16)
    assert L.ls_stage_pages(ctypes.byref(d), p, p, 8, A, 0, 4, A, A, None, 0, None) == 1
    assert "pinned" in ls.ls_last_error()
