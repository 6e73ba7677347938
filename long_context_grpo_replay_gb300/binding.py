"""Thin ctypes binding of libls, one Python function per C entry point, with
the same names.  Only argument marshalling happens here (torch tensors to
device pointers, structs, the current CUDA stream); every step of the replay
path runs in the library's kernels.  A missing library is an error: there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os
from pathlib import Path

__all__ = [
    "LsError", "lib", "library_path", "AttnDesc", "PromptKV", "Member",
    "LS_DTYPE_F32", "LS_DTYPE_BF16",
    "ls_kv_page_write", "ls_replay_workspace_size", "ls_replay_fwd", "ls_lse_merge",
    "ls_replay_bwd_preprocess", "ls_replay_bwd", "ls_replay_group",
    "ls_read_device_status", "ls_clear_device_status", "ls_status_string", "ls_last_error",
    "ls_trace_enable", "ls_trace_reset", "ls_trace_read", "ls_num_kernel_ids",
    "ls_kernel_name", "ls_launch_count", "ls_uses_tensor_cores", "kernel_trace",
    "desc_for", "prompt_from", "EXPORTED_SYMBOLS", "ls_replay_fwd_noalloc",
    "ls_replay_fwd_noalloc_scratch_bytes", "ls_prompt_prefill", "ls_prompt_prefill_workspace_size",
    "ls_replay_fwd_part", "ls_replay_bwd_part", "ls_sum_parts",
    "GdnDesc", "LS_GDN_EXACT", "LS_GDN_TENSOR_CORE", "LS_GDN_BWD_REUSES_FORWARD", "ls_gdn_workspace_size", "ls_gdn_replay_fwd",
    "ls_gdn_replay_bwd", "ls_stage_pages",
]

LS_DTYPE_F32 = 0
LS_DTYPE_BF16 = 1

EXPORTED_SYMBOLS = [
    "ls_kv_page_write", "ls_replay_workspace_size", "ls_replay_fwd", "ls_lse_merge",
    "ls_replay_bwd_preprocess", "ls_replay_bwd", "ls_replay_group", "ls_read_device_status",
    "ls_clear_device_status", "ls_status_string", "ls_last_error", "ls_trace_enable",
    "ls_trace_reset", "ls_trace_read", "ls_num_kernel_ids", "ls_kernel_name",
    "ls_launch_count", "ls_uses_tensor_cores", "ls_replay_fwd_noalloc",
    "ls_replay_fwd_noalloc_scratch_bytes", "ls_prompt_prefill", "ls_prompt_prefill_workspace_size",
    "ls_replay_fwd_part", "ls_replay_bwd_part", "ls_sum_parts",
    "ls_gdn_workspace_size", "ls_gdn_replay_fwd", "ls_gdn_replay_bwd", "ls_stage_pages",
]


class LsError(RuntimeError):
    def __init__(self, status: int, name: str, detail: str):
        super().__init__(f"{name}: {detail}")
        self.status = status
        self.name = name


class AttnDesc(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float)]


class PromptKV(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("pool_pages", ctypes.c_int64), ("page_table", ctypes.c_void_p),
                ("num_pages", ctypes.c_int64), ("prompt_len", ctypes.c_int64)]


class Member(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("d_o", ctypes.c_void_p), ("resp_len", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("delta", ctypes.c_void_p), ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p),
                ("dv", ctypes.c_void_p)]


LS_GDN_EXACT = 0
LS_GDN_TENSOR_CORE = 1
LS_GDN_BWD_REUSES_FORWARD = 1  # ls_gdn_desc.flags


class GdnDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("precision", ctypes.c_int32), ("flags", ctypes.c_int32)]


def library_path() -> Path:
    return Path(os.environ.get("LS_LIBRARY",
                               Path(__file__).resolve().parent / "_lib" / "libls.so"))


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libls; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not path.exists():
        raise RuntimeError(
            f"libls not found at {path}; build it first (python -c 'import __graft_entry__ as g; "
            "g.build()' or python long_context_grpo_replay_gb300/build.py)")
    L = ctypes.CDLL(str(path))
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "ls_kv_page_write": [ctypes.POINTER(AttnDesc), P, P, I64, P, I64, I64, I64, P, P, P, SZ, P],
        "ls_replay_workspace_size": [ctypes.POINTER(AttnDesc), ctypes.POINTER(PromptKV), I32,
                                     ctypes.POINTER(SZ)],
        "ls_replay_fwd": [ctypes.POINTER(AttnDesc), ctypes.POINTER(PromptKV), P, P, P, I32, P, P,
                          P, SZ, P],
        "ls_lse_merge": [I32, I64, I32, P, P, I32, P, P, P],
        "ls_replay_bwd_preprocess": [ctypes.POINTER(AttnDesc), P, P, I32, P, P],
        "ls_replay_bwd": [ctypes.POINTER(AttnDesc), ctypes.POINTER(PromptKV), P, P, P, P, P, P,
                          I32, P, P, P, P, SZ, P],
        "ls_replay_group": [ctypes.POINTER(AttnDesc), ctypes.POINTER(PromptKV), I32,
                            ctypes.POINTER(Member), P, SZ, P],
        "ls_prompt_prefill": [ctypes.POINTER(AttnDesc), P, P, P, I32, P, P, P, P, I64, P, I64, P,
                              SZ, P],
        "ls_prompt_prefill_workspace_size": [ctypes.POINTER(AttnDesc), I32, ctypes.POINTER(SZ)],
        "ls_sum_parts": [I32, I64, P, I32, P, P],
        "ls_replay_fwd_part": [ctypes.POINTER(AttnDesc), ctypes.POINTER(PromptKV), P, P, P, I32, I32,
                               P, P, P, SZ, P],
        "ls_replay_bwd_part": [ctypes.POINTER(AttnDesc), ctypes.POINTER(PromptKV), P, P, P, P, P, P,
                               I32, I32, P, P, P, P, SZ, P],
        "ls_gdn_workspace_size": [ctypes.POINTER(GdnDesc), I32, ctypes.POINTER(SZ)],
        "ls_gdn_replay_fwd": [ctypes.POINTER(GdnDesc), P, P, P, P, P, P, I32, P, P, P, SZ, P],
        "ls_gdn_replay_bwd": [ctypes.POINTER(GdnDesc), P, P, P, P, P, P, P, I32, P, P, P, P, P, P,
                              SZ, P],
        "ls_stage_pages": [ctypes.POINTER(AttnDesc), P, P, I64, P, I64, I32, P, P, P, SZ, P],
        "ls_read_device_status": [P, SZ, P],
        "ls_clear_device_status": [P, SZ, P],
        "ls_trace_enable": [I32],
        "ls_trace_reset": [],
        "ls_trace_read": [I32, ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_double)],
        "ls_uses_tensor_cores": [ctypes.POINTER(AttnDesc)],
        "ls_replay_fwd_noalloc": [ctypes.POINTER(AttnDesc), ctypes.POINTER(PromptKV), P, P, P,
                                  I32, P, P, P],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int32
    for name, res, args in [("ls_status_string", ctypes.c_char_p, [I32]),
                            ("ls_last_error", ctypes.c_char_p, []),
                            ("ls_num_kernel_ids", I32, []),
                            ("ls_kernel_name", ctypes.c_char_p, [I32]),
                            ("ls_launch_count", I64, []),
                            ("ls_replay_fwd_noalloc_scratch_bytes", SZ, [])]:
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def _check(status: int):
    if status != 0:
        L = lib()
        raise LsError(status, L.ls_status_string(status).decode(), L.ls_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(dt) -> int:
    import torch
    if dt == torch.float32:
        return LS_DTYPE_F32
    if dt == torch.bfloat16:
        return LS_DTYPE_BF16
    raise ValueError(f"unsupported dtype {dt}")


def desc_for(hq, hkv, head_dim, page_size, dtype, softmax_scale=None) -> AttnDesc:
    """Build an AttnDesc; dtype may be a torch dtype or an LS_DTYPE_* code."""
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    scale = softmax_scale if softmax_scale is not None else head_dim ** -0.5
    return AttnDesc(code, hq, hkv, head_dim, page_size, scale)


def prompt_from(k_pool, v_pool, page_table, prompt_len) -> PromptKV:
    """PromptKV over device tensors (pools [pool_pages, Hkv, S_p, d], int32 table)."""
    if prompt_len == 0:
        return PromptKV(None, None, 0, None, 0, 0)
    return PromptKV(_ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(page_table),
                    page_table.shape[0], prompt_len)


# ------------------------------------------------------------------ entry points
def ls_kv_page_write(desc, k_pool, v_pool, page_table, start_pos, k, v, ws=None, stream=None):
    _want_dtype(desc, k_pool, v_pool, k, v)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().ls_kv_page_write(ctypes.byref(desc), _ptr(k_pool), _ptr(v_pool),
                                  k_pool.shape[0], _ptr(page_table), page_table.shape[0],
                                  start_pos, k.shape[0], _ptr(k), _ptr(v), _ptr(ws), ws_bytes,
                                  _stream(stream)))


def ls_replay_workspace_size(desc, prompt, max_resp_len) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().ls_replay_workspace_size(ctypes.byref(desc), ctypes.byref(prompt),
                                          max_resp_len, ctypes.byref(out)))
    return out.value


def _nbytes(t):
    return t.numel() * t.element_size()


def _want_f32(*ts):
    import torch
    for t in ts:
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"expected a float32 tensor, got {t.dtype}")


def _want_dtype(desc, *ts):
    for t in ts:
        if t is not None and _dtype_code(t.dtype) != desc.dtype:
            raise TypeError(f"tensor dtype {t.dtype} does not match the descriptor dtype")


def ls_replay_fwd(desc, prompt, q, k_resp, v_resp, o, lse, ws, stream=None):
    _want_f32(lse)
    _want_dtype(desc, q, k_resp, v_resp, o)
    _check(lib().ls_replay_fwd(ctypes.byref(desc), ctypes.byref(prompt), _ptr(q), _ptr(k_resp),
                               _ptr(v_resp), q.shape[0], _ptr(o), _ptr(lse), _ptr(ws),
                               _nbytes(ws), _stream(stream)))


def ls_prompt_prefill_workspace_size(desc, n_tok) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().ls_prompt_prefill_workspace_size(ctypes.byref(desc), n_tok, ctypes.byref(out)))
    return out.value


def ls_prompt_prefill(desc, q, k, v, o, lse, k_pool, v_pool, page_table, ws, stream=None):
    """Capture a prompt: write its K/V into the pool pages and compute its
    causal self-attention o, lse (see ls.h)."""
    _want_f32(lse)
    _want_dtype(desc, q, k, v, o, k_pool, v_pool)
    _check(lib().ls_prompt_prefill(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), q.shape[0],
                                   _ptr(o), _ptr(lse), _ptr(k_pool), _ptr(v_pool), k_pool.shape[0],
                                   _ptr(page_table), page_table.shape[0], _ptr(ws), _nbytes(ws),
                                   _stream(stream)))


def ls_replay_fwd_part(desc, prompt, q, k_resp, v_resp, with_response, o_part, lse_part, ws,
                       stream=None):
    """One rank's exact float32 partial of the replay forward (see ls.h)."""
    _want_f32(o_part, lse_part)
    _want_dtype(desc, q, k_resp, v_resp)
    _check(lib().ls_replay_fwd_part(ctypes.byref(desc), ctypes.byref(prompt), _ptr(q), _ptr(k_resp),
                                    _ptr(v_resp), q.shape[0], 1 if with_response else 0,
                                    _ptr(o_part), _ptr(lse_part), _ptr(ws), _nbytes(ws),
                                    _stream(stream)))


def ls_replay_bwd_part(desc, prompt, q, k_resp, v_resp, d_o, lse, delta, with_response, dq_part,
                       dk=None, dv=None, ws=None, stream=None):
    """One rank's float32 share of dQ (and the response dK/dV on the rank
    that holds the response keys; see ls.h)."""
    _want_f32(lse, delta, dq_part)
    _want_dtype(desc, q, k_resp, v_resp, d_o, dk, dv)
    _check(lib().ls_replay_bwd_part(ctypes.byref(desc), ctypes.byref(prompt), _ptr(q), _ptr(k_resp),
                                    _ptr(v_resp), _ptr(d_o), _ptr(lse), _ptr(delta), q.shape[0],
                                    1 if with_response else 0, _ptr(dq_part), _ptr(dk), _ptr(dv),
                                    _ptr(ws), _nbytes(ws), _stream(stream)))


def ls_sum_parts(parts, out, stream=None):
    """out = parts.sum(0) in float32 accumulation (parts float32 [n, ...])."""
    _want_f32(parts)
    n = parts.shape[0]
    _check(lib().ls_sum_parts(n, out.numel(), _ptr(parts), _dtype_code(out.dtype), _ptr(out),
                              _stream(stream)))


def _gdn_desc(s0, q, precision, flags=0):
    """q [B, R, H, dk] (a group) or [R, H, dk] (one member)."""
    return GdnDesc(q.shape[0] if q.dim() == 4 else 1, s0.shape[0], s0.shape[2], s0.shape[1],
                   precision, flags)


def _resp_len(q):
    return q.shape[1] if q.dim() == 4 else q.shape[0]


def ls_gdn_workspace_size(desc, resp_len) -> int:
    """desc: GdnDesc(batch, heads, dk, dv, precision)."""
    out = ctypes.c_size_t(0)
    _check(lib().ls_gdn_workspace_size(ctypes.byref(desc), resp_len, ctypes.byref(out)))
    return out.value


def ls_gdn_replay_fwd(s0, q, k, v, g, beta, o, s_final=None, ws=None, stream=None,
                      precision=LS_GDN_EXACT):
    """Gated-DeltaNet replay from the captured state s0 [H, dv, dk] of one
    member (q [R, H, dk]) or a group (q [B, R, H, dk]); see ls.h.  float32
    buffers; precision LS_GDN_EXACT (ws may be None) or LS_GDN_TENSOR_CORE
    (ws of ls_gdn_workspace_size bytes)."""
    _want_f32(s0, q, k, v, g, beta, o, s_final)
    _check(lib().ls_gdn_replay_fwd(ctypes.byref(_gdn_desc(s0, q, precision)), _ptr(s0), _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(g), _ptr(beta), _resp_len(q), _ptr(o), _ptr(s_final),
                                   _ptr(ws), 0 if ws is None else _nbytes(ws), _stream(stream)))


def ls_gdn_replay_bwd(s0, q, k, v, g, beta, d_o, dq, dk, dv, dg, dbeta, ws, stream=None,
                      precision=LS_GDN_EXACT, reuse_forward=False):
    """Gradients of the replay for q, k, v, g, beta (none for s0; see ls.h).
    reuse_forward: ws holds the scratch of ls_gdn_replay_fwd on these same
    inputs (LS_GDN_BWD_REUSES_FORWARD)."""
    _want_f32(s0, q, k, v, g, beta, d_o, dq, dk, dv, dg, dbeta)
    desc = _gdn_desc(s0, q, precision, LS_GDN_BWD_REUSES_FORWARD if reuse_forward else 0)
    _check(lib().ls_gdn_replay_bwd(ctypes.byref(desc), _ptr(s0), _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(g), _ptr(beta), _ptr(d_o), _resp_len(q), _ptr(dq), _ptr(dk),
                                   _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(ws), _nbytes(ws),
                                   _stream(stream)))


def ls_stage_pages(desc, k_src, v_src, page_table, first_page, n_pages, k_dst, v_dst, ws=None,
                   stream=None):
    """Logical pages first_page .. first_page+n_pages-1 (slots from the
    device page_table) of pinned-host or device pools into staging pools;
    see ls.h."""
    _want_dtype(desc, k_src, v_src, k_dst, v_dst)
    _check(lib().ls_stage_pages(ctypes.byref(desc), _ptr(k_src), _ptr(v_src), k_src.shape[0],
                                _ptr(page_table), first_page, n_pages, _ptr(k_dst), _ptr(v_dst),
                                _ptr(ws), 0 if ws is None else _nbytes(ws), _stream(stream)))


def ls_replay_fwd_noalloc(desc, prompt, q, k_resp, v_resp, o, lse, stream=None):
    """ls_replay_fwd without a workspace: for callers that cannot allocate
    device memory; uses the library's fixed device scratch (see ls.h)."""
    _want_f32(lse)
    _want_dtype(desc, q, k_resp, v_resp, o)
    _check(lib().ls_replay_fwd_noalloc(ctypes.byref(desc), ctypes.byref(prompt), _ptr(q),
                                       _ptr(k_resp), _ptr(v_resp), q.shape[0], _ptr(o), _ptr(lse),
                                       _stream(stream)))


def ls_replay_fwd_noalloc_scratch_bytes() -> int:
    return lib().ls_replay_fwd_noalloc_scratch_bytes()


def ls_lse_merge(o_parts, lse_parts, o, lse=None, stream=None):
    n_parts, n_rows, d = o_parts.shape
    _want_f32(o_parts, lse_parts, lse)
    _check(lib().ls_lse_merge(n_parts, n_rows, d, _ptr(o_parts), _ptr(lse_parts),
                              _dtype_code(o.dtype), _ptr(o), _ptr(lse), _stream(stream)))


def ls_replay_bwd_preprocess(desc, o, d_o, delta, stream=None):
    _want_f32(delta)
    _want_dtype(desc, o, d_o)
    _check(lib().ls_replay_bwd_preprocess(ctypes.byref(desc), _ptr(o), _ptr(d_o), o.shape[0],
                                          _ptr(delta), _stream(stream)))


def ls_replay_bwd(desc, prompt, q, k_resp, v_resp, d_o, lse, delta, dq, dk, dv, ws, stream=None):
    _want_f32(lse, delta)
    _want_dtype(desc, q, k_resp, v_resp, d_o, dq, dk, dv)
    _check(lib().ls_replay_bwd(ctypes.byref(desc), ctypes.byref(prompt), _ptr(q), _ptr(k_resp),
                               _ptr(v_resp), _ptr(d_o), _ptr(lse), _ptr(delta), q.shape[0],
                               _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), _nbytes(ws),
                               _stream(stream)))


def ls_replay_group(desc, prompt, members, ws, stream=None):
    """members: sequence of dicts with tensors q, k, v, d_o, o, lse, delta, dq, dk, dv."""
    arr = (Member * max(1, len(members)))()
    for i, m in enumerate(members):
        _want_f32(m["lse"], m["delta"])
        _want_dtype(desc, m["q"], m["k"], m["v"], m["d_o"], m["o"], m["dq"], m["dk"], m["dv"])
        arr[i] = Member(_ptr(m["q"]), _ptr(m["k"]), _ptr(m["v"]), _ptr(m["d_o"]),
                        m["q"].shape[0], 0, _ptr(m["o"]), _ptr(m["lse"]), _ptr(m["delta"]),
                        _ptr(m["dq"]), _ptr(m["dk"]), _ptr(m["dv"]))
    _check(lib().ls_replay_group(ctypes.byref(desc), ctypes.byref(prompt), len(members), arr,
                                 _ptr(ws), _nbytes(ws), _stream(stream)))


def ls_read_device_status(ws, stream=None):
    _check(lib().ls_read_device_status(_ptr(ws), _nbytes(ws), _stream(stream)))


def ls_clear_device_status(ws, stream=None):
    _check(lib().ls_clear_device_status(_ptr(ws), _nbytes(ws), _stream(stream)))


def ls_status_string(status: int) -> str:
    return lib().ls_status_string(status).decode()


def ls_last_error() -> str:
    return lib().ls_last_error().decode()


def ls_trace_enable(on: bool = True):
    _check(lib().ls_trace_enable(1 if on else 0))


def ls_trace_reset():
    _check(lib().ls_trace_reset())


def ls_trace_read(kernel_id: int):
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check(lib().ls_trace_read(kernel_id, ctypes.byref(n), ctypes.byref(ms)))
    return n.value, ms.value


def ls_num_kernel_ids() -> int:
    return lib().ls_num_kernel_ids()


def ls_kernel_name(kernel_id: int) -> str:
    return lib().ls_kernel_name(kernel_id).decode()


def ls_launch_count() -> int:
    return lib().ls_launch_count()


def ls_uses_tensor_cores(desc) -> bool:
    return lib().ls_uses_tensor_cores(ctypes.byref(desc)) != 0


def kernel_trace() -> dict:
    """{kernel name: (launches, total ms)} accumulated since the last reset."""
    out = {}
    for k in range(ls_num_kernel_ids()):
        n, ms = ls_trace_read(k)
        if n:
            out[ls_kernel_name(k)] = (n, ms)
    return out
