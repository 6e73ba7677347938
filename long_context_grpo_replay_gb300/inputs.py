"""Seeded synthetic inputs for response-replay attention.

This module only draws random numbers and lays them out; it holds none of the
operator's arithmetic.  Both the CUDA path's tests and the float64 oracle take
their inputs from here, and nothing else is shared between them.

The workloads mirror the shapes of the LongStraw pages' Qwen full-attention
layers (review "论文综述：LongStraw…", section 三: GQA, 24 query heads, 4 KV
heads, head dim 256) at the prompt lengths of its results table (2,097,152
positions; stress prefix 4,456,448 positions) and group sizes G = 2 and 8.
The pages train on synthetic responses (DeepRead summary, *Strengths &
Weaknesses*), so no dataset stands behind these shapes.

Distributions: Q, K, V ~ N(0, 1)/sqrt(d); dO ~ N(0, 1).  Optional per-KV-head
K scale ~ U(0.5, 2) applied to prompt and response K alike.  Pools hold
``pool_factor`` times the pages the prompt needs; the page table is a seeded
random choice of distinct slots, and unused slots may be poisoned with NaN so
that any stray page read shows up.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Workload", "WORKLOADS", "make_prompt", "make_prompt_source", "make_member",
           "torch_dtype"]


@dataclass(frozen=True)
class Workload:
    name: str
    hq: int
    hkv: int
    head_dim: int
    page_size: int
    prompt_len: int
    resp_lens: tuple
    dtype: str  # "f32" | "bf16"
    seed: int
    pool_factor: int = 1
    poison: bool = False
    k_head_scale: bool = False
    note: str = field(default="", compare=False)

    @property
    def num_pages(self) -> int:
        return -(-self.prompt_len // self.page_size)

    @property
    def pool_pages(self) -> int:
        return max(1, self.num_pages * self.pool_factor)

    @property
    def group(self) -> int:
        return len(self.resp_lens)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


def _stress_lens(seed: int, g: int, lo: int = 512, hi: int = 8192) -> tuple:
    gen = torch.Generator().manual_seed(seed * 7919 + 17)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (g,), generator=gen))


WORKLOADS = {
    # tiny fp32: Hq=4, Hkv=1, d=64, 1024-token prompt in 16-token pages
    "tiny_f32": Workload("tiny_f32", 4, 1, 64, 16, 1024, (64, 64), "f32", 0),
    # bf16 P=32K in 256-token pages, R=2048, G=2
    "bf16_p32k_r2048": Workload("bf16_p32k_r2048", 24, 4, 256, 256, 32768, (2048, 2048),
                                "bf16", 2),
    # bf16 P=256K, G=8 x R=4096, per-KV-head K scale ~ U(0.5, 2)
    "bf16_p256k_r4096_g8": Workload("bf16_p256k_r4096_g8", 24, 4, 256, 256, 262144,
                                    (4096,) * 8, "bf16", 3, k_head_scale=True),
    # bf16 P=2M (8192 pages of 256), G=8 x R=4096
    "bf16_p2m_r4096_g8": Workload("bf16_p2m_r4096_g8", 24, 4, 256, 256, 2097152,
                                  (4096,) * 8, "bf16", 4),
    # bf16 P=2M, G=8 x R=64: the short-response KV-streaming variant
    "bf16_p2m_r64_g8": Workload("bf16_p2m_r64_g8", 24, 4, 256, 256, 2097152,
                                (64,) * 8, "bf16", 4),
    # bf16 P=256K, G=8 x R=64: the short-response case at a size an ncu capture
    # of every counter pass can hold (prompt K/V still larger than L2)
    "bf16_p256k_r64_g8": Workload("bf16_p256k_r64_g8", 24, 4, 256, 256, 262144,
                                  (64,) * 8, "bf16", 4),
    # bf16 stress: P=4,456,448 scattered over a 2x pool (unused slots NaN), ragged R
    "bf16_p4m_ragged_g8": Workload("bf16_p4m_ragged_g8", 24, 4, 256, 256, 4456448,
                                   _stress_lens(5, 8), "bf16", 5, pool_factor=2, poison=True),
}


def torch_dtype(w: Workload) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[w.dtype]


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7_919) % (1 << 62))
    return g


def _k_scales(w: Workload, device) -> torch.Tensor:
    if not w.k_head_scale:
        return torch.ones(w.hkv, device=device)
    g = _gen("cpu", w.seed, 3)
    return (0.5 + 1.5 * torch.rand(w.hkv, generator=g)).to(device)


def _randn_chunked(shape, gen, device, dtype, mult, chunk_rows=256):
    """N(0,1) * mult, drawn in chunks along dim 0 so that a multi-GB bf16
    tensor never needs a full fp32 temporary."""
    out = torch.empty(shape, device=device, dtype=dtype)
    for a in range(0, shape[0], chunk_rows):
        b = min(shape[0], a + chunk_rows)
        t = torch.randn((b - a,) + tuple(shape[1:]), generator=gen, device=device,
                        dtype=torch.float32)
        out[a:b] = (t * mult).to(dtype)
    return out


def make_prompt(w: Workload, device="cpu") -> dict:
    """Pools [pool_pages, Hkv, page_size, d] already holding the prompt pages,
    plus the int32 page table [num_pages] and the prompt length."""
    dt = torch_dtype(w)
    g = _gen(device, w.seed, 1)
    gcpu = _gen("cpu", w.seed, 2)
    if w.pool_factor == 1:
        pt = torch.randperm(w.num_pages, generator=gcpu)
    else:
        pt = torch.randperm(w.pool_pages, generator=gcpu)[: w.num_pages]
    pt = pt.to(torch.int32)
    shape = (w.pool_pages, w.hkv, w.page_size, w.head_dim)
    mult = 1.0 / math.sqrt(w.head_dim)
    rows = max(1, (1 << 24) // (w.hkv * w.page_size * w.head_dim))
    k_pool = _randn_chunked(shape, g, device, dt, mult, rows)
    v_pool = _randn_chunked(shape, g, device, dt, mult, rows)
    if w.k_head_scale:
        ks = _k_scales(w, device).to(torch.float32)
        for a in range(0, shape[0], rows):
            b = min(shape[0], a + rows)
            k_pool[a:b] = (k_pool[a:b].float() * ks[None, :, None, None]).to(dt)
    if w.poison and w.pool_factor > 1:
        used = torch.zeros(w.pool_pages, dtype=torch.bool)
        used[pt.long()] = True
        unused = (~used).nonzero().flatten().to(device)
        if unused.numel():
            k_pool[unused] = float("nan")
            v_pool[unused] = float("nan")
    if w.num_pages * w.page_size > w.prompt_len:
        # the tail of the last page is not prompt: poison it too
        last = int(pt[-1])
        tail = w.prompt_len - (w.num_pages - 1) * w.page_size
        k_pool[last, :, tail:] = float("nan")
        v_pool[last, :, tail:] = float("nan")
    return {"k_pool": k_pool, "v_pool": v_pool, "page_table": pt.to(device),
            "prompt_len": w.prompt_len}


def make_prompt_source(w: Workload, device="cpu", n_tok=None) -> dict:
    """Token-major prompt K/V [n_tok, Hkv, d] (what a prefill produces before
    the page write) and the page table for a pool of ``pool_pages`` slots."""
    dt = torch_dtype(w)
    n_tok = w.prompt_len if n_tok is None else n_tok
    g = _gen(device, w.seed, 4)
    gcpu = _gen("cpu", w.seed, 2)
    if w.pool_factor == 1:
        pt = torch.randperm(w.num_pages, generator=gcpu)
    else:
        pt = torch.randperm(w.pool_pages, generator=gcpu)[: w.num_pages]
    mult = 1.0 / math.sqrt(w.head_dim)
    rows = max(1, (1 << 24) // (w.hkv * w.head_dim))
    k = _randn_chunked((n_tok, w.hkv, w.head_dim), g, device, dt, mult, rows)
    v = _randn_chunked((n_tok, w.hkv, w.head_dim), g, device, dt, mult, rows)
    if w.k_head_scale:
        ks = _k_scales(w, device).to(torch.float32)
        k = (k.float() * ks[None, :, None]).to(dt)
    return {"k": k, "v": v, "page_table": pt.to(torch.int32).to(device)}


def make_member(w: Workload, member: int, device="cpu", resp_len=None) -> dict:
    """Member inputs: q [R, Hq, d], k/v [R, Hkv, d], d_o [R, Hq, d]."""
    dt = torch_dtype(w)
    R = w.resp_lens[member] if resp_len is None else resp_len
    g = _gen(device, w.seed, 100 + member)
    mult = 1.0 / math.sqrt(w.head_dim)
    q = (torch.randn((R, w.hq, w.head_dim), generator=g, device=device) * mult).to(dt)
    k = torch.randn((R, w.hkv, w.head_dim), generator=g, device=device) * mult
    k = (k * _k_scales(w, device)[None, :, None]).to(dt)
    v = (torch.randn((R, w.hkv, w.head_dim), generator=g, device=device) * mult).to(dt)
    d_o = torch.randn((R, w.hq, w.head_dim), generator=g, device=device).to(dt)
    return {"q": q, "k": k, "v": v, "d_o": d_o}


def make_head_sample(w: Workload, n_tok: int, device="cpu") -> dict:
    """The inputs one KV head's group of query heads sees, drawn alone with the
    distributions of make_member (a bounded sample for timing the oracle on a
    long prompt): q [1, Gq, d] (the last row), k/v [n_tok, 1, d]."""
    dt = torch_dtype(w)
    g = _gen(device, w.seed, 900)
    mult = 1.0 / math.sqrt(w.head_dim)
    gq = w.hq // w.hkv
    q = (torch.randn((1, gq, w.head_dim), generator=g, device=device) * mult).to(dt)
    k = (torch.randn((n_tok, 1, w.head_dim), generator=g, device=device) * mult).to(dt)
    v = (torch.randn((n_tok, 1, w.head_dim), generator=g, device=device) * mult).to(dt)
    return {"q": q, "k": k, "v": v}


def make_gdn_group(batch: int, heads: int, resp_len: int, seed: int, dk: int = 128,
                   dv: int = 128, device="cpu") -> dict:
    """Seeded float32 inputs of one gated-DeltaNet group replay, drawn on
    `device` (a CUDA generator's stream differs from the CPU one).

    s0 [H, dv, dk]: the captured prompt state shared by the group, N(0, 0.1^2).
    q, k [B, R, H, dk]: unit-norm rows (the layer normalises q and k before
    the recurrence), q further scaled by dk^-1/2.  v, d_o [B, R, H, dv]:
    N(0, 1).  g [B, R, H]: log of a decay in [0.85, 1).  beta [B, R, H]:
    write strength in [0.05, 0.95)."""
    gen = _gen(device, seed, 11)
    B, R, H = batch, resp_len, heads
    f32 = dict(generator=gen, device=device, dtype=torch.float32)

    def unit(x):
        return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-6)

    return {
        "s0": 0.1 * torch.randn((H, dv, dk), **f32),
        "q": unit(torch.randn((B, R, H, dk), **f32)) * dk ** -0.5,
        "k": unit(torch.randn((B, R, H, dk), **f32)),
        "v": torch.randn((B, R, H, dv), **f32),
        "g": torch.log(0.85 + 0.15 * torch.rand((B, R, H), **f32)),
        "beta": 0.05 + 0.9 * torch.rand((B, R, H), **f32),
        "d_o": torch.randn((B, R, H, dv), **f32),
    }
