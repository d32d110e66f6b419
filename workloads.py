"""Seeded synthetic inputs for split-KV paged decode attention.

This module is shared by the tests, the benchmark and the oracle's callers.  It
only draws random numbers and lays them out as a paged KV cache; it holds none
of the attention arithmetic.  FP8 inputs are produced by quantising the drawn
values with a per-tensor scale (input preparation: the method itself only ever
*reads* e4m3 codes and multiplies by ``kv_scale``).

Workloads follow the shapes discussed on the pages:

* "vLLM 0.30.0 FA4 SplitKV Bug: H100 Decode Can Be 48% Slower", sections
  "What SplitKV is trying to do" and "Gemma 4 exposes the failure clearly":
  one query token, few KV heads (2), contexts of ~260 and ~5.9k tokens.
* "Xqa decode kernels" (vLLM pull request #43232), section "Purpose" and the
  serving benchmark: BF16 queries over an FP8 KV cache in the HND layout,
  random 32,000-token prompts.
* "Shipped: 484.5 tok/s on one GB300 ...", table "What shipped": MLA decode of
  one request with 6 query tokens per step split 4 (or 8) ways.

Layout (HND pages): ``k_pages[num_pages][Hkv][P][Dk]``, ``v_pages`` likewise
with ``Dv``; ``block_table[B][max_pages]`` int32 physical page ids;
``q[B][T][Hq][Dk]`` bf16; ``seq_lens[B]`` int32 = visible keys including the
current T tokens.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one decode-attention call."""

    name: str
    batch: int
    q_tokens: int
    num_q_heads: int
    num_kv_heads: int
    qk_dim: int
    v_dim: int
    page_size: int
    kv_dtype: str  # "bf16" or "fp8_e4m3"
    lens: str  # "fixed:<L>", "uniform:<lo>:<hi>", "loguniform:<lo>:<hi>"
    std: float = 1.0
    v_shares_k: bool = False
    splits: tuple = (0,)  # num_splits values exercised; 0 = planner-chosen
    pool_slack: float = 1.0  # extra free pages in the pool, as a fraction of used
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.qk_dim)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The workloads, each with its own seed.
WORKLOADS = {
    "tiny_gqa_ctx260": Workload(
        "tiny_gqa_ctx260", 1, 1, 16, 2, 128, 128, 16, "bf16", "fixed:260",
        splits=(1, 4), pool_slack=2.76, seed=1001),
    "gqa_ctx5900": Workload(
        "gqa_ctx5900", 1, 1, 16, 2, 128, 128, 16, "bf16", "fixed:5900",
        splits=(1, 2, 4, 8, 16, 32, 0), pool_slack=0.39, seed=1002),
    "fp8_batch8_ctx32k": Workload(
        "fp8_batch8_ctx32k", 8, 1, 32, 4, 128, 128, 16, "fp8_e4m3",
        "uniform:28672:32768", splits=(0,), pool_slack=0.05, seed=1003),
    "mla_t6_ctx64k": Workload(
        "mla_t6_ctx64k", 1, 6, 128, 1, 576, 512, 64, "bf16", "fixed:65536",
        std=0.5, v_shares_k=True, splits=(1, 4, 8, 0), pool_slack=0.0, seed=1004),
    # the same MLA decode over a cache whose V rows are a separate 512-wide tensor
    "mla_sepv_t6_ctx64k": Workload(
        "mla_sepv_t6_ctx64k", 1, 6, 128, 1, 576, 512, 64, "bf16", "fixed:65536",
        std=0.5, v_shares_k=False, splits=(1, 4, 0), pool_slack=0.0, seed=1006),
    # the same MLA decode over an e4m3 latent cache with a per-tensor scale
    "mla_fp8_t6_ctx64k": Workload(
        "mla_fp8_t6_ctx64k", 1, 6, 128, 1, 576, 512, 64, "fp8_e4m3", "fixed:65536",
        std=0.5, v_shares_k=True, splits=(1, 4, 8, 0), pool_slack=0.0, seed=1007),
    # speculative decode: four query tokens of each G = 8 group (32 rows per
    # KV head, causal among themselves) over the 5.9k context
    "spec_t4_gqa_ctx5900": Workload(
        "spec_t4_gqa_ctx5900", 1, 4, 16, 2, 128, 128, 16, "bf16", "fixed:5900",
        splits=(1, 8, 0), pool_slack=0.39, seed=1008),
    "mixed_batch32_bf16": Workload(
        "mixed_batch32_bf16", 32, 1, 32, 8, 128, 128, 16, "bf16",
        "loguniform:256:131072", splits=(0,), pool_slack=0.02, seed=1005),
    "mixed_batch32_fp8": Workload(
        "mixed_batch32_fp8", 32, 1, 32, 8, 128, 128, 16, "fp8_e4m3",
        "loguniform:256:131072", splits=(0,), pool_slack=0.02, seed=1005),
}


def draw_seq_lens(w: Workload, rng: np.random.Generator) -> np.ndarray:
    kind, *args = w.lens.split(":")
    if kind == "fixed":
        lens = np.full(w.batch, int(args[0]), dtype=np.int64)
    elif kind == "uniform":
        lo, hi = int(args[0]), int(args[1])
        lens = rng.integers(lo, hi + 1, size=w.batch)
    elif kind == "loguniform":
        lo, hi = int(args[0]), int(args[1])
        lens = np.rint(np.exp(rng.uniform(math.log(lo), math.log(hi), size=w.batch)))
        lens = np.clip(lens, lo, hi).astype(np.int64)
    elif kind == "list":
        lens = np.array([int(a) for a in args], dtype=np.int64)
        assert lens.size == w.batch
    else:
        raise ValueError(w.lens)
    return lens.astype(np.int32)


@dataclasses.dataclass
class Inputs:
    """One seeded decode-attention call.  Tensors live on ``device``."""

    w: Workload
    q: torch.Tensor  # bf16 [B][T][Hq][Dk]
    k_pages: torch.Tensor  # bf16 or uint8 [N][Hkv][P][Dk] (HND) or [N][P][Hkv][Dk] (NHD)
    v_pages: Optional[torch.Tensor]  # None when V shares K's rows
    block_table: torch.Tensor  # int32 [B][max_pages]
    seq_lens: torch.Tensor  # int32 [B]
    seq_lens_host: np.ndarray  # int32 [B]
    kv_scale: float
    scale: float
    poison_page: int  # page filled with NaN (bf16) / 0x7F codes (e4m3)
    layout: str = "HND"  # order of the page pools' dimensions

    @property
    def num_pages(self) -> int:
        return self.k_pages.shape[0]

    @property
    def max_pages(self) -> int:
        return self.block_table.shape[1]


def _quantize_e4m3(x: torch.Tensor, kv_scale: float) -> torch.Tensor:
    """Per-tensor e4m3 quantisation of synthetic values (clamp, then RNE cast)."""
    y = torch.clamp(x / kv_scale, -E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None,
                poison: bool = True, lens: Optional[np.ndarray] = None,
                max_pages: Optional[int] = None, layout: str = "HND") -> Inputs:
    """Builds the inputs of workload ``w`` from ``seed`` (default ``w.seed``).

    * Lengths, page permutation and block tables come from numpy's PCG64.
    * Values come from ``torch.Generator`` on ``device`` (N(0, std^2), fp32,
      then cast), so large pools are drawn where they will be used.
    * With ``poison``, one extra physical page is filled with NaN (BF16) or
      e4m3 code 0x7F, every unused block-table entry points at it, and the
      slots past ``seq_len`` in each sequence's last page are poisoned too:
      a kernel that reads outside the visible keys shows it in its output.
    * ``layout="NHD"`` stores the same values with the slot and head axes of
      each page swapped (``[N][P][Hkv][D]``); everything else is unchanged.
    """
    if layout not in ("HND", "NHD"):
        raise ValueError(layout)
    seed = w.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    seq_lens = draw_seq_lens(w, rng) if lens is None else np.asarray(lens, np.int32)
    P = w.page_size
    n_pages = (seq_lens.astype(np.int64) + P - 1) // P
    used = int(n_pages.sum())
    pool = used + int(math.ceil(used * w.pool_slack)) + (1 if poison else 0)
    pool = max(pool, 1)
    if max_pages is None:
        max_pages = max(1, int(n_pages.max()) if n_pages.size else 1)
    perm = rng.permutation(pool - (1 if poison else 0))
    poison_page = pool - 1 if poison else -1
    table = np.full((w.batch, max_pages), poison_page if poison else 0, dtype=np.int32)
    off = 0
    for b in range(w.batch):
        n = int(n_pages[b])
        table[b, :n] = perm[off:off + n]
        off += n

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dev = torch.device(device)
    q = torch.randn((w.batch, w.q_tokens, w.num_q_heads, w.qk_dim), generator=g,
                    device=dev, dtype=torch.float32) * w.std
    kshape = (pool, w.num_kv_heads, P, w.qk_dim)
    vshape = (pool, w.num_kv_heads, P, w.v_dim)
    k = torch.randn(kshape, generator=g, device=dev, dtype=torch.float32) * w.std
    v = None
    if not w.v_shares_k:
        v = torch.randn(vshape, generator=g, device=dev, dtype=torch.float32) * w.std

    kv_scale = 1.0
    if w.kv_dtype == "fp8_e4m3":
        amax = float(k.abs().max())
        if v is not None:
            amax = max(amax, float(v.abs().max()))
        kv_scale = amax / E4M3_MAX
        k_t = _quantize_e4m3(k, kv_scale)
        v_t = _quantize_e4m3(v, kv_scale) if v is not None else None
        poison_val = 0x7F
    elif w.kv_dtype == "bf16":
        k_t = k.to(torch.bfloat16)
        v_t = v.to(torch.bfloat16) if v is not None else None
        poison_val = float("nan")
    else:
        raise ValueError(w.kv_dtype)
    del k, v

    if poison:
        k_t[poison_page].fill_(poison_val)
        if v_t is not None:
            v_t[poison_page].fill_(poison_val)
        for b in range(w.batch):
            L, n = int(seq_lens[b]), int(n_pages[b])
            if n and L % P:
                last = int(table[b, n - 1])
                k_t[last, :, L % P:, :].fill_(poison_val)
                if v_t is not None:
                    v_t[last, :, L % P:, :].fill_(poison_val)

    if layout == "NHD":
        k_t = k_t.transpose(1, 2).contiguous()
        v_t = v_t.transpose(1, 2).contiguous() if v_t is not None else None

    return Inputs(
        w=w,
        q=q.to(torch.bfloat16),
        k_pages=k_t,
        v_pages=v_t,
        block_table=torch.from_numpy(table).to(dev),
        seq_lens=torch.from_numpy(seq_lens.copy()).to(dev),
        seq_lens_host=seq_lens,
        kv_scale=kv_scale,
        scale=w.scale,
        poison_page=poison_page,
        layout=layout,
    )


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw storage of a bf16 (-> uint16) or e4m3 code (-> uint8) tensor, on the host."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.uint8:
        return t.numpy()
    raise TypeError(t.dtype)
