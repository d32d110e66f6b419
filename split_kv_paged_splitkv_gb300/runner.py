"""Convenience wrapper: plan, torch-allocated workspace and outputs, one decode.

Marshalling only -- torch allocates device memory and provides the stream;
the computation is ``splitkv_decode`` in libsplitkv.
"""
from __future__ import annotations

import torch

from . import (SPLITKV_BF16, SPLITKV_COMBINE_SEPARATE, SPLITKV_FP8_E4M3, SPLITKV_LAYOUT_HND,
               SPLITKV_LAYOUT_NHD, make_desc, splitkv_combine_workspace, splitkv_decode,
               splitkv_decode_partials,
               splitkv_decode_kv_scales, splitkv_plan, splitkv_plan_fixed,
               splitkv_plan_upload, splitkv_read_stats)


class DecodeSession:
    """Holds a plan and its uploaded workspace for one set of KV-cache tensors.

    ``q`` bf16 [B][T][Hq][Dk]; ``k_pages`` bf16 or uint8 (e4m3 codes)
    [N][Hkv][P][Dk] (``kv_layout`` HND) or [N][P][Hkv][Dk] (NHD); ``v_pages``
    likewise or None with ``v_shares_k``;
    ``block_table`` int32 [B][max_pages]; ``seq_lens`` int32 [B] on the device
    and ``seq_lens_host`` the same values on the host.
    """

    def __init__(self, q, k_pages, v_pages, block_table, seq_lens, seq_lens_host, *, scale,
                 kv_scale=1.0, num_splits=0, num_sms=0, v_dim=None, v_shares_k=False,
                 combine_mode=SPLITKV_COMBINE_SEPARATE, stream=None, k_scale=None, v_scale=None,
                 fixed=False, kv_layout=SPLITKV_LAYOUT_HND):
        B, T, Hq, Dk = q.shape
        if kv_layout == SPLITKV_LAYOUT_NHD:
            N, P, Hkv, _ = k_pages.shape
        else:
            N, Hkv, P, _ = k_pages.shape
        if v_dim is None:
            v_dim = Dk if v_pages is None else v_pages.shape[3]
        fp8 = k_pages.dtype == torch.uint8
        self.desc = make_desc(B, T, Hq, Hkv, Dk, v_dim, P, block_table.shape[1], N,
                              SPLITKV_FP8_E4M3 if fp8 else SPLITKV_BF16, int(v_shares_k),
                              combine_mode, kv_layout)
        # fixed: a capacity plan (num_splits items per sequence and head group)
        # whose kernels derive every item from the current device seq_lens,
        # so one captured CUDA graph serves any lengths
        self.fixed = fixed
        self.plan = (splitkv_plan_fixed(self.desc, num_splits) if fixed else
                     splitkv_plan(self.desc, seq_lens_host, num_splits, num_sms))
        self.num_splits = num_splits
        dev = q.device
        self.workspace = torch.empty(max(self.plan.workspace_size, 256), dtype=torch.uint8, device=dev)
        self.stream = stream
        splitkv_plan_upload(self.plan, self.workspace, self.workspace.numel(), stream)
        self.tensors = (q, k_pages, v_pages, block_table, seq_lens)
        self.scale, self.kv_scale = float(scale), float(kv_scale)
        self.k_scale, self.v_scale = k_scale, v_scale  # per-KV-head e4m3 scales, or None
        self.out = torch.empty((B, T, Hq, v_dim), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, T, Hq), dtype=torch.float32, device=dev)

    def run(self, out=None, lse=None, tensors=None):
        q, k, v, table, lens = tensors if tensors is not None else self.tensors
        o = self.out if out is None else out
        l = self.lse if lse is None else lse
        if self.k_scale is not None:
            splitkv_decode_kv_scales(self.plan, self.workspace, q, k, v, table, lens,
                                     self.num_splits, self.scale, self.k_scale, self.v_scale, o, l,
                                     self.stream)
        else:
            splitkv_decode(self.plan, self.workspace, q, k, v, table, lens, self.num_splits,
                           self.scale, self.kv_scale, o, l, self.stream)
        return self.out if out is None else out, self.lse if lse is None else lse

    def run_partials(self, out=None, lse=None, tensors=None):
        """The split-KV kernel alone (splitkv_decode_partials): rows of sequences
        with one split are final, the others wait for merge()."""
        q, k, v, table, lens = tensors if tensors is not None else self.tensors
        o = self.out if out is None else out
        l = self.lse if lse is None else lse
        splitkv_decode_partials(self.plan, self.workspace, q, k, v, table, lens, self.num_splits,
                                self.scale, self.kv_scale, o, l, self.stream)
        return o, l

    def merge(self, out=None, lse=None):
        """Merges the partials run_partials left in the workspace (splitkv_combine_workspace)."""
        o = self.out if out is None else out
        l = self.lse if lse is None else lse
        splitkv_combine_workspace(self.plan, self.workspace, o, l, self.stream)
        return o, l

    def stats(self):
        """(per-CTA log [n][4], device status word) -- synchronises the stream."""
        return splitkv_read_stats(self.plan, self.workspace, self.stream)
