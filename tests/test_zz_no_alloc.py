"""splitkv_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (code inside another framework's memory budget,
plugins that may not allocate after start-up, real-time loops that must not
stall on an allocation).  It keeps its workspace in a fixed 16 MiB device array
inside the library instead of a caller buffer.

The GPU test calls it through the C-ABI on four workloads in a row (bf16 GQA,
e4m3 GQA in NHD pages, MLA with a separate V tensor; each call must not see
the previous call's work list or tickets) and compares each result with
splitkv_decode's on a caller workspace, within the bars the other parity
tests use.  The file sorts last so that a run
stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads
import split_kv_paged_splitkv_gb300 as skv
from _support import LSE_TOL, OUT_TOL, need_gpu, session


def test_noalloc_rejects_plans_beyond_its_scratch():
    """A plan needing more than 16 MiB of workspace is refused before any GPU work."""
    B, Hkv, P = 64, 8, 16
    desc = skv.make_desc(B, 1, Hkv * 8, Hkv, 128, 128, P, 512, B * 512 + 1)
    plan = skv.splitkv_plan(desc, np.full(B, 512 * P, np.int32), 64, 148)
    assert plan.workspace_size > 16 << 20
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_decode_noalloc(plan, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 64,
                                   0.1, 1.0, 1 << 20, 1 << 20, 0)
    assert e.value.status == skv.SPLITKV_EWORKSPACE
    assert "16 MiB" in skv.splitkv_last_error()


@pytest.mark.gpu
def test_noalloc_matches_workspace_decode_on_two_calls():
    need_gpu()
    cases = [
        (workloads.WORKLOADS["gqa_ctx5900"], 0, "HND"),
        (workloads.WORKLOADS["tiny_gqa_ctx260"], 4, "HND"),
        # an e4m3 cache in NHD pages, and an MLA decode with a separate V tensor
        (workloads.Workload("noalloc_e4m3", 3, 1, 32, 4, 128, 128, 16, "fp8_e4m3",
                            "list:500:1200:33", pool_slack=0.5, seed=61), 0, "NHD"),
        (workloads.Workload("noalloc_mla", 1, 2, 128, 1, 576, 512, 64, "bf16", "list:700",
                            std=0.5, v_shares_k=False, pool_slack=0.5, seed=62), 3, "HND"),
    ]
    for w, splits, layout in cases:
        x = workloads.make_inputs(w, device="cuda", layout=layout)
        ref = session(x, splits)
        ref_out, ref_lse = ref.run()
        ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        skv.splitkv_decode_noalloc(ref.plan, x.q, x.k_pages, x.v_pages, x.block_table,
                                   x.seq_lens, splits, x.scale, x.kv_scale, out, lse)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert (out.float() - ref_out.float()).abs().max().item() <= OUT_TOL
        fin = torch.isfinite(ref_lse)
        assert torch.equal(torch.isfinite(lse), fin)
        assert (lse[fin] - ref_lse[fin]).abs().max().item() <= LSE_TOL
