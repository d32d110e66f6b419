"""splitkv_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (code inside another framework's memory budget,
plugins that may not allocate after start-up, real-time loops that must not
stall on an allocation).  It keeps its workspace in a fixed 16 MiB device array
inside the library instead of a caller buffer.

The GPU test calls it through the C-ABI, twice in a row, on each of five
workloads (bf16 GQA with the planner's splits, a short bf16 GQA at 4 splits,
an e4m3 cache in NHD pages, an MLA decode with a separate V tensor, an MLA
decode over an e4m3 latent cache in 16-key pages): every
call must reproduce splitkv_decode on a caller workspace bit for bit (same
kernels, same plan, so a stale work list or ticket from the previous call
would show), leave the device status word clear, and log the same per-CTA
page ranges; one workload is also checked against the fp64 oracle.  The free
device memory must not change across the calls.  The file sorts last so that
a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads
import split_kv_paged_splitkv_gb300 as skv
from _support import compare, need_gpu, oracle_direct, session


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
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_noalloc_read_stats(plan, 0)
    assert e.value.status == skv.SPLITKV_EWORKSPACE


_CASES = [
    (workloads.WORKLOADS["gqa_ctx5900"], 0, "HND"),
    (workloads.WORKLOADS["tiny_gqa_ctx260"], 4, "HND"),
    # an e4m3 cache in NHD pages, and an MLA decode with a separate V tensor
    (workloads.Workload("noalloc_e4m3", 3, 1, 32, 4, 128, 128, 16, "fp8_e4m3",
                        "list:500:1200:33", pool_slack=0.5, seed=61), 0, "NHD"),
    (workloads.Workload("noalloc_mla", 1, 2, 128, 1, 576, 512, 64, "bf16", "list:700",
                        std=0.5, v_shares_k=False, pool_slack=0.5, seed=62), 3, "HND"),
    # and an MLA decode over an e4m3 latent cache
    (workloads.Workload("noalloc_mla_e4m3", 1, 2, 128, 1, 576, 512, 16, "fp8_e4m3", "list:900",
                        std=0.5, v_shares_k=True, pool_slack=0.5, seed=63), 4, "HND"),
]


@pytest.mark.gpu
def test_noalloc_equals_workspace_decode_on_consecutive_calls():
    need_gpu()
    runs = []
    for w, splits, layout in _CASES:
        x = workloads.make_inputs(w, device="cuda", layout=layout)
        ref = session(x, splits)
        ref_out, ref_lse = ref.run()
        ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
        ref_log, ref_status = ref.stats()
        assert ref_status == 0
        # outputs made before any free-memory reading: nothing below allocates
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        runs.append((x, splits, ref, ref_out, ref_lse, ref_log, out, lse))

    def call_all():
        for x, splits, ref, ref_out, ref_lse, ref_log, out, lse in runs:
            for _ in range(2):  # two calls in a row on the shared array
                out.fill_(float("nan"))
                lse.fill_(float("nan"))
                skv.splitkv_decode_noalloc(ref.plan, x.q, x.k_pages, x.v_pages, x.block_table,
                                           x.seq_lens, splits, x.scale, x.kv_scale, out, lse)
                log, status = skv.splitkv_noalloc_read_stats(ref.plan)
                assert status == 0, (x.w.name, status)
                assert torch.equal(out, ref_out), x.w.name
                assert torch.equal(lse, ref_lse), x.w.name
                assert np.array_equal(log, ref_log), x.w.name

    call_all()  # first calls: the library's one-time set-up happens here
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    call_all()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before

    # and the e4m3 NHD case against the fp64 oracle
    x, _, _, _, _, _, out, lse = runs[2]
    ref_o, ref_l = oracle_direct(x)
    compare(out, lse, ref_o, ref_l, what="noalloc e4m3 NHD")
