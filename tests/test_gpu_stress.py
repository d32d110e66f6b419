"""Back-to-back calls in a CUDA graph, as bench.py runs them: no bounded wait
may time out (status word 0, no abort record in any CTA's log) and the last
call's output must equal, bit for bit, what one eager call writes.  Rare
synchronisation races (a barrier phase seen from two phases behind, a buffer
reused early) show up here as a status bit or as differing bits.
"""
import pytest
import torch

import workloads
import split_kv_paged_splitkv_gb300 as skv
from _support import need_gpu
from split_kv_paged_splitkv_gb300.runner import DecodeSession

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.mark.parametrize("name,mode,calls", [
    ("mla_t6_ctx64k", skv.SPLITKV_COMBINE_SEPARATE, 600),
    ("mla_sepv_t6_ctx64k", skv.SPLITKV_COMBINE_SEPARATE, 600),
    ("mla_fp8_t6_ctx64k", skv.SPLITKV_COMBINE_SEPARATE, 600),
    ("gqa_ctx5900", skv.SPLITKV_COMBINE_SEPARATE, 3000),
    ("gqa_ctx5900", skv.SPLITKV_COMBINE_FUSED, 3000),
    ("fp8_batch8_ctx32k", skv.SPLITKV_COMBINE_SEPARATE, 600),
    ("spec_t4_gqa_ctx5900", skv.SPLITKV_COMBINE_SEPARATE, 3000),
    ("spec_t4_gqa_ctx5900", skv.SPLITKV_COMBINE_FUSED, 3000),
    # two query tokens over the e4m3 batch: two KV heads and two row groups
    # per item in a multi-wave grid
    ("fp8_batch8_ctx32k@2", skv.SPLITKV_COMBINE_SEPARATE, 300),
])
def test_back_to_back_calls(name, mode, calls):
    w = workloads.WORKLOADS[name.split("@")[0]]
    if "@" in name:
        w = w.replace(q_tokens=int(name.split("@")[1]))
    x = workloads.make_inputs(w, device="cuda")
    s = DecodeSession(x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens, x.seq_lens_host,
                      scale=x.scale, kv_scale=x.kv_scale, num_splits=0, v_dim=w.v_dim,
                      v_shares_k=w.v_shares_k, combine_mode=mode)
    ref_o, ref_l = (t.clone() for t in s.run())
    torch.cuda.synchronize()
    # a second pool, so consecutive calls read different memory
    pools = [(x.k_pages, x.v_pages),
             (x.k_pages.clone(), None if x.v_pages is None else x.v_pages.clone())]
    per_graph = 20
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(per_graph):
            k, v = pools[i % 2]
            s.run(tensors=(x.q, k, v, x.block_table, x.seq_lens))
    for _ in range(calls // per_graph):
        g.replay()
    torch.cuda.synchronize()
    log, status = s.stats()
    assert status == 0, f"{name}: device status {status}"
    if w.num_kv_heads == 1:  # MLA: field 3 of the log is the abort record
        assert (log[:, 3] == 0).all(), f"{name}: CTAs gave up: {log[log[:, 3] != 0][:4]}"
    assert torch.equal(s.out, ref_o) and torch.equal(s.lse, ref_l), name
