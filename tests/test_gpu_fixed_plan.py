"""GPU checks of capacity plans (splitkv_plan_fixed).

* the work items the decode kernels derive from the device lengths -- read
  back through splitkv_plan_refresh / splitkv_read_items, which write the
  same list, and through the per-CTA log of page ranges -- equal the oracle
  planner's for the same num_splits (every used item), and the unused
  capacity items are marked and score nothing;
* decodes through a capacity plan match the fp64 oracle;
* one captured CUDA graph of decodes replayed over changing device lengths
  matches the oracle for each set of lengths.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import split_kv_paged_splitkv_gb300 as skv
from split_kv_paged_splitkv_gb300.runner import DecodeSession
from _support import compare, need_gpu, oracle_direct

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _gqa(lens, G=8, Hkv=2, T=1, P=16, fp8=False, seed=3):
    return workloads.Workload(
        "fixed", len(lens), T, G * Hkv, Hkv, 128, 128, P, "fp8_e4m3" if fp8 else "bf16",
        "list:" + ":".join(str(int(x)) for x in lens), pool_slack=0.5, seed=seed)


def _mla(lens, T=2, seed=5, v_shares_k=True, P=64, fp8=False):
    return workloads.Workload("fixed_mla", len(lens), T, 128, 1, 576, 512, P,
                              "fp8_e4m3" if fp8 else "bf16",
                              "list:" + ":".join(str(int(x)) for x in lens), std=0.5,
                              v_shares_k=v_shares_k, pool_slack=0.5, seed=seed)


def _session(x, S, mode=skv.SPLITKV_COMBINE_SEPARATE, lens_dev=None):
    return DecodeSession(x.q, x.k_pages, x.v_pages, x.block_table,
                         x.seq_lens if lens_dev is None else lens_dev, x.seq_lens_host,
                         scale=x.scale, kv_scale=x.kv_scale, num_splits=S, combine_mode=mode,
                         v_dim=x.w.v_dim, v_shares_k=x.w.v_shares_k, fixed=True)


def _oracle_at(x, lens):
    """Oracle output for the same pages and tables at other (shorter) lengths."""
    return oracle.attention_direct(
        workloads.bits(x.q), workloads.bits(x.k_pages),
        None if x.v_pages is None else workloads.bits(x.v_pages),
        x.block_table.cpu().numpy(), np.asarray(lens, np.int32), scale=x.scale,
        kv_dtype=x.w.kv_dtype, kv_scale=x.kv_scale, v_dim=x.w.v_dim, v_shares_k=x.w.v_shares_k)


@pytest.mark.parametrize("fp8,Hkv,G", [(False, 2, 8), (True, 8, 4), (True, 3, 2)])
def test_refreshed_work_list_equals_the_planner(fp8, Hkv, G):
    lens = [0, 5, 16 * 3 + 1, 16 * 40, 16 * 7]
    x = workloads.make_inputs(_gqa(lens, G=G, Hkv=Hkv, fp8=fp8), device="cuda")
    for S in (1, 4, 9):
        s = _session(x, S)
        s.run()
        log, status = s.stats()
        skv.splitkv_plan_refresh(s.plan, s.workspace, x.seq_lens)
        items = skv.splitkv_read_items(s.plan, s.workspace)
        # the kernels iterated exactly the page ranges of the refreshed list
        assert np.array_equal(log[:, 0], items[:, 4]) and np.array_equal(log[:, 1], items[:, 5])
        hpi = skv.splitkv_plan_heads_per_item(s.plan)
        U = Hkv // hpi
        assert items.shape[0] == len(lens) * U * S
        used = items[items[:, 3] > 0]
        ref = np.array(oracle.plan_items(lens, 16, Hkv, S, 132, heads_per_item=hpi), np.int32)
        key = lambda a: np.lexsort((a[:, 2], a[:, 1], a[:, 0]))
        assert np.array_equal(used[key(used)][:, :6], ref[key(ref)])
        # fixed partial slots: group g = b * U + u owns slots [g S, g S + S)
        for it in used:
            b, h, sp, Sb = it[:4]
            g = b * U + h // hpi
            assert it[6] == (g * S + sp if Sb > 1 else -1) and it[7] == (g if Sb > 1 else -1)
        assert status == 0
        assert (log[items[:, 3] == 0, 2] == 0).all()  # unused capacity items score nothing
        out, lse = s.out, s.lse
        ref_o, ref_l = oracle_direct(x)
        compare(out, lse, ref_o, ref_l, what=f"fixed S={S} fp8={fp8}")


@pytest.mark.parametrize("mode", [skv.SPLITKV_COMBINE_SEPARATE, skv.SPLITKV_COMBINE_FUSED])
@pytest.mark.parametrize("T,G", [(1, 8), (2, 8), (4, 8)])
def test_one_graph_serves_changing_lengths(mode, T, G):
    """Capture the decode once; change the device lengths; replay."""
    cap = [16 * 30 + 3, 16 * 61, 16 * 9 + 7]
    x = workloads.make_inputs(_gqa(cap, G=G, T=T, seed=11), device="cuda")
    lens_dev = x.seq_lens.clone()
    s = _session(x, 8, mode, lens_dev=lens_dev)
    s.run()  # eager warm-up (sets kernel attributes before capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s.run()
    for lens in (cap, [T, 16 * 61, 0], [16 * 2, 5 + T, 16 * 9 + 7], [16 * 30, 16 * 8 + 1, T + 1]):
        lens_dev.copy_(torch.tensor(lens, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = _oracle_at(x, lens)
        compare(s.out, s.lse, ref_o, ref_l, what=f"graph lens={lens} mode={mode}")
        assert s.stats()[1] == 0


@pytest.mark.parametrize("v_shares_k,P,fp8", [(True, 64, False), (False, 64, False), (True, 16, False),
                                               (False, 32, False), (True, 64, True), (True, 16, True)])
def test_mla_capacity_plan(v_shares_k, P, fp8):
    cap = [64 * 9 + 5, 64 * 3, 2]
    x = workloads.make_inputs(_mla(cap, v_shares_k=v_shares_k, P=P, fp8=fp8), device="cuda")
    lens_dev = x.seq_lens.clone()
    s = _session(x, 4, lens_dev=lens_dev)
    for lens in (cap, [64 * 2 + 1, 64 * 3, 0]):
        lens_dev.copy_(torch.tensor(lens, dtype=torch.int32))
        s.run()
        torch.cuda.synchronize()
        ref_o, ref_l = _oracle_at(x, lens)
        compare(s.out, s.lse, ref_o, ref_l, what=f"mla P={P} lens={lens}")
        log, status = s.stats()
        assert status == 0


def test_bad_device_length_is_reported_and_served_empty():
    cap = [16 * 5, 16 * 3]
    x = workloads.make_inputs(_gqa(cap), device="cuda")
    lens_dev = x.seq_lens.clone()
    s = _session(x, 2, lens_dev=lens_dev)
    lens_dev.copy_(torch.tensor([16 * 5, 16 * 1000], dtype=torch.int32))  # beyond the table
    s.run()
    torch.cuda.synchronize()
    assert s.stats()[1] & skv.SPLITKV_DEVERR_SEQLEN
    lse = s.lse.cpu().numpy()
    assert np.isneginf(lse[1]).all() and (s.out[1].float().cpu().numpy() == 0).all()
    ref_o, ref_l = _oracle_at(x, [16 * 5, 0])
    compare(s.out[:1], s.lse[:1], ref_o[:1], ref_l[:1], what="valid sequence next to a bad one")
