"""splitkv_decode in two steps (splitkv_decode_partials, then
splitkv_combine_workspace) writes exactly what the one-call decode writes in
SEPARATE mode, for every kernel family and for capacity plans; the partial
pass alone leaves single-split sequences final."""
import numpy as np
import pytest
import torch

import workloads
import split_kv_paged_splitkv_gb300 as skv
from _support import compare, need_gpu, oracle_direct
from split_kv_paged_splitkv_gb300.runner import DecodeSession

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _gqa(lens, fp8, T=1, G=8, Hkv=2, P=16):
    return workloads.Workload(
        "two_step", len(lens), T, G * Hkv, Hkv, 128, 128, P, "fp8_e4m3" if fp8 else "bf16",
        "list:" + ":".join(str(int(x)) for x in lens), pool_slack=0.5, seed=23 + fp8)


def _mla(lens, T, v_shares_k):
    return workloads.Workload("two_step_mla", len(lens), T, 128, 1, 576, 512, 64, "bf16",
                              "list:" + ":".join(str(int(x)) for x in lens), std=0.5,
                              v_shares_k=v_shares_k, pool_slack=0.5, seed=31 + T)


def _two_step_equals_decode(x, S, mode=skv.SPLITKV_COMBINE_SEPARATE, fixed=False):
    ref_o, ref_l = oracle_direct(x)
    one = DecodeSession(x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens, x.seq_lens_host,
                        scale=x.scale, kv_scale=x.kv_scale, num_splits=S, v_dim=x.w.v_dim,
                        v_shares_k=x.w.v_shares_k, combine_mode=skv.SPLITKV_COMBINE_SEPARATE,
                        fixed=fixed)
    two = DecodeSession(x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens, x.seq_lens_host,
                        scale=x.scale, kv_scale=x.kv_scale, num_splits=S, v_dim=x.w.v_dim,
                        v_shares_k=x.w.v_shares_k, combine_mode=mode, fixed=fixed)
    o1, l1 = one.run()
    two.out.fill_(float("nan"))
    two.lse.fill_(float("nan"))
    two.run_partials()
    # rows of single-split sequences are final after the partial pass alone
    if fixed:
        skv.splitkv_plan_refresh(two.plan, two.workspace, x.seq_lens)
        items = skv.splitkv_read_items(two.plan, two.workspace)
    else:
        items = skv.splitkv_plan_get_items(two.plan)
    single = sorted({int(b) for b, ns in zip(items[:, 0], items[:, 3]) if ns == 1})
    torch.cuda.synchronize()
    for b in single:
        assert torch.equal(two.out[b], o1[b]) and torch.equal(two.lse[b], l1[b]), b
    o2, l2 = two.merge()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    compare(o2, l2, ref_o, ref_l, what=f"S={S} mode={mode} fixed={fixed}")
    assert two.stats()[1] == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_gqa_two_step(fp8):
    x = workloads.make_inputs(_gqa([1, 16, 300, 1000, 0, 2000], fp8), device="cuda")
    for S in (1, 4, 0):
        _two_step_equals_decode(x, S)
    # a FUSED descriptor: the partial pass still leaves the merge to the second step
    _two_step_equals_decode(x, 4, mode=skv.SPLITKV_COMBINE_FUSED)


def test_gqa_two_step_capacity_plan():
    x = workloads.make_inputs(_gqa([5, 700, 1300, 64], False, T=2, G=4), device="cuda")
    _two_step_equals_decode(x, 3, fixed=True)


@pytest.mark.parametrize("v_shares_k", [True, False])
def test_mla_two_step(v_shares_k):
    x = workloads.make_inputs(_mla([6, 300, 1500], 6, v_shares_k), device="cuda")
    for S in (1, 3, 0):
        _two_step_equals_decode(x, S)
