"""GPU parity of the MLA split-KV path (tcgen05/TMEM kernel) against the fp64 oracle.

128 query heads per token share one 576-wide latent KV head; V is its first 512
columns; query tokens are causal among themselves.  Bars as elsewhere: max-abs
error <= 1e-2 on bf16 outputs, <= 1e-3 on fp32 LSE.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import split_kv_paged_splitkv_gb300 as skv
from _support import compare, need_gpu, oracle_direct, session

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _mla(lens, T, seed=3, v_shares_k=True, P=64):
    return workloads.Workload("mla_custom", len(lens), T, 128, 1, 576, 512, P, "bf16",
                              "list:" + ":".join(str(int(x)) for x in lens), std=0.5,
                              v_shares_k=v_shares_k, pool_slack=0.5, seed=seed)


@pytest.mark.parametrize("T", [1, 2, 6, 16])
@pytest.mark.parametrize("sepv", [False, True])
def test_mla_small_ragged(T, sepv):
    """V as the first 512 columns of the latent rows, or (sepv) its own tensor."""
    lens = [T, 64, 100, 130, 1000]
    x = workloads.make_inputs(_mla(lens, T, seed=10 + T + 5 * sepv, v_shares_k=not sepv),
                              device="cuda")
    ref_o, ref_l = oracle_direct(x)
    for S in (1, 2, 3, 0):
        s = session(x, S)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"T={T} S={S}")
        log, status = s.stats()
        assert status == 0, status
        items = skv.splitkv_plan_get_items(s.plan)
        # 2*T CTAs per item, in item order; every CTA scored its item's keys
        nonempty = np.repeat(items[:, 5] > items[:, 4], 2 * T)
        assert (log[nonempty, 2] > 0).all()
        assert (log[:, 3] == 0).all()


@pytest.mark.parametrize("name", ["mla_t6_ctx64k", "mla_sepv_t6_ctx64k"])
def test_mla_ctx64k_full(name):
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w, device="cuda")
    ref_o, ref_l = oracle_direct(x)
    for S in w.splits:
        s = session(x, S)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"S={S}")
        log, status = s.stats()
        assert status == 0 and (log[:, 2] > 0).all()


@pytest.mark.parametrize("P", [16, 32, 128, 192])
@pytest.mark.parametrize("sepv", [False, True])
def test_mla_page_sizes(P, sepv):
    """Pages smaller than the 64-key block (several boxes per block chunk,
    split boundaries inside a block) and larger ones (several blocks per
    page, split boundaries at page starts)."""
    T = 3
    lens = [T, 40, P + 7, 3 * P, 777, 2100]
    x = workloads.make_inputs(_mla(lens, T, seed=30 + P + sepv, v_shares_k=not sepv, P=P),
                              device="cuda")
    ref_o, ref_l = oracle_direct(x)
    for S in (1, 3, 7, 0):
        s = session(x, S)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"P={P} sepv={sepv} S={S}")
        log, status = s.stats()
        assert status == 0, status
        assert (log[:, 3] == 0).all()
