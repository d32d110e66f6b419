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
from split_kv_paged_splitkv_gb300.runner import DecodeSession

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _mla(lens, T, seed=3, v_shares_k=True, P=64, fp8=False):
    return workloads.Workload("mla_custom", len(lens), T, 128, 1, 576, 512, P,
                              "fp8_e4m3" if fp8 else "bf16",
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
        _check_cta_ranges(s, x, T)


def _check_cta_ranges(s, x, T):
    """The per-CTA log equals the plan exactly: 2*T CTAs per work item (token
    t, V half h), each iterating its item's page range [p0, p1) and scoring
    the keys min(p1 * P, L) - p0 * P of it, with no abort record."""
    items = skv.splitkv_plan_get_items(s.plan)
    log, _ = s.stats()
    assert len(log) == 2 * T * len(items)
    P = x.w.page_size
    L = x.seq_lens_host[items[:, 0]].astype(np.int64)
    keys = np.maximum(0, np.minimum(items[:, 5].astype(np.int64) * P, L) - items[:, 4] * P)
    assert np.array_equal(log[:, 0], np.repeat(items[:, 4], 2 * T))
    assert np.array_equal(log[:, 1], np.repeat(items[:, 5], 2 * T))
    assert np.array_equal(log[:, 2], np.repeat(keys, 2 * T))
    assert (log[:, 3] == 0).all()
    # and the planner's ranges equal the oracle's split table
    ref = oracle.plan_items(list(x.seq_lens_host), P, 1, s.num_splits,
                            torch.cuda.get_device_properties(0).multi_processor_count,
                            ctas_per_item=2 * T, ctas_per_sm=1)
    assert np.array_equal(items[:, :6], np.array(ref, np.int32).reshape(-1, 6))


@pytest.mark.parametrize("P", [16, 32, 64, 128])
@pytest.mark.parametrize("sepv,fp8", [(False, False), (True, False), (False, True)])
def test_mla_paged_gather_is_bit_exact(P, sepv, fp8):
    """The latent rows (576 wide, bf16 or e4m3 codes) and, with a separate V
    tensor, the V rows (512 wide), read through the block table with the
    decode kernel's tensor maps and shared-memory addressing, equal the CPU
    gather bit for bit."""
    lens = [3, P + 7, 777, 64 * 3]
    x = workloads.make_inputs(_mla(lens, 2, seed=70 + P + sepv, v_shares_k=not sepv, P=P, fp8=fp8),
                              device="cuda")
    desc = skv.make_desc(len(lens), 2, 128, 1, 576, 512, P, x.max_pages, x.num_pages,
                         skv.SPLITKV_FP8_E4M3 if fp8 else skv.SPLITKV_BF16, int(not sepv))
    tables = x.block_table.cpu().numpy()
    for b, L in enumerate(x.seq_lens_host):
        L = int(L)
        for pages, width in ((x.k_pages, 576),) + (((x.v_pages, 512),) if sepv else ()):
            dst = torch.zeros((L, width), dtype=pages.dtype, device="cuda")
            skv.splitkv_debug_gather(desc, pages, width, x.block_table, b, 0, L, dst)
            torch.cuda.synchronize()
            ref = oracle.gather_keys(workloads.bits(pages), tables[b], L, 0)
            assert np.array_equal(workloads.bits(dst), ref), (b, width)


@pytest.mark.parametrize("T", [1, 2, 6, 16])
def test_mla_fp8_small_ragged(T):
    """An e4m3 latent cache (V = its first 512 columns, one per-tensor scale):
    converted to f16 in shared memory, f16 tensor-core products."""
    lens = [T, 64, 100, 130, 1000]
    x = workloads.make_inputs(_mla(lens, T, seed=40 + T, fp8=True), device="cuda")
    ref_o, ref_l = oracle_direct(x)
    for S in (1, 2, 3, 0):
        s = session(x, S)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"fp8 T={T} S={S}")
        assert s.stats()[1] == 0
        _check_cta_ranges(s, x, T)


@pytest.mark.parametrize("P", [16, 32, 128, 192])
def test_mla_fp8_page_sizes(P):
    T = 3
    lens = [T, 40, P + 7, 3 * P, 777, 2100]
    x = workloads.make_inputs(_mla(lens, T, seed=50 + P, P=P, fp8=True), device="cuda")
    ref_o, ref_l = oracle_direct(x)
    for S in (1, 3, 7, 0):
        s = session(x, S)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"fp8 P={P} S={S}")
        assert s.stats()[1] == 0
        _check_cta_ranges(s, x, T)


@pytest.mark.parametrize("mag", [1e5, 1e-6, "spread"])
def test_mla_fp8_queries_of_any_bf16_magnitude(mag):
    """Queries far outside f16's range (the kernel scales each row by a power
    of two before its f16 products), or with components spread over 2^-20 ..
    2^16 within each row, with the cache scale set so that the scores stay of
    order one; outputs compared relative to their size."""
    T = 2
    lens = [T + 3, 300, 1000]
    x = workloads.make_inputs(_mla(lens, T, seed=60, fp8=True), device="cuda")
    if mag == "spread":
        rng = np.random.default_rng(61)
        e = torch.from_numpy(rng.uniform(-20, 16, size=tuple(x.q.shape))).float().cuda()
        q = (torch.sign(x.q.float()) * torch.exp2(e)).to(torch.bfloat16)
        kv_scale = float(np.float32(x.kv_scale / 2.0 ** 16))
    else:
        q = (x.q.float() * mag).to(torch.bfloat16)
        kv_scale = float(np.float32(x.kv_scale / mag))
    ref_o, ref_l = oracle.attention_direct(
        workloads.bits(q), workloads.bits(x.k_pages), None, x.block_table.cpu().numpy(),
        x.seq_lens_host, scale=x.scale, kv_dtype="fp8_e4m3", kv_scale=kv_scale, v_dim=512,
        v_shares_k=True)
    s = DecodeSession(q, x.k_pages, None, x.block_table, x.seq_lens, x.seq_lens_host,
                      scale=x.scale, kv_scale=kv_scale, num_splits=3, v_dim=512, v_shares_k=True)
    out, lse = s.run()
    assert s.stats()[1] == 0
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    assert np.abs(o - ref_o).max() <= 1e-2 * np.abs(ref_o).max()
    assert np.abs(lse.cpu().numpy() - ref_l).max() <= 1e-3


@pytest.mark.parametrize("name", ["mla_t6_ctx64k", "mla_sepv_t6_ctx64k", "mla_fp8_t6_ctx64k"])
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
        _check_cta_ranges(s, x, T)


@pytest.mark.parametrize("P", [16, 64])
@pytest.mark.parametrize("sepv,fp8", [(False, False), (True, False), (False, True)])
def test_mla_out_of_range_page_ids_are_flagged(P, sepv, fp8):
    """As for GQA: an entry >= num_pages and a negative one are read as page
    0, SPLITKV_DEVERR_PAGE is set, the output stays finite, and the intact
    sequences match the oracle."""
    T = 2
    lens = [640, 1024, 320]  # whole pages: no poisoned tail slots in page 0
    x = workloads.make_inputs(_mla(lens, T, seed=90 + P + sepv, v_shares_k=not sepv, P=P, fp8=fp8),
                              device="cuda")
    ref_o, ref_l = oracle_direct(x)
    bad = x.block_table.clone()
    bad[1, 2] = x.num_pages + 3
    bad[2, 0] = -1
    for S in (1, 3):
        s = session(x, S)
        out, lse = s.run(tensors=(x.q, x.k_pages, x.v_pages, bad, x.seq_lens))
        log, status = s.stats()
        assert status & skv.SPLITKV_DEVERR_PAGE, status
        assert not status & skv.SPLITKV_DEVERR_TIMEOUT
        assert torch.isfinite(out.float()).all()
        rows = [(0, t, h) for t in range(T) for h in range(128)]
        compare(out, lse, ref_o, ref_l, rows=rows, what=f"P={P} sepv={sepv} S={S}")
