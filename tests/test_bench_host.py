"""Host logic of bench.py (CPU only).

* The per-step inputs of the single-pool layout: R copies of the workload's
  pages scattered over one pool in random order, one block table per step.
  Through its own table every step must read exactly the workload's key and
  value rows (checked with the oracle's gather), and the steps' page sets
  must be disjoint, so that no step finds its pages in L2.
* The algorithmic byte and FLOP counts the roofline divides by, against
  closed forms for the workloads' shapes.
"""
import numpy as np
import pytest

import bench
import oracle
import workloads


@pytest.mark.parametrize("name,layout", [("tiny_gqa_ctx260", "HND"), ("tiny_gqa_ctx260", "NHD"),
                                         ("fp8_batch8_ctx32k", "HND")])
def test_single_pool_steps_read_the_workload_rows(name, layout):
    w = workloads.WORKLOADS[name]
    if w.batch > 1:  # keep the CPU test small: two short sequences of the same shape
        w = w.replace(batch=2, lens="list:300:1000")
    x = workloads.make_inputs(w, device="cpu", layout=layout)
    R = 3
    big_k, big_v, steps = bench.step_inputs(x, R, "single")
    assert big_k.shape[0] == R * x.k_pages.shape[0]
    used = []
    for k, v, t in steps:
        assert k is big_k and v is big_v
        pages = set()
        for b, L in enumerate(x.seq_lens_host):
            L = int(L)
            n = -(-L // w.page_size)
            pages |= set(t[b, :n].tolist())
            for h in range(w.num_kv_heads):
                for got, ref in ((k, x.k_pages), (v, x.v_pages)):
                    a = oracle.gather_keys(workloads.bits(got), t[b].numpy(), L, h, layout)
                    r = oracle.gather_keys(workloads.bits(ref), x.block_table[b].numpy(), L, h,
                                           layout)
                    assert np.array_equal(a, r)
        used.append(pages)
    for i in range(R):
        for j in range(i + 1, R):
            assert not (used[i] & used[j])


def test_rotating_pools_keep_the_table():
    x = workloads.make_inputs(workloads.WORKLOADS["tiny_gqa_ctx260"], device="cpu")
    _, _, steps = bench.step_inputs(x, 3, "rotate")
    assert steps[0][0] is x.k_pages
    for k, v, t in steps:
        assert t is x.block_table
        # (bit patterns: the poisoned page holds NaN)
        assert np.array_equal(workloads.bits(k), workloads.bits(x.k_pages))
        assert np.array_equal(workloads.bits(v), workloads.bits(x.v_pages))
    assert steps[1][0].data_ptr() != steps[2][0].data_ptr()


def test_algorithmic_counts():
    w = workloads.WORKLOADS["gqa_ctx5900"]
    lens = np.array([5900], np.int32)
    # keys x KV heads x (K + V rows of 128 bf16) + Q
    assert bench.algorithmic_bytes(w, lens) == 5900 * 2 * 2 * 128 * 2 + 16 * 128 * 2
    w8 = workloads.WORKLOADS["fp8_batch8_ctx32k"]
    lens8 = np.array([30000, 29000], np.int32)
    assert bench.algorithmic_bytes(w8, lens8) == 59000 * 4 * 2 * 128 + 8 * 32 * 128 * 2
    m = workloads.WORKLOADS["mla_t6_ctx64k"]
    lm = np.array([65536], np.int32)
    # latent rows read once (V shares them)
    assert bench.algorithmic_bytes(m, lm) == 65536 * 576 * 2 + 6 * 128 * 576 * 2
    # query token t sees L - T + 1 + t keys; 2 FLOP per multiply-add over 576 + 512
    vis = sum(65536 - 6 + 1 + t for t in range(6))
    assert bench.algorithmic_flops(m, lm) == 2.0 * 128 * vis * (576 + 512)
    assert bench.is_tensor_bound(m) and not bench.is_tensor_bound(w)
    sv = workloads.WORKLOADS["mla_sepv_t6_ctx64k"]
    assert bench.algorithmic_bytes(sv, lm) == 65536 * (576 + 512) * 2 + 6 * 128 * 576 * 2
    sp = workloads.WORKLOADS["spec_t4_gqa_ctx5900"]
    # the four tokens share the keys: KV counted once, Q for every token
    assert bench.algorithmic_bytes(sp, lens) == 5900 * 2 * 2 * 128 * 2 + 4 * 16 * 128 * 2
    f8 = workloads.WORKLOADS["mla_fp8_t6_ctx64k"]
    assert bench.algorithmic_bytes(f8, lm) == 65536 * 576 + 6 * 128 * 576 * 2


def test_packed_step_buffer_round_trips():
    """The end-to-end leg ships a step's inputs in one byte buffer: every
    tensor at a 256-byte-aligned offset, read back bit for bit through its
    view (e4m3 codes, bf16 with NaN poison, int32 tables)."""
    import torch
    x = workloads.make_inputs(workloads.WORKLOADS["fp8_batch8_ctx32k"].replace(
        batch=2, lens="list:300:1000"), device="cpu")
    src = [x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens]
    offs, n = bench._packed(src)
    assert all(o % 256 == 0 for o in offs)
    assert n == offs[-1] + x.seq_lens.numel() * 4
    for a, b, t in zip(offs, offs[1:], src):
        assert a + t.numel() * t.element_size() <= b
    buf = torch.zeros(n, dtype=torch.uint8)
    views = bench._views(buf, src, offs)
    for v, t in zip(views, src):
        v.copy_(t)
    for v, t in zip(bench._views(buf.clone(), src, offs), src):
        assert v.dtype == t.dtype and v.shape == t.shape
        assert torch.equal(v.reshape(-1).view(torch.uint8), t.reshape(-1).view(torch.uint8))
