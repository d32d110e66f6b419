"""Performance regression tests: correct output can hide a slow split-KV path.

"vLLM 0.30.0 FA4 SplitKV Bug: H100 Decode Can Be 48% Slower" (sections "Why
the result is still correct" and "The kernel-only sweep makes the bug
obvious"): when the requested split count never reached the kernel, every
extra split CTA got an empty KV range, the outputs stayed right, and only a
kernel-only sweep over num_splits showed the decode getting no faster.  The
same sweep guards this library: the 5,900-key single-sequence decode must get
faster at every step from 1 to 64 splits, and at 64 splits at least 8x faster
than unsplit.  Floors guard the other workloads: the long FP8 batch's split
kernel alone must move its algorithmic bytes at >= 0.70 of the measured HBM
copy bandwidth, the mixed-length bf16 batch of 32 at >= 0.85, the 6-token MLA
decode's split kernel must reach >= 0.36 of the measured bf16 tensor
throughput, and the whole 5,900-key call must stay under 7.5 us (each about
15 % below what this build measures); through a 64-split capacity plan (the
CUDA-graph serving path) it must stay under 7.6 us, which a capacity plan
that misses the one-wave kernel form does not.

Timing: CUDA-graph replay of back-to-back calls rotating over copies of the
KV pool whose total exceeds four times the L2 size, CUDA events on the
launching stream, after warm-up replays.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads
from _support import need_gpu, session

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _pools(x):
    l2 = int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 << 20))
    nbytes = x.k_pages.numel() * x.k_pages.element_size() + (
        0 if x.v_pages is None else x.v_pages.numel() * x.v_pages.element_size())
    R = max(2, math.ceil(4 * l2 / nbytes))
    pools = [(x.k_pages, x.v_pages)]
    pools += [(x.k_pages.clone(), None if x.v_pages is None else x.v_pages.clone())
              for _ in range(R - 1)]
    return pools


def _us_per_call(sess, x, pools, partials=False, reps=20):
    def step(i):
        k, v = pools[i % len(pools)]
        t = (x.q, k, v, x.block_table, x.seq_lens)
        if partials:
            sess.run_partials(tensors=t)
        else:
            sess.run(tensors=t)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(len(pools)):
            step(i)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    e1.synchronize()
    assert sess.stats()[1] == 0
    return e0.elapsed_time(e1) * 1e3 / (reps * len(pools))


def test_split_sweep_gets_faster():
    x = workloads.make_inputs(workloads.WORKLOADS["gqa_ctx5900"], device="cuda")
    pools = _pools(x)
    t = {}
    for S in (1, 4, 16, 64):
        sess = session(x, S)
        t[S] = _us_per_call(sess, x, pools)
        # every launched split CTA owned keys (the page's bug gave them none)
        log, status = sess.stats()
        assert status == 0 and (log[:, 2] > 0).all() and len(log) == 2 * S
    msg = ", ".join(f"S={S}: {v:.2f} us" for S, v in t.items())
    for a, b in ((1, 4), (4, 16), (16, 64)):
        assert t[b] < 0.95 * t[a], f"more splits did not speed the decode up ({msg})"
    assert t[1] >= 8 * t[64], f"64 splits less than 8x faster than 1 ({msg})"


def _peak(key, fallback):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))[key])
    return fallback  # one earlier measurement on this part


def _hbm_peak():
    return _peak("hbm_gbs", 6800.0)


def _kv_bytes(w, x):
    lens = x.seq_lens_host.astype(np.int64)
    kv = 1 if w.kv_dtype == "fp8_e4m3" else 2
    return int(lens.sum()) * w.num_kv_heads * 2 * w.qk_dim * kv + w.batch * w.num_q_heads * w.qk_dim * 2


def test_fp8_batch8_ctx32k_bandwidth_floor():
    w = workloads.WORKLOADS["fp8_batch8_ctx32k"]
    x = workloads.make_inputs(w, device="cuda")
    pools = _pools(x)
    sess = session(x, 0)
    us = _us_per_call(sess, x, pools, partials=True, reps=10)
    gbs = _kv_bytes(w, x) / (us * 1e-6) / 1e9
    peak = _hbm_peak()
    assert gbs >= 0.70 * peak, f"{gbs:.0f} GB/s is below 0.70 of {peak:.0f} GB/s ({us:.1f} us)"


def test_mixed_batch32_bf16_bandwidth_floor():
    w = workloads.WORKLOADS["mixed_batch32_bf16"]
    x = workloads.make_inputs(w, device="cuda")
    pools = _pools(x)
    sess = session(x, 0)
    us = _us_per_call(sess, x, pools, partials=True, reps=3)
    gbs = _kv_bytes(w, x) / (us * 1e-6) / 1e9
    peak = _hbm_peak()
    assert gbs >= 0.85 * peak, f"{gbs:.0f} GB/s is below 0.85 of {peak:.0f} GB/s ({us:.1f} us)"


def test_mla_t6_ctx64k_tensor_floor():
    w = workloads.WORKLOADS["mla_t6_ctx64k"]
    x = workloads.make_inputs(w, device="cuda")
    pools = _pools(x)
    sess = session(x, 0)
    us = _us_per_call(sess, x, pools, partials=True, reps=5)
    # query token t sees L - T + 1 + t keys; QK over 576 dims and PV over 512,
    # 2 FLOP per multiply-add, 128 heads
    L, T = int(x.seq_lens_host[0]), w.q_tokens
    visible = sum(L - T + 1 + t for t in range(T))
    tflops = 2.0 * w.num_q_heads * visible * (w.qk_dim + w.v_dim) / (us * 1e-6) / 1e12
    peak = _peak("bf16_tflops", 1900.0)
    assert tflops >= 0.36 * peak, f"{tflops:.0f} TFLOP/s is below 0.36 of {peak:.0f} ({us:.1f} us)"


def test_gqa_ctx5900_call_latency_ceiling():
    x = workloads.make_inputs(workloads.WORKLOADS["gqa_ctx5900"], device="cuda")
    pools = _pools(x)
    us = _us_per_call(session(x, 0), x, pools, reps=200)
    assert us <= 7.5, f"the 5,900-key call takes {us:.2f} us"


def test_gqa_ctx5900_capacity_plan_latency_ceiling():
    from split_kv_paged_splitkv_gb300.runner import DecodeSession
    x = workloads.make_inputs(workloads.WORKLOADS["gqa_ctx5900"], device="cuda")
    pools = _pools(x)
    sess = DecodeSession(x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens, x.seq_lens_host,
                         scale=x.scale, kv_scale=x.kv_scale, num_splits=64, fixed=True)
    us = _us_per_call(sess, x, pools, reps=200)
    assert us <= 7.6, f"the 5,900-key call through a capacity plan takes {us:.2f} us"
