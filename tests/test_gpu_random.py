"""Seeded random configurations against the fp64 oracle.

The fixed cases elsewhere vary one option at a time; these draw them jointly:
batch, query tokens, group size, KV heads, page size, cache type, page layout,
per-KV-head scales, split count, combine mode and ragged lengths (empty
sequences and exact page multiples included) for the GQA kernel, and tokens,
page size, lengths, split count, a separate V tensor or an e4m3 latent cache for the
MLA kernel.  Sizes stay
small enough for the oracle to finish in seconds.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import split_kv_paged_splitkv_gb300 as skv
from _support import compare, need_gpu, oracle_direct
from split_kv_paged_splitkv_gb300.runner import DecodeSession

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _lens(rng, B, P, T, max_len):
    out = []
    for _ in range(B):
        r = rng.random()
        if r < 0.1:
            out.append(0)
        elif r < 0.25:
            out.append(int(P * rng.integers(1, max(2, max_len // P))))  # exact page multiple
        else:
            out.append(int(rng.integers(T, max_len + 1)))
    return out


@pytest.mark.parametrize("case", range(48))
def test_random_gqa(case):
    rng = np.random.default_rng(500 + case)
    T = int(rng.choice([1, 1, 2, 3, 4]))
    G = int(rng.choice([g for g in (1, 2, 4, 5, 8) if T * g <= 32]))
    Hkv = int(rng.choice([1, 2, 3, 4]))
    P = int(rng.choice([16, 32, 64]))
    B = int(rng.integers(1, 5))
    fp8 = bool(rng.random() < 0.5)
    layout = "NHD" if rng.random() < 0.3 else "HND"
    lens = _lens(rng, B, P, T, 1800)
    w = workloads.Workload(f"rand{case}", B, T, G * Hkv, Hkv, 128, 128, P,
                           "fp8_e4m3" if fp8 else "bf16",
                           "list:" + ":".join(str(x) for x in lens), pool_slack=0.3,
                           seed=700 + case)
    x = workloads.make_inputs(w, device="cuda", layout=layout)
    per_head = fp8 and rng.random() < 0.4
    S = int(rng.choice([0, 0, 1, 2, 3, 7, 64]))
    mode = int(rng.choice([skv.SPLITKV_COMBINE_FUSED, skv.SPLITKV_COMBINE_SEPARATE]))
    kw = dict(scale=x.scale, kv_scale=x.kv_scale, num_splits=S, combine_mode=mode,
              kv_layout=skv.SPLITKV_LAYOUT_NHD if layout == "NHD" else skv.SPLITKV_LAYOUT_HND)
    what = f"T={T} G={G} Hkv={Hkv} P={P} B={B} fp8={fp8} {layout} S={S} mode={mode} lens={lens}"
    if per_head:
        c = float(x.kv_scale)
        ks = c * rng.uniform(0.4, 1.0, Hkv)
        vs = c * rng.uniform(0.4, 1.0, Hkv)
        ref_o, ref_l = oracle.attention_direct(
            workloads.bits(x.q), workloads.bits(x.k_pages), workloads.bits(x.v_pages),
            x.block_table.cpu().numpy(), x.seq_lens_host, scale=x.scale, kv_dtype="fp8_e4m3",
            k_scale=ks.astype(np.float32).astype(np.float64),
            v_scale=vs.astype(np.float32).astype(np.float64), layout=layout)
        kw.update(k_scale=torch.tensor(ks, dtype=torch.float32, device="cuda"),
                  v_scale=torch.tensor(vs, dtype=torch.float32, device="cuda"))
        what += " per-head scales"
    else:
        ref_o, ref_l = oracle_direct(x)
    s = DecodeSession(x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens, x.seq_lens_host, **kw)
    out, lse = s.run()
    compare(out, lse, ref_o, ref_l, what=what)
    log, status = s.stats()
    assert status == 0, (what, status)
    items = skv.splitkv_plan_get_items(s.plan)
    nonempty = items[:, 5] > items[:, 4]
    assert (log[nonempty, 2] > 0).all(), what


@pytest.mark.parametrize("case", range(10))
def test_random_mla(case):
    rng = np.random.default_rng(900 + case)
    T = int(rng.integers(1, 9))
    B = int(rng.integers(1, 3))
    P = int(rng.choice([16, 32, 64, 64, 128]))
    lens = _lens(rng, B, P, T, 1500)
    sepv = bool(rng.random() < 0.5)
    fp8 = not sepv and bool(np.random.default_rng(990 + case).random() < 0.5)  # e4m3 latent cache
    w = workloads.Workload(f"rand_mla{case}", B, T, 128, 1, 576, 512, P,
                           "fp8_e4m3" if fp8 else "bf16",
                           "list:" + ":".join(str(x) for x in lens), std=0.5,
                           v_shares_k=not sepv, pool_slack=0.3, seed=950 + case)
    x = workloads.make_inputs(w, device="cuda")
    S = int(rng.choice([0, 1, 2, 5]))
    ref_o, ref_l = oracle_direct(x)
    s = DecodeSession(x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens, x.seq_lens_host,
                      scale=x.scale, kv_scale=x.kv_scale, num_splits=S, v_dim=512,
                      v_shares_k=not sepv)
    out, lse = s.run()
    compare(out, lse, ref_o, ref_l,
            what=f"MLA T={T} B={B} P={P} sepv={sepv} fp8={fp8} S={S} lens={lens}")
    assert s.stats()[1] == 0
