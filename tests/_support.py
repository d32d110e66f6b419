"""Shared helpers for the GPU tests: run the library and the oracle on one input."""
import numpy as np
import torch

import oracle
import split_kv_paged_splitkv_gb300 as skv
import workloads
from split_kv_paged_splitkv_gb300.runner import DecodeSession

OUT_TOL = 1e-2  # max-abs error on bf16 outputs
LSE_TOL = 1e-3  # max-abs error on fp32 LSE


def need_gpu():
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def oracle_direct(x: workloads.Inputs, rows=None):
    w = x.w
    return oracle.attention_direct(
        workloads.bits(x.q), workloads.bits(x.k_pages),
        None if x.v_pages is None else workloads.bits(x.v_pages),
        x.block_table.cpu().numpy(), x.seq_lens_host, scale=x.scale, kv_dtype=w.kv_dtype,
        kv_scale=x.kv_scale, v_dim=w.v_dim, v_shares_k=w.v_shares_k, rows=rows,
        layout=x.layout)


def session(x: workloads.Inputs, num_splits=0, combine_mode=1, num_sms=0):
    return DecodeSession(x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens, x.seq_lens_host,
                         scale=x.scale, kv_scale=x.kv_scale, num_splits=num_splits,
                         num_sms=num_sms, v_dim=x.w.v_dim, v_shares_k=x.w.v_shares_k,
                         combine_mode=combine_mode,
                         kv_layout=skv.SPLITKV_LAYOUT_NHD if x.layout == "NHD" else skv.SPLITKV_LAYOUT_HND)


def compare(out, lse, ref_o, ref_l, rows=None, what=""):
    """Max-abs errors over all rows (or the given (b, t, h) rows); asserts the bar."""
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    if rows is not None:
        idx = tuple(np.array(rows).T)
        o, l, ref_o, ref_l = o[idx], l[idx], ref_o[idx], ref_l[idx]
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), f"{what}: -inf LSE pattern differs"
    eo = float(np.abs(o - ref_o).max()) if o.size else 0.0
    el = float(np.abs(l[fin] - ref_l[fin]).max()) if fin.any() else 0.0
    assert eo <= OUT_TOL, f"{what}: max |out - oracle| = {eo:.3e} > {OUT_TOL}"
    assert el <= LSE_TOL, f"{what}: max |lse - oracle| = {el:.3e} > {LSE_TOL}"
    return eo, el
