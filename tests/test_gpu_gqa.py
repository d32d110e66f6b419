"""GPU parity of the GQA split-KV path against the fp64 oracle, through the C-ABI.

Bars: max-abs error <= 1e-2 on bf16 outputs and <= 1e-3 on fp32 LSE; split
tables, per-CTA page ranges and the paged gather must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import split_kv_paged_splitkv_gb300 as skv
from _support import LSE_TOL, OUT_TOL, compare, need_gpu, oracle_direct, session
from split_kv_paged_splitkv_gb300.runner import DecodeSession

pytestmark = pytest.mark.gpu
W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _custom(lens, G=8, Hkv=2, T=1, P=16, fp8=False, seed=7):
    return workloads.Workload(
        "custom", len(lens), T, G * Hkv, Hkv, 128, 128, P, "fp8_e4m3" if fp8 else "bf16",
        "list:" + ":".join(str(int(x)) for x in lens), pool_slack=0.5, seed=seed)


# ------------------------------------------------------------------ gather

@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("P", [16, 64])
@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_paged_gather_is_bit_exact(fp8, P, layout):
    w = _custom([16 * 7 + 5, 3 * P + 1], P=P, fp8=fp8)
    x = workloads.make_inputs(w, device="cuda", layout=layout)
    kv_layout = skv.SPLITKV_LAYOUT_NHD if layout == "NHD" else skv.SPLITKV_LAYOUT_HND
    for b in range(2):
        L = int(x.seq_lens_host[b])
        for h in range(w.num_kv_heads):
            for which, pages in (("k", x.k_pages), ("v", x.v_pages)):
                dst = torch.zeros((L, 128), dtype=pages.dtype, device="cuda")
                skv.splitkv_debug_gather(skv.make_desc(2, 1, 16, 2, 128, 128, P, x.max_pages,
                                                       x.num_pages, int(fp8),
                                                       kv_layout=kv_layout),
                                         pages, 128, x.block_table, b, h, L, dst)
                torch.cuda.synchronize()
                ref = oracle.gather_keys(workloads.bits(pages), x.block_table[b].cpu().numpy(), L, h,
                                         layout)
                got = workloads.bits(dst)
                assert np.array_equal(got, ref), (which, b, h)


# ------------------------------------------------------------------ workloads 1 and 2

@pytest.mark.parametrize("mode", [skv.SPLITKV_COMBINE_FUSED, skv.SPLITKV_COMBINE_SEPARATE])
def test_tiny_gqa_ctx260(mode):
    x = workloads.make_inputs(W["tiny_gqa_ctx260"], device="cuda")
    ref_o, ref_l = oracle_direct(x)
    for S in (1, 4, 12):  # 12: a few rows over 9..16 splits merge in the one-pass form
        s = session(x, S, mode)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"S={S} mode={mode}")
        log, status = s.stats()
        assert status == 0


@pytest.mark.parametrize("mode", [skv.SPLITKV_COMBINE_FUSED, skv.SPLITKV_COMBINE_SEPARATE])
def test_gqa_ctx5900_split_sweep(mode):
    x = workloads.make_inputs(W["gqa_ctx5900"], device="cuda")
    ref_o, ref_l = oracle_direct(x)
    outs = []
    for S in W["gqa_ctx5900"].splits:
        s = session(x, S, mode)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"S={S}")
        outs.append(out.float().cpu().numpy())
        log, status = s.stats()
        assert status == 0
    # split invariance on the GPU itself
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= OUT_TOL


@pytest.mark.parametrize("mode", [skv.SPLITKV_COMBINE_FUSED, skv.SPLITKV_COMBINE_SEPARATE])
def test_spec_t4_gqa_ctx5900(mode):
    """Four speculative tokens of each G = 8 group over the 5.9k context (32
    query rows per KV head): every split count of the workload against the
    oracle, and the splits agree with one another."""
    x = workloads.make_inputs(W["spec_t4_gqa_ctx5900"], device="cuda")
    ref_o, ref_l = oracle_direct(x)
    for S in W["spec_t4_gqa_ctx5900"].splits:
        s = session(x, S, mode)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"T=4 S={S} mode={mode}")
        log, status = s.stats()
        assert status == 0 and (log[:, 2] > 0).all()


def test_split_ranges_and_nonempty_ctas():
    """Every launched CTA iterated exactly its planned page range and scored keys."""
    x = workloads.make_inputs(W["gqa_ctx5900"], device="cuda")
    for S in (1, 2, 4, 8, 16, 32, 64, 0):
        s = session(x, S, skv.SPLITKV_COMBINE_FUSED)  # fused: the merging CTA is logged
        s.run()
        log, status = s.stats()
        items = skv.splitkv_plan_get_items(s.plan)
        ref = np.array(oracle.plan_items(list(x.seq_lens_host), 16, 2, S, _sms(), ctas_per_sm=3),
                       np.int32)
        assert np.array_equal(items[:, :6], ref)
        assert np.array_equal(log[:, 0], items[:, 4]) and np.array_equal(log[:, 1], items[:, 5])
        n_pages = 369
        expect_keys = np.minimum(items[:, 5] * 16, 5900) - items[:, 4] * 16
        assert np.array_equal(log[:, 2], expect_keys)
        assert (log[:, 2] > 0).all()  # non-empty fraction = 1.0
        if S:
            assert len(items) == 2 * min(S, n_pages)
        assert status == 0
        # fused merge log: bit 0 = wrote the group's output, bit 1 = merged a
        # bundle of up to 8 consecutive splits (groups of more than 8 splits)
        split_items = items[items[:, 3] > 1]
        if len(split_items):
            groups = np.unique(split_items[:, 7])
            assert (log[:, 3] & 1).sum() == len(groups)
            bundles = sum(-(-int(split_items[split_items[:, 7] == g][0, 3]) // 8)
                          for g in groups if split_items[split_items[:, 7] == g][0, 3] > 8)
            assert ((log[:, 3] >> 1) & 1).sum() == bundles


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


# ------------------------------------------------------------------ ragged and edge cases

@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("G,Hkv", [(8, 2), (4, 2), (1, 3), (2, 1)])
@pytest.mark.parametrize("P", [16, 32, 64, 128])
def test_ragged_lengths(fp8, G, Hkv, P):
    lens = [1, 15, 16, 17, 255, 257, 1000, 0, 3 * P, 2 * P + 1]
    w = _custom(lens, G=G, Hkv=Hkv, P=P, fp8=fp8, seed=G * 10 + Hkv + P)
    x = workloads.make_inputs(w, device="cuda")
    ref_o, ref_l = oracle_direct(x)
    for S in (1, 3, 0):
        for mode in (0, 1):
            s = session(x, S, mode)
            out, lse = s.run()
            compare(out, lse, ref_o, ref_l, what=f"S={S} mode={mode}")
            log, status = s.stats()
            assert status == 0
            items = skv.splitkv_plan_get_items(s.plan)
            nonempty = items[:, 5] > items[:, 4]
            assert (log[nonempty, 2] > 0).all()


@pytest.mark.parametrize("T,G", [(2, 4), (8, 1), (4, 2), (3, 2),
                                 (2, 8), (4, 4), (3, 5), (16, 1), (5, 2),
                                 (3, 8), (4, 8), (6, 4), (16, 2), (5, 6)])
@pytest.mark.parametrize("fp8", [False, True])
def test_multi_token_causal(T, G, fp8):
    """Speculative decode: T query tokens, causal among themselves; T*G > 8
    takes the two-row-group kernel (query rows 8..15 of a KV head), T*G > 16
    the four-row-group one (up to 32 rows)."""
    lens = [T, T + 1, 37, 300, 16 * 5]
    w = _custom(lens, G=G, Hkv=2, T=T, fp8=fp8, seed=T * 7 + G)
    x = workloads.make_inputs(w, device="cuda")
    ref_o, ref_l = oracle_direct(x)
    # num_sms = 1 makes every plan of more than one item take the two-stage
    # (several CTAs per SM) kernel form; 0 plans for the device (one wave here)
    for sms in (0, 1):
        for S in (1, 2, 5):
            for mode in ((1, 0) if S == 5 else (1,)):
                s = session(x, S, mode, num_sms=sms)
                out, lse = s.run()
                compare(out, lse, ref_o, ref_l, what=f"T={T} G={G} S={S} mode={mode} sms={sms}")
                assert s.stats()[1] == 0


@pytest.mark.parametrize("T,G,Hkv", [(1, 8, 4), (1, 4, 8), (2, 8, 2), (1, 2, 3)])
def test_per_head_kv_scales(T, G, Hkv):
    """e4m3 cache with its own K and V scale per KV head (splitkv_decode_kv_scales),
    against the oracle dequantising K and V with those scales; also separate
    per-tensor K and V scales (all heads equal)."""
    w = _custom([T + 3, 233, 1000, 16 * 9], G=G, Hkv=Hkv, T=T, fp8=True, seed=40 + Hkv)
    x = workloads.make_inputs(w, device="cuda")
    rng = np.random.default_rng(Hkv * 10 + G)
    # at most the cache's own quantisation scale, so values keep the N(0, 1)
    # magnitude the absolute bf16 output bar is set for (one bf16 ulp is
    # 2^-5 for |out| in [4, 8))
    c = float(x.kv_scale)
    per_head = (c * rng.uniform(0.4, 1.0, Hkv), c * rng.uniform(0.4, 1.0, Hkv))
    per_tensor = (np.full(Hkv, 0.9 * c), np.full(Hkv, 0.6 * c))
    for ks, vs in (per_head, per_tensor):
        ref_o, ref_l = oracle.attention_direct(
            workloads.bits(x.q), workloads.bits(x.k_pages), workloads.bits(x.v_pages),
            x.block_table.cpu().numpy(), x.seq_lens_host, scale=x.scale, kv_dtype="fp8_e4m3",
            k_scale=ks.astype(np.float32).astype(np.float64),
            v_scale=vs.astype(np.float32).astype(np.float64))
        kt = torch.tensor(ks, dtype=torch.float32, device="cuda")
        vt = torch.tensor(vs, dtype=torch.float32, device="cuda")
        for S, mode in ((1, 1), (3, 1), (0, 0)):
            s = DecodeSession(x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens,
                              x.seq_lens_host, scale=x.scale, num_splits=S, combine_mode=mode,
                              k_scale=kt, v_scale=vt)
            out, lse = s.run()
            compare(out, lse, ref_o, ref_l, what=f"T={T} G={G} Hkv={Hkv} S={S}")
            assert s.stats()[1] == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_thirty_two_rows_per_head_long_context(fp8):
    """T*G = 32 (four tokens of a G = 8 group) over a long context with the
    planner's splits, one-wave and multi-wave grids."""
    for lens, Hkv in (([2048 + 9, 700, 16], 4), ([4000, 3000, 2500, 1800, 1200, 900, 600, 33], 8)):
        w = _custom(lens, G=8, Hkv=Hkv, T=4, fp8=fp8, seed=93 + Hkv)
        x = workloads.make_inputs(w, device="cuda")
        ref_o, ref_l = oracle_direct(x)
        s = session(x, 0)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"T=4 G=8 Hkv={Hkv} planner")
        assert s.stats()[1] == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_sixteen_rows_per_head_long_context(fp8):
    """T*G = 16 over a long context with the planner's splits: many tiles per
    warp, both row groups, merged partials."""
    w = _custom([2048 + 9, 700, 16], G=8, Hkv=4, T=2, fp8=fp8, seed=91)
    x = workloads.make_inputs(w, device="cuda")
    ref_o, ref_l = oracle_direct(x)
    s = session(x, 0)
    out, lse = s.run()
    compare(out, lse, ref_o, ref_l, what="T=2 G=8 Hkv=4 planner")
    log, status = s.stats()
    assert status == 0 and (log[:, 2] > 0).all()


@pytest.mark.parametrize("T,G,Hkv,fp8", [(1, 8, 2, False), (2, 8, 2, False), (1, 8, 3, True),
                                          (1, 8, 2, True), (2, 8, 2, True)])
def test_both_ring_depths(T, G, Hkv, fp8):
    """A grid of at most one CTA per SM runs the four-stage ring, a larger one
    the two-stage ring; a plan for a 4-SM machine forces the latter.  Covers
    each kernel instantiation: bf16 with one and two row groups, e4m3 with one
    and two KV heads per item, e4m3 with two row groups."""
    w = _custom([T + 1, 333, 1500, 16 * 7 + 3, 900], G=G, Hkv=Hkv, T=T, fp8=fp8, seed=T + G + Hkv)
    x = workloads.make_inputs(w, device="cuda")
    ref_o, ref_l = oracle_direct(x)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for num_sms, S in ((0, 2), (4, 6)):
        s = session(x, S, 1, num_sms=num_sms)
        n_items = skv.splitkv_plan_get_items(s.plan).shape[0]
        assert (n_items <= sms) if num_sms == 0 else (n_items > num_sms)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"T={T} G={G} Hkv={Hkv} num_sms={num_sms}")
        assert s.stats()[1] == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_items_longer_than_the_block_table_staging_chunk(fp8):
    """One split over 1,250+ pages: every producer warp restages the item's
    block-table entries chunk by chunk (1,024 at a time) mid-item, in the
    one-wave four-stage form (four producer warps) and, with a plan for four
    SMs, the two-stage form."""
    lens = [16 * 1250 + 5, 16 * 1100, 37]
    w = _custom(lens, G=8, Hkv=2, fp8=fp8, seed=17 + fp8)
    x = workloads.make_inputs(w, device="cuda")
    ref_o, ref_l = oracle_direct(x)
    for S, num_sms in ((1, 0), (1, 4), (2, 0)):
        s = session(x, S, 1, num_sms=num_sms)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"fp8={fp8} S={S} num_sms={num_sms}")
        log, status = s.stats()
        assert status == 0 and (log[:, 2] > 0).all()


@pytest.mark.parametrize("T,G,Hkv,fp8,P", [(1, 8, 2, False, 16), (2, 8, 2, False, 32),
                                            (1, 4, 3, False, 64), (1, 8, 4, True, 16),
                                            (1, 2, 3, True, 32), (2, 8, 2, True, 16)])
def test_nhd_pages(T, G, Hkv, fp8, P):
    """Pages stored NHD ([N][P][Hkv][D]) against the oracle reading the same
    layout, and bit-identical to the same values stored HND (the kernel's
    shared-memory tiles are the same in both)."""
    lens = [T, T + 16, 255, 1000, 0, 16 * 9 + 3]
    w = _custom(lens, G=G, Hkv=Hkv, T=T, fp8=fp8, P=P, seed=3 * T + G + Hkv)
    xn = workloads.make_inputs(w, device="cuda", layout="NHD")
    xh = workloads.make_inputs(w, device="cuda")
    assert xn.k_pages.shape[1] == w.page_size and xn.k_pages.shape[2] == Hkv
    ref_o, ref_l = oracle_direct(xn)
    for S, mode in ((1, 1), (3, 1), (0, 1), (5, 0)):
        sn = session(xn, S, mode)
        out_n, lse_n = sn.run()
        compare(out_n, lse_n, ref_o, ref_l, what=f"NHD T={T} G={G} Hkv={Hkv} S={S} mode={mode}")
        assert sn.stats()[1] == 0
        out_h, lse_h = session(xh, S, mode).run()
        assert torch.equal(out_n, out_h) and torch.equal(lse_n, lse_h)


# ------------------------------------------------------------------ workloads 3 and 5

def test_fp8_batch8_ctx32k_full():
    x = workloads.make_inputs(W["fp8_batch8_ctx32k"], device="cuda")
    ref_o, ref_l = oracle_direct(x)
    for mode in (0, 1):
        s = session(x, 0, mode)
        out, lse = s.run()
        compare(out, lse, ref_o, ref_l, what=f"mode={mode}")
        log, status = s.stats()
        assert status == 0 and (log[:, 2] > 0).all()


@pytest.mark.parametrize("name", ["mixed_batch32_bf16", "mixed_batch32_fp8"])
def test_mixed_batch32_full(name):
    """Full-size run (32 sequences of 256 to 131,072 keys, planner splits),
    every output row of every sequence against the oracle."""
    w = W[name]
    x = workloads.make_inputs(w, device="cuda")
    s = session(x, 0)
    out, lse = s.run()
    log, status = s.stats()
    assert status == 0 and (log[:, 2] > 0).all()
    ref_o, ref_l = oracle_direct(x)
    compare(out, lse, ref_o, ref_l, what=name)


# ------------------------------------------------------------------ query magnitudes (e4m3)

@pytest.mark.parametrize("T,G", [(1, 8), (2, 8), (1, 4), (4, 8)])
def test_e4m3_queries_of_any_bf16_magnitude(T, G):
    """The e4m3 path multiplies bf16 queries with f16 tensor-core products;
    each query row is scaled by a power of two into f16's range first.  Rows
    drawn at |q| ~ 1e5 (beyond f16's largest value), ~1e-6 (below its
    normal range), ~1 and with components spread over 2^-20 .. 2^16 in one
    row must match the oracle; K carries per-head scales that keep every
    row's scores of order one, so the softmax is not trivially flat."""
    lens = [T + 2, 300, 1000, 16 * 7]
    w = _custom(lens, G=G, Hkv=2, T=T, fp8=True, seed=80 + T + G)
    x = workloads.make_inputs(w, device="cuda")
    c = float(x.kv_scale)
    rng = np.random.default_rng(T * 10 + G)
    for mag in (1e5, 1e-6, "spread"):
        q = x.q.float().clone()
        if mag == "spread":
            # per component 2^e, e uniform in [-20, 16], random sign: row maxima
            # around 2^16 (> 65,504) with tiny components alongside
            e = torch.from_numpy(rng.uniform(-20, 16, size=tuple(q.shape))).float().to(q.device)
            q = torch.sign(q) * torch.exp2(e)
            kscale = c / 2.0 ** 16
        else:
            q = q * mag
            kscale = c / mag
        q = q.to(torch.bfloat16)
        ks = np.full(2, kscale, np.float32)
        vs = np.full(2, c, np.float32)
        ref_o, ref_l = oracle.attention_direct(
            workloads.bits(q), workloads.bits(x.k_pages), workloads.bits(x.v_pages),
            x.block_table.cpu().numpy(), x.seq_lens_host, scale=x.scale, kv_dtype="fp8_e4m3",
            k_scale=ks.astype(np.float64), v_scale=vs.astype(np.float64))
        kt = torch.tensor(ks, device="cuda")
        vt = torch.tensor(vs, device="cuda")
        for S in (1, 3):
            sess = DecodeSession(q, x.k_pages, x.v_pages, x.block_table, x.seq_lens,
                                 x.seq_lens_host, scale=x.scale, num_splits=S, k_scale=kt,
                                 v_scale=vt)
            out, lse = sess.run()
            compare(out, lse, ref_o, ref_l, what=f"|q| {mag} T={T} G={G} S={S}")
            assert sess.stats()[1] == 0
        # the per-tensor scale path with the same magnitudes: K and V share
        # kv_scale, so the outputs scale with it; compare relative to the
        # output's own size
        if mag != "spread":
            ref_o2, ref_l2 = oracle.attention_direct(
                workloads.bits(q), workloads.bits(x.k_pages), workloads.bits(x.v_pages),
                x.block_table.cpu().numpy(), x.seq_lens_host, scale=x.scale, kv_dtype="fp8_e4m3",
                kv_scale=float(np.float32(kscale)))
            sess = DecodeSession(q, x.k_pages, x.v_pages, x.block_table, x.seq_lens,
                                 x.seq_lens_host, scale=x.scale, kv_scale=kscale, num_splits=3)
            out, lse = sess.run()
            o = out.float().cpu().numpy()
            assert np.isfinite(o).all()
            peak = np.abs(ref_o2).max()
            assert np.abs(o - ref_o2).max() <= 1e-2 * peak, mag
            assert np.abs(lse.cpu().numpy() - ref_l2).max() <= LSE_TOL, mag


# ------------------------------------------------------------------ out-of-range page ids

@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("S", [1, 3, 0])
def test_out_of_range_page_ids_are_flagged(fp8, S):
    """A block-table entry >= num_pages and a negative one: the kernel reads
    page 0 in their place (never outside the pool), sets
    SPLITKV_DEVERR_PAGE in the status word, keeps the output finite, and the
    sequences whose tables are intact still match the oracle."""
    # lengths are whole pages, so no page (page 0 included) holds the poisoned
    # tail slots a partly filled last page carries
    w = _custom([304, 704, 1008, 208], G=8, Hkv=4, fp8=fp8, seed=95 + fp8)
    x = workloads.make_inputs(w, device="cuda")
    ref_o, ref_l = oracle_direct(x)
    bad = x.block_table.clone()
    bad[1, 5] = x.num_pages + 7
    bad[3, 2] = -4
    s = session(x, S)
    out, lse = s.run(tensors=(x.q, x.k_pages, x.v_pages, bad, x.seq_lens))
    log, status = s.stats()
    assert status & skv.SPLITKV_DEVERR_PAGE
    assert not status & skv.SPLITKV_DEVERR_TIMEOUT
    assert torch.isfinite(out.float()).all()
    rows = [(b, 0, h) for b in (0, 2) for h in range(w.num_q_heads)]
    compare(out, lse, ref_o, ref_l, rows=rows, what=f"intact sequences fp8={fp8} S={S}")
    # the status word is sticky until the next upload; a clean call after a
    # fresh upload reports nothing
    s2 = session(x, S)
    s2.run()
    assert s2.stats()[1] == 0


# ------------------------------------------------------------------ combine

def test_combine_matches_oracle_and_is_associative():
    rng = np.random.default_rng(3)
    S, R, D = 5, 7, 128
    o = rng.standard_normal((S, R, D)).astype(np.float32)
    l = (rng.standard_normal((S, R)) * 4).astype(np.float32)
    l[1, 2] = -np.inf
    l[:, 5] = -np.inf  # an all-empty row
    od = torch.from_numpy(o).cuda()
    ld = torch.from_numpy(l).cuda()

    def comb(o_, l_):
        n = o_.shape[0]
        out = torch.empty((R, D), dtype=torch.float32, device="cuda")
        lo = torch.empty(R, dtype=torch.float32, device="cuda")
        skv.splitkv_combine(o_.contiguous(), l_.contiguous(), n, R, D, None, out, lo)
        return out, lo

    full_o, full_l = comb(od, ld)
    torch.cuda.synchronize()
    for r in range(R):
        ro, rl = oracle.combine([(o[s, r].astype(np.float64), float(l[s, r])) for s in range(S)])
        assert np.abs(full_o[r].cpu().numpy() - ro).max() < 1e-5
        if np.isfinite(rl):
            assert abs(full_l[r].item() - rl) < 1e-5
        else:
            assert full_l[r].item() == -np.inf and (full_o[r] == 0).all()
    # ((0,1),2,3,4) == (0,1,2,3,4) and permutation invariance
    a_o, a_l = comb(od[:2], ld[:2])
    left_o, left_l = comb(torch.cat([a_o[None], od[2:]]), torch.cat([a_l[None], ld[2:]]))
    perm = [3, 0, 4, 2, 1]
    p_o, p_l = comb(od[perm], ld[perm])
    fin = torch.isfinite(full_l)
    for oo, ll in ((left_o, left_l), (p_o, p_l)):
        assert (oo - full_o).abs().max().item() < 1e-5
        assert (ll[fin] - full_l[fin]).abs().max().item() < 1e-5
    # -inf partial is the identity
    e_o, e_l = comb(torch.cat([od[:1], torch.zeros_like(od[:1])]),
                    torch.cat([ld[:1], torch.full_like(ld[:1], -np.inf)]))
    one_o, one_l = comb(od[:1], ld[:1])
    assert (e_o - one_o).abs().max().item() == 0 and torch.equal(e_l, one_l)


# ------------------------------------------------------------------ status word

def test_seq_len_mismatch_is_reported():
    x = workloads.make_inputs(W["tiny_gqa_ctx260"], device="cuda")
    s = session(x, 4)
    wrong = x.seq_lens.clone()
    wrong[0] -= 3
    s.run(tensors=(x.q, x.k_pages, x.v_pages, x.block_table, wrong))
    _, status = s.stats()
    assert status & skv.SPLITKV_DEVERR_SEQLEN


@pytest.mark.parametrize("S,R,D", [(200, 3, 512), (70, 2, 96), (1, 4, 128), (64, 5, 128),
                                   (16, 6, 512), (17, 3, 128), (12, 768, 512), (9, 2, 128),
                                   (13, 1100, 128)])
def test_combine_many_parts_and_widths(S, R, D):
    """More splits than one load round covers (running maximum across chunks),
    V widths that are not a multiple of 128, a single part, and -inf rows."""
    rng = np.random.default_rng(S * 7 + D)
    o = rng.standard_normal((S, R, D)).astype(np.float32)
    l = (rng.standard_normal((S, R)) * 6).astype(np.float32)
    l[rng.random((S, R)) < 0.2] = -np.inf
    l[:, 0] = -np.inf if S > 1 else l[:, 0]
    out = torch.empty((R, D), dtype=torch.float32, device="cuda")
    lo = torch.empty(R, dtype=torch.float32, device="cuda")
    skv.splitkv_combine(torch.from_numpy(o).cuda(), torch.from_numpy(l).cuda(), S, R, D, None, out, lo)
    torch.cuda.synchronize()
    for r in range(R):
        ro, rl = oracle.combine([(o[s, r].astype(np.float64), float(l[s, r])) for s in range(S)])
        assert np.abs(out[r].cpu().numpy() - ro).max() < 1e-5
        if np.isfinite(rl):
            assert abs(lo[r].item() - rl) < 1e-5
        else:
            assert lo[r].item() == -np.inf
