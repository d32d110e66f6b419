"""Host-side checks of the C-ABI library (no GPU needed).

* the library loads and exports every function ``include/splitkv.h`` declares;
* the planner's work list equals the oracle's restatement, exactly;
* argument validation returns the documented status codes before any CUDA call.
"""
import ctypes

import numpy as np
import pytest

import __graft_entry__

__graft_entry__.build()

import split_kv_paged_splitkv_gb300 as skv  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402


def test_library_exports_every_declared_function():
    names = skv.header_functions()
    assert "splitkv_decode" in names and "splitkv_plan" in names
    lib = ctypes.CDLL(skv.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def _desc(B=1, T=1, Hq=16, Hkv=2, D=128, Dv=128, P=16, maxp=512, N=600, fp8=False, mla=False,
          mode=0):
    return skv.make_desc(B, T, Hq, Hkv, D, Dv, P, maxp, N,
                         skv.SPLITKV_FP8_E4M3 if fp8 else skv.SPLITKV_BF16, int(mla), mode)


# Resident CTAs per SM the library's planner counts on for the GQA kernel
# (launch bounds and shared memory of the kernel allow three).
GQA_CTAS_PER_SM = 3


def _expected_hpi(Hkv, fp8, rows_per_head=8):
    if not fp8 or rows_per_head > 16:
        return 1
    return 2 if Hkv % 2 == 0 else 1


def _oracle_items(lens, P, Hkv, S, sms, hpi=1):
    return np.array(oracle.plan_items(list(lens), P, Hkv, S, sms, ctas_per_sm=GQA_CTAS_PER_SM,
                                      heads_per_item=hpi), dtype=np.int32).reshape(-1, 6)


def _check_plan(lens, P, Hkv, S, sms, Hq=None, fp8=False):
    maxp = max(1, max(-(-int(L) // P) for L in lens))
    d = _desc(B=len(lens), Hq=Hkv * (8 if Hq is None else Hq // Hkv), Hkv=Hkv, P=P, maxp=maxp,
              N=max(1, sum(-(-int(L) // P) for L in lens)), fp8=fp8)
    plan = skv.splitkv_plan(d, np.array(lens, np.int32), S, sms)
    hpi = skv.splitkv_plan_heads_per_item(plan)
    assert hpi == _expected_hpi(Hkv, fp8)
    items = skv.splitkv_plan_get_items(plan)
    ref = _oracle_items(lens, P, Hkv, S, sms, hpi)
    assert items.shape[0] == ref.shape[0]
    assert np.array_equal(items[:, :6], ref), (lens, S)
    # the split table per KV head: every head of an item, (b, h_kv, s, p0, p1)
    ranges = skv.splitkv_plan_get_ranges(plan)
    ref_rows = np.array([(b, h0 + hh, s_, p0, p1) for (b, h0, s_, _, p0, p1) in ref
                         for hh in range(hpi)], dtype=np.int32).reshape(-1, 5)
    assert np.array_equal(ranges, ref_rows), (lens, S)
    return items


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16, 32, 64, 0])
def test_plan_matches_oracle_gqa_ctx5900(S):
    items = _check_plan([5900], 16, 2, S, 148)
    n = 369
    if S:
        assert items.shape[0] == 2 * min(S, n)
    assert (items[:, 5] > items[:, 4]).all()


@pytest.mark.parametrize("w", ["tiny_gqa_ctx260", "fp8_batch8_ctx32k", "mixed_batch32_bf16",
                               "mixed_batch32_fp8"])
@pytest.mark.parametrize("sms", [148, 152])
def test_plan_matches_oracle_workloads(w, sms):
    wl = workloads.WORKLOADS[w]
    lens = workloads.draw_seq_lens(wl, np.random.default_rng(wl.seed))
    for S in wl.splits:
        _check_plan(lens, wl.page_size, wl.num_kv_heads, S, sms, fp8=wl.kv_dtype == "fp8_e4m3")


def test_plan_matches_oracle_random_batches():
    rng = np.random.default_rng(123)
    for trial in range(40):
        B = int(rng.integers(1, 12))
        lens = rng.integers(0, 3000, size=B)
        lens[rng.random(B) < 0.1] = 0
        P = int(rng.choice([16, 32, 64]))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        S = int(rng.choice([0, 0, 1, 3, 7, 64]))
        sms = int(rng.choice([1, 7, 148, 152]))
        _check_plan(list(lens), P, Hkv, S, sms, fp8=bool(rng.random() < 0.5))


def test_plan_slots_and_groups_are_consistent():
    lens = [260, 5900, 16, 0, 1000]
    d = _desc(B=5, maxp=400, N=1000)
    plan = skv.splitkv_plan(d, np.array(lens, np.int32), 4, 148)
    it = skv.splitkv_plan_get_items(plan)
    for row in it:
        b, h, s, S, p0, p1, slot, group = row
        if S == 1:
            assert slot == -1 and group == -1
        else:
            assert slot >= 0 and group >= 0
    multi = it[it[:, 3] > 1]
    # slots of one group are contiguous and start at a multiple... each group owns S slots
    for g in np.unique(multi[:, 7]):
        rows = multi[multi[:, 7] == g]
        slots = np.sort(rows[:, 6])
        assert np.array_equal(slots, np.arange(slots[0], slots[0] + rows[0, 3]))
        assert np.array_equal(np.sort(rows[:, 2]), np.arange(rows[0, 3]))
    assert skv.splitkv_workspace_size(plan) > 0


@pytest.mark.parametrize("bad,code", [
    (dict(P=8), skv.SPLITKV_EINVAL),
    (dict(Hq=15), skv.SPLITKV_EINVAL),
    (dict(D=96, Dv=96), skv.SPLITKV_EUNSUPPORTED),
    (dict(T=5, Hq=16, Hkv=2), skv.SPLITKV_EUNSUPPORTED),  # 5 * 8 query rows per KV head > 32
    (dict(N=0), skv.SPLITKV_EINVAL),
])
def test_plan_rejects_bad_descriptors(bad, code):
    d = _desc(**bad)
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_plan(d, np.array([100], np.int32), 1, 148)
    assert e.value.status == code


def test_mla_with_separate_v_is_planned():
    """The MLA shapes plan alike whether V shares the latent rows or not."""
    lens = np.array([5000], np.int32)
    items = []
    for vsk in (1, 0):
        d = skv.make_desc(1, 6, 128, 1, 576, 512, 64, 128, 200, skv.SPLITKV_BF16, vsk)
        items.append(skv.splitkv_plan_get_items(skv.splitkv_plan(d, lens, 4, 148)))
    assert np.array_equal(items[0], items[1])


def test_mla_e4m3_latent_cache_is_planned_and_separate_e4m3_v_is_not():
    """An e4m3 latent cache (V in its rows) plans like the bf16 one; an e4m3
    cache with a separate V tensor has no kernel."""
    lens = np.array([5000], np.int32)
    d16 = skv.make_desc(1, 6, 128, 1, 576, 512, 64, 128, 200, skv.SPLITKV_BF16, 1)
    d8 = skv.make_desc(1, 6, 128, 1, 576, 512, 64, 128, 200, skv.SPLITKV_FP8_E4M3, 1)
    assert np.array_equal(skv.splitkv_plan_get_items(skv.splitkv_plan(d16, lens, 4, 148)),
                          skv.splitkv_plan_get_items(skv.splitkv_plan(d8, lens, 4, 148)))
    d8v = skv.make_desc(1, 6, 128, 1, 576, 512, 64, 128, 200, skv.SPLITKV_FP8_E4M3, 0)
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_plan(d8v, lens, 4, 148)
    assert e.value.status == skv.SPLITKV_EUNSUPPORTED


@pytest.mark.parametrize("P,ok", [(16, True), (32, True), (64, True), (128, True), (192, True),
                                  (48, False), (80, False)])
def test_mla_page_sizes(P, ok):
    """The MLA kernel streams 64-key blocks: pages of 16 or 32 keys (several
    per block) or of a multiple of 64 keys (whole blocks per page)."""
    d = skv.make_desc(1, 2, 128, 1, 576, 512, P, 64 * 64 // P + 1, 8 * 64 * 64 // P,
                      skv.SPLITKV_BF16, 1)
    lens = np.array([64 * 64], np.int32)
    if ok:
        it = skv.splitkv_plan_get_items(skv.splitkv_plan(d, lens, 4, 148))
        assert it[:, 5].max() * P >= 64 * 64
    else:
        with pytest.raises(skv.SplitKVError) as e:
            skv.splitkv_plan(d, lens, 4, 148)
        assert e.value.status == skv.SPLITKV_EUNSUPPORTED


def test_two_step_entry_points_validate_before_any_cuda_call():
    plan = skv.splitkv_plan(_desc(B=1), np.array([300], np.int32), 2, 148)
    A = 1 << 20  # aligned, never dereferenced: validation fails first
    assert skv._lib.splitkv_combine_workspace(None, A, A, A, None) == skv.SPLITKV_EINVAL
    assert skv._lib.splitkv_combine_workspace(plan.handle, None, A, A, None) == skv.SPLITKV_EWORKSPACE
    assert skv._lib.splitkv_combine_workspace(plan.handle, A, None, A, None) == skv.SPLITKV_EINVAL
    assert skv._lib.splitkv_combine_workspace(plan.handle, A + 8, A, A, None) == skv.SPLITKV_EINVAL
    assert skv._lib.splitkv_combine_workspace(plan.handle, A, A, A + 2, None) == skv.SPLITKV_EINVAL
    st = skv._lib.splitkv_decode_partials(plan.handle, A, A, A, A, A, A, 0, 0.1, 1.0, None, None,
                                          None)
    assert st == skv.SPLITKV_EINVAL  # out is NULL


def test_kv_layout_field():
    """Both page layouts plan alike (the split table does not depend on the
    layout); any other value is rejected."""
    lens = np.array([700, 33], np.int32)
    items = []
    for layout in (skv.SPLITKV_LAYOUT_HND, skv.SPLITKV_LAYOUT_NHD):
        d = _desc(B=2)
        d.kv_layout = layout
        items.append(skv.splitkv_plan_get_items(skv.splitkv_plan(d, lens, 3, 148)))
    assert np.array_equal(items[0], items[1])
    d = _desc(B=2)
    d.kv_layout = 2
    with pytest.raises(skv.SplitKVError) as e:
        skv.splitkv_plan(d, lens, 3, 148)
    assert e.value.status == skv.SPLITKV_EINVAL


def test_plan_rejects_bad_lengths_and_splits():
    d = _desc(maxp=4)
    for lens, S in (([65], 1), ([-1], 1), ([10], 65), ([10], -1)):
        with pytest.raises(skv.SplitKVError) as e:
            skv.splitkv_plan(d, np.array(lens, np.int32), S, 148)
        assert e.value.status == skv.SPLITKV_EINVAL
    d2 = _desc(T=4, Hq=8, Hkv=4, maxp=4)
    with pytest.raises(skv.SplitKVError):
        skv.splitkv_plan(d2, np.array([3], np.int32), 1, 148)  # shorter than q_tokens


def test_decode_validates_before_any_cuda_call():
    d = _desc()
    plan = skv.splitkv_plan(d, np.array([100], np.int32), 2, 148)
    A = 1 << 20  # 16-byte aligned fake addresses; validation fails before use
    cases = [
        dict(workspace=None),
        dict(q=None),
        dict(q=A + 8),
        dict(num_splits=3),
        dict(scale=0.0),
    ]
    base = dict(workspace=A, q=A, k=A, v=A, table=A, lens=A, num_splits=2, scale=0.1,
                kv_scale=1.0, out=A, lse=A)
    for c in cases:
        args = dict(base)
        args.update(c)
        st = skv._lib.splitkv_decode(plan.handle, args["workspace"], args["q"], args["k"],
                                     args["v"], args["table"], args["lens"], args["num_splits"],
                                     args["scale"], args["kv_scale"], args["out"], args["lse"], None)
        assert st in (skv.SPLITKV_EINVAL, skv.SPLITKV_EWORKSPACE), (c, st)
        assert skv.splitkv_last_error()


def test_heads_per_item_is_one_above_sixteen_rows_per_head():
    for T, G, want in ((1, 8, 2), (2, 8, 2), (3, 4, 2), (2, 4, 2), (3, 8, 1), (4, 8, 1)):
        d = _desc(T=T, Hq=8 * G, Hkv=8, fp8=True)
        plan = skv.splitkv_plan(d, np.array([300], np.int32), 0, 148)
        assert skv.splitkv_plan_heads_per_item(plan) == _expected_hpi(8, True, T * G) == want


def test_decode_kv_scales_validates_before_any_cuda_call():
    A = 1 << 20
    fp8_plan = skv.splitkv_plan(_desc(fp8=True), np.array([100], np.int32), 2, 148)
    bf16_plan = skv.splitkv_plan(_desc(), np.array([100], np.int32), 2, 148)
    cases = [
        (fp8_plan, dict(ks=None), skv.SPLITKV_EINVAL),
        (fp8_plan, dict(vs=None), skv.SPLITKV_EINVAL),
        (fp8_plan, dict(ks=A + 2), skv.SPLITKV_EINVAL),
        (bf16_plan, dict(), skv.SPLITKV_EUNSUPPORTED),
        (fp8_plan, dict(q=None), skv.SPLITKV_EINVAL),
    ]
    for plan, c, code in cases:
        args = dict(q=A, ks=A, vs=A)
        args.update(c)
        st = skv._lib.splitkv_decode_kv_scales(plan.handle, A, args["q"], A, A, A, A, 2, 0.1,
                                               args["ks"], args["vs"], A, A, None)
        assert st == code, (c, st)
        assert skv.splitkv_last_error()


def test_fixed_plan_template_and_layout():
    """A capacity plan holds num_splits items per (sequence, head group), in
    (b, head group, s) order, all unused until the device refresh."""
    for fp8, Hkv, want_hpi in ((False, 2, 1), (True, 8, 2)):
        d = _desc(B=3, Hq=8 * Hkv, Hkv=Hkv, fp8=fp8, mode=skv.SPLITKV_COMBINE_SEPARATE)
        plan = skv.splitkv_plan_fixed(d, 4)
        assert skv.splitkv_plan_heads_per_item(plan) == want_hpi
        U = Hkv // want_hpi
        items = skv.splitkv_plan_get_items(plan)
        assert items.shape == (3 * U * 4, 8)
        b, u, s_ = np.meshgrid(np.arange(3), np.arange(U), np.arange(4), indexing="ij")
        assert np.array_equal(items[:, 0], b.ravel())
        assert np.array_equal(items[:, 1], u.ravel() * want_hpi)
        assert np.array_equal(items[:, 2], s_.ravel())
        assert (items[:, 3] == 0).all() and (items[:, 6] == -1).all() and (items[:, 7] == -1).all()
        assert skv.splitkv_plan_launches_per_call(plan) == 2
        assert skv.splitkv_workspace_size(plan) > 0
    one = skv.splitkv_plan_fixed(_desc(mode=skv.SPLITKV_COMBINE_SEPARATE), 1)
    assert skv.splitkv_plan_launches_per_call(one) == 1  # nothing to merge
    for bad in (0, 65):
        with pytest.raises(skv.SplitKVError):
            skv.splitkv_plan_fixed(_desc(), bad)


def test_refresh_and_read_items_validate_before_any_cuda_call():
    A = 1 << 20
    host_plan = skv.splitkv_plan(_desc(), np.array([100], np.int32), 2, 148)
    fixed = skv.splitkv_plan_fixed(_desc(), 2)
    assert skv._lib.splitkv_plan_refresh(host_plan.handle, A, A, None) == skv.SPLITKV_EINVAL
    assert skv._lib.splitkv_plan_refresh(fixed.handle, A, None, None) == skv.SPLITKV_EINVAL
    assert skv._lib.splitkv_plan_refresh(fixed.handle, None, A, None) == skv.SPLITKV_EWORKSPACE
    assert skv._lib.splitkv_plan_refresh(fixed.handle, A, A + 2, None) == skv.SPLITKV_EINVAL
    out = np.zeros((1, 8), np.int32)
    assert skv._lib.splitkv_read_items(fixed.handle, A, out.ctypes.data, 1, None) == skv.SPLITKV_EINVAL


def test_upload_checks_workspace_size():
    d = _desc()
    plan = skv.splitkv_plan(d, np.array([5900], np.int32), 8, 148)
    st = skv._lib.splitkv_plan_upload(plan.handle, 1 << 20, 16, None)
    assert st == skv.SPLITKV_EWORKSPACE


def test_combine_validates():
    st = skv._lib.splitkv_combine(1 << 20, 1 << 20, 0, 4, 128, 1 << 20, None, None, None)
    assert st == skv.SPLITKV_EINVAL
    for n_parts, dv in ((2, 130), (2, 0), (0, 128), (2, 6)):
        st = skv._lib.splitkv_combine(1 << 20, 1 << 20, n_parts, 4, dv, 1 << 20, None, None, None)
        assert st == skv.SPLITKV_EINVAL, (n_parts, dv)


def test_plan_matches_oracle_mla_cta_pairs():
    """MLA items launch a CTA pair per query token; the automatic split count
    plans over num_sms / (2 T) machines in both the library and the oracle."""
    for T, L, P in ((6, 65536, 64), (1, 4096, 64), (2, 300, 64), (16, 9000, 64),
                    (6, 65536, 16), (3, 777, 32), (6, 65536, 128)):
        maxp = -(-65536 // P)
        d = skv.make_desc(1, T, 128, 1, 576, 512, P, maxp, maxp + 8, skv.SPLITKV_BF16, 1)
        for S in (0, 1, 4, 8):
            plan = skv.splitkv_plan(d, np.array([L], np.int32), S, 148)
            items = skv.splitkv_plan_get_items(plan)
            ref = np.array(oracle.plan_items([L], P, 1, S, 148, ctas_per_item=2 * T), np.int32)
            assert np.array_equal(items[:, :6], ref), (T, L, P, S)


def test_launches_per_call():
    d_sep = _desc(mode=skv.SPLITKV_COMBINE_SEPARATE)
    d_fus = _desc(mode=skv.SPLITKV_COMBINE_FUSED)
    lens = np.array([5900], np.int32)
    assert skv.splitkv_plan_launches_per_call(skv.splitkv_plan(d_sep, lens, 8, 148)) == 2
    assert skv.splitkv_plan_launches_per_call(skv.splitkv_plan(d_fus, lens, 8, 148)) == 1
    assert skv.splitkv_plan_launches_per_call(skv.splitkv_plan(d_sep, lens, 1, 148)) == 1  # nothing to merge
