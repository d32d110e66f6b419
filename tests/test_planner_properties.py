"""Properties of the library's split plans, checked on the C++ planner itself.

Independent of the oracle's step-by-step restatement of the automatic policy:
whatever split count the policy picks, the plan must give every launched split
CTA a non-empty KV range ("vLLM 0.30.0 FA4 SplitKV Bug: H100 Decode Can Be 48%
Slower", section "The actual bug is one missing constructor argument"), tile
each sequence's pages exactly, honour a requested split count whenever the
sequence has that many pages, stay within the 64-split cap, and order items
longest first.  Random shapes, lengths, split requests and SM counts (CPU only;
the planner makes no CUDA call when num_sms is given).
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import split_kv_paged_splitkv_gb300 as skv  # noqa: E402

B_F, H_F, S_F, N_F, P0_F, P1_F, SLOT_F, GRP_F = range(8)


@st.composite
def plans(draw):
    mla = draw(st.booleans())
    P = draw(st.sampled_from([16, 32, 64, 128] if mla else [16, 32, 48, 64, 128]))
    B = draw(st.integers(1, 9))
    T = draw(st.integers(1, 6)) if mla else draw(st.integers(1, 2))
    if mla:
        Hq, Hkv, dk, dv = 128, 1, 576, 512
        fp8 = draw(st.booleans())
    else:
        Hkv = draw(st.sampled_from([1, 2, 3, 4, 8]))
        G = draw(st.sampled_from([1, 2, 4, 8]))
        Hq, dk, dv = Hkv * G, 128, 128
        fp8 = draw(st.booleans())
    max_pages = draw(st.integers(1, 300))
    lens = draw(st.lists(st.one_of(st.just(0), st.integers(T, max_pages * P)), min_size=B,
                         max_size=B))
    S = draw(st.sampled_from([0, 0, 1, 2, 3, 7, 16, 64]))
    sms = draw(st.sampled_from([1, 4, 37, 148, 152]))
    desc = skv.make_desc(B, T, Hq, Hkv, dk, dv, P, max_pages, B * max_pages + 1,
                         skv.SPLITKV_FP8_E4M3 if fp8 else skv.SPLITKV_BF16, int(mla))
    return desc, np.array(lens, np.int32), S, sms


@settings(max_examples=300, deadline=None)
@given(plans())
def test_every_split_owns_a_nonempty_balanced_range(case):
    desc, lens, S, sms = case
    plan = skv.splitkv_plan(desc, lens, S, sms)
    items = skv.splitkv_plan_get_items(plan)
    hpi = skv.splitkv_plan_heads_per_item(plan)
    P = desc.page_size
    groups = desc.num_kv_heads // hpi
    # longest first
    sizes = items[:, P1_F] - items[:, P0_F]
    assert (np.diff(sizes) <= 0).all()
    slots = items[items[:, SLOT_F] >= 0][:, SLOT_F]
    assert len(np.unique(slots)) == len(slots)
    for b, L in enumerate(lens):
        n = -(-int(L) // P)
        mine = items[items[:, B_F] == b]
        if n == 0:
            # one empty item per head group, nothing to merge
            assert len(mine) == groups and (mine[:, P0_F] == mine[:, P1_F]).all()
            assert (mine[:, SLOT_F] == -1).all()
            continue
        Sb = int(mine[0, N_F])
        assert (mine[:, N_F] == Sb).all()
        assert 1 <= Sb <= min(n, 64)
        if S > 0:
            assert Sb == min(S, n)  # the request reaches the kernel
        for h0 in range(0, desc.num_kv_heads, hpi):
            r = mine[mine[:, H_F] == h0]
            assert len(r) == Sb
            r = r[np.argsort(r[:, S_F])]
            assert (r[:, S_F] == np.arange(Sb)).all()
            assert r[0, P0_F] == 0 and r[-1, P1_F] == n
            assert (r[1:, P0_F] == r[:-1, P1_F]).all()  # contiguous tiling
            w = r[:, P1_F] - r[:, P0_F]
            assert w.min() >= 1 and w.max() - w.min() <= 1  # non-empty, balanced
            if Sb > 1:  # merged through one combine group, contiguous slots
                assert len(np.unique(r[:, GRP_F])) == 1 and r[0, GRP_F] >= 0
                assert (np.diff(r[:, SLOT_F]) == 1).all()
            else:
                assert (r[:, SLOT_F] == -1).all() and (r[:, GRP_F] == -1).all()
    # the same inputs give the same plan
    again = skv.splitkv_plan_get_items(skv.splitkv_plan(desc, lens, S, sms))
    assert np.array_equal(items, again)
