"""Pins for the fp64 oracle, checked against things other than the oracle itself.

* brute force in 60-digit arithmetic (mpmath) on tiny hand-built inputs, with
  the softmax written without max-subtraction;
* closed forms (identical keys, one key, one dominant key);
* invariants (number of splits, physical page permutation, page size, combine
  associativity and permutation, -inf as the combine's identity);
* library special cases (torch.softmax in float64, torch's e4m3 and bf16
  decoders);
* the hand-worked split tables in ``tests/golden``.
"""
import json
import math
import os

import mpmath
import numpy as np
import pytest
import torch

import oracle
from oracle import splitkv_oracle as O
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
mpmath.mp.dps = 60


def _bf16_bits(x):
    return workloads.bits(torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16))


def _tiny_problem(rng, L, D, Hq=2, Hkv=1, T=1, P=4, dv=None, shuffle=True):
    """A tiny paged problem in bf16 with a shuffled block table."""
    dv = D if dv is None else dv
    n = -(-L // P)
    pool = n + 3
    q = _bf16_bits(rng.standard_normal((1, T, Hq, D)))
    k = _bf16_bits(rng.standard_normal((pool, Hkv, P, D)))
    v = _bf16_bits(rng.standard_normal((pool, Hkv, P, dv)))
    phys = rng.permutation(pool)[:n] if shuffle else np.arange(n)
    table = np.full((1, n + 2), pool - 1, dtype=np.int32)
    table[0, :n] = phys
    return q, k, v, table, np.array([L], dtype=np.int32)


def _mp_attention(q_row, K, V, scale):
    """Brute force: exp of every score, direct sums, 60 digits."""
    s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b))
                                         for a, b in zip(q_row, k)) for k in K]
    e = [mpmath.exp(x) for x in s]
    tot = mpmath.fsum(e)
    out = [mpmath.fsum(e[j] * mpmath.mpf(float(V[j][d])) for j in range(len(K))) / tot
           for d in range(len(V[0]))]
    return [float(o) for o in out], float(mpmath.log(tot))


# ---------------------------------------------------------------- decoding

def test_e4m3_hand_values():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_codes.json")))
    for code, val in g["codes"].items():
        got = float(O.e4m3_to_float(np.array([int(code, 16)], np.uint8))[0])
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    for code in g["nan_codes"]:
        assert np.isnan(O.e4m3_to_float(np.array([int(code, 16)], np.uint8))[0])


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_float(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_bf16_decode_matches_torch():
    raw = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_to_float(raw)
    ref = torch.from_numpy(raw.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[ok], ref[ok])
    assert O.bf16_to_float(np.array([0x3F80], np.uint16))[0] == 1.0
    assert O.bf16_to_float(np.array([0xC000], np.uint16))[0] == -2.0


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("L,D,P", [(1, 2, 4), (3, 3, 2), (5, 4, 4), (8, 4, 3)])
def test_direct_matches_brute_force(L, D, P):
    rng = np.random.default_rng(L * 100 + D)
    q, k, v, table, lens = _tiny_problem(rng, L, D, Hq=2, Hkv=1, P=P)
    scale = 0.37
    out, lse = O.attention_direct(q, k, v, table, lens, scale=scale)
    for h in range(2):
        K = [O.bf16_to_float(k[table[0, j // P], 0, j % P]) for j in range(L)]
        V = [O.bf16_to_float(v[table[0, j // P], 0, j % P]) for j in range(L)]
        ref_o, ref_l = _mp_attention(O.bf16_to_float(q[0, 0, h]), K, V, scale)
        np.testing.assert_allclose(out[0, 0, h], ref_o, rtol=0, atol=1e-13)
        assert abs(lse[0, 0, h] - ref_l) < 1e-13


def test_nhd_layout_brute_force():
    """NHD pages ``[N][P][Hkv][D]``: key j of KV head h is row
    ``pages[table[j // P]][j % P][h]``, indexed here by hand (P != Hkv, so a
    swap of the slot and head axes cannot pass)."""
    rng = np.random.default_rng(17)
    L, D, P, Hkv, G = 7, 3, 3, 2, 2
    n = -(-L // P)
    pool = n + 2
    q = _bf16_bits(rng.standard_normal((1, 1, Hkv * G, D)))
    k = _bf16_bits(rng.standard_normal((pool, P, Hkv, D)))
    v = _bf16_bits(rng.standard_normal((pool, P, Hkv, D)))
    table = rng.permutation(pool)[:n].astype(np.int32)[None, :]
    lens = np.array([L], dtype=np.int32)
    out, lse = O.attention_direct(q, k, v, table, lens, scale=0.6, layout="NHD")
    for h in range(Hkv * G):
        hk = h // G
        K = [O.bf16_to_float(k[table[0, j // P], j % P, hk]) for j in range(L)]
        V = [O.bf16_to_float(v[table[0, j // P], j % P, hk]) for j in range(L)]
        ref_o, ref_l = _mp_attention(O.bf16_to_float(q[0, 0, h]), K, V, 0.6)
        np.testing.assert_allclose(out[0, 0, h], ref_o, atol=1e-13)
        assert abs(lse[0, 0, h] - ref_l) < 1e-13


def test_layout_invariance_is_bitwise():
    """The same rows stored HND and NHD give bit-identical results, in the
    direct and the split mode."""
    q, k, v, table, lens = _mid_problem(L=37, T=2, Hq=8, Hkv=2, P=4)
    k_n = np.ascontiguousarray(k.transpose(0, 2, 1, 3))
    v_n = np.ascontiguousarray(v.transpose(0, 2, 1, 3))
    o1, l1 = O.attention_direct(q, k, v, table, lens, scale=0.3)
    o2, l2 = O.attention_direct(q, k_n, v_n, table, lens, scale=0.3, layout="NHD")
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    o3, l3 = O.attention_split_mode(q, k, v, table, lens, num_splits=3, scale=0.3)
    o4, l4 = O.attention_split_mode(q, k_n, v_n, table, lens, num_splits=3, scale=0.3,
                                    layout="NHD")
    assert np.array_equal(o3, o4) and np.array_equal(l3, l4)


def test_causal_multi_token_brute_force():
    """Query token t of T sees keys 0 .. L-T+t (bottom-right aligned)."""
    rng = np.random.default_rng(7)
    L, T, D, P = 7, 3, 4, 2
    q, k, v, table, lens = _tiny_problem(rng, L, D, Hq=2, Hkv=2, T=T, P=P)
    out, lse = O.attention_direct(q, k, v, table, lens, scale=0.5)
    for t in range(T):
        for h in range(2):
            n_vis = L - T + t + 1
            K = [O.bf16_to_float(k[table[0, j // P], h, j % P]) for j in range(n_vis)]
            V = [O.bf16_to_float(v[table[0, j // P], h, j % P]) for j in range(n_vis)]
            ref_o, ref_l = _mp_attention(O.bf16_to_float(q[0, t, h]), K, V, 0.5)
            np.testing.assert_allclose(out[0, t, h], ref_o, atol=1e-13)
            assert abs(lse[0, t, h] - ref_l) < 1e-13


def test_latent_v_brute_force():
    """The latent cache (V shares the key rows): V_j is the first v_dim
    columns of K_j, for every query head of the one KV head, causal over T."""
    rng = np.random.default_rng(29)
    L, T, D, dv, P, Hq = 6, 2, 5, 3, 4, 3
    q, k, _, table, lens = _tiny_problem(rng, L, D, Hq=Hq, Hkv=1, T=T, P=P)
    out, lse = O.attention_direct(q, k, None, table, lens, scale=0.45, v_dim=dv,
                                  v_shares_k=True)
    assert out.shape == (1, T, Hq, dv)
    for t in range(T):
        for h in range(Hq):
            n_vis = L - T + t + 1
            K = [O.bf16_to_float(k[table[0, j // P], 0, j % P]) for j in range(n_vis)]
            V = [row[:dv] for row in K]
            ref_o, ref_l = _mp_attention(O.bf16_to_float(q[0, t, h]), K, V, 0.45)
            np.testing.assert_allclose(out[0, t, h], ref_o, atol=1e-13)
            assert abs(lse[0, t, h] - ref_l) < 1e-13


def test_fp8_brute_force_with_scale():
    """e4m3 keys/values are code * kv_scale in both the scores and the output."""
    rng = np.random.default_rng(11)
    L, D, P = 6, 4, 4
    q = _bf16_bits(rng.standard_normal((1, 1, 2, D)))
    k = rng.integers(0, 256, size=(3, 1, P, D)).astype(np.uint8)
    v = rng.integers(0, 256, size=(3, 1, P, D)).astype(np.uint8)
    k[(k & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    v[(v & 0x7F) == 0x7F] = 0x44
    table = np.array([[2, 0]], np.int32)
    kv_scale = 0.0123
    out, lse = O.attention_direct(q, k, v, table, np.array([L], np.int32), scale=0.3,
                                  kv_dtype="fp8_e4m3", kv_scale=kv_scale)
    for h in range(2):
        K = [O.e4m3_to_float(k[table[0, j // P], 0, j % P]) * kv_scale for j in range(L)]
        V = [O.e4m3_to_float(v[table[0, j // P], 0, j % P]) * kv_scale for j in range(L)]
        ref_o, ref_l = _mp_attention(O.bf16_to_float(q[0, 0, h]), K, V, 0.3)
        np.testing.assert_allclose(out[0, 0, h], ref_o, atol=1e-13)
        assert abs(lse[0, 0, h] - ref_l) < 1e-12


def _fp8_tiny(rng, L=6, D=4, P=4, Hq=4, Hkv=2, N=3):
    q = _bf16_bits(rng.standard_normal((1, 1, Hq, D)))
    k = rng.integers(0, 256, size=(N, Hkv, P, D)).astype(np.uint8)
    v = rng.integers(0, 256, size=(N, Hkv, P, D)).astype(np.uint8)
    k[(k & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    v[(v & 0x7F) == 0x7F] = 0x44
    table = np.array([[2, 0]], np.int32)
    return q, k, v, table, np.array([L], np.int32)


def test_fp8_per_head_kv_scales_brute_force():
    """Per-KV-head scales: K_j = code * k_scale[h_kv], V_j = code * v_scale[h_kv],
    with query head h reading KV head h // G."""
    rng = np.random.default_rng(12)
    L, P = 6, 4
    q, k, v, table, lens = _fp8_tiny(rng, L=L, P=P)
    ks, vs = [0.011, 0.037], [0.21, 0.053]
    out, lse = O.attention_direct(q, k, v, table, lens, scale=0.3, kv_dtype="fp8_e4m3",
                                  k_scale=ks, v_scale=vs)
    for h in range(4):
        hk = h // 2
        K = [O.e4m3_to_float(k[table[0, j // P], hk, j % P]) * ks[hk] for j in range(L)]
        V = [O.e4m3_to_float(v[table[0, j // P], hk, j % P]) * vs[hk] for j in range(L)]
        ref_o, ref_l = _mp_attention(O.bf16_to_float(q[0, 0, h]), K, V, 0.3)
        np.testing.assert_allclose(out[0, 0, h], ref_o, atol=1e-13)
        assert abs(lse[0, 0, h] - ref_l) < 1e-12


def test_fp8_v_scale_is_linear_and_k_scale_is_a_temperature():
    """Scaling V by c scales the output by c and leaves the LSE alone; scaling K
    by a is the same as scaling the softmax scale by a."""
    rng = np.random.default_rng(13)
    q, k, v, table, lens = _fp8_tiny(rng)
    base_o, base_l = O.attention_direct(q, k, v, table, lens, scale=0.3, kv_dtype="fp8_e4m3",
                                        k_scale=[0.02, 0.02], v_scale=[0.1, 0.1])
    o2, l2 = O.attention_direct(q, k, v, table, lens, scale=0.3, kv_dtype="fp8_e4m3",
                                k_scale=[0.02, 0.02], v_scale=[0.35, 0.35])
    np.testing.assert_allclose(o2, base_o * 3.5, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(l2, base_l, rtol=0, atol=1e-12)
    o3, l3 = O.attention_direct(q, k, v, table, lens, scale=0.3 * 0.02 / 0.05, kv_dtype="fp8_e4m3",
                                k_scale=[0.05, 0.05], v_scale=[0.1, 0.1])
    np.testing.assert_allclose(o3, base_o, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(l3, base_l, rtol=0, atol=1e-11)
    # a single per-tensor kv_scale is the special case k_scale = v_scale = kv_scale
    o4, l4 = O.attention_direct(q, k, v, table, lens, scale=0.3, kv_dtype="fp8_e4m3",
                                kv_scale=0.02)
    o5, l5 = O.attention_direct(q, k, v, table, lens, scale=0.3, kv_dtype="fp8_e4m3",
                                k_scale=[0.02, 0.02], v_scale=[0.02, 0.02])
    assert np.array_equal(o4, o5) and np.array_equal(l4, l5)


def test_head_mapping_uses_contiguous_groups():
    """With G = 2, query heads 2,3 read KV head 1.  Make KV head 1's keys all
    zero: those rows must average V (closed form) while heads 0,1 must not."""
    rng = np.random.default_rng(5)
    L, D, P = 6, 4, 2
    q, k, v, table, lens = _tiny_problem(rng, L, D, Hq=4, Hkv=2, P=P)
    k[:, 1] = 0
    out, lse = O.attention_direct(q, k, v, table, lens, scale=1.0)
    V1 = np.stack([O.bf16_to_float(v[table[0, j // P], 1, j % P]) for j in range(L)])
    for h in (2, 3):
        np.testing.assert_allclose(out[0, 0, h], V1.mean(0), atol=1e-14)
        assert abs(lse[0, 0, h] - math.log(L)) < 1e-14
    for h in (0, 1):
        assert np.abs(out[0, 0, h] - V1.mean(0)).max() > 1e-3


# ---------------------------------------------------------------- closed forms

def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    L, D, P = 37, 8, 4
    q, k, v, table, lens = _tiny_problem(rng, L, D, P=P)
    k[:] = k[0, 0, 0]  # every key the same row
    scale = 0.25
    out, lse = O.attention_direct(q, k, v, table, lens, scale=scale)
    V = np.stack([O.bf16_to_float(v[table[0, j // P], 0, j % P]) for j in range(L)])
    for h in range(2):
        s = scale * float(O.bf16_to_float(q[0, 0, h]) @ O.bf16_to_float(k[0, 0, 0]))
        np.testing.assert_allclose(out[0, 0, h], V.mean(0), rtol=0, atol=1e-14)
        assert abs(lse[0, 0, h] - (s + math.log(L))) < 1e-12


def test_single_key():
    rng = np.random.default_rng(4)
    q, k, v, table, lens = _tiny_problem(rng, 1, 5, P=4)
    out, lse = O.attention_direct(q, k, v, table, lens, scale=0.7)
    for h in range(2):
        s0 = 0.7 * float(O.bf16_to_float(q[0, 0, h]) @ O.bf16_to_float(k[table[0, 0], 0, 0]))
        np.testing.assert_array_equal(out[0, 0, h], O.bf16_to_float(v[table[0, 0], 0, 0]))
        assert abs(lse[0, 0, h] - s0) < 1e-15


def test_dominant_key():
    rng = np.random.default_rng(6)
    L, D, P = 20, 4, 4
    q, k, v, table, lens = _tiny_problem(rng, L, D, Hq=1, P=P)
    q[0, 0, 0] = _bf16_bits([1.0, 0, 0, 0])
    k[..., 0] = _bf16_bits(0.0)
    j = 13
    k[table[0, j // P], 0, j % P, 0] = _bf16_bits(50.0)
    out, lse = O.attention_direct(q, k, v, table, lens, scale=1.0)
    # the other 19 keys carry weight e^-50 each: out = V_13 up to 19 e^-50 max|V|
    tol = 19 * math.exp(-50) * 10
    np.testing.assert_allclose(out[0, 0, 0], O.bf16_to_float(v[table[0, j // P], 0, j % P]),
                               rtol=0, atol=tol)
    assert abs(lse[0, 0, 0] - 50.0) < 1e-14


def test_no_visible_keys():
    rng = np.random.default_rng(8)
    q, k, v, table, lens = _tiny_problem(rng, 4, 4, P=4)
    out, lse = O.attention_direct(q, k, v, table, np.array([0], np.int32), scale=1.0)
    assert np.all(out == 0) and np.all(lse == -math.inf)


# ---------------------------------------------------------------- library case

def test_matches_torch_softmax_float64():
    rng = np.random.default_rng(9)
    L, D, P = 50, 16, 8
    q, k, v, table, lens = _tiny_problem(rng, L, D, Hq=4, Hkv=2, P=P)
    out, lse = O.attention_direct(q, k, v, table, lens, scale=0.2)
    for h in range(4):
        hk = h // 2
        K = torch.from_numpy(np.stack([O.bf16_to_float(k[table[0, j // P], hk, j % P]) for j in range(L)]))
        V = torch.from_numpy(np.stack([O.bf16_to_float(v[table[0, j // P], hk, j % P]) for j in range(L)]))
        qt = torch.from_numpy(O.bf16_to_float(q[0, 0, h]))
        s = (K @ qt) * 0.2
        ref = torch.softmax(s, dim=0) @ V
        np.testing.assert_allclose(out[0, 0, h], ref.numpy(), atol=1e-14)
        assert abs(lse[0, 0, h] - torch.logsumexp(s, 0).item()) < 1e-13


# ---------------------------------------------------------------- invariants

def _mid_problem(seed=12, L=203, D=16, Hq=4, Hkv=2, T=1, P=8, fp8=False):
    rng = np.random.default_rng(seed)
    q, k, v, table, lens = _tiny_problem(rng, L, D, Hq=Hq, Hkv=Hkv, T=T, P=P)
    if fp8:
        k = rng.integers(0, 0x7E, size=k.shape).astype(np.uint8) | (rng.integers(0, 2, size=k.shape) << 7).astype(np.uint8)
        v = rng.integers(0, 0x7E, size=v.shape).astype(np.uint8)
    return q, k, v, table, lens


@pytest.mark.parametrize("fp8", [False, True])
def test_split_invariance(fp8):
    q, k, v, table, lens = _mid_problem(fp8=fp8)
    kw = dict(scale=0.25, kv_dtype="fp8_e4m3" if fp8 else "bf16", kv_scale=0.01 if fp8 else 1.0)
    ref_o, ref_l = O.attention_direct(q, k, v, table, lens, **kw)
    n = O.pages_of(int(lens[0]), k.shape[2])
    for S in list(range(1, n + 1)) + [n + 5, 0]:
        o, l = O.attention_split_mode(q, k, v, table, lens, num_splits=S, **kw)
        np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)


def test_split_invariance_causal_multi_token():
    q, k, v, table, lens = _mid_problem(L=37, T=6, Hq=8, Hkv=1, P=4)
    ref_o, ref_l = O.attention_direct(q, k, v, table, lens, scale=0.3)
    for S in range(1, 11):
        o, l = O.attention_split_mode(q, k, v, table, lens, num_splits=S, scale=0.3)
        np.testing.assert_allclose(o, ref_o, atol=1e-12)
        np.testing.assert_allclose(l, ref_l, atol=1e-12)


def test_page_permutation_invariance_is_bitwise():
    q, k, v, table, lens = _mid_problem()
    out, lse = O.attention_direct(q, k, v, table, lens, scale=0.25)
    rng = np.random.default_rng(1)
    perm = rng.permutation(k.shape[0])  # new position of old page i is perm[i]
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    table2 = perm[table].astype(np.int32)
    out2, lse2 = O.attention_direct(q, k2, v2, table2, lens, scale=0.25)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def _repage(pages, P_new, perm):
    """The key rows of a contiguous pool (pages 0..n-1 in table order) cut
    into pages of P_new rows; logical page i is stored at physical perm[i]."""
    N, Hkv, P, D = pages.shape
    rows = pages.transpose(1, 0, 2, 3).reshape(Hkv, N * P, D)  # [Hkv][keys][D]
    n_new = len(perm)
    pad = n_new * P_new - N * P
    rows = np.concatenate([rows, np.zeros((Hkv, pad, D), rows.dtype)], axis=1)
    logical = rows.reshape(Hkv, n_new, P_new, D).transpose(1, 0, 2, 3)
    out = np.empty_like(logical)
    out[perm] = logical
    return out


@pytest.mark.parametrize("P_old,P_new", [(4, 16), (16, 4), (8, 24)])
@pytest.mark.parametrize("latent", [False, True])
def test_page_size_is_transparent(P_old, P_new, latent):
    """Cutting the same key rows into pages of another size (the 576-wide
    latent rows with V as their first columns, or separate K and V) and
    scattering them over the pool changes nothing: bitwise for the direct
    definition, to rounding in split mode (whose page-granular split
    boundaries move)."""
    rng = np.random.default_rng(40 + P_old + P_new)
    L, T, Hq = 45, 3, 4
    D, dv = (12, 8) if latent else (6, 6)
    n = -(-L // P_old)
    q = _bf16_bits(rng.standard_normal((1, T, Hq, D)))
    k = _bf16_bits(rng.standard_normal((n, 1, P_old, D)))
    v = None if latent else _bf16_bits(rng.standard_normal((n, 1, P_old, dv)))
    table = np.arange(n, dtype=np.int32)[None, :]
    lens = np.array([L], np.int32)
    kw = dict(scale=0.3, v_dim=dv, v_shares_k=latent)
    ref = O.attention_direct(q, k, v, table, lens, **kw)
    perm = rng.permutation(-(-(n * P_old) // P_new)).astype(np.int32)
    k2 = _repage(k, P_new, perm)
    v2 = None if latent else _repage(v, P_new, perm)
    got = O.attention_direct(q, k2, v2, perm[None, :], lens, **kw)
    assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1])
    for S in (1, 2, 3):
        o, l = O.attention_split_mode(q, k2, v2, perm[None, :], lens, num_splits=S, **kw)
        np.testing.assert_allclose(o, ref[0], atol=1e-12)
        np.testing.assert_allclose(l, ref[1], atol=1e-12)


def _rand_part(rng, dim=6):
    return rng.standard_normal(dim), float(rng.standard_normal() * 3)


def test_combine_associative_and_permutation_invariant():
    rng = np.random.default_rng(21)
    a, b, c, d = (_rand_part(rng) for _ in range(4))
    left = O.combine([O.combine([a, b]), c])
    right = O.combine([a, O.combine([b, c])])
    flat = O.combine([a, b, c])
    for x in (left, right):
        np.testing.assert_allclose(x[0], flat[0], atol=1e-14)
        assert abs(x[1] - flat[1]) < 1e-14
    perm = O.combine([c, a, d, b])
    ref = O.combine([a, b, c, d])
    np.testing.assert_allclose(perm[0], ref[0], atol=1e-14)
    assert abs(perm[1] - ref[1]) < 1e-14


def test_combine_identity_and_empty():
    rng = np.random.default_rng(22)
    a = _rand_part(rng)
    empty = (np.zeros(6), -math.inf)
    x = O.combine([a, empty])
    np.testing.assert_allclose(x[0], a[0], atol=1e-15)
    assert abs(x[1] - a[1]) < 1e-15
    y = O.combine([empty, empty])
    assert np.all(y[0] == 0) and y[1] == -math.inf


def test_combine_closed_form_two_equal_halves():
    """Two partials with equal lse: lse grows by ln 2 and the outputs average."""
    o1, o2 = np.array([1.0, 2.0]), np.array([3.0, -2.0])
    o, l = O.combine([(o1, 0.5), (o2, 0.5)])
    np.testing.assert_allclose(o, [2.0, 0.0], atol=1e-15)
    assert abs(l - (0.5 + math.log(2))) < 1e-15


# ---------------------------------------------------------------- planner

def test_split_ranges_golden():
    g = json.load(open(os.path.join(GOLDEN, "split_ranges.json")))
    for case in g["cases"]:
        r = [list(x) for x in O.split_ranges(case["n"], case["S"])]
        if "ranges" in case:
            assert r == case["ranges"]
        else:
            assert r[:len(case["first"])] == case["first"]
            assert r[-len(case["last"]):] == case["last"]
    cc = g["ceil_chunk_contrast"]
    ours = O.split_ranges(cc["n"], cc["S"])
    assert sum(1 for a, b in ours if b > a) == cc["S"]
    chunk = -(-cc["n"] // cc["S"])
    ceil_rule = [(s * chunk, min(cc["n"], (s + 1) * chunk)) for s in range(cc["S"])]
    assert sum(1 for a, b in ceil_rule if b > a) == cc["nonempty"]


@pytest.mark.parametrize("n", [1, 2, 3, 17, 64, 369, 1000])
def test_split_ranges_tile_and_nonempty(n):
    for S in range(1, min(n, 70) + 1):
        r = O.split_ranges(n, S)
        assert r[0][0] == 0 and r[-1][1] == n
        assert all(r[i][1] == r[i + 1][0] for i in range(S - 1))
        sizes = [b - a for a, b in r]
        assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1


def test_plan_items_honours_num_splits_and_is_nonempty():
    lens = [260, 5900, 1, 16, 17, 0]
    for S in (1, 2, 4, 8, 16, 32, 64):
        items = O.plan_items(lens, 16, 2, S, 148)
        for b, L in enumerate(lens):
            n = O.pages_of(L, 16)
            mine = [it for it in items if it[0] == b]
            if n == 0:
                assert len(mine) == 2 and all(it[4] == it[5] for it in mine)
                continue
            assert len(mine) == 2 * min(S, n)
            assert all(it[5] > it[4] for it in mine)
            for h in range(2):
                rr = sorted((it[4], it[5]) for it in mine if it[1] == h)
                assert rr[0][0] == 0 and rr[-1][1] == n
        sizes = [it[5] - it[4] for it in items]
        assert sizes == sorted(sizes, reverse=True)


def test_makespan_lpt_hand_example():
    # LPT on 2 machines: 7 -> m0, 5 -> m1, 4 -> m1 (5<7), 3 -> m0 (7<9), 2 -> m0 (10 vs 9 -> m1)
    assert O._makespan([5, 3, 7, 2, 4], 2) == 11
    assert O._makespan([4, 4, 4], 3) == 4
    assert O._makespan([1] * 10, 3) == 4


def test_auto_splits_fill_the_machine_for_few_heads():
    """Two KV heads and one long sequence: the automatic choice must create
    many more split CTAs than KV heads (the point of split-KV)."""
    items = O.plan_items([5900], 16, 2, 0, 148)
    assert len(items) >= 64
    assert all(it[5] > it[4] for it in items)
    items1 = O.plan_items([260], 16, 2, 0, 148)
    assert all(it[5] > it[4] for it in items1)


def test_auto_splits_count_resident_slots():
    """One 100-page sequence, one KV head, 4 SMs.  Worked by hand with the
    cost model (item = 16 * pages + ITEM_OVERHEAD, plus COMBINE_COST * S):
    one resident CTA per SM -> 4 splits of 25 pages (504 beats 608 for 8
    splits); two per SM -> 8 machines, 8 splits of 12-13 pages (320)."""
    assert O.choose_splits([100], 1, 4, ctas_per_sm=1) == [4]
    assert O.choose_splits([100], 1, 4, ctas_per_sm=2) == [8]
    # an item that needs two CTAs halves the machines again
    assert O.choose_splits([100], 1, 4, ctas_per_item=2, ctas_per_sm=2) == [4]


def test_head_groups_share_the_sequence_ranges():
    lens = [5900, 300, 0]
    for S in (0, 1, 4):
        items = O.plan_items(lens, 16, 8, S, 152, ctas_per_sm=3, heads_per_item=4)
        assert sorted(set(it[1] for it in items)) == [0, 4]
        for b, L in enumerate(lens):
            n = O.pages_of(L, 16)
            rr = {h: sorted((it[4], it[5]) for it in items if it[0] == b and it[1] == h)
                  for h in (0, 4)}
            assert rr[0] == rr[4]
            if n:
                assert rr[0][0][0] == 0 and rr[0][-1][1] == n
                assert all(p1 > p0 for p0, p1 in rr[0])
                if S:
                    assert len(rr[0]) == min(S, n)
            else:
                assert rr[0] == [(0, 0)]


# ---------------------------------------------------------------- pin strength

def _pins_on_direct():
    test_direct_matches_brute_force(5, 4, 4)
    test_identical_keys_give_mean_of_values()
    test_causal_multi_token_brute_force()
    test_head_mapping_uses_contiguous_groups()
    test_nhd_layout_brute_force()
    test_latent_v_brute_force()


@pytest.mark.parametrize("mistake", ["no_scale", "neg_scores", "k_for_v", "lse_off_by_max",
                                     "head_mod", "causal_off_by_one", "page_slot_swap",
                                     "nhd_read_as_hnd", "latent_v_last_columns"])
def test_planted_mistakes_are_caught(monkeypatch, mistake):
    """Each plausible slip, planted in the oracle on the CPU, fails a pin."""
    orig_attend = O._softmax_attend
    orig_gather = O.gather_keys

    if mistake == "no_scale":
        monkeypatch.setattr(O, "_softmax_attend", lambda q, K, V, s: orig_attend(q, K, V, 1.0))
    elif mistake == "neg_scores":
        monkeypatch.setattr(O, "_softmax_attend", lambda q, K, V, s: orig_attend(-q, K, V, s))
    elif mistake == "k_for_v":
        monkeypatch.setattr(O, "_softmax_attend",
                            lambda q, K, V, s: orig_attend(q, K, K[:, :V.shape[1]] if K.shape[1] >= V.shape[1] else V * 2, s))
    elif mistake == "lse_off_by_max":
        def bad(q, K, V, s):
            o, l = orig_attend(q, K, V, s)
            return o, (l - float((s * (K @ q)).max()) if K.shape[0] else l)
        monkeypatch.setattr(O, "_softmax_attend", bad)
    elif mistake == "head_mod":
        orig_direct = O.attention_direct

        def bad_direct(q, k, v, table, lens, **kw):
            # map query head h to KV head h % Hkv instead of h // G
            Hq, Hkv = q.shape[2], k.shape[1]
            G = Hq // Hkv
            perm = [(h % Hkv) * G + h // Hkv for h in range(Hq)]
            o, l = orig_direct(q[:, :, perm], k, v, table, lens, **kw)
            inv = np.argsort(perm)
            return o[:, :, inv], l[:, :, inv]
        monkeypatch.setattr(O, "attention_direct", bad_direct)
    elif mistake == "causal_off_by_one":
        orig_direct = O.attention_direct

        def bad_direct(q, k, v, table, lens, **kw):
            return orig_direct(q, k, v, table, np.asarray(lens) - (1 if q.shape[1] > 1 else 0), **kw)
        monkeypatch.setattr(O, "attention_direct", bad_direct)
    elif mistake == "page_slot_swap":
        def bad_gather(pages, row, n, head, layout="HND"):
            P = O.page_size_of(pages, layout)
            out = orig_gather(pages, row, n, head, layout)
            return out[::-1].copy() if n > P else out
        monkeypatch.setattr(O, "gather_keys", bad_gather)
    elif mistake == "latent_v_last_columns":
        # V of the latent cache taken from the last v_dim columns of the key rows
        def bad_attend(q, K, V, s):
            dv = V.shape[1]
            if dv < K.shape[1] and np.array_equal(V, K[:, :dv]):
                V = K[:, K.shape[1] - dv:]
            return orig_attend(q, K, V, s)
        monkeypatch.setattr(O, "_softmax_attend", bad_attend)
    elif mistake == "nhd_read_as_hnd":
        # the slot and head axes of NHD pages taken in HND order
        monkeypatch.setattr(O, "gather_keys",
                            lambda pages, row, n, head, layout="HND": orig_gather(pages, row, n, head))
    # (the NHD axes read in HND order index past the slot axis when P != Hkv)
    with pytest.raises(IndexError if mistake == "nhd_read_as_hnd" else AssertionError):
        _pins_on_direct()
