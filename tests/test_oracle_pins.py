"""Pins for the fp64 oracle: each test checks the oracle against something
other than itself (a closed form, a printed worked example, an invariant, or
an independently written brute force)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from shared_prefix_decode_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    return torch.tensor(np.asarray(x), dtype=torch.float32).to(torch.bfloat16).double().numpy()


# ---------------------------------------------------------------- closed forms
def test_single_key_returns_its_value():
    """One key: softmax weight 1, so O = v exactly and LSE = the scaled score."""
    rng = np.random.default_rng(1)
    d = 64
    q, k, v = rng.standard_normal((1, d)), rng.standard_normal((1, d)), rng.standard_normal((1, d))
    scale = 0.37
    O, L = oracle.sdp(q, k, v, scale)
    assert np.array_equal(O[0], v[0])
    assert L[0] == pytest.approx(scale * float(q[0] @ k[0]), abs=1e-13)


def test_identical_keys_give_mean_value():
    """n identical keys: equal weights, O = mean(V), LSE = s + ln n."""
    rng = np.random.default_rng(2)
    d, n = 32, 37
    q = rng.standard_normal((3, d))
    k = np.repeat(rng.standard_normal((1, d)), n, axis=0)
    v = rng.standard_normal((n, d))
    O, L = oracle.sdp(q, k, v, 0.25)
    for r in range(3):
        np.testing.assert_allclose(O[r], v.mean(axis=0), atol=1e-13)
        assert L[r] == pytest.approx(0.25 * float(q[r] @ k[0]) + math.log(n), abs=1e-12)


def test_scores_use_scale_and_natural_log():
    """Two keys with scores a, b: LSE = ln(e^a + e^b), weights e^a/(e^a+e^b)."""
    d = 4
    q = np.array([[1.0, 0, 0, 0]])
    k = np.array([[2.0, 0, 0, 0], [-1.0, 0, 0, 0]])
    v = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
    scale = 0.5
    O, L = oracle.sdp(q, k, v, scale)
    a, b = 1.0, -0.5
    assert L[0] == pytest.approx(math.log(math.exp(a) + math.exp(b)), abs=1e-14)
    wa = math.exp(a) / (math.exp(a) + math.exp(b))
    np.testing.assert_allclose(O[0], [wa, 1 - wa, 0, 0], atol=1e-15)


def test_empty_key_set_is_zero_and_minus_inf():
    O, L = oracle.sdp(np.ones((2, 8)), np.zeros((0, 8)), np.zeros((0, 8)), 1.0)
    assert np.all(O == 0) and np.all(L == -np.inf)


def test_merge_with_empty_part_is_identity_and_both_empty_is_empty():
    rng = np.random.default_rng(3)
    O1 = rng.standard_normal((4, 16))
    L1 = rng.standard_normal(4)
    O, L = oracle.merge(O1, L1, np.zeros((4, 16)), np.full(4, -np.inf))
    np.testing.assert_array_equal(O, O1)
    np.testing.assert_array_equal(L, L1)
    O, L = oracle.merge(np.zeros((2, 16)), np.full(2, -np.inf), np.zeros((2, 16)),
                        np.full(2, -np.inf))
    assert np.all(O == 0) and np.all(L == -np.inf) and not np.any(np.isnan(O))


# ------------------------------------------------------------- invariants
def test_key_permutation_invariance():
    rng = np.random.default_rng(4)
    d, n = 48, 300
    q, K, V = rng.standard_normal((5, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    O, L = oracle.sdp(q, K, V, 0.2)
    p = rng.permutation(n)
    O2, L2 = oracle.sdp(q, K[p], V[p], 0.2)
    np.testing.assert_allclose(O2, O, atol=1e-12)
    np.testing.assert_allclose(L2, L, atol=1e-12)


def test_merge_identity_on_random_splits():
    """Hydragen Eq. 5: merging the (O, LSE) of two disjoint key parts equals
    attention over their concatenation."""
    rng = np.random.default_rng(5)
    d, n = 64, 500
    q, K, V = rng.standard_normal((7, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    q *= 3.0  # peaked softmax
    O, L = oracle.sdp(q, K, V, 1 / 8)
    for cut in (1, 17, 250, 499):
        mask = np.zeros(n, bool)
        mask[rng.permutation(n)[:cut]] = True
        Oa, La = oracle.sdp(q, K[mask], V[mask], 1 / 8)
        Ob, Lb = oracle.sdp(q, K[~mask], V[~mask], 1 / 8)
        Om, Lm = oracle.merge(Oa, La, Ob, Lb)
        np.testing.assert_allclose(Om, O, atol=1e-12)
        np.testing.assert_allclose(Lm, L, atol=1e-12)


def test_chunk_partial_states_reduce_to_full_attention():
    """ChunkAttention Eq. 1 + Eq. 2: partial (o, m, n) per chunk, reduced in an
    arbitrary order, then O / n equals softmax attention; m + ln n equals LSE."""
    rng = np.random.default_rng(6)
    d, n, c = 32, 333, 64
    q, K, V = rng.standard_normal(d), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    O, L = oracle.sdp(q[None], K, V, 0.3)
    chunks = [(s, min(s + c, n)) for s in range(0, n, c)]
    order = rng.permutation(len(chunks))
    state = [np.zeros(d), -math.inf, 0.0]
    for i in order:
        s, e = chunks[i]
        o_c, m_c, n_c = oracle.partial_attn(q, K[s:e], V[s:e], 0.3)
        oracle.attn_reduce(o_c, m_c, n_c, state)
    np.testing.assert_allclose(state[0] / state[2], O[0], atol=1e-12)
    assert state[1] + math.log(state[2]) == pytest.approx(L[0], abs=1e-12)


# -------------------------------------------- printed worked example (blog)
def test_blog_split_merge_example():
    """The shared-prefix KV caching blog's float64 check: prefix pass + per
    sequence suffix pass, merged, vs single pass; printed max error 3.05e-16."""
    g = json.load(open(os.path.join(GOLDEN, "blog_split_merge_check.json")))
    d, P, B, S = g["d"], g["P"], g["B"], g["S"]
    rng = np.random.default_rng(0)
    Kp, Vp = rng.standard_normal((P, d)), rng.standard_normal((P, d))
    Ks, Vs = rng.standard_normal((B, S, d)), rng.standard_normal((B, S, d))
    Q = rng.standard_normal((B, d))
    scale = 1 / math.sqrt(d)
    O1, L1 = oracle.sdp(Q, Kp, Vp, scale)
    O2, L2 = np.zeros((B, d)), np.zeros(B)
    for b in range(B):
        o, l = oracle.sdp(Q[b:b + 1], Ks[b], Vs[b], scale)
        O2[b], L2[b] = o[0], l[0]
    Om, _ = oracle.merge(O1, L1, O2, L2)
    ref = np.stack([oracle.sdp(Q[b:b + 1], np.vstack([Kp, Ks[b]]), np.vstack([Vp, Vs[b]]),
                               scale)[0][0] for b in range(B)])
    err = np.abs(Om - ref).max()
    assert err <= g["bound_used"], err
    assert err < 100 * g["printed_max_abs_error"]


# ------------------------------------------ brute force (independent numpy)
def _np_attention(q, K, V, scale):
    """Second, independent fp64 softmax attention (numpy / scipy)."""
    from scipy.special import logsumexp, softmax
    s = scale * (K @ q)
    return softmax(s) @ V, logsumexp(s)


def _np_cascade(wl):
    """Brute-force cascade: gather each sequence's keys with numpy fancy
    indexing from the page lists, then the numpy softmax above."""
    kp = wl.k_pool.double().numpy()
    vp = wl.v_pool.double().numpy()
    q = wl.q.double().numpy()
    ps = wl.page_size
    G = wl.Hq // wl.Hkv
    O = np.zeros((wl.B, wl.Hq, wl.d))
    L = np.zeros((wl.B, wl.Hq))
    for b in range(wl.B):
        pages, slots = [], []
        for lv in wl.levels:
            nodes = lv.nodes.numpy()
            ids = lv.page_ids.numpy()
            hit = np.nonzero((nodes[:, 0] <= b) & (b < nodes[:, 1]))[0]
            assert len(hit) <= 1
            if len(hit) == 0:
                continue
            _, _, kl, off = nodes[hit[0]]
            t = np.arange(kl)
            pages.append(ids[off + t // ps])
            slots.append(t % ps)
        pages = np.concatenate(pages) if pages else np.zeros(0, int)
        slots = np.concatenate(slots) if slots else np.zeros(0, int)
        for h in range(wl.Hq):
            K = kp[pages, h // G, slots, :]
            V = vp[pages, h // G, slots, :]
            if len(pages) == 0:
                O[b, h], L[b, h] = 0.0, -np.inf
            else:
                O[b, h], L[b, h] = _np_attention(q[b, h], K, V, wl.scale)
    return O, L


def test_sdp_matches_brute_force_tiny():
    rng = np.random.default_rng(7)
    for nk in (1, 2, 5, 64):
        q, K, V = rng.standard_normal((3, 16)), rng.standard_normal((nk, 16)), rng.standard_normal((nk, 16))
        O, L = oracle.sdp(q, K, V, 0.7)
        for r in range(3):
            o, l = _np_attention(q[r], K, V, 0.7)
            np.testing.assert_allclose(O[r], o, atol=1e-12)
            assert L[r] == pytest.approx(l, abs=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_cascade_matches_brute_force_tiny_trees(seed):
    """Tiny trees (B<=4, <=64 keys per sequence) with GQA, shuffled pages,
    two shared levels and ragged suffixes including empty ones."""
    wl = W.build_cascade("t", B=4, Hq=4, Hkv=2, d=16, page_size=4,
                         shared=[[(0, 4, 12)], [(0, 2, 8), (2, 4, 5)]],
                         suffix_range=(0, 9), seed=seed)
    O, L = oracle.cascade(wl)
    Ob, Lb = _np_cascade(wl)
    np.testing.assert_allclose(O.reshape(Ob.shape), Ob, atol=1e-12)
    np.testing.assert_allclose(L.reshape(Lb.shape), Lb, atol=1e-12)


def test_cascade_config_tiny_matches_brute_force():
    wl = W.make_config("tiny", seed=3)
    O, L = oracle.cascade(wl)
    Ob, Lb = _np_cascade(wl)
    np.testing.assert_allclose(O.reshape(Ob.shape), Ob, atol=1e-12)
    np.testing.assert_allclose(L.reshape(Lb.shape), Lb, atol=1e-12)


def test_zero_query_counts_visible_keys():
    """q = 0: every key has score 0, so LSE = ln(#visible keys) and O = their
    mean -- pins the number of keys each sequence sees (catches length
    off-by-ones in the tree walk)."""
    wl = W.build_cascade("z", B=5, Hq=2, Hkv=1, d=8, page_size=4,
                         shared=[[(0, 5, 7)], [(1, 3, 6)]], suffix_lens=[0, 3, 4, 1, 9], seed=1)
    wl.q.zero_()
    O, L = oracle.cascade(wl)
    n_vis = wl.seq_kv_len()
    assert n_vis == [7, 16, 17, 8, 16]
    for r, (b, h) in enumerate([(b, h) for b in range(5) for h in range(2)]):
        assert L[r] == pytest.approx(math.log(n_vis[b]), abs=1e-13)
    Ob, _ = _np_cascade(wl)
    np.testing.assert_allclose(O.reshape(Ob.shape), Ob, atol=1e-13)


def test_page_shuffle_invariance():
    """Physical page order is immaterial: same logical KV under two different
    page permutations gives the same output."""
    wl = W.build_cascade("s", B=3, Hq=4, Hkv=4, d=16, page_size=4,
                         shared=[[(0, 3, 16)]], suffix_lens=[5, 0, 11], seed=9, shuffle=False)
    O, L = oracle.cascade(wl)
    perm = torch.randperm(wl.num_pages, generator=torch.Generator().manual_seed(11))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(len(perm))
    wl.k_pool = wl.k_pool[inv].contiguous()  # logical page p now at physical perm[p]
    wl.v_pool = wl.v_pool[inv].contiguous()
    for lv in wl.levels:
        lv.page_ids = perm[lv.page_ids.long()].to(torch.int32)
    O2, L2 = oracle.cascade(wl)
    np.testing.assert_allclose(O2, O, atol=1e-12)
    np.testing.assert_allclose(L2, L, atol=1e-12)


def test_boundaries_zero_suffix_and_zero_prefix():
    """Zero-length suffix = prefix-only attention; P = 0 = pure suffix decode."""
    wl = W.build_cascade("b", B=2, Hq=2, Hkv=1, d=16, page_size=4,
                         shared=[[(0, 2, 10)]], suffix_lens=[0, 0], seed=4)
    O, L = oracle.cascade(wl)
    ids = wl.levels[0].page_ids.long()
    K = wl.k_pool[ids].permute(1, 0, 2, 3).reshape(1, -1, 16)[0, :10].double().numpy()
    V = wl.v_pool[ids].permute(1, 0, 2, 3).reshape(1, -1, 16)[0, :10].double().numpy()
    Op, Lp = oracle.sdp(wl.q.double().numpy().reshape(4, 16), K, V, wl.scale)
    np.testing.assert_allclose(O, Op, atol=1e-13)
    np.testing.assert_allclose(L, Lp, atol=1e-13)
    # no shared level, one empty sequence
    wl2 = W.build_cascade("c", B=2, Hq=2, Hkv=1, d=16, page_size=4, shared=[],
                          suffix_lens=[6, 0], seed=5)
    O2, L2 = oracle.cascade(wl2)
    assert np.all(O2[2:] == 0) and np.all(L2[2:] == -np.inf)
    Ob, Lb = _np_cascade(wl2)
    np.testing.assert_allclose(O2[:2], Ob.reshape(-1, 16)[:2], atol=1e-12)


def test_paged_decode_and_prefix_agree_with_cascade():
    """The per-sequence page-table form and the contiguous-prefix form are
    independently written gathers; both must agree with the tree form."""
    wl = W.make_config("tiny", seed=5)
    O, L = oracle.cascade(wl)
    pt, sl = W.full_page_tables(wl)
    Op, Lp = oracle.paged_decode(wl.q, wl.k_pool, wl.v_pool, pt, sl, wl.scale)
    np.testing.assert_allclose(Op.reshape(O.shape), O, atol=1e-12)
    np.testing.assert_allclose(Lp.reshape(L.shape), L, atol=1e-12)
    # contiguous [len][Hkv][d] prefix built from the shared level's pages
    wl0 = W.make_config("tiny", seed=5)
    wl0.levels = wl0.levels[:1]
    O0, L0 = oracle.cascade(wl0)
    ids = wl0.levels[0].page_ids.long()
    k = wl0.k_pool[ids].permute(0, 2, 1, 3).reshape(-1, wl0.Hkv, wl0.d)
    v = wl0.v_pool[ids].permute(0, 2, 1, 3).reshape(-1, wl0.Hkv, wl0.d)
    Oc, Lc = oracle.prefix(wl0.q, k, v, wl0.scale)
    np.testing.assert_allclose(Oc.reshape(O0.shape), O0, atol=1e-12)
    np.testing.assert_allclose(Lc.reshape(L0.shape), L0, atol=1e-12)


def test_probe_output_is_the_code_row():
    wl = W.make_config("tiny", seed=0)
    n = wl.seq_kv_len()
    targets = [0, n[1] - 1, 255, 256 if n[3] > 256 else 3]
    W.apply_probe(wl, targets)
    O, L = oracle.cascade(wl)
    for r, (b, h) in enumerate([(b, h) for b in range(wl.B) for h in range(wl.Hq)]):
        # every other weight is below e^-300: zero to fp32, ~1e-200 in fp64
        np.testing.assert_allclose(O[r], W.probe_expected(b, wl.d).double().numpy(), rtol=0,
                                   atol=1e-30)


def test_gqa_mapping_consecutive_heads():
    """Query heads h and h' read the same KV head iff h // G == h' // G: with
    identical q rows, heads of one group agree and heads of different groups
    differ."""
    wl = W.build_cascade("g", B=1, Hq=4, Hkv=2, d=16, page_size=4, shared=[],
                         suffix_lens=[9], seed=2)
    wl.q[0, :, :] = wl.q[0, 0, :]
    O, _ = oracle.cascade(wl)
    np.testing.assert_array_equal(O[0], O[1])
    np.testing.assert_array_equal(O[2], O[3])
    assert np.abs(O[0] - O[2]).max() > 1e-3


# ------------------------------------------------ reduced-precision KV (E4M3)
def test_e4m3_decoder_special_values():
    """The E4M3 values that close forms fix: +-0, the smallest subnormal
    2^-9, the largest subnormal 7 * 2^-9, the smallest normal 2^-6, 1, 1.875,
    2, the largest finite value 448 (S.1111.110) and the two NaN codes
    (S.1111.111); there are no infinities."""
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3F: 1.875,
             0x40: 2.0, 0x7E: 448.0, 0x80: -0.0, 0x81: -(2.0 ** -9), 0xB8: -1.0, 0xFE: -448.0}
    got = oracle.e4m3_decode(np.array(sorted(table), dtype=np.uint8))
    for (c, want), g in zip(sorted(table.items()), got):
        assert g == want, (hex(c), g, want)
    assert np.signbit(oracle.e4m3_decode(np.array([0x80], dtype=np.uint8))[0])
    nan = oracle.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.isnan(nan).all()
    allv = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.isfinite(allv).sum() == 254 and not np.isinf(allv).any()


def test_e4m3_decoder_is_monotone_symmetric_and_matches_torch():
    """Codes 0x00..0x7E decode to strictly increasing values (each step one
    unit in the last place of the lower code's binade: 2^-9 through the
    subnormals and the first binade, 2^(e-10) in binade e), the sign bit
    negates, and every code agrees with torch's independent float8_e4m3fn
    decoding."""
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    steps = np.diff(pos)
    assert (steps > 0).all()
    for c in range(1, 0x7F):
        e = max((c - 1) >> 3, 1)
        assert steps[c - 1] == 2.0 ** (e - 10), hex(c)
    neg = oracle.e4m3_decode((np.arange(0x7F) | 0x80).astype(np.uint8))
    np.testing.assert_array_equal(neg, -pos)
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_decode(codes)
    ok = np.isfinite(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    assert np.isnan(got[~ok]).all()


def _e4m3_pow2_workload(seed):
    """A tree whose last level reads E4M3 pools with power-of-two scales
    that differ per page, per KV head and between K and V, next to bf16
    pools holding the same values (code value x scale is exact in bf16:
    4 significant bits, exponents within range)."""
    wl = W.build_cascade("q8", B=5, Hq=4, Hkv=2, d=16, page_size=4, shared=[[(0, 5, 7)], [(0, 2, 5), (2, 5, 3)]],
                         suffix_range=(0, 9), seed=seed)
    g = torch.Generator().manual_seed(seed + 11)
    P = wl.num_pages
    shape = (P, wl.Hkv, wl.page_size, wl.d)
    # finite codes only (not S.1111.111)
    k8 = torch.randint(0, 254, shape, generator=g, dtype=torch.int32)
    v8 = torch.randint(0, 254, shape, generator=g, dtype=torch.int32)
    k8 = torch.where(k8 >= 0x7F, k8 + 1, k8).to(torch.uint8)
    v8 = torch.where(v8 >= 0x7F, v8 + 1, v8).to(torch.uint8)
    ks = torch.pow(2.0, torch.randint(-3, 4, (P, wl.Hkv), generator=g).double()).float()
    vs = torch.pow(2.0, torch.randint(-3, 4, (P, wl.Hkv), generator=g).double()).float()
    w8 = W.with_e4m3_levels(wl, levels=(-1,))
    w8.q8 = W.E4M3Pools(k8, v8, ks, vs)
    kd = (k8.view(torch.float8_e4m3fn).double() * ks.double()[:, :, None, None]).to(torch.bfloat16)
    vd = (v8.view(torch.float8_e4m3fn).double() * vs.double()[:, :, None, None]).to(torch.bfloat16)
    assert torch.equal(kd.double(), k8.view(torch.float8_e4m3fn).double() * ks.double()[:, :, None, None])
    # the bf16 twin: shared levels keep wl's pools, the last level the decoded values
    twin = W.build_cascade("q8", B=5, Hq=4, Hkv=2, d=16, page_size=4,
                           shared=[[(0, 5, 7)], [(0, 2, 5), (2, 5, 3)]], suffix_range=(0, 9), seed=seed)
    last = set(twin.levels[-1].page_ids.tolist())
    shared = set(p for lv in twin.levels[:-1] for p in lv.page_ids.tolist())
    assert not (last & shared)
    for p in last:
        twin.k_pool[p] = kd[p]
        twin.v_pool[p] = vd[p]
    return w8, twin


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_e4m3_levels_equal_their_decoded_bf16_twin(seed):
    """Cascade over a tree whose suffix level is stored as E4M3 codes and
    per-(page, KV head) scales equals the cascade over bf16 pools holding the
    decoded values (1e-12): pins which scale a key takes (its page, its KV
    head, K's or V's) and that only the marked level is decoded."""
    w8, twin = _e4m3_pow2_workload(seed)
    O8, L8 = oracle.cascade(w8)
    O, L = oracle.cascade(twin)
    np.testing.assert_allclose(O8, O, atol=1e-12, rtol=0)
    np.testing.assert_allclose(L8, L, atol=1e-12, rtol=0)


def test_e4m3_paged_decode_equals_decoded_bf16():
    """The per-sequence paged decode over E4M3 pools equals the bf16 paged
    decode over the decoded values (1e-12)."""
    own = W.build_cascade("q8s", B=5, Hq=4, Hkv=2, d=16, page_size=4, shared=[], suffix_range=(0, 9), seed=9)
    g = torch.Generator().manual_seed(5)
    P = own.num_pages
    k8 = torch.randint(0, 0x7F, (P, 2, 4, 16), generator=g, dtype=torch.int32).to(torch.uint8)
    v8 = torch.randint(0x80, 0xFF, (P, 2, 4, 16), generator=g, dtype=torch.int32).to(torch.uint8)
    ks = torch.pow(2.0, torch.randint(-2, 3, (P, 2), generator=g).double()).float()
    vs = torch.pow(2.0, torch.randint(-2, 3, (P, 2), generator=g).double()).float()
    kd = (k8.view(torch.float8_e4m3fn).double() * ks.double()[:, :, None, None]).to(torch.bfloat16)
    vd = (v8.view(torch.float8_e4m3fn).double() * vs.double()[:, :, None, None]).to(torch.bfloat16)
    pt, sl = W.full_page_tables(own)
    O8, L8 = oracle.paged_decode_e4m3(own.q, k8, v8, ks, vs, pt, sl, own.scale)
    O, L = oracle.paged_decode(own.q, kd, vd, pt, sl, own.scale)
    np.testing.assert_allclose(O8, O, atol=1e-12, rtol=0)
    np.testing.assert_allclose(L8, L, atol=1e-12, rtol=0)


# ------------------------------------------- planted mistakes must be caught
_PINS = [
    test_single_key_returns_its_value,
    test_identical_keys_give_mean_value,
    test_scores_use_scale_and_natural_log,
    test_merge_identity_on_random_splits,
    test_chunk_partial_states_reduce_to_full_attention,
    test_blog_split_merge_example,
    test_sdp_matches_brute_force_tiny,
    lambda: test_cascade_matches_brute_force_tiny_trees(0),
    test_zero_query_counts_visible_keys,
    test_paged_decode_and_prefix_agree_with_cascade,
    test_probe_output_is_the_code_row,
    test_gqa_mapping_consecutive_heads,
    test_e4m3_decoder_special_values,
    test_e4m3_decoder_is_monotone_symmetric_and_matches_torch,
    lambda: test_e4m3_levels_equal_their_decoded_bf16_twin(0),
    test_e4m3_paged_decode_equals_decoded_bf16,
]

_MUTANTS = {
    "dropped_scale": ("s[j] = scale * acc;", "s[j] = acc;"),
    "gqa_modulo": ("int kvh = h / G;\n        int nk", "int kvh = h % G;\n        int nk"),
    "short_node": ("for (t = 0; t < nd[2]; ++t)", "for (t = 0; t < nd[2] - 1; ++t)"),
    "merge_sign": ("(w1 * O1[r * d + i] + w2 * O2[r * d + i])", "(w1 * O1[r * d + i] - w2 * O2[r * d + i])"),
    "lse_without_max": ("double L = m + log(sum);", "double L = log(sum);"),
    "slot_reversed": ("long slot = t % L->page_size;",
                      "long slot = L->page_size - 1 - t % L->page_size;"),
    "reduce_wrong_factor": ("O[i] = x * o_c[i] + y * O[i];", "O[i] = y * o_c[i] + x * O[i];"),
    "e4m3_bias": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_subnormal": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    "e4m3_kv_scales_swapped": ("keys[n].k_scale = k_scales[l][page * Hkv + kvh];",
                               "keys[n].k_scale = v_scales[l][page * Hkv + kvh];"),
    "e4m3_scale_head_ignored": ("keys[n].v_scale = v_scales[l][page * Hkv + kvh];",
                                "keys[n].v_scale = v_scales[l][page * Hkv];"),
}


def _run_pins_with(so_path):
    """Child-process entry: run every pin against a compiled oracle variant and
    print how many failed."""
    failed = []
    with oracle.use_library(so_path):
        for pin in _PINS:
            try:
                pin()
            except (AssertionError, ValueError):
                failed.append(getattr(pin, "__name__", "lambda"))
    print("FAILED_PINS", len(failed), ",".join(failed))


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_pins_catch_planted_oracle_mistake(name, tmp_path):
    """Plant one mistake in a copy of the oracle source; at least one pin must
    fail (a crash of the mutant, e.g. an out-of-range read, also counts)."""
    import subprocess
    import sys
    src = open(oracle.source_path()).read()
    old, new = _MUTANTS[name]
    assert old in src, f"mutation anchor for {name} not found"
    c = tmp_path / "mut.c"
    so = tmp_path / "mut.so"
    c.write_text(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", str(so),
                           str(c), "-lm"])
    code = ("import sys; sys.path[:0] = [%r, %r]; import test_oracle_pins as t; "
            "t._run_pins_with(%r)" % (os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                                     os.path.dirname(os.path.abspath(__file__)), str(so)))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return  # the mutant crashed: caught
    line = [l for l in r.stdout.splitlines() if l.startswith("FAILED_PINS")][-1]
    assert int(line.split()[1]) > 0, f"planted mistake {name!r} passed every pin"


# ------------------------------------------------ parallel prompting layout
def test_parallel_prompting_fig2_mask():
    """The worked example printed as Figure 2 of Read Once, Answer Many: a
    3-token document, 3 streams with 1-token questions, decode step 2.  The
    layout generator reproduces the figure's slot ids and positions, and the
    oracle's Eq. 2 mask gives the new token of stream 1 exactly the slots the
    figure marks visible."""
    g = json.load(open(os.path.join(GOLDEN, "parallel_prompting_fig2_mask.json")))
    req = W.stream_requests(R=1, P=g["request"]["streams"], Hq=1, Hkv=1, d=8,
                            doc_len=g["request"]["document_tokens"],
                            q_len_range=(g["request"]["question_tokens_per_stream"],) * 2,
                            T=g["request"]["decode_step"], seed=0)
    sid, pos, _, _ = req.rows[0]
    assert sid.tolist() == g["slot_sid"] and pos.tolist() == g["position"]
    qy = g["query"]
    assert req.q_pos[qy["sid"]] == qy["position"]
    vis = oracle.stream_visible([qy["sid"]], [qy["position"]], g["slot_sid"], g["position"])[0]
    assert [g["slots"][i] for i in np.nonzero(vis)[0]] == g["visible_to_query"]


@pytest.mark.parametrize("seed", [0, 1])
def test_stream_mask_equals_its_cascade_form(seed):
    """Each stream of a Parallel Prompting request sees the document plus its
    own question and answers (Eq. 2), which is the prefix tree of one shared
    document node and one private node per stream: the oracle of the masked
    row equals the oracle of that tree, row by row (documents of 37 and 300
    tokens, up to 5 streams with questions of 1-4 tokens, 3 answer steps)."""
    req = W.stream_requests(R=2, P=5, Hq=4, Hkv=2, d=32, doc_len=37 if seed == 0 else 300,
                            q_len_range=(1, 4), T=3, seed=seed)
    wl = W.streams_as_tree(req, page_size=16)
    O, L = oracle.cascade(wl)
    G = req.Hq // req.Hkv
    q = req.q.double().numpy()
    row = 0
    for r in range(req.R):
        sid, pos, k, v = req.rows[r]
        for s in range(req.P):
            b = r * req.P + s
            for h in range(req.Hq):
                Om, Lm = oracle.stream_masked(q[b, h][None], k[:, h // G].double().numpy(),
                                              v[:, h // G].double().numpy(), [s], [req.q_pos[b]],
                                              sid.numpy(), pos.numpy(), req.scale)
                np.testing.assert_allclose(O[row], Om[0], atol=1e-12)
                assert L[row] == pytest.approx(Lm[0], abs=1e-12)
                row += 1
    # another stream's slots are never visible
    vis = oracle.stream_visible([0, 1], [req.q_pos[0], req.q_pos[1]], req.rows[0][0].numpy(),
                                req.rows[0][1].numpy())
    assert not (vis[0] & (req.rows[0][0].numpy() == 1)).any()
    assert not (vis[1] & (req.rows[0][0].numpy() == 0)).any()


_STREAM_MUTANTS = {
    "causal_strict": ("causal = slot_pos <= q_pos", "causal = slot_pos < q_pos"),
    "document_hidden": ("same = (slot_sid == -1) | (slot_sid == q_sid)", "same = slot_sid == q_sid"),
    "streams_unmasked": ("return causal & same", "return causal"),
}


@pytest.mark.parametrize("name", sorted(_STREAM_MUTANTS))
def test_stream_pins_catch_planted_mask_mistake(name, monkeypatch):
    """Plant one mistake in the oracle's stream mask (a copy of its source,
    loaded in place of the real one); the Figure 2 pin or the cascade-form
    pin must fail."""
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(oracle.stream_visible))
    old, new = _STREAM_MUTANTS[name]
    assert old in src, f"mutation anchor for {name} not found"
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    monkeypatch.setattr(oracle, "stream_visible", ns["stream_visible"])
    failed = 0
    for pin in (test_parallel_prompting_fig2_mask, lambda: test_stream_mask_equals_its_cascade_form(0)):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, f"planted mistake {name!r} passed every pin"


# ------------------------------------------------------ the plan, replayed
def _replay_plan(wl, capacity=0, num_sms=152, plan_wl=None):
    """The planner's output run on the oracle: each work item's rows attend
    (oracle.sdp) to the keys its record's pages hold over its key range, and
    each output row merges (oracle.merge) the partial states its merge list
    names.  The plan is built from ``plan_wl`` (default ``wl``); the keys,
    queries and current suffix lengths come from ``wl``.  Returns (O, LSE)
    in oracle.cascade's row order."""
    from shared_prefix_decode_gb300 import binding as hb
    levels = hb._levels_of(plan_wl if plan_wl is not None else wl)
    args = (levels, wl.B, wl.Hq, wl.Hkv, wl.d)
    items = hb.hp_cascade_plan_items(*args, capacity=capacity, num_sms=num_sms)
    pages = hb.hp_cascade_plan_item_pages(*args, capacity=capacity, num_sms=num_sms)
    tab = hb.hp_cascade_plan_merge_table(*args, capacity=capacity, num_sms=num_sms)
    G, ps = wl.G, wl.page_size
    K, V, q = wl.k_pool.double().numpy(), wl.v_pool.double().numpy(), wl.q.double().numpy()
    part = {}
    for it, pg in zip(items, pages):
        k0, k1 = it["k0"], it["k1"]
        if it["len_seq"] >= 0:  # a loop item ends at its sequence's current length
            k1 = min(k1, int(wl.levels[it["level"]].nodes[it["len_seq"], 2]))
        pid = [pg[t // ps - k0 // ps] for t in range(k0, k1)]
        slot = [t % ps for t in range(k0, k1)]
        seqs = range(it["seq_begin"], it["seq_begin"] + it["n_seq"])
        for h in range(it["kvh"], it["kvh"] + it["n_kvh"]):
            Q = np.stack([q[b, h * G + g] for b in seqs for g in range(G)])
            O, L = oracle.sdp(Q, K[pid, h, slot], V[pid, h, slot], wl.scale)
            for i, b in enumerate(seqs):
                s_ = b - it["seq_begin"]
                if it["tc"]:
                    row = it["part_row"] + (s_ // (128 // G)) * 128 + (s_ % (128 // G)) * G
                else:
                    row = it["part_row"] + ((h - it["kvh"]) * it["n_seq"] + s_) * G
                for g in range(G):
                    part[row + g] = (O[i * G + g], L[i * G + g])
    Oo = np.zeros((wl.B * wl.Hq, wl.d))
    Lo = np.full(wl.B * wl.Hq, -np.inf)
    for b in range(wl.B):
        for h in range(wl.Hq):
            o, l = np.zeros((1, wl.d)), np.full(1, -np.inf)
            for r in tab[b * wl.Hkv + h // G]:
                po, pl = part[r + h % G]
                o, l = oracle.merge(o, l, po[None], np.array([pl]))
            Oo[b * wl.Hq + h], Lo[b * wl.Hq + h] = o[0], l[0]
    return Oo, Lo


@pytest.mark.parametrize("name,kw", [("llama3_8b", {}), ("tree2", dict(B=32, prefix=256)),
                                     ("codellama13b", dict(B=24, prefix=512)), ("no_sharing", dict(B=6, prefix=300)),
                                     ("tiny", {})])
def test_plan_replayed_on_the_oracle_equals_the_definition(name, kw):
    """The plan (items, their record pages, the merge lists) computes the
    definition: replayed on the oracle it equals oracle.cascade row by row
    (1e-12), the benchmarked workload at full size included."""
    wl = W.make_config(name, seed=2, **kw)
    O, L = oracle.cascade(wl)
    Or, Lr = _replay_plan(wl)
    np.testing.assert_allclose(Or, O, atol=1e-12)
    fin = np.isfinite(L)
    assert np.array_equal(np.isfinite(Lr), fin)
    np.testing.assert_allclose(Lr[fin], L[fin], atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_plan_replayed_on_random_trees_and_loop_plans(seed):
    rng = np.random.default_rng(200 + seed)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8]))
    B = int(rng.integers(1, 40))
    shared = []
    for _ in range(int(rng.integers(1, 4))):
        cuts = sorted(set(rng.integers(1, B, size=int(rng.integers(0, 4))).tolist())) if B > 1 else []
        bounds = [0] + cuts + [B]
        shared.append([(a, b, int(rng.integers(0, 300))) for a, b in zip(bounds[:-1], bounds[1:])])
    wl = W.build_cascade(f"r{seed}", B=B, Hq=Hkv * G, Hkv=Hkv, d=64, page_size=int(rng.choice([16, 32])),
                         shared=shared, suffix_range=(0, 100), seed=seed)
    O, L = oracle.cascade(wl)
    Or, Lr = _replay_plan(wl, num_sms=int(rng.choice([16, 152])))
    np.testing.assert_allclose(Or, O, atol=1e-12)
    np.testing.assert_allclose(Lr[np.isfinite(L)], L[np.isfinite(L)], atol=1e-12)
    # the same tree as a decode loop: the plan built at the start, replayed
    # after each of five appended tokens with the grown suffixes
    cap = int(wl.levels[-1].nodes[:, 2].max()) + 5
    lw = W.with_suffix_capacity(wl, cap, seed=seed)
    start = W.CascadeWorkload(lw.name, lw.B, lw.Hq, lw.Hkv, lw.d, lw.page_size, lw.scale, lw.q, lw.k_pool,
                              lw.v_pool, [W.TreeLevel(l.nodes.clone(), l.page_ids) for l in lw.levels])
    for q, k, v in W.decode_tokens(lw, 5, seed=seed):
        W.append_token(lw, k, v)
        lw.q = q
        O, L = oracle.cascade(lw)
        Or, Lr = _replay_plan(lw, capacity=cap, plan_wl=start)
        np.testing.assert_allclose(Or, O, atol=1e-12)
        np.testing.assert_allclose(Lr, L, atol=1e-12)


@pytest.mark.parametrize("mid,ps", [(32, 16), (20, 16), (64, 32), (0, 16)])
def test_plan_with_fused_single_sequence_chains_replayed(mid, ps):
    """Trees whose sequences each own a question node below a shared document
    (page-aligned or not, or empty) above their suffix: the planner fuses a
    sequence's own nodes into one where it can, and the replayed plan still
    equals the definition, also as a decode loop as the suffixes grow."""
    B = 6
    wl = W.build_cascade("chain", B=B, Hq=8, Hkv=2, d=64, page_size=ps,
                         shared=[[(0, B, 100)], [(b, b + 1, mid) for b in range(B)]],
                         suffix_range=(0, 40), seed=mid)
    O, L = oracle.cascade(wl)
    Or, Lr = _replay_plan(wl)
    np.testing.assert_allclose(Or, O, atol=1e-12)
    np.testing.assert_allclose(Lr, L, atol=1e-12)
    cap = int(wl.levels[-1].nodes[:, 2].max()) + 3
    lw = W.with_suffix_capacity(wl, cap, seed=1)
    start = W.CascadeWorkload(lw.name, lw.B, lw.Hq, lw.Hkv, lw.d, lw.page_size, lw.scale, lw.q, lw.k_pool,
                              lw.v_pool, [W.TreeLevel(l.nodes.clone(), l.page_ids) for l in lw.levels])
    for q, k, v in W.decode_tokens(lw, 3, seed=1):
        W.append_token(lw, k, v)
        lw.q = q
        O, L = oracle.cascade(lw)
        Or, Lr = _replay_plan(lw, capacity=cap, plan_wl=start)
        np.testing.assert_allclose(Or, O, atol=1e-12)
        np.testing.assert_allclose(Lr, L, atol=1e-12)


def test_plans_of_the_gpu_random_trees_replayed():
    """The twelve random trees of the GPU parity tests: their plans,
    replayed on the oracle, equal the definition."""
    from test_gpu_parity import _random_tree
    for seed in range(12):
        wl = _random_tree(seed)
        O, L = oracle.cascade(wl)
        Or, Lr = _replay_plan(wl)
        np.testing.assert_allclose(Or, O, atol=1e-12, err_msg=f"tree {seed}")
        fin = np.isfinite(L)
        assert np.array_equal(np.isfinite(Lr), fin)
        np.testing.assert_allclose(Lr[fin], L[fin], atol=1e-12, err_msg=f"tree {seed}")


def test_deep_chunk_tree_replayed():
    """A ChunkAttention-style tree: a 64-token system prompt shared by all
    sequences, then each sequence's private keys as a chain of 16-token
    chunk nodes, one level per chunk (up to 20 levels).  The chunks of each
    sequence plan as one node, and the replayed plan equals the definition."""
    from shared_prefix_decode_gb300 import binding as hb
    B, ps = 5, 16
    lens = [0, 3, 7, 12, 19]  # chunks per sequence
    levels = [[(0, B, 64)]] + [[(b, b + 1, ps) for b in range(B) if lens[b] > c] for c in range(max(lens))]
    levels = [lv for lv in levels if lv]
    wl = W.build_cascade("chunks", B=B, Hq=8, Hkv=2, d=64, page_size=ps, shared=levels, suffix_lens=[5] * B,
                         seed=3)
    assert len(wl.levels) == 21
    items = hb.hp_cascade_plan_items(hb._levels_of(wl), wl.B, wl.Hq, wl.Hkv, wl.d)
    # each sequence's chunks and suffix are one node at its first chunk's
    # level; sequence 0 has no chunk, so its suffix stays at the last level
    own = {(it["seq_begin"], it["level"]) for it in items if it["n_seq"] == 1}
    assert own == {(0, 20)} | {(b, 1) for b in range(1, B)}
    O, L = oracle.cascade(wl)
    Or, Lr = _replay_plan(wl)
    np.testing.assert_allclose(Or, O, atol=1e-12)
    np.testing.assert_allclose(Lr, L, atol=1e-12)


def _realistic_forest(seed, B=24, ps=16):
    """A ChunkAttention-style forest: two system prompts, each shared by half
    of the sequences, then nested shared chunks down to pairs and triples of
    sequences (narrow nodes), then private suffixes."""
    h = B // 2
    lvl0 = [(0, h, 128), (h, B, 96)]
    lvl1 = [(0, 6, 64), (6, 12, 48), (12, 18, 32), (18, 24, 64)]
    lvl2 = [(b, min(b + 3, B), 16 * (1 + (b // 3) % 3)) for b in range(0, B, 3)]
    lvl3 = [(b, b + 2, 32) for b in range(0, B, 4)]
    return W.build_cascade(f"forest{seed}", B=B, Hq=8, Hkv=2, d=64, page_size=ps,
                           shared=[lvl0, lvl1, lvl2, lvl3], suffix_range=(1, 40), seed=seed)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_narrow_nodes_fused_into_chains_replayed(seed):
    """Narrow shared nodes (2-3 sequences, short) are read by each of their
    sequences inside its own node (fewer partial states, a few more bytes);
    the replayed plan still equals the definition."""
    from shared_prefix_decode_gb300 import binding as hb
    wl = _realistic_forest(seed)
    items = hb.hp_cascade_plan_items(hb._levels_of(wl), wl.B, wl.Hq, wl.Hkv, wl.d)
    # no item reads a node of 2-3 sequences as a shared item: they all joined
    assert all(it["n_seq"] == 1 or it["n_seq"] > 3 for it in items)
    O, L = oracle.cascade(wl)
    Or, Lr = _replay_plan(wl)
    np.testing.assert_allclose(Or, O, atol=1e-12)
    np.testing.assert_allclose(Lr, L, atol=1e-12)
