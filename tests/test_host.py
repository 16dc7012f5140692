"""Host-side tests (no GPU): the C-ABI library loads and exports every symbol
include/hp.h declares; the tree planner reproduces the pages' context list and
rejects invalid trees before any launch."""
import ctypes
import json
import os
import re

import pytest
import torch

from shared_prefix_decode_gb300 import binding as hb
from shared_prefix_decode_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def _header_functions():
    src = open(os.path.join(ROOT, "include", "hp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(hp_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_library_loads_and_exports_every_declared_symbol():
    lib = hb.library()
    declared = _header_functions()
    assert len(declared) >= 14
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in hp.h but not exported"
    assert set(declared) == set(hb.exported_symbols())
    assert lib.hp_build_arch() == 103
    assert lib.hp_abi_version() == 5


def test_status_strings():
    assert hb.status_str(0) == "ok"
    for s in range(1, 7):
        assert hb.status_str(s) and hb.status_str(s) != "unknown status"


def _pool():
    # a host buffer stands in for the pools: planning reads no pool memory
    return torch.zeros(64, dtype=torch.uint8)


def _fig2_levels(pool, ps=16):
    """ChunkAttention's Figure 2 tree as levels of chunk nodes, one page each."""
    g = json.load(open(os.path.join(GOLDEN, "chunkattention_fig2_contexts.json")))
    chunks = g["tree"]["chunks"]

    def depth(c):
        d = 0
        while chunks[c]["parent"] is not None:
            c = chunks[c]["parent"]
            d += 1
        return d

    by_level = {}
    for name, c in chunks.items():
        by_level.setdefault(depth(name), []).append((name, c["covers"]))
    levels, names, page = [], {}, 0
    for lvl in sorted(by_level):
        nodes, ids = [], []
        for n, (name, (i, j)) in enumerate(sorted(by_level[lvl], key=lambda x: x[1][0])):
            nodes.append((i, j, ps, len(ids)))
            ids.append(page)
            page += 1
            names[(lvl, n)] = name
        levels.append((pool.data_ptr(), pool.data_ptr(), 64, ps, nodes, ids))
    return g, levels, names


def test_chunkattention_fig2_context_list():
    pool = _pool()
    g, levels, names = _fig2_levels(pool)
    ctx = hb.hp_cascade_contexts(levels, B=3, Hq=4, Hkv=4, d=128)
    got = [[names[(l, n)], i, j] for (l, n, i, j, _) in ctx]
    assert got == g["contexts"]
    shared = [names[(l, n)] for (l, n, i, j, batched) in ctx if batched]
    assert shared == g["shared"]
    assert all((j - i > 1) == bool(batched) for (_, _, i, j, batched) in ctx)


def test_plan_stats_llama3_shape():
    """B=64 x G=4 rows share the prefix: 256 rows per KV head go to the
    tensor-core kernel; each sequence's suffix is a small-row item."""
    wl = W.make_config("llama3_8b", seed=0)
    levels = hb._levels_of(wl)
    n_tc, n_small, part_rows, n_merge = hb.hp_cascade_plan_stats(levels, wl.B, wl.Hq, wl.Hkv, wl.d,
                                                                 num_sms=152)
    # each KV head's 32 prefix tiles are split evenly into key ranges, and the
    # planner leaves some CTAs to the paged items: at most one item per CTA
    assert n_tc % 8 == 0 and 8 <= n_tc < 152
    assert n_small >= wl.B * wl.Hkv // 8  # items cover a group of 8 KV heads
    # every (b, kvh) merges the prefix splits that cover it plus its suffix splits
    assert n_merge >= wl.B * wl.Hkv * 2
    assert part_rows > 0


@pytest.mark.parametrize("name", ["tiny", "tree2", "doc_streams", "no_sharing"])
def test_plan_stats_configs(name):
    wl = W.make_config(name, seed=1, B=16 if name != "tiny" else None, prefix=512 if name != "tiny" else None)
    st = hb.hp_cascade_plan_stats(hb._levels_of(wl), wl.B, wl.Hq, wl.Hkv, wl.d, num_sms=152)
    assert all(x >= 0 for x in st)
    if name == "no_sharing":
        assert st[0] == 0


def test_plan_spreads_shared_nodes_of_narrow_groups():
    """Two-level tree (G = 1): a level-2 node's 16 sequences share one paged
    item, whose keys are loaded once -- its modelled cost must not scale with
    the sequence count, or the planner piles the private suffixes onto a few
    CTAs and gives the tensor-core items to a handful of CTAs (a step 3x the
    roofline).  Every KV head's shared prefix then gets its own CTAs."""
    wl = W.make_config("tree2", seed=0)
    n_tc, n_small, _, _ = hb.hp_cascade_plan_stats(hb._levels_of(wl), wl.B, wl.Hq, wl.Hkv, wl.d, num_sms=152)
    assert n_tc >= wl.Hkv


def _desc_levels(nodes, ids, num_pages=8, ps=16, pool=None):
    pool = pool if pool is not None else _pool()
    return [(pool.data_ptr(), pool.data_ptr(), num_pages, ps, nodes, ids)]


@pytest.mark.parametrize("nodes,ids,why", [
    ([(0, 5, 16, 0)], [0], "seq_end beyond B"),
    ([(2, 2, 16, 0)], [0], "empty sequence range"),
    ([(0, 2, 16, 0), (1, 3, 16, 1)], [0, 1], "overlapping nodes in one level"),
    ([(0, 2, 33, 0)], [0, 1], "page list too short"),
    ([(0, 2, 16, 0)], [8], "page id beyond the pool"),
    ([(0, 2, 16, 0)], [-1], "negative page id"),
    ([(0, 2, -1, 0)], [0], "negative length"),
])
def test_invalid_trees_are_rejected_on_the_host(nodes, ids, why):
    levels = _desc_levels(nodes, ids)
    assert hb.hp_cascade_plan_bytes(levels, 4, 4, 4, 128, num_sms=152) == 0, why
    with pytest.raises(hb.HpError):
        hb.hp_cascade_plan_stats(levels, 4, 4, 4, 128)


def test_unsupported_shapes_are_rejected():
    ok = _desc_levels([(0, 2, 16, 0)], [0])
    assert hb.hp_cascade_plan_bytes(ok, 4, 4, 4, 128, num_sms=152) > 0
    assert hb.hp_cascade_plan_bytes(ok, 4, 4, 4, 96, num_sms=152) == 0      # d
    assert hb.hp_cascade_plan_bytes(ok, 4, 6, 4, 128, num_sms=152) == 0     # Hq % Hkv
    assert hb.hp_cascade_plan_bytes(_desc_levels([(0, 2, 16, 0)], [0], ps=24), 4, 4, 4, 128,
                                    num_sms=152) == 0                        # page size
    assert hb.hp_cascade_plan_bytes(_desc_levels([(0, 2, 0, 0)], []), 4, 4, 4, 128, num_sms=152) > 0


def test_zero_length_nodes_make_no_items():
    levels = _desc_levels([(0, 4, 0, 0)], [])
    st = hb.hp_cascade_plan_stats(levels, 4, 4, 4, 128)
    assert st == (0, 0, 0, 0)


def test_workspace_sizes_are_positive_and_rejections_are_zero():
    assert hb.suffix_workspace_bytes(4, 32, 128, 16, 16) >= 256
    assert hb.suffix_workspace_bytes(4, 32, 96, 16, 16) == 0
    assert hb.prefix_workspace_bytes(64, 32, 8, 128, 4096) >= 256
    assert hb.prefix_workspace_bytes(64, 30, 8, 128, 4096) == 0


def test_decode_binding_rejects_wrong_step_tensors():
    """q, out, lse and the workspace are checked before the library is called:
    dtype, shape, unit inner stride and device."""
    class Plan:
        B, Hq, d = 2, 4, 64

    q = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    lse = torch.zeros(2, 4)
    ws = torch.zeros(256, dtype=torch.uint8)
    for bad in (q.float(), q[:, :, ::2], q[:1], q):  # wrong dtype, stride, shape, host memory
        with pytest.raises(ValueError):
            hb._check_step_tensors(Plan, bad, q, lse, ws)


# ------------------------------------------------------------ decode loop
def _loop_levels(B=4, ps=16, cap_pages=3, shared_len=32, lens=(5, 16, 0, 20), pool=None):
    """A shared node over all B sequences (pages 0..), then one suffix per
    sequence with cap_pages reserved pages each (distinct ids after the
    shared ones)."""
    pool = pool if pool is not None else _pool()
    n_sh = (shared_len + ps - 1) // ps
    shared = (pool.data_ptr(), pool.data_ptr(), 64, ps, [(0, B, shared_len, 0)], list(range(n_sh)))
    nodes = [(b, b + 1, lens[b], b * cap_pages) for b in range(B)]
    ids = [n_sh + i for i in range(B * cap_pages)]
    return [shared, (pool.data_ptr(), pool.data_ptr(), 64, ps, nodes, ids)]


def test_loop_plan_is_the_static_plan_plus_the_suffix_page_table():
    lv = _loop_levels()
    static = hb.hp_cascade_plan_bytes(lv, 4, 4, 4, 128, num_sms=152)
    loop = hb.hp_cascade_loop_plan_bytes(lv, 4, 4, 4, 128, capacity=48, num_sms=152)
    assert static > 0 and loop > static
    # capacity exactly the reserved pages, and a capacity of one token
    assert hb.hp_cascade_loop_plan_bytes(_loop_levels(lens=(1, 1, 0, 1), cap_pages=1), 4, 4, 4, 128,
                                         capacity=1, num_sms=152) > 0


@pytest.mark.parametrize("mutate,why", [
    (lambda lv: lv, "capacity beyond the reserved pages"),
    (lambda lv: [lv[0], lv[1][:4] + ([(0, 2, 5, 0), (2, 3, 0, 6), (3, 4, 20, 9)],) + lv[1][5:]],
     "a suffix node covering two sequences"),
    (lambda lv: [lv[0], lv[1][:5] + ([1] + lv[1][5][1:],)], "a suffix page that a shared node uses"),
    (lambda lv: [lv[0], lv[1][:5] + ([lv[1][5][3]] + lv[1][5][1:],)], "a page reserved for two suffixes"),
    (lambda lv: [lv[0], lv[1][:4] + ([(0, 1, 5, 0), (1, 2, 16, 3), (2, 3, 0, 6)],) + lv[1][5:]],
     "a sequence without a suffix node"),
])
def test_loop_plan_rejects_trees_it_cannot_grow(mutate, why):
    cap = 64 if why.startswith("capacity") else 48
    assert hb.hp_cascade_loop_plan_bytes(mutate(_loop_levels()), 4, 4, 4, 128, capacity=cap, num_sms=152) == 0, why


def test_loop_plan_rejects_bad_capacity_and_wide_groups():
    lv = _loop_levels()
    assert hb.hp_cascade_loop_plan_bytes(lv, 4, 4, 4, 128, capacity=0, num_sms=152) == 0
    assert hb.hp_cascade_loop_plan_bytes(lv, 4, 4, 4, 128, capacity=19, num_sms=152) == 0  # below a length
    assert hb.hp_cascade_loop_plan_bytes(lv, 4, 32, 1, 128, capacity=48, num_sms=152) == 0  # G = 32 > 16
    assert hb.hp_cascade_loop_plan_bytes(lv, 4, 16, 1, 128, capacity=48, num_sms=152) > 0   # G = 16


def test_suffix_capacity_and_host_append():
    wl = W.make_config("llama3_8b", B=5, prefix=48, seed=3)
    cap = 300
    w2 = W.with_suffix_capacity(wl, cap, seed=3)
    ps = wl.page_size
    last = w2.levels[-1]
    ids = last.page_ids.tolist()
    per = (cap + ps - 1) // ps
    assert len(ids) == wl.B * per and len(set(ids)) == len(ids)
    shared_ids = set(w2.levels[0].page_ids.tolist())
    assert not shared_ids & set(ids)
    # the visible keys are unchanged
    for a, b in zip(wl.levels[-1].nodes.tolist(), last.nodes.tolist()):
        assert a[2] == b[2]
        npg = (a[2] + ps - 1) // ps
        old = wl.levels[-1].page_ids[a[3]:a[3] + npg]
        assert torch.equal(wl.k_pool[old], w2.k_pool[last.page_ids[b[3]:b[3] + npg]])
    (q, k, v), = W.decode_tokens(w2, 1, seed=3)
    before = last.nodes[:, 2].clone()
    W.append_token(w2, k, v)
    assert torch.equal(last.nodes[:, 2], before + 1)
    for b in range(wl.B):
        t = int(before[b])
        page = ids[int(last.nodes[b, 3]) + t // ps]
        assert torch.equal(w2.k_pool[page, :, t % ps], k[b]) and torch.equal(w2.v_pool[page, :, t % ps], v[b])


def test_loop_binding_rejects_wrong_token_rows():
    """The new token's K and V rows are checked before the library is called:
    bf16 [B][Hkv][d], head dimension contiguous, on the GPU, equal strides."""
    class Plan:
        B, Hkv, d = 3, 2, 64

    k = torch.zeros(3, 2, 64, dtype=torch.bfloat16)
    for bad in (k.float(), k[:, :, ::2], k[:2], k):  # dtype, stride, shape, host memory
        with pytest.raises(ValueError):
            hb._check_token_rows(Plan, bad, bad)
    with pytest.raises(ValueError):
        hb.LoopPlan([], 1, 1, 1, 64, capacity=0)


# --------------------------------------------------- plan item invariants
def _check_plan_items(wl, capacity=0, num_sms=152):
    """Every key of every node is covered exactly once per (sequence, KV
    head), each item sits in the role its node's query rows call for
    (tensor cores above 16 rows), partial-row
    ranges are disjoint and inside the plan's, and each CTA runs its
    tensor-core items before its paged items."""
    levels = hb._levels_of(wl)
    items = hb.hp_cascade_plan_items(levels, wl.B, wl.Hq, wl.Hkv, wl.d, capacity=capacity, num_sms=num_sms)
    n_tc, n_small, n_part, _ = hb.hp_cascade_plan_stats(levels, wl.B, wl.Hq, wl.Hkv, wl.d, num_sms=num_sms) \
        if capacity == 0 else (None, None, None, None)
    G = wl.G
    last = len(wl.levels) - 1
    cover = {}
    total = {}
    spans = []
    prev_cta, seen_paged = -1, False
    for it in items:
        assert 0 <= it["cta"] < num_sms
        if it["cta"] != prev_cta:
            prev_cta, seen_paged = it["cta"], False
        node_rows = next((se - sb) * G for sb, se, _, _ in wl.levels[it["level"]].nodes.tolist()
                         if sb <= it["seq_begin"] < se)
        assert bool(it["tc"]) == (node_rows > 16), "role must follow the node's query rows"
        if it["tc"]:
            assert not seen_paged, "a tensor-core item after a paged item in one CTA"
            assert it["n_kvh"] == 1 and it["n_seq"] <= 2 * (128 // G)
            rows = -(-it["n_seq"] // (128 // G)) * 128
        else:
            seen_paged = True
            rows = it["n_seq"] * G * it["n_kvh"]
        assert 0 <= it["k0"] < it["k1"]
        loop_item = capacity > 0 and it["level"] == last
        assert it["len_seq"] == (it["seq_begin"] if loop_item else -1)
        spans.append((it["part_row"], it["part_row"] + rows))
        for b in range(it["seq_begin"], it["seq_begin"] + it["n_seq"]):
            for h in range(it["kvh"], it["kvh"] + it["n_kvh"]):
                cover.setdefault((it["level"], b, h), []).append((it["k0"], it["k1"]))
                total[(b, h)] = total.get((b, h), 0) + it["k1"] - it["k0"]
    spans.sort()
    for (a0, a1), (b0, _) in zip(spans, spans[1:]):
        assert a1 <= b0, "partial-row ranges overlap"
    if n_part is not None:
        assert spans[-1][1] <= n_part and len(items) == n_tc + n_small
    # per (level, sequence, head): one node (a tree node, or single-sequence
    # nodes of that sequence fused into the first of them), its keys covered
    # once from 0; per (sequence, head): every key of every node
    for key, rng in cover.items():
        rng = sorted(rng)
        assert rng[0][0] == 0, key
        for (x0, x1), (y0, _) in zip(rng, rng[1:]):
            assert x1 == y0, f"keys of (level, sequence, head) {key} not covered once"
    want_total = {}
    for l, lv in enumerate(wl.levels):
        for sb, se, kl, _ in lv.nodes.tolist():
            end = capacity if (capacity > 0 and l == last) else kl
            for b in range(sb, se):
                for h in range(wl.Hkv):
                    if end:
                        want_total[(b, h)] = want_total.get((b, h), 0) + end
    assert total == want_total
    # merge lists: row (b, kvh) merges exactly the partial rows of the items
    # covering it, at the item's row layout (tensor-core items: blocks of
    # 128 rows of 128 / G sequences; paged items: [head in group][sequence][g])
    tab = hb.hp_cascade_plan_merge_table(levels, wl.B, wl.Hq, wl.Hkv, wl.d, capacity=capacity, num_sms=num_sms)
    want = [[] for _ in range(wl.B * wl.Hkv)]
    spb = 128 // G
    for it in items:
        for b in range(it["seq_begin"], it["seq_begin"] + it["n_seq"]):
            s_ = b - it["seq_begin"]
            for h in range(it["kvh"], it["kvh"] + it["n_kvh"]):
                if it["tc"]:
                    row = it["part_row"] + (s_ // spb) * 128 + (s_ % spb) * G
                else:
                    row = it["part_row"] + ((h - it["kvh"]) * it["n_seq"] + s_) * G
                want[b * wl.Hkv + h].append(row)
    assert [sorted(x) for x in tab] == [sorted(x) for x in want]
    return items


@pytest.mark.parametrize("name", W.CONFIG_NAMES)
def test_plan_items_cover_every_key_once(name):
    wl = W.make_config(name, seed=0)
    items = _check_plan_items(wl)
    assert items


@pytest.mark.parametrize("seed", range(8))
def test_plan_items_on_random_trees(seed):
    import numpy as np
    rng = np.random.default_rng(100 + seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    B = int(rng.integers(1, 300))
    shared = []
    for _ in range(int(rng.integers(0, 4))):
        cuts = sorted(set(rng.integers(1, B, size=int(rng.integers(0, 6))).tolist())) if B > 1 else []
        bounds = [0] + cuts + [B]
        shared.append([(a, b, int(rng.integers(0, 3000))) for a, b in zip(bounds[:-1], bounds[1:])])
    wl = W.build_cascade(f"r{seed}", B=B, Hq=Hkv * G, Hkv=Hkv, d=int(rng.choice([64, 128])),
                         page_size=int(rng.choice([16, 32, 64])), shared=shared, suffix_range=(0, 400), seed=seed)
    _check_plan_items(wl, num_sms=int(rng.choice([16, 152])))


@pytest.mark.parametrize("name,kw,cap", [("llama3_8b", {}, 300), ("tree2", {}, 300), ("tiny", {}, 40),
                                         ("no_sharing", dict(B=16, prefix=512), 600)])
def test_loop_plan_items_reach_the_capacity(name, kw, cap):
    wl = W.with_suffix_capacity(W.make_config(name, seed=1, **kw), cap, seed=1)
    _check_plan_items(wl, capacity=cap)



def _chain_tree(seed, ps=16, mid=32, loop_cap=0):
    """A shared document, then one single-sequence node per sequence (a
    question of `mid` tokens), then the private suffixes."""
    B = 6
    return W.build_cascade(f"chain{seed}", B=B, Hq=8, Hkv=2, d=64, page_size=ps,
                           shared=[[(0, B, 100)], [(b, b + 1, mid) for b in range(B)]],
                           suffix_range=(1, 40), seed=seed)


def test_single_sequence_chains_are_fused():
    """A sequence's own question node (page-aligned) and its suffix are one
    planning node: its items sit at the question's level and cover both
    nodes' keys; none are left at the suffix's level.  A question that
    ends mid-page is not fused with a suffix (only the last fused node may
    end mid-page), nor is a growing decode-loop suffix."""
    wl = _chain_tree(0)
    items = _check_plan_items(wl)
    assert {it["level"] for it in items} == {0, 1}
    for b, (_, _, kl, _) in enumerate(wl.levels[2].nodes.tolist()):
        assert max(it["k1"] for it in items if it["level"] == 1 and it["seq_begin"] == b) == 32 + kl
    ragged = _chain_tree(0, mid=20)
    assert {it["level"] for it in _check_plan_items(ragged)} == {0, 1, 2}
    loop = W.with_suffix_capacity(wl, 64, seed=0)
    assert {it["level"] for it in _check_plan_items(loop, capacity=64)} == {0, 1, 2}


def _fused_by_seq(items):
    by_seq = {}
    for it in items:
        if it["n_seq"] == 1:
            by_seq.setdefault(it["seq_begin"], set()).add((it["level"], max(
                x["k1"] for x in items if x["n_seq"] == 1 and x["seq_begin"] == it["seq_begin"]
                and x["level"] == it["level"])))
    return by_seq


def test_chunkattention_fig2_private_chunks_are_planned_as_one():
    """In ChunkAttention's Figure 2 tree, sequence 1 owns chunks C4 then C6
    and sequence 2 owns C5 then C7 (one page each).  The context list keeps
    them apart, as the page lists it; with 64-token chunks and 32 KV heads
    (re-reading a shared chunk per sequence costs more than a merge part)
    the planner walks each private pair as one node of two pages at C4's /
    C5's level, and sequence 0's single C3 stays as it is."""
    pool = _pool()
    ps = 64
    g, levels, names = _fig2_levels(pool, ps=ps)
    items = hb.hp_cascade_plan_items(levels, 3, 32, 32, 128, num_sms=152)
    lvl = {names[k]: k[0] for k in names}
    by_seq = _fused_by_seq(items)
    assert by_seq[0] == {(lvl["C3"], ps)}
    assert by_seq[1] == {(lvl["C4"], 2 * ps)}
    assert by_seq[2] == {(lvl["C5"], 2 * ps)}


def test_chunkattention_fig2_narrow_shared_chunks_join_the_chains():
    """The same tree with 16-token chunks and 4 KV heads: re-reading the
    shared chunks C0, C1, C2 (three sequences each) per sequence costs less
    than their merge parts, so each sequence becomes one node at C0's level:
    C0 C1 C2 C3 for sequence 0, C0 C1 C2 C4 C6 and C0 C1 C2 C5 C7 for
    sequences 1 and 2."""
    pool = _pool()
    ps = 16
    g, levels, names = _fig2_levels(pool, ps=ps)
    items = hb.hp_cascade_plan_items(levels, 3, 4, 4, 128, num_sms=152)
    lvl = {names[k]: k[0] for k in names}
    assert all(it["n_seq"] == 1 for it in items)
    by_seq = _fused_by_seq(items)
    assert by_seq == {0: {(lvl["C0"], 4 * ps)}, 1: {(lvl["C0"], 5 * ps)}, 2: {(lvl["C0"], 5 * ps)}}
    # the chunks are read per sequence: no item covers two sequences
    tab = hb.hp_cascade_plan_merge_table(levels, 3, 4, 4, 128, num_sms=152)
    for row, parts in enumerate(tab):
        b, h = divmod(row, 4)
        mine = [it for it in items if it["seq_begin"] == b and it["kvh"] <= h < it["kvh"] + it["n_kvh"]]
        assert len(parts) == len(mine)  # one part per key range of the sequence's single node


def test_deep_trees_and_pool_slot_limit():
    """Up to 64 levels plan as long as at most 8 distinct pool sets serve
    them; 65 levels, or a ninth pool set, are rejected."""
    pool = _pool()
    node = [(0, 2, 16, 0)]
    deep = [(pool.data_ptr(), pool.data_ptr(), 8, 16, node, [0]) for _ in range(64)]
    assert hb.hp_cascade_plan_bytes(deep, 4, 4, 4, 128, num_sms=152) > 0
    assert hb.hp_cascade_plan_bytes(deep + deep[:1], 4, 4, 4, 128, num_sms=152) == 0
    bufs = [torch.zeros(64, dtype=torch.uint8) for _ in range(9)]
    eight = [(b.data_ptr(), b.data_ptr(), 8, 16, node, [0]) for b in bufs[:8]]
    assert hb.hp_cascade_plan_bytes(eight + eight[:4], 4, 4, 4, 128, num_sms=152) > 0
    nine = [(b.data_ptr(), b.data_ptr(), 8, 16, node, [0]) for b in bufs]
    assert hb.hp_cascade_plan_bytes(nine, 4, 4, 4, 128, num_sms=152) == 0
    # the same pools with another page size are another pool set
    other_ps = [(bufs[0].data_ptr(), bufs[0].data_ptr(), 8, 32, node, [0])]
    assert hb.hp_cascade_plan_bytes(eight[:7] + other_ps, 4, 4, 4, 128, num_sms=152) > 0
    assert hb.hp_cascade_plan_bytes(eight + other_ps, 4, 4, 4, 128, num_sms=152) == 0


# ------------------------------------------------ reduced-precision (E4M3) levels
@pytest.mark.parametrize("name,kw", [("llama3_8b", {}), ("tree2", dict(B=32, prefix=256)),
                                     ("codellama13b", dict(B=32, prefix=256)), ("no_sharing", {})])
def test_e4m3_suffix_plans_cover_every_key_once(name, kw):
    """Trees whose suffix level holds E4M3 codes plan like their bf16 twins:
    the same coverage, roles and merge lists."""
    wl = W.with_e4m3_levels(W.make_config(name, seed=0, **kw))
    items = _check_plan_items(wl)
    assert any(not it["tc"] for it in items)


def test_e4m3_levels_are_rejected_where_the_kernels_do_not_read_them():
    """E4M3 storage is for the per-sequence pass: a batched node in an E4M3
    level, a per-sequence node left in bf16 next to an E4M3 level, d = 64,
    missing scales and decode-loop plans are refused on the host."""
    wl = W.make_config("llama3_8b", seed=0, B=8, prefix=256)
    bad_tc = W.with_e4m3_levels(wl, levels=(0, -1))
    assert hb.hp_cascade_plan_bytes(hb._levels_of(bad_tc), wl.B, wl.Hq, wl.Hkv, wl.d, num_sms=152) == 0
    # a narrow shared node (4 sequences x G=4 = 16 rows: per-sequence pass) kept in bf16
    narrow = W.build_cascade("n", B=8, Hq=32, Hkv=8, d=128, page_size=16, shared=[[(0, 4, 64), (4, 8, 64)]],
                             suffix_range=(1, 40), seed=1)
    mixed = W.with_e4m3_levels(narrow, levels=(-1,))
    assert hb.hp_cascade_plan_bytes(hb._levels_of(mixed), 8, 32, 8, 128, num_sms=152) == 0
    both = W.with_e4m3_levels(narrow, levels=(0, -1))
    assert hb.hp_cascade_plan_bytes(hb._levels_of(both), 8, 32, 8, 128, num_sms=152) > 0
    tiny = W.with_e4m3_levels(W.make_config("tiny", seed=0))  # d = 64
    assert hb.hp_cascade_plan_bytes(hb._levels_of(tiny), tiny.B, tiny.Hq, tiny.Hkv, tiny.d, num_sms=152) == 0
    lv = hb._levels_of(W.with_e4m3_levels(wl))
    lv[-1] = lv[-1][:7] + (None, None)
    assert hb.hp_cascade_plan_bytes(lv, wl.B, wl.Hq, wl.Hkv, wl.d, num_sms=152) == 0
    cap = W.with_suffix_capacity(wl, 300)
    loop = W.with_e4m3_levels(cap)
    assert hb.hp_cascade_loop_plan_bytes(hb._levels_of(loop), wl.B, wl.Hq, wl.Hkv, wl.d, 300, num_sms=152) == 0
    assert hb.hp_cascade_loop_plan_bytes(hb._levels_of(cap), wl.B, wl.Hq, wl.Hkv, wl.d, 300, num_sms=152) > 0


def test_e4m3_unique_bytes_and_quantiser():
    """An E4M3 level stores one byte per element plus two f32 scales per
    (page, KV head); the quantiser's scales map each slice's largest
    magnitude to 448, and decoding its codes stays within half an E4M3 step."""
    wl = W.make_config("llama3_8b", seed=0, B=8, prefix=64)
    w8 = W.with_e4m3_levels(wl)
    assert [lv.e4m3 for lv in w8.levels] == [False, True]
    ps = wl.page_size
    suf = wl.levels[-1].nodes.tolist()
    toks = sum(n[2] for n in suf)
    pages = sum((n[2] + ps - 1) // ps for n in suf)
    assert w8.unique_kv_bytes() == 64 * wl.Hkv * wl.d * 4 + toks * wl.Hkv * wl.d * 2 + pages * wl.Hkv * 8
    q8 = w8.q8
    x = wl.k_pool.float()
    amax = x.abs().amax(dim=(2, 3))
    assert torch.allclose(q8.k_scale * 448.0, amax, rtol=1e-6)
    dec = q8.k.view(torch.float8_e4m3fn).float() * q8.k_scale[:, :, None, None]
    # relative step of E4M3 is 2^-3 in the normal range: error <= 2^-4 of the value's binade
    err = (dec - x).abs()
    assert (err <= x.abs() * 2.0 ** -4 + q8.k_scale[:, :, None, None] * 2.0 ** -10).all()


# ------------------------------------------------ Parallel Prompting rows
def test_stream_rows_paged_layout():
    """Each request's row sits in its pages slot by slot, with its stream
    ids and positions; slots past the row are never visible (-2)."""
    req = W.stream_requests(R=3, P=4, Hq=4, Hkv=2, d=64, doc_len=37, q_len_range=(1, 9), T=3, seed=2)
    rows = W.stream_rows_paged(req, page_size=16, seed=1)
    for r, (sid, pos, k, v) in enumerate(req.rows):
        nk = sid.numel()
        assert int(rows.row_len[r]) == nk
        for t in range(nk):
            page = int(rows.row_pages[r, t // 16])
            assert torch.equal(rows.k_pool[page, :, t % 16], k[t]) and torch.equal(rows.v_pool[page, :, t % 16], v[t])
        assert torch.equal(rows.slot_sid[r, :nk], sid) and torch.equal(rows.slot_pos[r, :nk], pos)
        assert (rows.slot_sid[r, nk:] == -2).all()
    assert rows.slot_sid.shape[1] % 4 == 0 and rows.slot_sid.shape[1] >= rows.row_pages.shape[1] * 16
    assert rows.q_sid.tolist() == [s for _ in range(3) for s in range(4)]


def test_stream_workspace_sizes_and_rejections():
    assert hb.stream_workspace_bytes(2, 16, 32, 32, 128, 40, 16) > 0
    assert hb.stream_workspace_bytes(2, 64, 32, 8, 128, 40, 16) > 0
    assert hb.stream_workspace_bytes(0, 16, 32, 32, 128, 40, 16) == 0
    assert hb.stream_workspace_bytes(2, 16, 32, 32, 96, 40, 16) == 0
    assert hb.stream_workspace_bytes(2, 16, 64, 2, 128, 40, 16) == 0  # 32 query heads per KV head


def test_host_workspace_bytes():
    """hp_cascade_host_workspace_bytes: the step's workspace rounded up to
    256 bytes, then a B x Hq x d bf16 copy of q; 0 for an invalid info."""
    info = hb.HpPlanInfo()
    info.B, info.Hq, info.Hkv, info.d, info.ws_bytes = 64, 32, 8, 128, 1000
    assert hb.library().hp_cascade_host_workspace_bytes(ctypes.byref(info)) == 1024 + 64 * 32 * 128 * 2
    info.ws_bytes = 4096
    assert hb.library().hp_cascade_host_workspace_bytes(ctypes.byref(info)) == 4096 + 64 * 32 * 128 * 2
    info.d = 96
    assert hb.library().hp_cascade_host_workspace_bytes(ctypes.byref(info)) == 0
    assert hb.library().hp_cascade_host_workspace_bytes(None) == 0


def test_e4m3_paged_work_split_into_about_four_items_per_cta():
    """The per-sequence-only workload (B=64, 32 heads, 2048 tokens each):
    bf16 paged items are about one per CTA (HBM-bound, fewer partial states),
    E4M3 ones about four per CTA (consumer-bound, spread evenly); a short
    E4M3 workload keeps one per CTA."""
    bf = W.make_config("no_sharing", seed=2)
    q8 = W.with_e4m3_levels(bf)
    _, n_bf, _, _ = hb.hp_cascade_plan_stats(hb._levels_of(bf), bf.B, bf.Hq, bf.Hkv, bf.d)
    _, n_q8, _, _ = hb.hp_cascade_plan_stats(hb._levels_of(q8), q8.B, q8.Hq, q8.Hkv, q8.d)
    assert n_bf == 256 and 4 * 152 * 0.9 <= n_q8 <= 4 * 152 * 1.4
    short = W.with_e4m3_levels(W.make_config("no_sharing", seed=2, B=16, prefix=400))
    _, n_short, _, _ = hb.hp_cascade_plan_stats(hb._levels_of(short), short.B, short.Hq, short.Hkv, short.d)
    assert n_short <= 2 * 152
