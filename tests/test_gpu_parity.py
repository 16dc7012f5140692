"""GPU parity: every entry point of the C ABI against the fp64 oracle on the
same seeded inputs.

Tolerances: O max-abs <= 2e-2 and mean-abs <= 2e-3, LSE abs <= 1e-3 for bf16
inputs (the stated accuracy bar); merge of f32 states within f32 rounding;
index probes bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from shared_prefix_decode_gb300 import binding as hb
from shared_prefix_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_ABS = 2e-2, 2e-3, 1e-3
DEV = "cuda"


def _check(out, lse, O, L, what=""):
    o = out.double().cpu().numpy().reshape(O.shape)
    l = lse.double().cpu().numpy().reshape(L.shape)
    fin = np.isfinite(L)
    assert np.array_equal(np.isfinite(l), fin), f"{what}: empty rows differ"
    assert np.all(l[~fin] == -np.inf) and np.all(o[~fin] == 0), f"{what}: empty rows must be (0, -inf)"
    d_o = np.abs(o - O)
    d_l = np.abs(l[fin] - L[fin]) if fin.any() else np.zeros(1)
    assert d_o.max() <= O_MAX, f"{what}: max|dO| {d_o.max():.3g}"
    assert d_o.mean() <= O_MEAN, f"{what}: mean|dO| {d_o.mean():.3g}"
    assert d_l.max() <= LSE_ABS, f"{what}: max|dLSE| {d_l.max():.3g}"
    return float(d_o.max()), float(d_l.max())


def _status_ok(ws):
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(ws) == hb.HP_OK


# ------------------------------------------------------------------ merge
@pytest.mark.parametrize("d", [64, 128, 100])
def test_merge_states(d):
    g = torch.Generator().manual_seed(d)
    rows = 1000
    oa, ob = torch.randn(rows, d, generator=g), torch.randn(rows, d, generator=g)
    la, lb = torch.randn(rows, generator=g) * 5, torch.randn(rows, generator=g) * 5
    la[:10] = -math.inf          # first part empty
    lb[10:20] = -math.inf        # second part empty
    la[20:25] = lb[20:25] = -math.inf  # both empty
    lb[25:30] = la[25:30] + 80   # far apart
    O, L = oracle.merge(oa.numpy(), la.numpy(), ob.numpy(), lb.numpy())
    out, lse = hb.hp_merge_states(oa.to(DEV), la.to(DEV), ob.to(DEV), lb.to(DEV))
    o, l = out.cpu().double().numpy(), lse.cpu().double().numpy()
    np.testing.assert_allclose(o, O, atol=2e-6, rtol=1e-5)
    fin = np.isfinite(L)
    np.testing.assert_allclose(l[fin], L[fin], atol=2e-5)
    assert np.all(l[~fin] == -np.inf) and np.all(o[~fin] == 0)
    # in place, and bf16 output
    oa_d = oa.to(DEV)
    hb.hp_merge_states(oa_d, la.to(DEV), ob.to(DEV), lb.to(DEV), out=oa_d)
    np.testing.assert_allclose(oa_d.cpu().double().numpy(), O, atol=2e-6, rtol=1e-5)
    ob16, _ = hb.hp_merge_states(oa.to(DEV), la.to(DEV), ob.to(DEV), lb.to(DEV), out_dtype=torch.bfloat16)
    np.testing.assert_allclose(ob16.cpu().double().numpy(), O, atol=2e-2)


# ---------------------------------------------------- paged decode (suffix)
def _paged_case(name, seed, **kw):
    wl = W.make_config(name, seed=seed, **kw)
    pt, sl = W.full_page_tables(wl)
    return wl, pt, sl


@pytest.mark.parametrize("name,kw", [
    ("tiny", {}),
    ("llama3_8b", dict(B=6, prefix=256)),
    ("codellama13b", dict(B=3, prefix=128)),
    ("tree2", dict(B=16, prefix=256)),
    ("no_sharing", dict(B=4, prefix=300)),
])
@pytest.mark.parametrize("seed", [0, 1])
def test_suffix_decode_paged(name, kw, seed):
    wl, pt, sl = _paged_case(name, seed, **kw)
    O, L = oracle.paged_decode(wl.q, wl.k_pool, wl.v_pool, pt, sl, wl.scale)
    wg = wl.to(DEV)
    ws = hb.alloc_workspace(hb.suffix_workspace_bytes(wl.B, wl.Hq, wl.d, pt.shape[1], wl.page_size), DEV)
    out, lse = hb.hp_suffix_decode_paged(wg.q, wg.k_pool, wg.v_pool, pt.to(DEV), sl.to(DEV), wl.scale,
                                         ws=ws, out_dtype=torch.float32)
    _status_ok(ws)
    _check(out, lse, O, L, f"paged {name}")


def test_suffix_decode_edge_lengths():
    """Lengths 0, 1, 15, 16, 17, a full table, and a page table wider than
    needed; G = 4 and d = 128."""
    lens = [0, 1, 15, 16, 17, 33, 64, 127]
    wl = W.build_cascade("e", B=len(lens), Hq=8, Hkv=2, d=128, page_size=16, shared=[],
                         suffix_lens=lens, seed=3)
    pt, sl = W.full_page_tables(wl)
    pt = torch.cat([pt, torch.zeros(pt.shape[0], 3, dtype=torch.int32)], 1)
    O, L = oracle.paged_decode(wl.q, wl.k_pool, wl.v_pool, pt, sl, wl.scale)
    wg = wl.to(DEV)
    out, lse = hb.hp_suffix_decode_paged(wg.q, wg.k_pool, wg.v_pool, pt.to(DEV), sl.to(DEV), wl.scale,
                                         out_dtype=torch.float32)
    torch.cuda.synchronize()
    _check(out, lse, O, L, "edge lengths")


def test_suffix_decode_bad_page_sets_bounds_status():
    wl = W.build_cascade("x", B=2, Hq=4, Hkv=1, d=64, page_size=16, shared=[], suffix_lens=[40, 20], seed=1)
    pt, sl = W.full_page_tables(wl)
    pt[0, 1] = wl.num_pages + 5  # out of range
    wg = wl.to(DEV)
    ws = hb.alloc_workspace(hb.suffix_workspace_bytes(2, 4, 64, pt.shape[1], 16), DEV)
    out, lse = hb.hp_suffix_decode_paged(wg.q, wg.k_pool, wg.v_pool, pt.to(DEV), sl.to(DEV), wl.scale, ws=ws)
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(ws) == hb.HP_ERR_BOUNDS
    assert torch.isfinite(out.float()).all()
    # sequence 1 is untouched by the bad page
    O, L = oracle.paged_decode(wl.q[1:], wl.k_pool, wl.v_pool, pt[1:], sl[1:], wl.scale)
    _check(out[1:], lse[1:], O, L, "bounds: clean row")
    # the status word was cleared by the read
    assert hb.hp_read_device_status(ws) == hb.HP_OK


# ---------------------------------------------------- contiguous prefix
def _contig_prefix(wl):
    ids = wl.levels[0].page_ids.long()
    kv_len = int(wl.levels[0].nodes[0, 2])
    k = wl.k_pool[ids].permute(0, 2, 1, 3).reshape(-1, wl.Hkv, wl.d)[:kv_len].contiguous()
    v = wl.v_pool[ids].permute(0, 2, 1, 3).reshape(-1, wl.Hkv, wl.d)[:kv_len].contiguous()
    return k, v


@pytest.mark.parametrize("Hq,Hkv,d,B,P", [
    (4, 1, 64, 4, 256),      # GQA 4, 16 rows
    (32, 8, 128, 64, 4096),  # Llama-3-8B shape, 256 rows per KV head
    (32, 8, 128, 10, 1000),  # ragged tail tile, 40 rows
    (8, 8, 128, 300, 384),   # MHA, 300 rows -> two row chunks
    (16, 2, 64, 33, 130),    # G = 8, d = 64, tail of 2 keys
])
def test_prefix_attn(Hq, Hkv, d, B, P):
    g = torch.Generator().manual_seed(B + P)
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(P, Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(P, Hkv, d, generator=g).to(torch.bfloat16)
    scale = 1 / math.sqrt(d)
    O, L = oracle.prefix(q, k, v, scale)
    out, lse = hb.hp_prefix_attn(q.to(DEV), k.to(DEV), v.to(DEV), scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    _check(out, lse, O, L, f"prefix {Hq}/{Hkv}/{d} B={B} P={P}")


@pytest.mark.parametrize("d,Hq,Hkv,B", [(128, 4, 1, 40), (64, 8, 2, 20)])
def test_prefix_attn_running_max_rescale(d, Hq, Hkv, B):
    """Scores that grow by about 17 log2 units from one 128-key tile to the
    next: every tile moves the reference max past the lazy-rescale threshold,
    so O is rescaled in TMEM at every tile."""
    g = torch.Generator().manual_seed(11 + d)
    P, scale = 1024, 1 / math.sqrt(d)
    base = torch.randn(d, generator=g)
    base = base / base.norm() * 4.0
    q = (base + 0.1 * torch.randn(B, Hq, d, generator=g)).to(torch.bfloat16)
    ramp = (torch.arange(P) // 128).float() * 12.0 / scale  # + 12 natural units per tile
    k = torch.randn(P, Hkv, d, generator=g) + (ramp[:, None, None] * base / base.norm() ** 2)
    k = k.to(torch.bfloat16)
    v = torch.randn(P, Hkv, d, generator=g).to(torch.bfloat16)
    O, L = oracle.prefix(q, k, v, scale)
    out, lse = hb.hp_prefix_attn(q.to(DEV), k.to(DEV), v.to(DEV), scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    _check(out, lse, O, L, f"rescale d={d}")


def test_prefix_attn_row_window_and_strides():
    """rows [3, 3+20) only; K/V as a strided view of a wider [len][2*Hkv][d]."""
    g = torch.Generator().manual_seed(5)
    B, Hq, Hkv, d, P = 30, 8, 2, 128, 640
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16)
    kw = torch.randn(P, 2 * Hkv, d, generator=g).to(torch.bfloat16)
    vw = torch.randn(P, 2 * Hkv, d, generator=g).to(torch.bfloat16)
    k, v = kw[:, ::2], vw[:, ::2]
    O, L = oracle.prefix(q[3:23], k.contiguous(), v.contiguous(), 0.1)
    out = torch.full((B, Hq, d), 7.0, device=DEV)
    lse = torch.full((B, Hq), 7.0, device=DEV)
    kd, vd = kw.to(DEV)[:, ::2], vw.to(DEV)[:, ::2]
    hb.hp_prefix_attn(q.to(DEV), kd, vd, 0.1, row_begin=3, rows=20, out=out, lse=lse)
    torch.cuda.synchronize()
    _check(out[3:23], lse[3:23], O, L, "row window")
    assert torch.all(out[:3] == 7.0) and torch.all(out[23:] == 7.0)


def test_prefix_attn_empty_prefix():
    q = torch.randn(4, 4, 64).to(torch.bfloat16).to(DEV)
    k = torch.zeros(0, 1, 64, dtype=torch.bfloat16, device=DEV)
    out, lse = hb.hp_prefix_attn(q, k, k, 0.125, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(lse == -math.inf)


# ------------------------------------------------------------- cascade
SMALL_CASES = [
    ("tiny", {}),
    ("llama3_8b", dict(B=8, prefix=512)),
    ("codellama13b", dict(B=12, prefix=384)),
    ("tree2", dict(B=32, prefix=256)),
    ("doc_streams", dict(B=20, prefix=640)),
    ("no_sharing", dict(B=6, prefix=200)),
]


@pytest.mark.parametrize("name,kw", SMALL_CASES)
@pytest.mark.parametrize("seed", [0, 1, 2, 3, 4])
def test_cascade_small(name, kw, seed):
    wl = W.make_config(name, seed=seed, **kw)
    O, L = oracle.cascade(wl)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    out, lse = plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
    _status_ok(plan.ws)
    _check(out, lse, O, L, f"cascade {name} seed {seed}")


def test_cascade_llama3_full_all_rows():
    """The benchmarked workload at full size: B=64, 32/8 heads, d=128, 4K
    prefix, suffixes U[1,256], shuffled 16-token pages; every output row."""
    for seed in (0, 1):
        wl = W.make_config("llama3_8b", seed=seed)
        O, L = oracle.cascade(wl)
        wg = wl.to(DEV)
        plan = hb.CascadePlan.from_workload(wg)
        out, lse = plan.decode(wg.q, wl.scale)  # bf16 output, as benchmarked
        _status_ok(plan.ws)
        _check(out, lse, O, L, f"llama3 full seed {seed}")


def _sample_rows(wl, n, seed):
    g = torch.Generator().manual_seed(seed)
    bs = torch.randint(0, wl.B, (n,), generator=g).tolist()
    hs = torch.randint(0, wl.Hq, (n,), generator=g).tolist()
    rows = sorted(set(zip(bs, hs)) | {(0, 0), (wl.B - 1, wl.Hq - 1)})
    return rows


@pytest.mark.parametrize("name", ["codellama13b", "tree2", "doc_streams", "no_sharing"])
def test_cascade_full_size_all_rows(name):
    """Every output row of the full-size workload, seed 0."""
    wl = W.make_config(name, seed=0)
    O, L = oracle.cascade(wl)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    out, lse = plan.decode(wg.q, wl.scale)
    _status_ok(plan.ws)
    _check(out, lse, O, L, f"{name} full, every row")


@pytest.mark.parametrize("name", ["codellama13b", "tree2", "doc_streams", "no_sharing"])
@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_cascade_full_size_sampled(name, seed):
    wl = W.make_config(name, seed=seed)
    rows = _sample_rows(wl, 96, 7 + seed)
    O, L = oracle.cascade(wl, rows)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    out, lse = plan.decode(wg.q, wl.scale)
    _status_ok(plan.ws)
    idx_b = torch.tensor([r[0] for r in rows])
    idx_h = torch.tensor([r[1] for r in rows])
    _check(out.cpu()[idx_b, idx_h], lse.cpu()[idx_b, idx_h], O, L, f"{name} full sampled")
    # property at any size: every row is finite and its LSE at least the
    # largest single score bound log(1) for a non-empty key set is finite
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


# ------------------------------------------------- bit-exact index probes
def _nodes_of(wl, b):
    """(level, node index, seq_begin, kv_len, offset of the node in b's
    context) of every node covering sequence b, in level order."""
    out, off = [], 0
    for li, lv in enumerate(wl.levels):
        for i, (sb, se, kl, _) in enumerate(lv.nodes.tolist()):
            if sb <= b < se:
                out.append((li, i, sb, kl, off))
                off += kl
                break
    return out


def _probe_targets(wl, where):
    """Collision-free probe targets, one per sequence, by rule (no fallback):
    the i-th sequence of a node probes token i-derived slots of it, so two
    sequences never probe the same stored token.
      first:     each sequence its first non-empty node, token i (every node's
                 first token is probed by the node's first sequence);
      last:      its last non-empty node, token kv_len - 1 - i;
      page_edge: the node at level b mod depth, token i*ps + (ps - 1 if b is
                 odd else 0); when that passes the node's end, the same edge of
                 its private node;
      level<k>:  its node at level k, token i (every node of level k probed)."""
    ps = wl.page_size
    tg = []
    for b in range(wl.B):
        nodes = [n for n in _nodes_of(wl, b) if n[3] > 0]
        if where == "first":
            li, _, sb, kl, off = nodes[0]
            t = b - sb
        elif where == "last":
            li, _, sb, kl, off = nodes[-1]
            t = kl - 1 - (b - sb)
        elif where == "page_edge":
            li, _, sb, kl, off = nodes[b % len(nodes)]
            t = (b - sb) * ps + (ps - 1 if b % 2 else 0)
            if t >= kl:
                li, _, sb, kl, off = next(n for n in nodes if n[2] == b and wl.levels[n[0]].nodes[n[1], 1] == b + 1)
                t = min(kl - 1, ps - 1 if b % 2 else 0)
        elif where.startswith("level"):
            k = int(where[5:])
            li, _, sb, kl, off = next(n for n in nodes if n[0] == k)
            t = b - sb
        else:
            raise ValueError(where)
        assert 0 <= t < kl, (where, b, t, kl)
        tg.append(off + t)
    return tg


def _distinct_targets(wl, seed):
    """One target per sequence, spread over every level; targets inside a
    shared node are distinct tokens so no two sequences' probes collide."""
    g = torch.Generator().manual_seed(seed)
    n = wl.seq_kv_len()
    used = set()
    tg = []
    for b in range(wl.B):
        for _ in range(1000):
            t = int(torch.randint(0, n[b], (1,), generator=g))
            # locate (level, node) to test collision on shared tokens
            off, key = t, None
            for li, lv in enumerate(wl.levels):
                hit = [(i, nd) for i, nd in enumerate(lv.nodes.tolist()) if nd[0] <= b < nd[1]]
                if not hit:
                    continue
                i, nd = hit[0]
                if off < nd[2]:
                    key = (li, i, off)
                    break
                off -= nd[2]
            if key not in used:
                used.add(key)
                tg.append(t)
                break
    return tg


def _run_probe(wl, tg, what):
    W.apply_probe(wl, tg)  # raises if two targets share a stored token
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    out, lse = plan.decode(wg.q, wl.scale)  # bf16 output
    _status_ok(plan.ws)
    out = out.cpu()
    for b in range(wl.B):
        want = W.probe_expected(b, wl.d)
        got = out[b]
        bad = (got.view(torch.int16) != want.view(torch.int16)[None, :]).any(dim=1)
        assert not bad.any(), f"{what}: sequence {b} (target {tg[b]}) heads {bad.nonzero().flatten().tolist()}"


PROBE_CASES = [
    ("tiny", {}),
    ("llama3_8b", dict(B=16, prefix=512)),
    ("tree2", dict(B=32, prefix=256)),
    ("codellama13b", dict(B=8, prefix=256)),
    ("doc_streams", dict(B=24, prefix=320)),
]


@pytest.mark.parametrize("name,kw", PROBE_CASES)
@pytest.mark.parametrize("mode", ["random", "first", "last", "page_edge"])
def test_probe_bit_exact(name, kw, mode):
    wl = W.make_config(name, seed=11, **kw)
    tg = _distinct_targets(wl, 3) if mode == "random" else _probe_targets(wl, mode)
    _run_probe(wl, tg, f"{name} {mode}")


@pytest.mark.parametrize("level", [0, 1, 2])
def test_probe_bit_exact_every_node_of_each_tree2_level(level):
    """tree2 at B=32: level 0 (one node), level 1 (8 nodes of 4 sequences),
    level 2 (the suffixes): every node's tokens probed by its sequences."""
    wl = W.make_config("tree2", seed=12, B=32, prefix=256)
    tg = _probe_targets(wl, f"level{level}")
    _run_probe(wl, tg, f"tree2 level {level}")


@pytest.mark.parametrize("mode", ["first", "last", "page_edge"])
def test_probe_bit_exact_codellama13b_full_batch(mode):
    """B = 256 sequences at G = 1: the shared node's 256 query rows run on
    the tensor cores (two 128-row blocks), probed bit for bit."""
    wl = W.make_config("codellama13b", seed=13, prefix=1024)
    tg = _probe_targets(wl, mode)
    _run_probe(wl, tg, f"codellama13b B=256 {mode}")


def test_probe_bit_exact_paged_decode():
    wl = W.make_config("llama3_8b", seed=2, B=8, prefix=256)
    W.apply_probe(wl, _distinct_targets(wl, 9))
    pt, sl = W.full_page_tables(wl)
    wg = wl.to(DEV)
    out, _ = hb.hp_suffix_decode_paged(wg.q, wg.k_pool, wg.v_pool, pt.to(DEV), sl.to(DEV), wl.scale)
    torch.cuda.synchronize()
    out = out.cpu()
    for b in range(wl.B):
        assert torch.equal(out[b].view(torch.int16), W.probe_expected(b, wl.d).view(torch.int16)[None].expand(wl.Hq, -1))


# -------------------------------------------- determinism, graphs, plans
def test_cascade_deterministic_and_graph_replay():
    wl = W.make_config("llama3_8b", seed=4, B=16, prefix=1024)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    o1, l1 = plan.decode(wg.q, wl.scale)
    o2, l2 = plan.decode(wg.q, wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    out = torch.empty_like(o1)
    lse = torch.empty_like(l1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan.decode(wg.q, wl.scale, out=out, lse=lse)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g):
        plan.decode(wg.q, wl.scale, out=out, lse=lse)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, o1) and torch.equal(lse, l1)
    # new queries in the same buffer, replay again
    wg.q.copy_(torch.randn_like(wg.q, dtype=torch.float32).to(torch.bfloat16))
    g.replay()
    o3, l3 = plan.decode(wg.q, wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, o3) and torch.equal(lse, l3)


def test_cascade_stale_plan_info_is_reported():
    wl = W.make_config("tiny", seed=0)
    wg = wl.to(DEV)
    p1 = hb.CascadePlan.from_workload(wg)
    p2 = hb.CascadePlan.from_workload(wg)
    p1.info.tag = p2.info.tag  # info of another plan
    p1.decode(wg.q, wl.scale)
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(p1.ws) == hb.HP_ERR_ARG


def test_cascade_matches_naive_per_sequence_decode():
    """The cascade result equals per-sequence paged decode over the whole
    context (the prefix re-read per sequence), within the same tolerance."""
    wl = W.make_config("llama3_8b", seed=3, B=16, prefix=1024)
    pt, sl = W.full_page_tables(wl)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    oc, lc = plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
    on, ln = hb.hp_suffix_decode_paged(wg.q, wg.k_pool, wg.v_pool, pt.to(DEV), sl.to(DEV), wl.scale,
                                       out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert (oc - on).abs().max().item() <= O_MAX
    assert (lc - ln).abs().max().item() <= LSE_ABS


def test_cascade_device_timeout_is_reported_and_the_context_stays_usable():
    """Failure detection without a fault: with hp_test_withhold_first_tile on,
    one CTA arms a tile barrier but issues no copy, so its bounded waits (2 s of
    %globaltimer) run out; the kernel drains, frees its tensor memory and
    returns, and the step reports HP_ERR_DEVICE_TIMEOUT through the status
    word.  The next step on the same workspace is correct."""
    wl = W.make_config("llama3_8b", seed=2, B=8, prefix=512)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    assert plan.info.n_tc_items > 0  # CTA 0 runs a tensor-core item
    hb.library().hp_test_withhold_first_tile(1)
    try:
        plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        hb.library().hp_test_withhold_first_tile(0)
    assert hb.hp_read_device_status(plan.ws) == hb.HP_ERR_DEVICE_TIMEOUT
    out, lse = plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
    _status_ok(plan.ws)
    O, L = oracle.cascade(wl)
    _check(out, lse, O, L, "after a device timeout")


def _random_tree(seed):
    """A random cascade: 1-3 shared levels, each a random partition of the
    sequences into contiguous nodes (lengths 0..300, some single-sequence),
    private suffixes 0..100, random GQA group size, head dim and page size."""
    rng = np.random.default_rng(seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    ps = int(rng.choice([16, 32, 64]))
    B = int(rng.integers(1, 41))
    shared = []
    for _ in range(int(rng.integers(1, 4))):
        cuts = sorted(set(rng.integers(1, B, size=int(rng.integers(0, 4))).tolist())) if B > 1 else []
        bounds = [0] + cuts + [B]
        shared.append([(a, b, int(rng.integers(0, 301))) for a, b in zip(bounds[:-1], bounds[1:])])
    return W.build_cascade(f"random{seed}", B=B, Hq=Hkv * G, Hkv=Hkv, d=d, page_size=ps, shared=shared,
                           suffix_range=(0, 100), seed=seed)


@pytest.mark.parametrize("seed", range(12))
def test_cascade_random_trees(seed):
    """Irregular trees through the whole path (planner, both roles, merge):
    every output row against the oracle."""
    wl = _random_tree(seed)
    O, L = oracle.cascade(wl)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    out, lse = plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
    _status_ok(plan.ws)
    _check(out, lse, O, L, f"random tree {seed}: B={wl.B} Hq={wl.Hq} Hkv={wl.Hkv} d={wl.d} ps={wl.page_size}")


# ------------------------------------------------------------ decode loop
def _loop_host(name, kw, steps, seed):
    if name == "edges":
        # suffixes of length 0, 1 and at page edges; capacity just covers the loop
        wl = W.build_cascade("edges", B=6, Hq=8, Hkv=2, d=128, page_size=16, shared=[[(0, 6, 100)]],
                             suffix_lens=[0, 1, 15, 16, 17, 33], seed=seed)
    else:
        wl = W.make_config(name, seed=seed, **kw)
    cap = int(wl.levels[-1].nodes[:, 2].max()) + steps
    return W.with_suffix_capacity(wl, cap, seed=seed), cap


@pytest.mark.parametrize("name,kw,steps", [
    ("llama3_8b", dict(B=8, prefix=512), 40),
    ("tiny", {}, 24),
    ("tree2", dict(B=16, prefix=128), 20),
    ("no_sharing", dict(B=4, prefix=100), 20),
    ("edges", {}, 34),
])
def test_decode_loop_matches_oracle_every_step(name, kw, steps):
    """A decode loop through the C ABI: each step appends one token per
    sequence into its suffix pages and attends over the grown suffixes with
    the plan built once.  Every step's rows against the oracle over the same
    tree with the token appended on the host; at the end the device pools and
    lengths equal the host's, byte for byte."""
    host, cap = _loop_host(name, kw, steps, seed=5)
    dev = host.to(DEV)
    plan = hb.LoopPlan.from_workload(dev, cap)
    for s, (q, k, v) in enumerate(W.decode_tokens(host, steps, seed=5)):
        plan.append(k.to(DEV), v.to(DEV))
        out, lse = plan.decode(q.to(DEV), host.scale, out_dtype=torch.float32)
        W.append_token(host, k, v)
        host.q = q
        O, L = oracle.cascade(host)
        _check(out, lse, O, L, f"decode loop {name} step {s}")
    _status_ok(plan.ws)
    assert torch.equal(plan.suffix_len.cpu(), host.levels[-1].nodes[:, 2])
    assert torch.equal(dev.k_pool.cpu(), host.k_pool) and torch.equal(dev.v_pool.cpu(), host.v_pool)


def test_decode_loop_as_one_graph():
    """A 32-step loop (append + decode per step) captured as one CUDA graph
    and replayed from the same starting state gives the eager loop's results
    bit for bit."""
    steps = 32
    host, cap = _loop_host("llama3_8b", dict(B=8, prefix=256), steps, seed=9)
    toks = W.decode_tokens(host, steps, seed=9)
    qs, ks, vs = (torch.stack([t[i] for t in toks]).to(DEV) for i in range(3))
    dev = host.to(DEV)
    plan = hb.LoopPlan.from_workload(dev, cap)
    k0, v0, n0 = dev.k_pool.clone(), dev.v_pool.clone(), plan.suffix_len.clone()
    B, Hq, d = host.B, host.Hq, host.d
    oe = torch.empty(steps, B, Hq, d, device=DEV)
    le = torch.empty(steps, B, Hq, device=DEV)
    for s in range(steps):
        plan.append(ks[s], vs[s])
        plan.decode(qs[s], host.scale, out=oe[s], lse=le[s])
    torch.cuda.synchronize()
    _status_ok(plan.ws)
    og, lg = torch.zeros_like(oe), torch.zeros_like(le)

    def reset():
        dev.k_pool.copy_(k0)
        dev.v_pool.copy_(v0)
        plan.suffix_len.copy_(n0)

    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        reset()
        plan.append(ks[0], vs[0])  # warm-up on the capture stream
        plan.decode(qs[0], host.scale, out=og[0], lse=lg[0])
    torch.cuda.current_stream().wait_stream(st)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for s in range(steps):
            plan.append(ks[s], vs[s])
            plan.decode(qs[s], host.scale, out=og[s], lse=lg[s])
    for _ in range(2):
        reset()
        og.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(og, oe) and torch.equal(lg, le)
        assert torch.equal(plan.suffix_len, n0 + steps)
    _status_ok(plan.ws)
    # the same loop with the append fused into each step, as one graph
    gf = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gf):
        for s in range(steps):
            plan.decode_append(qs[s], ks[s], vs[s], host.scale, out=og[s], lse=lg[s])
    for _ in range(2):
        reset()
        og.zero_()
        gf.replay()
        torch.cuda.synchronize()
        assert torch.equal(og, oe) and torch.equal(lg, le)
        assert torch.equal(plan.suffix_len, n0 + steps)
    _status_ok(plan.ws)


def test_decode_loop_length_errors_are_reported():
    """Lengths the loop plan cannot serve are reported through the status
    word, inside the reserved pages: an append at the capacity writes nothing
    and keeps the length; a decode with a length below the plan-time suffix
    (here 0) flags HP_ERR_BOUNDS.  A loop plan through the plain decode call,
    and a plain plan through the loop calls, are argument errors."""
    host, cap = _loop_host("llama3_8b", dict(B=4, prefix=128), 4, seed=2)
    dev = host.to(DEV)
    plan = hb.LoopPlan.from_workload(dev, cap)
    (q, k, v), = W.decode_tokens(host, 1, seed=2)
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    full = plan.suffix_len.clone()
    full[1] = cap
    plan.suffix_len.copy_(full)
    kp = dev.k_pool.clone()
    plan.append(k, v)
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(plan.ws) == hb.HP_ERR_BOUNDS
    n = plan.suffix_len.cpu()
    assert n[1] == cap and n[0] == full[0] + 1
    changed = (dev.k_pool != kp).flatten(1).any(1).nonzero().flatten().tolist()
    assert len(changed) == 3  # one page for each of the other three sequences
    plan.decode(q, host.scale)  # length == capacity is valid
    _status_ok(plan.ws)
    # the fused step at the capacity: nothing written for that sequence, its
    # length kept, the others appended
    kp = dev.k_pool.clone()
    before = plan.suffix_len.clone()
    plan.decode_append(q, k, v, host.scale)
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(plan.ws) == hb.HP_ERR_BOUNDS
    n = plan.suffix_len.cpu()
    assert n[1] == cap and torch.equal(n[[0, 2, 3]], before.cpu()[[0, 2, 3]] + 1)
    assert len((dev.k_pool != kp).flatten(1).any(1).nonzero()) == 3
    low = plan.suffix_len.clone()
    low[2] = 0
    hb.hp_cascade_decode_loop(plan, q, host.scale, suffix_len=low)
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(plan.ws) == hb.HP_ERR_BOUNDS
    with pytest.raises(hb.HpError):
        hb.hp_cascade_decode(plan, q, host.scale)
    static = hb.CascadePlan.from_workload(dev)
    with pytest.raises(hb.HpError):
        hb.hp_cascade_decode_loop(static, q, host.scale, suffix_len=plan.suffix_len)
    static.suffix_len = plan.suffix_len
    with pytest.raises(hb.HpError):
        hb.hp_cascade_append_kv(static, k, v)
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(plan.ws) == hb.HP_OK


@pytest.mark.parametrize("name,kw,steps", [
    ("llama3_8b", dict(B=8, prefix=512), 24),
    ("tree2", dict(B=16, prefix=128), 12),
    ("tiny", {}, 16),
    ("edges", {}, 34),
])
def test_decode_loop_fused_append_equals_separate_calls(name, kw, steps):
    """hp_cascade_decode_append (the token written by the persistent kernel,
    the length advanced by the merge) against hp_cascade_append_kv +
    hp_cascade_decode_loop on a second copy of the same tree: every step's
    results bit for bit, and the pools and lengths at the end; every eighth
    step also against the oracle."""
    host, cap = _loop_host(name, kw, steps, seed=7)
    da, db = host.to(DEV), host.to(DEV)
    pa = hb.LoopPlan.from_workload(da, cap)
    pb = hb.LoopPlan.from_workload(db, cap)
    for s, (q, k, v) in enumerate(W.decode_tokens(host, steps, seed=7)):
        qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
        pa.append(kd, vd)
        oa, la = pa.decode(qd, host.scale, out_dtype=torch.float32)
        ob, lb = pb.decode_append(qd, kd, vd, host.scale, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob) and torch.equal(la, lb), f"step {s}"
        W.append_token(host, k, v)
        if s % 8 == 7 or s == steps - 1:
            host.q = q
            O, L = oracle.cascade(host)
            _check(ob, lb, O, L, f"fused decode loop {name} step {s}")
    _status_ok(pa.ws)
    _status_ok(pb.ws)
    assert torch.equal(pa.suffix_len, pb.suffix_len)
    assert torch.equal(pb.suffix_len.cpu(), host.levels[-1].nodes[:, 2])
    assert torch.equal(da.k_pool, db.k_pool) and torch.equal(da.v_pool, db.v_pool)


def test_decode_loop_full_size_sampled():
    """The benchmarked shape at full size (B=64, 32/8 heads, d=128, 4K shared
    prefix, suffixes U[1,256]) as a decode loop: 8 fused steps, each checked
    on 64 sampled rows against the oracle over the host-appended tree."""
    steps = 8
    host, cap = _loop_host("llama3_8b", {}, steps, seed=11)
    dev = host.to(DEV)
    plan = hb.LoopPlan.from_workload(dev, cap)
    g = torch.Generator().manual_seed(11)
    for s, (q, k, v) in enumerate(W.decode_tokens(host, steps, seed=11)):
        out, lse = plan.decode_append(q.to(DEV), k.to(DEV), v.to(DEV), host.scale, out_dtype=torch.float32)
        W.append_token(host, k, v)
        host.q = q
        bs = torch.randint(0, host.B, (64,), generator=g).tolist()
        hs = torch.randint(0, host.Hq, (64,), generator=g).tolist()
        rows = list(zip(bs, hs))
        O, L = oracle.cascade(host, rows)
        o = torch.stack([out[b, h] for b, h in rows])
        l = torch.stack([lse[b, h] for b, h in rows])
        _check(o, l, O, L, f"full-size decode loop step {s}")
    _status_ok(plan.ws)
    assert torch.equal(plan.suffix_len.cpu(), host.levels[-1].nodes[:, 2])


# ------------------------------------------------ general forests (deep, many pools, narrow nodes)
def _forest(seed, B=24, ps=16):
    """Two system prompts, nested shared chunks down to pairs and triples of
    sequences, private suffixes (ChunkAttention's realistic trees)."""
    h = B // 2
    lvl0 = [(0, h, 128), (h, B, 96)]
    lvl1 = [(0, 6, 64), (6, 12, 48), (12, 18, 32), (18, 24, 64)]
    lvl2 = [(b, min(b + 3, B), 16 * (1 + (b // 3) % 3)) for b in range(0, B, 3)]
    lvl3 = [(b, b + 2, 32) for b in range(0, B, 4)]
    return W.build_cascade(f"forest{seed}", B=B, Hq=8, Hkv=2, d=64, page_size=ps,
                           shared=[lvl0, lvl1, lvl2, lvl3], suffix_range=(1, 40), seed=seed)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_cascade_forest_with_narrow_nodes(seed):
    """Narrow shared nodes joined into their sequences' nodes (read per
    sequence), wider ones on the tensor cores, every row against the oracle."""
    wl = _forest(seed)
    items = hb.hp_cascade_plan_items(hb._levels_of(wl), wl.B, wl.Hq, wl.Hkv, wl.d)
    assert all(it["n_seq"] == 1 or it["n_seq"] > 3 for it in items)
    O, L = oracle.cascade(wl)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    out, lse = plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
    _status_ok(plan.ws)
    _check(out, lse, O, L, f"forest {seed}")


def test_cascade_deep_chunk_tree_21_levels():
    """A 64-token prompt shared by all sequences, then each sequence's keys
    as a chain of 16-token chunk nodes, one level per chunk (21 levels)."""
    B, ps = 5, 16
    lens = [0, 3, 7, 12, 19]
    levels = [[(0, B, 64)]] + [[(b, b + 1, ps) for b in range(B) if lens[b] > c] for c in range(max(lens))]
    levels = [lv for lv in levels if lv]
    wl = W.build_cascade("chunks", B=B, Hq=8, Hkv=2, d=64, page_size=ps, shared=levels, suffix_lens=[5] * B, seed=3)
    assert len(wl.levels) == 21
    O, L = oracle.cascade(wl)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    out, lse = plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
    _status_ok(plan.ws)
    _check(out, lse, O, L, "21-level chunk tree")


@pytest.mark.parametrize("n_pools", [2, 5, 8])
def test_cascade_levels_over_several_pools(n_pools):
    """A 12-level tree whose levels live in n_pools distinct pool pairs
    (copies of one pool: the values, and so the oracle, are the same); the
    plan keeps one tensor-map slot per pool set."""
    B = 16
    shared = [[(0, B, 64)], [(0, 8, 48), (8, 16, 32)]] + \
             [[(b, b + 4, 16 * (1 + l % 2)) for b in range(0, B, 4)] for l in range(4)] + \
             [[(b, b + 1, 16) for b in range(B)] for _ in range(5)]
    wl = W.build_cascade("pools", B=B, Hq=16, Hkv=4, d=128, page_size=16, shared=shared, suffix_range=(0, 30), seed=4)
    assert len(wl.levels) == 12
    O, L = oracle.cascade(wl)
    wg = wl.to(DEV)
    pools = [(wg.k_pool.clone(), wg.v_pool.clone()) for _ in range(n_pools)]
    levels = []
    for i, lv in enumerate(wg.levels):
        kp, vp = pools[i % n_pools]
        levels.append((kp.data_ptr(), vp.data_ptr(), wg.num_pages, wg.page_size, lv.nodes.tolist(),
                       lv.page_ids.cpu().tolist()))
    plan = hb.CascadePlan(levels, wl.B, wl.Hq, wl.Hkv, wl.d, device=DEV)
    assert plan.info.num_levels == n_pools
    out, lse = plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
    _status_ok(plan.ws)
    _check(out, lse, O, L, f"{n_pools} pools")
