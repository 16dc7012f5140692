"""GPU parity of the reduced-precision KV path: private suffixes (and every
other node of the per-sequence pass) stored as E4M3 codes with one f32 scale
per (page, KV head) for K and for V, against the fp64 oracle that decodes
the same codes by the format's definition.

The quantised values are the inputs: the oracle and the kernels see the same
codes and scales, so the tolerances are the bf16 ones (O max-abs 2e-2,
mean-abs 2e-3, LSE abs 1e-3).
"""
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
    assert np.all(o[~fin] == 0), f"{what}: empty rows must be 0"
    d_o = np.abs(o - O)
    d_l = np.abs(l[fin] - L[fin]) if fin.any() else np.zeros(1)
    assert d_o.max() <= O_MAX, f"{what}: max|dO| {d_o.max():.3g}"
    assert d_o.mean() <= O_MEAN, f"{what}: mean|dO| {d_o.mean():.3g}"
    assert d_l.max() <= LSE_ABS, f"{what}: max|dLSE| {d_l.max():.3g}"


def _status_ok(ws):
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(ws) == hb.HP_OK


CASES = [
    ("llama3_8b", dict(B=8, prefix=512)),
    ("codellama13b", dict(B=32, prefix=384)),
    ("tree2", dict(B=32, prefix=256)),
    ("doc_streams", dict(B=20, prefix=640)),
    ("no_sharing", dict(B=6, prefix=200)),
]


@pytest.mark.parametrize("name,kw", CASES)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_e4m3_suffix_cascade_every_row(name, kw, seed):
    wl = W.with_e4m3_levels(W.make_config(name, seed=seed, **kw))
    O, L = oracle.cascade(wl)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    out, lse = plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
    _status_ok(plan.ws)
    _check(out, lse, O, L, f"e4m3 {name} seed {seed}")


def test_e4m3_suffix_cascade_benchmarked_shape_full_size():
    """B=64, 32/8 heads, 4K bf16 prefix, E4M3 suffixes U[1,256]: every row."""
    wl = W.with_e4m3_levels(W.make_config("llama3_8b", seed=3))
    O, L = oracle.cascade(wl)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    out, lse = plan.decode(wg.q, wl.scale)
    _status_ok(plan.ws)
    _check(out, lse, O, L, "e4m3 llama3 full")


def test_e4m3_scales_per_page_and_head_are_applied():
    """Scales far from 1 that differ per page, per KV head and between K and
    V (codes kept): the output follows the decoded values, not the codes."""
    wl = W.with_e4m3_levels(W.make_config("llama3_8b", seed=4, B=8, prefix=256))
    g = torch.Generator().manual_seed(9)
    P, Hkv = wl.q8.k_scale.shape
    wl.q8.k_scale = wl.q8.k_scale * torch.pow(2.0, torch.randint(-4, 3, (P, Hkv), generator=g).float())
    wl.q8.v_scale = wl.q8.v_scale * torch.pow(2.0, torch.randint(-6, 7, (P, Hkv), generator=g).float())
    O, L = oracle.cascade(wl)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    out, lse = plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
    _status_ok(plan.ws)
    scale_o = max(1.0, float(np.abs(O).max()))
    o = out.double().cpu().numpy().reshape(O.shape)
    assert np.abs(o - O).max() <= O_MAX * scale_o
    assert np.abs(lse.double().cpu().numpy().reshape(L.shape) - L).max() <= LSE_ABS * 4


def _paged_e4m3(wl):
    pt, sl = W.full_page_tables(wl)
    q8 = W.quantize_e4m3(wl.k_pool, wl.v_pool)
    return pt, sl, q8


@pytest.mark.parametrize("name,kw", [("llama3_8b", dict(B=8, prefix=512)), ("no_sharing", dict(B=4, prefix=333)),
                                     ("tree2", dict(B=16, prefix=128))])
def test_e4m3_paged_decode(name, kw):
    wl = W.make_config(name, seed=5, **kw)
    pt, sl, q8 = _paged_e4m3(wl)
    O, L = oracle.paged_decode_e4m3(wl.q, q8.k, q8.v, q8.k_scale, q8.v_scale, pt, sl, wl.scale)
    g8 = q8.to(DEV)
    out, lse = hb.hp_suffix_decode_paged_e4m3(wl.q.to(DEV), g8.k, g8.v, g8.k_scale, g8.v_scale, pt.to(DEV),
                                              sl.to(DEV), wl.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    _check(out, lse, O, L, f"e4m3 paged {name}")


def test_e4m3_paged_decode_edge_lengths():
    """Lengths 0, 1, 15, 16, 17, 31, 33 and 64 in one call (ragged last
    chunks, an empty sequence)."""
    lens = [0, 1, 15, 16, 17, 31, 33, 64]
    wl = W.build_cascade("edge", B=len(lens), Hq=8, Hkv=2, d=128, page_size=16, shared=[], suffix_lens=lens, seed=6)
    pt, sl, q8 = _paged_e4m3(wl)
    O, L = oracle.paged_decode_e4m3(wl.q, q8.k, q8.v, q8.k_scale, q8.v_scale, pt, sl, wl.scale)
    g8 = q8.to(DEV)
    ws = hb.alloc_workspace(hb.suffix_workspace_bytes(wl.B, wl.Hq, wl.d, pt.shape[1], 16), DEV)
    out, lse = hb.hp_suffix_decode_paged_e4m3(wl.q.to(DEV), g8.k, g8.v, g8.k_scale, g8.v_scale, pt.to(DEV),
                                              sl.to(DEV), wl.scale, ws=ws, out_dtype=torch.float32)
    _status_ok(ws)
    _check(out, lse, O, L, "e4m3 edge lengths")
    assert torch.all(out[0] == 0) and torch.all(torch.isinf(lse[0]))


def test_e4m3_paged_decode_bad_page_sets_bounds_status():
    wl = W.make_config("llama3_8b", seed=7, B=4, prefix=64)
    pt, sl, q8 = _paged_e4m3(wl)
    pt[1, 0] = 10 ** 6
    g8 = q8.to(DEV)
    ws = hb.alloc_workspace(hb.suffix_workspace_bytes(wl.B, wl.Hq, wl.d, pt.shape[1], 16), DEV)
    hb.hp_suffix_decode_paged_e4m3(wl.q.to(DEV), g8.k, g8.v, g8.k_scale, g8.v_scale, pt.to(DEV), sl.to(DEV),
                                   wl.scale, ws=ws)
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(ws) == hb.HP_ERR_BOUNDS


def test_e4m3_cascade_equals_e4m3_paged_decode():
    """The cascade over a tree with E4M3 suffixes and a bf16 prefix, against
    the same tree decoded per sequence with every level in E4M3 would differ
    (the prefix is quantised there); instead, with no shared level the two
    entry points read the same codes and must agree to the bar."""
    wl = W.with_e4m3_levels(W.make_config("no_sharing", seed=8, B=8, prefix=300))
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    oc, lc = plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
    pt, sl = W.full_page_tables(wl)
    on, ln = hb.hp_suffix_decode_paged_e4m3(wg.q, wg.q8.k, wg.q8.v, wg.q8.k_scale, wg.q8.v_scale, pt.to(DEV),
                                            sl.to(DEV), wl.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert (oc - on).abs().max().item() <= O_MAX
    assert (lc - ln).abs().max().item() <= LSE_ABS


def test_e4m3_per_sequence_workload_full_size_sampled_rows():
    """The per-sequence-only workload at full size (B=64, 32 heads, 2048
    tokens each) in E4M3, where the planner splits the consumer-bound paged
    work into about four items per CTA: 96 sampled rows against the oracle."""
    wl = W.with_e4m3_levels(W.make_config("no_sharing", seed=2))
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    assert plan.info.n_small_items >= 4 * 152 * 0.9
    out, lse = plan.decode(wg.q, wl.scale, out_dtype=torch.float32)
    _status_ok(plan.ws)
    g = torch.Generator().manual_seed(4)
    flat = torch.randperm(wl.B * wl.Hq, generator=g)[:96].tolist()
    O, L = oracle.cascade(wl, rows=[(f // wl.Hq, f % wl.Hq) for f in flat])
    o = out.double().cpu().numpy().reshape(wl.B * wl.Hq, wl.d)[flat]
    l = lse.double().cpu().numpy().reshape(wl.B * wl.Hq)[flat]
    _check(torch.from_numpy(o), torch.from_numpy(l), O, L, "e4m3 no_sharing full size")
