"""The allocation-free paged decode entry point.

hp_suffix_decode_paged_noalloc serves callers that cannot give the library
device memory (no allocator of their own at the C ABI, all device memory held
by a caching allocator, or no tolerance for cudaMalloc's implicit
synchronisation); its scratch is a fixed array inside the library.  These
tests call it through the C ABI and compare it with hp_suffix_decode_paged,
which takes a caller-provided workspace, on two calls in a row.  The file is
named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from shared_prefix_decode_gb300 import binding as hb
from shared_prefix_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_ABS = 2e-2, 2e-3, 1e-3


def _noalloc(q, k_pool, v_pool, page_table, seq_lens, scale, out, lse):
    B, Hq, d = q.shape
    P, Hkv, ps, _ = k_pool.shape
    return hb.library().hp_suffix_decode_paged_noalloc(
        q.data_ptr(), q.stride(0), q.stride(1), B, k_pool.data_ptr(), v_pool.data_ptr(), P, ps,
        page_table.data_ptr(), page_table.stride(0), seq_lens.data_ptr(), Hq, Hkv, d, ctypes.c_float(scale),
        out.data_ptr(), hb.HP_F32 if out.dtype == torch.float32 else hb.HP_BF16, out.stride(0), out.stride(1),
        lse.data_ptr(), lse.stride(0), torch.cuda.current_stream().cuda_stream)


def _case(name, seed, **kw):
    wl = W.make_config(name, seed=seed, **kw)
    pt, sl = W.full_page_tables(wl)
    wg = wl.to("cuda")
    return wl, wg, pt.to("cuda"), sl.to("cuda")


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    cases = [_case("llama3_8b", 5, B=8, prefix=512), _case("tree2", 6, B=16, prefix=256)]
    results = []
    for wl, wg, pt, sl in cases:
        out = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.float32, device="cuda")
        lse = torch.empty(wl.B, wl.Hq, dtype=torch.float32, device="cuda")
        assert _noalloc(wg.q, wg.k_pool, wg.v_pool, pt, sl, wl.scale, out, lse) == hb.HP_OK
        results.append((out, lse))
    torch.cuda.synchronize()
    for (wl, wg, pt, sl), (out, lse) in zip(cases, results):
        ref_o, ref_l = hb.hp_suffix_decode_paged(wg.q, wg.k_pool, wg.v_pool, pt, sl, wl.scale,
                                                 out_dtype=torch.float32)
        torch.cuda.synchronize()
        d = (out - ref_o).abs()
        assert d.max().item() <= O_MAX and d.mean().item() <= O_MEAN
        assert (lse - ref_l).abs().max().item() <= LSE_ABS


def test_noalloc_repeated_call_is_stable_and_bf16_output():
    wl, wg, pt, sl = _case("tiny", 2)
    outs = []
    for _ in range(2):
        out = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(wl.B, wl.Hq, dtype=torch.float32, device="cuda")
        assert _noalloc(wg.q, wg.k_pool, wg.v_pool, pt, sl, wl.scale, out, lse) == hb.HP_OK
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    ref_o, ref_l = hb.hp_suffix_decode_paged(wg.q, wg.k_pool, wg.v_pool, pt, sl, wl.scale)
    torch.cuda.synchronize()
    assert (outs[0][0].float() - ref_o.float()).abs().max().item() <= O_MAX
    assert (outs[0][1] - ref_l).abs().max().item() <= LSE_ABS


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """B * Hq partial rows of (d + 1) floats must fit the fixed 16 MiB array."""
    B, Hq, Hkv, d = 4096, 16, 16, 128  # 65,536 rows x 516 B > 16 MiB
    q = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(1, Hkv, 16, d, dtype=torch.bfloat16, device="cuda")
    pt = torch.zeros(B, 1, dtype=torch.int32, device="cuda")
    sl = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, Hq, d, dtype=torch.float32, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    assert _noalloc(q, pool, pool, pt, sl, 0.1, out, lse) == hb.HP_ERR_WORKSPACE
