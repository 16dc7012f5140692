"""The allocation-free paged decode entry point.

hp_suffix_decode_paged_noalloc serves callers that cannot give the library
device memory: a program that reaches it only through the C ABI and has no
device allocator of its own, a process whose caching allocator already holds
all device memory, or a path that cannot pay for cudaMalloc's implicit
synchronisation.  Its scratch is a fixed 16 MiB array inside the library;
each key split of a call needs B*Hq partial rows of 2d + 4 bytes (bf16 O row
plus f32 LSE), so one split fits up to 64,525 rows at d = 128.  These tests
call it through the C ABI and compare it with the fp64 oracle and with
hp_suffix_decode_paged (which takes a caller-provided workspace), on two
calls in a row.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
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
    return wl, wg, pt, sl


def _against_oracle(out, lse, q_cpu, wl, pt, sl):
    O, L = oracle.paged_decode(q_cpu, wl.k_pool, wl.v_pool, pt, sl, wl.scale)
    o = out.double().cpu().numpy()
    d = np.abs(o - O)
    assert d.max() <= O_MAX and d.mean() <= O_MEAN, (d.max(), d.mean())
    assert np.abs(lse.double().cpu().numpy() - L).max() <= LSE_ABS


def test_noalloc_matches_oracle_and_workspace_entry_on_two_calls_in_a_row():
    cases = [_case("llama3_8b", 5, B=8, prefix=512), _case("tree2", 6, B=16, prefix=256)]
    results = []
    for wl, wg, pt, sl in cases:
        out = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.float32, device="cuda")
        lse = torch.empty(wl.B, wl.Hq, dtype=torch.float32, device="cuda")
        assert _noalloc(wg.q, wg.k_pool, wg.v_pool, pt.cuda(), sl.cuda(), wl.scale, out, lse) == hb.HP_OK
        results.append((out, lse))
    torch.cuda.synchronize()
    for (wl, wg, pt, sl), (out, lse) in zip(cases, results):
        _against_oracle(out, lse, wl.q, wl, pt, sl)
        ref_o, ref_l = hb.hp_suffix_decode_paged(wg.q, wg.k_pool, wg.v_pool, pt.cuda(), sl.cuda(), wl.scale,
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
        assert _noalloc(wg.q, wg.k_pool, wg.v_pool, pt.cuda(), sl.cuda(), wl.scale, out, lse) == hb.HP_OK
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    _against_oracle(outs[0][0], outs[0][1], wl.q, wl, pt, sl)


def test_noalloc_benchmarked_shape_uses_wider_splits():
    """B=64, 32/8 heads, a 4096-token prefix plus suffixes: 2048 rows per
    split, so the scratch holds 31 splits and the call widens them to 256
    keys (17 splits); every row against the oracle."""
    wl, wg, pt, sl = _case("llama3_8b", 7)
    out = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.float32, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, dtype=torch.float32, device="cuda")
    for _ in range(2):
        assert _noalloc(wg.q, wg.k_pool, wg.v_pool, pt.cuda(), sl.cuda(), wl.scale, out, lse) == hb.HP_OK
    torch.cuda.synchronize()
    _against_oracle(out, lse, wl.q, wl, pt, sl)


def test_noalloc_broadcast_query_reads_q_without_a_tensor_map():
    """q with a zero batch stride (one query row set shared by every
    sequence): the queries are read by the consumer warps, not by TMA."""
    wl, wg, pt, sl = _case("llama3_8b", 8, B=6, prefix=304)
    q1 = wg.q[:1].expand(wl.B, wl.Hq, wl.d)
    assert q1.stride(0) == 0
    out = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.float32, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, dtype=torch.float32, device="cuda")
    assert _noalloc(q1, wg.k_pool, wg.v_pool, pt.cuda(), sl.cuda(), wl.scale, out, lse) == hb.HP_OK
    torch.cuda.synchronize()
    _against_oracle(out, lse, wl.q[:1].expand(wl.B, wl.Hq, wl.d).contiguous(), wl, pt, sl)


@pytest.mark.parametrize("rows,ok", [(64525, True), (64526, False)])
def test_noalloc_scratch_limit(rows, ok):
    """One split of B*Hq rows of 2*128 + 4 bytes must fit the 16 MiB array
    (less its header): 64,525 rows fit, one more is rejected."""
    B, Hq, Hkv, d = rows, 1, 1, 128
    g = torch.Generator(device="cuda").manual_seed(3)
    q = torch.randn(B, Hq, d, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(1, Hkv, 16, d, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(1, Hkv, 16, d, generator=g, device="cuda").to(torch.bfloat16)
    pt = torch.zeros(B, 1, dtype=torch.int32, device="cuda")
    sl = torch.ones(B, dtype=torch.int32, device="cuda")  # each sequence sees key 0 of page 0
    out = torch.empty(B, Hq, d, dtype=torch.float32, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    st = _noalloc(q, k, v, pt, sl, 0.1, out, lse)
    if not ok:
        assert st == hb.HP_ERR_WORKSPACE
        return
    assert st == hb.HP_OK
    torch.cuda.synchronize()
    # one visible key: O is its value row exactly, LSE its scaled score
    assert torch.equal(out[:, 0], v[0, 0, 0].float().expand(B, d))
    s = (q[:, 0].double() * k[0, 0, 0].double()).sum(-1) * 0.1
    assert (lse[:, 0].double() - s).abs().max().item() <= LSE_ABS
