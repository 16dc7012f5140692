"""GPU tests of hp_cascade_decode_host: the cascade step with q read from,
and O / LSE written to, page-locked host memory.  The step computes on an
exact copy of q, so its result must equal hp_cascade_decode's bit for bit;
it is also held to the oracle at the usual bar (O max-abs 2e-2, mean-abs
2e-3, LSE abs 1e-3).
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
DEV = "cuda"


def _host_bufs(wl, out_dtype=torch.bfloat16):
    q_host = wl.q.pin_memory()
    out_host = torch.full((wl.B, wl.Hq, wl.d), float("nan"), dtype=out_dtype).pin_memory()
    lse_host = torch.full((wl.B, wl.Hq), float("nan"), dtype=torch.float32).pin_memory()
    return q_host, out_host, lse_host


@pytest.mark.parametrize("name,kw", [("llama3_8b", dict(B=16, prefix=512)), ("tree2", dict(B=32, prefix=256)),
                                     ("codellama13b", dict(B=32, prefix=384)), ("no_sharing", dict(B=4, prefix=100)),
                                     ("tiny", {}), ("doc_streams", dict(B=24, prefix=640))])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_host_step_equals_device_step_and_oracle(name, kw, out_dtype):
    wl = W.make_config(name, seed=2, **kw)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    ref_o, ref_l = plan.decode(wg.q, wl.scale, out_dtype=out_dtype)
    ws = hb.alloc_workspace(hb.host_workspace_bytes(plan), DEV)
    q_host, out_host, lse_host = _host_bufs(wl, out_dtype)
    hb.hp_cascade_decode_host(plan, q_host, wl.scale, out_host, lse_host, ws)
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(ws) == hb.HP_OK
    assert torch.equal(out_host, ref_o.cpu()) and torch.equal(lse_host, ref_l.cpu())
    O, L = oracle.cascade(wl)
    d = np.abs(out_host.double().numpy().reshape(O.shape) - O)
    assert d.max() <= O_MAX and d.mean() <= O_MEAN
    fin = np.isfinite(L)
    assert np.abs(lse_host.double().numpy().reshape(L.shape)[fin] - L[fin]).max() <= LSE_ABS


def test_host_step_strided_q_and_no_lse():
    """q_host as a view with padded rows; no LSE buffer."""
    wl = W.make_config("llama3_8b", seed=5, B=8, prefix=256)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    ref_o, _ = plan.decode(wg.q, wl.scale)
    wide = torch.zeros(wl.B, wl.Hq + 3, wl.d + 64, dtype=torch.bfloat16).pin_memory()
    wide[:, :wl.Hq, :wl.d] = wl.q
    q_view = wide[:, :wl.Hq, :wl.d]
    out_host = torch.zeros(wl.B, wl.Hq, wl.d, dtype=torch.bfloat16).pin_memory()
    ws = hb.alloc_workspace(hb.host_workspace_bytes(plan), DEV)
    hb.hp_cascade_decode_host(plan, q_view, wl.scale, out_host, None, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_host, ref_o.cpu())


def test_host_steps_in_one_graph():
    """Three steps over three pinned query sets, captured in one CUDA graph
    and replayed twice: each output equals its device-resident step."""
    wl = W.make_config("llama3_8b", seed=7, B=16, prefix=512)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    ws = hb.alloc_workspace(hb.host_workspace_bytes(plan), DEV)
    g = torch.Generator().manual_seed(11)
    qs = [torch.randn(wl.B, wl.Hq, wl.d, generator=g).to(torch.bfloat16) for _ in range(3)]
    bufs = [(q.pin_memory(),) + _host_bufs(wl)[1:] for q in qs]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for qh, oh, lh in bufs:  # warm-up outside the capture
            hb.hp_cascade_decode_host(plan, qh, wl.scale, oh, lh, ws, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for qh, oh, lh in bufs:
            hb.hp_cascade_decode_host(plan, qh, wl.scale, oh, lh, ws, stream=stream)
    for _ in range(2):
        for _, oh, lh in bufs:
            oh.fill_(float("nan"))
            lh.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for q, (_, oh, lh) in zip(qs, bufs):
            ro, rl = plan.decode(q.to(DEV), wl.scale)
            torch.cuda.synchronize()
            assert torch.equal(oh, ro.cpu()) and torch.equal(lh, rl.cpu())
    assert hb.hp_read_device_status(ws) == hb.HP_OK


def _raw_call(plan, q_ptr, out_ptr, lse_ptr, ws, ws_bytes=None, q_sb=None):
    hq, d = plan.Hq, plan.d
    return hb.library().hp_cascade_decode_host(
        plan.plan.data_ptr(), ctypes.byref(plan.info), q_ptr, hq * d if q_sb is None else q_sb, d,
        ctypes.c_float(0.088), out_ptr, hb.HP_BF16, hq * d, d, lse_ptr, hq, ws.data_ptr(),
        ws.numel() if ws_bytes is None else ws_bytes, None)


def test_host_step_rejects_memory_that_is_not_page_locked():
    """Pageable host memory and device memory are argument errors, found
    before any launch."""
    wl = W.make_config("llama3_8b", seed=1, B=4, prefix=64)
    wg = wl.to(DEV)
    plan = hb.CascadePlan.from_workload(wg)
    ws = hb.alloc_workspace(hb.host_workspace_bytes(plan), DEV)
    q_pin, o_pin, l_pin = _host_bufs(wl)
    q_pageable = wl.q.clone()
    o_pageable = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.bfloat16)
    o_dev = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.bfloat16, device=DEV)
    assert _raw_call(plan, q_pageable.data_ptr(), o_pin.data_ptr(), l_pin.data_ptr(), ws) == hb.HP_ERR_ARG
    assert _raw_call(plan, q_pin.data_ptr(), o_pageable.data_ptr(), l_pin.data_ptr(), ws) == hb.HP_ERR_ARG
    assert _raw_call(plan, wg.q.data_ptr(), o_pin.data_ptr(), l_pin.data_ptr(), ws) == hb.HP_ERR_ARG
    assert _raw_call(plan, q_pin.data_ptr(), o_dev.data_ptr(), l_pin.data_ptr(), ws) == hb.HP_ERR_ARG
    # a workspace without room for the q copy
    assert (_raw_call(plan, q_pin.data_ptr(), o_pin.data_ptr(), l_pin.data_ptr(), ws,
                      ws_bytes=plan.info.ws_bytes) == hb.HP_ERR_WORKSPACE)
    # a q stride that is not a multiple of 8 elements
    assert (_raw_call(plan, q_pin.data_ptr(), o_pin.data_ptr(), l_pin.data_ptr(), ws,
                      q_sb=wl.Hq * wl.d + 4) == hb.HP_ERR_UNSUPPORTED)
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(ws) == hb.HP_OK
