"""GPU parity of the Parallel Prompting row kernel (hp_stream_decode): each
request's KV row -- document, questions, interleaved answers -- read in place
with the stream mask of Read Once, Answer Many (Section 3, Eq. 2) applied per
key inside the kernel, against the oracle's masked attention
(oracle.stream_masked) on the layouts the page's correctness checks name:
documents of 37, 300 and 1000 tokens with 1 to 64 streams, prefill-like and
decode positions.  Tolerances as everywhere: O max-abs 2e-2, mean-abs 2e-3,
LSE 1e-3; the Figure 2 probe is bit-exact.
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


def _bf16(t):
    return t.float().numpy().astype(np.float64)


def _oracle_rows(req, rows_cpu):
    """Per request and head: the oracle's masked attention of the request's
    P queries over its row (query head h reads KV head h // G)."""
    G = req.Hq // req.Hkv
    O = np.zeros((req.R * req.P, req.Hq, req.d))
    L = np.zeros((req.R * req.P, req.Hq))
    for r, (sid, pos, k, v) in enumerate(req.rows):
        q_sid = rows_cpu.q_sid[r * req.P:(r + 1) * req.P].numpy()
        q_pos = rows_cpu.q_pos[r * req.P:(r + 1) * req.P].numpy()
        for h in range(req.Hq):
            Q = _bf16(req.q[r * req.P:(r + 1) * req.P, h])
            o, l = oracle.stream_masked(Q, _bf16(k[:, h // G]), _bf16(v[:, h // G]), q_sid, q_pos, sid.numpy(),
                                        pos.numpy(), req.scale)
            O[r * req.P:(r + 1) * req.P, h] = o
            L[r * req.P:(r + 1) * req.P, h] = l
    return O, L


def _check(out, lse, O, L, what):
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    d = np.abs(o - O)
    assert d.max() <= O_MAX, f"{what}: max|dO| {d.max():.3g}"
    assert d.mean() <= O_MEAN, f"{what}: mean|dO| {d.mean():.3g}"
    fin = np.isfinite(L)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.abs(l[fin] - L[fin]).max() <= LSE_ABS, f"{what}: max|dLSE| {np.abs(l[fin] - L[fin]).max():.3g}"


def _run(req, page_size=16, seed=0, out_dtype=torch.float32):
    rows = W.stream_rows_paged(req, page_size=page_size, seed=seed)
    g = rows.to(DEV)
    ws = hb.alloc_workspace(hb.stream_workspace_bytes(req.R, req.P, req.Hq, req.Hkv, req.d, g.row_pages.shape[1],
                                                      page_size), DEV)
    out, lse = hb.hp_stream_decode(req.q.to(DEV), g, req.P, req.scale, ws=ws, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(ws) == hb.HP_OK
    return rows, out, lse


@pytest.mark.parametrize("doc_len", [37, 300, 1000])
@pytest.mark.parametrize("P", [1, 3, 16, 64])
@pytest.mark.parametrize("heads", [(4, 4), (8, 2)])
def test_stream_decode_matches_masked_oracle(doc_len, P, heads):
    """Two requests, decode step 4 (each stream's newest answer token),
    questions of 3..12 tokens, d = 128; MHA and GQA (4 query heads per KV
    head)."""
    Hq, Hkv = heads
    req = W.stream_requests(R=2, P=P, Hq=Hq, Hkv=Hkv, d=128, doc_len=doc_len, q_len_range=(3, 12), T=4,
                            seed=doc_len + P + Hq)
    rows, out, lse = _run(req, seed=P)
    O, L = _oracle_rows(req, rows)
    _check(out, lse, O, L, f"doc {doc_len} P {P} heads {heads}")


@pytest.mark.parametrize("T", [1, 2])
@pytest.mark.parametrize("page_size", [16, 64])
def test_stream_decode_d64_pages_and_early_steps(T, page_size):
    req = W.stream_requests(R=3, P=5, Hq=4, Hkv=1, d=64, doc_len=300, q_len_range=(1, 20), T=T, seed=7 + T)
    rows, out, lse = _run(req, page_size=page_size, seed=T, out_dtype=torch.bfloat16)
    O, L = _oracle_rows(req, rows)
    _check(out, lse, O, L, f"d64 T {T} page {page_size}")


@pytest.mark.parametrize("P,Hkv", [(64, 1), (64, 2), (32, 4), (16, 8)])
@pytest.mark.parametrize("d", [64, 128])
def test_stream_decode_every_stage_shape(P, Hkv, d):
    """Every (chunks per stage, heads per item) form the planner picks (MHA,
    16 streams per consumer warp): 64 streams over 1 or 2 KV heads give
    items of 1 or 2 heads and four chunks per stage, 32 streams over 4 heads
    items of 4 heads and two chunks, 16 streams over 8 heads items of 8
    heads and one chunk; at d = 64 and d = 128."""
    req = W.stream_requests(R=2, P=P, Hq=Hkv, Hkv=Hkv, d=d, doc_len=300, q_len_range=(5, 40), T=3,
                            seed=20 + Hkv + d)
    rows, out, lse = _run(req, seed=Hkv)
    O, L = _oracle_rows(req, rows)
    _check(out, lse, O, L, f"Hkv {Hkv} d {d}")


def test_stream_decode_prefill_positions():
    """Queries that are not the newest token of their stream (earlier
    positions): the causal half of the mask hides the stream's later tokens."""
    req = W.stream_requests(R=2, P=4, Hq=4, Hkv=4, d=128, doc_len=37, q_len_range=(2, 6), T=6, seed=11)
    g = torch.Generator().manual_seed(3)
    # pull each query back by 0..5 positions (still at or after its question)
    req.q_pos = [p - int(torch.randint(0, 6, (1,), generator=g)) for p in req.q_pos]
    rows, out, lse = _run(req, seed=2)
    O, L = _oracle_rows(req, rows)
    _check(out, lse, O, L, "prefill positions")


def test_stream_decode_figure2_probe_bit_exact():
    """Figure 2 of Read Once, Answer Many: a 3-token document, 3 streams with
    1-token questions, decode step 2 (12 slots).  Stream 1's query points at
    e_0; slot a1^1 (stream 1, position 4) scores high, a2^0 (stream 0) higher
    and a2^1 (stream 1, position 5) highest.  At position 5 the output of
    stream 1 is a2^1's value row bit for bit (a2^0 is another stream's); at
    position 4 it is a1^1's (a2^1 lies in its future).  Every other weight
    underflows to 0."""
    for q_pos1, want_slot in ((5, 10), (4, 7)):
        req = W.stream_requests(R=1, P=3, Hq=1, Hkv=1, d=128, doc_len=3, q_len_range=(1, 1), T=2, seed=0)
        sid, pos, k, v = req.rows[0]
        assert sid.tolist() == [-1, -1, -1, 0, 1, 2, 0, 1, 2, 0, 1, 2]
        assert pos.tolist() == [0, 1, 2, 3, 3, 3, 4, 4, 4, 5, 5, 5]
        k.zero_()
        e0 = torch.zeros(128)
        e0[0] = 1.0
        k[7, 0] = (64.0 * e0).to(torch.bfloat16)   # a1^1
        k[9, 0] = (128.0 * e0).to(torch.bfloat16)  # a2^0: another stream
        k[10, 0] = (96.0 * e0).to(torch.bfloat16)  # a2^1: stream 1, position 5
        for t in range(12):
            v[t, 0] = W.probe_expected(t, 128)
        req.q = torch.zeros(3, 1, 128, dtype=torch.bfloat16)
        req.q[1, 0] = (64.0 * e0).to(torch.bfloat16)
        req.q_pos = [5, q_pos1, 5]
        rows, out, lse = _run(req, seed=1, out_dtype=torch.bfloat16)
        assert torch.equal(out[1, 0].cpu(), W.probe_expected(want_slot, 128)), f"query at position {q_pos1}"
        O, L = _oracle_rows(req, rows)
        _check(out, lse, O, L, "figure 2")


def test_stream_decode_equals_cascade_form():
    """The same requests through the cascade path (document as a node shared
    by the request's streams, each stream's own slots as a private node)
    give the same attention."""
    req = W.stream_requests(R=3, P=8, Hq=8, Hkv=2, d=128, doc_len=300, q_len_range=(4, 16), T=3, seed=5)
    rows, out, lse = _run(req, seed=4)
    tree = W.streams_as_tree(req)
    tg = tree.to(DEV)
    plan = hb.CascadePlan.from_workload(tg)
    oc, lc = plan.decode(tg.q, tree.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert (out - oc).abs().max().item() <= O_MAX
    assert (lse - lc).abs().max().item() <= LSE_ABS


def test_stream_decode_bad_page_sets_bounds_status():
    req = W.stream_requests(R=2, P=3, Hq=4, Hkv=4, d=128, doc_len=37, q_len_range=(2, 4), T=2, seed=9)
    rows = W.stream_rows_paged(req)
    rows.row_pages[1, 0] = 10 ** 6
    g = rows.to(DEV)
    ws = hb.alloc_workspace(hb.stream_workspace_bytes(req.R, req.P, req.Hq, req.Hkv, req.d, g.row_pages.shape[1], 16),
                            DEV)
    hb.hp_stream_decode(req.q.to(DEV), g, req.P, req.scale, ws=ws)
    torch.cuda.synchronize()
    assert hb.hp_read_device_status(ws) == hb.HP_ERR_BOUNDS
