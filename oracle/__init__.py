"""fp64 CPU oracle for shared-prefix (cascade) decode attention.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
CUDA library never imports, links or calls it, and it never imports the CUDA
library: the two share only the seeded input generator.

The arithmetic lives in ``hp_oracle.c`` (plain loops, double precision,
OpenMP over output rows); this module marshals numpy / torch CPU arrays into
it.  Each wrapper names the passage it follows:

* ``sdp``            - SDP(Q,K,V) and LSE(Q,K), Hydragen "Attention
                       Decomposition Across Subsequences" (the LSE definition).
* ``merge``          - two-part exact merge, Hydragen Eq. 5 with the
                       max-subtracted combine_lse step.
* ``partial_attn`` / ``attn_reduce`` - ChunkAttention Eq. 1 and Eq. 2.
* ``cascade``        - attention of each sequence over the concatenation of
                       its tree nodes' keys (Hydragen "Hierarchical Sharing";
                       ChunkAttention prefix tree), i.e. the unsplit definition.
* ``paged_decode``   - per-sequence attention through a page table.
* ``prefix``         - attention of a batch of queries against one contiguous
                       prefix laid out [len][Hkv][d].
* ``e4m3_decode``    - the value of an 8-bit E4M3 code, by the format's
                       definition (sign, 4 exponent bits with bias 7, 3
                       mantissa bits, subnormals, no infinities); levels of a
                       workload stored as E4M3 codes times an f32 scale per
                       (page, KV head) are decoded element by element before
                       the same definition runs (Hydragen, "Implications and
                       Future Directions": KV quantisation for the
                       memory-bound suffix pass).
* ``paged_decode_e4m3`` - ``paged_decode`` over E4M3 pools.
* ``stream_visible`` / ``stream_masked`` - the Parallel Prompting stream mask
                       (Read Once, Answer Many, Section 3, Eq. 2): one KV row
                       per request holding the document and every stream's
                       interleaved tokens; a query of stream s sees the
                       document and stream s's own earlier slots.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hp_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libhp_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_fp = ctypes.POINTER(ctypes.c_float)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, -O2, OpenMP)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.hpo_sdp_f64.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp, _dp, _dp,
                                        ctypes.c_double, _dp, _dp]
            lib.hpo_merge.argtypes = [ctypes.c_long, ctypes.c_int, _dp, _dp, _dp, _dp, _dp, _dp]
            lib.hpo_partial_attn.argtypes = [ctypes.c_int, ctypes.c_int, _dp, _dp, _dp,
                                             ctypes.c_double, _dp, _dp, _dp]
            lib.hpo_attn_reduce.argtypes = [ctypes.c_int, _dp, ctypes.c_double, ctypes.c_double,
                                            _dp, _dp, _dp]
            lib.hpo_cascade.argtypes = [ctypes.c_int] * 4 + [ctypes.c_double, _u16p, ctypes.c_int,
                                        ctypes.POINTER(_u16p), ctypes.POINTER(_u16p), _i32p, _i32p,
                                        ctypes.POINTER(_i32p), ctypes.POINTER(_i32p),
                                        ctypes.c_long, _i32p, _dp, _dp]
            lib.hpo_cascade.restype = ctypes.c_int
            lib.hpo_paged_decode.argtypes = [ctypes.c_int] * 4 + [
                ctypes.c_double, _u16p, ctypes.c_long, ctypes.c_long, _u16p, _u16p, ctypes.c_int,
                _i32p, ctypes.c_int, _i32p, _dp, _dp]
            lib.hpo_paged_decode.restype = ctypes.c_int
            lib.hpo_prefix.argtypes = [ctypes.c_int] * 4 + [
                ctypes.c_double, _u16p, ctypes.c_long, ctypes.c_long, _u16p, _u16p, ctypes.c_long,
                ctypes.c_long, ctypes.c_int, _dp, _dp]
            lib.hpo_prefix.restype = ctypes.c_int
            lib.hpo_e4m3_decode.argtypes = [ctypes.c_long, _u8p, _dp]
            lib.hpo_cascade_q.argtypes = [ctypes.c_int] * 4 + [
                ctypes.c_double, _u16p, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p),
                ctypes.POINTER(ctypes.c_void_p), _i32p, ctypes.POINTER(_fp), ctypes.POINTER(_fp), _i32p, _i32p,
                ctypes.POINTER(_i32p), ctypes.POINTER(_i32p), ctypes.c_long, _i32p, _dp, _dp]
            lib.hpo_cascade_q.restype = ctypes.c_int
            lib.hpo_paged_decode_e4m3.argtypes = [ctypes.c_int] * 4 + [
                ctypes.c_double, _u16p, ctypes.c_long, ctypes.c_long, _u8p, _u8p, _fp, _fp, ctypes.c_int,
                _i32p, ctypes.c_int, _i32p, _dp, _dp]
            lib.hpo_paged_decode_e4m3.restype = ctypes.c_int
            lib.hpo_num_threads.restype = ctypes.c_int
            lib.hpo_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().hpo_num_threads())


def set_num_threads(n: int) -> None:
    _load().hpo_set_num_threads(int(n))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray, typ):
    return a.ctypes.data_as(typ)


def _bf16_bits(t) -> np.ndarray:
    """Raw bf16 bits of a CPU torch bf16 tensor as a contiguous uint16 array."""
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16:
        raise TypeError("expected a torch.bfloat16 tensor")
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def sdp(Q, K, V, scale: float):
    """Q [nq,d], K/V [nk,d] (fp64) -> (O [nq,d], lse [nq])."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    nq, d = Q.shape
    nk = K.shape[0]
    O = np.zeros((nq, d))
    L = np.zeros(nq)
    _load().hpo_sdp_f64(nq, nk, d, _ptr(Q, _dp), _ptr(K, _dp), _ptr(V, _dp), float(scale),
                        _ptr(O, _dp), _ptr(L, _dp))
    return O, L


def merge(O1, L1, O2, L2):
    """Exact two-part merge of (O, LSE) states; rows x d."""
    O1, L1, O2, L2 = _f64(O1), _f64(L1), _f64(O2), _f64(L2)
    n, d = O1.shape
    O = np.zeros((n, d))
    L = np.zeros(n)
    _load().hpo_merge(n, d, _ptr(O1, _dp), _ptr(L1, _dp), _ptr(O2, _dp), _ptr(L2, _dp),
                      _ptr(O, _dp), _ptr(L, _dp))
    return O, L


def partial_attn(q, Kc, Vc, scale: float):
    """ChunkAttention Eq. 1 for one query row: returns (o, m, n)."""
    q, Kc, Vc = _f64(q), _f64(Kc), _f64(Vc)
    d = q.shape[0]
    c = Kc.shape[0]
    o = np.zeros(d)
    m = ctypes.c_double()
    n = ctypes.c_double()
    _load().hpo_partial_attn(d, c, _ptr(q, _dp), _ptr(Kc, _dp), _ptr(Vc, _dp), float(scale),
                             _ptr(o, _dp), ctypes.byref(m), ctypes.byref(n))
    return o, m.value, n.value


def attn_reduce(o_c, m_c: float, n_c: float, state):
    """ChunkAttention Eq. 2: fold chunk state into ``state = [O, m, n]`` (in place)."""
    O, m, n = state
    O = _f64(O).copy()
    o_c = _f64(o_c)
    mm = ctypes.c_double(m)
    nn = ctypes.c_double(n)
    _load().hpo_attn_reduce(O.shape[0], _ptr(o_c, _dp), float(m_c), float(n_c), _ptr(O, _dp),
                            ctypes.byref(mm), ctypes.byref(nn))
    state[0], state[1], state[2] = O, mm.value, nn.value
    return state


def _u8_bytes(t) -> np.ndarray:
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8:
        raise TypeError("expected a torch.uint8 tensor of E4M3 codes")
    return t.detach().cpu().contiguous().numpy()


def _f32(t) -> np.ndarray:
    return np.ascontiguousarray(t.detach().cpu().numpy().astype(np.float32))


def e4m3_decode(codes) -> np.ndarray:
    """Values of 8-bit E4M3 codes (any shape of uint8) as float64."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.zeros(c.shape, dtype=np.float64)
    _load().hpo_e4m3_decode(c.size, _ptr(c, _u8p), _ptr(out, _dp))
    return out


def _cascade_e4m3(wl, rows_np):
    """``cascade`` for a workload with levels marked e4m3 (their keys and
    values decoded from wl.q8's codes and scales)."""
    lib = _load()
    n = rows_np.shape[0]
    q = _bf16_bits(wl.q)
    kp, vp = _bf16_bits(wl.k_pool), _bf16_bits(wl.v_pool)
    k8 = v8 = ks = vs = None
    if wl.q8 is not None:
        k8, v8 = _u8_bytes(wl.q8.k), _u8_bytes(wl.q8.v)
        ks, vs = _f32(wl.q8.k_scale), _f32(wl.q8.v_scale)
    nl = len(wl.levels)
    keep = []
    k_arr = (ctypes.c_void_p * max(nl, 1))()
    v_arr = (ctypes.c_void_p * max(nl, 1))()
    ks_arr = (_fp * max(nl, 1))()
    vs_arr = (_fp * max(nl, 1))()
    dt = np.zeros(max(nl, 1), dtype=np.int32)
    nodes_arr = (_i32p * max(nl, 1))()
    ids_arr = (_i32p * max(nl, 1))()
    ps_arr = np.full(max(nl, 1), wl.page_size, dtype=np.int32)
    nn_arr = np.zeros(max(nl, 1), dtype=np.int32)
    for i, lv in enumerate(wl.levels):
        nodes = np.ascontiguousarray(lv.nodes.cpu().numpy().astype(np.int32))
        ids = np.ascontiguousarray(lv.page_ids.cpu().numpy().astype(np.int32))
        if ids.size == 0:
            ids = np.zeros(1, dtype=np.int32)
        keep += [nodes, ids]
        if lv.e4m3:
            if k8 is None:
                raise ValueError("a level is marked e4m3 but the workload has no E4M3 pools")
            dt[i] = 1
            k_arr[i] = k8.ctypes.data
            v_arr[i] = v8.ctypes.data
            ks_arr[i] = _ptr(ks, _fp)
            vs_arr[i] = _ptr(vs, _fp)
        else:
            k_arr[i] = kp.ctypes.data
            v_arr[i] = vp.ctypes.data
        nodes_arr[i] = _ptr(nodes, _i32p)
        ids_arr[i] = _ptr(ids, _i32p)
        nn_arr[i] = nodes.shape[0]
    O = np.zeros((n, wl.d))
    L = np.zeros(n)
    rc = lib.hpo_cascade_q(wl.B, wl.Hq, wl.Hkv, wl.d, float(wl.scale), _ptr(q, _u16p), nl, k_arr, v_arr,
                           _ptr(dt, _i32p), ks_arr, vs_arr, _ptr(ps_arr, _i32p), _ptr(nn_arr, _i32p), nodes_arr,
                           ids_arr, n, _ptr(rows_np, _i32p), _ptr(O, _dp), _ptr(L, _dp))
    if rc != 0:
        raise ValueError(f"hpo_cascade_q rejected its arguments ({rc})")
    return O, L


def cascade(wl, rows: Optional[Sequence[Sequence[int]]] = None):
    """Attention of rows (b, h) of a ``CascadeWorkload`` over each sequence's
    concatenated tree keys.  Default: every row.  Returns (O [n,d], lse [n])."""
    lib = _load()
    if any(getattr(lv, "e4m3", False) for lv in wl.levels):
        if rows is None:
            rows = [(b, h) for b in range(wl.B) for h in range(wl.Hq)]
        return _cascade_e4m3(wl, np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2)))
    if rows is None:
        rows = [(b, h) for b in range(wl.B) for h in range(wl.Hq)]
    rows_np = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    n = rows_np.shape[0]
    q = _bf16_bits(wl.q)
    kp = _bf16_bits(wl.k_pool)
    vp = _bf16_bits(wl.v_pool)
    nl = len(wl.levels)
    keep = []
    k_arr = (_u16p * max(nl, 1))()
    v_arr = (_u16p * max(nl, 1))()
    nodes_arr = (_i32p * max(nl, 1))()
    ids_arr = (_i32p * max(nl, 1))()
    ps_arr = np.full(max(nl, 1), wl.page_size, dtype=np.int32)
    nn_arr = np.zeros(max(nl, 1), dtype=np.int32)
    for i, lv in enumerate(wl.levels):
        nodes = np.ascontiguousarray(lv.nodes.cpu().numpy().astype(np.int32))
        ids = np.ascontiguousarray(lv.page_ids.cpu().numpy().astype(np.int32))
        if ids.size == 0:
            ids = np.zeros(1, dtype=np.int32)
        keep += [nodes, ids]
        k_arr[i] = _ptr(kp, _u16p)
        v_arr[i] = _ptr(vp, _u16p)
        nodes_arr[i] = _ptr(nodes, _i32p)
        ids_arr[i] = _ptr(ids, _i32p)
        nn_arr[i] = nodes.shape[0]
    O = np.zeros((n, wl.d))
    L = np.zeros(n)
    rc = lib.hpo_cascade(wl.B, wl.Hq, wl.Hkv, wl.d, float(wl.scale), _ptr(q, _u16p), nl, k_arr,
                         v_arr, _ptr(ps_arr, _i32p), _ptr(nn_arr, _i32p), nodes_arr, ids_arr, n,
                         _ptr(rows_np, _i32p), _ptr(O, _dp), _ptr(L, _dp))
    if rc != 0:
        raise ValueError(f"hpo_cascade rejected its arguments ({rc})")
    return O, L


def stream_visible(q_sid, q_pos, slot_sid, slot_pos) -> np.ndarray:
    """Read Once, Answer Many, Section 3, Eq. 2: a query of stream q_sid at
    position q_pos may attend to a slot iff the slot is not after it (causal
    over positions; streams share positions) and the slot belongs to the
    document (sid -1) or to the query's own stream.  Returns the [nq, nk]
    boolean mask."""
    q_sid = np.asarray(q_sid).reshape(-1, 1)
    q_pos = np.asarray(q_pos).reshape(-1, 1)
    slot_sid = np.asarray(slot_sid).reshape(1, -1)
    slot_pos = np.asarray(slot_pos).reshape(1, -1)
    causal = slot_pos <= q_pos
    same = (slot_sid == -1) | (slot_sid == q_sid)
    return causal & same


def stream_masked(Q, K, V, q_sid, q_pos, slot_sid, slot_pos, scale: float):
    """Attention of query rows Q [nq, d] over one request's KV row K, V
    [nk, d] under the stream mask (``stream_visible``): each row is SDP over
    its visible slots (``sdp``).  Returns (O [nq, d], lse [nq]); a row with
    no visible slot gets (0, -inf)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    vis = stream_visible(q_sid, q_pos, slot_sid, slot_pos)
    O = np.zeros((Q.shape[0], Q.shape[1]))
    L = np.full(Q.shape[0], -np.inf)
    for i in range(Q.shape[0]):
        idx = np.nonzero(vis[i])[0]
        if idx.size:
            o, l = sdp(Q[i:i + 1], K[idx], V[idx], scale)
            O[i], L[i] = o[0], l[0]
    return O, L


def paged_decode(q, k_pool, v_pool, page_table, seq_lens, scale: float):
    """q [B,Hq,d] bf16; pools [P,Hkv,ps,d] bf16; page_table [B,W] int32;
    seq_lens [B] int32 -> (O [B,Hq,d], lse [B,Hq])."""
    lib = _load()
    B, Hq, d = q.shape
    _, Hkv, ps, _ = k_pool.shape
    qb = _bf16_bits(q)
    kp, vp = _bf16_bits(k_pool), _bf16_bits(v_pool)
    pt = np.ascontiguousarray(np.asarray(page_table, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    O = np.zeros((B, Hq, d))
    L = np.zeros((B, Hq))
    rc = lib.hpo_paged_decode(B, Hq, Hkv, d, float(scale), _ptr(qb, _u16p), Hq * d, d,
                              _ptr(kp, _u16p), _ptr(vp, _u16p), ps, _ptr(pt, _i32p),
                              pt.shape[1], _ptr(sl, _i32p), _ptr(O, _dp), _ptr(L, _dp))
    if rc != 0:
        raise ValueError("hpo_paged_decode rejected its arguments")
    return O, L


def paged_decode_e4m3(q, k8, v8, k_scale, v_scale, page_table, seq_lens, scale: float):
    """``paged_decode`` over E4M3 pools: k8/v8 uint8 [P,Hkv,ps,d] codes,
    k_scale/v_scale f32 [P,Hkv] -> (O [B,Hq,d], lse [B,Hq])."""
    lib = _load()
    B, Hq, d = q.shape
    _, Hkv, ps, _ = k8.shape
    qb = _bf16_bits(q)
    kb, vb = _u8_bytes(k8), _u8_bytes(v8)
    ks, vs = _f32(k_scale), _f32(v_scale)
    pt = np.ascontiguousarray(np.asarray(page_table, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    O = np.zeros((B, Hq, d))
    L = np.zeros((B, Hq))
    rc = lib.hpo_paged_decode_e4m3(B, Hq, Hkv, d, float(scale), _ptr(qb, _u16p), Hq * d, d, _ptr(kb, _u8p),
                                   _ptr(vb, _u8p), _ptr(ks, _fp), _ptr(vs, _fp), ps, _ptr(pt, _i32p), pt.shape[1],
                                   _ptr(sl, _i32p), _ptr(O, _dp), _ptr(L, _dp))
    if rc != 0:
        raise ValueError("hpo_paged_decode_e4m3 rejected its arguments")
    return O, L


def prefix(q, k, v, scale: float):
    """q [nb,Hq,d] bf16; k/v [len,Hkv,d] bf16 -> (O [nb,Hq,d], lse [nb,Hq])."""
    lib = _load()
    nb, Hq, d = q.shape
    ln, Hkv, _ = k.shape
    qb = _bf16_bits(q)
    kb, vb = _bf16_bits(k), _bf16_bits(v)
    O = np.zeros((nb, Hq, d))
    L = np.zeros((nb, Hq))
    rc = lib.hpo_prefix(nb, Hq, Hkv, d, float(scale), _ptr(qb, _u16p), Hq * d, d,
                        _ptr(kb, _u16p), _ptr(vb, _u16p), Hkv * d, d, ln, _ptr(O, _dp),
                        _ptr(L, _dp))
    if rc != 0:
        raise ValueError("hpo_prefix rejected its arguments")
    return O, L


class use_library:
    """Context manager that routes the wrappers through another compiled copy of
    the oracle (used by the tests that plant a mistake in the oracle source and
    check that the pins catch it)."""

    def __init__(self, so_path: str):
        self.so_path = so_path
        self._saved = None

    def __enter__(self):
        global _lib
        base = _load()
        lib = ctypes.CDLL(self.so_path)
        for name in ("hpo_sdp_f64", "hpo_merge", "hpo_partial_attn", "hpo_attn_reduce",
                     "hpo_cascade", "hpo_paged_decode", "hpo_prefix", "hpo_num_threads",
                     "hpo_set_num_threads", "hpo_e4m3_decode", "hpo_cascade_q", "hpo_paged_decode_e4m3"):
            f, g = getattr(lib, name), getattr(base, name)
            f.argtypes = g.argtypes
            f.restype = g.restype
        with _lock:
            self._saved = _lib
            _lib = lib
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self._saved
        return False


def source_path() -> str:
    return _SRC
