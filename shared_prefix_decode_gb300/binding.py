"""ctypes binding of the C ABI in include/hp.h.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libhp.so.  There is no fallback -- if the library is missing or
fails to load, every call raises.  PyTorch supplies device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import List, Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libhp.so")

HP_OK, HP_ERR_ARG, HP_ERR_UNSUPPORTED, HP_ERR_WORKSPACE, HP_ERR_CUDA, HP_ERR_BOUNDS, HP_ERR_DEVICE_TIMEOUT = range(7)
HP_BF16, HP_F32 = 0, 1
HP_KV_BF16, HP_KV_E4M3 = 0, 1

c_i32, c_i64, c_f32, c_vp, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class HpTreeNode(ctypes.Structure):
    _fields_ = [("seq_begin", c_i32), ("seq_end", c_i32), ("kv_len", c_i32), ("page_off", c_i32)]


class HpTreeLevel(ctypes.Structure):
    _fields_ = [("k_pool", c_vp), ("v_pool", c_vp), ("num_pages", c_i32), ("page_size", c_i32),
                ("num_nodes", c_i32), ("nodes", ctypes.POINTER(HpTreeNode)),
                ("page_ids", ctypes.POINTER(c_i32)), ("num_page_ids", c_i32), ("kv_type", c_i32),
                ("k_scale", c_vp), ("v_scale", c_vp)]


class HpTreeDesc(ctypes.Structure):
    _fields_ = [("num_levels", c_i32), ("B", c_i32), ("Hq", c_i32), ("Hkv", c_i32), ("d", c_i32),
                ("levels", ctypes.POINTER(HpTreeLevel)), ("num_sms", c_i32)]


class HpPlanInfo(ctypes.Structure):
    _fields_ = [("B", c_i32), ("Hq", c_i32), ("Hkv", c_i32), ("d", c_i32), ("n_tc_items", c_i32),
                ("n_small_items", c_i32), ("grid", c_i32), ("rec_stride", c_i32),
                ("num_levels", c_i32), ("merge_stride", c_i32),
                ("n_part_rows", c_i64), ("plan_bytes", c_i64), ("ws_bytes", c_i64),
                ("tag", ctypes.c_uint64)]


# name -> (restype, argtypes); the exported surface of hp.h
_SIGNATURES = {
    "hp_status_str": (ctypes.c_char_p, [c_i32]),
    "hp_build_arch": (c_i32, []),
    "hp_abi_version": (c_i32, []),
    "hp_merge_states": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_vp, c_i64, c_i32, c_vp]),
    "hp_suffix_workspace_bytes": (c_sz, [c_i32, c_i32, c_i32, c_i32, c_i32]),
    "hp_suffix_decode_paged": (c_i32, [c_vp, c_i64, c_i64, c_i32, c_vp, c_vp, c_i32, c_i32, c_vp, c_i32,
                                       c_vp, c_i32, c_i32, c_i32, c_f32, c_vp, c_i32, c_i64, c_i64,
                                       c_vp, c_i64, c_vp, c_sz, c_vp]),
    "hp_suffix_decode_paged_noalloc": (c_i32, [c_vp, c_i64, c_i64, c_i32, c_vp, c_vp, c_i32, c_i32, c_vp,
                                               c_i32, c_vp, c_i32, c_i32, c_i32, c_f32, c_vp, c_i32, c_i64,
                                               c_i64, c_vp, c_i64, c_vp]),
    "hp_suffix_decode_paged_e4m3": (c_i32, [c_vp, c_i64, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_vp,
                                            c_i32, c_vp, c_i32, c_i32, c_i32, c_f32, c_vp, c_i32, c_i64, c_i64,
                                            c_vp, c_i64, c_vp, c_sz, c_vp]),
    "hp_stream_workspace_bytes": (c_sz, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32]),
    "hp_stream_decode": (c_i32, [c_vp, c_i64, c_i64, c_i32, c_i32, c_vp, c_vp, c_i32, c_i32, c_vp, c_i32, c_vp, c_vp,
                                 c_vp, c_i32, c_vp, c_vp, c_i32, c_i32, c_i32, c_f32, c_vp, c_i32, c_i64, c_i64, c_vp,
                                 c_i64, c_vp, c_sz, c_vp]),
    "hp_prefix_workspace_bytes": (c_sz, [c_i32, c_i32, c_i32, c_i32, c_i32]),
    "hp_prefix_attn": (c_i32, [c_vp, c_i64, c_i64, c_i32, c_i32, c_vp, c_vp, c_i64, c_i64, c_i32,
                               c_i32, c_i32, c_i32, c_f32, c_vp, c_i32, c_i64, c_i64, c_vp, c_i64,
                               c_vp, c_sz, c_vp]),
    "hp_cascade_plan_bytes": (c_sz, [ctypes.POINTER(HpTreeDesc)]),
    "hp_cascade_plan": (c_i32, [ctypes.POINTER(HpTreeDesc), c_vp, c_sz, ctypes.POINTER(HpPlanInfo), c_vp]),
    "hp_cascade_decode": (c_i32, [c_vp, ctypes.POINTER(HpPlanInfo), c_vp, c_i64, c_i64, c_f32, c_vp,
                                  c_i32, c_i64, c_i64, c_vp, c_i64, c_vp, c_sz, c_vp]),
    "hp_cascade_host_workspace_bytes": (c_sz, [ctypes.POINTER(HpPlanInfo)]),
    "hp_cascade_decode_host": (c_i32, [c_vp, ctypes.POINTER(HpPlanInfo), c_vp, c_i64, c_i64, c_f32, c_vp,
                                       c_i32, c_i64, c_i64, c_vp, c_i64, c_vp, c_sz, c_vp]),
    "hp_cascade_decode_profiled": (c_i32, [c_vp, ctypes.POINTER(HpPlanInfo), c_vp, c_i64, c_i64, c_f32, c_vp,
                                           c_i32, c_i64, c_i64, c_vp, c_i64, c_vp, c_sz, c_vp,
                                           ctypes.POINTER(c_vp)]),
    "hp_cascade_loop_plan_bytes": (c_sz, [ctypes.POINTER(HpTreeDesc), c_i32]),
    "hp_cascade_loop_plan": (c_i32, [ctypes.POINTER(HpTreeDesc), c_i32, c_vp, c_sz, ctypes.POINTER(HpPlanInfo),
                                     c_vp]),
    "hp_cascade_append_kv": (c_i32, [c_vp, ctypes.POINTER(HpPlanInfo), c_vp, c_vp, c_i64, c_i64, c_vp, c_vp,
                                     c_sz, c_vp]),
    "hp_cascade_decode_loop": (c_i32, [c_vp, ctypes.POINTER(HpPlanInfo), c_vp, c_vp, c_i64, c_i64, c_f32, c_vp,
                                       c_i32, c_i64, c_i64, c_vp, c_i64, c_vp, c_sz, c_vp]),
    "hp_cascade_decode_append": (c_i32, [c_vp, ctypes.POINTER(HpPlanInfo), c_vp, c_vp, c_vp, c_i64, c_i64, c_vp,
                                         c_i64, c_i64, c_f32, c_vp, c_i32, c_i64, c_i64, c_vp, c_i64, c_vp, c_sz,
                                         c_vp]),
    "hp_cascade_contexts": (c_i32, [ctypes.POINTER(HpTreeDesc), ctypes.POINTER(c_i32), c_i32]),
    "hp_cascade_plan_stats": (c_i32, [ctypes.POINTER(HpTreeDesc), ctypes.POINTER(c_i64)]),
    "hp_cascade_plan_items": (c_i32, [ctypes.POINTER(HpTreeDesc), c_i32, ctypes.POINTER(c_i32), c_i32]),
    "hp_cascade_plan_merge_table": (c_i32, [ctypes.POINTER(HpTreeDesc), c_i32, ctypes.POINTER(c_i32), c_i64]),
    "hp_cascade_plan_item_pages": (c_i64, [ctypes.POINTER(HpTreeDesc), c_i32, ctypes.POINTER(c_i64),
                                           ctypes.POINTER(c_i32), c_i64]),
    "hp_read_device_status": (c_i32, [c_vp, c_vp]),
    "hp_test_withhold_first_tile": (None, [c_i32]),
}

_lib = None
_lock = threading.Lock()


class HpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} (status {status})")


def library() -> ctypes.CDLL:
    """Load libhp.so (built by ``shared_prefix_decode_gb300.build``).  Raises
    if it is missing: there is no other implementation to fall back to."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing; run "
                                   "`python -m shared_prefix_decode_gb300.build` (nvcc, sm_103a)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def exported_symbols() -> List[str]:
    return list(_SIGNATURES)


def status_str(status: int) -> str:
    return library().hp_status_str(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != HP_OK:
        raise HpError(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dt(dtype) -> int:
    if dtype == torch.bfloat16:
        return HP_BF16
    if dtype == torch.float32:
        return HP_F32
    raise ValueError(f"output dtype must be bfloat16 or float32, not {dtype}")


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A zeroed workspace (the first word is the device status word)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ----------------------------------------------------------------- merge
def hp_merge_states(o_a: torch.Tensor, lse_a: torch.Tensor, o_b: torch.Tensor, lse_b: torch.Tensor,
                    out: Optional[torch.Tensor] = None, lse_out: Optional[torch.Tensor] = None,
                    out_dtype=torch.float32, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Exact two-state merge; o_* f32 [rows, d], lse_* f32 [rows]."""
    _need(o_a.dtype == torch.float32 and o_b.dtype == torch.float32, "states must be float32")
    _need(o_a.is_contiguous() and o_b.is_contiguous(), "states must be contiguous")
    rows, d = o_a.shape
    if out is None:
        out = torch.empty(rows, d, dtype=out_dtype, device=o_a.device)
    if lse_out is None:
        lse_out = torch.empty(rows, dtype=torch.float32, device=o_a.device)
    _check(library().hp_merge_states(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(out),
                                     _dt(out.dtype), _ptr(lse_out), rows, d, _stream(stream)),
           "hp_merge_states")
    return out, lse_out


# ----------------------------------------------------- paged suffix decode
def suffix_workspace_bytes(B: int, Hq: int, d: int, pt_stride: int, page_size: int) -> int:
    return int(library().hp_suffix_workspace_bytes(B, Hq, d, pt_stride, page_size))


def hp_suffix_decode_paged(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           page_table: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                           ws: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                           stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """q [B,Hq,d] bf16; pools [P,Hkv,ps,d] bf16; page_table [B,W] int32;
    seq_lens [B] int32 (device)."""
    B, Hq, d = q.shape
    P, Hkv, ps, d2 = k_pool.shape
    _need(d2 == d and v_pool.shape == k_pool.shape, "pool shape mismatch")
    _need(page_table.dtype == torch.int32 and seq_lens.dtype == torch.int32, "int32 tables")
    _need(page_table.is_contiguous() and k_pool.is_contiguous() and v_pool.is_contiguous(), "contiguous")
    if out is None:
        out = torch.empty(B, Hq, d, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = alloc_workspace(suffix_workspace_bytes(B, Hq, d, page_table.shape[1], ps), q.device)
    _check(library().hp_suffix_decode_paged(
        _ptr(q), q.stride(0), q.stride(1), B, _ptr(k_pool), _ptr(v_pool), P, ps, _ptr(page_table),
        page_table.stride(0), _ptr(seq_lens), Hq, Hkv, d, float(scale), _ptr(out), _dt(out.dtype),
        out.stride(0), out.stride(1), _ptr(lse), lse.stride(0), _ptr(ws), ws.numel(), _stream(stream)),
        "hp_suffix_decode_paged")
    return out, lse


def hp_suffix_decode_paged_e4m3(q: torch.Tensor, k8: torch.Tensor, v8: torch.Tensor, k_scale: torch.Tensor,
                                v_scale: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                                out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                                ws: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                                stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """hp_suffix_decode_paged over E4M3 pools: k8/v8 uint8 [P,Hkv,ps,d] codes,
    k_scale/v_scale f32 [P,Hkv] (device)."""
    B, Hq, d = q.shape
    P, Hkv, ps, d2 = k8.shape
    _need(d2 == d and v8.shape == k8.shape and k8.dtype == torch.uint8 and v8.dtype == torch.uint8,
          "E4M3 pools must be uint8 [P,Hkv,ps,d]")
    _need(k_scale.dtype == torch.float32 and v_scale.dtype == torch.float32 and tuple(k_scale.shape) == (P, Hkv)
          and tuple(v_scale.shape) == (P, Hkv) and k_scale.is_contiguous() and v_scale.is_contiguous(),
          "scales must be contiguous f32 [P,Hkv]")
    _need(page_table.dtype == torch.int32 and seq_lens.dtype == torch.int32, "int32 tables")
    _need(page_table.is_contiguous() and k8.is_contiguous() and v8.is_contiguous(), "contiguous")
    if out is None:
        out = torch.empty(B, Hq, d, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = alloc_workspace(suffix_workspace_bytes(B, Hq, d, page_table.shape[1], ps), q.device)
    _check(library().hp_suffix_decode_paged_e4m3(
        _ptr(q), q.stride(0), q.stride(1), B, _ptr(k8), _ptr(v8), _ptr(k_scale), _ptr(v_scale), P, ps,
        _ptr(page_table), page_table.stride(0), _ptr(seq_lens), Hq, Hkv, d, float(scale), _ptr(out), _dt(out.dtype),
        out.stride(0), out.stride(1), _ptr(lse), lse.stride(0), _ptr(ws), ws.numel(), _stream(stream)),
        "hp_suffix_decode_paged_e4m3")
    return out, lse


# ------------------------------------------------- Parallel Prompting rows
def stream_workspace_bytes(R: int, P: int, Hq: int, Hkv: int, d: int, pt_stride: int, page_size: int) -> int:
    return int(library().hp_stream_workspace_bytes(R, P, Hq, Hkv, d, pt_stride, page_size))


def hp_stream_decode(q: torch.Tensor, rows, P: int, scale: float, out: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                     stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """q [R*P, Hq, d] bf16; ``rows`` a ``workloads.StreamRows`` on the GPU
    (pools, row page table and lengths, slot stream ids and positions, query
    stream ids and positions)."""
    RP, Hq, d = q.shape
    _need(RP % P == 0, "q must hold R * P query rows")
    R = RP // P
    Pn, Hkv, ps, d2 = rows.k_pool.shape
    _need(d2 == d and rows.v_pool.shape == rows.k_pool.shape, "pool shape mismatch")
    for t, n in ((rows.row_pages, "row_pages"), (rows.row_len, "row_len"), (rows.slot_sid, "slot_sid"),
                 (rows.slot_pos, "slot_pos"), (rows.q_sid, "q_sid"), (rows.q_pos, "q_pos")):
        _need(t.dtype == torch.int32 and t.is_contiguous() and t.is_cuda, f"{n} must be contiguous int32 on the GPU")
    _need(tuple(rows.row_len.shape) == (R,) and tuple(rows.q_sid.shape) == (RP,) and
          tuple(rows.q_pos.shape) == (RP,) and rows.row_pages.shape[0] == R and rows.slot_sid.shape == rows.slot_pos.shape
          and rows.slot_sid.shape[0] == R, "row arrays do not match R and P")
    if out is None:
        out = torch.empty(RP, Hq, d, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(RP, Hq, dtype=torch.float32, device=q.device)
    pt = rows.row_pages.shape[1]
    if ws is None:
        ws = alloc_workspace(stream_workspace_bytes(R, P, Hq, Hkv, d, pt, ps), q.device)
    _check(library().hp_stream_decode(
        _ptr(q), q.stride(0), q.stride(1), R, P, _ptr(rows.k_pool), _ptr(rows.v_pool), Pn, ps, _ptr(rows.row_pages),
        pt, _ptr(rows.row_len), _ptr(rows.slot_sid), _ptr(rows.slot_pos), rows.slot_sid.shape[1], _ptr(rows.q_sid),
        _ptr(rows.q_pos), Hq, Hkv, d, float(scale), _ptr(out), _dt(out.dtype), out.stride(0), out.stride(1),
        _ptr(lse), lse.stride(0), _ptr(ws), ws.numel(), _stream(stream)), "hp_stream_decode")
    return out, lse


# --------------------------------------------------- contiguous prefix
def prefix_workspace_bytes(rows: int, Hq: int, Hkv: int, d: int, prefix_len: int) -> int:
    return int(library().hp_prefix_workspace_bytes(rows, Hq, Hkv, d, prefix_len))


def hp_prefix_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float, row_begin: int = 0,
                   rows: Optional[int] = None, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                   out_dtype=torch.bfloat16, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """q [B,Hq,d] bf16; k/v [len,Hkv,d] bf16 (strided rows allowed)."""
    B, Hq, d = q.shape
    ln, Hkv, d2 = k.shape
    _need(d2 == d and v.shape == k.shape and v.stride() == k.stride(), "prefix shape mismatch")
    _need(k.stride(2) == 1, "head dimension must be contiguous")
    if rows is None:
        rows = B - row_begin
    if out is None:
        out = torch.empty(B, Hq, d, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = alloc_workspace(prefix_workspace_bytes(rows, Hq, Hkv, d, ln), q.device)
    _check(library().hp_prefix_attn(
        _ptr(q), q.stride(0), q.stride(1), row_begin, rows, _ptr(k), _ptr(v), k.stride(0), k.stride(1),
        ln, Hq, Hkv, d, float(scale), _ptr(out), _dt(out.dtype), out.stride(0), out.stride(1), _ptr(lse),
        lse.stride(0), _ptr(ws), ws.numel(), _stream(stream)), "hp_prefix_attn")
    return out, lse


# ------------------------------------------------------------- cascade
class _Desc:
    """Keeps the ctypes arrays of a tree descriptor alive."""

    def __init__(self, levels, B: int, Hq: int, Hkv: int, d: int, num_sms: int = 0):
        self.keep = []
        arr = (HpTreeLevel * max(len(levels), 1))()
        for i, lv in enumerate(levels):
            # (k_pool, v_pool, num_pages, page_size, nodes, page_ids[, kv_type, k_scale, v_scale])
            k_pool, v_pool, num_pages, page_size, nodes, page_ids = lv[:6]
            kv_type, k_scale, v_scale = tuple(lv[6:9]) if len(lv) >= 9 else (HP_KV_BF16, None, None)
            nodes = [tuple(int(x) for x in n) for n in nodes]
            n_arr = (HpTreeNode * max(len(nodes), 1))(*[HpTreeNode(*n) for n in nodes])
            ids = [int(x) for x in page_ids]
            i_arr = (c_i32 * max(len(ids), 1))(*ids)
            self.keep += [n_arr, i_arr]
            arr[i] = HpTreeLevel(k_pool, v_pool, num_pages, page_size, len(nodes),
                                 ctypes.cast(n_arr, ctypes.POINTER(HpTreeNode)),
                                 ctypes.cast(i_arr, ctypes.POINTER(c_i32)), len(ids), int(kv_type), k_scale, v_scale)
        self.keep.append(arr)
        self.desc = HpTreeDesc(len(levels), B, Hq, Hkv, d, ctypes.cast(arr, ctypes.POINTER(HpTreeLevel)),
                               num_sms)


def _levels_of(wl) -> list:
    """Tree levels of a ``workloads.CascadeWorkload`` (pools must be on the GPU
    for planning; host-only inspection accepts CPU pools).  Levels marked
    e4m3 read the workload's E4M3 pools and scales."""
    out = []
    for lv in wl.levels:
        if getattr(lv, "e4m3", False):
            q8 = wl.q8
            out.append((q8.k.data_ptr(), q8.v.data_ptr(), wl.num_pages, wl.page_size, lv.nodes.tolist(),
                        lv.page_ids.cpu().tolist(), HP_KV_E4M3, q8.k_scale.data_ptr(), q8.v_scale.data_ptr()))
        else:
            out.append((wl.k_pool.data_ptr(), wl.v_pool.data_ptr(), wl.num_pages, wl.page_size,
                        lv.nodes.tolist(), lv.page_ids.cpu().tolist()))
    return out


def hp_cascade_contexts(levels, B, Hq, Hkv, d) -> List[Tuple[int, int, int, int, int]]:
    """(level, node, seq_begin, seq_end, batched) context list (host only)."""
    D = _Desc(levels, B, Hq, Hkv, d, num_sms=1)
    n = library().hp_cascade_contexts(ctypes.byref(D.desc), None, 0)
    if n < 0:
        raise HpError(HP_ERR_ARG, "hp_cascade_contexts")
    buf = (c_i32 * (5 * max(n, 1)))()
    library().hp_cascade_contexts(ctypes.byref(D.desc), buf, n)
    return [tuple(buf[5 * i:5 * i + 5]) for i in range(n)]


def hp_cascade_plan_stats(levels, B, Hq, Hkv, d, num_sms: int = 152) -> Tuple[int, int, int, int]:
    D = _Desc(levels, B, Hq, Hkv, d, num_sms=num_sms)
    st = (c_i64 * 4)()
    if library().hp_cascade_plan_stats(ctypes.byref(D.desc), st) != 0:
        raise HpError(HP_ERR_ARG, "hp_cascade_plan_stats")
    return tuple(int(x) for x in st)


PLAN_ITEM_FIELDS = ("level", "seq_begin", "n_seq", "kvh", "n_kvh", "k0", "k1", "part_row", "cta", "tc", "len_seq")


def hp_cascade_plan_items(levels, B, Hq, Hkv, d, capacity: int = 0, num_sms: int = 152) -> List[dict]:
    """The plan's work items (host only), CTA by CTA: dicts of PLAN_ITEM_FIELDS."""
    D = _Desc(levels, B, Hq, Hkv, d, num_sms=num_sms)
    n = library().hp_cascade_plan_items(ctypes.byref(D.desc), int(capacity), None, 0)
    if n < 0:
        raise HpError(HP_ERR_ARG, "hp_cascade_plan_items")
    buf = (c_i32 * (11 * max(n, 1)))()
    library().hp_cascade_plan_items(ctypes.byref(D.desc), int(capacity), buf, n)
    return [dict(zip(PLAN_ITEM_FIELDS, buf[11 * i:11 * i + 11])) for i in range(n)]


def hp_cascade_plan_item_pages(levels, B, Hq, Hkv, d, capacity: int = 0, num_sms: int = 152) -> List[List[int]]:
    """Per item (hp_cascade_plan_items' order) the page ids its record carries."""
    D = _Desc(levels, B, Hq, Hkv, d, num_sms=num_sms)
    lib = library()
    n_items = lib.hp_cascade_plan_items(ctypes.byref(D.desc), int(capacity), None, 0)
    if n_items < 0:
        raise HpError(HP_ERR_ARG, "hp_cascade_plan_item_pages")
    offs = (c_i64 * (n_items + 1))()
    total = lib.hp_cascade_plan_item_pages(ctypes.byref(D.desc), int(capacity), offs, None, 0)
    pages = (c_i32 * max(total, 1))()
    lib.hp_cascade_plan_item_pages(ctypes.byref(D.desc), int(capacity), offs, pages, total)
    return [list(pages[offs[i]:offs[i + 1]]) for i in range(n_items)]


def hp_cascade_plan_merge_table(levels, B, Hq, Hkv, d, capacity: int = 0, num_sms: int = 152) -> List[List[int]]:
    """The plan's merge lists (host only): entry b*Hkv + kvh lists the partial
    rows (query head g = 0 of the group) merged into row (b, kvh*G + g)."""
    D = _Desc(levels, B, Hq, Hkv, d, num_sms=num_sms)
    stride = library().hp_cascade_plan_merge_table(ctypes.byref(D.desc), int(capacity), None, 0)
    if stride < 0:
        raise HpError(HP_ERR_ARG, "hp_cascade_plan_merge_table")
    n = B * Hkv * stride
    buf = (c_i32 * max(n, 1))()
    library().hp_cascade_plan_merge_table(ctypes.byref(D.desc), int(capacity), buf, n)
    return [list(buf[i * stride + 1:i * stride + 1 + buf[i * stride]]) for i in range(B * Hkv)]


def hp_cascade_plan_bytes(levels, B, Hq, Hkv, d, num_sms: int = 0) -> int:
    D = _Desc(levels, B, Hq, Hkv, d, num_sms=num_sms)
    return int(library().hp_cascade_plan_bytes(ctypes.byref(D.desc)))


class CascadePlan:
    """A device-resident plan for one prefix tree (re-plan when the tree
    changes).  Owns the plan buffer and a workspace sized for it."""

    def __init__(self, levels, B: int, Hq: int, Hkv: int, d: int, device="cuda", stream=None,
                 num_sms: int = 0, workspace: bool = True, capacity: int = 0):
        D = _Desc(levels, B, Hq, Hkv, d, num_sms=num_sms)
        lib = library()
        if capacity:
            nbytes = int(lib.hp_cascade_loop_plan_bytes(ctypes.byref(D.desc), int(capacity)))
        else:
            nbytes = int(lib.hp_cascade_plan_bytes(ctypes.byref(D.desc)))
        if nbytes == 0:
            raise HpError(HP_ERR_ARG, "hp_cascade_loop_plan_bytes" if capacity else "hp_cascade_plan_bytes")
        self.plan = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.info = HpPlanInfo()
        if capacity:
            _check(lib.hp_cascade_loop_plan(ctypes.byref(D.desc), int(capacity), _ptr(self.plan), nbytes,
                                            ctypes.byref(self.info), _stream(stream)), "hp_cascade_loop_plan")
        else:
            _check(lib.hp_cascade_plan(ctypes.byref(D.desc), _ptr(self.plan), nbytes,
                                       ctypes.byref(self.info), _stream(stream)), "hp_cascade_plan")
        self.B, self.Hq, self.Hkv, self.d = B, Hq, Hkv, d
        self.capacity = int(capacity)
        self.ws = alloc_workspace(self.info.ws_bytes, device) if workspace else None

    @classmethod
    def from_workload(cls, wl, **kw) -> "CascadePlan":
        return cls(_levels_of(wl), wl.B, wl.Hq, wl.Hkv, wl.d, device=wl.q.device, **kw)

    def decode(self, q: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
               lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
               out_dtype=torch.bfloat16, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        return hp_cascade_decode(self, q, scale, out=out, lse=lse, ws=ws, out_dtype=out_dtype, stream=stream)


def hp_cascade_plan(levels, B, Hq, Hkv, d, device="cuda", stream=None, num_sms: int = 0) -> CascadePlan:
    return CascadePlan(levels, B, Hq, Hkv, d, device=device, stream=stream, num_sms=num_sms)


def _check_step_tensors(plan: CascadePlan, q: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
                        ws: torch.Tensor):
    """The layouts hp_cascade_decode reads: q [B][Hq][d] bf16 and out
    [B][Hq][d] with unit stride along d, lse [B][Hq] f32 with unit stride
    along heads, all on the device; the workspace a byte tensor."""
    _need(q.dim() == 3 and tuple(q.shape) == (plan.B, plan.Hq, plan.d), "q shape does not match the plan")
    _need(q.dtype == torch.bfloat16 and q.is_cuda and q.stride(2) == 1, "q must be bf16 on the GPU, d contiguous")
    _need(tuple(out.shape) == tuple(q.shape) and out.dtype in (torch.bfloat16, torch.float32) and out.is_cuda
          and out.stride(2) == 1, "out must be [B][Hq][d] bf16 or f32 on the GPU, d contiguous")
    _need(tuple(lse.shape) == (plan.B, plan.Hq) and lse.dtype == torch.float32 and lse.is_cuda
          and lse.stride(1) == 1, "lse must be [B][Hq] f32 on the GPU, heads contiguous")
    _need(ws is not None and ws.dtype == torch.uint8 and ws.is_cuda, "workspace must be a uint8 GPU tensor")


def hp_cascade_decode(plan: CascadePlan, q: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                      out_dtype=torch.bfloat16, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    B, Hq, d = q.shape
    if out is None:
        out = torch.empty(B, Hq, d, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = plan.ws
    _check_step_tensors(plan, q, out, lse, ws)
    _check(library().hp_cascade_decode(
        _ptr(plan.plan), ctypes.byref(plan.info), _ptr(q), q.stride(0), q.stride(1), float(scale), _ptr(out),
        _dt(out.dtype), out.stride(0), out.stride(1), _ptr(lse), lse.stride(0), _ptr(ws), ws.numel(),
        _stream(stream)), "hp_cascade_decode")
    return out, lse


def host_workspace_bytes(plan: CascadePlan) -> int:
    n = int(library().hp_cascade_host_workspace_bytes(ctypes.byref(plan.info)))
    if n == 0:
        raise HpError(HP_ERR_ARG, "hp_cascade_host_workspace_bytes")
    return n


def hp_cascade_decode_host(plan: CascadePlan, q_host: torch.Tensor, scale: float, out_host: torch.Tensor,
                           lse_host: Optional[torch.Tensor], ws: torch.Tensor, stream=None) -> None:
    """One step with q read from, and O / LSE written to, page-locked host
    tensors (``tensor.pin_memory()``); ws: a GPU byte tensor of at least
    host_workspace_bytes(plan)."""
    _need(q_host.dim() == 3 and tuple(q_host.shape) == (plan.B, plan.Hq, plan.d), "q shape does not match the plan")
    _need(q_host.dtype == torch.bfloat16 and not q_host.is_cuda and q_host.is_pinned() and q_host.stride(2) == 1,
          "q_host must be a pinned bf16 host tensor, d contiguous")
    _need(tuple(out_host.shape) == tuple(q_host.shape) and out_host.dtype in (torch.bfloat16, torch.float32)
          and not out_host.is_cuda and out_host.is_pinned() and out_host.stride(2) == 1,
          "out_host must be a pinned [B][Hq][d] bf16 or f32 host tensor, d contiguous")
    if lse_host is not None:
        _need(tuple(lse_host.shape) == (plan.B, plan.Hq) and lse_host.dtype == torch.float32
              and not lse_host.is_cuda and lse_host.is_pinned() and lse_host.stride(1) == 1,
              "lse_host must be a pinned [B][Hq] f32 host tensor, heads contiguous")
    _need(ws is not None and ws.dtype == torch.uint8 and ws.is_cuda, "workspace must be a uint8 GPU tensor")
    _check(library().hp_cascade_decode_host(
        _ptr(plan.plan), ctypes.byref(plan.info), _ptr(q_host), q_host.stride(0), q_host.stride(1), float(scale),
        _ptr(out_host), _dt(out_host.dtype), out_host.stride(0), out_host.stride(1),
        None if lse_host is None else _ptr(lse_host), 0 if lse_host is None else lse_host.stride(0), _ptr(ws),
        ws.numel(), _stream(stream)), "hp_cascade_decode_host")


def hp_cascade_decode_profiled(plan: CascadePlan, q: torch.Tensor, scale: float, out: torch.Tensor,
                               lse: torch.Tensor, events: Sequence[Optional[torch.cuda.Event]],
                               ws: Optional[torch.Tensor] = None, stream=None) -> None:
    """hp_cascade_decode that records events[0..2] around its two kernels
    (events[3] is not used)."""
    _check_step_tensors(plan, q, out, lse, plan.ws if ws is None else ws)
    ev = (c_vp * 4)(*[None if e is None else e.cuda_event for e in events])
    _check(library().hp_cascade_decode_profiled(
        _ptr(plan.plan), ctypes.byref(plan.info), _ptr(q), q.stride(0), q.stride(1), float(scale), _ptr(out),
        _dt(out.dtype), out.stride(0), out.stride(1), _ptr(lse), lse.stride(0), _ptr(plan.ws if ws is None else ws),
        (plan.ws if ws is None else ws).numel(), _stream(stream), ev), "hp_cascade_decode_profiled")


# ---------------------------------------------------------- decode loop
def hp_cascade_loop_plan_bytes(levels, B, Hq, Hkv, d, capacity: int, num_sms: int = 0) -> int:
    D = _Desc(levels, B, Hq, Hkv, d, num_sms=num_sms)
    return int(library().hp_cascade_loop_plan_bytes(ctypes.byref(D.desc), int(capacity)))


class LoopPlan(CascadePlan):
    """A decode-loop plan (hp_cascade_loop_plan): the tree's last level holds
    each sequence's suffix, with pages reserved up to ``capacity`` tokens.
    ``suffix_len`` (device int32 [B], owned here) starts at the suffixes'
    plan-time lengths; ``append`` writes one token per sequence and moves it
    on, ``decode`` attends over the current lengths."""

    def __init__(self, levels, B: int, Hq: int, Hkv: int, d: int, capacity: int, device="cuda",
                 stream=None, num_sms: int = 0):
        _need(int(capacity) >= 1, "capacity must be at least 1")
        super().__init__(levels, B, Hq, Hkv, d, device=device, stream=stream, num_sms=num_sms,
                         capacity=int(capacity))
        lens = [0] * B
        for sb, se, kl, _ in levels[-1][4]:
            lens[int(sb)] = int(kl)
        self.suffix_len = torch.tensor(lens, dtype=torch.int32, device=device)

    @classmethod
    def from_workload(cls, wl, capacity: int, **kw) -> "LoopPlan":
        return cls(_levels_of(wl), wl.B, wl.Hq, wl.Hkv, wl.d, capacity, device=wl.q.device, **kw)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
        hp_cascade_append_kv(self, k_new, v_new, stream=stream)

    def decode_append(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, scale: float,
                      out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                      out_dtype=torch.bfloat16, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        return hp_cascade_decode_append(self, q, k_new, v_new, scale, out=out, lse=lse, out_dtype=out_dtype,
                                        stream=stream)

    def decode(self, q: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
               lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
               out_dtype=torch.bfloat16, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        return hp_cascade_decode_loop(self, q, scale, out=out, lse=lse, ws=ws, out_dtype=out_dtype, stream=stream)


def _check_token_rows(plan, k_new: torch.Tensor, v_new: torch.Tensor):
    shape = (plan.B, plan.Hkv, plan.d)
    for t, nm in ((k_new, "k_new"), (v_new, "v_new")):
        _need(tuple(t.shape) == shape and t.dtype == torch.bfloat16 and t.is_cuda and t.stride(2) == 1,
              f"{nm} must be bf16 [B][Hkv][d] on the GPU, d contiguous")
    _need(k_new.stride() == v_new.stride(), "k_new and v_new must have the same strides")


def hp_cascade_append_kv(plan: LoopPlan, k_new: torch.Tensor, v_new: torch.Tensor, ws: Optional[torch.Tensor] = None,
                         stream=None) -> None:
    """One token per sequence: k_new / v_new bf16 [B][Hkv][d] (head dimension
    contiguous) go to position plan.suffix_len[b] of each suffix."""
    _check_token_rows(plan, k_new, v_new)
    ws = plan.ws if ws is None else ws
    _need(ws is not None and ws.dtype == torch.uint8 and ws.is_cuda, "workspace must be a uint8 GPU tensor")
    _check(library().hp_cascade_append_kv(
        _ptr(plan.plan), ctypes.byref(plan.info), _ptr(k_new), _ptr(v_new), k_new.stride(0), k_new.stride(1),
        _ptr(plan.suffix_len), _ptr(ws), ws.numel(), _stream(stream)), "hp_cascade_append_kv")


def hp_cascade_decode_loop(plan: LoopPlan, q: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
                           lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                           out_dtype=torch.bfloat16, stream=None,
                           suffix_len: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    B, Hq, d = q.shape
    if out is None:
        out = torch.empty(B, Hq, d, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = plan.ws
    lens = plan.suffix_len if suffix_len is None else suffix_len
    _need(lens.dtype == torch.int32 and lens.is_cuda and tuple(lens.shape) == (plan.B,) and lens.is_contiguous(),
          "suffix_len must be a contiguous int32 [B] GPU tensor")
    _check_step_tensors(plan, q, out, lse, ws)
    _check(library().hp_cascade_decode_loop(
        _ptr(plan.plan), ctypes.byref(plan.info), _ptr(lens), _ptr(q), q.stride(0), q.stride(1), float(scale),
        _ptr(out), _dt(out.dtype), out.stride(0), out.stride(1), _ptr(lse), lse.stride(0), _ptr(ws), ws.numel(),
        _stream(stream)), "hp_cascade_decode_loop")
    return out, lse


def hp_cascade_decode_append(plan: LoopPlan, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                             scale: float, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                             ws: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                             stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Append and decode in one step's two launches (plan.suffix_len advances)."""
    B, Hq, d = q.shape
    if out is None:
        out = torch.empty(B, Hq, d, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = plan.ws
    _check_token_rows(plan, k_new, v_new)
    _check_step_tensors(plan, q, out, lse, ws)
    lens = plan.suffix_len
    _check(library().hp_cascade_decode_append(
        _ptr(plan.plan), ctypes.byref(plan.info), _ptr(lens), _ptr(k_new), _ptr(v_new), k_new.stride(0),
        k_new.stride(1), _ptr(q), q.stride(0), q.stride(1), float(scale), _ptr(out), _dt(out.dtype), out.stride(0),
        out.stride(1), _ptr(lse), lse.stride(0), _ptr(ws), ws.numel(), _stream(stream)), "hp_cascade_decode_append")
    return out, lse


def hp_read_device_status(ws: torch.Tensor, stream=None) -> int:
    """Reads and clears the workspace status word (synchronises the stream)."""
    return int(library().hp_read_device_status(_ptr(ws), _stream(stream)))
