"""Seeded synthetic inputs for shared-prefix (cascade) decode attention.

This module only builds inputs: query tensors, paged KV pools, page tables and
the per-level prefix-tree descriptor.  It holds none of the attention
arithmetic, so both the CUDA path and the fp64 oracle consume exactly the same
tensors.

Storage model (Hydragen, "Hierarchical Sharing"; ChunkAttention, "Prefix-Aware
KV Cache (PAKV): The Prefix Tree Structure"):

* all KV lives in one page pool per workload, laid out ``[page][Hkv][ps][d]``
  (bf16).  A shared prefix is the same physical pages for every sequence that
  shares it.
* the tree is given level by level.  A level is a list of nodes
  ``(seq_begin, seq_end, kv_len, page_off)``: the node's ``kv_len`` tokens are
  visible to the contiguous sequence range ``[seq_begin, seq_end)`` and sit in
  pages ``page_ids[page_off : page_off + ceil(kv_len / ps)]``.
* a private suffix is a level whose nodes cover one sequence each.
* sequence ``b`` sees, in order, the tokens of the node that covers it at each
  level.  A level may leave a sequence uncovered (it then contributes nothing).

Random draws (seeded ``torch.Generator``): lengths with ``torch.randint``
(inclusive ranges), the physical page permutation with ``torch.randperm``, then
q, K, V as N(0,1) fp32 rounded to bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import torch

__all__ = [
    "TreeLevel",
    "CascadeWorkload",
    "build_cascade",
    "make_config",
    "CONFIG_NAMES",
    "full_page_tables",
    "apply_probe",
    "with_suffix_capacity",
    "append_token",
    "decode_tokens",
    "StreamRequests",
    "stream_requests",
    "streams_as_tree",
    "StreamRows",
    "stream_rows_paged",
    "E4M3Pools",
    "quantize_e4m3",
    "with_e4m3_levels",
]

E4M3_MAX = 448.0  # largest finite value of the E4M3 format


@dataclass
class TreeLevel:
    """One level of the prefix tree.

    ``nodes`` is an int32 tensor ``[n, 4]`` of ``(seq_begin, seq_end, kv_len,
    page_off)``; ``page_ids`` an int32 tensor of physical page ids.
    """

    nodes: torch.Tensor
    page_ids: torch.Tensor
    e4m3: bool = False  # keys and values of this level come from the workload's E4M3 pools

    @property
    def num_nodes(self) -> int:
        return int(self.nodes.shape[0])


@dataclass
class E4M3Pools:
    """Reduced-precision copies of a workload's pools: E4M3 codes (raw bytes,
    uint8 ``[num_pages, Hkv, ps, d]``) with one f32 scale per (page, KV head)
    for K and for V; the stored value of a code is its E4M3 value times the
    scale of its page and head."""

    k: torch.Tensor
    v: torch.Tensor
    k_scale: torch.Tensor  # f32 [num_pages, Hkv]
    v_scale: torch.Tensor

    def to(self, device) -> "E4M3Pools":
        return E4M3Pools(self.k.to(device), self.v.to(device), self.k_scale.to(device), self.v_scale.to(device))


@dataclass
class CascadeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    scale: float
    q: torch.Tensor  # [B, Hq, d] bf16
    k_pool: torch.Tensor  # [num_pages, Hkv, ps, d] bf16
    v_pool: torch.Tensor
    levels: List[TreeLevel] = field(default_factory=list)
    seed: int = 0
    part: str = "all"  # make_config's part: the whole workload, or one pass of it
    q8: Optional[E4M3Pools] = None  # pools of the levels marked e4m3

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[0])

    def seq_kv_len(self) -> List[int]:
        """Total number of keys each sequence attends over."""
        out = [0] * self.B
        for lv in self.levels:
            for sb, se, kl, _ in lv.nodes.tolist():
                for b in range(sb, se):
                    out[b] += kl
        return out

    def unique_kv_tokens(self) -> int:
        """Stored tokens: each node's tokens once, however many sequences share them."""
        return sum(int(lv.nodes[:, 2].sum()) for lv in self.levels)

    def unique_kv_bytes(self) -> int:
        """Bytes of K and V stored once: 2 bytes per element for bf16 levels,
        1 for E4M3 levels plus their two f32 scales per (page, KV head)."""
        tot = 0
        for lv in self.levels:
            toks = int(lv.nodes[:, 2].sum())
            if lv.e4m3:
                pages = sum((int(n[2]) + self.page_size - 1) // self.page_size for n in lv.nodes.tolist())
                tot += toks * self.Hkv * self.d * 2 + pages * self.Hkv * 8
            else:
                tot += toks * self.Hkv * self.d * 4
        return tot

    def shared_flops(self) -> int:
        """4 * rows * keys * d over nodes that cover more than one sequence
        (the batched matrix-matrix part)."""
        tot = 0
        for lv in self.levels:
            for sb, se, kl, _ in lv.nodes.tolist():
                if se - sb > 1:
                    tot += 4 * (se - sb) * self.Hq * kl * self.d
        return tot

    def to(self, device) -> "CascadeWorkload":
        lv = [TreeLevel(l.nodes.clone(), l.page_ids.to(device), l.e4m3) for l in self.levels]
        return CascadeWorkload(self.name, self.B, self.Hq, self.Hkv, self.d, self.page_size,
                               self.scale, self.q.to(device), self.k_pool.to(device),
                               self.v_pool.to(device), lv, self.seed, self.part,
                               self.q8.to(device) if self.q8 is not None else None)


def build_cascade(
    name: str,
    *,
    B: int,
    Hq: int,
    Hkv: int,
    d: int,
    page_size: int,
    shared: Sequence[Sequence[Tuple[int, int, int]]],
    suffix_lens: Optional[Sequence[int]] = None,
    suffix_range: Optional[Tuple[int, int]] = None,
    seed: int = 0,
    scale: Optional[float] = None,
    shuffle: bool = True,
    extra_suffix_range: Optional[Tuple[int, int]] = None,
    device=None,
) -> CascadeWorkload:
    """Build a workload.

    ``shared`` lists the shared levels, each a list of ``(seq_begin, seq_end,
    kv_len)`` nodes.  Private suffix lengths are either given or drawn from
    ``suffix_range`` (inclusive); ``extra_suffix_range`` adds a second drawn
    length to each suffix (question + answer-so-far).  ``device``: where q, K
    and V are drawn (a CUDA device draws them there from a generator of that
    device, seeded alike: the same tree and distributions, other values --
    for timing runs of the large shapes; the oracle's inputs come from the
    CPU draw).
    """
    g = torch.Generator().manual_seed(seed)
    if suffix_lens is None:
        lo, hi = suffix_range if suffix_range is not None else (0, 0)
        suffix_lens = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
        if extra_suffix_range is not None:
            lo2, hi2 = extra_suffix_range
            extra = torch.randint(lo2, hi2 + 1, (B,), generator=g).tolist()
            suffix_lens = [a + b for a, b in zip(suffix_lens, extra)]
    suffix_lens = [int(x) for x in suffix_lens]
    assert len(suffix_lens) == B

    ps = page_size
    # logical page allocation, in tree order: shared levels, then suffixes
    level_specs = [list(lv) for lv in shared] + [[(b, b + 1, suffix_lens[b]) for b in range(B)]]
    n_logical = 0
    level_nodes = []
    for spec in level_specs:
        rows = []
        for sb, se, kl in spec:
            npg = (kl + ps - 1) // ps
            rows.append((sb, se, kl, n_logical, npg))
            n_logical += npg
        level_nodes.append(rows)
    n_pages = max(n_logical, 1)
    perm = torch.randperm(n_pages, generator=g) if shuffle else torch.arange(n_pages)

    dev = torch.device(device) if device is not None else torch.device("cpu")
    gv = g if dev.type == "cpu" else torch.Generator(device=dev).manual_seed(seed)
    q = torch.randn(B, Hq, d, generator=gv, device=dev).to(torch.bfloat16)
    k_pool = torch.randn(n_pages, Hkv, ps, d, generator=gv, device=dev).to(torch.bfloat16)
    v_pool = torch.randn(n_pages, Hkv, ps, d, generator=gv, device=dev).to(torch.bfloat16)

    levels = []
    for rows in level_nodes:
        ids = []
        nodes = []
        for sb, se, kl, first, npg in rows:
            nodes.append((sb, se, kl, len(ids)))
            ids.extend(perm[first:first + npg].tolist())
        levels.append(TreeLevel(torch.tensor(nodes, dtype=torch.int32).reshape(-1, 4),
                                torch.tensor(ids, dtype=torch.int32)))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return CascadeWorkload(name, B, Hq, Hkv, d, ps, float(scale), q, k_pool, v_pool, levels, seed)


# Named workloads.  Shapes follow the attention shapes of the models the pages
# use (Llama-3-8B, CodeLlama-13b, Llama-2-7B, CodeLlama-7B); weights are never
# needed because attention cost depends only on shapes and lengths.
CONFIG_NAMES = ("tiny", "llama3_8b", "codellama13b", "tree2", "doc_streams", "no_sharing")


def make_config(name: str, seed: int = 0, B: Optional[int] = None, prefix: Optional[int] = None,
                shuffle: bool = True, part: str = "all", device=None) -> CascadeWorkload:
    """Named workloads; ``B``/``prefix`` override the batch and the first-level
    prefix length to make smaller variants of the same structure.  ``part``:
    "all" (the workload), "prefix" (its shared levels alone: every private
    suffix empty) or "suffix" (its private suffixes alone: no shared level),
    to time or profile one pass of the step on its own.  ``device`` as in
    ``build_cascade``."""
    if part not in ("all", "prefix", "suffix"):
        raise ValueError(f"part must be all, prefix or suffix, not {part!r}")

    def mk(shared, **kw):
        if part == "suffix":
            shared = []
        if part == "prefix":
            kw.pop("suffix_range", None)
            kw.pop("extra_suffix_range", None)
            kw["suffix_lens"] = [0] * kw["B"]
        wl = build_cascade(name, shared=shared, seed=seed, shuffle=shuffle, device=device, **kw)
        wl.part = part
        return wl

    if name == "tiny":
        B_ = B or 4
        P = 256 if prefix is None else prefix
        return mk([[(0, B_, P)]] if P > 0 else [], B=B_, Hq=4, Hkv=1, d=64, page_size=16,
                  suffix_range=(0, 32), scale=1.0 / math.sqrt(64))
    if name == "llama3_8b":
        B_ = B or 64
        P = 4096 if prefix is None else prefix
        return mk([[(0, B_, P)]] if P > 0 else [], B=B_, Hq=32, Hkv=8, d=128, page_size=16,
                  suffix_range=(1, 256))
    if name == "codellama13b":
        B_ = B or 256
        P = 16384 if prefix is None else prefix
        return mk([[(0, B_, P)]] if P > 0 else [], B=B_, Hq=40, Hkv=40, d=128, page_size=16,
                  suffix_range=(1, 512))
    if name == "tree2":
        # global prefix shared by all sequences, then 8 contiguous subgroups
        # sharing a second-level prefix, then private suffixes; 64-token chunks
        B_ = B or 128
        P = 2048 if prefix is None else prefix
        groups = 8
        per = B_ // groups
        P2 = 1024 if prefix is None else max(prefix // 2, 64)
        lvl2 = [(gi * per, (gi + 1) * per, P2) for gi in range(groups)]
        return mk([[(0, B_, P)], lvl2], B=B_, Hq=32, Hkv=32, d=128, page_size=64, suffix_range=(64, 256))
    if name == "doc_streams":
        # one document shared by all streams; each stream's private segment is
        # its question (32..64 tokens) plus its answer so far (0..256 tokens)
        B_ = B or 256
        P = 16384 if prefix is None else prefix
        return mk([[(0, B_, P)]] if P > 0 else [], B=B_, Hq=32, Hkv=32, d=128, page_size=16,
                  suffix_range=(32, 64), extra_suffix_range=(0, 256))
    if name == "no_sharing":
        B_ = B or 64
        L = 2048 if prefix is None else prefix
        return mk([], B=B_, Hq=32, Hkv=32, d=128, page_size=16, suffix_lens=[L] * B_)
    raise ValueError(f"unknown config {name!r}; known: {CONFIG_NAMES}")


def full_page_tables(wl: CascadeWorkload) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-sequence page table over the whole concatenated context (shared
    pages aliased into every sequence that sees them), for per-sequence paged
    decode.  Requires every level but the last to hold whole pages.

    Returns ``(page_table [B, max_pages] int32, seq_lens [B] int32)``.
    """
    ps = wl.page_size
    per_seq: List[List[int]] = [[] for _ in range(wl.B)]
    lens = [0] * wl.B
    for li, lv in enumerate(wl.levels):
        ids = lv.page_ids.tolist()
        for sb, se, kl, off in lv.nodes.tolist():
            npg = (kl + ps - 1) // ps
            for b in range(sb, se):
                if lens[b] % ps != 0:
                    raise ValueError("a non-final level holds a partial page")
                per_seq[b].extend(ids[off:off + npg])
                lens[b] += kl
    width = max(1, max(len(p) for p in per_seq))
    pt = torch.zeros(wl.B, width, dtype=torch.int32)
    for b, p in enumerate(per_seq):
        if p:
            pt[b, :len(p)] = torch.tensor(p, dtype=torch.int32)
    return pt, torch.tensor(lens, dtype=torch.int32)


# ------------------------------------------------------------ decode loop
def with_suffix_capacity(wl: CascadeWorkload, capacity: int, seed: int = 0) -> CascadeWorkload:
    """The same workload with every private suffix's page list reserved up to
    ``capacity`` tokens, for a decode loop that appends one token per sequence
    per step.  The new pages go at the end of the pool, filled with N(0,1)
    bf16 (what a reused page would hold: never visible until written), and
    are handed out in a seeded random order.  The last level must hold one
    node per sequence, node b covering sequence b."""
    last = wl.levels[-1]
    nodes = last.nodes.tolist()
    assert len(nodes) == wl.B and all(n[0] == b and n[1] == b + 1 for b, n in enumerate(nodes))
    ps = wl.page_size
    cap_pages = (capacity + ps - 1) // ps
    assert all(n[2] <= capacity for n in nodes)
    g = torch.Generator().manual_seed(seed + 7919)
    extra = sum(cap_pages - (n[2] + ps - 1) // ps for n in nodes)
    base = wl.num_pages
    order = (base + torch.randperm(max(extra, 1), generator=g))[:extra].tolist()
    shape = (extra, wl.Hkv, ps, wl.d)
    k_pool = torch.cat([wl.k_pool.cpu(), torch.randn(shape, generator=g).to(torch.bfloat16)])
    v_pool = torch.cat([wl.v_pool.cpu(), torch.randn(shape, generator=g).to(torch.bfloat16)])
    ids_old = last.page_ids.tolist()
    ids, new_nodes, it = [], [], 0
    for sb, se, kl, off in nodes:
        npg = (kl + ps - 1) // ps
        new_nodes.append((sb, se, kl, len(ids)))
        ids.extend(ids_old[off:off + npg])
        ids.extend(order[it:it + cap_pages - npg])
        it += cap_pages - npg
    levels = [TreeLevel(l.nodes.clone(), l.page_ids.cpu().clone()) for l in wl.levels[:-1]]
    levels.append(TreeLevel(torch.tensor(new_nodes, dtype=torch.int32).reshape(-1, 4),
                            torch.tensor(ids, dtype=torch.int32)))
    return CascadeWorkload(wl.name, wl.B, wl.Hq, wl.Hkv, wl.d, ps, wl.scale, wl.q.cpu().clone(), k_pool,
                           v_pool, levels, wl.seed)


def decode_tokens(wl: CascadeWorkload, steps: int, seed: int = 0):
    """Seeded inputs of a decode loop: per step, a new query [B][Hq][d] and
    the new token's K and V rows [B][Hkv][d] (N(0,1) rounded to bf16)."""
    g = torch.Generator().manual_seed(seed + 104729)
    out = []
    for _ in range(steps):
        q = torch.randn(wl.B, wl.Hq, wl.d, generator=g).to(torch.bfloat16)
        k = torch.randn(wl.B, wl.Hkv, wl.d, generator=g).to(torch.bfloat16)
        v = torch.randn(wl.B, wl.Hkv, wl.d, generator=g).to(torch.bfloat16)
        out.append((q, k, v))
    return out


def append_token(wl: CascadeWorkload, k_new: torch.Tensor, v_new: torch.Tensor) -> None:
    """Host-side append (in place, CPU tensors): sequence b's new K / V rows
    go to slot kv_len % ps of page ``page_ids[page_off + kv_len // ps]`` of its
    suffix, and its kv_len grows by one."""
    last = wl.levels[-1]
    ps = wl.page_size
    ids = last.page_ids.tolist()
    for b, (sb, se, kl, off) in enumerate(last.nodes.tolist()):
        page = ids[off + kl // ps]
        wl.k_pool[page, :, kl % ps, :] = k_new[b].cpu()
        wl.v_pool[page, :, kl % ps, :] = v_new[b].cpu()
        last.nodes[b, 2] = kl + 1


# ------------------------------------------------- parallel prompting layout
@dataclass
class StreamRequests:
    """Requests in the Parallel Prompting layout (Read Once, Answer Many,
    Section 3): one KV row per request holding the document, then the P
    streams' questions one after another, then the answer tokens interleaved
    by step (step 1 of streams 0..P-1, then step 2, ...).  Slot ids: -1 for
    the document, s for stream s's question and answers.  Positions: the
    document's run from 0; every stream's start right after the document.

    ``rows[r]`` = (slot_sid [nk], slot_pos [nk], K [nk, Hkv, d], V [nk, Hkv, d])
    for request r; ``q`` [R*P, Hq, d] the step's queries, stream s of request
    r being sequence r*P + s (the newest answer token of each stream, at
    ``q_pos``).
    """

    R: int
    P: int
    Hq: int
    Hkv: int
    d: int
    doc_len: int
    q_lens: List[List[int]]
    T: int
    scale: float
    rows: list
    q: torch.Tensor
    q_pos: List[int]


def stream_requests(R: int, P: int, Hq: int, Hkv: int, d: int, doc_len: int, q_len_range: Tuple[int, int],
                    T: int, seed: int = 0) -> StreamRequests:
    """Seeded requests at decode step T (T >= 1 answer tokens per stream, the
    last one being the step's new token).  Question lengths are drawn from
    ``q_len_range`` (inclusive), then K, V and q as N(0,1) rounded to bf16."""
    g = torch.Generator().manual_seed(seed)
    lo, hi = q_len_range
    q_lens = [torch.randint(lo, hi + 1, (P,), generator=g).tolist() for _ in range(R)]
    rows, q_pos = [], []
    for r in range(R):
        sid = [-1] * doc_len
        pos = list(range(doc_len))
        for s in range(P):
            sid += [s] * q_lens[r][s]
            pos += [doc_len + i for i in range(q_lens[r][s])]
        for t in range(T):
            for s in range(P):
                sid.append(s)
                pos.append(doc_len + q_lens[r][s] + t)
        nk = len(sid)
        k = torch.randn(nk, Hkv, d, generator=g).to(torch.bfloat16)
        v = torch.randn(nk, Hkv, d, generator=g).to(torch.bfloat16)
        rows.append((torch.tensor(sid, dtype=torch.int32), torch.tensor(pos, dtype=torch.int32), k, v))
        q_pos += [doc_len + q_lens[r][s] + T - 1 for s in range(P)]
    q = torch.randn(R * P, Hq, d, generator=g).to(torch.bfloat16)
    return StreamRequests(R, P, Hq, Hkv, d, doc_len, q_lens, T, 1.0 / math.sqrt(d), rows, q, q_pos)


def streams_as_tree(req: StreamRequests, page_size: int = 16) -> CascadeWorkload:
    """The same requests as a prefix tree (the form the cascade path runs):
    sequence r*P + s is stream s of request r; level 0 holds each request's
    document as a node shared by its P streams, level 1 each stream's own
    slots (question, then answers, in row order) as a private node.  Every
    node starts on a fresh page; pages are laid out in node order."""
    ps = page_size
    pages_k, pages_v = [], []

    def put(k, v):
        first = len(pages_k)
        n = k.shape[0]
        for p0 in range(0, n, ps):
            pk = torch.zeros(req.Hkv, ps, req.d, dtype=torch.bfloat16)
            pv = torch.zeros(req.Hkv, ps, req.d, dtype=torch.bfloat16)
            m = min(ps, n - p0)
            pk[:, :m] = k[p0:p0 + m].transpose(0, 1)
            pv[:, :m] = v[p0:p0 + m].transpose(0, 1)
            pages_k.append(pk)
            pages_v.append(pv)
        return list(range(first, len(pages_k)))

    doc_nodes, doc_ids, own_nodes, own_ids = [], [], [], []
    for r, (sid, _, k, v) in enumerate(req.rows):
        doc = (sid == -1).nonzero().flatten()
        doc_nodes.append((r * req.P, (r + 1) * req.P, int(doc.numel()), len(doc_ids)))
        doc_ids += put(k[doc], v[doc])
        for s in range(req.P):
            own = (sid == s).nonzero().flatten()
            own_nodes.append((r * req.P + s, r * req.P + s + 1, int(own.numel()), len(own_ids)))
            own_ids += put(k[own], v[own])
    if not pages_k:
        pages_k.append(torch.zeros(req.Hkv, ps, req.d, dtype=torch.bfloat16))
        pages_v.append(torch.zeros(req.Hkv, ps, req.d, dtype=torch.bfloat16))
    levels = [TreeLevel(torch.tensor(doc_nodes, dtype=torch.int32).reshape(-1, 4),
                        torch.tensor(doc_ids, dtype=torch.int32)),
              TreeLevel(torch.tensor(own_nodes, dtype=torch.int32).reshape(-1, 4),
                        torch.tensor(own_ids, dtype=torch.int32))]
    return CascadeWorkload("parallel_prompting", req.R * req.P, req.Hq, req.Hkv, req.d, ps, req.scale,
                           req.q.clone(), torch.stack(pages_k), torch.stack(pages_v), levels, 0)


# ------------------------------------------------- reduced-precision pools
def quantize_e4m3(k_pool: torch.Tensor, v_pool: torch.Tensor) -> E4M3Pools:
    """E4M3 copies of bf16 pools ``[num_pages, Hkv, ps, d]``: per (page, KV
    head) the scale is the largest magnitude over the page's tokens and
    columns divided by 448 (1 for an all-zero slice), and each element is
    rounded to the nearest E4M3 value of element / scale (ties to even, by
    torch's float8_e4m3fn conversion).  Input preparation only: the attention
    arithmetic never runs here."""
    out = []
    for pool in (k_pool, v_pool):
        x = pool.float()
        amax = x.abs().amax(dim=(2, 3))
        sc = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
        y = (x / sc[:, :, None, None]).clamp(-E4M3_MAX, E4M3_MAX)
        out.append((y.to(torch.float8_e4m3fn).view(torch.uint8).contiguous(), sc.contiguous()))
    return E4M3Pools(out[0][0], out[1][0], out[0][1], out[1][1])


def with_e4m3_levels(wl: CascadeWorkload, levels="paged") -> CascadeWorkload:
    """The same workload with some levels read from E4M3 copies of its pools
    (``quantize_e4m3`` of every page; the levels keep their page ids).
    ``levels``: level indices, or "paged" (default) for every level whose
    nodes all run the per-sequence pass (at most 16 query rows: sequences x
    Hq/Hkv) -- the private suffixes and narrow shared nodes."""
    if levels == "paged":
        levels = [i for i, lv in enumerate(wl.levels)
                  if all((int(n[1]) - int(n[0])) * wl.G <= 16 for n in lv.nodes.tolist())]
    marks = {l % len(wl.levels) for l in levels}
    lv = [TreeLevel(l.nodes.clone(), l.page_ids.clone(), i in marks or l.e4m3) for i, l in enumerate(wl.levels)]
    return CascadeWorkload(wl.name, wl.B, wl.Hq, wl.Hkv, wl.d, wl.page_size, wl.scale, wl.q, wl.k_pool, wl.v_pool,
                           lv, wl.seed, wl.part, quantize_e4m3(wl.k_pool, wl.v_pool))


@dataclass
class StreamRows:
    """Parallel Prompting requests stored for hp_stream_decode: each
    request's KV row in pages of a shared pool, with its slots' stream ids
    and positions, and each query's stream id and position."""

    k_pool: torch.Tensor     # bf16 [num_pages, Hkv, ps, d]
    v_pool: torch.Tensor
    row_pages: torch.Tensor  # int32 [R, pt_stride]
    row_len: torch.Tensor    # int32 [R]
    slot_sid: torch.Tensor   # int32 [R, sid_stride]; -2 past the row (never visible)
    slot_pos: torch.Tensor   # int32 [R, sid_stride]
    q_sid: torch.Tensor      # int32 [R * P]
    q_pos: torch.Tensor      # int32 [R * P]
    page_size: int

    def to(self, device) -> "StreamRows":
        return StreamRows(*(t.to(device) for t in (self.k_pool, self.v_pool, self.row_pages, self.row_len,
                                                    self.slot_sid, self.slot_pos, self.q_sid, self.q_pos)),
                          self.page_size)


def stream_rows_paged(req: StreamRequests, page_size: int = 16, seed: int = 0, shuffle: bool = True) -> StreamRows:
    """The rows of ``stream_requests`` in a paged pool: row r's slot t at
    page row_pages[r, t // page_size], position t % page_size; the pages of
    all rows in one seeded random physical order.  Unused page slots hold
    N(0,1) bf16 (never visible: past the row's length)."""
    ps = page_size
    npg = [(row[0].numel() + ps - 1) // ps for row in req.rows]
    total = max(1, sum(npg))
    g = torch.Generator().manual_seed(seed + 5101)
    perm = torch.randperm(total, generator=g) if shuffle else torch.arange(total)
    k_pool = torch.randn(total, req.Hkv, ps, req.d, generator=g).to(torch.bfloat16)
    v_pool = torch.randn(total, req.Hkv, ps, req.d, generator=g).to(torch.bfloat16)
    pt_stride = max(1, max(npg))
    sid_stride = (pt_stride * ps + 3) // 4 * 4
    row_pages = torch.zeros(req.R, pt_stride, dtype=torch.int32)
    slot_sid = torch.full((req.R, sid_stride), -2, dtype=torch.int32)
    slot_pos = torch.full((req.R, sid_stride), 2 ** 30, dtype=torch.int32)
    row_len = torch.zeros(req.R, dtype=torch.int32)
    first = 0
    for r, (sid, pos, k, v) in enumerate(req.rows):
        nk = sid.numel()
        pages = perm[first:first + npg[r]]
        first += npg[r]
        row_pages[r, :npg[r]] = pages.to(torch.int32)
        for t0 in range(0, nk, ps):
            m = min(ps, nk - t0)
            p_ = int(pages[t0 // ps])
            k_pool[p_, :, :m] = k[t0:t0 + m].transpose(0, 1)
            v_pool[p_, :, :m] = v[t0:t0 + m].transpose(0, 1)
        slot_sid[r, :nk] = sid
        slot_pos[r, :nk] = pos
        row_len[r] = nk
    q_sid = torch.tensor([s for _ in range(req.R) for s in range(req.P)], dtype=torch.int32)
    q_pos = torch.tensor(req.q_pos, dtype=torch.int32)
    return StreamRows(k_pool, v_pool, row_pages, row_len, slot_sid, slot_pos, q_sid, q_pos, ps)


def _probe_code(b: int, d: int) -> torch.Tensor:
    """A bf16-exact value row unique to sequence ``b`` (and to each column)."""
    i = torch.arange(d)
    return (((b * 131 + i * 7) % 256) - 128).to(torch.float32) / 16.0


def apply_probe(wl: CascadeWorkload, targets: Sequence[int], alpha: float = 64.0,
                beta: float = 64.0) -> CascadeWorkload:
    """Turn a workload into an indexing probe (in place; returns it).

    Sequence ``b`` gets the query ``alpha * s_b * e_{j_b}`` for every head (a
    signed basis direction distinct per sequence, so one sequence's target key
    scores ~0 or very negative for every other sequence), and the key at
    logical position ``targets[b]`` of its concatenated context becomes
    ``beta * s_b * e_{j_b}`` for every KV head, with the value row set to a code
    unique to ``b``.  All other scores sit far below the target's, so the exact
    softmax output of row ``(b, h)`` is the code row itself.
    """
    d = wl.d
    if wl.B > 2 * d:
        raise ValueError("probe needs B <= 2*d distinct signed directions")
    ps = wl.page_size
    q = torch.zeros(wl.B, wl.Hq, d, dtype=torch.float32)
    locs = []
    for b in range(wl.B):
        j, sgn = b % d, (1.0 if b < d else -1.0)
        q[b, :, j] = alpha * sgn
        # walk b's levels to find the physical slot of logical token targets[b]
        t = int(targets[b])
        loc = None
        for lv in wl.levels:
            ids = lv.page_ids.tolist()
            for sb, se, kl, off in lv.nodes.tolist():
                if sb <= b < se:
                    if t < kl:
                        loc = (ids[off + t // ps], t % ps)
                    t -= kl
                    break
            if loc is not None:
                break
        if loc is None:
            raise ValueError(f"target {targets[b]} beyond sequence {b}'s context")
        locs.append((b, j, sgn, loc))
    slots = [loc for _, _, _, loc in locs]
    if len(set(slots)) != len(slots):
        raise ValueError("two probe targets share one physical slot")
    wl.q = q.to(torch.bfloat16)
    for b, j, sgn, (page, slot) in locs:
        krow = torch.zeros(d)
        krow[j] = beta * sgn
        wl.k_pool[page, :, slot, :] = krow.to(torch.bfloat16)
        wl.v_pool[page, :, slot, :] = _probe_code(b, d).to(torch.bfloat16)
    return wl


def probe_expected(b: int, d: int) -> torch.Tensor:
    return _probe_code(b, d).to(torch.bfloat16)
