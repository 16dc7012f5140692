// hp_tc_role.cuh -- the tensor-core role: batched attention of stacked
// queries against one shared tree node, for one work item, by a 384-thread
// CTA.  Shared by the standalone prefix kernel and the fused cascade kernel.
//
// Method: the queries of every sequence below a shared node are stacked into
// one matrix (Hydragen, "Inter-Sequence Batched Prefix Attention"; with GQA
// the G query heads of a KV head are further rows, shared-prefix KV caching
// blog, "Splitting attention at the prefix boundary"), so S = Q K^T and
// O = P V are matrix-matrix products and the node's KV is read once.  The key
// range of a node is split across items (ChunkAttention's extra partition of
// the chunk axis, "The Chunk-First Phase Kernel in Detail"); an item runs an
// online softmax over its 128-key tiles (the running max / sum state of
// ChunkAttention Eq. 1-2) and writes a partial (O, LSE) per row, merged later
// by log-sum-exp.
//
// One item: up to two blocks of 128 query rows x one key range.  A block
// holds 128 / G sequences x G heads (rows s*G + g), loaded by one TMA box per
// 64 columns straight from q[b][h][:], so the rows of a block need no
// staging by threads.  Roles:
//   warp 0      TMA producer: Q, then K and V tiles (128 keys x d, 128-byte
//               swizzle) through a 2-stage ring, all boxes of a tile issued
//               by several lanes at once (a TMA box costs about the same
//               whatever its size; one thread issuing boxes one by one caps
//               an SM far below HBM bandwidth).
//   warp 1      TMEM owner and MMA issuer (one thread):
//               S_mb = Q_mb K^T (A, B from shared memory) into TMEM,
//               O_mb += P_mb V   (A = P from TMEM, B = V from shared memory).
//   warps 4-7   softmax for block 0, warps 8-11 for block 1: read a 128-column
//               score row from TMEM, max / exp2 / row sum, write P (bf16)
//               over the S columns, rescale O in TMEM when the max grows by
//               more than 2^8 (the reference max is kept otherwise; exact,
//               since the final O / l uses the same reference), and at the end
//               stage O / l (bf16) in shared memory as 128-row x 64-column boxes
//               that one thread writes out with TMA tensor stores (the
//               partial rows of a block are 128 reserved rows of the
//               workspace).  The loops walk the row in 32-column chunks
//               (short code: a cold instruction cache costs microseconds
//               when HBM is saturated).
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [384,384+d).
// The two row blocks ping-pong: S of block 1 is computed while block 0 runs
// its softmax, and S of tile j+1 is issued right after P V of tile j.
//
// Register split: warpgroup 0 (producer, MMA, two idle warps) lowers its
// count, the softmax warpgroups raise theirs; the caller issues setmaxnreg at
// the top of each branch.
#pragma once

#include <cuda_runtime.h>

#include "hp_internal.h"
#include "hp_ptx.cuh"

namespace hp {
namespace tcr {

constexpr int kThreads = 384;
constexpr uint32_t kRegsLaunch = 168, kRegsCtl = 136, kRegsSoftmax = 184;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax == kThreads * kRegsLaunch, "register split");
constexpr float kTau = 8.0f;  // lazy rescale threshold, log2 units
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct Layout {
    static constexpr int kHalves = D / 64;
    static constexpr int kRegion = 128 * 128;  // [128 rows][64 bf16] swizzled, 16 KB
    static constexpr int kTile = kHalves * kRegion;
    static constexpr int kQ = 0;  // [mb][half] regions
    static constexpr int kK = kQ + 2 * kTile;
    static constexpr int kV = kK + 2 * kTile;
    static constexpr int kEnd = kV + 2 * kTile;  // O staging reuses K (block 0) and V (block 1)
    static constexpr int kOBox = 128 * 128;      // [128 rows][64 bf16], 128-byte swizzle
    static_assert(2 * kTile >= (D / 64) * kOBox, "O staging must fit one ring");
};

// barrier slots (8 bytes each) at the caller's barrier area
enum { B_KFULL = 0, B_KEMPTY = 2, B_VFULL = 4, B_VEMPTY = 6, B_S = 8, B_P = 10, B_O = 12, B_DRAIN = 14,
       B_Q = 15, B_COUNT = 16 };
// Byte offsets in the caller's 256-byte barrier area.
constexpr int kBarTmemSlot = 192, kBarAbort = 196;
static_assert(B_COUNT * 8 <= kBarTmemSlot, "barrier area");

struct ItemGeo {
    int seq_begin, n_seq, kvh, k0, k1, part_row;
    int spb;               // sequences per 128-row block: 128 / G
    int paged, ps, box, num_pages;
    const int32_t *pages;  // paged: page of key t is pages[t / ps - k0 / ps] (generic address)
    const void *map_k;
    const void *map_v;
    const void *map_q;
};

// Per-CTA resources of the role.
struct Ctx {
    uint8_t *smem;        // 1024-aligned base of the role's layout
    uint32_t sbase;       // its shared-window address
    uint32_t bar0;        // B_COUNT barriers
    uint32_t *tmem_slot;  // TMEM base address written by tcgen05.alloc
    volatile int *abort;
    uint32_t *status;
};

struct Args {
    int G;
    float scale_log2;  // > 0
    const void *map_o;  // partial O rows [rows][D] bf16: box 64 columns x 128 rows, 128-byte swizzle
    float *part_lse;
};

__device__ __forceinline__ uint32_t bar_at(const Ctx &c, int i) { return c.bar0 + 8u * (uint32_t)i; }

__device__ __forceinline__ void named_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void mbar_inval(uint32_t bar)
{
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ int n_tiles_of(const ItemGeo &g) { return (g.k1 - g.k0 + kTcTile - 1) / kTcTile; }
__device__ __forceinline__ int n_blocks_of(const ItemGeo &g) { return (g.n_seq + g.spb - 1) / g.spb; }

__device__ __forceinline__ bool item_ok(const ItemGeo &g)
{
    const int nmb = n_blocks_of(g);
    return g.spb >= 1 && nmb >= 1 && nmb <= 2 && g.k1 > g.k0 &&
           (!g.paged || (g.box >= 1 && kTcTile % g.box == 0 && g.ps % g.box == 0));
}

// One thread: (re)initialise the role's barriers.  `reinit` when an earlier
// item used them (the CTA has synchronised since).
__device__ __forceinline__ void init_barriers(const Ctx &c, bool reinit)
{
    for (int i = 0; i < B_COUNT; ++i) {
        if (reinit)
            mbar_inval(bar_at(c, i));
        mbar_init(bar_at(c, i), (i == B_P || i == B_P + 1) ? 128u : 1u);
    }
    *c.abort = 0;
    fence_mbar_init();
}

// Issue the TMA copies of one 128-key tile (K or V) into `dst`, one box per
// lane (box, column half).  Boxes past the item's keys read page num_pages,
// which the map zero-fills.
template <int D>
__device__ __forceinline__ void issue_tile(const Ctx &c, const ItemGeo &g, const void *map, uint32_t dst,
                                           uint32_t bar, int tile, int lane)
{
    constexpr int kHalves = D / 64;
    if (lane == 0)
        mbar_arrive_expect_tx(bar, Layout<D>::kTile);
    __syncwarp();
    const int kt0 = g.k0 + tile * kTcTile;
    if (g.paged) {
        const int nbox = kTcTile / g.box;
        const int pbase = g.k0 / g.ps;
        for (int l = lane; l < nbox * kHalves; l += 32) {
            const int bx = l / kHalves, h = l - bx * kHalves;
            const int t = kt0 + bx * g.box;
            int page = g.num_pages;
            if (t < g.k1) {
                page = g.pages[t / g.ps - pbase];
                if ((unsigned)page >= (unsigned)g.num_pages) {
                    atomicOr(c.status, kStBounds);
                    page = g.num_pages;
                }
            }
            tma_load_4d_h(dst + h * Layout<D>::kRegion + bx * g.box * 128, map, bar, h * 64, t % g.ps, g.kvh, page,
                          l2_evict_first());
        }
    } else if (lane < kHalves) {
        tma_load_3d_h(dst + lane * Layout<D>::kRegion, map, bar, lane * 64, g.kvh, kt0, l2_evict_first());
    }
}

// ---------------------------------------------------------------- phase A
// Warp 0: the item's Q blocks and its first two tiles.  `withhold` (failure
// detection tests only): arm the first K tile's barrier for its bytes but
// issue no copy, so the waits on it run out their time limit.
template <int D>
__device__ __forceinline__ void producer_prologue(const Ctx &c, const ItemGeo &g, const Args &a, int lane,
                                                  bool withhold = false)
{
    using L = Layout<D>;
    constexpr int kHalves = D / 64;
    const int nmb = n_blocks_of(g);
    if (lane == 0)
        mbar_arrive_expect_tx(bar_at(c, B_Q), (uint32_t)(nmb * kHalves * g.spb * a.G * 128));
    __syncwarp();
    if (lane < nmb * kHalves) {
        const int mb = lane / kHalves, h = lane % kHalves;
        tma_load_3d(c.sbase + L::kQ + (mb * kHalves + h) * L::kRegion, g.map_q, bar_at(c, B_Q), h * 64,
                    g.kvh * a.G, g.seq_begin + mb * g.spb);
    }
    const int n_tiles = n_tiles_of(g);
    const int pre = n_tiles < 2 ? n_tiles : 2;
    for (int j = 0; j < pre; ++j) {
        if (withhold && j == 0) {
            if (lane == 0)
                mbar_arrive_expect_tx(bar_at(c, B_KFULL + 0), L::kTile);
            __syncwarp();
        } else {
            issue_tile<D>(c, g, g.map_k, c.sbase + L::kK + j * L::kTile, bar_at(c, B_KFULL + j), j, lane);
        }
        issue_tile<D>(c, g, g.map_v, c.sbase + L::kV + j * L::kTile, bar_at(c, B_VFULL + j), j, lane);
    }
}

// ---------------------------------------------------------------- phase B
template <int D>
__device__ __forceinline__ void producer_loop(const Ctx &c, const ItemGeo &g, int lane)
{
    using L = Layout<D>;
    const int n_tiles = n_tiles_of(g);
    const int pre = n_tiles < 2 ? n_tiles : 2;
    auto wait_warp = [&](int b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar_at(c, b), parity, c.status, c.abort)) != 0;
    };
    int issued = pre;
    for (int j = pre; j < n_tiles; ++j) {
        const int st = j & 1;
        const uint32_t ph = (uint32_t)(j >> 1) & 1u;
        if (!wait_warp(B_KEMPTY + st, ph ^ 1u))
            break;
        issue_tile<D>(c, g, g.map_k, c.sbase + L::kK + st * L::kTile, bar_at(c, B_KFULL + st), j, lane);
        if (!wait_warp(B_VEMPTY + st, ph ^ 1u)) {
            if (lane == 0)
                mbar_wait_drain(bar_at(c, B_KFULL + st), ph);  // K of tile j is in flight
            break;
        }
        issue_tile<D>(c, g, g.map_v, c.sbase + L::kV + st * L::kTile, bar_at(c, B_VFULL + st), j, lane);
        issued = j + 1;
    }
    // every load issued has landed before the item ends
    if (lane == 0) {
        mbar_wait_drain(bar_at(c, B_Q), 0u);
        for (int j = max(0, issued - 2); j < issued; ++j) {
            const uint32_t ph = (uint32_t)(j >> 1) & 1u;
            mbar_wait_drain(bar_at(c, B_KFULL + (j & 1)), ph);
            mbar_wait_drain(bar_at(c, B_VFULL + (j & 1)), ph);
        }
    }
}

// One thread (warp 1, lane 0).
template <int D>
__device__ __forceinline__ void mma_loop(const Ctx &c, const ItemGeo &g, uint32_t tmem)
{
    using L = Layout<D>;
    constexpr int kHalves = D / 64;
    constexpr uint32_t kIdescQK = umma_idesc_bf16(128, 128, false);
    constexpr uint32_t kIdescPV = umma_idesc_bf16(128, D, true);
    const int nmb = n_blocks_of(g);
    const int n_tiles = n_tiles_of(g);
    const uint32_t qa = c.sbase + L::kQ;
    auto issue_s = [&](int mb, int st) {
        for (int ks = 0; ks < D / 16; ++ks) {
            const int h = ks >> 2, kin = ks & 3;
            const uint64_t a = umma_desc_sw128(qa + (mb * kHalves + h) * L::kRegion + kin * 32, 16, 1024);
            const uint64_t b =
                umma_desc_sw128(c.sbase + L::kK + st * L::kTile + h * L::kRegion + kin * 32, 16, 1024);
            tc_mma_ss(tmem + mb * 128, a, b, kIdescQK, ks > 0 ? 1u : 0u);
        }
        tc_commit(bar_at(c, B_S + mb));
    };
    auto issue_pv = [&](int mb, int st, int j) {
        for (int ks = 0; ks < kTcTile / 16; ++ks) {
            const uint64_t b = umma_desc_sw128(c.sbase + L::kV + st * L::kTile + ks * 2048, L::kRegion, 1024);
            tc_mma_ts(tmem + 256 + mb * 128, tmem + mb * 128 + ks * 8, b, kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(bar_at(c, B_O + mb));
    };
    bool ok = mbar_wait(bar_at(c, B_Q), 0u, c.status, c.abort) &&
              mbar_wait(bar_at(c, B_KFULL + 0), 0u, c.status, c.abort);
    if (ok) {
        tc_fence_after();
        for (int mb = 0; mb < nmb; ++mb)
            issue_s(mb, 0);
        tc_commit(bar_at(c, B_KEMPTY + 0));
    }
    for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j & 1;
        const uint32_t ph = (uint32_t)(j >> 1) & 1u;
        if (!(ok = mbar_wait(bar_at(c, B_VFULL + st), ph, c.status, c.abort)))
            break;
        const bool more = j + 1 < n_tiles;
        const int st1 = (j + 1) & 1;
        for (int mb = 0; mb < nmb; ++mb) {
            if (!(ok = mbar_wait(bar_at(c, B_P + mb), (uint32_t)j & 1u, c.status, c.abort)))
                break;
            tc_fence_after();
            issue_pv(mb, st, j);
            if (more) {
                if (mb == 0) {
                    if (!(ok = mbar_wait(bar_at(c, B_KFULL + st1), (uint32_t)((j + 1) >> 1) & 1u, c.status,
                                         c.abort)))
                        break;
                    tc_fence_after();
                }
                issue_s(mb, st1);
            }
        }
        if (!ok)
            break;
        tc_commit(bar_at(c, B_VEMPTY + st));
        if (more)
            tc_commit(bar_at(c, B_KEMPTY + st1));
    }
    // every MMA issued has completed before the item ends
    tc_commit(bar_at(c, B_DRAIN));
    mbar_wait_drain(bar_at(c, B_DRAIN), 0u);
}

// Warps 4-11 (mb = 0 for warps 4-7, 1 for 8-11).  Each thread owns one row
// of its block (its TMEM lane).
template <int D>
__device__ __forceinline__ void softmax_loop(const Ctx &c, const ItemGeo &g, const Args &a, uint32_t tmem,
                                             int warp, int lane, int tid)
{
    using L = Layout<D>;
    constexpr int kHalves = D / 64;
    const int rows_total = g.n_seq * a.G;
    const int rpb = g.spb * a.G;  // rows per block
    const int nmb = n_blocks_of(g);
    const int n_tiles = n_tiles_of(g);
    const int mb = (warp - 4) >> 2;
    const int rr = tid - 128 * (1 + mb);  // row within the block == TMEM lane
    const int rows_here = min(rpb, rows_total - mb * rpb);
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = tl + mb * 128;
    const uint32_t o_col = tl + 256 + mb * 128;
    const float cs = a.scale_log2;
    const uint64_t cs2 = f32x2_pack(cs, cs);
    auto wait_warp = [&](int b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar_at(c, b), parity, c.status, c.abort)) != 0;
    };
    float m_run = -INFINITY;  // reference max, log2 units
    float l_run = 0.f;
    bool ok = mb < nmb;
    uint32_t r[32];
    for (int j = 0; ok && j < n_tiles; ++j) {
        if (!(ok = wait_warp(B_S + mb, (uint32_t)j & 1u)))
            break;
        tc_fence_after();
        const int nvalid = min(kTcTile, g.k1 - (g.k0 + j * kTcTile));
        // largest valid score (the scale is positive: the largest scaled
        // score is the largest raw score times the scale)
        float mx = -INFINITY;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
            tmem_ld32(s_col + cc * 32, r);
            tmem_ld_wait();
            const int lim = nvalid - cc * 32;
            if (lim >= 32) {
#pragma unroll
                for (int i = 0; i < 32; i += 2)
                    mx = fmax3(mx, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    mx = fmaxf(mx, i < lim ? __uint_as_float(r[i]) : -INFINITY);
            }
        }
        const float tmax = mx * cs;
        const bool need = tmax > m_run + kTau;
        const float alpha = need ? fast_exp2(m_run - tmax) : 1.f;
        if (need) {
            l_run *= alpha;
            m_run = tmax;
        }
        // P = exp2(s * c - m) as bf16 pairs over the S columns (chunk cc's P
        // lands in columns already read); invalid keys get P = 0.  Pairs of
        // scores go through the packed f32x2 fma / add.
        const float nm = -m_run;
        const uint64_t nm2 = f32x2_pack(nm, nm);
        uint64_t acc2 = f32x2_pack(0.f, 0.f);
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
            tmem_ld32(s_col + cc * 32, r);
            tmem_ld_wait();
            const int lim = nvalid - cc * 32;
            uint32_t pk[16];
            if (lim >= 32) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                                           cs2, nm2),
                                 x0, x1);
                    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                    acc2 = f32x2_add(acc2, f32x2_pack(p0, p1));
                    pk[i] = pack_bf16x2(p0, p1);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float p0 = fast_exp2(fmaf(__uint_as_float(r[2 * i]), cs, nm));
                    float p1 = fast_exp2(fmaf(__uint_as_float(r[2 * i + 1]), cs, nm));
                    p0 = 2 * i < lim ? p0 : 0.f;
                    p1 = 2 * i + 1 < lim ? p1 : 0.f;
                    acc2 = f32x2_add(acc2, f32x2_pack(p0, p1));
                    pk[i] = pack_bf16x2(p0, p1);
                }
            }
            tmem_st16(s_col + cc * 16, pk);
        }
        float lsum0, lsum1;
        f32x2_unpack(acc2, lsum0, lsum1);
        const float lsum = lsum0 + lsum1;
        l_run += lsum;
        // O was accumulated against the old reference max: rescale it once
        // the previous P V has landed (rare: the max grew by more than 2^kTau)
        if (j > 0 && __any_sync(0xffffffffu, need)) {
            if (!(ok = wait_warp(B_O + mb, (uint32_t)(j - 1) & 1u)))
                break;
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                tmem_ld32(o_col + cc * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                tmem_st32(o_col + cc * 32, r);
            }
        }
        tmem_st_wait();
        if (mb == 0 && nvalid < kTcTile) {
            // last, partial tile: rows past the node hold whatever the pool
            // holds there; zero their V so 0 * garbage stays 0
            const int st = j & 1;
            if (!(ok = wait_warp(B_VFULL + st, (uint32_t)(j >> 1) & 1u)))
                break;
            if (rr >= nvalid) {
                for (int h = 0; h < kHalves; ++h) {
                    uint4 *vrow = reinterpret_cast<uint4 *>(c.smem + L::kV + st * L::kTile + h * L::kRegion + rr * 128);
#pragma unroll
                    for (int qd = 0; qd < 8; ++qd)
                        vrow[qd] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(bar_at(c, B_P + mb));
    }
    // Epilogue: O / l into shared memory (block 0 over the K ring, block 1
    // over the V ring, both idle once the last P V has completed) as D/64
    // bf16 boxes of [128 rows][64 columns] in the 128-byte swizzled order the
    // tensor map expects (conflict-free: 8 consecutive rows hit 8 distinct
    // 16-byte slots), then one thread of the block stores the boxes to
    // partial rows part_row + mb*128 .. +127 and waits until they have been
    // read.
    const bool have = ok && mb < nmb;
    uint8_t *stg = c.smem + (mb == 0 ? L::kK : L::kV);
    if (have && wait_warp(B_O + mb, (uint32_t)(n_tiles - 1) & 1u)) {
        tc_fence_after();
        const float inv = 1.f / l_run;
        uint32_t r2[32];
#pragma unroll 1
        for (int bx = 0; bx < D / 64; ++bx) {
            tmem_ld32(o_col + bx * 64, r);
            tmem_ld32(o_col + bx * 64 + 32, r2);
            tmem_ld_wait();
            uint8_t *row = stg + bx * L::kOBox + rr * 128;
#pragma unroll
            for (int i = 0; i < 8; ++i) {  // 16-byte piece i: columns bx*64 + 8i .. +7
                const uint32_t *src = i < 4 ? &r[8 * i] : &r2[8 * (i - 4)];
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv);
                v.y = pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv);
                v.z = pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv);
                v.w = pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv);
                *reinterpret_cast<uint4 *>(row + ((i ^ (rr & 7)) << 4)) = v;
            }
        }
        if (rr < rows_here)
            a.part_lse[g.part_row + mb * 128 + rr] = (m_run + fast_log2(l_run)) * kLn2;
        fence_proxy_async_smem();
    }
    tc_fence_before();
    named_sync(1 + mb, 128);
    if (have && rr == 0) {
        for (int bx = 0; bx < D / 64; ++bx)
            tma_store_2d(a.map_o, smem_u32(stg + bx * L::kOBox), bx * 64, g.part_row + mb * 128);
        bulk_commit_group();
        bulk_wait_read_all();
    }
}

}  // namespace tcr
}  // namespace hp
