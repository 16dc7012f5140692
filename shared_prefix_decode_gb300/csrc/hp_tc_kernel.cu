// hp_tc_kernel.cu -- batched attention of stacked queries against one shared
// tree node, on the tcgen05 tensor cores.
//
// Method: the queries of every sequence below a shared node are stacked into
// one matrix (Hydragen, "Inter-Sequence Batched Prefix Attention"; with GQA
// the G query heads of a KV head are further rows, shared-prefix KV caching
// blog, "Splitting attention at the prefix boundary"), so S = Q K^T and
// O = P V are matrix-matrix products and the node's KV is read once.  The key
// range of a node is split across CTAs (ChunkAttention's extra partition of
// the chunk axis, "The Chunk-First Phase Kernel in Detail"); each CTA runs an
// online softmax over its 128-key tiles (the running max / sum state of
// ChunkAttention Eq. 1-2) and writes a partial (O, LSE) per row, merged later
// by log-sum-exp.
//
// One CTA = one work item: up to 256 query rows (two M=128 blocks) x one key
// range.  Warp roles (384 threads):
//   warp 0      TMA producer: K and V tiles (128 keys x d, 128-byte swizzle)
//               through a 2-stage ring; paged pools use one box per page run.
//   warp 1      TMEM owner and MMA issuer (one thread):
//               S_mb = Q_mb K^T (A, B from shared memory) into TMEM,
//               O_mb += P_mb V   (A = P from TMEM, B = V from shared memory).
//   warps 2-3   help stage Q, then idle.
//   warps 4-7   softmax for rows 0-127, warps 8-11 for rows 128-255: read S
//               from TMEM, online max / exp2 / row sum, write P (bf16) over
//               the S columns, rescale O in TMEM when the max grows by more
//               than 2^8 (the reference max is kept otherwise; exact, since
//               the final O / l uses the same reference).
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [384,384+d).
// The two row blocks ping-pong: S of block 1 is computed while block 0 runs
// its softmax, and S of tile j+1 is issued right after P V of tile j.
#include <cuda_runtime.h>

#include "hp_internal.h"
#include "hp_ptx.cuh"

namespace hp {

namespace {

constexpr int kMaxBoxes = 1024;

template <int D>
struct TcLayout {
    static constexpr int kHalves = D / 64;
    static constexpr int kRegion = 128 * 128;  // [128 rows][64 bf16] swizzled, 16 KB
    static constexpr int kTile = kHalves * kRegion;
    static constexpr int kQ = 0;  // [mb][half] regions
    static constexpr int kK = kQ + 2 * kTile;
    static constexpr int kV = kK + 2 * kTile;
    static constexpr int kBar = kV + 2 * kTile;
    static constexpr int kPages = kBar + 256;  // staged page ids of the item's boxes
    static constexpr int kBytes = kPages + 4 * kMaxBoxes;
};

// barrier slots
enum { B_KFULL = 0, B_KEMPTY = 2, B_VFULL = 4, B_VEMPTY = 6, B_S = 8, B_P = 10, B_O = 12, B_DRAIN = 14,
       B_COUNT = 15 };

constexpr int kThreads = 384;
// Register split: warpgroup 0 (producer, MMA, two helper warps) lowers its
// count, the two softmax warpgroups raise theirs; the sum equals the launch
// allocation (384 threads x kRegsLaunch), which the host checks before the
// first launch.
constexpr uint32_t kRegsLaunch = 168, kRegsCtl = 136, kRegsSoftmax = 184;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax == kThreads * kRegsLaunch, "register split");
constexpr float kTau = 8.0f;  // lazy rescale threshold, log2 units
constexpr float kLn2 = 0.69314718055994530942f;

struct ItemGeo {
    int seq_begin, n_seq, kvh, k0, k1, part_row;
    const int32_t *pages;  // the node's page list (paged mode)
    int paged, ps, box, num_pages;
    const void *map_k;
    const void *map_v;
};

__device__ __forceinline__ ItemGeo resolve_item(const TcParams &p, int idx)
{
    ItemGeo g;
    if (p.plan != nullptr) {
        const WorkItem it = plan_array<WorkItem>(p.plan, p.plan->off_tc)[idx];
        const LevelDev &lv = p.plan->levels[it.level];
        const CUtensorMap *maps = plan_array<CUtensorMap>(p.plan, p.plan->off_maps);
        g.seq_begin = it.seq_begin;
        g.n_seq = it.n_seq;
        g.kvh = it.kvh;
        g.k0 = it.k0;
        g.k1 = it.k1;
        g.pages = plan_array<int32_t>(p.plan, p.plan->off_page_ids) + it.page_base;
        g.part_row = it.part_row;
        g.paged = 1;
        g.ps = lv.page_size;
        g.box = lv.tc_box;
        g.num_pages = lv.num_pages;
        g.map_k = maps + it.level * kMapsPerLevel + 0;
        g.map_v = maps + it.level * kMapsPerLevel + 1;
    } else {
        const int split = idx % p.imp_n_split;
        const int t = idx / p.imp_n_split;
        const int kvh = t % p.Hkv;
        const int rc = t / p.Hkv;
        g.seq_begin = p.imp_row_begin + rc * p.imp_seqs_per_item;
        g.n_seq = min(p.imp_seqs_per_item, p.imp_rows - rc * p.imp_seqs_per_item);
        g.kvh = kvh;
        g.k0 = split * p.imp_split_len;
        g.k1 = min(g.k0 + p.imp_split_len, p.imp_len);
        g.pages = nullptr;
        g.part_row = idx * p.imp_seqs_per_item * p.G;
        g.paged = 0;
        g.ps = 0;
        g.box = kTcTile;
        g.num_pages = 0;
        g.map_k = &p.map_k;
        g.map_v = &p.map_v;
    }
    return g;
}

// Issue the TMA copies of one 128-key tile (K or V) into `dst`.  Paged items
// take the page of each box from the ids staged in shared memory.
// Issue the TMA copies of one 128-key tile (K or V) into `dst`, one box per
// lane (box, column half) so that all boxes leave in one warp instruction: a
// single thread issuing small boxes one after another is limited to a
// fraction of HBM bandwidth, several lanes issuing together are not.  Paged
// items take the page of each box from the ids staged in shared memory.
template <int D>
__device__ __forceinline__ void issue_tile(const ItemGeo &g, const int32_t *s_pages, const void *map,
                                           uint32_t dst, uint32_t bar, int tile, int lane)
{
    constexpr int kHalves = D / 64;
    if (lane == 0)
        mbar_arrive_expect_tx(bar, TcLayout<D>::kTile);
    __syncwarp();
    const int kt0 = g.k0 + tile * kTcTile;
    if (g.paged) {
        const int nbox = kTcTile / g.box;
        for (int l = lane; l < nbox * kHalves; l += 32) {
            const int bx = l / kHalves, h = l - bx * kHalves;
            const int t = kt0 + bx * g.box;
            tma_load_4d(dst + h * TcLayout<D>::kRegion + bx * g.box * 128, map, bar, h * 64, t % g.ps, g.kvh,
                        s_pages[tile * nbox + bx]);
        }
    } else if (lane < kHalves) {
        tma_load_3d(dst + lane * TcLayout<D>::kRegion, map, bar, lane * 64, g.kvh, kt0);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) hp_tc_kernel(const __grid_constant__ TcParams p)
{
    using L = TcLayout<D>;
    constexpr int kHalves = D / 64;
    constexpr uint32_t kIdescQK = umma_idesc_bf16(128, 128, false);
    constexpr uint32_t kIdescPV = umma_idesc_bf16(128, D, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kBar;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kBar + 128);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L::kBar + 132);
    int32_t *s_pages = reinterpret_cast<int32_t *>(smem + L::kPages);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (p.plan != nullptr && (p.plan->magic != kPlanMagic || p.plan->tag != p.tag)) {
        if (threadIdx.x == 0)
            atomicOr(p.status, kStPlan);
        return;  // uniform across the CTA: nothing allocated yet
    }
    const ItemGeo g = resolve_item(p, blockIdx.x);
    const int rows_total = g.n_seq * p.G;
    const int nmb = (rows_total + 127) >> 7;
    const int n_tiles = (g.k1 - g.k0 + kTcTile - 1) / kTcTile;
    const int n_boxes = g.paged ? n_tiles * (kTcTile / g.box) : 0;
    if (nmb > 2 || n_tiles <= 0 || n_boxes > kMaxBoxes) {
        if (threadIdx.x == 0)
            atomicOr(p.status, kStPlan);
        return;  // uniform across the CTA: nothing allocated yet
    }
    const int pre = n_tiles < 2 ? n_tiles : 2;  // tiles issued before the CTA barrier

    // warp-uniform bounded wait
    auto wait_warp = [&](int b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar(b), parity, p.status, abort)) != 0;
    };

    if (warp == 0) {
        // Barriers, then the page id of every box of the item (ids out of
        // range become the zero-filled page num_pages and set the bounds
        // flag), then the first tiles' copies -- these overlap Q staging.
        if (lane == 0) {
            for (int i = 0; i < B_COUNT; ++i)
                mbar_init(bar(i), (i == B_P || i == B_P + 1) ? 128u : 1u);
            *abort = 0;
            fence_mbar_init();
            prefetch_tensormap(g.map_k);
            prefetch_tensormap(g.map_v);
        }
        if (g.paged) {
            const int nbox = kTcTile / g.box;
            for (int i = lane; i < n_boxes; i += 32) {
                const int t = g.k0 + (i / nbox) * kTcTile + (i % nbox) * g.box;
                int page = g.num_pages;
                if (t < g.k1) {
                    page = __ldg(g.pages + t / g.ps);
                    if ((unsigned)page >= (unsigned)g.num_pages) {
                        atomicOr(p.status, kStBounds);
                        page = g.num_pages;
                    }
                }
                s_pages[i] = page;
            }
        }
        __syncwarp();
        for (int j = 0; j < pre; ++j) {
            issue_tile<D>(g, s_pages, g.map_k, sbase + L::kK + j * L::kTile, bar(B_KFULL + j), j, lane);
            issue_tile<D>(g, s_pages, g.map_v, sbase + L::kV + j * L::kTile, bar(B_VFULL + j), j, lane);
        }
    } else {
        if (warp == 1) {
            tmem_alloc(smem_u32(tmem_slot), 512);
            tmem_relinquish();
        }
        // Stage Q (rows r = s*G + g of the item; rows past the item are zero)
        // in the 128-byte-swizzled K-major layout the MMA descriptors
        // describe.  Warps 1-11; all loads of a thread before its stores.
        constexpr int kQThreads = kThreads - 32;
        constexpr int kCpr = D / 8;  // 16-byte chunks per row
        constexpr int kPer = (2 * 128 * kCpr + kQThreads - 1) / kQThreads;
        const int qt = tid - 32;
        const int total = nmb * 128 * kCpr;
        uint4 buf[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = qt + k * kQThreads;
            const int r = i / kCpr;
            buf[k] = make_uint4(0u, 0u, 0u, 0u);
            if (i < total && r < rows_total) {
                const int c = i % kCpr;
                const int s = r / p.G;
                const int gg = r - s * p.G;
                const uint16_t *src =
                    p.q + (int64_t)(g.seq_begin + s) * p.q_sb + (int64_t)(g.kvh * p.G + gg) * p.q_sh + c * 8;
                buf[k] = __ldg(reinterpret_cast<const uint4 *>(src));
            }
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = qt + k * kQThreads;
            if (i < total) {
                const int r = i / kCpr, c = i % kCpr;
                const int mb = r >> 7, rr = r & 127, h = c >> 3, cc = c & 7;
                uint8_t *dst = smem + L::kQ + ((mb * kHalves + h) * 128 + rr) * 128 + ((cc ^ (rr & 7)) << 4);
                *reinterpret_cast<uint4 *>(dst) = buf[k];
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Registers: the softmax warpgroups hold a whole 128-column score row
    if (warp < 4)
        setmaxnreg_dec<kRegsCtl>();
    else
        setmaxnreg_inc<kRegsSoftmax>();

    if (warp == 0) {
        // ------------------------------------------------------ producer
        int issued = pre;
        for (int j = pre; j < n_tiles; ++j) {
            const int st = j & 1;
            const uint32_t ph = (uint32_t)(j >> 1) & 1u;
            if (!wait_warp(B_KEMPTY + st, ph ^ 1u))
                break;
            issue_tile<D>(g, s_pages, g.map_k, sbase + L::kK + st * L::kTile, bar(B_KFULL + st), j, lane);
            if (!wait_warp(B_VEMPTY + st, ph ^ 1u)) {
                if (lane == 0)
                    mbar_wait_drain(bar(B_KFULL + st), ph);  // K of tile j is in flight
                break;
            }
            issue_tile<D>(g, s_pages, g.map_v, sbase + L::kV + st * L::kTile, bar(B_VFULL + st), j, lane);
            issued = j + 1;
        }
        // drain: every load issued has landed before the CTA exits
        if (lane == 0) {
            for (int j = max(0, issued - 2); j < issued; ++j) {
                const uint32_t ph = (uint32_t)(j >> 1) & 1u;
                mbar_wait_drain(bar(B_KFULL + (j & 1)), ph);
                mbar_wait_drain(bar(B_VFULL + (j & 1)), ph);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t qa = sbase + L::kQ;
            auto issue_s = [&](int mb, int st) {
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int h = ks >> 2, kin = ks & 3;
                    const uint64_t a =
                        umma_desc_sw128(qa + (mb * kHalves + h) * L::kRegion + kin * 32, 16, 1024);
                    const uint64_t b =
                        umma_desc_sw128(sbase + L::kK + st * L::kTile + h * L::kRegion + kin * 32, 16, 1024);
                    tc_mma_ss(tmem + mb * 128, a, b, kIdescQK, ks > 0 ? 1u : 0u);
                }
                tc_commit(bar(B_S + mb));
            };
            auto issue_pv = [&](int mb, int st, int j) {
                for (int ks = 0; ks < kTcTile / 16; ++ks) {
                    const uint64_t b =
                        umma_desc_sw128(sbase + L::kV + st * L::kTile + ks * 2048, L::kRegion, 1024);
                    tc_mma_ts(tmem + 256 + mb * 128, tmem + mb * 128 + ks * 8, b, kIdescPV,
                              (j > 0 || ks > 0) ? 1u : 0u);
                }
                tc_commit(bar(B_O + mb));
            };
            bool ok = mbar_wait(bar(B_KFULL + 0), 0u, p.status, abort);
            if (ok) {
                tc_fence_after();
                for (int mb = 0; mb < nmb; ++mb)
                    issue_s(mb, 0);
                tc_commit(bar(B_KEMPTY + 0));
            }
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int st = j & 1;
                const uint32_t ph = (uint32_t)(j >> 1) & 1u;
                if (!(ok = mbar_wait(bar(B_VFULL + st), ph, p.status, abort)))
                    break;
                const bool more = j + 1 < n_tiles;
                const int st1 = (j + 1) & 1;
                for (int mb = 0; mb < nmb; ++mb) {
                    if (!(ok = mbar_wait(bar(B_P + mb), (uint32_t)j & 1u, p.status, abort)))
                        break;
                    tc_fence_after();
                    issue_pv(mb, st, j);
                    if (more) {
                        if (mb == 0) {
                            if (!(ok = mbar_wait(bar(B_KFULL + st1), (uint32_t)((j + 1) >> 1) & 1u,
                                                 p.status, abort)))
                                break;
                            tc_fence_after();
                        }
                        issue_s(mb, st1);
                    }
                }
                if (!ok)
                    break;
                tc_commit(bar(B_VEMPTY + st));
                if (more)
                    tc_commit(bar(B_KEMPTY + st1));
            }
            // every MMA issued has completed before TMEM is released
            tc_commit(bar(B_DRAIN));
            mbar_wait_drain(bar(B_DRAIN), 0u);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------ softmax
        const int mb = (warp - 4) >> 2;
        const int rr = tid - 128 * (1 + mb);  // row within the block == TMEM lane
        const int row = mb * 128 + rr;
        const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_col = tl + mb * 128;
        const uint32_t o_col = tl + 256 + mb * 128;
        const float c = p.scale_log2;  // > 0 (checked on the host)
        float m_run = -INFINITY;       // reference max, log2 units
        float l_run = 0.f;
        bool ok = mb < nmb;
        uint32_t sv[128];
        uint32_t r[32];
        for (int j = 0; ok && j < n_tiles; ++j) {
            if (!(ok = wait_warp(B_S + mb, (uint32_t)j & 1u)))
                break;
            tc_fence_after();
            const int nvalid = min(kTcTile, g.k1 - (g.k0 + j * kTcTile));
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                tmem_ld32(s_col + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[cc * 32]));
            tmem_ld_wait();
            // the scale is positive, so the largest scaled score is the
            // largest raw score times the scale
            float mx = -INFINITY;
            if (nvalid >= kTcTile) {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    mx = fmaxf(mx, __uint_as_float(sv[i]));
            } else {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i < nvalid)
                        mx = fmaxf(mx, __uint_as_float(sv[i]));
            }
            const float tmax = mx * c;
            const bool need = tmax > m_run + kTau;
            const float alpha = need ? fast_exp2(m_run - tmax) : 1.f;
            if (need) {
                l_run *= alpha;
                m_run = tmax;
            }
            // P = exp2(s * c - m) as bf16 pairs over the S columns (the score
            // row is dead afterwards, which keeps the rescale below cheap in
            // registers)
            const float nm = -m_run;
            float lsum = 0.f;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c0 = cc * 32 + 2 * i;
                    float p0 = fast_exp2(fmaf(__uint_as_float(sv[c0]), c, nm));
                    float p1 = fast_exp2(fmaf(__uint_as_float(sv[c0 + 1]), c, nm));
                    if (nvalid < kTcTile) {
                        p0 = c0 < nvalid ? p0 : 0.f;
                        p1 = c0 + 1 < nvalid ? p1 : 0.f;
                    }
                    lsum += p0 + p1;
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st16(s_col + cc * 16, pk);
            }
            l_run += lsum;
            // O was accumulated against the old reference max: rescale it
            // once the previous P V has landed (rare: only when the max grows
            // by more than 2^kTau)
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                if (!(ok = wait_warp(B_O + mb, (uint32_t)(j - 1) & 1u)))
                    break;
                tc_fence_after();
#pragma unroll
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
                // last, partial tile: rows past the node hold whatever the
                // pool holds there; zero their V so 0 * garbage stays 0
                const int st = j & 1;
                if (!(ok = wait_warp(B_VFULL + st, (uint32_t)(j >> 1) & 1u)))
                    break;
                if (rr >= nvalid) {
                    for (int h = 0; h < kHalves; ++h) {
                        uint4 *vrow =
                            reinterpret_cast<uint4 *>(smem + L::kV + st * L::kTile + h * L::kRegion + rr * 128);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            vrow[q] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(bar(B_P + mb));
        }
        if (ok && mb < nmb) {
            if (wait_warp(B_O + mb, (uint32_t)(n_tiles - 1) & 1u)) {
                tc_fence_after();
                const float inv = 1.f / l_run;
                const float lse = (m_run + fast_log2(l_run)) * kLn2;
                float *dst = p.part_o + (size_t)(g.part_row + row) * D;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    tmem_ld32(o_col + cc * 32, r);
                    tmem_ld_wait();
                    if (row < rows_total) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            float4 v = make_float4(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv,
                                                   __uint_as_float(r[i + 2]) * inv,
                                                   __uint_as_float(r[i + 3]) * inv);
                            *reinterpret_cast<float4 *>(dst + cc * 32 + i) = v;
                        }
                    }
                }
                if (row < rows_total)
                    p.part_lse[g.part_row + row] = lse;
            }
        }
        tc_fence_before();
    }

    // Lanes 1-31 of warps 0 and 1 reach this point while their lane 0 still
    // runs the producer / MMA loop: converge each warp before the CTA barrier
    // (an aligned barrier must be reached by whole warps), so TMEM is freed
    // only after every role has finished.
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t launch_tc_d(const TcParams &p, int grid, cudaStream_t s)
{
    static bool configured = false;
    const int bytes = TcLayout<D>::kBytes + 1024;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(hp_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess)
            return e;
        // the register split assumes this launch allocation per thread
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, hp_tc_kernel<D>)) != cudaSuccess)
            return e;
        if (fa.numRegs != (int)kRegsLaunch)
            return cudaErrorInvalidConfiguration;
        configured = true;
    }
    hp_tc_kernel<D><<<grid, kThreads, bytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t tc_smem_bytes(int d)
{
    return d == 64 ? TcLayout<64>::kBytes + 1024 : TcLayout<128>::kBytes + 1024;
}

cudaError_t launch_tc(const TcParams &p, int grid, int d, cudaStream_t s)
{
    if (grid <= 0)
        return cudaSuccess;
    return d == 64 ? launch_tc_d<64>(p, grid, s) : launch_tc_d<128>(p, grid, s);
}

}  // namespace hp
