// hp_small_kernel.cu -- paged decode of up to 16 query rows per KV head
// against one key range (a private suffix, or a node shared by very few
// sequences).
//
// Method: the sequence-first phase of ChunkAttention ("The Sequence-First
// Phase Kernel in Detail") / Hydragen's suffix attention: per sequence, the
// keys of its private chunks are walked through the page list, with an
// online softmax carrying the running (m, n, O) state of ChunkAttention
// Eq. 1-2.  The G query heads that share a KV head are processed together
// (each KV byte is loaded once for the whole group).
//
// One CTA = one producer warp + up to four consumer warps.  A work item is
// (sequences, a group of nh <= 4 consecutive KV heads, a key range); consumer
// warp w computes KV head kvh0 + w.  A page holds all KV heads of its tokens
// contiguously, so one TMA box covers 16 tokens x 64 columns x nh heads
// (8 KB at nh = 4): the TMA engine costs about the same per box whatever its
// size, and 2 KB one-head boxes would cap an SM at a fraction of HBM
// bandwidth.  The producer fills a 3-stage ring of K and V chunks (128-byte
// swizzled, so the ldmatrix reads are conflict free); the consumers release a
// stage by arriving on its "empty" barrier.  Scores and P V use the m16n8k16
// bf16 MMA with f32 accumulation: rows are the (up to 16) query rows, S = Q K^T
// for 16 keys is two n8 tiles, and O = P V reuses the S accumulator layout as
// the A operand.  CTAs walk their items back to back; the producer runs ahead
// across item boundaries.
#include <cuda_runtime.h>

#include "hp_internal.h"
#include "hp_ptx.cuh"

namespace hp {

namespace {

constexpr int kConsumers = 4;  // consumer warps = largest KV-head group
constexpr int kThreadsSmall = (kConsumers + 1) * 32;
constexpr int kStages = 3;
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct SmallLayout {
    static constexpr int kHalves = D / 64;
    static constexpr int kHeadBox = 16 * 128;            // one head: [16 tokens][64 bf16], swizzled
    static constexpr int kHalf = kConsumers * kHeadBox;  // one column half of the head group
    static constexpr int kChunk = kHalves * kHalf;       // K (or V) of one 16-token chunk
    static constexpr int kStage = 2 * kChunk;            // K then V
    static constexpr int kBar = kStages * kStage;
    static constexpr int kFlags = kBar + 2 * kStages * 8;  // full[], empty[] then per-stage flags
    static constexpr int kBytes = kFlags + kStages * 4 + 64;
};

struct SItem {
    int valid;
    int seq_begin, n_seq, kvh0, k0, k1, part_row;
    const int32_t *pages;
    int ps, num_pages;
    const void *map_k;
    const void *map_v;
};

__device__ __forceinline__ SItem get_item(const SmallParams &p, int idx)
{
    SItem it;
    if (p.plan != nullptr) {
        const WorkItem w = plan_array<WorkItem>(p.plan, p.plan->off_small)[idx];
        const LevelDev &lv = p.plan->levels[w.level];
        const CUtensorMap *maps = plan_array<CUtensorMap>(p.plan, p.plan->off_maps);
        it.seq_begin = w.seq_begin;
        it.n_seq = w.n_seq;
        it.kvh0 = w.kvh;
        it.k0 = w.k0;
        it.k1 = w.k1;
        it.part_row = w.part_row;
        it.pages = plan_array<int32_t>(p.plan, p.plan->off_page_ids) + w.page_base;
        it.ps = lv.page_size;
        it.num_pages = lv.num_pages;
        it.map_k = maps + w.level * kMapsPerLevel + 2;
        it.map_v = maps + w.level * kMapsPerLevel + 3;
    } else {
        const int split = idx % p.n_split;
        const int t = idx / p.n_split;
        const int groups = p.Hkv / p.nh;
        const int grp = t % groups;
        const int b = t / groups;
        int len = __ldg(p.seq_lens + b);
        const int cap = p.pt_stride * p.page_size;
        if (len < 0 || len > cap) {
            atomicOr(p.status, kStBounds);
            len = len < 0 ? 0 : cap;
        }
        it.seq_begin = b;
        it.n_seq = 1;
        it.kvh0 = grp * p.nh;
        it.k0 = split * p.split_len;
        it.k1 = min(it.k0 + p.split_len, len);
        it.part_row = idx * p.nh * p.G;
        it.pages = p.page_table + (int64_t)b * p.pt_stride;
        it.ps = p.page_size;
        it.num_pages = p.num_pages;
        it.map_k = &p.map_k;
        it.map_v = &p.map_v;
    }
    it.valid = it.k0 < it.k1;
    return it;
}

// A walk over the chunks of this CTA's items (items c, c + grid, ...).  The
// producer's walk also holds, in register `pg` of lane l, the page id of
// chunk blk*32 + l of the current item (loaded by all lanes at once).
struct Cursor {
    int item;     // current item index (>= n_items when done)
    int chunk;    // chunk within the item
    int nchunks;  // chunks of the item
    int pg;       // page id block (producer walk only)
    int blk;      // which 32-chunk block pg holds
    SItem it;
};

__device__ __forceinline__ void cursor_load_pages(Cursor &c, int lane)
{
    c.blk = c.chunk >> 5;
    const int ch = c.blk * 32 + lane;
    c.pg = ch < c.nchunks ? __ldg(c.it.pages + (c.it.k0 + ch * kChunk) / c.it.ps) : 0;
}

__device__ __forceinline__ void cursor_seek(const SmallParams &p, int n_items, int stride, Cursor &c,
                                            bool with_pages, int lane)
{
    while (c.item < n_items) {
        c.it = get_item(p, c.item);
        if (c.it.valid) {
            c.chunk = 0;
            c.nchunks = (c.it.k1 - c.it.k0 + kChunk - 1) / kChunk;
            if (with_pages) {
                cursor_load_pages(c, lane);
                if (p.plan != nullptr && c.item + stride < n_items && lane == 0)
                    asm volatile("prefetch.global.L1 [%0];" ::"l"(
                        plan_array<WorkItem>(p.plan, p.plan->off_small) + c.item + stride));
            }
            return;
        }
        c.item += stride;
    }
}

__device__ __forceinline__ void cursor_next(const SmallParams &p, int n_items, int stride, Cursor &c,
                                            bool with_pages, int lane)
{
    if (++c.chunk >= c.nchunks) {
        c.item += stride;
        cursor_seek(p, n_items, stride, c, with_pages, lane);
    } else if (with_pages && (c.chunk >> 5) != c.blk) {
        cursor_load_pages(c, lane);
    }
}

// Issue the TMA copies of the producer's current chunk (called by all lanes
// of the producer warp; lanes 0 .. 2*(d/64)-1 each issue one box: K or V,
// one column half, every head of the group).  *bad is set when the page id
// is out of range: the boxes are then zero-filled and the consumers mask the
// chunk.
template <int D>
__device__ __forceinline__ void issue_chunk(const SmallParams &p, const Cursor &c, uint32_t stage_addr,
                                            uint32_t bar, volatile int *bad, int lane)
{
    using L = SmallLayout<D>;
    constexpr int kHalves = D / 64;
    int page = __shfl_sync(0xffffffffu, c.pg, c.chunk & 31);
    const bool oob = (unsigned)page >= (unsigned)c.it.num_pages;
    if (oob)
        page = c.it.num_pages;
    if (lane == 0) {
        if (oob)
            atomicOr(p.status, kStBounds);
        *bad = oob ? 1 : 0;
        mbar_arrive_expect_tx(bar, 2 * kHalves * p.nh * L::kHeadBox);
    }
    __syncwarp();
    if (lane < 2 * kHalves) {
        const int t = c.it.k0 + c.chunk * kChunk;
        const int h = lane % kHalves;
        const bool is_v = lane >= kHalves;
        tma_load_4d(stage_addr + (is_v ? L::kChunk : 0) + h * L::kHalf, is_v ? c.it.map_v : c.it.map_k, bar,
                    h * 64, t % c.it.ps, c.it.kvh0, page);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreadsSmall) hp_small_kernel(const __grid_constant__ SmallParams p)
{
    using L = SmallLayout<D>;
    constexpr int kHalves = D / 64;
    constexpr int kKs = D / 16;  // k-steps of the S MMA
    constexpr int kNt = D / 8;   // n8 tiles of O

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full0 = sbase + L::kBar;
    const uint32_t empty0 = full0 + kStages * 8;
    volatile int *bad = reinterpret_cast<volatile int *>(smem + L::kFlags);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L::kFlags + kStages * 4);

    if (p.plan != nullptr && (p.plan->magic != kPlanMagic || p.plan->tag != p.tag)) {
        if (threadIdx.x == 0)
            atomicOr(p.status, kStPlan);
        return;
    }
    const int nh = p.nh;
    const int n_items = p.n_items;
    const int stride = gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, (uint32_t)nh);
        }
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    auto wait_warp = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, p.status, abort)) != 0;
    };

    if (warp == kConsumers) {
        // -------------------------------------------------------- producer
        Cursor prod{(int)blockIdx.x, 0, 0, 0, -1, {}};
        cursor_seek(p, n_items, stride, prod, true, lane);
        if (lane == 0 && prod.item < n_items) {
            prefetch_tensormap(prod.it.map_k);
            prefetch_tensormap(prod.it.map_v);
        }
        uint32_t k = 0;
        for (; prod.item < n_items; ++k) {
            const uint32_t st = k % kStages;
            if (k >= (uint32_t)kStages && !wait_warp(empty0 + 8 * st, ((k / kStages) - 1) & 1u))
                break;
            issue_chunk<D>(p, prod, sbase + st * L::kStage, full0 + 8 * st, bad + st, lane);
            cursor_next(p, n_items, stride, prod, true, lane);
        }
        // every copy issued has landed before the CTA exits
        if (lane == 0)
            for (uint32_t j = k > (uint32_t)kStages ? k - kStages : 0; j < k; ++j)
                mbar_wait_drain(full0 + 8 * (j % kStages), (j / kStages) & 1u);
    } else if (warp < nh) {
        // -------------------------------------------------------- consumer
        Cursor cons{(int)blockIdx.x, 0, 0, 0, -1, {}};
        cursor_seek(p, n_items, stride, cons, false, lane);
        uint32_t qa[kKs][4];
        float o[kNt][4];
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        const int r0 = lane >> 2, r1 = r0 + 8;
        const int tq = 2 * (lane & 3);
        const uint32_t hoff = (uint32_t)warp * L::kHeadBox;  // this warp's head within a box
        uint32_t k = 0;
        while (cons.item < n_items) {
            const SItem &it = cons.it;
            const int rows = it.n_seq * p.G;
            const int kvh = it.kvh0 + warp;
            if (cons.chunk == 0) {
                // new item: query fragments (A operand, rows r0 / r1) and state
                const uint16_t *q0 = nullptr, *q1 = nullptr;
                if (r0 < rows)
                    q0 = p.q + (int64_t)(it.seq_begin + r0 / p.G) * p.q_sb + (int64_t)(kvh * p.G + r0 % p.G) * p.q_sh;
                if (r1 < rows)
                    q1 = p.q + (int64_t)(it.seq_begin + r1 / p.G) * p.q_sb + (int64_t)(kvh * p.G + r1 % p.G) * p.q_sh;
#pragma unroll
                for (int ks = 0; ks < kKs; ++ks) {
                    qa[ks][0] = q0 ? __ldg(reinterpret_cast<const uint32_t *>(q0 + ks * 16 + tq)) : 0u;
                    qa[ks][1] = q1 ? __ldg(reinterpret_cast<const uint32_t *>(q1 + ks * 16 + tq)) : 0u;
                    qa[ks][2] = q0 ? __ldg(reinterpret_cast<const uint32_t *>(q0 + ks * 16 + 8 + tq)) : 0u;
                    qa[ks][3] = q1 ? __ldg(reinterpret_cast<const uint32_t *>(q1 + ks * 16 + 8 + tq)) : 0u;
                }
#pragma unroll
                for (int n = 0; n < kNt; ++n)
                    o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
                m0 = m1 = -INFINITY;
                l0 = l1 = 0.f;
            }
            const uint32_t st = k % kStages;
            const uint32_t kst = sbase + st * L::kStage + hoff;
            const uint32_t vst = kst + L::kChunk;
            if (!wait_warp(full0 + 8 * st, (k / kStages) & 1u))
                break;

            const int t0 = it.k0 + cons.chunk * kChunk;
            int nvalid = min(kChunk, it.k1 - t0);
            if (bad[st])
                nvalid = 0;
            if (nvalid < kChunk) {
                // rows past the valid keys: zero this head's V so that
                // 0 * (whatever the pool holds there) stays 0
                uint8_t *vp = smem + (vst - sbase);
                const int nz = (kChunk - nvalid) * 8 * kHalves;
                for (int i = lane; i < nz; i += 32) {
                    const int row = nvalid + i / (8 * kHalves);
                    const int rem = i % (8 * kHalves);
                    const int h = rem >> 3, c = rem & 7;
                    *reinterpret_cast<uint4 *>(vp + h * L::kHalf + row * 128 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }

            // S = Q K^T over 16 keys: n8 tile 0 = keys 0-7, tile 1 = keys 8-15
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
            {
                const int mi = lane >> 3, ri = lane & 7;
                const int tok = ri + ((mi >> 1) << 3);
#pragma unroll
                for (int ks = 0; ks < kKs; ++ks) {
                    const int dch = 2 * ks + (mi & 1);
                    const uint32_t addr = kst + (dch >> 3) * L::kHalf + tok * 128 + (((dch & 7) ^ (tok & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(addr, b0, b1, b2, b3);
                    mma_bf16_16816(s0, qa[ks], b0, b1);
                    mma_bf16_16816(s1, qa[ks], b2, b3);
                }
            }
            // online softmax (rows r0: elements 0,1; rows r1: elements 2,3)
            const float c = p.scale_log2;
            float x[2][4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tk = tq + (e & 1);
                x[0][e] = tk < nvalid ? s0[e] * c : -INFINITY;
                x[1][e] = tk + 8 < nvalid ? s1[e] * c : -INFINITY;
            }
            float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
            float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float ms0 = mn0 == -INFINITY ? 0.f : mn0;  // all keys so far masked: nothing to scale
            const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
            const float a0 = fast_exp2(m0 - ms0), a1 = fast_exp2(m1 - ms1);
            m0 = mn0;
            m1 = mn1;
            if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                for (int n = 0; n < kNt; ++n) {
                    o[n][0] *= a0;
                    o[n][1] *= a0;
                    o[n][2] *= a1;
                    o[n][3] *= a1;
                }
                l0 *= a0;
                l1 *= a1;
            }
            uint32_t pa[4];
            pa[0] = pack_bf16x2(fast_exp2(x[0][0] - ms0), fast_exp2(x[0][1] - ms0));
            pa[1] = pack_bf16x2(fast_exp2(x[0][2] - ms1), fast_exp2(x[0][3] - ms1));
            pa[2] = pack_bf16x2(fast_exp2(x[1][0] - ms0), fast_exp2(x[1][1] - ms0));
            pa[3] = pack_bf16x2(fast_exp2(x[1][2] - ms1), fast_exp2(x[1][3] - ms1));
            l0 += bf16lo_to_f32(pa[0]) + bf16hi_to_f32(pa[0]) + bf16lo_to_f32(pa[2]) + bf16hi_to_f32(pa[2]);
            l1 += bf16lo_to_f32(pa[1]) + bf16hi_to_f32(pa[1]) + bf16lo_to_f32(pa[3]) + bf16hi_to_f32(pa[3]);

            // O += P V
            {
                const int mi = lane >> 3, ri = lane & 7;
                const int tok = ri + ((mi & 1) << 3);
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    const int dch = 2 * dp + (mi >> 1);
                    const uint32_t addr = vst + (dch >> 3) * L::kHalf + tok * 128 + (((dch & 7) ^ (tok & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(addr, b0, b1, b2, b3);
                    mma_bf16_16816(o[2 * dp], pa, b0, b1);
                    mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
                }
            }
            // release the stage to the producer
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty0 + 8 * st);
            ++k;

            if (cons.chunk + 1 >= cons.nchunks) {
                float L0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
                L0 += __shfl_xor_sync(0xffffffffu, L0, 2);
                float L1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
                L1 += __shfl_xor_sync(0xffffffffu, L1, 2);
                const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f;
                const float inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
                const int base = it.part_row + warp * rows;  // this head's rows
                if (r0 < rows) {
                    float *dst = p.part_o + (size_t)(base + r0) * D + tq;
#pragma unroll
                    for (int n = 0; n < kNt; ++n)
                        *reinterpret_cast<float2 *>(dst + n * 8) = make_float2(o[n][0] * inv0, o[n][1] * inv0);
                    if ((lane & 3) == 0)
                        p.part_lse[base + r0] = L0 > 0.f ? (m0 + fast_log2(L0)) * kLn2 : -INFINITY;
                }
                if (r1 < rows) {
                    float *dst = p.part_o + (size_t)(base + r1) * D + tq;
#pragma unroll
                    for (int n = 0; n < kNt; ++n)
                        *reinterpret_cast<float2 *>(dst + n * 8) = make_float2(o[n][2] * inv1, o[n][3] * inv1);
                    if ((lane & 3) == 0)
                        p.part_lse[base + r1] = L1 > 0.f ? (m1 + fast_log2(L1)) * kLn2 : -INFINITY;
                }
            }
            cursor_next(p, n_items, stride, cons, false, lane);
        }
    }
    __syncwarp();
}

template <int D>
cudaError_t launch_small_d(const SmallParams &p, int grid, cudaStream_t s)
{
    static bool configured = false;
    const int bytes = SmallLayout<D>::kBytes + 1024;
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(hp_small_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    hp_small_kernel<D><<<grid, kThreadsSmall, bytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t small_smem_bytes(int d)
{
    return d == 64 ? SmallLayout<64>::kBytes + 1024 : SmallLayout<128>::kBytes + 1024;
}

int small_heads_per_item(int Hkv)
{
    return Hkv % 4 == 0 ? 4 : (Hkv % 2 == 0 ? 2 : 1);
}

cudaError_t launch_small(const SmallParams &p, int grid, int d, cudaStream_t s)
{
    if (grid <= 0)
        return cudaSuccess;
    return d == 64 ? launch_small_d<64>(p, grid, s) : launch_small_d<128>(p, grid, s);
}

}  // namespace hp
