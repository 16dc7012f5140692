// hp_small_role.cuh -- the paged-decode role: up to 16 query rows per KV
// head against one key range (a private suffix, or a node shared by very few
// sequences).  Shared by the standalone paged-decode kernel and the fused
// cascade kernel.
//
// Method: the sequence-first phase of ChunkAttention ("The Sequence-First
// Phase Kernel in Detail") / Hydragen's suffix attention: per sequence, the
// keys of its private chunks are walked through the page list, with an
// online softmax carrying the running (m, n, O) state of ChunkAttention
// Eq. 1-2.  The G query heads that share a KV head are processed together
// (each KV byte is loaded once for the whole group).
//
// A work item is (sequences, a group of nh consecutive KV heads, a key
// range); consumer warp w computes KV head kvh0 + w.  A page holds all KV
// heads of its tokens contiguously, so one TMA box covers 16 tokens x 64
// columns x nh heads: the TMA engine costs about the same per box whatever its
// size, and one-head 2 KB boxes would cap an SM far below HBM bandwidth.  One
// producer warp fills a ring of K and V chunks (128-byte swizzled, so the
// ldmatrix reads are conflict free) and writes, per stage, the item fields
// the consumers need; the consumers release a stage by arriving on its
// "empty" barrier.  With an item's first chunk the producer also loads the
// item's query rows (one sequence: G rows per head of the group) into the
// stage's Q slot, so a new item costs the consumers no dependent global load.
// Scores and P V use the m16n8k16 bf16 MMA with f32 accumulation: rows are
// the (up to 16) query rows of a head, S = Q K^T for 16 keys is two n8
// tiles, and O = P V reuses the S accumulator layout as the A operand.  The
// producer runs ahead across item boundaries.
//
// Reduced-precision KV (Q8 instantiations, d = 128): the pools hold E4M3
// codes, one byte per element, with an f32 scale per (page, KV head) for K
// and one for V (Hydragen, "Implications and Future Directions": the suffix
// pass is memory-bound and quantising its KV cache halves its bytes).  A
// stage holds the 16-token chunk's codes (one box of 16 tokens x 128 bytes x
// nh heads per K and per V) and the chunk's scales, which the producer copies
// with cp.async tracked by the stage's barrier.  The consumers decode codes
// to f16 in registers, exactly: K codes with integer bit operations (up to a
// power of two), V codes with the hardware conversion (the two spread the
// work over two pipes), and use the f16 MMA: the queries are rounded from
// bf16 to f16 once per item (exact for |q| in f16's normal range), scores
// are scaled by the chunk's K scale, and P is weighted by the chunk's V
// scale before it is rounded to f16 for P V.  The fragment layouts are in
// consumer_q8.
#pragma once

#include <cuda_runtime.h>

#include "hp_internal.h"
#include "hp_ptx.cuh"

namespace hp {
namespace smr {

constexpr float kLn2 = 0.69314718055994530942f;

// Shared memory of the role for NC consumer warps, S stages and a Q slot of
// QR rows per stage; Q8: E4M3 pools (d = 128); SM: the stream mask of a
// Parallel Prompting row (each stage also holds its keys' stream ids and
// positions: up to 8 chunks of 16 keys).
template <int D, int NC, int S, int QR, bool Q8 = false, bool SM = false>
struct Layout {
    static_assert(!Q8 || D == 128, "E4M3 pools: d = 128");
    static constexpr int kHalves = D / 64;
    static constexpr int kHeadBox = 16 * 128;     // one head: [16 tokens][64 bf16] or [16 tokens][128 E4M3], swizzled
    static constexpr int kHalf = NC * kHeadBox;   // one column half of the head group (bf16)
    static constexpr int kChunk = Q8 ? kHalf : kHalves * kHalf;  // K (or V) of one 16-token chunk
    static constexpr int kQRows = QR;                // Q slot: nh * G <= QR rows of one sequence
    static constexpr int kQHalf = kQRows * 128;
    static constexpr int kQSlot = kHalves * kQHalf;
    static constexpr int kScales = Q8 ? 1024 : 0;  // Q8: K scales [NC], then V scales at +128 bytes (f32)
    static constexpr int kMask = SM ? 1024 : 0;    // SM: stream ids of chunk c at 64c, positions at 512 + 64c (int32)
    static constexpr int kStage = 2 * kChunk + kQSlot + kScales + kMask;  // K, V, Q slot, scales, mask
    static constexpr int kEnd = S * kStage;
    static_assert(NC * 4 <= 128, "scale slots");
};

// What the consumers need about the chunk in a stage.
struct StageMeta {
    int seq_begin, n_seq, kvh0, part_row;
    int nvalid;  // valid keys of the chunk (0 when its page id was out of range)
    int first, last;
    int qslot;   // first chunk only: the item's Q rows are in this stage's Q slot
    int pairs;   // the item has at least kPairChunks chunks (E4M3 consumers take them two at a time)
    int oob;     // rows stages: bit c set when chunk c's page id was out of range
};


template <int N>
struct Int {
    static constexpr int value = N;
};

// The geometry of one item.
struct Desc {
    int valid;
    int seq_begin, n_seq, kvh0, k0, k1, part_row;
    const int32_t *pages;  // page of key t: pages[t / ps - pbase] (generic address)
    int pbase;
    int ps, num_pages;
    const void *map_k;
    const void *map_v;
    // Parallel Prompting row (SM): stream id and position of key t of the
    // row at slot_sid[t] / slot_pos[t] (16-byte aligned, readable to the end
    // of the 16-key chunk holding the row's last key)
    const int32_t *slot_sid = nullptr;
    const int32_t *slot_pos = nullptr;
    // E4M3 pools: scale of (page, KV head h) at k_scale[page * Hkv + h]
    const float *k_scale = nullptr;
    const float *v_scale = nullptr;
    int Hkv = 0;
    // A decode step with the append fused: the item holds the step's new
    // token (its last key).  The producer copies the token's K and V rows of
    // the item's nh heads (head h at src + h * src_sh) to the pool (head h
    // at dst + h * dst_sh) before it loads the item's last chunk.  Null: no
    // token to write.
    const uint16_t *tok_k_src = nullptr;
    const uint16_t *tok_v_src = nullptr;
    uint16_t *tok_k_dst = nullptr;
    uint16_t *tok_v_dst = nullptr;
    int64_t tok_src_sh = 0;
    int64_t tok_dst_sh = 0;
};

struct Ctx {
    uint8_t *smem;   // 1024-aligned base of the ring
    uint32_t sbase;
    uint32_t full0;  // S "full" barriers (count 1 + transaction bytes)
    uint32_t empty0; // S "empty" barriers (count nh)
    StageMeta *meta; // S entries
    uint32_t zero16; // 16 zero bytes (shared address): ldmatrix rows past the item
    volatile int *abort;
    uint32_t *status;
};

struct Args {
    const uint16_t *q;      // rows read by the consumers when Q is not in the slot
    int64_t q_sb, q_sh;
    const void *map_q;      // box 64 columns x (nh * G) heads x 1 row (nh * G <= QR); null: no Q slot
    int G, nh;
    float scale_log2;
    uint16_t *part_o;  // bf16
    float *part_lse;
    // SM: consumer warp w serves head w / n_sg of the item's group and its
    // streams (query sequences) (w % n_sg) * ns_pg .. + ns_pg - 1 (ns_pg * G
    // <= 16 rows), writing partial rows part_row + w * ns_pg * G ..; query
    // sequence b carries stream id q_sid[b] and position q_pos[b]
    int n_sg = 1, ns_pg = 0;
    const int32_t *q_sid = nullptr;
    const int32_t *q_pos = nullptr;
};

// Producer warp: walks items k = 0, 1, ... of `src` (src(k, pre) -> Desc,
// with n_items entries; pre = src.prefetch(k), loaded for 32 items at a time,
// one per lane, so that a value an item needs from global memory is not a
// dependent load at the item's start), then closes the ring with a sentinel
// stage (n_seq = -1, completed by a plain arrival) that tells the consumers
// to stop.  All 32 lanes call it.
template <int D, int NC, int S, int QR, class Src, bool Q8 = false>
__device__ __forceinline__ void producer(const Ctx &c, const Args &a, const Src &src, int n_items, int lane)
{
    using L = Layout<D, NC, S, QR, Q8>;
    constexpr int kHalves = D / 64;
    auto wait_warp = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, c.status, c.abort)) != 0;
    };
    uint32_t k = 0;  // chunks issued
    bool ok = true;
    bool prefetched = false;
    int pre = 0;
    for (int it = 0; ok && it < n_items; ++it) {
        if (Src::kPrefetch && (it & 31) == 0)
            pre = src.prefetch(it + lane < n_items ? it + lane : -1);
        const Desc d = src(it, Src::kPrefetch ? __shfl_sync(0xffffffffu, pre, it & 31) : 0);
        if (!d.valid)
            continue;
        // the step's new token (a decode step with the append fused): its K
        // and V rows are loaded now and stored before the item's last chunk
        constexpr int kPer = D / 8;  // 16-byte pieces of one head's row
        constexpr int kTokRegs = Src::kTokens ? (2 * 8 * kPer + 31) / 32 : 1;  // nh <= 8
        uint4 tok[kTokRegs];
        const int ntok = Src::kTokens && d.tok_k_dst != nullptr ? 2 * a.nh * kPer : 0;
#pragma unroll
        for (int r = 0; r < kTokRegs; ++r) {
            const int i = lane + 32 * r;
            if (i < ntok) {
                const bool is_v = i >= ntok / 2;
                const int j = is_v ? i - ntok / 2 : i;
                tok[r] = *reinterpret_cast<const uint4 *>((is_v ? d.tok_v_src : d.tok_k_src) +
                                                          (j / kPer) * d.tok_src_sh + (j % kPer) * 8);
            }
        }
        if (!prefetched && lane == 0) {
            prefetch_tensormap(d.map_k);
            prefetch_tensormap(d.map_v);
            prefetched = true;
        }
        const int nchunks = (d.k1 - d.k0 + kChunk - 1) / kChunk;
        const bool qslot = a.map_q != nullptr && d.n_seq == 1;
        int pg = 0;
        for (int ch = 0; ch < nchunks; ++ch, ++k) {
            if ((ch & 31) == 0) {  // page ids of the next 32 chunks, one per lane
                const int cc = ch + lane;
                pg = cc < nchunks ? d.pages[(d.k0 + cc * kChunk) / d.ps - d.pbase] : 0;
            }
            const uint32_t st = k % S;
            if (k >= (uint32_t)S && !(ok = wait_warp(c.empty0 + 8 * st, ((k / S) - 1) & 1u)))
                break;
            int page = __shfl_sync(0xffffffffu, pg, ch & 31);
            const bool oob = (unsigned)page >= (unsigned)d.num_pages;
            if (oob)
                page = d.num_pages;  // zero-filled boxes, chunk masked
            const int t = d.k0 + ch * kChunk;
            const uint32_t bar = c.full0 + 8 * st;
            if (Src::kTokens && ntok > 0 && ch + 1 == nchunks) {
                // the new token, in this chunk: its rows go to the pool first,
                // visible to the copy below (generic writes, proxy fence, warp
                // barrier, then the TMA issue)
#pragma unroll
                for (int r = 0; r < kTokRegs; ++r) {
                    const int i = lane + 32 * r;
                    if (i < ntok) {
                        const bool is_v = i >= ntok / 2;
                        const int j = is_v ? i - ntok / 2 : i;
                        *reinterpret_cast<uint4 *>((is_v ? d.tok_v_dst : d.tok_k_dst) + (j / kPer) * d.tok_dst_sh +
                                                   (j % kPer) * 8) = tok[r];
                    }
                }
                fence_proxy_async_global();
                __syncwarp();
            }
            if constexpr (Q8) {
                // the chunk's scales: K of heads kvh0 .. kvh0 + nh - 1 by lanes
                // 8.., V by lanes 16..; tracked by the stage's barrier (its
                // pending count rises before the producer's own arrival)
                const int hi = lane & 7;
                if (lane >= 8 && lane < 24 && hi < a.nh) {
                    const bool is_v = lane >= 16;
                    const uint32_t dst = c.sbase + st * L::kStage + 2 * L::kChunk + L::kQSlot + (is_v ? 128 : 0) + 4 * hi;
                    if (oob) {
                        st_shared_f32(dst, 0.f);
                    } else {
                        cp_async_4(dst, (is_v ? d.v_scale : d.k_scale) + (int64_t)page * d.Hkv + d.kvh0 + hi);
                        cp_async_mbar_arrive(bar);
                    }
                }
                __syncwarp();
            }
            if (lane == 0) {
                if (oob)
                    atomicOr(c.status, kStBounds);
                StageMeta m;
                m.seq_begin = d.seq_begin;
                m.n_seq = d.n_seq;
                m.kvh0 = d.kvh0;
                m.part_row = d.part_row;
                m.nvalid = oob ? 0 : min(kChunk, d.k1 - t);
                m.first = ch == 0;
                m.last = ch + 1 == nchunks;
                m.qslot = ch == 0 && qslot;
                m.pairs = nchunks >= kPairChunks;
                c.meta[st] = m;
                mbar_arrive_expect_tx(bar, (Q8 ? 2 : 2 * kHalves) * a.nh * L::kHeadBox +
                                               (m.qslot ? kHalves * a.nh * a.G * 128 : 0));
            }
            __syncwarp();
            constexpr int kBoxLanes = Q8 ? 2 : 2 * kHalves;  // K and V boxes (one per column half for bf16)
            if (lane < kBoxLanes) {
                const int h = Q8 ? 0 : lane % kHalves;
                const bool is_v = Q8 ? lane == 1 : lane >= kHalves;
                tma_load_4d_h(c.sbase + st * L::kStage + (is_v ? L::kChunk : 0) + h * L::kHalf,
                              is_v ? d.map_v : d.map_k, bar, h * 64, t % d.ps, d.kvh0, page, l2_evict_first());
            } else if (ch == 0 && qslot && lane < kBoxLanes + kHalves) {
                const int h = lane - kBoxLanes;
                tma_load_3d(c.sbase + st * L::kStage + 2 * L::kChunk + h * L::kQHalf, a.map_q, bar, h * 64,
                            d.kvh0 * a.G, d.seq_begin);
            }
        }
    }
    // sentinel stage
    {
        const uint32_t st = k % S;
        if (k >= (uint32_t)S)
            wait_warp(c.empty0 + 8 * st, ((k / S) - 1) & 1u);
        if (lane == 0) {
            StageMeta m{};
            m.n_seq = -1;
            c.meta[st] = m;
            mbar_arrive(c.full0 + 8 * st);
        }
        __syncwarp();
        ++k;
    }
    // every copy issued has landed before the role ends
    if (lane == 0)
        for (uint32_t j = k > (uint32_t)S ? k - S : 0; j < k; ++j)
            mbar_wait_drain(c.full0 + 8 * (j % S), (j / S) & 1u);
}

// Consumer warp w (0 <= w < nh): processes the chunks in ring order until
// the producer's sentinel stage.
template <int D, int NC, int S, int QR>
__device__ __forceinline__ void consumer(const Ctx &c, const Args &a, int w, int lane)
{
    using L = Layout<D, NC, S, QR>;
    constexpr int kHalves = D / 64;
    constexpr int kKs = D / 16;  // k-steps of the S MMA
    constexpr int kNt = D / 8;   // n8 tiles of O
    auto wait_warp = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, c.status, c.abort)) != 0;
    };
    uint32_t qa[kKs][4];
    float o[kNt][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int r0 = lane >> 2, r1 = r0 + 8;
    const int tq = 2 * (lane & 3);
    const uint32_t hoff = (uint32_t)w * L::kHeadBox;  // this warp's head within a box
    for (uint32_t k = 0;; ++k) {
        const uint32_t st = k % S;
        if (!wait_warp(c.full0 + 8 * st, (k / S) & 1u))
            break;
        const StageMeta m = c.meta[st];
        if (m.n_seq < 0)
            break;  // sentinel: the producer's walk is over
        const int seq0 = m.seq_begin;
        const int rows = m.n_seq * a.G;
        const int kvh = m.kvh0 + w;
        if (m.first && m.qslot) {
            // new item, Q rows in the stage: head w's rows are slot rows
            // w*G .. w*G+G-1; rows past G read a zero chunk
            const int mi = lane >> 3, ri = (lane & 7) + ((mi & 1) << 3);
            const uint32_t qs = c.sbase + st * L::kStage + 2 * L::kChunk;
            const int srow = w * a.G + ri;
#pragma unroll
            for (int ks = 0; ks < kKs; ++ks) {
                const int dch = 2 * ks + (mi >> 1);
                const uint32_t addr = ri < rows ? qs + (dch >> 3) * L::kQHalf + srow * 128 +
                                                      (((dch & 7) ^ (srow & 7)) << 4)
                                                : c.zero16;
                ldmatrix_x4(addr, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
            }
#pragma unroll
            for (int n = 0; n < kNt; ++n)
                o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        } else if (m.first) {
            // new item: query fragments (A operand, rows r0 / r1) and state
            const uint16_t *q0 = nullptr, *q1 = nullptr;
            if (r0 < rows)
                q0 = a.q + (int64_t)(seq0 + r0 / a.G) * a.q_sb + (int64_t)(kvh * a.G + r0 % a.G) * a.q_sh;
            if (r1 < rows)
                q1 = a.q + (int64_t)(seq0 + r1 / a.G) * a.q_sb + (int64_t)(kvh * a.G + r1 % a.G) * a.q_sh;
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
        const uint32_t kst = c.sbase + st * L::kStage + hoff;
        const uint32_t vst = kst + L::kChunk;
        const int nvalid = m.nvalid;
        if (nvalid < kChunk) {
            // rows past the valid keys: zero this head's V so that
            // 0 * (whatever the pool holds there) stays 0
            uint8_t *vp = c.smem + (vst - c.sbase);
            const int nz = (kChunk - nvalid) * 8 * kHalves;
            for (int i = lane; i < nz; i += 32) {
                const int row = nvalid + i / (8 * kHalves);
                const int rem = i % (8 * kHalves);
                const int h = rem >> 3, ch = rem & 7;
                *reinterpret_cast<uint4 *>(vp + h * L::kHalf + row * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
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
        const float cs = a.scale_log2;
        float x[2][4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int tk = tq + (e & 1);
            x[0][e] = tk < nvalid ? s0[e] * cs : -INFINITY;
            x[1][e] = tk + 8 < nvalid ? s1[e] * cs : -INFINITY;
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
            mbar_arrive(c.empty0 + 8 * st);

        if (m.last) {
            float L0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
            L0 += __shfl_xor_sync(0xffffffffu, L0, 2);
            float L1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
            L1 += __shfl_xor_sync(0xffffffffu, L1, 2);
            const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f;
            const float inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
            const int base = m.part_row + w * rows;  // this warp's rows
            if (r0 < rows) {
                uint16_t *dst = a.part_o + (size_t)(base + r0) * D + tq;
#pragma unroll
                for (int n = 0; n < kNt; ++n)
                    *reinterpret_cast<uint32_t *>(dst + n * 8) = pack_bf16x2(o[n][0] * inv0, o[n][1] * inv0);
                if ((lane & 3) == 0)
                    a.part_lse[base + r0] = L0 > 0.f ? (m0 + fast_log2(L0)) * kLn2 : -INFINITY;
            }
            if (r1 < rows) {
                uint16_t *dst = a.part_o + (size_t)(base + r1) * D + tq;
#pragma unroll
                for (int n = 0; n < kNt; ++n)
                    *reinterpret_cast<uint32_t *>(dst + n * 8) = pack_bf16x2(o[n][2] * inv1, o[n][3] * inv1);
                if ((lane & 3) == 0)
                    a.part_lse[base + r1] = L1 > 0.f ? (m1 + fast_log2(L1)) * kLn2 : -INFINITY;
            }
        }
    }
}

// Four E4M3 codes (one 32-bit word, bytes b0..b3) -> two f16 pairs holding
// the codes' values times 2^-8, exactly: lo = (b0, b2), hi = (b1, b3), the
// first byte of each pair in the low half.  Each byte's sign stays on top of
// its 16-bit half and its 7 other bits move to bits 7..13: the 4 exponent
// bits land in f16's exponent field (f16's bias 15 against E4M3's 7: the
// factor 2^-8) and the 3 mantissa bits on top of f16's mantissa; subnormal
// codes (exponent 0) land on f16 subnormals with the same factor.  Integer
// ALU operations only.
// Two E4M3 codes (bits 0-7 and 8-15) -> two f16 values, exact (low half
// from the low byte), by the hardware conversion.
__device__ __forceinline__ uint32_t e4m3x2_cvt(uint32_t two_codes)
{
    uint32_t r;
    asm("{.reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t;}" : "=r"(r) : "r"(two_codes));
    return r;
}
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t x, uint32_t &lo, uint32_t &hi)
{
    hi = (x & 0x80008000u) | ((x >> 1) & 0x3F803F80u);
    lo = ((x << 8) & 0x80008000u) | ((x << 7) & 0x3F803F80u);
}

// E4M3 consumer warp w (0 <= w < nh), d = 128: as `consumer`, with codes
// decoded to f16 in registers (K codes as values x 2^-8 by integer
// operations, the factor 2^8 put back into the K scale of the scores; V
// codes as their values by the hardware conversion) and the
// operands of both products swapped so that the keys fill the MMA's 16 rows
// and the head's query rows its 8 columns: with up to 8 query rows (G <= 8,
// one sequence) a chunk costs 16 MMAs instead of 32; 9..16 rows take a
// second column tile.
//   - S^T = K Q^T: k-step i of thread (g, t) takes bytes 32t+4i .. 32t+4i+3
//     of key rows g and g+8; its A registers pair bytes (0, 2) and (1, 3),
//     and the query fragments (B) pair the same columns, so the head
//     dimension is summed in a permuted order (the same for Q and K).  Even
//     and odd k-steps accumulate separately (independent MMA chains).
//   - The scores of a query are spread over the 8 lanes of one t (keys g and
//     g + 8 each): maxima and sums are warp reductions over those lanes.
//   - O'^T = V^T P^T: P^T's B fragments are the f16 score tiles transposed
//     with movmatrix; V^T's A fragments pair the codes of keys (2t, 2t+1)
//     and (2t+8, 2t+9) (byte permutes put the two keys' codes of a column
//     side by side for the conversion) of thread (g, t)'s columns
//     16g .. 16g+15, m-tile j
//     taking columns 16g + 2j and 16g + 2j + 1, so thread (g, t) ends with
//     columns 16g .. 16g+15 of query rows 2t and 2t+1 (of each column tile).
//   - The V scale of a chunk enters as P * (vsc / vref), vref being the first
//     nonzero V scale of the item, so P stays near [0, 1] when it is rounded
//     to f16 and O' needs no rescaling between chunks; O = O' vref / l.
//     A chunk whose V scale is 0 adds nothing to O (its weights still count
//     in the denominator).
template <int D, int NC, int S, int QR>
__device__ __forceinline__ void consumer_q8(const Ctx &c, const Args &a, int w, int lane)
{
    using L = Layout<D, NC, S, QR, true>;
    static_assert(D == 128, "E4M3 pools: d = 128");
    static_assert(S >= 2, "two stages held at once");
    constexpr int kKs = D / 16;  // k-steps of S^T = K Q^T
    constexpr int kMt = D / 16;  // m16 tiles of O^T
    constexpr float kDecode = 256.f;  // a K code decoded by integer operations = value * 2^-8
    auto wait_warp = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, c.status, c.abort)) != 0;
    };
    // qb[ks][nt][0|1]: query rows nt*8 + g, column pairs (32t+4ks, +2) / (+1, +3)
    uint32_t qb[kKs][2][2];
    float o[kMt][2][4];
    // per column tile: running max and sum of query rows nt*8 + 2t, + 1
    float mq[2][2], lq[2][2];
    float vref = 0.f;
    const int g = lane >> 2, t = lane & 3;
    const uint32_t hoff = (uint32_t)w * L::kHeadBox;  // this warp's head within a box
    int rows = 0;
    bool two = false;  // a second column tile (9..16 query rows)
    // One pass over NU (1 or 2) consecutive chunks of an item, in stages
    // st[0..NU): with two, their scores share one softmax update and their
    // decoding and MMAs interleave.
    auto pass = [&](auto nu, const uint32_t(&st)[2]) {
        constexpr int NU = decltype(nu)::value;
        uint32_t kst[NU], vst[NU];
        int nvalid[NU];
        float ksc[NU], vsc[NU];
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const uint32_t stage = c.sbase + st[u] * L::kStage;
            kst[u] = stage + hoff;
            vst[u] = stage + L::kChunk + hoff;
            nvalid[u] = c.meta[st[u]].nvalid;
            ksc[u] = ld_shared_f32(stage + 2 * L::kChunk + L::kQSlot + 4 * w);
            vsc[u] = ld_shared_f32(stage + 2 * L::kChunk + L::kQSlot + 128 + 4 * w);
            if (nvalid[u] < kChunk) {
                // rows past the valid keys: zero this head's V codes so that
                // 0 * (whatever the pool holds there) stays 0
                uint8_t *vp = c.smem + (vst[u] - c.sbase);
                const int nz = (kChunk - nvalid[u]) * 8;
                for (int i = lane; i < nz; i += 32)
                    *reinterpret_cast<uint4 *>(vp + (nvalid[u] + i / 8) * 128 + (i % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
            }
        }
        __syncwarp();

        // S^T = K Q^T: rows = keys (g, g + 8), columns = query rows 2t, 2t+1;
        // the k-steps in two halves of four.  With one chunk, even and odd
        // k-steps accumulate separately (independent MMA chains).
        constexpr int NA = NU == 1 ? 2 : NU;  // accumulators
        float sc[NA][2][4];
#pragma unroll
        for (int u = 0; u < NA; ++u)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    sc[u][nt][e] = 0.f;
#pragma unroll
        for (int hk = 0; hk < 2; ++hk) {
            uint4 kw[NU][2];  // [chunk][key row g | g + 8]: bytes 32t + 16hk .. +15
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                const int k0r = g, k1r = g + 8;
                kw[u][0] = ld_shared_v4(kst[u] + k0r * 128 + (((2 * t + hk) ^ (k0r & 7)) << 4));
                kw[u][1] = ld_shared_v4(kst[u] + k1r * 128 + (((2 * t + hk) ^ (k1r & 7)) << 4));
            }
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
                const int ks = 4 * hk + kq;
#pragma unroll
                for (int u = 0; u < NU; ++u) {
                    auto word = [&](const uint4 &v) {
                        return kq == 0 ? v.x : kq == 1 ? v.y : kq == 2 ? v.z : v.w;
                    };
                    uint32_t ak[4];
                    e4m3x4_to_f16(word(kw[u][0]), ak[0], ak[2]);
                    e4m3x4_to_f16(word(kw[u][1]), ak[1], ak[3]);
                    const int acc = NU == 1 ? (ks & 1) : u;
                    mma_f16_16816(sc[acc][0], ak, qb[ks][0][0], qb[ks][0][1]);
                    if (two)
                        mma_f16_16816(sc[acc][1], ak, qb[ks][1][0], qb[ks][1][1]);
                }
            }
        }
        if constexpr (NU == 1) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    sc[0][nt][e] += sc[1][nt][e];
        }
        // online softmax per query column over the pass's keys: element e of
        // tile nt of chunk u is key (e < 2 ? g : g + 8) of the chunk, query
        // row nt*8 + 2t + (e & 1); each chunk's K scale (and the decoding
        // factor) multiplies its scores
        float cs[NU], pv[NU];
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            cs[u] = a.scale_log2 * ksc[u] * kDecode;
            if (vref == 0.f)
                vref = vsc[u];
        }
#pragma unroll
        for (int u = 0; u < NU; ++u)
            pv[u] = vref != 0.f ? vsc[u] / vref : 0.f;  // 0: the chunk adds nothing to O
        uint32_t pb[NU][2][2];  // [chunk][column tile]: P^T fragments (keys 0-7, 8-15)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            if (nt == 1 && !two)
                break;
            float x[NU][4];
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int u = 0; u < NU; ++u) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = e < 2 ? g : g + 8;
                    x[u][e] = key < nvalid[u] ? sc[u][nt][e] * cs[u] : -INFINITY;
                }
                mx[0] = fmax3(mx[0], x[u][0], x[u][2]);
                mx[1] = fmax3(mx[1], x[u][1], x[u][3]);
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], off));
                mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], off));
            }
            float al[2], ms[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float mn = fmaxf(mq[nt][i], mx[i]);
                ms[i] = mn == -INFINITY ? 0.f : mn;  // all keys so far masked: nothing to scale
                al[i] = fast_exp2(mq[nt][i] - ms[i]);
                mq[nt][i] = mn;
                lq[nt][i] *= al[i];
            }
            if (__any_sync(0xffffffffu, al[0] != 1.f || al[1] != 1.f)) {
#pragma unroll
                for (int j = 0; j < kMt; ++j) {
                    o[j][nt][0] *= al[0];
                    o[j][nt][2] *= al[0];
                    o[j][nt][1] *= al[1];
                    o[j][nt][3] *= al[1];
                }
            }
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                float p[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    p[e] = fast_exp2(x[u][e] - ms[e & 1]);
                lq[nt][0] += p[0] + p[2];
                lq[nt][1] += p[1] + p[3];
                // [keys g][queries 2t, 2t+1] per 8x8 block, transposed to
                // [query g][keys 2t, 2t+1]: the B fragments of P^T
                pb[u][nt][0] = movmatrix_trans(pack_f16x2(p[0] * pv[u], p[1] * pv[u]));
                pb[u][nt][1] = movmatrix_trans(pack_f16x2(p[2] * pv[u], p[3] * pv[u]));
            }
        }

        // O'^T += V^T P^T
        const int ta = 2 * t, tb = 2 * t + 1;
        uint4 vw[NU][4];
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            vw[u][0] = ld_shared_v4(vst[u] + ta * 128 + ((g ^ (ta & 7)) << 4));
            vw[u][1] = ld_shared_v4(vst[u] + tb * 128 + ((g ^ (tb & 7)) << 4));
            vw[u][2] = ld_shared_v4(vst[u] + (ta + 8) * 128 + ((g ^ (ta & 7)) << 4));
            vw[u][3] = ld_shared_v4(vst[u] + (tb + 8) * 128 + ((g ^ (tb & 7)) << 4));
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                auto word = [&](const uint4 &v) { return q4 == 0 ? v.x : q4 == 1 ? v.y : q4 == 2 ? v.z : v.w; };
                const uint32_t A = word(vw[u][0]), B = word(vw[u][1]), C = word(vw[u][2]), E = word(vw[u][3]);
                // m-tiles 2q4 and 2q4+1: columns 16g + 4q4 + (0, 1) and (2, 3)
                uint32_t a0[4], a1[4];
                const uint32_t ab0 = __byte_perm(A, B, 0x5140), ce0 = __byte_perm(C, E, 0x5140);
                const uint32_t ab1 = __byte_perm(A, B, 0x7362), ce1 = __byte_perm(C, E, 0x7362);
                a0[0] = e4m3x2_cvt(ab0);
                a0[1] = e4m3x2_cvt(ab0 >> 16);
                a0[2] = e4m3x2_cvt(ce0);
                a0[3] = e4m3x2_cvt(ce0 >> 16);
                a1[0] = e4m3x2_cvt(ab1);
                a1[1] = e4m3x2_cvt(ab1 >> 16);
                a1[2] = e4m3x2_cvt(ce1);
                a1[3] = e4m3x2_cvt(ce1 >> 16);
                mma_f16_16816(o[2 * q4][0], a0, pb[u][0][0], pb[u][0][1]);
                mma_f16_16816(o[2 * q4 + 1][0], a1, pb[u][0][0], pb[u][0][1]);
                if (two) {
                    mma_f16_16816(o[2 * q4][1], a0, pb[u][1][0], pb[u][1][1]);
                    mma_f16_16816(o[2 * q4 + 1][1], a1, pb[u][1][0], pb[u][1][1]);
                }
            }
        }
        // release the stages to the producer
        __syncwarp();
        if (lane == 0)
#pragma unroll
            for (int u = 0; u < NU; ++u)
                mbar_arrive(c.empty0 + 8 * st[u]);
    };

    for (uint32_t k = 0;;) {
        const uint32_t st0 = k % S;
        if (!wait_warp(c.full0 + 8 * st0, (k / S) & 1u))
            break;
        const StageMeta m = c.meta[st0];
        if (m.n_seq < 0)
            break;  // sentinel: the producer's walk is over
        const int kvh = m.kvh0 + w;
        if (m.first) {
            const uint32_t stage = c.sbase + st0 * L::kStage;
            rows = m.n_seq * a.G;
            two = rows > 8;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int r = nt * 8 + g;
                uint4 x[4];
                if (r < rows && m.qslot) {
                    const int srow = w * a.G + r;
                    const uint32_t qs = stage + 2 * L::kChunk + (t >> 1) * L::kQHalf + srow * 128;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        x[cc] = ld_shared_v4(qs + (((4 * (t & 1) + cc) ^ (srow & 7)) << 4));
                } else if (r < rows) {
                    const uint16_t *q = a.q + (int64_t)(m.seq_begin + r / a.G) * a.q_sb +
                                        (int64_t)(kvh * a.G + r % a.G) * a.q_sh + 32 * t;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        x[cc] = __ldg(reinterpret_cast<const uint4 *>(q) + cc);
                } else {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        x[cc] = make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    qb[2 * cc][nt][0] = pack_f16x2(bf16lo_to_f32(x[cc].x), bf16lo_to_f32(x[cc].y));
                    qb[2 * cc][nt][1] = pack_f16x2(bf16hi_to_f32(x[cc].x), bf16hi_to_f32(x[cc].y));
                    qb[2 * cc + 1][nt][0] = pack_f16x2(bf16lo_to_f32(x[cc].z), bf16lo_to_f32(x[cc].w));
                    qb[2 * cc + 1][nt][1] = pack_f16x2(bf16hi_to_f32(x[cc].z), bf16hi_to_f32(x[cc].w));
                }
            }
#pragma unroll
            for (int j = 0; j < kMt; ++j)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    o[j][nt][0] = o[j][nt][1] = o[j][nt][2] = o[j][nt][3] = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
                mq[nt][0] = mq[nt][1] = -INFINITY, lq[nt][0] = lq[nt][1] = 0.f;
            vref = 0.f;
        }
        // a long item's chunk that is not its last: its successor is in the
        // next stage
        const bool pair = m.pairs && !m.last;
        const uint32_t st[2] = {st0, (k + 1) % S};
        if (pair && !wait_warp(c.full0 + 8 * st[1], ((k + 1) / S) & 1u))
            break;
        const bool last = pair ? c.meta[st[1]].last : m.last;
        if (pair)
            pass(Int<2>{}, st);
        else
            pass(Int<1>{}, st);
        k += pair ? 2u : 1u;

        if (last) {
            const int base = m.part_row + w * rows;  // this head's rows
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                if (nt == 1 && !two)
                    break;
                float Lq[2] = {lq[nt][0], lq[nt][1]};
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    Lq[0] += __shfl_xor_sync(0xffffffffu, Lq[0], off);
                    Lq[1] += __shfl_xor_sync(0xffffffffu, Lq[1], off);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int r = nt * 8 + 2 * t + i;
                    if (r >= rows)
                        continue;
                    const float inv = Lq[i] > 0.f ? vref / Lq[i] : 0.f;
                    // columns 16g + 2j (element i) and 16g + 2j + 1 (element 2 + i) of m-tile j
                    uint32_t pk[8];
#pragma unroll
                    for (int j = 0; j < kMt; ++j)
                        pk[j] = pack_bf16x2(o[j][nt][i] * inv, o[j][nt][2 + i] * inv);
                    uint4 *dst = reinterpret_cast<uint4 *>(a.part_o + (size_t)(base + r) * D + 16 * g);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    if (g == 0)
                        a.part_lse[base + r] = Lq[i] > 0.f ? (mq[nt][i] + fast_log2(Lq[i])) * kLn2 : -INFINITY;
                }
            }
        }
    }
}

// ------------------------------------------------------ Parallel Prompting
// The rows of hp_stream_decode (Read Once, Answer Many, Section 3): one KV
// row per request holds the document, the questions and the interleaved
// answers; each key carries a stream id (-1 for the document) and a
// position, and a query of stream s at position p sees key k iff
// pos[k] <= p and (sid[k] = -1 or sid[k] = s) (Eq. 2).  Consumer warp w of
// an item serves KV head w / n_sg of the item's nh heads and the group of
// ns_pg streams (w % n_sg); the group's 16 query rows see each chunk
// through the mask.  A stage holds SC consecutive chunks of the row (SC *
// nh <= NC head boxes), so that an item of few heads still keeps the ring's
// bytes in flight and each warp has SC independent chunks per pass: chunk c
// of a stage occupies head slots c * nh .. c * nh + nh - 1 of each column
// half, its stream ids sit at mask + 64c and its positions at mask + 512 +
// 64c.

// Producer warp of the rows: as `producer`, a stage per SC chunks.  All 32
// lanes call it.
template <int D, int NC, int S, int SC, class Src>
__device__ __forceinline__ void producer_rows(const Ctx &c, const Args &a, const Src &src, int n_items, int lane)
{
    using L = Layout<D, NC, S, 0, false, true>;
    constexpr int kHalves = D / 64;
    constexpr int kBoxes = 2 * kHalves;  // K and V boxes of one chunk
    static_assert(SC >= 1 && 32 % SC == 0 && SC * kBoxes <= 16 && SC <= 8, "lanes and mask slots");
    auto wait_warp = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, c.status, c.abort)) != 0;
    };
    uint32_t k = 0;  // stages issued
    bool ok = true;
    bool prefetched = false;
    for (int it = 0; ok && it < n_items; ++it) {
        const Desc d = src(it, 0);
        if (!d.valid)
            continue;
        if (!prefetched && lane == 0) {
            prefetch_tensormap(d.map_k);
            prefetch_tensormap(d.map_v);
            prefetched = true;
        }
        const int nchunks = (d.k1 - d.k0 + kChunk - 1) / kChunk;
        int pg = 0;
        for (int ch0 = 0; ch0 < nchunks; ch0 += SC, ++k) {
            if ((ch0 & 31) == 0) {  // page ids of the next 32 chunks, one per lane
                const int cc = ch0 + lane;
                pg = cc < nchunks ? d.pages[(d.k0 + cc * kChunk) / d.ps - d.pbase] : 0;
            }
            const uint32_t st = k % S;
            if (k >= (uint32_t)S && !(ok = wait_warp(c.empty0 + 8 * st, ((k / S) - 1) & 1u)))
                break;
            const int n_sub = min(SC, nchunks - ch0);
            // lane u < n_sub: the page of chunk u of the stage
            const int cp = __shfl_sync(0xffffffffu, pg, (ch0 + lane) & 31);
            const unsigned oob =
                __ballot_sync(0xffffffffu, lane < n_sub && (unsigned)cp >= (unsigned)d.num_pages);
            const int t0 = d.k0 + ch0 * kChunk;
            const uint32_t bar = c.full0 + 8 * st;
            const uint32_t stage = c.sbase + st * L::kStage;
            if (lane == 0) {
                if (oob)
                    atomicOr(c.status, kStBounds);
                StageMeta m{};
                m.seq_begin = d.seq_begin;
                m.n_seq = d.n_seq;
                m.kvh0 = d.kvh0;
                m.part_row = d.part_row;
                m.nvalid = min(SC * kChunk, d.k1 - t0);
                m.first = ch0 == 0;
                m.last = ch0 + SC >= nchunks;
                m.oob = (int)oob;
                c.meta[st] = m;
                mbar_arrive_expect_tx(bar, (uint32_t)n_sub * (kBoxes * a.nh * L::kHeadBox + 128));
            }
            __syncwarp();
            // lanes 0 .. n_sub * kBoxes - 1: the K and V boxes of chunk
            // lane / kBoxes; lanes 16 .. 16 + 2 n_sub - 1: its ids / positions
            const int bu = lane < 16 ? lane / kBoxes : (lane - 16) >> 1;
            int page = __shfl_sync(0xffffffffu, cp, bu < SC ? bu : 0);
            if ((oob >> bu) & 1u)
                page = d.num_pages;  // zero-filled boxes, chunk masked
            if (lane < n_sub * kBoxes) {
                const int b = lane % kBoxes, h = b % kHalves;
                const bool is_v = b >= kHalves;
                tma_load_4d_h(stage + (is_v ? L::kChunk : 0) + h * L::kHalf + bu * a.nh * L::kHeadBox,
                              is_v ? d.map_v : d.map_k, bar, h * 64, (t0 + bu * kChunk) % d.ps, d.kvh0, page,
                              l2_evict_first());
            } else if (lane >= 16 && lane < 16 + 2 * n_sub) {
                const bool is_pos = (lane - 16) & 1;
                const uint32_t mk = stage + 2 * L::kChunk + L::kQSlot + L::kScales;
                bulk_load_h(mk + (is_pos ? 512 : 0) + 64 * bu, (is_pos ? d.slot_pos : d.slot_sid) + t0 + bu * kChunk,
                            64, bar, l2_evict_first());
            }
        }
    }
    // sentinel stage
    {
        const uint32_t st = k % S;
        if (k >= (uint32_t)S)
            wait_warp(c.empty0 + 8 * st, ((k / S) - 1) & 1u);
        if (lane == 0) {
            StageMeta m{};
            m.n_seq = -1;
            c.meta[st] = m;
            mbar_arrive(c.full0 + 8 * st);
        }
        __syncwarp();
        ++k;
    }
    // every copy issued has landed before the role ends
    if (lane == 0)
        for (uint32_t j = k > (uint32_t)S ? k - S : 0; j < k; ++j)
            mbar_wait_drain(c.full0 + 8 * (j % S), (j / S) & 1u);
}

// Consumer warp w of the rows (w < nh * n_sg).  Per stage: S = Q K^T for
// each of its SC chunks (independent MMA chains), the mask and the scale,
// one online-softmax update over the stage's 16 SC keys, then P V per chunk.
template <int D, int NC, int S, int SC>
__device__ __forceinline__ void consumer_rows(const Ctx &c, const Args &a, int w, int lane)
{
    using L = Layout<D, NC, S, 0, false, true>;
    constexpr int kHalves = D / 64;
    constexpr int kKs = D / 16;  // k-steps of the S MMA
    constexpr int kNt = D / 8;   // n8 tiles of O
    auto wait_warp = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, c.status, c.abort)) != 0;
    };
    uint32_t qa[kKs][4];
    float o[kNt][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int r0 = lane >> 2, r1 = r0 + 8;
    const int tq = 2 * (lane & 3);
    const int hw = w / a.n_sg;  // head of the item's group
    const int sj = w % a.n_sg;  // stream group
    int qsid0 = 0, qsid1 = 0, qpos0 = 0, qpos1 = 0;  // rows r0 / r1's stream and position
    int rows = 0;
    for (uint32_t k = 0;; ++k) {
        const uint32_t st = k % S;
        if (!wait_warp(c.full0 + 8 * st, (k / S) & 1u))
            break;
        const StageMeta m = c.meta[st];
        if (m.n_seq < 0)
            break;  // sentinel: the producer's walk is over
        const int seq0 = m.seq_begin + sj * a.ns_pg;
        rows = max(0, min(a.ns_pg, m.n_seq - sj * a.ns_pg)) * a.G;
        if (m.first) {
            // new item: query fragments (A operand, rows r0 / r1), their
            // streams and positions, and the state
            const int kvh = m.kvh0 + hw;
            const uint16_t *q0 = nullptr, *q1 = nullptr;
            if (r0 < rows)
                q0 = a.q + (int64_t)(seq0 + r0 / a.G) * a.q_sb + (int64_t)(kvh * a.G + r0 % a.G) * a.q_sh;
            if (r1 < rows)
                q1 = a.q + (int64_t)(seq0 + r1 / a.G) * a.q_sb + (int64_t)(kvh * a.G + r1 % a.G) * a.q_sh;
            qsid0 = r0 < rows ? __ldg(a.q_sid + seq0 + r0 / a.G) : 0;
            qpos0 = r0 < rows ? __ldg(a.q_pos + seq0 + r0 / a.G) : 0;
            qsid1 = r1 < rows ? __ldg(a.q_sid + seq0 + r1 / a.G) : 0;
            qpos1 = r1 < rows ? __ldg(a.q_pos + seq0 + r1 / a.G) : 0;
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
        const uint32_t stage = c.sbase + st * L::kStage;
        const uint32_t mk = stage + 2 * L::kChunk + L::kQSlot + L::kScales;
        int valid[SC];  // valid keys of each chunk
        bool zeroed = false;
#pragma unroll
        for (int u = 0; u < SC; ++u) {
            valid[u] = ((m.oob >> u) & 1) ? 0 : max(0, min(kChunk, m.nvalid - u * kChunk));
            if (valid[u] < kChunk) {
                // rows past the valid keys (or a chunk the stage does not
                // hold): zero this head's V so that 0 * (whatever the stage
                // holds there) stays 0
                uint8_t *vp = c.smem + (stage - c.sbase) + L::kChunk + (u * a.nh + hw) * L::kHeadBox;
                const int nz = (kChunk - valid[u]) * 8 * kHalves;
                for (int i = lane; i < nz; i += 32) {
                    const int row = valid[u] + i / (8 * kHalves);
                    const int rem = i % (8 * kHalves);
                    const int h = rem >> 3, ch = rem & 7;
                    *reinterpret_cast<uint4 *>(vp + h * L::kHalf + row * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                zeroed = true;
            }
        }
        if (zeroed) {
            fence_proxy_async_smem();
            __syncwarp();
        }

        // The stream mask first (rows r0: elements 0,1; rows r1: elements
        // 2,3; key of tile t, element e: 8t + tq + (e & 1)): a chunk that no
        // query row of this warp sees (another stream group's question or
        // answer tokens) costs the warp no MMA.
        bool see[SC][2][4];
        bool vis_all = true;
        unsigned vis = 0;
#pragma unroll
        for (int u = 0; u < SC; ++u) {
            bool any = false;
#pragma unroll
            for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int key = tile * 8 + tq + j;
                    const int sid = ld_shared_s32(mk + 64 * u + 4 * key);
                    const int pos = ld_shared_s32(mk + 512 + 64 * u + 4 * key);
                    const bool in = key < valid[u];
                    see[u][tile][j] = in && pos <= qpos0 && (sid == -1 || sid == qsid0);
                    see[u][tile][2 + j] = in && pos <= qpos1 && (sid == -1 || sid == qsid1);
                    any = any || see[u][tile][j] || see[u][tile][2 + j];
                }
            const bool v = __any_sync(0xffffffffu, any);
            vis |= (unsigned)v << u;
            vis_all = vis_all && v;
        }

        // S = Q K^T per chunk: n8 tile 0 = keys 0-7, tile 1 = keys 8-15
        float x[SC][2][4];
        {
            const int mi = lane >> 3, ri = lane & 7;
            const int tok = ri + ((mi >> 1) << 3);
#pragma unroll
            for (int u = 0; u < SC; ++u)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    x[u][0][e] = x[u][1][e] = 0.f;
            auto s_chunk = [&](int u, int ks) {
                const int dch = 2 * ks + (mi & 1);
                const uint32_t kst = stage + (u * a.nh + hw) * L::kHeadBox;
                const uint32_t addr = kst + (dch >> 3) * L::kHalf + tok * 128 + (((dch & 7) ^ (tok & 7)) << 4);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(addr, b0, b1, b2, b3);
                mma_bf16_16816(x[u][0], qa[ks], b0, b1);
                mma_bf16_16816(x[u][1], qa[ks], b2, b3);
            };
            if (vis_all) {  // every chunk: interleaved MMA chains
#pragma unroll
                for (int ks = 0; ks < kKs; ++ks)
#pragma unroll
                    for (int u = 0; u < SC; ++u)
                        s_chunk(u, ks);
            } else {
#pragma unroll
                for (int u = 0; u < SC; ++u)
                    if ((vis >> u) & 1u)
#pragma unroll
                        for (int ks = 0; ks < kKs; ++ks)
                            s_chunk(u, ks);
            }
        }
        // scale and mask
        const float cs = a.scale_log2;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int u = 0; u < SC; ++u) {
#pragma unroll
            for (int tile = 0; tile < 2; ++tile) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    x[u][tile][e] = see[u][tile][e] ? x[u][tile][e] * cs : -INFINITY;
                mx0 = fmax3(mx0, x[u][tile][0], x[u][tile][1]);
                mx1 = fmax3(mx1, x[u][tile][2], x[u][tile][3]);
            }
        }
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
        // the row sums take the weights before their rounding to bf16 for
        // P V (the LSE keeps f32 accuracy)
        uint32_t pa[SC][4];
#pragma unroll
        for (int u = 0; u < SC; ++u) {
            float p[2][4];
#pragma unroll
            for (int tile = 0; tile < 2; ++tile)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    p[tile][e] = fast_exp2(x[u][tile][e] - (e < 2 ? ms0 : ms1));
            pa[u][0] = pack_bf16x2(p[0][0], p[0][1]);
            pa[u][1] = pack_bf16x2(p[0][2], p[0][3]);
            pa[u][2] = pack_bf16x2(p[1][0], p[1][1]);
            pa[u][3] = pack_bf16x2(p[1][2], p[1][3]);
            l0 += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
            l1 += (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
        }

        // O += P V, chunk by chunk (the chunks this warp sees)
        {
            const int mi = lane >> 3, ri = lane & 7;
            const int tok = ri + ((mi & 1) << 3);
            auto pv_chunk = [&](int u, int dp) {
                const int dch = 2 * dp + (mi >> 1);
                const uint32_t vst = stage + L::kChunk + (u * a.nh + hw) * L::kHeadBox;
                const uint32_t addr = vst + (dch >> 3) * L::kHalf + tok * 128 + (((dch & 7) ^ (tok & 7)) << 4);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(addr, b0, b1, b2, b3);
                mma_bf16_16816(o[2 * dp], pa[u], b0, b1);
                mma_bf16_16816(o[2 * dp + 1], pa[u], b2, b3);
            };
            if (vis_all) {
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp)
#pragma unroll
                    for (int u = 0; u < SC; ++u)
                        pv_chunk(u, dp);
            } else {
#pragma unroll
                for (int u = 0; u < SC; ++u)
                    if ((vis >> u) & 1u)
#pragma unroll
                        for (int dp = 0; dp < D / 16; ++dp)
                            pv_chunk(u, dp);
            }
        }
        // release the stage to the producer
        __syncwarp();
        if (lane == 0)
            mbar_arrive(c.empty0 + 8 * st);

        if (m.last) {
            float L0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
            L0 += __shfl_xor_sync(0xffffffffu, L0, 2);
            float L1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
            L1 += __shfl_xor_sync(0xffffffffu, L1, 2);
            const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f;
            const float inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
            const int base = m.part_row + w * a.ns_pg * a.G;  // this warp's rows
            if (r0 < rows) {
                uint16_t *dst = a.part_o + (size_t)(base + r0) * D + tq;
#pragma unroll
                for (int n = 0; n < kNt; ++n)
                    *reinterpret_cast<uint32_t *>(dst + n * 8) = pack_bf16x2(o[n][0] * inv0, o[n][1] * inv0);
                if ((lane & 3) == 0)
                    a.part_lse[base + r0] = L0 > 0.f ? (m0 + fast_log2(L0)) * kLn2 : -INFINITY;
            }
            if (r1 < rows) {
                uint16_t *dst = a.part_o + (size_t)(base + r1) * D + tq;
#pragma unroll
                for (int n = 0; n < kNt; ++n)
                    *reinterpret_cast<uint32_t *>(dst + n * 8) = pack_bf16x2(o[n][2] * inv1, o[n][3] * inv1);
                if ((lane & 3) == 0)
                    a.part_lse[base + r1] = L1 > 0.f ? (m1 + fast_log2(L1)) * kLn2 : -INFINITY;
            }
        }
    }
}

}  // namespace smr
}  // namespace hp
