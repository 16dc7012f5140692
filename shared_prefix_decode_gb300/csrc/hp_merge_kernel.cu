// hp_merge_kernel.cu -- exact log-sum-exp merge of partial attention states.
//
// Each output row (b, h) has a fixed, ordered list of partial states
// (O_i normalised over its own keys, LSE_i); the merge is Hydragen Eq. 5
// applied to all of them at once in its max-subtracted form (combine_lse):
//   M = max_i LSE_i;  w_i = e^(LSE_i - M);  O = sum_i w_i O_i / sum_i w_i;
//   LSE = M + ln sum_i w_i.
// An empty part has LSE = -inf and weight exactly 0; a row with no parts, or
// only empty ones, gets O = 0 and LSE = -inf.  The order of the parts is
// fixed by the plan, so results are deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "hp_internal.h"
#include "hp_ptx.cuh"

namespace hp {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMergeWarps = 4;
constexpr int kChunkParts = 16;  // parts of a row loaded together

// Partial row of entry e of output row (b, h).
struct PartList {
    int n;
    const int32_t *trow;  // plan mode: the (b, kvh) row of the merge table
    int b, kvh, g;
};

__device__ __forceinline__ int part_row(const MergeParams &p, const PartList &L, int e)
{
    if (p.plan != nullptr)
        return __ldg(L.trow + 1 + e) + L.g;
    if (p.mode == 1) {
        // small-kernel items (b, head group, split), rows (head in group, g)
        const int groups = p.Hkv / p.nh;
        const int item = ((L.b * groups + L.kvh / p.nh) * p.n_split + e);
        return (item * p.nh + L.kvh % p.nh) * p.G + L.g;
    }
    // mode 2: contiguous prefix items (rc, kvh, split) of two 128-row blocks
    const int rel = L.b - p.row_begin;
    const int rc = rel / p.seqs_per_item, sl = rel % p.seqs_per_item;
    const int item = (rc * p.Hkv + L.kvh) * p.n_split + e;
    return (int)tc_part_row((int64_t)item * 2 * kTcTile, sl, L.g, p.G);
}

template <int VPT>  // values per lane: d / 32
__global__ void __launch_bounds__(kMergeWarps * 32) hp_merge_kernel(const MergeParams p)
{
    // a kernel launched after this one as a programmatic dependent (the next
    // step's persistent kernel) may start its plan-only set-up meanwhile
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kMergeWarps + warp;
    const int64_t n_rows = (int64_t)p.B * p.Hq;
    if (row >= n_rows)
        return;
    PartList L;
    L.b = (int)(row / p.Hq);
    const int h = (int)(row % p.Hq);
    L.kvh = h / p.G;
    L.g = h % p.G;
    int pr_a = 0, pr_b = 0;
    if (p.plan != nullptr) {
        // the table row (count, then the parts) and the plan's identity in
        // one round of independent loads
        L.trow = p.tab + (size_t)(L.b * p.Hkv + L.kvh) * p.tab_stride;
        const uint32_t magic = p.plan->magic;
        const uint64_t tag = p.plan->tag;
        L.n = __ldg(L.trow);
        const int ea = lane + 1 < p.tab_stride ? __ldg(L.trow + 1 + lane) : 0;
        const int eb = lane + 33 < p.tab_stride ? __ldg(L.trow + 33 + lane) : 0;
        if (magic != kPlanMagic || tag != p.tag || L.n < 0 || L.n >= p.tab_stride) {
            if (lane == 0)
                atomicOr(p.status, kStPlan);
            return;
        }
        pr_a = ea + L.g;
        pr_b = eb + L.g;
    } else {
        L.trow = nullptr;
        if (p.mode == 1) {
            int len = __ldg(p.seq_lens + L.b);
            len = max(0, len);
            L.n = min(p.n_split, (len + p.split_len - 1) / p.split_len);
        } else {
            L.n = p.n_split;
        }
        pr_a = lane < L.n ? part_row(p, L, lane) : 0;
        pr_b = lane + 32 < L.n ? part_row(p, L, lane + 32) : 0;
    }
    // Everything above depends on the plan alone: when launched as a
    // dependent of the kernel that writes the partial states, it overlaps that
    // kernel's tail.
    if (p.wait_prior)
        asm volatile("griddepcontrol.wait;" ::: "memory");  // the partial states are complete

    // Online merge over chunks of up to kChunkParts parts: every LSE and O row
    // of a chunk is loaded before any is used (one memory round trip per
    // chunk), then the chunk joins the running state -- max M, denominator,
    // weighted sum, rescaled when M grows.  The parts are taken in their fixed
    // order, so the result is deterministic.  Every lane reads the same LSEs
    // and its own VPT columns of each O row.
    float M = -INFINITY, den = 0.f;
    float acc[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i)
        acc[i] = 0.f;
    for (int e0 = 0; e0 < L.n; e0 += kChunkParts) {
        const int cnt = min(kChunkParts, L.n - e0);
        float ls[kChunkParts];
        float v[kChunkParts][VPT];
#pragma unroll
        for (int k = 0; k < kChunkParts; ++k) {
            const int e = e0 + k;
            int pr = __shfl_sync(0xffffffffu, e < 32 ? pr_a : pr_b, e & 31);
            if (e >= 64 && k < cnt)
                pr = part_row(p, L, e);
            ls[k] = -INFINITY;
#pragma unroll
            for (int i = 0; i < VPT; ++i)
                v[k][i] = 0.f;
            if (k < cnt) {
                ls[k] = __ldg(p.part_lse + pr);
                const uint16_t *src = p.part_o + (size_t)pr * p.d + lane * VPT;  // bf16
                if (VPT == 4) {
                    const uint2 x = __ldg(reinterpret_cast<const uint2 *>(src));
                    v[k][0] = bf16lo_to_f32(x.x);
                    v[k][1] = bf16hi_to_f32(x.x);
                    v[k][2] = bf16lo_to_f32(x.y);
                    v[k][3] = bf16hi_to_f32(x.y);
                } else {
                    const uint32_t x = __ldg(reinterpret_cast<const uint32_t *>(src));
                    v[k][0] = bf16lo_to_f32(x);
                    v[k][1] = bf16hi_to_f32(x);
                }
            }
        }
        float mc = M;
#pragma unroll
        for (int k = 0; k < kChunkParts; ++k)
            mc = fmaxf(mc, ls[k]);
        if (mc == -INFINITY)
            continue;  // every part so far is empty
        const float sc = fast_exp2((M - mc) * kLog2e);  // 0 while M = -inf
        den *= sc;
#pragma unroll
        for (int i = 0; i < VPT; ++i)
            acc[i] *= sc;
#pragma unroll
        for (int k = 0; k < kChunkParts; ++k) {
            const float w = fast_exp2((ls[k] - mc) * kLog2e);  // 0 for an empty part
            den += w;
#pragma unroll
            for (int i = 0; i < VPT; ++i)
                acc[i] = fmaf(w, v[k][i], acc[i]);
        }
        M = mc;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int64_t off = (int64_t)L.b * p.o_sb + (int64_t)h * p.o_sh + lane * VPT;
    if (p.out_f32) {
        float *dst = reinterpret_cast<float *>(p.out) + off;
#pragma unroll
        for (int i = 0; i < VPT; ++i)
            dst[i] = acc[i] * inv;
    } else {
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + off;
#pragma unroll
        for (int i = 0; i < VPT; i += 2)
            *reinterpret_cast<__nv_bfloat162 *>(dst + i) = __floats2bfloat162_rn(acc[i] * inv, acc[i + 1] * inv);
    }
    if (lane == 0 && p.lse != nullptr)
        p.lse[(int64_t)L.b * p.lse_sb + h] = den > 0.f ? M + __logf(den) : -INFINITY;
}

// Grouped merge: one warp per kRowsPerWarp = 512 / D consecutive query heads
// of one KV head.  Those heads share their list of parts, and a part's rows
// for them are contiguous, so lane l owns 16 columns of row l / (32 /
// kRowsPerWarp): per part, one LSE and one 32-byte load per lane.  Same
// online merge and part order as hp_merge_kernel.
constexpr int kGroupWarps = 2;
constexpr int kGroupChunk = 16;

template <int D>
__global__ void __launch_bounds__(kGroupWarps * 32) hp_merge_group_kernel(const MergeParams p)
{
    constexpr int kRowsPerWarp = 512 / D, kLanesPerRow = 32 / kRowsPerWarp, kVals = D / kLanesPerRow;
    static_assert(kVals == 16, "16 columns per lane");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per_kvh = p.G / kRowsPerWarp;  // warps per (b, kvh)
    const int64_t gw = (int64_t)blockIdx.x * kGroupWarps + warp;
    if (gw >= (int64_t)p.B * p.Hkv * per_kvh)
        return;
    PartList L;
    L.b = (int)(gw / ((int64_t)p.Hkv * per_kvh));
    const int rem = (int)(gw % ((int64_t)p.Hkv * per_kvh));
    L.kvh = rem / per_kvh;
    const int g = (rem % per_kvh) * kRowsPerWarp + lane / kLanesPerRow;  // this lane's head in the group
    const int c0 = (lane % kLanesPerRow) * kVals;                       // and its first column
    L.g = 0;  // rows below are of head 0; each lane adds its own g
    int base_a = 0, base_b = 0;
    if (p.plan != nullptr) {
        L.trow = p.tab + (size_t)(L.b * p.Hkv + L.kvh) * p.tab_stride;
        const uint32_t magic = p.plan->magic;
        const uint64_t tag = p.plan->tag;
        L.n = __ldg(L.trow);
        base_a = lane + 1 < p.tab_stride ? __ldg(L.trow + 1 + lane) : 0;
        base_b = lane + 33 < p.tab_stride ? __ldg(L.trow + 33 + lane) : 0;
        if (magic != kPlanMagic || tag != p.tag || L.n < 0 || L.n >= p.tab_stride) {
            if (lane == 0)
                atomicOr(p.status, kStPlan);
            return;
        }
    } else {
        L.trow = nullptr;
        if (p.mode == 1) {
            int len = __ldg(p.seq_lens + L.b);
            len = max(0, len);
            L.n = min(p.n_split, (len + p.split_len - 1) / p.split_len);
        } else {
            L.n = p.n_split;
        }
        base_a = lane < L.n ? part_row(p, L, lane) : 0;
        base_b = lane + 32 < L.n ? part_row(p, L, lane + 32) : 0;
    }
    if (p.wait_prior)
        asm volatile("griddepcontrol.wait;" ::: "memory");  // the partial states are complete
    float M = -INFINITY, den = 0.f;
    float acc[kVals];
#pragma unroll
    for (int i = 0; i < kVals; ++i)
        acc[i] = 0.f;
    {
        for (int e0 = 0; e0 < L.n; e0 += kGroupChunk) {
            const int cnt = min(kGroupChunk, L.n - e0);
            float ls[kGroupChunk];
            uint4 v[kGroupChunk][2];
#pragma unroll
            for (int k = 0; k < kGroupChunk; ++k) {
                const int e = e0 + k;
                int pr = __shfl_sync(0xffffffffu, e < 32 ? base_a : base_b, e & 31);
                if (e >= 64 && k < cnt)
                    pr = part_row(p, L, e);
                pr += g;
                ls[k] = -INFINITY;
                v[k][0] = v[k][1] = make_uint4(0u, 0u, 0u, 0u);
                if (k < cnt) {
                    // L2 only (.cg): each partial row is read once
                    ls[k] = __ldcg(p.part_lse + pr);
                    const uint4 *src = reinterpret_cast<const uint4 *>(p.part_o + (size_t)pr * D + c0);
                    v[k][0] = __ldcg(src);
                    v[k][1] = __ldcg(src + 1);
                }
            }
            float mc = M;
#pragma unroll
            for (int k = 0; k < kGroupChunk; ++k)
                mc = fmaxf(mc, ls[k]);
            if (mc == -INFINITY)
                continue;  // every part so far is empty
            const float sc = fast_exp2((M - mc) * kLog2e);  // 0 while M = -inf
            den *= sc;
#pragma unroll
            for (int i = 0; i < kVals; ++i)
                acc[i] *= sc;
#pragma unroll
            for (int k = 0; k < kGroupChunk; ++k) {
                const float w = fast_exp2((ls[k] - mc) * kLog2e);  // 0 for an empty part
                den += w;
                const uint32_t x[8] = {v[k][0].x, v[k][0].y, v[k][0].z, v[k][0].w,
                                       v[k][1].x, v[k][1].y, v[k][1].z, v[k][1].w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    acc[2 * j] = fmaf(w, bf16lo_to_f32(x[j]), acc[2 * j]);
                    acc[2 * j + 1] = fmaf(w, bf16hi_to_f32(x[j]), acc[2 * j + 1]);
                }
            }
            M = mc;
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int h = L.kvh * p.G + g;
    const int64_t off = (int64_t)L.b * p.o_sb + (int64_t)h * p.o_sh + c0;
    if (p.out_f32) {
        float *dst = reinterpret_cast<float *>(p.out) + off;
#pragma unroll
        for (int j = 0; j < kVals; j += 2)
            *reinterpret_cast<float2 *>(dst + j) = make_float2(acc[j] * inv, acc[j + 1] * inv);
    } else {
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + off;
#pragma unroll
        for (int j = 0; j < kVals; j += 2)
            *reinterpret_cast<__nv_bfloat162 *>(dst + j) = __floats2bfloat162_rn(acc[j] * inv, acc[j + 1] * inv);
    }
    if (lane % kLanesPerRow == 0 && p.lse != nullptr)
        p.lse[(int64_t)L.b * p.lse_sb + h] = den > 0.f ? M + __logf(den) : -INFINITY;
}

// Two-state merge of arbitrary d: one warp per row.
__global__ void __launch_bounds__(kMergeWarps * 32)
    hp_merge2_kernel(const float *oa, const float *la, const float *ob, const float *lb, void *o, int out_f32,
                     float *lse, int64_t rows, int d)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kMergeWarps + warp;
    if (r >= rows)
        return;
    const float A = la[r], Bv = lb[r];
    const float M = fmaxf(A, Bv);
    float wa = 0.f, wb = 0.f;
    if (M != -INFINITY) {
        wa = fast_exp2((A - M) * kLog2e);
        wb = fast_exp2((Bv - M) * kLog2e);
    }
    const float den = wa + wb;
    const float inv = den > 0.f ? 1.f / den : 0.f;
    // every lane reads its inputs before any lane writes (in-place merges)
    for (int i = lane; i < d; i += 32) {
        const float x = oa[r * d + i], y = ob[r * d + i];
        const float v = (wa * x + wb * y) * inv;
        if (out_f32)
            reinterpret_cast<float *>(o)[r * d + i] = v;
        else
            reinterpret_cast<__nv_bfloat16 *>(o)[r * d + i] = __float2bfloat16_rn(v);
    }
    if (lane == 0 && lse != nullptr)
        lse[r] = den > 0.f ? M + __logf(den) : -INFINITY;
}

}  // namespace

// The merge kernels run between kernels that use (almost) all shared memory:
// keep the same carveout so the SMs need no reconfiguration in between.
static cudaError_t merge_configure()
{
    static const cudaError_t e = [] {
        cudaError_t r = cudaFuncSetAttribute(hp_merge_kernel<4>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             (int)cudaSharedmemCarveoutMaxShared);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(hp_merge_kernel<2>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(hp_merge2_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(hp_merge_group_kernel<128>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(hp_merge_group_kernel<64>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        return r;
    }();
    return e;
}

// The grouped kernel when a KV head's query heads split into whole warps of
// 512 / d heads; the per-row kernel otherwise.
static bool use_group(const MergeParams &p) { return (p.d == 128 && p.G % 4 == 0) || (p.d == 64 && p.G % 8 == 0); }

template <class K>
static cudaError_t launch_with(K kernel, const MergeParams &p, int64_t warps, int per_cta, bool dependent, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + per_cta - 1) / per_cta));
    cfg.blockDim = dim3(per_cta * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

static cudaError_t launch_merge_any(const MergeParams &p_in, int64_t out_rows, bool dependent, cudaStream_t s)
{
    if (out_rows <= 0)
        return cudaSuccess;
    if (cudaError_t e = merge_configure(); e != cudaSuccess)
        return e;
    MergeParams p = p_in;
    p.wait_prior = dependent ? 1 : 0;
    if (use_group(p)) {
        const int64_t warps = out_rows / (512 / p.d);
        return p.d == 128 ? launch_with(hp_merge_group_kernel<128>, p, warps, kGroupWarps, dependent, s)
                          : launch_with(hp_merge_group_kernel<64>, p, warps, kGroupWarps, dependent, s);
    }
    return p.d == 128 ? launch_with(hp_merge_kernel<4>, p, out_rows, kMergeWarps, dependent, s)
                      : launch_with(hp_merge_kernel<2>, p, out_rows, kMergeWarps, dependent, s);
}

cudaError_t launch_merge(const MergeParams &p, int64_t out_rows, cudaStream_t s)
{
    return launch_merge_any(p, out_rows, false, s);
}

cudaError_t launch_merge_dependent(const MergeParams &p, int64_t out_rows, cudaStream_t s)
{
    return launch_merge_any(p, out_rows, true, s);
}

cudaError_t launch_merge2(const float *oa, const float *la, const float *ob, const float *lb, void *o,
                          int out_f32, float *lse, int64_t rows, int d, cudaStream_t s)
{
    if (rows <= 0)
        return cudaSuccess;
    if (cudaError_t e = merge_configure(); e != cudaSuccess)
        return e;
    const int64_t grid = (rows + kMergeWarps - 1) / kMergeWarps;
    hp_merge2_kernel<<<(unsigned)grid, kMergeWarps * 32, 0, s>>>(oa, la, ob, lb, o, out_f32, lse, rows, d);
    return cudaGetLastError();
}

}  // namespace hp
