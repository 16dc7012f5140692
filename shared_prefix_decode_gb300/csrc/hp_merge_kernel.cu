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

// Partial row of entry e of output row (b, h); returns -1 past the end.
struct PartList {
    int n;
    int base;    // plan mode: CSR begin
    int b, kvh, g;
};

__device__ __forceinline__ int part_row(const MergeParams &p, const PartList &L, int e)
{
    if (p.plan != nullptr)
        return __ldg(plan_array<int32_t>(p.plan, p.plan->off_merge_idx) + L.base + e) + L.g;
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
    if (p.plan != nullptr) {
        if (p.plan->magic != kPlanMagic || p.plan->tag != p.tag) {
            if (lane == 0)
                atomicOr(p.status, kStPlan);
            return;
        }
        const int32_t *mptr = plan_array<int32_t>(p.plan, p.plan->off_merge_ptr);
        L.base = __ldg(mptr + L.b * p.Hkv + L.kvh);
        L.n = __ldg(mptr + L.b * p.Hkv + L.kvh + 1) - L.base;
    } else if (p.mode == 1) {
        int len = __ldg(p.seq_lens + L.b);
        len = max(0, len);
        L.n = min(p.n_split, (len + p.split_len - 1) / p.split_len);
        L.base = 0;
    } else {
        L.n = p.n_split;
        L.base = 0;
    }
    // Everything above depends on the plan alone: when launched as a
    // dependent of the kernel that writes the partial states, it overlaps that
    // kernel's tail, and so does the lookup of this lane's first two parts.
    const int pr_a = lane < L.n ? part_row(p, L, lane) : 0;
    const int pr_b = lane + 32 < L.n ? part_row(p, L, lane + 32) : 0;
    if (p.wait_prior)
        asm volatile("griddepcontrol.wait;" ::: "memory");  // the partial states are complete
    auto row_of = [&](int e) { return e == lane ? pr_a : (e == lane + 32 ? pr_b : part_row(p, L, e)); };

    // Lanes own parts e = lane, lane + 32, ...: gather their rows and LSEs in
    // parallel, then the weighted sum walks the parts in their fixed order
    // with the row loads of 8 parts in flight at a time.
    float M = -INFINITY;
    for (int e = lane; e < L.n; e += 32)
        M = fmaxf(M, __ldg(p.part_lse + row_of(e)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i)
        acc[i] = 0.f;
    float den = 0.f;
    if (M != -INFINITY) {
        for (int e0 = 0; e0 < L.n; e0 += 32) {
            const int e = e0 + lane;
            int pr = 0;
            float w = 0.f;
            if (e < L.n) {
                pr = row_of(e);
                w = fast_exp2((__ldg(p.part_lse + pr) - M) * kLog2e);
            }
            den += w;
            const int cnt = min(32, L.n - e0);
            for (int k0 = 0; k0 < cnt; k0 += 8) {
                float wk[8];
                float v[8][VPT];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int kk = min(k0 + k, 31);
                    wk[k] = __shfl_sync(0xffffffffu, w, kk);
                    const int prk = __shfl_sync(0xffffffffu, pr, kk);
                    if (k0 + k < cnt) {
                        const float *src = p.part_o + (size_t)prk * p.d + lane * VPT;
                        if (VPT == 4) {
                            const float4 x = __ldg(reinterpret_cast<const float4 *>(src));
                            v[k][0] = x.x;
                            v[k][1] = x.y;
                            v[k][2] = x.z;
                            v[k][3] = x.w;
                        } else {
                            const float2 x = __ldg(reinterpret_cast<const float2 *>(src));
                            v[k][0] = x.x;
                            v[k][1] = x.y;
                        }
                    } else {
                        wk[k] = 0.f;
#pragma unroll
                        for (int i = 0; i < VPT; ++i)
                            v[k][i] = 0.f;
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k)
#pragma unroll
                    for (int i = 0; i < VPT; ++i)
                        acc[i] += wk[k] * v[k][i];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            den += __shfl_xor_sync(0xffffffffu, den, o);
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

cudaError_t launch_merge(const MergeParams &p, int64_t out_rows, cudaStream_t s)
{
    if (out_rows <= 0)
        return cudaSuccess;
    const int64_t grid = (out_rows + kMergeWarps - 1) / kMergeWarps;
    if (p.d == 128)
        hp_merge_kernel<4><<<(unsigned)grid, kMergeWarps * 32, 0, s>>>(p);
    else
        hp_merge_kernel<2><<<(unsigned)grid, kMergeWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_merge_dependent(const MergeParams &p_in, int64_t out_rows, cudaStream_t s)
{
    if (out_rows <= 0)
        return cudaSuccess;
    MergeParams p = p_in;
    p.wait_prior = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((out_rows + kMergeWarps - 1) / kMergeWarps));
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.d == 128)
        return cudaLaunchKernelEx(&cfg, hp_merge_kernel<4>, p);
    return cudaLaunchKernelEx(&cfg, hp_merge_kernel<2>, p);
}

cudaError_t launch_merge2(const float *oa, const float *la, const float *ob, const float *lb, void *o,
                          int out_f32, float *lse, int64_t rows, int d, cudaStream_t s)
{
    if (rows <= 0)
        return cudaSuccess;
    const int64_t grid = (rows + kMergeWarps - 1) / kMergeWarps;
    hp_merge2_kernel<<<(unsigned)grid, kMergeWarps * 32, 0, s>>>(oa, la, ob, lb, o, out_f32, lse, rows, d);
    return cudaGetLastError();
}

}  // namespace hp
