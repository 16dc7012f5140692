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
#include "hp_merge_row.cuh"
#include "hp_ptx.cuh"

namespace hp {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
// One warp (one output row) per CTA: a CTA's resources are released as soon
// as its row is merged (with four rows per CTA the step measured 0.37 us
// longer on the Llama-3-8B shape).
constexpr int kMergeWarps = 1;

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
    if (p.mode == 3) {
        // stream-row items (request, head group, stream block, split); rows
        // [warp (head in group, stream group)][stream in group][g]
        const int r = L.b / p.P, sidx = L.b % p.P;
        const int sb = sidx / p.spi, si = sidx % p.spi;
        const int groups = p.Hkv / p.nh;
        const int item = ((r * groups + L.kvh / p.nh) * p.n_sblk + sb) * p.n_split + e;
        const int w = (L.kvh % p.nh) * p.n_sg + si / p.ns_pg;
        return item * p.rows_item + (w * p.ns_pg + si % p.ns_pg) * p.G + L.g;
    }
    // mode 2: contiguous prefix items (rc, kvh, split) of two 128-row blocks
    const int rel = L.b - p.row_begin;
    const int rc = rel / p.seqs_per_item, sl = rel % p.seqs_per_item;
    const int item = (rc * p.Hkv + L.kvh) * p.n_split + e;
    return (int)tc_part_row((int64_t)item * 2 * kTcTile, sl, L.g, p.G);
}

template <int VPT>  // values per lane: d / 32
__global__ void __launch_bounds__(kMergeWarps * 32) hp_merge_kernel(const __grid_constant__ MergeParams p)
{
    // a following cascade launch may start its set-up on the SMs this grid
    // frees; it waits for this grid to complete before it touches memory
    // this kernel reads or writes
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
        if (p.mode == 1 || p.mode == 3) {
            int len = __ldg(p.seq_lens + (p.mode == 3 ? L.b / p.P : L.b));
            len = max(0, len);
            L.n = min(p.n_split, (len + p.split_len - 1) / p.split_len);
        } else {
            L.n = p.n_split;
        }
        pr_a = lane < L.n ? part_row(p, L, lane) : 0;
        pr_b = lane + 32 < L.n ? part_row(p, L, lane + 32) : 0;
    }
    if (p.wait_prior)
        asm volatile("griddepcontrol.wait;" ::: "memory");  // the partial states are complete
    if (p.len_inc != nullptr && h == 0 && lane == 0) {
        // the step appended its token: the suffix is one longer from now on
        const int len = p.len_inc[L.b];
        if (len >= 0 && len < p.len_capacity)
            p.len_inc[L.b] = len + 1;
    }
    const size_t esz = p.out_f32 ? 4 : 2;
    mrg::RowOut o;
    o.out = static_cast<uint8_t *>(p.out) + ((int64_t)L.b * p.o_sb + (int64_t)h * p.o_sh) * esz;
    o.out_f32 = p.out_f32;
    o.lse = p.lse != nullptr ? p.lse + (int64_t)L.b * p.lse_sb + h : nullptr;
    if (L.trow != nullptr) {
        // parts past the first 64: straight from the table row
        const int32_t *trow = L.trow;
        const int g = L.g;
        mrg::merge_row<VPT * 32, 8>(p.part_o, p.part_lse, L.n, pr_a, pr_b,
                                    [trow, g](int e) { return __ldg(trow + 1 + e) + g; }, lane, o);
    } else {
        mrg::merge_row<VPT * 32, 8>(p.part_o, p.part_lse, L.n, pr_a, pr_b,
                                    [&p, L](int e) { return part_row(p, L, e); }, lane, o);
    }
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
    static DeviceOnce once;
    return once.run([] {
        cudaError_t r = cudaFuncSetAttribute(hp_merge_kernel<4>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             (int)cudaSharedmemCarveoutMaxShared);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(hp_merge_kernel<2>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(hp_merge2_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);

        return r;
    });
}

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
