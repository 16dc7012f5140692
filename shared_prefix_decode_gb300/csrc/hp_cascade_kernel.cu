// hp_cascade_kernel.cu -- one persistent launch for the whole cascade step
// (except the merge): every CTA (one per SM) runs the work items the host
// planner scheduled on it -- first its shared-node items on the tensor cores
// (hp_tc_role.cuh: the batched prefix pass of Hydragen's "Inter-Sequence
// Batched Prefix Attention", split along keys as in ChunkAttention's
// chunk-first phase), then its paged items (hp_small_role.cuh: the per
// sequence pass of ChunkAttention's sequence-first phase).  The schedule is a
// longest-first greedy assignment computed on the host from the tree, so the
// prefix pass is spread over many SMs (each SM's TMA engine bounds what one
// SM can pull in small boxes) while the other SMs stream suffixes, and all
// SMs stream suffixes once their prefix work is done.
//
// 384 threads: warpgroup 0 = TMA producer (warp 0), MMA issuer (warp 1), two
// helpers; warpgroups 1-2 = softmax warps of the tensor-core role, and the 8
// consumer warps of the paged role.  The paged role's ring overlays the
// tensor-core role's shared memory once that role is done.
//
// Every partial (O, LSE) row goes to the workspace; the merge kernel, launched
// as a programmatic dependent of this one, combines them.
#include <cuda_runtime.h>

#include "hp_internal.h"
#include "hp_ptx.cuh"
#include "hp_small_role.cuh"
#include "hp_tc_role.cuh"

namespace hp {

namespace {

constexpr int kThreads = tcr::kThreads;
constexpr int kNC = 8;  // paged-role consumer warps (warps 4..11)
constexpr int kSmallStages = 3;

template <int D>
struct FusedLayout {
    using T = tcr::Layout<D>;
    using S = smr::Layout<D, kNC, kSmallStages>;
    static constexpr int kRing = T::kEnd > S::kEnd ? T::kEnd : S::kEnd;
    static constexpr int kTcBar = kRing;           // tcr::B_COUNT barriers, then tmem slot, abort
    static constexpr int kSmBar = kTcBar + 256;    // full[S], empty[S]
    static constexpr int kMeta = kSmBar + 64;      // StageMeta[S], then abort
    static constexpr int kPages = kMeta + 256;     // tcr::kMaxBoxes page ids
    static constexpr int kBytes = kPages + 4 * tcr::kMaxBoxes;
    static_assert(2 * kSmallStages * 8 <= 64, "small barriers");
    static_assert(kSmallStages * (int)sizeof(smr::StageMeta) + 4 <= 256, "stage metadata");
};

__device__ __forceinline__ tcr::ItemGeo tc_geo(const PlanHeader *ph, int idx)
{
    const WorkItem it = plan_array<WorkItem>(ph, ph->off_tc)[idx];
    const LevelDev &lv = ph->levels[it.level];
    const CUtensorMap *maps = plan_array<CUtensorMap>(ph, ph->off_maps);
    tcr::ItemGeo g;
    g.seq_begin = it.seq_begin;
    g.n_seq = it.n_seq;
    g.kvh = it.kvh;
    g.k0 = it.k0;
    g.k1 = it.k1;
    g.pages = plan_array<int32_t>(ph, ph->off_page_ids) + it.page_base;
    g.part_row = it.part_row;
    g.paged = 1;
    g.ps = lv.page_size;
    g.box = lv.tc_box;
    g.num_pages = lv.num_pages;
    g.map_k = maps + it.level * kMapsPerLevel + 0;
    g.map_v = maps + it.level * kMapsPerLevel + 1;
    return g;
}

// This CTA's paged items: entries of its schedule after its tensor-core items.
struct PlanSmallItems {
    const PlanHeader *ph;
    const int32_t *list;  // schedule entries (small items numbered after the tensor-core ones)
    __device__ smr::Desc operator()(int k) const
    {
        const WorkItem w = plan_array<WorkItem>(ph, ph->off_small)[list[k] - ph->n_tc];
        const LevelDev &lv = ph->levels[w.level];
        const CUtensorMap *maps = plan_array<CUtensorMap>(ph, ph->off_maps);
        smr::Desc d;
        d.seq_begin = w.seq_begin;
        d.n_seq = w.n_seq;
        d.kvh0 = w.kvh;
        d.k0 = w.k0;
        d.k1 = w.k1;
        d.part_row = w.part_row;
        d.pages = plan_array<int32_t>(ph, ph->off_page_ids) + w.page_base;
        d.ps = lv.page_size;
        d.num_pages = lv.num_pages;
        d.map_k = maps + w.level * kMapsPerLevel + 2;
        d.map_v = maps + w.level * kMapsPerLevel + 3;
        d.valid = d.k0 < d.k1;
        return d;
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) hp_cascade_kernel(const __grid_constant__ CascadeParams p)
{
    using FL = FusedLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const PlanHeader *ph = p.plan;
    if (ph->magic != kPlanMagic || ph->tag != p.tag || (int)gridDim.x != ph->grid) {
        if (tid == 0)
            atomicOr(p.status, kStPlan);
        return;  // uniform across the CTA
    }
    // let the merge kernel launch as soon as every CTA has started; it waits
    // for this grid to finish before reading the partial states
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int32_t *cta_ptr = plan_array<int32_t>(ph, ph->off_cta_ptr);
    const int32_t *cta_ntc = plan_array<int32_t>(ph, ph->off_cta_ntc);
    const int32_t *cta_items = plan_array<int32_t>(ph, ph->off_cta_items);
    const int beg = __ldg(cta_ptr + blockIdx.x);
    const int end = __ldg(cta_ptr + blockIdx.x + 1);
    const int n_tc = __ldg(cta_ntc + blockIdx.x);
    const int n_small = end - beg - n_tc;

    tcr::Ctx tc;
    tc.smem = smem;
    tc.sbase = smem_u32(smem);
    tc.bar0 = tc.sbase + FL::kTcBar;
    tc.tmem_slot = reinterpret_cast<uint32_t *>(smem + FL::kTcBar + 128);
    tc.abort = reinterpret_cast<volatile int *>(smem + FL::kTcBar + 132);
    tc.s_pages = reinterpret_cast<int32_t *>(smem + FL::kPages);
    tc.status = p.status;
    const tcr::Args ta{p.q, p.q_sb, p.q_sh, ph->G, p.scale_log2, p.part_o, p.part_lse};

    smr::Ctx sc;
    sc.smem = smem;
    sc.sbase = tc.sbase;
    sc.full0 = tc.sbase + FL::kSmBar;
    sc.empty0 = sc.full0 + kSmallStages * 8;
    sc.meta = reinterpret_cast<smr::StageMeta *>(smem + FL::kMeta);
    sc.abort = reinterpret_cast<volatile int *>(smem + FL::kMeta + kSmallStages * sizeof(smr::StageMeta));
    sc.status = p.status;
    const smr::Args sa{p.q, p.q_sb, p.q_sh, ph->G, ph->small_nh, p.scale_log2, p.part_o, p.part_lse};

    if (tid == 0) {
        for (int s = 0; s < kSmallStages; ++s) {
            mbar_init(sc.full0 + 8 * s, 1);
            mbar_init(sc.empty0 + 8 * s, (uint32_t)ph->small_nh);
        }
        *sc.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp < 4) {
        setmaxnreg_dec<tcr::kRegsCtl>();
        uint32_t tmem = 0;
        for (int i = 0; i < n_tc; ++i) {
            const tcr::ItemGeo g = tc_geo(ph, __ldg(cta_items + beg + i));
            if (warp == 0)
                tcr::producer_prologue<D>(tc, g, i > 0, lane);
            else {
                if (warp == 1 && i == 0) {
                    tmem_alloc(smem_u32(tc.tmem_slot), 512);
                    tmem_relinquish();
                }
                tcr::stage_q<D, kThreads - 32>(tc, g, ta, tid - 32);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            tcr::named_sync(0, kThreads);
            tc_fence_after();
            tmem = *tc.tmem_slot;
            if (warp == 0)
                tcr::producer_loop<D>(tc, g, lane);
            else if (warp == 1 && lane == 0)
                tcr::mma_loop<D>(tc, g, ph->G, tmem);
            __syncwarp();
            tc_fence_before();
            tcr::named_sync(0, kThreads);
        }
        if (n_tc > 0 && warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
        if (warp == 0)
            smr::producer<D, kNC, kSmallStages>(sc, sa, PlanSmallItems{ph, cta_items + beg + n_tc}, n_small, lane);
    } else {
        setmaxnreg_inc<tcr::kRegsSoftmax>();
        for (int i = 0; i < n_tc; ++i) {
            const tcr::ItemGeo g = tc_geo(ph, __ldg(cta_items + beg + i));
            tcr::stage_q<D, kThreads - 32>(tc, g, ta, tid - 32);
            fence_proxy_async_smem();
            tc_fence_before();
            tcr::named_sync(0, kThreads);
            tc_fence_after();
            const uint32_t tmem = *tc.tmem_slot;
            tcr::softmax_loop<D>(tc, g, ta, tmem, warp, lane, tid);
            // the epilogue wrote shared memory that TMA refills next
            fence_proxy_async_smem();
            tc_fence_before();
            tcr::named_sync(0, kThreads);
        }
        if (warp - 4 < ph->small_nh)
            smr::consumer<D, kNC, kSmallStages>(sc, sa, warp - 4, lane);
    }
    __syncwarp();
}

template <int D>
cudaError_t launch_cascade_d(const CascadeParams &p, int grid, cudaStream_t s)
{
    static bool configured = false;
    const int bytes = FusedLayout<D>::kBytes + 1024;
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(hp_cascade_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess)
            return e;
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, hp_cascade_kernel<D>)) != cudaSuccess)
            return e;
        if (fa.numRegs != (int)tcr::kRegsLaunch)
            return cudaErrorInvalidConfiguration;  // the register split assumes this allocation
        configured = true;
    }
    hp_cascade_kernel<D><<<grid, kThreads, bytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

int cascade_heads_per_item(int Hkv)
{
    return Hkv % 8 == 0 ? 8 : (Hkv % 4 == 0 ? 4 : (Hkv % 2 == 0 ? 2 : 1));
}

cudaError_t launch_cascade(const CascadeParams &p, int grid, int d, cudaStream_t s)
{
    if (grid <= 0)
        return cudaSuccess;
    return d == 64 ? launch_cascade_d<64>(p, grid, s) : launch_cascade_d<128>(p, grid, s);
}

}  // namespace hp
