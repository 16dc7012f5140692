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
//
// Three instantiations: the static step, the decode loop's (Loop = true),
// in which suffix items end at the sequences' current lengths on the device
// and, with the append fused, the paged producer writes each sequence's new
// token into its suffix pages before it loads that chunk, and the static
// step over trees whose paged levels hold E4M3 codes (Q8 = true, d = 128:
// the paged role's ring then holds 5 stages of half-size chunks).
#include <cuda_runtime.h>

#include "hp_internal.h"
#include "hp_ptx.cuh"
#include "hp_small_role.cuh"
#include "hp_tc_role.cuh"

namespace hp {

namespace {

constexpr int kThreads = tcr::kThreads;
constexpr int kNC = 8;  // paged-role consumer warps (warps 4..11)
constexpr int kQRows = 32;  // paged-role Q slot rows per stage: nh * G <= 32

// Q8: the paged role reads E4M3 pools (half-size chunks, more stages)
template <int D, bool Q8>
struct FusedLayout {
    static constexpr int kSmallStages = Q8 ? 5 : 3;
    using T = tcr::Layout<D>;
    using S = smr::Layout<D, kNC, kSmallStages, kQRows, Q8>;
    static constexpr int kRing = T::kEnd > S::kEnd ? T::kEnd : S::kEnd;
    static constexpr int kTcBar = kRing;           // tcr::B_COUNT barriers, tmem slot, abort (256 bytes)
    static constexpr int kSmBar = kTcBar + 256;    // full[S], empty[S]
    static constexpr int kMeta = kSmBar + 128;     // StageMeta[S]
    static constexpr int kZero = kMeta + 256;      // 16 zero bytes, then the paged role's abort flag
    static constexpr int kRecBar = kZero + 32;     // the record's barrier
    static constexpr int kRec = kRecBar + 32;      // the CTA record
    static constexpr int kBytes = kRec + kRecMaxBytes;
    static_assert(tcr::kBarAbort + 4 <= 256, "tensor-core barrier area");
    static_assert(2 * kSmallStages * 8 <= 128, "paged barriers");
    static_assert(kSmallStages * (int)sizeof(smr::StageMeta) <= 256, "stage metadata");
    static_assert(kRec % 16 == 0, "bulk copy destination");
};

__device__ __forceinline__ const CUtensorMap *level_maps(const CascadeParams &p, int level)
{
    return reinterpret_cast<const CUtensorMap *>(p.plan + kPlanMapsOff) + level * kMapsPerLevel;
}

__device__ __forceinline__ tcr::ItemGeo tc_geo(const CascadeParams &p, const RecItem &it, const int32_t *pages)
{
    tcr::ItemGeo g;
    g.seq_begin = it.seq_begin;
    g.n_seq = it.n_seq;
    g.kvh = it.kvh;
    g.k0 = it.k0;
    g.k1 = it.k1;
    g.part_row = it.part_row;
    g.spb = kTcTile / p.G;
    g.paged = 1;
    g.ps = it.ps;
    g.box = it.box;
    g.num_pages = it.num_pages;
    g.pages = pages + it.page_off;
    g.map_k = level_maps(p, it.level) + 0;
    g.map_v = level_maps(p, it.level) + 1;
    g.map_q = &p.q_tc;
    return g;
}

// The paged items of this CTA's record.  In a decode loop a suffix item's
// key range ends at its sequence's current length (at most the planned end,
// which is the capacity for the suffix's last item).  A length that leaves
// the item empty or passes the capacity is reported; the item then keeps one
// key, inside its reserved pages, so the step stays in bounds.
// Loop: the decode-loop instantiation (lengths on the device, the append
// possibly fused); the static step's instantiation carries none of that code.
template <bool Loop, bool Q8>
struct RecordItems {
    static constexpr bool kPrefetch = Loop, kTokens = Loop;
    const CascadeParams *p;
    const RecItem *items;  // the record's paged items
    const int32_t *pages;  // the record's page list
    // a suffix item's current length (decode loops), loaded ahead
    __device__ int prefetch(int k) const
    {
        if (!Loop || k < 0 || p->suffix_len == nullptr)
            return 0;
        const int s = items[k].len_seq;
        return s >= 0 ? p->suffix_len[s] : 0;
    }
    __device__ smr::Desc operator()(int k, int pre_len) const
    {
        const RecItem w = items[k];
        smr::Desc d;
        d.seq_begin = w.seq_begin;
        d.n_seq = w.n_seq;
        d.kvh0 = w.kvh;
        d.k0 = w.k0;
        d.k1 = w.k1;
        if (Loop && w.len_seq >= 0 && p->suffix_len) {
            const int len = pre_len;
            // with the append fused, the step's own token is key `len`
            const bool app = p->k_new != nullptr && len >= 0 && len < p->loop_capacity;
            const int n = app ? len + 1 : len;
            d.k1 = min(w.k1, n);
            if (d.k1 <= w.k0 || n > p->loop_capacity || (p->k_new != nullptr && !app)) {
                atomicOr(p->status, kStBounds);
                d.k1 = max(d.k1, w.k0 + 1);
            }
            if (app && len >= w.k0 && len < w.k1) {
                const int pid = pages[w.page_off + len / w.ps - w.k0 / w.ps];
                if ((unsigned)pid < (unsigned)w.num_pages) {
                    const int64_t dst = (((int64_t)pid * p->Hkv + w.kvh) * w.ps + len % w.ps) * (int64_t)p->d;
                    d.tok_k_src = p->k_new + (int64_t)w.len_seq * p->kv_sb + (int64_t)w.kvh * p->kv_sh;
                    d.tok_v_src = p->v_new + (int64_t)w.len_seq * p->kv_sb + (int64_t)w.kvh * p->kv_sh;
                    d.tok_k_dst = p->loop_k_pool + dst;
                    d.tok_v_dst = p->loop_v_pool + dst;
                    d.tok_src_sh = p->kv_sh;
                    d.tok_dst_sh = (int64_t)w.ps * p->d;
                }
            }
        }
        d.part_row = w.part_row;
        d.pages = pages + w.page_off;
        d.pbase = w.k0 / w.ps;
        d.ps = w.ps;
        d.num_pages = w.num_pages;
        d.map_k = level_maps(*p, w.level) + 2;
        d.map_v = level_maps(*p, w.level) + 3;
        if (Q8) {
            d.k_scale = p->k_scale[w.level];
            d.v_scale = p->v_scale[w.level];
            d.Hkv = p->Hkv;
        }
        d.valid = d.k0 < d.k1;
        return d;
    }
};

template <int D, bool Loop, bool Q8>
__global__ void __launch_bounds__(kThreads, 1) hp_cascade_kernel(const __grid_constant__ CascadeParams p)
{
    using FL = FusedLayout<D, Q8>;
    constexpr int kSmallStages = FL::kSmallStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // let the merge kernel launch as soon as every CTA has started; it waits
    // for this grid to finish before reading the partial states
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    tcr::Ctx tc;
    tc.smem = smem;
    tc.sbase = smem_u32(smem);
    tc.bar0 = tc.sbase + FL::kTcBar;
    tc.tmem_slot = reinterpret_cast<uint32_t *>(smem + FL::kTcBar + tcr::kBarTmemSlot);
    tc.abort = reinterpret_cast<volatile int *>(smem + FL::kTcBar + tcr::kBarAbort);
    tc.status = p.status;
    const tcr::Args ta{p.G, p.scale_log2, &p.o_tc, p.part_lse};

    smr::Ctx sc;
    sc.smem = smem;
    sc.sbase = tc.sbase;
    sc.full0 = tc.sbase + FL::kSmBar;
    sc.empty0 = sc.full0 + kSmallStages * 8;
    sc.meta = reinterpret_cast<smr::StageMeta *>(smem + FL::kMeta);
    sc.zero16 = tc.sbase + FL::kZero;
    sc.abort = reinterpret_cast<volatile int *>(smem + FL::kZero + 16);
    sc.status = p.status;
    const smr::Args sa{p.q,  p.q_sb,          p.q_sh,   p.q_slot ? &p.q_sm : nullptr, p.G, p.small_nh,
                       p.scale_log2, p.part_o, p.part_lse};

    const uint32_t rec_bar = tc.sbase + FL::kRecBar;
    const RecHead *rec = reinterpret_cast<const RecHead *>(smem + FL::kRec);
    if (tid == 0) {
        // the record first: everything else of the CTA's work depends on it
        mbar_init(rec_bar, 1);
        tcr::init_barriers(tc, false);
        for (int s = 0; s < kSmallStages; ++s) {
            mbar_init(sc.full0 + 8 * s, 1);
            mbar_init(sc.empty0 + 8 * s, (uint32_t)p.small_nh);
        }
        *sc.abort = 0;
        fence_mbar_init();
        mbar_arrive_expect_tx(rec_bar, (uint32_t)p.rec_stride);
        // evict_last: the plan is re-read every step, the pools stream through
        bulk_load_h(tc.sbase + FL::kRec, p.plan + kPlanRecOff + (size_t)blockIdx.x * p.rec_stride,
                    (uint32_t)p.rec_stride, rec_bar, l2_evict_last());
    } else if (tid == 32) {
        prefetch_tensormap(&p.q_tc);
        prefetch_tensormap(&p.o_tc);
        if (p.q_slot)
            prefetch_tensormap(&p.q_sm);
        for (int l = 0; l < p.num_levels; ++l)
            for (int m = 0; m < kMapsPerLevel; ++m)
                prefetch_tensormap(level_maps(p, l) + m);
    } else if (tid >= 64 && tid < 68) {
        reinterpret_cast<uint32_t *>(smem + FL::kZero)[tid - 64] = 0u;
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tc.tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tc.tmem_slot;
    // This grid may start before the kernel ahead of it in the stream has
    // finished (programmatic dependent launch).  Only the set-up above and
    // the record load (plan memory, written by uploads alone) come before
    // this point; q, the pools and the workspace are touched after it.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // the record: its tag must match the launch's, its contents its size
    bool good = mbar_wait(rec_bar, 0u, p.status, tc.abort);
    int n_tc = 0, n_small = 0;
    if (good) {
        n_tc = rec->n_tc;
        n_small = rec->n_small;
        good = rec->tag == p.tag && n_tc >= 0 && n_small >= 0 &&
               (int64_t)sizeof(RecHead) + (int64_t)sizeof(RecItem) * (n_tc + n_small) + 4 * (int64_t)rec->n_pages <=
                   p.rec_stride;
        if (!good && tid == 0)
            atomicOr(p.status, kStPlan);
    }
    if (!good) {
        n_tc = 0;
        n_small = 0;
    }
    const RecItem *items = reinterpret_cast<const RecItem *>(rec + 1);
    const int32_t *pages = reinterpret_cast<const int32_t *>(items + n_tc + n_small);

    if (warp < 4) {
        setmaxnreg_dec<tcr::kRegsCtl>();
        for (int i = 0; i < n_tc; ++i) {
            const tcr::ItemGeo g = tc_geo(p, items[i], pages);
            if (i > 0) {
                // barriers of the previous item: re-initialise before any wait
                if (tid == 0)
                    tcr::init_barriers(tc, true);
                __syncwarp();
            }
            if (warp == 0 && tcr::item_ok(g))
                tcr::producer_prologue<D>(tc, g, ta, lane, p.withhold != 0 && blockIdx.x == 0 && i == 0);
            if (i > 0) {
                fence_proxy_async_smem();
                tcr::named_sync(0, kThreads);
            }
            if (tcr::item_ok(g)) {
                if (warp == 0)
                    tcr::producer_loop<D>(tc, g, lane);
                else if (warp == 1 && lane == 0)
                    tcr::mma_loop<D>(tc, g, tmem);
            } else if (tid == 0) {
                atomicOr(p.status, kStPlan);
            }
            __syncwarp();
            tc_fence_before();
            tcr::named_sync(0, kThreads);
        }
        // (a CTA without paged items skips the role: its code is not fetched
        // at the end of the step's longest chain)
        if (warp == 0 && n_small > 0)
            smr::producer<D, kNC, kSmallStages, kQRows, RecordItems<Loop, Q8>, Q8>(
                sc, sa, RecordItems<Loop, Q8>{&p, items + n_tc, pages}, n_small, lane);
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
    } else {
        setmaxnreg_inc<tcr::kRegsSoftmax>();
        for (int i = 0; i < n_tc; ++i) {
            const tcr::ItemGeo g = tc_geo(p, items[i], pages);
            if (i > 0)
                tcr::named_sync(0, kThreads);
            if (tcr::item_ok(g))
                tcr::softmax_loop<D>(tc, g, ta, tmem, warp, lane, tid);
            // the epilogue wrote shared memory that TMA refills next
            fence_proxy_async_smem();
            tc_fence_before();
            tcr::named_sync(0, kThreads);
        }
        if (warp - 4 < p.small_nh && n_small > 0) {
            if constexpr (Q8)
                smr::consumer_q8<D, kNC, kSmallStages, kQRows>(sc, sa, warp - 4, lane);
            else
                smr::consumer<D, kNC, kSmallStages, kQRows>(sc, sa, warp - 4, lane);
        }
    }
    __syncwarp();
}

template <int D, bool Loop, bool Q8>
cudaError_t launch_cascade_d(const CascadeParams &p, int grid, cudaStream_t s)
{
    static DeviceOnce once;  // per instantiation and device
    const int bytes = FusedLayout<D, Q8>::kBytes + 1024;
    static_assert(FusedLayout<D, Q8>::kBytes + 1024 <= 227 * 1024, "shared memory per CTA");
    cudaError_t e = once.run([bytes] {
        cudaError_t r =
            cudaFuncSetAttribute(hp_cascade_kernel<D, Loop, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (r != cudaSuccess)
            return r;
        cudaFuncAttributes fa;
        if ((r = cudaFuncGetAttributes(&fa, hp_cascade_kernel<D, Loop, Q8>)) != cudaSuccess)
            return r;
        // the register split assumes this allocation
        return fa.numRegs == (int)tcr::kRegsLaunch ? cudaSuccess : cudaErrorInvalidConfiguration;
    });
    if (e != cudaSuccess)
        return e;
    // launched as a programmatic dependent: the CTAs may set up (barriers,
    // TMEM, the record) while the previous kernel in the stream drains; the
    // kernel waits for that kernel to complete before it reads its inputs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, hp_cascade_kernel<D, Loop, Q8>, p);
}

}  // namespace

int cascade_q_rows() { return kQRows; }

int cascade_heads_per_item(int Hkv)
{
    return Hkv % 8 == 0 ? 8 : (Hkv % 4 == 0 ? 4 : (Hkv % 2 == 0 ? 2 : 1));
}

cudaError_t launch_cascade(const CascadeParams &p, int grid, int d, cudaStream_t s)
{
    if (grid <= 0)
        return cudaSuccess;
    if (p.q8)
        return d == 128 && p.suffix_len == nullptr ? launch_cascade_d<128, false, true>(p, grid, s)
                                                   : cudaErrorInvalidValue;
    if (p.suffix_len != nullptr)
        return d == 64 ? launch_cascade_d<64, true, false>(p, grid, s) : launch_cascade_d<128, true, false>(p, grid, s);
    return d == 64 ? launch_cascade_d<64, false, false>(p, grid, s) : launch_cascade_d<128, false, false>(p, grid, s);
}

}  // namespace hp
