// hp_tc_kernel.cu -- standalone batched prefix attention (hp_prefix_attn):
// one CTA per work item of the tensor-core role (hp_tc_role.cuh), items
// derived from the grid over a contiguous [len][Hkv][d] prefix.
#include <cuda_runtime.h>

#include "hp_internal.h"
#include "hp_ptx.cuh"
#include "hp_tc_role.cuh"

namespace hp {

namespace {

template <int D>
struct TcKernelLayout {
    using R = tcr::Layout<D>;
    static constexpr int kBar = R::kEnd;
    static constexpr int kBytes = kBar + 256;
};

// Item idx of a contiguous prefix: (row chunk, KV head, key split).
__device__ __forceinline__ tcr::ItemGeo contiguous_item(const TcParams &p, int idx)
{
    tcr::ItemGeo g;
    const int split = idx % p.imp_n_split;
    const int t = idx / p.imp_n_split;
    const int kvh = t % p.Hkv;
    const int rc = t / p.Hkv;
    g.seq_begin = p.imp_row_begin + rc * p.imp_seqs_per_item;
    g.n_seq = min(p.imp_seqs_per_item, p.imp_rows - rc * p.imp_seqs_per_item);
    g.kvh = kvh;
    g.k0 = split * p.imp_split_len;
    g.k1 = min(g.k0 + p.imp_split_len, p.imp_len);
    g.part_row = idx * 2 * kTcTile;
    g.spb = kTcTile / p.G;
    g.paged = 0;
    g.ps = 0;
    g.box = kTcTile;
    g.num_pages = 0;
    g.pages = nullptr;
    g.map_k = &p.map_k;
    g.map_v = &p.map_v;
    g.map_q = &p.map_q;
    return g;
}

template <int D>
__global__ void __launch_bounds__(tcr::kThreads, 1) hp_tc_kernel(const __grid_constant__ TcParams p)
{
    using KL = TcKernelLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    tcr::Ctx c;
    c.smem = smem;
    c.sbase = smem_u32(smem);
    c.bar0 = c.sbase + KL::kBar;
    c.tmem_slot = reinterpret_cast<uint32_t *>(smem + KL::kBar + tcr::kBarTmemSlot);
    c.abort = reinterpret_cast<volatile int *>(smem + KL::kBar + tcr::kBarAbort);
    c.status = p.status;
    const tcr::Args a{p.G, p.scale_log2, &p.map_o, p.part_lse};

    const tcr::ItemGeo g = contiguous_item(p, blockIdx.x);
    if (!tcr::item_ok(g)) {
        if (tid == 0)
            atomicOr(p.status, kStPlan);
        return;  // uniform across the CTA: nothing allocated yet
    }
    if (tid == 0) {
        tcr::init_barriers(c, false);
        prefetch_tensormap(g.map_q);
        prefetch_tensormap(g.map_k);
        prefetch_tensormap(g.map_v);
        prefetch_tensormap(&p.map_o);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(c.tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *c.tmem_slot;
    if (warp < 4) {
        setmaxnreg_dec<tcr::kRegsCtl>();
        if (warp == 0) {
            tcr::producer_prologue<D>(c, g, a, lane);
            tcr::producer_loop<D>(c, g, lane);
        } else if (warp == 1 && lane == 0) {
            tcr::mma_loop<D>(c, g, tmem);
        }
        __syncwarp();
        tc_fence_before();
        tcr::named_sync(0, tcr::kThreads);
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
    } else {
        setmaxnreg_inc<tcr::kRegsSoftmax>();
        tcr::softmax_loop<D>(c, g, a, tmem, warp, lane, tid);
        tc_fence_before();
        tcr::named_sync(0, tcr::kThreads);
    }
}

template <int D>
cudaError_t launch_tc_d(const TcParams &p, int grid, cudaStream_t s)
{
    static DeviceOnce once;  // per instantiation and device
    const int bytes = TcKernelLayout<D>::kBytes + 1024;
    cudaError_t e = once.run([bytes] {
        cudaError_t r = cudaFuncSetAttribute(hp_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (r != cudaSuccess)
            return r;
        // the register split assumes this launch allocation per thread
        cudaFuncAttributes fa;
        if ((r = cudaFuncGetAttributes(&fa, hp_tc_kernel<D>)) != cudaSuccess)
            return r;
        return fa.numRegs == (int)tcr::kRegsLaunch ? cudaSuccess : cudaErrorInvalidConfiguration;
    });
    if (e != cudaSuccess)
        return e;
    hp_tc_kernel<D><<<grid, tcr::kThreads, bytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t tc_smem_bytes(int d)
{
    return d == 64 ? TcKernelLayout<64>::kBytes + 1024 : TcKernelLayout<128>::kBytes + 1024;
}

cudaError_t launch_tc(const TcParams &p, int grid, int d, cudaStream_t s)
{
    if (grid <= 0)
        return cudaSuccess;
    return d == 64 ? launch_tc_d<64>(p, grid, s) : launch_tc_d<128>(p, grid, s);
}

}  // namespace hp
