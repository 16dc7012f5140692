// hp_small_kernel.cu -- standalone paged decode (hp_suffix_decode_paged, its
// allocation-free variant, and hp_suffix_decode_paged_e4m3): the
// paged-decode role (hp_small_role.cuh) with one producer warp and four
// consumer warps per CTA; CTA c walks items c, c + grid, ... of (sequence,
// KV-head group, key split).  Q8: E4M3 pools with per-(page, KV head) scales.
// Also the Parallel Prompting row kernel (hp_stream_decode): the same role in
// its stream-mask mode, one producer and eight consumer warps per CTA.
#include <cuda_runtime.h>

#include "hp_internal.h"
#include "hp_ptx.cuh"
#include "hp_small_role.cuh"

namespace hp {

namespace {

constexpr int kConsumers = 4;
constexpr int kThreadsSmall = (kConsumers + 1) * 32;
constexpr int kQRows = 16;  // Q slot rows per stage: nh * G <= 16

// bf16 pools: 3 stages of 16-token chunks; E4M3 pools: 5 (half the bytes each)
template <int D, bool Q8>
struct SmallKernelLayout {
    static constexpr int kStages = Q8 ? 5 : 3;
    using R = smr::Layout<D, kConsumers, kStages, kQRows, Q8>;
    static constexpr int kBar = R::kEnd;
    static constexpr int kMeta = kBar + 2 * kStages * 8;
    static constexpr int kZero = kMeta + 256;  // 16 zero bytes, then the abort flag
    static constexpr int kBytes = kZero + 32;
    static_assert(kStages * (int)sizeof(smr::StageMeta) <= 256, "stage metadata");
};

// Items of the page-table form: idx -> (sequence, head group, split).
struct TableItems {
    const SmallParams *p;
    int first, stride;
    static constexpr bool kPrefetch = false, kTokens = false;
    __device__ int prefetch(int) const { return 0; }
    __device__ smr::Desc operator()(int k, int) const
    {
        const int idx = first + k * stride;
        smr::Desc d;
        const int split = idx % p->n_split;
        const int t = idx / p->n_split;
        const int groups = p->Hkv / p->nh;
        const int grp = t % groups;
        const int b = t / groups;
        int len = __ldg(p->seq_lens + b);
        const int cap = p->pt_stride * p->page_size;
        if (len < 0 || len > cap) {
            atomicOr(p->status, kStBounds);
            len = len < 0 ? 0 : cap;
        }
        d.seq_begin = b;
        d.n_seq = 1;
        d.kvh0 = grp * p->nh;
        d.k0 = split * p->split_len;
        d.k1 = min(d.k0 + p->split_len, len);
        d.part_row = idx * p->nh * p->G;
        d.pages = p->page_table + (int64_t)b * p->pt_stride;
        d.pbase = 0;
        d.ps = p->page_size;
        d.num_pages = p->num_pages;
        d.map_k = &p->map_k;
        d.map_v = &p->map_v;
        d.k_scale = p->k_scale;
        d.v_scale = p->v_scale;
        d.Hkv = p->Hkv;
        d.valid = d.k0 < d.k1;
        return d;
    }
};

template <int D, bool Q8>
__global__ void __launch_bounds__(kThreadsSmall) hp_small_kernel(const __grid_constant__ SmallParams p)
{
    using KL = SmallKernelLayout<D, Q8>;
    constexpr int kStages = KL::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    smr::Ctx c;
    c.smem = smem;
    c.sbase = smem_u32(smem);
    c.full0 = c.sbase + KL::kBar;
    c.empty0 = c.full0 + kStages * 8;
    c.meta = reinterpret_cast<smr::StageMeta *>(smem + KL::kMeta);
    c.zero16 = c.sbase + KL::kZero;
    c.abort = reinterpret_cast<volatile int *>(smem + KL::kZero + 16);
    c.status = p.status;
    smr::Args a{p.q, p.q_sb, p.q_sh, p.q_slot ? &p.map_q : nullptr, p.G, p.nh, p.scale_log2, p.part_o, p.part_lse};
    if (threadIdx.x < 4)
        reinterpret_cast<uint32_t *>(smem + KL::kZero)[threadIdx.x] = 0u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(c.full0 + 8 * s, 1);
            mbar_init(c.empty0 + 8 * s, (uint32_t)p.nh);
        }
        *c.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int n_items = p.n_items > (int)blockIdx.x ? (p.n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    if (warp == kConsumers)
        smr::producer<D, kConsumers, kStages, kQRows, TableItems, Q8>(
            c, a, TableItems{&p, (int)blockIdx.x, (int)gridDim.x}, n_items, lane);
    else if (warp < p.nh) {
        if constexpr (Q8)
            smr::consumer_q8<D, kConsumers, kStages, kQRows>(c, a, warp, lane);
        else
            smr::consumer<D, kConsumers, kStages, kQRows>(c, a, warp, lane);
    }
    __syncwarp();
}

// ------------------------------------------------ Parallel Prompting rows
// Read Once, Answer Many, Section 3: one KV row per request holds the
// document and every stream's question and answer tokens; the stream mask
// (Eq. 2) keeps each stream's query on the document and its own tokens.  An
// item is (request r, nh KV heads, a block of spi streams, a key range): the
// row's chunks are loaded once for all the block's streams, and consumer warp
// w computes head w / n_sg for streams (w % n_sg) * ns_pg .. of the block.
// Warpgroup 0: the producer warp (warp 0) and three idle warps, which give
// their registers to warpgroups 1 and 2: the eight consumer warps (4..11).
constexpr int kStreamConsumers = 8;
constexpr int kStreamThreads = 384;
constexpr uint32_t kStreamRegsLaunch = 168, kStreamRegsCtl = 56, kStreamRegsConsumer = 224;
static_assert(128 * kStreamRegsCtl + 256 * kStreamRegsConsumer == kStreamThreads * kStreamRegsLaunch,
              "register split");

// A stage holds NC head-chunks (SC chunks of nh heads, SC * nh = NC): the
// fewer the heads of an item, the smaller the stage and the more stages the
// ring holds (up to 8), so the bytes in flight stay about the same.
template <int D, int NC>
struct StreamKernelLayout {
    static constexpr int kStageBytes = smr::Layout<D, NC, 1, 0, false, true>::kStage;
    static constexpr int kStages = (200 * 1024 / kStageBytes) < 8 ? (200 * 1024 / kStageBytes) : 8;
    using R = smr::Layout<D, NC, kStages, 0, false, true>;
    static constexpr int kBar = R::kEnd;
    static constexpr int kMeta = kBar + 2 * kStages * 8;
    static constexpr int kZero = kMeta + 512;  // 16 zero bytes, then the abort flag
    static constexpr int kBytes = kZero + 32;
    static_assert(kStages >= 3 && kStages * (int)sizeof(smr::StageMeta) <= 512, "stage metadata");
};

struct StreamItems {
    const StreamParams *p;
    int first, stride;
    static constexpr bool kPrefetch = false, kTokens = false;
    __device__ int prefetch(int) const { return 0; }
    __device__ smr::Desc operator()(int k, int) const
    {
        const int idx = first + k * stride;
        smr::Desc d;
        const int split = idx % p->n_split;
        int t = idx / p->n_split;
        const int sb = t % p->n_sblk;
        t /= p->n_sblk;
        const int groups = p->Hkv / p->nh;
        const int grp = t % groups;
        const int r = t / groups;
        int len = __ldg(p->row_len + r);
        const int cap = p->pt_stride * p->page_size;
        if (len < 0 || len > cap) {
            atomicOr(p->status, kStBounds);
            len = len < 0 ? 0 : cap;
        }
        d.seq_begin = r * p->P + sb * p->spi;
        d.n_seq = min(p->spi, p->P - sb * p->spi);
        d.kvh0 = grp * p->nh;
        d.k0 = split * p->split_len;
        d.k1 = min(d.k0 + p->split_len, len);
        d.part_row = idx * p->rows_item;
        d.pages = p->row_pages + (int64_t)r * p->pt_stride;
        d.pbase = 0;
        d.ps = p->page_size;
        d.num_pages = p->num_pages;
        d.map_k = &p->map_k;
        d.map_v = &p->map_v;
        d.slot_sid = p->slot_sid + (int64_t)r * p->sid_stride;
        d.slot_pos = p->slot_pos + (int64_t)r * p->sid_stride;
        d.valid = d.k0 < d.k1;
        return d;
    }
};

template <int D, int SC, int NC>
__global__ void __launch_bounds__(kStreamThreads, 1) hp_stream_kernel(const __grid_constant__ StreamParams p)
{
    using KL = StreamKernelLayout<D, NC>;
    constexpr int kS = KL::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    smr::Ctx c;
    c.smem = smem;
    c.sbase = smem_u32(smem);
    c.full0 = c.sbase + KL::kBar;
    c.empty0 = c.full0 + kS * 8;
    c.meta = reinterpret_cast<smr::StageMeta *>(smem + KL::kMeta);
    c.zero16 = c.sbase + KL::kZero;
    c.abort = reinterpret_cast<volatile int *>(smem + KL::kZero + 16);
    c.status = p.status;
    smr::Args a{p.q, p.q_sb, p.q_sh, nullptr, p.G, p.nh, p.scale_log2, p.part_o, p.part_lse};
    a.n_sg = p.n_sg;
    a.ns_pg = p.ns_pg;
    a.q_sid = p.q_sid;
    a.q_pos = p.q_pos;
    const int n_warps = p.nh * p.n_sg;  // consumer warps of an item
    if (threadIdx.x < 4)
        reinterpret_cast<uint32_t *>(smem + KL::kZero)[threadIdx.x] = 0u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(c.full0 + 8 * s, 1);
            mbar_init(c.empty0 + 8 * s, (uint32_t)n_warps);
        }
        *c.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int n_items = p.n_items > (int)blockIdx.x ? (p.n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    if (warp < 4) {
        setmaxnreg_dec<kStreamRegsCtl>();
        if (warp == 0)
            smr::producer_rows<D, NC, kS, SC, StreamItems>(c, a, StreamItems{&p, (int)blockIdx.x, (int)gridDim.x},
                                                           n_items, lane);
    } else {
        setmaxnreg_inc<kStreamRegsConsumer>();
        if (warp - 4 < n_warps)
            smr::consumer_rows<D, NC, kS, SC>(c, a, warp - 4, lane);
    }
    __syncwarp();
}

template <int D, int SC, int NC>
cudaError_t launch_stream_d(const StreamParams &p, int grid, cudaStream_t s)
{
    static DeviceOnce once;  // per instantiation and device
    const int bytes = StreamKernelLayout<D, NC>::kBytes + 1024;
    static_assert(StreamKernelLayout<D, NC>::kBytes + 1024 <= 227 * 1024, "shared memory per CTA");
    cudaError_t e = once.run([bytes] {
        cudaError_t r =
            cudaFuncSetAttribute(hp_stream_kernel<D, SC, NC>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (r != cudaSuccess)
            return r;
        cudaFuncAttributes fa;
        if ((r = cudaFuncGetAttributes(&fa, hp_stream_kernel<D, SC, NC>)) != cudaSuccess)
            return r;
        // the register split assumes this allocation
        return fa.numRegs == (int)kStreamRegsLaunch ? cudaSuccess : cudaErrorInvalidConfiguration;
    });
    if (e != cudaSuccess)
        return e;
    hp_stream_kernel<D, SC, NC><<<grid, kStreamThreads, bytes, s>>>(p);
    return cudaGetLastError();
}

// (chunks per stage, heads per item) as the planner chooses them: up to 8
// head-chunks per stage, at most four chunks.
template <int D>
cudaError_t launch_stream_sc(const StreamParams &p, int grid, cudaStream_t s)
{
    const int nc = p.sc * p.nh;
    if (p.sc == 1 && nc == 8)
        return launch_stream_d<D, 1, 8>(p, grid, s);
    if (p.sc == 2 && nc == 8)
        return launch_stream_d<D, 2, 8>(p, grid, s);
    if (p.sc == 4 && nc == 8)
        return launch_stream_d<D, 4, 8>(p, grid, s);
    if (p.sc == 4 && nc == 4)
        return launch_stream_d<D, 4, 4>(p, grid, s);
    return cudaErrorInvalidValue;
}

template <int D, bool Q8>
cudaError_t launch_small_d(const SmallParams &p, int grid, cudaStream_t s)
{
    static DeviceOnce once;  // per instantiation and device
    const int bytes = SmallKernelLayout<D, Q8>::kBytes + 1024;
    cudaError_t e = once.run([bytes] {
        return cudaFuncSetAttribute(hp_small_kernel<D, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    });
    if (e != cudaSuccess)
        return e;
    hp_small_kernel<D, Q8><<<grid, kThreadsSmall, bytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stream(const StreamParams &p, int grid, int d, cudaStream_t s)
{
    if (grid <= 0)
        return cudaSuccess;
    if (p.sc * p.nh > kStreamConsumers)
        return cudaErrorInvalidValue;
    return d == 64 ? launch_stream_sc<64>(p, grid, s) : launch_stream_sc<128>(p, grid, s);
}

size_t small_smem_bytes(int d, bool q8)
{
    if (q8)
        return SmallKernelLayout<128, true>::kBytes + 1024;
    return d == 64 ? SmallKernelLayout<64, false>::kBytes + 1024 : SmallKernelLayout<128, false>::kBytes + 1024;
}

int small_q_rows() { return kQRows; }

int small_heads_per_item(int Hkv)
{
    return Hkv % 4 == 0 ? 4 : (Hkv % 2 == 0 ? 2 : 1);
}

cudaError_t launch_small(const SmallParams &p, int grid, int d, cudaStream_t s)
{
    if (grid <= 0)
        return cudaSuccess;
    if (p.q8)
        return d == 128 ? launch_small_d<128, true>(p, grid, s) : cudaErrorInvalidValue;
    return d == 64 ? launch_small_d<64, false>(p, grid, s) : launch_small_d<128, false>(p, grid, s);
}

}  // namespace hp
