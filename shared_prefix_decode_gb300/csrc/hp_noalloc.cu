// hp_noalloc.cu -- paged decode for callers that cannot allocate device
// memory.
//
// hp_suffix_decode_paged needs a caller-provided workspace for its partial
// (O, LSE) states.  Some callers have no way to provide one: a host program or
// plugin that reaches this library only through its C ABI and has no device
// allocator of its own, code running where a caching allocator already owns
// all device memory so that cudaMalloc would fail, or a latency-critical path
// that must not pay for cudaMalloc's implicit device synchronisation.  This
// file gives them hp_suffix_decode_paged_noalloc, which keeps its scratch in a
// fixed device array that is part of the library itself.
//
// The array below is created when the library's device code is loaded and
// stays resident on every GPU that loads it until the process exits.  Its
// device address is looked up (cudaGetSymbolAddress, with the device
// current) during the first call in each CUDA context -- the first call on a
// device, and again after cudaDeviceReset has replaced that device's context
// and the array may have moved.  Every call shares the one array, so calls
// that run at the same time on the GPU (on different streams, or from
// different host threads) overwrite each other's partial states: serialise
// them.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "hp_host.h"
#include "hp_internal.h"

namespace {

// Largest scratch this entry point uses: the device status word plus the
// partial rows of one call.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_hp_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_lock;
struct ScratchAddr {
    unsigned long long ctx_id;  // the CUDA context the address belongs to (0: none yet)
    void *ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

// Unique id of the current CUDA context (ids are never reused), via the
// driver entry points the runtime hands out; 0 if it cannot be read.
unsigned long long current_context_id()
{
    static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
        cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array in the current device's context,
// looked up once per context.  Returns nullptr if the lookup failed.
void *scratch_on_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    // (before the first runtime call on a device its context may not exist
    // yet: id 0, and the lookup below creates it)
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> g(g_setup_lock);
    ScratchAddr &a = g_scratch[dev];
    if (a.ptr == nullptr || ctx == 0 || a.ctx_id != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_hp_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            a.ptr = nullptr;
            return nullptr;
        }
        a.ptr = p;
        a.ctx_id = current_context_id();
    }
    return a.ptr;
}

}  // namespace

extern "C" hp_status hp_suffix_decode_paged_noalloc(const void *q, int64_t q_sb, int64_t q_sh, int32_t B,
                                                    const void *k_pool, const void *v_pool, int32_t num_pages,
                                                    int32_t page_size, const int32_t *page_table,
                                                    int32_t pt_stride, const int32_t *seq_lens, int32_t Hq,
                                                    int32_t Hkv, int32_t d, float scale, void *out,
                                                    hp_dtype out_dt, int64_t o_sb, int64_t o_sh, float *lse,
                                                    int64_t lse_sb, hp_stream_t stream)
{
    using namespace hp;
    if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !out)
        return HP_ERR_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || num_pages < 1 || pt_stride < 1 || !std::isfinite(scale))
        return HP_ERR_ARG;
    if ((d != 64 && d != 128) || page_size < 16 || page_size > 256 || page_size % 16 || Hq / Hkv > kSmallRows)
        return HP_ERR_UNSUPPORTED;
    if (out_dt != HP_BF16 && out_dt != HP_F32)
        return HP_ERR_ARG;
    const size_t esz = out_dt == HP_F32 ? 4 : 2;
    const size_t lane_bytes = esz * (size_t)(d / 32);
    if (!aligned(q, 16) || q_sb % 8 || q_sh % 8 || q_sb < 0 || q_sh < 0 || !aligned(out, lane_bytes) ||
        (o_sb * (int64_t)esz) % (int64_t)lane_bytes || (o_sh * (int64_t)esz) % (int64_t)lane_bytes ||
        !aligned(k_pool, 16) || !aligned(v_pool, 16))
        return HP_ERR_UNSUPPORTED;
    if ((int64_t)pt_stride * page_size > INT32_MAX)
        return HP_ERR_UNSUPPORTED;

    // Split each sequence into as few key ranges as fit the scratch: at
    // least 64 keys per range, and no more ranges than the scratch holds.
    // Each split needs B * Hq partial rows of 2d + 4 bytes (the bf16 O row
    // and its f32 LSE); one split fits while B * Hq <= 64,525 at d = 128
    // (127,096 at d = 64).
    const int max_len = pt_stride * page_size;
    const size_t per_row = (size_t)d * 2 + 4;  // partial O row (bf16) + its LSE
    const size_t avail = kNoAllocScratchBytes - 2 * kWsHeader;
    const int64_t rows_per_split = (int64_t)B * Hq;
    const int64_t max_splits = (int64_t)(avail / per_row) / rows_per_split;
    if (max_splits < 1)
        return HP_ERR_WORKSPACE;  // B * Hq partial rows exceed the fixed scratch
    int64_t split = 64;
    while (ceil_div(max_len, split) > max_splits)
        split *= 2;
    const int n_split = (int)ceil_div(max_len, split);
    const int64_t part_rows = rows_per_split * n_split;

    void *scratch = scratch_on_current_device();
    if (!scratch)
        return HP_ERR_CUDA;
    uint8_t *base = static_cast<uint8_t *>(scratch);
    const size_t off_lse = kWsHeader;
    const size_t off_o = round_up(off_lse + (size_t)part_rows * 4, 256);
    if (off_o + (size_t)part_rows * d * 2 > kNoAllocScratchBytes)
        return HP_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the status word is the only scratch that must start at zero
    if (cudaMemsetAsync(base, 0, sizeof(uint32_t), s) != cudaSuccess)
        return HP_ERR_CUDA;

    SmallParams sp;
    std::memset(&sp, 0, sizeof(sp));
    const int nh = small_heads_per_item(Hkv);
    if (!encode_pool_map(&sp.map_k, k_pool, num_pages, Hkv, page_size, d, kChunk, nh) ||
        !encode_pool_map(&sp.map_v, v_pool, num_pages, Hkv, page_size, d, kChunk, nh))
        return HP_ERR_CUDA;
    const int G = Hq / Hkv;
    // Q rows by TMA with each item's first chunk when the strides allow a
    // tensor map; the consumers read them themselves otherwise
    sp.q_slot = nh * G <= small_q_rows() && (B == 1 || q_sb > 0) && (Hq == 1 || q_sh > 0) &&
                encode_q_map(&sp.map_q, q, B, Hq, d, q_sb, q_sh, nh * G, 1);
    sp.q = static_cast<const uint16_t *>(q);
    sp.q_sb = q_sb;
    sp.q_sh = q_sh;
    sp.G = G;
    sp.Hkv = Hkv;
    sp.scale_log2 = scale * 1.4426950408889634f;
    sp.n_items = B * (Hkv / nh) * n_split;
    sp.nh = nh;
    sp.page_table = page_table;
    sp.pt_stride = pt_stride;
    sp.seq_lens = seq_lens;
    sp.B = B;
    sp.num_pages = num_pages;
    sp.page_size = page_size;
    sp.split_len = (int)split;
    sp.n_split = n_split;
    sp.part_o = reinterpret_cast<uint16_t *>(base + off_o);
    sp.part_lse = reinterpret_cast<float *>(base + off_lse);
    sp.status = reinterpret_cast<uint32_t *>(base);
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int per_sm = (int)std::max<size_t>(1, std::min<size_t>(4, (size_t)(227 * 1024) / small_smem_bytes(d)));
    const int grid = (int)std::min<int64_t>(sp.n_items, (int64_t)sms * per_sm);
    if (launch_small(sp, grid, d, s) != cudaSuccess)
        return HP_ERR_CUDA;

    MergeParams mp;
    std::memset(&mp, 0, sizeof(mp));
    mp.part_o = sp.part_o;
    mp.part_lse = sp.part_lse;
    mp.d = d;
    mp.G = G;
    mp.Hq = Hq;
    mp.Hkv = Hkv;
    mp.B = B;
    mp.plan = nullptr;
    mp.mode = 1;
    mp.seq_lens = seq_lens;
    mp.split_len = (int)split;
    mp.n_split = n_split;
    mp.nh = nh;
    mp.out = out;
    mp.out_f32 = out_dt == HP_F32;
    mp.o_sb = o_sb;
    mp.o_sh = o_sh;
    mp.lse = lse;
    mp.lse_sb = lse_sb;
    mp.status = sp.status;
    return launch_merge(mp, (int64_t)B * Hq, s) == cudaSuccess ? HP_OK : HP_ERR_CUDA;
}
