// hp_api.cu -- host side of the C ABI declared in include/hp.h: argument
// validation, TMA descriptor encoding, plan upload (the planner itself is
// hp_plan.cu), and the launches.  No entry point here allocates device
// memory or synchronises, except hp_cascade_plan (waits for its upload) and
// hp_read_device_status.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <numeric>
#include <queue>
#include <unordered_map>
#include <vector>

#include <cudaTypedefs.h>

#include "hp_host.h"
#include "hp_internal.h"
#include "hp_plan.h"

using namespace hp;

namespace {

constexpr int32_t kAbiVersion = 5;
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------- utilities


PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}


// Contiguous prefix: token t, head g at base + t*st + g*sh (elements);
// box = 64 columns x 1 head x 128 tokens.
bool encode_prefix_map(CUtensorMap *m, const void *base, int len, int Hkv, int d, int64_t st, int64_t sh)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hkv, (cuuint64_t)len};
    cuuint64_t strides[2] = {(cuuint64_t)sh * 2, (cuuint64_t)st * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kTcTile};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Partial O rows [rows][d] bf16 for the tensor-core role's stores: box 64
// columns x 128 rows, 128-byte swizzle.
bool encode_o_map(CUtensorMap *m, uint16_t *part_o, int64_t rows, int d)
{
    auto fn = encode_fn();
    if (!fn || rows < 1)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kTcTile};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, part_o, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// q rows are read by TMA (16-byte aligned base and strides, positive
// strides where the dimension has more than one entry).
bool q_layout_ok(const void *q, int64_t q_sb, int64_t q_sh, int B, int Hq)
{
    return aligned(q, 16) && q_sb % 8 == 0 && q_sh % 8 == 0 && (B == 1 || q_sb > 0) && (Hq == 1 || q_sh > 0) &&
           q_sb >= 0 && q_sh >= 0 && q_sb < ((int64_t)1 << 38) && q_sh < ((int64_t)1 << 38);
}

bool out_layout_ok(const void *out, hp_dtype dt, int64_t o_sb, int64_t o_sh, int d)
{
    if (dt != HP_BF16 && dt != HP_F32)
        return false;
    // the merge writes pairs of values; rows and strides aligned to d/32
    // values (a rule of earlier lane layouts, kept: stricter than pairs need)
    const size_t esz = dt == HP_F32 ? 4 : 2;
    const size_t lane_bytes = esz * (size_t)(d / 32);
    return aligned(out, lane_bytes) && (o_sb * (int64_t)esz) % (int64_t)lane_bytes == 0 &&
           (o_sh * (int64_t)esz) % (int64_t)lane_bytes == 0;
}

// CTAs of the small-row kernel resident per SM (shared memory bound); its
// grid is one such wave, each warp walking several items.
int small_ctas_per_sm(int d, bool q8 = false)
{
    return (int)std::max<size_t>(1, std::min<size_t>(4, (size_t)(227 * 1024) / small_smem_bytes(d, q8)));
}



// ------------------------------------------------------ standalone splits
// Key split of the standalone paged decode: items are (sequence, KV-head
// group, split); aim for about three items per resident CTA, at least 64 keys
// each.
int suffix_split_len(int B, int Hkv, int max_len, int sms, int d)
{
    const int nh = small_heads_per_item(Hkv);
    const int64_t chunks = (int64_t)B * (Hkv / nh) * ceil_div(std::max(max_len, 1), kChunk);
    const int64_t target = (int64_t)sms * small_ctas_per_sm(d) * 3;
    const int64_t per = std::max<int64_t>(4, ceil_div(chunks, target));
    return (int)(per * kChunk);
}

struct PrefixGeo {
    int spi, n_rc, n_split, split_len, n_items;
    int64_t part_rows;
};

PrefixGeo prefix_geo(int rows, int G, int Hkv, int len, int sms)
{
    PrefixGeo g{};
    g.spi = 2 * (kTcTile / G);
    g.spi = std::min(g.spi, std::max(rows, 1));
    g.n_rc = (int)ceil_div(rows, g.spi);
    const int64_t tiles = ceil_div(std::max(len, 1), kTcTile);
    const int64_t per = std::max<int64_t>(2, ceil_div((int64_t)g.n_rc * Hkv * tiles, sms));
    g.split_len = (int)(per * kTcTile);
    g.n_split = len > 0 ? (int)ceil_div(len, g.split_len) : 0;
    g.n_items = g.n_rc * Hkv * g.n_split;
    g.part_rows = (int64_t)g.n_items * 2 * kTcTile;  // two 128-row blocks per item
    return g;
}

uint64_t new_tag()
{
    static std::atomic<uint64_t> ctr{0};
    const uint64_t t = (uint64_t)std::chrono::steady_clock::now().time_since_epoch().count();
    return (t * 0x9E3779B97F4A7C15ull) ^ (++ctr * 0xBF58476D1CE4E5B9ull) ^ 0x68706c616e000000ull;
}

uint32_t *status_ptr(void *ws) { return reinterpret_cast<uint32_t *>(ws); }

// Failure detection tests: set by hp_test_withhold_first_tile.
std::atomic<int> g_withhold{0};

// Plans this library wrote, by device address: the persistent kernel copies
// its schedule record from plan + kPlanRecOff + cta * rec_stride before it can
// check the plan's tag, so a decode call is only launched when the grid and
// record stride it was given stay inside the plan image last written there.
// A decode-loop plan also keeps, on the host, what its appends need.
struct PlanExtent {
    uint64_t tag;
    int64_t total_bytes;
    int32_t loop_capacity;  // 0: not a decode-loop plan
    int32_t leaf_stride, page_size, num_pages;
    int64_t off_leaf_tab;
    void *k_pool, *v_pool;  // the suffix level's pools
    // E4M3 paged levels: the scales of each pool slot
    int32_t q8;
    const float *k_scale[kMaxLevels];
    const float *v_scale[kMaxLevels];
};
std::mutex g_plans_mu;
std::unordered_map<const void *, PlanExtent> g_plans;

void register_plan(const void *plan_dev, const PlanExtent &e)
{
    std::lock_guard<std::mutex> lk(g_plans_mu);
    g_plans[plan_dev] = e;
}

// The plan last written at plan_dev, if info's geometry stays inside it.
bool plan_extent(const void *plan_dev, const hp_plan_info *info, PlanExtent *out)
{
    std::lock_guard<std::mutex> lk(g_plans_mu);
    auto it = g_plans.find(plan_dev);
    if (it == g_plans.end())
        return false;
    const int64_t need = (int64_t)plan_tab_offset(info->grid, info->rec_stride) +
                         4 * (int64_t)info->B * info->Hkv * info->merge_stride;
    if (info->merge_stride < 1 || need > it->second.total_bytes)
        return false;
    *out = it->second;
    return true;
}

}  // namespace

int hp::device_sms()
{
    static std::atomic<int> cached{0};
    int v = cached.load();
    if (v > 0)
        return v;
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) {
        cached.store(n);
        return n;
    }
    cudaGetLastError();  // clear a sticky "no device" error
    return 152;          // GB300
}

bool hp::encode_pool_map(CUtensorMap *m, const void *pool, int num_pages, int Hkv, int ps, int d, int box_tok,
                         int box_heads, bool e4m3)
{
    auto fn = encode_fn();
    if (!fn || (e4m3 && d != 128))
        return false;
    const cuuint64_t es_b = e4m3 ? 1 : 2;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)ps, (cuuint64_t)Hkv, (cuuint64_t)num_pages};
    cuuint64_t strides[3] = {(cuuint64_t)d * es_b, (cuuint64_t)ps * d * es_b, (cuuint64_t)Hkv * ps * d * es_b};
    cuuint32_t box[4] = {e4m3 ? (cuuint32_t)d : 64u, (cuuint32_t)box_tok, (cuuint32_t)box_heads, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(pool),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

hp::WsLayout hp::ws_layout(int64_t part_rows, int d)
{
    WsLayout w;
    w.off_lse = kWsHeader;
    w.off_o = round_up(w.off_lse + (size_t)std::max<int64_t>(part_rows, 1) * 4, 256);
    w.total = round_up(w.off_o + (size_t)std::max<int64_t>(part_rows, 1) * d * 2, 256);
    return w;
}

// Queries q[b][h][:] (bf16; strides in elements, 16-byte multiples): box
// 64 columns x box_h heads x box_b rows, 128-byte swizzle, rows past B
// zero-filled.
bool hp::encode_q_map(CUtensorMap *m, const void *q, int B, int Hq, int d, int64_t q_sb, int64_t q_sh, int box_h,
                  int box_b)
{
    auto fn = encode_fn();
    if (!fn || box_h < 1 || box_h > 256 || box_b < 1 || box_b > 256)
        return false;
    const cuuint64_t sh = Hq > 1 ? (cuuint64_t)q_sh * 2 : (cuuint64_t)d * 2;
    const cuuint64_t sb = B > 1 ? (cuuint64_t)q_sb * 2 : sh * (cuuint64_t)Hq;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hq, (cuuint64_t)B};
    cuuint64_t strides[2] = {sh, sb};
    cuuint32_t box[3] = {64, (cuuint32_t)box_h, (cuuint32_t)box_b};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// ----------------------------------------------- Parallel Prompting rows
namespace {

struct StreamGeo {
    int ns_pg, n_sg, nh, sc, spi, n_sblk, rows_item, split_len, n_split;
    int64_t n_items, part_rows;
};

// Items of hp_stream_decode: consumer warps of an item serve (head, group of
// ns_pg streams) pairs, at most 8; the streams of a request share one pass
// over its row when their groups fit one item.
StreamGeo stream_geo(int R, int P, int G, int Hkv, int max_len, int sms)
{
    StreamGeo g{};
    g.ns_pg = std::max(1, std::min(kSmallRows / G, P));
    const int n_sg_all = (int)ceil_div(P, g.ns_pg);
    g.n_sg = std::min(n_sg_all, 8);
    g.nh = 1;
    for (int nh = 8; nh >= 1; nh /= 2)
        if (nh * g.n_sg <= 8 && Hkv % nh == 0) {
            g.nh = nh;
            break;
        }
    // an item of fewer than 8 heads takes several chunks per ring stage
    g.sc = std::min(4, 8 / g.nh);
    g.spi = g.n_sg * g.ns_pg;
    g.n_sblk = (int)ceil_div(P, g.spi);
    g.rows_item = g.nh * g.n_sg * g.ns_pg * G;
    const int64_t units = (int64_t)R * (Hkv / g.nh) * g.n_sblk;
    const int64_t chunks = ceil_div(std::max(max_len, 1), kChunk);
    // The key splits: items go to the CTAs in turn, so the step lasts about
    // ceil(items / SMs) items of ceil(chunks / splits) chunks each; take the
    // split count with the shortest such makespan (ties: fewer splits, fewer
    // partial states to merge), items of at least 4 chunks.
    int64_t per = chunks, best = -1;
    for (int64_t ns = 1; ns <= 256; ++ns) {
        const int64_t p_ns = ceil_div(chunks, ns);
        if (ns > 1 && p_ns < 4)
            break;
        const int64_t cost = ceil_div(units * ns, (int64_t)std::max(sms, 1)) * p_ns;
        if (best < 0 || cost < best) {
            best = cost;
            per = p_ns;
        }
    }
    g.split_len = (int)(per * kChunk);
    g.n_split = (int)ceil_div(std::max(max_len, 1), g.split_len);
    g.n_items = units * g.n_split;
    g.part_rows = g.n_items * g.rows_item;
    return g;
}

}  // namespace

// =================================================================== C ABI
extern "C" {

const char *hp_status_str(hp_status s)
{
    switch (s) {
    case HP_OK: return "ok";
    case HP_ERR_ARG: return "invalid argument";
    case HP_ERR_UNSUPPORTED: return "unsupported shape or layout";
    case HP_ERR_WORKSPACE: return "workspace or plan buffer too small or misaligned";
    case HP_ERR_CUDA: return "CUDA runtime error";
    case HP_ERR_BOUNDS: return "device: page id or length out of range";
    case HP_ERR_DEVICE_TIMEOUT: return "device: bounded wait ran out";
    }
    return "unknown status";
}

int32_t hp_build_arch(void) { return 103; }
int32_t hp_abi_version(void) { return kAbiVersion; }

hp_status hp_merge_states(const float *o_a, const float *lse_a, const float *o_b, const float *lse_b,
                          void *o_out, hp_dtype out_dt, float *lse_out, int64_t rows, int32_t d,
                          hp_stream_t stream)
{
    if (rows < 0 || d < 1 || (out_dt != HP_BF16 && out_dt != HP_F32))
        return HP_ERR_ARG;
    if (rows == 0)
        return HP_OK;
    if (!o_a || !lse_a || !o_b || !lse_b || !o_out)
        return HP_ERR_ARG;
    cudaError_t e = launch_merge2(o_a, lse_a, o_b, lse_b, o_out, out_dt == HP_F32, lse_out, rows, d,
                                  reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? HP_OK : HP_ERR_CUDA;
}

size_t hp_suffix_workspace_bytes(int32_t B, int32_t Hq, int32_t d, int32_t pt_stride, int32_t page_size)
{
    if (B < 1 || Hq < 1 || !supported_d(d) || pt_stride < 1 || page_size < 16)
        return 0;
    const int max_len = pt_stride * page_size;
    // the workspace bound assumes the most KV heads per group (Hkv = Hq)
    const int split = suffix_split_len(B, Hq, max_len, device_sms(), d);
    const int64_t n_split_max = ceil_div(max_len, std::min(split, 4 * kChunk));
    return ws_layout((int64_t)B * Hq * n_split_max, d).total;
}

static hp_status suffix_decode_impl(const void *q, int64_t q_sb, int64_t q_sh, int32_t B, const void *k_pool,
                                    const void *v_pool, const float *k_scale, const float *v_scale, bool q8,
                                    int32_t num_pages, int32_t page_size, const int32_t *page_table, int32_t pt_stride,
                                    const int32_t *seq_lens, int32_t Hq, int32_t Hkv, int32_t d, float scale, void *out,
                                    hp_dtype out_dt, int64_t o_sb, int64_t o_sh, float *lse, int64_t lse_sb, void *ws,
                                    size_t ws_bytes, hp_stream_t stream)
{
    if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !out || !ws)
        return HP_ERR_ARG;
    if (q8 && (!k_scale || !v_scale || !aligned(k_scale, 4) || !aligned(v_scale, 4)))
        return HP_ERR_ARG;
    if (q8 && d != 128)
        return HP_ERR_UNSUPPORTED;
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || num_pages < 1 || pt_stride < 1 || !std::isfinite(scale))
        return HP_ERR_ARG;
    if (!supported_d(d) || page_size < 16 || page_size > 256 || page_size % 16 || Hq / Hkv > kSmallRows)
        return HP_ERR_UNSUPPORTED;
    if (!q_layout_ok(q, q_sb, q_sh, B, Hq) || !out_layout_ok(out, out_dt, o_sb, o_sh, d) || !aligned(k_pool, 16) ||
        !aligned(v_pool, 16))
        return HP_ERR_UNSUPPORTED;
    if ((int64_t)pt_stride * page_size > INT32_MAX)
        return HP_ERR_UNSUPPORTED;
    const int G = Hq / Hkv;
    const int max_len = pt_stride * page_size;
    const int sms = device_sms();
    const int split = suffix_split_len(B, Hkv, max_len, sms, d);
    const int n_split = (int)ceil_div(max_len, split);
    const int nh = small_heads_per_item(Hkv);
    const WsLayout wl = ws_layout((int64_t)B * Hq * n_split, d);
    if (ws_bytes < wl.total || !aligned(ws, 256))
        return HP_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *wsb = static_cast<uint8_t *>(ws);

    SmallParams sp;
    std::memset(&sp, 0, sizeof(sp));
    if (!encode_pool_map(&sp.map_k, k_pool, num_pages, Hkv, page_size, d, kChunk, nh, q8) ||
        !encode_pool_map(&sp.map_v, v_pool, num_pages, Hkv, page_size, d, kChunk, nh, q8))
        return HP_ERR_CUDA;
    sp.q8 = q8 ? 1 : 0;
    sp.k_scale = k_scale;
    sp.v_scale = v_scale;
    sp.q_slot = nh * G <= small_q_rows();
    if (sp.q_slot && !encode_q_map(&sp.map_q, q, B, Hq, d, q_sb, q_sh, nh * G, 1))
        return HP_ERR_CUDA;
    sp.q = static_cast<const uint16_t *>(q);
    sp.q_sb = q_sb;
    sp.q_sh = q_sh;
    sp.G = G;
    sp.Hkv = Hkv;
    sp.scale_log2 = scale * kLog2e;
    sp.n_items = B * (Hkv / nh) * n_split;
    sp.nh = nh;
    sp.page_table = page_table;
    sp.pt_stride = pt_stride;
    sp.seq_lens = seq_lens;
    sp.B = B;
    sp.num_pages = num_pages;
    sp.page_size = page_size;
    sp.split_len = split;
    sp.n_split = n_split;
    sp.part_o = reinterpret_cast<uint16_t *>(wsb + wl.off_o);
    sp.part_lse = reinterpret_cast<float *>(wsb + wl.off_lse);
    sp.status = status_ptr(ws);
    const int grid = (int)std::min<int64_t>(sp.n_items, (int64_t)sms * small_ctas_per_sm(d, q8));
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
    mp.mode = 1;
    mp.seq_lens = seq_lens;
    mp.split_len = split;
    mp.n_split = n_split;
    mp.nh = nh;
    mp.out = out;
    mp.out_f32 = out_dt == HP_F32;
    mp.o_sb = o_sb;
    mp.o_sh = o_sh;
    mp.lse = lse;
    mp.lse_sb = lse_sb;
    mp.status = status_ptr(ws);
    return launch_merge(mp, (int64_t)B * Hq, s) == cudaSuccess ? HP_OK : HP_ERR_CUDA;
}

hp_status hp_suffix_decode_paged(const void *q, int64_t q_sb, int64_t q_sh, int32_t B, const void *k_pool,
                                 const void *v_pool, int32_t num_pages, int32_t page_size,
                                 const int32_t *page_table, int32_t pt_stride, const int32_t *seq_lens,
                                 int32_t Hq, int32_t Hkv, int32_t d, float scale, void *out, hp_dtype out_dt,
                                 int64_t o_sb, int64_t o_sh, float *lse, int64_t lse_sb, void *ws,
                                 size_t ws_bytes, hp_stream_t stream)
{
    return suffix_decode_impl(q, q_sb, q_sh, B, k_pool, v_pool, nullptr, nullptr, false, num_pages, page_size,
                              page_table, pt_stride, seq_lens, Hq, Hkv, d, scale, out, out_dt, o_sb, o_sh, lse,
                              lse_sb, ws, ws_bytes, stream);
}

hp_status hp_suffix_decode_paged_e4m3(const void *q, int64_t q_sb, int64_t q_sh, int32_t B, const void *k_pool,
                                      const void *v_pool, const float *k_scale, const float *v_scale,
                                      int32_t num_pages, int32_t page_size, const int32_t *page_table,
                                      int32_t pt_stride, const int32_t *seq_lens, int32_t Hq, int32_t Hkv, int32_t d,
                                      float scale, void *out, hp_dtype out_dt, int64_t o_sb, int64_t o_sh,
                                      float *lse, int64_t lse_sb, void *ws, size_t ws_bytes, hp_stream_t stream)
{
    return suffix_decode_impl(q, q_sb, q_sh, B, k_pool, v_pool, k_scale, v_scale, true, num_pages, page_size,
                              page_table, pt_stride, seq_lens, Hq, Hkv, d, scale, out, out_dt, o_sb, o_sh, lse,
                              lse_sb, ws, ws_bytes, stream);
}

size_t hp_stream_workspace_bytes(int32_t R, int32_t P, int32_t Hq, int32_t Hkv, int32_t d, int32_t pt_stride,
                                 int32_t page_size)
{
    if (R < 1 || P < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || Hq / Hkv > kSmallRows || !supported_d(d) ||
        pt_stride < 1 || page_size < 16 || page_size % 16)
        return 0;
    const StreamGeo g = stream_geo(R, P, Hq / Hkv, Hkv, pt_stride * page_size, device_sms());
    return ws_layout(g.part_rows, d).total;
}

hp_status hp_stream_decode(const void *q, int64_t q_sb, int64_t q_sh, int32_t R, int32_t P, const void *k_pool,
                           const void *v_pool, int32_t num_pages, int32_t page_size, const int32_t *row_pages,
                           int32_t pt_stride, const int32_t *row_len, const int32_t *slot_sid,
                           const int32_t *slot_pos, int32_t sid_stride, const int32_t *q_sid, const int32_t *q_pos,
                           int32_t Hq, int32_t Hkv, int32_t d, float scale, void *out, hp_dtype out_dt,
                           int64_t o_sb, int64_t o_sh, float *lse, int64_t lse_sb, void *ws, size_t ws_bytes,
                           hp_stream_t stream)
{
    if (!q || !k_pool || !v_pool || !row_pages || !row_len || !slot_sid || !slot_pos || !q_sid || !q_pos || !out ||
        !ws)
        return HP_ERR_ARG;
    if (R < 1 || P < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || num_pages < 1 || pt_stride < 1 || !std::isfinite(scale))
        return HP_ERR_ARG;
    if (!supported_d(d) || page_size < 16 || page_size > 256 || page_size % 16 || Hq / Hkv > kSmallRows)
        return HP_ERR_UNSUPPORTED;
    if ((int64_t)pt_stride * page_size > INT32_MAX || (int64_t)R * P > INT32_MAX / 2)
        return HP_ERR_UNSUPPORTED;
    // the slot arrays are read 16 slots at a time by bulk copies
    if (sid_stride % 4 || (int64_t)sid_stride < (int64_t)pt_stride * page_size || !aligned(slot_sid, 16) ||
        !aligned(slot_pos, 16))
        return HP_ERR_UNSUPPORTED;
    if (q_sb % 8 || q_sh % 8 || q_sb < 0 || q_sh < 0 || !aligned(q, 16) || !out_layout_ok(out, out_dt, o_sb, o_sh, d) ||
        !aligned(k_pool, 16) || !aligned(v_pool, 16))
        return HP_ERR_UNSUPPORTED;
    const int G = Hq / Hkv;
    const int sms = device_sms();
    const StreamGeo g = stream_geo(R, P, G, Hkv, pt_stride * page_size, sms);
    const WsLayout wl = ws_layout(g.part_rows, d);
    if (ws_bytes < wl.total || !aligned(ws, 256))
        return HP_ERR_WORKSPACE;
    if (g.n_items > INT32_MAX || g.part_rows > INT32_MAX)
        return HP_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *wsb = static_cast<uint8_t *>(ws);

    StreamParams sp;
    std::memset(&sp, 0, sizeof(sp));
    if (!encode_pool_map(&sp.map_k, k_pool, num_pages, Hkv, page_size, d, kChunk, g.nh) ||
        !encode_pool_map(&sp.map_v, v_pool, num_pages, Hkv, page_size, d, kChunk, g.nh))
        return HP_ERR_CUDA;
    sp.G = G;
    sp.Hkv = Hkv;
    sp.scale_log2 = scale * kLog2e;
    sp.n_items = (int32_t)g.n_items;
    sp.R = R;
    sp.P = P;
    sp.row_pages = row_pages;
    sp.pt_stride = pt_stride;
    sp.row_len = row_len;
    sp.slot_sid = slot_sid;
    sp.slot_pos = slot_pos;
    sp.sid_stride = sid_stride;
    sp.q_sid = q_sid;
    sp.q_pos = q_pos;
    sp.num_pages = num_pages;
    sp.page_size = page_size;
    sp.split_len = g.split_len;
    sp.n_split = g.n_split;
    sp.nh = g.nh;
    sp.n_sg = g.n_sg;
    sp.ns_pg = g.ns_pg;
    sp.sc = g.sc;
    sp.spi = g.spi;
    sp.n_sblk = g.n_sblk;
    sp.rows_item = g.rows_item;
    sp.q = static_cast<const uint16_t *>(q);
    sp.q_sb = q_sb;
    sp.q_sh = q_sh;
    sp.part_o = reinterpret_cast<uint16_t *>(wsb + wl.off_o);
    sp.part_lse = reinterpret_cast<float *>(wsb + wl.off_lse);
    sp.status = status_ptr(ws);
    const int grid = (int)std::min<int64_t>(g.n_items, (int64_t)sms);
    if (launch_stream(sp, grid, d, s) != cudaSuccess)
        return HP_ERR_CUDA;

    MergeParams mp;
    std::memset(&mp, 0, sizeof(mp));
    mp.part_o = sp.part_o;
    mp.part_lse = sp.part_lse;
    mp.d = d;
    mp.G = G;
    mp.Hq = Hq;
    mp.Hkv = Hkv;
    mp.B = R * P;
    mp.mode = 3;
    mp.seq_lens = row_len;
    mp.split_len = g.split_len;
    mp.n_split = g.n_split;
    mp.nh = g.nh;
    mp.P = P;
    mp.spi = g.spi;
    mp.n_sblk = g.n_sblk;
    mp.ns_pg = g.ns_pg;
    mp.n_sg = g.n_sg;
    mp.rows_item = g.rows_item;
    mp.out = out;
    mp.out_f32 = out_dt == HP_F32;
    mp.o_sb = o_sb;
    mp.o_sh = o_sh;
    mp.lse = lse;
    mp.lse_sb = lse_sb;
    mp.status = status_ptr(ws);
    return launch_merge(mp, (int64_t)R * P * Hq, s) == cudaSuccess ? HP_OK : HP_ERR_CUDA;
}

size_t hp_prefix_workspace_bytes(int32_t rows, int32_t Hq, int32_t Hkv, int32_t d, int32_t prefix_len)
{
    if (rows < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || !supported_d(d) || prefix_len < 0)
        return 0;
    const PrefixGeo g = prefix_geo(rows, Hq / Hkv, Hkv, prefix_len, device_sms());
    return ws_layout(g.part_rows, d).total;
}

hp_status hp_prefix_attn(const void *q, int64_t q_sb, int64_t q_sh, int32_t row_begin, int32_t rows, const void *k,
                         const void *v, int64_t kv_st, int64_t kv_sh, int32_t prefix_len, int32_t Hq, int32_t Hkv,
                         int32_t d, float scale, void *out, hp_dtype out_dt, int64_t o_sb, int64_t o_sh,
                         float *lse, int64_t lse_sb, void *ws, size_t ws_bytes, hp_stream_t stream)
{
    if (!q || !out || !ws || rows < 1 || row_begin < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || prefix_len < 0 ||
        !std::isfinite(scale) || !(scale > 0.f))
        return HP_ERR_ARG;
    if (prefix_len > 0 && (!k || !v))
        return HP_ERR_ARG;
    if (!supported_d(d) || Hq / Hkv > kTcTile)
        return HP_ERR_UNSUPPORTED;
    if (!q_layout_ok(q, q_sb, q_sh, row_begin + rows, Hq) || !out_layout_ok(out, out_dt, o_sb, o_sh, d))
        return HP_ERR_UNSUPPORTED;
    if (prefix_len > 0 &&
        (!aligned(k, 16) || !aligned(v, 16) || kv_st % 8 || kv_sh % 8 || kv_st <= 0 || kv_sh < 0))
        return HP_ERR_UNSUPPORTED;
    const int G = Hq / Hkv;
    const int sms = device_sms();
    const PrefixGeo g = prefix_geo(rows, G, Hkv, prefix_len, sms);
    const WsLayout wl = ws_layout(g.part_rows, d);
    if (ws_bytes < wl.total || !aligned(ws, 256))
        return HP_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *wsb = static_cast<uint8_t *>(ws);

    TcParams tp;
    std::memset(&tp, 0, sizeof(tp));
    if (g.n_items > 0) {
        if (!encode_prefix_map(&tp.map_k, k, prefix_len, Hkv, d, kv_st, kv_sh) ||
            !encode_prefix_map(&tp.map_v, v, prefix_len, Hkv, d, kv_st, kv_sh) ||
            !encode_q_map(&tp.map_q, q, row_begin + rows, Hq, d, q_sb, q_sh, G, kTcTile / G) ||
            !encode_o_map(&tp.map_o, reinterpret_cast<uint16_t *>(wsb + wl.off_o), g.part_rows, d))
            return HP_ERR_CUDA;
        tp.G = G;
        tp.Hkv = Hkv;
        tp.scale_log2 = scale * kLog2e;
        tp.n_items = g.n_items;
        tp.imp_row_begin = row_begin;
        tp.imp_rows = rows;
        tp.imp_seqs_per_item = g.spi;
        tp.imp_split_len = g.split_len;
        tp.imp_n_split = g.n_split;
        tp.imp_len = prefix_len;
        tp.part_lse = reinterpret_cast<float *>(wsb + wl.off_lse);
        tp.status = status_ptr(ws);
        if (launch_tc(tp, g.n_items, d, s) != cudaSuccess)
            return HP_ERR_CUDA;
    }
    MergeParams mp;
    std::memset(&mp, 0, sizeof(mp));
    mp.part_o = reinterpret_cast<const uint16_t *>(wsb + wl.off_o);
    mp.part_lse = reinterpret_cast<float *>(wsb + wl.off_lse);
    mp.d = d;
    mp.G = G;
    mp.Hq = Hq;
    mp.Hkv = Hkv;
    mp.B = rows;  // output rows b - row_begin
    mp.mode = 2;
    mp.n_split = g.n_split;
    mp.seqs_per_item = g.spi;
    mp.row_begin = 0;
    mp.rows = rows;
    mp.n_rc = g.n_rc;
    // rows are addressed relative to row_begin
    const size_t esz = out_dt == HP_F32 ? 4 : 2;
    mp.out = static_cast<uint8_t *>(out) + (size_t)row_begin * o_sb * esz;
    mp.out_f32 = out_dt == HP_F32;
    mp.o_sb = o_sb;
    mp.o_sh = o_sh;
    mp.lse = lse ? lse + (size_t)row_begin * lse_sb : nullptr;
    mp.lse_sb = lse_sb;
    mp.status = status_ptr(ws);
    return launch_merge(mp, (int64_t)rows * Hq, s) == cudaSuccess ? HP_OK : HP_ERR_CUDA;
}

size_t hp_cascade_plan_bytes(const hp_tree_desc *desc)
{
    HostPlan P;
    if (build_plan(desc, P, false) != HP_OK)
        return 0;
    return (size_t)P.hdr.total_bytes;
}

static hp_status cascade_plan_impl(const hp_tree_desc *desc, int capacity, void *plan_dev, size_t plan_bytes,
                                   hp_plan_info *info, hp_stream_t stream)
{
    if (!plan_dev || !info)
        return HP_ERR_ARG;
    HostPlan P;
    hp_status st = build_plan(desc, P, true, capacity);
    if (st != HP_OK)
        return st;
    PlanHeader &H = P.hdr;
    if (plan_bytes < (size_t)H.total_bytes || !aligned(plan_dev, 256))
        return HP_ERR_WORKSPACE;
    H.tag = new_tag();
    std::vector<uint8_t> img((size_t)H.total_bytes, 0);
    std::memcpy(img.data(), &H, sizeof(H));
    if (!P.maps.empty())
        std::memcpy(img.data() + kPlanMapsOff, P.maps.data(), sizeof(CUtensorMap) * P.maps.size());
    for (size_t c = 0; c < P.records.size(); ++c) {
        uint8_t *dst = img.data() + kPlanRecOff + c * (size_t)H.rec_stride;
        std::memcpy(dst, P.records[c].data(), P.records[c].size());
        std::memcpy(dst, &H.tag, sizeof(H.tag));  // RecHead::tag
    }
    std::memcpy(img.data() + H.off_merge_tab, P.merge_tab.data(), 4 * P.merge_tab.size());
    if (!P.leaf_tab.empty())
        std::memcpy(img.data() + H.off_leaf_tab, P.leaf_tab.data(), 4 * P.leaf_tab.size());
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(plan_dev, img.data(), img.size(), cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return HP_ERR_CUDA;
    PlanExtent ext{};
    ext.tag = H.tag;
    ext.total_bytes = H.total_bytes;
    ext.q8 = P.q8 ? 1 : 0;
    for (size_t sl = 0; sl < P.slot_kv.size() && sl < (size_t)kMaxLevels; ++sl) {
        ext.k_scale[sl] = P.slot_k_scale[sl];
        ext.v_scale[sl] = P.slot_v_scale[sl];
    }
    if (capacity > 0) {
        const hp_tree_level &S = desc->levels[desc->num_levels - 1];
        ext.loop_capacity = capacity;
        ext.leaf_stride = H.leaf_stride;
        ext.page_size = S.page_size;
        ext.num_pages = S.num_pages;
        ext.off_leaf_tab = H.off_leaf_tab;
        ext.k_pool = const_cast<void *>(S.k_pool);
        ext.v_pool = const_cast<void *>(S.v_pool);
    }
    register_plan(plan_dev, ext);
    std::memset(info, 0, sizeof(*info));
    info->B = H.B;
    info->Hq = H.Hq;
    info->Hkv = H.Hkv;
    info->d = H.d;
    info->n_tc_items = H.n_tc;
    info->n_small_items = H.n_small;
    info->grid = H.grid;
    info->rec_stride = H.rec_stride;
    info->num_levels = H.num_levels;
    info->merge_stride = H.merge_stride;
    info->n_part_rows = H.n_part_rows;
    info->plan_bytes = H.total_bytes;
    info->ws_bytes = H.ws_bytes;
    info->tag = H.tag;
    return HP_OK;
}

hp_status hp_cascade_plan(const hp_tree_desc *desc, void *plan_dev, size_t plan_bytes, hp_plan_info *info,
                          hp_stream_t stream)
{
    return cascade_plan_impl(desc, 0, plan_dev, plan_bytes, info, stream);
}

size_t hp_cascade_loop_plan_bytes(const hp_tree_desc *desc, int32_t capacity)
{
    HostPlan P;
    if (capacity < 1 || build_plan(desc, P, false, capacity) != HP_OK)
        return 0;
    return (size_t)P.hdr.total_bytes;
}

hp_status hp_cascade_loop_plan(const hp_tree_desc *desc, int32_t capacity, void *plan_dev, size_t plan_bytes,
                               hp_plan_info *info, hp_stream_t stream)
{
    if (capacity < 1)
        return HP_ERR_ARG;
    return cascade_plan_impl(desc, capacity, plan_dev, plan_bytes, info, stream);
}

// The arguments of a cascade step, checked before anything is launched;
// fills *ext from the plan.
static hp_status decode_args(const void *plan_dev, const hp_plan_info *info, const void *q, int64_t q_sb,
                             int64_t q_sh, float scale, const void *out, hp_dtype out_dt, int64_t o_sb, int64_t o_sh,
                             const void *ws, size_t ws_bytes, const int32_t *suffix_len, const void *k_new,
                             const void *v_new, int64_t kv_sb, int64_t kv_sh, PlanExtent *ext)
{
    if (!plan_dev || !info || !q || !out || !ws || !std::isfinite(scale) || !(scale > 0.f))
        return HP_ERR_ARG;
    if (info->B < 1 || info->Hq < 1 || info->Hkv < 1 || info->Hq % info->Hkv || !supported_d(info->d))
        return HP_ERR_ARG;
    if (!q_layout_ok(q, q_sb, q_sh, info->B, info->Hq) || !out_layout_ok(out, out_dt, o_sb, o_sh, info->d))
        return HP_ERR_UNSUPPORTED;
    if (info->Hq / info->Hkv > kTcTile || info->grid < 1 || info->num_levels < 1 ||
        info->num_levels > kMaxLevels || info->rec_stride < (int32_t)sizeof(RecHead) ||
        info->rec_stride > kRecMaxBytes || info->rec_stride % 128)
        return HP_ERR_ARG;
    if (!plan_extent(plan_dev, info, ext))
        return HP_ERR_ARG;
    // a decode-loop plan runs with the current suffix lengths, a plain plan without
    if ((ext->loop_capacity > 0) != (suffix_len != nullptr) || (suffix_len && !aligned(suffix_len, 4)))
        return HP_ERR_ARG;
    if (k_new && (!v_new || !aligned(k_new, 16) || !aligned(v_new, 16) || kv_sb <= 0 || kv_sh <= 0 || kv_sb % 8 ||
                  kv_sh % 8))
        return HP_ERR_UNSUPPORTED;
    if (ws_bytes < (size_t)info->ws_bytes || !aligned(ws, 256))
        return HP_ERR_WORKSPACE;
    return HP_OK;
}

static hp_status cascade_decode_impl(const void *plan_dev, const hp_plan_info *info, const void *q,
                                     int64_t q_sb, int64_t q_sh, float scale, void *out, hp_dtype out_dt,
                                     int64_t o_sb, int64_t o_sh, float *lse, int64_t lse_sb, void *ws,
                                     size_t ws_bytes, hp_stream_t stream, void *const *events,
                                     const int32_t *suffix_len = nullptr, const void *k_new = nullptr,
                                     const void *v_new = nullptr, int64_t kv_sb = 0, int64_t kv_sh = 0)
{
    auto mark = [&](int i) {
        if (events && events[i])
            cudaEventRecordWithFlags(static_cast<cudaEvent_t>(events[i]), reinterpret_cast<cudaStream_t>(stream),
                                     cudaEventRecordExternal);
    };
    PlanExtent ext;
    const hp_status st = decode_args(plan_dev, info, q, q_sb, q_sh, scale, out, out_dt, o_sb, o_sh, ws, ws_bytes,
                                     suffix_len, k_new, v_new, kv_sb, kv_sh, &ext);
    if (st != HP_OK)
        return st;
    const WsLayout wl = ws_layout(info->n_part_rows, info->d);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    const PlanHeader *plan = static_cast<const PlanHeader *>(plan_dev);
    const int G = info->Hq / info->Hkv;
    uint16_t *part_o = reinterpret_cast<uint16_t *>(wsb + wl.off_o);
    float *part_lse = reinterpret_cast<float *>(wsb + wl.off_lse);

    mark(0);
    if (info->n_tc_items + info->n_small_items > 0) {
        CascadeParams cp;
        std::memset(&cp, 0, sizeof(cp));
        const int nh = cascade_heads_per_item(info->Hkv);
        cp.q_slot = nh * G <= cascade_q_rows();
        if (!encode_q_map(&cp.q_tc, q, info->B, info->Hq, info->d, q_sb, q_sh, G, kTcTile / G) ||
            (cp.q_slot && !encode_q_map(&cp.q_sm, q, info->B, info->Hq, info->d, q_sb, q_sh, nh * G, 1)) ||
            !encode_o_map(&cp.o_tc, part_o, std::max<int64_t>(info->n_part_rows, 1), info->d))
            return HP_ERR_CUDA;
        cp.plan = static_cast<const uint8_t *>(plan_dev);
        cp.tag = info->tag;
        cp.rec_stride = info->rec_stride;
        cp.num_levels = info->num_levels;
        cp.G = G;
        cp.small_nh = nh;
        cp.q = static_cast<const uint16_t *>(q);
        cp.q_sb = q_sb;
        cp.q_sh = q_sh;
        cp.scale_log2 = scale * kLog2e;
        cp.part_o = part_o;
        cp.part_lse = part_lse;
        cp.status = status_ptr(ws);
        // failure detection tests only (hp_test_withhold_first_tile)
        cp.withhold = g_withhold.load(std::memory_order_relaxed);
        cp.suffix_len = suffix_len;
        cp.loop_capacity = ext.loop_capacity;
        cp.k_new = static_cast<const uint16_t *>(k_new);
        cp.v_new = static_cast<const uint16_t *>(v_new);
        cp.kv_sb = kv_sb;
        cp.kv_sh = kv_sh;
        cp.loop_k_pool = static_cast<uint16_t *>(ext.k_pool);
        cp.loop_v_pool = static_cast<uint16_t *>(ext.v_pool);
        cp.Hkv = info->Hkv;
        cp.d = info->d;
        cp.q8 = ext.q8;
        for (int sl = 0; sl < kMaxLevels; ++sl) {
            cp.k_scale[sl] = ext.k_scale[sl];
            cp.v_scale[sl] = ext.v_scale[sl];
        }
        if (launch_cascade(cp, info->grid, info->d, s) != cudaSuccess)
            return HP_ERR_CUDA;
    }
    mark(1);
    MergeParams mp;
    std::memset(&mp, 0, sizeof(mp));
    mp.part_o = part_o;
    mp.part_lse = part_lse;
    mp.d = info->d;
    mp.G = G;
    mp.Hq = info->Hq;
    mp.Hkv = info->Hkv;
    mp.B = info->B;
    mp.plan = plan;
    mp.tag = info->tag;
    mp.tab = reinterpret_cast<const int32_t *>(static_cast<const uint8_t *>(plan_dev) +
                                               plan_tab_offset(info->grid, info->rec_stride));
    mp.tab_stride = info->merge_stride;
    mp.out = out;
    mp.out_f32 = out_dt == HP_F32;
    mp.o_sb = o_sb;
    mp.o_sh = o_sh;
    mp.lse = lse;
    mp.lse_sb = lse_sb;
    mp.status = status_ptr(ws);
    if (k_new) {
        mp.len_inc = const_cast<int32_t *>(suffix_len);
        mp.len_capacity = ext.loop_capacity;
    }
    // the merge overlaps its launch with the fused kernel's tail unless an
    // event was recorded in between
    const bool dependent = !(events && events[1]);
    if ((dependent ? launch_merge_dependent(mp, (int64_t)info->B * info->Hq, s)
                   : launch_merge(mp, (int64_t)info->B * info->Hq, s)) != cudaSuccess)
        return HP_ERR_CUDA;
    mark(2);
    return HP_OK;
}

hp_status hp_cascade_decode(const void *plan_dev, const hp_plan_info *info, const void *q, int64_t q_sb,
                            int64_t q_sh, float scale, void *out, hp_dtype out_dt, int64_t o_sb, int64_t o_sh,
                            float *lse, int64_t lse_sb, void *ws, size_t ws_bytes, hp_stream_t stream)
{
    return cascade_decode_impl(plan_dev, info, q, q_sb, q_sh, scale, out, out_dt, o_sb, o_sh, lse, lse_sb, ws,
                               ws_bytes, stream, nullptr);
}

// The device-accessible address of page-locked host memory, or null when
// p is not page-locked host memory (device memory, pageable memory, an
// unknown pointer).
static void *pinned_host_address(const void *p)
{
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer leaves no sticky error behind
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

size_t hp_cascade_host_workspace_bytes(const hp_plan_info *info)
{
    if (!info || info->B < 1 || info->Hq < 1 || !supported_d(info->d) || info->ws_bytes < 1)
        return 0;
    return round_up((size_t)info->ws_bytes, 256) + (size_t)info->B * info->Hq * info->d * 2;
}

hp_status hp_cascade_decode_host(const void *plan_dev, const hp_plan_info *info, const void *q_host, int64_t q_sb,
                                 int64_t q_sh, float scale, void *out_host, hp_dtype out_dt, int64_t o_sb,
                                 int64_t o_sh, float *lse_host, int64_t lse_sb, void *ws, size_t ws_bytes,
                                 hp_stream_t stream)
{
    if (!plan_dev || !info || !q_host || !out_host || !ws)
        return HP_ERR_ARG;
    const size_t need = hp_cascade_host_workspace_bytes(info);
    if (need == 0)
        return HP_ERR_ARG;
    if (!q_layout_ok(q_host, q_sb, q_sh, info->B, info->Hq))
        return HP_ERR_UNSUPPORTED;
    if (ws_bytes < need || !aligned(ws, 256))
        return HP_ERR_WORKSPACE;
    void *q_dev = pinned_host_address(q_host);
    void *out_dev = pinned_host_address(out_host);
    void *lse_dev = lse_host ? pinned_host_address(lse_host) : nullptr;
    if (!q_dev || !out_dev || (lse_host && !lse_dev) || !aligned(q_dev, 16))
        return HP_ERR_ARG;
    uint16_t *staged = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + round_up((size_t)info->ws_bytes, 256));
    // the copy-in is launched only once the step's own arguments have been
    // checked, so an argument error launches nothing
    PlanExtent ext;
    const hp_status st = decode_args(plan_dev, info, staged, (int64_t)info->Hq * info->d, info->d, scale, out_dev,
                                     out_dt, o_sb, o_sh, ws, ws_bytes, nullptr, nullptr, nullptr, 0, 0, &ext);
    if (st != HP_OK)
        return st;
    StageParams sp;
    sp.src = static_cast<const uint16_t *>(q_dev);
    sp.sb = q_sb;
    sp.sh = q_sh;
    sp.B = info->B;
    sp.Hq = info->Hq;
    sp.d = info->d;
    sp.dst = staged;
    if (launch_stage(sp, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return HP_ERR_CUDA;
    return cascade_decode_impl(plan_dev, info, staged, (int64_t)info->Hq * info->d, info->d, scale, out_dev, out_dt,
                               o_sb, o_sh, static_cast<float *>(lse_dev), lse_sb, ws, ws_bytes, stream, nullptr);
}

hp_status hp_cascade_decode_loop(const void *plan_dev, const hp_plan_info *info, const int32_t *suffix_len,
                                 const void *q, int64_t q_sb, int64_t q_sh, float scale, void *out, hp_dtype out_dt,
                                 int64_t o_sb, int64_t o_sh, float *lse, int64_t lse_sb, void *ws, size_t ws_bytes,
                                 hp_stream_t stream)
{
    if (!suffix_len)
        return HP_ERR_ARG;
    return cascade_decode_impl(plan_dev, info, q, q_sb, q_sh, scale, out, out_dt, o_sb, o_sh, lse, lse_sb, ws,
                               ws_bytes, stream, nullptr, suffix_len);
}

hp_status hp_cascade_decode_append(const void *plan_dev, const hp_plan_info *info, int32_t *suffix_len,
                                   const void *k_new, const void *v_new, int64_t kv_sb, int64_t kv_sh, const void *q,
                                   int64_t q_sb, int64_t q_sh, float scale, void *out, hp_dtype out_dt, int64_t o_sb,
                                   int64_t o_sh, float *lse, int64_t lse_sb, void *ws, size_t ws_bytes,
                                   hp_stream_t stream)
{
    if (!suffix_len || !k_new || !v_new)
        return HP_ERR_ARG;
    return cascade_decode_impl(plan_dev, info, q, q_sb, q_sh, scale, out, out_dt, o_sb, o_sh, lse, lse_sb, ws,
                               ws_bytes, stream, nullptr, suffix_len, k_new, v_new, kv_sb, kv_sh);
}

hp_status hp_cascade_append_kv(const void *plan_dev, const hp_plan_info *info, const void *k_new, const void *v_new,
                               int64_t kv_sb, int64_t kv_sh, int32_t *suffix_len, void *ws, size_t ws_bytes,
                               hp_stream_t stream)
{
    if (!plan_dev || !info || !k_new || !v_new || !suffix_len || !ws)
        return HP_ERR_ARG;
    if (info->B < 1 || info->Hkv < 1 || !supported_d(info->d) || info->grid < 1 || info->rec_stride < 1)
        return HP_ERR_ARG;
    PlanExtent ext;
    if (!plan_extent(plan_dev, info, &ext) || ext.loop_capacity < 1)
        return HP_ERR_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(suffix_len, 4) || kv_sb <= 0 || kv_sh <= 0 ||
        kv_sb % 8 || kv_sh % 8)
        return HP_ERR_UNSUPPORTED;
    if (ws_bytes < kWsHeader || !aligned(ws, 256))
        return HP_ERR_WORKSPACE;
    AppendParams ap;
    std::memset(&ap, 0, sizeof(ap));
    ap.leaf_tab = reinterpret_cast<const int32_t *>(static_cast<const uint8_t *>(plan_dev) + ext.off_leaf_tab);
    ap.leaf_stride = ext.leaf_stride;
    ap.capacity = ext.loop_capacity;
    ap.page_size = ext.page_size;
    ap.num_pages = ext.num_pages;
    ap.B = info->B;
    ap.Hkv = info->Hkv;
    ap.d = info->d;
    ap.k_pool = static_cast<uint16_t *>(ext.k_pool);
    ap.v_pool = static_cast<uint16_t *>(ext.v_pool);
    ap.k_new = static_cast<const uint16_t *>(k_new);
    ap.v_new = static_cast<const uint16_t *>(v_new);
    ap.kv_sb = kv_sb;
    ap.kv_sh = kv_sh;
    ap.suffix_len = suffix_len;
    ap.status = status_ptr(ws);
    return launch_append(ap, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? HP_OK : HP_ERR_CUDA;
}

hp_status hp_cascade_decode_profiled(const void *plan_dev, const hp_plan_info *info, const void *q,
                                     int64_t q_sb, int64_t q_sh, float scale, void *out, hp_dtype out_dt,
                                     int64_t o_sb, int64_t o_sh, float *lse, int64_t lse_sb, void *ws,
                                     size_t ws_bytes, hp_stream_t stream, void *const *events)
{
    return cascade_decode_impl(plan_dev, info, q, q_sb, q_sh, scale, out, out_dt, o_sb, o_sh, lse, lse_sb, ws,
                               ws_bytes, stream, events);
}

int32_t hp_cascade_contexts(const hp_tree_desc *desc, int32_t *out, int32_t cap)
{
    if (validate_desc(desc) != HP_OK)
        return -1;
    std::vector<int32_t> ctx;
    build_contexts(desc, ctx);
    const int32_t n = (int32_t)(ctx.size() / 5);
    if (out)
        std::memcpy(out, ctx.data(), sizeof(int32_t) * 5 * (size_t)std::min(n, std::max(cap, 0)));
    return n;
}

int32_t hp_cascade_plan_stats(const hp_tree_desc *desc, int64_t *stats4)
{
    HostPlan P;
    if (!stats4 || build_plan(desc, P, false) != HP_OK)
        return -1;
    stats4[0] = P.hdr.n_tc;
    stats4[1] = P.hdr.n_small;
    stats4[2] = P.hdr.n_part_rows;
    stats4[3] = P.hdr.n_merge;
    return 0;
}

int32_t hp_cascade_plan_items(const hp_tree_desc *desc, int32_t capacity, int32_t *out, int32_t cap)
{
    HostPlan P;
    if (capacity < 0 || build_plan(desc, P, false, capacity) != HP_OK)
        return -1;
    const int32_t n = (int32_t)(P.tc.size() + P.small.size());
    if (!out)
        return n;
    int32_t k = 0;
    auto put = [&](const WorkItem &w, int cta, int tc) {
        if (k >= cap)
            return;
        int32_t *e = out + (size_t)k * 11;
        const int32_t v[11] = {w.level, w.seq_begin, w.n_seq, w.kvh, tc ? 1 : P.hdr.small_nh, w.k0, w.k1,
                               w.part_row, cta, tc, w.len_seq};
        std::memcpy(e, v, sizeof(v));
        ++k;
    };
    for (size_t c = 0; c < P.cta_tc.size(); ++c) {
        for (int32_t id : P.cta_tc[c])
            put(P.tc[id], (int)c, 1);
        for (int32_t id : P.cta_small[c])
            put(P.small[id], (int)c, 0);
    }
    return n;
}

int64_t hp_cascade_plan_item_pages(const hp_tree_desc *desc, int32_t capacity, int64_t *offsets, int32_t *pages,
                                   int64_t cap)
{
    HostPlan P;
    if (capacity < 0 || build_plan(desc, P, false, capacity) != HP_OK)
        return -1;
    // the page ids each item's record entry carries, in hp_cascade_plan_items' order
    int64_t total = 0, k = 0;
    auto put = [&](const WorkItem &w) {
        const int ps = P.level_ps[w.level];
        const int64_t first = w.k0 / ps, n = item_pages(w, ps);
        if (offsets)
            offsets[k] = total;
        for (int64_t i = 0; i < n; ++i, ++total)
            if (pages && total < cap)
                pages[total] = P.page_ids[(size_t)(w.page_base + first + i)];
        ++k;
    };
    for (size_t c = 0; c < P.cta_tc.size(); ++c) {
        for (int32_t id : P.cta_tc[c])
            put(P.tc[id]);
        for (int32_t id : P.cta_small[c])
            put(P.small[id]);
    }
    if (offsets)
        offsets[k] = total;
    return total;
}

int32_t hp_cascade_plan_merge_table(const hp_tree_desc *desc, int32_t capacity, int32_t *out, int64_t cap)
{
    HostPlan P;
    if (capacity < 0 || build_plan(desc, P, false, capacity) != HP_OK)
        return -1;
    if (out)
        std::memcpy(out, P.merge_tab.data(),
                    sizeof(int32_t) * (size_t)std::min<int64_t>((int64_t)P.merge_tab.size(), std::max<int64_t>(cap, 0)));
    return P.hdr.merge_stride;
}

void hp_test_withhold_first_tile(int32_t enable) { g_withhold.store(enable != 0 ? 1 : 0); }

hp_status hp_read_device_status(void *ws, hp_stream_t stream)
{
    if (!ws)
        return HP_ERR_ARG;
    uint32_t word = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(ws, 0, sizeof(word), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return HP_ERR_CUDA;
    if (word & kStTimeout)
        return HP_ERR_DEVICE_TIMEOUT;
    if (word & kStBounds)
        return HP_ERR_BOUNDS;
    if (word & kStPlan)
        return HP_ERR_ARG;
    return HP_OK;
}

} // extern "C"
