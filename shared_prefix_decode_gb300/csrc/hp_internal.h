// hp_internal.h -- structures shared by the host library and the kernels:
// the device-resident plan (work items, page ids, merge lists, TMA tensor
// maps) and the launch entry points of each kernel translation unit.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/hp.h"

namespace hp {

// One-time set-up per device, for state the CUDA runtime keeps per device
// (a kernel's shared-memory limit and carveout): run(f) calls f with the
// device current, the first time any thread reaches it on that device;
// other threads wait for it.  A failed f is tried again by the next caller.
class DeviceOnce {
  public:
    template <class F>
    cudaError_t run(F &&f)
    {
        int dev = -1;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return e;
        if (dev < 0 || dev >= kMaxDev)
            return cudaErrorInvalidDevice;
        if (done_[dev].load(std::memory_order_acquire))
            return cudaSuccess;
        std::lock_guard<std::mutex> g(mu_);
        if (done_[dev].load(std::memory_order_relaxed))
            return cudaSuccess;
        e = f();
        if (e == cudaSuccess)
            done_[dev].store(true, std::memory_order_release);
        return e;
    }

  private:
    static constexpr int kMaxDev = 64;
    std::mutex mu_;
    std::atomic<bool> done_[kMaxDev] = {};
};

// A plan keeps pool information and tensor maps per distinct pool set (a
// "pool slot": K pool, V pool, page count, page size), at most kMaxLevels of
// them; a tree may have up to kMaxTreeLevels levels that share them.
constexpr int kMaxLevels = 8;
constexpr int kMaxTreeLevels = 64;
constexpr uint32_t kPlanMagic = 0x31504C48u;  // "HLP1"
constexpr int kTcTile = 128;                  // keys per tensor-core tile
constexpr int kTcMaxRows = 256;               // query rows per tensor-core item (2 x M=128)
constexpr int kSmallRows = 16;                // query rows per small item (one m16 tile)
// E4M3 paged items of at least this many 16-key chunks are consumed two
// chunks per pass (more independent work per consumer warp); shorter ones
// chunk by chunk, where waiting for a second stage costs more than the
// overlap gains.
constexpr int kPairChunks = 12;
constexpr int kChunk = 16;                    // keys per small-kernel chunk
constexpr size_t kWsHeader = 256;             // status word + reserved
// Partial attention states in the workspace: LSE as f32, O / l as bf16 (raw
// bits) -- the partial rows are written once and read once, and their bytes
// cross the SMs' ports twice; bf16 keeps 8 significant bits, the precision
// of the bf16 output.

// Device status bits (the first word of every workspace).
enum : uint32_t { kStBounds = 1u, kStTimeout = 2u, kStPlan = 4u };

// One unit of work: query rows (sequences [seq_begin, seq_begin+n_seq) x the
// G heads of KV head kvh) against keys [k0, k1) of one tree node.  Its rows
// land in partial rows part_row + s*G + g.  (Host-side planning form.)
struct WorkItem {
    int32_t level;
    int32_t seq_begin;
    int32_t n_seq;
    int32_t kvh;
    int32_t k0, k1;
    int32_t page_base;  // index in the level's page-id list of the node's first page
    int32_t part_row;
    int32_t len_seq;    // decode-loop suffix items: the sequence whose length ends the range; else -1
    int32_t k1_model;   // the key end the cost model assumes (k1, or a loop item's mean end)
};
static_assert(sizeof(WorkItem) == 40, "WorkItem layout");

struct LevelDev {
    const void *k_pool;
    const void *v_pool;
    int32_t num_pages;
    int32_t page_size;
    int32_t tc_box;     // tokens per TMA box of the tensor-core maps (gcd(page_size, 128))
    int32_t pad;
};

// Tensor maps per level: [0] K for the tensor-core role, [1] V likewise,
// [2] K for the paged role (16-token boxes of a head group), [3] V likewise.
constexpr int kMapsPerLevel = 4;

struct alignas(64) PlanHeader {
    uint32_t magic;
    uint32_t version;
    uint64_t tag;
    int32_t B, Hq, Hkv, d, G, num_levels;
    int32_t n_tc, n_small, n_part_rows, n_merge;
    int32_t small_nh;       // KV heads per paged item
    int32_t grid;           // CTAs of the fused kernel (one record per CTA)
    int32_t rec_stride;     // bytes per CTA record (multiple of 128)
    int32_t merge_stride;   // int32 per merge-table row
    int64_t off_merge_tab;  // [B*Hkv][merge_stride] int32: count, then partial rows of (b, g = 0)
    int64_t total_bytes;
    int64_t ws_bytes;
    int64_t ws_off_lse;     // byte offsets into the workspace
    int64_t ws_off_o;
    // decode-loop plans (loop_capacity > 0): the suffix level, and each
    // sequence's suffix pages for appends, [B][leaf_stride] int32 at
    // off_leaf_tab (after the merge table)
    int32_t loop_capacity, loop_level;
    int32_t leaf_stride, pad0;
    int64_t off_leaf_tab;
    LevelDev levels[kMaxLevels];
};

// Fixed places in the plan image: the tensor maps (kMapsPerLevel per level,
// kMaxLevels slots), then one record per CTA of the fused kernel.
constexpr size_t kPlanMapsOff = (sizeof(PlanHeader) + 127) / 128 * 128;
constexpr size_t kPlanRecOff = kPlanMapsOff + (size_t)kMaxLevels * kMapsPerLevel * sizeof(CUtensorMap);
// The merge table follows the records.
inline size_t plan_tab_offset(int grid, int rec_stride)
{
    return (kPlanRecOff + (size_t)grid * rec_stride + 63) / 64 * 64;
}

// ------------------------------------------------------------ CTA records
// Everything one CTA of the fused kernel needs to start its work, fetched
// with a single bulk copy: its items (tensor-core items first) and the page
// ids of their key ranges.  The page of key t of an item is
// pages[page_off + t / ps - k0 / ps].
struct RecHead {
    uint64_t tag;
    int32_t n_tc, n_small;
    int32_t n_pages;
    int32_t pad[3];
};
struct RecItem {
    int32_t seq_begin, n_seq, kvh, k0, k1, part_row;
    int32_t level, page_off;  // level: the pool slot (tensor maps) of the item's keys
    int32_t ps, box, num_pages;
    int32_t len_seq;  // decode-loop suffix items: the sequence whose current length ends [k0, k1); else -1
};
static_assert(sizeof(RecHead) == 32 && sizeof(RecItem) == 48, "record layout");
constexpr int kRecMaxBytes = 8192;

// ----------------------------------------------------------- kernel params
// Standalone tensor-core kernel over a contiguous prefix (hp_prefix_attn).
struct TcParams {
    CUtensorMap map_k;  // [len][Hkv][d]: box 64 columns x 1 head x 128 tokens
    CUtensorMap map_v;
    CUtensorMap map_q;  // [B][Hq][d]: box 64 columns x G heads x (128 / G) rows
    CUtensorMap map_o;  // partial O [rows][d] bf16: box 64 columns x 128 rows
    int32_t G, Hkv;
    float scale_log2;   // softmax scale * log2(e)
    int32_t n_items;    // item i owns partial rows [256 i, 256 i + 256)
    int32_t imp_row_begin, imp_rows, imp_seqs_per_item, imp_split_len, imp_n_split, imp_len;
    float *part_lse;
    uint32_t *status;
};

// Standalone paged decode kernel (hp_suffix_decode_paged and its
// allocation-free variant): items (b, kvh group, split) from a page table.
struct SmallParams {
    CUtensorMap map_k;  // head-group boxes: 64 columns x 16 tokens x nh heads
    CUtensorMap map_v;
    CUtensorMap map_q;  // [B][Hq][d]: box 64 columns x (nh * G) heads x 1 row
    int32_t G, Hkv;
    float scale_log2;
    int32_t n_items;
    const int32_t *page_table;
    int32_t pt_stride;
    const int32_t *seq_lens;
    int32_t B, num_pages, page_size, split_len, n_split;
    int32_t nh;  // KV heads per item (a group of consecutive heads; 1, 2 or 4)
    int32_t q_slot;  // map_q is valid (nh * G <= small_q_rows()): Q rows arrive with each item's first chunk
    const uint16_t *q;  // otherwise the consumers read q[b][h][:] themselves
    int64_t q_sb, q_sh;
    uint16_t *part_o;   // bf16
    float *part_lse;
    uint32_t *status;
    // E4M3 pools (q8 != 0): codes [num_pages][Hkv][page_size][d] bytes, scales
    // of (page, KV head) at k_scale / v_scale[page * Hkv + head]
    int32_t q8;
    const float *k_scale;
    const float *v_scale;
};

// Parallel Prompting rows (hp_stream_decode): items (request, KV-head group,
// stream block, key split) over each request's one KV row, with the stream
// mask applied per key.
struct StreamParams {
    CUtensorMap map_k;  // head-group boxes: 64 columns x 16 tokens x nh heads
    CUtensorMap map_v;
    int32_t G, Hkv;
    float scale_log2;
    int32_t n_items;
    int32_t R, P;          // requests, streams per request (query sequence r * P + s)
    const int32_t *row_pages;  // [R][pt_stride] page ids of each request's row
    int32_t pt_stride;
    const int32_t *row_len;    // [R] slots of each row
    const int32_t *slot_sid;   // [R][sid_stride] stream id per slot (-1: document)
    const int32_t *slot_pos;   // [R][sid_stride] position per slot
    int32_t sid_stride;
    const int32_t *q_sid;      // [R * P] stream id of each query
    const int32_t *q_pos;      // [R * P] position of each query
    int32_t num_pages, page_size, split_len, n_split;
    int32_t nh;                // KV heads per item
    int32_t n_sg, ns_pg;       // stream groups per item (one consumer warp each per head), streams per group
    int32_t spi, n_sblk;       // streams per item (n_sg * ns_pg), stream blocks per request
    int32_t rows_item;         // partial rows per item: nh * n_sg * ns_pg * G
    int32_t sc;                // chunks of 16 keys per ring stage (1, 2 or 4; sc * nh <= 8)
    const uint16_t *q;
    int64_t q_sb, q_sh;
    uint16_t *part_o;
    float *part_lse;
    uint32_t *status;
};

// Fused cascade kernel (tensor-core and paged roles, one persistent launch).
struct CascadeParams {
    CUtensorMap q_tc;      // box 64 columns x G heads x (128 / G) rows
    CUtensorMap q_sm;      // box 64 columns x (nh * G) heads x 1 row
    CUtensorMap o_tc;      // partial O [rows][d] bf16: box 64 columns x 128 rows (tensor-core stores)
    const uint8_t *plan;   // plan image (maps at kPlanMapsOff, records at kPlanRecOff)
    uint64_t tag;
    int32_t rec_stride;
    int32_t num_levels;
    int32_t G, small_nh;
    int32_t q_slot;        // q_sm is valid (small_nh * G <= cascade_q_rows())
    const uint16_t *q;     // otherwise the paged role reads q[b][h][:] itself
    int64_t q_sb, q_sh;
    float scale_log2;
    uint16_t *part_o;      // bf16 (paged role; the tensor-core role stores through o_tc)
    float *part_lse;
    uint32_t *status;
    int32_t withhold;      // failure detection tests: CTA 0 withholds its first K tile
    // decode-loop plans: suffix item ends come from suffix_len[len_seq]
    const int32_t *suffix_len;
    int32_t loop_capacity;
    // the append fused into the step (k_new != null): the suffix of sequence
    // b also holds the token k_new / v_new[b] at position suffix_len[b], which
    // the paged producer writes into the suffix pools (bf16
    // [num_pages][Hkv][ps][d]) before it loads that chunk
    const uint16_t *k_new;
    const uint16_t *v_new;
    int64_t kv_sb, kv_sh;
    uint16_t *loop_k_pool;
    uint16_t *loop_v_pool;
    int32_t Hkv, d;
    // trees whose paged levels hold E4M3 codes (q8 != 0): the scales of each
    // pool slot, (page, KV head) at k_scale[slot][page * Hkv + head]
    int32_t q8;
    const float *k_scale[kMaxLevels];
    const float *v_scale[kMaxLevels];
};

// Decode-loop append: one token per sequence into its suffix pages.
// Copy-in of host-resident queries (hp_host_io_kernel.cu): src rows
// (b, h) at src + b * sb + h * sh (elements, device-accessible address of
// page-locked host memory) to dst[(b * Hq + h) * d ..] in device memory.
struct StageParams {
    const uint16_t *src;
    int64_t sb, sh;
    int B, Hq, d;
    uint16_t *dst;
};

struct AppendParams {
    const int32_t *leaf_tab;  // [B][leaf_stride] page ids (the plan's)
    int32_t leaf_stride, capacity, page_size, num_pages;
    int32_t B, Hkv, d;
    uint16_t *k_pool;  // bf16 [num_pages][Hkv][page_size][d]
    uint16_t *v_pool;
    const uint16_t *k_new;  // bf16 row (b, h) at b*kv_sb + h*kv_sh
    const uint16_t *v_new;
    int64_t kv_sb, kv_sh;
    int32_t *suffix_len;
    uint32_t *status;
};

// Merge kernel: combines the partial rows of each output row.
struct MergeParams {
    const uint16_t *part_o;  // bf16
    const float *part_lse;
    int32_t d, G, Hq, Hkv, B;
    // plan mode (plan != nullptr): the plan's merge table, one row per (b, kvh)
    const PlanHeader *plan;
    uint64_t tag;
    const int32_t *tab;
    int32_t tab_stride;
    // implicit modes (plan == nullptr)
    int32_t mode;            // 1: paged decode splits; 2: contiguous prefix splits; 3: stream rows
    const int32_t *seq_lens; // mode 1
    int32_t split_len, n_split, seqs_per_item, row_begin, rows, n_rc;
    int32_t nh;  // mode 1, 3: KV heads per item
    // mode 3 (Parallel Prompting rows; seq_lens = the rows' lengths [R])
    int32_t P, spi, n_sblk, ns_pg, n_sg, rows_item;
    int32_t wait_prior;  // launched as a programmatic dependent: wait for the prior grid first
    void *out;
    int32_t out_f32;
    int64_t o_sb, o_sh;
    float *lse;
    int64_t lse_sb;
    uint32_t *status;
    // the append fused into the step: after the partial states are complete,
    // suffix_len[b] < len_capacity moves on by one (row (b, 0) does it)
    int32_t *len_inc;
    int32_t len_capacity;
};

template <typename T>
__host__ __device__ inline const T *plan_array(const PlanHeader *h, int64_t off)
{
    return reinterpret_cast<const T *>(reinterpret_cast<const uint8_t *>(h) + off);
}

// Launchers (return the cudaGetLastError() after the launch).
cudaError_t launch_tc(const TcParams &p, int grid, int d, cudaStream_t s);
cudaError_t launch_small(const SmallParams &p, int grid, int d, cudaStream_t s);
cudaError_t launch_stream(const StreamParams &p, int grid, int d, cudaStream_t s);
cudaError_t launch_merge(const MergeParams &p, int64_t out_rows, cudaStream_t s);
// The merge as a programmatic dependent launch of the preceding kernel.
cudaError_t launch_merge_dependent(const MergeParams &p, int64_t out_rows, cudaStream_t s);
cudaError_t launch_cascade(const CascadeParams &p, int grid, int d, cudaStream_t s);
cudaError_t launch_append(const AppendParams &p, cudaStream_t s);
cudaError_t launch_stage(const StageParams &p, cudaStream_t s);
int cascade_heads_per_item(int Hkv);
int cascade_q_rows();  // paged-role Q slot rows of the fused kernel
int small_q_rows();    // Q slot rows of the standalone paged kernel
cudaError_t launch_merge2(const float *oa, const float *la, const float *ob, const float *lb,
                          void *o, int out_f32, float *lse, int64_t rows, int d, cudaStream_t s);
size_t tc_smem_bytes(int d);
// TMA map of the queries q[b][h][:] (bf16, strides in elements): box 64
// columns x box_h heads x box_b rows, 128-byte swizzle.
bool encode_q_map(CUtensorMap *m, const void *q, int B, int Hq, int d, int64_t q_sb, int64_t q_sh, int box_h,
                  int box_b);
// Rows of a tensor-core item: block mb of 128 / G sequences owns partial rows
// part_row + 128 mb .. + 127; sequence s, head g of the item is row
// part_row + 128 (s / spb) + (s % spb) G + g with spb = 128 / G.
__host__ __device__ inline int64_t tc_part_row(int64_t part_row, int s, int g, int G)
{
    const int spb = kTcTile / G;
    return part_row + (int64_t)(s / spb) * kTcTile + (int64_t)(s % spb) * G + g;
}
size_t small_smem_bytes(int d, bool q8 = false);
int small_heads_per_item(int Hkv);

}  // namespace hp
