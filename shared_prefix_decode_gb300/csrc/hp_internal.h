// hp_internal.h -- structures shared by the host library and the kernels:
// the device-resident plan (work items, page ids, merge lists, TMA tensor
// maps) and the launch entry points of each kernel translation unit.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/hp.h"

namespace hp {

constexpr int kMaxLevels = 8;
constexpr uint32_t kPlanMagic = 0x31504C48u;  // "HLP1"
constexpr int kTcTile = 128;                  // keys per tensor-core tile
constexpr int kTcMaxRows = 256;               // query rows per tensor-core item (2 x M=128)
constexpr int kSmallRows = 16;                // query rows per small item (one m16 tile)
constexpr int kChunk = 16;                    // keys per small-kernel chunk
constexpr size_t kWsHeader = 256;             // status word + reserved

// Device status bits (the first word of every workspace).
enum : uint32_t { kStBounds = 1u, kStTimeout = 2u, kStPlan = 4u };

// One unit of work: query rows (sequences [seq_begin, seq_begin+n_seq) x the
// G heads of KV head kvh) against keys [k0, k1) of one tree node.  Its rows
// land in partial rows part_row + s*G + g.
struct WorkItem {
    int32_t level;
    int32_t seq_begin;
    int32_t n_seq;
    int32_t kvh;
    int32_t k0, k1;
    int32_t page_base;  // index in the plan's page-id array of the node's first page
    int32_t part_row;
};
static_assert(sizeof(WorkItem) == 32, "WorkItem layout");

struct LevelDev {
    const void *k_pool;
    const void *v_pool;
    int32_t num_pages;
    int32_t page_size;
    int32_t tc_box;     // tokens per TMA box of the tensor-core maps (gcd(page_size, 128))
    int32_t pad;
};

// Tensor maps per level: [0] K for the tensor-core kernel, [1] V likewise,
// [2] K for the small kernel (16-token boxes), [3] V likewise.
constexpr int kMapsPerLevel = 4;

struct alignas(64) PlanHeader {
    uint32_t magic;
    uint32_t version;
    uint64_t tag;
    int32_t B, Hq, Hkv, d, G, num_levels;
    int32_t n_tc, n_small, n_part_rows, n_merge;
    int32_t small_nh;       // KV heads per small-row item
    int32_t grid;           // CTAs of the fused kernel (one schedule per CTA)
    int64_t off_maps;       // byte offsets from the plan base
    int64_t off_tc;
    int64_t off_small;
    int64_t off_page_ids;
    int64_t off_merge_ptr;  // [B*Hkv + 1] int32
    int64_t off_merge_idx;  // [n_merge] int32: partial row of (b, g = 0)
    int64_t off_cta_ptr;    // [grid + 1] int32: each CTA's schedule in cta_items
    int64_t off_cta_ntc;    // [grid] int32: how many of them are tensor-core items
    int64_t off_cta_items;  // int32: tensor-core item i as i, small item j as n_tc + j
    int64_t total_bytes;
    int64_t ws_bytes;
    int64_t ws_off_lse;     // byte offsets into the workspace
    int64_t ws_off_o;
    LevelDev levels[kMaxLevels];
};

// ----------------------------------------------------------- kernel params
// Tensor-core (prefix / shared-node) kernel.
struct TcParams {
    CUtensorMap map_k;  // used when maps == nullptr (contiguous prefix)
    CUtensorMap map_v;
    const uint16_t *q;
    int64_t q_sb, q_sh;
    int32_t G, Hkv;
    float scale_log2;   // softmax scale * log2(e)
    // item source: the device plan (items, maps, page ids are found through
    // its header), or implicit items over a contiguous prefix (plan == nullptr)
    const PlanHeader *plan;
    uint64_t tag;             // expected plan tag (plan mode)
    int32_t n_items;
    // implicit mode
    int32_t imp_row_begin, imp_rows, imp_seqs_per_item, imp_split_len, imp_n_split, imp_len;
    float *part_o;
    float *part_lse;
    uint32_t *status;
};

// Small-row (paged decode) kernel.
struct SmallParams {
    CUtensorMap map_k;  // used when maps == nullptr (standalone paged decode)
    CUtensorMap map_v;
    const uint16_t *q;
    int64_t q_sb, q_sh;
    int32_t G, Hkv;
    float scale_log2;
    // plan mode (plan != nullptr): items, maps and page ids via the header
    const PlanHeader *plan;
    uint64_t tag;
    int32_t n_items;
    // standalone mode: items (b, kvh, split) from the page table
    const int32_t *page_table;
    int32_t pt_stride;
    const int32_t *seq_lens;
    int32_t B, num_pages, page_size, split_len, n_split, seqs_per_item;
    int32_t nh;  // KV heads per item (a group of consecutive heads; 1, 2 or 4)
    float *part_o;
    float *part_lse;
    uint32_t *status;
};

// Fused cascade kernel (tensor-core and paged roles, one persistent launch).
struct CascadeParams {
    const PlanHeader *plan;
    uint64_t tag;
    const uint16_t *q;
    int64_t q_sb, q_sh;
    float scale_log2;
    float *part_o;
    float *part_lse;
    uint32_t *status;
};

// Merge kernel: combines the partial rows of each output row.
struct MergeParams {
    const float *part_o;
    const float *part_lse;
    int32_t d, G, Hq, Hkv, B;
    // plan mode (plan != nullptr): CSR over (b, kvh) found through the header
    const PlanHeader *plan;
    uint64_t tag;
    // implicit modes (plan == nullptr)
    int32_t mode;            // 1: paged decode splits; 2: contiguous prefix splits
    const int32_t *seq_lens; // mode 1
    int32_t split_len, n_split, seqs_per_item, row_begin, rows, n_rc;
    int32_t nh;  // mode 1: KV heads per small-kernel item
    int32_t wait_prior;  // launched as a programmatic dependent: wait for the prior grid first
    void *out;
    int32_t out_f32;
    int64_t o_sb, o_sh;
    float *lse;
    int64_t lse_sb;
    uint32_t *status;
};

template <typename T>
__host__ __device__ inline const T *plan_array(const PlanHeader *h, int64_t off)
{
    return reinterpret_cast<const T *>(reinterpret_cast<const uint8_t *>(h) + off);
}

// Launchers (return the cudaGetLastError() after the launch).
cudaError_t launch_tc(const TcParams &p, int grid, int d, cudaStream_t s);
cudaError_t launch_small(const SmallParams &p, int grid, int d, cudaStream_t s);
cudaError_t launch_merge(const MergeParams &p, int64_t out_rows, cudaStream_t s);
// The merge as a programmatic dependent launch of the preceding kernel.
cudaError_t launch_merge_dependent(const MergeParams &p, int64_t out_rows, cudaStream_t s);
cudaError_t launch_cascade(const CascadeParams &p, int grid, int d, cudaStream_t s);
int cascade_heads_per_item(int Hkv);
cudaError_t launch_merge2(const float *oa, const float *la, const float *ob, const float *lb,
                          void *o, int out_f32, float *lse, int64_t rows, int d, cudaStream_t s);
size_t tc_smem_bytes(int d);
size_t small_smem_bytes(int d);
int small_heads_per_item(int Hkv);

}  // namespace hp
