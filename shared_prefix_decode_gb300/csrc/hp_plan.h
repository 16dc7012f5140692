// hp_plan.h -- the host planner of the cascade step: from a tree descriptor
// to work items, the persistent kernel's schedule records and the merge
// table (ChunkAttention's context generation, "Context Generation and
// GPU-CPU Coordination"; Hydragen's "Hierarchical Sharing").
#pragma once

#include <cstdint>
#include <vector>

#include "hp_internal.h"

namespace hp {

// A node as the planner schedules it: a tree node, or several single-sequence
// nodes of one sequence fused into one (their keys back to back, over the
// concatenation of their page lists).
struct PNode {
    int level;  // the level whose pools and tensor maps the items use
    int seq_begin, seq_end;
    int64_t kv_len;
    int32_t page_base;  // index in the plan's page-id list of the node's first page
    bool loop;          // a decode-loop suffix (grows at run time)
};

// One item for the scheduler: its modelled cost and its record bytes.
struct Job {
    double cost;
    int32_t id;
    bool tc;
    int64_t rec_bytes;
};

struct HostPlan {
    PlanHeader hdr;
    std::vector<PNode> nodes;
    std::vector<CUtensorMap> maps;
    std::vector<WorkItem> tc, small;
    std::vector<int32_t> page_ids;     // all levels' page ids, concatenated
    std::vector<int32_t> level_ps;     // page size per level
    std::vector<int32_t> level_slot;   // pool slot of each level (levels with the same pools share one)
    std::vector<int32_t> level_kv;     // hp_kv_type of each level
    // per pool slot: hp_kv_type and the E4M3 scale arrays (device pointers)
    std::vector<int32_t> slot_kv;
    std::vector<const float *> slot_k_scale, slot_v_scale;
    bool q8 = false;  // the paged levels hold E4M3 codes
    std::vector<int32_t> merge_tab;  // [B*Hkv][merge_stride]
    std::vector<int32_t> leaf_tab;   // decode loop: [B][leaf_stride] suffix page ids
    std::vector<std::vector<int32_t>> cta_tc, cta_small;  // item ids per CTA of the fused kernel
    // the items as scheduler jobs, longest first (tensor-core, paged, both),
    // valid until make_items runs again
    std::vector<Job> jobs_tc, jobs_sm, jobs_all;
    bool jobs_ready = false;
    std::vector<std::vector<uint8_t>> records;           // one per CTA, without the tag
    std::vector<int32_t> contexts;  // (level, node, seq_begin, seq_end, pass) x n
};

// Page ids an item's record entry holds: the pages of keys [k0, k1).
inline int64_t item_pages(const WorkItem &w, int ps) { return (int64_t)(w.k1 - 1) / ps - w.k0 / ps + 1; }

// Checks a tree descriptor (HP_OK, HP_ERR_ARG or HP_ERR_UNSUPPORTED).
hp_status validate_desc(const hp_tree_desc *d);

// Context list in the pages' order: shared nodes level by level, then each
// sequence's private nodes in level order; (level, node, seq_begin, seq_end,
// batched) per entry.
void build_contexts(const hp_tree_desc *d, std::vector<int32_t> &out);

// The whole plan of a tree into P (capacity > 0: a decode-loop plan);
// `encode` also encodes the TMA descriptors of the pools.
hp_status build_plan(const hp_tree_desc *d, HostPlan &P, bool encode, int capacity = 0);

}  // namespace hp
