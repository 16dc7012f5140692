// hp_plan.cu -- the host planner: validation, planning nodes (with a
// sequence's own nodes fused), work items split along the key axis, the
// cost-model split of the persistent grid between the two roles, the
// longest-first schedule, the per-CTA records and the merge table.
#include <algorithm>
#include <cstring>
#include <numeric>
#include <queue>
#include <utility>
#include <vector>

#include "hp_host.h"
#include "hp_plan.h"

namespace hp {

namespace {

// Time model of the fused kernel (ns), from timelines of the step on GB300:
// every CTA waits for its record; a tensor-core item pays for its Q, the
// latency of its first tiles and its epilogue, then per 128-key tile (TMA
// and exp2 bound, proportional to d); a CTA with paged items waits for its
// first chunks, then each item streams its KV.
struct CostModel {
    // ns; a tensor-core tile costs tc_tile with two 128-row blocks, tc_tile1
    // with one (timelines: about 2.1-2.5 us and 1.85 us at d = 128; 2.6 us
    // gave the shortest steps over 2.0-3.3 us on the workloads with many
    // tiles per CTA: document + streams 165.4 against 167.9 us at 2.3,
    // CodeLlama-13b with E4M3 suffixes 227.6 against 236.1)
    double cta = 1500, tc_item = 6000, tc_tile = 2600, tc_tile1 = 1850, sm_start = 1000, sm_item = 200,
           sm_bytes_per_ns = 60;
    double tc(const WorkItem &w, int G, int d) const
    {
        const bool two = w.n_seq > kTcTile / G;
        return tc_item + (two ? tc_tile : tc_tile1) * (double)ceil_div(w.k1_model - w.k0, kTcTile) * d / 128.0;
    }
    // a paged item loads its keys and values once for all its sequences
    // (bytes_kv: bytes of one key's K and V elements, 4 for bf16, 2 for E4M3)
    double small(const WorkItem &w, int d, int nh, int bytes_kv = 4) const
    {
        return sm_item + (double)(w.k1_model - w.k0) * nh * d * bytes_kv / sm_bytes_per_ns;
    }
};


// Longest-first greedy assignment of `jobs` to CTAs [c0, c1), each CTA's
// record kept within kRecMaxBytes; false when a job fits no record.
bool lpt(const std::vector<Job> &jobs, int c0, int c1, std::vector<double> &load, std::vector<int64_t> &used,
         std::vector<int> &n_sm, std::vector<std::vector<int32_t>> *tc_of, std::vector<std::vector<int32_t>> *sm_of,
         double start_cost)
{
    // the least-loaded CTA with room in its record (the lowest index among
    // equal loads), from a heap of (load, CTA)
    using Slot = std::pair<double, int>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int c = c0; c < c1; ++c)
        heap.push({load[c], c});
    std::vector<Slot> full;
    for (const Job &j : jobs) {
        int best = -1;
        while (!heap.empty()) {
            const Slot e = heap.top();
            heap.pop();
            if (used[e.second] + j.rec_bytes <= kRecMaxBytes) {
                best = e.second;
                break;
            }
            full.push_back(e);
        }
        for (const Slot &e : full)
            heap.push(e);
        full.clear();
        if (best < 0)
            return false;
        if (!j.tc && n_sm[best]++ == 0)
            load[best] += start_cost;
        if (tc_of)
            (j.tc ? *tc_of : *sm_of)[best].push_back(j.id);
        load[best] += j.cost;
        used[best] += j.rec_bytes;
        heap.push({load[best], best});
    }
    return true;
}

// Schedule of the fused kernel's items over `grid` CTAs: CTAs [0, n_tc_ctas)
// take the tensor-core items, the others the paged items -- or, `mixed`,
// every CTA the paged items once its tensor-core items are done (n_tc_ctas =
// grid: every CTA may take both, tensor-core items first).  Returns the
// modelled makespan, or a negative value when the records cannot hold the
// items.
double schedule(HostPlan &P, int grid, int n_tc_ctas, bool mixed, int d, const CostModel &cm, bool record = true)
{
    if (!P.jobs_ready) {
        auto longest_first = [](std::vector<Job> &v) {
            std::stable_sort(v.begin(), v.end(), [](const Job &a, const Job &b) { return a.cost > b.cost; });
        };
        P.jobs_tc.clear();
        P.jobs_sm.clear();
        for (size_t i = 0; i < P.tc.size(); ++i) {
            const WorkItem &w = P.tc[i];
            P.jobs_tc.push_back({cm.tc(w, P.hdr.G, d), (int32_t)i, true,
                                 (int64_t)sizeof(RecItem) + 4 * item_pages(w, P.level_ps[w.level])});
        }
        const int nh = P.hdr.small_nh;
        for (size_t j = 0; j < P.small.size(); ++j) {
            const WorkItem &w = P.small[j];
            // an E4M3 chunk is half the bytes, but decoding its codes costs the
            // consumers about as long as a bf16 chunk takes to stream (ncu:
            // the E4M3 role executes twice the instructions per key):
            // modelled at the bf16 rate per key when the item is consumed two
            // chunks per pass, at 1.5 times that rate chunk by chunk (timed
            // on the benchmarked shape with E4M3 suffixes and on CodeLlama-13b)
            const bool paired = ceil_div(w.k1_model - w.k0, (int64_t)kChunk) >= kPairChunks;
            P.jobs_sm.push_back({cm.small(w, d, nh, P.q8 && !paired ? 6 : 4), (int32_t)j, false,
                                 (int64_t)sizeof(RecItem) + 4 * item_pages(w, P.level_ps[w.level])});
        }
        P.jobs_all = P.jobs_tc;
        P.jobs_all.insert(P.jobs_all.end(), P.jobs_sm.begin(), P.jobs_sm.end());
        longest_first(P.jobs_tc);
        longest_first(P.jobs_sm);
        longest_first(P.jobs_all);
        P.jobs_ready = true;
    }
    const std::vector<Job> &tcj = P.jobs_tc, &smj = P.jobs_sm;
    std::vector<double> load(grid, cm.cta);
    std::vector<int64_t> used(grid, (int64_t)sizeof(RecHead));
    std::vector<int> n_sm(grid, 0);
    auto *tc_of = record ? &P.cta_tc : nullptr;
    auto *sm_of = record ? &P.cta_small : nullptr;
    if (record) {
        P.cta_tc.assign(grid, {});
        P.cta_small.assign(grid, {});
    }
    bool ok;
    if (n_tc_ctas >= grid) {
        ok = lpt(P.jobs_all, 0, grid, load, used, n_sm, tc_of, sm_of, cm.sm_start);
    } else {
        ok = lpt(tcj, 0, n_tc_ctas, load, used, n_sm, tc_of, sm_of, cm.sm_start) &&
             lpt(smj, mixed ? 0 : n_tc_ctas, grid, load, used, n_sm, tc_of, sm_of, cm.sm_start);
    }
    if (!ok)
        return -1.0;
    return *std::max_element(load.begin(), load.end());
}

// The records of the schedule in P (one per CTA, tag left zero).
void build_records(HostPlan &P)
{
    const int grid = (int)P.cta_tc.size();
    P.records.assign(grid, {});
    for (int c = 0; c < grid; ++c) {
        RecHead h{};
        h.n_tc = (int32_t)P.cta_tc[c].size();
        h.n_small = (int32_t)P.cta_small[c].size();
        std::vector<RecItem> items;
        std::vector<int32_t> pages;
        auto add = [&](const WorkItem &w) {
            const int ps = P.level_ps[w.level];
            const int slot = P.level_slot[w.level];
            const LevelDev &L = P.hdr.levels[slot];
            RecItem r{};
            r.seq_begin = w.seq_begin;
            r.n_seq = w.n_seq;
            r.kvh = w.kvh;
            r.k0 = w.k0;
            r.k1 = w.k1;
            r.part_row = w.part_row;
            r.level = slot;
            r.page_off = (int32_t)pages.size();
            r.ps = ps;
            r.box = L.tc_box;
            r.num_pages = L.num_pages;
            r.len_seq = w.len_seq;
            const int64_t first = w.k0 / ps, n = item_pages(w, ps);
            for (int64_t i = 0; i < n; ++i)
                pages.push_back(P.page_ids[(size_t)(w.page_base + first + i)]);
            items.push_back(r);
        };
        for (int32_t id : P.cta_tc[c])
            add(P.tc[id]);
        for (int32_t id : P.cta_small[c])
            add(P.small[id]);
        h.n_pages = (int32_t)pages.size();
        std::vector<uint8_t> &rec = P.records[c];
        rec.resize(sizeof(RecHead) + sizeof(RecItem) * items.size() + 4 * pages.size());
        std::memcpy(rec.data(), &h, sizeof(h));
        if (!items.empty())
            std::memcpy(rec.data() + sizeof(RecHead), items.data(), sizeof(RecItem) * items.size());
        if (!pages.empty())
            std::memcpy(rec.data() + sizeof(RecHead) + sizeof(RecItem) * items.size(), pages.data(),
                        4 * pages.size());
    }
}

// Work items of the tree for the given key splits (tensor-core items: one KV
// head, up to two blocks of 128 / G sequences; paged items: a group of nh KV
// heads of a node's sequences), with their partial rows and, when `lists`
// is given, the merge list of every (b, kvh).  Returns the partial row count.
// With capacity > 0 (a decode-loop plan) the last level's suffixes are split
// over their plan-time length as usual, but each suffix's last item reaches
// to the capacity (a suffix of length 0 gets one item [0, capacity)); at run
// time the items end at the sequence's current length.
int64_t make_items(const hp_tree_desc *d, int G, int nh, int64_t tc_split, int64_t small_split, HostPlan &P,
                   std::vector<std::vector<int32_t>> *lists, int capacity = 0)
{
    P.tc.clear();
    P.small.clear();
    P.jobs_ready = false;
    int64_t part = 0;
    for (const PNode &N : P.nodes) {
        const int l = N.level;
        const bool loop = N.loop;
        if (N.kv_len == 0 && !loop)
            continue;
        const int64_t klen = loop ? std::max<int64_t>(N.kv_len, 1) : N.kv_len;
        const int nseq = N.seq_end - N.seq_begin;
        const bool tc = (int64_t)nseq * G > kSmallRows;
        const int spc = tc ? 2 * (kTcTile / G) : nseq;
        const int64_t split = tc ? tc_split : small_split;
        // tensor-core items take one KV head; small-row items a group of
        // nh heads whose rows are laid out [head in group][sequence][g]
        const int hstep = tc ? 1 : nh;
        for (int s0 = N.seq_begin; s0 < N.seq_end; s0 += spc) {
            const int ns = std::min(spc, N.seq_end - s0);
            for (int kvh = 0; kvh < d->Hkv; kvh += hstep)
                for (int64_t k0 = 0; k0 < klen; k0 += split) {
                    WorkItem w;
                    w.level = l;
                    w.seq_begin = s0;
                    w.n_seq = ns;
                    w.kvh = kvh;
                    w.k0 = (int32_t)k0;
                    w.k1 = (int32_t)std::min<int64_t>(k0 + split, klen);
                    w.len_seq = loop ? s0 : -1;
                    w.k1_model = w.k1;
                    if (loop && w.k1 == klen) {
                        // reaches to the capacity; over the loop it holds
                        // half of the headroom on average
                        w.k1 = capacity;
                        w.k1_model = (int32_t)std::max<int64_t>(k0 + 1, (N.kv_len + (int64_t)capacity) / 2);
                    }
                    w.page_base = N.page_base;
                    w.part_row = (int32_t)std::min<int64_t>(part, INT32_MAX);
                    if (tc) {
                        // 128 rows per block of 128 / G sequences (the
                        // block is stored whole by a TMA tensor store)
                        if (lists)
                            for (int b = s0; b < s0 + ns; ++b)
                                (*lists)[(size_t)b * d->Hkv + kvh].push_back(
                                    (int32_t)std::min<int64_t>(tc_part_row(part, b - s0, 0, G), INT32_MAX));
                        part += ceil_div(ns, kTcTile / G) * kTcTile;
                    } else {
                        if (lists)
                            for (int hw = 0; hw < hstep; ++hw)
                                for (int b = s0; b < s0 + ns; ++b)
                                    (*lists)[(size_t)b * d->Hkv + kvh + hw].push_back(
                                        (int32_t)(part + ((int64_t)hw * ns + (b - s0)) * G));
                        part += (int64_t)ns * G * hstep;
                    }
                    (tc ? P.tc : P.small).push_back(w);
                }
        }
    }
    return part;
}


// A decode-loop tree: the last level holds one single-sequence node per
// sequence (node n covers sequence n), each with page ids for `capacity`
// tokens that no other node of the same pools uses, and every suffix's rows
// fit one paged item (G <= 16).
hp_status validate_loop(const hp_tree_desc *d, int capacity)
{
    if (capacity < 1 || capacity > (1 << 24))
        return HP_ERR_ARG;
    if (d->Hq / d->Hkv > kSmallRows)
        return HP_ERR_UNSUPPORTED;
    const int last = d->num_levels - 1;
    const hp_tree_level &S = d->levels[last];
    if (S.num_nodes != d->B)
        return HP_ERR_ARG;
    const int64_t cap_pages = ceil_div(capacity, S.page_size);
    std::vector<char> mine((size_t)S.num_pages, 0);
    for (int n = 0; n < S.num_nodes; ++n) {
        const hp_tree_node &N = S.nodes[n];
        if (N.seq_begin != n || N.seq_end != n + 1 || N.kv_len > capacity)
            return HP_ERR_ARG;
        if ((int64_t)N.page_off + cap_pages > S.num_page_ids)
            return HP_ERR_ARG;
        for (int64_t i = 0; i < cap_pages; ++i) {
            const int32_t pid = S.page_ids[N.page_off + i];
            if (pid < 0 || pid >= S.num_pages || mine[(size_t)pid])
                return HP_ERR_ARG;  // out of range, or reserved twice
            mine[(size_t)pid] = 1;
        }
    }
    // pages of the other levels in the same pools stay read-only
    for (int l = 0; l < last; ++l) {
        const hp_tree_level &L = d->levels[l];
        if (L.k_pool != S.k_pool && L.v_pool != S.v_pool && L.k_pool != S.v_pool && L.v_pool != S.k_pool)
            continue;
        for (int n = 0; n < L.num_nodes; ++n) {
            const hp_tree_node &N = L.nodes[n];
            const int64_t npg = ceil_div(N.kv_len, L.page_size);
            for (int64_t i = 0; i < npg; ++i) {
                const int32_t pid = L.page_ids[N.page_off + i];
                if (L.page_size != S.page_size || (pid < S.num_pages && mine[(size_t)pid]))
                    return HP_ERR_ARG;
            }
        }
    }
    return HP_OK;
}


// The nodes the planner schedules, level by level in tree order.  Several
// single-sequence nodes of one sequence on the paged path (G <= 16 rows) are
// fused into one: attention over a set of keys does not depend on their
// order, so one item can walk the nodes' keys back to back over the
// concatenation of their page lists.  That needs every node but the last to
// end on a page boundary, and all of them to use the same pools and page
// size.  The fused node takes the place of its first member; the sequence
// then has one partial state, not one per node, for the same bytes.  Nodes
// that grow in a decode loop stay on their own.
//
// A narrow shared node -- 2 or 3 sequences, still on the paged path, page
// aligned -- can join its sequences' chains too: each of them then reads the
// node's keys itself, and each loses a partial state and a merge part
// ("every merge has a cost", shared-prefix KV caching blog, "Prefix trees:
// multi-level sharing"; ChunkAttention's realistic trees have many such
// nodes).  It joins when the extra reads cost less than the merge parts they
// save (narrow_pays), and only when every one of its sequences has an own
// node to fuse it with.  Concatenated page lists are appended to P.page_ids.
namespace {

// Modelled cost of one more merge part per output row (ns): the merge
// kernel's time grows by about this much per part of its rows.
constexpr double kMergePartNs = 120.0;
// HBM bytes per ns the re-reads are charged at.
constexpr double kReadBytesPerNs = 6000.0;

bool narrow_pays(const hp_tree_desc *d, const hp_tree_node &N, int page_size, int G)
{
    const int ns = N.seq_end - N.seq_begin;
    if (ns < 2 || ns > 3 || ns * G > kSmallRows || N.kv_len <= 0 || N.kv_len % page_size)
        return false;
    const double extra = (double)(ns - 1) * N.kv_len * d->Hkv * d->d * 4.0 / kReadBytesPerNs;
    return extra < kMergePartNs;
}

}  // namespace

void plan_nodes(const hp_tree_desc *d, int G, int capacity, const std::vector<int32_t> &level_page_off, HostPlan &P)
{
    const int last = d->num_levels - 1;
    P.nodes.clear();
    auto fusable = [&](int l, const hp_tree_node &N) {
        return N.seq_end - N.seq_begin == 1 && G <= kSmallRows && N.kv_len > 0 && !(capacity > 0 && l == last);
    };
    auto same_pools = [&](int a, int b) {
        const hp_tree_level &A = d->levels[a], &Bl = d->levels[b];
        return A.k_pool == Bl.k_pool && A.v_pool == Bl.v_pool && A.num_pages == Bl.num_pages &&
               A.page_size == Bl.page_size && A.kv_type == Bl.kv_type && A.k_scale == Bl.k_scale &&
               A.v_scale == Bl.v_scale;
    };
    const int nl = d->num_levels;
    // own[l][b]: the fusable node of level l that covers only sequence b, or -1;
    // wide[l][b]: the narrow shared node of level l covering b, if it may join
    std::vector<std::vector<int>> own(nl, std::vector<int>(d->B, -1)), wide(nl, std::vector<int>(d->B, -1));
    std::vector<std::vector<char>> narrow(nl);
    for (int l = 0; l < nl; ++l) {
        narrow[l].assign(d->levels[l].num_nodes, 0);
        for (int n = 0; n < d->levels[l].num_nodes; ++n) {
            const hp_tree_node &N = d->levels[l].nodes[n];
            if (fusable(l, N))
                own[l][N.seq_begin] = n;
            else if (!(capacity > 0 && l == last) && narrow_pays(d, N, d->levels[l].page_size, G))
                narrow[l][n] = 1;
        }
    }
    // the chain of sequence b: its own nodes and the joining narrow nodes,
    // same pools as the first, page-aligned ones first, at most one ragged
    // node last
    auto chain_of = [&](int b) {
        std::vector<std::pair<int, int>> cand;
        for (int l = 0; l < nl; ++l) {
            int n = own[l][b];
            if (n < 0)
                n = wide[l][b];
            if (n >= 0 && (cand.empty() || same_pools(cand[0].first, l)))
                cand.emplace_back(l, n);
        }
        std::vector<std::pair<int, int>> chain;
        int ragged = -1;
        for (size_t i = 0; i < cand.size(); ++i) {
            const hp_tree_level &L = d->levels[cand[i].first];
            if (L.nodes[cand[i].second].kv_len % L.page_size == 0)
                chain.push_back(cand[i]);
            else if (ragged < 0)
                ragged = (int)i;
        }
        if (ragged >= 0)
            chain.push_back(cand[ragged]);
        return chain;
    };
    auto has_own = [&](const std::vector<std::pair<int, int>> &ch) {
        for (const auto &m : ch)
            if (own[m.first][d->levels[m.first].nodes[m.second].seq_begin] == m.second &&
                d->levels[m.first].nodes[m.second].seq_end - d->levels[m.first].nodes[m.second].seq_begin == 1)
                return true;
        return false;
    };
    // Narrow nodes join when every one of their sequences' chains takes them
    // along with an own node; otherwise they stay whole (each round only
    // withdraws nodes, so the rounds end).
    for (;;) {
        for (int l = 0; l < nl; ++l)
            std::fill(wide[l].begin(), wide[l].end(), -1);
        for (int l = 0; l < nl; ++l)
            for (int n = 0; n < d->levels[l].num_nodes; ++n)
                if (narrow[l][n]) {
                    const hp_tree_node &N = d->levels[l].nodes[n];
                    for (int b = N.seq_begin; b < N.seq_end; ++b)
                        wide[l][b] = n;
                }
        bool changed = false;
        for (int l = 0; l < nl; ++l)
            for (int n = 0; n < d->levels[l].num_nodes; ++n) {
                if (!narrow[l][n])
                    continue;
                const hp_tree_node &N = d->levels[l].nodes[n];
                bool ok = true;
                for (int b = N.seq_begin; b < N.seq_end && ok; ++b) {
                    const auto ch = chain_of(b);
                    ok = has_own(ch) && std::find(ch.begin(), ch.end(), std::make_pair(l, n)) != ch.end();
                }
                if (!ok) {
                    narrow[l][n] = 0;
                    changed = true;
                }
            }
        if (!changed)
            break;
    }
    for (int l = 0; l < nl; ++l)
        std::fill(wide[l].begin(), wide[l].end(), -1);
    for (int l = 0; l < nl; ++l)
        for (int n = 0; n < d->levels[l].num_nodes; ++n)
            if (narrow[l][n]) {
                const hp_tree_node &N = d->levels[l].nodes[n];
                for (int b = N.seq_begin; b < N.seq_end; ++b)
                    wide[l][b] = n;
            }
    // heads[l][n]: the fused chains that take the place of node (l, n) (a
    // narrow node heads one chain per sequence); skip[l][n]: fused away
    std::vector<std::vector<std::vector<std::vector<std::pair<int, int>>>>> heads(nl);
    std::vector<std::vector<char>> skip(nl);
    for (int l = 0; l < nl; ++l) {
        heads[l].assign(d->levels[l].num_nodes, {});
        skip[l].assign(d->levels[l].num_nodes, 0);
    }
    for (int b = 0; b < d->B; ++b) {
        const auto chain = chain_of(b);
        if (chain.size() < 2)
            continue;
        // the fused node sits where its first member (in tree order) was
        const auto head = *std::min_element(chain.begin(), chain.end());
        heads[head.first][head.second].push_back(chain);
        for (const auto &m : chain)
            skip[m.first][m.second] = 1;
    }
    for (int l = 0; l < nl; ++l) {
        const hp_tree_level &L = d->levels[l];
        for (int n = 0; n < L.num_nodes; ++n) {
            const auto &chains = heads[l][n];
            if (skip[l][n] && chains.empty())
                continue;
            const hp_tree_node &N = L.nodes[n];
            if (chains.empty()) {
                PNode pn;
                pn.level = l;
                pn.seq_begin = N.seq_begin;
                pn.seq_end = N.seq_end;
                pn.loop = capacity > 0 && l == last;
                pn.kv_len = N.kv_len;
                pn.page_base = level_page_off[l] + N.page_off;
                P.nodes.push_back(pn);
                continue;
            }
            for (const auto &ch : chains) {
                // the sequence of the chain: its own node's (a narrow head covers several)
                int b = -1;
                for (const auto &m : ch) {
                    const hp_tree_node &M = d->levels[m.first].nodes[m.second];
                    if (M.seq_end - M.seq_begin == 1)
                        b = M.seq_begin;
                }
                PNode pn;
                pn.level = l;
                pn.seq_begin = b;
                pn.seq_end = b + 1;
                pn.loop = false;
                pn.kv_len = 0;
                pn.page_base = (int32_t)P.page_ids.size();
                for (const auto &m : ch) {
                    const hp_tree_level &ML = d->levels[m.first];
                    const hp_tree_node &MN = ML.nodes[m.second];
                    const int64_t npg = ceil_div(MN.kv_len, ML.page_size);
                    P.page_ids.insert(P.page_ids.end(), ML.page_ids + MN.page_off, ML.page_ids + MN.page_off + npg);
                    pn.kv_len += MN.kv_len;
                }
                P.nodes.push_back(pn);
            }
        }
    }
}

}  // namespace

// Checks a tree descriptor.
hp_status validate_desc(const hp_tree_desc *d)
{
    if (!d || !d->levels || d->num_levels < 1 || d->B < 1 || d->Hq < 1 || d->Hkv < 1 || d->Hq % d->Hkv)
        return HP_ERR_ARG;
    if (d->num_levels > kMaxTreeLevels || !supported_d(d->d) || d->Hq / d->Hkv > kTcTile)
        return HP_ERR_UNSUPPORTED;
    for (int l = 0; l < d->num_levels; ++l) {
        const hp_tree_level &L = d->levels[l];
        if (L.num_nodes < 0 || L.num_page_ids < 0 || L.num_pages < 1)
            return HP_ERR_ARG;
        if (L.page_size < 16 || L.page_size > 256 || L.page_size % 16)
            return HP_ERR_UNSUPPORTED;
        if (!L.k_pool || !L.v_pool || !aligned(L.k_pool, 16) || !aligned(L.v_pool, 16))
            return HP_ERR_ARG;
        if (L.kv_type != HP_KV_BF16 && L.kv_type != HP_KV_E4M3)
            return HP_ERR_ARG;
        if (L.kv_type == HP_KV_E4M3) {
            if (d->d != 128)
                return HP_ERR_UNSUPPORTED;
            if (!L.k_scale || !L.v_scale || !aligned(L.k_scale, 4) || !aligned(L.v_scale, 4))
                return HP_ERR_ARG;
        }
        if ((L.num_nodes > 0 && !L.nodes) || (L.num_page_ids > 0 && !L.page_ids))
            return HP_ERR_ARG;
        std::vector<std::pair<int, int>> ranges;
        for (int n = 0; n < L.num_nodes; ++n) {
            const hp_tree_node &N = L.nodes[n];
            if (N.seq_begin < 0 || N.seq_end > d->B || N.seq_begin >= N.seq_end || N.kv_len < 0 || N.page_off < 0)
                return HP_ERR_ARG;
            const int64_t npg = ceil_div(N.kv_len, L.page_size);
            if ((int64_t)N.page_off + npg > L.num_page_ids)
                return HP_ERR_ARG;
            for (int64_t i = 0; i < npg; ++i) {
                const int32_t pid = L.page_ids[N.page_off + i];
                if (pid < 0 || pid >= L.num_pages)
                    return HP_ERR_ARG;
            }
            ranges.emplace_back(N.seq_begin, N.seq_end);
        }
        std::sort(ranges.begin(), ranges.end());
        for (size_t i = 1; i < ranges.size(); ++i)
            if (ranges[i].first < ranges[i - 1].second)
                return HP_ERR_ARG;  // nodes of one level must cover disjoint sequences
    }
    return HP_OK;
}

void build_contexts(const hp_tree_desc *d, std::vector<int32_t> &out)
{
    out.clear();
    for (int l = 0; l < d->num_levels; ++l)
        for (int n = 0; n < d->levels[l].num_nodes; ++n) {
            const hp_tree_node &N = d->levels[l].nodes[n];
            if (N.seq_end - N.seq_begin > 1)
                out.insert(out.end(), {l, n, N.seq_begin, N.seq_end, 1});
        }
    for (int b = 0; b < d->B; ++b)
        for (int l = 0; l < d->num_levels; ++l)
            for (int n = 0; n < d->levels[l].num_nodes; ++n) {
                const hp_tree_node &N = d->levels[l].nodes[n];
                if (N.seq_begin == b && N.seq_end == b + 1)
                    out.insert(out.end(), {l, n, N.seq_begin, N.seq_end, 0});
            }
}

hp_status build_plan(const hp_tree_desc *d, HostPlan &P, bool encode, int capacity)
{
    hp_status st = validate_desc(d);
    if (st == HP_OK && capacity != 0)
        st = validate_loop(d, capacity);
    if (st != HP_OK)
        return st;
    const int G = d->Hq / d->Hkv;
    const int sms = d->num_sms > 0 ? d->num_sms : device_sms();
    PlanHeader &H = P.hdr;
    std::memset(&H, 0, sizeof(H));
    H.magic = kPlanMagic;
    H.version = 1;
    H.B = d->B;
    H.Hq = d->Hq;
    H.Hkv = d->Hkv;
    H.d = d->d;
    H.G = G;

    // page ids of all levels, concatenated; one pool slot per distinct pool set
    std::vector<int32_t> level_page_off(d->num_levels);
    std::vector<int> slot_level;  // the first level of each slot
    P.level_ps.assign(d->num_levels, 0);
    P.level_slot.assign(d->num_levels, 0);
    P.level_kv.assign(d->num_levels, HP_KV_BF16);
    P.slot_kv.clear();
    P.slot_k_scale.clear();
    P.slot_v_scale.clear();
    for (int l = 0; l < d->num_levels; ++l) {
        const hp_tree_level &L = d->levels[l];
        P.level_ps[l] = L.page_size;
        P.level_kv[l] = L.kv_type;
        level_page_off[l] = (int32_t)P.page_ids.size();
        P.page_ids.insert(P.page_ids.end(), L.page_ids, L.page_ids + L.num_page_ids);
        int slot = 0;
        while (slot < (int)slot_level.size()) {
            const hp_tree_level &S = d->levels[slot_level[slot]];
            if (S.k_pool == L.k_pool && S.v_pool == L.v_pool && S.num_pages == L.num_pages &&
                S.page_size == L.page_size && S.kv_type == L.kv_type && S.k_scale == L.k_scale &&
                S.v_scale == L.v_scale)
                break;
            ++slot;
        }
        if (slot == (int)slot_level.size()) {
            if (slot == kMaxLevels)
                return HP_ERR_UNSUPPORTED;  // more distinct pools than a plan holds tensor maps for
            slot_level.push_back(l);
            LevelDev &LD = H.levels[slot];
            LD.k_pool = L.k_pool;
            LD.v_pool = L.v_pool;
            LD.num_pages = L.num_pages;
            LD.page_size = L.page_size;
            LD.tc_box = std::gcd(L.page_size, kTcTile);
            LD.pad = L.kv_type;
            P.slot_kv.push_back(L.kv_type);
            P.slot_k_scale.push_back(L.kv_type == HP_KV_E4M3 ? L.k_scale : nullptr);
            P.slot_v_scale.push_back(L.kv_type == HP_KV_E4M3 ? L.v_scale : nullptr);
        }
        P.level_slot[l] = slot;
    }
    H.num_levels = (int32_t)slot_level.size();

    plan_nodes(d, G, capacity, level_page_off, P);

    // E4M3 levels: only nodes of the per-sequence pass, and then every node
    // of that pass in an E4M3 level (the kernel's paged role runs one
    // storage); none in decode-loop plans
    P.q8 = false;
    for (int l = 0; l < d->num_levels; ++l)
        P.q8 = P.q8 || P.level_kv[l] == HP_KV_E4M3;
    if (P.q8) {
        if (capacity > 0)
            return HP_ERR_UNSUPPORTED;
        for (const PNode &N : P.nodes) {
            if (N.kv_len == 0)
                continue;
            const bool tc = (int64_t)(N.seq_end - N.seq_begin) * G > kSmallRows;
            if (tc == (P.level_kv[N.level] == HP_KV_E4M3))
                return HP_ERR_UNSUPPORTED;
        }
    }

    // Work sizes: 128-key tiles of the shared (tensor-core) nodes, 16-key
    // chunks of the paged ones.
    const int nh = cascade_heads_per_item(d->Hkv);
    H.small_nh = nh;
    int64_t tc_tiles = 0, small_chunks = 0;
    for (const PNode &N : P.nodes) {
        const int64_t rows = (int64_t)(N.seq_end - N.seq_begin) * G;
        if (N.kv_len == 0)
            continue;
        if (rows > kSmallRows) {
            const int spc = 2 * (kTcTile / G);
            tc_tiles += ceil_div(N.seq_end - N.seq_begin, spc) * d->Hkv * ceil_div(N.kv_len, kTcTile);
        } else {
            small_chunks += (int64_t)(d->Hkv / nh) * ceil_div(N.kv_len, kChunk);
        }
    }

    // Split of the CTAs between the two roles: n_tc CTAs run the tensor-core
    // items (about one each: the key split is the shared tiles over n_tc), the
    // others stream the paged items (about one each: fewer, longer items
    // mean fewer partial states for the merge; measured against three per
    // CTA, the benchmarked step 18.2 against 18.9 us, the per-sequence-only
    // workload 303.8 against 320.7); the n_tc with the shortest modelled
    // makespan wins.  Without one of the two kinds, or with
    // a single CTA, every CTA may take both.
    const CostModel cm;
    auto splits_for = [&](int n_tc_ctas, int64_t &tc_split, int64_t &small_split) {
        const int64_t per = std::max<int64_t>(1, ceil_div(tc_tiles, std::max(1, n_tc_ctas)));
        tc_split = kTcTile * std::min(kMaxTcTiles, per);
        const int n_sm = std::max(1, sms - (n_tc_ctas < sms ? n_tc_ctas : 0));
        // E4M3 paged items are bound by their consumers, not by HBM: with
        // long per-CTA work, four items per CTA spread it evenly (an item
        // per CTA leaves some CTAs two and others one when the nodes do not
        // divide by the CTAs; per-sequence-only workload 224.0 against
        // 254.5 us); with short work the extra items cost more than they
        // balance (benchmarked step with E4M3 suffixes: 21.6 against 19.8)
        const int64_t per_cta = ceil_div(small_chunks, (int64_t)n_sm);
        const int64_t parts = P.q8 && per_cta >= 64 ? 4 : 1;
        small_split = kChunk * std::max<int64_t>(2, ceil_div(small_chunks, (int64_t)n_sm * parts));
    };
    int best_k = sms;
    bool best_mixed = false;
    if (tc_tiles > 0 && small_chunks > 0 && sms > 1) {
        double best = -1.0;
        int64_t made_ts = -1, made_ss = -1;  // the splits P's items were made for
        for (int mixed = 0; mixed < 2; ++mixed)
            for (int k = 1; k < sms; ++k) {
                int64_t ts, ss;
                splits_for(k, ts, ss);
                if (ts != made_ts || ss != made_ss) {
                    make_items(d, G, nh, ts, ss, P, nullptr, capacity);
                    made_ts = ts;
                    made_ss = ss;
                }
                const double t = schedule(P, sms, k, mixed != 0, d->d, cm, false);
                if (t >= 0.0 && (best < 0.0 || t < best)) {
                    best = t;
                    best_k = k;
                    best_mixed = mixed != 0;
                }
            }
    }
    int64_t tc_split, small_split;
    splits_for(best_k, tc_split, small_split);

    // Items and partial rows, level by level; merge lists per (b, kvh).
    std::vector<std::vector<int32_t>> lists((size_t)d->B * d->Hkv);
    const int64_t part = make_items(d, G, nh, tc_split, small_split, P, &lists, capacity);
    if (part > INT32_MAX)
        return HP_ERR_UNSUPPORTED;
    // merge table: one row per (b, kvh), its count then its partial rows
    size_t max_parts = 0, n_merge = 0;
    for (const auto &l : lists) {
        max_parts = std::max(max_parts, l.size());
        n_merge += l.size();
    }
    H.merge_stride = (int32_t)round_up(max_parts + 1, 4);
    P.merge_tab.assign(lists.size() * (size_t)H.merge_stride, 0);
    for (size_t i = 0; i < lists.size(); ++i) {
        int32_t *row = &P.merge_tab[i * (size_t)H.merge_stride];
        row[0] = (int32_t)lists[i].size();
        std::copy(lists[i].begin(), lists[i].end(), row + 1);
    }
    H.n_tc = (int32_t)P.tc.size();
    H.n_small = (int32_t)P.small.size();
    H.grid = sms;
    if (schedule(P, sms, best_k, best_mixed, d->d, cm) < 0.0)
        return HP_ERR_UNSUPPORTED;  // the step's page lists exceed what the CTAs' records hold
    build_records(P);
    H.n_part_rows = (int32_t)part;
    H.n_merge = (int32_t)n_merge;

    // device layout: header, maps and records at fixed offsets, merge lists
    size_t rec_max = sizeof(RecHead);
    for (const auto &r : P.records)
        rec_max = std::max(rec_max, r.size());
    H.rec_stride = (int32_t)round_up(rec_max, 128);
    size_t off = plan_tab_offset(sms, H.rec_stride);
    H.off_merge_tab = (int64_t)off;
    off += 4 * P.merge_tab.size();
    if (capacity > 0) {
        // each sequence's suffix pages, for the appends of the loop
        const int last = d->num_levels - 1;
        const hp_tree_level &S = d->levels[last];
        H.loop_capacity = capacity;
        H.loop_level = last;
        H.leaf_stride = (int32_t)ceil_div(capacity, S.page_size);
        off = round_up(off, 64);
        H.off_leaf_tab = (int64_t)off;
        P.leaf_tab.assign((size_t)d->B * H.leaf_stride, 0);
        for (int b = 0; b < d->B; ++b)
            std::copy(S.page_ids + S.nodes[b].page_off, S.page_ids + S.nodes[b].page_off + H.leaf_stride,
                      P.leaf_tab.begin() + (size_t)b * H.leaf_stride);
        off += 4 * P.leaf_tab.size();
    }
    H.total_bytes = (int64_t)round_up(off, 256);
    const WsLayout ws = ws_layout(part, d->d);
    H.ws_off_lse = (int64_t)ws.off_lse;
    H.ws_off_o = (int64_t)ws.off_o;
    H.ws_bytes = (int64_t)ws.total;

    build_contexts(d, P.contexts);

    if (encode) {
        P.maps.resize((size_t)kMapsPerLevel * slot_level.size());
        for (size_t sl = 0; sl < slot_level.size(); ++sl) {
            const hp_tree_level &L = d->levels[slot_level[sl]];
            const int tcb = H.levels[sl].tc_box;
            CUtensorMap *m = &P.maps[sl * kMapsPerLevel];
            if (L.kv_type == HP_KV_E4M3) {
                // paged boxes only; the tensor-core slots hold copies (never used)
                if (!encode_pool_map(m + 2, L.k_pool, L.num_pages, d->Hkv, L.page_size, d->d, kChunk, nh, true) ||
                    !encode_pool_map(m + 3, L.v_pool, L.num_pages, d->Hkv, L.page_size, d->d, kChunk, nh, true))
                    return HP_ERR_CUDA;
                m[0] = m[2];
                m[1] = m[3];
                continue;
            }
            if (!encode_pool_map(m + 0, L.k_pool, L.num_pages, d->Hkv, L.page_size, d->d, tcb) ||
                !encode_pool_map(m + 1, L.v_pool, L.num_pages, d->Hkv, L.page_size, d->d, tcb) ||
                !encode_pool_map(m + 2, L.k_pool, L.num_pages, d->Hkv, L.page_size, d->d, kChunk, nh) ||
                !encode_pool_map(m + 3, L.v_pool, L.num_pages, d->Hkv, L.page_size, d->d, kChunk, nh))
                return HP_ERR_CUDA;
        }
    }
    return HP_OK;
}

}  // namespace hp
