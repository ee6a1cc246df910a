// cascade_plan.cu -- host-side grouping of sequences for cascade attention.
//
// The pages offer cascade attention as an opt-in for groups of sequences that
// share a long enough whole-page prefix, gated by a minimum member count and a
// minimum number of shared pages [mlxcel manual "KV Cache", §"Paged Decode
// Storage and Kernels"; the CASCADE_MIN_MEMBERS / CASCADE_MIN_SHARED_PAGES
// controls].  They do not say how the groups are found; this planner reads the
// plainest meaning of "share a prefix" for a paged cache: the same physical
// blocks at the same leading positions of the block tables.
//
//   1. A sequence's whole pages are its first min(ctx / 16, max_blocks) blocks.
//   2. Sequences with at least min_shared_blocks whole pages are sorted by
//      their whole-page block ids (lexicographic, a shorter list that is a prefix
//      of a longer one first, ties by index), so that sequences sharing deeper
//      prefixes sit next to each other.
//   3. A run of neighbours whose pairwise common prefix is at least
//      min_shared_blocks forms a group; groups of fewer than min_members are
//      dropped.
//   4. A group is cut into ceil(n / item_width) items of near-equal size, in
//      sorted order; an item shares the minimum common prefix of its adjacent
//      members, and items smaller than min_members are dropped.
// Pure host code: no CUDA call.
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

struct TableView {
    const int32_t* bt;
    int32_t max_blocks;
    const int32_t* row(int s) const { return bt + size_t(s) * max_blocks; }
};

int common_prefix(const TableView& t, int a, int la, int b, int lb) {
    const int n = std::min(la, lb);
    const int32_t* ra = t.row(a);
    const int32_t* rb = t.row(b);
    int i = 0;
    while (i < n && ra[i] == rb[i]) ++i;
    return i;
}

}  // namespace

extern "C" pkv_status pkv_cascade_plan(const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
                                       int32_t max_blocks_per_seq, int32_t min_members, int32_t min_shared_blocks,
                                       int32_t item_width, int32_t max_items, int32_t* members, int32_t* item_blocks,
                                       int32_t* num_items) {
    if (!num_items) return PKV_ERR_INVALID_ARG;
    *num_items = 0;
    if (num_seqs < 0 || max_blocks_per_seq < 0 || item_width < 1 || item_width > 16 || max_items < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!block_tables || !context_lens)) return PKV_ERR_INVALID_ARG;
    if (max_items > 0 && (!members || !item_blocks)) return PKV_ERR_INVALID_ARG;
    for (int64_t i = 0; i < int64_t(max_items) * item_width; ++i) members[i] = -1;
    for (int i = 0; i < max_items; ++i) item_blocks[i] = 0;
    if (min_members < 1) min_members = 1;
    if (min_shared_blocks < 1) min_shared_blocks = 1;

    const TableView t{block_tables, max_blocks_per_seq};
    std::vector<int> whole(size_t(std::max(num_seqs, 0)));
    std::vector<int> cand;
    for (int s = 0; s < num_seqs; ++s) {
        const int ctx = std::max(context_lens[s], 0);
        whole[s] = std::min(ctx / pkv::kBlockSize, max_blocks_per_seq);
        if (whole[s] >= min_shared_blocks) cand.push_back(s);
    }
    std::sort(cand.begin(), cand.end(), [&](int a, int b) {
        const int32_t* ra = t.row(a);
        const int32_t* rb = t.row(b);
        const int n = std::min(whole[a], whole[b]);
        for (int i = 0; i < n; ++i)
            if (ra[i] != rb[i]) return ra[i] < rb[i];
        if (whole[a] != whole[b]) return whole[a] < whole[b];
        return a < b;
    });
    // lcp[i]: whole pages shared by cand[i] and cand[i + 1]
    std::vector<int> lcp(cand.size() > 0 ? cand.size() - 1 : 0);
    for (size_t i = 0; i + 1 < cand.size(); ++i)
        lcp[i] = common_prefix(t, cand[i], whole[cand[i]], cand[i + 1], whole[cand[i + 1]]);

    int out = 0;
    size_t g0 = 0;
    while (g0 < cand.size() && out < max_items) {
        size_t g1 = g0 + 1;   // group [g0, g1)
        while (g1 < cand.size() && lcp[g1 - 1] >= min_shared_blocks) ++g1;
        const int n = int(g1 - g0);
        if (n >= min_members && n >= 2) {
            const int items = (n + item_width - 1) / item_width;
            const int base = n / items, extra = n % items;
            size_t k = g0;
            for (int it = 0; it < items && out < max_items; ++it) {
                const int sz = base + (it < extra ? 1 : 0);
                if (sz >= min_members && sz >= 2) {
                    int shared = whole[cand[k]];
                    for (int j = 0; j + 1 < sz; ++j) shared = std::min(shared, lcp[k + j]);
                    for (int j = 0; j < sz; ++j) members[size_t(out) * item_width + j] = cand[k + j];
                    item_blocks[out] = shared;
                    ++out;
                }
                k += size_t(sz);
            }
        }
        g0 = g1;
    }
    *num_items = out;
    return PKV_OK;
}
