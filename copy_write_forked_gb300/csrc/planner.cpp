// Sharing planner: which logical blocks a set of queried branches read from
// the same physical blocks.
//
// Dendrite article (ainews.cool, section 技术深度解析): a fork at position t
// leaves positions 0..t-1 shared with the parent and gives the child new leaf
// nodes for positions >= t; attention gathers K/V from the shared ancestor
// path and the branch's own leaf path.  With block tables this means: after a
// fork at t the child's table entries 0..floor(t/bs)-1 equal the parent's and
// stay equal for good (a full block is never written again), while the block
// holding position t (if partly filled) may later be copied on write and so
// counts as the child's own.
//
// For queried branch b and logical block i, the owner of (b, i) is found by
// walking up: while b has a parent and i < floor(fork_len(b)/bs), move to the
// parent.  Branches with the same owner for block i share the physical block.
// Walking from b upwards, node a owns blocks [start_a, cap) of b, where start_a
// = floor(fork_len(a)/bs) (0 for a root) and cap is the smallest fork cut met
// so far (ceil(len(b)/bs) at b itself).  Grouping those ranges by owner node
// and cutting at every distinct cap yields maximal block ranges read by a fixed
// set of queried branches: the segments.
#include <algorithm>
#include <cstring>
#include <unordered_map>

#include "dendrite_internal.h"

namespace dendrite {

void plan_segments(int32_t n_nodes, const int32_t* parent, const int32_t* fork_len,
                   const int32_t* len, int32_t bs, const int32_t* queried, int32_t n_queried,
                   std::vector<Segment>& segs, std::vector<int32_t>& members) {
    segs.clear();
    members.clear();
    struct Rec { int32_t grp, cap, member; };
    static thread_local std::vector<int32_t> slot, order, mem, count;
    static thread_local std::vector<Rec> recs, sorted;
    slot.assign(n_nodes, -1);
    order.clear();
    recs.clear();
    // walk every queried branch up to its root: owner node -> [start, cap)
    for (int32_t qi = 0; qi < n_queried; ++qi) {
        int32_t node = queried[qi];
        int32_t cap = (len[node] + bs - 1) / bs;
        while (cap > 0) {
            const int32_t start = parent[node] >= 0 ? fork_len[node] / bs : 0;
            if (start < cap) {
                if (slot[node] < 0) {
                    slot[node] = (int32_t)order.size();
                    order.push_back(node);
                }
                recs.push_back({slot[node], cap, qi});
            }
            if (parent[node] < 0) break;
            cap = std::min(cap, start);
            node = parent[node];
        }
    }
    // group by owner (first-visit order) with one counting pass; within a
    // group the records stay in increasing member order
    const int32_t n_grp = (int32_t)order.size();
    count.assign(n_grp + 1, 0);
    for (const Rec& r : recs) count[r.grp + 1]++;
    for (int32_t g = 0; g < n_grp; ++g) count[g + 1] += count[g];
    sorted.resize(recs.size());
    {
        static thread_local std::vector<int32_t> cursor;
        cursor.assign(count.begin(), count.end() - 1);
        for (const Rec& r : recs) sorted[cursor[r.grp]++] = r;
    }
    for (int32_t gi = 0; gi < n_grp; ++gi) {
        const size_t g0 = count[gi], g1 = count[gi + 1];
        const int32_t node = order[gi];
        const int32_t start = parent[node] >= 0 ? fork_len[node] / bs : 0;
        bool uniform = true;
        for (size_t k = g0 + 1; k < g1 && uniform; ++k) uniform = sorted[k].cap == sorted[g0].cap;
        if (uniform) {   // every member reads [start, cap): one segment, members already in order
            Segment sg;
            sg.block_start = start;
            sg.block_count = sorted[g0].cap - start;
            sg.member_offset = (int32_t)members.size();
            for (size_t k = g0; k < g1; ++k) members.push_back(sorted[k].member);
            sg.n_members = (int32_t)(g1 - g0);
            sg.rep_node = queried[sorted[g0].member];
            segs.push_back(sg);
            continue;
        }
        // caps descending (members ascending within a cap); the ascending
        // cuts then take the smallest cap first, and the members of
        // [lo, cut) are the records with cap >= cut, a prefix of the group
        std::stable_sort(sorted.begin() + g0, sorted.begin() + g1,
                         [](const Rec& a, const Rec& b) { return a.cap > b.cap; });
        int32_t lo = start;
        size_t end = g1;
        while (end > g0) {
            const int32_t cut = sorted[end - 1].cap;
            if (cut > lo) {
                Segment sg;
                sg.block_start = lo;
                sg.block_count = cut - lo;
                sg.member_offset = (int32_t)members.size();
                mem.clear();
                for (size_t k = g0; k < end; ++k) mem.push_back(sorted[k].member);
                std::sort(mem.begin(), mem.end());
                members.insert(members.end(), mem.begin(), mem.end());
                sg.n_members = (int32_t)mem.size();
                sg.rep_node = queried[mem.front()];
                segs.push_back(sg);
                lo = cut;
            }
            while (end > g0 && sorted[end - 1].cap == cut) --end;
        }
    }
}

}  // namespace dendrite

extern "C" int dendrite_plan_segments(int32_t n_nodes, const int32_t* parent, const int32_t* fork_len,
                                      const int32_t* len, int32_t block_size,
                                      const int32_t* queried, int32_t n_queried,
                                      dendrite_segment* segs, int32_t seg_cap, int32_t* n_segs,
                                      int32_t* members, int32_t member_cap, int32_t* n_members) {
    if (n_nodes < 0 || n_queried < 0 || block_size <= 0 || !n_segs || !n_members) return DENDRITE_EINVAL;
    if (n_nodes > 0 && (!parent || !fork_len || !len)) return DENDRITE_EINVAL;
    if (n_queried > 0 && !queried) return DENDRITE_EINVAL;
    for (int32_t i = 0; i < n_nodes; ++i) {
        if (parent[i] < -1 || parent[i] >= n_nodes || len[i] < 0 || fork_len[i] < 0) return DENDRITE_EINVAL;
        if (parent[i] >= 0 && fork_len[i] > len[i]) return DENDRITE_EINVAL;
    }
    // reject cycles: every parent chain must end at a root within n_nodes steps
    for (int32_t i = 0; i < n_nodes; ++i) {
        int32_t x = i, steps = 0;
        while (x >= 0 && steps <= n_nodes) { x = parent[x]; ++steps; }
        if (x >= 0) return DENDRITE_EINVAL;
    }
    std::vector<char> seen(n_nodes, 0);
    for (int32_t q = 0; q < n_queried; ++q) {
        if (queried[q] < 0 || queried[q] >= n_nodes || seen[queried[q]]) return DENDRITE_EINVAL;
        seen[queried[q]] = 1;
    }
    std::vector<dendrite::Segment> s;
    std::vector<int32_t> m;
    dendrite::plan_segments(n_nodes, parent, fork_len, len, block_size, queried, n_queried, s, m);
    *n_segs = (int32_t)s.size();
    *n_members = (int32_t)m.size();
    if ((int32_t)s.size() > seg_cap || (int32_t)m.size() > member_cap) return DENDRITE_ELIMIT;
    for (size_t i = 0; i < s.size(); ++i) {
        segs[i].rep = s[i].rep_node;
        segs[i].block_start = s[i].block_start;
        segs[i].block_count = s[i].block_count;
        segs[i].member_offset = s[i].member_offset;
        segs[i].n_members = s[i].n_members;
    }
    if (!m.empty()) std::memcpy(members, m.data(), m.size() * sizeof(int32_t));
    return DENDRITE_OK;
}
