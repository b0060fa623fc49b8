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
    struct Rec { int32_t cap, member; };
    static thread_local std::vector<int32_t> slot, order, cnt, cap0, cur, mem, first_block, flat;
    static thread_local std::vector<char> mixed;
    static thread_local std::vector<Rec> recs;
    slot.assign(n_nodes, -1);
    first_block.resize(n_nodes);   // a node's first own block (0 for a root)
    for (int32_t i = 0; i < n_nodes; ++i) first_block[i] = parent[i] >= 0 ? fork_len[i] / bs : 0;
    order.clear();
    cnt.clear();
    cap0.clear();
    mixed.clear();
    // Walk every queried branch up to its root (owner node -> [start, cap)),
    // twice.  The first walk numbers the owners in first-visit order, counts
    // each one's records and notes whether all its records share one cap;
    // the second writes each owner's members (in increasing member order)
    // into its own range, and their caps for owners with several.
    int32_t n_rec = 0;
    for (int32_t qi = 0; qi < n_queried; ++qi) {
        int32_t node = queried[qi];
        int32_t cap = (len[node] + bs - 1) / bs;
        while (cap > 0) {
            const int32_t start = first_block[node];
            if (start < cap) {
                int32_t g = slot[node];
                if (g < 0) {
                    g = slot[node] = (int32_t)order.size();
                    order.push_back(node);
                    cnt.push_back(0);
                    cap0.push_back(cap);
                    mixed.push_back(0);
                }
                cnt[g]++;
                mixed[g] |= cap != cap0[g];
                ++n_rec;
            }
            if (parent[node] < 0) break;
            cap = std::min(cap, start);
            node = parent[node];
        }
    }
    const int32_t n_grp = (int32_t)order.size();
    cur.resize(n_grp + 1);
    cur[0] = 0;
    for (int32_t g = 0; g < n_grp; ++g) cur[g + 1] = cur[g] + cnt[g];
    flat.resize(n_rec);
    recs.resize(n_rec);
    {
        static thread_local std::vector<int32_t> pos;
        pos.assign(cur.begin(), cur.end() - 1);
        for (int32_t qi = 0; qi < n_queried; ++qi) {
            int32_t node = queried[qi];
            int32_t cap = (len[node] + bs - 1) / bs;
            while (cap > 0) {
                const int32_t start = first_block[node];
                if (start < cap) {
                    const int32_t g = slot[node];
                    const int32_t at = pos[g]++;
                    flat[at] = qi;
                    if (mixed[g]) recs[at] = Rec{cap, qi};
                }
                if (parent[node] < 0) break;
                cap = std::min(cap, start);
                node = parent[node];
            }
        }
    }
    members.reserve(n_rec);
    for (int32_t gi = 0; gi < n_grp; ++gi) {
        const int32_t g0 = cur[gi], g1 = cur[gi + 1];
        const int32_t node = order[gi];
        const int32_t start = first_block[node];
        if (!mixed[gi]) {   // every member reads [start, cap): one segment, members already in order
            Segment sg;
            sg.block_start = start;
            sg.block_count = cap0[gi] - start;
            sg.member_offset = (int32_t)members.size();
            members.insert(members.end(), flat.begin() + g0, flat.begin() + g1);
            sg.n_members = g1 - g0;
            sg.rep_node = queried[flat[g0]];
            sg.owner = node;
            segs.push_back(sg);
            continue;
        }
        // caps descending (members ascending within a cap); the ascending
        // cuts then take the smallest cap first, and the members of
        // [lo, cut) are the records with cap >= cut, a prefix of the group
        std::stable_sort(recs.begin() + g0, recs.begin() + g1,
                         [](const Rec& a, const Rec& b) { return a.cap > b.cap; });
        int32_t lo = start;
        int32_t end = g1;
        while (end > g0) {
            const int32_t cut = recs[end - 1].cap;
            if (cut > lo) {
                Segment sg;
                sg.block_start = lo;
                sg.block_count = cut - lo;
                sg.member_offset = (int32_t)members.size();
                mem.clear();
                for (int32_t k = g0; k < end; ++k) mem.push_back(recs[k].member);
                std::sort(mem.begin(), mem.end());
                members.insert(members.end(), mem.begin(), mem.end());
                sg.n_members = (int32_t)mem.size();
                sg.rep_node = queried[mem.front()];
                sg.owner = node;
                segs.push_back(sg);
                lo = cut;
            }
            while (end > g0 && recs[end - 1].cap == cut) --end;
        }
    }
}


// Folding.  Every segment costs each of its rows a partial (max, sum, acc) row,
// written by a partial kernel and read again by the merge, plus a fresh load of
// the row's query, and each of its row groups a unit start.  In a deep tree of
// short nodes (MCTS: 32 tokens a node) most segments are two blocks long and
// these per-row and per-unit costs outweigh the reading of the blocks.  Folding
// a segment s lets every segment that follows s in some member's path read s's
// range again with its own rows: each following segment is extended down to
// s's first block, s's own units and partial rows disappear, and its blocks are
// read once per following segment (mostly from L2, as the units of those
// segments run next to one another).  Members whose path ends in s keep a
// segment of their own over s's range.  The segments still read every
// (member, block) pair exactly once, and each is still read through one
// physical block per position for all its members, because every member of a
// following segment is a member of s.  Decisions run in increasing block
// order, so a segment's range already includes what was folded into it when
// its own turn comes.
namespace {

// Estimated SM time, in ns, of one kv head's row group of `rows` rows: per
// 16-token block, and per unit (start, query load, partial rows written and
// merged).  Fitted to per-CTA timelines of the partial kernels on GB300.
int64_t group_block_ns(bool tc, int32_t rows) {
    if (tc) return rows <= 128 ? 275 : 325;
    const int32_t rt = rows <= 16 ? 1 : rows <= 32 ? 2 : 4;
    return 60 * (1 + rt);
}
int64_t group_unit_ns(bool tc, int32_t rows) { return (tc ? 3000 : 1000) + 29 * (int64_t)rows; }

// Estimated time of one block for a row group of R rows (one unit).
int64_t tile_ns(const FoldParams& fp, int64_t R) {
    const bool tc = fp.tc_rows >= 0 && R > fp.tc_rows;
    return group_block_ns(tc, (int32_t)std::min<int64_t>(R, tc ? kMaxUnitRowsTc : fp.small_rows));
}

// Estimate for R rows over T blocks, split into row groups as the plan splits
// them; with_units adds the per-unit part.
int64_t estimate_ns(const FoldParams& fp, int64_t T, int64_t R, bool with_units) {
    const bool tc = fp.tc_rows >= 0 && R > fp.tc_rows;
    const int32_t g = tc ? kMaxUnitRowsTc : fp.small_rows;
    const int64_t full = R / g, rem = R - full * g;
    int64_t ns = full * (T * group_block_ns(tc, g) + (with_units ? group_unit_ns(tc, g) : 0));
    if (rem) ns += T * group_block_ns(tc, (int32_t)rem) + (with_units ? group_unit_ns(tc, (int32_t)rem) : 0);
    return ns;
}

// The segment before each segment in its members' block order (the same for
// all of them): the previous segment of the same owner, or for an owner's
// first segment, the segment ending at its first block in the group of the
// nearest ancestor that owns the block before it (-1: none).  Needs each
// owner node's segments consecutive in segs, in ascending blocks.
void segment_prev(const std::vector<Segment>& segs, int32_t n_nodes, const int32_t* parent,
                  const int32_t* fork_len, int32_t bs, std::vector<int32_t>& prev) {
    static thread_local std::vector<int32_t> node_first, node_count;
    const int32_t S = (int32_t)segs.size();
    node_first.assign(n_nodes, -1);
    node_count.assign(n_nodes, 0);
    for (int32_t si = 0; si < S; ++si) {
        const int32_t o = segs[si].owner;
        if (node_first[o] < 0) node_first[o] = si;
        node_count[o]++;
    }
    prev.assign(S, -1);
    for (int32_t si = 0; si < S; ++si) {
        const Segment& sg = segs[si];
        if (si > node_first[sg.owner]) {
            prev[si] = si - 1;
            continue;
        }
        const int32_t b = sg.block_start;
        if (b == 0) continue;
        int32_t a = parent[sg.owner];
        while (a >= 0 && parent[a] >= 0 && fork_len[a] / bs > b - 1) a = parent[a];
        if (a < 0 || node_first[a] < 0) continue;
        // the owner's segment that ends at b
        int32_t lo = node_first[a], hi = node_first[a] + node_count[a] - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (segs[mid].block_start <= b - 1) lo = mid; else hi = mid - 1;
        }
        if (segs[lo].block_start + segs[lo].block_count == b) prev[si] = lo;
    }
}

}  // namespace

void fold_segments(const FoldParams& fp, int32_t n_nodes, const int32_t* parent, const int32_t* fork_len,
                   const int32_t* len, int32_t block_size, const int32_t* queried, int32_t n_queried,
                   std::vector<Segment>& segs, std::vector<int32_t>& members, const std::vector<int32_t>* prev_in) {
    const int32_t S = (int32_t)segs.size();
    if (fp.fold_pct < 0 || S < 2 || fp.rows_per_member <= 0) return;
    static thread_local std::vector<int32_t> prev, koff, kseg, eoff, emem, order, ext, qblocks;
    static thread_local std::vector<char> folded;
    const int32_t bs = block_size;
    // each queried branch's block count
    qblocks.resize(n_queried);
    for (int32_t q = 0; q < n_queried; ++q) qblocks[q] = (len[queried[q]] + bs - 1) / bs;
    if (prev_in && (int32_t)prev_in->size() == S) prev = *prev_in;
    else segment_prev(segs, n_nodes, parent, fork_len, bs, prev);
    // the segments after each segment, and the members whose blocks end there
    koff.assign(S + 1, 0);
    eoff.resize(S + 1);
    emem.resize(members.size());
    {
        int32_t e = 0;
        for (int32_t si = 0; si < S; ++si) {   // members stay in ascending order within a segment
            if (prev[si] >= 0) koff[prev[si] + 1]++;
            const Segment& sg = segs[si];
            const int32_t end = sg.block_start + sg.block_count;
            eoff[si] = e;
            const int32_t* mp = members.data() + sg.member_offset;
            for (int32_t k = 0; k < sg.n_members; ++k) {
                const int32_t m = mp[k];
                emem[e] = m;
                e += qblocks[m] == end;
            }
        }
        eoff[S] = e;
    }
    for (int32_t si = 0; si < S; ++si) koff[si + 1] += koff[si];
    kseg.resize(koff[S]);
    {
        static thread_local std::vector<int32_t> kc;
        kc.assign(koff.begin(), koff.end() - 1);
        for (int32_t si = 0; si < S; ++si)
            if (prev[si] >= 0) kseg[kc[prev[si]]++] = si;
    }
    // decide in increasing block order
    {
        // counting sort by first block (stable)
        int32_t max_start = 0;
        for (const Segment& sg : segs) max_start = std::max(max_start, sg.block_start);
        static thread_local std::vector<int32_t> cnt;
        cnt.assign((size_t)max_start + 2, 0);
        for (const Segment& sg : segs) cnt[sg.block_start + 1]++;
        for (int32_t b = 0; b <= max_start; ++b) cnt[b + 1] += cnt[b];
        order.resize(S);
        for (int32_t si = 0; si < S; ++si) order[cnt[segs[si].block_start]++] = si;
    }
    ext.resize(S);
    for (int32_t si = 0; si < S; ++si) ext[si] = segs[si].block_start;
    folded.assign(S, 0);
    const int64_t rpm = fp.rows_per_member;
    bool any = false;
    for (const int32_t si : order) {
        if (koff[si + 1] == koff[si]) continue;   // nothing follows it
        const Segment& sg = segs[si];
        const int64_t T = (int64_t)sg.block_start + sg.block_count - ext[si];
        const int64_t keep = estimate_ns(fp, T, sg.n_members * rpm, true);
        int64_t fold = 0;
        for (int32_t k = koff[si]; k < koff[si + 1]; ++k)
            fold += estimate_ns(fp, T, segs[kseg[k]].n_members * rpm, false);
        if (eoff[si + 1] > eoff[si]) fold += estimate_ns(fp, T, (eoff[si + 1] - eoff[si]) * rpm, true);
        if (fold * 100 < keep * fp.fold_pct) {
            folded[si] = 1;
            any = true;
            for (int32_t k = koff[si]; k < koff[si + 1]; ++k) ext[kseg[k]] = ext[si];
        }
    }
    if (!any) return;
    // rebuild in the original order; a folded segment's place goes to the
    // segment of the members that end in it, if any
    static thread_local std::vector<Segment> out;
    static thread_local std::vector<int32_t> out_members;
    out.clear();
    out_members.clear();
    for (int32_t si = 0; si < S; ++si) {
        const Segment& sg = segs[si];
        const int32_t end = sg.block_start + sg.block_count;
        Segment o;
        o.block_start = ext[si];
        o.block_count = end - ext[si];
        o.member_offset = (int32_t)out_members.size();
        if (!folded[si]) {
            o.owner = sg.owner;
            o.rep_node = sg.rep_node;
            o.n_members = sg.n_members;
            o.x_off = sg.x_off;
            o.n_x = sg.n_x;
            out_members.insert(out_members.end(), members.begin() + sg.member_offset,
                               members.begin() + sg.member_offset + sg.n_members);
        } else {
            if (eoff[si + 1] == eoff[si]) continue;
            o.owner = sg.owner;
            o.rep_node = queried[emem[eoff[si]]];
            o.n_members = eoff[si + 1] - eoff[si];
            out_members.insert(out_members.end(), emem.begin() + eoff[si], emem.begin() + eoff[si + 1]);
        }
        out.push_back(o);
    }
    segs.swap(out);
    members.swap(out_members);
}

// Packing.  A segment s whose members continue into following segments that
// have no followers of their own (leaves of the segment tree: the private
// tails of speculative draft paths, of beam leaves, of MCTS leaves) costs
// every follower a unit start, a query load and a partial row per member row,
// for a few blocks each.  Packing gives s the followers' tiles as extra
// tiles, each masked to the members of the follower it came from, so one unit
// per kv head reads s's blocks with all its rows and then each follower's
// blocks with that follower's rows; a row's partial then covers all of its
// blocks, and the followers' units, partial rows and merge reads disappear.
// The price is that every extra tile is multiplied with all of s's rows (the
// row tiles of s's unit), so long private tails (the stress leaves) stay on
// their own.  Decisions run in decreasing block order, so a follower has
// absorbed its own followers before its turn comes and a packed follower's
// extra tiles move up with its own.
void pack_segments(const FoldParams& fp, int32_t pack_pct, int32_t n_nodes, const int32_t* parent,
                   const int32_t* fork_len, int32_t block_size, std::vector<Segment>& segs,
                   std::vector<int32_t>& members, std::vector<ExtraTile>& xt, std::vector<int32_t>* prev_out) {
    xt.clear();
    if (prev_out) prev_out->clear();
    const int32_t S = (int32_t)segs.size();
    if (pack_pct < 0 || S < 2 || fp.rows_per_member <= 0) return;
    static thread_local std::vector<int32_t> prev, koff, kseg, order, open_followers, cnt;
    // absorbed followers of each segment (a list in absorption order) and its extra tiles so far
    static thread_local std::vector<int32_t> nx, first_abs, next_abs, last_abs;
    static thread_local std::vector<char> gone;
    segment_prev(segs, n_nodes, parent, fork_len, block_size, prev);
    koff.assign(S + 1, 0);
    for (int32_t si = 0; si < S; ++si)
        if (prev[si] >= 0) koff[prev[si] + 1]++;
    for (int32_t si = 0; si < S; ++si) koff[si + 1] += koff[si];
    kseg.resize(koff[S]);
    {
        static thread_local std::vector<int32_t> kc;
        kc.assign(koff.begin(), koff.end() - 1);
        for (int32_t si = 0; si < S; ++si)
            if (prev[si] >= 0) kseg[kc[prev[si]]++] = si;
    }
    open_followers.resize(S);
    for (int32_t si = 0; si < S; ++si) open_followers[si] = koff[si + 1] - koff[si];
    // decreasing first block (a counting sort): followers come before the segment they follow
    {
        int32_t max_start = 0;
        for (const Segment& sg : segs) max_start = std::max(max_start, sg.block_start);
        cnt.assign((size_t)max_start + 2, 0);
        for (const Segment& sg : segs) cnt[max_start - sg.block_start + 1]++;
        for (int32_t k = 0; k <= max_start; ++k) cnt[k + 1] += cnt[k];
        order.resize(S);
        for (int32_t si = 0; si < S; ++si) order[cnt[max_start - segs[si].block_start]++] = si;
    }
    nx.assign(S, 0);
    first_abs.assign(S, -1);
    next_abs.assign(S, -1);
    last_abs.assign(S, -1);
    gone.assign(S, 0);
    const int64_t rpm = fp.rows_per_member;
    bool any = false;
    for (const int32_t si : order) {
        const int32_t k0 = koff[si], k1 = koff[si + 1];
        if (k0 == k1) continue;
        const Segment& sg = segs[si];
        const int64_t R = (int64_t)sg.n_members * rpm;
        const bool tc = fp.tc_rows >= 0 && R > fp.tc_rows;
        if (sg.n_members > kMaxPackMembers || R > (tc ? kMaxUnitRowsTc : fp.small_rows)) continue;
        // every follower closed, and none read by all of sg's members (a
        // chain, which folding joins without masks)
        bool closed = true;
        for (int32_t k = k0; k < k1 && closed; ++k)
            closed = open_followers[kseg[k]] == 0 && segs[kseg[k]].n_members < sg.n_members;
        if (!closed) continue;
        int64_t T = sg.block_count + (int64_t)nx[si];
        int64_t apart = estimate_ns(fp, T, R, true);
        for (int32_t k = k0; k < k1; ++k) {
            const Segment& f = segs[kseg[k]];
            const int64_t Tf = f.block_count + (int64_t)nx[kseg[k]];
            apart += estimate_ns(fp, Tf, (int64_t)f.n_members * rpm, true);
            T += Tf;
        }
        // the tcgen05 kernel stages a unit's extra tiles in shared memory
        const int64_t X = T - sg.block_count;
        if (tc && X > kMaxTcExtraTiles) continue;
        // on the mma.sync kernel an extra tile also costs the producer its
        // entry's load: about twice a tile's time, measured on beam leaves
        const int64_t packed_ns = estimate_ns(fp, T, R, true) + (tc ? 0 : X * tile_ns(fp, R));
        if (packed_ns * 100 >= apart * pack_pct) continue;
        for (int32_t k = k0; k < k1; ++k) {
            const int32_t fi = kseg[k];
            if (first_abs[si] < 0) first_abs[si] = fi; else next_abs[last_abs[si]] = fi;
            last_abs[si] = fi;
            gone[fi] = 1;
        }
        nx[si] = (int32_t)X;
        open_followers[si] = 0;
        any = true;
    }
    if (!any) {
        if (prev_out) *prev_out = prev;
        return;
    }
    // Rebuild in the original order without the absorbed segments.  A kept
    // segment's extra tiles are its absorbed followers' blocks in absorption
    // order, each follower's own blocks before those of the followers it had
    // absorbed, masked to that follower's members (their bit positions in the
    // kept segment's member list; both lists ascending).
    // (The member list is left as it is: the kept segments keep their
    // ranges in it, and the absorbed segments' ranges are no longer read.)
    static thread_local std::vector<Segment> out;
    out.clear();
    for (int32_t si = 0; si < S; ++si) {
        if (gone[si]) continue;
        const Segment& sg = segs[si];
        Segment o = sg;
        o.x_off = (int32_t)xt.size();
        const int32_t* sm = members.data() + sg.member_offset;
        auto emit = [&](auto&& self, int32_t fi) -> void {
            const Segment& f = segs[fi];
            const int32_t* fm = members.data() + f.member_offset;
            uint32_t fmask = 0;
            for (int32_t a = 0, b = 0; a < f.n_members; ++a) {
                while (sm[b] != fm[a]) ++b;
                fmask |= 1u << b;
            }
            for (int32_t i = 0; i < f.block_count; ++i) xt.push_back(ExtraTile{f.rep_node, f.block_start + i, fmask});
            for (int32_t g = first_abs[fi]; g >= 0; g = next_abs[g]) self(self, g);
        };
        for (int32_t g = first_abs[si]; g >= 0; g = next_abs[g]) emit(emit, g);
        o.n_x = (int32_t)xt.size() - o.x_off;
        out.push_back(o);
    }
    // the kept segments' predecessors (an absorbed segment had no followers,
    // so it is nobody's predecessor): their new indices
    if (prev_out) {
        static thread_local std::vector<int32_t> idx;
        idx.assign(S, -1);
        int32_t k = 0;
        for (int32_t si = 0; si < S; ++si)
            if (!gone[si]) idx[si] = k++;
        prev_out->resize(k);
        for (int32_t si = 0; si < S; ++si)
            if (!gone[si]) (*prev_out)[idx[si]] = prev[si] >= 0 ? idx[prev[si]] : -1;
    }
    segs.swap(out);
}

}  // namespace dendrite

namespace {

int check_forest(int32_t n_nodes, const int32_t* parent, const int32_t* fork_len, const int32_t* len,
                 int32_t block_size, const int32_t* queried, int32_t n_queried) {
    if (n_nodes < 0 || n_queried < 0 || block_size <= 0) return DENDRITE_EINVAL;
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
    return DENDRITE_OK;
}

int export_segments(const std::vector<dendrite::Segment>& s, const std::vector<int32_t>& m, dendrite_segment* segs,
                    int32_t seg_cap, int32_t* n_segs, int32_t* members, int32_t member_cap, int32_t* n_members) {
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

}  // namespace

extern "C" int dendrite_plan_segments(int32_t n_nodes, const int32_t* parent, const int32_t* fork_len,
                                      const int32_t* len, int32_t block_size,
                                      const int32_t* queried, int32_t n_queried,
                                      dendrite_segment* segs, int32_t seg_cap, int32_t* n_segs,
                                      int32_t* members, int32_t member_cap, int32_t* n_members) {
    if (!n_segs || !n_members) return DENDRITE_EINVAL;
    DENDRITE_TRY(check_forest(n_nodes, parent, fork_len, len, block_size, queried, n_queried));
    std::vector<dendrite::Segment> s;
    std::vector<int32_t> m;
    dendrite::plan_segments(n_nodes, parent, fork_len, len, block_size, queried, n_queried, s, m);
    return export_segments(s, m, segs, seg_cap, n_segs, members, member_cap, n_members);
}

extern "C" int dendrite_plan_segments_folded(int32_t n_nodes, const int32_t* parent, const int32_t* fork_len,
                                             const int32_t* len, int32_t block_size,
                                             const int32_t* queried, int32_t n_queried,
                                             int32_t rows_per_member, int32_t tc_min_rows, int32_t fold_pct,
                                             dendrite_segment* segs, int32_t seg_cap, int32_t* n_segs,
                                             int32_t* members, int32_t member_cap, int32_t* n_members) {
    if (!n_segs || !n_members || rows_per_member <= 0 || tc_min_rows < -1 || fold_pct < -1) return DENDRITE_EINVAL;
    DENDRITE_TRY(check_forest(n_nodes, parent, fork_len, len, block_size, queried, n_queried));
    std::vector<dendrite::Segment> s;
    std::vector<int32_t> m;
    dendrite::plan_segments(n_nodes, parent, fork_len, len, block_size, queried, n_queried, s, m);
    const dendrite::FoldParams fp{rows_per_member, tc_min_rows == 0 ? dendrite::kTcMinRowsDefault : tc_min_rows,
                                  dendrite::kMaxUnitRowsBf16,
                                  fold_pct == 0 ? dendrite::kFoldPctDefault : fold_pct};
    dendrite::fold_segments(fp, n_nodes, parent, fork_len, len, block_size, queried, n_queried, s, m);
    return export_segments(s, m, segs, seg_cap, n_segs, members, member_cap, n_members);
}

extern "C" int dendrite_plan_segments_packed(int32_t n_nodes, const int32_t* parent, const int32_t* fork_len,
                                             const int32_t* len, int32_t block_size,
                                             const int32_t* queried, int32_t n_queried,
                                             int32_t rows_per_member, int32_t tc_min_rows, int32_t fold_pct,
                                             int32_t pack_pct, dendrite_segment* segs, int32_t seg_cap,
                                             int32_t* n_segs, int32_t* members, int32_t member_cap,
                                             int32_t* n_members, int32_t* extra_off, dendrite_extra_tile* extras,
                                             int32_t extra_cap, int32_t* n_extras) {
    if (!n_segs || !n_members || !n_extras || rows_per_member <= 0 || tc_min_rows < -1 || fold_pct < -1 ||
        pack_pct < -1)
        return DENDRITE_EINVAL;
    DENDRITE_TRY(check_forest(n_nodes, parent, fork_len, len, block_size, queried, n_queried));
    std::vector<dendrite::Segment> s;
    std::vector<int32_t> m;
    std::vector<dendrite::ExtraTile> xt;
    dendrite::plan_segments(n_nodes, parent, fork_len, len, block_size, queried, n_queried, s, m);
    const dendrite::FoldParams fp{rows_per_member, tc_min_rows == 0 ? dendrite::kTcMinRowsDefault : tc_min_rows,
                                  dendrite::kMaxUnitRowsBf16,
                                  fold_pct == 0 ? dendrite::kFoldPctDefault : fold_pct};
    std::vector<int32_t> prev;
    dendrite::pack_segments(fp, pack_pct == 0 ? dendrite::kPackPctDefault : pack_pct, n_nodes, parent, fork_len,
                            block_size, s, m, xt, &prev);
    dendrite::fold_segments(fp, n_nodes, parent, fork_len, len, block_size, queried, n_queried, s, m, &prev);
    *n_extras = (int32_t)xt.size();
    const int rc = export_segments(s, m, segs, seg_cap, n_segs, members, member_cap, n_members);
    if (rc != DENDRITE_OK || (int32_t)xt.size() > extra_cap) return rc != DENDRITE_OK ? rc : DENDRITE_ELIMIT;
    if (extra_off) {
        for (size_t i = 0; i < s.size(); ++i) extra_off[i] = s[i].x_off;
        extra_off[s.size()] = (int32_t)xt.size();
    }
    for (size_t i = 0; i < xt.size(); ++i)
        extras[i] = dendrite_extra_tile{xt[i].rep_node, xt[i].blk, xt[i].mask, 0};
    return DENDRITE_OK;
}
