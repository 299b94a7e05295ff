// Host-side work planner of the tensor-core split decode (plain C++, no CUDA):
// splits each batch element's segments of tiles into contiguous runs, one per CTA,
// with one partial slot per (CTA, segment piece). Kept in a header of its own so
// that the CPU tests compile it and check its invariants.
#pragma once

#include <stdint.h>

#include <algorithm>
#include <utility>
#include <vector>

namespace slimkv {
namespace plan {

// Work plan: contiguous unit ranges per CTA with balanced cost, one partial slot
// per (CTA, segment piece), and the slot range of every batch element.
struct WorkPlan {
    int n_ctas = 0;
    std::vector<int> u_begin, slot_base, batch_slot, slot_seg;
    int slots = 0;
};

// Segments of one batch element in unit order: (tiles, cost per tile).
struct SegList {
    std::vector<std::pair<int, int>> segs;
};

// Fixed cost of a piece in tile-cost units (about 1.6 tiles): its first tile waits for
// a query image and takes the rescale path, and its end waits for the last value MMAs
// and writes a partial. The planner avoids splitting a segment across CTAs unless
// that pays for itself.
constexpr int kPieceCost = 8;

inline WorkPlan make_plan(int B, const SegList& sl, int max_ctas) {
    // runs of equal-cost units in unit order (batch-major, then segment)
    int64_t total = 0, units = 0;
    int cmax = 1;
    for (int b = 0; b < B; ++b)
        for (auto& r : sl.segs) {
            total += (int64_t)r.first * r.second;
            units += r.first;
            cmax = std::max(cmax, r.second);
        }
    const int G = (int)std::max<int64_t>(1, std::min<int64_t>(max_ctas, units));
    // Greedy packing with per-CTA budget T: a CTA takes units in order until the next
    // one would exceed T; every piece (a CTA's run inside one segment) costs
    // kPieceCost on top of its units. `visit(u, new_cta, b, seg)` sees every unit
    // boundary where a CTA or a piece starts; returns the number of CTAs.
    auto pack = [&](int64_t T, auto&& visit) {
        int ctas = 1;
        int64_t cur = 0, u = 0;
        for (int b = 0; b < B; ++b)
            for (int si = 0; si < (int)sl.segs.size(); ++si) {
                const auto& r = sl.segs[si];
                int n = r.first;
                bool open = false;   // a piece of this segment is open in the current CTA
                while (n > 0) {
                    if (!open) {
                        if (cur > 0 && cur + kPieceCost + r.second > T) {
                            ++ctas;
                            cur = 0;
                            visit(u, true, b, si);
                        } else {
                            visit(u, false, b, si);
                        }
                        cur += kPieceCost;
                        open = true;
                    }
                    int64_t room = (T - cur) / r.second;
                    if (room == 0) {
                        ++ctas;
                        cur = kPieceCost;
                        visit(u, true, b, si);
                        room = (T - cur) / r.second;
                    }
                    const int take = (int)std::min<int64_t>(n, room);
                    cur += (int64_t)take * r.second;
                    u += take;
                    n -= take;
                }
            }
        return ctas;
    };
    auto no_visit = [](int64_t, bool, int, int) {};
    int64_t lo = std::max<int64_t>(cmax + kPieceCost, (total + G - 1) / G),
            hi = std::max<int64_t>(lo, total + (int64_t)kPieceCost * B * (int64_t)sl.segs.size());
    while (lo < hi) {
        const int64_t mid = (lo + hi) / 2;
        if (pack(mid, no_visit) <= G) hi = mid;
        else lo = mid + 1;
    }
    const int64_t T = lo;
    WorkPlan w;
    std::vector<int> piece_cta;   // CTA of each piece, in unit order
    std::vector<int> piece_b;
    w.u_begin.push_back(0);
    bool first = true;
    pack(T, [&](int64_t u, bool new_cta, int b, int si) {
        if (new_cta && !first) w.u_begin.push_back((int)u);
        first = false;
        piece_cta.push_back((int)w.u_begin.size() - 1);
        piece_b.push_back(b);
        w.slot_seg.push_back(si);
    });
    w.u_begin.push_back((int)units);
    w.n_ctas = (int)w.u_begin.size() - 1;
    // slots in piece order: CTA i's pieces are consecutive, and batch b owns a
    // contiguous slot range because units are batch-major
    w.slot_base.assign(w.n_ctas, -1);
    w.batch_slot.assign(B + 1, -1);
    for (int s = 0; s < (int)piece_cta.size(); ++s) {
        if (w.slot_base[piece_cta[s]] < 0) w.slot_base[piece_cta[s]] = s;
        if (w.batch_slot[piece_b[s]] < 0) w.batch_slot[piece_b[s]] = s;
    }
    w.batch_slot[B] = (int)piece_cta.size();
    w.slots = (int)piece_cta.size();
    return w;
}

// First slot of batch element b whose piece lies in a segment with index >= seg
// (batch_slot[b + 1] if none): with the segments of a batch element in kind order,
// the slots of b below it hold the partials of the segments before `seg`.
inline int first_slot_from_seg(const WorkPlan& w, int b, int seg) {
    int s = w.batch_slot[b];
    while (s < w.batch_slot[b + 1] && w.slot_seg[s] < seg) ++s;
    return s;
}

}  // namespace plan
}  // namespace slimkv
