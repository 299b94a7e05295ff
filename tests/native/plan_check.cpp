// Invariants of the split-decode work planner (latent_kv_cache_decode_b300/csrc/work_plan.h),
// checked against the decode kernel's own derivation of pieces: a CTA's run starts a new
// piece at its first unit and at every segment start inside it.
#include <cstdio>
#include <cstdlib>

#include "work_plan.h"

using namespace slimkv::plan;

static int check(int B, const SegList& sl, int G, int* n_ctas, int* max_pieces, int* min_units, int* max_units) {
    const WorkPlan w = make_plan(B, sl, G);
    std::vector<int> seg_start;
    int u = 0;
    for (int b = 0; b < B; ++b)
        for (auto& r : sl.segs) {
            if (r.first > 0) seg_start.push_back(u);
            u += r.first;
        }
    const int units = u;
    if (w.u_begin.empty() || w.u_begin.front() != 0 || w.u_begin.back() != units) return 1;
    if ((int)w.u_begin.size() != w.n_ctas + 1 || w.n_ctas < 1 || w.n_ctas > G) return 2;
    int pieces = 0, maxp = 0, minu = 1 << 30, maxu = 0;
    for (int c = 0; c < w.n_ctas; ++c) {
        if (w.u_begin[c + 1] <= w.u_begin[c]) return 3;   // no empty CTA
        int p = 0;
        for (int x = w.u_begin[c]; x < w.u_begin[c + 1]; ++x)
            if (x == w.u_begin[c] || std::binary_search(seg_start.begin(), seg_start.end(), x)) ++p;
        if (w.slot_base[c] != pieces) return 4;
        pieces += p;
        maxp = std::max(maxp, p);
        minu = std::min(minu, w.u_begin[c + 1] - w.u_begin[c]);
        maxu = std::max(maxu, w.u_begin[c + 1] - w.u_begin[c]);
    }
    if (pieces != w.slots || (int)w.batch_slot.size() != B + 1 || w.batch_slot[B] != pieces) return 5;
    // every piece starts at a CTA start or a segment start: the workspace reserves one
    // partial slot per segment plus a fixed margin above the largest grid
    if (w.slots > w.n_ctas + (int)seg_start.size()) return 7;
    // batch element b's slots are contiguous and hold exactly its pieces
    for (int b = 0; b < B; ++b)
        if (w.batch_slot[b + 1] < w.batch_slot[b]) return 6;
    // every slot records its piece's segment; inside a batch element the segments rise, so
    // first_slot_from_seg splits b's slots into those before and from a given segment
    if ((int)w.slot_seg.size() != w.slots) return 8;
    for (int b = 0; b < B; ++b) {
        for (int s = w.batch_slot[b] + 1; s < w.batch_slot[b + 1]; ++s)
            if (w.slot_seg[s] < w.slot_seg[s - 1]) return 9;
        for (int seg = 0; seg <= (int)sl.segs.size(); ++seg) {
            const int m = first_slot_from_seg(w, b, seg);
            if (m < w.batch_slot[b] || m > w.batch_slot[b + 1]) return 12;
            for (int s = w.batch_slot[b]; s < w.batch_slot[b + 1]; ++s)
                if ((s < m) != (w.slot_seg[s] < seg)) return 13;
        }
    }
    if (n_ctas) *n_ctas = w.n_ctas;
    if (max_pieces) *max_pieces = maxp;
    if (min_units) *min_units = minu;
    if (max_units) *max_units = maxu;
    return 0;
}

int main() {
    // the 128K / 16x layer: per batch element 64 latent tiles and 8 raw segments of 8 tiles,
    // each tile costing 5 (four 32 KB slots + 1)
    SegList h;
    h.segs.push_back({64, 5});
    for (int g = 0; g < 8; ++g) h.segs.push_back({8, 5});
    int n = 0, mp = 0, mn = 0, mx = 0;
    if (check(8, h, 148, &n, &mp, &mn, &mx)) return 10;
    std::printf("headline: %d CTAs, max %d pieces, %d..%d tiles\n", n, mp, mn, mx);
    if (n != 128 || mp != 1 || mn != 8 || mx != 8) return 11;
    srand(1);
    for (int t = 0; t < 20000; ++t) {
        SegList s;
        const int ns = 1 + rand() % 12;
        int units = 0;
        for (int i = 0; i < ns; ++i) {
            s.segs.push_back({rand() % 40, 1 + rand() % 9});
            units += s.segs.back().first;
        }
        const int B = 1 + rand() % 9, G = 1 + rand() % 160;
        if (units == 0) continue;
        const int e = check(B, s, G, nullptr, nullptr, nullptr, nullptr);
        if (e) {
            std::printf("case %d failed with %d\n", t, e);
            return 20 + e;
        }
    }
    std::printf("random cases ok\n");
    return 0;
}
