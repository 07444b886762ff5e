// spin_budget.cu -- per-layer block budgets (host side of the library).
//
// "Sparse Attention Still Has a Dense Problem" (the SPIN project page), section "Per-layer
// block budgets", Figures 5-6: a layer's miss rate is the fraction of the dense indexer's
// top-K slots that fall into skipped blocks; a dense probe step every P decoding steps
// measures each layer's miss curve (its miss rate at each budget); the budgets minimise the
// worst layer's miss rate while the total budget across layers stays at the target block
// sparsity, and they are published to a device-side table.
//
// Budgets here are kept fractions on a grid of G + 1 points (p_g = g * 10000 / G basis
// points, G divides 10000).  The curve at p is measured against the selection the method
// makes at that budget without its random exploration share: the budget rule's m blocks, the
// forced first and last blocks, then the best m - f blocks by predicted block score (equal
// scores: lower block id).  The selections are nested in m, so one ordering of the blocks and
// a prefix count of the dense top-K hits per position give every point of the curve.  A
// batch's curve is the mean of its requests' curves.
//
// The allocation finds the smallest attainable worst miss tau* by bisection over the
// curves' distinct values (a layer's fewest points reaching miss <= tau only falls as tau
// grows), gives each layer those points, and hands the spare points out one at a time to the
// layer with the largest miss at its current point (equal misses: the layer with fewer
// points, then the lower index, so flat curves keep the uniform budget; a layer at the top of
// the grid takes none), through a max-heap.
#include <algorithm>
#include <cmath>
#include <queue>
#include <vector>

#include "spin_common.cuh"
#include "spin_internal.h"

namespace spin {

int64_t budget_blocks_host(int64_t nb, int64_t top_k, int32_t rho_bp) {
    const int64_t floor_k = (top_k + kBlock - 1) / kBlock;
    const int64_t keep = ((int64_t)(10000 - rho_bp) * nb + 9999) / 10000;
    const int64_t m = floor_k > keep ? floor_k : keep;
    return m < nb ? m : nb;
}

// One request's curve, accumulated into acc[n_points]; returns false when the dense top-K
// holds no valid slot (the request is then left out of the mean).
static bool miss_curve_one(const float* S, int32_t nb, const int32_t* topk, int32_t top_k, int32_t n_points,
                           double* acc) {
    int64_t nvalid = 0;
    for (int32_t k = 0; k < top_k; ++k) nvalid += topk[k] >= 0;
    if (nvalid == 0) return false;
    // free blocks in selection order: predicted score descending, block id ascending
    std::vector<int32_t> order;
    order.reserve(nb);
    for (int32_t j = 1; j + 1 < nb; ++j) order.push_back(j);
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return S[a] > S[b]; });
    std::vector<int32_t> pos(nb, -1);  // position among the free blocks (-1: forced)
    for (size_t p = 0; p < order.size(); ++p) pos[order[p]] = (int32_t)p;
    std::vector<int64_t> hits(order.size() + 1, 0);
    for (int32_t k = 0; k < top_k; ++k) {
        if (topk[k] < 0) continue;
        const int32_t p = pos[topk[k] / kBlock];
        if (p >= 0) ++hits[p + 1];
    }
    for (size_t p = 1; p < hits.size(); ++p) hits[p] += hits[p - 1];  // hits[t]: in the first t free blocks
    const int64_t free_hits = hits[order.size()];
    const int32_t f = nb > 1 ? 2 : 1;
    const int32_t G = n_points - 1;
    for (int32_t g = 0; g < n_points; ++g) {
        const int32_t keep_bp = (int32_t)((int64_t)g * 10000 / G);
        const int64_t m = budget_blocks_host(nb, top_k, 10000 - keep_bp);
        const int64_t t = std::min<int64_t>(std::max<int64_t>(m - f, 0), (int64_t)order.size());
        acc[g] += (double)(free_hits - hits[t]) / (double)nvalid;
    }
    return true;
}

void mean_miss_curve_host(const float* S, int32_t n_req, int64_t s_stride, const int32_t* nb,
                          const int32_t* topk, int32_t top_k, int32_t n_points, float* miss) {
    std::vector<double> acc(n_points, 0.0);
    int32_t used = 0;
    for (int32_t r = 0; r < n_req; ++r) {
        std::vector<double> one(n_points, 0.0);
        if (!miss_curve_one(S + (int64_t)r * s_stride, nb[r], topk + (int64_t)r * top_k, top_k, n_points,
                            one.data()))
            continue;
        for (int32_t g = 0; g < n_points; ++g) acc[g] += one[g];
        ++used;
    }
    for (int32_t g = 0; g < n_points; ++g) miss[g] = used ? (float)(acc[g] / used) : 0.0f;
}

void allocate_budgets_host(const float* miss, int32_t n_layers, int32_t n_points, int32_t target_g,
                           int32_t g_min, int32_t* g_out) {
    const int32_t G = n_points - 1;
    const int64_t total = (int64_t)n_layers * target_g;
    auto at = [&](int32_t l, int32_t g) { return miss[(int64_t)l * n_points + g]; };
    std::vector<float> taus;
    for (int32_t l = 0; l < n_layers; ++l)
        for (int32_t g = g_min; g <= G; ++g) taus.push_back(at(l, g));
    std::sort(taus.begin(), taus.end());
    taus.erase(std::unique(taus.begin(), taus.end()), taus.end());
    auto need = [&](int32_t l, float tau) {
        for (int32_t g = g_min; g <= G; ++g)
            if (at(l, g) <= tau) return g;
        return -1;
    };
    auto fits = [&](float tau) {
        int64_t s = 0;
        for (int32_t l = 0; l < n_layers; ++l) {
            const int32_t g = need(l, tau);
            if (g < 0) return false;
            s += g;
        }
        return s <= total;
    };
    // the largest value fits (every layer reaches it at g_min or later, and the total is at
    // least n_layers * g_min), so the bisection ends on the smallest value that fits
    size_t lo = 0, hi = taus.size() - 1;
    while (lo < hi) {
        const size_t mid = (lo + hi) / 2;
        if (fits(taus[mid])) hi = mid;
        else lo = mid + 1;
    }
    int64_t used = 0;
    for (int32_t l = 0; l < n_layers; ++l) {
        g_out[l] = need(l, taus[lo]);
        used += g_out[l];
    }
    // spare points: largest miss first; on equal misses fewer points, then lower layer
    struct Cand {
        float miss;
        int32_t g, l;
    };
    auto worse = [](const Cand& a, const Cand& b) {
        if (a.miss != b.miss) return a.miss < b.miss;
        if (a.g != b.g) return a.g > b.g;
        return a.l > b.l;
    };
    std::priority_queue<Cand, std::vector<Cand>, decltype(worse)> heap(worse);
    for (int32_t l = 0; l < n_layers; ++l)
        if (g_out[l] < G) heap.push({at(l, g_out[l]), g_out[l], l});
    for (int64_t s = used; s < total && !heap.empty(); ++s) {
        const int32_t l = heap.top().l;
        heap.pop();
        ++g_out[l];
        if (g_out[l] < G) heap.push({at(l, g_out[l]), g_out[l], l});
    }
}

}  // namespace spin
