// Dedicated ownership: LPT assignment of matrices to owner ranks with a same-layer spread rule
// (DMuon "Core Concepts", section "均衡划分": global balance of the per-rank work, and the parameters of
// one layer spread over different ranks so their broadcasts run concurrently). Host-only.
#include <algorithm>
#include <cstring>
#include <numeric>
#include <unordered_map>
#include <vector>

#include "dmuon.h"
#include "internal.h"

namespace dmuon {
namespace {

double matrix_cost(int64_t rows, int64_t cols, int model) {
  const double m = static_cast<double>(std::min(rows, cols));
  const double n = static_cast<double>(std::max(rows, cols));
  switch (model) {
    case DMUON_COST_GRAM_FLOPS: return 6.0 * m * m * n + 17.0 * m * m * m;
    case DMUON_COST_DIRECT_FLOPS: return 15.0 * m * m * n + 5.0 * m * m * m;
    default: return static_cast<double>(rows) * static_cast<double>(cols);
  }
}

}  // namespace
}  // namespace dmuon

using namespace dmuon;

extern "C" int dmuon_assign_owners(int count, const int64_t* rows, const int64_t* cols, const int* layer_ids,
                                   int nranks, int cost_model, int* owner_out, double* loads_out) {
  try {
    if (count < 1) return set_error(DMUON_ERR_INVALID_ARG, "count must be >= 1");
    if (!rows || !cols || !owner_out) return set_error(DMUON_ERR_INVALID_ARG, "rows, cols and owner_out must not be NULL");
    if (nranks < 1 || nranks > 65536) return set_error(DMUON_ERR_INVALID_ARG, "nranks must be in [1, 65536]");
    if (cost_model != DMUON_COST_ELEMENTS && cost_model != DMUON_COST_GRAM_FLOPS && cost_model != DMUON_COST_DIRECT_FLOPS)
      return set_error(DMUON_ERR_INVALID_ARG, "unknown cost_model");
    for (int i = 0; i < count; ++i) {
      if (rows[i] < 1 || cols[i] < 1) return set_error(DMUON_ERR_INVALID_ARG, "matrix sizes must be >= 1");
      if (layer_ids && layer_ids[i] < 0) return set_error(DMUON_ERR_INVALID_ARG, "layer ids must be >= 0");
    }
    std::vector<double> cost(count);
    for (int i = 0; i < count; ++i) cost[i] = matrix_cost(rows[i], cols[i], cost_model);
    std::vector<int> order(count);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });

    std::vector<double> load(nranks, 0.0);
    // Matrices of each layer already placed on each rank (only the layers seen so far).
    std::unordered_map<int, std::vector<int>> per_layer;
    for (int idx : order) {
      int best = 0;
      if (layer_ids) {
        std::vector<int>& held = per_layer[layer_ids[idx]];
        if (held.empty()) held.assign(nranks, 0);
        const int fewest = *std::min_element(held.begin(), held.end());
        best = -1;
        for (int r = 0; r < nranks; ++r)
          if (held[r] == fewest && (best < 0 || load[r] < load[best])) best = r;
        held[best] += 1;
      } else {
        for (int r = 1; r < nranks; ++r)
          if (load[r] < load[best]) best = r;
      }
      owner_out[idx] = best;
      load[best] += cost[idx];
    }
    if (loads_out) std::memcpy(loads_out, load.data(), sizeof(double) * nranks);
    return DMUON_OK;
  } catch (const std::exception& e) {
    return set_error(DMUON_ERR_OOM, e.what());
  }
}
