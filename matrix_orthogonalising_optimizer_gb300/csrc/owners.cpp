// Owner assignment for the per-owner Muon step (host code only).
//
// DMuon gives every weight matrix a single owner rank, which alone keeps the
// matrix's optimizer state and runs its Newton-Schulz update.  The update's
// cost depends strongly on the matrix shape, so a round-robin assignment
// leaves straggling ranks; DMuon instead chooses the owners that minimise the
// predicted makespan -- the largest per-rank sum of predicted costs -- posed
// as a mixed-integer program, with a greedy heuristic for very large
// instances (DMuon technical summary on gist.science, section 2.3
// "compute-aware load balancing").
//
// The single-GPU library has no ranks; this computes the assignment a
// multi-rank caller would use, from costs it supplies (measured per bucket,
// or the plan's per-matrix FLOPs).
//   greedy: longest processing time first -- matrices in decreasing cost
//           (ties: lower index first), each to the currently least-loaded
//           rank (ties: lower rank).
//   exact:  the optimum of the makespan program, found by depth-first branch
//           and bound over the matrices in the greedy order, starting from
//           the greedy solution; a branch is cut when its load bound cannot
//           beat the best makespan found, and among ranks still empty only
//           the first is tried (they are interchangeable).
// The reported makespan is recomputed from the final assignment, each rank's
// costs summed in increasing matrix index, so it does not depend on the
// search order.
#include <algorithm>
#include <cmath>
#include <numeric>
#include <string>
#include <vector>

#include "dmuon.h"

namespace dmuon {
void set_last_error(const std::string& msg);
}

namespace {

constexpr int64_t kExactMaxCount = 32;
constexpr int64_t kExactMaxNodes = 200000000;

int fail(int code, const std::string& msg) {
    dmuon::set_last_error(msg);
    return code;
}

std::vector<int64_t> greedy_order(const double* costs, int64_t count) {
    std::vector<int64_t> order(static_cast<size_t>(count));
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) { return costs[a] > costs[b]; });
    return order;
}

void greedy(const double* costs, const std::vector<int64_t>& order, int32_t ranks, int32_t* owner) {
    std::vector<double> load(static_cast<size_t>(ranks), 0.0);
    for (int64_t i : order) {
        int32_t best = 0;
        for (int32_t r = 1; r < ranks; ++r)
            if (load[r] < load[best]) best = r;
        owner[i] = best;
        load[best] += costs[i];
    }
}

double makespan_of(const double* costs, int64_t count, int32_t ranks, const int32_t* owner) {
    std::vector<double> load(static_cast<size_t>(ranks), 0.0);
    for (int64_t i = 0; i < count; ++i) load[owner[i]] += costs[i];
    return count > 0 ? *std::max_element(load.begin(), load.end()) : 0.0;
}

struct Search {
    const double* costs;
    std::vector<int64_t> order;
    std::vector<double> suffix;  // suffix[k] = sum of costs of order[k..]
    int32_t ranks;
    std::vector<double> load;
    std::vector<int32_t> cur, best_assign;  // indexed by matrix
    double best;
    int64_t nodes = 0;
    bool exhausted = false;

    void dfs(size_t k, double cur_max, double assigned) {
        if (++nodes > kExactMaxNodes) {
            exhausted = true;
            return;
        }
        if (k == order.size()) {
            if (cur_max < best) {
                best = cur_max;
                best_assign = cur;
            }
            return;
        }
        const double bound = std::max(cur_max, (assigned + suffix[k]) / ranks);
        if (bound >= best) return;
        const int64_t i = order[k];
        bool tried_empty = false;
        for (int32_t r = 0; r < ranks && !exhausted; ++r) {
            if (load[r] == 0.0) {
                if (tried_empty) continue;
                tried_empty = true;
            }
            const double old = load[r], nl = old + costs[i];
            if (nl >= best) continue;
            load[r] = nl;
            cur[i] = r;
            dfs(k + 1, std::max(cur_max, nl), assigned + costs[i]);
            load[r] = old;
        }
    }
};

}  // namespace

extern "C" int dmuon_assign_owners(const double* costs, int64_t count, int32_t ranks, int32_t method, int32_t* owner,
                                   double* makespan) {
    if (count < 0 || ranks < 1 || (count > 0 && (!costs || !owner)))
        return fail(DMUON_ERR_INVALID_ARG, "dmuon_assign_owners: bad count, ranks or NULL array");
    if (method != DMUON_ASSIGN_GREEDY && method != DMUON_ASSIGN_EXACT)
        return fail(DMUON_ERR_INVALID_ARG, "dmuon_assign_owners: unknown method");
    for (int64_t i = 0; i < count; ++i)
        if (!std::isfinite(costs[i]) || costs[i] < 0.0)
            return fail(DMUON_ERR_INVALID_ARG, "dmuon_assign_owners: cost " + std::to_string(i) +
                                                   " is negative or not finite");
    if (method == DMUON_ASSIGN_EXACT && count > kExactMaxCount)
        return fail(DMUON_ERR_INVALID_ARG, "dmuon_assign_owners: the exact method takes at most " +
                                               std::to_string(kExactMaxCount) + " matrices; use the greedy one");
    const std::vector<int64_t> order = greedy_order(costs, count);
    greedy(costs, order, ranks, owner);
    if (method == DMUON_ASSIGN_EXACT && count > 0) {
        // the search's own load sums run in the greedy order: start from the
        // greedy makespan measured that way
        Search s;
        s.costs = costs;
        s.order = order;
        s.ranks = ranks;
        s.suffix.assign(order.size() + 1, 0.0);
        for (size_t k = order.size(); k-- > 0;) s.suffix[k] = s.suffix[k + 1] + costs[order[k]];
        std::vector<double> gl(static_cast<size_t>(ranks), 0.0);
        for (int64_t i : order) gl[owner[i]] += costs[i];
        s.best = *std::max_element(gl.begin(), gl.end());
        s.best_assign.assign(owner, owner + count);
        s.load.assign(static_cast<size_t>(ranks), 0.0);
        s.cur.assign(static_cast<size_t>(count), 0);
        s.dfs(0, 0.0, 0.0);
        if (s.exhausted)
            return fail(DMUON_ERR_INVALID_ARG, "dmuon_assign_owners: exact search exceeded " +
                                                   std::to_string(kExactMaxNodes) + " nodes; use the greedy method");
        std::copy(s.best_assign.begin(), s.best_assign.end(), owner);
    }
    if (makespan) *makespan = makespan_of(costs, count, ranks, owner);
    return DMUON_OK;
}
