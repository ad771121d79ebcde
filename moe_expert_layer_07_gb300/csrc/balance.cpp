// Balanced expert permutation (Moreh report "21K output tokens/s DeepSeek
// inference on MI300X with Expert Parallelism", section "Load balancing
// across GPUs"): group the experts into equal-size sets whose summed
// activation counts are as even as possible, then renumber them so every
// set is a contiguous block of physical ids.  The report calls it a variant
// of balanced number partitioning and gives no algorithm; this one minimises
// the largest set total:
//   E <= 16  exact branch and bound (items in decreasing count, a new set is
//            opened only as the first empty one, bound = current best);
//   E > 16   greedy (largest count first into the lightest set with room)
//            followed by improving swaps between the heaviest set and any
//            other, best swap first, until none lowers the heaviest set.
// Host-only code.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <numeric>
#include <vector>

#include "../../include/moe_gb300.h"

namespace {

struct Partition {
    std::vector<int> set_of;   // per expert
    std::vector<int64_t> load;
};

Partition greedy(const std::vector<int64_t> &c, int S, int m) {
    const int E = (int)c.size();
    std::vector<int> order(E);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return c[a] > c[b]; });
    Partition p;
    p.set_of.assign(E, -1);
    p.load.assign(S, 0);
    std::vector<int> size(S, 0);
    for (int e : order) {
        int best = -1;
        for (int s = 0; s < S; ++s)
            if (size[s] < m && (best < 0 || p.load[s] < p.load[best])) best = s;
        p.set_of[e] = best;
        p.load[best] += c[e];
        ++size[best];
    }
    return p;
}

void improve_by_swaps(const std::vector<int64_t> &c, int S, Partition &p) {
    const int E = (int)c.size();
    for (int iter = 0; iter < 100000; ++iter) {
        int A = 0;
        for (int s = 1; s < S; ++s)
            if (p.load[s] > p.load[A]) A = s;
        int64_t best_new = p.load[A];
        int ba = -1, bb = -1;
        for (int a = 0; a < E; ++a) {
            if (p.set_of[a] != A) continue;
            for (int b = 0; b < E; ++b) {
                const int B = p.set_of[b];
                if (B == A || c[b] >= c[a]) continue;
                const int64_t d = c[a] - c[b];
                const int64_t nm = std::max(p.load[A] - d, p.load[B] + d);
                if (nm < best_new) {
                    best_new = nm;
                    ba = a;
                    bb = b;
                }
            }
        }
        if (ba < 0) return;
        const int B = p.set_of[bb];
        const int64_t d = c[ba] - c[bb];
        p.load[A] -= d;
        p.load[B] += d;
        std::swap(p.set_of[ba], p.set_of[bb]);
    }
}

struct Exact {
    const std::vector<int64_t> &c;
    std::vector<int> order;
    int S, m;
    std::vector<int64_t> load;
    std::vector<int> size, assign, best_assign;
    int64_t best;

    Exact(const std::vector<int64_t> &counts, int S_, int m_, const Partition &seed)
        : c(counts), S(S_), m(m_) {
        const int E = (int)c.size();
        order.resize(E);
        std::iota(order.begin(), order.end(), 0);
        std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return c[a] > c[b]; });
        load.assign(S, 0);
        size.assign(S, 0);
        assign.assign(E, -1);
        best_assign = seed.set_of;
        best = *std::max_element(seed.load.begin(), seed.load.end());
    }
    void run(int i, int64_t cur_max) {
        if (cur_max >= best) return;
        if (i == (int)order.size()) {
            best = cur_max;
            best_assign = assign;
            return;
        }
        const int e = order[i];
        bool tried_empty = false;
        for (int s = 0; s < S; ++s) {
            if (size[s] == m) continue;
            if (size[s] == 0) {
                if (tried_empty) continue;   // empty sets are interchangeable
                tried_empty = true;
            }
            load[s] += c[e];
            ++size[s];
            assign[e] = s;
            run(i + 1, std::max(cur_max, load[s]));
            assign[e] = -1;
            --size[s];
            load[s] -= c[e];
        }
    }
};

// Sets are numbered by their lowest logical id; inside a set, logical ids
// ascend; set s holds physical ids [s*m, (s+1)*m).
void write_layout(const Partition &p, int S, int m, int32_t *log2phys, int32_t *phys2log) {
    const int E = (int)p.set_of.size();
    std::vector<int> first(S, E);
    for (int e = 0; e < E; ++e) first[p.set_of[e]] = std::min(first[p.set_of[e]], e);
    std::vector<int> set_rank(S);
    std::iota(set_rank.begin(), set_rank.end(), 0);
    std::sort(set_rank.begin(), set_rank.end(), [&](int a, int b) { return first[a] < first[b]; });
    std::vector<int> slot_of_set(S);
    for (int r = 0; r < S; ++r) slot_of_set[set_rank[r]] = r;
    std::vector<int> fill(S, 0);
    for (int e = 0; e < E; ++e) {
        const int s = slot_of_set[p.set_of[e]];
        const int phys = s * m + fill[s]++;
        log2phys[e] = phys;
        phys2log[phys] = e;
    }
}

}  // namespace

extern "C" int expert_balance_permutation(const int64_t *counts, int32_t num_experts,
                                          int32_t num_sets, int32_t *log2phys, int32_t *phys2log,
                                          double *max_over_mean) {
    if (!counts || !log2phys || !phys2log || num_experts <= 0 || num_sets <= 0 ||
        num_experts % num_sets)
        return MOE_ERR_INVALID_ARG;
    const int E = num_experts, S = num_sets, m = E / S;
    std::vector<int64_t> c(counts, counts + E);
    for (int64_t v : c)
        if (v < 0) return MOE_ERR_INVALID_ARG;

    Partition p = greedy(c, S, m);
    improve_by_swaps(c, S, p);
    if (E <= 16) {
        Exact ex(c, S, m, p);
        ex.run(0, 0);
        p.set_of = ex.best_assign;
        p.load.assign(S, 0);
        for (int e = 0; e < E; ++e) p.load[p.set_of[e]] += c[e];
    }

    write_layout(p, S, m, log2phys, phys2log);
    if (max_over_mean) {
        const int64_t total = std::accumulate(c.begin(), c.end(), (int64_t)0);
        const int64_t mx = *std::max_element(p.load.begin(), p.load.end());
        *max_over_mean = total > 0 ? (double)mx * S / (double)total : 1.0;
    }
    return MOE_OK;
}

namespace {

// Co-activation kept inside sets: sum of A[a][b], a < b, same set.
int64_t intra(const std::vector<int> &set_of, const int64_t *A, int E) {
    int64_t v = 0;
    for (int a = 0; a < E; ++a)
        for (int b = a + 1; b < E; ++b)
            if (set_of[a] == set_of[b]) v += A[(size_t)a * E + b];
    return v;
}

// Exhaustive search (tiny E): the lowest unplaced expert opens a set, which
// is completed with every combination of the remaining ones under the bound.
struct AffinityExact {
    const std::vector<int64_t> &c;
    const int64_t *A;
    int E, m;
    int64_t bound, best = -1;
    std::vector<int> set_of, best_set_of;
    int next_set = 0;
    AffinityExact(const std::vector<int64_t> &counts, const int64_t *aff, int E_, int m_, int64_t b)
        : c(counts), A(aff), E(E_), m(m_), bound(b), set_of(E_, -1) {}
    void run(int64_t acc) {
        int first = -1;
        for (int e = 0; e < E; ++e)
            if (set_of[e] < 0) {
                first = e;
                break;
            }
        if (first < 0) {
            if (acc > best) {
                best = acc;
                best_set_of = set_of;
            }
            return;
        }
        const int s = next_set++;
        std::vector<int> members{first};
        set_of[first] = s;
        choose(first + 1, members, c[first], acc);
        set_of[first] = -1;
        --next_set;
    }
    void choose(int from, std::vector<int> &members, int64_t load, int64_t acc) {
        if ((int)members.size() == m) {
            int64_t gain = 0;
            for (size_t i = 0; i < members.size(); ++i)
                for (size_t j = i + 1; j < members.size(); ++j)
                    gain += A[(size_t)members[i] * E + members[j]];
            run(acc + gain);
            return;
        }
        for (int e = from; e < E; ++e) {
            if (set_of[e] >= 0 || load + c[e] > bound) continue;
            set_of[e] = set_of[members[0]];
            members.push_back(e);
            choose(e + 1, members, load + c[e], acc);
            members.pop_back();
            set_of[e] = -1;
        }
    }
};

}  // namespace

// Affinity-aware placement (SGLang/H20 article, section "Expert Affinity
// EPLB": co-locate experts that are often selected together).  Start from
// the balanced partition (largest set total L*), then maximise the
// co-activation kept inside sets while every set total stays within
// max(L*, floor((1 + slack) * mean)): exhaustively for E <= 16, otherwise by
// best-improvement swaps between sets.
extern "C" int expert_set_imbalance(const int64_t *counts, const int32_t *log2phys,
                                    int32_t num_experts, int32_t num_sets,
                                    double *max_over_mean) {
    if (!counts || !max_over_mean || num_experts <= 0 || num_sets <= 0 ||
        num_experts % num_sets)
        return MOE_ERR_INVALID_ARG;
    const int E = num_experts, S = num_sets, m = E / S;
    std::vector<int64_t> load(S, 0);
    std::vector<char> seen(E, 0);
    for (int e = 0; e < E; ++e) {
        const int p = log2phys ? log2phys[e] : e;
        if (counts[e] < 0 || p < 0 || p >= E || seen[p]) return MOE_ERR_INVALID_ARG;
        seen[p] = 1;
        load[p / m] += counts[e];
    }
    const int64_t total = std::accumulate(load.begin(), load.end(), (int64_t)0);
    const int64_t mx = *std::max_element(load.begin(), load.end());
    *max_over_mean = total > 0 ? (double)mx * S / (double)total : 1.0;
    return MOE_OK;
}

extern "C" int expert_affinity_permutation(const int64_t *counts, const int64_t *coact,
                                           int32_t num_experts, int32_t num_sets,
                                           double load_slack, int32_t *log2phys,
                                           int32_t *phys2log, double *max_over_mean,
                                           double *intra_fraction) {
    if (!counts || !coact || !log2phys || !phys2log || num_experts <= 0 || num_sets <= 0 ||
        num_experts % num_sets || !(load_slack >= 0.0))
        return MOE_ERR_INVALID_ARG;
    const int E = num_experts, S = num_sets, m = E / S;
    std::vector<int64_t> c(counts, counts + E);
    for (int64_t v : c)
        if (v < 0) return MOE_ERR_INVALID_ARG;
    for (int a = 0; a < E; ++a)
        for (int b = 0; b < E; ++b)
            if (coact[(size_t)a * E + b] < 0 || coact[(size_t)a * E + b] != coact[(size_t)b * E + a])
                return MOE_ERR_INVALID_ARG;

    Partition p = greedy(c, S, m);
    improve_by_swaps(c, S, p);
    if (E <= 16) {
        Exact ex(c, S, m, p);
        ex.run(0, 0);
        p.set_of = ex.best_assign;
    }
    p.load.assign(S, 0);
    for (int e = 0; e < E; ++e) p.load[p.set_of[e]] += c[e];
    const int64_t balanced_max = *std::max_element(p.load.begin(), p.load.end());
    const int64_t total = std::accumulate(c.begin(), c.end(), (int64_t)0);
    const int64_t bound = std::max<int64_t>(
        balanced_max, (int64_t)std::floor((1.0 + load_slack) * (double)total / S));

    if (E <= 16) {
        AffinityExact ax(c, coact, E, m, bound);
        ax.run(0);
        if (ax.best >= 0) p.set_of = ax.best_set_of;
    } else {
        // W[e][s] = co-activation of expert e with the members of set s
        std::vector<int64_t> W((size_t)E * S, 0);
        for (int a = 0; a < E; ++a)
            for (int b = 0; b < E; ++b) W[(size_t)a * S + p.set_of[b]] += coact[(size_t)a * E + b];
        for (int iter = 0; iter < 100000; ++iter) {
            int64_t best_gain = 0;
            int ba = -1, bb = -1;
            for (int a = 0; a < E; ++a) {
                const int sa = p.set_of[a];
                for (int b = a + 1; b < E; ++b) {
                    const int sb = p.set_of[b];
                    if (sa == sb) continue;
                    const int64_t la = p.load[sa] - c[a] + c[b], lb = p.load[sb] - c[b] + c[a];
                    if (la > bound || lb > bound) continue;
                    const int64_t ab = coact[(size_t)a * E + b];
                    const int64_t gain = (W[(size_t)a * S + sb] - ab - W[(size_t)a * S + sa]) +
                                         (W[(size_t)b * S + sa] - ab - W[(size_t)b * S + sb]);
                    if (gain > best_gain) {
                        best_gain = gain;
                        ba = a;
                        bb = b;
                    }
                }
            }
            if (ba < 0) break;
            const int sa = p.set_of[ba], sb = p.set_of[bb];
            for (int e = 0; e < E; ++e) {
                W[(size_t)e * S + sa] += coact[(size_t)e * E + bb] - coact[(size_t)e * E + ba];
                W[(size_t)e * S + sb] += coact[(size_t)e * E + ba] - coact[(size_t)e * E + bb];
            }
            p.load[sa] += c[bb] - c[ba];
            p.load[sb] += c[ba] - c[bb];
            std::swap(p.set_of[ba], p.set_of[bb]);
        }
    }
    p.load.assign(S, 0);
    for (int e = 0; e < E; ++e) p.load[p.set_of[e]] += c[e];
    write_layout(p, S, m, log2phys, phys2log);
    if (max_over_mean) {
        const int64_t mx = *std::max_element(p.load.begin(), p.load.end());
        *max_over_mean = total > 0 ? (double)mx * S / (double)total : 1.0;
    }
    if (intra_fraction) {
        int64_t all = 0;
        for (int a = 0; a < E; ++a)
            for (int b = a + 1; b < E; ++b) all += coact[(size_t)a * E + b];
        *intra_fraction = all > 0 ? (double)intra(p.set_of, coact, E) / (double)all : 1.0;
    }
    return MOE_OK;
}
