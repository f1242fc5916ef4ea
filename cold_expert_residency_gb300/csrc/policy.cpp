// Adaptive residency policy (host side, between steps).
//
// "We Built the Counter", section 2: a side thread reads the usage table every
// N steps, keeps a decaying average and queues swaps decided against a CPU
// copy of each layer's hot/cold lists; section 9 gives the defaults (read
// every 64 steps, 500-step half-life, <= 2 swaps per layer per read, 1.5x
// hysteresis, minimum average 8, <= 8 swaps per step).  The average is an
// exponentially weighted mean of the per-read pick counts, normalised by the
// decayed weight sum so that it is unbiased from the first read.
//
// The same section lets an operator ask for the placement chosen at start-up
// back, and checks that swapping back to it loses nothing.  The restore
// planner gives those swaps for any saved placement.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <new>
#include <string>
#include <vector>

#include "../../include/moe_residency.h"

// The library's thread-local error message (moe_abi.cu); the header that
// declares it also carries CUDA types, which this host-only file does without.
namespace moe {
int set_error(int code, const std::string &msg);
}
using moe::set_error;

struct moe_policy {
    int E;
    double decay, hysteresis, min_avg;
    int max_pairs;
    std::vector<uint32_t> last;
    std::vector<double> acc;
    double wsum = 0.0;
};

extern "C" {

int moe_policy_create(int experts, double read_every, double half_life, double hysteresis, double min_avg,
                      int max_pairs, const int32_t *counts_now, moe_policy **out) {
    if (!out || experts < 1 || !(read_every > 0) || !(half_life > 0) || !(hysteresis >= 1.0) || max_pairs < 0)
        return set_error(MOE_EINVAL, "invalid policy parameter");
    moe_policy *p = new (std::nothrow) moe_policy();
    if (!p) return set_error(MOE_ENOMEM, "out of host memory");
    p->E = experts;
    p->decay = std::pow(0.5, read_every / half_life);
    p->hysteresis = hysteresis;
    p->min_avg = min_avg;
    p->max_pairs = max_pairs;
    try {
        p->last.assign(experts, 0u);
        p->acc.assign(experts, 0.0);
    } catch (const std::bad_alloc &) {
        delete p;
        return set_error(MOE_ENOMEM, "out of host memory");
    }
    if (counts_now)
        for (int e = 0; e < experts; ++e) p->last[e] = (uint32_t)counts_now[e];
    *out = p;
    return MOE_OK;
}

int moe_policy_destroy(moe_policy *p) {
    delete p;
    return MOE_OK;
}

static int policy_read(moe_policy *p, const int32_t *counts, const int32_t *row_map, int32_t *promote,
                       int32_t *demote) {
    const int E = p->E;
    for (int e = 0; e < E; ++e) {
        const uint32_t now = (uint32_t)counts[e];
        p->acc[e] = p->decay * p->acc[e] + (double)(uint32_t)(now - p->last[e]);
        p->last[e] = now;
    }
    p->wsum = p->decay * p->wsum + 1.0;
    std::vector<double> avg(E);
    for (int e = 0; e < E; ++e) avg[e] = p->acc[e] / p->wsum;

    std::vector<int> cold, hot;
    for (int e = 0; e < E; ++e) {
        if (row_map[e] < 0) {
            if (avg[e] >= p->min_avg) cold.push_back(e);
        } else {
            hot.push_back(e);
        }
    }
    // most-used cold first, least-used hot first; equal averages by expert id
    std::stable_sort(cold.begin(), cold.end(), [&](int a, int b) { return avg[a] > avg[b]; });
    std::stable_sort(hot.begin(), hot.end(), [&](int a, int b) { return avg[a] < avg[b]; });
    const int lim = std::min({p->max_pairs, (int)cold.size(), (int)hot.size()});
    int n = 0;
    for (; n < lim; ++n) {
        if (!(avg[cold[n]] > p->hysteresis * avg[hot[n]])) break;
        promote[n] = cold[n];
        demote[n] = hot[n];
    }
    return n;
}

static int plan_restore(int experts, const int32_t *row_map, const int32_t *target, int max_pairs,
                        int32_t *promote, int32_t *demote) {
    std::vector<int> in, out;       // experts to bring into HBM, experts to move out
    for (int e = 0; e < experts; ++e) {
        const bool hot = row_map[e] >= 0, want = target[e] >= 0;
        if (hot != want) (want ? in : out).push_back(e);
    }
    if (in.size() != out.size())    // swaps never change the hot bank's size
        return set_error(MOE_EINVAL, "the two maps hold different numbers of hot experts");
    const int n = std::min((int)in.size(), max_pairs);
    for (int i = 0; i < n; ++i) {
        promote[i] = in[i];
        demote[i] = out[i];
    }
    return n;
}

int moe_policy_read(moe_policy *p, const int32_t *counts, const int32_t *row_map, int32_t *promote,
                    int32_t *demote) {
    if (!p || !counts || !row_map || !promote || !demote) return set_error(MOE_EINVAL, "null argument");
    try {
        return policy_read(p, counts, row_map, promote, demote);
    } catch (const std::bad_alloc &) {
        return set_error(MOE_ENOMEM, "out of host memory");
    }
}

int moe_plan_restore(int experts, const int32_t *row_map, const int32_t *target, int max_pairs,
                     int32_t *promote, int32_t *demote) {
    if (experts < 1 || !row_map || !target || max_pairs < 0 || ((!promote || !demote) && max_pairs > 0))
        return set_error(MOE_EINVAL, "invalid argument");
    try {
        return plan_restore(experts, row_map, target, max_pairs, promote, demote);
    } catch (const std::bad_alloc &) {
        return set_error(MOE_ENOMEM, "out of host memory");
    }
}

}  // extern "C"
