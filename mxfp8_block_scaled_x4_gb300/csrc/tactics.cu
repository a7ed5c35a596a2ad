// tactics.cu -- the tactic table: measured GEMM schedules per problem class.
//
// The pages leave tactic selection to later work (vLLM PR #52204: "This PR
// does not add tactic hints"; FlashInfer PR #1214 review: an "autotuner for
// these kernels ... with benching/perf tuning").  Here a tactic is a
// GemmSchedule; the table maps (device, call kind, power-of-two bucket of M,
// N, K, experts) to the schedule an autotuning run measured fastest.  The
// calls consult the table before the built-in heuristic.  Host code only.
#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "internal.h"

namespace mxk {

namespace {

struct Key {
    int dev, kind;
    int64_t mb, n, k, e;
    bool operator<(const Key& o) const {
        return std::tie(dev, kind, mb, n, k, e) < std::tie(o.dev, o.kind, o.mb, o.n, o.k, o.e);
    }
};

std::mutex g_mu;
std::map<Key, GemmSchedule> g_table;

Key make_key(int dev, int kind, int64_t m, int64_t n, int64_t k, int64_t experts) {
    return Key{dev, kind, m_bucket(m), n, k, experts};
}

}  // namespace

int64_t m_bucket(int64_t m) {
    int64_t b = 1;
    while (b < m) b <<= 1;
    return b;
}

bool schedule_valid(const GemmSchedule& s, int kind, int64_t k) {
    const int tt = s.tokens_per_tile;
    const bool grouped = kind == kTacticGrouped || kind == kTacticGated;
    if (s.dual)
        return (kind == kTacticLinear || kind == kTacticGemm) && (tt == 144 || tt == 160 || tt == 176 || tt == 192) &&
               s.pipes == 2;
    if (tt != 16 && tt != 32 && tt != 64 && tt != 128 && tt != 256) return false;
    if (s.pipes == 2 && tt > 64) return false;
    // Four pipelines: 16-token tiles (not gated) and 32-token tiles.
    if (s.pipes == 4 && !((tt == 16 && kind != kTacticGated) || tt == 32)) return false;
    if (s.pipes != 1 && s.pipes != 2 && s.pipes != 4) return false;
    if (kind == kTacticGated && tt > 128) return false;
    if (s.persistent) {
        if (s.split_k != 1 || s.fuse_quant) return false;
    } else {
        if (grouped || tt > 128) return false;
        if (s.split_k < 1 || s.split_k > 8 || s.split_k > k / 128) return false;
        if (s.fuse_quant && kind != kTacticLinear) return false;
    }
    return true;
}

bool tactic_lookup(int dev, int kind, int64_t m, int64_t n, int64_t k, int64_t experts, GemmSchedule* out) {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_table.find(make_key(dev, kind, m, n, k, experts));
    if (it == g_table.end()) return false;
    *out = it->second;
    return true;
}

void tactic_store(int dev, int kind, int64_t m, int64_t n, int64_t k, int64_t experts, const GemmSchedule& s) {
    std::lock_guard<std::mutex> lock(g_mu);
    g_table[make_key(dev, kind, m, n, k, experts)] = s;
}

void tactic_clear() {
    std::lock_guard<std::mutex> lock(g_mu);
    g_table.clear();
}

int64_t tactic_count() {
    std::lock_guard<std::mutex> lock(g_mu);
    return static_cast<int64_t>(g_table.size());
}

std::vector<GemmSchedule> candidate_schedules(int kind, int64_t m, int64_t k) {
    std::vector<GemmSchedule> out;
    auto add = [&](int tt, int split, bool persistent, bool fuse, int pipes, bool dual) {
        GemmSchedule s;
        s.tokens_per_tile = tt;
        s.split_k = split;
        s.persistent = persistent;
        s.fuse_quant = fuse;
        s.pipes = pipes;
        s.dual = dual;
        if (schedule_valid(s, kind, k)) out.push_back(s);
    };
    const bool grouped = kind == kTacticGrouped || kind == kTacticGated;
    const int pipes_of[3] = {1, 2, 4};
    for (int tt : {16, 32, 64, 128, 256}) {
        // Persistent tiles: every kind.
        for (int pp : pipes_of) add(tt, 1, true, false, pp, false);
        if (grouped || tt > 128) continue;
        // One tile per cluster of `split` CTAs: dense, tiles not far beyond M.
        if (tt > 2 * m_bucket(m) && tt > 16) continue;
        for (int split : {1, 2, 3, 4, 6, 8})
            for (int pp : pipes_of) {
                add(tt, split, false, false, pp, false);
                if (kind == kTacticLinear && m <= 128) add(tt, split, false, true, pp, false);
            }
    }
    if (!grouped && m > 128) {
        for (int tt : {192, 176, 160, 144}) add(tt, 1, true, false, 2, true);
    }
    return out;
}

}  // namespace mxk
