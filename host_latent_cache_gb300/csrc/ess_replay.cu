// Replay of hot-pool eviction policies over a trace of selections (host code
// only).
//
// hwcomputing.csdn.net FlashOffloading analysis, section "evaluation", the
// decode ablation and its Figure 8: the top-k indices of every step are
// collected once, then an offline simulator replays the same access sequence
// with only the eviction policy changed (Random, LRU, Score: evict low-score
// tokens, LIM: a score threshold plus a chunk scan) and counts the misses per
// request, summed over the MTP ways.
//
// One step of one request: the union of the ways' selections is resolved
// against the token -> slot map; hits are stamped with the step; the slots
// not holding a union token are the candidates, empty slots first in slot
// order, then the resident ones by the policy's key, ties to the lower slot;
// the i-th miss (ascending token) takes the i-th candidate.  Keys: LRU the
// last step of use; Random a SplitMix64 draw (Steele, Lea and Flood, "Fast
// Splittable Pseudorandom Number Generators", OOPSLA 2014) keyed by (seed,
// request, step) and the slot; Score the token's score this step, the
// maximum over the ways; LIM none, i.e. slot order (its threshold read as
// the top-k cutoff, which every candidate is below).
#include <algorithm>
#include <vector>

#include "ess_internal.h"

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

// the (i+1)-th output of SplitMix64 seeded with key
uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * kGamma); }

uint64_t step_key(uint64_t seed, int64_t request, int64_t step) {
  uint64_t k = seed;
  k = mix64((k ^ static_cast<uint64_t>(request)) + kGamma);
  k = mix64((k ^ static_cast<uint64_t>(step)) + kGamma);
  return k;
}

struct Cand {
  int resident;     // 0: empty slot, 1: resident
  uint64_t ukey;    // Random
  int64_t ikey;     // LRU
  double fkey;      // Score
  int slot;
};

}  // namespace

extern "C" ess_status ess_replay_misses(int32_t n_steps, int32_t n_ways, const int64_t* offsets,
                                        const int32_t* tokens, const float* scores, int32_t T,
                                        int32_t C, int32_t policy, uint64_t seed,
                                        int64_t request, int32_t* union_misses,
                                        int32_t* way_misses) {
  if (n_steps < 0 || n_ways < 1 || T < 1 || C < 1 || policy < ESS_EVICT_LRU ||
      policy > ESS_EVICT_LIM || (n_steps > 0 && (!offsets || !tokens || !union_misses ||
                                                 !way_misses)) ||
      (policy == ESS_EVICT_SCORE && n_steps > 0 && !scores))
    return ESS_ERR_INVALID_ARG;
  std::vector<int32_t> slot_of(T, -1), slot_token(C, -1);
  std::vector<int64_t> last_used(C, -1);
  std::vector<uint8_t> held(C, 0);
  std::vector<int32_t> uni, miss;
  std::vector<Cand> cand;
  for (int s = 0; s < n_steps; ++s) {
    uni.clear();
    int wm = 0;
    for (int m = 0; m < n_ways; ++m) {
      const int64_t a = offsets[s * n_ways + m], b = offsets[s * n_ways + m + 1];
      if (a < 0 || b < a) return ESS_ERR_INVALID_ARG;
      for (int64_t e = a; e < b; ++e) {
        const int32_t t = tokens[e];
        if (t < 0 || t >= T) return ESS_ERR_INVALID_ARG;
        if (slot_of[t] < 0) ++wm;
        uni.push_back(t);
      }
    }
    std::sort(uni.begin(), uni.end());
    uni.erase(std::unique(uni.begin(), uni.end()), uni.end());
    if (static_cast<int64_t>(uni.size()) > C) return ESS_ERR_CAPACITY;
    std::fill(held.begin(), held.end(), 0);
    miss.clear();
    for (int32_t t : uni) {
      if (slot_of[t] >= 0) {
        last_used[slot_of[t]] = s;       // hits are stamped first
        held[slot_of[t]] = 1;
      } else {
        miss.push_back(t);
      }
    }
    cand.clear();
    const uint64_t key = step_key(seed, request, s);
    for (int v = 0; v < C; ++v) {
      if (held[v]) continue;
      Cand c{slot_token[v] >= 0 ? 1 : 0, 0, 0, 0.0, v};
      if (c.resident) {
        if (policy == ESS_EVICT_LRU) c.ikey = last_used[v];
        if (policy == ESS_EVICT_RANDOM) c.ukey = draw(key, static_cast<uint64_t>(v));
        if (policy == ESS_EVICT_SCORE) {
          float best = scores[(static_cast<int64_t>(s) * n_ways) * T + slot_token[v]];
          for (int m = 1; m < n_ways; ++m)
            best = std::max(best, scores[(static_cast<int64_t>(s) * n_ways + m) * T + slot_token[v]]);
          c.fkey = best;
        }
      }
      cand.push_back(c);
    }
    const size_t n = miss.size();
    std::partial_sort(cand.begin(), cand.begin() + n, cand.end(), [](const Cand& x, const Cand& y) {
      if (x.resident != y.resident) return x.resident < y.resident;
      if (x.ikey != y.ikey) return x.ikey < y.ikey;
      if (x.ukey != y.ukey) return x.ukey < y.ukey;
      if (x.fkey != y.fkey) return x.fkey < y.fkey;
      return x.slot < y.slot;
    });
    for (size_t i = 0; i < n; ++i) {
      const int v = cand[i].slot;
      if (slot_token[v] >= 0) slot_of[slot_token[v]] = -1;
      slot_of[miss[i]] = v;
      slot_token[v] = miss[i];
      last_used[v] = s;
    }
    union_misses[s] = static_cast<int32_t>(n);
    way_misses[s] = wm;
  }
  return ESS_OK;
}
