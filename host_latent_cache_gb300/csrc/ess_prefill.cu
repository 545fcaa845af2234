// Binding table of the prefill layer schedule with four device buffers
// (host code only).
//
// hwcomputing.csdn.net FlashOffloading analysis, section "prefill side: four
// whole-layer buffers hide the transfers": B0 stays bound to layer 0 for the
// whole prefill and B1..B3 rotate over the later layers through a binding
// table; a buffer may take a new layer only once its previous layer's last
// compute and its write-back to host memory are done; at layer i's
// scheduling point the schedule prefetches layer onload_layer_map[i].
//
// The plan binds the rotating buffers round-robin in load order (the layers
// no entry of the map prefetches are loaded up front, then the prefetches in
// scheduling order) and names, for every load, the layer whose release it
// waits for.  A load can only wait for a layer whose write-back is issued
// before the load: on separate copy streams layer i's write-back is issued
// before its prefetch, on one serial copy stream after it.
#include <vector>

#include "ess_internal.h"

extern "C" ess_status ess_prefill_plan(int32_t n_layers, const int32_t* onload_layer_map,
                                       int32_t rotating, int32_t shared_copy, int32_t* buffer,
                                       int32_t* load_at, int32_t* reuse_after) {
  if (n_layers < 1 || rotating < 1 || !onload_layer_map || !buffer || !load_at || !reuse_after)
    return ESS_ERR_INVALID_ARG;
  const int L = n_layers;
  constexpr int kNotLoaded = -2;
  std::vector<int> at(L, kNotLoaded);      // scheduling point that loads each layer
  for (int i = 0; i < L; ++i) {
    const int j = onload_layer_map[i];
    if (j == -1) continue;
    if (j < 1 || j >= L || at[j] != kNotLoaded) return ESS_ERR_INVALID_ARG;
    at[j] = i;
  }
  std::vector<int> order;                  // load order
  for (int j = 1; j < L; ++j)
    if (at[j] == kNotLoaded) {
      at[j] = -1;                          // up front
      order.push_back(j);
    }
  for (int i = 0; i < L; ++i)
    if (onload_layer_map[i] >= 1) order.push_back(onload_layer_map[i]);
  buffer[0] = 0;
  load_at[0] = -1;
  reuse_after[0] = -1;
  std::vector<int> last(rotating + 1, -1);
  for (size_t n = 0; n < order.size(); ++n) {
    const int j = order[n];
    const int b = 1 + static_cast<int>(n % static_cast<size_t>(rotating));
    buffer[j] = b;
    load_at[j] = at[j];
    reuse_after[j] = last[b];
    last[b] = j;
  }
  for (int j = 1; j < L; ++j) {
    const int p = reuse_after[j], i = load_at[j];
    if (p < 0) continue;
    const bool issued_before = i >= 0 && (shared_copy ? p < i : p <= i);
    if (!issued_before) return ESS_ERR_INVALID_ARG;   // the buffer would still be held
  }
  return ESS_OK;
}
