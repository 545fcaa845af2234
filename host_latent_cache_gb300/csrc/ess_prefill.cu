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

// ---------------------------------------------------------------------------
// The engine that runs the schedule: whole-layer KV moves between pinned host
// memory and the device buffers on copy streams, the caller's per-layer
// compute runs on the compute stream, and events carry every dependency of
// the page's lifecycle (a load waits for its scheduling point and for the
// release of its buffer's previous layer; a compute waits for its load; a
// write-back follows its compute; a release follows the write-back).
extern "C" ess_status ess_prefill_run(int32_t n_layers, const int32_t* onload_layer_map,
                                      int32_t rotating, int32_t shared_copy,
                                      void* const* host_kv, size_t layer_bytes, size_t wb_offset,
                                      size_t wb_bytes, void* const* buffers,
                                      ess_prefill_compute_fn compute, void* user,
                                      ess_stream_t compute_stream, ess_stream_t h2d_stream,
                                      ess_stream_t d2h_stream) {
  if (n_layers < 1 || rotating < 1 || !host_kv || !buffers || !compute || layer_bytes == 0 ||
      wb_offset > layer_bytes || wb_bytes > layer_bytes - wb_offset)
    return ESS_ERR_INVALID_ARG;
  const int L = n_layers;
  for (int l = 1; l < L; ++l)
    if (!host_kv[l]) return ESS_ERR_INVALID_ARG;
  for (int b = 0; b <= rotating; ++b)
    if (!buffers[b]) return ESS_ERR_INVALID_ARG;
  std::vector<int32_t> buffer(L), load_at(L), reuse_after(L);
  const ess_status ps = ess_prefill_plan(n_layers, onload_layer_map, rotating, shared_copy,
                                         buffer.data(), load_at.data(), reuse_after.data());
  if (ps != ESS_OK) return ps;
  cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
  cudaStream_t hs = static_cast<cudaStream_t>(h2d_stream);
  cudaStream_t ds = shared_copy ? hs : static_cast<cudaStream_t>(d2h_stream);
  // events: loaded, computed, released and the start of each scheduling point
  std::vector<cudaEvent_t> ev(4 * static_cast<size_t>(L), nullptr);
  auto destroy = [&]() {
    for (cudaEvent_t e : ev)
      if (e) cudaEventDestroy(e);
  };
  for (auto& e : ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      destroy();
      return ESS_ERR_CUDA;
    }
  cudaEvent_t* loaded = ev.data();
  cudaEvent_t* computed = loaded + L;
  cudaEvent_t* released = computed + L;
  cudaEvent_t* point = released + L;
  bool ok = true;
  auto load = [&](int j, cudaEvent_t after) {
    if (after) ok = ok && cudaStreamWaitEvent(hs, after, 0) == cudaSuccess;
    if (reuse_after[j] >= 0)
      ok = ok && cudaStreamWaitEvent(hs, released[reuse_after[j]], 0) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(buffers[buffer[j]], host_kv[j], layer_bytes,
                               cudaMemcpyHostToDevice, hs) == cudaSuccess;
    ok = ok && cudaEventRecord(loaded[j], hs) == cudaSuccess;
  };
  for (int j = 1; j < L; ++j)       // the layers no scheduling point prefetches
    if (load_at[j] == -1) load(j, nullptr);
  // A load waits on an event that must already be recorded when it is enqueued:
  // on one copy stream the plan only lets point i's prefetch reuse a buffer
  // released before layer i, and the prefetch goes ahead of i's write-back;
  // on separate streams it may take layer i's own buffer, so it is enqueued
  // after i's write-back (it still starts no earlier than compute(i)).
  auto prefetch = [&](int i) {
    for (int j = 1; j < L; ++j)
      if (load_at[j] == i) load(j, point[i]);
  };
  for (int i = 0; i < L && ok; ++i) {
    ok = ok && cudaEventRecord(point[i], cs) == cudaSuccess;
    if (shared_copy) prefetch(i);
    if (i >= 1) ok = ok && cudaStreamWaitEvent(cs, loaded[i], 0) == cudaSuccess;
    if (!ok) break;
    compute(user, i, buffers[buffer[i]], compute_stream);
    ok = ok && cudaEventRecord(computed[i], cs) == cudaSuccess;
    if (i >= 1) {                   // layer 0 stays in B0
      ok = ok && cudaStreamWaitEvent(ds, computed[i], 0) == cudaSuccess;
      if (wb_bytes)
        ok = ok && cudaMemcpyAsync(static_cast<char*>(host_kv[i]) + wb_offset,
                                   static_cast<char*>(buffers[buffer[i]]) + wb_offset, wb_bytes,
                                   cudaMemcpyDeviceToHost, ds) == cudaSuccess;
      ok = ok && cudaEventRecord(released[i], ds) == cudaSuccess;
    }
    if (!shared_copy) prefetch(i);
  }
  // the compute stream ends after every write-back, so one wait on it covers the pass
  for (int i = 1; i < L && ok; ++i) ok = cudaStreamWaitEvent(cs, released[i], 0) == cudaSuccess;
  destroy();
  return ok ? ESS_OK : ESS_ERR_CUDA;
}
