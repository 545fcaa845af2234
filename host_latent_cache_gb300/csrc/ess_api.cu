// Host side of the C ABI declared in ess.h: workspace layout, argument
// checks, tensor-map encoding and the launch sequences of each entry point.

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "ess_internal.h"
#include "ess_sync.cuh"

namespace ess {
namespace {

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

ess_status check_config(const ess_config* c) {
  if (!c) return ESS_ERR_INVALID_ARG;
  if (c->n_layers < 1 || c->batch < 1 || c->max_T < 1 || c->C < 1 || c->page < 1 || c->k < 1 ||
      c->mtp < 1 || c->idx_heads < 1 || c->idx_dim < 1 || c->mla_heads < 1)
    return ESS_ERR_INVALID_ARG;
  if (c->max_T % c->page != 0) return ESS_ERR_INVALID_ARG;
  if (c->max_T % 4 != 0) return ESS_ERR_UNSUPPORTED;   // 16-byte rows of key scales
  if (!(c->sm_scale > 0.0f)) return ESS_ERR_INVALID_ARG;
  if (c->miss_mode != ESS_MISS_FUSED && c->miss_mode != ESS_MISS_STAGED) return ESS_ERR_INVALID_ARG;
  if (c->idx_dtype != ESS_FP8_E4M3 && c->idx_dtype != ESS_BF16) return ESS_ERR_INVALID_ARG;
  const int esz = c->idx_dtype == ESS_FP8_E4M3 ? 1 : 2;
  if (c->idx_dim * esz != kKeyRowBytes) return ESS_ERR_UNSUPPORTED;
  if (c->mtp > kMaxWays) return ESS_ERR_UNSUPPORTED;
  if (c->mtp * c->idx_heads > 256) return ESS_ERR_UNSUPPORTED;
  if (c->mtp > 1 && c->idx_heads % 32 != 0) return ESS_ERR_UNSUPPORTED;
  if ((c->mtp * c->idx_heads) % 4 != 0) return ESS_ERR_UNSUPPORTED;  // 16-byte weight rows
  if (c->mla_heads > 128) return ESS_ERR_UNSUPPORTED;
  if (c->latent_dim != kLatent || c->rope_dim != kRowDim - kLatent) return ESS_ERR_UNSUPPORTED;
  if (static_cast<long long>(c->mtp) * c->k > kMaxWayK) return ESS_ERR_UNSUPPORTED;
  if (static_cast<long long>(c->batch) * c->max_T > 0x7fffffffLL) return ESS_ERR_UNSUPPORTED;
  // the miss union never exceeds min(M*k, T) rows, so it always fits
  const long long need = std::min<long long>(static_cast<long long>(c->mtp) * c->k, c->max_T);
  if (c->C < need) return ESS_ERR_CAPACITY;
  // every kernel's shared memory must fit one CTA
  if (indexer_smem_need(*c) > kMaxSmemPerCta || select_smem_need(*c) > kMaxSmemPerCta)
    return ESS_ERR_UNSUPPORTED;
  return ESS_OK;
}

Layout compute_layout(const ess_config& c) {
  Layout L;
  const size_t B = c.batch, M = c.mtp, T = c.max_T, C = c.C, k = c.k, H = c.mla_heads,
               HI = c.idx_heads;
  L.nch = (c.k + kAttnRows - 1) / kAttnRows;
  size_t o = 0;
  L.o_T = o;        o = align256(o + B * 4);
  L.o_tiles = o;    o = align256(o + (B + 1) * 4);
  L.o_step = o;     o = align256(o + B * 4);
  L.o_stats = o;    o = align256(o + kStatFields * 8);
  L.o_cslots = o;   o = align256(o + B * T * 4);
  L.o_stoken = o;   o = align256(o + B * C * 4);
  L.o_lused = o;    o = align256(o + B * C * 4);
  L.o_order = o;    o = align256(o + 2 * B * C * 4);
  L.o_pool = o;     o = align256(o + B * C * kRowBytes);
  L.o_T0 = o;       o = align256(o + B * 4);
  L.o_tail = o;     o = align256(o + B * 2 * c.page * kRowBytes);
  L.o_guess = o;    o = align256(o + B * M * 4);
  L.layer_bytes = o;
  o = L.layer_bytes * c.n_layers;
  L.o_scores = o;   o = align256(o + B * M * T * 4);
  L.o_tidx = o;     o = align256(o + B * M * k * 4);
  L.o_tslot = o;    o = align256(o + B * M * k * 4);
  L.o_nmw = o;      o = align256(o + B * M * 4);
  L.o_mtok = o;     o = align256(o + B * M * k * 4);
  L.o_mslot = o;    o = align256(o + B * M * k * 4);
  L.o_nmiss = o;    o = align256(o + B * 4);
  L.o_vict = o;     o = align256(o + B * M * k * 4);
  L.o_hist = o;     o = align256(o + B * M * kHistBins * 4);
  L.o_po = o;       o = align256(o + B * M * L.nch * H * kLatent * 2);
  L.o_pml = o;      o = align256(o + B * M * L.nch * H * 8);
  L.o_hq = o;       o = align256(o + B * M * HI * kKeyRowBytes);
  L.o_hw = o;       o = align256(o + B * M * HI * 4);
  L.o_hqm = o;      o = align256(o + B * M * H * kRowBytes);
  L.o_hout = o;     o = align256(o + B * M * H * kLatent * 4);
  L.o_status = o;   o = align256(o + 256);
  L.o_fhist = o;    o = align256(o + B * M * kFineBins * 4);
  L.o_tflag = o;    o = align256(o + B * M * ((T + 31) / 32) * 4);
  L.o_ready = o;    o = align256(o + B * kCounterStride * 4);
  L.o_adone = o;    o = align256(o + B * M * kCounterStride * 4);
  L.total = o;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool layer_ok(const ess_pool* p, int layer) {
  return p && layer >= 0 && layer < p->cfg.n_layers && p->layers[layer].bound;
}

ess_status cuda_status(cudaError_t e) { return e == cudaSuccess ? ESS_OK : ESS_ERR_CUDA; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

}  // namespace

bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                   uint64_t inner_elems, uint64_t outer_rows, uint64_t row_stride_bytes,
                   uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn || !aligned16(base) || (row_stride_bytes & 15u)) return false;
  cuuint64_t dims[2] = {inner_elems, outer_rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The LRU order list of a layer from host copies of last_used [B][C] and step
// [B]: slots by (last_used, slot), in the list that the next step reads.
cudaError_t write_order(const ess_pool& p, int layer, const std::vector<int32_t>& lu,
                        const std::vector<int32_t>& sp) {
  const ess_config& c = p.cfg;
  const size_t B = c.batch;
  std::vector<int32_t> ord(c.C);
  for (size_t b = 0; b < B; ++b) {
    for (int i = 0; i < c.C; ++i) ord[i] = i;
    const int32_t* l = lu.data() + b * c.C;
    std::sort(ord.begin(), ord.end(), [l](int32_t x, int32_t y) {
      return l[x] != l[y] ? l[x] < l[y] : x < y;
    });
    int32_t* dst = p.layers[layer].order + (static_cast<size_t>(sp[b] & 1) * B + b) * c.C;
    const cudaError_t e = cudaMemcpy(dst, ord.data(), c.C * 4, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_reset(const ess_pool& p, int layer, cudaStream_t st) {
  const ess_config& c = p.cfg;
  const Layer& L = p.layers[layer];
  const size_t B = c.batch;
  cudaError_t e;
  if ((e = cudaMemsetAsync(L.cache_slots, 0xff, B * c.max_T * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(L.slot_token, 0xff, B * c.C * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(L.last_used, 0xff, B * c.C * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(L.step, 0, B * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.scr.ghist, 0, B * c.mtp * kHistBins * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.scr.fhist, 0, B * c.mtp * kFineBins * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(L.guess, 0, B * c.mtp * 4, st)) != cudaSuccess) return e;
  if ((e = launch_order_reset(p, layer, st)) != cudaSuccess) return e;
  return cudaMemsetAsync(L.stats, 0, kStatFields * 8, st);
}

}  // namespace ess

using namespace ess;

extern "C" {

const char* ess_status_string(ess_status s) {
  switch (s) {
    case ESS_OK: return "ok";
    case ESS_ERR_INVALID_ARG: return "invalid argument";
    case ESS_ERR_CAPACITY: return "miss union exceeds the hot pool";
    case ESS_ERR_UNSUPPORTED: return "unsupported shape or value range";
    case ESS_ERR_OOM: return "workspace too small";
    case ESS_ERR_CUDA: return "CUDA error";
    case ESS_ERR_TIMEOUT: return "device wait timed out";
    case ESS_ERR_DEVICE_CHECK: return "device bounds check failed";
  }
  return "unknown status";
}

ess_status ess_host_alloc(size_t bytes, void** out) {
  if (!out || bytes == 0) return ESS_ERR_INVALID_ARG;
  *out = nullptr;
  void* p = nullptr;
  if (cudaHostAlloc(&p, bytes, cudaHostAllocPortable | cudaHostAllocMapped) != cudaSuccess) {
    cudaGetLastError();
    return ESS_ERR_OOM;
  }
  std::memset(p, 0, bytes);
  *out = p;
  return ESS_OK;
}

ess_status ess_host_free(void* ptr) {
  if (!ptr) return ESS_ERR_INVALID_ARG;
  return cudaFreeHost(ptr) == cudaSuccess ? ESS_OK : ESS_ERR_CUDA;
}

ess_status ess_pool_device_bytes(const ess_config* cfg, size_t* bytes) {
  if (!bytes) return ESS_ERR_INVALID_ARG;
  const ess_status s = check_config(cfg);
  if (s != ESS_OK) return s;
  *bytes = compute_layout(*cfg).total;
  return ESS_OK;
}

ess_status ess_pool_create(const ess_config* cfg, void* dev_workspace, size_t ws_bytes,
                           ess_pool** out) {
  if (!out) return ESS_ERR_INVALID_ARG;
  *out = nullptr;
  const ess_status s = check_config(cfg);
  if (s != ESS_OK) return s;
  if (!dev_workspace || (reinterpret_cast<uintptr_t>(dev_workspace) & 255u)) return ESS_ERR_INVALID_ARG;
  const Layout L = compute_layout(*cfg);
  if (ws_bytes < L.total) return ESS_ERR_OOM;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ESS_ERR_CUDA;
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, dev_workspace) != cudaSuccess || pa.type != cudaMemoryTypeDevice)
    return ESS_ERR_INVALID_ARG;
  ess_pool* p = new (std::nothrow) ess_pool;
  if (!p) return ESS_ERR_OOM;
  p->cfg = *cfg;
  p->n_launch = &p->launches;
  p->ws = static_cast<char*>(dev_workspace);
  p->ws_bytes = ws_bytes;
  p->device = dev;
  p->lay = L;
  if (cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    delete p;
    return ESS_ERR_CUDA;
  }
  p->layers = new (std::nothrow) Layer[cfg->n_layers];
  if (!p->layers) {
    delete p;
    return ESS_ERR_OOM;
  }
  for (int l = 0; l < cfg->n_layers; ++l) {
    char* base = p->ws + L.layer_bytes * l;
    Layer& y = p->layers[l];
    y.T_dev = reinterpret_cast<int32_t*>(base + L.o_T);
    y.tile_off = reinterpret_cast<int32_t*>(base + L.o_tiles);
    y.step = reinterpret_cast<int32_t*>(base + L.o_step);
    y.stats = reinterpret_cast<long long*>(base + L.o_stats);
    y.cache_slots = reinterpret_cast<int32_t*>(base + L.o_cslots);
    y.slot_token = reinterpret_cast<int32_t*>(base + L.o_stoken);
    y.last_used = reinterpret_cast<int32_t*>(base + L.o_lused);
    y.order = reinterpret_cast<int32_t*>(base + L.o_order);
    y.pool = reinterpret_cast<uint16_t*>(base + L.o_pool);
    y.T0_dev = reinterpret_cast<int32_t*>(base + L.o_T0);
    y.tail = reinterpret_cast<uint16_t*>(base + L.o_tail);
    y.guess = reinterpret_cast<uint32_t*>(base + L.o_guess);
  }
  Scratch& r = p->scr;
  r.scores = reinterpret_cast<float*>(p->ws + L.o_scores);
  r.topk_idx = reinterpret_cast<int32_t*>(p->ws + L.o_tidx);
  r.topk_slot = reinterpret_cast<int32_t*>(p->ws + L.o_tslot);
  r.n_miss_way = reinterpret_cast<int32_t*>(p->ws + L.o_nmw);
  r.miss_tok = reinterpret_cast<int32_t*>(p->ws + L.o_mtok);
  r.miss_slot = reinterpret_cast<int32_t*>(p->ws + L.o_mslot);
  r.n_miss = reinterpret_cast<int32_t*>(p->ws + L.o_nmiss);
  r.vlist = reinterpret_cast<int32_t*>(p->ws + L.o_vict);
  r.ghist = reinterpret_cast<uint32_t*>(p->ws + L.o_hist);
  r.part_o = reinterpret_cast<uint16_t*>(p->ws + L.o_po);
  r.part_ml = reinterpret_cast<float2*>(p->ws + L.o_pml);
  r.h_qidx = reinterpret_cast<uint8_t*>(p->ws + L.o_hq);
  r.h_w = reinterpret_cast<float*>(p->ws + L.o_hw);
  r.h_qmla = reinterpret_cast<uint16_t*>(p->ws + L.o_hqm);
  r.h_out = reinterpret_cast<float*>(p->ws + L.o_hout);
  r.status = reinterpret_cast<int32_t*>(p->ws + L.o_status);
  r.fhist = reinterpret_cast<uint32_t*>(p->ws + L.o_fhist);
  r.tflag = reinterpret_cast<uint32_t*>(p->ws + L.o_tflag);
  r.ready = reinterpret_cast<int32_t*>(p->ws + L.o_ready);
  r.attn_done = reinterpret_cast<int32_t*>(p->ws + L.o_adone);
  r.nwords = (cfg->max_T + 31) / 32;
  cudaError_t e = cudaSuccess;
  for (int l = 0; l < cfg->n_layers && e == cudaSuccess; ++l) {
    e = launch_reset(*p, l, nullptr);
    if (e == cudaSuccess)
      e = cudaMemset(p->layers[l].pool, 0, static_cast<size_t>(cfg->batch) * cfg->C * kRowBytes);
  }
  if (e == cudaSuccess) e = cudaMemset(r.status, 0, 256);
  if (e == cudaSuccess)
    e = cudaMemset(r.ready, 0, (L.o_adone - L.o_ready) + static_cast<size_t>(cfg->batch) *
                                                           cfg->mtp * kCounterStride * 4);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    delete[] p->layers;
    delete p;
    return ESS_ERR_CUDA;
  }
  *out = p;
  return ESS_OK;
}

ess_status ess_pool_destroy(ess_pool* pool) {
  if (!pool) return ESS_ERR_INVALID_ARG;
  delete[] pool->layers;
  delete pool;
  return ESS_OK;
}

ess_status bind_layer(ess_pool* pool, int layer, const void* host_latent,
                      const int32_t* page_table, const void* idx_keys, const float* idx_scale,
                      const int32_t* T_host, bool compact);

ess_status ess_pool_bind_layer(ess_pool* pool, int layer, const void* host_latent,
                               const int32_t* page_table, const void* idx_keys,
                               const float* idx_scale, const int32_t* T_host) {
  return bind_layer(pool, layer, host_latent, page_table, idx_keys, idx_scale, T_host, false);
}

ess_status ess_pool_bind_layer_compact(ess_pool* pool, int layer, const void* host_compact,
                                       const int32_t* page_table, const void* idx_keys,
                                       const float* idx_scale, const int32_t* T_host) {
  return bind_layer(pool, layer, host_compact, page_table, idx_keys, idx_scale, T_host, true);
}

ess_status bind_layer(ess_pool* pool, int layer, const void* host_latent,
                      const int32_t* page_table, const void* idx_keys, const float* idx_scale,
                      const int32_t* T_host, bool compact) {
  if (!pool || layer < 0 || layer >= pool->cfg.n_layers || !host_latent || !idx_keys || !T_host)
    return ESS_ERR_INVALID_ARG;
  const ess_config& c = pool->cfg;
  if (!aligned16(idx_keys) || !aligned16(host_latent) || (idx_scale && !aligned16(idx_scale)))
    return ESS_ERR_INVALID_ARG;
  void* dev_alias = nullptr;
  if (cudaHostGetDevicePointer(&dev_alias, const_cast<void*>(host_latent), 0) != cudaSuccess) {
    cudaGetLastError();
    return ESS_ERR_INVALID_ARG;  // not pinned / registered host memory
  }
  std::vector<int32_t> tiles(c.batch + 1, 0);
  int tmax = 0;
  for (int b = 0; b < c.batch; ++b) {
    if (T_host[b] < 0 || T_host[b] > c.max_T) return ESS_ERR_INVALID_ARG;
    tiles[b + 1] = tiles[b] + (T_host[b] + kIdxTile - 1) / kIdxTile;
    tmax = T_host[b] > tmax ? T_host[b] : tmax;
  }
  Layer& L = pool->layers[layer];
  if (!encode_map_2d(&L.kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, idx_keys, kKeyRowBytes,
                     static_cast<uint64_t>(c.batch) * c.max_T, kKeyRowBytes, kKeyRowBytes, kIdxTile))
    return ESS_ERR_CUDA;
  if (cudaMemcpy(L.T_dev, T_host, c.batch * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(L.T0_dev, T_host, c.batch * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(L.tile_off, tiles.data(), (c.batch + 1) * 4, cudaMemcpyHostToDevice) != cudaSuccess)
    return ESS_ERR_CUDA;
  L.T0_host.assign(T_host, T_host + c.batch);
  L.n_appended = 0;
  L.host_latent = static_cast<const uint16_t*>(dev_alias);
  L.compact = compact;
  L.page_table = page_table;
  L.idx_keys = static_cast<const uint8_t*>(idx_keys);
  L.idx_scale = idx_scale;
  L.total_tiles = tiles[c.batch];
  L.T_hmax = tmax;
  L.bound = true;
  return ESS_OK;
}

ess_status ess_pool_reset(ess_pool* pool, int layer, ess_stream_t stream) {
  if (!pool || layer < 0 || layer >= pool->cfg.n_layers) return ESS_ERR_INVALID_ARG;
  return cuda_status(launch_reset(*pool, layer, static_cast<cudaStream_t>(stream)));
}

ess_status ess_append(ess_pool* pool, int layer, const void* latent_row, const void* key_row,
                      const float* key_scale, ess_stream_t stream) {
  if (!pool || layer < 0 || layer >= pool->cfg.n_layers || !latent_row || !key_row)
    return ESS_ERR_INVALID_ARG;
  const ess_config& c = pool->cfg;
  Layer& L = pool->layers[layer];
  if (!L.bound || !aligned16(latent_row) || !aligned16(key_row)) return ESS_ERR_INVALID_ARG;
  if (L.idx_scale && !key_scale) return ESS_ERR_INVALID_ARG;
  if (L.compact) return ESS_ERR_UNSUPPORTED;   // pages would have to be encoded on the way out
  const int n = L.n_appended + 1;   // tokens appended after this call
  for (int b = 0; b < c.batch; ++b)
    if (L.T0_host[b] + n > c.max_T) return ESS_ERR_CAPACITY;
  const cudaError_t e = launch_append(*pool, layer, latent_row, key_row, key_scale,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return ESS_ERR_CUDA;
  // the host copies of T_b that size the indexer and selection launches
  int tiles = 0, tmax = 0;
  for (int b = 0; b < c.batch; ++b) {
    const int T = L.T0_host[b] + n;
    tiles += (T + kIdxTile - 1) / kIdxTile;
    tmax = T > tmax ? T : tmax;
  }
  L.n_appended = n;
  L.append_pending = true;
  L.total_tiles = tiles;
  L.T_hmax = tmax;
  return ESS_OK;
}

ess_status ess_indexer_scores(ess_pool* pool, int layer, const void* q_idx, const float* w,
                              float* scores, ess_stream_t stream) {
  if (!layer_ok(pool, layer) || !q_idx || !w || !scores || !aligned16(q_idx) || !aligned16(w))
    return ESS_ERR_INVALID_ARG;
  return cuda_status(launch_indexer(*pool, layer, q_idx, w, scores, false,
                                    static_cast<cudaStream_t>(stream)));
}

ess_status ess_select_manage(ess_pool* pool, int layer, const float* scores, int32_t* topk_idx,
                             int32_t* topk_slot, int32_t* n_miss_way, int32_t* miss_tok,
                             int32_t* miss_slot, int32_t* n_miss, ess_stream_t stream) {
  if (!layer_ok(pool, layer) || !scores || !topk_idx || !topk_slot || !n_miss_way || !miss_tok ||
      !miss_slot || !n_miss || !aligned16(scores))
    return ESS_ERR_INVALID_ARG;
  return cuda_status(launch_select(*pool, layer, scores, false, topk_idx, topk_slot, n_miss_way,
                                   miss_tok, miss_slot, n_miss, static_cast<cudaStream_t>(stream)));
}

ess_status ess_indexer_topk(ess_pool* pool, int layer, const void* q_idx, const float* w,
                            int32_t* topk_idx, int32_t* topk_slot, int32_t* n_miss_way,
                            int32_t* miss_tok, int32_t* miss_slot, int32_t* n_miss,
                            ess_stream_t stream) {
  if (!layer_ok(pool, layer) || !q_idx || !w || !aligned16(q_idx) || !aligned16(w) || !topk_idx ||
      !topk_slot ||
      !n_miss_way || !miss_tok || !miss_slot || !n_miss)
    return ESS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the indexer also fills the score histogram that the selection starts from
  cudaError_t e = launch_indexer(*pool, layer, q_idx, w, pool->scr.scores, true, st);
  if (e != cudaSuccess) return ESS_ERR_CUDA;
  return cuda_status(launch_select(*pool, layer, pool->scr.scores, true, topk_idx, topk_slot,
                                   n_miss_way, miss_tok, miss_slot, n_miss, st));
}

ess_status ess_stage_misses(ess_pool* pool, int layer, const int32_t* miss_tok,
                            const int32_t* miss_slot, const int32_t* n_miss,
                            ess_stream_t stream) {
  if (!layer_ok(pool, layer) || !miss_tok || !miss_slot || !n_miss) return ESS_ERR_INVALID_ARG;
  return cuda_status(
      launch_stage(*pool, layer, miss_tok, miss_slot, n_miss, static_cast<cudaStream_t>(stream)));
}

ess_status ess_sparse_mla_decode(ess_pool* pool, int layer, const void* q_mla,
                                 const int32_t* topk_idx, const int32_t* topk_slot, float* out,
                                 ess_stream_t stream) {
  if (!layer_ok(pool, layer) || !q_mla || !topk_idx || !topk_slot || !out || !aligned16(q_mla) ||
      !aligned16(out))
    return ESS_ERR_INVALID_ARG;
  // the caller's lists may come from anywhere: the kernel waits for all
  // preceding work before it reads them
  return cuda_status(launch_attention(*pool, layer, q_mla, topk_idx, topk_slot, out,
                                      pool->cfg.miss_mode == ESS_MISS_STAGED, false,
                                      static_cast<cudaStream_t>(stream)));
}

ess_status ess_step_profiled(ess_pool* pool, int layer, const void* q_idx, const float* w,
                             const void* q_mla, float* out, ess_stream_t stream,
                             void* const* events) {
  if (!layer_ok(pool, layer) || !q_idx || !w || !q_mla || !out || !aligned16(q_idx) ||
      !aligned16(w) || !aligned16(q_mla) || !aligned16(out))
    return ESS_ERR_INVALID_ARG;
  Scratch& r = pool->scr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto mark = [&](int i) -> bool {
    return !events || !events[i] ||
           cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) == cudaSuccess;
  };
  if (!mark(0)) return ESS_ERR_CUDA;
  if (launch_indexer(*pool, layer, q_idx, w, r.scores, true, st) != cudaSuccess || !mark(1))
    return ESS_ERR_CUDA;
  if (launch_select(*pool, layer, r.scores, true, r.topk_idx, r.topk_slot, r.n_miss_way,
                    r.miss_tok, r.miss_slot, r.n_miss, st) != cudaSuccess)
    return ESS_ERR_CUDA;
  const bool staged = pool->cfg.miss_mode == ESS_MISS_STAGED;
  if (staged && launch_stage(*pool, layer, r.miss_tok, r.miss_slot, r.n_miss, st) != cudaSuccess)
    return ESS_ERR_CUDA;
  if (!mark(2)) return ESS_ERR_CUDA;
  // fused: the kernel just before is the LRU finishing kernel of the selection
  // that wrote the lists, so the attention may start beside it
  if (launch_attention(*pool, layer, q_mla, r.topk_idx, r.topk_slot, out, staged, !staged, st) !=
          cudaSuccess ||
      !mark(3))
    return ESS_ERR_CUDA;
  return ESS_OK;
}

ess_status ess_step(ess_pool* pool, int layer, const void* q_idx, const float* w,
                    const void* q_mla, float* out, ess_stream_t stream) {
  return ess_step_profiled(pool, layer, q_idx, w, q_mla, out, stream, nullptr);
}

ess_status ess_step_host(ess_pool* pool, int layer, const void* q_idx_host, const float* w_host,
                         const void* q_mla_host, float* out_host, ess_stream_t stream) {
  if (!layer_ok(pool, layer) || !q_idx_host || !w_host || !q_mla_host || !out_host)
    return ESS_ERR_INVALID_ARG;
  const ess_config& c = pool->cfg;
  Scratch& r = pool->scr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t BM = static_cast<size_t>(c.batch) * c.mtp;
  // mapped pinned buffers: the GPU reads the inputs and writes the output over
  // the host link itself, inside the step's chain of kernels
  void *dq = nullptr, *dw = nullptr, *dqm = nullptr, *dout = nullptr;
  auto alias = [](const void* h, void** d) {
    return cudaHostGetDevicePointer(d, const_cast<void*>(h), 0) == cudaSuccess;
  };
  if (alias(q_idx_host, &dq) && alias(w_host, &dw) && alias(q_mla_host, &dqm) &&
      alias(out_host, &dout) && aligned16(dq) && aligned16(dw) && aligned16(dqm) &&
      aligned16(dout)) {
    if (launch_inputs_in(*pool, dq, dw, dqm, st) != cudaSuccess) return ESS_ERR_CUDA;
    return ess_step(pool, layer, r.h_qidx, r.h_w, r.h_qmla, static_cast<float*>(dout), stream);
  }
  cudaGetLastError();   // a buffer that is not mapped: copy through the staging
  if (cudaMemcpyAsync(r.h_qidx, q_idx_host, BM * c.idx_heads * kKeyRowBytes,
                      cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(r.h_w, w_host, BM * c.idx_heads * 4, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(r.h_qmla, q_mla_host, BM * c.mla_heads * kRowBytes, cudaMemcpyHostToDevice,
                      st) != cudaSuccess)
    return ESS_ERR_CUDA;
  const ess_status s = ess_step(pool, layer, r.h_qidx, r.h_w, r.h_qmla, r.h_out, stream);
  if (s != ESS_OK) return s;
  if (cudaMemcpyAsync(out_host, r.h_out, BM * c.mla_heads * kLatent * 4, cudaMemcpyDeviceToHost,
                      st) != cudaSuccess)
    return ESS_ERR_CUDA;
  return ESS_OK;
}

ess_status ess_pipeline_step(ess_pool* const* pools, int n_pools, int n_layers,
                             const void* const* q_idx, const float* const* w,
                             const void* const* q_mla, float* const* out,
                             const ess_stream_t* streams) {
  if (!pools || n_pools < 1 || n_layers < 1 || !q_idx || !w || !q_mla || !out || !streams)
    return ESS_ERR_INVALID_ARG;
  for (int i = 0; i < n_pools; ++i)
    if (!pools[i] || pools[i]->cfg.n_layers < n_layers) return ESS_ERR_INVALID_ARG;
  // issue layer by layer, alternating micro-batches, so each stream has work
  // queued while the other one runs
  for (int l = 0; l < n_layers; ++l) {
    for (int i = 0; i < n_pools; ++i) {
      const int x = i * n_layers + l;
      const ess_status s = ess_step(pools[i], l, q_idx[x], w[x], q_mla[x], out[x], streams[i]);
      if (s != ESS_OK) return s;
    }
  }
  return ESS_OK;
}

ess_status ess_pool_get_state(ess_pool* pool, int layer, int32_t* cache_slots,
                              int32_t* slot_token, int32_t* last_used, int32_t* step) {
  if (!pool || layer < 0 || layer >= pool->cfg.n_layers) return ESS_ERR_INVALID_ARG;
  const ess_config& c = pool->cfg;
  const Layer& L = pool->layers[layer];
  const size_t B = c.batch;
  if (cudaDeviceSynchronize() != cudaSuccess) return ESS_ERR_CUDA;
  if (cache_slots && cudaMemcpy(cache_slots, L.cache_slots, B * c.max_T * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return ESS_ERR_CUDA;
  if (slot_token && cudaMemcpy(slot_token, L.slot_token, B * c.C * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return ESS_ERR_CUDA;
  if (last_used && cudaMemcpy(last_used, L.last_used, B * c.C * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return ESS_ERR_CUDA;
  if (step && cudaMemcpy(step, L.step, B * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return ESS_ERR_CUDA;
  return ESS_OK;
}

ess_status ess_pool_set_state(ess_pool* pool, int layer, const int32_t* cache_slots,
                              const int32_t* slot_token, const int32_t* last_used,
                              const int32_t* step) {
  if (!pool || layer < 0 || layer >= pool->cfg.n_layers) return ESS_ERR_INVALID_ARG;
  const ess_config& c = pool->cfg;
  const Layer& L = pool->layers[layer];
  const size_t B = c.batch;
  if (cache_slots) {
    for (size_t i = 0; i < B * c.max_T; ++i)
      if (cache_slots[i] < -1 || cache_slots[i] >= c.C) return ESS_ERR_INVALID_ARG;
  }
  if (slot_token) {
    for (size_t i = 0; i < B * c.C; ++i)
      if (slot_token[i] < -1 || slot_token[i] >= c.max_T) return ESS_ERR_INVALID_ARG;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return ESS_ERR_CUDA;
  // the LRU order list is derived from last_used and step: rebuild it
  std::vector<int32_t> lu(B * c.C), sp(B);
  if (last_used) std::memcpy(lu.data(), last_used, lu.size() * 4);
  else if (cudaMemcpy(lu.data(), L.last_used, lu.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return ESS_ERR_CUDA;
  if (step) std::memcpy(sp.data(), step, sp.size() * 4);
  else if (cudaMemcpy(sp.data(), L.step, sp.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return ESS_ERR_CUDA;
  for (size_t b = 0; b < B; ++b) {
    if (sp[b] < 0) return ESS_ERR_INVALID_ARG;
    for (int i = 0; i < c.C; ++i)
      if (lu[b * c.C + i] < -1 || lu[b * c.C + i] >= sp[b]) return ESS_ERR_INVALID_ARG;
  }
  if (cache_slots && cudaMemcpy(L.cache_slots, cache_slots, B * c.max_T * 4, cudaMemcpyHostToDevice) != cudaSuccess) return ESS_ERR_CUDA;
  if (slot_token && cudaMemcpy(L.slot_token, slot_token, B * c.C * 4, cudaMemcpyHostToDevice) != cudaSuccess) return ESS_ERR_CUDA;
  if (last_used && cudaMemcpy(L.last_used, last_used, B * c.C * 4, cudaMemcpyHostToDevice) != cudaSuccess) return ESS_ERR_CUDA;
  if (step && cudaMemcpy(L.step, step, B * 4, cudaMemcpyHostToDevice) != cudaSuccess) return ESS_ERR_CUDA;
  if (write_order(*pool, layer, lu, sp) != cudaSuccess) return ESS_ERR_CUDA;
  // the rows of the resident tokens come from the authoritative host copy
  if (L.bound) {
    if (launch_refill(*pool, layer, nullptr) != cudaSuccess) return ESS_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return ESS_ERR_CUDA;
  }
  return ESS_OK;
}

ess_status ess_host_gather(const void* host_rows, int64_t n_host_rows, int32_t row_bytes,
                           const int64_t* rows, int64_t n_rows, void* dst, int32_t* bad_row,
                           ess_stream_t stream) {
  if (!host_rows || !dst || n_host_rows < 0 || n_rows < 0 || row_bytes <= 0 || row_bytes % 16 ||
      !aligned16(host_rows) || !aligned16(dst))
    return ESS_ERR_INVALID_ARG;
  if (!rows && n_rows > n_host_rows) return ESS_ERR_INVALID_ARG;
  void* dev_alias = nullptr;
  if (cudaHostGetDevicePointer(&dev_alias, const_cast<void*>(host_rows), 0) != cudaSuccess) {
    cudaGetLastError();
    return ESS_ERR_INVALID_ARG;  // not pinned / mapped host memory
  }
  return cuda_status(launch_host_gather(dev_alias, rows, n_rows, n_host_rows, row_bytes, dst,
                                        bad_row, static_cast<cudaStream_t>(stream)));
}

ess_status ess_pool_set_eviction(ess_pool* pool, int32_t policy, uint64_t seed) {
  if (!pool || policy < ESS_EVICT_LRU || policy > ESS_EVICT_LIM) return ESS_ERR_INVALID_ARG;
  const ess_config& c = pool->cfg;
  if (policy == ESS_EVICT_LRU && pool->evict_policy != ESS_EVICT_LRU) {
    // the LRU list was not kept under the other order: rebuild it from the stamps
    if (cudaDeviceSynchronize() != cudaSuccess) return ESS_ERR_CUDA;
    std::vector<int32_t> lu(static_cast<size_t>(c.batch) * c.C), sp(c.batch);
    for (int l = 0; l < c.n_layers; ++l) {
      const Layer& L = pool->layers[l];
      if (cudaMemcpy(lu.data(), L.last_used, lu.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
          cudaMemcpy(sp.data(), L.step, sp.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
          write_order(*pool, l, lu, sp) != cudaSuccess)
        return ESS_ERR_CUDA;
    }
  }
  pool->evict_policy = policy;
  pool->evict_seed = seed;
  return ESS_OK;
}

ess_status ess_pool_get_rows(ess_pool* pool, int layer, void* rows_host) {
  if (!pool || !rows_host || layer < 0 || layer >= pool->cfg.n_layers) return ESS_ERR_INVALID_ARG;
  const ess_config& c = pool->cfg;
  if (cudaDeviceSynchronize() != cudaSuccess) return ESS_ERR_CUDA;
  const size_t n = static_cast<size_t>(c.batch) * c.C * kRowBytes;
  return cuda_status(cudaMemcpy(rows_host, pool->layers[layer].pool, n, cudaMemcpyDeviceToHost));
}

ess_status ess_pool_kernel_launches(const ess_pool* pool, int64_t* count) {
  if (!pool || !count) return ESS_ERR_INVALID_ARG;
  *count = pool->launches;
  return ESS_OK;
}

ess_status ess_pool_read_stats(ess_pool* pool, int layer, ess_stats* out, int reset) {
  if (!pool || !out || layer < 0 || layer >= pool->cfg.n_layers) return ESS_ERR_INVALID_ARG;
  long long v[kStatFields];
  const Layer& L = pool->layers[layer];
  if (cudaDeviceSynchronize() != cudaSuccess) return ESS_ERR_CUDA;
  if (cudaMemcpy(v, L.stats, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return ESS_ERR_CUDA;
  out->steps = v[0];
  out->hits = v[1];
  out->misses = v[2];
  out->union_size = v[3];
  out->miss_rows = v[4];
  out->miss_bytes = v[5];
  out->guided = v[6];
  out->fine_cuts = v[7];
  if (reset && cudaMemset(L.stats, 0, sizeof(v)) != cudaSuccess) return ESS_ERR_CUDA;
  return ESS_OK;
}

ess_status ess_pool_poll(ess_pool* pool, ess_stream_t stream) {
  if (!pool) return ESS_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ESS_ERR_CUDA;
  int32_t st = 0;
  if (cudaMemcpy(&st, pool->scr.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return ESS_ERR_CUDA;
  if (st != 0 && cudaMemset(pool->scr.status, 0, 4) != cudaSuccess) return ESS_ERR_CUDA;
  return static_cast<ess_status>(st);
}

}  // extern "C"
