// Decode append: the newest token of every request joins the layer.
//
// hwcomputing.csdn.net FlashOffloading analysis, section "architecture: one
// master copy, two residency policies" and its Figure 2: on the decode side
// the device keeps the model's own indexer state, the hot cache of C slots,
// the cache_slots table and two tail blocks that take the newly produced KV;
// the authoritative KV lives in host memory, paged by (request, layer, token
// block) behind a block table.
//
// The page names the parts but not the steps; the reading taken here:
//   - token t of request b is written to row t mod (2 * page) of the
//     request's two-page device ring, and its indexer key (and scale) to row
//     t of the layer's indexer cache, so the next indexer pass scores it;
//   - when t completes a page, the appended rows of that page are written
//     back to their host rows through the block table;
//   - a ring row is overwritten by token t + 2 * page, so rows of the newest
//     two pages (tokens >= page * floor(T_b / page) - page) are read from the
//     ring and older ones from the host copy;
//   - cache_slots stays -1 for a new token: it is not in the hot cache, and a
//     step that selects it loads it into a slot like any other miss (from the
//     ring while it is there).
#include "ess_device.cuh"

namespace ess {
namespace {

struct AppendArgs {
  const uint16_t* latent;     // [B][D] bf16: the new rows
  const uint8_t* key;         // [B][128 bytes]: the new indexer key rows
  const float* key_scale;     // [B], used when the layer has per-token scales
  uint8_t* idx_keys;          // [B][T][128 bytes]
  float* idx_scale;           // [B][T] or null
  uint16_t* tail;             // [B][2 * page][D]
  uint16_t* host;             // [B][T][D] device alias of the pinned host rows
  const int32_t* page_table;  // [B][T / page] or null
  int32_t* Tb;                // [B]
  const int32_t* T0;          // [B] T_b at the bind
  int32_t* tile_off;          // [B+1] prefix of indexer tiles
  int* status;
  int T, page, npages;
  int n_before;               // tokens appended to every request before this call
};

constexpr int kAppendThreads = 256;
constexpr int kRowVec = kRowBytes / 16;      // 72 16-byte units per latent row
constexpr int kKeyVec = kKeyRowBytes / 16;   // 8 per key row

// One CTA per request, launched as a programmatic dependent.  Its own
// dependents may start at once: every kernel of the library waits for this
// grid to finish (griddepcontrol.wait) before it reads T_b, the keys or the
// ring.
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const AppendArgs a) {
  pdl_wait_previous();   // the previous step still reads T_b, the ring and the keys
  pdl_launch_dependents();
  const int b = blockIdx.x, tid = threadIdx.x;
  const int t = a.T0[b] + a.n_before;
  const bool bad = t < 0 || t >= a.T || a.Tb[b] != t;
  __syncthreads();       // every thread has read T_b before it changes below
  if (bad) {
    if (tid == 0) set_status(a.status, ESS_ERR_DEVICE_CHECK);
    return;
  }
  const int ring = 2 * a.page;
  uint16_t* trow = a.tail + (static_cast<size_t>(b) * ring + t % ring) * kRowDim;
  if (tid < kRowVec) {
    reinterpret_cast<uint4*>(trow)[tid] =
        reinterpret_cast<const uint4*>(a.latent + static_cast<size_t>(b) * kRowDim)[tid];
  } else if (tid >= 128 && tid < 128 + kKeyVec) {
    const int q = tid - 128;
    reinterpret_cast<uint4*>(a.idx_keys + (static_cast<size_t>(b) * a.T + t) * kKeyRowBytes)[q] =
        reinterpret_cast<const uint4*>(a.key + static_cast<size_t>(b) * kKeyRowBytes)[q];
  } else if (tid == 160) {
    if (a.idx_scale) a.idx_scale[static_cast<size_t>(b) * a.T + t] = a.key_scale[b];
  } else if (tid == 192) {
    // T_b and this request's end of the tile prefix; every request grows by
    // one token, so the prefix follows from the bind-time lengths
    a.Tb[b] = t + 1;
    int tiles = 0;
    for (int i = 0; i <= b; ++i) tiles += (a.T0[i] + a.n_before + 1 + kIdxTile - 1) / kIdxTile;
    a.tile_off[b + 1] = tiles;
  }
  if ((t + 1) % a.page != 0) return;

  // t completes its page: copy the page's appended rows to the host copy
  __syncthreads();       // the new row is in the ring
  const int pg = t / a.page;
  int hrow0 = pg * a.page;
  if (a.page_table) {
    const int pp = a.page_table[static_cast<size_t>(b) * a.npages + pg];
    if (pp < 0 || pp >= a.npages) {
      if (tid == 0) set_status(a.status, ESS_ERR_DEVICE_CHECK);
      return;
    }
    hrow0 = pp * a.page;
  }
  const int first = a.T0[b] > pg * a.page ? a.T0[b] : pg * a.page;   // first appended token
  const int n = (t + 1 - first) * kRowVec;
  for (int i = tid; i < n; i += kAppendThreads) {
    const int tok = first + i / kRowVec, q = i % kRowVec;
    const uint4 v =
        reinterpret_cast<const uint4*>(a.tail + (static_cast<size_t>(b) * ring + tok % ring) * kRowDim)[q];
    reinterpret_cast<uint4*>(a.host + (static_cast<size_t>(b) * a.T + hrow0 + tok % a.page) * kRowDim)[q] = v;
  }
}

}  // namespace

cudaError_t launch_append(const ess_pool& p, int layer, const void* latent, const void* key,
                          const float* key_scale, cudaStream_t st) {
  const ess_config& c = p.cfg;
  const Layer& L = p.layers[layer];
  AppendArgs a;
  a.latent = static_cast<const uint16_t*>(latent);
  a.key = static_cast<const uint8_t*>(key);
  a.key_scale = key_scale;
  // the caller's indexer cache and host copy grow with the context: the
  // binding hands them over for these writes
  a.idx_keys = const_cast<uint8_t*>(L.idx_keys);
  a.idx_scale = const_cast<float*>(L.idx_scale);
  a.tail = L.tail;
  a.host = const_cast<uint16_t*>(L.host_latent);
  a.page_table = L.page_table;
  a.Tb = L.T_dev;
  a.T0 = L.T0_dev;
  a.tile_off = L.tile_off;
  a.status = p.scr.status;
  a.T = c.max_T;
  a.page = c.page;
  a.npages = c.max_T / c.page;
  a.n_before = L.n_appended;
  const cudaError_t e = launch_pdl(append_kernel, dim3(c.batch), dim3(kAppendThreads), 0, st, a);
  if (e == cudaSuccess) count_launch(p);
  return e;
}

// ---------------------------------------------------------------------------
// Step inputs straight from mapped pinned host memory: three segments of
// 16-byte units (indexer queries, head weights, MLA queries) copied into the
// pool's staging by the GPU's own threads.  The host reads are issued before
// the wait for the previous grid (nothing on the device writes the caller's
// host inputs), so they overlap that grid's tail; the staging is written
// after it (the previous step's attention reads the staged MLA queries).
namespace {

struct InSeg {
  const uint4* src;
  uint4* dst;
  long long n;   // 16-byte units
};

constexpr int kInPerThread = 2;

__global__ void __launch_bounds__(256) inputs_in_kernel(const InSeg s0, const InSeg s1,
                                                        const InSeg s2) {
  // The indexer after this kernel may launch at once: it loads its first key
  // tiles beside the previous step's last kernel, as it does without this one,
  // and waits for this grid (and so for that kernel) before it reads a query.
  pdl_launch_dependents();
  const long long i0 =
      (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * kInPerThread;
  uint4 v[kInPerThread];
  uint4* d[kInPerThread];
#pragma unroll
  for (int u = 0; u < kInPerThread; ++u) {
    long long i = i0 + u;
    d[u] = nullptr;
    if (i < s0.n) {
      v[u] = s0.src[i];
      d[u] = s0.dst + i;
    } else if ((i -= s0.n) < s1.n) {
      v[u] = s1.src[i];
      d[u] = s1.dst + i;
    } else if ((i -= s1.n) < s2.n) {
      v[u] = s2.src[i];
      d[u] = s2.dst + i;
    }
  }
  pdl_wait_previous();
#pragma unroll
  for (int u = 0; u < kInPerThread; ++u)
    if (d[u]) *d[u] = v[u];
}

}  // namespace

cudaError_t launch_inputs_in(const ess_pool& p, const void* q_idx_dev, const void* w_dev,
                             const void* q_mla_dev, cudaStream_t st) {
  const ess_config& c = p.cfg;
  const long long BM = static_cast<long long>(c.batch) * c.mtp;
  InSeg s0{static_cast<const uint4*>(q_idx_dev), reinterpret_cast<uint4*>(p.scr.h_qidx),
           BM * c.idx_heads * kKeyRowBytes / 16};
  InSeg s1{static_cast<const uint4*>(w_dev), reinterpret_cast<uint4*>(p.scr.h_w),
           BM * c.idx_heads * 4 / 16};
  InSeg s2{static_cast<const uint4*>(q_mla_dev), reinterpret_cast<uint4*>(p.scr.h_qmla),
           BM * c.mla_heads * kRowBytes / 16};
  const long long n = s0.n + s1.n + s2.n;
  const long long per_cta = 256LL * kInPerThread;
  const cudaError_t e =
      launch_pdl(inputs_in_kernel, dim3(static_cast<unsigned>((n + per_cta - 1) / per_cta)),
                 dim3(256), 0, st, s0, s1, s2);
  if (e == cudaSuccess) count_launch(p);
  return e;
}

}  // namespace ess
