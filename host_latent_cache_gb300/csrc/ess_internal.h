// Internal declarations shared by the host API and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "ess.h"

namespace ess {

constexpr int kRowDim = 576;          // D = 512 latent + 64 RoPE (bf16)
constexpr int kRowBytes = kRowDim * 2;
constexpr int kLatent = 512;
constexpr int kMaxWays = 4;
constexpr int kMaxWayK = 8192;        // M * k cap of the selection lists
constexpr int kKeyRowBytes = 128;     // one indexer key row

constexpr int kIdxThreads = 320;      // 10 warps: TMA, MMA, 2 groups of 4 epilogue warps
constexpr int kHistBins = 4096;       // score histogram on the top 12 bits of the ordered key
// Guided selection: the indexer also flags every token whose key lies at or
// above a guessed coarse bin g (the previous step's threshold bin less one)
// and counts the keys of bins g .. g + kFineWin - 1 on 8 more bits.
constexpr int kFineWin = 4;           // coarse bins covered by the fine histogram
constexpr int kFineSub = 256;         // fine bins per coarse bin
constexpr int kFineBins = kFineWin * kFineSub;
// key-tile ring: as many 16 KB stages as fit one CTA, up to kIdxMaxStages
#ifndef ESS_IDX_MAX_STAGES
#define ESS_IDX_MAX_STAGES 6
#endif
constexpr int kIdxMaxStages = ESS_IDX_MAX_STAGES;
constexpr int kIdxMinStages = 2;
// tiles per chunk: the indexer's barrier rounds move up to this many 128-token
// tiles (three: three 48 KB ring stages fit beside the rest, where four-tile
// chunks leave room for two 64 KB stages only)
#ifndef ESS_IDX_SUB
#define ESS_IDX_SUB 3
#endif
constexpr int kIdxSubMax = ESS_IDX_SUB;
constexpr int kIdxTile = 128;         // tokens per tile (MMA M)

constexpr int kSelCluster = 8;        // CTAs per request in the selection kernel
constexpr int kSelThreads = 512;

constexpr int kAttnRows = 128;        // selected rows per attention CTA
constexpr int kAttnThreads = 128;
constexpr int kAttnQStages = 4;

constexpr int kStatFields = 8;        // ess_stats fields kept on the device

// Bindings and state of one layer (device pointers point into the workspace
// or at caller buffers).
struct Layer {
  bool bound = false;
  const uint16_t* host_latent = nullptr;  // device-accessible alias of the pinned host rows
  bool compact = false;           // host rows are compact 656-byte rows (no appends)
  const int32_t* page_table = nullptr;
  const uint8_t* idx_keys = nullptr;
  const float* idx_scale = nullptr;
  int32_t* T_dev = nullptr;       // [B]
  int32_t* tile_off = nullptr;    // [B+1] prefix of indexer tiles
  int32_t total_tiles = 0;
  int32_t T_hmax = 0;             // max over requests of T_b
  // decode append: tokens t >= T0_b were appended after the bind; the two
  // newest pages of them sit in a device ring until the host copy takes over
  int32_t* T0_dev = nullptr;      // [B] T_b at the bind
  uint16_t* tail = nullptr;       // [B][2 * page][D] bf16, token t at row t % (2 * page)
  std::vector<int32_t> T0_host;   // host copy of T0_dev
  int32_t n_appended = 0;         // tokens appended to every request since the bind
  // an append kernel was launched after the last indexer launch: the next
  // indexer must wait for it before reading tile prefixes or key rows
  mutable bool append_pending = false;
  CUtensorMap kmap;               // keys as [B*T rows][128 B], 128x128 boxes, 128B swizzle
  // state
  int32_t* cache_slots = nullptr; // [B][T]
  int32_t* slot_token = nullptr;  // [B][C]
  int32_t* last_used = nullptr;   // [B][C]
  int32_t* step = nullptr;        // [B]
  int32_t* order = nullptr;       // [2][B][C] slots in (last_used, slot) order, by step parity
  uint32_t* guess = nullptr;      // [B][M] coarse bin the next indexer flags from (0: none)
  uint16_t* pool = nullptr;       // [B][C][D] bf16
  long long* stats = nullptr;     // [kStatFields]
};

struct Scratch {
  float* scores = nullptr;        // [B][M][T]
  int32_t* topk_idx = nullptr;    // [B][M][k]
  int32_t* topk_slot = nullptr;   // [B][M][k]
  int32_t* n_miss_way = nullptr;  // [B][M]
  int32_t* miss_tok = nullptr;    // [B][M*k]
  int32_t* miss_slot = nullptr;   // [B][M*k]
  int32_t* n_miss = nullptr;      // [B]
  int32_t* vlist = nullptr;       // [B][M*k] victims in LRU order
  uint32_t* ghist = nullptr;      // [B][M][kHistBins] score histogram
  uint32_t* fhist = nullptr;      // [B][M][kFineBins] fine histogram over the guessed window
  uint32_t* tflag = nullptr;      // [B][M][nwords] bit t % 32 of word t / 32: key >= guess
  int nwords = 0;                 // flag words per (request, way): ceil(max_T / 32)
  uint16_t* part_o = nullptr;     // [B][M][nch][H][512] fp16, 16-byte units XOR-swizzled by head
  float2* part_ml = nullptr;      // [B][M][nch][H]
  uint8_t* h_qidx = nullptr;      // staging for ess_step_host
  float* h_w = nullptr;
  uint16_t* h_qmla = nullptr;
  float* h_out = nullptr;
  int32_t* status = nullptr;      // device status word
  // completion counters, one 128-byte line apart, zeroed by the first
  // selection CTA of their request: [B] selection CTAs (or the victim CTA,
  // counting for all of them) done writing request b's lists; [B][M]
  // attention CTAs done writing the partials of (request b, way m)
  int32_t* ready = nullptr;
  int32_t* attn_done = nullptr;
};

// Workspace layout computed from a config (offsets in bytes).
struct Layout {
  size_t total = 0;
  size_t layer_bytes = 0;
  // per layer (relative to the layer base)
  size_t o_T, o_tiles, o_cslots, o_stoken, o_lused, o_step, o_pool, o_stats, o_order, o_T0,
      o_tail, o_guess;
  // scratch (absolute)
  size_t o_scores, o_tidx, o_tslot, o_nmw, o_mtok, o_mslot, o_nmiss, o_vict, o_hist, o_po, o_pml,
      o_hq, o_hw, o_hqm, o_hout, o_status, o_fhist, o_tflag, o_ready, o_adone;
  int nch = 0;                    // attention chunks per (request, way)
};

}  // namespace ess

struct ess_pool {
  ess_config cfg;
  char* ws = nullptr;
  size_t ws_bytes = 0;
  int device = 0;
  int num_sms = 0;
  ess::Layout lay;
  ess::Layer* layers = nullptr;
  ess::Scratch scr;
  int32_t evict_policy = ESS_EVICT_LRU;  // victim order of the decode kernels
  unsigned long long evict_seed = 0;     // key of the Random order
  long long launches = 0;          // kernels launched by this pool's calls
  long long* n_launch = nullptr;   // -> launches (copies of the handle count into it)
};

namespace ess {

inline void count_launch(const ess_pool& p) {
  if (p.n_launch) ++*p.n_launch;
}

// Every kernel asks for the largest shared-memory carveout, even one that
// uses little shared memory: the carveout an SM is given for one kernel's CTAs
// decides whether a programmatic dependent with a large footprint (the
// attention kernel beside the LRU finishing kernel, the indexer beside the
// merge kernel) can be resident on that SM at the same time.
template <typename... KArgs>
cudaError_t prefer_max_smem(void (*kernel)(KArgs...)) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              static_cast<int>(cudaSharedmemCarveoutMaxShared));
}

// Launches a kernel as a programmatic dependent of the previous kernel on the
// stream: its CTAs may be scheduled before that kernel has finished, so every
// kernel of this library waits (griddepcontrol.wait) before it touches global
// memory, and lets its own dependents launch once it is running.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = prefer_max_smem(kernel);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Largest shared memory one CTA of a kernel asks for under a config, and the
// per-CTA limit of this architecture (227 KiB).  Configs above it are refused
// when validated, instead of failing at launch.
constexpr size_t kMaxSmemPerCta = 232448;
size_t indexer_smem_need(const ess_config& c);
size_t select_smem_need(const ess_config& c);

// Kernel launchers (one per kernel file).  They assume validated arguments.
// with_hist: also accumulate the per-(request, way) score histogram in the
// pool's scratch (it must be zero; the selection kernel zeroes it after use).
cudaError_t launch_indexer(const ess_pool& p, int layer, const void* q_idx, const float* w,
                           float* scores, bool with_hist, cudaStream_t st);
// Two kernels: the selection proper (lists, miss union, victims) and the LRU
// finishing kernel (state rewrite, next LRU list, step counter).
// hist_given: the indexer filled the histogram; otherwise the kernel builds it.
cudaError_t launch_select(const ess_pool& p, int layer, const float* scores, bool hist_given,
                          int32_t* topk_idx, int32_t* topk_slot, int32_t* n_miss_way,
                          int32_t* miss_tok, int32_t* miss_slot, int32_t* n_miss, cudaStream_t st);
cudaError_t launch_order_reset(const ess_pool& p, int layer, cudaStream_t st);
cudaError_t launch_stage(const ess_pool& p, int layer, const int32_t* miss_tok,
                         const int32_t* miss_slot, const int32_t* n_miss, cudaStream_t st);
// early: the kernel launched just before on st is the LRU finishing kernel
// of the selection that wrote topk_idx / topk_slot (see AttnArgs::early)
cudaError_t launch_attention(const ess_pool& p, int layer, const void* q_mla,
                             const int32_t* topk_idx, const int32_t* topk_slot, float* out,
                             bool misses_staged, bool early, cudaStream_t st);
cudaError_t launch_reset(const ess_pool& p, int layer, cudaStream_t st);
// rows of a device-mapped pinned host array -> dst (rows NULL: rows 0..n-1);
// a row index outside [0, n_host_rows) sets *status (when given) to 1
cudaError_t launch_host_gather(const void* host_dev, const int64_t* rows, int64_t n_rows,
                               int64_t n_host_rows, int row_bytes, void* dst, int* status,
                               cudaStream_t st);
// the step inputs of ess_step_host from device aliases of mapped pinned host
// buffers into the pool's staging (one kernel, a programmatic dependent)
cudaError_t launch_inputs_in(const ess_pool& p, const void* q_idx_dev, const void* w_dev,
                             const void* q_mla_dev, cudaStream_t st);
// reload the pool rows of every resident token from the host copy
cudaError_t launch_refill(const ess_pool& p, int layer, cudaStream_t st);
cudaError_t launch_append(const ess_pool& p, int layer, const void* latent, const void* key,
                          const float* key_scale, cudaStream_t st);

// Encodes a 2-D tiled tensor map; returns false on failure.
bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                   uint64_t inner_elems, uint64_t outer_rows, uint64_t row_stride_bytes,
                   uint32_t box_inner, uint32_t box_rows);

}  // namespace ess
