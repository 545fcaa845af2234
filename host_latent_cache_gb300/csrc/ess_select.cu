// (a2)-(a4), (a8): exact top-k, hit/miss resolution against cache_slots,
// the miss union over the MTP ways, LRU victim choice and the state rewrite.
//
// hwcomputing.csdn.net FlashOffloading analysis, section "decode side (1)":
//  - cache_slots is a per-request, per-layer int32 token->slot vector with
//    -1 for "not resident", so a lookup is O(1) and management costs
//    O(k) + O(|Miss|) instead of a scan of the hot cache;
//  - five steps per layer and step: (1) look up every way's top-k,
//    (2) union of the misses over the ways, (3) take the union of the top-k
//    out of C_b and pick as many victims as misses, (4) pair each miss with
//    a victim and rewrite cache_slots, (5) copy the misses into the paired
//    slots; loads equal evictions so |C_b| never changes;
//  - LIM emits the top-k slot list and copy triples (DRAM source, HBM
//    destination, count) and puts the misses at the head of the list.
// "ESS: Latent-Cache Offload": the GPU sparse pool keeps its hot subset
// under LRU.
//
// One cluster of kSelCluster CTAs handles one request; CTA r owns tokens
// [r*n_local, (r+1)*n_local) and positions/slots [r*c_local, (r+1)*c_local).
//
// Top-k: a histogram of the top 12 bits of the order-preserving score keys
// (filled by the indexer, or built here for caller scores) gives the bin
// that holds the k-th largest score.  One ordered pass lists the tokens
// above that bin (selected) and in it (candidates).  When the indexer has
// flagged the tokens at or above the previous step's cut less one bin and
// the cut has not fallen below that bin, the pass reads only the flagged
// tokens, and when the cut's bin is one of the four the indexer's fine
// histogram covers, the candidates are those of one 4096-wide fine bin.
// The candidates' keys are gathered through distributed shared memory into
// every CTA and ranked one against another (up to 128) or by MSB radix
// passes over their low 20 bits, which fix the exact threshold; equal keys
// go to the lowest token.  If a CTA's list could overflow, the kernel falls
// back to radix passes over every token.  Every path gives the same exact
// result; all lists come out in ascending token order.
//
// LRU: the slots are kept in a list sorted by (last_used, slot), double
// buffered by step parity.  After the hits are stamped, the unstamped
// entries in list order are exactly the eviction order, so the first
// |Miss| of them are the victims, already in the order that pairs the i-th
// miss with the i-th victim; the next list is the remaining unstamped
// entries followed by the stamped slots in slot order.  The stamps of the
// step are also set in a bitmap over the slots, kept in distributed shared
// memory (CTA r holds the words of its slot range and every CTA ORs its
// hits into them), which each CTA copies whole to look its list entries up.
//
// Two kernels share this work: select_kernel produces everything the step
// reads (the emitted lists, the miss union and its victims), and
// lru_finish_kernel, which only the next step depends on, rewrites the state
// and closes the next LRU list while the attention kernel runs.  Each
// select_kernel CTA counts itself in a per-request counter once its share of
// the lists is written, so a step's attention CTAs start on their own
// request's lists without waiting for the slowest request.
#include <algorithm>
#include <mutex>

#include "ess_device.cuh"
#include "ess_sync.cuh"

namespace ess {
namespace {

constexpr int CL = kSelCluster;
constexpr int NT = kSelThreads;
constexpr int NW = NT / 32;


constexpr int kDigBits = 10;               // radix digit width of the exact passes
constexpr int kDig = 1 << kDigBits;
constexpr int kDirectRank = 128;           // gathered candidates ranked one against another

struct SelArgs {
  const float* scores;        // [B][M][T]
  uint32_t* ghist;            // [B][M][kHistBins]
  int hist_given;             // 1: filled by the indexer; 0: build it here
  // guided selection (with the indexer's histogram only): the coarse bin the
  // indexer flagged from per (request, way), rewritten here for the next step;
  // the indexer's fine histogram and flag bitmap
  uint32_t* guess;            // [B][M] or null
  uint32_t* fhist;            // [B][M][kFineBins]
  const uint32_t* tflag;      // [B][M][nwords]
  int nwords;
  int32_t* cache_slots;       // [B][T]
  int32_t* slot_token;        // [B][C]
  int32_t* last_used;         // [B][C]
  int32_t* step;              // [B]
  int32_t* order;             // [2][B][C]
  const int32_t* Tb;          // [B]
  int32_t* topk_idx;          // [B][M][k]
  int32_t* topk_slot;         // [B][M][k]
  int32_t* n_miss_way;        // [B][M]
  int32_t* miss_tok;          // [B][M*k]
  int32_t* miss_slot;         // [B][M*k]
  int32_t* n_miss;            // [B]
  int32_t* vlist;             // [B][M*k] victims in LRU order
  long long* stats;           // [kStatFields]
  int* status;
  int B, M, k, T, C;
  int policy;                 // ESS_EVICT_*: LRU keeps the order list; the others
                              // leave the victims to victim_kernel
  unsigned long long seed;    // key of the Random victim order
  // [B] counters or null: request b's lists are complete once its counter
  // reaches kSelCluster (each selection CTA adds 1 under LRU; the victim CTA
  // adds kSelCluster); [B][M] counters of the attention kernel's chunk CTAs.
  // Both are zeroed by the request's first CTA.
  int* ready;
  int* attn_done;
  // the layer's host rows, so that each miss's address translation starts
  // while the selection still runs (a prefetch; nothing waits for it)
  const uint8_t* host;        // device alias of the pinned host rows
  const int32_t* page_table;  // [B][T/page] or null
  const int32_t* T0;          // [B] rows t >= T0_b may still sit in the device ring
  int page, row_bytes;
  int n_local;                // tokens per CTA (multiple of 4)
  int c_local;                // slots / order positions per CTA
  int resident;               // scores staged in shared memory
  int lcap;                   // token-list capacity per CTA
  int gcap;                   // gathered-candidate capacity per CTA
  uint32_t keys_bytes;        // size of the staged-scores region
};

struct SelShared {
  uint32_t hist[2][kMaxWays * kDig];
  uint32_t tot[kMaxWays * kDig];
  int scanbuf[2][NW];
  int wcount[NW];
  uint32_t prefix[kMaxWays], selmask[kMaxWays];
  int remaining[kMaxWays], eq_local[kMaxWays], eq_before[kMaxWays], eq_total[kMaxWays];
  int active[kMaxWays], quota[kMaxWays], rank_needed[kMaxWays];
  int last_lo, last_dmask;
  int b1[kMaxWays], take1[kMaxWays], cand1[kMaxWays];  // coarse threshold bin per way
  uint32_t g[kMaxWays];               // guessed coarse bin the indexer flagged from (0: none)
  int fine[kMaxWays], fb[kMaxWays];   // the cut's fine bin within b1, when the fine histogram has it
  int fallback;
  int nl;
  int ncand[kMaxWays];                // this CTA's candidates per way (read through DSMEM)
  int gcnt[kMaxWays][CL];             // every CTA's candidate count per way (read once)
  int gsel;                           // 1: candidates are gathered into every CTA
  // published for the other CTAs of the cluster (read through DSMEM)
  int pub_overflow, pub_nmiss, pub_nu, pub_hit[kMaxWays], pub_miss[kMaxWays], pub_unst;
  // cluster-wide values derived from the publications
  int n_miss_total, nu_total, miss_off, hit_off[kMaxWays], wmiss_off[kMaxWays], nmw[kMaxWays];
  int hits_total[kMaxWays];
  int unst_before, unst_total;
  int ndefer;                         // misses whose slot waits for the victims
  int step_b;
  unsigned long long bar;
};

__device__ __forceinline__ void hist_add_warp(uint32_t* h, uint32_t bin, bool ok) {
  const unsigned act = __ballot_sync(0xffffffffu, ok);
  if (ok) {
    const unsigned peers = __match_any_sync(act, bin);
    if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(peers) - 1))
      atomicAdd(&h[bin], static_cast<uint32_t>(__popc(peers)));
  }
}

// Exclusive block-wide prefix of v (512 threads); total returned through tot.
// The scratch is double-buffered so one __syncthreads per call suffices.
__device__ __forceinline__ int block_scan(int v, int& tot, SelShared& sh, int& parity) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  int* buf = sh.scanbuf[parity];
  parity ^= 1;
  if (lane == 31) buf[warp] = x;
  __syncthreads();
  int pre = 0, t = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const int u = buf[i];
    pre += (i < warp) ? u : 0;
    t += u;
  }
  tot = t;
  return pre + x - v;
}

// Ordered positions for a block-wide compaction (same `run` in every thread).
__device__ __forceinline__ int ordered_pos(int v, int& run, SelShared& sh, int& parity) {
  int tot;
  const int p = run + block_scan(v, tot, sh, parity);
  run += tot;
  return p;
}

// Exclusive prefix of per-warp counts (one __syncthreads; callers keep the
// wcount buffer free until every thread has passed the next barrier).
__device__ __forceinline__ int warp_base(int wcnt, int& total, SelShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) sh.wcount[warp] = wcnt;
  __syncthreads();
  int pre = 0, t = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const int u = sh.wcount[i];
    pre += (i < warp) ? u : 0;
    t += u;
  }
  total = t;
  return pre;
}

// Sum of a shared-memory word over the CTAs of the cluster (and over ranks
// below upto_rank).
__device__ __forceinline__ uint32_t sum_over_cluster(const void* local, uint32_t upto_rank,
                                                     uint32_t* before) {
  const uint32_t a = smem_u32(local);
  uint32_t v[CL];
#pragma unroll
  for (uint32_t r = 0; r < CL; ++r) v[r] = ld_dsmem_u32(dsmem_addr(a, r));
  uint32_t s = 0, b = 0;
#pragma unroll
  for (uint32_t r = 0; r < CL; ++r) {
    if (r < upto_rank) b += v[r];
    s += v[r];
  }
  if (before) *before = b;
  return s;
}

// Cluster-wide exact selection of the remaining[m] largest keys (keys <
// 2^nbits) per active way over the elements for which keyf(m, i, key) is
// true; elements of rank r precede those of rank r+1, and equal keys go to
// the lowest element.  MSB-first passes of kDigBits-bit digits; per-CTA
// histograms are summed through distributed shared memory.  Leaves prefix[m]
// (threshold key), remaining[m] (how many threshold-equal elements to take,
// lowest first) and eq_local / eq_before / eq_total of threshold-equal
// elements.  Precondition: a cluster_sync separates this call from any
// earlier remote read of sh.hist.
template <class KeyFn>
__device__ void cluster_select(KeyFn keyf, int n_valid, int nw, int nbits, SelShared& sh,
                               uint32_t rank) {
  const int tid = threadIdx.x;
  if (tid < kMaxWays) {
    sh.prefix[tid] = 0;
    sh.selmask[tid] = 0;
  }
  for (int i = tid; i < 2 * kMaxWays * kDig; i += NT) (&sh.hist[0][0])[i] = 0;
  __syncthreads();
  const int passes = (nbits + kDigBits - 1) / kDigBits;
  for (int p = 0; p < passes; ++p) {
    const int hi = nbits - kDigBits * p;
    const int lo = hi - kDigBits > 0 ? hi - kDigBits : 0;
    const uint32_t dmask = (1u << (hi - lo)) - 1u;
    uint32_t* H = sh.hist[p & 1];
    for (int m = 0; m < nw; ++m) {
      if (!sh.active[m]) continue;
      const uint32_t pre = sh.prefix[m], msk = sh.selmask[m];
      for (int base = 0; base < n_valid; base += NT) {
        const int i = base + tid;
        uint32_t key = 0u;
        bool ok = i < n_valid && keyf(m, i, key);
        ok = ok && ((key & msk) == pre);
        hist_add_warp(H + m * kDig, (key >> lo) & dmask, ok);
      }
    }
    __syncthreads();
    cluster_sync();
    for (int i = tid; i < nw * kDig; i += NT) {
      if (!sh.active[i / kDig]) continue;
      sh.tot[i] = sum_over_cluster(&H[i], 0, nullptr);
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < nw && sh.active[warp]) {
      // lane l covers bins kDig-1-32l-j, j = 0..31 (descending)
      const int m = warp;
      const int need = sh.remaining[m];
      const uint32_t* T = sh.tot + m * kDig + kDig - 1 - 32 * lane;
      int s32 = 0;
#pragma unroll 8
      for (int j = 0; j < 32; ++j) s32 += static_cast<int>(T[-j]);
      int incl = s32;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned bal = __ballot_sync(0xffffffffu, incl >= need);
      const int L = bal ? __ffs(bal) - 1 : 31;
      if (lane == L) {
        const uint32_t* TL = sh.tot + m * kDig + kDig - 1 - 32 * L;
        int acc = incl - s32;
        int j = 0;
        for (; j < 31; ++j) {
          const int cj = static_cast<int>(TL[-j]);
          if (acc + cj >= need) break;
          acc += cj;
        }
        const uint32_t digit = static_cast<uint32_t>(kDig - 1 - 32 * L - j);
        sh.prefix[m] |= digit << lo;
        sh.selmask[m] |= dmask << lo;
        sh.remaining[m] = need - acc;
      }
    }
    if (tid == 0) {
      sh.last_lo = lo;
      sh.last_dmask = static_cast<int>(dmask);
    }
    __syncthreads();
    if (p + 1 < passes)
      for (int i = tid; i < kMaxWays * kDig; i += NT) sh.hist[(p + 1) & 1][i] = 0;
    __syncthreads();
  }
  if (passes > 0 && tid < nw && sh.active[tid]) {
    const int m = tid;
    const uint32_t dig = (sh.prefix[m] >> sh.last_lo) & static_cast<uint32_t>(sh.last_dmask);
    const uint32_t* h = &sh.hist[(passes - 1) & 1][m * kDig + dig];
    uint32_t before = 0;
    const uint32_t total = sum_over_cluster(h, rank, &before);
    sh.eq_local[m] = static_cast<int>(*h);
    sh.eq_before[m] = static_cast<int>(before);
    sh.eq_total[m] = static_cast<int>(total);
  }
  __syncthreads();
}

// Quota of threshold-equal elements this CTA takes, and whether they must be
// ranked (only the CTA where the cut falls inside its equal elements).
__device__ __forceinline__ void set_quota(SelShared& sh, int nw) {
  const int m = threadIdx.x;
  if (m < nw && sh.active[m]) {
    int q = sh.remaining[m] - sh.eq_before[m];
    q = q < 0 ? 0 : (q > sh.eq_local[m] ? sh.eq_local[m] : q);
    sh.quota[m] = q;
    sh.rank_needed[m] = (q > 0 && q < sh.eq_local[m]) ? 1 : 0;
  }
}

// MW: the number of MTP ways, fixed at compile time so every per-way loop over
// the tokens unrolls to exactly the ways that exist
template <int MW>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(NT, 1)
    select_kernel(const SelArgs a) {
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ SelShared sh;
  pdl_wait_previous();
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int b = blockIdx.x / CL;
  constexpr int M = MW;
  const int MK = M * a.k;
  const int Tb = a.Tb[b];
  const int keff = a.k < Tb ? a.k : Tb;
  const int r0 = static_cast<int>(rank) * a.n_local;
  int nloc = Tb - r0;
  nloc = nloc < 0 ? 0 : (nloc > a.n_local ? a.n_local : nloc);
  float* keys_s = reinterpret_cast<float*>(dsm);                      // [M][n_local]
  int* ltok = reinterpret_cast<int*>(dsm + a.keys_bytes);             // [lcap] token list
  int* lslot = ltok + a.lcap;                                         // [lcap] resolved slot
  int* cslot = lslot + a.lcap;                                        // [c_local] this CTA's LRU list slice
  uint32_t* ckey = reinterpret_cast<uint32_t*>(cslot + a.c_local);    // [M][lcap] candidate keys
  uint32_t* gkey = ckey + M * a.lcap;                                 // [gcap] gathered keys
  const int segw = a.c_local / 32;                                    // bitmap words per slot range
  uint32_t* hseg = gkey + a.gcap;        // [segw] stamps of this CTA's slot range (ORed remotely)
  uint32_t* hall = hseg + segw;          // [CL * segw] all stamps, copied after [S3]
  uint32_t* umask = hall + CL * segw;    // [segw] unstamped entries of this CTA's list positions
  uint8_t* grank = reinterpret_cast<uint8_t*>(umask + segw);          // [gcap] source rank
  uint8_t* lflag = grank + a.gcap;                                    // [lcap] way bits
  const int n_local = a.n_local, lcap = a.lcap, Tmax = a.T;
  const bool resident = a.resident != 0;
  const size_t bT = static_cast<size_t>(b) * a.T;
  const size_t bC = static_cast<size_t>(b) * a.C;
  uint32_t* gh = a.ghist + static_cast<size_t>(b) * M * kHistBins;
  const unsigned lt = lanemask_lt();
  int parity = 0;

  if (tid == 0) {
    // the previous step's readers of the counter completed before this grid
    // passed its wait; this step's readers launch after the resolve below
    if (a.ready != nullptr && rank == 0) {
      atomicExch(a.ready + b * kCounterStride, 0);
      for (int m = 0; m < M; ++m) atomicExch(a.attn_done + (b * M + m) * kCounterStride, 0);
    }
    sh.step_b = a.step[b];  // (also read directly as step0)
    sh.nl = 0;
    sh.fallback = 0;
    sh.pub_overflow = sh.pub_nmiss = sh.pub_nu = sh.pub_unst = 0;
    sh.ndefer = 0;
    for (int m = 0; m < kMaxWays; ++m) {
      sh.pub_hit[m] = sh.pub_miss[m] = 0;
      sh.active[m] = 0;
      sh.g[m] = (a.guess != nullptr && m < M) ? a.guess[b * M + m] : 0u;
      sh.fine[m] = 0;
    }
    mbar_init(smem_u32(&sh.bar), 1);
    fence_mbar_init();
  }
  // the stamp words of this CTA's slots; remote ORs into them come only after
  // a cluster barrier that every CTA reaches after this
  for (int i = tid; i < segw; i += NT) hseg[i] = 0u;
  __syncthreads();

  // this CTA's positions of the current LRU list (read after the hits are stamped)
  const int step0 = a.step[b];
  const int p0 = static_cast<int>(rank) * a.c_local;
  const bool lru = a.policy == ESS_EVICT_LRU;
  int cl = lru ? a.C - p0 : 0;   // other policies do not use the LRU list
  cl = cl < 0 ? 0 : (cl > a.c_local ? a.c_local : cl);
  const int32_t* ocur = a.order + (static_cast<size_t>(step0 & 1) * a.B + b) * a.C;
  int32_t* onxt = a.order + (static_cast<size_t>((step0 & 1) ^ 1) * a.B + b) * a.C;

  const bool sel_all = keff >= Tb;  // every token is selected (includes T_b = 0)
  // the indexer's histogram is final once the previous grid is: this
  // thread's bins (4095 - 8t - j, j = 0..7, per way) are read while the
  // scores are still landing
  const bool pre_hist = !sel_all && a.hist_given;
  uint32_t c8p[M][8];
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int j = 0; j < 8; ++j)
      c8p[m][j] = pre_hist ? gh[m * kHistBins + kHistBins - 1 - 8 * tid - j] : 0u;
  // so are the indexer's flag words (this thread's first word of the CTA's
  // range, the ways OR-ed) and its fine histogram (2M words per thread)
  const bool pre_guide = pre_hist && a.tflag != nullptr;
  const int fw0 = r0 >> 5, fw1 = (r0 + nloc + 31) >> 5;
  uint32_t tw_pre = 0u;
  if (pre_guide && nloc > 0 && fw0 + tid < fw1)
#pragma unroll
    for (int m = 0; m < M; ++m)
      tw_pre |= a.tflag[(static_cast<size_t>(b) * M + m) * a.nwords + fw0 + tid];
  static_assert(kFineBins % NT == 0, "fine bins spread evenly over the threads");
  constexpr int FPT = M * kFineBins / NT;
  uint32_t fpre[FPT];
#pragma unroll
  for (int j = 0; j < FPT; ++j)
    fpre[j] = pre_guide ? a.fhist[static_cast<size_t>(b) * M * kFineBins + tid + j * NT] : 0u;

  // ---------------------------------------------------------------- scores
  // The scores (and the order slice) land in shared memory by bulk copy; the
  // wait for them comes before the first code that reads them there, so the
  // bin search and the guided listing (which reads its few scores from global
  // memory) run while they land.
  const bool load_scores = resident && nloc > 0;
  // the order list slice is copied in 16-byte units when aligned, else by threads
  const bool bulk_order = cl > 0 && (cl & 3) == 0 && (p0 & 3) == 0 && (a.C & 3) == 0;
  auto wait_bulk = [&]() {   // idempotent: phase 0 stays complete
    if ((load_scores || bulk_order) && !mbar_wait(smem_u32(&sh.bar), 0, nullptr))
      set_status(a.status, ESS_ERR_TIMEOUT);
  };
  {
    const int cnt = ((nloc + 3) / 4) * 4 <= Tmax - r0 ? ((nloc + 3) / 4) * 4 : Tmax - r0;
    if (tid == 0 && (load_scores || bulk_order)) {
      uint32_t bytes = (load_scores ? cnt * 4 * M : 0) + (bulk_order ? cl * 4 : 0);
      mbar_arrive_expect_tx(smem_u32(&sh.bar), bytes);
      if (load_scores)
        for (int m = 0; m < M; ++m)
          bulk_load(smem_u32(keys_s + m * n_local),
                    a.scores + (static_cast<size_t>(b) * M + m) * Tmax + r0,
                    static_cast<uint32_t>(cnt * 4), smem_u32(&sh.bar));
      if (bulk_order)
        bulk_load(smem_u32(cslot), ocur + p0, static_cast<uint32_t>(cl * 4), smem_u32(&sh.bar));
    }
    if (!bulk_order)
      for (int i = tid; i < cl; i += NT) cslot[i] = ocur[p0 + i];
    // the fine bins go to shared memory, free until the candidate passes
    if (pre_guide)
#pragma unroll
      for (int j = 0; j < FPT; ++j) (&sh.hist[0][0])[tid + j * NT] = fpre[j];
    __syncthreads();
  }
  const float* gscores = a.scores + static_cast<size_t>(b) * M * Tmax + r0;
  auto score_key = [=](int m, int i) -> uint32_t {
    const float f = resident ? keys_s[m * n_local + i] : gscores[static_cast<size_t>(m) * Tmax + i];
    return float_key(f + 0.0f);  // +0 and -0 compare equal, as scores do
  };

  // ---------------------------------------------------------------- (a2) top-k
  if (!sel_all && !a.hist_given) {
    wait_bulk();
    // caller scores: build the 12-bit histogram of this request
    for (int m = 0; m < M; ++m)
      for (int base = 0; base < nloc; base += NT) {
        const int i = base + tid;
        const bool ok = i < nloc;
        hist_add_warp(gh + m * kHistBins, ok ? score_key(m, i) >> 20 : 0u, ok);
      }
    __syncthreads();
    cluster_sync();
  }
  if (!sel_all) {
#pragma unroll
    for (int m = 0; m < M; ++m) {
      // thread t owns bins 4095 - 8t - j, j = 0..7 (descending order)
      int c8[8];
      int s8 = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c8[j] = static_cast<int>(pre_hist ? c8p[m][j]
                                          : gh[m * kHistBins + kHistBins - 1 - 8 * tid - j]);
        s8 += c8[j];
      }
      int tot;
      const int excl = block_scan(s8, tot, sh, parity);
      if (excl < keff && keff <= excl + s8) {
        // first of this thread's bins (descending) where the count reaches keff;
        // unrolled so c8 stays in registers
        int acc = excl, jsel = 7, cj = c8[7];
        bool found = false;
#pragma unroll
        for (int j = 0; j < 7; ++j) {
          if (!found) {
            if (acc + c8[j] >= keff) {
              found = true;
              jsel = j;
              cj = c8[j];
            } else {
              acc += c8[j];
            }
          }
        }
        sh.b1[m] = kHistBins - 1 - 8 * tid - jsel;
        sh.take1[m] = keff - acc;
        sh.cand1[m] = cj;
      }
      if (tid == 0 && tot != Tb) sh.fallback = 1;  // histogram does not describe these scores
    }
    __syncthreads();
  }
  bool fast = !sel_all && !sh.fallback;
  const bool have_b1 = fast;   // the coarse bins describe this step's scores
  // Guided: every way's threshold bin lies at or above the bin its flags start
  // from, so the flagged tokens hold the whole selection and its candidates.
  bool guided = fast && a.tflag != nullptr;
  for (int m = 0; m < M; ++m)
    guided = guided && sh.g[m] != 0u && static_cast<uint32_t>(sh.b1[m]) >= sh.g[m];
  if (guided) {
    // a way whose threshold bin the fine histogram covers takes its cut on 8
    // more key bits: candidates are the keys of one fine bin
    if (warp < M) {
      const int m = warp;
      const uint32_t d = static_cast<uint32_t>(sh.b1[m]) - sh.g[m];
      int fine = 0;
      if (d < static_cast<uint32_t>(kFineWin)) {
        const uint32_t* F = &sh.hist[0][0] + m * kFineBins + d * kFineSub;
        // lane l owns fine bins 255 - 8l - j, j = 0..7 (descending)
        int c8[8];
        int s8 = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c8[j] = static_cast<int>(F[kFineSub - 1 - 8 * lane - j]);
          s8 += c8[j];
        }
        int incl = s8;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int tot = __shfl_sync(0xffffffffu, incl, 31);
        const int need = sh.take1[m];
        if (tot == sh.cand1[m]) {   // the fine bins add up to the coarse bin
          fine = 1;
          const unsigned bal = __ballot_sync(0xffffffffu, incl >= need);
          if (lane == __ffs(bal) - 1) {
            int acc = incl - s8, jsel = 7, cj = c8[7];
            bool found = false;
#pragma unroll
            for (int j = 0; j < 7; ++j) {
              if (!found) {
                if (acc + c8[j] >= need) {
                  found = true;
                  jsel = j;
                  cj = c8[j];
                } else {
                  acc += c8[j];
                }
              }
            }
            sh.fb[m] = kFineSub - 1 - 8 * lane - jsel;
            sh.take1[m] = need - acc;
            sh.cand1[m] = cj;
          }
        }
      }
      if (lane == 0) sh.fine[m] = fine;
    }
    __syncthreads();
  }
  // cache slots of the listed tokens, read as soon as the list is out and
  // carried through the filter (its first four rounds), so that the resolve
  // reads them from shared memory
  int csr[4] = {-1, -1, -1, -1};
  bool cs_ready = false;
  if (sel_all) {
    for (int i = tid; i < nloc; i += NT) {
      ltok[i] = r0 + i;
      lflag[i] = static_cast<uint8_t>((1u << M) - 1u);
    }
    if (tid == 0) sh.nl = nloc;
    wait_bulk();
    __syncthreads();
    cluster_sync();   // every CTA's stamp words are zero (the other paths pass one too)
  }
  if (fast) {
    // one ordered pass over this CTA's tokens, each warp over its own
    // contiguous range: tokens above the coarse bin are selected (low
    // nibble), tokens in it are candidates (high nibble)
    uint32_t lo_k[kMaxWays], hi_k[kMaxWays];
#pragma unroll
    for (int m = 0; m < kMaxWays; ++m) {
      const bool use = m < M;
      const uint32_t bin = use ? static_cast<uint32_t>(sh.b1[m]) : 0xFFFu;
      const bool all_in = use && sh.take1[m] == sh.cand1[m];
      if (use && sh.fine[m]) {
        // the cut's fine bin: 4096 keys wide
        const uint32_t lo = (bin << 20) | (static_cast<uint32_t>(sh.fb[m]) << 12);
        lo_k[m] = lo;
        hi_k[m] = all_in ? lo : (lo == 0xFFFFF000u ? 0xFFFFFFFFu : lo + 4096u);
        continue;
      }
      lo_k[m] = bin << 20;                                    // key >= lo: at or above the bin
      hi_k[m] = all_in ? (bin << 20) : ((bin + 1u) << 20);    // key >= hi: selected outright
      if (!use) lo_k[m] = hi_k[m] = 0xFFFFFFFFu;
      if (use && bin == 0xFFFu && !all_in) hi_k[m] = 0xFFFFFFFFu;  // top bin: nothing above it
    }
    auto coarse_flags = [=](int i) -> uint32_t {
      uint32_t f = 0;
#pragma unroll
      for (int m = 0; m < kMaxWays; ++m) {
        if (m >= M) break;
        const uint32_t key = score_key(m, i);
        if (key >= hi_k[m]) f |= 1u << m;
        else if (key >= lo_k[m]) f |= 16u << m;
      }
      return f;
    };
    // the flags of one token from its scores (M ways)
    auto flags_of = [=](const float* sv) -> uint32_t {
      uint32_t f = 0;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint32_t key = float_key(sv[m] + 0.0f);
        if (key >= hi_k[m]) f |= 1u << m;
        else if (key >= lo_k[m]) f |= 16u << m;
      }
      return f;
    };
    auto flags_global = [=](int i) -> uint32_t {
      float sv[M];
#pragma unroll
      for (int m = 0; m < M; ++m) sv[m] = gscores[static_cast<size_t>(m) * Tmax + i];
      return flags_of(sv);
    };
    int total;
    if (guided) {
      // the flagged tokens only: one flag word per thread (the ways' words
      // OR-ed, clipped to this CTA's tokens).  The scores of a word's first
      // eight flagged tokens are read from global memory together, the rest
      // one by one; the tokens that the keys place at or above the cut are
      // counted, given ordered positions, and listed.
      const int w0 = r0 >> 5, w1 = (r0 + nloc + 31) >> 5;
      int run = 0;
      for (int wb = w0; wb < w1; wb += NT) {
        const int w = wb + tid;
        uint32_t bits = 0u;
        if (w < w1 && nloc > 0) {
          if (wb == w0) {
            bits = tw_pre;
          } else {
#pragma unroll
            for (int m = 0; m < M; ++m)
              bits |= a.tflag[(static_cast<size_t>(b) * M + m) * a.nwords + w];
          }
          const int tlo = w * 32, thi = r0 + nloc;
          if (tlo < r0) bits &= 0xFFFFFFFFu << (r0 - tlo);
          if (thi - tlo < 32) bits &= (1u << (thi - tlo)) - 1u;
        }
        constexpr int NB = 8;
        int jj[NB];
        uint32_t x = bits;
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          jj[u] = -1;
          if (x != 0u) {
            jj[u] = __ffs(x) - 1;
            x &= x - 1u;
          }
        }
        const uint32_t rest = x;   // flagged tokens past the first eight
        float sv[NB][M];
#pragma unroll
        for (int u = 0; u < NB; ++u)
#pragma unroll
          for (int m = 0; m < M; ++m)
            sv[u][m] = jj[u] >= 0 ? gscores[static_cast<size_t>(m) * Tmax + (w * 32 + jj[u] - r0)]
                                  : 0.0f;
        uint32_t fl[NB];
        uint32_t q = 0u;
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          fl[u] = jj[u] >= 0 ? flags_of(sv[u]) : 0u;
          q += fl[u] ? 1u : 0u;
        }
        for (uint32_t y = rest; y != 0u; y &= y - 1u)
          q += flags_global(w * 32 + (__ffs(y) - 1) - r0) ? 1u : 0u;
        int p = ordered_pos(static_cast<int>(q), run, sh, parity);
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          if (fl[u] == 0u) continue;
          if (p < lcap) {
            ltok[p] = w * 32 + jj[u];
            lflag[p] = static_cast<uint8_t>(fl[u]);
          }
          ++p;
        }
        for (uint32_t y = rest; y != 0u; y &= y - 1u) {
          const int i = w * 32 + (__ffs(y) - 1) - r0;
          const uint32_t f = flags_global(i);
          if (f == 0u) continue;
          if (p < lcap) {
            ltok[p] = r0 + i;
            lflag[p] = static_cast<uint8_t>(f);
          }
          ++p;
        }
      }
      total = run;
      wait_bulk();   // the candidate keys and the filter read the staged scores
    } else {
    wait_bulk();
    const int per_w = (((nloc + NW - 1) / NW) + 31) & ~31;
    const int wlo = warp * per_w;
    const int whi = wlo + per_w < nloc ? wlo + per_w : nloc;
    // one pass: each warp stages its flagged tokens (in the candidate-key
    // gather buffer, unused until later) and copies them to their place once
    // the warps' counts are known; a warp whose range flags more than its
    // staging holds lists its range a second time instead
    constexpr int WSTAGE = 128;
    uint32_t* stok = gkey + warp * WSTAGE;
    uint8_t* sflg = grank + warp * WSTAGE;
    int wcnt = 0;
    // eight 32-token groups per iteration: their score reads are in flight
    // together (they come from global memory when the scores do not fit in
    // shared memory)
    constexpr int G = 8;
    for (int base = wlo; base < whi; base += 32 * G) {
      uint32_t f4[G];
#pragma unroll
      for (int u = 0; u < G; ++u) {
        const int i = base + 32 * u + lane;
        f4[u] = i < whi ? coarse_flags(i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < G; ++u) {
        const int i = base + 32 * u + lane;
        const unsigned bal = __ballot_sync(0xffffffffu, f4[u] != 0);
        if (f4[u]) {
          const int p = wcnt + __popc(bal & lt);
          if (p < WSTAGE) {
            stok[p] = static_cast<uint32_t>(r0 + i);
            sflg[p] = static_cast<uint8_t>(f4[u]);
          }
        }
        wcnt += __popc(bal);
      }
    }
    __syncwarp();
    int pos = warp_base(wcnt, total, sh);
    if (wcnt <= WSTAGE) {
      for (int j = lane; j < wcnt; j += 32) {
        const int p = pos + j;
        if (p < lcap) {
          ltok[p] = static_cast<int>(stok[j]);
          lflag[p] = sflg[j];
        }
      }
    } else {
      for (int base = wlo; base < whi; base += 32) {
        const int i = base + lane;
        const uint32_t f = i < whi ? coarse_flags(i) : 0u;
        const unsigned bal = __ballot_sync(0xffffffffu, f != 0);
        if (f) {
          const int p = pos + __popc(bal & lt);
          if (p < lcap) {
            ltok[p] = r0 + i;
            lflag[p] = static_cast<uint8_t>(f);
          }
        }
        pos += __popc(bal);
      }
    }
    }
    const int nl = total < lcap ? total : lcap;
    // candidates of each way in list order, with their low 20 key bits
    if (tid < M) {
      sh.active[tid] = sh.take1[tid] < sh.cand1[tid] ? 1 : 0;
      sh.remaining[tid] = sh.take1[tid];
    }
    __syncthreads();
    for (int m = 0; m < M; ++m) {
      if (!sh.active[m]) {
        if (tid == 0) sh.ncand[m] = 0;
        continue;
      }
      int run = 0;
      for (int base = 0; base < nl; base += NT) {
        const int e = base + tid;
        const bool c = e < nl && (lflag[e] & (16u << m));
        const int p = ordered_pos(c ? 1 : 0, run, sh, parity);
        if (c) ckey[m * lcap + p] = score_key(m, ltok[e] - r0) & 0xFFFFFu;
      }
      if (tid == 0) sh.ncand[m] = run;
    }
    if (tid == 0) {
      sh.nl = nl;
      sh.pub_overflow = total > lcap ? 1 : 0;
      int need = 0;
      for (int m = 0; m < M; ++m) need += sh.active[m] ? sh.cand1[m] : 0;
      sh.gsel = need <= a.gcap ? 1 : 0;   // same in every CTA: from the shared histogram
    }
    __syncthreads();
    cluster_sync();  // lists and candidate keys complete; overflow flags published
    // every CTA's overflow flag and candidate counts, in one round of remote reads
    if (tid < CL) {
      const uint32_t r = static_cast<uint32_t>(tid);
      const uint32_t ovf = ld_dsmem_u32(dsmem_addr(smem_u32(&sh.pub_overflow), r));
      uint32_t nc[M];
#pragma unroll
      for (int m = 0; m < M; ++m) nc[m] = ld_dsmem_u32(dsmem_addr(smem_u32(&sh.ncand[m]), r));
#pragma unroll
      for (int m = 0; m < M; ++m) sh.gcnt[m][tid] = static_cast<int>(nc[m]);
      if (ovf) sh.fallback = 1;
    }
    __syncthreads();
    fast = !sh.fallback;
    // (read after the list barrier: loads still in flight at a cluster
    // barrier's release would hold it up)
    if (fast) {
      const int nl = sh.nl;
#pragma unroll
      for (int q = 0; q < 4; ++q) {   // the filter's entry-to-thread mapping
        const int e = q * NT + tid;
        csr[q] = e < nl ? a.cache_slots[bT + ltok[e]] : -1;
      }
    }
  }
  if (fast) {
    const int nl = sh.nl;
    bool any = false;
    for (int m = 0; m < M; ++m) any |= sh.active[m] != 0;
    if (any && sh.gsel) {
      // gather every CTA's candidate keys (in cluster order) and find the
      // exact threshold locally: the same result in every CTA, no more barriers
      for (int m = 0; m < M; ++m) {
        if (!sh.active[m]) continue;
        // every CTA's count (read with the overflow flags), then all the remote reads at once
        int roff[CL + 1];
        roff[0] = 0;
#pragma unroll
        for (int r = 0; r < CL; ++r) roff[r + 1] = roff[r] + sh.gcnt[m][r];
        const int off = roff[CL];
        const int ngc = off < a.gcap ? off : a.gcap;
        const int need0 = sh.remaining[m];   // unchanged until after the next barrier
        const uint32_t kbase = smem_u32(ckey + m * lcap);
        for (int g = tid; g < ngc; g += NT) {
          int r = 0;
#pragma unroll
          for (int q = 1; q < CL; ++q) r += g >= roff[q] ? 1 : 0;
          int base = 0;
#pragma unroll
          for (int q = 0; q < CL; ++q) base = (q == r) ? roff[q] : base;
          gkey[g] = ld_dsmem_u32(dsmem_addr(kbase, static_cast<uint32_t>(r)) + 4u * (g - base));
          grank[g] = static_cast<uint8_t>(r);
        }
        __syncthreads();
        const int ng = off < a.gcap ? off : a.gcap;
        uint32_t pre = 0;
        if (ng <= kDirectRank) {
          // few candidates: each one's rank among them (equal keys by their
          // place in cluster order, i.e. by token); rank need - 1 is the cut
          if (tid < ng) {
            const uint32_t kg = gkey[tid];
            int gt = 0, eqb = 0;
            for (int i = 0; i < ng; ++i) {
              const uint32_t ki = gkey[i];
              gt += ki > kg ? 1 : 0;
              eqb += (ki == kg && i < tid) ? 1 : 0;
            }
            if (gt + eqb == need0 - 1) {
              sh.prefix[m] = kg;
              sh.remaining[m] = need0 - gt;   // threshold-equal candidates to take
            }
          }
          __syncthreads();
          pre = sh.prefix[m];
        } else {
        // exact take1-th largest of the gathered keys: two 10-bit passes
        uint32_t* H = sh.hist[0];
        uint32_t msk = 0;
        int need = sh.remaining[m];
        for (int p = 0; p < 2; ++p) {
          const int lo = p == 0 ? 10 : 0;
          for (int i = tid; i < kDig; i += NT) H[i] = 0;
          __syncthreads();
          for (int i = tid; i < ng; i += NT) {
            const uint32_t k = gkey[i];
            if ((k & msk) == pre) atomicAdd(&H[(k >> lo) & (kDig - 1)], 1u);
          }
          __syncthreads();
          {
            // thread t owns bins kDig-1-2t and kDig-2-2t (descending): one
            // block-wide prefix finds the bin where the count reaches need
            static_assert(2 * NT == kDig, "two bins per thread");
            const int hb = kDig - 1 - 2 * tid;
            const int c0 = static_cast<int>(H[hb]), c1 = static_cast<int>(H[hb - 1]);
            int tot2;
            const int excl = block_scan(c0 + c1, tot2, sh, parity);
            if (excl < need && need <= excl + c0 + c1) {
              const bool upper = excl + c0 >= need;
              sh.prefix[m] = pre | (static_cast<uint32_t>(upper ? hb : hb - 1) << lo);
              sh.remaining[m] = need - (upper ? excl : excl + c0);
            }
          }
          __syncthreads();
          pre = sh.prefix[m];
          msk |= static_cast<uint32_t>(kDig - 1) << lo;
          need = sh.remaining[m];
          __syncthreads();
        }
        }
        // threshold-equal candidates: this CTA's count and those of lower ranks
        if (tid == 0) {
          sh.eq_local[m] = 0;
          sh.eq_before[m] = 0;
        }
        __syncthreads();
        int el = 0, eb = 0;
        for (int i = tid; i < ng; i += NT) {
          if (gkey[i] != pre) continue;
          const uint32_t r = grank[i];
          el += r == rank ? 1 : 0;
          eb += r < rank ? 1 : 0;
        }
        for (int o = 16; o; o >>= 1) {
          el += __shfl_xor_sync(0xffffffffu, el, o);
          eb += __shfl_xor_sync(0xffffffffu, eb, o);
        }
        if (lane == 0 && (el || eb)) {
          atomicAdd(&sh.eq_local[m], el);
          atomicAdd(&sh.eq_before[m], eb);
        }
        __syncthreads();
      }
      set_quota(sh, M);
      __syncthreads();
    } else if (any) {
      auto cand_key = [&](int m, int e, uint32_t& key) -> bool {
        if (!(lflag[e] & (16u << m))) return false;
        key = score_key(m, ltok[e] - r0) & 0xFFFFFu;
        return true;
      };
      cluster_select(cand_key, nl, M, 20, sh, rank);
      set_quota(sh, M);
      __syncthreads();
    }
    // filter the list in place into the union of the ways' selections
    int eqrun[kMaxWays] = {0, 0, 0, 0};
    int nu = 0;
    for (int base = 0; base < nl; base += NT) {
      const int e = base + tid;
      int tok = 0;
      uint32_t f = 0;
      if (e < nl) {
        tok = ltok[e];
        f = lflag[e];
      }
      int cs = -1;
      if (base < 4 * NT) {
        cs = csr[0];
        csr[0] = csr[1];
        csr[1] = csr[2];
        csr[2] = csr[3];
      } else if (e < nl) {
        cs = a.cache_slots[bT + tok];
      }
      uint32_t sel = f & 0xFu;
#pragma unroll
      for (int m = 0; m < kMaxWays; ++m) {
        if (m >= M) break;
        if (!sh.active[m]) continue;
        const bool cm = (f >> (4 + m)) & 1u;
        const uint32_t k20 = cm ? (score_key(m, tok - r0) & 0xFFFFFu) : 0u;
        const uint32_t thr = sh.prefix[m];
        const bool eq = cm && k20 == thr;
        if (cm && k20 > thr) sel |= 1u << m;
        if (sh.rank_needed[m]) {
          const int r = ordered_pos(eq ? 1 : 0, eqrun[m], sh, parity);
          if (eq && r < sh.quota[m]) sel |= 1u << m;
        } else if (eq && sh.quota[m] > 0) {
          sel |= 1u << m;
        }
      }
      const int pos = ordered_pos(sel ? 1 : 0, nu, sh, parity);
      if (sel) {
        ltok[pos] = tok;
        lflag[pos] = static_cast<uint8_t>(sel);
        lslot[pos] = cs;
      }
    }
    cs_ready = true;
    if (tid == 0) sh.nl = nu;
    __syncthreads();
  } else if (!sel_all) {
    // fallback: exact radix passes over every token
    wait_bulk();
    if (tid < M) {
      sh.active[tid] = 1;
      sh.remaining[tid] = keff;
    }
    __syncthreads();
    auto all_key = [&](int m, int i, uint32_t& key) -> bool {
      key = score_key(m, i);
      return true;
    };
    cluster_select(all_key, nloc, M, 32, sh, rank);
    set_quota(sh, M);
    __syncthreads();
    int eqrun[kMaxWays] = {0, 0, 0, 0};
    int nu = 0;
    for (int base = 0; base < nloc; base += NT * 4) {
      const int i0 = base + tid * 4;
      uint32_t selbits[4] = {0, 0, 0, 0};
#pragma unroll
      for (int m = 0; m < kMaxWays; ++m) {
        if (m >= M) break;
        const uint32_t thr = sh.prefix[m];
        bool eq[4];
        int neq = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool valid = (i0 + j) < nloc;
          const uint32_t key = valid ? score_key(m, i0 + j) : 0u;
          eq[j] = valid && key == thr;
          neq += eq[j];
          if (valid && key > thr) selbits[j] |= 1u << m;
        }
        if (sh.rank_needed[m]) {
          int r = ordered_pos(neq, eqrun[m], sh, parity);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (eq[j]) {
              if (r < sh.quota[m]) selbits[j] |= 1u << m;
              ++r;
            }
        } else if (sh.quota[m] > 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (eq[j]) selbits[j] |= 1u << m;
        }
      }
      int cu = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) cu += selbits[j] ? 1 : 0;
      int pos = ordered_pos(cu, nu, sh, parity);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (selbits[j]) {
          if (pos < a.lcap) {
            ltok[pos] = r0 + i0 + j;
            lflag[pos] = static_cast<uint8_t>(selbits[j]);
          } else {
            set_status(a.status, ESS_ERR_DEVICE_CHECK);
          }
          ++pos;
        }
    }
    if (tid == 0) sh.nl = nu < a.lcap ? nu : a.lcap;
    __syncthreads();
  }
  const int nu = sh.nl;

  // ---------------------------------------------------------------- (a3) resolve
  // The LRU finishing kernel may launch now: its CTAs take their SMs while
  // this kernel finishes, and only wait for it.  Launched at this kernel's
  // start instead, they slowed its first phases by a few microseconds.
  pdl_launch_dependents();
  // a miss among this thread's first entries: its page-table entry is read
  // now and used for the prefetch of its host row after [S3]
  int pf_page = -1;
  for (int e = tid; e < nu; e += NT) {
    const int t = ltok[e];
    int s = cs_ready ? lslot[e] : a.cache_slots[bT + t];
    if (s >= a.C || s < -1) {
      set_status(a.status, ESS_ERR_DEVICE_CHECK);
      s = -1;
    }
    lslot[e] = s;
    if (s >= 0) {
      // the hit's stamp in last_used is written after the last cluster barrier
      // (nothing in this kernel reads it; a store still in flight would hold a
      // barrier's release); the stamp bitmap carries it to the LRU scan
      if (lru) {
        const int ow = s / a.c_local, o = s - ow * a.c_local;
        red_or_dsmem(dsmem_addr(smem_u32(hseg + (o >> 5)), static_cast<uint32_t>(ow)),
                     1u << (o & 31));
      }
    }
    const uint32_t mk = lflag[e];
    for (int m = 0; m < M; ++m)
      if (mk & (1u << m)) atomicAdd(s >= 0 ? &sh.pub_hit[m] : &sh.pub_miss[m], 1);
    if (s < 0) atomicAdd(&sh.pub_nmiss, 1);
    if (s < 0 && e == tid && a.host != nullptr && a.page_table != nullptr)
      pf_page = a.page_table[static_cast<size_t>(b) * (a.T / a.page) + t / a.page];
  }
  if (tid == 0) sh.pub_nu = nu;
  __syncthreads();
  cluster_sync();  // [S3] stamps visible, per-CTA counts published
  // the whole stamp bitmap, every CTA's words (the remote ORs are complete),
  // 16 bytes a thread; the first round's reads are in flight with the sums
  const int nv4 = lru ? CL * segw / 4 : 0;
  uint4 hv = make_uint4(0u, 0u, 0u, 0u);
  if (tid < nv4) {
    const int w = 4 * tid, r = w / segw;
    hv = ld_dsmem_v4(dsmem_addr(smem_u32(hseg + (w - r * segw)), static_cast<uint32_t>(r)));
  }
  // the cluster sums, each in a warp of its own so that their remote reads overlap
  if (tid == 0) {
    uint32_t before = 0;
    sh.n_miss_total = static_cast<int>(sum_over_cluster(&sh.pub_nmiss, rank, &before));
    sh.miss_off = static_cast<int>(before);
  } else if (tid == 32) {
    sh.nu_total = static_cast<int>(sum_over_cluster(&sh.pub_nu, rank, nullptr));
  } else if (tid >= 64 && tid < 64 + M) {
    uint32_t before = 0;
    sh.nmw[tid - 64] = static_cast<int>(sum_over_cluster(&sh.pub_miss[tid - 64], rank, &before));
    sh.wmiss_off[tid - 64] = static_cast<int>(before);
  } else if (tid >= 96 && tid < 96 + M) {
    uint32_t before = 0;
    sh.hits_total[tid - 96] = static_cast<int>(sum_over_cluster(&sh.pub_hit[tid - 96], rank, &before));
    sh.hit_off[tid - 96] = static_cast<int>(before);
  }
  // LRU positions of this CTA in the current order list
  const int per_wc = (((cl + NW - 1) / NW) + 31) & ~31;
  const int clo = warp * per_wc;
  const int chi = clo + per_wc < cl ? clo + per_wc : cl;
  if (tid < nv4) *reinterpret_cast<uint4*>(hall + 4 * tid) = hv;
  for (int q = tid + NT; q < nv4; q += NT) {
    const int w = 4 * q, r = w / segw;
    *reinterpret_cast<uint4*>(hall + w) =
        ld_dsmem_v4(dsmem_addr(smem_u32(hseg + (w - r * segw)), static_cast<uint32_t>(r)));
  }
  __syncthreads();
  int wpre = 0;   // unstamped entries of the warps before this one
  {
    // unstamped entries among my positions of the list, 32 at a time: their
    // mask is kept for the placement after [S4]
    int wcnt = 0;
    for (int base = clo; base < chi; base += 32) {
      const int i = base + lane;
      bool un = false;
      if (i < chi) {
        int sl = cslot[i];
        if (sl < 0 || sl >= a.C) {
          set_status(a.status, ESS_ERR_DEVICE_CHECK);
          sl = 0;
          cslot[i] = 0;
        }
        un = ((hall[sl >> 5] >> (sl & 31)) & 1u) == 0u;
      }
      const unsigned bal = __ballot_sync(0xffffffffu, un);
      if (lane == 0) umask[base >> 5] = bal;
      wcnt += __popc(bal);
    }
    int total;
    wpre = warp_base(wcnt, total, sh);
    if (tid == 0) sh.pub_unst = total;
  }
  __syncthreads();
  cluster_arrive();  // [S4] unstamped counts published (the miss union goes on meanwhile)
  int n_miss_total = sh.n_miss_total;
  if (n_miss_total > a.C || n_miss_total > MK) {  // cannot happen when C >= min(M*k, T)
    if (tid == 0) set_status(a.status, ESS_ERR_CAPACITY);
    n_miss_total = 0;
  }
  {
    // the miss union in ascending token order
    int run = sh.miss_off;
    for (int base = 0; base < nu; base += NT) {
      const int e = base + tid;
      const bool f = e < nu && lslot[e] < 0;
      const int pos = ordered_pos(f ? 1 : 0, run, sh, parity);
      if (f && pos < MK) {
        const int t = ltok[e];
        lslot[e] = -2 - pos;   // a miss: its index in the request's miss union
        a.miss_tok[static_cast<size_t>(b) * MK + pos] = t;
        if (a.host != nullptr && t < a.T0[b]) {
          const int pg = !a.page_table ? 0
                         : base == 0   ? pf_page
                                       : a.page_table[static_cast<size_t>(b) * (a.T / a.page) +
                                                      t / a.page];
          const int pr = a.page_table ? pg * a.page + t % a.page : t;
          if (pr >= 0 && pr < a.T)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(
                a.host + (static_cast<size_t>(b) * a.T + pr) * a.row_bytes));
        }
      }
    }
  }
  cluster_wait();  // [S4]
  if (tid == 0) {
    uint32_t before = 0;
    sh.unst_total = static_cast<int>(sum_over_cluster(&sh.pub_unst, rank, &before));
    sh.unst_before = static_cast<int>(before);
  }
  __syncthreads();
  // Unstamped slots in LRU order: the first |Miss| are the victims, the rest
  // open the next list (each warp places its own contiguous positions); with
  // another policy cl is 0 and victim_kernel lists the victims.  The victims,
  // which other CTAs read, go out before the barrier; the next list after it.
  const int upos0 = sh.unst_before + wpre;
  if (sh.unst_before < n_miss_total) {
    int pos = upos0;
    for (int base = clo; base < chi && pos < n_miss_total; base += 32) {
      const unsigned msk = umask[base >> 5];
      if ((msk >> lane) & 1u) {
        const int p = pos + __popc(msk & lt);
        if (p < n_miss_total) a.vlist[static_cast<size_t>(b) * MK + p] = cslot[base + lane];
      }
      pos += __popc(msk);
    }
  }
  cluster_arrive();  // [S5] victims listed (the lists go out meanwhile)
  {
    int pos = upos0;
    for (int base = clo; base < chi; base += 32) {
      const unsigned msk = umask[base >> 5];
      if ((msk >> lane) & 1u) {
        const int p = pos + __popc(msk & lt) - n_miss_total;
        if (p >= 0 && p < a.C) onxt[p] = cslot[base + lane];
      }
      pos += __popc(msk);
    }
    // the hits' stamps (misses' slots are stamped by lru_finish_kernel)
    for (int e = tid; e < nu; e += NT) {
      const int s = lslot[e];
      if (s >= 0) a.last_used[bC + s] = sh.step_b;
    }
  }

  // ---------------------------------------------------------------- emit per-way lists
  // Misses first, then hits, each in token order.  Under LRU a miss's slot is
  // its victim's, listed by whichever CTA holds that position of the LRU list:
  // it is written after [S5] from a deferred (way, position, miss index).
  uint32_t* defer = ckey;   // the candidate keys are no longer needed
  for (int m = 0; m < M; ++m) {
    int runm = sh.wmiss_off[m];
    int runh = sh.nmw[m] + sh.hit_off[m];
    const size_t wo = (static_cast<size_t>(b) * M + m) * a.k;
    for (int base = 0; base < nu; base += NT) {
      const int e = base + tid;
      bool fm = false, fh = false;
      int t = 0, s = -1;
      if (e < nu && (lflag[e] & (1u << m))) {
        t = ltok[e];
        s = lslot[e];
        fm = s < 0;
        fh = !fm;
      }
      // one scan for both lists: misses in the low half-word, hits in the high
      int tot;
      const int ex = block_scan((fm ? 1 : 0) | (fh ? 1 << 16 : 0), tot, sh, parity);
      const int pm = runm + (ex & 0xFFFF), ph = runh + (ex >> 16);
      runm += tot & 0xFFFF;
      runh += tot >> 16;
      if (fm && pm < a.k) {
        const int mi = -2 - s;
        a.topk_idx[wo + pm] = t;
        if (lru) {
          const int d = atomicAdd(&sh.ndefer, 1);
          // way (2 bits), position (13 bits: k <= 8192), miss index + 1 (14 bits, 0: none)
          defer[d] = (static_cast<uint32_t>(m) << 27) | (static_cast<uint32_t>(pm) << 14) |
                     static_cast<uint32_t>(mi >= 0 && mi < MK ? mi + 1 : 0);
        } else {
          a.topk_slot[wo + pm] = -2 - mi;   // its miss index; victim_kernel puts ~slot here
        }
      }
      if (fh && ph < a.k) {
        a.topk_idx[wo + ph] = t;
        a.topk_slot[wo + ph] = s;
      }
    }
  }
  cluster_wait();  // [S5] no shared memory is read remotely after this
  __syncthreads();
  if (n_miss_total > 0 && lru) {
    // the i-th miss goes to the i-th victim (the state rewrite and the rest of
    // the next LRU list are left to lru_finish_kernel)
    const int per = (n_miss_total + CL - 1) / CL;
    const int i0 = static_cast<int>(rank) * per;
    const int i1 = i0 + per < n_miss_total ? i0 + per : n_miss_total;
    for (int i = i0 + tid; i < i1; i += NT)
      a.miss_slot[static_cast<size_t>(b) * MK + i] = a.vlist[static_cast<size_t>(b) * MK + i];
  }
  for (int i = tid; i < sh.ndefer; i += NT) {
    const uint32_t d = defer[i];
    const int m = static_cast<int>(d >> 27), pm = static_cast<int>((d >> 14) & 0x1FFF);
    const int mi = static_cast<int>(d & 0x3FFF) - 1;
    const int ns = (mi >= 0 && mi < n_miss_total) ? a.vlist[static_cast<size_t>(b) * MK + mi] : 0;
    a.topk_slot[(static_cast<size_t>(b) * M + m) * a.k + pm] = ~ns;
  }
  if (rank == 0 && tid == 0) {
    for (int m = 0; m < M; ++m) a.n_miss_way[b * M + m] = sh.nmw[m];
    a.n_miss[b] = n_miss_total;
  }
  if (lru && a.ready != nullptr) {
    // this CTA's share of request b's lists is out
    __syncthreads();
    if (tid == 0) count_done(a.ready + b * kCounterStride, 1);
  }
  if (rank == 0 && tid == 0) {
    if (a.stats) {
      long long h = 0, mi = 0;
      for (int m = 0; m < M; ++m) {
        h += sh.hits_total[m];
        mi += sh.nmw[m];
      }
      atomicAdd(reinterpret_cast<unsigned long long*>(&a.stats[0]), 1ull);
      atomicAdd(reinterpret_cast<unsigned long long*>(&a.stats[1]), static_cast<unsigned long long>(h));
      atomicAdd(reinterpret_cast<unsigned long long*>(&a.stats[2]), static_cast<unsigned long long>(mi));
      atomicAdd(reinterpret_cast<unsigned long long*>(&a.stats[3]),
                static_cast<unsigned long long>(sh.nu_total));
      atomicAdd(reinterpret_cast<unsigned long long*>(&a.stats[4]),
                static_cast<unsigned long long>(n_miss_total));
      atomicAdd(reinterpret_cast<unsigned long long*>(&a.stats[5]),
                static_cast<unsigned long long>(n_miss_total) * kRowBytes);
      if (guided) {
        int nf = 0;
        for (int m = 0; m < M; ++m) nf += sh.fine[m];
        atomicAdd(reinterpret_cast<unsigned long long*>(&a.stats[6]), 1ull);
        atomicAdd(reinterpret_cast<unsigned long long*>(&a.stats[7]),
                  static_cast<unsigned long long>(nf));
      }
    }
  }
  // every CTA read the histogram before [S3]: clear it for the next step
  if (rank == 0)
    for (int i = tid; i < M * kHistBins; i += NT) gh[i] = 0u;
  if (rank == 0 && a.guess != nullptr) {
    // the same for the fine histogram; every CTA read its guesses at the
    // start: the next step's indexer flags from one bin below this cut
    uint32_t* fh = a.fhist + static_cast<size_t>(b) * M * kFineBins;
    for (int i = tid; i < M * kFineBins; i += NT) fh[i] = 0u;
    if (tid < M) {
      const int b1 = sh.b1[tid];
      a.guess[b * M + tid] = (have_b1 && b1 >= 2) ? static_cast<uint32_t>(b1 - 1) : 0u;
    }
  }
}

// (a4) the rest of the LRU update, after the lists are out: each miss's
// victim slot takes the miss (cache_slots / slot_token / last_used), the
// stamped slots (hits and victims) close the next LRU list in slot order,
// and the request's step counter advances.  Nothing downstream in the same
// step reads what this kernel writes, so the attention kernel can run beside
// it; the next step's selection reads it.
struct LruShared {
  int pub_stamp;       // stamped slots in this CTA's slot range (read through DSMEM)
  int stamp_before, stamp_total;
  int wcount[NW];
};

__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(NT, 1)
    lru_finish_kernel(const SelArgs a) {
  // whatever follows waits before it reads what the selection wrote: with
  // griddepcontrol.wait, or (a step's attention) on the selection's counters,
  // so it may launch before this grid's own wait is over
  pdl_launch_dependents();
  pdl_wait_previous();
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ LruShared sh;
  uint8_t* cflag = dsm;                                        // [c_local] stamped flags
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int b = blockIdx.x / CL;
  const int MK = a.M * a.k;
  const int Tb = a.Tb[b];
  const size_t bT = static_cast<size_t>(b) * a.T;
  const size_t bC = static_cast<size_t>(b) * a.C;
  const unsigned lt = lanemask_lt();
  const int step_b = a.step[b];
  const int p0 = static_cast<int>(rank) * a.c_local;
  // the LRU list is kept only under the LRU policy (cl = 0 skips its upkeep)
  int cl = a.policy == ESS_EVICT_LRU ? a.C - p0 : 0;
  cl = cl < 0 ? 0 : (cl > a.c_local ? a.c_local : cl);
  int32_t* onxt = a.order + (static_cast<size_t>((step_b & 1) ^ 1) * a.B + b) * a.C;
  int n_miss_total = a.n_miss[b];
  if (n_miss_total < 0 || n_miss_total > MK || n_miss_total > a.C) n_miss_total = 0;
  if (tid == 0) sh.pub_stamp = 0;
  __syncthreads();
  {
    // stamped slots of my range: the hits (stamped by the selection) and the
    // victims (from the victim list; their last_used is rewritten below)
    int cnt = 0;
    constexpr int U = 8;   // loads in flight per thread
    for (int i0 = tid; i0 < cl; i0 += NT * U) {
      int lu[U];
#pragma unroll
      for (int u = 0; u < U; ++u) lu[u] = (i0 + u * NT < cl) ? a.last_used[bC + p0 + i0 + u * NT] : 0;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * NT;
        if (i < cl) {
          const bool h = lu[u] == step_b;
          cflag[i] = h ? 1 : 0;
          cnt += h ? 1 : 0;
        }
      }
    }
    __syncthreads();
    for (int i = tid; i < n_miss_total; i += NT) {
      const int v = a.vlist[static_cast<size_t>(b) * MK + i];
      if (v >= p0 && v < p0 + cl) {
        cflag[v - p0] = 1;
        ++cnt;
      }
    }
    for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0 && cnt) atomicAdd(&sh.pub_stamp, cnt);
  }
  __syncthreads();
  cluster_sync();  // [L1] every CTA has read last_used; stamped counts published
  if (tid == 0) {
    uint32_t before = 0;
    sh.stamp_total = static_cast<int>(sum_over_cluster(&sh.pub_stamp, rank, &before));
    sh.stamp_before = static_cast<int>(before);
  }
  if (n_miss_total > 0) {
    // pair the i-th miss with the i-th victim, split across the cluster
    const int per = (n_miss_total + CL - 1) / CL;
    const int i0 = static_cast<int>(rank) * per;
    const int i1 = i0 + per < n_miss_total ? i0 + per : n_miss_total;
    for (int i = i0 + tid; i < i1; i += NT) {
      const int v = a.vlist[static_cast<size_t>(b) * MK + i];
      const int t = a.miss_tok[static_cast<size_t>(b) * MK + i];
      if (v < 0 || v >= a.C || t < 0 || t >= Tb) {
        set_status(a.status, ESS_ERR_DEVICE_CHECK);
        continue;
      }
      const int old = a.slot_token[bC + v];
      if (old >= 0 && old < a.T) a.cache_slots[bT + old] = -1;
      a.cache_slots[bT + t] = v;
      a.slot_token[bC + v] = t;
      a.last_used[bC + v] = step_b;
    }
  }
  __syncthreads();
  {
    // stamped slots close the next list in slot order
    const int per_wc = (((cl + NW - 1) / NW) + 31) & ~31;
    const int clo = warp * per_wc;
    const int chi = clo + per_wc < cl ? clo + per_wc : cl;
    int wcnt = 0;
    for (int base = clo; base < chi; base += 32) {
      const int i = base + lane;
      wcnt += __popc(__ballot_sync(0xffffffffu, i < chi && cflag[i]));
    }
    if (lane == 0) sh.wcount[warp] = wcnt;
    __syncthreads();
    int pos = a.C - sh.stamp_total + sh.stamp_before;
    for (int w = 0; w < warp; ++w) pos += sh.wcount[w];
    for (int base = clo; base < chi; base += 32) {
      const int i = base + lane;
      const bool f = i < chi && cflag[i];
      const unsigned bal = __ballot_sync(0xffffffffu, f);
      if (f) {
        const int p = pos + __popc(bal & lt);
        if (p >= 0 && p < a.C) onxt[p] = p0 + i;
      }
      pos += __popc(bal);
    }
  }
  __syncthreads();
  cluster_sync();  // [L2] the stamped counts have been read everywhere
  if (rank == 0 && tid == 0) a.step[b] = step_b + 1;
}

// (a4) victims under the Random, Score and LIM orders ([FO] "evaluation",
// the decode ablation: the same access sequence with only the eviction policy
// changed).  One CTA per request, after the selection kernel has stamped the
// hits and built the miss union.  Candidates are the slots whose token is not
// in the union: empty slots first in slot order, then the resident ones by
// the policy's key (Score: the token's score this step, the maximum over the
// ways; Random: a SplitMix64 draw keyed by (seed, request, step) and the slot;
// LIM: none, i.e. slot order), ties to the lower slot.  The first |Miss| are
// the victims, in that order: an exact radix select finds them, a bitonic
// sort orders them.  Then the paired slots go to miss_slot and into the
// misses' topk_slot entries (~slot), which the selection left as miss indices.
constexpr int kVicThreads = 1024;

__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

struct VicShared {
  unsigned int hist[256];
  int scan[kVicThreads / 32];
  int need;
  unsigned long long prefix, mask;
};

// Shared memory of victim_kernel: the sort buffer (ns entries of key + slot),
// then, when they fit, each slot's class (1 byte) and, for Score, its 32-bit
// key; without them the kernel reads them again from global memory.
struct VicSmem {
  int ns;
  bool cls_cached, key_cached;
  size_t bytes;
};

VicSmem vic_smem(const ess_config& c) {
  VicSmem v;
  const int need = std::min(c.mtp * c.k, c.C);
  v.ns = 1;
  while (v.ns < need) v.ns <<= 1;
  const size_t sort = static_cast<size_t>(v.ns) * 12;
  const size_t budget = kMaxSmemPerCta - sizeof(VicShared) - 1024;
  const size_t cls = (static_cast<size_t>(c.C) + 15) / 16 * 16;
  const size_t key = static_cast<size_t>(c.C) * 4;
  v.cls_cached = sort + cls <= budget;
  v.key_cached = v.cls_cached && sort + cls + key <= budget;
  v.bytes = sort + (v.cls_cached ? cls : 0) + (v.key_cached ? key : 0);
  return v;
}

__global__ void __launch_bounds__(kVicThreads, 1)
    victim_kernel(const SelArgs a, int ns, int cls_cached, int key_cached) {
  pdl_wait_previous();
  pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ VicShared sh;
  unsigned long long* skey = reinterpret_cast<unsigned long long*>(dsm);   // [ns]
  int* sslot = reinterpret_cast<int*>(skey + ns);                          // [ns]
  uint8_t* scls = reinterpret_cast<uint8_t*>(sslot + ns);                  // [C] if cached
  uint32_t* skey32 = reinterpret_cast<uint32_t*>(scls + (a.C + 15) / 16 * 16);  // [C] if cached
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int M = a.M, C = a.C, MK = a.M * a.k;
  const size_t bC = static_cast<size_t>(b) * C;
  const int step_b = a.step[b];
  int n = a.n_miss[b];
  if (n < 0 || n > MK || n > C) n = 0;
  int32_t* vl = a.vlist + static_cast<size_t>(b) * MK;
  const bool score = a.policy == ESS_EVICT_SCORE, random = a.policy == ESS_EVICT_RANDOM;
  // slots [s0, s1) belong to this thread, in slot order across threads
  const int per = (C + kVicThreads - 1) / kVicThreads;
  const int s0 = tid * per < C ? tid * per : C;
  const int s1 = s0 + per < C ? s0 + per : C;
  const unsigned long long rkey =
      mix64((mix64((a.seed ^ static_cast<unsigned long long>(b)) + 0x9E3779B97F4A7C15ULL) ^
             static_cast<unsigned long long>(step_b)) + 0x9E3779B97F4A7C15ULL);
  // class of a slot from global memory: 0 not a candidate (its token is in the
  // union: stamped this step), 1 empty, 2 resident; and a resident's key
  auto classify_global = [&](int sl, unsigned long long& key) -> int {
    if (a.last_used[bC + sl] == step_b) return 0;
    const int t = a.slot_token[bC + sl];
    if (t < 0) return 1;
    if (score) {
      float best = a.scores[(static_cast<size_t>(b) * M) * a.T + t];
      for (int m = 1; m < M; ++m)
        best = fmaxf(best, a.scores[(static_cast<size_t>(b) * M + m) * a.T + t]);
      key = float_key(best + 0.0f);
    } else if (random) {
      key = mix64(rkey + static_cast<unsigned long long>(sl + 1) * 0x9E3779B97F4A7C15ULL);
    } else {
      key = 0;   // LIM: slot order
    }
    return 2;
  };
  auto classify = [&](int sl, unsigned long long& key) -> int {
    if (!cls_cached) return classify_global(sl, key);
    const int c = scls[sl];
    if (c == 2) {
      if (score) {
        if (key_cached) key = skey32[sl];
        else classify_global(sl, key);
      } else if (random) {
        key = mix64(rkey + static_cast<unsigned long long>(sl + 1) * 0x9E3779B97F4A7C15ULL);
      } else {
        key = 0;
      }
    }
    return c;
  };
  // exclusive prefix over threads of v (block-wide), total in tot
  auto bscan = [&](int v, int& tot) -> int {
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) sh.scan[warp] = x;
    __syncthreads();
    int pre = 0, t = 0;
    for (int i = 0; i < kVicThreads / 32; ++i) {
      const int u = sh.scan[i];
      pre += i < warp ? u : 0;
      t += u;
    }
    tot = t;
    return pre + x - v;
  };
  // one pass from global memory: classes (and Score keys) into shared memory,
  // eight slots' loads in flight at a time; and the count of empty slots
  int ne = 0;
  for (int g = s0; g < s1; g += 8) {
    int lu[8], tk[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      lu[u] = g + u < s1 ? a.last_used[bC + g + u] : step_b;
      tk[u] = g + u < s1 ? a.slot_token[bC + g + u] : -1;
    }
    float best[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      best[u] = 0.0f;
      if (score && lu[u] != step_b && tk[u] >= 0) {
        best[u] = a.scores[(static_cast<size_t>(b) * M) * a.T + tk[u]];
        for (int m = 1; m < M; ++m)
          best[u] = fmaxf(best[u], a.scores[(static_cast<size_t>(b) * M + m) * a.T + tk[u]]);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (g + u >= s1) break;
      const int c = lu[u] == step_b ? 0 : (tk[u] < 0 ? 1 : 2);
      ne += c == 1 ? 1 : 0;
      if (cls_cached) scls[g + u] = static_cast<uint8_t>(c);
      if (key_cached) skey32[g + u] = float_key(best[u] + 0.0f);
    }
  }
  __syncthreads();
  // empty candidates come first, in slot order
  int E;
  int pe = bscan(ne, E);
  for (int sl = s0; sl < s1 && pe < n; ++sl) {
    unsigned long long k;
    if (classify(sl, k) == 1) vl[pe++] = sl;
  }
  const int R = n > E ? n - E : 0;   // resident victims
  if (R > 0) {
    // exact radix select, smallest first, 8-bit digits from the top of the key
    const int nbits = random ? 64 : (score ? 32 : 0);
    if (tid == 0) {
      sh.prefix = 0;
      sh.mask = 0;
      sh.need = R;
    }
    __syncthreads();   // (LIM has no pass that would synchronise before the reads below)
    for (int hi = nbits; hi > 0; hi -= 8) {
      const int lo = hi - 8;
      for (int i = tid; i < 256; i += kVicThreads) sh.hist[i] = 0;
      __syncthreads();
      const unsigned long long pre = sh.prefix, msk = sh.mask;
      for (int sl = s0; sl < s1; ++sl) {
        unsigned long long k = 0;
        if (classify(sl, k) == 2 && (k & msk) == pre) atomicAdd(&sh.hist[(k >> lo) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 8l..8l+7 (ascending)
        int c8[8], s8 = 0;
        for (int j = 0; j < 8; ++j) {
          c8[j] = static_cast<int>(sh.hist[8 * lane + j]);
          s8 += c8[j];
        }
        int incl = s8;
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int need = sh.need;
        const int excl = incl - s8;
        if (excl < need && need <= incl) {
          int acc = excl, j = 0;
          for (; j < 7; ++j) {
            if (acc + c8[j] >= need) break;
            acc += c8[j];
          }
          sh.prefix = pre | (static_cast<unsigned long long>(8 * lane + j) << lo);
          sh.mask = msk | (255ULL << lo);
          sh.need = need - acc;
        }
      }
      __syncthreads();
    }
    // residents below the threshold key, and the lowest-slot equal ones
    const unsigned long long thr = sh.prefix;
    const int take_eq = sh.need;
    int nlt = 0, neq = 0;
    for (int sl = s0; sl < s1; ++sl) {
      unsigned long long k = 0;
      if (classify(sl, k) == 2) {
        nlt += k < thr ? 1 : 0;
        neq += k == thr ? 1 : 0;
      }
    }
    int tot_lt, tot_eq;
    int plt = bscan(nlt, tot_lt);
    int peq = bscan(neq, tot_eq);
    for (int sl = s0; sl < s1; ++sl) {
      unsigned long long k = 0;
      if (classify(sl, k) != 2) continue;
      int pos = -1;
      if (k < thr) pos = plt++;
      else if (k == thr && peq < take_eq) pos = tot_lt + peq++;
      if (pos >= 0 && pos < ns) {
        skey[pos] = k;
        sslot[pos] = sl;
      }
    }
    if (tid == 0 && (tot_lt + take_eq != R || R > ns)) set_status(a.status, ESS_ERR_DEVICE_CHECK);
    // bitonic sort of the R victims by (key, slot), padded to a power of two
    int N = 1;
    while (N < R) N <<= 1;
    if (N > ns) N = ns;
    for (int i = R + tid; i < N; i += kVicThreads) {
      skey[i] = ~0ULL;
      sslot[i] = 0x7fffffff;
    }
    __syncthreads();
    for (int kk = 2; kk <= N; kk <<= 1) {
      for (int j = kk >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < N; i += kVicThreads) {
          const int l = i ^ j;
          if (l > i) {
            const bool up = (i & kk) == 0;
            const unsigned long long ki = skey[i], kl = skey[l];
            const int si = sslot[i], sl2 = sslot[l];
            const bool gt = ki > kl || (ki == kl && si > sl2);
            if (gt == up) {
              skey[i] = kl;
              skey[l] = ki;
              sslot[i] = sl2;
              sslot[l] = si;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int i = tid; i < R && i < N; i += kVicThreads) vl[E + i] = sslot[i];
  }
  __syncthreads();
  // the paired slots: copy triples and the misses' slot entries
  for (int i = tid; i < n; i += kVicThreads) a.miss_slot[static_cast<size_t>(b) * MK + i] = vl[i];
  for (int m = 0; m < M; ++m) {
    const size_t wo = (static_cast<size_t>(b) * M + m) * a.k;
    const int nm = a.n_miss_way[b * M + m];
    for (int e = tid; e < nm && e < a.k; e += kVicThreads) {
      const int mi = -2 - a.topk_slot[wo + e];
      if (mi < 0 || mi >= n) {
        set_status(a.status, ESS_ERR_DEVICE_CHECK);
        continue;
      }
      a.topk_slot[wo + e] = ~vl[mi];
    }
  }
  if (a.ready != nullptr) {
    __syncthreads();
    if (tid == 0) count_done(a.ready + b * kCounterStride, kSelCluster);
  }
}

__global__ void order_reset_kernel(int32_t* order, int n_per_list, int C) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < 2 * n_per_list) order[i] = (i % n_per_list) % C;
}

}  // namespace

cudaError_t launch_order_reset(const ess_pool& p, int layer, cudaStream_t st) {
  const ess_config& c = p.cfg;
  const int n = c.batch * c.C;
  order_reset_kernel<<<(2 * n + 255) / 256, 256, 0, st>>>(p.layers[layer].order, n, c.C);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch(p);
  return e;
}

namespace {

// Shared-memory sizes of the selection kernel for a largest request length
// T_hmax: the per-CTA token range, the list capacities, and the bytes of the
// lists (fixed) and of the staged scores (res_bytes).
struct SelSizes {
  int nl, c_local, lcap, gcap;
  size_t res_bytes, fixed;
};

constexpr size_t kSelKeysBudget = 160 * 1024;   // leaves room for the static shared state

SelSizes sel_sizes(const ess_config& c, int T_hmax) {
  SelSizes z;
  z.nl = (T_hmax + CL - 1) / CL;
  z.nl = ((z.nl + 3) / 4) * 4;
  if (z.nl < 4) z.nl = 4;
  // slots per CTA: a multiple of 128, so that each CTA's range of the stamp
  // bitmap is whole 16-byte units of words
  z.c_local = ((c.C + CL - 1) / CL + 127) / 128 * 128;
  const int MK = c.mtp * c.k;
  z.lcap = z.nl < MK ? z.nl : MK;   // the union of one CTA's tokens never exceeds this
  z.lcap = (z.lcap + 3) / 4 * 4;    // keeps the arrays after the list 16-byte aligned
  z.gcap = 4096;
  z.res_bytes = static_cast<size_t>(c.mtp) * z.nl * 4;
  // lists, the LRU slice, candidate keys, gathered keys and ranks, and the
  // stamp bitmap words (own range, all ranges, unstamped masks)
  z.fixed = static_cast<size_t>(z.lcap) * (9 + 4 * c.mtp) + static_cast<size_t>(z.c_local) * 4 +
            static_cast<size_t>(z.gcap) * 5 + static_cast<size_t>(z.c_local / 32) * (CL + 2) * 4 +
            64;
  return z;
}

}  // namespace

// Largest shared memory (static + dynamic) one selection CTA can ask for over
// every request length up to max_T: the lists grow with the length, and the
// staged scores are used only while they fit the budget.
size_t select_smem_need(const ess_config& c) {
  const SelSizes z = sel_sizes(c, c.max_T);
  return sizeof(SelShared) + (z.fixed > kSelKeysBudget ? z.fixed : kSelKeysBudget);
}

cudaError_t launch_select(const ess_pool& p, int layer, const float* scores, bool hist_given,
                          int32_t* topk_idx, int32_t* topk_slot, int32_t* n_miss_way,
                          int32_t* miss_tok, int32_t* miss_slot, int32_t* n_miss, cudaStream_t st) {
  const ess_config& c = p.cfg;
  const Layer& L = p.layers[layer];
  SelArgs a;
  a.scores = scores;
  a.ghist = p.scr.ghist;
  a.hist_given = hist_given ? 1 : 0;
  a.guess = hist_given ? L.guess : nullptr;
  a.fhist = p.scr.fhist;
  a.tflag = hist_given ? p.scr.tflag : nullptr;
  a.nwords = p.scr.nwords;
  a.cache_slots = L.cache_slots;
  a.slot_token = L.slot_token;
  a.last_used = L.last_used;
  a.step = L.step;
  a.order = L.order;
  a.Tb = L.T_dev;
  a.topk_idx = topk_idx;
  a.topk_slot = topk_slot;
  a.n_miss_way = n_miss_way;
  a.miss_tok = miss_tok;
  a.miss_slot = miss_slot;
  a.n_miss = n_miss;
  a.vlist = p.scr.vlist;
  a.host = reinterpret_cast<const uint8_t*>(L.host_latent);
  a.page_table = L.page_table;
  a.T0 = L.T0_dev;
  a.page = c.page;
  a.row_bytes = L.compact ? kCompactRowBytes : kRowBytes;
  a.stats = L.stats;
  a.status = p.scr.status;
  a.B = c.batch;
  a.M = c.mtp;
  a.k = c.k;
  a.T = c.max_T;
  a.C = c.C;
  a.policy = p.evict_policy;
  a.seed = p.evict_seed;
  a.ready = p.scr.ready;
  a.attn_done = p.scr.attn_done;
  const SelSizes z = sel_sizes(c, L.T_hmax);
  a.n_local = z.nl;
  a.c_local = z.c_local;
  a.lcap = z.lcap;
  a.gcap = z.gcap;
  const size_t res_bytes = z.res_bytes;
  const size_t fixed = z.fixed;
  a.resident = (res_bytes + fixed <= kSelKeysBudget) ? 1 : 0;
  size_t kb = a.resident ? res_bytes : 0;
  kb = (kb + 15) / 16 * 16;
  a.keys_bytes = static_cast<uint32_t>(kb);
  const size_t smem = kb + fixed;
  void (*kern)(SelArgs) = c.mtp == 1 ? select_kernel<1>
                        : c.mtp == 2 ? select_kernel<2>
                        : c.mtp == 3 ? select_kernel<3>
                                     : select_kernel<4>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(c.batch * CL), dim3(NT), smem, st, a);
  if (e != cudaSuccess) return e;
  count_launch(p);
  if (a.policy != ESS_EVICT_LRU) {
    const VicSmem v = vic_smem(c);
    e = cudaFuncSetAttribute(victim_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(v.bytes));
    if (e != cudaSuccess) return e;
    e = launch_pdl(victim_kernel, dim3(c.batch), dim3(kVicThreads), v.bytes, st, a, v.ns,
                   v.cls_cached ? 1 : 0, v.key_cached ? 1 : 0);
    if (e != cudaSuccess) return e;
    count_launch(p);
  }
  const size_t smem_b = (static_cast<size_t>(a.c_local) + 15) / 16 * 16;
  e = cudaFuncSetAttribute(lru_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_b));
  if (e != cudaSuccess) return e;
  e = launch_pdl(lru_finish_kernel, dim3(c.batch * CL), dim3(NT), smem_b, st, a);
  if (e == cudaSuccess) count_launch(p);
  return e;
}

// ---------------------------------------------------------------------------
// Selection whose scratch needs no allocation by the caller.
//
// For callers that cannot allocate device memory when they select: an engine
// that hands out all of its device memory at start-up, or a thread on which an
// allocation would synchronise the device and stall decoding.  The selection
// kernel needs two scratch buffers besides its inputs, outputs and the pool
// state: the per-(request, way) score histogram and the victim list.  This
// variant takes them from a fixed array compiled into the library instead of
// the pool's workspace.  Every GPU that loads the library holds the array
// until the process exits; every call shares it, so calls that overlap on the
// GPU race.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kSelectStaticScratchBytes = size_t(2) << 20;  // 2 MiB

static __device__ __align__(256) unsigned char g_select_scratch[kSelectStaticScratchBytes];

// Device address of g_select_scratch, looked up once per device (the name is
// only a host-side stand-in for the device array).
std::mutex g_scratch_mu;
void* g_scratch_addr[128] = {nullptr};

// dev must be the current device: the lookup returns the current device's copy.
cudaError_t select_scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  cudaError_t e;
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

size_t align256_sz(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace
}  // namespace ess

extern "C" ess_status ess_select_manage_noalloc(ess_pool* pool, int layer, const float* scores,
                                                int32_t* topk_idx, int32_t* topk_slot,
                                                int32_t* n_miss_way, int32_t* miss_tok,
                                                int32_t* miss_slot, int32_t* n_miss,
                                                ess_stream_t stream) {
  using namespace ess;
  if (!pool || layer < 0 || layer >= pool->cfg.n_layers || !pool->layers[layer].bound ||
      !scores || !topk_idx || !topk_slot || !n_miss_way || !miss_tok || !miss_slot || !n_miss ||
      (reinterpret_cast<uintptr_t>(scores) & 15u))
    return ESS_ERR_INVALID_ARG;
  const ess_config& c = pool->cfg;
  const size_t bm = static_cast<size_t>(c.batch) * c.mtp;
  const size_t hist_bytes = align256_sz(bm * kHistBins * sizeof(uint32_t));
  const size_t vlist_bytes = align256_sz(bm * c.k * sizeof(int32_t));
  if (hist_bytes + vlist_bytes > kSelectStaticScratchBytes) return ESS_ERR_OOM;
  // the array is looked up (and later used) on the pool's device, which must be
  // the current one, as for every call on the pool
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return ESS_ERR_CUDA;
  if (cur != pool->device) return ESS_ERR_INVALID_ARG;
  void* base = nullptr;
  if (select_scratch_address(pool->device, &base) != cudaSuccess) return ESS_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the histogram is accumulated with atomics, so it must start at zero
  if (cudaMemsetAsync(base, 0, hist_bytes, st) != cudaSuccess) return ESS_ERR_CUDA;
  ess_pool view = *pool;  // same layers and state; only the two scratch buffers differ
  view.scr.ghist = static_cast<uint32_t*>(base);
  view.scr.vlist = reinterpret_cast<int32_t*>(static_cast<char*>(base) + hist_bytes);
  const cudaError_t e = launch_select(view, layer, scores, false, topk_idx, topk_slot, n_miss_way,
                                      miss_tok, miss_slot, n_miss, st);
  return e == cudaSuccess ? ESS_OK : ESS_ERR_CUDA;
}
