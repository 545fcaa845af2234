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
// [r*n_local, (r+1)*n_local) and slots [r*c_local, (r+1)*c_local).  The top-k
// threshold is found exactly by MSB-first radix passes whose per-CTA
// histograms are summed through distributed shared memory; ties at the
// threshold go to the lowest token (lowest slot for victims).  All lists
// come out in ascending token order, which fixes the pairing of the i-th
// miss with the i-th victim in (last_used, slot) order.
#include "ess_device.cuh"

namespace ess {
namespace {

constexpr int CL = kSelCluster;
constexpr int NT = kSelThreads;
constexpr int NW = NT / 32;

struct SelArgs {
  const float* scores;        // [B][M][T]
  int32_t* cache_slots;       // [B][T]
  int32_t* slot_token;        // [B][C]
  int32_t* last_used;         // [B][C]
  int32_t* step;              // [B]
  const int32_t* Tb;          // [B]
  int32_t* topk_idx;          // [B][M][k]
  int32_t* topk_slot;         // [B][M][k]
  int32_t* n_miss_way;        // [B][M]
  int32_t* miss_tok;          // [B][M*k]
  int32_t* miss_slot;         // [B][M*k]
  int32_t* n_miss;            // [B]
  unsigned long long* vict;   // [B][M*k]
  long long* stats;           // [kStatFields]
  int* status;
  int B, M, k, T, C;
  int n_local;                // tokens per CTA (multiple of 4)
  int c_local;                // slots per CTA
  int resident;               // scores staged in shared memory
  int ucap;                   // union-list capacity per CTA
  uint32_t keys_bytes;        // size of the keys / sort region
};

struct SelShared {
  uint32_t hist[2][kMaxWays * 256];
  uint32_t tot[kMaxWays * 256];
  int scanbuf[2][NW];
  uint32_t prefix[kMaxWays], selmask[kMaxWays];
  int remaining[kMaxWays], eq_local[kMaxWays], eq_before[kMaxWays], eq_total[kMaxWays];
  int active[kMaxWays], quota[kMaxWays], rank_needed[kMaxWays], eq_run[kMaxWays];
  int last_lo, last_dmask;
  int nu;
  // published for the other CTAs of the cluster (read through DSMEM)
  int pub_nmiss, pub_nu, pub_hit[kMaxWays], pub_miss[kMaxWays];
  int pub_lumin, pub_lumax, pub_vcnt;
  // cluster-wide values derived from the publications
  int n_miss_total, nu_total, miss_off, hit_off[kMaxWays], wmiss_off[kMaxWays], nmw[kMaxWays];
  int hits_total[kMaxWays];
  int lu_min, lu_max, vict_off;
  int step_b;
  unsigned long long bar;
  int abort;
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

__device__ __forceinline__ uint32_t sum_over_cluster(const void* local, uint32_t upto_rank,
                                                     uint32_t* before) {
  const uint32_t a = smem_u32(local);
  uint32_t s = 0, b = 0;
  for (uint32_t r = 0; r < CL; ++r) {
    const uint32_t v = ld_dsmem_u32(dsmem_addr(a, r));
    if (r < upto_rank) b += v;
    s += v;
  }
  if (before) *before = b;
  return s;
}

// Cluster-wide exact selection of the remaining[m] largest keys (keys <
// 2^nbits) per active way; elements of rank r precede those of rank r+1, and
// equal keys go to the lowest element.  Leaves prefix[m] (threshold key),
// remaining[m] (how many threshold-equal elements to take, lowest first) and
// eq_local / eq_before / eq_total of threshold-equal elements.
// Precondition: a cluster_sync separates this call from any earlier remote
// read of sh.hist.
template <class KeyFn>
__device__ void cluster_select(KeyFn keyf, int n_valid, int nw, int nbits, SelShared& sh,
                               uint32_t rank) {
  const int tid = threadIdx.x;
  if (tid < kMaxWays) {
    sh.prefix[tid] = 0;
    sh.selmask[tid] = 0;
  }
  for (int i = tid; i < 2 * kMaxWays * 256; i += NT) (&sh.hist[0][0])[i] = 0;
  __syncthreads();
  const int passes = (nbits + 7) / 8;
  for (int p = 0; p < passes; ++p) {
    const int hi = nbits - 8 * p;
    const int lo = hi - 8 > 0 ? hi - 8 : 0;
    const uint32_t dmask = (hi - lo >= 32) ? 0xffffffffu : ((1u << (hi - lo)) - 1u);
    uint32_t* H = sh.hist[p & 1];
    for (int m = 0; m < nw; ++m) {
      if (!sh.active[m]) continue;
      const uint32_t pre = sh.prefix[m], msk = sh.selmask[m];
      for (int base = 0; base < n_valid; base += NT) {
        const int i = base + tid;
        bool ok = i < n_valid;
        const uint32_t key = ok ? keyf(m, i) : 0u;
        ok = ok && ((key & msk) == pre);
        hist_add_warp(H + m * 256, (key >> lo) & dmask, ok);
      }
    }
    __syncthreads();
    cluster_sync();
    for (int i = tid; i < nw * 256; i += NT) {
      if (!sh.active[i >> 8]) continue;
      sh.tot[i] = sum_over_cluster(&H[i], 0, nullptr);
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < nw && sh.active[warp]) {
      const int m = warp;
      const int need = sh.remaining[m];
      int c8[8];
      int s8 = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c8[j] = static_cast<int>(sh.tot[m * 256 + 255 - 8 * lane - j]);
        s8 += c8[j];
      }
      int incl = s8;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned bal = __ballot_sync(0xffffffffu, incl >= need);
      const int L = bal ? __ffs(bal) - 1 : 31;
      if (lane == L) {
        int acc = incl - s8;
        int j = 0;
        for (; j < 7; ++j) {
          if (acc + c8[j] >= need) break;
          acc += c8[j];
        }
        const uint32_t digit = static_cast<uint32_t>(255 - 8 * L - j);
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
      for (int i = tid; i < kMaxWays * 256; i += NT) sh.hist[(p + 1) & 1][i] = 0;
    __syncthreads();
  }
  if (passes > 0 && tid < nw && sh.active[tid]) {
    const int m = tid;
    const uint32_t dig = (sh.prefix[m] >> sh.last_lo) & static_cast<uint32_t>(sh.last_dmask);
    const uint32_t* h = &sh.hist[(passes - 1) & 1][m * 256 + dig];
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
    sh.eq_run[m] = 0;
  }
}

__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(NT, 1)
    select_kernel(const SelArgs a) {
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ SelShared sh;
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_ctarank();
  const int b = blockIdx.x / CL;
  const int M = a.M;
  const int MK = M * a.k;
  const int Tb = a.Tb[b];
  const int keff = a.k < Tb ? a.k : Tb;
  const int r0 = static_cast<int>(rank) * a.n_local;
  int nloc = Tb - r0;
  nloc = nloc < 0 ? 0 : (nloc > a.n_local ? a.n_local : nloc);
  float* keys_s = reinterpret_cast<float*>(dsm);                        // [M][n_local] or sort buffer
  int* lu_s = reinterpret_cast<int*>(dsm + a.keys_bytes);               // [c_local]
  int* utok = lu_s + a.c_local;                                         // [ucap]
  int* uslot = utok + a.ucap;                                           // [ucap]
  uint8_t* umask = reinterpret_cast<uint8_t*>(uslot + a.ucap);          // [ucap]
  const size_t bT = static_cast<size_t>(b) * a.T;
  const size_t bC = static_cast<size_t>(b) * a.C;
  int parity = 0;

  if (tid == 0) {
    sh.step_b = a.step[b];
    sh.nu = 0;
    sh.abort = 0;
    sh.pub_nmiss = 0;
    sh.pub_nu = 0;
    sh.pub_vcnt = 0;
    for (int m = 0; m < kMaxWays; ++m) {
      sh.pub_hit[m] = 0;
      sh.pub_miss[m] = 0;
      sh.active[m] = 0;
    }
    mbar_init(smem_u32(&sh.bar), 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---------------------------------------------------------------- scores
  if (a.resident && nloc > 0) {
    const int cnt = ((nloc + 3) / 4) * 4 <= a.T - r0 ? ((nloc + 3) / 4) * 4 : a.T - r0;
    if (tid == 0) {
      mbar_arrive_expect_tx(smem_u32(&sh.bar), static_cast<uint32_t>(cnt * 4 * M));
      for (int m = 0; m < M; ++m)
        bulk_load(smem_u32(keys_s + m * a.n_local),
                  a.scores + (static_cast<size_t>(b) * M + m) * a.T + r0,
                  static_cast<uint32_t>(cnt * 4), smem_u32(&sh.bar));
    }
    if (!mbar_wait(smem_u32(&sh.bar), 0, nullptr)) {
      set_status(a.status, ESS_ERR_TIMEOUT);
      sh.abort = 1;
    }
  }
  const float* gscores = a.scores + static_cast<size_t>(b) * M * a.T + r0;
  auto score_key = [&](int m, int i) -> uint32_t {
    const float f = a.resident ? keys_s[m * a.n_local + i] : gscores[static_cast<size_t>(m) * a.T + i];
    return float_key(f);
  };

  // ---------------------------------------------------------------- (a2) top-k
  const bool sel_all = keff >= Tb;  // every token is selected (includes T_b = 0)
  if (tid < M) {
    sh.active[tid] = sel_all ? 0 : 1;
    sh.remaining[tid] = keff;
  }
  __syncthreads();
  if (!sel_all) {
    cluster_select(score_key, nloc, M, 32, sh, rank);
    set_quota(sh, M);
    __syncthreads();
  }
  // ordered compaction of the union of the ways' selections into utok/umask
  {
    int nu = 0;
    int eqrun[kMaxWays] = {0, 0, 0, 0};  // threshold-equal elements seen so far (same in all threads)
    for (int base = 0; base < nloc; base += NT * 4) {
      const int i0 = base + tid * 4;
      uint32_t selbits[4] = {0, 0, 0, 0};
      for (int m = 0; m < M; ++m) {
        uint32_t key[4];
        bool valid[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          valid[j] = (i0 + j) < nloc;
          key[j] = valid[j] ? score_key(m, i0 + j) : 0u;
        }
        if (sel_all) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (valid[j]) selbits[j] |= 1u << m;
          continue;
        }
        const uint32_t thr = sh.prefix[m];
        bool eq[4];
        int neq = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          eq[j] = valid[j] && key[j] == thr;
          neq += eq[j];
          if (valid[j] && key[j] > thr) selbits[j] |= 1u << m;
        }
        if (sh.rank_needed[m]) {  // uniform
          int tot;
          int r = block_scan(neq, tot, sh, parity);
          r += eqrun[m];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (eq[j]) {
              if (r < sh.quota[m]) selbits[j] |= 1u << m;
              ++r;
            }
          eqrun[m] += tot;
        } else if (sh.quota[m] > 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (eq[j]) selbits[j] |= 1u << m;
        }
      }
      int cu = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) cu += selbits[j] ? 1 : 0;
      int tot;
      int pos = nu + block_scan(cu, tot, sh, parity);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (selbits[j]) {
          if (pos < a.ucap) {
            utok[pos] = r0 + i0 + j;
            umask[pos] = static_cast<uint8_t>(selbits[j]);
          } else {
            set_status(a.status, ESS_ERR_DEVICE_CHECK);
          }
          ++pos;
        }
      nu += tot;
    }
    if (tid == 0) sh.nu = nu < a.ucap ? nu : a.ucap;
    __syncthreads();
  }
  const int nu = sh.nu;

  // ---------------------------------------------------------------- (a3) resolve
  for (int e = tid; e < nu; e += NT) {
    const int t = utok[e];
    int s = a.cache_slots[bT + t];
    if (s >= a.C || s < -1) {
      set_status(a.status, ESS_ERR_DEVICE_CHECK);
      s = -1;
    }
    uslot[e] = s;
    if (s >= 0) a.last_used[bC + s] = sh.step_b;   // hits are stamped first
    const uint32_t mk = umask[e];
    for (int m = 0; m < M; ++m)
      if (mk & (1u << m)) atomicAdd(s >= 0 ? &sh.pub_hit[m] : &sh.pub_miss[m], 1);
    if (s < 0) atomicAdd(&sh.pub_nmiss, 1);
  }
  if (tid == 0) sh.pub_nu = nu;
  __threadfence();
  __syncthreads();
  cluster_sync();  // (1) per-CTA counts published
  if (tid == 0) {
    uint32_t before = 0;
    sh.n_miss_total = static_cast<int>(sum_over_cluster(&sh.pub_nmiss, rank, &before));
    sh.miss_off = static_cast<int>(before);
    sh.nu_total = static_cast<int>(sum_over_cluster(&sh.pub_nu, rank, nullptr));
  }
  if (tid < M) {
    uint32_t before = 0;
    sh.nmw[tid] = static_cast<int>(sum_over_cluster(&sh.pub_miss[tid], rank, &before));
    sh.wmiss_off[tid] = static_cast<int>(before);
    sh.hits_total[tid] = static_cast<int>(sum_over_cluster(&sh.pub_hit[tid], rank, &before));
    sh.hit_off[tid] = static_cast<int>(before);
  }
  __syncthreads();
  const int n_miss_total = sh.n_miss_total;
  if (n_miss_total > a.C || n_miss_total > MK) {  // cannot happen when C >= min(M*k, T)
    if (tid == 0) set_status(a.status, ESS_ERR_CAPACITY);
  }
  // (2) the miss union in ascending token order
  {
    int run = sh.miss_off;
    for (int base = 0; base < nu; base += NT) {
      const int e = base + tid;
      const bool f = e < nu && uslot[e] < 0;
      int tot;
      const int pos = run + block_scan(f ? 1 : 0, tot, sh, parity);
      if (f && pos < MK) a.miss_tok[static_cast<size_t>(b) * MK + pos] = utok[e];
      run += tot;
    }
  }
  __threadfence();
  __syncthreads();
  cluster_sync();  // (2) stamps and miss list visible

  // ---------------------------------------------------------------- (a4) LRU victims
  const bool do_victims = n_miss_total > 0 && n_miss_total <= a.C && n_miss_total <= MK;
  if (do_victims) {
    const int s0 = static_cast<int>(rank) * a.c_local;
    int cl = a.C - s0;
    cl = cl < 0 ? 0 : (cl > a.c_local ? a.c_local : cl);
    int mn = 0x7fffffff, mx = -0x7fffffff - 1;
    for (int i = tid; i < cl; i += NT) {
      const int v = a.last_used[bC + s0 + i];
      lu_s[i] = v;
      mn = v < mn ? v : mn;
      mx = v > mx ? v : mx;
    }
    for (int o = 16; o; o >>= 1) {
      mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (tid == 0) {
      sh.pub_lumin = 0x7fffffff;
      sh.pub_lumax = -0x7fffffff - 1;
    }
    __syncthreads();
    if ((tid & 31) == 0) {
      atomicMin(&sh.pub_lumin, mn);
      atomicMax(&sh.pub_lumax, mx);
    }
    __syncthreads();
    cluster_sync();  // (3)
    if (tid == 0) {
      int gmn = 0x7fffffff, gmx = -0x7fffffff - 1;
      for (uint32_t r = 0; r < CL; ++r) {
        gmn = min(gmn, static_cast<int>(ld_dsmem_u32(dsmem_addr(smem_u32(&sh.pub_lumin), r))));
        gmx = max(gmx, static_cast<int>(ld_dsmem_u32(dsmem_addr(smem_u32(&sh.pub_lumax), r))));
      }
      sh.lu_min = gmn;
      sh.lu_max = gmx;
      sh.active[0] = n_miss_total < a.C ? 1 : 0;
      for (int m = 1; m < kMaxWays; ++m) sh.active[m] = 0;
      sh.remaining[0] = n_miss_total;
    }
    __syncthreads();
    const int lu_max = sh.lu_max;
    const uint32_t range = static_cast<uint32_t>(lu_max - sh.lu_min);
    const int nbits = range == 0 ? 0 : 32 - __clz(static_cast<int>(range));
    // larger key = older slot; equal keys go to the lowest slot
    auto lu_key = [&](int, int i) -> uint32_t { return static_cast<uint32_t>(lu_max - lu_s[i]); };
    const bool take_all = !sh.active[0];
    if (!take_all) {
      if (nbits > 0) {
        cluster_select(lu_key, cl, 1, nbits, sh, rank);
      } else {
        if (tid == 0) {
          sh.prefix[0] = 0;
          sh.eq_local[0] = cl;
          const int bef = s0 < a.C ? s0 : a.C;
          sh.eq_before[0] = bef;
          sh.eq_total[0] = a.C;
        }
        __syncthreads();
      }
      set_quota(sh, 1);
      __syncthreads();
    }
    // victims in slot order: count, exchange, write
    const uint32_t thr = sh.prefix[0];
    int vcnt = 0;
    for (int base = 0; base < cl; base += NT) {
      const int i = base + tid;
      int f = 0;
      if (i < cl) f = take_all ? 1 : (lu_key(0, i) > thr ? 1 : 0);
      vcnt += f;
    }
    for (int o = 16; o; o >>= 1) vcnt += __shfl_xor_sync(0xffffffffu, vcnt, o);
    if ((tid & 31) == 0) atomicAdd(&sh.pub_vcnt, vcnt);
    __syncthreads();
    if (tid == 0 && !take_all) sh.pub_vcnt += sh.quota[0];
    __syncthreads();
    cluster_sync();  // (4)
    if (tid == 0) {
      uint32_t before = 0;
      sum_over_cluster(&sh.pub_vcnt, rank, &before);
      sh.vict_off = static_cast<int>(before);
    }
    __syncthreads();
    {
      int run = sh.vict_off;
      int eqr = 0;
      for (int base = 0; base < cl; base += NT) {
        const int i = base + tid;
        bool f = false;
        if (i < cl) {
          if (take_all) {
            f = true;
          } else {
            const uint32_t kk = lu_key(0, i);
            if (kk > thr) f = true;
          }
        }
        bool e = false;
        if (!take_all && i < cl && lu_key(0, i) == thr) e = true;
        if (!take_all && sh.rank_needed[0]) {
          int tot;
          const int r = eqr + block_scan(e ? 1 : 0, tot, sh, parity);
          if (e && r < sh.quota[0]) f = true;
          eqr += tot;
        } else if (!take_all && e && sh.quota[0] > 0) {
          f = true;
        }
        int tot;
        const int pos = run + block_scan(f ? 1 : 0, tot, sh, parity);
        if (f && pos < MK) {
          const int slot = s0 + i;
          const uint32_t lub = static_cast<uint32_t>(lu_s[i]) ^ 0x80000000u;
          a.vict[static_cast<size_t>(b) * MK + pos] =
              (static_cast<unsigned long long>(lub) << 32) | static_cast<uint32_t>(slot);
        }
        run += tot;
      }
    }
    __threadfence();
    __syncthreads();
    cluster_sync();  // (5) victims gathered
    if (rank == 0) {
      // sort the victims by (last_used, slot) and pair them with the misses
      unsigned long long* sb = reinterpret_cast<unsigned long long*>(keys_s);
      const int n = n_miss_total;
      int np2 = 1;
      while (np2 < n) np2 <<= 1;
      for (int i = tid; i < np2; i += NT)
        sb[i] = i < n ? a.vict[static_cast<size_t>(b) * MK + i] : ~0ull;
      __syncthreads();
      for (int kk = 2; kk <= np2; kk <<= 1) {
        for (int jj = kk >> 1; jj > 0; jj >>= 1) {
          for (int i = tid; i < np2; i += NT) {
            const int ix = i ^ jj;
            if (ix > i) {
              const unsigned long long x = sb[i], y = sb[ix];
              const bool up = (i & kk) == 0;
              if ((x > y) == up) {
                sb[i] = y;
                sb[ix] = x;
              }
            }
          }
          __syncthreads();
        }
      }
      const int step_b = sh.step_b;
      for (int i = tid; i < n; i += NT) {
        const int v = static_cast<int>(sb[i] & 0xffffffffu);
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
        a.miss_slot[static_cast<size_t>(b) * MK + i] = v;
      }
    }
    __threadfence();
    __syncthreads();
    cluster_sync();  // (6) new slots visible
  }

  // ---------------------------------------------------------------- emit per-way lists
  for (int m = 0; m < M; ++m) {
    int runm = sh.wmiss_off[m];
    int runh = sh.nmw[m] + sh.hit_off[m];
    const size_t wo = (static_cast<size_t>(b) * M + m) * a.k;
    for (int base = 0; base < nu; base += NT) {
      const int e = base + tid;
      bool fm = false, fh = false;
      int t = 0, s = -1;
      if (e < nu && (umask[e] & (1u << m))) {
        t = utok[e];
        s = uslot[e];
        fm = s < 0;
        fh = !fm;
      }
      int totm, toth;
      const int pm = runm + block_scan(fm ? 1 : 0, totm, sh, parity);
      const int ph = runh + block_scan(fh ? 1 : 0, toth, sh, parity);
      if (fm && pm < a.k) {
        const int ns = a.cache_slots[bT + t];
        a.topk_idx[wo + pm] = t;
        a.topk_slot[wo + pm] = ~ns;
      }
      if (fh && ph < a.k) {
        a.topk_idx[wo + ph] = t;
        a.topk_slot[wo + ph] = s;
      }
      runm += totm;
      runh += toth;
    }
  }
  if (rank == 0 && tid == 0) {
    for (int m = 0; m < M; ++m) a.n_miss_way[b * M + m] = sh.nmw[m];
    a.n_miss[b] = n_miss_total;
    a.step[b] = sh.step_b + 1;
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
    }
  }
  __syncthreads();
  cluster_sync();  // nobody leaves while others may read its shared memory
}

}  // namespace

cudaError_t launch_select(const ess_pool& p, int layer, const float* scores, int32_t* topk_idx,
                          int32_t* topk_slot, int32_t* n_miss_way, int32_t* miss_tok,
                          int32_t* miss_slot, int32_t* n_miss, cudaStream_t st) {
  const ess_config& c = p.cfg;
  const Layer& L = p.layers[layer];
  SelArgs a;
  a.scores = scores;
  a.cache_slots = L.cache_slots;
  a.slot_token = L.slot_token;
  a.last_used = L.last_used;
  a.step = L.step;
  a.Tb = L.T_dev;
  a.topk_idx = topk_idx;
  a.topk_slot = topk_slot;
  a.n_miss_way = n_miss_way;
  a.miss_tok = miss_tok;
  a.miss_slot = miss_slot;
  a.n_miss = n_miss;
  a.vict = p.scr.vict;
  a.stats = L.stats;
  a.status = p.scr.status;
  a.B = c.batch;
  a.M = c.mtp;
  a.k = c.k;
  a.T = c.max_T;
  a.C = c.C;
  int nl = (L.T_hmax + CL - 1) / CL;
  nl = ((nl + 3) / 4) * 4;
  if (nl < 4) nl = 4;
  a.n_local = nl;
  a.c_local = (c.C + CL - 1) / CL;
  const int MK = c.mtp * c.k;
  a.ucap = MK < c.mtp * nl ? MK : c.mtp * nl;
  int np2 = 1;
  while (np2 < MK) np2 <<= 1;
  const size_t sort_bytes = static_cast<size_t>(np2) * 8;
  const size_t res_bytes = static_cast<size_t>(c.mtp) * nl * 4;
  const size_t fixed = static_cast<size_t>(a.c_local) * 4 + static_cast<size_t>(a.ucap) * 9 + 64;
  const size_t budget = 200 * 1024;
  a.resident = (res_bytes + fixed <= budget) ? 1 : 0;
  size_t kb = a.resident ? (res_bytes > sort_bytes ? res_bytes : sort_bytes) : sort_bytes;
  kb = (kb + 15) / 16 * 16;
  a.keys_bytes = static_cast<uint32_t>(kb);
  const size_t smem = kb + fixed;
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  select_kernel<<<c.batch * CL, NT, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace ess
