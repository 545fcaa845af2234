// (a1) Lightning-indexer scores over the GPU-resident indexer cache.
//
// "ESS: Latent-Cache Offload" (foosynaptic tech notes), table "double cache
// and ESS division of labour": the indexer cache holds one light vector per
// position and is scored over the whole context every step, so it stays on
// the GPU.  Score of position s for query way m:
//     S = fl32( scale_s * sum_h w_h * ReLU(q_h . k_s) ).
//
// Persistent, warp-specialised kernel, one CTA per SM:
//   warp 0     (one lane) streams 128-token key tiles (128 B per token) with
//              TMA into a ring of as many 16 KB stages as shared memory holds
//              (up to 12), and at each request boundary starts asynchronous
//              loads of that request's queries (TMA, 128B swizzle) and head
//              weights (bulk copy) without pausing the key stream.  Key tiles
//              of tokens present at the bind depend on no earlier kernel, so
//              the first ring's worth is requested before the wait for the
//              previous grid, overlapping the stream's ramp-up with its tail;
//   warp 1     (one lane) issues tcgen05.mma: D[128 tokens][N] = K_tile * Q^T
//              with e4m3 (kind::f8f6f4) or bf16 (kind::f16) inputs and fp32
//              accumulators in TMEM, N = ways x heads padded to 32;
//   warps 2-9  two groups of four epilogue warps taking alternate tiles: a
//              thread reads its token's row of D from TMEM, applies ReLU, the
//              head weights and the key scale, stores the score and counts it
//              in a shared-memory histogram of the top 12 bits of its ordered
//              key, which is added to a per-(request, way) global histogram
//              at the end of each request's run of tiles (one histogram per
//              way, flushed and cleared between two barriers).  Given a
//              guessed coarse bin g per (request, way), it also sets the
//              token's bit in a flag bitmap when its key lies in bin g or
//              above (one ballot per 32 tokens) and counts keys of bins
//              g .. g + 3 in a fine histogram on 8 more bits, so that the
//              selection can skip the tokens far below the cut.
// The key tiles are the only large HBM stream; the kernel is bound by HBM
// bandwidth (about 132 B per token and request).
#include "ess_device.cuh"

namespace ess {
namespace {

struct IdxArgs {
  const float* w;            // [B][M][H_I]
  const float* scale;        // [B][T] or null (1.0)
  const int32_t* Tb;         // [B]
  const int32_t* tile_off;   // [B+1]
  const uint8_t* q;          // [B][M][H_I][128 B]
  float* scores;             // [B][M][T]
  uint32_t* ghist;           // [B][M][kHistBins] or null
  const uint32_t* guess;     // [B][M] guessed coarse bin (0: none), or null
  uint32_t* fhist;           // [B][M][kFineBins] (with guess)
  uint32_t* tflag;           // [B][M][nwords] (with guess)
  int nwords;
  int* status;
  int B, M, HI, NP, T, total_tiles, A;
  int S;                     // key-ring stages (chunks)
  int U;                     // tiles per chunk, the unit of the barrier rounds
  int early;                 // 1: no append since the last indexer launch on this layer
};

constexpr uint32_t kTileBytes = kIdxTile * kKeyRowBytes;  // 16 KB
constexpr int kMaxAcc = 8;   // TMEM accumulators in flight (A * N <= 512 columns)

// Walks a CTA's tiles in order over the concatenated requests: request b
// owns tiles [lo, hi); the tile prefix is read only when the request changes.
struct TileCursor {
  const int32_t* off;
  int B, b, lo, hi;
  __device__ __forceinline__ void start(const int32_t* o, int nb, int g) {
    off = o;
    B = nb;
    b = 0;
    lo = 0;
    hi = nb > 1 ? o[1] : 0x7fffffff;
    advance(g);
  }
  __device__ __forceinline__ void advance(int g) {
    while (b + 1 < B && g >= hi) {
      ++b;
      lo = hi;
      hi = b + 1 < B ? off[b + 1] : 0x7fffffff;
    }
  }
};

// Walks a CTA's tiles in chunks of up to U consecutive tiles of one request
// (the unit of every barrier round below), identically in every role.
struct ChunkWalker {
  TileCursor tc;
  int g, g1, U;
  __device__ __forceinline__ void start(const int32_t* off, int B, int g0_, int g1_, int U_) {
    tc.start(off, B, g0_);
    g = g0_;
    g1 = g1_;
    U = U_;
  }
  // request b, its first tile j0 in the chunk, n tiles; the chunk ends the
  // request's run of tiles in this CTA when last is set
  __device__ __forceinline__ bool next(int& b, int& j0, int& n, bool& last) {
    if (g >= g1) return false;
    tc.advance(g);
    b = tc.b;
    j0 = g - tc.lo;
    const int end = tc.hi < g1 ? tc.hi : g1;
    n = end - g < U ? end - g : U;
    g += n;
    last = g >= end;
    return true;
  }
};

// MW: the number of ways, fixed at compile time so that the epilogue's
// per-way code unrolls to exactly the ways that exist
template <bool FP8, int MW>
__global__ void __launch_bounds__(kIdxThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                   const IdxArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int NP = a.NP;
  const int A = a.A;
  const int S = a.S;
  const int U = a.U;
  const uint32_t stage_bytes = static_cast<uint32_t>(U) * kTileBytes;
  uint8_t* kst = smem;                                   // S x U x 16 KB key tiles
  uint8_t* qbuf = kst + S * stage_bytes;                 // 2 x NP x 128 B queries
  float* wbuf = reinterpret_cast<float*>(qbuf + 2 * NP * 128);  // 2 x NP weights
  uint32_t* hist = reinterpret_cast<uint32_t*>(wbuf + 2 * NP);   // M x kHistBins
  // the fine histograms follow the coarse ones: M x kFineBins
  const int HC = a.ghist ? a.M * kHistBins : 0;
  const int HB = HC + (a.ghist && a.guess ? a.M * kFineBins : 0);
  uint64_t* bars = reinterpret_cast<uint64_t*>(hist + HB);
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;
  uint64_t* acce = accf + kMaxAcc;
  uint64_t* qfull = acce + kMaxAcc;
  uint64_t* qempty = qfull + 2;
  uint64_t* epdone = qempty + 2;      // every epilogue thread has counted its tokens
  uint64_t* fldone = epdone + 2;      // the histogram is flushed and clear again
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fldone + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* consumed = abort_flag + 1;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int g0 = static_cast<int>((static_cast<long long>(blockIdx.x) * a.total_tiles) / gridDim.x);
  const int g1 =
      static_cast<int>((static_cast<long long>(blockIdx.x + 1) * a.total_tiles) / gridDim.x);
  const int MH = a.M * a.HI;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < kMaxAcc; ++i) {
      mbar_init(smem_u32(&accf[i]), 1);
      mbar_init(smem_u32(&acce[i]), 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&qfull[i]), 1);
      mbar_init(smem_u32(&qempty[i]), 1 + 256);
      mbar_init(smem_u32(&epdone[i]), 256);
      mbar_init(smem_u32(&fldone[i]), 256);
    }
    *abort_flag = 0;
    *consumed = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < HB; i += kIdxThreads) hist[i] = 0;
  for (int i = tid; i < 2 * NP; i += kIdxThreads) wbuf[i] = 0.0f;
  uint32_t ncols = 32;
  while (ncols < static_cast<uint32_t>(A * U * NP)) ncols <<= 1;
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), ncols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&qmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the keys of chunk it: n tiles from tile j0 of request b into stage it % S
  // (the epilogue threads read their tokens' key scales from global memory)
  auto issue_chunk = [&](int it, int b, int j0, int n) {
    const int s = it % S;
    mbar_arrive_expect_tx(smem_u32(&full[s]), static_cast<uint32_t>(n) * kTileBytes);
    for (int u = 0; u < n; ++u)
      tma_load_2d(smem_u32(kst + s * stage_bytes + u * kTileBytes), &kmap, smem_u32(&full[s]), 0,
                  b * a.T + (j0 + u) * kIdxTile);
  };
  // Early mode: no append kernel has run on this layer since its last indexer,
  // so the tile prefix and the key rows of the first chunks are
  // final already; the first ring's worth is requested before the wait.
  int n_early = 0;
  if (warp == 0 && a.early) {
    if (lane == 0) {
      ChunkWalker cw;
      cw.start(a.tile_off, a.B, g0, g1, U);
      int b, j0, n;
      bool last;
      while (n_early < S && cw.next(b, j0, n, last)) issue_chunk(n_early++, b, j0, n);
    }
    n_early = __shfl_sync(0xffffffffu, n_early, 0);
  }
  pdl_wait_previous();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------ producer
    ChunkWalker cw;
    cw.start(a.tile_off, a.B, g0, g1, U);
    int cur_b = -1, seg = -1, it = 0;
    int b, j0, n;
    bool last;
    bool ok = true;
    for (; ok && cw.next(b, j0, n, last); ++it) {
      if (b != cur_b) {
        ++seg;
        const int qb = seg & 1;
        int w_ok = 1;
        if (lane == 0) {
          if (seg >= 2)
            w_ok = mbar_wait(smem_u32(&qempty[qb]), ((seg >> 1) - 1) & 1, abort_flag) ? 1 : 0;
          if (w_ok) {
            // queries: NP rows x 128 B by TMA (128B swizzle = the MMA operand
            // layout; rows past M*H_I belong to other requests or are zero and
            // only meet zero weights); weights: M*H_I floats by bulk copy
            mbar_arrive_expect_tx(smem_u32(&qfull[qb]), static_cast<uint32_t>(NP * 128 + MH * 4));
            tma_load_2d(smem_u32(qbuf + qb * NP * 128), &qmap, smem_u32(&qfull[qb]), 0, b * MH);
            bulk_load(smem_u32(wbuf + qb * NP), a.w + static_cast<size_t>(b) * MH,
                      static_cast<uint32_t>(MH * 4), smem_u32(&qfull[qb]));
          }
        }
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        cur_b = b;
      }
      int w_ok = 1;
      if (lane == 0 && it >= n_early) {
        const int s = it % S;
        if (it >= S) w_ok = mbar_wait(smem_u32(&empty[s]), ((it / S) - 1) & 1, abort_flag) ? 1 : 0;
        if (w_ok) issue_chunk(it, b, j0, n);
      }
      w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
      if (!w_ok) ok = false;
    }
    if (!ok) {
      if (lane == 0) {
        set_status(a.status, ESS_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
    // drain: wait (bounded) for every issued copy to land
    if (lane == 0 && *abort_flag) {
      const int issued = it > n_early ? it : n_early;
      for (int i = *consumed; i < issued; ++i)
        mbar_wait(smem_u32(&full[i % S]), (i / S) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = FP8 ? make_idesc(kFmtE4M3, kFmtE4M3, 0, NP, 128)
                                 : make_idesc(kFmtBF16, kFmtBF16, 0, NP, 128);
      ChunkWalker cw;
      cw.start(a.tile_off, a.B, g0, g1, U);
      int cur_b = -1, seg = -1, it = 0;
      int b, j0, n;
      bool last;
      for (; cw.next(b, j0, n, last); ++it) {
        if (b != cur_b) {
          if (seg >= 0) umma_commit(smem_u32(&qempty[seg & 1]));
          ++seg;
          if (!mbar_wait(smem_u32(&qfull[seg & 1]), (seg >> 1) & 1, abort_flag)) break;
          cur_b = b;
        }
        const int s = it % S;
        if (!mbar_wait(smem_u32(&full[s]), (it / S) & 1, abort_flag)) break;
        *consumed = it + 1;
        const int acc = it % A;
        if (it >= A && !mbar_wait(smem_u32(&acce[acc]), ((it / A) - 1) & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t b_base = smem_u32(qbuf + (seg & 1) * NP * 128);
        for (int u = 0; u < n; ++u) {
          const uint32_t a_base = smem_u32(kst + s * stage_bytes + u * kTileBytes);
          const uint32_t d = tmem_base + static_cast<uint32_t>((acc * U + u) * NP);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = make_sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd = make_sdesc_sw128(b_base + kk * 32, 16, 1024);
            if (FP8)
              umma_f8(d, ad, bd, idesc, kk > 0);
            else
              umma_f16(d, ad, bd, idesc, kk > 0);
          }
        }
        umma_commit(smem_u32(&empty[s]));
        umma_commit(smem_u32(&accf[acc]));
      }
      if (seg >= 0) umma_commit(smem_u32(&qempty[seg & 1]));
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..9)
    const int grp = (warp - 2) >> 2;         // chunks with it % 2 == grp
    const int quad = warp & 3;               // TMEM lanes 32*quad .. +31
    const int row = quad * 32 + lane;        // token row of each tile
    const int te = tid - 64;                 // 0..255
    ChunkWalker cw;
    cw.start(a.tile_off, a.B, g0, g1, U);
    int cur_b = -1, seg = -1, it = 0;
    int Tcur = 0;
    uint32_t gm[kMaxWays] = {0u, 0u, 0u, 0u};   // guessed coarse bin per way (0: none)
    int b, j0, n;
    bool last;
    bool ok = true;
    // 64-column TMEM loads when no chunk of columns straddles two ways
    const bool wide = (NP % 64 == 0) && (MW == 1 || a.HI % 64 == 0);
    // sum_h w_h * ReLU(D[row][h]) of every way, from the NP columns at taddr;
    // every product and partial sum is exact under the score contract, so
    // four independent chains per chunk give the same result as one
    auto head_sums = [&](uint32_t taddr, const float* wq, float* sm) {
#pragma unroll
      for (int m = 0; m < kMaxWays; ++m) sm[m] = 0.0f;
      if (NP == 32) {
        float v[32];
        tmem_ld32(taddr, v);
        float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 w4 = *reinterpret_cast<const float4*>(wq + i);
          p0 = fmaf(w4.x, fmaxf(v[i], 0.0f), p0);
          p1 = fmaf(w4.y, fmaxf(v[i + 1], 0.0f), p1);
          p2 = fmaf(w4.z, fmaxf(v[i + 2], 0.0f), p2);
          p3 = fmaf(w4.w, fmaxf(v[i + 3], 0.0f), p3);
        }
        sm[0] = (p0 + p1) + (p2 + p3);
      } else if (wide) {
        for (int c = 0; c < NP / 64; ++c) {
          float v[64];
          tmem_ld64(taddr + c * 64, v);
          float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
          for (int i = 0; i < 64; i += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(wq + c * 64 + i);
            p0 = fmaf(w4.x, fmaxf(v[i], 0.0f), p0);
            p1 = fmaf(w4.y, fmaxf(v[i + 1], 0.0f), p1);
            p2 = fmaf(w4.z, fmaxf(v[i + 2], 0.0f), p2);
            p3 = fmaf(w4.w, fmaxf(v[i + 3], 0.0f), p3);
          }
          const float part = (p0 + p1) + (p2 + p3);
          // columns c*64 .. belong to way c*64 / H_I (here H_I % 64 == 0 or M == 1)
          const int m = (MW == 1) ? 0 : (c * 64) / a.HI;
          if (m == 0) sm[0] += part;
          else if (m == 1) sm[1] += part;
          else if (m == 2) sm[2] += part;
          else sm[3] += part;
        }
      } else {
        // 32-column chunks: a way of 32 heads, or N = 96 / 160 / 224
        for (int c = 0; c < NP / 32; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(wq + c * 32 + i);
            p0 = fmaf(w4.x, fmaxf(v[i], 0.0f), p0);
            p1 = fmaf(w4.y, fmaxf(v[i + 1], 0.0f), p1);
            p2 = fmaf(w4.z, fmaxf(v[i + 2], 0.0f), p2);
            p3 = fmaf(w4.w, fmaxf(v[i + 3], 0.0f), p3);
          }
          const float part = (p0 + p1) + (p2 + p3);
          const int m = (MW == 1) ? 0 : (c * 32) / a.HI;   // H_I % 32 == 0 when M > 1
          if (m == 0) sm[0] += part;
          else if (m == 1) sm[1] += part;
          else if (m == 2) sm[2] += part;
          else sm[3] += part;
        }
      }
    };
    for (; ok && cw.next(b, j0, n, last); ++it) {
      if (b != cur_b) {
        ++seg;
        if (!mbar_wait(smem_u32(&qfull[seg & 1]), (seg >> 1) & 1, abort_flag)) break;
        cur_b = b;
        Tcur = a.Tb[b];
#pragma unroll
        for (int m = 0; m < kMaxWays; ++m)
          gm[m] = (HB > HC && m < MW) ? a.guess[b * MW + m] : 0u;
      }
      if ((it & 1) == grp) {
        // this thread's key scales of the chunk, read while its MMAs run
        float scv[kIdxSubMax];
#pragma unroll
        for (int u = 0; u < kIdxSubMax; ++u) {
          const int t = (j0 + u) * kIdxTile + row;
          scv[u] = (u < n && t < Tcur && a.scale != nullptr)
                       ? __ldg(a.scale + static_cast<size_t>(b) * a.T + t)
                       : 1.0f;
        }
        const int acc = it % A;
        ok = mbar_wait(smem_u32(&accf[acc]), (it / A) & 1, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float* wq = wbuf + (seg & 1) * NP;
        // the head sums of the chunk's tiles (unrolled over kIdxSubMax so that
        // they stay in registers)
        float smv[kIdxSubMax][kMaxWays];
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll
        for (int u = 0; u < kIdxSubMax; ++u)
          if (u < n) head_sums(lane_base + static_cast<uint32_t>((acc * U + u) * NP), wq, smv[u]);
        tc_fence_before();
        mbar_arrive(smem_u32(&acce[acc]));
#pragma unroll
        for (int u = 0; u < kIdxSubMax; ++u) {
          if (u >= n) continue;   // the same in every lane
          const int t = (j0 + u) * kIdxTile + row;
          const bool valid = t < Tcur;
          const float sc = scv[u];
          const int word = (j0 + u) * (kIdxTile / 32) + quad;   // this warp's 32 tokens
#pragma unroll
          for (int m = 0; m < kMaxWays; ++m) {   // unrolled: the sums stay in registers
            if (m >= MW) break;
            uint32_t key = 0u;
            if (valid) {
              const float sv = __fmul_rn(smv[u][m], sc) + 0.0f;  // one rounding; +0 for zero
              a.scores[(static_cast<size_t>(b) * a.M + m) * a.T + t] = sv;
              key = float_key(sv);
              if (HB) atomicAdd(hist + m * kHistBins + (key >> 20), 1u);
              const uint32_t d = (key >> 20) - gm[m];
              if (gm[m] != 0u && d < static_cast<uint32_t>(kFineWin))
                atomicAdd(hist + HC + m * kFineBins + d * kFineSub + ((key >> 12) & (kFineSub - 1)),
                          1u);
            }
            if (gm[m] != 0u) {   // the same in every lane
              const unsigned f = __ballot_sync(0xffffffffu, valid && (key >> 20) >= gm[m]);
              if (lane == 0 && word < a.nwords)
                a.tflag[(static_cast<size_t>(b) * a.M + m) * a.nwords + word] = f;
            }
          }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      // end of this request's run of tiles: release the query buffer and
      // publish the histogram once every epilogue thread has counted
      if (last) {
        mbar_arrive(smem_u32(&qempty[seg & 1]));
        if (HB) {
          mbar_arrive(smem_u32(&epdone[seg & 1]));
          if (!mbar_wait(smem_u32(&epdone[seg & 1]), (seg >> 1) & 1, abort_flag)) break;
          uint32_t* gh = a.ghist + static_cast<size_t>(b) * a.M * kHistBins;
          uint32_t* gf = HB > HC ? a.fhist + static_cast<size_t>(b) * a.M * kFineBins : nullptr;
          for (int i = te; i < HB; i += 256) {
            const uint32_t v = hist[i];
            if (v) {
              atomicAdd(i < HC ? gh + i : gf + (i - HC), v);
              hist[i] = 0;
            }
          }
          // nobody counts the next request's tokens before the clear is complete
          mbar_arrive(smem_u32(&fldone[seg & 1]));
          if (!mbar_wait(smem_u32(&fldone[seg & 1]), (seg >> 1) & 1, abort_flag)) break;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, ncols);
  }
}

size_t indexer_smem_bytes(int S, int U, int NP, int HB) {
  return 1024 + static_cast<size_t>(S) * U * kTileBytes + 2u * NP * 128 + 2u * NP * 4 +
         HB * 4u + (2 * S + 2 * kMaxAcc + 8) * 8 + 16;
}

// Tiles per chunk and key-ring stages for a query width: as many tiles per
// chunk as keep U x N <= 256 TMEM columns (so at least two chunks' sums are
// in flight), then as many stages as fit one CTA (at most kIdxMaxStages),
// fewer tiles per chunk when not even kIdxMinStages stages fit.
void indexer_shape(int NP, int HB, int* U_out, int* S_out) {
  int U = 256 / NP < kIdxSubMax ? 256 / NP : kIdxSubMax;
  if (U < 1) U = 1;
  for (;; --U) {
    int S = kIdxMaxStages;
    while (S > kIdxMinStages && indexer_smem_bytes(S, U, NP, HB) > kMaxSmemPerCta) --S;
    if (indexer_smem_bytes(S, U, NP, HB) <= kMaxSmemPerCta || U == 1) {
      *U_out = U;
      *S_out = S;
      return;
    }
  }
}

}  // namespace

// Shared memory of one indexer CTA with the fused score histogram in its
// smallest shape (the kernel has no static shared memory).
size_t indexer_smem_need(const ess_config& c) {
  const int NP = ((c.mtp * c.idx_heads + 31) / 32) * 32;
  const int HB = c.mtp * (kHistBins + kFineBins);
  int U, S;
  indexer_shape(NP, HB, &U, &S);
  return indexer_smem_bytes(S, U, NP, HB);
}

cudaError_t launch_indexer(const ess_pool& p, int layer, const void* q_idx, const float* w,
                           float* scores, bool with_hist, cudaStream_t st) {
  const ess_config& c = p.cfg;
  const Layer& L = p.layers[layer];
  if (L.total_tiles == 0) return cudaSuccess;
  IdxArgs a;
  a.w = w;
  a.scale = L.idx_scale;
  a.Tb = L.T_dev;
  a.tile_off = L.tile_off;
  a.q = static_cast<const uint8_t*>(q_idx);
  a.scores = scores;
  a.ghist = with_hist ? p.scr.ghist : nullptr;
  // the flags and the fine histogram go with the histogram: the selection
  // that reads it follows on the stream and keeps the guesses
  a.guess = with_hist ? L.guess : nullptr;
  a.fhist = p.scr.fhist;
  a.tflag = p.scr.tflag;
  a.nwords = p.scr.nwords;
  a.status = p.scr.status;
  a.B = c.batch;
  a.M = c.mtp;
  a.HI = c.idx_heads;
  a.NP = ((c.mtp * c.idx_heads + 31) / 32) * 32;
  a.T = c.max_T;
  a.total_tiles = L.total_tiles;
  const int HB = with_hist ? c.mtp * (kHistBins + kFineBins) : 0;
  indexer_shape(a.NP, HB, &a.U, &a.S);
  a.A = 512 / (a.U * a.NP) < kMaxAcc ? 512 / (a.U * a.NP) : kMaxAcc;
  a.early = L.append_pending ? 0 : 1;
  CUtensorMap qmap;
  if (!encode_map_2d(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_idx, kKeyRowBytes,
                     static_cast<uint64_t>(c.batch) * c.mtp * c.idx_heads, kKeyRowBytes,
                     kKeyRowBytes, static_cast<uint32_t>(a.NP)))
    return cudaErrorInvalidValue;
  const int grid = L.total_tiles < p.num_sms ? L.total_tiles : p.num_sms;
  const size_t smem = indexer_smem_bytes(a.S, a.U, a.NP, HB);
  cudaError_t e;
  using Kern = void (*)(CUtensorMap, CUtensorMap, IdxArgs);
  static const Kern kern_fp8[kMaxWays] = {indexer_kernel<true, 1>, indexer_kernel<true, 2>,
                                          indexer_kernel<true, 3>, indexer_kernel<true, 4>};
  static const Kern kern_bf16[kMaxWays] = {indexer_kernel<false, 1>, indexer_kernel<false, 2>,
                                           indexer_kernel<false, 3>, indexer_kernel<false, 4>};
  const Kern kern = (c.idx_dtype == ESS_FP8_E4M3 ? kern_fp8 : kern_bf16)[c.mtp - 1];
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(grid), dim3(kIdxThreads), smem, st, L.kmap, qmap, a);
  if (e == cudaSuccess) {
    count_launch(p);
    // this launch waits for any append before it, so the next one may load early
    p.layers[layer].append_pending = false;
  }
  return e;
}

}  // namespace ess
