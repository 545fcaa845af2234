// (a5) Sparse absorbed-MLA attention with a gather that forks per row, and
// (a6) the separate miss-staging copy.
//
// hwcomputing.csdn.net FlashOffloading analysis, section "decode side (2)":
// SparseFlashAttention gathers the selected rows, then runs Q x K, softmax
// and A x V; CopySFA moves the host copy into that gather and forks on
// hit/miss: a hit row is read from the HBM hot cache, a miss row is read
// from pinned host memory straight on chip and written to its slot on the
// way (three memory accesses instead of four for copy-then-attend).
// "ESS: Latent-Cache Offload": each latent entry is c^KV[512] + k^R[64];
// the logits use all 576 dims, the output the first 512.
//
// One CTA handles 128 selected rows of one (request, way), assigned with a
// stride over the emitted list so the misses at its head spread over all
// CTAs.  Rows are gathered with 16-byte cp.async straight from the pool
// (HBM) or from pinned host memory (UVA) into 128B-swizzled shared memory
// (a miss among the newest appended tokens comes from their device ring);
// tcgen05.mma computes S[128 heads][128 rows] = Q * R^T (bf16, fp32 in
// TMEM) one 64-dim block at a time as rows land; the softmax numerator P is
// formed in fp32 and split into two bf16 terms P = P_hi + P_lo (about 16
// significant bits, so the output stays within the tolerance), and
// O[128][512] = P_hi * V + P_lo * V accumulates in TMEM with V read in place
// as the N-major operand.
// Each CTA leaves its (max, sum) per head and its unnormalised O [H][512] as
// a partial: O leaves TMEM through shared memory in four 128-dim quarters,
// each written out by one bulk copy.  A second kernel, launched as a
// programmatic dependent of this one, merges the partials of every (request,
// way) with the usual log-sum-exp weights.
#include "ess_device.cuh"
#include "ess_sync.cuh"

namespace ess {
namespace {

constexpr int NCH_ROWS = kAttnRows;      // rows per CTA
constexpr int QST = kAttnQStages;
constexpr uint32_t kBlk = 16384;         // one [128 rows x 64 dims] bf16 block
constexpr int kDimBlocks = kRowDim / 64; // 9
constexpr uint32_t kRowsBytes = kDimBlocks * kBlk;   // 147456
constexpr uint32_t kQBytes = QST * kBlk;             // 65536
constexpr int kMergeBatch = 8;       // chunk partials in flight per merge thread
constexpr int kMergeMinBlocks = 8;   // merge CTAs per SM the register budget allows

struct AttnArgs {
  const int32_t* topk_idx;    // [B][M][k]
  const int32_t* topk_slot;   // [B][M][k]
  const int32_t* Tb;          // [B]
  const int32_t* page_table;  // [B][T/page] or null
  uint16_t* pool;             // [B][C][576]
  const uint16_t* host;       // [B][T][576] (device alias of pinned host memory)
  const uint16_t* tail;       // [B][2*page][576] ring of the newest appended rows
  const int32_t* T0;          // [B] tokens >= T0_b were appended after the bind
  uint16_t* part_o;           // [B][M][nch][H][512] fp16 (unit u of head h at u ^ (h & 7))
  float2* part_ml;            // [B][M][nch][H]
  int* status;
  int B, M, H, k, nch, C, T, page, npages;
  float c2;                   // sm_scale * log2(e)
  int staged;
  int compact;                // host rows are compact 656-byte rows, widened on the way
  // 1: the previous kernel on the stream is the LRU finishing kernel of the
  // selection that wrote the lists read here.  The grid may launch while that
  // selection still runs: each CTA waits for its request's counter in ready
  // instead, and the wait for the finishing kernel moves to the end so the
  // two run side by side.  Each CTA then counts its partial out in
  // attn_done, on which the merge kernel waits instead of this whole grid.
  int early;
  const int* ready;           // [B] completion counters of the selection (early only)
  int* attn_done;             // [B][M] completion counters of this grid (early only)
};

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap qmap, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* rows = smem;                       // 9 blocks
  uint8_t* qst = smem + kRowsBytes;           // 4 stages; P (fp16) reuses stages 0-1
  uint64_t* bars = reinterpret_cast<uint64_t*>(qst + kQBytes);
  uint64_t* qfull = bars;                     // [4]
  uint64_t* qempty = qfull + QST;             // [4]
  uint64_t* blk = qempty + QST;               // [9]
  uint64_t* sfull = blk + kDimBlocks;         // [1]
  uint64_t* ofull = sfull + 1;                // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ofull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int c = blockIdx.x, m = blockIdx.y, b = blockIdx.z;
  const size_t wo = (static_cast<size_t>(b) * a.M + m) * a.k;
  const int qrow0 = (b * a.M + m) * a.H;
  // early: the merge kernel waits on the counters, so it may launch as soon as
  // every CTA of this grid is resident
  if (a.early) pdl_launch_dependents();

  if (tid == 0) {
    for (int i = 0; i < QST; ++i) {
      mbar_init(smem_u32(&qfull[i]), 1);
      mbar_init(smem_u32(&qempty[i]), 1);
    }
    for (int i = 0; i < kDimBlocks; ++i) mbar_init(smem_u32(&blk[i]), kAttnThreads);
    mbar_init(smem_u32(sfull), 1);
    mbar_init(smem_u32(ofull), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything above touched only this CTA's shared memory and TMEM.  Early:
  // T_b was final before the selection ahead of this grid could launch.
  if (!a.early) pdl_wait_previous();
  const int Tb = a.Tb[b];
  const int nsel = a.k < Tb ? a.k : Tb;
  // appended tokens of the two newest pages are read from the device ring
  const int tail_lo = max(a.T0[b], (Tb / a.page - 1) * a.page);
  // rows j = 0..cnt-1 hold entries c + j * nch of the emitted list
  int cnt = 0;
  if (c < nsel) cnt = (nsel - 1 - c) / a.nch + 1;
  if (cnt > NCH_ROWS) cnt = NCH_ROWS;

  // query blocks 0..3 into the stage ring
  if (tid == 32) {
    tma_prefetch_desc(&qmap);
    for (int s = 0; s < QST; ++s) {
      mbar_arrive_expect_tx(smem_u32(&qfull[s]), kBlk);
      tma_load_2d(smem_u32(qst + s * kBlk), &qmap, smem_u32(&qfull[s]), s * 64, qrow0);
    }
  }
  if (a.early) {
    // request b's lists are out once every selection CTA of it has counted
    // itself (all of them are resident: they let the finishing kernel, and it
    // this grid, launch).  Past the limit the chunk is treated as empty.
    __shared__ int lists_ok;
    if (tid == 0) {
      lists_ok = wait_count(a.ready + b * kCounterStride, kSelCluster) ? 1 : 0;
      if (!lists_ok) set_status(a.status, ESS_ERR_TIMEOUT);
    }
    __syncthreads();
    if (!lists_ok) cnt = 0;
  }

  // ------------------------------------------------ gather
  // Thread j resolves row j (its entry, hit/miss, source address); warp w then
  // gathers its rows 32w..32w+31 cooperatively: for each 64-dim block, 8 lanes
  // cover one row's 128 bytes, so every instruction moves four full lines.
  const int j = tid;
  const int lane = tid & 31;
  bool valid = j < cnt;
  bool miss = false;
  bool cmiss = false;          // a compact host row: widened below instead of copied
  int slot = 0;
  const uint16_t* src = nullptr;
  if (valid) {
    const int e = c + j * a.nch;
    const int t = __ldcg(a.topk_idx + wo + e);     // through L2: written by the selection
    const int s = __ldcg(a.topk_slot + wo + e);
    miss = s < 0;
    slot = miss ? ~s : s;
    int prow = t;
    if (a.page_table) {
      const int pg = (t >= 0 && t < Tb) ? t / a.page : 0;
      prow = a.page_table[static_cast<size_t>(b) * a.npages + pg] * a.page + t % a.page;
    }
    if (t < 0 || t >= Tb || slot < 0 || slot >= a.C || prow < 0 || prow >= a.T) {
      set_status(a.status, ESS_ERR_DEVICE_CHECK);
      valid = false;
    } else if (miss && !a.staged && a.compact) {
      cmiss = true;   // widened below
      src = reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(a.host) +
                                              (static_cast<size_t>(b) * a.T + prow) *
                                                  kCompactRowBytes);
    } else if (miss && !a.staged) {
      src = t >= tail_lo
                ? a.tail + (static_cast<size_t>(b) * 2 * a.page + t % (2 * a.page)) * kRowDim
                : a.host + (static_cast<size_t>(b) * a.T + prow) * kRowDim;
    } else {
      src = a.pool + (static_cast<size_t>(b) * a.C + slot) * kRowDim;
    }
  }
  const unsigned valid_mask = __ballot_sync(0xffffffffu, valid);
  const unsigned cmiss_mask = __ballot_sync(0xffffffffu, cmiss);
  const unsigned copy_mask = valid_mask & ~cmiss_mask;
  const int sub = lane >> 3;   // row within a group of four
  const int ch = lane & 7;     // 16-byte chunk within the 128-byte block row
  for (int kb = 0; kb < kDimBlocks; ++kb) {
    uint8_t* dst = rows + kb * kBlk;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int rl = q * 4 + sub;                 // row of this warp, 0..31
      const int r = warp * 32 + rl;
      const uint64_t sp = __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(src), rl);
      const uint32_t off = sw128_off(r, ch);
      if ((copy_mask >> rl) & 1u)
        cp_async16(smem_u32(dst + off), reinterpret_cast<const uint16_t*>(sp) + kb * 64 + ch * 8);
      else if (!((valid_mask >> rl) & 1u))
        *reinterpret_cast<uint4*>(dst + off) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
  }
  // compact host rows: the warp widens its own, up to four rows' loads in flight
  // (plain stores; each thread's fence before it publishes a block covers them)
  for (unsigned cm = cmiss_mask; cm;) {
    int rls[4];
    CompactLane cl[4];
    int nb = 0;
    for (; nb < 4 && cm; ++nb) {
      rls[nb] = __ffs(cm) - 1;
      cm &= cm - 1;
      const uint64_t sp = __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(src), rls[nb]);
      cl[nb] = compact_load(reinterpret_cast<const uint8_t*>(sp), lane);
    }
    for (int i = 0; i < nb; ++i) {
      const int r = warp * 32 + rls[i];
      uint4 lo, hi;
      compact_widen(cl[i], lane, lo, hi);
      // dims 16 lane .. +15: block lane / 4, 16-byte chunks 2 (lane % 4) and + 1
      uint8_t* blk0 = rows + (lane >> 2) * kBlk;
      *reinterpret_cast<uint4*>(blk0 + sw128_off(r, (lane & 3) * 2)) = lo;
      *reinterpret_cast<uint4*>(blk0 + sw128_off(r, (lane & 3) * 2 + 1)) = hi;
      if (lane >= 1 && lane < 9)   // RoPE dims 512 + 8 (lane - 1): block 8, chunk lane - 1
        *reinterpret_cast<uint4*>(rows + 8 * kBlk + sw128_off(r, lane - 1)) = cl[i].extra;
    }
  }
  __syncwarp();
  // as each 64-dim block lands: publish it; thread 0 multiplies, thread 32 refills Q
  const uint32_t idesc_qk = make_idesc(kFmtBF16, kFmtBF16, 0, 128, 128);
  bool ok = true;
  for (int kb = 0; kb < kDimBlocks; ++kb) {
    cp_async_wait_dyn(kDimBlocks - 1 - kb);
    fence_proxy_async_smem();
    mbar_arrive(smem_u32(&blk[kb]));
    if (tid == 0 && ok) {
      const int s = kb % QST;
      ok = mbar_wait(smem_u32(&blk[kb]), 0, abort_flag) &&
           mbar_wait(smem_u32(&qfull[s]), (kb / QST) & 1, abort_flag);
      if (ok) {
        tc_fence_after();
        const uint32_t qa = smem_u32(qst + s * kBlk);
        const uint32_t ra = smem_u32(rows + kb * kBlk);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_f16(tmem, make_sdesc_sw128(qa + kk * 32, 16, 1024),
                   make_sdesc_sw128(ra + kk * 32, 16, 1024), idesc_qk, (kb | kk) != 0);
        umma_commit(smem_u32(&qempty[s]));
      } else {
        set_status(a.status, ESS_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
    if (tid == 32 && ok && kb + QST < kDimBlocks) {
      const int s = kb % QST;
      ok = mbar_wait(smem_u32(&qempty[s]), (kb / QST) & 1, abort_flag);
      if (ok) {
        mbar_arrive_expect_tx(smem_u32(&qfull[s]), kBlk);
        tma_load_2d(smem_u32(qst + s * kBlk), &qmap, smem_u32(&qfull[s]), (kb + QST) * 64, qrow0);
      } else {
        set_status(a.status, ESS_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  }
  if (tid == 0 && ok) umma_commit(smem_u32(sfull));

  // FUSED miss path: write each host row through to its pool slot (the warp
  // that gathered the row copies it, 16 bytes per lane)
  cp_async_wait<0>();
  __syncwarp();
  {
    const unsigned miss_mask = __ballot_sync(0xffffffffu, valid && miss && !a.staged);
    for (unsigned mm = miss_mask; mm; mm &= mm - 1) {
      const int rl = __ffs(mm) - 1;
      const int r = warp * 32 + rl;
      const int sl = __shfl_sync(0xffffffffu, slot, rl);
      uint16_t* dstp = a.pool + (static_cast<size_t>(b) * a.C + sl) * kRowDim;
      for (int q = lane; q < kRowBytes / 16; q += 32) {
        const int kb = q >> 3, cc = q & 7;
        *reinterpret_cast<uint4*>(dstp + kb * 64 + cc * 8) =
            *reinterpret_cast<const uint4*>(rows + kb * kBlk + sw128_off(r, cc));
      }
    }
  }
  __syncwarp();

  // ------------------------------------------------ softmax over this CTA's rows
  const bool s_ok = mbar_wait(smem_u32(sfull), 0, abort_flag);
  const bool all_ok = __syncthreads_and(s_ok ? 1 : 0) != 0;
  float mx = -INFINITY, l = 0.0f;
  if (all_ok) {
    tc_fence_after();
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int cc = 0; cc < 4; ++cc) {
      float v[32];
      tmem_ld32(trow + cc * 32, v);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (cc * 32 + i < cnt) mx = fmaxf(mx, v[i]);
    }
    const float base = (cnt > 0) ? mx * a.c2 : 0.0f;
    // [128 heads x 128 rows] bf16, two 64-row blocks each: P_hi in stages 0-1,
    // P_lo in stages 2-3 (the query stages are free once S is complete)
    uint8_t* Phi = qst;
    uint8_t* Plo = qst + 2 * kBlk;
    for (int cc = 0; cc < 4; ++cc) {
      float v[32];
      tmem_ld32(trow + cc * 32, v);
      float p[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        p[i] = (cc * 32 + i < cnt) ? ex2_approx(fmaf(v[i], a.c2, -base)) : 0.0f;
        l += p[i];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 4 chunks of 8 rows
        const int col = cc * 32 + q * 8;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = p[q * 8 + 2 * e], x1 = p[q * 8 + 2 * e + 1];
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
          const float2 hf = __bfloat1622float2(h2);
          const __nv_bfloat162 l2 = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
          hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
          lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
        }
        const uint32_t off = (col >> 6) * kBlk + sw128_off(tid, (col & 63) >> 3);
        *reinterpret_cast<uint4*>(Phi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(Plo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    mx = (cnt > 0) ? base : -INFINITY;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && all_ok) {
    tc_fence_after();
    // O[128 x 512] = (P_hi + P_lo)[128 x 128] * V[128 x 512]; V is N-major (dims contiguous)
    const uint32_t idesc_pv = make_idesc(kFmtBF16, kFmtBF16, 1, 256, 128);
    const uint32_t ra = smem_u32(rows);
    for (int kt = 0; kt < 8; ++kt) {
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint32_t pa = smem_u32(qst + part * 2 * kBlk);
        const uint64_t ad = make_sdesc_sw128(pa + (kt >> 2) * kBlk + (kt & 3) * 32, 16, 1024);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint64_t bd = make_sdesc_sw128(ra + half * 4 * kBlk + kt * 2048, kBlk, 1024);
          umma_f16(tmem + half * 256, ad, bd, idesc_pv, (kt | part) != 0);
        }
      }
    }
    umma_commit(smem_u32(ofull));
  }
  // ------------------------------------------------ partial output
  const bool o_ok = all_ok && mbar_wait(smem_u32(ofull), 0, abort_flag);
  const bool all_o = __syncthreads_and(o_ok ? 1 : 0) != 0;
  const size_t pr = (static_cast<size_t>(b) * a.M + m) * a.nch + c;
  if (all_o) {
    // O leaves TMEM through shared memory as fp16 (the row blocks are free
    // once PV is done): [head][512 dims], the 16-byte unit u (8 dims) of head h
    // stored at u ^ (h & 7) so the shared-memory writes spread over every bank,
    // then one bulk copy writes the CTA's partial out.  The unnormalised sums
    // are bounded by the row count times the largest latent value, far inside
    // fp16 range; the merge weights and the final output stay fp32.
    tc_fence_after();
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    if (warp * 32 < a.H) {   // tcgen05.ld is warp-wide: the condition is per warp
      for (int cc = 0; cc < kLatent / 32; ++cc) {
        float v[32];
        tmem_ld32(trow + cc * 32, v);
        if (tid < a.H) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int u = cc * 4 + e;
            uint4 pk;
            pk.x = half2_bits(v[8 * e + 0], v[8 * e + 1]);
            pk.y = half2_bits(v[8 * e + 2], v[8 * e + 3]);
            pk.z = half2_bits(v[8 * e + 4], v[8 * e + 5]);
            pk.w = half2_bits(v[8 * e + 6], v[8 * e + 7]);
            *reinterpret_cast<uint4*>(rows + tid * (kLatent * 2) + ((u ^ (tid & 7)) << 4)) = pk;
          }
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_store(a.part_o + pr * a.H * kLatent, smem_u32(rows),
                 static_cast<uint32_t>(a.H) * kLatent * 2u);
      bulk_commit();
    }
    if (tid < a.H) a.part_ml[pr * a.H + tid] = make_float2(mx, l);
  } else {
    if (tid < a.H) a.part_ml[pr * a.H + tid] = make_float2(-INFINITY, 0.0f);
  }
  if (tid == 0) bulk_wait_all();
  if (a.early) pdl_wait_previous();   // finish only after the LRU finishing kernel
  else pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (a.early && tid == 0) {
    // the partial is out (the bulk copy complete, every (max, sum) written
    // before the barrier) and the finishing kernel has completed: count it
    fence_proxy_async_global();
    count_done(a.attn_done + (b * a.M + m) * kCounterStride, 1);
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// out[b][m][h][:] = sum_c 2^(mx_c - M) O_c[h][:] / sum_c 2^(mx_c - M) l_c over the
// chunk partials of (request b, way m), M the running maximum (merged
// kMergeBatch chunks at a time, rescaling the running sums when M grows).  One
// CTA per (head, request-way); thread t owns dims 4t..4t+3.  Launched as a
// programmatic dependent of the attention kernel: it waits for that grid
// before reading the partials, or, inside a step (done given), only for the
// counter of its own (request, way).  Eight chunks' loads are in flight per thread
// (two rounds of L2 latency instead of four), with few enough registers that
// every CTA is still resident beside the attention CTAs (a second wave would
// add its whole latency to the step).
__global__ void __launch_bounds__(128, kMergeMinBlocks) merge_kernel(const uint16_t* __restrict__ part_o,
                                                    const float2* __restrict__ part_ml,
                                                    float* __restrict__ out, int H, int nch,
                                                    const int* done, int* status) {
  const int h = blockIdx.x, bm = blockIdx.y, t = threadIdx.x;
  if (done != nullptr) {
    // the nch chunk CTAs of (request, way) bm count themselves once their
    // partials are out; the attention CTAs are all resident before this grid
    // launches.  Past the limit the error is recorded and the merge goes on.
    if (t == 0 && !wait_count(done + bm * kCounterStride, nch)) set_status(status, ESS_ERR_TIMEOUT);
    __syncthreads();
  } else {
    pdl_wait_previous();
  }
  pdl_launch_dependents();
  const float2* ml = part_ml + static_cast<size_t>(bm) * nch * H + h;
  // dims 4t..4t+3 of head h: half of the 16-byte unit t/2, stored at unit (t/2) ^ (h & 7)
  const int u = (t >> 1) ^ (h & 7);
  const uint2* po = reinterpret_cast<const uint2*>(
      part_o + (static_cast<size_t>(bm) * nch * H + h) * kLatent + u * 8 + (t & 1) * 4);
  const size_t cstride = static_cast<size_t>(H) * (kLatent / 4);   // one chunk, in uint2 units
  float M = -INFINITY, L = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < nch; c0 += kMergeBatch) {
    float2 e[kMergeBatch];
    uint2 v[kMergeBatch];
#pragma unroll
    for (int q = 0; q < kMergeBatch; ++q) {
      const int c = c0 + q;
      e[q] = c < nch ? __ldcg(ml + static_cast<size_t>(c) * H) : make_float2(-INFINITY, 0.0f);
      v[q] = c < nch ? __ldcg(po + static_cast<size_t>(c) * cstride) : make_uint2(0u, 0u);
    }
    float Mg = M;
#pragma unroll
    for (int q = 0; q < kMergeBatch; ++q)
      if (e[q].y > 0.0f) Mg = fmaxf(Mg, e[q].x);
    const float r = (M == -INFINITY) ? 0.0f : exp2f(M - Mg);
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
    L *= r;
#pragma unroll
    for (int q = 0; q < kMergeBatch; ++q) {
      if (e[q].y > 0.0f) {   // a chunk with no rows leaves no O partial
        const float w = exp2f(e[q].x - Mg);
        const float2 lo = half2_bits_to_float2(v[q].x), hi = half2_bits_to_float2(v[q].y);
        L = fmaf(w, e[q].y, L);
        acc.x = fmaf(w, lo.x, acc.x);
        acc.y = fmaf(w, lo.y, acc.y);
        acc.z = fmaf(w, hi.x, acc.z);
        acc.w = fmaf(w, hi.y, acc.w);
      }
    }
    M = Mg;
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  reinterpret_cast<float4*>(out + (static_cast<size_t>(bm) * H + h) * kLatent)[t] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

// (a6) one warp per miss row: host (or ring) row of miss_tok -> pool slot miss_slot
__global__ void __launch_bounds__(256) stage_kernel(const int32_t* __restrict__ miss_tok,
                                                    const int32_t* __restrict__ miss_slot,
                                                    const int32_t* __restrict__ n_miss,
                                                    const int32_t* __restrict__ Tb,
                                                    const int32_t* __restrict__ page_table,
                                                    const uint16_t* __restrict__ host,
                                                    const uint16_t* __restrict__ tail,
                                                    const int32_t* __restrict__ T0,
                                                    uint16_t* __restrict__ pool, int MK, int C,
                                                    int T, int page, int npages, int compact,
                                                    int* status) {
  pdl_wait_previous();
  pdl_launch_dependents();
  const int b = blockIdx.y;
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n_miss[b]) return;
  const int t = miss_tok[static_cast<size_t>(b) * MK + i];
  const int v = miss_slot[static_cast<size_t>(b) * MK + i];
  int prow = t;
  if (page_table && t >= 0 && t < Tb[b])
    prow = page_table[static_cast<size_t>(b) * npages + t / page] * page + t % page;
  if (t < 0 || t >= Tb[b] || v < 0 || v >= C || prow < 0 || prow >= T) {
    if (lane == 0) set_status(status, ESS_ERR_DEVICE_CHECK);
    return;
  }
  if (compact) {   // a compact host row, widened to bf16 (the warp is converged here)
    compact_row_to_bf16(reinterpret_cast<const uint8_t*>(host) +
                            (static_cast<size_t>(b) * T + prow) * kCompactRowBytes,
                        pool + (static_cast<size_t>(b) * C + v) * kRowDim, lane);
    return;
  }
  // appended tokens of the two newest pages come from the device ring
  const int tail_lo = max(T0[b], (Tb[b] / page - 1) * page);
  const uint4* s = reinterpret_cast<const uint4*>(
      t >= tail_lo ? tail + (static_cast<size_t>(b) * 2 * page + t % (2 * page)) * kRowDim
                   : host + (static_cast<size_t>(b) * T + prow) * kRowDim);
  uint4* d = reinterpret_cast<uint4*>(pool + (static_cast<size_t>(b) * C + v) * kRowDim);
  uint4 r[3];
#pragma unroll
  for (int q = 0; q < 3; ++q)
    if (lane + 32 * q < kRowBytes / 16) r[q] = s[lane + 32 * q];
#pragma unroll
  for (int q = 0; q < 3; ++q)
    if (lane + 32 * q < kRowBytes / 16) d[lane + 32 * q] = r[q];
}

// Reload the rows of every resident token from the host copy (or the ring of
// appended rows) into its pool slot: slot s of request b holds token
// slot_token[b][s] after a restored state.  One warp per slot.
__global__ void __launch_bounds__(256) refill_kernel(const int32_t* __restrict__ slot_token,
                                                     const int32_t* __restrict__ Tb,
                                                     const int32_t* __restrict__ page_table,
                                                     const uint16_t* __restrict__ host,
                                                     const uint16_t* __restrict__ tail,
                                                     const int32_t* __restrict__ T0,
                                                     uint16_t* __restrict__ pool, int C, int T,
                                                     int page, int npages, int compact,
                                                     int* status) {
  const int b = blockIdx.y;
  const int s = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (s >= C) return;
  const int t = slot_token[static_cast<size_t>(b) * C + s];
  if (t < 0) return;
  const int tb = Tb[b];
  int prow = t;
  if (page_table && t < tb)
    prow = page_table[static_cast<size_t>(b) * npages + t / page] * page + t % page;
  if (t >= tb || prow < 0 || prow >= T) {
    if (lane == 0) set_status(status, ESS_ERR_DEVICE_CHECK);
    return;
  }
  if (compact) {
    compact_row_to_bf16(reinterpret_cast<const uint8_t*>(host) +
                            (static_cast<size_t>(b) * T + prow) * kCompactRowBytes,
                        pool + (static_cast<size_t>(b) * C + s) * kRowDim, lane);
    return;
  }
  const int tail_lo = max(T0[b], (tb / page - 1) * page);
  const uint4* src = reinterpret_cast<const uint4*>(
      t >= tail_lo ? tail + (static_cast<size_t>(b) * 2 * page + t % (2 * page)) * kRowDim
                   : host + (static_cast<size_t>(b) * T + prow) * kRowDim);
  uint4* d = reinterpret_cast<uint4*>(pool + (static_cast<size_t>(b) * C + s) * kRowDim);
  for (int q = lane; q < kRowBytes / 16; q += 32) d[q] = src[q];
}

// Rows of a pinned host array -> device memory, one warp per row, 16-byte
// loads: the miss path's access pattern, for measuring the host link.
__global__ void __launch_bounds__(256) host_gather_kernel(const uint4* __restrict__ host,
                                                          const int64_t* __restrict__ rows,
                                                          int64_t n_rows, int64_t n_host_rows,
                                                          int vec_per_row, uint4* __restrict__ dst,
                                                          int* status) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n_rows) return;
  const int64_t r = rows ? rows[i] : i;
  if (r < 0 || r >= n_host_rows) {
    if (lane == 0 && status) atomicCAS(status, 0, 1);
    return;
  }
  const uint4* s = host + r * vec_per_row;
  uint4* d = dst + i * vec_per_row;
  for (int q = lane; q < vec_per_row; q += 32) d[q] = s[q];
}

size_t attn_smem_bytes() { return 1024 + kRowsBytes + kQBytes + 24 * 8 + 16; }

}  // namespace

cudaError_t launch_attention(const ess_pool& p, int layer, const void* q_mla,
                             const int32_t* topk_idx, const int32_t* topk_slot, float* out,
                             bool misses_staged, bool early, cudaStream_t st) {
  const ess_config& c = p.cfg;
  const Layer& L = p.layers[layer];
  CUtensorMap qmap;
  if (!encode_map_2d(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q_mla, kRowDim,
                     static_cast<uint64_t>(c.batch) * c.mtp * c.mla_heads, kRowBytes, 64, 128))
    return cudaErrorInvalidValue;
  AttnArgs a;
  a.topk_idx = topk_idx;
  a.topk_slot = topk_slot;
  a.Tb = L.T_dev;
  a.page_table = L.page_table;
  a.pool = L.pool;
  a.host = L.host_latent;
  a.tail = L.tail;
  a.T0 = L.T0_dev;
  a.part_o = p.scr.part_o;
  a.part_ml = p.scr.part_ml;
  a.status = p.scr.status;
  a.B = c.batch;
  a.M = c.mtp;
  a.H = c.mla_heads;
  a.k = c.k;
  a.nch = p.lay.nch;
  a.C = c.C;
  a.T = c.max_T;
  a.page = c.page;
  a.npages = c.max_T / c.page;
  a.c2 = c.sm_scale * 1.4426950408889634f;
  a.staged = misses_staged ? 1 : 0;
  a.compact = L.compact ? 1 : 0;
  a.early = (early && !misses_staged) ? 1 : 0;
  a.ready = p.scr.ready;
  a.attn_done = p.scr.attn_done;
  const size_t smem = attn_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.nch, c.mtp, c.batch);
  e = launch_pdl(attn_kernel, grid, dim3(kAttnThreads), smem, st, qmap, a);
  if (e != cudaSuccess) return e;
  count_launch(p);
  e = launch_pdl(merge_kernel, dim3(c.mla_heads, c.batch * c.mtp), dim3(128), 0, st,
                 static_cast<const uint16_t*>(p.scr.part_o), static_cast<const float2*>(p.scr.part_ml),
                 out, c.mla_heads, a.nch,
                 static_cast<const int*>(a.early ? p.scr.attn_done : nullptr), p.scr.status);
  if (e == cudaSuccess) count_launch(p);
  return e;
}

cudaError_t launch_stage(const ess_pool& p, int layer, const int32_t* miss_tok,
                         const int32_t* miss_slot, const int32_t* n_miss, cudaStream_t st) {
  const ess_config& c = p.cfg;
  const Layer& L = p.layers[layer];
  const int MK = c.mtp * c.k;
  dim3 grid((MK + 7) / 8, c.batch);
  const cudaError_t e =
      launch_pdl(stage_kernel, grid, dim3(256), 0, st, miss_tok, miss_slot, n_miss,
                 static_cast<const int32_t*>(L.T_dev), static_cast<const int32_t*>(L.page_table),
                 L.host_latent, static_cast<const uint16_t*>(L.tail),
                 static_cast<const int32_t*>(L.T0_dev), L.pool, MK, c.C, c.max_T, c.page,
                 c.max_T / c.page, L.compact ? 1 : 0, p.scr.status);
  if (e == cudaSuccess) count_launch(p);
  return e;
}

cudaError_t launch_refill(const ess_pool& p, int layer, cudaStream_t st) {
  const ess_config& c = p.cfg;
  const Layer& L = p.layers[layer];
  dim3 grid((c.C + 7) / 8, c.batch);
  refill_kernel<<<grid, 256, 0, st>>>(L.slot_token, L.T_dev, L.page_table, L.host_latent, L.tail,
                                      L.T0_dev, L.pool, c.C, c.max_T, c.page, c.max_T / c.page,
                                      L.compact ? 1 : 0, p.scr.status);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch(p);
  return e;
}

cudaError_t launch_host_gather(const void* host_dev, const int64_t* rows, int64_t n_rows,
                               int64_t n_host_rows, int row_bytes, void* dst, int* status,
                               cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  const int64_t blocks = (n_rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  host_gather_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      static_cast<const uint4*>(host_dev), rows, n_rows, n_host_rows, row_bytes / 16,
      static_cast<uint4*>(dst), status);
  return cudaGetLastError();
}

}  // namespace ess
