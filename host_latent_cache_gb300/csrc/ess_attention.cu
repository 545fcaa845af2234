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
// (HBM) or from pinned host memory (UVA) into 128B-swizzled shared memory;
// tcgen05.mma computes S[128 heads][128 rows] = Q * R^T (bf16, fp32 in
// TMEM) one 64-dim block at a time as rows land, the softmax numerator P is
// formed in fp32 and stored as fp16, the 512 value dims of the rows are
// converted in place to fp16, and O[128][512] = P * V accumulates in TMEM.
// Per-CTA (max, sum, O) partials are merged by a second kernel.
#include "ess_device.cuh"

namespace ess {
namespace {

constexpr int NCH_ROWS = kAttnRows;      // rows per CTA
constexpr int QST = kAttnQStages;
constexpr uint32_t kBlk = 16384;         // one [128 rows x 64 dims] bf16 block
constexpr int kDimBlocks = kRowDim / 64; // 9
constexpr uint32_t kRowsBytes = kDimBlocks * kBlk;   // 147456
constexpr uint32_t kQBytes = QST * kBlk;             // 65536

struct AttnArgs {
  const int32_t* topk_idx;    // [B][M][k]
  const int32_t* topk_slot;   // [B][M][k]
  const int32_t* Tb;          // [B]
  const int32_t* page_table;  // [B][T/page] or null
  uint16_t* pool;             // [B][C][576]
  const uint16_t* host;       // [B][T][576] (device alias of pinned host memory)
  float* part_o;              // [B][M][nch][H][512]
  float2* part_ml;            // [B][M][nch][H]
  int* status;
  int B, M, H, k, nch, C, T, page, npages;
  float c2;                   // sm_scale * log2(e)
  int staged;
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
  const int Tb = a.Tb[b];
  const int nsel = a.k < Tb ? a.k : Tb;
  // rows j = 0..cnt-1 hold entries c + j * nch of the emitted list
  int cnt = 0;
  if (c < nsel) cnt = (nsel - 1 - c) / a.nch + 1;
  if (cnt > NCH_ROWS) cnt = NCH_ROWS;
  const size_t wo = (static_cast<size_t>(b) * a.M + m) * a.k;
  const int qrow0 = (b * a.M + m) * a.H;

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

  // query blocks 0..3 into the stage ring
  if (tid == 32) {
    tma_prefetch_desc(&qmap);
    for (int s = 0; s < QST; ++s) {
      mbar_arrive_expect_tx(smem_u32(&qfull[s]), kBlk);
      tma_load_2d(smem_u32(qst + s * kBlk), &qmap, smem_u32(&qfull[s]), s * 64, qrow0);
    }
  }

  // ------------------------------------------------ gather: thread j owns row j
  const int j = tid;
  bool valid = j < cnt;
  bool miss = false;
  int slot = 0;
  const uint16_t* src = nullptr;
  if (valid) {
    const int e = c + j * a.nch;
    const int t = a.topk_idx[wo + e];
    const int s = a.topk_slot[wo + e];
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
    } else if (miss && !a.staged) {
      src = a.host + (static_cast<size_t>(b) * a.T + prow) * kRowDim;
    } else {
      src = a.pool + (static_cast<size_t>(b) * a.C + slot) * kRowDim;
    }
  }
  for (int kb = 0; kb < kDimBlocks; ++kb) {
    uint8_t* dst = rows + kb * kBlk;
    for (int ch = 0; ch < 8; ++ch) {
      const uint32_t off = sw128_off(j, ch);
      if (valid)
        cp_async16(smem_u32(dst + off), src + kb * 64 + ch * 8);
      else
        *reinterpret_cast<uint4*>(dst + off) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
  }
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

  // FUSED miss path: write the host row through to its pool slot
  if (valid && miss && !a.staged) {
    uint16_t* dstp = a.pool + (static_cast<size_t>(b) * a.C + slot) * kRowDim;
    for (int kb = 0; kb < kDimBlocks; ++kb)
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(dstp + kb * 64 + ch * 8) =
            *reinterpret_cast<const uint4*>(rows + kb * kBlk + sw128_off(j, ch));
  }

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
    uint8_t* P = qst;  // [128 heads x 128 rows] fp16, two 64-row blocks
    for (int cc = 0; cc < 4; ++cc) {
      float v[32];
      tmem_ld32(trow + cc * 32, v);
      float p[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        p[i] = (cc * 32 + i < cnt) ? exp2f(fmaf(v[i], a.c2, -base)) : 0.0f;
        l += p[i];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 4 chunks of 8 rows
        const int col = cc * 32 + q * 8;
        uint4 pk;
        __half2 h0 = __floats2half2_rn(p[q * 8 + 0], p[q * 8 + 1]);
        __half2 h1 = __floats2half2_rn(p[q * 8 + 2], p[q * 8 + 3]);
        __half2 h2 = __floats2half2_rn(p[q * 8 + 4], p[q * 8 + 5]);
        __half2 h3 = __floats2half2_rn(p[q * 8 + 6], p[q * 8 + 7]);
        pk.x = *reinterpret_cast<uint32_t*>(&h0);
        pk.y = *reinterpret_cast<uint32_t*>(&h1);
        pk.z = *reinterpret_cast<uint32_t*>(&h2);
        pk.w = *reinterpret_cast<uint32_t*>(&h3);
        *reinterpret_cast<uint4*>(P + (col >> 6) * kBlk + sw128_off(tid, (col & 63) >> 3)) = pk;
      }
    }
    mx = (cnt > 0) ? base : -INFINITY;
    // value dims of this thread's row: bf16 -> fp16 in place (blocks 0..7)
    bool over = false;
    for (int kb = 0; kb < kLatent / 64; ++kb) {
      for (int ch = 0; ch < 8; ++ch) {
        uint4* pp = reinterpret_cast<uint4*>(rows + kb * kBlk + sw128_off(j, ch));
        uint4 u = *pp;
        uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float lo = __uint_as_float(w4[q] << 16);
          const float hi = __uint_as_float(w4[q] & 0xffff0000u);
          over |= fabsf(lo) > 65504.0f || fabsf(hi) > 65504.0f;
          __half2 h = __floats2half2_rn(lo, hi);
          w4[q] = *reinterpret_cast<uint32_t*>(&h);
        }
        *pp = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
    if (over) set_status(a.status, ESS_ERR_UNSUPPORTED);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && all_ok) {
    tc_fence_after();
    // O[128 x 512] = P[128 x 128] * V[128 x 512]; V is N-major (dims contiguous)
    const uint32_t idesc_pv = make_idesc(kFmtF16, kFmtF16, 1, 256, 128);
    const uint32_t pa = smem_u32(qst);
    const uint32_t ra = smem_u32(rows);
    for (int kt = 0; kt < 8; ++kt) {
      const uint64_t ad = make_sdesc_sw128(pa + (kt >> 2) * kBlk + (kt & 3) * 32, 16, 1024);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint64_t bd = make_sdesc_sw128(ra + half * 4 * kBlk + kt * 2048, kBlk, 1024);
        umma_f16(tmem + half * 256, ad, bd, idesc_pv, kt > 0);
      }
    }
    umma_commit(smem_u32(ofull));
  }
  // ------------------------------------------------ partial output
  const bool o_ok = all_ok && mbar_wait(smem_u32(ofull), 0, abort_flag);
  const bool all_o = __syncthreads_and(o_ok ? 1 : 0) != 0;
  const size_t pr = (static_cast<size_t>(b) * a.M + m) * a.nch + c;
  if (all_o) {
    tc_fence_after();
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float* dst = a.part_o + (pr * a.H + tid) * kLatent;
    for (int cc = 0; cc < kLatent / 32; ++cc) {
      float v[32];
      tmem_ld32(trow + cc * 32, v);
      if (tid < a.H) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(dst + cc * 32 + q * 4) =
              make_float4(v[q * 4], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
      }
    }
    if (tid < a.H) a.part_ml[pr * a.H + tid] = make_float2(mx, l);
  } else if (tid < a.H) {
    a.part_ml[pr * a.H + tid] = make_float2(-INFINITY, 0.0f);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// out[b][m][h][:] = sum_c 2^(mx_c - M) O_c / sum_c 2^(mx_c - M) l_c
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ part_o,
                                                      const float2* __restrict__ part_ml,
                                                      float* __restrict__ out, int H, int nch) {
  const int row = blockIdx.x;            // (b*M + m)*H + h
  const int bm = row / H, h = row % H;
  const float2* ml = part_ml + static_cast<size_t>(bm) * nch * H + h;
  float M = -INFINITY;
  for (int c = 0; c < nch; ++c) M = fmaxf(M, ml[static_cast<size_t>(c) * H].x);
  float4 acc = make_float4(0, 0, 0, 0);
  float L = 0.0f;
  if (M != -INFINITY) {
    for (int c = 0; c < nch; ++c) {
      const float2 v = ml[static_cast<size_t>(c) * H];
      if (v.y <= 0.0f) continue;
      const float wgt = exp2f(v.x - M);
      L += wgt * v.y;
      const float4 o = *reinterpret_cast<const float4*>(
          part_o + ((static_cast<size_t>(bm) * nch + c) * H + h) * kLatent + threadIdx.x * 4);
      acc.x = fmaf(wgt, o.x, acc.x);
      acc.y = fmaf(wgt, o.y, acc.y);
      acc.z = fmaf(wgt, o.z, acc.z);
      acc.w = fmaf(wgt, o.w, acc.w);
    }
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  *reinterpret_cast<float4*>(out + static_cast<size_t>(row) * kLatent + threadIdx.x * 4) =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

// (a6) one warp per miss row: host row of miss_tok -> pool slot miss_slot
__global__ void __launch_bounds__(256) stage_kernel(const int32_t* __restrict__ miss_tok,
                                                    const int32_t* __restrict__ miss_slot,
                                                    const int32_t* __restrict__ n_miss,
                                                    const int32_t* __restrict__ Tb,
                                                    const int32_t* __restrict__ page_table,
                                                    const uint16_t* __restrict__ host,
                                                    uint16_t* __restrict__ pool, int MK, int C,
                                                    int T, int page, int npages, int* status) {
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
  const uint4* s = reinterpret_cast<const uint4*>(host + (static_cast<size_t>(b) * T + prow) * kRowDim);
  uint4* d = reinterpret_cast<uint4*>(pool + (static_cast<size_t>(b) * C + v) * kRowDim);
  uint4 r[3];
#pragma unroll
  for (int q = 0; q < 3; ++q)
    if (lane + 32 * q < kRowBytes / 16) r[q] = s[lane + 32 * q];
#pragma unroll
  for (int q = 0; q < 3; ++q)
    if (lane + 32 * q < kRowBytes / 16) d[lane + 32 * q] = r[q];
}

size_t attn_smem_bytes() { return 1024 + kRowsBytes + kQBytes + 24 * 8 + 16; }

}  // namespace

cudaError_t launch_attention(const ess_pool& p, int layer, const void* q_mla,
                             const int32_t* topk_idx, const int32_t* topk_slot, float* out,
                             bool misses_staged, cudaStream_t st) {
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
  const size_t smem = attn_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.nch, c.mtp, c.batch);
  attn_kernel<<<grid, kAttnThreads, smem, st>>>(qmap, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  combine_kernel<<<c.batch * c.mtp * c.mla_heads, 128, 0, st>>>(p.scr.part_o, p.scr.part_ml, out,
                                                                c.mla_heads, a.nch);
  return cudaGetLastError();
}

cudaError_t launch_stage(const ess_pool& p, int layer, const int32_t* miss_tok,
                         const int32_t* miss_slot, const int32_t* n_miss, cudaStream_t st) {
  const ess_config& c = p.cfg;
  const Layer& L = p.layers[layer];
  const int MK = c.mtp * c.k;
  dim3 grid((MK + 7) / 8, c.batch);
  stage_kernel<<<grid, 256, 0, st>>>(miss_tok, miss_slot, n_miss, L.T_dev, L.page_table,
                                     L.host_latent, L.pool, MK, c.C, c.max_T, c.page,
                                     c.max_T / c.page, p.scr.status);
  return cudaGetLastError();
}

}  // namespace ess
