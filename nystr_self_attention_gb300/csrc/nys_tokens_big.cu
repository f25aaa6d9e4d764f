// Token rows on the tensor cores for large landmark counts and head widths
// (m up to 256, d = 128), whose operands do not fit the pipelined token
// kernel's shared memory. Same computation:
//   out[t] = softmax(Q[t] K~^T / sqrt(d)) W + sum_j w[h][j] V[t + j - (ks-1)/2]
// ("Nyströmformer" review page, Proposed method, bullets 3 and 6).
//
// Shared memory holds K~ (m x d), W^T (d x m) and the conv's Toeplitz
// operand per head (as its distinct 64 x 64 blocks: a block depends only on
// its block diagonal), ONE buffer shared by the Q tile and the V halo, and
// two 2 KB boxes per worker warp in which output rows are staged for TMA
// stores. TMEM: F/P
// (m columns), PW and CV accumulators (d columns each). One CTA per SM
// walks a contiguous range of 128-token tiles with five warps:
//   warp 4, one thread: TMA copies and tcgen05 products, in program order
//     per tile j:  F(j) = Q K~^T (once P V of tile j-1 is done) -> V halo
//     into the freed buffer -> CV(j) = T V (during the softmax of j) -> the
//     next Q tile into the buffer CV(j) freed -> PW(j) = P W (after the
//     softmax)
//   warps 0-3: softmax of tile j (thread = token row, P over F in TMEM),
//     then its epilogue out = PW / rowsum + CV, while F(j+1) is computed
// Every wait is bounded; a wait that runs out sets the status word, both
// roles wind down, copies in flight are awaited and TMEM is freed.
#include <cuda_bf16.h>

#include <algorithm>

#include "nys_internal.h"
#include "nys_sm100.h"
#include "nys_tma_host.h"

namespace nys {
namespace {

using namespace sm100;

struct BigMaps {
  CUtensorMap q, v, kt, wt;
  CUtensorMap out;  // stores: boxes of 32 tokens x 32 columns (SWIZZLE_64B)
};

struct BigParams {
  const float* conv_w;
  __nv_bfloat16* out;
  int* status;
  int H, n, d, m, m_pad, ks, kc;
  int tiles_per_head, total_tiles, tiles_per_cta;
  float c;  // softmax scale * log2(e)
  uint32_t off_kt, off_wt, off_t, off_qv, off_stage;
  int nbox;  // 64-column boxes of the conv's K (the V halo's rows)
  uint32_t kt_bytes, wt_bytes, q_bytes, v_bytes;
};

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int DP = 128, DC = 2;  // head width 128: two 64-column chunks
constexpr size_t kSmemBudget = 227 * 1024 - 1024;
constexpr int kThreads = 160;
constexpr uint32_t kStageBytes = 4 * 4096;  // output staging, two 2 KB boxes per worker warp

struct BigBars {
  uint64_t kw, q, v;           // TMA: K~ / W^T, Q tile, V halo
  uint64_t f, cv, pw;          // products done
  uint64_t p, epi, t;          // softmax warps: P written, accumulators read, Toeplitz built
  uint64_t fin;
};

__device__ __forceinline__ bool wait_or_fail(uint64_t* bar, uint32_t parity, int* status,
                                             volatile int* abort_flag) {
  if (mbar_wait(bar, parity, abort_flag, kWaitNs)) return true;
  if (!*abort_flag) {
    *abort_flag = 1;
    atomicExch(status, (int)NYS_ERR_TIMEOUT);
  }
  return false;
}

__global__ void __launch_bounds__(kThreads, 1) tokens_big(const __grid_constant__ BigMaps maps,
                                                          const __grid_constant__ BigParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* kts = sm + p.off_kt;
  uint8_t* wts = sm + p.off_wt;
  uint8_t* tbs = sm + p.off_t;
  uint8_t* qv = sm + p.off_qv;
  uint8_t* stage = sm + p.off_stage;  // output staging: two 32 x 32 bf16 boxes per worker warp
  __shared__ BigBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  volatile int* abort_flag = &abort_sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rad = p.ks > 0 ? (p.ks - 1) / 2 : 0;
  const int g0 = blockIdx.x * p.tiles_per_cta;
  const int ntiles = min(p.total_tiles, g0 + p.tiles_per_cta) - g0;
  const int tph = p.tiles_per_head;

  if (tid == 0) {
    mbar_init(&bars.kw, 1);
    mbar_init(&bars.q, 1);
    mbar_init(&bars.v, 1);
    mbar_init(&bars.f, 1);
    mbar_init(&bars.cv, 1);
    mbar_init(&bars.pw, 1);
    mbar_init(&bars.p, 128);
    mbar_init(&bars.epi, 128);
    mbar_init(&bars.t, 128);
    mbar_init(&bars.fin, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base_sh, 512);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t COL_F = 0, COL_PW = 256, COL_CV = 384;

  if (warp == 4) {
    // ------------------------------------------------------------- control
    if (lane == 0 && ntiles > 0) {
      tma_prefetch(&maps.q);
      tma_prefetch(&maps.v);
      tma_prefetch(&maps.kt);
      tma_prefetch(&maps.wt);
      const uint32_t idf = idesc_bf16(128, p.m_pad, false, false);
      const uint32_t idw = idesc_bf16(128, DP, false, false);
      const uint32_t idc = idesc_bf16(128, DP, false, true);
      uint32_t n_kw = 0, n_q = 0, n_v = 0, n_t = 0;  // copies issued / Toeplitz blocks awaited
      int cur_bh = -1, cur_h = -1;
      int bh = g0 / tph, t = g0 - (g0 / tph) * tph;  // head and tile within it
      auto load_q = [&](int tile_bh, int tile_t) {
        mbar_arrive_expect_tx(&bars.q, p.q_bytes);
        for (int dc = 0; dc < DC; ++dc) tma_load_3d(qv + dc * 16384, &maps.q, &bars.q, dc * 64, tile_t * 128, tile_bh);
        ++n_q;
      };
      load_q(bh, t);
      for (int j = 0; j < ntiles; ++j) {
        const int h = bh % p.H;
        // F(j): the F region is free once P V of tile j-1 is done
        if (j > 0 && !wait_or_fail(&bars.pw, (j - 1) & 1, p.status, abort_flag)) break;
        if (bh != cur_bh) {
          mbar_arrive_expect_tx(&bars.kw, p.kt_bytes + p.wt_bytes);
          for (int dc = 0; dc < DC; ++dc)
            tma_load_3d(kts + dc * (p.m_pad * 128), &maps.kt, &bars.kw, dc * 64, 0, bh);
          for (int mc = 0; mc * 64 < p.m_pad; ++mc)
            tma_load_3d(wts + mc * (DP * 128), &maps.wt, &bars.kw, mc * 64, 0, bh);
          ++n_kw;
          if (!wait_or_fail(&bars.kw, (n_kw - 1) & 1, p.status, abort_flag)) break;
          cur_bh = bh;
        }
        if (!wait_or_fail(&bars.q, (n_q - 1) & 1, p.status, abort_flag)) break;
        tc_fence_after_sync();
        {
          const uint64_t a0 = smem_desc(smem_u32(qv), 16, 1024, SW_128B);
          const uint64_t b0 = smem_desc(smem_u32(kts), 16, 1024, SW_128B);
#pragma unroll
          for (int kk = 0; kk < DP / 16; ++kk)
            mma_bf16(tmem + COL_F, a0 + (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2),
                     b0 + (uint64_t)((kk >> 2) * (p.m_pad * 8) + (kk & 3) * 2), idf, kk > 0);
          mma_commit(&bars.f);
        }
        if (p.kc > 0) {
          // V halo into the buffer F(j) has consumed
          if (!wait_or_fail(&bars.f, j & 1, p.status, abort_flag)) break;
          mbar_arrive_expect_tx(&bars.v, p.v_bytes);
          for (int dc = 0; dc < DC; ++dc)
            tma_load_3d(qv + dc * (p.kc * 128), &maps.v, &bars.v, dc * 64, t * 128 - rad, bh);
          ++n_v;
          // CV(j): V loaded, Toeplitz block of head h built, CV accumulator
          // read by the epilogue of tile j-1
          bool ok = wait_or_fail(&bars.v, (n_v - 1) & 1, p.status, abort_flag);
          if (ok && h != cur_h) {
            ++n_t;
            ok = wait_or_fail(&bars.t, (n_t - 1) & 1, p.status, abort_flag);
            cur_h = h;
          }
          if (ok && j > 0) ok = wait_or_fail(&bars.epi, (j - 1) & 1, p.status, abort_flag);
          if (!ok) break;
          tc_fence_after_sync();
          // K-box c of the Toeplitz operand is the 128-row window [B_c; B_c-1]
          // of the compact block list, which starts at block nbox - 1 - c
          const uint64_t a0 = smem_desc(smem_u32(tbs), 16, 1024, SW_128B);
          const uint64_t v0 = smem_desc(smem_u32(qv), p.kc * 128, 1024, SW_128B);
          for (int kk = 0; kk < p.kc / 16; ++kk)
            mma_bf16(tmem + COL_CV, a0 + (uint64_t)((p.nbox - 1 - (kk >> 2)) * 512 + (kk & 3) * 2),
                     v0 + (uint64_t)(kk * 128), idc, kk > 0);
          mma_commit(&bars.cv);
          // the next Q tile into the buffer CV(j) frees
          if (j + 1 < ntiles) {
            if (!wait_or_fail(&bars.cv, j & 1, p.status, abort_flag)) break;
            load_q(t + 1 == tph ? bh + 1 : bh, t + 1 == tph ? 0 : t + 1);
          }
        } else {
          if (j > 0 && !wait_or_fail(&bars.epi, (j - 1) & 1, p.status, abort_flag)) break;
          if (j + 1 < ntiles) {
            if (!wait_or_fail(&bars.f, j & 1, p.status, abort_flag)) break;
            load_q(t + 1 == tph ? bh + 1 : bh, t + 1 == tph ? 0 : t + 1);
          }
        }
        // PW(j) once the softmax has written P
        if (!wait_or_fail(&bars.p, j & 1, p.status, abort_flag)) break;
        tc_fence_after_sync();
        {
          const uint64_t w0 = smem_desc(smem_u32(wts), 16, 1024, SW_128B);
          for (int kk = 0; kk < p.m_pad / 16; ++kk)
            mma_bf16_tA(tmem + COL_PW, tmem + COL_F + kk * 8,
                        w0 + (uint64_t)((kk >> 2) * (DP * 8) + (kk & 3) * 2), idw, kk > 0);
          mma_commit(&bars.pw);
        }
        if (++t == tph) {
          t = 0;
          ++bh;
        }
      }
      if (*abort_flag) {
        // wait (bounded) for the copies still in flight
        if (n_kw) mbar_wait(&bars.kw, (n_kw - 1) & 1, nullptr, kWaitNs);
        if (n_q) mbar_wait(&bars.q, (n_q - 1) & 1, nullptr, kWaitNs);
        if (n_v) mbar_wait(&bars.v, (n_v - 1) & 1, nullptr, kWaitNs);
      }
      // no product of this CTA may be in flight when TMEM is freed
      mma_commit(&bars.fin);
      mbar_wait(&bars.fin, 0, nullptr, kWaitNs);
    }
  } else {
    // ---------------------------------------- softmax and epilogue, warps 0-3
    const uint32_t lo = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t fcol = tmem + lo + COL_F;
    const bool full_m = p.m == p.m_pad && (p.m_pad & 63) == 0;
    int bh = g0 / tph, t = g0 - (g0 / tph) * tph, cur_h = -1;
    for (int j = 0; j < ntiles; ++j) {
      const int h = bh % p.H;
      if (p.kc > 0 && h != cur_h) {
        // Toeplitz operand of head h: element (t, u) is w[u - t] (t the
        // tile's token, u the halo row), so its 64 x 64 block (r, c) depends
        // on c - r only: B_k[t'][u'] = w[64 k + u' - t']. Stored once each,
        // as the list B_(nbox-1), ..., B_0, B_-1 (= 0) of 8 KB blocks; thread
        // tid writes row tid % 64 of every other block. Its previous reader,
        // CV(j-1), completed before PW(j-1), which the epilogue of tile j-1
        // waited for.
        const float* wh = p.conv_w + (size_t)h * p.ks;
        const int tr = tid & 63;
        for (int blk = tid >> 6; blk <= p.nbox; blk += 2) {
          const int k = p.nbox - 1 - blk;
          for (int u0 = 0; u0 < 64; u0 += 8) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int ua = 64 * k + u0 + 2 * e - tr, ub = ua + 1;
              const float fa = (ua >= 0 && ua < p.ks) ? __ldg(wh + ua) : 0.f;
              const float fb = (ub >= 0 && ub < p.ks) ? __ldg(wh + ub) : 0.f;
              wv[e] = pack_bf16x2(fa, fb);
            }
            *reinterpret_cast<uint4*>(tbs + blk * 8192 + sw128_offset(tr, u0 * 2)) =
                make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
        fence_async_smem();
        mbar_arrive(&bars.t);
        cur_h = h;
      }
      // softmax of F(j): P (bf16) over F
      if (!__all_sync(0xffffffffu, wait_or_fail(&bars.f, j & 1, p.status, abort_flag))) break;
      tc_fence_after_sync();
      float mx = -INFINITY, l = 0.f;
      if (full_m) {
        for (int c0 = 0; c0 < p.m_pad; c0 += 64) {
          uint32_t r0[32], r1[32];
          tmem_ld32(fcol + c0, r0);
          tmem_ld32(fcol + c0 + 32, r1);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            mx = fmaxf(mx, fmaxf(__uint_as_float(r0[e]), __uint_as_float(r1[e])));
        }
      } else {
        for (int c0 = 0; c0 < p.m_pad; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(fcol + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c0 + e < p.m) mx = fmaxf(mx, __uint_as_float(r[e]));
        }
      }
      const float mc = mx * p.c;
      for (int c0 = 0; c0 < p.m_pad; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(fcol + c0, r);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float a = (full_m || c0 + 2 * e < p.m) ? fast_exp2(fmaf(__uint_as_float(r[2 * e]), p.c, -mc)) : 0.f;
          const float b = (full_m || c0 + 2 * e + 1 < p.m) ? fast_exp2(fmaf(__uint_as_float(r[2 * e + 1]), p.c, -mc)) : 0.f;
          l += a + b;
          pk[e] = pack_bf16x2(a, b);
        }
        tmem_st16(fcol + (c0 >> 1), pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars.p);
      // epilogue: out = PW / l + CV once PW(j) (and CV(j) before it) is done
      if (!__all_sync(0xffffffffu, wait_or_fail(&bars.pw, j & 1, p.status, abort_flag))) break;
      tc_fence_after_sync();
      // out rows, 32 columns at a time, staged in one of this warp's two
      // swizzled boxes (alternating) and written by a TMA store (rows past n
      // are clipped by the store); a box is rewritten once the store issued
      // from it two rounds earlier has read it
      const float inv_l = 1.f / l;
      const bool in_seq = t * 128 + warp * 32 < p.n;  // no box that starts past the sequence
#pragma unroll
      for (int c0 = 0; c0 < DP; c0 += 32) {
        uint8_t* box = stage + warp * 4096 + ((c0 >> 5) & 1) * 2048;
        uint32_t a[32], b[32];
        tmem_ld32(tmem + lo + COL_PW + c0, a);
        if (p.kc > 0) tmem_ld32(tmem + lo + COL_CV + c0, b);
        tmem_ld_wait();
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float x0 = __uint_as_float(a[2 * e]) * inv_l, x1 = __uint_as_float(a[2 * e + 1]) * inv_l;
          if (p.kc > 0) {
            x0 += __uint_as_float(b[2 * e]);
            x1 += __uint_as_float(b[2 * e + 1]);
          }
          o[e] = pack_bf16x2(x0, x1);
        }
        if (lane == 0) bulk_wait_read1();
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 4; ++e)
          *reinterpret_cast<uint4*>(box + sw64_offset(lane, 16 * e)) =
              make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0 && in_seq) {
          tma_store_3d(&maps.out, box, c0, t * 128 + warp * 32, (int)bh);
          bulk_commit();
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&bars.epi);
      if (++t == tph) {
        t = 0;
        ++bh;
      }
    }
  }
  if (warp < 4 && lane == 0) bulk_wait0();  // this warp's output stores are done
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

struct BigPlan {
  int m_pad, kc, nbox;
  uint32_t kt_bytes, wt_bytes, t_bytes, q_bytes, v_bytes, qv_bytes;
  size_t smem;
};

bool plan_big(const Shape& s, BigPlan* pl) {
  if (s.dtype != NYS_BF16 || s.d != 128) return false;
  pl->m_pad = ((s.m + 31) / 32) * 32;
  pl->kc = s.ks > 0 ? ((128 + s.ks - 1 + 15) / 16) * 16 : 0;
  if (pl->m_pad > 256 || pl->kc > 256) return false;
  pl->kt_bytes = (uint32_t)pl->m_pad * DP * 2;
  pl->wt_bytes = (uint32_t)((pl->m_pad + 63) / 64) * DP * 128;
  pl->nbox = (pl->kc + 63) / 64;
  pl->t_bytes = pl->kc > 0 ? (uint32_t)(pl->nbox + 1) * 8192 : 0;  // compact Toeplitz blocks
  pl->q_bytes = 128 * DP * 2;
  pl->v_bytes = (uint32_t)pl->kc * DP * 2;
  pl->qv_bytes = std::max(pl->q_bytes, pl->v_bytes);
  pl->smem = (size_t)pl->kt_bytes + pl->wt_bytes + pl->t_bytes + pl->qv_bytes + kStageBytes + 1024;
  return pl->smem <= kSmemBudget;
}

}  // namespace

bool tokens_big_supported(const Shape& s) {
  BigPlan pl;
  return plan_big(s, &pl);
}

int launch_tokens_big(const Shape& s, const void* q, const void* v, const void* kt_bf16,
                      const void* wt_bf16, const float* conv_w, void* out, int* status,
                      int num_sms, cudaStream_t stream) {
  BigPlan pl;
  if (!plan_big(s, &pl)) return NYS_ERR_UNSUPPORTED;
  const uint64_t BH = (uint64_t)s.bh();
  const int m64 = s.m64();
  BigMaps maps;
  {
    const uint64_t dims[3] = {(uint64_t)s.d, (uint64_t)s.n, BH};
    const uint64_t strides[2] = {(uint64_t)s.d * 2, (uint64_t)s.n * s.d * 2};
    const uint32_t boxq[3] = {64, 128, 1};
    const uint32_t boxv[3] = {64, (uint32_t)(pl.kc > 0 ? pl.kc : 16), 1};
    const uint32_t boxo[3] = {32, 32, 1};
    if (!make_tensor_map(&maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, boxq,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&maps.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, dims, strides, boxo,
                         CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_tensor_map(&maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, v, dims, strides, boxv,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
  }
  {
    const uint64_t dims[3] = {(uint64_t)DP, (uint64_t)m64, BH};
    const uint64_t strides[2] = {(uint64_t)DP * 2, (uint64_t)m64 * DP * 2};
    const uint32_t box[3] = {64, (uint32_t)pl.m_pad, 1};
    if (!make_tensor_map(&maps.kt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kt_bf16, dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
  }
  {
    const uint64_t dims[3] = {(uint64_t)m64, (uint64_t)DP, BH};
    const uint64_t strides[2] = {(uint64_t)m64 * 2, (uint64_t)m64 * DP * 2};
    const uint32_t box[3] = {64, (uint32_t)DP, 1};
    if (!make_tensor_map(&maps.wt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, wt_bf16, dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
  }
  BigParams p{};
  p.conv_w = conv_w;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.status = status;
  p.H = s.H;
  p.n = s.n;
  p.d = s.d;
  p.m = s.m;
  p.m_pad = pl.m_pad;
  p.ks = s.ks;
  p.kc = pl.kc;
  p.tiles_per_head = (s.n + 127) / 128;
  p.total_tiles = (int)(BH * p.tiles_per_head);
  const int ctas = std::min(p.total_tiles, num_sms);
  p.tiles_per_cta = (p.total_tiles + ctas - 1) / ctas;
  const int grid = (p.total_tiles + p.tiles_per_cta - 1) / p.tiles_per_cta;
  p.c = (1.0f / sqrtf((float)s.d)) * 1.4426950408889634f;
  p.kt_bytes = pl.kt_bytes;
  p.wt_bytes = pl.wt_bytes;
  p.q_bytes = pl.q_bytes;
  p.v_bytes = pl.v_bytes;
  p.off_kt = 0;
  p.off_wt = pl.kt_bytes;
  p.off_t = p.off_wt + pl.wt_bytes;
  p.off_qv = p.off_t + pl.t_bytes;
  p.off_stage = p.off_qv + pl.qv_bytes;
  p.nbox = pl.nbox;
  if (cudaFuncSetAttribute(tokens_big, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem) !=
      cudaSuccess)
    return set_cuda_error(cudaGetLastError());
  KernelScope scope("tokens_big", stream);
  tokens_big<<<grid, kThreads, pl.smem, stream>>>(maps, p);
  return launch_status();
}

}  // namespace nys
