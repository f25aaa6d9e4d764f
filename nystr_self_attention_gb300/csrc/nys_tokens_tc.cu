// Token rows on the tensor cores (bf16 inputs, fp32 accumulate):
//   out[t] = softmax(Q[t] K~^T / sqrt(d)) W + sum_j w[h][j] V[t + j - (ks-1)/2]
// ("Nyströmformer" review page, Proposed method, bullets 3 and 6).
//
// One CTA of 128 threads walks a contiguous range of 128-token tiles
// (persistent over the whole batch). Per tile:
//   F   = Q_tile K~^T            tcgen05, A = Q (smem, TMA), B = K~ (smem)
//   P   = exp(F - rowmax)        thread = row, read from TMEM, written back
//                                into the same TMEM columns as packed bf16
//   PW  = P W                    tcgen05, A = P (TMEM), B = W^T (smem)
//   CV  = T V_halo               tcgen05, A = banded Toeplitz of the conv
//                                taps (smem), B = V rows t0-r .. (MN-major)
//   out = PW / rowsum + CV       thread = row, bf16 store
// Q and the V halo come in by TMA through a two-stage ring; K~, W^T and the
// Toeplitz block are reloaded only when the head changes. Every wait is
// bounded; a wait that runs out sets the status word and the CTA winds down.
#include <cuda_bf16.h>

#include <algorithm>

#include "nys_internal.h"
#include "nys_sm100.h"
#include "nys_tma_host.h"

namespace nys {
namespace {

using namespace sm100;

struct TokMaps {
  CUtensorMap q, v, kt, wt;
};

struct TokParams {
  const float* conv_w;
  __nv_bfloat16* out;
  int* status;
  int H, n, d, m, m_pad, ks, kc;  // m_pad: multiple of 32; kc: conv K extent (0: no conv)
  int tiles_per_head, total_tiles, tiles_per_cta;
  float c;  // softmax scale * log2(e)
  uint32_t tmem_cols;
  uint32_t off_q, off_v, off_kt, off_wt, off_t;  // smem offsets from the 1024-aligned base
  uint32_t q_stage, v_stage, kt_bytes, wt_bytes;
};

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ void fail(int* status, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicExch(status, (int)NYS_ERR_TIMEOUT);
}

template <int DP>
__global__ void __launch_bounds__(128, 1) tokens_tc(const __grid_constant__ TokMaps maps,
                                                    const TokParams p) {
  constexpr int DC = DP / 64;  // 64-column chunks of d
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  __shared__ uint64_t bar_full[2], bar_kw, bar_mma;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  volatile int* abort_flag = &abort_sh;

  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_init(&bar_kw, 1);
    mbar_init(&bar_mma, 1);
    abort_sh = 0;
    fence_barrier_init();
    tma_prefetch(&maps.q);
    tma_prefetch(&maps.v);
    tma_prefetch(&maps.kt);
    tma_prefetch(&maps.wt);
  }
  if (warp == 0) tmem_alloc(&tmem_base_sh, p.tmem_cols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t COL_F = 0, COL_PW = p.m_pad, COL_CV = p.m_pad + DP;
  const int rad = p.ks > 0 ? (p.ks - 1) / 2 : 0;

  const int g0 = blockIdx.x * p.tiles_per_cta;
  const int g1 = min(p.total_tiles, g0 + p.tiles_per_cta);

  uint32_t pend = 0;                  // bit s: a load into stage s not yet waited on
  uint32_t nload0 = 0, nload1 = 0;    // loads issued into stage 0 / 1
  bool kw_pending = false;
  auto issue_load = [&](int stage, int g) {
    const int bh = g / p.tiles_per_head, t0 = (g % p.tiles_per_head) * 128;
    uint8_t* qs = sm + p.off_q + stage * p.q_stage;
    uint8_t* vs = sm + p.off_v + stage * p.v_stage;
    mbar_arrive_expect_tx(&bar_full[stage], p.q_stage + (p.kc > 0 ? p.v_stage : 0));
#pragma unroll
    for (int dc = 0; dc < DC; ++dc) tma_load_3d(qs + dc * 16384, &maps.q, &bar_full[stage], dc * 64, t0, bh);
    if (p.kc > 0) {
#pragma unroll
      for (int dc = 0; dc < DC; ++dc)
        tma_load_3d(vs + dc * (p.kc * 128), &maps.v, &bar_full[stage], dc * 64, t0 - rad, bh);
    }
    pend |= 1u << stage;
    if (stage) ++nload1; else ++nload0;
  };
  auto issue_f = [&](int stage) {
    const uint32_t qs = smem_u32(sm + p.off_q + stage * p.q_stage);
    const uint32_t ks_ = smem_u32(sm + p.off_kt);
    const uint32_t id = idesc_bf16(128, p.m_pad, false, false);
#pragma unroll
    for (int kk = 0; kk < DP / 16; ++kk) {
      const uint64_t a = smem_desc(qs + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, SW_128B);
      const uint64_t b = smem_desc(ks_ + (kk >> 2) * (p.m_pad * 128) + (kk & 3) * 32, 16, 1024, SW_128B);
      mma_bf16(tmem + COL_F, a, b, id, kk > 0);
    }
    mma_commit(&bar_mma);
  };

  if (tid == 0) {
    if (g0 < g1) issue_load(0, g0);
    if (g0 + 1 < g1) issue_load(1, g0 + 1);
  }

  uint32_t mma_phase = 0, kw_phase = 0;
  int cur_bh = -1, cur_h = -1;
  bool f_issued = false;  // F of the current tile already in flight
  for (int g = g0; g < g1; ++g) {
    const int j = g - g0, s = j & 1;
    const int bh = g / p.tiles_per_head, t0 = (g % p.tiles_per_head) * 128;
    const int h = bh % p.H;
    // (A) head change: K~, W^T by TMA; the conv's Toeplitz block by threads
    if (bh != cur_bh) {
      if (tid == 0) {
        mbar_arrive_expect_tx(&bar_kw, p.kt_bytes + p.wt_bytes);
        for (int dc = 0; dc < DC; ++dc)
          tma_load_3d(sm + p.off_kt + dc * (p.m_pad * 128), &maps.kt, &bar_kw, dc * 64, 0, bh);
        for (int mc = 0; mc < p.m_pad / 64 + ((p.m_pad & 63) ? 1 : 0); ++mc)
          tma_load_3d(sm + p.off_wt + mc * (DP * 128), &maps.wt, &bar_kw, mc * 64, 0, bh);
        kw_pending = true;
      }
      if (p.kc > 0 && h != cur_h) {
        // row t of the Toeplitz block: column u holds w[u - t] for 0 <= u - t < ks
        const int t = tid;
        const float* wh = p.conv_w + (size_t)h * p.ks;
        uint8_t* tb = sm + p.off_t;
        const int kc64 = (p.kc + 63) & ~63;
        for (int u0 = 0; u0 < kc64; u0 += 8) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int ua = u0 + 2 * e - t, ub = ua + 1;
            const float fa = (ua >= 0 && ua < p.ks && u0 + 2 * e < p.kc) ? wh[ua] : 0.f;
            const float fb = (ub >= 0 && ub < p.ks && u0 + 2 * e + 1 < p.kc) ? wh[ub] : 0.f;
            wv[e] = pack_bf16x2(fa, fb);
          }
          uint8_t* dst = tb + (u0 >> 6) * 16384 + sw128_offset(t, (u0 & 63) * 2);
          *reinterpret_cast<uint4*>(dst) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
        fence_async_smem();
        cur_h = h;
      }
      if (tid == 0) {
        if (!mbar_wait(&bar_kw, kw_phase, abort_flag, kWaitNs)) fail(p.status, abort_flag);
        else kw_pending = false;
      }
      kw_phase ^= 1;
      cur_bh = bh;
      f_issued = false;
      __syncthreads();
      if (*abort_flag) break;
    }
    // (B) F = Q K~^T
    if (tid == 0 && !f_issued) {
      if (!mbar_wait(&bar_full[s], (j >> 1) & 1, abort_flag, kWaitNs)) {
        fail(p.status, abort_flag);
      } else {
        pend &= ~(1u << s);
        tc_fence_after_sync();
        issue_f(s);
      }
    }
    if (!mbar_wait(&bar_mma, mma_phase, abort_flag, kWaitNs)) fail(p.status, abort_flag);
    mma_phase ^= 1;
    __syncthreads();
    if (*abort_flag) break;
    tc_fence_after_sync();
    // (C) softmax over the m landmarks of row `tid`; P (bf16) overwrites F
    float mx = -INFINITY;
    for (int c0 = 0; c0 < p.m_pad; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + COL_F + c0, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (c0 + e < p.m) mx = fmaxf(mx, __uint_as_float(r[e]));
    }
    const float mc = mx * p.c;
    float l = 0.f;
    for (int c0 = 0; c0 < p.m_pad; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + COL_F + c0, r);
      tmem_ld_wait();
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float a = (c0 + 2 * e < p.m) ? fast_exp2(fmaf(__uint_as_float(r[2 * e]), p.c, -mc)) : 0.f;
        const float b = (c0 + 2 * e + 1 < p.m) ? fast_exp2(fmaf(__uint_as_float(r[2 * e + 1]), p.c, -mc)) : 0.f;
        l += a + b;
        pk[e] = pack_bf16x2(a, b);
      }
      tmem_st16(tmem + lane_off + COL_F + (c0 >> 1), pk);
    }
    tmem_st_wait();
    tc_fence_before_sync();
    __syncthreads();
    // (D) PW = P W ; CV = T V_halo
    if (tid == 0) {
      tc_fence_after_sync();
      const uint32_t ws_ = smem_u32(sm + p.off_wt);
      const uint32_t idw = idesc_bf16(128, DP, false, false);
      for (int kk = 0; kk < p.m_pad / 16; ++kk) {
        const uint64_t b = smem_desc(ws_ + (kk >> 2) * (DP * 128) + (kk & 3) * 32, 16, 1024, SW_128B);
        mma_bf16_tA(tmem + COL_PW, tmem + COL_F + kk * 8, b, idw, kk > 0);
      }
      if (p.kc > 0) {
        const uint32_t ts = smem_u32(sm + p.off_t);
        const uint32_t vs = smem_u32(sm + p.off_v + s * p.v_stage);
        const uint32_t idc = idesc_bf16(128, DP, false, true);
        for (int kk = 0; kk < p.kc / 16; ++kk) {
          const uint64_t a = smem_desc(ts + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, SW_128B);
          const uint64_t b = smem_desc(vs + kk * 2048, p.kc * 128, 1024, SW_128B);
          mma_bf16(tmem + COL_CV, a, b, idc, kk > 0);
        }
      }
      mma_commit(&bar_mma);
    }
    if (!mbar_wait(&bar_mma, mma_phase, abort_flag, kWaitNs)) fail(p.status, abort_flag);
    mma_phase ^= 1;
    __syncthreads();
    if (*abort_flag) break;
    tc_fence_after_sync();
    // (E) stage s is free: prefetch tile g+2; start F of tile g+1 (same head)
    f_issued = false;
    if (tid == 0) {
      if (g + 2 < g1) issue_load(s, g + 2);
      if (g + 1 < g1 && (g + 1) / p.tiles_per_head == bh) {
        const int s1 = (j + 1) & 1;
        if (!mbar_wait(&bar_full[s1], ((j + 1) >> 1) & 1, abort_flag, kWaitNs)) {
          fail(p.status, abort_flag);
        } else {
          pend &= ~(1u << s1);
          tc_fence_after_sync();
          issue_f(s1);
        }
      }
    }
    if (g + 1 < g1 && (g + 1) / p.tiles_per_head == bh) f_issued = true;
    // (F) out = PW / l + CV, bf16
    const int t = t0 + tid;
    const float inv_l = 1.f / l;
    __nv_bfloat16* orow = p.out + ((size_t)bh * p.n + t) * p.d;
#pragma unroll
    for (int c0 = 0; c0 < DP; c0 += 32) {
      uint32_t a[32], b[32];
      tmem_ld32(tmem + lane_off + COL_PW + c0, a);
      if (p.kc > 0) tmem_ld32(tmem + lane_off + COL_CV + c0, b);
      tmem_ld_wait();
      if (t < p.n && c0 < p.d) {
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
        uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e] = make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
      }
    }
    tc_fence_before_sync();
    __syncthreads();
  }
  // wind down: after an abort, wait (bounded) for copies still in flight
  if (tid == 0 && *abort_flag) {
    if (pend & 1u) mbar_wait(&bar_full[0], (nload0 - 1) & 1, nullptr, kWaitNs);
    if (pend & 2u) mbar_wait(&bar_full[1], (nload1 - 1) & 1, nullptr, kWaitNs);
    if (kw_pending) mbar_wait(&bar_kw, kw_phase ^ 1, nullptr, kWaitNs);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, p.tmem_cols);
}

int dpad_of(int d) { return d <= 64 ? 64 : 128; }

}  // namespace

// Shared-memory bytes the tensor-core token kernel needs for this shape
// (0 if the shape is outside what it handles).
size_t tokens_tc_smem(const Shape& s) {
  if (s.dtype != NYS_BF16) return 0;
  const int DP = dpad_of(s.d);
  const int m_pad = ((s.m + 31) / 32) * 32;
  const int kc = s.ks > 0 ? ((128 + s.ks - 1 + 15) / 16) * 16 : 0;
  if (kc > 256 || m_pad > 256) return 0;
  const size_t q_stage = 128 * DP * 2, v_stage = (size_t)kc * DP * 2;
  const size_t kt = (size_t)m_pad * DP * 2, wt = (size_t)((m_pad + 63) / 64) * DP * 128;
  const size_t tb = kc > 0 ? (size_t)((kc + 63) / 64) * 16384 : 0;
  const size_t total = 2 * q_stage + 2 * v_stage + kt + wt + tb + 1024;
  return total <= 227 * 1024 ? total : 0;
}

int launch_tokens_tc(const Shape& s, const void* q, const void* v, const void* kt_bf16,
                     const void* wt_bf16, const float* conv_w, void* out, int* status,
                     int num_sms, cudaStream_t stream) {
  const size_t smem = tokens_tc_smem(s);
  if (smem == 0) return NYS_ERR_UNSUPPORTED;
  const int DP = dpad_of(s.d);
  const int m_pad = ((s.m + 31) / 32) * 32;
  const int m64 = ((s.m + 63) / 64) * 64;
  const int kc = s.ks > 0 ? ((128 + s.ks - 1 + 15) / 16) * 16 : 0;
  const uint64_t BH = (uint64_t)s.bh();

  TokMaps maps;
  {
    const uint64_t dims[3] = {(uint64_t)s.d, (uint64_t)s.n, BH};
    const uint64_t strides[2] = {(uint64_t)s.d * 2, (uint64_t)s.n * s.d * 2};
    const uint32_t boxq[3] = {64, 128, 1};
    const uint32_t boxv[3] = {64, (uint32_t)(kc > 0 ? kc : 16), 1};
    if (!make_tensor_map(&maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, boxq,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, v, dims, strides, boxv,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return NYS_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {(uint64_t)DP, (uint64_t)m64, BH};
    const uint64_t strides[2] = {(uint64_t)DP * 2, (uint64_t)m64 * DP * 2};
    const uint32_t box[3] = {64, (uint32_t)m_pad, 1};
    if (!make_tensor_map(&maps.kt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kt_bf16, dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B))
      return NYS_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {(uint64_t)m64, (uint64_t)DP, BH};
    const uint64_t strides[2] = {(uint64_t)m64 * 2, (uint64_t)m64 * DP * 2};
    const uint32_t box[3] = {64, (uint32_t)DP, 1};
    if (!make_tensor_map(&maps.wt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, wt_bf16, dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B))
      return NYS_ERR_CUDA;
  }

  TokParams p{};
  p.conv_w = conv_w;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.status = status;
  p.H = s.H;
  p.n = s.n;
  p.d = s.d;
  p.m = s.m;
  p.m_pad = m_pad;
  p.ks = s.ks;
  p.kc = kc;
  p.tiles_per_head = (s.n + 127) / 128;
  p.total_tiles = (int)(BH * p.tiles_per_head);
  const int ctas = std::min(p.total_tiles, num_sms);
  p.tiles_per_cta = (p.total_tiles + ctas - 1) / ctas;
  const int grid = (p.total_tiles + p.tiles_per_cta - 1) / p.tiles_per_cta;
  p.c = (1.0f / sqrtf((float)s.d)) * 1.4426950408889634f;
  const uint32_t need = (uint32_t)(m_pad + 2 * DP);
  uint32_t cols = 32;
  while (cols < need) cols <<= 1;
  p.tmem_cols = cols;
  p.q_stage = 128 * DP * 2;
  p.v_stage = (uint32_t)kc * DP * 2;
  p.kt_bytes = (uint32_t)m_pad * DP * 2;
  p.wt_bytes = (uint32_t)((m_pad + 63) / 64) * DP * 128;
  p.off_q = 0;
  p.off_v = 2 * p.q_stage;
  p.off_kt = p.off_v + 2 * p.v_stage;
  p.off_wt = p.off_kt + p.kt_bytes;
  p.off_t = p.off_wt + p.wt_bytes;

  auto kern = DP == 64 ? tokens_tc<64> : tokens_tc<128>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return NYS_ERR_CUDA;
  KernelScope scope("tokens_tc", stream);
  kern<<<grid, 128, smem, stream>>>(maps, p);
  return cudaGetLastError() == cudaSuccess ? NYS_OK : NYS_ERR_CUDA;
}

}  // namespace nys
