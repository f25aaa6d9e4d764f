// Landmark rows on the tensor cores (bf16 inputs, fp32 accumulate):
//   G = softmax(Q~ K^T / sqrt(d)) V
// ("Nyströmformer" review page, Proposed method, bullets 3 and 6), computed
// as a split over keys: each CTA takes 128 landmark rows of one head and a
// contiguous range of 128-key tiles, and writes the unnormalised partial
// O = sum_j exp(s_ij - M_i) V_j with its (M_i, L_i = sum_j exp(s_ij - M_i)).
// The m x n scores never leave the chip. Per key tile:
//   S = Q~ K_tile^T           tcgen05, A = Q~ (smem), B = K tile (smem, TMA)
//   online softmax            thread = landmark row, from TMEM; the running
//                             max is re-based only when it grows by more
//                             than 2^8 (the accumulator is then rescaled in
//                             TMEM); P (bf16) overwrites S in TMEM
//   O += P V_tile             tcgen05, A = P (TMEM), B = V tile (MN-major)
// K and V tiles come in by TMA through a two-stage ring. Every wait is
// bounded; a wait that runs out sets the status word and the CTA winds down.
#include <cuda_bf16.h>

#include <algorithm>

#include "nys_internal.h"
#include "nys_sm100.h"
#include "nys_tma_host.h"

namespace nys {
namespace {

using namespace sm100;

struct RowMaps {
  CUtensorMap qt, k, v;
};

struct RowParams {
  float* gpart;  // [B*H][splits][m][d]
  float* gml;    // [B*H][splits][m][2]: (max in units of scaled scores, sum)
  int* status;
  int n, d, m, splits, tiles_per_split, n_tiles;
  float c;      // scale * log2(e)
  float scale;  // 1/sqrt(d)
  uint32_t tmem_cols;
};

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRebase = 8.0f;  // re-base the running max when it grows by > 2^8

__device__ __forceinline__ void fail(int* status, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicExch(status, (int)NYS_ERR_TIMEOUT);
}

template <int DP>
__global__ void __launch_bounds__(128, 1) rows_tc(const __grid_constant__ RowMaps maps,
                                               const RowParams p) {
  constexpr int DC = DP / 64;
  constexpr uint32_t TILE = DC * 16384;  // one 128-row tile of K or V, bytes
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* q_s = sm;               // [DC][128 rows][128 B]
  uint8_t* k_s = sm + TILE;        // [2][DC][128][128 B]
  uint8_t* v_s = sm + 3 * TILE;    // [2][DC][128][128 B]
  __shared__ uint64_t bar_q, bar_full[2], bar_mma;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  volatile int* abort_flag = &abort_sh;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int rb = blockIdx.x, split = blockIdx.y, bh = blockIdx.z;
  const int tile0 = split * p.tiles_per_split;
  const int ntile = min(p.n_tiles, tile0 + p.tiles_per_split) - tile0;
  const int row = rb * 128 + tid;

  if (tid == 0) {
    mbar_init(&bar_q, 1);
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_init(&bar_mma, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base_sh, p.tmem_cols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  constexpr uint32_t COL_S = 0, COL_O = 128;

  uint32_t pend = 0;                  // bit s: a load into stage s not yet waited on
  uint32_t nload0 = 0, nload1 = 0;    // loads issued into stage 0 / 1
  bool q_pending = false;
  auto issue_load = [&](int stage, int j) {
    const int key0 = (tile0 + j) * 128;
    mbar_arrive_expect_tx(&bar_full[stage], 2 * TILE);
#pragma unroll
    for (int dc = 0; dc < DC; ++dc) {
      tma_load_3d(k_s + stage * TILE + dc * 16384, &maps.k, &bar_full[stage], dc * 64, key0, bh);
      tma_load_3d(v_s + stage * TILE + dc * 16384, &maps.v, &bar_full[stage], dc * 64, key0, bh);
    }
    pend |= 1u << stage;
    if (stage) ++nload1; else ++nload0;
  };
  if (tid == 0 && ntile > 0) {
    mbar_arrive_expect_tx(&bar_q, TILE);
#pragma unroll
    for (int dc = 0; dc < DC; ++dc) tma_load_3d(q_s + dc * 16384, &maps.qt, &bar_q, dc * 64, rb * 128, bh);
    q_pending = true;
    issue_load(0, 0);
    if (ntile > 1) issue_load(1, 1);
    if (!mbar_wait(&bar_q, 0, abort_flag, kWaitNs)) fail(p.status, abort_flag);
    else q_pending = false;
  }

  float m_run = -INFINITY, l_run = 0.f;
  uint32_t mma_phase = 0;
  const bool live = row < p.m;
  for (int j = 0; j < ntile; ++j) {
    const int s = j & 1;
    // S = Q~ K_tile^T
    if (tid == 0 && !*abort_flag) {
      if (!mbar_wait(&bar_full[s], (j >> 1) & 1, abort_flag, kWaitNs)) {
        fail(p.status, abort_flag);
      } else {
        pend &= ~(1u << s);
        tc_fence_after_sync();
        const uint32_t qa = smem_u32(q_s), kb = smem_u32(k_s + s * TILE);
        const uint32_t id = idesc_bf16(128, 128, false, false);
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk) {
          const uint64_t a = smem_desc(qa + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, SW_128B);
          const uint64_t b = smem_desc(kb + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, SW_128B);
          mma_bf16(tmem + COL_S, a, b, id, kk > 0);
        }
        mma_commit(&bar_mma);
      }
    }
    if (!mbar_wait(&bar_mma, mma_phase, abort_flag, kWaitNs)) fail(p.status, abort_flag);
    mma_phase ^= 1;
    __syncthreads();
    if (*abort_flag) break;
    tc_fence_after_sync();
    // online softmax of this row over the tile's keys. TMEM loads and
    // stores are warp-collective, so every lane takes part; padding rows
    // (row >= m) only feed zeros to the P V product.
    const int key0 = (tile0 + j) * 128;
    {
      float tmax = -INFINITY;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + COL_S + c0, r);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (key0 + c0 + e < p.n) tmax = fmaxf(tmax, __uint_as_float(r[e]));
        }
      }
      const bool rebase = live && (m_run == -INFINITY || (tmax - m_run) * p.c > kRebase);
      float alpha = 1.f;
      if (rebase) {
        alpha = (m_run == -INFINITY) ? 0.f : fast_exp2((m_run - tmax) * p.c);
        l_run *= alpha;
        m_run = tmax;
      }
      if (j > 0 && __any_sync(0xffffffffu, rebase)) {
        // rescale the accumulator rows (all earlier MMAs are done)
#pragma unroll
        for (int c0 = 0; c0 < DP; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + COL_O + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tmem_st32(tmem + lane_off + COL_O + c0, r);
        }
      }
      const float mc = m_run * p.c;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + COL_S + c0, r);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int ka = key0 + c0 + 2 * e;
          const float a = (live && ka < p.n) ? fast_exp2(fmaf(__uint_as_float(r[2 * e]), p.c, -mc)) : 0.f;
          const float b = (live && ka + 1 < p.n) ? fast_exp2(fmaf(__uint_as_float(r[2 * e + 1]), p.c, -mc)) : 0.f;
          l_run += a + b;
          pk[e] = pack_bf16x2(a, b);
        }
        tmem_st16(tmem + lane_off + COL_S + (c0 >> 1), pk);
      }
    }
    tmem_st_wait();
    tc_fence_before_sync();
    __syncthreads();
    // O += P V_tile
    if (tid == 0) {
      tc_fence_after_sync();
      const uint32_t vb = smem_u32(v_s + s * TILE);
      const uint32_t id = idesc_bf16(128, DP, false, true);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t b = smem_desc(vb + kk * 2048, 16384, 1024, SW_128B);
        mma_bf16_tA(tmem + COL_O, tmem + COL_S + kk * 8, b, id, (j > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(&bar_mma);
    }
    if (!mbar_wait(&bar_mma, mma_phase, abort_flag, kWaitNs)) fail(p.status, abort_flag);
    mma_phase ^= 1;
    __syncthreads();
    if (*abort_flag) break;
    tc_fence_after_sync();
    if (tid == 0 && j + 2 < ntile) issue_load(s, j + 2);
  }
  // partial result of this CTA: O row (unnormalised), max, sum
  if (!*abort_flag && ntile > 0) {
    const size_t prow = ((size_t)bh * p.splits + split) * p.m + row;
    float* o = p.gpart + prow * p.d;
#pragma unroll
    for (int c0 = 0; c0 < DP; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + COL_O + c0, r);
      tmem_ld_wait();
      if (live && c0 < p.d) {
        float4* dst = reinterpret_cast<float4*>(o + c0);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          dst[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                               __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
      }
    }
    if (live) {
      p.gml[prow * 2 + 0] = m_run * p.scale;
      p.gml[prow * 2 + 1] = l_run;
    }
  }
  if (tid == 0 && *abort_flag) {
    if (q_pending) mbar_wait(&bar_q, 0, nullptr, kWaitNs);
    if (pend & 1u) mbar_wait(&bar_full[0], (nload0 - 1) & 1, nullptr, kWaitNs);
    if (pend & 2u) mbar_wait(&bar_full[1], (nload1 - 1) & 1, nullptr, kWaitNs);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, p.tmem_cols);
}

}  // namespace

// Key splits and tiles of the tensor-core landmark-row kernel (host math).
void rows_tc_split(const Shape& s, int* splits, int* tiles_per_split) {
  const int n_tiles = (s.n + 127) / 128;
  const long long rb = (s.m + 127) / 128;
  long long want = (2 * 152 + rb * s.bh() - 1) / (rb * s.bh());
  if (want > n_tiles) want = n_tiles;
  if (want < 1) want = 1;
  const int tps = (int)((n_tiles + want - 1) / want);
  *tiles_per_split = tps;
  *splits = (n_tiles + tps - 1) / tps;
}

int launch_rows_tc(const Shape& s, const void* qt_bf16, const void* k, const void* v, float* gpart,
                   float* gml, int splits, int tiles_per_split, int* status, cudaStream_t stream) {
  const int DP = s.dpad();
  const int m64 = s.m64();
  const uint64_t BH = (uint64_t)s.bh();
  RowMaps maps;
  {
    const uint64_t dims[3] = {(uint64_t)DP, (uint64_t)m64, BH};
    const uint64_t strides[2] = {(uint64_t)DP * 2, (uint64_t)m64 * DP * 2};
    const uint32_t box[3] = {64, 128, 1};
    if (!make_tensor_map(&maps.qt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, qt_bf16, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return NYS_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {(uint64_t)s.d, (uint64_t)s.n, BH};
    const uint64_t strides[2] = {(uint64_t)s.d * 2, (uint64_t)s.n * s.d * 2};
    const uint32_t box[3] = {64, 128, 1};
    if (!make_tensor_map(&maps.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, v, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return NYS_ERR_CUDA;
  }
  RowParams p{};
  p.gpart = gpart;
  p.gml = gml;
  p.status = status;
  p.n = s.n;
  p.d = s.d;
  p.m = s.m;
  const int sp = splits, tps = tiles_per_split;
  p.splits = sp;
  p.tiles_per_split = tps;
  p.n_tiles = (s.n + 127) / 128;
  p.scale = 1.0f / sqrtf((float)s.d);
  p.c = p.scale * 1.4426950408889634f;
  p.tmem_cols = DP == 64 ? 256 : 256;
  const int TILE = (DP / 64) * 16384;
  const size_t smem = 5 * (size_t)TILE + 1024;
  auto kern = DP == 64 ? rows_tc<64> : rows_tc<128>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return NYS_ERR_CUDA;
  KernelScope scope("rows_tc", stream);
  kern<<<dim3((s.m + 127) / 128, sp, (unsigned)BH), 128, smem, stream>>>(maps, p);
  return cudaGetLastError() == cudaSuccess ? NYS_OK : NYS_ERR_CUDA;
}

}  // namespace nys
