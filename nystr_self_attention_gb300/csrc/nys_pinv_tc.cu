// Landmark kernel, iterative pseudo-inverse and W = Z G on the tensor cores
// ("Nyströmformer" review page, Proposed method, bullets 2, 3 and 5), for
// m <= 128 landmarks:
//   G   = merge of the key-split partials of softmax(Q~ K^T s) V
//   A_S = softmax(Q~ K~^T s)   scores as three tf32 products of the hi/lo
//                              split of Q~ and K~ (hi*hi + hi*lo + lo*hi,
//                              the error-corrected tf32 GEMM of Ootomo and
//                              Yokota, 2022): close to fp32 accuracy
//   Z_0 = A_S^T / (||A_S||_1 ||A_S||_inf)
//   iters x:  X = A_S Z;  Y1 = X (7I - X);  Y2 = X (15I - Y1);
//             Z <- 1/4 Z (13I - Y2)               tcgen05 kind::tf32
//   W   = Z G                                      tcgen05 kind::tf32
// The products run on tf32 operands with fp32 accumulation and fp32
// storage; the update is the paper's own (Z recomputed through A_S Z every
// step), not a reformulation.
//
// m is padded to MP = 32, 64 or 128 (the zero padding is exact: the padded
// block of every iterate stays zero) and hp = 128 / MP heads (fewer if d
// is large) share one CTA of 256 threads, stacked along the 128 TMEM lanes:
// row i of head slot h is lane h MP + i. One M = 128 MMA then serves all hp
// heads: the B operand stacks the heads' right factors along N, and each
// head reads only its own diagonal block of the 128 x (hp MP) result (the
// off-diagonal blocks mix heads and are never read). A_S is the A operand
// of X = A_S Z from shared memory; X and Z are A operands in TMEM; each
// product's B operand is written, transposed, into one shared-memory
// buffer by the epilogue of the product before it.
//
// Z-only mode (z given): no merge and no W; Z goes out in fp32 so that the
// kernel can run before the key-split partials exist. The second kernel
// here, w_tc, then forms W = Z G from Z and the G merged by merge_g (16 to
// 64 columns of a head per CTA).
#include <cuda_bf16.h>

#include <algorithm>

#include "nys_internal.h"
#include "nys_sm100.h"

namespace nys {
namespace {

using namespace sm100;

struct PinvParams {
  const float* qt;     // [B*H][m][d] fp32
  const float* kt;     // [B*H][m][d] fp32
  const float* gpart;  // [B*H][splits][m][d]
  const float* gml;    // [B*H][splits][m][2]
  float* g;            // [B*H][m][d]  stage export
  float* a_s;          // [B*H][m][m]  stage export
  float* z;            // [B*H][m][m]  Z out (stage export; the Z-only mode's result)
  float* w;            // [B*H][m][d]  stage export
  __nv_bfloat16* wt;   // [B*H][dpad][m64] zero padded
  int* status;
  int BH, m, d, dpad, m64, splits, iters;
  int z_only;     // Z only: no merge of the partials, no W
  uint32_t stall_ns;  // > 0: wait this long on a phase nothing completes (timeout test)
  int hp;         // heads per CTA
  float scale;    // 1/sqrt(d)
  float c;        // scale * log2(e)
  uint32_t tmem_cols;
  uint32_t abuf_off, bbuf_off, klo_off;  // smem offsets (G^T at 0)
  uint32_t abuf_lo_off, bbuf_lo_off, gbuf_lo_off;  // three-product mode: lo halves
};

constexpr uint64_t kWaitNs = 2000000000ull;

// byte offset of element (row, col) of a K-major SWIZZLE_128B fp32 operand
// with `rows` rows: 32-column chunks of [rows x 128 B]
__device__ __forceinline__ uint32_t kmaj_off(int row, int col, int rows) {
  return (uint32_t)(col >> 5) * (uint32_t)(rows * 128) + sw128_offset(row, (col & 31) * 4);
}

// v[e] -> element (j0 + e, col) for e < 32: one column of 32 rows. The
// swizzle term depends on e only through e % 8, so the 32 addresses are 8
// register offsets plus immediates.
__device__ __forceinline__ void store_col32(uint8_t* buf, int rows, int col, int j0,
                                            const float (&v)[32]) {
  uint8_t* base = buf + (uint32_t)(col >> 5) * (uint32_t)(rows * 128) + (uint32_t)j0 * 128u +
                  (uint32_t)(col & 3) * 4u;
  const uint32_t L = (uint32_t)(col & 31) >> 2;
#pragma unroll
  for (int e = 0; e < 32; ++e)
    *reinterpret_cast<float*>(base + e * 128 + ((L ^ (uint32_t)(e & 7)) << 4)) = v[e];
}

// v[e] -> element (j0 + e, col) for e < 16 (j0 % 8 == 0), as store_col32
__device__ __forceinline__ void store_col16(uint8_t* buf, int rows, int col, int j0,
                                            const float (&v)[16]) {
  uint8_t* base = buf + (uint32_t)(col >> 5) * (uint32_t)(rows * 128) + (uint32_t)j0 * 128u +
                  (uint32_t)(col & 3) * 4u;
  const uint32_t L = (uint32_t)(col & 31) >> 2;
#pragma unroll
  for (int e = 0; e < 16; ++e)
    *reinterpret_cast<float*>(base + e * 128 + ((L ^ (uint32_t)(e & 7)) << 4)) = v[e];
}

// four consecutive elements (row, c .. c+3), c % 4 == 0, as one 16-byte store
__device__ __forceinline__ void store_row4(uint8_t* buf, int rows, int row, int c, float4 v) {
  *reinterpret_cast<float4*>(buf + kmaj_off(row, c, rows)) = v;
}

__device__ __forceinline__ float ld_elem(const uint8_t* buf, int rows, int row, int col) {
  return *reinterpret_cast<const float*>(buf + kmaj_off(row, col, rows));
}

__device__ __forceinline__ float tf32_hi(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// 256 threads: warp w works on TMEM lane quarter w % 4 (rows 32 (w % 4) ..
// + 31); the two warps of a quarter split each row's 32-column chunks
// (half h = w / 4 takes the chunks with index % 2 == h).
constexpr int kThreads = 256;

// tf32 hi / lo split: hi keeps the leading 11 significand bits (exact in
// tf32), lo = x - hi (exact in fp32)
__device__ __forceinline__ void split_tf32(float x, float& h, float& l) {
  h = tf32_hi(x);
  l = x - h;
}

// X3: every product as three tf32 products of its operands' hi / lo halves
// (A_hi B_hi + A_lo B_hi + A_hi B_lo), for fp32 inputs (MP <= 64): the lo
// halves of A_S, of the B operand and of G^T sit in shared memory beside
// the hi halves, those of Z and X in TMEM beside theirs.
// THREE: each update in three dependent levels of products instead of four
// (X = A_S Z; X X and Z X side by side over one B operand; Z' = 1/4 (13 Z -
// 15 Z X + Z X (7X - X^2)) accumulated onto 13 Z - 15 Z X), with a second
// accumulator in TMEM: where one CTA per SM runs anyway.
template <int MP, bool X3, bool THREE>
__global__ void __launch_bounds__(kThreads, (MP == 128 || X3 || THREE) ? 1 : 2)
    pinv_tc(const __grid_constant__ PinvParams p) {
  constexpr int NCH = MP / 32;  // 32-column chunks of a head's m x m block
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int hp = p.hp, NP = hp * MP;  // N of the stacked m x m products (<= 128)
  const int NW = hp * p.d;            // N of the stacked W = Z G (<= 256)
  uint8_t* gbuf = sm;                 // G^T, heads stacked:   [NW rows x MP]
  uint8_t* abuf = sm + p.abuf_off;    // A_S (A operand):      [128 rows x MP]
  uint8_t* bbuf = sm + p.bbuf_off;    // B operand:            [NP rows x MP]
  uint8_t* khi = abuf;                // K~ hi / lo, stacked:  [NP rows x d]
  uint8_t* klo = sm + p.klo_off;      //   (score step only, over abuf / bbuf)
  uint8_t* abuf_lo = sm + p.abuf_lo_off;  // X3 only
  uint8_t* bbuf_lo = sm + p.bbuf_lo_off;
  uint8_t* gbuf_lo = sm + p.gbuf_lo_off;
  __shared__ uint64_t bar_mma;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float red_rmax[2][128], red_rsum[2][128], red_rs[2][128], red_cs[2][128];
  __shared__ float red_q[2][4];  // per lane quarter: largest row / column abs-sum
  volatile int* abort_flag = &abort_sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int row = quarter * 32 + lane;     // TMEM lane
  const int hs = row / MP, li = row % MP;  // head slot (warp-uniform), row in the head
  const int bh = (int)blockIdx.x * hp + hs;
  const bool head_ok = hs < hp && bh < p.BH;  // warp-uniform
  const int m = p.m, d = p.d;
  const bool live = head_ok && li < m;
  const bool in_np = row < NP;

  __shared__ uint64_t bar_fin, bar_never;
  if (tid == 0) {
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_fin, 1);
    mbar_init(&bar_never, 1);  // nothing ever arrives on it
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base_sh, p.tmem_cols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // The timeout path on demand: before any copy or product is in flight, a
  // bounded wait on a phase that nothing completes runs out, and the CTA
  // winds down as after any timeout (status word set, no further work).
  if (p.stall_ns > 0) {
    if (tid == 0 && !mbar_wait(&bar_never, 0, nullptr, p.stall_ns)) {
      *abort_flag = 1;
      atomicExch(p.status, (int)NYS_ERR_TIMEOUT);
    }
    __syncthreads();
  }
  const uint32_t tmem = tmem_base_sh;
  const uint32_t lo = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t COL_Z = 0, COL_X = MP, COL_D = 2 * MP;  // main loop
  // THREE: the second accumulator (Z X) after the product region; X3: lo
  // halves of Z and X after those
  const uint32_t COL_D2 = COL_D + (uint32_t)max(NP, NW);
  const uint32_t COL_ZL = COL_D2 + (THREE ? (uint32_t)NP : 0u), COL_XL = COL_ZL + MP;
  const uint32_t COL_QH = 0, COL_QL = d, COL_S = 2 * d;  // score step
  const uint32_t dblk = (uint32_t)(hs * MP);  // this head's block of a stacked result

  uint32_t phase = 0;
  // tf32 product D (+)= A x B, M = 128, N = b_rows, K = k_dim. A from TMEM
  // columns a_col.. or, if a_smem is set, from shared memory (K-major,
  // 128 rows); B from shared memory (K-major, b_rows rows).
  auto issue1 = [&](uint32_t d_col, uint32_t a_col, const uint8_t* a_smem, const uint8_t* b,
                    int b_rows, int k_dim, bool acc_first) {
    const uint64_t b0 = smem_desc(smem_u32(b), 16, 1024, SW_128B);
    const uint32_t id = idesc_tf32(128, b_rows);
    const uint32_t bchunk = (uint32_t)b_rows * 8u;  // (b_rows * 128 B) >> 4
    if (a_smem) {
      const uint64_t a0 = smem_desc(smem_u32(a_smem), 16, 1024, SW_128B);
#pragma unroll 4
      for (int kk = 0; kk < k_dim / 8; ++kk) {
        const uint32_t step = (uint32_t)(kk & 3) * 2u;  // 8 tf32 = 32 B
        mma_tf32(tmem + d_col, a0 + (uint64_t)((uint32_t)(kk >> 2) * 1024u + step),
                 b0 + (uint64_t)((uint32_t)(kk >> 2) * bchunk + step), id,
                 (kk > 0 || acc_first) ? 1u : 0u);
      }
    } else {
#pragma unroll 4
      for (int kk = 0; kk < k_dim / 8; ++kk) {
        const uint64_t bd = b0 + (uint64_t)((uint32_t)(kk >> 2) * bchunk + (uint32_t)(kk & 3) * 2u);
        mma_tf32_tA(tmem + d_col, tmem + a_col + kk * 8, bd, id, (kk > 0 || acc_first) ? 1u : 0u);
      }
    }
  };
  // one product; X3: A_hi B_hi + A_lo B_hi + A_hi B_lo, the lo halves at
  // a_col_lo / a_smem_lo and b_lo
  auto issue = [&](uint32_t d_col, uint32_t a_col, uint32_t a_col_lo, const uint8_t* a_smem,
                   const uint8_t* a_smem_lo, const uint8_t* b, const uint8_t* b_lo, int b_rows,
                   int k_dim, bool acc = false) {
    issue1(d_col, a_col, a_smem, b, b_rows, k_dim, acc);
    if constexpr (X3) {
      issue1(d_col, a_col_lo, a_smem ? a_smem_lo : nullptr, b, b_rows, k_dim, true);
      issue1(d_col, a_col, a_smem, b_lo, b_rows, k_dim, true);
    }
  };
  auto wait_mma = [&]() {
    if (!mbar_wait(&bar_mma, phase, abort_flag, kWaitNs)) {
      *abort_flag = 1;
      atomicExch(p.status, (int)NYS_ERR_TIMEOUT);
    }
    phase ^= 1;
    tc_fence_after_sync();
  };

  // ---- 1) the merge of G runs after the iteration (W is its only user);
  // its partial rows are prefetched into L2 here so that it then waits on
  // L2 rather than on DRAM
  const bool z_only = p.z_only != 0;  // uniform
  if (!z_only && live)
    for (int sp = 0; sp < p.splits; ++sp) {
      const size_t prow = ((size_t)bh * p.splits + sp) * m + li;
      for (int c0 = half * 32; c0 < d; c0 += 64)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.gpart + prow * d + c0));
      if (half == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.gml + prow * 2));
    }

  // ---- 2) scores S = Q~ K~^T in 3xTF32: Q~ hi / lo rows -> TMEM (A), K~
  // hi / lo rows -> shared memory (B, head slot hs at rows hs MP ..)
  {
    const float* qrow = p.qt + ((size_t)(live ? bh : 0) * m + (live ? li : 0)) * d;
    const float* krow = p.kt + ((size_t)(live ? bh : 0) * m + (live ? li : 0)) * d;
    for (int c0 = half * 32; c0 < d; c0 += 64) {
      // all 16 loads in flight before the first shared-memory store
      float4 kv[8], qv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        kv[e] = live ? __ldg(reinterpret_cast<const float4*>(krow + c0) + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        qv[e] = live ? __ldg(reinterpret_cast<const float4*>(qrow + c0) + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (in_np) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 kh = make_float4(tf32_hi(kv[e].x), tf32_hi(kv[e].y), tf32_hi(kv[e].z), tf32_hi(kv[e].w));
          store_row4(khi, NP, row, c0 + 4 * e, kh);
          store_row4(klo, NP, row, c0 + 4 * e,
                     make_float4(kv[e].x - kh.x, kv[e].y - kh.y, kv[e].z - kh.z, kv[e].w - kh.w));
        }
      }
      uint32_t qh[32], ql[32];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float q4[4] = {qv[e].x, qv[e].y, qv[e].z, qv[e].w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float hh = tf32_hi(q4[t]);
          qh[4 * e + t] = __float_as_uint(hh);
          ql[4 * e + t] = __float_as_uint(q4[t] - hh);
        }
      }
      tmem_st32(tmem + lo + COL_QH + c0, qh);
      tmem_st32(tmem + lo + COL_QL + c0, ql);
    }
  }
  fence_async_smem();
  tmem_st_wait();
  tc_fence_before_sync();
  __syncthreads();
  if (tid == 0 && !*abort_flag) {
    tc_fence_after_sync();
    issue1(COL_S, COL_QH, nullptr, khi, NP, d, false);
    issue1(COL_S, COL_QH, nullptr, klo, NP, d, true);
    issue1(COL_S, COL_QL, nullptr, khi, NP, d, true);
    mma_commit(&bar_mma);
  }
  wait_mma();
  __syncthreads();

  // ---- 3) row softmax over the head's own block of S (scale 1/sqrt(d));
  // half h takes the chunks c = h, h + 2 (both in flight at once), the two
  // halves combine the row max and sum through shared memory. A_S rows ->
  // abuf (A operand of X = A_S Z).
  {
    const int nmine = head_ok ? (NCH - half + 1) >> 1 : 0;  // 0, 1 or 2, warp-uniform
    const int j0 = half * 32, j1 = (half + 2) * 32;
    uint32_t r0[32], r1[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) r0[e] = r1[e] = 0u;
    if (nmine > 0) tmem_ld32(tmem + lo + COL_S + dblk + j0, r0);
    if (nmine > 1) tmem_ld32(tmem + lo + COL_S + dblk + j1, r1);
    tmem_ld_wait();
    float pm = -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      if (nmine > 0 && j0 + e < m) pm = fmaxf(pm, __uint_as_float(r0[e]));
      if (nmine > 1 && j1 + e < m) pm = fmaxf(pm, __uint_as_float(r1[e]));
    }
    red_rmax[half][row] = pm;
    __syncthreads();
    const float mc = fmaxf(red_rmax[0][row], red_rmax[1][row]) * p.c;
    float ps = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float x0 = (live && nmine > 0 && j0 + e < m) ? fast_exp2(fmaf(__uint_as_float(r0[e]), p.c, -mc)) : 0.f;
      const float x1 = (live && nmine > 1 && j1 + e < m) ? fast_exp2(fmaf(__uint_as_float(r1[e]), p.c, -mc)) : 0.f;
      ps += x0 + x1;
      r0[e] = __float_as_uint(x0);
      r1[e] = __float_as_uint(x1);
    }
    red_rsum[half][row] = ps;
    __syncthreads();
    const float inv = live ? 1.f / (red_rsum[0][row] + red_rsum[1][row]) : 0.f;
    float rs = 0.f;
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      float a[8];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        a[t] = __uint_as_float(r0[e + t]) * inv;
        a[4 + t] = __uint_as_float(r1[e + t]) * inv;
        rs += fabsf(a[t]) + fabsf(a[4 + t]);
      }
      if (half < NCH) store_row4(abuf, 128, row, j0 + e, make_float4(a[0], a[1], a[2], a[3]));
      if (half + 2 < NCH) store_row4(abuf, 128, row, j1 + e, make_float4(a[4], a[5], a[6], a[7]));
    }
    red_rs[half][row] = rs;
  }
  __syncthreads();
  // ||A_S||_1 per head: thread (row hs MP + j, half) sums column j of its
  // head over half of the rows (four independent partial sums)
  {
    float c4[4] = {0.f, 0.f, 0.f, 0.f};
    if (live) {
      const int i0 = half * (MP >> 1), i1 = i0 + (MP >> 1);
      for (int i = i0; i < i1; i += 4) {
#pragma unroll
        for (int t = 0; t < 4; ++t) c4[t] += fabsf(ld_elem(abuf, 128, hs * MP + i + t, li));
      }
    }
    red_cs[half][row] = (c4[0] + c4[1]) + (c4[2] + c4[3]);
  }
  __syncthreads();
  // per lane quarter: largest row abs-sum and largest column abs-sum
  if (half == 0) {
    float rs = live ? red_rs[0][row] + red_rs[1][row] : 0.f;
    float cs = live ? red_cs[0][row] + red_cs[1][row] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      rs = fmaxf(rs, __shfl_xor_sync(0xffffffffu, rs, o));
      cs = fmaxf(cs, __shfl_xor_sync(0xffffffffu, cs, o));
    }
    if (lane == 0) {
      red_q[0][quarter] = rs;
      red_q[1][quarter] = cs;
    }
  }
  __syncthreads();
  float alpha = 0.f;
  {
    // the lane quarters of this head: [hs MP / 32, (hs + 1) MP / 32)
    float ninf = 0.f, n1 = 0.f;
    for (int q = hs * MP / 32; q < (hs + 1) * MP / 32 && q < 4; ++q) {
      ninf = fmaxf(ninf, red_q[0][q]);
      n1 = fmaxf(n1, red_q[1][q]);
    }
    if (head_ok) alpha = 1.f / (n1 * ninf);
  }
  // Z_0 = alpha A_S^T -> TMEM: row i of Z_0 is alpha * column i of A_S
  if (head_ok) {
    for (int c = half; c < NCH; c += 2) {
      uint32_t r[32], rl[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x = alpha * ld_elem(abuf, 128, hs * MP + c * 32 + e, li);
        float h = x, l = 0.f;
        if constexpr (X3) split_tf32(x, h, l);
        r[e] = __float_as_uint(h);
        rl[e] = __float_as_uint(l);
      }
      tmem_st32(tmem + lo + COL_Z + c * 32, r);
      if constexpr (X3) tmem_st32(tmem + lo + COL_ZL + c * 32, rl);
    }
  }
  // B operand of X = A_S Z_0: row hs MP + j holds column j of Z_0, i.e.
  // alpha * row j of A_S
  if (in_np)
    for (int c = half; c < NCH; c += 2)
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        float4 v = *reinterpret_cast<const float4*>(abuf + kmaj_off(row, c * 32 + e, 128));
        v.x *= alpha; v.y *= alpha; v.z *= alpha; v.w *= alpha;
        if constexpr (X3) {
          float4 h, l;
          split_tf32(v.x, h.x, l.x);
          split_tf32(v.y, h.y, l.y);
          split_tf32(v.z, h.z, l.z);
          split_tf32(v.w, h.w, l.w);
          store_row4(bbuf, NP, row, c * 32 + e, h);
          store_row4(bbuf_lo, NP, row, c * 32 + e, l);
        } else {
          store_row4(bbuf, NP, row, c * 32 + e, v);
        }
      }
  fence_async_smem();
  tmem_st_wait();
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (X3) {
    // A_S -> hi in place and lo beside it (the norms and Z_0 have read it;
    // the stage export reads hi + lo, which is A_S exactly)
    for (int c = half; c < NCH; c += 2)
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const uint32_t off = kmaj_off(row, c * 32 + e, 128);
        const float4 v = *reinterpret_cast<const float4*>(abuf + off);
        float4 h, l;
        split_tf32(v.x, h.x, l.x);
        split_tf32(v.y, h.y, l.y);
        split_tf32(v.z, h.z, l.z);
        split_tf32(v.w, h.w, l.w);
        *reinterpret_cast<float4*>(abuf + off) = h;
        *reinterpret_cast<float4*>(abuf_lo + off) = l;
      }
    fence_async_smem();
    __syncthreads();
  }

  // ---- 4) the iteration
  // Stage export of A_S (abuf is constant from here on): seven rows per
  // call, one per warp 1-7, coalesced. It runs while thread 0 issues a
  // product's MMAs, when the other threads would only wait; warp 0 (the
  // issuer's) takes no rows, so the export never delays the issue.
  int exp_row = 0;
  auto export_rows = [&]() {
    const int r = exp_row + warp - 1;
    exp_row += kThreads / 32 - 1;
    if (warp == 0) return;
    if (r >= hp * m) return;
    const int h2 = r / m, i = r - h2 * m;
    const int bh2 = (int)blockIdx.x * hp + h2;
    if (bh2 >= p.BH) return;
    float* a_out = p.a_s + ((size_t)bh2 * m + i) * m;
    for (int j = lane; j < m; j += 32)
      a_out[j] = X3 ? ld_elem(abuf, 128, h2 * MP + i, j) + ld_elem(abuf_lo, 128, h2 * MP + i, j)
                    : ld_elem(abuf, 128, h2 * MP + i, j);
  };
  auto gemm = [&](uint32_t a_col, const uint8_t* a_smem) {
    if (tid == 0) {
      tc_fence_after_sync();
      issue(COL_D, a_col, a_col == COL_Z ? COL_ZL : COL_XL, a_smem, abuf_lo, bbuf, bbuf_lo, NP, MP);
      mma_commit(&bar_mma);
    }
    if (exp_row < hp * m) export_rows();
    wait_mma();
  };
  // epilogue: the head's block of this row of D -> sign * scale * D + diag
  // * I, written transposed as the next product's B operand (element
  // (i, j) of the head -> storage row hs MP + j, column i); optionally also
  // scale * D -> TMEM columns to_col.. (an A operand).
  auto store_chunk = [&](int j0, uint32_t (&r)[32], float diag, float sign, float scale_,
                         int to_col) {
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float x = scale_ * __uint_as_float(r[e]);
      r[e] = __float_as_uint(x);
      v[e] = fmaf(sign, x, (j0 + e == li) ? diag : 0.f);
    }
    if constexpr (X3) {
      float vl[32];
      uint32_t rl[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        split_tf32(v[e], v[e], vl[e]);
        float h, l;
        split_tf32(__uint_as_float(r[e]), h, l);
        r[e] = __float_as_uint(h);
        rl[e] = __float_as_uint(l);
      }
      store_col32(bbuf_lo, NP, li, hs * MP + j0, vl);
      if (to_col >= 0) tmem_st32(tmem + lo + (to_col == (int)COL_X ? COL_XL : COL_ZL) + j0, rl);
    }
    store_col32(bbuf, NP, li, hs * MP + j0, v);
    if (to_col >= 0) tmem_st32(tmem + lo + (uint32_t)to_col + j0, r);
  };
  auto store_bt = [&](float diag, float sign, float scale_, int to_col) {
    if (head_ok) {
      if constexpr (NCH == 4) {  // chunks half and half + 2: both loads in flight
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem + lo + COL_D + dblk + half * 32, r0);
        tmem_ld32(tmem + lo + COL_D + dblk + (half + 2) * 32, r1);
        tmem_ld_wait();
        store_chunk(half * 32, r0, diag, sign, scale_, to_col);
        store_chunk((half + 2) * 32, r1, diag, sign, scale_, to_col);
      } else {
        for (int c = half; c < NCH; c += 2) {
          uint32_t r[32];
          tmem_ld32(tmem + lo + COL_D + dblk + c * 32, r);
          tmem_ld_wait();
          store_chunk(c * 32, r, diag, sign, scale_, to_col);
        }
      }
    }
    fence_async_smem();
    tmem_st_wait();
    tc_fence_before_sync();
    __syncthreads();
  };
  // three levels: X X -> D and Z X -> D2 over one B operand (X)
  auto gemm2 = [&]() {
    if (tid == 0) {
      tc_fence_after_sync();
      issue(COL_D, COL_X, COL_XL, nullptr, nullptr, bbuf, bbuf_lo, NP, MP);
      issue(COL_D2, COL_Z, COL_ZL, nullptr, nullptr, bbuf, bbuf_lo, NP, MP);
      mma_commit(&bar_mma);
    }
    if (exp_row < hp * m) export_rows();
    wait_mma();
  };
  // D (holding 13 Z - 15 Z X) += Z X (7X - X^2): A = Z X (TMEM, in X's columns)
  auto gemm3 = [&]() {
    if (tid == 0) {
      tc_fence_after_sync();
      issue(COL_D, COL_X, COL_XL, nullptr, nullptr, bbuf, bbuf_lo, NP, MP, true);
      mma_commit(&bar_mma);
    }
    if (exp_row < hp * m) export_rows();
    wait_mma();
  };
  // the level-2 epilogue, 16 columns at a time of this row of the head's
  // blocks of X X (D), Z X (D2), X and Z: B <- 7X - X^2 (transposed), X's
  // columns <- Z X (the A operand of the last level), D <- 13 Z - 15 Z X
  auto epi2 = [&]() {
    if (head_ok) {
      for (int c = half; c < MP / 16; c += 2) {
        const int j0 = c * 16;
        uint32_t x2[16], zx[16], xv[16], zv[16], xl[16], zl[16];
        tmem_ld16(tmem + lo + COL_D + dblk + j0, x2);
        tmem_ld16(tmem + lo + COL_D2 + dblk + j0, zx);
        tmem_ld16(tmem + lo + COL_X + j0, xv);
        tmem_ld16(tmem + lo + COL_Z + j0, zv);
        if constexpr (X3) {
          tmem_ld16(tmem + lo + COL_XL + j0, xl);
          tmem_ld16(tmem + lo + COL_ZL + j0, zl);
        }
        tmem_ld_wait();
        float b[16], bl[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float x = __uint_as_float(xv[e]) + (X3 ? __uint_as_float(xl[e]) : 0.f);
          const float z = __uint_as_float(zv[e]) + (X3 ? __uint_as_float(zl[e]) : 0.f);
          const float zxe = __uint_as_float(zx[e]);
          b[e] = fmaf(7.f, x, -__uint_as_float(x2[e]));
          zv[e] = __float_as_uint(fmaf(13.f, z, -15.f * zxe));
          if constexpr (X3) {
            split_tf32(b[e], b[e], bl[e]);
            float h, l;
            split_tf32(zxe, h, l);
            zx[e] = __float_as_uint(h);
            xl[e] = __float_as_uint(l);
          }
        }
        store_col16(bbuf, NP, li, hs * MP + j0, b);
        if constexpr (X3) {
          store_col16(bbuf_lo, NP, li, hs * MP + j0, bl);
          tmem_st16(tmem + lo + COL_XL + j0, xl);
        }
        tmem_st16(tmem + lo + COL_X + j0, zx);
        tmem_st16(tmem + lo + COL_D + dblk + j0, zv);
      }
    }
    fence_async_smem();
    tmem_st_wait();
    tc_fence_before_sync();
    __syncthreads();
  };
  for (int it = 0; THREE && it < p.iters && !*abort_flag; ++it) {
    gemm(0, abuf);                          // X = A_S Z
    if (*abort_flag) break;
    store_bt(0.f, 1.f, 1.f, (int)COL_X);    // B <- X ; X -> TMEM
    gemm2();                                // X X, Z X
    if (*abort_flag) break;
    epi2();                                 // B <- 7X - X^2 ; Z X -> TMEM ; D <- 13Z - 15ZX
    gemm3();                                // D += Z X (7X - X^2)
    if (*abort_flag) break;
    store_bt(0.f, 1.f, 0.25f, (int)COL_Z);  // Z <- D / 4 ; B <- Z by columns
  }
  for (int it = 0; !THREE && it < p.iters && !*abort_flag; ++it) {
    gemm(0, abuf);                          // X = A_S Z
    if (*abort_flag) break;
    store_bt(7.f, -1.f, 1.f, (int)COL_X);   // B <- 7I - X ; X -> TMEM
    gemm(COL_X, nullptr);                   // Y = X (7I - X)
    if (*abort_flag) break;
    store_bt(15.f, -1.f, 1.f, -1);          // B <- 15I - Y
    gemm(COL_X, nullptr);                   // Y = X (15I - ...)
    if (*abort_flag) break;
    store_bt(13.f, -1.f, 1.f, -1);          // B <- 13I - Y
    gemm(COL_Z, nullptr);                   // Y = Z (13I - ...)
    if (*abort_flag) break;
    store_bt(0.f, 1.f, 0.25f, (int)COL_Z);  // Z <- Y / 4 ; B <- Z by columns
  }
  while (exp_row < hp * m) export_rows();  // what the products did not cover
  // ---- 5a) G = merge of the key-split partials (row li of head bh); G^T
  // into gbuf (B of W = Z G, head slot hs at rows hs d ..). One pass over
  // the splits, two at a time with all their loads in flight: a running
  // (max, denominator) rescales the accumulated rows as in an online
  // softmax; an empty partial (max = -inf, rows never written) contributes
  // nothing.
  if (!z_only) {
    float* grow_out = p.g + ((size_t)(live ? bh : 0) * m + (live ? li : 0)) * d;
    for (int c0 = half * 32; c0 < d; c0 += 64) {
      float acc[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) acc[e] = 0.f;
      if (live) {
        float gm = -INFINITY, den = 0.f;
        for (int sp = 0; sp < p.splits; sp += 2) {
          const bool two = sp + 1 < p.splits;
          const size_t pr0 = ((size_t)bh * p.splits + sp) * m + li;
          const size_t pr1 = two ? pr0 + (size_t)m : pr0;
          const float2 ml0 = __ldg(reinterpret_cast<const float2*>(p.gml) + pr0);
          const float2 ml1 = __ldg(reinterpret_cast<const float2*>(p.gml) + pr1);
          const float4* s0 = reinterpret_cast<const float4*>(p.gpart + pr0 * d + c0);
          const float4* s1 = reinterpret_cast<const float4*>(p.gpart + pr1 * d + c0);
          float4 v0[8], v1[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            v0[e] = __ldg(s0 + e);
            v1[e] = __ldg(s1 + e);
          }
          const bool ok0 = ml0.x != -INFINITY, ok1 = two && ml1.x != -INFINITY;
          const float cm = fmaxf(gm, fmaxf(ok0 ? ml0.x : -INFINITY, ok1 ? ml1.x : -INFINITY));
          if (cm == -INFINITY) continue;  // nothing yet
          const float r = gm == -INFINITY ? 0.f : expf(gm - cm);
          const float f0 = ok0 ? expf(ml0.x - cm) : 0.f;
          const float f1 = ok1 ? expf(ml1.x - cm) : 0.f;
          den = den * r + (ok0 ? ml0.y * f0 : 0.f) + (ok1 ? ml1.y * f1 : 0.f);
          gm = cm;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 a0 = ok0 ? v0[e] : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 a1 = ok1 ? v1[e] : make_float4(0.f, 0.f, 0.f, 0.f);
            acc[4 * e] = fmaf(acc[4 * e], r, fmaf(a0.x, f0, a1.x * f1));
            acc[4 * e + 1] = fmaf(acc[4 * e + 1], r, fmaf(a0.y, f0, a1.y * f1));
            acc[4 * e + 2] = fmaf(acc[4 * e + 2], r, fmaf(a0.z, f0, a1.z * f1));
            acc[4 * e + 3] = fmaf(acc[4 * e + 3], r, fmaf(a0.w, f0, a1.w * f1));
          }
        }
        const float inv = 1.f / den;
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] *= inv;
        float4* go = reinterpret_cast<float4*>(grow_out + c0);
#pragma unroll
        for (int e = 0; e < 8; ++e) go[e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
      }
      if (hs < hp) {
        if constexpr (X3) {
          float al[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) split_tf32(acc[e], acc[e], al[e]);
          store_col32(gbuf_lo, NW, li, hs * d + c0, al);
        }
        store_col32(gbuf, NW, li, hs * d + c0, acc);
      }
    }
  }

  fence_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  // ---- 5) Z (TMEM columns COL_Z.., this thread's row) out
  if (p.z && !*abort_flag && head_ok) {  // warp-uniform: the TMEM loads are collective
    float* zrow = p.z + ((size_t)bh * m + (live ? li : 0)) * m;
    for (int c0 = half * 32; c0 < m; c0 += 64) {
      uint32_t r[32];
      tmem_ld32(tmem + lo + COL_Z + c0, r);
      if constexpr (X3) {
        uint32_t rl[32];
        tmem_ld32(tmem + lo + COL_ZL + c0, rl);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(rl[e]));
      }
      tmem_ld_wait();
      if (!live) continue;
      if (c0 + 32 <= m && (m & 3) == 0) {
        float4* zo = reinterpret_cast<float4*>(zrow + c0);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          zo[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                              __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (c0 + e < m) zrow[c0 + e] = __uint_as_float(r[e]);
      }
    }
  }
  // ---- 5) W = Z G (head slot hs in columns hs d ..)
  if (!z_only && !*abort_flag) {
    if (tid == 0) {
      tc_fence_after_sync();
      issue(COL_D, COL_Z, COL_ZL, nullptr, nullptr, gbuf, gbuf_lo, NW, MP);
      mma_commit(&bar_mma);
    }
    wait_mma();
    if (!*abort_flag && head_ok) {
      float* wrow = p.w + ((size_t)bh * m + (live ? li : 0)) * d;
      __nv_bfloat16* wt = p.wt + (size_t)bh * p.dpad * p.m64;
      for (int c0 = half * 32; c0 < d; c0 += 64) {
        uint32_t r[32];
        tmem_ld32(tmem + lo + COL_D + hs * d + c0, r);
        tmem_ld_wait();
        if (live) {
          float4* wo = reinterpret_cast<float4*>(wrow + c0);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            wo[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
        }
        // W^T (bf16, zero padded to m64 columns): column li, and li + MP
        // where MP < m64 (the bf16 token kernels' operand; fp32: none)
        for (int lj = li; p.wt && lj < p.m64; lj += MP) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            wt[(size_t)(c0 + e) * p.m64 + lj] =
                __float2bfloat16_rn(lj == li && live ? __uint_as_float(r[e]) : 0.f);
        }
      }
      if (half == 0 && p.wt)
        for (int lj = li; lj < p.m64; lj += MP)
          for (int c = d; c < p.dpad; ++c) wt[(size_t)c * p.m64 + lj] = __float2bfloat16_rn(0.f);
    }
  }
  // no product of this CTA may still be in flight when its TMEM is freed
  // (after a timeout the last products were not waited for)
  if (tid == 0) {
    mma_commit(&bar_fin);
    mbar_wait(&bar_fin, 0, nullptr, kWaitNs);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, p.tmem_cols);
}

// W = Z G for the plan that computes Z beside the landmark-row pass (Z
// needs only the landmarks; G is merged from the key-split partials by a
// CUDA-core kernel after that pass). CTA (cb, head) forms the NC columns
// [NC cb, NC cb + NC) of W: Z -> shared memory (A operand, K-major, zero
// padded to 128 x MP), those columns of G written transposed (B operand,
// K-major, N = NC), one tf32 product M = 128, N = NC, K = MP into TMEM; then
// W (fp32 stage export) and W^T as bf16 [dpad][m64] with zero padding (CTA 0
// also writes the zero columns d .. dpad - 1). Global loads are
// row-contiguous across a warp's lanes.
struct WParams {
  const float* z;      // [B*H][m][m]
  const float* g;      // [B*H][m][d]  G (merged)
  float* w;            // [B*H][m][d]  stage export
  __nv_bfloat16* wt;   // [B*H][dpad][m64]
  int* status;
  int m, d, dpad, m64;
};

// NC: columns of W per CTA (16, 32 or 64)
template <int MP, int NC>
__global__ void __launch_bounds__(kThreads, 3) w_tc(const __grid_constant__ WParams p) {
  constexpr int NQ = NC / 4;                          // float4s of a G row block
  constexpr uint32_t kCols = NC < 32 ? 32u : (uint32_t)NC;  // TMEM columns
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* abuf = sm;                  // Z:   [128 rows x MP]
  uint8_t* gbuf = sm + 128 * MP * 4;   // G^T: [NC rows x MP]
  __shared__ uint64_t bar_mma;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m = p.m, d = p.d, c0 = (int)blockIdx.x * NC;
  const long long bh = blockIdx.y;
  if (tid == 0) {
    mbar_init(&bar_mma, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base_sh, kCols);

  // Z: float4 (r, q) = Z[r][4q .. 4q + 3], q fastest; zeros outside m x m
  {
    constexpr int Q = MP / 4, NV = 128 * Q / kThreads;
    const float* zh = p.z + bh * m * m;
    float4 v[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      const int e = tid + u * kThreads, r = e / Q, c = (e % Q) * 4;
      if ((m & 3) == 0)
        v[u] = r < m && c < m ? __ldg(reinterpret_cast<const float4*>(zh + (size_t)r * m + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
      else {
        const float* zr = zh + (size_t)(r < m ? r : 0) * m;
        v[u] = make_float4(r < m && c < m ? __ldg(zr + c) : 0.f, r < m && c + 1 < m ? __ldg(zr + c + 1) : 0.f,
                           r < m && c + 2 < m ? __ldg(zr + c + 2) : 0.f, r < m && c + 3 < m ? __ldg(zr + c + 3) : 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      const int e = tid + u * kThreads;
      store_row4(abuf, 128, e / Q, (e % Q) * 4, v[u]);
    }
  }

  // G columns c0 .. c0 + NC - 1: element (i, q) = columns c0 + 4q .. + 3 of
  // row i, q fastest, all loads of a thread in flight; element (i, c0 + j)
  // goes to gbuf storage row j, column i (rows i >= m: zeros)
  {
    constexpr int NE = (MP * NQ + kThreads - 1) / kThreads;
    float4 gv[NE];
#pragma unroll
    for (int u = 0; u < NE; ++u) {
      const int e = tid + u * kThreads, i = e / NQ, q = e % NQ;
      gv[u] = e < MP * NQ && i < m ? __ldg(reinterpret_cast<const float4*>(p.g + (bh * m + i) * d + c0) + q)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < NE; ++u) {
      const int e = tid + u * kThreads, i = e / NQ, q = e % NQ;
      if (e >= MP * NQ) break;
      *reinterpret_cast<float*>(gbuf + kmaj_off(4 * q, i, NC)) = gv[u].x;
      *reinterpret_cast<float*>(gbuf + kmaj_off(4 * q + 1, i, NC)) = gv[u].y;
      *reinterpret_cast<float*>(gbuf + kmaj_off(4 * q + 2, i, NC)) = gv[u].z;
      *reinterpret_cast<float*>(gbuf + kmaj_off(4 * q + 3, i, NC)) = gv[u].w;
    }
  }
  fence_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  const uint32_t tmem = tmem_base_sh;
  if (tid == 0) {
    tc_fence_after_sync();
    const uint64_t a0 = smem_desc(smem_u32(abuf), 16, 1024, SW_128B);
    const uint64_t b0 = smem_desc(smem_u32(gbuf), 16, 1024, SW_128B);
    const uint32_t id = idesc_tf32(128, NC);
    constexpr uint32_t bchunk = NC * 8u;  // (NC rows * 128 B) >> 4
#pragma unroll
    for (int kk = 0; kk < MP / 8; ++kk) {
      const uint32_t step = (uint32_t)(kk & 3) * 2u;
      mma_tf32(tmem, a0 + (uint64_t)((uint32_t)(kk >> 2) * 1024u + step),
               b0 + (uint64_t)((uint32_t)(kk >> 2) * bchunk + step), id, kk > 0 ? 1u : 0u);
    }
    mma_commit(&bar_mma);
  }
  const bool ok = mbar_wait(&bar_mma, 0, &abort_sh, kWaitNs);
  if (!ok) {
    abort_sh = 1;
    atomicExch(p.status, (int)NYS_ERR_TIMEOUT);
  }
  tc_fence_after_sync();
  // warps 0-3: W row `row` = TMEM lane row, the block's NC columns
  if (warp < 4 && __all_sync(0xffffffffu, ok)) {
    const int row = warp * 32 + lane;
    __nv_bfloat16* wt = p.wt + bh * p.dpad * p.m64 + row;
#pragma unroll
    for (int j0 = 0; j0 < NC; j0 += 16) {
      uint32_t r[16];
      tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + j0, r);
      tmem_ld_wait();
      if (row < m) {
        float4* wo = reinterpret_cast<float4*>(p.w + (bh * m + row) * d + c0 + j0);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          wo[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                              __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
      }
      if (row < p.m64) {
#pragma unroll
        for (int e = 0; e < 16; ++e)
          wt[(size_t)(c0 + j0 + e) * p.m64] = __float2bfloat16_rn(row < m ? __uint_as_float(r[e]) : 0.f);
      }
    }
    if (blockIdx.x == 0 && row < p.m64)
      for (int c = d; c < p.dpad; ++c) wt[(size_t)c * p.m64] = __float2bfloat16_rn(0.f);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kCols);
}

// m rounded up to 32, 64 or 128
int mpad_of(int m) { return m <= 32 ? 32 : (m <= 64 ? 64 : 128); }

}  // namespace

bool pinv_tc_supported(const Shape& s) {
  if (s.dtype == NYS_FP32)  // three tf32 products per product
    return s.m <= 64 && s.d % 32 == 0 && s.d <= 64 && s.iters <= kX3MaxIters;
  return s.dtype == NYS_BF16 && s.m <= 128 && s.iters <= kTf32MaxIters;
}

// heads stacked per CTA: as many as the 128 TMEM lanes and a 256-column W
// product take, no more than there are
int heads_per_cta(const Shape& s) {
  return (int)std::min<long long>(std::min(128 / mpad_of(s.m), 256 / s.d), s.bh());
}

int pinv_tc_ctas(const Shape& s) {
  const int hp = heads_per_cta(s);
  return (int)((s.bh() + hp - 1) / hp);
}

int launch_pinv_tc(const Shape& s, const float* qt, const float* kt, const float* gpart,
                   const float* gml, float* g, float* a_s, float* z, float* w, void* wt_bf16,
                   int splits, int* status, cudaStream_t stream) {
  if (!pinv_tc_supported(s)) return NYS_ERR_UNSUPPORTED;
  PinvParams p{};
  p.z = z;
  p.z_only = gpart == nullptr ? 1 : 0;
  p.stall_ns = debug_stall_ns();
  p.qt = qt;
  p.kt = kt;
  p.gpart = gpart;
  p.gml = gml;
  p.g = g;
  p.a_s = a_s;
  p.w = w;
  p.wt = static_cast<__nv_bfloat16*>(wt_bf16);
  p.status = status;
  p.BH = (int)s.bh();
  p.m = s.m;
  p.d = s.d;
  p.dpad = s.dpad();
  p.m64 = s.m64();
  p.splits = splits;
  p.iters = s.iters;
  p.scale = 1.0f / sqrtf((float)s.d);
  p.c = p.scale * 1.4426950408889634f;
  const int MP = mpad_of(s.m);
  const bool x3 = s.dtype == NYS_FP32;
  p.hp = heads_per_cta(s);
  const int NP = p.hp * MP, NW = p.hp * s.d;
  // three levels per update where the CTAs run one per SM anyway (the
  // second accumulator takes TMEM that two CTAs per SM would share)
  const int grid_ctas = (p.BH + p.hp - 1) / p.hp;
  const uint32_t base_cols = (x3 ? 4 : 2) * MP + std::max(NP, NW);
  const bool three = (x3 || grid_ctas <= plan_sms()) && base_cols + NP <= 512;
  const uint32_t need = std::max<uint32_t>(2 * s.d + NP, base_cols + (three ? NP : 0));
  uint32_t cols = 32;
  while (cols < need) cols <<= 1;
  p.tmem_cols = cols;
  const size_t gbytes = (size_t)NW * MP * 4;
  const size_t abytes = (size_t)128 * MP * 4;
  const size_t bbytes = (size_t)NP * MP * 4;
  const size_t kbytes = (size_t)NP * s.d * 4;  // K~ hi / lo (score step only)
  p.abuf_off = (uint32_t)gbytes;
  p.bbuf_off = (uint32_t)(gbytes + abytes);
  p.klo_off = (uint32_t)(gbytes + kbytes);
  const size_t base = gbytes + std::max(abytes + bbytes, 2 * kbytes);
  p.abuf_lo_off = (uint32_t)base;
  p.bbuf_lo_off = (uint32_t)(base + abytes);
  p.gbuf_lo_off = (uint32_t)(base + abytes + bbytes);
  const size_t smem = (x3 ? base + abytes + bbytes + gbytes : base) + 1024;
  auto kern = x3 ? (MP == 32 ? pinv_tc<32, true, true> : pinv_tc<64, true, true>)
           : three ? (MP == 32 ? pinv_tc<32, false, true> : (MP == 64 ? pinv_tc<64, false, true> : pinv_tc<128, false, true>))
                   : (MP == 32 ? pinv_tc<32, false, false> : (MP == 64 ? pinv_tc<64, false, false> : pinv_tc<128, false, false>));
  // (two CTAs per SM for MP <= 64: the largest shared-memory carveout)
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return set_cuda_error(cudaGetLastError());
  const unsigned grid = (unsigned)((p.BH + p.hp - 1) / p.hp);
  KernelScope scope("pinv_tc", stream);
  kern<<<grid, kThreads, smem, stream>>>(p);
  return launch_status();
}

int launch_w_tc(const Shape& s, const float* z, const float* g, float* w, void* wt_bf16,
                int* status, cudaStream_t stream) {
  if (s.dtype != NYS_BF16 || !pinv_tc_supported(s) || s.d % 16 != 0) return NYS_ERR_UNSUPPORTED;
  WParams p{};
  p.z = z;
  p.g = g;
  p.w = w;
  p.wt = static_cast<__nv_bfloat16*>(wt_bf16);
  p.status = status;
  p.m = s.m;
  p.d = s.d;
  p.dpad = s.dpad();
  p.m64 = s.m64();
  const int MP = mpad_of(s.m);
  // whole heads per CTA (d <= 64) when the heads alone fill the GPU, else
  // 16-column blocks for more CTAs in flight
  const int NC = (s.bh() >= plan_sms() && s.d <= 64) ? s.d : 16;
  const size_t smem = (size_t)(128 + NC) * MP * 4 + 1024;
  void (*kern)(WParams) = nullptr;
  if (NC == 16) kern = MP == 32 ? w_tc<32, 16> : (MP == 64 ? w_tc<64, 16> : w_tc<128, 16>);
  else if (NC == 32) kern = MP == 32 ? w_tc<32, 32> : (MP == 64 ? w_tc<64, 32> : w_tc<128, 32>);
  else kern = MP == 32 ? w_tc<32, 64> : (MP == 64 ? w_tc<64, 64> : w_tc<128, 64>);
  // three CTAs per SM: the largest shared-memory carveout
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return set_cuda_error(cudaGetLastError());
  KernelScope scope("w_tc", stream);
  kern<<<dim3((unsigned)(s.d / NC), (unsigned)s.bh()), kThreads, smem, stream>>>(p);
  return launch_status();
}

}  // namespace nys
