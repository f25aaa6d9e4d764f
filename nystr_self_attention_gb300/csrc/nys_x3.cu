// fp32 inputs on the tensor cores: the landmark-row and token-row products
// ("Nyströmformer" review page, Proposed method, bullets 3 and 6)
//   landmark rows: for a range of 128-key tiles of one head, the partial
//                  (O, max, sum) of softmax(Q~ K^T s) V
//   token rows:    softmax(Q K~^T s) W for one tile of 128 tokens (the
//                  attention term; the convolution is added after it)
// Both are one operation: a block of up to 128 query rows attends to tiles
// of up to 128 keys with an online softmax. The products run in tcgen05
// kind::tf32 as three products of the operands' hi/lo split (hi = x with
// the low 13 significand bits cleared, exact in tf32; lo = x - hi, exact in
// fp32): A B ~ A_hi B_hi + A_lo B_hi + A_hi B_lo (the error-corrected tf32
// product of Ootomo and Yokota, 2022), which keeps fp32 accuracy.
//
// One CTA of 256 threads per work item. Shared memory holds the hi and lo
// halves of the query block (A of S = Q K^T), of the key tile (B of S) and
// of the value tile transposed (B of O += P V), each K-major SWIZZLE_128B.
// TMEM: S (128 columns, then P hi in place), P lo (128), O (d columns).
// Thread (warp w, lane l) owns query row 32 (w % 4) + l and half w / 4 of
// the row's key and value columns. The next tile's loads are in flight
// while P V runs. Every wait is bounded; a wait that runs out sets the
// status word and the CTA winds down without further products.
#include <cuda_runtime.h>

#include <algorithm>

#include "nys_internal.h"
#include "nys_sm100.h"

namespace nys {
namespace {

using namespace sm100;

struct X3Params {
  const float* q;       // landmark rows: Q~ [BH][m][d]; token rows: Q [BH][n][d]
  const float* k;       // landmark rows: K [BH][n][d];  token rows: K~ [BH][m][d]
  const float* v;       // landmark rows: V [BH][n][d];  token rows: W [BH][m][d]
  float* o;             // landmark rows: partial O [BH][splits][m][d]; token rows: out [BH][n][d]
  float* ml;            // landmark rows: [BH][splits][m][2] (max of the scaled scores, sum)
  const int* lengths;   // landmark rows: keys at or past lengths[b] take no part (null: none)
  const float* vseq;    // token rows with the conv: V [BH][n][d]
  const float* conv_w;  // token rows with the conv: [H][ks] taps (null: no conv)
  int* status;
  int H, n, d, m;
  int splits, tiles_per_split;  // landmark rows
  int tiles_per_head;           // token rows
  int ks;                       // token rows: conv taps (0: the attention term alone)
  float c;                      // scale * log2(e)
  float scale;                  // 1 / sqrt(d)
};

constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kConvRun = 16;  // conv outputs per item: consecutive rows of one column
constexpr uint32_t COL_S = 0, COL_PL = 128, COL_O = 256, kTmemCols = 512;

__device__ __forceinline__ float tf32_hi(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// byte offset of element (row, col) of a K-major SWIZZLE_128B fp32 operand
// with `rows` rows: 32-column chunks of [rows x 128 B]
__device__ __forceinline__ uint32_t kmaj(int row, int col, int rows) {
  return (uint32_t)(col >> 5) * (uint32_t)(rows * 128) + sw128_offset(row, (col & 31) * 4);
}

// A block of 128 rows x DP columns, row-major in global memory (row pitch
// d), into the hi / lo K-major operands (128 rows). Rows >= nrows and
// columns >= d are zero. Thread task e = tid + 256 i: row e / (DP/4), four
// columns (e % (DP/4)) * 4: coalesced 16-byte loads, conflict-free 16-byte
// stores.
template <int DP>
struct RowRegs {
  static constexpr int kPer = 128 * (DP / 4) / kThreads;
  float4 x[kPer];
};

template <int DP>
__device__ __forceinline__ void load_rows(const float* src, int nrows, int d, RowRegs<DP>& r) {
  constexpr int C4 = DP / 4;
#pragma unroll
  for (int i = 0; i < RowRegs<DP>::kPer; ++i) {
    const int e = (int)threadIdx.x + kThreads * i, row = e / C4, c = (e % C4) * 4;
    r.x[i] = (row < nrows && c < d) ? __ldg(reinterpret_cast<const float4*>(src + (size_t)row * d + c))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <int DP>
__device__ __forceinline__ void store_rows(const RowRegs<DP>& r, uint8_t* hi, uint8_t* lo) {
  constexpr int C4 = DP / 4;
#pragma unroll
  for (int i = 0; i < RowRegs<DP>::kPer; ++i) {
    const int e = (int)threadIdx.x + kThreads * i, row = e / C4, c = (e % C4) * 4;
    const float4 x = r.x[i];
    const float4 h = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
    const uint32_t off = kmaj(row, c, 128);
    *reinterpret_cast<float4*>(hi + off) = h;
    *reinterpret_cast<float4*>(lo + off) = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
  }
}

// A tile of 128 rows (keys) x DP columns, row-major in global memory, into
// the hi / lo K-major operands of its transpose (DP rows, K = the 128
// keys). Task e = tid + 256 i: key e % 128, eight columns 8 (e / 128); the
// 32 lanes of a warp take 32 consecutive keys and one column group, so each
// scalar store of the transpose hits 32 distinct banks.
template <int DP>
struct ColRegs {
  static constexpr int kPer = 128 * (DP / 8) / kThreads;
  float4 x[kPer][2];
};

template <int DP>
__device__ __forceinline__ void load_cols(const float* src, int nrows, int d, ColRegs<DP>& r) {
#pragma unroll
  for (int i = 0; i < ColRegs<DP>::kPer; ++i) {
    const int e = (int)threadIdx.x + kThreads * i, key = e & 127, c0 = (e >> 7) * 8;
    const float4* p = reinterpret_cast<const float4*>(src + (size_t)key * d + c0);
    const bool ok = key < nrows;
    r.x[i][0] = (ok && c0 < d) ? __ldg(p) : make_float4(0.f, 0.f, 0.f, 0.f);
    r.x[i][1] = (ok && c0 + 4 < d) ? __ldg(p + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <int DP>
__device__ __forceinline__ void store_cols(const ColRegs<DP>& r, uint8_t* hi, uint8_t* lo) {
#pragma unroll
  for (int i = 0; i < ColRegs<DP>::kPer; ++i) {
    const int e = (int)threadIdx.x + kThreads * i, key = e & 127, c0 = (e >> 7) * 8;
    const float x[8] = {r.x[i][0].x, r.x[i][0].y, r.x[i][0].z, r.x[i][0].w,
                        r.x[i][1].x, r.x[i][1].y, r.x[i][1].z, r.x[i][1].w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const float h = tf32_hi(x[t]);
      const uint32_t off = kmaj(c0 + t, key, DP);
      *reinterpret_cast<float*>(hi + off) = h;
      *reinterpret_cast<float*>(lo + off) = x[t] - h;
    }
  }
}

// D (+)= A B^T in three tf32 products, one thread. A: 128 rows x k_dim,
// K-major in shared memory (a_hi / a_lo) or, with a_hi == nullptr, in TMEM
// at addresses a_col_hi / a_col_lo (one tf32 per column); B: b_rows rows x k_dim,
// K-major in shared memory. `acc`: accumulate onto D (else D is overwritten).
__device__ __forceinline__ void issue_x3(uint32_t d_tmem, const uint8_t* a_hi, const uint8_t* a_lo,
                                         uint32_t a_col_hi, uint32_t a_col_lo, const uint8_t* b_hi,
                                         const uint8_t* b_lo, int b_rows, int k_dim, bool acc) {
  const uint32_t id = idesc_tf32(128, b_rows);
  const uint32_t bchunk = (uint32_t)b_rows * 8u;  // (b_rows x 128 B) >> 4
#pragma unroll
  for (int pass = 0; pass < 3; ++pass) {
    // (hi, hi), (lo, hi), (hi, lo)
    const uint8_t* b = pass == 2 ? b_lo : b_hi;
    const uint64_t b0 = smem_desc(smem_u32(b), 16, 1024, SW_128B);
    if (a_hi) {
      const uint64_t a0 = smem_desc(smem_u32(pass == 1 ? a_lo : a_hi), 16, 1024, SW_128B);
      for (int kk = 0; kk < k_dim / 8; ++kk) {
        const uint32_t step = (uint32_t)(kk & 3) * 2u;  // 8 tf32 = 32 B
        mma_tf32(d_tmem, a0 + (uint64_t)((uint32_t)(kk >> 2) * 1024u + step),
                 b0 + (uint64_t)((uint32_t)(kk >> 2) * bchunk + step), id,
                 (acc || pass > 0 || kk > 0) ? 1u : 0u);
      }
    } else {
      const uint32_t a_col = pass == 1 ? a_col_lo : a_col_hi;
      for (int kk = 0; kk < k_dim / 8; ++kk)
        mma_tf32_tA(d_tmem, a_col + (uint32_t)kk * 8u,
                    b0 + (uint64_t)((uint32_t)(kk >> 2) * bchunk + (uint32_t)(kk & 3) * 2u), id,
                    (acc || pass > 0 || kk > 0) ? 1u : 0u);
    }
  }
}

template <int DP, bool ROWS>
__global__ void __launch_bounds__(kThreads, 1) attn_x3(const X3Params p) {
  constexpr uint32_t kBlk = 128u * DP * 4u;  // one 128 x DP (or DP x 128) fp32 operand
  constexpr int HC = DP / 2;                 // O columns per half row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* q_hi = sm;
  uint8_t* q_lo = sm + kBlk;
  uint8_t* k_hi = sm + 2 * kBlk;
  uint8_t* k_lo = sm + 3 * kBlk;
  uint8_t* v_hi = sm + 4 * kBlk;  // V^T: DP rows, K = the tile's keys
  uint8_t* v_lo = sm + 5 * kBlk;
  __shared__ uint64_t bar, bar_fin;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float red[2][2][128];  // [max, sum][half][row]
  volatile int* abort_flag = &abort_sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;

  // ---- the work item
  const int d = p.d, m = p.m;
  long long bh;
  int split = 0, tile0, ntiles, q_rows, klen;
  const float *qsrc, *ksrc, *vsrc;
  if constexpr (ROWS) {
    bh = blockIdx.x / p.splits;
    split = (int)(blockIdx.x - bh * p.splits);
    klen = p.lengths ? min(p.n, max(0, p.lengths[bh / p.H])) : p.n;
    const int tiles = (klen + 127) / 128;
    tile0 = split * p.tiles_per_split;
    ntiles = max(0, min(tiles, tile0 + p.tiles_per_split) - tile0);
    q_rows = m;
    qsrc = p.q + (size_t)bh * m * d;
    ksrc = p.k + (size_t)bh * p.n * d;
    vsrc = p.v + (size_t)bh * p.n * d;
  } else {
    bh = blockIdx.x / p.tiles_per_head;
    const int t = (int)(blockIdx.x - bh * p.tiles_per_head);
    tile0 = 0;
    ntiles = 1;
    klen = m;
    q_rows = min(128, p.n - t * 128);
    qsrc = p.q + ((size_t)bh * p.n + (size_t)t * 128) * d;
    ksrc = p.k + (size_t)bh * m * d;
    vsrc = p.v + (size_t)bh * m * d;
  }

  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&bar_fin, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base_sh, kTmemCols);
  // the query block and the first tile
  {
    RowRegs<DP> qr, kr;
    ColRegs<DP> vr;
    load_rows<DP>(qsrc, q_rows, d, qr);
    if (ntiles > 0) {
      const size_t k0 = (size_t)tile0 * 128;
      load_rows<DP>(ksrc + k0 * d, klen - (int)k0, d, kr);
      load_cols<DP>(vsrc + k0 * d, klen - (int)k0, d, vr);
    }
    store_rows<DP>(qr, q_hi, q_lo);
    if (ntiles > 0) {
      store_rows<DP>(kr, k_hi, k_lo);
      store_cols<DP>(vr, v_hi, v_lo);
    }
  }
  fence_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t trow = tmem + lane_base;

  uint32_t phase = 0;
  auto wait_bar = [&]() {
    if (!mbar_wait(&bar, phase, abort_flag, kWaitNs) && !*abort_flag) {
      *abort_flag = 1;
      atomicExch(p.status, (int)NYS_ERR_TIMEOUT);
    }
    phase ^= 1;
    tc_fence_after_sync();
  };

  float mrun = -INFINITY, lrun = 0.f;  // this row's running max (raw score) and sum
  for (int j = 0; j < ntiles; ++j) {
    const int nk = min(128, klen - (tile0 + j) * 128);  // keys of this tile
    // S = Q K^T (and, by the commit's ordering, P V of tile j-1 done)
    if (tid == 0 && !*abort_flag) {
      issue_x3(tmem + COL_S, q_hi, q_lo, 0, 0, k_hi, k_lo, 128, DP, false);
      mma_commit(&bar);
    }
    wait_bar();
    __syncthreads();
    const bool alive = !*abort_flag;  // uniform: read after the barrier
    // ---- online softmax of this row over the tile's keys
    const int cb = 64 * half;
    uint32_t r0[32], r1[32];
    if (alive) {
      tmem_ld32(trow + COL_S + cb, r0);
      tmem_ld32(trow + COL_S + cb + 32, r1);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) r0[e] = r1[e] = 0u;
    }
    float pm = -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      if (cb + e < nk) pm = fmaxf(pm, __uint_as_float(r0[e]));
      if (cb + 32 + e < nk) pm = fmaxf(pm, __uint_as_float(r1[e]));
    }
    red[0][half][row] = pm;
    __syncthreads();
    const float mnew = fmaxf(mrun, fmaxf(red[0][0][row], red[0][1][row]));  // finite: nk >= 1
    const float alpha = mrun == -INFINITY ? 0.f : fast_exp2((mrun - mnew) * p.c);
    float ps = 0.f;
    {
      uint32_t lo_[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x = cb + e < nk ? fast_exp2((__uint_as_float(r0[e]) - mnew) * p.c) : 0.f;
        const float h = tf32_hi(x);
        ps += x;
        r0[e] = __float_as_uint(h);
        lo_[e] = __float_as_uint(x - h);
      }
      if (alive) {
        tmem_st32(trow + COL_S + cb, r0);
        tmem_st32(trow + COL_PL + cb, lo_);
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x = cb + 32 + e < nk ? fast_exp2((__uint_as_float(r1[e]) - mnew) * p.c) : 0.f;
        const float h = tf32_hi(x);
        ps += x;
        r1[e] = __float_as_uint(h);
        lo_[e] = __float_as_uint(x - h);
      }
      if (alive) {
        tmem_st32(trow + COL_S + cb + 32, r1);
        tmem_st32(trow + COL_PL + cb + 32, lo_);
      }
    }
    // O of the earlier tiles rescaled to the new max (P V of tile j-1 is done)
    if (alive && j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
      if constexpr (HC == 32) {
        uint32_t o[32];
        tmem_ld32(trow + COL_O + half * HC, o);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st32(trow + COL_O + half * HC, o);
      } else {
        uint32_t o[16];
        tmem_ld16(trow + COL_O + half * HC, o);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st16(trow + COL_O + half * HC, o);
      }
    }
    red[1][half][row] = ps;
    tmem_st_wait();
    tc_fence_before_sync();
    __syncthreads();
    lrun = lrun * alpha + (red[1][0][row] + red[1][1][row]);
    mrun = mnew;
    // O += P V
    if (tid == 0 && !*abort_flag) {
      tc_fence_after_sync();
      issue_x3(tmem + COL_O, nullptr, nullptr, tmem + COL_S, tmem + COL_PL, v_hi, v_lo, DP, 128, j > 0);
      mma_commit(&bar);
    }
    if (j + 1 < ntiles) {
      // the next tile's loads in flight while P V runs; K is free (S of
      // this tile is done), V once P V is
      const size_t k0 = (size_t)(tile0 + j + 1) * 128;
      RowRegs<DP> kr;
      ColRegs<DP> vr;
      load_rows<DP>(ksrc + k0 * d, klen - (int)k0, d, kr);
      load_cols<DP>(vsrc + k0 * d, klen - (int)k0, d, vr);
      store_rows<DP>(kr, k_hi, k_lo);
      wait_bar();
      store_cols<DP>(vr, v_hi, v_lo);
      fence_async_smem();
      tc_fence_before_sync();
      __syncthreads();
    }
  }
  if (ntiles > 0) wait_bar();  // the last P V
  __syncthreads();
  const bool alive = !*abort_flag;

  // ---- results: this row's half of O
  float o[HC];
  if (alive && ntiles > 0) {
    if constexpr (HC == 32) {
      uint32_t r[32];
      tmem_ld32(trow + COL_O + half * HC, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(r[e]);
    } else {
      uint32_t r[16];
      tmem_ld16(trow + COL_O + half * HC, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) o[e] = __uint_as_float(r[e]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < HC; ++e) o[e] = 0.f;
  }
  const int c0 = half * HC;
  const bool fuse_conv = !ROWS && p.ks > 0;  // uniform
  float* att_s = reinterpret_cast<float*>(sm);  // with the conv: the tile's attention term [128][DP]
  if (alive && row < q_rows) {
    float* dst;
    if constexpr (ROWS) {
      const size_t prow = ((size_t)bh * p.splits + split) * m + row;
      dst = p.o + prow * d;
      if (half == 0) {
        // an empty range (all its keys are padding) leaves max = -inf
        p.ml[prow * 2 + 0] = ntiles > 0 ? mrun * p.scale : -INFINITY;
        p.ml[prow * 2 + 1] = lrun;
      }
    } else {
      const int t = (int)(blockIdx.x - bh * p.tiles_per_head);
      // the operand buffers are free (the last P V is done): with the conv,
      // the attention term waits there for it
      dst = fuse_conv ? att_s + (size_t)row * DP : p.o + ((size_t)bh * p.n + (size_t)t * 128 + row) * d;
      const float inv = 1.f / lrun;
#pragma unroll
      for (int e = 0; e < HC; ++e) o[e] *= inv;
    }
#pragma unroll
    for (int e = 0; e < HC; e += 4)
      if (c0 + e < d) *reinterpret_cast<float4*>(dst + c0 + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
  }
  if constexpr (!ROWS) {
    if (fuse_conv && alive) {  // uniform
      // out[t][c] = att[t][c] + sum_j w[h][j] V[t + j - (ks - 1)/2][c], V
      // rows outside [0, n) zero, in fp32 FMAs: the tile's V rows with the
      // halo and the head's taps staged in the free operand buffers; an
      // item is kConvRun consecutive rows of one column, the V window in a
      // ring of registers whose indices the tap loop (unrolled in blocks of
      // kConvRun) keeps static: a tap costs one weight, one new V value and
      // kConvRun FMAs
      const int rad = (p.ks - 1) / 2, vrows = 128 + 2 * rad;
      float* v_s = att_s + 128 * DP;            // [vrows][DP]: V rows tok0 - rad ..
      float* w_s = v_s + (size_t)vrows * DP;    // [ks]
      const int tok0 = (int)(blockIdx.x - bh * p.tiles_per_head) * 128;
      const float* vb = p.vseq + (size_t)bh * p.n * d;
      const int d4 = d >> 2;
      for (int e = tid; e < vrows * d4; e += kThreads) {
        const int r = e / d4, c4 = (e - r * d4) * 4, u = tok0 - rad + r;
        const float4 x = (u >= 0 && u < p.n) ? __ldg(reinterpret_cast<const float4*>(vb + (size_t)u * d + c4))
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(v_s + (size_t)r * DP + c4) = x;
      }
      const float* wh = p.conv_w + (size_t)(bh % p.H) * p.ks;
      for (int j = tid; j < p.ks; j += kThreads) w_s[j] = wh[j];
      __syncthreads();
      const int ks_full = p.ks - p.ks % kConvRun;  // taps in whole blocks
      for (int item = tid; item < (128 / kConvRun) * d; item += kThreads) {
        const int c = item % d, r0 = (item / d) * kConvRun;
        if (tok0 + r0 >= p.n) continue;
        float acc[kConvRun], xw[kConvRun];
        const float* x = v_s + (size_t)r0 * DP + c;
#pragma unroll
        for (int r = 0; r < kConvRun; ++r) {
          acc[r] = 0.f;
          xw[r] = x[r * DP];  // before tap j, row r0 + j + r sits in xw[(j + r) % kConvRun]
        }
        const float* xp = x + kConvRun * DP;  // row r0 + j + kConvRun: xp[j * DP]
        const float* wp = w_s;
        // whole blocks: ks is odd, so a block never holds the last tap and
        // every next row lies inside the staged rows
        for (int jb = 0; jb < ks_full; jb += kConvRun) {
#pragma unroll
          for (int jj = 0; jj < kConvRun; ++jj) {
            const float wj = wp[jj];
#pragma unroll
            for (int r = 0; r < kConvRun; ++r) acc[r] = fmaf(wj, xw[(jj + r) % kConvRun], acc[r]);
            xw[jj] = xp[jj * DP];
          }
          wp += kConvRun;
          xp += kConvRun * DP;
        }
#pragma unroll
        for (int jj = 0; jj < kConvRun; ++jj) {
          const int j = ks_full + jj;
          if (j >= p.ks) break;
          const float wj = wp[jj];
#pragma unroll
          for (int r = 0; r < kConvRun; ++r) acc[r] = fmaf(wj, xw[(jj + r) % kConvRun], acc[r]);
          if (j + 1 < p.ks) xw[jj] = xp[jj * DP];
        }
        float* dst = p.o + ((size_t)bh * p.n + tok0 + r0) * d + c;
#pragma unroll
        for (int r = 0; r < kConvRun; ++r)
          if (tok0 + r0 + r < p.n) dst[(size_t)r * d] = att_s[(size_t)(r0 + r) * DP + c] + acc[r];
      }
    }
  }

  // wind-down: no product of this CTA may still be in flight
  if (tid == 0) {
    mma_commit(&bar_fin);
    mbar_wait(&bar_fin, 0, nullptr, kWaitNs);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int DP>
size_t x3_smem() {
  return std::max<size_t>(6u * 128u * DP * 4u + 1024u, 120u * 1024u);  // one CTA per SM
}

template <int DP, bool ROWS>
int launch_x3(const X3Params& p, long long items, const char* name, cudaStream_t stream) {
  if (items <= 0) return NYS_OK;
  if (items > 0x7FFFFFFFll) return NYS_ERR_UNSUPPORTED;
  const size_t smem = x3_smem<DP>();
  if (cudaFuncSetAttribute(attn_x3<DP, ROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return set_cuda_error(cudaGetLastError());
  KernelScope ks_(name, stream);
  attn_x3<DP, ROWS><<<(unsigned)items, kThreads, smem, stream>>>(p);
  return launch_status();
}

X3Params base_params(const Shape& s, int* status) {
  X3Params p{};
  p.status = status;
  p.H = s.H;
  p.n = s.n;
  p.d = s.d;
  p.m = s.m;
  p.scale = 1.0f / sqrtf((float)s.d);
  p.c = p.scale * 1.4426950408889634f;
  return p;
}

}  // namespace

bool x3_supported(const Shape& s) {
  return s.dtype == NYS_FP32 && s.d <= 64 && s.d % 4 == 0 && s.m <= 128;
}

void x3_rows_split(const Shape& s, int* splits, int* tiles_per_split) {
  const int tiles = (s.n + 127) / 128;
  const long long want = std::max(1ll, (long long)plan_sms() / std::max(1ll, s.bh()));
  const int sp = (int)std::min<long long>(tiles, want);
  *tiles_per_split = (tiles + sp - 1) / sp;
  *splits = (tiles + *tiles_per_split - 1) / *tiles_per_split;
}

int launch_rows_x3(const Shape& s, const float* qt, const void* k, const void* v, float* gpart,
                   float* gml, int splits, int tiles_per_split, int* status, cudaStream_t stream) {
  if (!x3_supported(s)) return NYS_ERR_UNSUPPORTED;
  if ((long long)splits * tiles_per_split < (s.n + 127) / 128) return NYS_ERR_ARG;
  X3Params p = base_params(s, status);
  p.q = qt;
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.o = gpart;
  p.ml = gml;
  p.lengths = s.lengths;
  p.splits = splits;
  p.tiles_per_split = tiles_per_split;
  const long long items = s.bh() * splits;
  return s.d <= 32 ? launch_x3<32, true>(p, items, "rows_x3", stream)
                   : launch_x3<64, true>(p, items, "rows_x3", stream);
}

int launch_tokens_x3(const Shape& s, const void* q, const void* v, const float* kt, const float* w,
                     const float* conv_w, void* out, int* status, cudaStream_t stream) {
  if (!x3_supported(s)) return NYS_ERR_UNSUPPORTED;
  if (s.ks > 0 && (!conv_w || s.ks % 2 == 0)) return NYS_ERR_ARG;
  X3Params p = base_params(s, status);
  p.q = static_cast<const float*>(q);
  p.k = kt;
  p.v = w;
  p.vseq = static_cast<const float*>(v);
  p.conv_w = s.ks > 0 ? conv_w : nullptr;
  p.ks = s.ks;
  p.o = static_cast<float*>(out);
  p.tiles_per_head = (s.n + 127) / 128;
  const long long items = s.bh() * p.tiles_per_head;
  return s.d <= 32 ? launch_x3<32, false>(p, items, "tokens_x3", stream)
                   : launch_x3<64, false>(p, items, "tokens_x3", stream);
}

}  // namespace nys
