// Landmark kernel, iterative pseudo-inverse and W = Z G on the tensor cores
// ("Nyströmformer" review page, Proposed method, bullets 2, 3 and 5), for
// m <= 128 landmarks, one CTA of 256 threads per head (row i of every
// m x m matrix in TMEM lane i):
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
// step), not a reformulation. A_S, Z and X stay in TMEM as A operands
// (row i in lane i); each product's B operand is written, transposed, into
// one shared-memory buffer by the epilogue of the product before it.
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
  float* w;            // [B*H][m][d]  stage export
  __nv_bfloat16* wt;   // [B*H][dpad][m64] zero padded
  int* status;
  int m, d, m_pad, dpad, m64, splits, iters;
  float scale;
  uint32_t tmem_cols;
  uint32_t gbuf_off;  // smem offset of the G^T buffer
  uint32_t klo_off;   // smem offset of the K~ lo split (prologue)
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

// four consecutive elements (row, c .. c+3), c % 4 == 0, as one 16-byte store
__device__ __forceinline__ void store_row4(uint8_t* buf, int rows, int row, int c, float4 v) {
  *reinterpret_cast<float4*>(buf + kmaj_off(row, c, rows)) = v;
}

__device__ __forceinline__ float tf32_hi(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// 256 threads: warp w works on TMEM lane quarter w % 4 (rows 32 (w % 4) ..
// + 31); the two warps of a quarter split each row's 32-column chunks
// (half h = w / 4 takes the chunks with index % 2 == h).
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads, 2) pinv_tc(const PinvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* bbuf = sm;               // B operand [MP rows x MP] fp32
  uint8_t* gbuf = sm + p.gbuf_off;  // G^T       [d rows x MP]  fp32
  uint8_t* khi = sm;                // K~ hi / lo [MP rows x d] (prologue only)
  uint8_t* klo = sm + p.klo_off;
  __shared__ uint64_t bar_mma;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float red_row[4], red_col[kThreads];
  volatile int* abort_flag = &abort_sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int row = quarter * 32 + lane;
  const int bh = blockIdx.x;
  const int m = p.m, d = p.d, MP = p.m_pad;
  const bool live = row < m;
  const bool in_mp = row < MP;
  const int nch = MP >> 5;  // 32-column chunks of an m x m matrix

  if (tid == 0) {
    mbar_init(&bar_mma, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base_sh, p.tmem_cols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t lo = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t COL_A = 0, COL_Z = MP, COL_X = 2 * MP, COL_Y = 3 * MP;
  const uint32_t COL_QH = 0, COL_QL = d, COL_S = 2 * d;  // prologue only

  uint32_t phase = 0;
  // tf32 product D = A (TMEM columns a_col..) x B (smem, b_rows rows = N),
  // K = k_dim. Descriptors: one base, then start-address increments.
  auto issue = [&](uint32_t d_col, uint32_t a_col, const uint8_t* b, int b_rows, int k_dim,
                   bool acc_first) {
    const uint64_t d0 = smem_desc(smem_u32(b), 16, 1024, SW_128B);
    const uint32_t id = idesc_tf32(128, b_rows);
    const uint32_t chunk16 = (uint32_t)b_rows * 8u;  // (b_rows * 128 B) >> 4
#pragma unroll 4
    for (int kk = 0; kk < k_dim / 8; ++kk) {
      const uint64_t bd = d0 + (uint64_t)((uint32_t)(kk >> 2) * chunk16 + (uint32_t)(kk & 3) * 2u);
      mma_tf32_tA(tmem + d_col, tmem + a_col + kk * 8, bd, id, (kk > 0 || acc_first) ? 1u : 0u);
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

  // ---- 1) A_S scores S = Q~ K~^T in 3xTF32 on the tensor cores
  {
    const float* krow = p.kt + ((size_t)bh * m + (live ? row : 0)) * d;
    const float* qrow = p.qt + ((size_t)bh * m + (live ? row : 0)) * d;
    for (int c0 = half * 32; c0 < d; c0 += 64) {
      uint32_t qh[32], ql[32];
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 kv = live ? *reinterpret_cast<const float4*>(krow + c0 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 qv = live ? *reinterpret_cast<const float4*>(qrow + c0 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 kh = make_float4(tf32_hi(kv.x), tf32_hi(kv.y), tf32_hi(kv.z), tf32_hi(kv.w));
        const float4 kl = make_float4(kv.x - kh.x, kv.y - kh.y, kv.z - kh.z, kv.w - kh.w);
        if (in_mp) {
          store_row4(khi, MP, row, c0 + e, kh);
          store_row4(klo, MP, row, c0 + e, kl);
        }
        const float q4[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float hh = tf32_hi(q4[t]);
          qh[e + t] = __float_as_uint(hh);
          ql[e + t] = __float_as_uint(q4[t] - hh);
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
  if (tid == 0) {
    tc_fence_after_sync();
    issue(COL_S, COL_QH, khi, MP, d, false);
    issue(COL_S, COL_QH, klo, MP, d, true);
    issue(COL_S, COL_QL, khi, MP, d, true);
    mma_commit(&bar_mma);
  }
  wait_mma();
  __syncthreads();
  // row softmax of the scores (scale 1/sqrt(d)) by the first half of the
  // CTA; A_S -> TMEM (A operand) and -> bbuf rows
  if (half == 0) {
    float rmax = -INFINITY;
    for (int j0 = 0; j0 < MP; j0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + lo + COL_S + j0, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (j0 + e < m) rmax = fmaxf(rmax, __uint_as_float(r[e]));
    }
    float sum = 0.f;
    for (int j0 = 0; j0 < MP; j0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + lo + COL_S + j0, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x = (live && j0 + e < m) ? expf((__uint_as_float(r[e]) - rmax) * p.scale) : 0.f;
        sum += x;
        r[e] = __float_as_uint(x);
      }
      tmem_st32(tmem + lo + COL_S + j0, r);
    }
    tmem_st_wait();
    const float inv = live ? 1.f / sum : 0.f;
    float rs = 0.f;
    for (int j0 = 0; j0 < MP; j0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + lo + COL_S + j0, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x = __uint_as_float(r[e]) * inv;
        r[e] = __float_as_uint(x);
        rs += fabsf(x);
      }
      // A_S row -> A operand (only dead Q~ / score columns are overwritten)
      tmem_st32(tmem + lo + COL_A + j0, r);
      if (in_mp) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          store_row4(bbuf, MP, row, j0 + e,
                     make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                                 __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])));
      }
    }
    // ||A_S||_inf: largest row abs-sum
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rs = fmaxf(rs, __shfl_xor_sync(0xffffffffu, rs, o));
    if (lane == 0) red_row[quarter] = rs;
    tmem_st_wait();
  }
  __syncthreads();
  // ||A_S||_1: largest column abs-sum. Thread (row j, half h) sums column j
  // over half of the rows with four independent partial sums.
  {
    float c4[4] = {0.f, 0.f, 0.f, 0.f};
    if (in_mp) {
      const int i0 = half * (MP >> 1), i1 = i0 + (MP >> 1);
      for (int i = i0; i < i1; i += 4) {
#pragma unroll
        for (int t = 0; t < 4; ++t)
          c4[t] += fabsf(*reinterpret_cast<const float*>(bbuf + kmaj_off(i + t, row, MP)));
      }
    }
    red_col[tid] = (c4[0] + c4[1]) + (c4[2] + c4[3]);
  }
  // stage export of A_S: coalesced copy of the bbuf rows
  {
    float* a_out = p.a_s + (size_t)bh * m * m;
    for (int e = tid; e < m * m; e += kThreads)
      a_out[e] = *reinterpret_cast<const float*>(bbuf + kmaj_off(e / m, e % m, MP));
  }
  __syncthreads();
  if (warp == 0) {
    float cs = 0.f;
    for (int j = lane; j < 128; j += 32) cs = fmaxf(cs, red_col[j] + red_col[j + 128]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cs = fmaxf(cs, __shfl_xor_sync(0xffffffffu, cs, o));
    if (lane == 0) red_col[0] = cs;
  }
  __syncthreads();
  const float alpha = 1.f / (red_col[0] * fmaxf(fmaxf(red_row[0], red_row[1]), fmaxf(red_row[2], red_row[3])));
  // Z_0 = alpha A_S^T: row i of Z_0 is alpha * column i of A_S -> TMEM
  for (int c = half; c < nch; c += 2) {
    uint32_t r[32];
#pragma unroll
    for (int e = 0; e < 32; ++e)
      r[e] = __float_as_uint(in_mp ? alpha * *reinterpret_cast<const float*>(bbuf + kmaj_off(c * 32 + e, row, MP)) : 0.f);
    tmem_st32(tmem + lo + COL_Z + c * 32, r);
  }
  __syncthreads();  // every column read done before the rows are rescaled
  // B operand of X = A_S Z_0: Z_0 stored by columns = alpha * A_S rows
  if (in_mp)
    for (int c = half; c < nch; c += 2)
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        float4* e4 = reinterpret_cast<float4*>(bbuf + kmaj_off(row, c * 32 + e, MP));
        float4 v = *e4;
        v.x *= alpha; v.y *= alpha; v.z *= alpha; v.w *= alpha;
        *e4 = v;
      }
  // ---- 2) G = merge of the key-split partials; G^T into gbuf (B of W = Z G)
  {
    float gm = -INFINITY;
    if (live)
      for (int sp = 0; sp < p.splits; ++sp)
        gm = fmaxf(gm, p.gml[(((size_t)bh * p.splits + sp) * m + row) * 2]);
    float den = 0.f;
    if (live)
      for (int sp = 0; sp < p.splits; ++sp) {
        const size_t prow = ((size_t)bh * p.splits + sp) * m + row;
        if (p.gml[prow * 2] == -INFINITY) continue;  // empty partial
        den += p.gml[prow * 2 + 1] * expf(p.gml[prow * 2] - gm);
      }
    const float inv = live ? 1.f / den : 0.f;
    float* grow_out = p.g + ((size_t)bh * m + (live ? row : 0)) * d;
    for (int c0 = half * 32; c0 < d; c0 += 64) {
      float acc[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) acc[e] = 0.f;
      if (live) {
        for (int sp = 0; sp < p.splits; ++sp) {
          const size_t prow = ((size_t)bh * p.splits + sp) * m + row;
          if (p.gml[prow * 2] == -INFINITY) continue;  // empty partial: O never written
          const float f = expf(p.gml[prow * 2] - gm);
          const float4* src = reinterpret_cast<const float4*>(p.gpart + prow * d + c0);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 v = src[e];
            acc[4 * e] += v.x * f;
            acc[4 * e + 1] += v.y * f;
            acc[4 * e + 2] += v.z * f;
            acc[4 * e + 3] += v.w * f;
          }
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] *= inv;
        float4* go = reinterpret_cast<float4*>(grow_out + c0);
#pragma unroll
        for (int e = 0; e < 8; ++e) go[e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
      }
      if (in_mp) store_col32(gbuf, d, row, c0, acc);
    }
  }
  fence_async_smem();
  tmem_st_wait();
  tc_fence_before_sync();
  __syncthreads();

  // ---- 3) the iteration
  auto gemm = [&](uint32_t d_col, uint32_t a_col, const uint8_t* b, int b_rows) {
    if (tid == 0) {
      tc_fence_after_sync();
      issue(d_col, a_col, b, b_rows, MP, false);
      mma_commit(&bar_mma);
    }
    wait_mma();
  };
  // epilogue: this row of D -> sign * scale * D + diag * I, written
  // transposed as the next product's B operand (element (i, j) -> storage
  // row j, column i); optionally also Z <- scale * D in TMEM.
  auto store_bt = [&](float diag, float sign, float scale_, uint32_t col, bool to_z) {
    for (int c = half; c < nch; c += 2) {
      const int j0 = c * 32;
      uint32_t r[32];
      tmem_ld32(tmem + lo + col + j0, r);
      tmem_ld_wait();
      float v[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x = scale_ * __uint_as_float(r[e]);
        r[e] = __float_as_uint(x);
        v[e] = fmaf(sign, x, (j0 + e == row) ? diag : 0.f);
      }
      if (in_mp) store_col32(bbuf, MP, row, j0, v);
      if (to_z) tmem_st32(tmem + lo + COL_Z + j0, r);
    }
    fence_async_smem();
    tmem_st_wait();
    tc_fence_before_sync();
    __syncthreads();
  };
  for (int it = 0; it < p.iters && !*abort_flag; ++it) {
    gemm(COL_X, COL_A, bbuf, MP);             // X = A_S Z
    if (*abort_flag) break;
    store_bt(7.f, -1.f, 1.f, COL_X, false);   // B <- 7I - X
    gemm(COL_Y, COL_X, bbuf, MP);             // Y = X (7I - X)
    if (*abort_flag) break;
    store_bt(15.f, -1.f, 1.f, COL_Y, false);  // B <- 15I - Y
    gemm(COL_Y, COL_X, bbuf, MP);             // Y = X (15I - ...)
    if (*abort_flag) break;
    store_bt(13.f, -1.f, 1.f, COL_Y, false);  // B <- 13I - Y
    gemm(COL_Y, COL_Z, bbuf, MP);             // Y = Z (13I - ...)
    if (*abort_flag) break;
    store_bt(0.f, 1.f, 0.25f, COL_Y, true);   // Z <- Y / 4 ; B <- Z by columns
  }
  // ---- 4) W = Z G
  if (!*abort_flag) {
    gemm(COL_Y, COL_Z, gbuf, d);
    if (!*abort_flag) {
      float* wrow = p.w + ((size_t)bh * m + (live ? row : 0)) * d;
      __nv_bfloat16* wt = p.wt + (size_t)bh * p.dpad * p.m64;
      for (int c0 = half * 32; c0 < d; c0 += 64) {
        uint32_t r[32];
        tmem_ld32(tmem + lo + COL_Y + c0, r);
        tmem_ld_wait();
        if (live) {
          float4* wo = reinterpret_cast<float4*>(wrow + c0);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            wo[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
        }
        if (row < p.m64) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            wt[(size_t)(c0 + e) * p.m64 + row] = __float2bfloat16_rn(live ? __uint_as_float(r[e]) : 0.f);
        }
      }
      if (half == 0 && row < p.m64)
        for (int c = d; c < p.dpad; ++c) wt[(size_t)c * p.m64 + row] = __float2bfloat16_rn(0.f);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, p.tmem_cols);
}

// m rounded up to 32, 64 or 128 (zero padding of A_S is exact: the
// padded block of every iterate stays zero)
int mpad_of(int m) { return m <= 32 ? 32 : (m <= 64 ? 64 : 128); }

}  // namespace

bool pinv_tc_supported(const Shape& s) { return s.dtype == NYS_BF16 && s.m <= 128; }

int launch_pinv_tc(const Shape& s, const float* qt, const float* kt, const float* gpart,
                   const float* gml, float* g, float* a_s, float* w, void* wt_bf16, int splits,
                   int* status, cudaStream_t stream) {
  if (!pinv_tc_supported(s)) return NYS_ERR_UNSUPPORTED;
  PinvParams p{};
  p.qt = qt;
  p.kt = kt;
  p.gpart = gpart;
  p.gml = gml;
  p.g = g;
  p.a_s = a_s;
  p.w = w;
  p.wt = static_cast<__nv_bfloat16*>(wt_bf16);
  p.status = status;
  p.m = s.m;
  p.d = s.d;
  p.m_pad = mpad_of(s.m);
  p.dpad = s.dpad();
  p.m64 = s.m64();
  p.splits = splits;
  p.iters = s.iters;
  p.scale = 1.0f / sqrtf((float)s.d);
  const uint32_t need = std::max<uint32_t>(3 * p.m_pad + std::max(p.m_pad, s.d),
                                           2 * s.d + p.m_pad);
  uint32_t cols = 32;
  while (cols < need) cols <<= 1;
  p.tmem_cols = cols;
  const size_t bbytes = (size_t)p.m_pad * p.m_pad * 4;
  const size_t gbytes = (size_t)s.d * p.m_pad * 4;
  p.gbuf_off = (uint32_t)bbytes;
  // K~ hi / lo (prologue only) share space with the operand buffers
  const size_t kbytes = (size_t)p.m_pad * s.d * 4;
  p.klo_off = (uint32_t)kbytes;
  const size_t smem = std::max(bbytes + gbytes, 2 * kbytes) + 1024;
  if (cudaFuncSetAttribute(pinv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return NYS_ERR_CUDA;
  KernelScope scope("pinv_tc", stream);
  pinv_tc<<<(unsigned)s.bh(), kThreads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? NYS_OK : NYS_ERR_CUDA;
}

}  // namespace nys
