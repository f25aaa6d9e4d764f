// Plain CUDA-core (SIMT) kernels for every step of the forward pass, fp32
// arithmetic throughout. They are the path for float32 inputs, where the
// output must stay within 1e-4 of an fp64 result and tensor-core rounding
// (bf16 / tf32 operands) would not do.
//
// Steps (the "Nyströmformer" review page, Proposed method, bullets 2-6):
//   landmarks   Q~, K~ = segment means                          (bullet 4)
//   rows        G = softmax(Q~ K^T s) V, split over keys with an
//               online softmax; partial (sum, max, sum-of-exp)  (bullets 3, 6)
//   pinv        merge partials; A_S = softmax(Q~ K~^T s); Z_0 = A_S^T /
//               (||A_S||_1 ||A_S||_inf); iters x cubic update; W = Z G
//                                                               (bullets 2, 5)
//   tokens      out = softmax(Q K~^T s) W + DWConv(V)           (bullets 3, 6)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "nys_internal.h"

namespace nys {
namespace {

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float x) { *p = x; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ---------------------------------------------------------------- landmarks
// Segment i of n rows split into m: rows [lo, lo + len) with
// lo = floor(i n / m), so every segment has n/m rows when m divides n and
// floor(n/m) or ceil(n/m) rows otherwise (m <= n: none is empty).
__device__ __forceinline__ void segment_rows(int i, int n, int m, int& lo, int& len) {
  lo = (int)((long long)i * n / m);
  len = (int)((long long)(i + 1) * n / m) - lo;
}

// grid (ceil(m64*dpad/256), B*H), block 256: one thread per landmark element
// of the padded [m64][dpad] grid. Writes Q~, K~ (fp32, [m][d]) and, when
// kt_b is given, K~ as bf16 [m64][dpad] with zeros in the padding.
template <typename T>
__global__ void __launch_bounds__(256)
landmarks_simt(const T* __restrict__ q, const T* __restrict__ k, float* __restrict__ qt,
               float* __restrict__ kt, __nv_bfloat16* __restrict__ qt_b,
               __nv_bfloat16* __restrict__ kt_b, int n, int d, int m, int m64, int dpad,
               const int* __restrict__ lengths, int H) {
  const long long bh = blockIdx.y;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= m64 * dpad) return;
  const int i = idx / dpad, c = idx % dpad;
  if (i >= m || c >= d) {
    if (kt_b) kt_b[(size_t)bh * m64 * dpad + idx] = __float2bfloat16_rn(0.f);
    if (qt_b) qt_b[(size_t)bh * m64 * dpad + idx] = __float2bfloat16_rn(0.f);
    return;
  }
  int lo, seg;
  segment_rows(i, lengths ? lengths[bh / H] : n, m, lo, seg);
  const size_t base = ((size_t)bh * n + (size_t)lo) * d + c;
  float sq = 0.f, sk = 0.f;
  for (int t = 0; t < seg; ++t) {
    sq += ld(q + base + (size_t)t * d);
    if (k) sk += ld(k + base + (size_t)t * d);
  }
  const float mq = sq / (float)seg, mk = sk / (float)seg;
  qt[((size_t)bh * m + i) * d + c] = mq;
  if (k) kt[((size_t)bh * m + i) * d + c] = mk;
  if (kt_b) kt_b[(size_t)bh * m64 * dpad + idx] = __float2bfloat16_rn(mk);
  if (qt_b) qt_b[(size_t)bh * m64 * dpad + idx] = __float2bfloat16_rn(mq);
}

// Segment means with one warp per (tensor, head, segment). A segment is
// len consecutive rows, i.e. one contiguous block of len*d elements; lanes
// stream it with 16-byte loads. With V elements per load and VPR = d / V
// loads per row dividing 32, lane l always sees column group l % VPR, so
// the per-column sums finish with shuffles over lanes l, l+VPR, ... .
// Warps for padding rows (m <= i < m64) write zeros to the bf16 copies.
// grid: (ceil(2 * B*H * m64 / 8)), block 256.
template <typename T>
__global__ void __launch_bounds__(256)
landmarks_vec(const T* __restrict__ q, const T* __restrict__ k, float* __restrict__ qt,
              float* __restrict__ kt, __nv_bfloat16* __restrict__ qt_b,
              __nv_bfloat16* __restrict__ kt_b, long long n_heads, int n, int d, int m, int m64,
              int dpad, const int* __restrict__ lengths, int H) {
  constexpr int V = 16 / sizeof(T);
  const long long job = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (job >= 2 * n_heads * m64) return;
  const int tensor = (int)(job / (n_heads * m64));
  const long long rest = job - (long long)tensor * n_heads * m64;
  const long long bh = rest / m64;
  const int i = (int)(rest % m64);
  __nv_bfloat16* outb = tensor == 0 ? qt_b : kt_b;
  if (i >= m) {
    if (outb)
      for (int c = lane; c < dpad; c += 32) outb[((size_t)bh * m64 + i) * dpad + c] = __float2bfloat16_rn(0.f);
    return;
  }
  int lo, seg;
  segment_rows(i, lengths ? lengths[bh / H] : n, m, lo, seg);
  const int vpr = d / V;
  const T* src = (tensor == 0 ? q : k) + ((size_t)bh * n + (size_t)lo) * d;
  const uint4* src4 = reinterpret_cast<const uint4*>(src);
  const int nvec = seg * vpr;
  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  // eight 16-byte loads in flight per lane, then the sums
  int v = lane;
  for (; v + 7 * 32 < nvec; v += 8 * 32) {
    uint4 u[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) u[r] = __ldg(src4 + v + 32 * r);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const T* x = reinterpret_cast<const T*>(&u[r]);
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] += ld(x + e);
    }
  }
  for (; v < nvec; v += 32) {
    const uint4 u = __ldg(src4 + v);
    const T* x = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] += ld(x + e);
  }
  for (int o = vpr; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
  if (lane < vpr) {
    const float inv = 1.f / (float)seg;
    float* out = (tensor == 0 ? qt : kt) + ((size_t)bh * m + i) * d + lane * V;
#pragma unroll
    for (int e = 0; e < V; ++e) out[e] = acc[e] * inv;
    if (outb) {
      __nv_bfloat16* ob = outb + ((size_t)bh * m64 + i) * dpad + lane * V;
#pragma unroll
      for (int e = 0; e < V; ++e) ob[e] = __float2bfloat16_rn(acc[e] * inv);
    }
  }
  if (outb)
    for (int c = d + lane; c < dpad; c += 32) outb[((size_t)bh * m64 + i) * dpad + c] = __float2bfloat16_rn(0.f);
}

// Small segments (ceil(n/m) * d / V <= 128 16-byte vectors): one warp takes
// SPW = 32 / VPR consecutive segments of one (tensor, head); lane l owns
// segment l / VPR and column group l % VPR (V columns) and sums that
// segment's rows for its columns itself (no shuffles), eight rows' loads in
// flight at a time; a warp-wide load covers SPW rows of 16 * VPR bytes. The
// warp runs to the longest segment's length; shorter segments' lanes skip
// the rows past their own end.
// Padding rows (m <= i < m64) get zeros in the bf16 copies.
// grid: (ceil(2 * B*H * ceil(m64 / SPW) / 8)), block 256.
template <typename T>
__global__ void __launch_bounds__(256)
landmarks_small(const T* __restrict__ q, const T* __restrict__ k, float* __restrict__ qt,
                float* __restrict__ kt, __nv_bfloat16* __restrict__ qt_b,
                __nv_bfloat16* __restrict__ kt_b, long long n_heads, int n, int d, int m, int m64,
                int dpad, const int* __restrict__ lengths, int H) {
  constexpr int V = 16 / sizeof(T);
  const int vpr = d / V, spw = 32 / vpr;
  const int nblk = (m64 + spw - 1) / spw;
  const long long job = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (job >= 2 * n_heads * nblk) return;
  const int tensor = (int)(job / (n_heads * nblk));
  const long long rest = job - (long long)tensor * n_heads * nblk;
  const long long bh = rest / nblk;
  const int sl = lane / vpr, cg = lane - sl * vpr;
  const int i = (int)(rest % nblk) * spw + sl;
  const int seg_max = (int)(((long long)n + m - 1) / m);
  __nv_bfloat16* outb = tensor == 0 ? qt_b : kt_b;
  if (i >= m64) return;
  if (i >= m) {
    if (outb)
      for (int c = cg * V; c < dpad; c += vpr * V)
#pragma unroll
        for (int e = 0; e < V; ++e) outb[((size_t)bh * m64 + i) * dpad + c + e] = __float2bfloat16_rn(0.f);
    return;
  }
  int lo, seg;
  segment_rows(i, lengths ? lengths[bh / H] : n, m, lo, seg);  // seg <= seg_max (length <= n)
  const uint4* src = reinterpret_cast<const uint4*>((tensor == 0 ? q : k) + ((size_t)bh * n + (size_t)lo) * d) + cg;
  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  for (int r0 = 0; r0 < seg_max; r0 += 8) {
    uint4 u[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) u[r] = r0 + r < seg ? __ldg(src + (size_t)(r0 + r) * vpr) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const T* x = reinterpret_cast<const T*>(&u[r]);
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] += ld(x + e);
    }
  }
  const float inv = 1.f / (float)seg;
  // V consecutive means as 16-byte stores (cg * V elements into a row of
  // d >= 8: 16-byte aligned)
  float* out = (tensor == 0 ? qt : kt) + ((size_t)bh * m + i) * d + cg * V;
#pragma unroll
  for (int e = 0; e < V; e += 4)
    *reinterpret_cast<float4*>(out + e) = make_float4(acc[e] * inv, acc[e + 1] * inv, acc[e + 2] * inv, acc[e + 3] * inv);
  if (outb) {
    __nv_bfloat16* ob = outb + ((size_t)bh * m64 + i) * dpad + cg * V;
    if constexpr (V == 8) {
      __nv_bfloat162 h2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) h2[e] = __floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
      *reinterpret_cast<uint4*>(ob) = *reinterpret_cast<const uint4*>(h2);
    } else {
#pragma unroll
      for (int e = 0; e < V; ++e) ob[e] = __float2bfloat16_rn(acc[e] * inv);
    }
    for (int c = d + cg * V; c < dpad; c += vpr * V)
#pragma unroll
      for (int e = 0; e < V; ++e) outb[((size_t)bh * m64 + i) * dpad + c + e] = __float2bfloat16_rn(0.f);
  }
}

// -------------------------------------------------------------------- rows
// grid (ceil(m/8), splits, B*H), block 128. CTA: 8 landmark rows x one key
// range, keys in chunks of 32. Writes unnormalised partial O, and (max, sum).
constexpr int RW_ROWS = 8, RW_KEYS = 32;

template <typename T>
__global__ void __launch_bounds__(128)
rows_simt(const float* __restrict__ qt, const T* __restrict__ k, const T* __restrict__ v,
          float* __restrict__ gpart, float* __restrict__ gml, int n, int d, int m, int splits,
          int keys_per_split, float scale, const int* __restrict__ lengths, int H) {
  extern __shared__ float sm[];
  float* sq = sm;                          // [8][d]
  float* sk = sq + RW_ROWS * d;            // [32][d+1]
  float* sv = sk + RW_KEYS * (d + 1);      // [32][d]
  float* sp = sv + RW_KEYS * d;            // [8][32]
  float* salpha = sp + RW_ROWS * RW_KEYS;  // [8]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r0 = blockIdx.x * RW_ROWS, split = blockIdx.y;
  const long long bh = blockIdx.z;
  for (int e = tid; e < RW_ROWS * d; e += 128) {
    const int r = e / d, c = e % d;
    sq[e] = (r0 + r < m) ? qt[((size_t)bh * m + r0 + r) * d + c] * scale : 0.f;
  }
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
  const int key0 = split * keys_per_split;
  // keys past the head's length (padding) take no part: a range that lies
  // wholly in the padding leaves an empty partial (max = -inf)
  const int key1 = min(lengths ? lengths[bh / H] : n, key0 + keys_per_split);
  const T* kb = k + (size_t)bh * n * d;
  const T* vb = v + (size_t)bh * n * d;
  for (int kc = key0; kc < key1; kc += RW_KEYS) {
    const int nk = min(RW_KEYS, key1 - kc);
    __syncthreads();
    for (int e = tid; e < RW_KEYS * d; e += 128) {
      const int j = e / d, c = e % d;
      float kv = 0.f, vv = 0.f;
      if (j < nk) {
        kv = ld(kb + (size_t)(kc + j) * d + c);
        vv = ld(vb + (size_t)(kc + j) * d + c);
      }
      sk[j * (d + 1) + c] = kv;
      sv[j * d + c] = vv;
    }
    __syncthreads();
    for (int p = tid; p < RW_ROWS * RW_KEYS; p += 128) {
      const int r = p / RW_KEYS, j = p % RW_KEYS;
      float s = 0.f;
      for (int c = 0; c < d; ++c) s += sq[r * d + c] * sk[j * (d + 1) + c];
      sp[p] = (j < nk) ? s : -INFINITY;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = warp * 2 + rr;
      const float s = sp[r * RW_KEYS + lane];
      const float mnew = fmaxf(mrun[rr], warp_max(s));
      const float p = (lane < nk) ? expf(s - mnew) : 0.f;
      const float alpha = expf(mrun[rr] - mnew);
      lrun[rr] = lrun[rr] * alpha + warp_sum(p);
      mrun[rr] = mnew;
      sp[r * RW_KEYS + lane] = p;
      if (lane == 0) salpha[r] = alpha;
    }
    __syncthreads();
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int e = tid + 128 * jj;
      if (e < RW_ROWS * d) {
        const int r = e / d, c = e % d;
        float a = acc[jj] * salpha[r];
        for (int j = 0; j < nk; ++j) a += sp[r * RW_KEYS + j] * sv[j * d + c];
        acc[jj] = a;
      }
    }
  }
  const size_t pbase = ((size_t)bh * splits + split) * m;
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) {
    const int e = tid + 128 * jj;
    if (e < RW_ROWS * d) {
      const int r = e / d, c = e % d;
      if (r0 + r < m) gpart[(pbase + r0 + r) * d + c] = acc[jj];
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = r0 + warp * 2 + rr;
      if (r < m) {
        gml[(pbase + r) * 2 + 0] = mrun[rr];
        gml[(pbase + r) * 2 + 1] = lrun[rr];
      }
    }
  }
}

// ---------------------------------------------------------------- merge G
// G = merge of the key-split partials (bullets 3 and 6: softmax(Q~ K^T s) V
// from the per-range sums). One thread per float4 of G (a column of CTAs
// per head: no 64-bit index divisions); splits in batches of SB (no more
// than there are, up to eight) with all their loads in flight, a running
// (max, denominator) that rescales the accumulated sum as in an online
// softmax; an empty partial (max = -inf) was never written and contributes
// nothing.
// grid (B*H, ceil(m * d / 4 / 256)), block 256.
template <int SB>  // splits per batch of loads (2, 4 or 8)
__global__ void __launch_bounds__(256)
merge_g(const float* __restrict__ gp, const float* __restrict__ gml, float* __restrict__ g, int m,
        int d, int splits) {
  const int d4 = d >> 2;
  const int e = (int)blockIdx.y * 256 + (int)threadIdx.x;  // float4 of this head's G
  if (e >= m * d4) return;
  const long long bh = blockIdx.x;
  const int i = e / d4;
  const float2* ml = reinterpret_cast<const float2*>(gml) + (bh * splits * m + i);
  const float4* src = reinterpret_cast<const float4*>(gp) + bh * splits * m * d4 + e;
  const size_t sstride = (size_t)m * d4;  // float4s between splits
  float gm = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sp = 0; sp < splits; sp += SB) {
    float2 mk[SB];
    float4 o[SB];
#pragma unroll
    for (int k = 0; k < SB; ++k) {
      const int s2 = sp + k < splits ? sp + k : sp;
      mk[k] = __ldg(ml + (size_t)s2 * m);
      o[k] = __ldg(src + (size_t)s2 * sstride);
    }
    float cm = gm;
#pragma unroll
    for (int k = 0; k < SB; ++k)
      if (sp + k < splits && mk[k].x != -INFINITY) cm = fmaxf(cm, mk[k].x);
    if (cm == -INFINITY) continue;  // only empty partials so far
    const float rs = gm == -INFINITY ? 0.f : expf(gm - cm);
    den *= rs;
    acc = make_float4(acc.x * rs, acc.y * rs, acc.z * rs, acc.w * rs);
#pragma unroll
    for (int k = 0; k < SB; ++k)
      if (sp + k < splits && mk[k].x != -INFINITY) {
        const float f = expf(mk[k].x - cm);
        den = fmaf(mk[k].y, f, den);
        acc = make_float4(fmaf(o[k].x, f, acc.x), fmaf(o[k].y, f, acc.y), fmaf(o[k].z, f, acc.z),
                          fmaf(o[k].w, f, acc.w));
      }
    gm = cm;
  }
  const float inv = 1.f / den;
  reinterpret_cast<float4*>(g)[bh * m * d4 + e] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

// -------------------------------------------------------------------- pinv
// Block-wide C = diag * I + alpha * A B on float matrices in global memory
// (the head's workspace, L2-resident). B is [K][N] row-major, or [N][K]
// row-major when b_trans. 256 threads, 64x64 output tiles, 4x4 per thread.
// C must not alias A or B.
constexpr int GT = 64, GK = 16, GP = GT + 4;

__device__ void block_gemm(const float* A, int lda, const float* Bm, int ldb, bool b_trans,
                           float* C, int ldc, int M, int N, int K, float alpha, float diag,
                           float* smem) {
  float* As = smem;            // [GK][GP]: As[kk][row]
  float* Bs = smem + GK * GP;  // [GK][GP]: Bs[kk][col]
  const int tid = threadIdx.x, tr = tid / 16, tc = tid % 16;
  for (int m0 = 0; m0 < M; m0 += GT) {
    for (int n0 = 0; n0 < N; n0 += GT) {
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
      for (int k0 = 0; k0 < K; k0 += GK) {
        __syncthreads();
        for (int e = tid; e < GT * GK; e += 256) {
          const int r = e / GK, kk = e % GK, gr = m0 + r, gk = k0 + kk;
          As[kk * GP + r] = (gr < M && gk < K) ? A[(size_t)gr * lda + gk] : 0.f;
        }
        for (int e = tid; e < GT * GK; e += 256) {
          int kk, c;
          if (b_trans) { c = e / GK; kk = e % GK; } else { kk = e / GT; c = e % GT; }
          const int gk = k0 + kk, gc = n0 + c;
          float x = 0.f;
          if (gk < K && gc < N) x = b_trans ? Bm[(size_t)gc * ldb + gk] : Bm[(size_t)gk * ldb + gc];
          Bs[kk * GP + c] = x;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < GK; ++kk) {
          float a[4], b[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) a[i] = As[kk * GP + tr * 4 + i];
#pragma unroll
          for (int j = 0; j < 4; ++j) b[j] = Bs[kk * GP + tc * 4 + j];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] += a[i] * b[j];
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int gr = m0 + tr * 4 + i, gc = n0 + tc * 4 + j;
          if (gr < M && gc < N) C[(size_t)gr * ldc + gc] = alpha * acc[i][j] + (gr == gc ? diag : 0.f);
        }
      }
    }
  }
  __syncthreads();
}

// C = diag * I + alpha * A B for m x m matrices (m <= 64) held in shared
// memory with row pitch kResPitch, zero past m (and C kept so: the diagonal
// term only inside m). 256 threads, a 4 x 4 block of C each; the products
// run from shared memory without a barrier per step. C must not alias A or B.
constexpr int kResPitch = 68, kResM = 64;
constexpr int kCoefMax = 4096;  // split weights kept in shared memory: splits * m at most

__device__ void smem_gemm64(const float* A, const float* B, float* C, int m, float alpha, float diag) {
  const int tid = threadIdx.x, tr = tid >> 4, tc = tid & 15;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k = 0; k < m; ++k) {
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = A[(4 * tr + i) * kResPitch + k];
    const float4 b = *reinterpret_cast<const float4*>(B + k * kResPitch + 4 * tc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[i][0] = fmaf(a[i], b.x, acc[i][0]);
      acc[i][1] = fmaf(a[i], b.y, acc[i][1]);
      acc[i][2] = fmaf(a[i], b.z, acc[i][2]);
      acc[i][3] = fmaf(a[i], b.w, acc[i][3]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * tr + i;
    float4 o;
    o.x = alpha * acc[i][0] + (r == 4 * tc && r < m ? diag : 0.f);
    o.y = alpha * acc[i][1] + (r == 4 * tc + 1 && r < m ? diag : 0.f);
    o.z = alpha * acc[i][2] + (r == 4 * tc + 2 && r < m ? diag : 0.f);
    o.w = alpha * acc[i][3] + (r == 4 * tc + 3 && r < m ? diag : 0.f);
    *reinterpret_cast<float4*>(C + r * kResPitch + 4 * tc) = o;
  }
  __syncthreads();
}

// grid (B*H), block 256. Everything for one head: merge the key-split
// partials into G, form A_S, run the iteration, write W = Z G. For m <= 64
// the iteration runs on matrices resident in shared memory (dynamic, five
// 64 x 64 blocks); larger m streams them through the head's workspace.
__global__ void __launch_bounds__(256, 1)
pinv_simt(const float* __restrict__ qt_all, const float* __restrict__ kt_all,
          const float* __restrict__ gpart, const float* __restrict__ gml, float* __restrict__ g_all,
          float* __restrict__ a_all, float* __restrict__ z_all, float* __restrict__ w_all,
          float* __restrict__ scratch_all, __nv_bfloat16* __restrict__ wt_b, int d, int m,
          int splits, int iters, float scale, int m64, int dpad) {
  __shared__ float smem[2 * GK * GP];
  __shared__ float red[2][8];
  extern __shared__ float dsm[];  // m <= 64: A_S, Z, X, U, T resident
  const long long bh = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t md = (size_t)m * d, mm = (size_t)m * m;
  const float* qt = qt_all + bh * md;
  const float* kt = kt_all + bh * md;
  float* g = g_all + bh * md;
  float* A = a_all + bh * mm;
  float* Z = z_all + bh * mm;
  float* W = w_all + bh * md;
  float* X = scratch_all + bh * 3 * mm;
  float* U = X + mm;
  float* V = U + mm;

  // 1) G = merge over splits of (O_s, max_s, sum_s)
  if (m <= kResM && splits * m <= kCoefMax) {  // uniform
    // each row's split weights f_s / den once, in shared memory after the
    // resident matrices; then every element is a weighted sum (an empty
    // partial, max -inf, has weight 0 and its rows are never read)
    float* coef = dsm + 5 * kResM * kResPitch;  // [splits][m]
    for (int i = tid; i < m; i += 256) {
      const float2* ml = reinterpret_cast<const float2*>(gml) + (size_t)bh * splits * m + i;
      float mx = -INFINITY;
      for (int s = 0; s < splits; ++s) mx = fmaxf(mx, ml[(size_t)s * m].x);
      float den = 0.f;
      for (int s = 0; s < splits; ++s) {
        const float2 v = ml[(size_t)s * m];
        const float f = v.x == -INFINITY ? 0.f : expf(v.x - mx);
        den += v.y * f;
        coef[s * m + i] = f;
      }
      const float inv = 1.f / den;
      for (int s = 0; s < splits; ++s) coef[s * m + i] *= inv;
    }
    __syncthreads();
    for (size_t e = tid; e < md; e += 256) {
      const int i = (int)(e / d), c = (int)(e % d);
      const float* gp = gpart + ((size_t)bh * splits * m + i) * d + c;
      float num = 0.f;
#pragma unroll 4
      for (int s = 0; s < splits; ++s) {
        const float w = coef[s * m + i];
        if (w != 0.f) num = fmaf(w, gp[(size_t)s * m * d], num);
      }
      g[e] = num;
    }
  } else
  for (size_t e = tid; e < md; e += 256) {
    const int i = (int)(e / d);
    float mx = -INFINITY;
    for (int s = 0; s < splits; ++s) mx = fmaxf(mx, gml[(((size_t)bh * splits + s) * m + i) * 2]);
    float num = 0.f, den = 0.f;
    for (int s = 0; s < splits; ++s) {
      const size_t row = ((size_t)bh * splits + s) * m + i;
      if (gml[row * 2] == -INFINITY) continue;  // empty partial: O never written
      const float f = expf(gml[row * 2] - mx);
      num += gpart[row * d + (e % d)] * f;
      den += gml[row * 2 + 1] * f;
    }
    g[e] = num / den;
  }
  // 2) A_S = softmax(Q~ K~^T s), rows by warps
  block_gemm(qt, d, kt, d, true, A, m, m, m, d, scale, 0.f, smem);
  for (int i = warp; i < m; i += 8) {
    float mx = -INFINITY;
    for (int j = lane; j < m; j += 32) mx = fmaxf(mx, A[(size_t)i * m + j]);
    mx = warp_max(mx);
    float sum = 0.f;
    for (int j = lane; j < m; j += 32) {
      const float p = expf(A[(size_t)i * m + j] - mx);
      A[(size_t)i * m + j] = p;
      sum += p;
    }
    sum = warp_sum(sum);
    const float inv = 1.f / sum;
    for (int j = lane; j < m; j += 32) A[(size_t)i * m + j] *= inv;
  }
  __syncthreads();
  // 3) Z_0 = A^T / (max column abs-sum * max row abs-sum)
  if (m <= kResM) {
    // A_S resident in shared memory from here on; the norms and Z_0 from it
    float* sA = dsm;
    float* zc = sA + kResM * kResPitch;      // Z
    float* zt = sA + 4 * kResM * kResPitch;  // T, then the next Z
    float* sX = sA + 2 * kResM * kResPitch;
    float* sU = sA + 3 * kResM * kResPitch;
    for (int e = tid; e < kResM * kResM; e += 256) {
      const int i = e / kResM, j = e % kResM;
      sA[i * kResPitch + j] = (i < m && j < m) ? A[(size_t)i * m + j] : 0.f;
    }
    __syncthreads();
    // thread j < m: column j's and row j's abs-sums, in index order
    float cs = 0.f, rs = 0.f;
    if (tid < m)
      for (int i = 0; i < m; ++i) {
        cs += fabsf(sA[i * kResPitch + tid]);
        rs += fabsf(sA[tid * kResPitch + i]);
      }
    float cm = warp_max(cs), rm = warp_max(rs);
    if (lane == 0) { red[0][warp] = cm; red[1][warp] = rm; }
    __syncthreads();
    if (tid == 0) {
      float c = 0.f, r = 0.f;
      for (int w = 0; w < 8; ++w) { c = fmaxf(c, red[0][w]); r = fmaxf(r, red[1][w]); }
      red[0][0] = 1.f / (c * r);
    }
    __syncthreads();
    const float alpha = red[0][0];
    for (int e = tid; e < kResM * kResM; e += 256) {
      const int i = e / kResM, j = e % kResM;
      zc[i * kResPitch + j] = sA[j * kResPitch + i] * alpha;
    }
    __syncthreads();
    // 4) Z <- 1/4 Z (13I - X (15I - X (7I - X))), X = A Z, in shared memory
    for (int it = 0; it < iters; ++it) {
      smem_gemm64(sA, zc, sX, m, 1.f, 0.f);  // X = A Z
      for (int e = tid; e < kResM * kResM; e += 256) {  // U = 7I - X
        const int i = e / kResM, j = e % kResM;
        sU[i * kResPitch + j] = (i == j && i < m ? 7.f : 0.f) - sX[i * kResPitch + j];
      }
      __syncthreads();
      smem_gemm64(sX, sU, zt, m, -1.f, 15.f);      // T = 15I - X U
      smem_gemm64(sX, zt, sU, m, -1.f, 13.f);      // U = 13I - X T
      smem_gemm64(zc, sU, zt, m, 0.25f, 0.f);      // Z' = Z U / 4
      float* t = zc;
      zc = zt;
      zt = t;
    }
    for (int e = tid; e < m * m; e += 256) Z[e] = zc[(e / m) * kResPitch + (e % m)];
    __syncthreads();
  }
  if (m > kResM) {  // uniform
  float cmax = 0.f, rmax = 0.f;
  for (int j = tid; j < m; j += 256) {
    float cs = 0.f, rs = 0.f;
    for (int i = 0; i < m; ++i) {
      cs += fabsf(A[(size_t)i * m + j]);
      rs += fabsf(A[(size_t)j * m + i]);
    }
    cmax = fmaxf(cmax, cs);
    rmax = fmaxf(rmax, rs);
  }
  cmax = warp_max(cmax);
  rmax = warp_max(rmax);
  if (lane == 0) { red[0][warp] = cmax; red[1][warp] = rmax; }
  __syncthreads();
  if (tid == 0) {
    float c = 0.f, r = 0.f;
    for (int w = 0; w < 8; ++w) { c = fmaxf(c, red[0][w]); r = fmaxf(r, red[1][w]); }
    red[0][0] = 1.f / (c * r);
  }
  __syncthreads();
  const float alpha0 = red[0][0];
  for (size_t e = tid; e < mm; e += 256) {
    const int i = (int)(e / m), j = (int)(e % m);
    Z[e] = A[(size_t)j * m + i] * alpha0;
  }
  __syncthreads();
  }
  // 4) (m > 64) Z <- 1/4 Z (13I - X (15I - X (7I - X))), X = A Z, through the workspace
  float* zc = Z;
  float* zn = V;
  for (int it = 0; m > kResM && it < iters; ++it) {
    block_gemm(A, m, zc, m, false, X, m, m, m, m, 1.f, 0.f, smem);            // X = A Z
    for (size_t e = tid; e < mm; e += 256)                                       // U = 7I - X
      U[e] = ((e / m) == (e % m) ? 7.f : 0.f) - X[e];
    __syncthreads();
    block_gemm(X, m, U, m, false, zn, m, m, m, m, -1.f, 15.f, smem);            // zn = 15I - X U
    block_gemm(X, m, zn, m, false, U, m, m, m, m, -1.f, 13.f, smem);            // U = 13I - X zn
    block_gemm(zc, m, U, m, false, zn, m, m, m, m, 0.25f, 0.f, smem);           // zn = Z U / 4
    float* t = zc; zc = zn; zn = t;
  }
  if (zc != Z) {
    for (size_t e = tid; e < mm; e += 256) Z[e] = zc[e];
    __syncthreads();
  }
  // 5) W = Z G
  block_gemm(Z, m, g, d, false, W, d, m, d, m, 1.f, 0.f, smem);
  // 6) W^T as bf16 [dpad][m64], zero padded, for the tensor-core token kernel
  if (wt_b) {
    __nv_bfloat16* wt = wt_b + (size_t)bh * dpad * m64;
    for (int e = tid; e < dpad * m64; e += 256) {
      const int c = e / m64, i = e % m64;
      wt[e] = __float2bfloat16_rn((c < d && i < m) ? W[(size_t)i * d + c] : 0.f);
    }
  }
}

// ------------------------------------------------------------------ tokens
// grid (ceil(n/32), B*H), block 256. CTA: 32 tokens; online softmax over
// landmark chunks of 32, then the depthwise conv of V and the store.
constexpr int TK_ROWS = 32, TK_LM = 32;

template <typename T>
__global__ void __launch_bounds__(256)
tokens_simt(const T* __restrict__ q, const T* __restrict__ v, const float* __restrict__ kt_all,
            const float* __restrict__ w_all, const float* __restrict__ conv_w, T* __restrict__ out,
            int H, int n, int d, int m, int ks, float scale) {
  extern __shared__ float sm[];
  float* sq = sm;                            // [32][d]
  float* sk = sq + TK_ROWS * d;              // [32][d+1]
  float* sw = sk + TK_LM * (d + 1);          // [32][d]
  float* sp = sw + TK_LM * d;                // [32][33]
  float* salpha = sp + TK_ROWS * 33;         // [32]
  float* sl = salpha + TK_ROWS;              // [32]
  float* svh = sl + TK_ROWS;                 // [32 + ks - 1][d]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * TK_ROWS;
  const long long bh = blockIdx.y;
  const int h = (int)(bh % H);
  const T* qb = q + (size_t)bh * n * d;
  const T* vb = v + (size_t)bh * n * d;
  const float* kt = kt_all + (size_t)bh * m * d;
  const float* W = w_all + (size_t)bh * m * d;
  for (int e = tid; e < TK_ROWS * d; e += 256) {
    const int r = e / d, c = e % d;
    sq[e] = (t0 + r < n) ? ld(qb + (size_t)(t0 + r) * d + c) * scale : 0.f;
  }
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  float mrun[4], lrun[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) { mrun[j] = -INFINITY; lrun[j] = 0.f; }
  for (int l0 = 0; l0 < m; l0 += TK_LM) {
    const int nl = min(TK_LM, m - l0);
    __syncthreads();
    for (int e = tid; e < TK_LM * d; e += 256) {
      const int i = e / d, c = e % d;
      sk[i * (d + 1) + c] = (i < nl) ? kt[(size_t)(l0 + i) * d + c] : 0.f;
      sw[i * d + c] = (i < nl) ? W[(size_t)(l0 + i) * d + c] : 0.f;
    }
    __syncthreads();
    for (int p = tid; p < TK_ROWS * TK_LM; p += 256) {
      const int r = p / TK_LM, i = p % TK_LM;
      float s = 0.f;
      for (int c = 0; c < d; ++c) s += sq[r * d + c] * sk[i * (d + 1) + c];
      sp[r * 33 + i] = (i < nl) ? s : -INFINITY;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = warp * 4 + rr;
      const float s = sp[r * 33 + lane];
      const float mnew = fmaxf(mrun[rr], warp_max(s));
      const float p = (lane < nl) ? expf(s - mnew) : 0.f;
      const float alpha = expf(mrun[rr] - mnew);
      lrun[rr] = lrun[rr] * alpha + warp_sum(p);
      mrun[rr] = mnew;
      sp[r * 33 + lane] = p;
      if (lane == 0) salpha[r] = alpha;
    }
    __syncthreads();
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const int e = tid + 256 * jj;
      if (e < TK_ROWS * d) {
        const int r = e / d, c = e % d;
        float a = acc[jj] * salpha[r];
        for (int i = 0; i < nl; ++i) a += sp[r * 33 + i] * sw[i * d + c];
        acc[jj] = a;
      }
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) sl[warp * 4 + rr] = lrun[rr];
  }
  // V rows t0 - r .. t0 + 31 + r (zero outside [0, n)) for the conv
  const int rad = ks > 0 ? (ks - 1) / 2 : 0;
  const int vrows = TK_ROWS + 2 * rad;
  for (int e = tid; e < vrows * d; e += 256) {
    const int u = t0 - rad + e / d, c = e % d;
    svh[e] = (ks > 0 && u >= 0 && u < n) ? ld(vb + (size_t)u * d + c) : 0.f;
  }
  __syncthreads();
  const float* wh = conv_w ? conv_w + (size_t)h * ks : nullptr;
#pragma unroll
  for (int jj = 0; jj < 16; ++jj) {
    const int e = tid + 256 * jj;
    if (e < TK_ROWS * d) {
      const int r = e / d, c = e % d;
      if (t0 + r < n) {
        float o = acc[jj] / sl[r];
        float cv = 0.f;
        for (int j = 0; j < ks; ++j) cv += wh[j] * svh[(r + j) * d + c];
        st(out + (size_t)bh * n * d + (size_t)(t0 + r) * d + c, o + cv);
      }
    }
  }
}

// -------------------------------------------------------------- conv, mask
// The depthwise convolution added to an output that holds the attention
// term alone, for the forms the fused token kernels do not cover: filters
// per channel ([H][d][ks]: channel c of head h has its own taps) and padded
// sequences (a batch entry's rows at or past its length are padding: they
// read as zero in the convolution and their output rows are zero). With
// ks = 0 it only zeroes the padding rows.
//   out[t][c] = t < L ? out[t][c] + sum_j w[j] V[t + j - (ks-1)/2][c] : 0,
//   V rows outside [0, L) read as zero, L = the entry's length (n if none).
// grid (ceil(n / (CV_ROWS nblk)), B*H), block CV_THREADS: a CTA takes nblk
// (at most CV_BLOCKS) consecutive blocks of CV_ROWS output rows of one head. The
// head's taps are staged once (tap-major, so that consecutive channels read
// consecutive words); per block, its V rows with the halo are staged in
// shared memory by 16-byte asynchronous copies (rows outside [0, len) zero),
// with two buffers (nbuf = 2) the next block's while this one is computed.
// A work item is CV_RUN consecutive rows of one column: the
// V window lives in a ring of CV_RUN registers, and with the tap loop
// unrolled in blocks of CV_RUN the ring's indices are static, so a tap costs
// one weight, one new V value and CV_RUN FMAs.
constexpr int CV_ROWS = 64, CV_THREADS = 256, CV_RUN = 16, CV_BLOCKS = 8;

// A block's V rows are staged in the input type. NARROW (bf16, or d <= 64):
// the staged rows and taps leave room for three CTAs per SM, so registers
// are capped to allow them (the attention term added after the taps so its
// loads overlap them); fp32 with d = 128 is bound by shared memory to two
// CTAs, and registers are capped for two.
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes sixteen
// zero bytes and reads nothing
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T, bool PER_CHANNEL, bool NARROW>
__global__ void __launch_bounds__(CV_THREADS, NARROW ? 3 : 2)
conv_mask(const T* __restrict__ v, const float* __restrict__ w, T* __restrict__ out, int H, int n,
          int d, int ks, const int* __restrict__ lengths, int nblk, int nbuf) {
  constexpr bool per_channel = PER_CHANNEL;
  extern __shared__ float sm[];
  const long long bh = blockIdx.y;
  const int h = (int)(bh % H);
  const int len = lengths ? lengths[bh / H] : n;
  const int rad = ks > 0 ? (ks - 1) / 2 : 0;
  const int vrows = CV_ROWS + 2 * rad;
  T* sv = reinterpret_cast<T*>(sm);                                  // [nbuf][vrows][d], input type
  float* sw = reinterpret_cast<float*>(sv + (size_t)nbuf * vrows * d);  // per channel: [ks][d]; per head: [ks]
  const T* vb = v + (size_t)bh * n * d;
  T* ob = out + (size_t)bh * n * d;
  const int tb0 = blockIdx.x * nblk * CV_ROWS;
  if (ks > 0 && tb0 < len) {
    if (per_channel) {
      // the head's [d][ks] taps, read in order, stored tap-major; eight
      // loads in flight per thread
      const float* wh = w + (size_t)h * d * ks;
      const int total = ks * d;
      for (int e0 = threadIdx.x; e0 < total; e0 += 8 * CV_THREADS) {
        float t[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int e = e0 + k * CV_THREADS;
          t[k] = e < total ? __ldg(wh + e) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int e = e0 + k * CV_THREADS;
          if (e < total) sw[(size_t)(e % ks) * d + e / ks] = t[k];
        }
      }
    } else {
      for (int j = threadIdx.x; j < ks; j += CV_THREADS) sw[j] = w[(size_t)h * ks + j];
    }
  }
  const int wstride = per_channel ? d : 1;  // word step between taps in sw
  const int ks_full = ks - ks % CV_RUN;     // taps in whole blocks of CV_RUN
  // block blk's V rows [t0 - rad, t0 + CV_ROWS + rad) into buffer blk % nbuf,
  // as one commit group (empty where the block has no conv work)
  constexpr int kEl = 16 / (int)sizeof(T);  // elements per 16-byte piece
  const int pr = d / kEl;                   // pieces per row (d is a multiple of 8)
  auto stage = [&](int blk) {
    const int t0 = tb0 + blk * CV_ROWS;
    if (ks > 0 && t0 < n && t0 < len) {
      T* dst = sv + (size_t)(blk % nbuf) * vrows * d;
      for (int e = threadIdx.x; e < vrows * pr; e += CV_THREADS) {
        const int row = e / pr, c = (e - row * pr) * kEl;
        const int u = t0 - rad + row;
        const bool in = u >= 0 && u < len;
        cp_async16(dst + (size_t)row * d + c, in ? vb + (size_t)u * d + c : vb, in ? 16 : 0);
      }
    }
    cp_async_commit();
  };
  stage(0);
  for (int blk = 0; blk < nblk; ++blk) {
    const int t0 = tb0 + blk * CV_ROWS;
    if (t0 >= n) break;  // uniform across the CTA
    const bool work = ks > 0 && t0 < len;
    const T* svb = sv + (size_t)(blk % nbuf) * vrows * d;
    if (nbuf == 1 && blk > 0) stage(blk);
    if (nbuf == 2 && blk + 1 < nblk && t0 + CV_ROWS < n) {
      stage(blk + 1);  // into block blk - 1's buffer, released at the end of its iteration
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // block blk's rows (and the taps) are in shared memory
    for (int item = threadIdx.x; item < (CV_ROWS / CV_RUN) * d; item += CV_THREADS) {
      const int c = item % d, r0 = (item / d) * CV_RUN;
      if (t0 + r0 >= n) continue;
      // the attention term already in out: all of the run's loads issued
      // before the taps (stored rows could alias later loads, so loads
      // after a store would wait); NARROW adds them after the taps, so that
      // their latency hides behind the FMAs
      float att[CV_RUN], acc[CV_RUN];
#pragma unroll
      for (int r = 0; r < CV_RUN; ++r) {
        const int t = t0 + r0 + r;
        const float a = (t < n && t < len) ? ld(ob + (size_t)t * d + c) : 0.f;
        att[r] = NARROW ? a : 0.f;
        acc[r] = NARROW ? 0.f : a;
      }
      if (work) {
        // ring: before tap j, V row (r0 + j + r) of the staged block sits in
        // xw[(j + r) % CV_RUN]; after it, the slot of row r0 + j takes row
        // r0 + j + CV_RUN (staged for every j < ks - 1)
        const T* x = svb + (size_t)r0 * d + c;
        const float* wp = sw + (per_channel ? c : 0);  // tap j of this channel: wp[j * wstride]
        const T* xp = x + (size_t)CV_RUN * d;          // row r0 + j + CV_RUN: xp[j * d]
        float xw[CV_RUN];
#pragma unroll
        for (int r = 0; r < CV_RUN; ++r) xw[r] = to_f(x[(size_t)r * d]);
        // whole blocks: no tap past ks, and (ks odd, CV_RUN even) never the
        // last tap, so every next row is inside the staged block
        for (int jb = 0; jb < ks_full; jb += CV_RUN) {
#pragma unroll
          for (int jj = 0; jj < CV_RUN; ++jj) {
            const float wj = wp[jj * wstride];
#pragma unroll
            for (int r = 0; r < CV_RUN; ++r) acc[r] = fmaf(wj, xw[(jj + r) % CV_RUN], acc[r]);
            xw[jj] = to_f(xp[jj * d]);
          }
          wp += CV_RUN * wstride;
          xp += CV_RUN * d;
        }
        // the last ks % CV_RUN taps
#pragma unroll
        for (int jj = 0; jj < CV_RUN; ++jj) {
          const int j = ks_full + jj;
          if (j >= ks) break;
          const float wj = wp[jj * wstride];
#pragma unroll
          for (int r = 0; r < CV_RUN; ++r) acc[r] = fmaf(wj, xw[(jj + r) % CV_RUN], acc[r]);
          if (j + 1 < ks) xw[jj] = to_f(xp[jj * d]);
        }
      }
#pragma unroll
      for (int r = 0; r < CV_RUN; ++r) {
        const int t = t0 + r0 + r;
        if (t >= n) break;
        st(ob + (size_t)t * d + c, t < len ? att[r] + acc[r] : 0.f);
      }
    }
    __syncthreads();  // every reader of this block's buffer is done before it is refilled
  }
}

template <typename T>
int conv_mask_t(const Shape& s, const void* v, const float* conv_w, void* out, cudaStream_t stream) {
  const int rad = s.ks > 0 ? (s.ks - 1) / 2 : 0;
  const bool per_channel = s.conv_layout == NYS_CONV_PER_CHANNEL;
  const bool narrow = sizeof(T) == 2 || s.d <= 64;
  // two V buffers (the next block's rows copied during this block's taps)
  // unless that leaves fewer CTAs per SM than one buffer: measured, a third
  // resident CTA hides more than the copy overlap does
  const size_t vbuf = sizeof(T) * (size_t)(CV_ROWS + 2 * rad) * s.d;
  const size_t taps = sizeof(float) * (size_t)s.ks * (per_channel ? s.d : 1);
  auto resident = [&](size_t bytes) {  // CTAs per SM: the launch bound, then shared memory
    return std::min<size_t>(narrow ? 3 : 2, (228 * 1024) / (bytes + 1024));
  };
  const int nbuf = 2 * vbuf + taps <= 227 * 1024 && resident(2 * vbuf + taps) >= resident(vbuf + taps) ? 2 : 1;
  const size_t smem = s.ks > 0 ? nbuf * vbuf + taps : 0;
  auto kern = per_channel ? (narrow ? conv_mask<T, true, true> : conv_mask<T, true, false>)
                          : (narrow ? conv_mask<T, false, true> : conv_mask<T, false, false>);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return set_cuda_error(cudaGetLastError());
  KernelScope ks_("conv_mask", stream);
  // blocks per CTA: up to CV_BLOCKS (the taps staged once for all of them),
  // fewer where that would leave SMs idle. (One wave of longer CTAs, sized
  // to the resident slots, was slower at B8 H8 n8192 d64: short CTAs let the
  // block scheduler even out the SMs' work as they finish.)
  const long long blocks = (long long)((s.n + CV_ROWS - 1) / CV_ROWS) * s.bh();
  const long long ctas_min = 2ll * plan_sms();
  const int nblk = (int)std::max(1ll, std::min<long long>(CV_BLOCKS, blocks / ctas_min));
  const dim3 grid((s.n + CV_ROWS * nblk - 1) / (CV_ROWS * nblk), (unsigned)s.bh());
  kern<<<grid, CV_THREADS, smem, stream>>>(static_cast<const T*>(v), s.ks > 0 ? conv_w : nullptr,
                                          static_cast<T*>(out), s.H, s.n, s.d, s.ks, s.lengths, nblk,
                                          s.ks > 0 ? nbuf : 1);
  return launch_status();
}

template <typename T>
int landmarks_t(const Shape& s, const void* q, const void* k, float* qt, float* kt,
                __nv_bfloat16* qt_b, __nv_bfloat16* kt_b, cudaStream_t stream) {
  const T* qq = static_cast<const T*>(q);
  const T* kk = static_cast<const T*>(k);
  const int vpr = s.d / (16 / (int)sizeof(T));
  const LandmarkKernel which = landmark_kernel(s);
  // Q's jobs come first (the job's tensor is its slowest index): without K,
  // only they are launched
  const long long tensors = k ? 2 : 1;
  if (which == LandmarkKernel::Small) {
    const int spw = 32 / vpr;
    const long long jobs = tensors * s.bh() * ((s.m64() + spw - 1) / spw);
    const unsigned grid = (unsigned)((jobs + 7) / 8);
    KernelScope ks_("landmarks_small", stream);
    landmarks_small<T><<<grid, 256, 0, stream>>>(qq, kk, qt, kt, qt_b, kt_b, s.bh(), s.n, s.d, s.m, s.m64(), s.dpad(),
                                                  s.lengths, s.H);
  } else if (which == LandmarkKernel::Vec) {
    const long long jobs = tensors * s.bh() * s.m64();
    KernelScope ks_("landmarks_vec", stream);
    landmarks_vec<T><<<(unsigned)((jobs + 7) / 8), 256, 0, stream>>>(
        qq, kk, qt, kt, qt_b, kt_b, s.bh(), s.n, s.d, s.m, s.m64(), s.dpad(), s.lengths, s.H);
  } else {
    KernelScope ks_("landmarks_simt", stream);
    landmarks_simt<T><<<dim3((s.m64() * s.dpad() + 255) / 256, (unsigned)s.bh()), 256, 0, stream>>>(
        qq, kk, qt, kt, qt_b, kt_b, s.n, s.d, s.m, s.m64(), s.dpad(), s.lengths, s.H);
  }
  return launch_status();
}

template <typename T>
int rows_t(const Shape& s, const float* qt, const void* k, const void* v, float* gp, float* gml,
           int splits, cudaStream_t stream) {
  const float scale = 1.0f / sqrtf((float)s.d);
  const int kps = (s.n + splits - 1) / splits;
  const size_t smem = sizeof(float) * (RW_ROWS * s.d + RW_KEYS * (s.d + 1) + RW_KEYS * s.d +
                                       RW_ROWS * RW_KEYS + RW_ROWS);
  KernelScope ks_("rows_simt", stream);
  rows_simt<T><<<dim3((s.m + RW_ROWS - 1) / RW_ROWS, splits, (unsigned)s.bh()), 128, smem, stream>>>(
      qt, static_cast<const T*>(k), static_cast<const T*>(v), gp, gml, s.n, s.d, s.m, splits, kps,
      scale, s.lengths, s.H);
  return launch_status();
}

template <typename T>
int tokens_t(const Shape& s, const void* q, const void* v, const float* kt, const float* w,
             const float* conv_w, void* out, cudaStream_t stream) {
  const float scale = 1.0f / sqrtf((float)s.d);
  const int rad = s.ks > 0 ? (s.ks - 1) / 2 : 0;
  const size_t smem = sizeof(float) * (TK_ROWS * s.d + TK_LM * (s.d + 1) + TK_LM * s.d +
                                       TK_ROWS * 33 + 2 * TK_ROWS + (TK_ROWS + 2 * rad) * s.d);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(tokens_simt<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return set_cuda_error(cudaGetLastError());
  KernelScope ks_("tokens_simt", stream);
  tokens_simt<T><<<dim3((s.n + TK_ROWS - 1) / TK_ROWS, (unsigned)s.bh()), 256, smem, stream>>>(
      static_cast<const T*>(q), static_cast<const T*>(v), kt, w, conv_w, static_cast<T*>(out), s.H,
      s.n, s.d, s.m, s.ks, scale);
  return launch_status();
}

}  // namespace

LandmarkKernel landmark_kernel(const Shape& s) {
  const int vpr = s.d / (16 / (s.dtype == NYS_FP32 ? 4 : 2));  // 16-byte vectors per row
  const long long nvec = (long long)s.seg_max() * vpr;
  if (32 % vpr == 0 && nvec <= 128) return LandmarkKernel::Small;
  if (32 % vpr == 0) return LandmarkKernel::Vec;
  return LandmarkKernel::Simt;
}

int launch_landmarks(const Shape& s, const void* q, const void* k, float* qt, float* kt,
                     __nv_bfloat16* qt_b, __nv_bfloat16* kt_b, cudaStream_t stream) {
  return s.dtype == NYS_FP32 ? landmarks_t<float>(s, q, k, qt, kt, qt_b, kt_b, stream)
                             : landmarks_t<__nv_bfloat16>(s, q, k, qt, kt, qt_b, kt_b, stream);
}

int launch_rows_simt(const Shape& s, const float* qt, const void* k, const void* v, float* gp,
                     float* gml, int splits, cudaStream_t stream) {
  return s.dtype == NYS_FP32 ? rows_t<float>(s, qt, k, v, gp, gml, splits, stream)
                             : rows_t<__nv_bfloat16>(s, qt, k, v, gp, gml, splits, stream);
}

int launch_pinv_simt(const Shape& s, const float* qt, const float* kt, const float* gp,
                     const float* gml, float* g, float* a, float* z, float* w, float* scratch,
                     __nv_bfloat16* wt_b, int splits, cudaStream_t stream) {
  const size_t dsmem = s.m <= kResM ? sizeof(float) * (5 * kResM * kResPitch + kCoefMax) : 0;
  if (dsmem > 48 * 1024 &&
      cudaFuncSetAttribute(pinv_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsmem) != cudaSuccess)
    return set_cuda_error(cudaGetLastError());
  KernelScope ks_("pinv_simt", stream);
  pinv_simt<<<(unsigned)s.bh(), 256, dsmem, stream>>>(qt, kt, gp, gml, g, a, z, w, scratch, wt_b, s.d,
                                                  s.m, splits, s.iters,
                                                  1.0f / sqrtf((float)s.d), s.m64(), s.dpad());
  return launch_status();
}

int launch_merge_g(const Shape& s, const float* gp, const float* gml, float* g, int splits,
                   cudaStream_t stream) {
  if (s.d % 4 != 0) return NYS_ERR_UNSUPPORTED;
  const int per_head4 = s.m * (s.d / 4);
  KernelScope ks_("merge_g", stream);
  const dim3 grid((unsigned)s.bh(), (unsigned)((per_head4 + 255) / 256));
  if (splits <= 2)
    merge_g<2><<<grid, 256, 0, stream>>>(gp, gml, g, s.m, s.d, splits);
  else if (splits <= 4)
    merge_g<4><<<grid, 256, 0, stream>>>(gp, gml, g, s.m, s.d, splits);
  else
    merge_g<8><<<grid, 256, 0, stream>>>(gp, gml, g, s.m, s.d, splits);
  return launch_status();
}

int launch_conv_mask(const Shape& s, const void* v, const float* conv_w, void* out,
                     cudaStream_t stream) {
  if (s.d > CV_THREADS) return NYS_ERR_UNSUPPORTED;
  return s.dtype == NYS_FP32 ? conv_mask_t<float>(s, v, conv_w, out, stream)
                             : conv_mask_t<__nv_bfloat16>(s, v, conv_w, out, stream);
}

int launch_tokens_simt(const Shape& s, const void* q, const void* v, const float* kt,
                       const float* w, const float* conv_w, void* out, cudaStream_t stream) {
  return s.dtype == NYS_FP32 ? tokens_t<float>(s, q, v, kt, w, conv_w, out, stream)
                             : tokens_t<__nv_bfloat16>(s, q, v, kt, w, conv_w, out, stream);
}

}  // namespace nys
