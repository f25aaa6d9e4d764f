// Landmark kernel, iterative pseudo-inverse and W = Z G on the tensor cores
// for 128 < m <= 256 landmarks ("Nyströmformer" review page, Proposed method,
// bullets 2, 3 and 5):
//   A_S = softmax(Q~ K~^T s)    scores in 3xTF32 (hi*hi + hi*lo + lo*hi)
//   Z_0 = A_S^T / (||A_S||_1 ||A_S||_inf)
//   iters x:  Z <- 1/4 Z (13I - 15X + 7X^2 - X^3),  X = A_S Z
//                                                  tcgen05 kind::f16 (fp16 operands)
//   W   = Z G                                      tcgen05 kind::tf32
// Each update is evaluated in three dependent levels of products instead of
// the four of the nested (Horner) form, since its cost is the latency of the
// chain, not the MMAs:
//   level 0:  X = A_S Z
//   level 1:  X X and Z X (one right factor, two left factors, side by side)
//   level 2:  Z' = 1/4 (13 Z - 15 Z X + Z X (7X - X^2))
// The update is the same polynomial in A_S and Z (X is recomputed from A_S
// and Z every update); only the grouping of its terms differs.
// An m x m fp32 matrix (256 KB at m = 256) does not fit one SM, so a
// cluster of four CTAs works on one head: CTA (r, c) owns rows
// [128 r, 128 r + 128) and columns [128 c, 128 c + 128) of every product
// (128 x 128 accumulators in TMEM; its block of Z stays in TMEM across the
// updates, and level 2 accumulates onto 13 Z - 15 Z X written there by the
// level-1 epilogue). Product operands live in global memory (L2 resident) as
// one fp16 row-major copy each (Z, X, Z X, 7X - X^2): a left factor is read
// K-major from it, a right factor MN-major (64-row K-chunks of the same
// rows), so each product block is written once. TMA streams 64-wide
// K-chunks into a two-stage shared-memory ring, and level 1's two products
// share one stream of their right factor. Each epilogue writes the next
// level's operands, then the cluster synchronises before they are read.
// Why fp16 operands: the chain's time goes to moving operands (an SM writes
// to L2 at about 32 bytes per clock, and a tf32 product reads shared memory
// as fast as TMA fills it), and fp16 halves those bytes. Its 11-bit
// significand (rounded to nearest) is finer than tf32's truncated one, and
// its range holds the iterates: Z_k = A_S^T q(A_S A_S^T) shares A_S's
// singular vectors, and with x = sigma z per singular value sigma the update
// maps x in [0, 1] into [0, 1] and grows it at most 13/4-fold, so
// z_k <= min(1/sigma, (13/4)^k alpha sigma) <= (13/4)^(k/2) (alpha <= 1):
// ||Z||_2 < 112 after at most 8 updates, far below fp16's 65504. Entries
// below fp16's normal range carry absolute errors near 6e-8. Accumulation stays fp32 (TMEM), Z itself stays fp32 in
// TMEM across the updates, and W = Z G runs in tf32 from the fp32 Z.
//
// Warps 0-3: epilogue / softmax (thread = row, TMEM lane = row); warp 4:
// TMA producer; warp 5: TMEM owner and tcgen05 issuer. Every mbarrier wait
// is bounded; after a timeout the CTA skips its remaining work but still
// takes part in every cluster barrier, so its peers never wait on it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>

#include "nys_internal.h"
#include "nys_sm100.h"
#include "nys_tma_host.h"

namespace nys {
namespace {

using namespace sm100;

// Loads: the fp16 operand matrices [B*H][m][mp] as left factors (A_S, Z, X,
// Z X: boxes of 128 rows x 64 columns) and as right factors (Z, X, 7X - X^2:
// boxes of 64 rows x 64 columns, read MN-major), then the fp32 maps of
// W = Z G: G^T [B*H][d][m] and Z [B*H][m][m]
enum MapIdx {
  MAP_A = 0, MAP_Z = 1, MAP_XR = 2, MAP_ZX = 3, MAP_BZ = 4, MAP_BX = 5, MAP_GT = 6, MAP_Z32 = 7,
  MAP_BY = 8, kLoadMaps = 9
};

// Stores: row-major 32 x 64 boxes (SWIZZLE_128B) of A_S, Z, X, Z X and
// 7X - X^2 (fp16); then A_S fp32 in 32 x 32 boxes (SWIZZLE_128B) and Z_0
// fp16 from its transposed staging, 32 x 32 boxes (SWIZZLE_64B)
enum StoreIdx { ST_Y = 4, ST_AS32 = 6, ST_Z16T = 7, kStoreMaps = 8 };

struct BigPinvMaps {
  CUtensorMap m[kLoadMaps];
  CUtensorMap st[kStoreMaps];
};

struct BigPinvParams {
  const float* qt;     // [B*H][m][d] fp32
  const float* kt;     // [B*H][m][d] fp32
  const float* gpart;  // [B*H][splits][m][d]
  const float* gml;    // [B*H][splits][m][2]
  float* g;            // [B*H][m][d]
  float* a_s;          // [B*H][m][m]   A_S (fp32)
  float* z;            // [B*H][m][m]   Z_0, then the last update's Z (fp32)
  __half* a16;         // [B*H][m][mp]  A_S                       (fp16 operands,
  __half* z16;         // [B*H][m][mp]  Z (row-major)              row pitch mp)
  __half* xr16;        // [B*H][m][mp]  X = A_S Z (row-major)
  __half* zx16;        // [B*H][m][mp]  Z X (row-major)
  __half* y16;         // [B*H][m][mp]  7X - X^2 (row-major)
  float* gt;           // [B*H][d][m]   G^T
  float* w;            // [B*H][m][d]
  __nv_bfloat16* wt;   // [B*H][dpad][m64] zero padded
  int* status;
  int m, mp, d, dpad, m64, splits, iters;
  float scale;
};

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kThreads = 192;
// The operand ring: two stages of two K-chunks each. A stage holds, per
// chunk, the 128 x 64 fp16 boxes of up to two left factors and the right
// factor's 64 K-rows x 128 columns as two 64 x 64 boxes (W: one <= 128 x 32
// fp32 box, K-major), behind one mbarrier: an mbarrier round trip costs
// about as much as streaming 16 KB, so stages are made large, not many.
constexpr int kStages = 2;
constexpr uint32_t kStageBytes = 98304;
constexpr uint32_t kOffA2 = 32768, kOffB = 65536;  // A1 chunks at 0 and 16 KB
constexpr uint32_t kTmemCols = 512;
// TMEM column bases of the four 128-column accumulators
constexpr uint32_t kR0 = 0;    // scores / A_S, then this CTA's block of Z
constexpr uint32_t kR1 = 128;  // X (level 0), W
constexpr uint32_t kR2 = 256;  // X X
constexpr uint32_t kR3 = 384;  // Z X

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// generic-proxy global writes <-> async-proxy (TMA) reads
__device__ __forceinline__ void fence_proxy_async_all() {
  asm volatile("fence.proxy.async;" ::: "memory");
}

// read a float of CTA `rank`'s copy of the shared variable at `p`
__device__ __forceinline__ float ld_peer(const float* p, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

__device__ __forceinline__ float tf32_hi(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kThreads, 1)
    pinv_big(const __grid_constant__ BigPinvMaps maps, const BigPinvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  __shared__ uint64_t full[kStages], empty[kStages], done, fin;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float rmax_sh[128], rsum_sh[128], rs_sh[128], cs_sh[128], red[8];
  volatile int* abort_flag = &abort_sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int r = (int)(rank >> 1), c = (int)(rank & 1);
  const int bh = blockIdx.x >> 2;
  const int m = p.m, d = p.d;
  const int gi = 128 * r + tid;  // this worker's row (warps 0-3)
  const bool worker = warp < 4;
  const bool rv = worker && gi < m;
  const size_t mm = (size_t)m * m;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    mbar_init(&fin, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(&tmem_base_sh, kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
  cluster_sync_all();  // every CTA of the cluster is running before any DSMEM access

  uint32_t ph_done = 0;
  auto wait_done = [&]() -> bool {
    bool ok = mbar_wait(&done, ph_done, abort_flag, kWaitNs);
    if (!ok && !*abort_flag) {
      *abort_flag = 1;
      atomicExch(p.status, (int)NYS_ERR_TIMEOUT);
    }
    ph_done ^= 1;
    tc_fence_after_sync();
    return ok;
  };

  // ---- 1) G = merge of the key-split partials: rows of this row block,
  // columns [c d/2, (c+1) d/2). G -> g (row-major), G^T -> gt. One pass
  // over the splits per 8-column chunk, four splits at a time with all
  // their loads in flight; a running (max, denominator) rescales the
  // accumulated row as in an online softmax, and an empty partial (max =
  // -inf, rows never written) contributes nothing. Only W = Z G reads G, so
  // the chunks are merged one per update level, while the workers would
  // otherwise wait for the level's products.
  constexpr int kMw = 8;              // columns per merge chunk
  const int n_merge = (d >> 1) / kMw;  // chunks of this CTA's columns of G
  auto merge_chunk = [&](int chunk) {
    if (!rv) return;
    const int hw = d >> 1;
    float* grow = p.g + ((size_t)bh * m + gi) * d;
    float* gtb = p.gt + (size_t)bh * d * m;
    const float2* ml_base = reinterpret_cast<const float2*>(p.gml) + (size_t)bh * p.splits * m + gi;
    const float* gp_base = p.gpart + ((size_t)bh * p.splits * m + gi) * d;
    {
      const int j0 = c * hw + kMw * chunk;
      float acc[kMw];
#pragma unroll
      for (int e = 0; e < kMw; ++e) acc[e] = 0.f;
      float gm = -INFINITY, den = 0.f;
      for (int sp = 0; sp < p.splits; sp += 4) {
        float2 ml[4];
        float4 v[4][kMw / 4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int spk = sp + k < p.splits ? sp + k : sp;
          ml[k] = __ldg(ml_base + (size_t)spk * m);
          const float4* src = reinterpret_cast<const float4*>(gp_base + (size_t)spk * m * d + j0);
#pragma unroll
          for (int e = 0; e < kMw / 4; ++e) v[k][e] = __ldg(src + e);
        }
        bool ok[4];
        float cm = gm;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ok[k] = sp + k < p.splits && ml[k].x != -INFINITY;
          if (ok[k]) cm = fmaxf(cm, ml[k].x);
        }
        if (cm == -INFINITY) continue;  // nothing yet
        const float r = gm == -INFINITY ? 0.f : expf(gm - cm);
        float f[4];
        den *= r;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          f[k] = ok[k] ? expf(ml[k].x - cm) : 0.f;
          den += ok[k] ? ml[k].y * f[k] : 0.f;
        }
        gm = cm;
#pragma unroll
        for (int e = 0; e < kMw; ++e) acc[e] *= r;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (ok[k]) {
#pragma unroll
            for (int e = 0; e < kMw / 4; ++e) {
              acc[4 * e] = fmaf(v[k][e].x, f[k], acc[4 * e]);
              acc[4 * e + 1] = fmaf(v[k][e].y, f[k], acc[4 * e + 1]);
              acc[4 * e + 2] = fmaf(v[k][e].z, f[k], acc[4 * e + 2]);
              acc[4 * e + 3] = fmaf(v[k][e].w, f[k], acc[4 * e + 3]);
            }
          }
      }
      const float inv = 1.f / den;
#pragma unroll
      for (int e = 0; e < kMw; ++e) acc[e] *= inv;
      float4* go = reinterpret_cast<float4*>(grow + j0);
#pragma unroll
      for (int e = 0; e < kMw / 4; ++e) go[e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
#pragma unroll
      for (int e = 0; e < kMw; ++e) gtb[(size_t)(j0 + e) * m + gi] = acc[e];
    }
  };
  if (p.iters == 0)
    for (int k = 0; k < n_merge; ++k) merge_chunk(k);

  // ---- 2) scores S = Q~ K~^T (rows of block r, columns of block c) in
  // 3xTF32. Per pass, up to two 32-column chunks of d; chunk slot layout:
  // Q hi | Q lo | K hi | K lo, 16 KB each.
  {
    const int gk = 128 * c + tid;  // K~ row = score column handled by this thread
    const bool qv_ok = rv, kv_ok = worker && gk < m;
    const float* qrow = p.qt + ((size_t)bh * m + (qv_ok ? gi : 0)) * d;
    const float* krow = p.kt + ((size_t)bh * m + (kv_ok ? gk : 0)) * d;
    const int nchunk = d >> 5;
    for (int pass = 0; pass * 2 < nchunk; ++pass) {
      const int ch0 = pass * 2, nch = min(2, nchunk - ch0);
      if (worker) {
        for (int cc = 0; cc < nch; ++cc) {
          uint8_t* slot = sm + cc * 65536;
          const int col0 = (ch0 + cc) * 32;
          // all 16 loads in flight before the first shared-memory store
          float4 q4[8], k4[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            q4[e] = qv_ok ? __ldg(reinterpret_cast<const float4*>(qrow + col0) + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            k4[e] = kv_ok ? __ldg(reinterpret_cast<const float4*>(krow + col0) + e) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 qh = make_float4(tf32_hi(q4[e].x), tf32_hi(q4[e].y), tf32_hi(q4[e].z), tf32_hi(q4[e].w));
            const float4 kh = make_float4(tf32_hi(k4[e].x), tf32_hi(k4[e].y), tf32_hi(k4[e].z), tf32_hi(k4[e].w));
            const uint32_t off = sw128_offset(tid, e * 16);
            *reinterpret_cast<float4*>(slot + off) = qh;
            *reinterpret_cast<float4*>(slot + 16384 + off) =
                make_float4(q4[e].x - qh.x, q4[e].y - qh.y, q4[e].z - qh.z, q4[e].w - qh.w);
            *reinterpret_cast<float4*>(slot + 32768 + off) = kh;
            *reinterpret_cast<float4*>(slot + 49152 + off) =
                make_float4(k4[e].x - kh.x, k4[e].y - kh.y, k4[e].z - kh.z, k4[e].w - kh.w);
          }
        }
        fence_async_smem();
      }
      tc_fence_before_sync();
      __syncthreads();
      if (warp == 5 && lane == 0 && !*abort_flag) {
        tc_fence_after_sync();
        const uint32_t id = idesc_tf32(128, 128);
        for (int cc = 0; cc < nch; ++cc) {
          const uint64_t qh = smem_desc(smem_u32(sm + cc * 65536), 16, 1024, SW_128B);
          const uint64_t ql = qh + (16384 >> 4), kh = qh + (32768 >> 4), kl = qh + (49152 >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t first = (pass == 0 && cc == 0 && kk == 0) ? 0u : 1u;
            mma_tf32(tmem, qh + kk * 2, kh + kk * 2, id, first);
            mma_tf32(tmem, qh + kk * 2, kl + kk * 2, id, 1u);
            mma_tf32(tmem, ql + kk * 2, kh + kk * 2, id, 1u);
          }
        }
        mma_commit(&done);
      }
      if (worker) wait_done();
      tc_fence_before_sync();
      __syncthreads();
    }
  }

  // ---- 3) softmax across the column pair (c = 0, 1) of this row block
  float a_row_sum = 0.f;  // this CTA's part of the row sum of A_S
  if (worker) {
    float mx = -INFINITY;
    if (!*abort_flag)
      for (int j0 = 0; j0 < 128; j0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lo + j0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (128 * c + j0 + e < m) mx = fmaxf(mx, __uint_as_float(v[e]));
      }
    rmax_sh[tid] = mx;
  }
  cluster_sync_all();
  float part = 0.f;
  if (worker && !*abort_flag) {
    const float rmax = fmaxf(rmax_sh[tid], ld_peer(&rmax_sh[tid], rank ^ 1u));
    for (int j0 = 0; j0 < 128; j0 += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lo + j0, v);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x = (rv && 128 * c + j0 + e < m) ? expf((__uint_as_float(v[e]) - rmax) * p.scale) : 0.f;
        part += x;
        v[e] = __float_as_uint(x);
      }
      tmem_st32(tmem + lo + j0, v);
    }
    tmem_st_wait();
  }
  if (worker) rsum_sh[tid] = part;
  cluster_sync_all();
  // The normalised block is staged in shared memory, in fp32 as four
  // SWIZZLE_128B boxes [128 rows x 32 columns] (also read back for the
  // column sums) and in fp16 as two [128 rows x 64 columns] boxes; each warp
  // stores its 32 rows of both by TMA (clipped at m).
  uint8_t* as_stage = sm;
  uint8_t* a16_stage = sm + 65536;
  if (worker && !*abort_flag) {
    const float own = rsum_sh[tid], peer = ld_peer(&rsum_sh[tid], rank ^ 1u);
    const float sum = c == 0 ? own + peer : peer + own;  // same order in both CTAs
    const float inv = rv ? 1.f / sum : 0.f;
    for (int j0 = 0; j0 < 128; j0 += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lo + j0, v);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float x = __uint_as_float(v[e]) * inv;
        v[e] = __float_as_uint(x);
        a_row_sum += fabsf(x);
      }
      tmem_st32(tmem + lo + j0, v);
      uint8_t* box = as_stage + (j0 >> 5) * 16384;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(box + sw128_offset(tid, q * 16)) =
            make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const __half2 h2 = __floats2half2_rn(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
        pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      uint8_t* hbox = a16_stage + (j0 >> 6) * 16384;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(hbox + sw128_offset(tid, (j0 & 63) * 2 + q * 16)) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
    tmem_st_wait();
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      for (int b = 0; b < 4; ++b)
        tma_store_3d(&maps.st[ST_AS32], as_stage + b * 16384 + warp * 4096, 128 * c + 32 * b, 128 * r + 32 * warp, bh);
      for (int b = 0; b < 2; ++b)
        tma_store_3d(&maps.st[MAP_A], a16_stage + b * 16384 + warp * 4096, 128 * c + 64 * b, 128 * r + 32 * warp, bh);
      bulk_commit();
    }
  }
  __syncthreads();
  if (worker) {
    // this CTA's part of column tid's abs-sum (four independent partials)
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
    if (!*abort_flag) {
      const uint8_t* cbox = as_stage + (tid >> 5) * 16384;
      for (int i = 0; i < 128; i += 4) {
#pragma unroll
        for (int t = 0; t < 4; ++t)
          s4[t] += fabsf(*reinterpret_cast<const float*>(cbox + sw128_offset(i + t, (tid & 31) * 4)));
      }
    }
    cs_sh[tid] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
    rs_sh[tid] = a_row_sum;
  }
  cluster_sync_all();
  // ||A_S||_1 and ||A_S||_inf from the four CTAs' partials, combined in a
  // fixed order so that every CTA of the cluster gets the same alpha
  if (worker) {
    float cmax = 0.f, rmaxs = 0.f;
    for (int b = 0; b < 2; ++b) {
      const float col = ld_peer(&cs_sh[tid], (uint32_t)b) + ld_peer(&cs_sh[tid], (uint32_t)(2 + b));
      if (128 * b + tid < m) cmax = fmaxf(cmax, col);
      const float row = ld_peer(&rs_sh[tid], (uint32_t)(2 * b)) + ld_peer(&rs_sh[tid], (uint32_t)(2 * b + 1));
      if (128 * b + tid < m) rmaxs = fmaxf(rmaxs, row);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      rmaxs = fmaxf(rmaxs, __shfl_xor_sync(0xffffffffu, rmaxs, o));
    }
    if (lane == 0) {
      red[warp] = cmax;
      red[4 + warp] = rmaxs;
    }
  }
  __syncthreads();
  // Z_0 = alpha A_S^T row-major: the transposed A_S block, fp32 by plain
  // coalesced stores and fp16 by TMA
  if (worker && !*abort_flag) {
    const float n1 = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const float ninf = fmaxf(fmaxf(red[4], red[5]), fmaxf(red[6], red[7]));
    const float alpha = 1.f / (n1 * ninf);
    float* z = p.z + bh * mm;
    // fp16 staging of the transpose, SWIZZLE_64B tiles of 32 x 32 (32 block
    // columns per tile)
    uint8_t* z16_stage = sm + 131072 + warp * 8192;
    for (int j0 = 0; j0 < 128; j0 += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lo + kR0 + j0, v);
      tmem_ld_wait();
      if (rv) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int gj = 128 * c + j0 + e;
          if (gj < m) z[(size_t)gj * m + gi] = alpha * __uint_as_float(v[e]);
        }
      }
      uint8_t* tt = z16_stage + (j0 >> 5) * 2048;
#pragma unroll
      for (int e = 0; e < 32; ++e)
        *reinterpret_cast<__half*>(tt + sw64_offset(e, lane * 2)) = __float2half_rn(alpha * __uint_as_float(v[e]));
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      for (int k = 0; k < 4; ++k)
        tma_store_3d(&maps.st[ST_Z16T], z16_stage + k * 2048, 128 * r + 32 * warp, 128 * c + 32 * k, bh);
      bulk_commit();
    }
  }
  // every store of the prologue has landed (and read its staging) before
  // the products start
  if (worker && lane == 0) bulk_wait0();
  __syncwarp();
  cluster_sync_all();
  // this CTA's block of Z_0 into TMEM (zero beyond m), where it stays across
  // the updates
  if (worker && !*abort_flag) {
    const float* zrow = p.z + bh * mm + (size_t)(rv ? gi : 0) * m;
    for (int j0 = 0; j0 < 128; j0 += 32) {
      uint32_t v[32];
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const int gj = 128 * c + j0 + e;
        const float4 q = (rv && gj < m) ? *reinterpret_cast<const float4*>(zrow + gj)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
        v[e] = __float_as_uint(q.x);
        v[e + 1] = __float_as_uint(q.y);
        v[e + 2] = __float_as_uint(q.z);
        v[e + 3] = __float_as_uint(q.w);
      }
      tmem_st32(tmem + lo + kR0 + j0, v);
    }
    tmem_st_wait();
  }
  tc_fence_before_sync();
  fence_proxy_async_all();
  cluster_sync_all();
  fence_proxy_async_all();
  tc_fence_after_sync();

  // ---- 4) the products: three levels per update, then W = Z G. Right
  // factors: Z (level 0), X (level 1), 7X - X^2 (level 2), G^T (W).
  const int nprod = 3 * p.iters + 1;
  const int hw = d >> 1;
  uint32_t kg_prod = 0, kg_mma = 0;   // ring positions of the producer / issuer
  uint32_t n_full[kStages] = {};      // loads issued per stage (producer)
  int it = 0, lv = 0;                 // update and level of product pi
  for (int pi = 0; pi < nprod; ++pi) {
    const bool is_w = pi == nprod - 1;
    // Update products (fp16): K-chunks of 64, every operand streamed (the
    // right factor MN-major: 64 of its rows, as two boxes of 64 columns);
    // level 1 runs its two products over one stream of the shared right
    // factor. W (tf32): K-chunks of 32 columns; its left factor Z is read
    // from TMEM (R0) for the K-block this CTA holds and streamed for the
    // other.
    const int amap1 = is_w ? MAP_Z32 : (lv == 0 ? MAP_A : (lv == 1 ? MAP_XR : MAP_ZX));
    const int bmap = is_w ? MAP_GT : (lv == 0 ? MAP_BZ : (lv == 1 ? MAP_BX : MAP_BY));
    const bool two = !is_w && lv == 1;
    const int kw = is_w ? 32 : 64;  // K-chunk width (elements)
    const int b_row0 = c * hw;  // W: this CTA's rows of G^T
    const int n_cols = is_w ? hw : 128;
    const uint32_t b_bytes = (uint32_t)n_cols * 128u;
    // stage j of a product holds K-chunks 2j and 2j + 1 (a chunk past m is
    // read as zeros and adds nothing)
    const int nst = ((m + kw - 1) / kw + 1) >> 1;
    if (warp == 4) {
      if (lane == 0 && !*abort_flag) {
        for (int j = 0; j < nst; ++j, ++kg_prod) {
          const int st = (int)(kg_prod % kStages);
          if (kg_prod >= (uint32_t)kStages &&
              !mbar_wait(&empty[st], ((kg_prod / kStages) - 1) & 1, abort_flag, kWaitNs)) {
            if (!*abort_flag) {
              *abort_flag = 1;
              atomicExch(p.status, (int)NYS_ERR_TIMEOUT);
            }
            break;
          }
          // W: the 32-column chunks 2j, 2j + 1 lie in K-block (2j) / 4
          const bool from_tmem = is_w && ((2 * j) >> 2) == c;
          uint8_t* sa = sm + st * kStageBytes;
          mbar_arrive_expect_tx(&full[st], 2u * (b_bytes + (from_tmem ? 0u : (two ? 32768u : 16384u))));
          ++n_full[st];
          for (int q = 0; q < 2; ++q) {
            const int kx = kw * (2 * j + q);
            if (!from_tmem) {
              tma_load_3d(sa + q * 16384, &maps.m[amap1], &full[st], kx, 128 * r, bh);
              if (two) tma_load_3d(sa + kOffA2 + q * 16384, &maps.m[MAP_Z], &full[st], kx, 128 * r, bh);
            }
            if (is_w) {
              tma_load_3d(sa + kOffB + q * 16384, &maps.m[bmap], &full[st], kx, b_row0, bh);
            } else {
              tma_load_3d(sa + kOffB + q * 16384, &maps.m[bmap], &full[st], 128 * c, kx, bh);
              tma_load_3d(sa + kOffB + q * 16384 + 8192, &maps.m[bmap], &full[st], 128 * c + 64, kx, bh);
            }
          }
        }
      }
      __syncwarp();
    } else if (warp == 5) {
      if (lane == 0 && !*abort_flag) {
        const uint32_t id = is_w ? idesc_tf32(128, n_cols) : idesc_f16(128, n_cols, true);
        // accumulators: X (level 0) and W in R1; X X in R2 and Z X in R3
        // (level 1); level 2 accumulates onto 13 Z - 15 Z X in R0
        const uint32_t d1 = (is_w || lv == 0) ? kR1 : (lv == 1 ? kR2 : kR0);
        bool ok = true;
        for (int j = 0; j < nst; ++j, ++kg_mma) {
          const int st = (int)(kg_mma % kStages);
          if (!mbar_wait(&full[st], (kg_mma / kStages) & 1, abort_flag, kWaitNs)) {
            if (!*abort_flag) {
              *abort_flag = 1;
              atomicExch(p.status, (int)NYS_ERR_TIMEOUT);
            }
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const bool from_tmem = is_w && ((2 * j) >> 2) == c;
          const uint32_t sb = smem_u32(sm + st * kStageBytes);
          // one accumulator at a time: switching accumulators between
          // consecutive MMAs halves their throughput
          for (int pr = 0; pr < (two ? 2 : 1); ++pr) {
            const uint32_t dacc = pr ? kR3 : d1;
            const uint32_t aoff = pr ? kOffA2 : 0u;
            const bool fresh = j == 0 && !(lv == 2 && !is_w);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const uint32_t ta = tmem + kR0 + (uint32_t)(((2 * j + q) & 3) * 32);
              const uint64_t a0 = smem_desc(sb + aoff + q * 16384, 16, 1024, SW_128B);
              // W: K-major, K-steps of 8 (32 bytes); else MN-major (column
              // halves 8 KB apart), K-steps of 16 rows (2 KB)
              const uint64_t b0 = is_w ? smem_desc(sb + kOffB + q * 16384, 16, 1024, SW_128B)
                                       : smem_desc(sb + kOffB + q * 16384, 8192, 1024, SW_128B);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acc = (fresh && q == 0 && kk == 0) ? 0u : 1u;
                if (!is_w)
                  mma_bf16(tmem + dacc, a0 + kk * 2, b0 + kk * 128, id, acc);  // kind::f16, fp16 by idesc
                else if (from_tmem)
                  mma_tf32_tA(tmem + dacc, ta + kk * 8, b0 + kk * 2, id, acc);
                else
                  mma_tf32(tmem + dacc, a0 + kk * 2, b0 + kk * 2, id, acc);
              }
            }
          }
          mma_commit(&empty[st]);
        }
        if (ok) mma_commit(&done);
      }
      __syncwarp();
    } else {
      // epilogue: thread = row gi of the product block. Before an update
      // level's products are done, merge the next chunk of G (the last
      // update level merges whatever is left).
      if (!is_w && !*abort_flag) {
        if (pi < nprod - 2) {
          if (pi < n_merge) merge_chunk(pi);
        } else if (pi == nprod - 2) {
          for (int k = pi; k < n_merge; ++k) merge_chunk(k);
        }
      }
      const bool ok_epi = __all_sync(0xffffffffu, wait_done());  // warp-uniform: TMEM loads are warp-wide
      if (is_w && ok_epi) {
        float* wrow = p.w + ((size_t)bh * m + (rv ? gi : 0)) * d + c * hw;
        __nv_bfloat16* wt = p.wt + (size_t)bh * p.dpad * p.m64;
        for (int j0 = 0; j0 < hw; j0 += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lo + kR1 + j0, v);
          tmem_ld_wait();
          if (rv) {
#pragma unroll
            for (int e = 0; e < 16; e += 4)
              *reinterpret_cast<float4*>(wrow + j0 + e) =
                  make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                              __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
          }
          if (gi < p.m64) {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              wt[(size_t)(c * hw + j0 + e) * p.m64 + gi] = __float2bfloat16_rn(rv ? __uint_as_float(v[e]) : 0.f);
          }
        }
        if (c == 1 && gi < p.m64)
          for (int j = d; j < p.dpad; ++j) wt[(size_t)j * p.m64 + gi] = __float2bfloat16_rn(0.f);
      } else if (!is_w) {
        // level 0: X (R1)            -> xr
        // level 1: Z X (R3)          -> zx, 7X - X^2 -> y,
        //          R0 <- 13 Z - 15 Z X
        // level 2: Z' = R0 / 4 -> R0, z; after the last update also the
        //          fp32 Z (for W and the stage export)
        // The blocks are rounded to fp16 and staged, row-major, in the (now
        // idle) operand ring as two SWIZZLE_128B boxes of [128 rows x 64
        // columns] each; every 64 columns each warp stores its 32 rows of
        // the box while the next columns are staged. The stores clip what
        // lies beyond m.
        const int rm_map = lv == 0 ? MAP_XR : (lv == 1 ? MAP_ZX : MAP_Z);
        const bool last_z = lv == 2 && it == p.iters - 1;
        uint8_t* rm_stage = sm;          // box b: block columns [64 b, 64 b + 64)
        uint8_t* y_stage = sm + 32768;   // level 1: 7X - X^2, the same way
        float* z32 = p.z + ((size_t)bh * m + (rv ? gi : 0)) * m + 128 * c;
        const bool store = ok_epi && !*abort_flag;
        auto stage16 = [&](uint8_t* stage, const float* x, int jc) {
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const __half2 h2 = __floats2half2_rn(x[2 * e], x[2 * e + 1]);
            pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          uint8_t* box = stage + (jc >> 6) * 16384;
          const uint32_t byte0 = (uint32_t)(jc & 63) * 2u;
          *reinterpret_cast<uint4*>(box + sw128_offset(tid, byte0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(box + sw128_offset(tid, byte0 + 16)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        };
        for (int j0 = 0; ok_epi && j0 < 128; j0 += 32) {
          for (int h = 0; h < 32; h += 16) {
            const int jc = j0 + h;
            float rmv[16];
            if (lv == 0) {
              uint32_t v[16];
              tmem_ld16(tmem + lo + kR1 + jc, v);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) rmv[e] = __uint_as_float(v[e]);
            } else if (lv == 1) {
              uint32_t vx[16], vx2[16], vzx[16], vz[16];
              tmem_ld16(tmem + lo + kR1 + jc, vx);
              tmem_ld16(tmem + lo + kR2 + jc, vx2);
              tmem_ld16(tmem + lo + kR3 + jc, vzx);
              tmem_ld16(tmem + lo + kR0 + jc, vz);
              tmem_ld_wait();
              float yv[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float zx = __uint_as_float(vzx[e]);
                rmv[e] = zx;
                yv[e] = fmaf(7.f, __uint_as_float(vx[e]), -__uint_as_float(vx2[e]));
                vz[e] = __float_as_uint(fmaf(13.f, __uint_as_float(vz[e]), -15.f * zx));
              }
              tmem_st16(tmem + lo + kR0 + jc, vz);
              stage16(y_stage, yv, jc);
            } else {
              uint32_t v[16];
              tmem_ld16(tmem + lo + kR0 + jc, v);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                rmv[e] = 0.25f * __uint_as_float(v[e]);
                v[e] = __float_as_uint(rmv[e]);
              }
              tmem_st16(tmem + lo + kR0 + jc, v);
              if (last_z && rv) {
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                  if (128 * c + jc + e < m)
                    *reinterpret_cast<float4*>(z32 + jc + e) = make_float4(rmv[e], rmv[e + 1], rmv[e + 2], rmv[e + 3]);
              }
            }
            stage16(rm_stage, rmv, jc);
          }
          // every 64 columns: this warp's rows of the box leave while the
          // next columns are staged
          if ((j0 & 63) == 32) {
            fence_async_smem();
            __syncwarp();
            if (lane == 0 && store) {
              const int bx = j0 >> 6;
              tma_store_3d(&maps.st[rm_map], rm_stage + bx * 16384 + warp * 4096, 128 * c + 64 * bx,
                           128 * r + 32 * warp, bh);
              if (lv == 1)
                tma_store_3d(&maps.st[ST_Y], y_stage + bx * 16384 + warp * 4096, 128 * c + 64 * bx,
                             128 * r + 32 * warp, bh);
              bulk_commit();
            }
          }
        }
        if (lv != 0) tmem_st_wait();
        if (lane == 0 && store) bulk_wait0();  // written before the cluster barrier publishes them
        __syncwarp();
      }
    }
    tc_fence_before_sync();
    fence_proxy_async_all();
    cluster_sync_all();
    fence_proxy_async_all();
    tc_fence_after_sync();
    if (++lv == 3) {
      lv = 0;
      ++it;
    }
  }

  // ---- teardown: no copy or MMA of this CTA may still be in flight
  if (warp == 4 && lane == 0 && *abort_flag) {
    for (int s = 0; s < kStages; ++s)
      if (n_full[s]) mbar_wait(&full[s], (n_full[s] - 1) & 1, nullptr, kWaitNs);
  }
  if (warp == 5 && lane == 0) {
    mma_commit(&fin);
    mbar_wait(&fin, 0, nullptr, kWaitNs);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
  cluster_sync_all();  // peers may still read this CTA's shared memory until here
}

constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + 1024;

}  // namespace

bool pinv_big_supported(const Shape& s) {
  return s.dtype == NYS_BF16 && s.m > 128 && s.m <= 256 && s.m % 4 == 0 && s.d % 32 == 0 &&
         s.d <= 128 && s.iters <= kTf32MaxIters;
}

int launch_pinv_big(const Shape& s, const float* qt, const float* kt, const float* gpart,
                    const float* gml, float* g, float* a_s, float* z, float* scratch, float* w,
                    void* wt_bf16, int splits, int* status, cudaStream_t stream) {
  if (!pinv_big_supported(s)) return NYS_ERR_UNSUPPORTED;
  const size_t BH = (size_t)s.bh(), mm = (size_t)s.m * s.m;
  BigPinvParams p{};
  p.qt = qt;
  p.kt = kt;
  p.gpart = gpart;
  p.gml = gml;
  p.g = g;
  p.a_s = a_s;
  // scratch holds, for the whole batch, the five fp16 operand matrices
  // [B*H][m][mp] (A_S, Z, X, Z X, 7X - X^2; mp = m rounded up to 8, so that
  // every row starts on a 16-byte boundary) in its first 4 m^2 floats, then
  // G^T. Z (fp32) lives in `z` (stage export).
  const int mp = (s.m + 7) & ~7;
  const size_t hm = BH * (size_t)s.m * mp;  // halves per fp16 matrix
  __half* h16 = reinterpret_cast<__half*>(scratch);
  p.z = z;
  p.a16 = h16;
  p.z16 = h16 + hm;
  p.xr16 = h16 + 2 * hm;
  p.zx16 = h16 + 3 * hm;
  p.y16 = h16 + 4 * hm;
  p.gt = scratch + 4 * BH * mm;
  p.w = w;
  p.wt = static_cast<__nv_bfloat16*>(wt_bf16);
  p.status = status;
  p.m = s.m;
  p.mp = mp;
  p.d = s.d;
  p.dpad = s.dpad();
  p.m64 = s.m64();
  p.splits = splits;
  p.iters = s.iters;
  p.scale = 1.0f / sqrtf((float)s.d);

  BigPinvMaps maps;
  memset(&maps, 0, sizeof(maps));
  {
    // left factors (128 x 64 boxes) and row-major stores (32 x 64) of A_S, Z,
    // X, Z X and 7X - X^2; right factors (64 x 64 boxes) of Z, X, 7X - X^2
    const uint64_t dims[3] = {(uint64_t)s.m, (uint64_t)s.m, BH};
    const uint64_t strides[2] = {(uint64_t)mp * 2, (uint64_t)s.m * mp * 2};
    const uint32_t box[3] = {64, 128, 1}, bbox[3] = {64, 64, 1}, sbox[3] = {64, 32, 1};
    const __half* left[4] = {p.a16, p.z16, p.xr16, p.zx16};
    for (int i = 0; i < 4; ++i)
      if (!make_tensor_map(&maps.m[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, left[i], dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B))
        return tensor_map_error(__FILE__, __LINE__);
    const __half* rows[5] = {p.a16, p.z16, p.xr16, p.zx16, p.y16};  // store index = position
    for (int i = 0; i < 5; ++i)
      if (!make_tensor_map(&maps.st[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, rows[i], dims, strides, sbox,
                           CU_TENSOR_MAP_SWIZZLE_128B))
        return tensor_map_error(__FILE__, __LINE__);
    const int bidx[3] = {MAP_BZ, MAP_BX, MAP_BY};
    const __half* right[3] = {p.z16, p.xr16, p.y16};
    for (int i = 0; i < 3; ++i)
      if (!make_tensor_map(&maps.m[bidx[i]], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, right[i], dims, strides,
                           bbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return tensor_map_error(__FILE__, __LINE__);
  }
  {
    const uint64_t dims[3] = {(uint64_t)s.m, (uint64_t)s.d, BH};
    const uint64_t strides[2] = {(uint64_t)s.m * 4, (uint64_t)s.d * s.m * 4};
    const uint32_t box[3] = {32, (uint32_t)(s.d / 2), 1};
    if (!make_tensor_map(&maps.m[MAP_GT], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.gt, dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
  }
  {
    const uint64_t dims[3] = {(uint64_t)s.m, (uint64_t)s.m, BH};
    const uint64_t strides[2] = {(uint64_t)s.m * 4, (uint64_t)mm * 4};
    const uint32_t box[3] = {32, 128, 1}, sbox[3] = {32, 32, 1};
    if (!make_tensor_map(&maps.m[MAP_Z32], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.z, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&maps.st[ST_AS32], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.a_s, dims, strides, sbox,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
    const uint64_t hstrides[2] = {(uint64_t)mp * 2, (uint64_t)s.m * mp * 2};
    if (!make_tensor_map(&maps.st[ST_Z16T], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, p.z16, dims, hstrides, sbox,
                         CU_TENSOR_MAP_SWIZZLE_64B))
      return tensor_map_error(__FILE__, __LINE__);
  }
  if (cudaFuncSetAttribute(pinv_big, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
      cudaSuccess)
    return set_cuda_error(cudaGetLastError());
  KernelScope scope("pinv_big", stream);
  pinv_big<<<(unsigned)(4 * BH), kThreads, kSmemBytes, stream>>>(maps, p);
  return launch_status();
}

}  // namespace nys
