// K-means rounds of clustered attention on the tensor cores ("Fast
// Transformers with Clustered Attention" review page, Proposed method,
// bullets 1 and 2), for bf16 queries with d in {64, 128} and C <= 128
// clusters. One round per launch of `kmeans_round_tc`, over 128-query tiles:
//   assignment  S = Q mu^T (128 x C_pad) as three bf16 products: mu is split
//               into hi + mid + lo (bf16 each, 24 bits of mu together) and Q
//               is exact in bf16, so S matches fp32 to rounding; then
//               a(i) = argmin_c |mu_c|^2 - 2 S[i, c] (ties: the lowest c),
//               the squared norms taken from the fp32 centroids
//   update      the members' sums onehot(a)^T Q (C_pad x d, one bf16 product
//               per tile with exact products and fp32 accumulation in TMEM,
//               reusing the Q tile as the MN-major right factor) and the
//               member counts, per CTA over its range of tiles of one head
// and `kmeans_reduce` sums the CTAs' partial sums in a fixed order (so a
// round is deterministic), divides by the counts (an empty cluster keeps its
// centroid), and prepares the next round's bf16 split and squared norms.
//
// Four worker warps (thread = query row of the tile, a TMEM lane, in the
// assignment; = cluster row for the members' sums) and an issuer warp whose
// lane 0 issues the TMA copies and the MMAs, driven by the workers' mbarrier
// arrivals. One CTA per SM. At d = 64 the Q tiles go through a ring of
// four buffers and the scores through two TMEM buffers, two tiles ahead of
// the members' product: tile j + 2's scores are issued right after tile j's
// product, into the buffer the workers read tile j's from. At d = 128 (three
// Q buffers, one score buffer) the next tile's scores are issued as soon as
// every worker has read this tile's. Either way the tensor cores work while
// the workers take the argmin and build the one-hot tile.
// Every mbarrier wait is bounded; a wait that runs out sets the status word
// and the CTA winds down (copies and products in flight awaited, TMEM
// freed).
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "nys_internal.h"
#include "nys_sm100.h"
#include "nys_tma_host.h"

namespace nys {
namespace {

using namespace sm100;

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kThreads = 160;  // four worker warps and the issuer warp
// TMEM: scores (C_pad columns; two buffers when the scores run two tiles
// ahead), members' sums (d columns)
constexpr uint32_t kColS = 0, kColU = 128, kColS2 = 256;
constexpr int kNQMax = 4;
// Q tile buffers, and how many tiles the scores run ahead of the members'
// product: d = 64 keeps four tiles of Q and two score buffers, so that a
// tile's scores never wait for the workers to read the previous tile's; at
// d = 128 shared memory holds three tiles and one score buffer.
__host__ __device__ constexpr int km_nq(int dch) { return dch == 1 ? 4 : 3; }
__host__ __device__ constexpr int km_ahead(int dch) { return dch == 1 ? 2 : 1; }

struct KmMaps {
  CUtensorMap q;    // bf16 [B*H][n][d], box 64 x 128
  CUtensorMap mu3;  // bf16 [B*H*3][C_pad][d] (hi, mid, lo per head), box 64 x C_pad
};

struct KmParams {
  const float* norms;  // [B*H][C_pad]  |mu_c|^2 of the fp32 centroids
  int* assign;         // [B*H][n]
  float* part;         // [B*H][S][C_pad][d]  members' sums per CTA
  int* cnt;            // [B*H][S][C_pad]     member counts per CTA
  int* status;
  int n, d, C, C_pad, tiles_per_head, tiles_per_cta, S;
  uint32_t off_mu, off_q, off_oh;  // shared-memory layout
};

struct KmBars {
  uint64_t mu, q[kNQMax], asg[2], upd, fin;
  uint64_t rd, ready;  // workers: a tile's scores read; its one-hot tile written
};

__device__ __forceinline__ bool km_wait(uint64_t* bar, uint32_t parity, int* status,
                                        volatile int* abort_flag) {
  if (mbar_wait(bar, parity, abort_flag, kWaitNs)) return true;
  if (!*abort_flag) {
    *abort_flag = 1;
    atomicExch(status, (int)NYS_ERR_TIMEOUT);
  }
  return false;
}

// grid (S, B*H): CTA (s, bh) runs tiles [s tpc, (s + 1) tpc) of head bh.
// DCH = d / 64 column boxes of Q and mu.
template <int DCH>
__global__ void __launch_bounds__(kThreads, 1) kmeans_round_tc(const __grid_constant__ KmMaps maps,
                                                               const KmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* mus = sm + p.off_mu;  // [3][DCH] boxes of C_pad rows x 128 B
  constexpr int kNQ = km_nq(DCH), kAhead = km_ahead(DCH);
  constexpr uint32_t kCols = kAhead == 2 ? 512 : 256;
  uint8_t* qb = sm + p.off_q;    // [kNQ][DCH] boxes of 128 rows x 128 B
  uint8_t* oh = sm + p.off_oh;   // one-hot^T: [2] boxes of 128 cluster rows x 64 queries (bf16)
  __shared__ KmBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ __align__(16) float norm_s[128];  // |mu_c|^2; +inf for c >= C (never the argmin)
  __shared__ int cnt_s[128];
  volatile int* abort_flag = &abort_sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool worker = warp < 4;
  const int s = blockIdx.x;
  const long long bh = blockIdx.y;
  const int t0 = s * p.tiles_per_cta;
  const int ntiles = max(0, min(p.tiles_per_head, t0 + p.tiles_per_cta) - t0);
  const uint32_t q_bytes = (uint32_t)DCH * 16384u;
  const uint32_t mu_box = (uint32_t)p.C_pad * 128u;

  if (tid == 0) {
    mbar_init(&bars.mu, 1);
    for (int r = 0; r < kNQ; ++r) mbar_init(&bars.q[r], 1);
    mbar_init(&bars.asg[0], 1);
    mbar_init(&bars.asg[1], 1);
    mbar_init(&bars.upd, 1);
    mbar_init(&bars.rd, 128);
    mbar_init(&bars.ready, 128);
    mbar_init(&bars.fin, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (worker) {
    norm_s[tid] = tid < p.C ? p.norms[bh * p.C_pad + tid] : INFINITY;
    cnt_s[tid] = 0;
  }
  // the one-hot tile starts all zero; each worker later clears only its own 1
  for (int e = tid; e < 2 * 128 * 128 / 16; e += kThreads)
    reinterpret_cast<uint4*>(oh)[e] = make_uint4(0u, 0u, 0u, 0u);
  fence_async_smem();
  if (warp == 0) tmem_alloc(&tmem_base_sh, kCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 4) {
    // ---------------------------------------------- issuer: copies, products
    if (lane == 0 && ntiles > 0) {
      uint32_t n_mu = 0, n_q[kNQ] = {};  // copies issued per buffer
      const uint32_t id_s = idesc_bf16(128, p.C_pad, false, false);
      const uint32_t id_u = idesc_bf16(128, 64 * DCH, false, true);
      auto load_q = [&](int jt) {  // tile t0 + jt into buffer jt % kNQ
        const int r = jt % kNQ;
        mbar_arrive_expect_tx(&bars.q[r], q_bytes);
        for (int c = 0; c < DCH; ++c)
          tma_load_3d(qb + (r * DCH + c) * 16384, &maps.q, &bars.q[r], 64 * c, (t0 + jt) * 128, (int)bh);
        ++n_q[r];
      };
      // scores of tile jt: Q mu^T as Q mu_hi^T + Q mu_mid^T + Q mu_lo^T, into
      // score buffer jt % 2 (with two buffers), completing on asg[jt % 2]
      auto scores = [&](int jt) -> bool {
        const int r = jt % kNQ;
        if (!km_wait(&bars.q[r], (n_q[r] - 1) & 1, p.status, abort_flag)) return false;
        tc_fence_after_sync();
        for (int k = 0; k < 3; ++k)
          for (int kk = 0; kk < 4 * DCH; ++kk) {
            const uint64_t a = smem_desc(smem_u32(qb + (r * DCH + (kk >> 2)) * 16384), 16, 1024, SW_128B);
            const uint64_t bd = smem_desc(smem_u32(mus + (k * DCH + (kk >> 2)) * mu_box), 16, 1024, SW_128B);
            mma_bf16(tmem + ((kAhead == 2 && (jt & 1)) ? kColS2 : kColS), a + (uint64_t)((kk & 3) * 2),
                     bd + (uint64_t)((kk & 3) * 2), id_s, (k > 0 || kk > 0) ? 1u : 0u);
          }
        mma_commit(&bars.asg[jt & 1]);
        return true;
      };
      tma_prefetch(&maps.q);
      tma_prefetch(&maps.mu3);
      mbar_arrive_expect_tx(&bars.mu, 3u * DCH * mu_box);
      for (int k = 0; k < 3; ++k)
        for (int c = 0; c < DCH; ++c)
          tma_load_3d(mus + (k * DCH + c) * mu_box, &maps.mu3, &bars.mu, 64 * c, 0, (int)(bh * 3 + k));
      n_mu = 1;
      for (int jt = 0; jt < kNQ - 1 && jt < ntiles; ++jt) load_q(jt);
      bool ok = km_wait(&bars.mu, 0, p.status, abort_flag);
      for (int jt = 0; ok && jt < kAhead && jt < ntiles; ++jt) ok = scores(jt);
      for (int j = 0; ok && j < ntiles; ++j) {
        // one score buffer: tile j + 1's scores once every worker has read tile j's
        if (kAhead == 1) {
          ok = km_wait(&bars.rd, j & 1, p.status, abort_flag);
          if (ok && j + 1 < ntiles) ok = scores(j + 1);
        }
        // tile j's members' product once its one-hot tile is written (the
        // workers waited for tile j - 1's product before writing it, and
        // had read tile j's scores)
        if (ok) ok = km_wait(&bars.ready, j & 1, p.status, abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
        const int r = j % kNQ;
        const uint64_t q0 = smem_desc(smem_u32(qb + r * DCH * 16384), 16384, 1024, SW_128B);
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t a = smem_desc(smem_u32(oh + (kk >> 2) * 16384), 16, 1024, SW_128B);
          mma_bf16(tmem + kColU, a + (uint64_t)((kk & 3) * 2), q0 + (uint64_t)(kk * 128), id_u,
                   (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars.upd);
        // two score buffers: tile j + 2's scores into the buffer tile j's
        // scores were read from (its Q tile landed one tile earlier)
        if (kAhead == 2 && j + 2 < ntiles && !scores(j + 2)) break;
        // tile j + kNQ - 1 into the buffer of tile j - 1, whose product is
        // done (the workers waited for it before this tile's one-hot tile)
        if (j + kNQ - 1 < ntiles) load_q(j + kNQ - 1);
      }
      if (*abort_flag) {
        // no copy of this CTA may still be in flight
        if (n_mu) mbar_wait(&bars.mu, 0, nullptr, kWaitNs);
        for (int r = 0; r < kNQ; ++r)
          if (n_q[r]) mbar_wait(&bars.q[r], (n_q[r] - 1) & 1, nullptr, kWaitNs);
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------- workers: thread = query row
    const uint32_t lo = static_cast<uint32_t>(warp * 32) << 16;
    int prev_a = -1;  // where this thread's query put its 1 in the one-hot tile
    for (int j = 0; j < ntiles; ++j) {
      const int tile = t0 + j;
      // assignment: nearest centroid of this thread's query
      const bool ok = km_wait(&bars.asg[j & 1], (j >> 1) & 1, p.status, abort_flag);
      const bool go = __all_sync(0xffffffffu, ok);  // warp-uniform: TMEM loads are warp-wide
      tc_fence_after_sync();
      // four independent running minima (column c in chain c % 4) over the
      // 128 score columns, loaded at once (columns C_pad and up are inside
      // the score region, and the +inf norms past C keep them out);
      // strict < keeps a chain's lowest index among equal scores, and the
      // chains combine by (score, index)
      float bv[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
      int bc[4] = {0, 0, 0, 0};
      if (go) {
        uint32_t v[4][32];
        const uint32_t scol = (kAhead == 2 && (j & 1)) ? kColS2 : kColS;
#pragma unroll
        for (int h = 0; h < 4; ++h) tmem_ld32(tmem + lo + scol + 32 * h, v[h]);
        tmem_ld_wait();
        const float4* n4 = reinterpret_cast<const float4*>(norm_s);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 nr = n4[(32 * h + e) >> 2];
            const float nn[4] = {nr.x, nr.y, nr.z, nr.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float score = fmaf(-2.f, __uint_as_float(v[h][e + k]), nn[k]);
              if (score < bv[k]) {
                bv[k] = score;
                bc[k] = 32 * h + e + k;
              }
            }
          }
        }
      }
      float best = bv[0];
      int best_c = bc[0];
#pragma unroll
      for (int k = 1; k < 4; ++k)
        if (bv[k] < best || (bv[k] == best && bc[k] < best_c)) {
          best = bv[k];
          best_c = bc[k];
        }
      tc_fence_before_sync();
      mbar_arrive(&bars.rd);  // the scores of tile j are read
      const int i = tile * 128 + tid;
      const bool valid = go && i < p.n;
      if (valid) {
        p.assign[bh * p.n + i] = best_c;
        atomicAdd(&cnt_s[best_c], 1);
      }
      // one-hot^T for the members' product: this thread's column, once the
      // product of tile j-1 has read the tile
      if (j >= 1) km_wait(&bars.upd, (j - 1) & 1, p.status, abort_flag);
      uint8_t* ohb = oh + (tid >> 6) * 16384;
      if (prev_a >= 0) *reinterpret_cast<uint16_t*>(ohb + sw128_offset(prev_a, (tid & 63) * 2)) = 0;
      prev_a = valid ? best_c : -1;
      if (valid) *reinterpret_cast<uint16_t*>(ohb + sw128_offset(best_c, (tid & 63) * 2)) = 0x3F80;  // bf16 1
      fence_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&bars.ready);
    }
    // the last members' product done
    if (ntiles > 0) km_wait(&bars.upd, (ntiles - 1) & 1, p.status, abort_flag);
  }
  tc_fence_before_sync();
  __syncthreads();  // counts complete; the members' sums in TMEM
  tc_fence_after_sync();

  // this CTA's members' sums and counts; thread = cluster row
  if (worker) {
    const uint32_t lo = static_cast<uint32_t>(warp * 32) << 16;
    const bool go = __all_sync(0xffffffffu, !*abort_flag) && ntiles > 0;
    float* prow = p.part + (((size_t)bh * p.S + s) * p.C_pad + (tid < p.C_pad ? tid : 0)) * p.d;
    for (int c0 = 0; c0 < p.d; c0 += 32) {
      uint32_t v[32];
      if (go) {
        tmem_ld32(tmem + lo + kColU + c0, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;
      }
      if (tid < p.C_pad) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<uint4*>(prow + c0 + e) = make_uint4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
    }
    if (tid < p.C_pad) p.cnt[((size_t)bh * p.S + s) * p.C_pad + tid] = cnt_s[tid];
  }

  // wind-down: no product of this CTA may still be in flight
  if (warp == 4 && lane == 0) {
    mma_commit(&bars.fin);
    mbar_wait(&bars.fin, 0, nullptr, kWaitNs);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kCols);
}

// grid (ceil(C_pad / cpb), B*H), block 256: thread (centroid c, columns
// [j, j + 4)), d / 4 threads per centroid and cpb = 256 / (d / 4) centroids
// per CTA (d = 64 or 128), every load in flight at once. With S > 0: the new
// centroid = the CTAs' members' sums added in CTA order, over the summed
// counts (an empty cluster keeps mu_old); with S = 0 the centroid is mu_old
// as it is. Either way it writes the bf16 split (hi, mid, lo) of the
// centroid and its squared norm (reduced over the centroid's lanes) for the
// next assignment; rows c >= C are zero.
constexpr int kRedThreads = 256;

__device__ __forceinline__ uint2 pack_bf16x4(float a, float b, float c, float d) {
  return make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, d));
}

__global__ void __launch_bounds__(kRedThreads) kmeans_reduce(const float* __restrict__ part,
                                                             const int* __restrict__ cnt,
                                                             const float* __restrict__ mu_old,
                                                             float* __restrict__ mu_new,
                                                             __nv_bfloat16* __restrict__ mu3,
                                                             float* __restrict__ norms, int S, int d,
                                                             int C, int C_pad) {
  const int tpc = d >> 2, cpb = kRedThreads / tpc;
  const int c = blockIdx.x * cpb + (int)threadIdx.x / tpc, j = ((int)threadIdx.x % tpc) * 4;
  const long long bh = blockIdx.y;
  float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c < C) {
    const size_t o = ((size_t)bh * C + c) * d + j;
    x = *reinterpret_cast<const float4*>(mu_old + o);
    if (S > 0) {
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
      int count = 0;
      for (int s = 0; s < S; ++s) {
        const size_t r = ((size_t)bh * S + s) * C_pad + c;
        const float4 v = *reinterpret_cast<const float4*>(part + r * d + j);
        sum.x += v.x;
        sum.y += v.y;
        sum.z += v.z;
        sum.w += v.w;
        count += cnt[r];
      }
      if (count > 0) {
        const float f = (float)count;
        x = make_float4(sum.x / f, sum.y / f, sum.z / f, sum.w / f);
      }
      *reinterpret_cast<float4*>(mu_new + o) = x;
    }
  }
  if (c < C_pad) {
    const float xs[4] = {x.x, x.y, x.z, x.w};
    float hi[4], mid[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat16 h = __float2bfloat16_rn(xs[e]);
      const float r1 = xs[e] - __bfloat162float(h);
      const __nv_bfloat16 m2 = __float2bfloat16_rn(r1);
      hi[e] = __bfloat162float(h);
      mid[e] = __bfloat162float(m2);
      lo[e] = r1 - mid[e];
    }
    const size_t base = ((size_t)bh * 3 * C_pad + c) * d + j;
    *reinterpret_cast<uint2*>(mu3 + base) = pack_bf16x4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint2*>(mu3 + base + (size_t)C_pad * d) = pack_bf16x4(mid[0], mid[1], mid[2], mid[3]);
    *reinterpret_cast<uint2*>(mu3 + base + 2 * (size_t)C_pad * d) = pack_bf16x4(lo[0], lo[1], lo[2], lo[3]);
  }
  float sq = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
  for (int off = tpc >> 1; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
  if (c < C_pad && j == 0) norms[(size_t)bh * C_pad + c] = sq;
}

struct KmPlan {
  int C_pad, T_h, tpc, S, dch;
  uint32_t off_mu, off_q, off_oh;
  size_t smem;
};

KmPlan km_plan(const Shape& s) {
  KmPlan k{};
  k.dch = s.d / 64;
  k.C_pad = (s.m + 15) & ~15;
  k.T_h = (s.n + 127) / 128;
  // one CTA per SM (the shared-memory request below keeps it so), at most
  // one wave: floor(SMs / heads) CTAs per head, whole tiles each
  const int bh = (int)std::min<long long>(s.bh(), 1 << 30);
  const int want = std::max(1, plan_sms() / bh);
  k.tpc = std::max(1, (k.T_h + want - 1) / want);
  k.S = (k.T_h + k.tpc - 1) / k.tpc;
  k.off_mu = 0;
  k.off_q = k.off_mu + 3u * k.dch * k.C_pad * 128u;
  k.off_oh = k.off_q + (uint32_t)km_nq(k.dch) * k.dch * 16384u;
  // more than half an SM's shared memory, so that one CTA (256 or 512 TMEM columns) holds an SM
  k.smem = std::max<size_t>((size_t)k.off_oh + 2 * 16384 + 1024, 116 * 1024);
  return k;
}

}  // namespace

bool kmeans_tc_supported(const Shape& s) {
  if (s.dtype != NYS_BF16 || (s.d != 64 && s.d != 128) || s.m < 1 || s.m > 128) return false;
  // dynamic shared memory, leaving room for the kernel's static part
  return km_plan(s).smem <= 225 * 1024;
}

KmWorkspace kmeans_tc_workspace(const Shape& s) {
  const KmPlan k = km_plan(s);
  KmWorkspace w{};
  w.S = k.S;
  w.C_pad = k.C_pad;
  w.mu3_bytes = (size_t)s.bh() * 3 * k.C_pad * s.d * 2;
  w.norm_bytes = (size_t)s.bh() * k.C_pad * 4;
  w.part_bytes = (size_t)s.bh() * k.S * k.C_pad * s.d * 4;
  w.cnt_bytes = (size_t)s.bh() * k.S * k.C_pad * 4;
  return w;
}

int launch_kmeans_prep(const Shape& s, const float* mu, void* mu3, float* norms, cudaStream_t st) {
  const KmPlan k = km_plan(s);
  KernelScope scope("kmeans_reduce", st);
  const int cpb = kRedThreads / (s.d / 4);
  kmeans_reduce<<<dim3((unsigned)((k.C_pad + cpb - 1) / cpb), (unsigned)s.bh()), kRedThreads, 0, st>>>(
      nullptr, nullptr, mu, nullptr, static_cast<__nv_bfloat16*>(mu3), norms, 0, s.d, s.m, k.C_pad);
  return launch_status();
}

int launch_kmeans_round_tc(const Shape& s, const void* q, const void* mu3, const float* norms,
                           int* assign, float* part, int* cnt, const float* mu_old, float* mu_new,
                           float* norms_next, void* mu3_next, int* status, cudaStream_t st) {
  if (!kmeans_tc_supported(s)) return NYS_ERR_UNSUPPORTED;
  const KmPlan k = km_plan(s);
  const uint64_t BH = (uint64_t)s.bh();
  KmMaps maps;
  memset(&maps, 0, sizeof(maps));
  {
    const uint64_t dims[3] = {(uint64_t)s.d, (uint64_t)s.n, BH};
    const uint64_t strides[2] = {(uint64_t)s.d * 2, (uint64_t)s.n * s.d * 2};
    const uint32_t box[3] = {64, 128, 1};
    if (!make_tensor_map(&maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
  }
  {
    const uint64_t dims[3] = {(uint64_t)s.d, (uint64_t)k.C_pad, BH * 3};
    const uint64_t strides[2] = {(uint64_t)s.d * 2, (uint64_t)k.C_pad * s.d * 2};
    const uint32_t box[3] = {64, (uint32_t)k.C_pad, 1};
    if (!make_tensor_map(&maps.mu3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, mu3, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
  }
  KmParams p{};
  p.norms = norms;
  p.assign = assign;
  p.part = part;
  p.cnt = cnt;
  p.status = status;
  p.n = s.n;
  p.d = s.d;
  p.C = s.m;
  p.C_pad = k.C_pad;
  p.tiles_per_head = k.T_h;
  p.tiles_per_cta = k.tpc;
  p.S = k.S;
  p.off_mu = k.off_mu;
  p.off_q = k.off_q;
  p.off_oh = k.off_oh;
  const dim3 grid((unsigned)k.S, (unsigned)BH);
  {
    KernelScope scope("kmeans_round_tc", st);
    if (k.dch == 1) {
      if (cudaFuncSetAttribute(kmeans_round_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)k.smem) != cudaSuccess)
        return set_cuda_error(cudaGetLastError());
      kmeans_round_tc<1><<<grid, kThreads, k.smem, st>>>(maps, p);
    } else {
      if (cudaFuncSetAttribute(kmeans_round_tc<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)k.smem) != cudaSuccess)
        return set_cuda_error(cudaGetLastError());
      kmeans_round_tc<2><<<grid, kThreads, k.smem, st>>>(maps, p);
    }
    const int rc = launch_status();
    if (rc != NYS_OK) return rc;
  }
  KernelScope scope("kmeans_reduce", st);
  const int cpb = kRedThreads / (s.d / 4);
  kmeans_reduce<<<dim3((unsigned)((k.C_pad + cpb - 1) / cpb), (unsigned)BH), kRedThreads, 0, st>>>(
      part, cnt, mu_old, mu_new, static_cast<__nv_bfloat16*>(mu3_next), norms_next, k.S, s.d, s.m,
      k.C_pad);
  return launch_status();
}

}  // namespace nys
