// Token rows on the tensor cores (bf16 inputs, fp32 accumulate):
//   out[t] = softmax(Q[t] K~^T / sqrt(d)) W + sum_j w[h][j] V[t + j - (ks-1)/2]
// ("Nyströmformer" review page, Proposed method, bullets 3 and 6).
//
// Persistent CTAs walk contiguous ranges of 128-token tiles. Warp roles:
//   warp 0       TMA producer: Q tiles (ring of 2-3 stages, freed once F is
//                done), V halos (ring of 2, freed once the conv is done), and
//                per head K~ and W^T (1-2 buffers); Q and V streams advance
//                independently
//   warp 1       tcgen05 issuer of the F and conv streams (the conv does
//                not wait for the softmax); warp 16 issuer of the PW stream
//                (each tcgen05.mma costs its issuing thread tens of cycles):
//                  F  = Q_tile K~^T          A = Q (smem), B = K~ (smem)
//                  PW = P W                  A = P (TMEM), B = W^T (smem)
//                  CV = T V_halo             A = banded Toeplitz of the conv
//                                            taps (smem), B = V (MN-major)
//   warps 2-3    build the Toeplitz block of the next head's taps (the first
//                head's block is built by the whole CTA up front)
//   warps 4-7    softmax of even tiles, warps 8-11 softmax of odd tiles:
//                thread = row, reads F from TMEM, writes P (bf16) back over
//                it, row sum to shared memory
//   warps 12-15  epilogue: out = PW / rowsum + CV, bf16 store
// F/P and the PW/CV accumulators are double-buffered in TMEM. Every wait is
// bounded; a wait that runs out sets the status word, every role winds down,
// copies in flight are awaited and TMEM is freed.
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
  int nq, nkw, nt;  // Q stages; buffers of the per-head K~/W^T and Toeplitz blocks
  float c;          // softmax scale * log2(e)
  uint32_t tmem_cols;
  uint32_t off_q, off_v, off_kt, off_t, off_l;  // smem offsets from the aligned base
  uint32_t q_stage, v_stage, kt_bytes, wt_bytes, t_bytes;
};

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s
constexpr int kThreads = 544;
constexpr int kNV = 2;  // V halo stages
// dynamic shared memory budget: the 227 KB per-block opt-in limit less the
// kernel's static shared memory (barriers) and a margin
constexpr size_t kSmemBudget = 227 * 1024 - 1024;

struct Bars {
  uint64_t qfull[3], qempty[3];      // Q tile ring
  uint64_t vfull[2], vempty[2];      // V halo ring
  uint64_t kw_full[2], kw_empty[2];  // per-head K~ / W^T
  uint64_t t_ready[2], t_empty[2];   // per-head Toeplitz block
  uint64_t f_full[2], p_full[2], pw_done[2];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t l_full[4];
};

__device__ __forceinline__ void set_fail(int* status, volatile int* abort_flag) {
  if (!*abort_flag) {
    *abort_flag = 1;
    atomicExch(status, (int)NYS_ERR_TIMEOUT);
  }
}

__device__ __forceinline__ bool wait_or_fail(uint64_t* bar, uint32_t parity, int* status,
                                             volatile int* abort_flag) {
  if (mbar_wait(bar, parity, abort_flag, kWaitNs)) return true;
  set_fail(status, abort_flag);
  return false;
}

// A walk over the CTA's tiles that tracks the head and the tile within it
// incrementally (the polling loops below do no division).
struct TileWalk {
  int j;       // tile within the CTA's range
  int bh, t;   // head, tile within the head
  bool first;  // first tile of a head (or of the range)
  __device__ void init(int g0, int tph) {
    j = 0;
    bh = g0 / tph;
    t = g0 - bh * tph;
    first = true;
  }
  __device__ bool last(int tph, int ntiles) const { return t == tph - 1 || j == ntiles - 1; }
  __device__ void next(int tph) {
    ++j;
    first = ++t == tph;
    if (first) {
      t = 0;
      ++bh;
    }
  }
};

// Slot and phase parity of a ring of n buffers, advanced one use at a time.
struct Ring {
  int i;
  uint32_t ph;
  __device__ void init() {
    i = 0;
    ph = 0;
  }
  __device__ void next(int n) {
    if (++i == n) {
      i = 0;
      ph ^= 1u;
    }
  }
};

// The Toeplitz operand of the conv: element (t, u) is w[u - t] (t the tile's
// token, u the halo row), so its 64 x 64 block (r, c) depends on c - r only:
// B_k[t'][u'] = w[64 k + u' - t']. It is kept as the list B_(nbox-1), ...,
// B_0, B_-1 (= 0) of 8 KB blocks; K-box c of the operand (128 rows) is then
// the window [B_c; B_c-1], which starts at block nbox - 1 - c. One 16-byte
// chunk (8 taps, columns u0 ..) of row t' of list block blk:
__device__ __forceinline__ void toeplitz_chunk(uint8_t* tbuf, const float* wh, int ks, int nbox,
                                               int blk, int t, int u0) {
  const int base = 64 * (nbox - 1 - blk) + u0 - t;  // tap index of column u0
  uint32_t wv[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int ua = base + 2 * e, ub = ua + 1;
    const float fa = (ua >= 0 && ua < ks) ? __ldg(wh + ua) : 0.f;
    const float fb = (ub >= 0 && ub < ks) ? __ldg(wh + ub) : 0.f;
    wv[e] = pack_bf16x2(fa, fb);
  }
  *reinterpret_cast<uint4*>(tbuf + blk * 8192 + sw128_offset(t, u0 * 2)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
}

template <int DP>
__global__ void __launch_bounds__(kThreads, 1) tokens_tc(const __grid_constant__ TokMaps maps,
                                                         const TokParams p) {
  constexpr int DC = DP / 64;  // 64-column chunks of d
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  volatile int* abort_flag = &abort_sh;
  float* lbuf = reinterpret_cast<float*>(sm + p.off_l);  // [4][128] row sums

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g0 = blockIdx.x * p.tiles_per_cta;
  const int g1 = min(p.total_tiles, g0 + p.tiles_per_cta);
  const int ntiles = g1 - g0;
  const int rad = p.ks > 0 ? (p.ks - 1) / 2 : 0;
  const int nbox = (p.kc + 63) >> 6;  // 64-column boxes of the conv's K
  auto head_of = [&](int g) { return g / p.tiles_per_head; };

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) {
      mbar_init(&bars.qfull[i], 1);
      mbar_init(&bars.qempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.vfull[i], 1);
      mbar_init(&bars.vempty[i], 1);
      mbar_init(&bars.kw_full[i], 1);
      mbar_init(&bars.kw_empty[i], 1);
      mbar_init(&bars.t_ready[i], 64);
      mbar_init(&bars.t_empty[i], 1);
      mbar_init(&bars.f_full[i], 1);
      mbar_init(&bars.p_full[i], 128);
      mbar_init(&bars.pw_done[i], 1);
      mbar_init(&bars.acc_full[i], p.kc > 0 ? 2 : 1);  // PW and CV commits
      mbar_init(&bars.acc_empty[i], 128);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&bars.l_full[i], 128);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, p.tmem_cols);
  // the first head's Toeplitz block, by the whole CTA
  if (p.kc > 0 && ntiles > 0) {
    const float* wh = p.conv_w + (size_t)(head_of(g0) % p.H) * p.ks;
    for (int task = tid; task < (nbox + 1) * 64 * 8; task += kThreads)
      toeplitz_chunk(sm + p.off_t, wh, p.ks, nbox, task >> 9, (task >> 3) & 63, (task & 7) * 8);
    fence_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (p.kc > 0 && ntiles > 0 && (warp == 2 || warp == 3)) mbar_arrive(&bars.t_ready[0]);
  const uint32_t tmem = tmem_base_sh;
  // TMEM columns: F/P buffers [2][m_pad], then accumulators [2][PW | CV]
  const uint32_t COL_F0 = 0, COL_ACC0 = 2 * p.m_pad;
  const uint32_t ACC_W = 2 * DP;
  const uint32_t kw_bytes = p.kt_bytes + p.wt_bytes;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && ntiles > 0) {
      tma_prefetch(&maps.q);
      tma_prefetch(&maps.v);
      tma_prefetch(&maps.kt);
      tma_prefetch(&maps.wt);
      const int tph = p.tiles_per_head;
      TileWalk wq, wv;
      wq.init(g0, tph);
      wv.init(g0, tph);
      Ring rq, rv, rk;  // Q stages, V stages, per-head K~ / W^T buffers
      rq.init();
      rv.init();
      rk.init();
      const int nv_tiles = p.kc > 0 ? ntiles : 0;
      int heads = 0;  // per-head loads issued
      uint32_t nq_issued[3] = {0, 0, 0}, nv_issued[2] = {0, 0}, nkw_issued[2] = {0, 0};
      uint64_t t_last = globaltimer_ns();
      while (wq.j < ntiles || wv.j < nv_tiles) {
        bool prog = false;
        if (wq.j < ntiles) {
          const bool new_head = wq.first;
          const bool kw_ok = !new_head || heads < p.nkw || mbar_test(&bars.kw_empty[rk.i], rk.ph ^ 1u);
          const bool q_ok = wq.j < p.nq || mbar_test(&bars.qempty[rq.i], rq.ph ^ 1u);
          if (kw_ok && q_ok) {
            if (new_head) {
              const int kb = rk.i;
              uint8_t* kts = sm + p.off_kt + kb * kw_bytes;
              uint8_t* wts = kts + p.kt_bytes;
              mbar_arrive_expect_tx(&bars.kw_full[kb], kw_bytes);
              for (int dc = 0; dc < DC; ++dc)
                tma_load_3d(kts + dc * (p.m_pad * 128), &maps.kt, &bars.kw_full[kb], dc * 64, 0, wq.bh);
              for (int mc = 0; mc * 64 < p.m_pad; ++mc)
                tma_load_3d(wts + mc * (DP * 128), &maps.wt, &bars.kw_full[kb], mc * 64, 0, wq.bh);
              ++nkw_issued[kb];
              ++heads;
              rk.next(p.nkw);
            }
            const int sq = rq.i;
            uint8_t* qs = sm + p.off_q + sq * p.q_stage;
            mbar_arrive_expect_tx(&bars.qfull[sq], p.q_stage);
            for (int dc = 0; dc < DC; ++dc)
              tma_load_3d(qs + dc * 16384, &maps.q, &bars.qfull[sq], dc * 64, wq.t * 128, wq.bh);
            ++nq_issued[sq];
            rq.next(p.nq);
            wq.next(tph);
            prog = true;
          }
        }
        if (wv.j < wq.j && wv.j < nv_tiles) {
          const int sv = rv.i;
          if (wv.j < kNV || mbar_test(&bars.vempty[sv], rv.ph ^ 1u)) {
            uint8_t* vs = sm + p.off_v + sv * p.v_stage;
            mbar_arrive_expect_tx(&bars.vfull[sv], p.v_stage);
            for (int dc = 0; dc < DC; ++dc)
              tma_load_3d(vs + dc * (p.kc * 128), &maps.v, &bars.vfull[sv], dc * 64,
                          wv.t * 128 - rad, wv.bh);
            ++nv_issued[sv];
            rv.next(kNV);
            wv.next(tph);
            prog = true;
          }
        }
        if (prog) {
          t_last = globaltimer_ns();
        } else {
          if (*abort_flag) break;
          if (globaltimer_ns() - t_last > kWaitNs) {
            set_fail(p.status, abort_flag);
            break;
          }
          __nanosleep(64);  // back off: leave issue slots to the working warps
        }
      }
      if (*abort_flag) {
        // wait (bounded) for this warp's copies still in flight
        for (int i = 0; i < 3; ++i)
          if (nq_issued[i]) mbar_wait(&bars.qfull[i], (nq_issued[i] - 1) & 1, nullptr, kWaitNs);
        for (int i = 0; i < 2; ++i) {
          if (nv_issued[i]) mbar_wait(&bars.vfull[i], (nv_issued[i] - 1) & 1, nullptr, kWaitNs);
          if (nkw_issued[i]) mbar_wait(&bars.kw_full[i], (nkw_issued[i] - 1) & 1, nullptr, kWaitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------- MMA issuer, F and conv streams
    if (lane == 0 && ntiles > 0) {
      const uint32_t idf = idesc_bf16(128, p.m_pad, false, false);
      const uint32_t idc = idesc_bf16(128, DP, false, true);
      const int ncv = p.kc > 0 ? ntiles : 0;
      const int tph = p.tiles_per_head;
      TileWalk wf, wc;
      wf.init(g0, tph);
      wc.init(g0, tph);
      Ring rqf, rkf, rtc, rvc;  // Q stages, K~ buffers, Toeplitz buffers, V stages
      rqf.init();
      rkf.init();
      rtc.init();
      rvc.init();
      int kcur = 0, tcur = 0;  // buffers of the current head
      uint64_t t_last = globaltimer_ns();
      while (wf.j < ntiles || wc.j < ncv) {
        bool prog = false;
        // F stream: F(j) = Q K~^T into F buffer j & 1
        if (wf.j < ntiles) {
          const int jf = wf.j;
          const bool new_head = wf.first;
          const bool ok = (!new_head || mbar_test(&bars.kw_full[rkf.i], rkf.ph)) &&
                          mbar_test(&bars.qfull[rqf.i], rqf.ph) &&
                          (jf < 2 || mbar_test(&bars.pw_done[jf & 1], ((jf >> 1) - 1) & 1));
          if (ok) {
            if (new_head) {
              kcur = rkf.i;
              rkf.next(p.nkw);
            }
            tc_fence_after_sync();
            const uint64_t a0 = smem_desc(smem_u32(sm + p.off_q + rqf.i * p.q_stage), 16, 1024, SW_128B);
            const uint64_t b0 = smem_desc(smem_u32(sm + p.off_kt + kcur * kw_bytes), 16, 1024, SW_128B);
            const uint32_t dcol = tmem + COL_F0 + (jf & 1) * p.m_pad;
#pragma unroll
            for (int kk = 0; kk < DP / 16; ++kk)
              mma_bf16(dcol, a0 + (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2),
                       b0 + (uint64_t)((kk >> 2) * (p.m_pad * 8) + (kk & 3) * 2), idf, kk > 0);
            mma_commit(&bars.f_full[jf & 1]);
            mma_commit(&bars.qempty[rqf.i]);
            rqf.next(p.nq);
            wf.next(tph);
            prog = true;
          }
        }
        // conv stream: CV(j) = T V_halo into accumulator j & 1 (does not
        // wait for the softmax)
        if (wc.j < ncv) {
          const int jc = wc.j;
          const bool new_head = wc.first;
          const bool ok = (!new_head || mbar_test(&bars.t_ready[rtc.i], rtc.ph)) &&
                          mbar_test(&bars.vfull[rvc.i], rvc.ph) &&
                          (jc < 2 || mbar_test(&bars.acc_empty[jc & 1], ((jc >> 1) - 1) & 1));
          if (ok) {
            if (new_head) {
              tcur = rtc.i;
              rtc.next(p.nt);
            }
            tc_fence_after_sync();
            const uint32_t acc = tmem + COL_ACC0 + (jc & 1) * ACC_W;
            const uint64_t a0 = smem_desc(smem_u32(sm + p.off_t + tcur * p.t_bytes), 16, 1024, SW_128B);
            const uint64_t v0 = smem_desc(smem_u32(sm + p.off_v + rvc.i * p.v_stage), p.kc * 128, 1024, SW_128B);
            for (int kk = 0; kk < p.kc / 16; ++kk)
              mma_bf16(acc + DP, a0 + (uint64_t)((nbox - 1 - (kk >> 2)) * 512 + (kk & 3) * 2),
                       v0 + (uint64_t)(kk * 128), idc, kk > 0);
            mma_commit(&bars.vempty[rvc.i]);
            mma_commit(&bars.acc_full[jc & 1]);
            if (wc.last(tph, ntiles)) mma_commit(&bars.t_empty[tcur]);
            rvc.next(kNV);
            wc.next(tph);
            prog = true;
          }
        }
        if (prog) {
          t_last = globaltimer_ns();
        } else {
          if (*abort_flag) break;
          if (globaltimer_ns() - t_last > kWaitNs) {
            set_fail(p.status, abort_flag);
            break;
          }
          __nanosleep(64);  // back off: leave issue slots to the working warps
        }
      }
    }
  } else if (warp == 16) {
    // ---------------------------------------------- MMA issuer, PW stream
    if (lane == 0 && ntiles > 0) {
      const uint32_t idw = idesc_bf16(128, DP, false, false);
      const int tph = p.tiles_per_head;
      TileWalk wp;
      wp.init(g0, tph);
      Ring rkp;  // per-head W^T buffers
      rkp.init();
      int kcur = 0;
      uint64_t t_last = globaltimer_ns();
      while (wp.j < ntiles) {
        bool prog = false;
        // PW stream: PW(j) = P W into accumulator j & 1
        {
          const int jp = wp.j;
          const bool ok = mbar_test(&bars.p_full[jp & 1], (jp >> 1) & 1) &&
                          (jp < 2 || mbar_test(&bars.acc_empty[jp & 1], ((jp >> 1) - 1) & 1));
          if (ok) {
            if (wp.first) {
              kcur = rkp.i;
              rkp.next(p.nkw);
            }
            tc_fence_after_sync();
            const uint32_t acc = tmem + COL_ACC0 + (jp & 1) * ACC_W;
            const uint64_t b0 = smem_desc(smem_u32(sm + p.off_kt + kcur * kw_bytes + p.kt_bytes), 16, 1024, SW_128B);
            const uint32_t pcol = tmem + COL_F0 + (jp & 1) * p.m_pad;
            for (int kk = 0; kk < p.m_pad / 16; ++kk)
              mma_bf16_tA(acc, pcol + kk * 8, b0 + (uint64_t)((kk >> 2) * (DP * 8) + (kk & 3) * 2), idw, kk > 0);
            mma_commit(&bars.acc_full[jp & 1]);
            mma_commit(&bars.pw_done[jp & 1]);
            if (wp.last(tph, ntiles)) mma_commit(&bars.kw_empty[kcur]);
            wp.next(tph);
            prog = true;
          }
        }
        if (prog) {
          t_last = globaltimer_ns();
        } else {
          if (*abort_flag) break;
          if (globaltimer_ns() - t_last > kWaitNs) {
            set_fail(p.status, abort_flag);
            break;
          }
          __nanosleep(64);  // back off: leave issue slots to the working warps
        }
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------- Toeplitz builders
    if (p.kc > 0 && ntiles > 0) {
      const int lt = tid - 64;  // row lt of every block
      int hi = 0, cur_bh = head_of(g0);
      for (int j = 1; j < ntiles; ++j) {
        const int bh = head_of(g0 + j);
        if (bh == cur_bh) continue;
        cur_bh = bh;
        ++hi;
        const int tb = hi % p.nt;
        if (hi >= p.nt && !wait_or_fail(&bars.t_empty[tb], ((hi / p.nt) - 1) & 1, p.status, abort_flag)) break;
        const float* wh = p.conv_w + (size_t)(bh % p.H) * p.ks;
        uint8_t* tbuf = sm + p.off_t + tb * p.t_bytes;
        for (int blk = 0; blk <= nbox; ++blk)
          for (int u0 = 0; u0 < 64; u0 += 8) toeplitz_chunk(tbuf, wh, p.ks, nbox, blk, lt, u0);
        fence_async_smem();
        mbar_arrive(&bars.t_ready[tb]);
      }
    }
  } else if (warp < 12) {
    // ------------------------------------- softmax: warps 4-7 even tiles,
    // warps 8-11 odd tiles (F buffer = tile parity)
    const int grp = (warp - 4) >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t fcol = tmem + lo + COL_F0 + grp * p.m_pad;
    const bool full_m = p.m == p.m_pad && (p.m_pad & 63) == 0;
    for (int j = grp; j < ntiles; j += 2) {
      if (!__all_sync(0xffffffffu, wait_or_fail(&bars.f_full[grp], (j >> 1) & 1, p.status, abort_flag))) break;
      tc_fence_after_sync();
      float mx = -INFINITY, l = 0.f;
      if (full_m) {
        // m is a multiple of 64: no masks. Tile max with two 32-column
        // chunks in flight at a time.
        for (int c0 = 0; c0 < p.m_pad; c0 += 64) {
          uint32_t r0[32], r1[32];
          tmem_ld32(fcol + c0, r0);
          tmem_ld32(fcol + c0 + 32, r1);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            mx = fmaxf(mx, fmaxf(__uint_as_float(r0[e]), __uint_as_float(r1[e])));
        }
        const float mc = mx * p.c;
        for (int c0 = 0; c0 < p.m_pad; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(fcol + c0, r);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float a = fast_exp2(fmaf(__uint_as_float(r[2 * e]), p.c, -mc));
            const float b = fast_exp2(fmaf(__uint_as_float(r[2 * e + 1]), p.c, -mc));
            l += a + b;
            pk[e] = pack_bf16x2(a, b);
          }
          tmem_st16(fcol + (c0 >> 1), pk);
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
        const float mc = mx * p.c;
        for (int c0 = 0; c0 < p.m_pad; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(fcol + c0, r);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float a = (c0 + 2 * e < p.m) ? fast_exp2(fmaf(__uint_as_float(r[2 * e]), p.c, -mc)) : 0.f;
            const float b = (c0 + 2 * e + 1 < p.m) ? fast_exp2(fmaf(__uint_as_float(r[2 * e + 1]), p.c, -mc)) : 0.f;
            l += a + b;
            pk[e] = pack_bf16x2(a, b);
          }
          tmem_st16(fcol + (c0 >> 1), pk);
        }
      }
      tmem_st_wait();
      lbuf[(j & 3) * 128 + row] = l;
      tc_fence_before_sync();
      mbar_arrive(&bars.p_full[grp]);
      mbar_arrive(&bars.l_full[j & 3]);
    }
  } else if (warp < 16) {
    // ------------------------------------------------------------ epilogue
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
    for (int j = 0; j < ntiles; ++j) {
      const int ab = j & 1;
      const int g = g0 + j, bh = head_of(g), t = (g % p.tiles_per_head) * 128 + row;
      bool ok = wait_or_fail(&bars.acc_full[ab], (j >> 1) & 1, p.status, abort_flag);
      ok = ok && wait_or_fail(&bars.l_full[j & 3], (j >> 2) & 1, p.status, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after_sync();
      const float inv_l = 1.f / lbuf[(j & 3) * 128 + row];
      const uint32_t acc = tmem + lo + COL_ACC0 + ab * ACC_W;
      __nv_bfloat16* orow = p.out + ((size_t)bh * p.n + t) * p.d;
      uint4 o4[DP / 8];
#pragma unroll
      for (int c0 = 0; c0 < DP; c0 += 32) {
        uint32_t a[32], b[32];
        tmem_ld32(acc + c0, a);
        if (p.kc > 0) tmem_ld32(acc + DP + c0, b);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t w4[4];
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            const int i0 = 8 * e + 2 * f;
            float x0 = __uint_as_float(a[i0]) * inv_l, x1 = __uint_as_float(a[i0 + 1]) * inv_l;
            if (p.kc > 0) {
              x0 += __uint_as_float(b[i0]);
              x1 += __uint_as_float(b[i0 + 1]);
            }
            w4[f] = pack_bf16x2(x0, x1);
          }
          o4[c0 / 8 + e] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&bars.acc_empty[ab]);
      if (t < p.n) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int e = 0; e < DP / 8; ++e)
          if (e * 8 < p.d) dst[e] = o4[e];
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, p.tmem_cols);
}

int dpad_of(int d) { return d <= 64 ? 64 : 128; }

struct TokPlan {
  int DP, m_pad, m64, kc, nq, nkw, nt;
  uint32_t q_stage, v_stage, kt_bytes, wt_bytes, t_bytes, tmem_cols;
  size_t smem;
};

bool plan_tokens(const Shape& s, TokPlan* pl) {
  if (s.dtype != NYS_BF16) return false;
  pl->DP = dpad_of(s.d);
  pl->m_pad = ((s.m + 31) / 32) * 32;
  pl->m64 = s.m64();
  pl->kc = s.ks > 0 ? ((128 + s.ks - 1 + 15) / 16) * 16 : 0;
  if (pl->kc > 256 || pl->m_pad > 256) return false;
  pl->q_stage = 128 * pl->DP * 2;
  pl->v_stage = (uint32_t)pl->kc * pl->DP * 2;
  pl->kt_bytes = (uint32_t)pl->m_pad * pl->DP * 2;
  pl->wt_bytes = (uint32_t)((pl->m_pad + 63) / 64) * pl->DP * 128;
  pl->t_bytes = pl->kc > 0 ? (uint32_t)((pl->kc + 63) / 64 + 1) * 8192 : 0;  // compact blocks
  const uint32_t need = 2 * pl->m_pad + 4 * pl->DP;
  if (need > 512) return false;
  uint32_t cols = 32;
  while (cols < need) cols <<= 1;
  pl->tmem_cols = cols;
  const size_t fixed = kNV * (size_t)pl->v_stage + 4 * 128 * 4 + 1024;
  const size_t kw = pl->kt_bytes + pl->wt_bytes;
  // preferred first: three Q stages and two buffers of each per-head block;
  // with one buffer the pipeline drains at a head change
  const int choices[6][3] = {{3, 2, 2}, {3, 2, 1}, {2, 2, 2}, {2, 2, 1}, {3, 1, 1}, {2, 1, 1}};
  for (const auto& ch : choices) {
    const size_t total = fixed + ch[0] * (size_t)pl->q_stage + ch[1] * kw + ch[2] * (size_t)pl->t_bytes;
    if (total <= kSmemBudget) {
      pl->nq = ch[0];
      pl->nkw = ch[1];
      pl->nt = ch[2];
      pl->smem = total;
      return true;
    }
  }
  return false;
}

}  // namespace

// Shared-memory bytes the tensor-core token kernel needs for this shape
// (0 if the shape is outside what it handles).
size_t tokens_tc_smem(const Shape& s) {
  TokPlan pl;
  return plan_tokens(s, &pl) ? pl.smem : 0;
}

int launch_tokens_tc(const Shape& s, const void* q, const void* v, const void* kt_bf16,
                     const void* wt_bf16, const float* conv_w, void* out, int* status,
                     int num_sms, cudaStream_t stream) {
  TokPlan pl;
  if (!plan_tokens(s, &pl)) return NYS_ERR_UNSUPPORTED;
  const uint64_t BH = (uint64_t)s.bh();
  const int DP = pl.DP;

  TokMaps maps;
  {
    const uint64_t dims[3] = {(uint64_t)s.d, (uint64_t)s.n, BH};
    const uint64_t strides[2] = {(uint64_t)s.d * 2, (uint64_t)s.n * s.d * 2};
    const uint32_t boxq[3] = {64, 128, 1};
    const uint32_t boxv[3] = {64, (uint32_t)(pl.kc > 0 ? pl.kc : 16), 1};
    if (!make_tensor_map(&maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, boxq,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, v, dims, strides, boxv,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
  }
  {
    const uint64_t dims[3] = {(uint64_t)DP, (uint64_t)pl.m64, BH};
    const uint64_t strides[2] = {(uint64_t)DP * 2, (uint64_t)pl.m64 * DP * 2};
    const uint32_t box[3] = {64, (uint32_t)pl.m_pad, 1};
    if (!make_tensor_map(&maps.kt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kt_bf16, dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
  }
  {
    const uint64_t dims[3] = {(uint64_t)pl.m64, (uint64_t)DP, BH};
    const uint64_t strides[2] = {(uint64_t)pl.m64 * 2, (uint64_t)pl.m64 * DP * 2};
    const uint32_t box[3] = {64, (uint32_t)DP, 1};
    if (!make_tensor_map(&maps.wt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, wt_bf16, dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
  }

  TokParams p{};
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
  p.nq = pl.nq;
  p.nkw = pl.nkw;
  p.nt = pl.nt;
  p.tiles_per_head = (s.n + 127) / 128;
  p.total_tiles = (int)(BH * p.tiles_per_head);
  const int ctas = std::min(p.total_tiles, num_sms);
  p.tiles_per_cta = (p.total_tiles + ctas - 1) / ctas;
  const int grid = (p.total_tiles + p.tiles_per_cta - 1) / p.tiles_per_cta;
  p.c = (1.0f / sqrtf((float)s.d)) * 1.4426950408889634f;
  p.tmem_cols = pl.tmem_cols;
  p.q_stage = pl.q_stage;
  p.v_stage = pl.v_stage;
  p.kt_bytes = pl.kt_bytes;
  p.wt_bytes = pl.wt_bytes;
  p.t_bytes = pl.t_bytes;
  p.off_q = 0;
  p.off_v = p.nq * p.q_stage;
  p.off_kt = p.off_v + kNV * p.v_stage;
  p.off_t = p.off_kt + p.nkw * (p.kt_bytes + p.wt_bytes);
  p.off_l = p.off_t + p.nt * p.t_bytes;

  auto kern = DP == 64 ? tokens_tc<64> : tokens_tc<128>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem) !=
      cudaSuccess)
    return set_cuda_error(cudaGetLastError());
  KernelScope scope("tokens_tc", stream);
  kern<<<grid, kThreads, pl.smem, stream>>>(maps, p);
  return launch_status();
}

}  // namespace nys
