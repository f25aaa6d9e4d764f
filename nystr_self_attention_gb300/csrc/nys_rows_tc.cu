// Landmark rows on the tensor cores (bf16 inputs, fp32 accumulate):
//   G = softmax(Q~ K^T / sqrt(d)) V
// ("Nyströmformer" review page, Proposed method, bullets 3 and 6), computed
// as partial sums over key ranges: each partial is the unnormalised
// O = sum_j exp(s_ij - M_i) V_j with (M_i, L_i = sum_j exp(s_ij - M_i)); the
// pseudo-inverse kernels merge them. The m x n scores never leave the chip.
//
// Persistent CTAs, one per SM, each take an equal contiguous range of the
// flattened (head, 128-key tile) space; the part of the range inside one
// head is a "unit" and yields that CTA's partial for the head. Two
// softmax warpgroups work in ping-pong on two independent streams of work
// items, each with its own S/P buffer and O accumulator in TMEM:
//   m > 128:  group g = landmark rows [128 g, 128 g + 128): both groups use
//             every K/V tile, so K and V are read once for all m rows;
//   m <= 128: group g = alternate key tiles of the unit; at the unit's end
//             group 0 combines both groups' (max, sum, O) into the one
//             partial.
// Per item (group g, key tile j):
//   S_g = Q~_g K_j^T         tcgen05, A = Q~ (smem), B = K tile (smem)
//   online softmax           thread = landmark row, from TMEM; the running
//                            max is re-based only when it grows by more than
//                            2^8 (O_g is then rescaled in TMEM); P (bf16)
//                            overwrites S_g in TMEM
//   O_g += P_g V_j           tcgen05, A = P (TMEM), B = V tile (MN-major)
// Warps 0-3 / 4-7: softmax groups (and each group's epilogue); warp 8: TMA
// producer (Q~ per unit, K and V tiles through one slot ring); warp 9: TMEM
// owner and issuer of the S products; warp 10: issuer of the P V products
// (a tcgen05.mma costs its issuing thread tens of cycles, so the two
// streams issue from separate threads). S of a group's next item waits for
// the P V that reads its P; one group's softmax overlaps the other group's
// products.
// Every wait is bounded; a wait that runs out sets the status word, every
// role winds down, copies in flight are awaited and TMEM is freed.
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
  CUtensorMap gp;  // gpart as [rows][d] fp32, 32 x 32 boxes (d <= 64)
};

struct RowParams {
  float* gpart;  // [B*H][parts][m][d]
  float* gml;    // [B*H][parts][m][2]: (max in units of scaled scores, sum)
  int* status;
  int n, d, m;
  int n_tiles;     // 128-key tiles per head
  int tpc;         // tiles per CTA range
  int total;       // heads * n_tiles (this launch)
  int parts;       // partials per head in gpart / gml
  int pieces_max;  // CTA ranges that can touch one head
  int big;         // 1: groups are row blocks (m > 128); 0: groups alternate tiles
  int nq, ns;      // Q~ buffers; K/V slots
  float c;         // scale * log2(e)
  float scale;     // 1/sqrt(d)
  const int* lengths;  // per batch entry: keys past it are padding (null: n)
  int H;
};

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRebase = 8.0f;  // re-base the running max when it grows by > 2^8
constexpr int kThreads = 352;
constexpr size_t kSmemBudget = 227 * 1024 - 1024;

struct Bars {
  uint64_t full[8], empty[8];  // K/V slots
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2], o_full[2], o_empty[2];
  uint64_t x_ready;  // m <= 128: group 1's (max, sum) of the unit handed to group 0
  uint64_t fin;
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

// As wait_or_fail, for a whole warp that waits together (a uniform result).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status,
                                          volatile int* abort_flag) {
  return __all_sync(0xffffffffu, wait_or_fail(bar, parity, status, abort_flag));
}

// The part of this CTA's tile range [pos, r1) that lies in one head.
struct Unit {
  int bh, tile0, ntile, piece;
  bool last_piece;  // the unit ends where the head ends
};

__device__ __forceinline__ bool next_unit(const RowParams& p, int& pos, int r1, Unit& u) {
  if (pos >= r1) return false;
  u.bh = pos / p.n_tiles;
  u.tile0 = pos - u.bh * p.n_tiles;
  const int head_end = (u.bh + 1) * p.n_tiles;
  const int e = min(r1, head_end);
  u.ntile = e - pos;
  u.piece = (int)blockIdx.x - (u.bh * p.n_tiles) / p.tpc;
  u.last_piece = e == head_end;
  pos = e;
  return true;
}

// Walks the work items of this CTA in order (used by the issuer twice: the
// S stream runs two items ahead of the P V stream). Ring slots and phase
// parities are tracked incrementally (no division in the issuing thread).
struct Cursor {
  int pos, r1;
  Unit u;
  bool valid;
  int loc, U;     // item within the unit, items in the unit
  int t;          // item index over the CTA
  int unit_no;    // units before this one
  int ks, vs;     // K / V slot of the current tile
  uint32_t kph, vph;  // their full-barrier parities
  __device__ void init(const RowParams& p, int r0, int r1_) {
    pos = r0;
    r1 = r1_;
    valid = next_unit(p, pos, r1, u);
    loc = 0;
    U = valid ? (p.big ? 2 * u.ntile : u.ntile) : 0;
    t = 0;
    unit_no = 0;
    ks = 0;
    vs = 1 % p.ns;
    kph = 0;
    vph = 0u;
  }
  __device__ void next_tile(const RowParams& p) {
    ks += 2;
    if (ks >= p.ns) { ks -= p.ns; kph ^= 1u; }
    vs += 2;
    if (vs >= p.ns) { vs -= p.ns; vph ^= 1u; }
  }
  __device__ void advance(const RowParams& p) {
    if (!p.big || (loc & 1)) next_tile(p);
    ++loc;
    ++t;
    if (loc == U) {
      ++unit_no;
      valid = next_unit(p, pos, r1, u);
      loc = 0;
      U = valid ? (p.big ? 2 * u.ntile : u.ntile) : 0;
    }
  }
  __device__ int group(const RowParams& p) const { return p.big ? (loc & 1) : (t & 1); }
  __device__ bool first_use(const RowParams& p) const { return !p.big || (loc & 1) == 0; }
  __device__ bool last_use(const RowParams& p) const { return !p.big || (loc & 1) == 1; }
  __device__ int qbuf(const RowParams& p) const { return p.nq == 2 ? (unit_no & 1) : 0; }
  __device__ uint32_t qph(const RowParams& p) const {
    return (uint32_t)(p.nq == 2 ? (unit_no >> 1) : unit_no) & 1u;
  }
};

template <int DP>
__global__ void __launch_bounds__(kThreads, 1) rows_tc(const __grid_constant__ RowMaps maps,
                                                       const __grid_constant__ RowParams p) {
  constexpr int DC = DP / 64;
  constexpr uint32_t TILE = DC * 16384;  // one 128-row tile of Q~, K or V, bytes
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const uint32_t qbuf_bytes = (p.big ? 2u : 1u) * TILE;
  // d <= 64: each softmax warp stages its 32 partial rows here (two
  // 32-column SWIZZLE_128B boxes) for a TMA store
  constexpr uint32_t kStageWarp = DP == 64 ? 8192 : 0;
  uint8_t* q_s = sm;                                    // [nq][1 or 2 tiles]
  uint8_t* stage_s = sm + p.nq * qbuf_bytes;            // [8 warps][kStageWarp]
  uint8_t* kv_s = stage_s + 8 * kStageWarp;             // [ns][TILE]
  __shared__ Bars bars;
  __shared__ float xm_s[128], xl_s[128];  // group 1's (max, sum) per row, m <= 128
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  volatile int* abort_flag = &abort_sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = (int)blockIdx.x * p.tpc;
  const int r1 = min(p.total, r0 + p.tpc);

  if (tid == 0) {
    for (int i = 0; i < p.ns; ++i) {
      mbar_init(&bars.full[i], 1);
      mbar_init(&bars.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 128);
      mbar_init(&bars.pv_done[i], 1);
      mbar_init(&bars.o_full[i], 1);
      mbar_init(&bars.o_empty[i], 128);
    }
    mbar_init(&bars.fin, 2);
    mbar_init(&bars.x_ready, 128);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(&tmem_base_sh, 512);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  // TMEM columns: S/P of group g at 128 g; O of group g at 256 + g DP
  constexpr uint32_t COL_O = 256;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (no divergence); lane 0 issues the copies.
    const bool leader = lane == 0;
    if (leader) {
      tma_prefetch(&maps.qt);
      tma_prefetch(&maps.k);
      tma_prefetch(&maps.v);
    }
    int pos = r0, unit_no = 0;
    uint32_t L = 0;     // K/V loads issued
    int slot = 0;       // L % ns
    uint32_t eph = 0;   // (L / ns) & 1
    Unit u;
    bool ok = true;
    while (ok && next_unit(p, pos, r1, u)) {
      const int qb = p.nq == 2 ? (unit_no & 1) : 0;
      const uint32_t qph = (uint32_t)(p.nq == 2 ? (unit_no >> 1) : unit_no) & 1u;
      if (unit_no >= p.nq && !warp_wait(&bars.q_empty[qb], qph ^ 1u, p.status, abort_flag)) {
        ok = false;
        break;
      }
      if (leader) {
        uint8_t* qs = q_s + qb * qbuf_bytes;
        mbar_arrive_expect_tx(&bars.q_full[qb], qbuf_bytes);
        for (int blk = 0; blk < (p.big ? 2 : 1); ++blk)
#pragma unroll
          for (int dc = 0; dc < DC; ++dc)
            tma_load_3d(qs + blk * TILE + dc * 16384, &maps.qt, &bars.q_full[qb], dc * 64, blk * 128, u.bh);
      }
      ++unit_no;
      for (int tl = 0; tl < u.ntile && ok; ++tl) {
        for (int kind = 0; kind < 2; ++kind, ++L) {
          const int s = slot;
          if (L >= (uint32_t)p.ns && !warp_wait(&bars.empty[s], eph ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          if (++slot == p.ns) {
            slot = 0;
            eph ^= 1u;
          }
          if (leader) {
            uint8_t* dst = kv_s + s * TILE;
            mbar_arrive_expect_tx(&bars.full[s], TILE);
#pragma unroll
            for (int dc = 0; dc < DC; ++dc)
              tma_load_3d(dst + dc * 16384, kind ? &maps.v : &maps.k, &bars.full[s], dc * 64,
                          (u.tile0 + tl) * 128, u.bh);
          }
        }
      }
    }
    if (*abort_flag && leader) {
      // wait (bounded) for this warp's copies still in flight
      for (int s = 0; s < p.ns; ++s) {
        const uint32_t cnt = L > (uint32_t)s ? (L - s + p.ns - 1) / p.ns : 0;
        if (cnt) mbar_wait(&bars.full[s], (cnt - 1) & 1, nullptr, kWaitNs);
      }
      for (int qb = 0; qb < p.nq; ++qb) {
        const int cnt = unit_no > qb ? (unit_no - qb + p.nq - 1) / p.nq : 0;
        if (cnt) mbar_wait(&bars.q_full[qb], (cnt - 1) & 1, nullptr, kWaitNs);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ---------------------------------------------- MMA issuer, S stream
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, 128, false, false);
      Cursor cs;
      cs.init(p, r0, r1);
      uint32_t sc0 = 0, sc1 = 0;  // S products issued per group
      while (cs.valid) {
        const int g = cs.group(p);
        const int qb = cs.qbuf(p);
        const uint32_t sc = g ? sc1 : sc0;
        if (cs.loc == 0 && !wait_or_fail(&bars.q_full[qb], cs.qph(p), p.status, abort_flag)) break;
        const int sk = cs.ks;
        if (cs.first_use(p) && !wait_or_fail(&bars.full[sk], cs.kph, p.status, abort_flag)) break;
        // S_g is P_g of the group's previous item until that item's P V is done
        if (sc > 0 && !wait_or_fail(&bars.pv_done[g], (sc - 1) & 1, p.status, abort_flag)) break;
        tc_fence_after_sync();
        const uint64_t a0 = smem_desc(smem_u32(q_s + qb * qbuf_bytes + (p.big ? g * TILE : 0)), 16, 1024, SW_128B);
        const uint64_t b0 = smem_desc(smem_u32(kv_s + sk * TILE), 16, 1024, SW_128B);
        const uint32_t dS = tmem + 128 * g;
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk) {
          const uint64_t off = (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2);  // (16 KB chunk, 32 B step) >> 4
          mma_bf16(dS, a0 + off, b0 + off, id_s, kk > 0);
        }
        mma_commit(&bars.s_full[g]);
        if (cs.last_use(p)) mma_commit(&bars.empty[sk]);
        if (cs.loc == cs.U - 1) mma_commit(&bars.q_empty[qb]);
        if (g) ++sc1; else ++sc0;
        cs.advance(p);
      }
      // no MMA of this thread may be in flight when TMEM is freed
      mma_commit(&bars.fin);
    }
  } else if (warp == 10) {
    // -------------------------------------------- MMA issuer, P V stream
    if (lane == 0) {
      const uint32_t id_pv = idesc_bf16(128, DP, false, true);
      Cursor cp;
      cp.init(p, r0, r1);
      uint32_t pcnt0 = 0, pcnt1 = 0;
      bool had0 = false, had1 = false;  // group has had a P V in the current unit
      while (cp.valid) {
        const int g = cp.group(p);
        const uint32_t pc = g ? pcnt1 : pcnt0;
        const bool had = g ? had1 : had0;
        if (!wait_or_fail(&bars.p_full[g], pc & 1, p.status, abort_flag)) break;
        if (!had && cp.unit_no > 0 &&
            !wait_or_fail(&bars.o_empty[g], (cp.unit_no - 1) & 1, p.status, abort_flag))
          break;
        const int sv = cp.vs;
        if (cp.first_use(p) && !wait_or_fail(&bars.full[sv], cp.vph, p.status, abort_flag)) break;
        const bool unit_end = cp.loc == cp.U - 1;
        // at the end of a unit, a group without a P V in it hands its
        // (empty) accumulator over too: wait for its previous epilogue
        if (unit_end && cp.unit_no > 0) {
          if (!had0 && g != 0 && !wait_or_fail(&bars.o_empty[0], (cp.unit_no - 1) & 1, p.status, abort_flag)) break;
          if (!had1 && g != 1 && !wait_or_fail(&bars.o_empty[1], (cp.unit_no - 1) & 1, p.status, abort_flag)) break;
        }
        tc_fence_after_sync();
        const uint64_t v0 = smem_desc(smem_u32(kv_s + sv * TILE), 16384, 1024, SW_128B);
        const uint32_t dO = tmem + COL_O + g * DP, aP = tmem + 128 * g;
        mma_bf16_tA(dO, aP, v0, id_pv, had ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < 8; ++kk)  // 16 keys = 2 KB of V, 8 TMEM columns of P
          mma_bf16_tA(dO, aP + kk * 8, v0 + (uint64_t)(kk * 128), id_pv, 1u);
        mma_commit(&bars.pv_done[g]);
        if (cp.last_use(p)) mma_commit(&bars.empty[sv]);
        if (unit_end) {
          // unit done: both groups' accumulators go to their epilogues
          mma_commit(&bars.o_full[0]);
          mma_commit(&bars.o_full[1]);
        }
        if (g) { ++pcnt1; had1 = true; } else { ++pcnt0; had0 = true; }
        if (unit_end) had0 = had1 = false;
        cp.advance(p);
      }
      mma_commit(&bars.fin);
    }
  } else {
    // ---------------------------------------------- softmax group g
    const int g = warp >> 2;
    const int lr = (warp & 3) * 32 + lane;  // TMEM lane = row of the group's block
    const uint32_t lo = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t scol = tmem + lo + 128 * g;
    const uint32_t ocol = tmem + lo + COL_O + g * DP;
    const int row = p.big ? 128 * g + lr : lr;
    const bool live = row < p.m;
    const bool warp_live = __any_sync(0xffffffffu, live);
    const bool warp_all_live = __all_sync(0xffffffffu, live);
    uint32_t cnt_s = 0, cnt_o = 0;
    int pos = r0, tglob = 0;
    Unit u;
    while (next_unit(p, pos, r1, u)) {
      const int U = p.big ? 2 * u.ntile : u.ntile;
      // keys of this head: padding past its length gives P = 0 (a tile that
      // lies wholly in the padding leaves the running max at -inf)
      const int nk = p.lengths ? p.lengths[u.bh / p.H] : p.n;
      float m_run = -INFINITY, l_run = 0.f;
      int mine = 0;
      bool ok = true;
      for (int t = tglob + ((g - tglob) & 1); t < tglob + U; t += 2) {
        const int local = t - tglob;
        const int key0 = (u.tile0 + (p.big ? (local >> 1) : local)) * 128;
        if (!__all_sync(0xffffffffu, wait_or_fail(&bars.s_full[g], cnt_s & 1, p.status, abort_flag))) {
          ok = false;
          break;
        }
        ++cnt_s;
        tc_fence_after_sync();
        if (warp_live) {
          // tile max: all four column chunks of S in flight at once; on a
          // full tile of live rows the chunks stay in registers for the
          // exponentials (S is read from TMEM once)
          float tmax = -INFINITY;
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32(scol, r0);
          tmem_ld32(scol + 32, r1);
          tmem_ld32(scol + 64, r2);
          tmem_ld32(scol + 96, r3);
          tmem_ld_wait();
          const bool fast = warp_all_live && key0 + 128 <= nk;  // warp-uniform
          if (key0 + 128 <= nk) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              tmax = fmaxf(tmax, fmaxf(fmaxf(__uint_as_float(r0[e]), __uint_as_float(r1[e])),
                                       fmaxf(__uint_as_float(r2[e]), __uint_as_float(r3[e]))));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              if (key0 + e < nk) tmax = fmaxf(tmax, __uint_as_float(r0[e]));
              if (key0 + 32 + e < nk) tmax = fmaxf(tmax, __uint_as_float(r1[e]));
              if (key0 + 64 + e < nk) tmax = fmaxf(tmax, __uint_as_float(r2[e]));
              if (key0 + 96 + e < nk) tmax = fmaxf(tmax, __uint_as_float(r3[e]));
            }
          }
          const bool rebase = live && (m_run == -INFINITY || (tmax - m_run) * p.c > kRebase);
          float alpha = 1.f;
          if (rebase) {
            alpha = (m_run == -INFINITY) ? 0.f : fast_exp2((m_run - tmax) * p.c);
            l_run *= alpha;
            m_run = tmax;
          }
          const float mc = m_run * p.c;
          if (fast) {
            // P = 2^(S c - M c), no masks, from the registers; P of chunk c
            // goes to columns c0 / 2 .. (already read)
            auto exp_chunk = [&](int c0, const uint32_t (&r)[32]) {
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float a = fast_exp2(fmaf(__uint_as_float(r[2 * e]), p.c, -mc));
                const float b = fast_exp2(fmaf(__uint_as_float(r[2 * e + 1]), p.c, -mc));
                l_run += a + b;
                pk[e] = pack_bf16x2(a, b);
              }
              tmem_st16(scol + (c0 >> 1), pk);
            };
            exp_chunk(0, r0);
            exp_chunk(32, r1);
            exp_chunk(64, r2);
            exp_chunk(96, r3);
          } else if (key0 >= nk) {
            // a tile wholly past the head's keys (padding): P = 0
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = 0u;
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32) tmem_st16(scol + (c0 >> 1), pk);
          } else {
            // padding rows and keys past the end give P = 0
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
              uint32_t r[32];
              tmem_ld32(scol + c0, r);
              tmem_ld_wait();
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int ka = key0 + c0 + 2 * e;
                const float a = (live && ka < nk) ? fast_exp2(fmaf(__uint_as_float(r[2 * e]), p.c, -mc)) : 0.f;
                const float b = (live && ka + 1 < nk) ? fast_exp2(fmaf(__uint_as_float(r[2 * e + 1]), p.c, -mc)) : 0.f;
                l_run += a + b;
                pk[e] = pack_bf16x2(a, b);
              }
              tmem_st16(scol + (c0 >> 1), pk);
            }
          }
          if (mine > 0 && __any_sync(0xffffffffu, rebase)) {
            // rescale the accumulator rows before this item's P V (the
            // group's earlier P V are done: S of this item waited for them)
#pragma unroll 1
            for (int c0 = 0; c0 < DP; c0 += 32) {
              uint32_t r[32];
              tmem_ld32(ocol + c0, r);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tmem_st32(ocol + c0, r);
            }
          }
          tmem_st_wait();
        }
        // warps whose rows are all padding leave P as it is: those rows of
        // O are never read
        tc_fence_before_sync();
        mbar_arrive(&bars.p_full[g]);
        ++mine;
      }
      if (!ok) break;
      // epilogue of this unit: one partial O (unnormalised), max, sum. For
      // m > 128 each group writes its rows; for m <= 128 the two groups
      // covered alternate key tiles of the same rows: group 1 hands its
      // (max, sum) to group 0, which writes the combined partial and frees
      // both accumulators. A unit without items writes (max, sum) = (-inf,
      // 0): the merges skip such partials.
      if (!__all_sync(0xffffffffu, wait_or_fail(&bars.o_full[g], cnt_o & 1, p.status, abort_flag))) break;
      ++cnt_o;
      tc_fence_after_sync();
      if (!p.big && g == 1) {
        xm_s[lr] = mine > 0 ? m_run : -INFINITY;
        xl_s[lr] = mine > 0 ? l_run : 0.f;
        mbar_arrive(&bars.x_ready);
        tglob += U;
        continue;
      }
      float m_out = mine > 0 ? m_run : -INFINITY, l_out = mine > 0 ? l_run : 0.f;
      float a0 = 1.f, a1 = 0.f;  // weights of this group's and group 1's O
      if (!p.big) {
        if (!__all_sync(0xffffffffu, wait_or_fail(&bars.x_ready, (cnt_o - 1) & 1, p.status, abort_flag))) break;
        const float m1 = xm_s[lr], l1 = xl_s[lr];
        const float mx = fmaxf(m_out, m1);
        a0 = m_out == -INFINITY ? 0.f : fast_exp2((m_out - mx) * p.c);
        a1 = m1 == -INFINITY ? 0.f : fast_exp2((m1 - mx) * p.c);
        l_out = l_out * a0 + l1 * a1;
        m_out = mx;
      }
      const uint32_t ocol1 = tmem + lo + COL_O + DP;  // group 1's O, same rows
      // combined chunk of O: a0 O_g + a1 O_1 (a zero weight drops its term,
      // whatever an accumulator without items holds)
      auto o_chunk = [&](int c0, uint32_t (&r)[32]) {
        tmem_ld32(ocol + c0, r);
        if (!p.big) {
          uint32_t r1[32];
          tmem_ld32(ocol1 + c0, r1);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float x0 = a0 != 0.f ? a0 * __uint_as_float(r[e]) : 0.f;
            const float x1 = a1 != 0.f ? a1 * __uint_as_float(r1[e]) : 0.f;
            r[e] = __float_as_uint(x0 + x1);
          }
        } else {
          tmem_ld_wait();
        }
      };
      const int part = u.piece;
      const size_t prow = ((size_t)u.bh * p.parts + part) * p.m + row;
      if (warp_live && __any_sync(0xffffffffu, m_out != -INFINITY)) {
        if (kStageWarp > 0 && warp_all_live) {
          uint8_t* st = stage_s + warp * kStageWarp;
          if (lane == 0) bulk_wait_read0();  // this warp's previous store has read st
          __syncwarp();
#pragma unroll
          for (int b = 0; b < DP / 32; ++b) {
            uint32_t r[32];
            o_chunk(32 * b, r);
            uint8_t* box = st + b * 4096 + lane * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(box + ((c ^ (lane & 7)) << 4)) =
                  make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            for (int b = 0; b < DP / 32; ++b)
              if (32 * b < p.d) tma_store_2d(&maps.gp, st + b * 4096, 32 * b, (int)prow);
            bulk_commit();
          }
        } else {
          float* o = p.gpart + prow * p.d;
#pragma unroll
          for (int c0 = 0; c0 < DP; c0 += 32) {
            uint32_t r[32];
            o_chunk(c0, r);
            if (live && c0 < p.d) {
              float4* dst = reinterpret_cast<float4*>(o + c0);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                     __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&bars.o_empty[g]);
      if (!p.big) mbar_arrive(&bars.o_empty[1]);  // group 1's accumulator, read above
      if (live) {
        p.gml[prow * 2 + 0] = m_out * p.scale;  // -inf for an empty partial
        p.gml[prow * 2 + 1] = l_out;
      }
      // the head's last range also marks the partial slots no range uses
      if (u.last_piece && live) {
        for (int pc = u.piece + 1; pc < p.pieces_max; ++pc) {
          const size_t prow2 = ((size_t)u.bh * p.parts + pc) * p.m + row;
          p.gml[prow2 * 2 + 0] = -INFINITY;
          p.gml[prow2 * 2 + 1] = 0.f;
        }
      }
      tglob += U;
    }
    if (kStageWarp > 0 && lane == 0) bulk_wait0();  // staged stores done before exit
  }
  // both issuing threads have committed to fin: once it completes, no MMA
  // of this CTA is in flight
  if (warp == 9 && lane == 0) mbar_wait(&bars.fin, 0, nullptr, kWaitNs);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

int nq_of(const Shape& s) { return s.m > 128 ? 1 : 2; }

}  // namespace

// Ranges of the tensor-core landmark-row kernel (host math): every CTA of a
// full-GPU launch gets tiles_per_cta consecutive tiles of the flattened
// (head, tile) space; a head is touched by at most pieces ranges, each giving
// one partial.
void rows_tc_split(const Shape& s, int ctas, int* parts, int* tiles_per_cta) {
  const long long kCtas = ctas > 0 ? ctas : 1;
  const long long n_tiles = (s.n + 127) / 128;
  const long long total = n_tiles * s.bh();
  long long tpc = (total + kCtas - 1) / kCtas;
  if (tpc < 1) tpc = 1;
  long long pieces = (n_tiles + tpc - 1) / tpc + 1;
  if (pieces > n_tiles) pieces = n_tiles;
  *tiles_per_cta = (int)tpc;
  *parts = (int)pieces;
}

int launch_rows_tc(const Shape& s, const void* qt_bf16, const void* k, const void* v, float* gpart,
                   float* gml, int parts, int tiles_per_cta, int* status, cudaStream_t stream) {
  if (s.m > 256) return NYS_ERR_UNSUPPORTED;
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
      return tensor_map_error(__FILE__, __LINE__);
  }
  {
    const uint64_t dims[3] = {(uint64_t)s.d, (uint64_t)s.n, BH};
    const uint64_t strides[2] = {(uint64_t)s.d * 2, (uint64_t)s.n * s.d * 2};
    const uint32_t box[3] = {64, 128, 1};
    if (!make_tensor_map(&maps.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, v, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
  }
  if (DP == 64) {
    const uint64_t dims[2] = {(uint64_t)s.d, BH * (uint64_t)parts * (uint64_t)s.m};
    const uint64_t strides[1] = {(uint64_t)s.d * 4};
    const uint32_t box[2] = {32, 32};
    if (!make_tensor_map(&maps.gp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, gpart, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return tensor_map_error(__FILE__, __LINE__);
  }
  RowParams p{};
  p.gpart = gpart;
  p.gml = gml;
  p.status = status;
  p.n = s.n;
  p.d = s.d;
  p.m = s.m;
  p.n_tiles = (s.n + 127) / 128;
  p.tpc = tiles_per_cta;
  p.total = (int)(BH * p.n_tiles);
  p.parts = parts;
  p.big = s.m > 128 ? 1 : 0;
  p.pieces_max = parts;
  p.scale = 1.0f / sqrtf((float)s.d);
  p.c = p.scale * 1.4426950408889634f;
  p.lengths = s.lengths;
  p.H = s.H;
  const size_t tile = (size_t)(DP / 64) * 16384;
  p.nq = nq_of(s);
  const size_t qbytes = (size_t)p.nq * (p.big ? 2 : 1) * tile;
  const size_t stage = DP == 64 ? 8 * 8192 : 0;
  size_t ns = (kSmemBudget - qbytes - stage) / tile;
  if (ns > 8) ns = 8;
  if (ns < 2) return NYS_ERR_UNSUPPORTED;
  p.ns = (int)ns;
  const size_t smem = qbytes + stage + ns * tile + 1024;
  const int grid = (p.total + p.tpc - 1) / p.tpc;
  auto kern = DP == 64 ? rows_tc<64> : rows_tc<128>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return set_cuda_error(cudaGetLastError());
  KernelScope scope("rows_tc", stream);
  kern<<<grid, kThreads, smem, stream>>>(maps, p);
  return launch_status();
}

}  // namespace nys
