// Clustered attention, centroid path ("Fast Transformers with Clustered
// Attention" review page, Proposed method, bullets 1, 2 and 4): per head the
// queries are grouped by K-means, attention is computed once per centroid
// and every query receives its cluster's row:
//   mu    = segment means of Q over C segments (initial centroids)
//   iters x:  a(i) = argmin_c |q_i - mu_c|^2   (ties: lowest c)
//             mu_c = mean of {q_i : a(i) = c}  (no member: unchanged)
//   G     = softmax(mu K^T / sqrt(d)) V        (C x d, key-split online softmax)
//   out_i = G[a(i)]
// It shares the Nyström path's kernels for the segment means and for
// softmax(. K^T s) V (the landmark-row kernels with the centroids in place of
// the landmarks, then the merge of the key-split partials). K-means runs on
// the tensor cores for bf16 queries with d in {64, 128} and C <= 128
// (nys_kmeans_tc.cu: the distances to fp32 accuracy, the members' sums as a
// one-hot product, deterministic), and otherwise in the CUDA-core kernels
// below in fp32 (the update sums a cluster's queries in index order). The
// broadcast is a CUDA-core kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nys_internal.h"

namespace nys {
namespace {

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

constexpr int kAssignThreads = 128;
constexpr int kTileC = 32;  // centroids per shared-memory tile

// grid (ceil(n / 128), B*H), block 128: thread = query. The query row sits
// in registers (DM >= d columns, zero past d); tiles of 32 centroids and
// their squared norms are staged in shared memory. The nearest centroid
// minimises |mu_c|^2 - 2 q . mu_c (|q|^2 is common to all c): one FMA per
// element.
template <typename T, int DM>
__global__ void __launch_bounds__(kAssignThreads)
kmeans_assign(const T* __restrict__ q, const float* __restrict__ mu, int* __restrict__ assign,
              int n, int d, int C) {
  __shared__ __align__(16) float smu[kTileC * DM];
  __shared__ float snorm[kTileC];
  const long long bh = blockIdx.y;
  const int t = blockIdx.x * kAssignThreads + threadIdx.x;
  const bool ok = t < n;
  float qr[DM];
  const T* qrow = q + ((size_t)bh * n + (ok ? t : 0)) * d;
#pragma unroll
  for (int j = 0; j < DM; ++j) qr[j] = (ok && j < d) ? ldf(qrow + j) : 0.f;
  const float* mh = mu + (size_t)bh * C * d;
  float best = INFINITY;
  int best_c = 0;
  for (int c0 = 0; c0 < C; c0 += kTileC) {
    const int nc = min(kTileC, C - c0);
    __syncthreads();
    for (int e = threadIdx.x; e < kTileC * DM; e += kAssignThreads) {
      const int c = e / DM, j = e % DM;
      smu[e] = (c < nc && j < d) ? mh[(size_t)(c0 + c) * d + j] : 0.f;
    }
    __syncthreads();
    if (threadIdx.x < kTileC) {
      float nrm = 0.f;
      for (int j = 0; j < DM; ++j) nrm = fmaf(smu[threadIdx.x * DM + j], smu[threadIdx.x * DM + j], nrm);
      snorm[threadIdx.x] = nrm;
    }
    __syncthreads();
    for (int c = 0; c < nc; ++c) {
      const float4* m = reinterpret_cast<const float4*>(smu + c * DM);
      float dot0 = 0.f, dot1 = 0.f;
#pragma unroll
      for (int j = 0; j < DM / 4; ++j) {
        const float4 mv = m[j];
        dot0 = fmaf(qr[4 * j], mv.x, dot0);
        dot1 = fmaf(qr[4 * j + 1], mv.y, dot1);
        dot0 = fmaf(qr[4 * j + 2], mv.z, dot0);
        dot1 = fmaf(qr[4 * j + 3], mv.w, dot1);
      }
      const float score = fmaf(-2.f, dot0 + dot1, snorm[c]);
      if (score < best) {  // strict: a tie keeps the lower index
        best = score;
        best_c = c0 + c;
      }
    }
  }
  if (ok) assign[(size_t)bh * n + t] = best_c;
}

constexpr int kUpdThreads = 128;

// grid (C, B*H), block 128: CTA = one cluster of one head. 128 assignments
// at a time: each warp ballots which of its 32 queries belong to the
// cluster; then thread j (j < d) adds column j of the members in index order
// (reproducible). The new centroid is the mean, or the old centroid for an
// empty cluster.
template <typename T>
__global__ void __launch_bounds__(kUpdThreads)
kmeans_update(const T* __restrict__ q, const int* __restrict__ assign,
              const float* __restrict__ mu_old, float* __restrict__ mu_new, int n, int d, int C) {
  __shared__ uint32_t masks[kUpdThreads / 32];
  const int c = blockIdx.x;
  const long long bh = blockIdx.y;
  const int j = threadIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int* ah = assign + (size_t)bh * n;
  const T* qh = q + (size_t)bh * n * d;
  float s = 0.f;
  int cnt = 0;
  for (int i0 = 0; i0 < n; i0 += kUpdThreads) {
    const int i = i0 + threadIdx.x;
    const bool member = i < n && __ldg(ah + i) == c;
    const uint32_t mk = __ballot_sync(0xffffffffu, member);
    __syncthreads();  // the previous chunk's masks have been read
    if (lane == 0) masks[warp] = mk;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kUpdThreads / 32; ++w) {
      uint32_t b = masks[w];
      cnt += __popc(b);
      while (b) {
        const int bit = __ffs(b) - 1;
        b &= b - 1;
        if (j < d) s += ldf(qh + (size_t)(i0 + 32 * w + bit) * d + j);
      }
    }
  }
  if (j < d) {
    const size_t o = ((size_t)bh * C + c) * d + j;
    mu_new[o] = cnt > 0 ? s / (float)cnt : mu_old[o];
  }
}

// bf16 copy of the centroids, [B*H][m64][dpad], zero padded: the A operand of
// the tensor-core landmark-row kernel. grid (m64, B*H), block dpad.
__global__ void pack_centroids(const float* __restrict__ mu, __nv_bfloat16* __restrict__ mb, int C,
                               int d, int m64, int dpad) {
  const int c = blockIdx.x, j = threadIdx.x;
  const long long bh = blockIdx.y;
  const float x = (c < C && j < d) ? mu[((size_t)bh * C + c) * d + j] : 0.f;
  mb[((size_t)bh * m64 + c) * dpad + j] = __float2bfloat16_rn(x);
}

// out[i] = G[a(i)]. One thread per 8 elements (d % 8 == 0: one 16-byte
// store in bf16, two in fp32); grid (ceil(n d / 8 / 256), B*H).
template <typename T>
__global__ void __launch_bounds__(256)
broadcast_rows(const float* __restrict__ g, const int* __restrict__ assign, T* __restrict__ out,
               int n, int d, int C) {
  const long long bh = blockIdx.y;
  const int e = blockIdx.x * 256 + threadIdx.x;  // group of 8 elements of this head
  const int d8 = d / 8;
  if (e >= n * d8) return;
  const int i = e / d8, j = (e - i * d8) * 8;
  const int a = __ldg(assign + (size_t)bh * n + i);
  const float4* src = reinterpret_cast<const float4*>(g + ((size_t)bh * C + a) * d + j);
  const float4 x0 = __ldg(src), x1 = __ldg(src + 1);
  T* o = out + ((size_t)bh * n + i) * d + j;
  if constexpr (sizeof(T) == 4) {
    reinterpret_cast<float4*>(o)[0] = x0;
    reinterpret_cast<float4*>(o)[1] = x1;
  } else {
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(x0.x, x0.y), h1 = __floats2bfloat162_rn(x0.z, x0.w);
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(x1.x, x1.y), h3 = __floats2bfloat162_rn(x1.z, x1.w);
    uint4 u;
    u.x = *reinterpret_cast<const uint32_t*>(&h0);
    u.y = *reinterpret_cast<const uint32_t*>(&h1);
    u.z = *reinterpret_cast<const uint32_t*>(&h2);
    u.w = *reinterpret_cast<const uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(o) = u;
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct ClusteredLayout {
  Layout attn;  // the landmark-row partials, G, the status word, scratch
  size_t assign, mu_a, mu_b, total;
  bool tc;                          // K-means on the tensor cores
  size_t mu3, norms, part, cnt;     // its workspace (tc only)
};

ClusteredLayout clustered_layout(const Shape& s) {
  ClusteredLayout L{};
  L.attn = make_layout(s);
  size_t off = L.attn.total;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
  L.assign = take((size_t)s.bh() * s.n * 4);
  L.mu_a = take((size_t)s.bh() * s.m * s.d * 4);
  L.mu_b = take((size_t)s.bh() * s.m * s.d * 4);
  L.tc = kmeans_tc_supported(s);
  if (L.tc) {
    const KmWorkspace w = kmeans_tc_workspace(s);
    L.mu3 = take(w.mu3_bytes);
    L.norms = take(w.norm_bytes);
    L.part = take(w.part_bytes);
    L.cnt = take(w.cnt_bytes);
  }
  L.total = off;
  return L;
}

template <typename T, int DM>
int launch_assign(const Shape& s, const void* q, const float* mu, int* assign, cudaStream_t st) {
  KernelScope scope("kmeans_assign", st);
  kmeans_assign<T, DM><<<dim3((s.n + kAssignThreads - 1) / kAssignThreads, (unsigned)s.bh()),
                         kAssignThreads, 0, st>>>(static_cast<const T*>(q), mu, assign, s.n, s.d,
                                                  s.m);
  return launch_status();
}

template <typename T>
int assign_t(const Shape& s, const void* q, const float* mu, int* assign, cudaStream_t st) {
  if (s.d <= 32) return launch_assign<T, 32>(s, q, mu, assign, st);
  if (s.d <= 64) return launch_assign<T, 64>(s, q, mu, assign, st);
  return launch_assign<T, 128>(s, q, mu, assign, st);
}

template <typename T>
int update_t(const Shape& s, const void* q, const int* assign, const float* mu_old, float* mu_new,
             cudaStream_t st) {
  KernelScope scope("kmeans_update", st);
  kmeans_update<T><<<dim3((unsigned)s.m, (unsigned)s.bh()), kUpdThreads, 0, st>>>(
      static_cast<const T*>(q), assign, mu_old, mu_new, s.n, s.d, s.m);
  return launch_status();
}

template <typename T>
int broadcast_t(const Shape& s, const float* g, const int* assign, void* out, cudaStream_t st) {
  const int groups = s.n * (s.d / 8);
  KernelScope scope("broadcast_rows", st);
  broadcast_rows<T><<<dim3((groups + 255) / 256, (unsigned)s.bh()), 256, 0, st>>>(
      g, assign, static_cast<T*>(out), s.n, s.d, s.m);
  return launch_status();
}

int check_clustered(int B, int H, int n, int d, int C, int iters, int dtype) {
  const int rc = check_shape(B, H, n, d, C, 0, 0, dtype);
  if (rc != NYS_OK) return rc;
  if (iters < 1 || iters > 64) return NYS_ERR_SHAPE;
  return NYS_OK;
}

}  // namespace
}  // namespace nys

using namespace nys;

extern "C" {

size_t nystrom_clustered_workspace_bytes(int B, int H, int n, int d, int C, int dtype) {
  if (check_clustered(B, H, n, d, C, 1, dtype) != NYS_OK) return 0;
  return clustered_layout(Shape{B, H, n, d, C, 0, 0, dtype}).total;
}

long long nystrom_clustered_stage_offset(int B, int H, int n, int d, int C, int iters, int dtype,
                                         int stage) {
  if (check_clustered(B, H, n, d, C, iters, dtype) != NYS_OK) return -1;
  const ClusteredLayout L = clustered_layout(Shape{B, H, n, d, C, 0, 0, dtype});
  // the centroids alternate between the two buffers, starting in mu_a
  const size_t last = (iters & 1) ? L.mu_b : L.mu_a;
  const size_t prev = (iters & 1) ? L.mu_a : L.mu_b;
  switch (stage) {
    case NYS_CSTAGE_ASSIGN: return (long long)L.assign;
    case NYS_CSTAGE_CENTROIDS_PREV: return (long long)prev;
    case NYS_CSTAGE_CENTROIDS: return (long long)last;
    case NYS_CSTAGE_G: return (long long)L.attn.g;
    default: return -1;
  }
}

int nystrom_clustered_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int H,
                               int n, int d, int C, int iters, int dtype, void* workspace,
                               size_t ws_bytes, nys_stream_t stream) {
  if (!q || !k || !v || !out) return NYS_ERR_ARG;
  int rc = check_clustered(B, H, n, d, C, iters, dtype);
  if (rc != NYS_OK) return rc;
  const uintptr_t a = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                      reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out);
  if (a & 15u) return NYS_ERR_ALIGN;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return NYS_ERR_ALIGN;
  const Shape s{B, H, n, d, C, 0, 0, dtype};
  const ClusteredLayout L = clustered_layout(s);
  if (workspace && ws_bytes < L.total) return NYS_ERR_NOMEM;
  int dev = 0;
  rc = check_device(&dev);
  if (rc != NYS_OK) return rc;
  char* ws = static_cast<char*>(workspace);
  if (!ws) {
    ws = static_cast<char*>(cached_workspace(dev, L.total, stream, &rc));
    if (!ws) return rc;
  }
  rc = begin_call(ws, L.attn, stream, dev);
  if (rc != NYS_OK) return rc;
  const bool bf16 = dtype == NYS_BF16;
  auto at = [&](size_t off) { return ws + off; };
  float* mu[2] = {reinterpret_cast<float*>(at(L.mu_a)), reinterpret_cast<float*>(at(L.mu_b))};
  int* assign = reinterpret_cast<int*>(at(L.assign));
  // initial centroids: segment means of Q (K is not read)
  rc = launch_landmarks(s, q, nullptr, mu[0], nullptr, nullptr, nullptr, stream);
  if (rc != NYS_OK) return error_in("initial centroids", rc);
  int* status = reinterpret_cast<int*>(at(L.attn.status));
  int cur = 0;
  if (L.tc) {
    void* mu3 = at(L.mu3);
    float* norms = reinterpret_cast<float*>(at(L.norms));
    rc = launch_kmeans_prep(s, mu[0], mu3, norms, stream);
    if (rc != NYS_OK) return error_in("K-means set-up", rc);
    for (int it = 0; it < iters; ++it) {
      rc = launch_kmeans_round_tc(s, q, mu3, norms, assign, reinterpret_cast<float*>(at(L.part)),
                                  reinterpret_cast<int*>(at(L.cnt)), mu[cur], mu[cur ^ 1], norms, mu3,
                                  status, stream);
      if (rc != NYS_OK) return error_in("K-means round", rc);
      cur ^= 1;
    }
  } else {
    for (int it = 0; it < iters; ++it) {
      rc = bf16 ? assign_t<__nv_bfloat16>(s, q, mu[cur], assign, stream)
                : assign_t<float>(s, q, mu[cur], assign, stream);
      if (rc != NYS_OK) return error_in("K-means assignment", rc);
      rc = bf16 ? update_t<__nv_bfloat16>(s, q, assign, mu[cur], mu[cur ^ 1], stream)
                : update_t<float>(s, q, assign, mu[cur], mu[cur ^ 1], stream);
      if (rc != NYS_OK) return error_in("K-means update", rc);
      cur ^= 1;
    }
  }
  // G = softmax(mu K^T / sqrt(d)) V with the centroids as the landmark rows
  float* gp = reinterpret_cast<float*>(at(L.attn.g_part));
  float* gml = reinterpret_cast<float*>(at(L.attn.g_ml));
  float* g = reinterpret_cast<float*>(at(L.attn.g));
  if (bf16) {
    __nv_bfloat16* mb = reinterpret_cast<__nv_bfloat16*>(at(L.attn.qt_bf16));
    {
      KernelScope scope("pack_centroids", stream);
      pack_centroids<<<dim3((unsigned)s.m64(), (unsigned)s.bh()), s.dpad(), 0, stream>>>(
          mu[cur], mb, C, d, s.m64(), s.dpad());
      rc = launch_status();
    }
    if (rc != NYS_OK) return error_in("centroid packing", rc);
    rc = launch_rows_tc(s, mb, k, v, gp, gml, L.attn.splits, L.attn.tiles_per_split, status, stream);
  } else {
    rc = launch_rows_simt(s, mu[cur], k, v, gp, gml, L.attn.splits, stream);
  }
  if (rc != NYS_OK) return error_in("centroid rows", rc);
  rc = launch_merge_g(s, gp, gml, g, L.attn.splits, stream);
  if (rc != NYS_OK) return error_in("merge of G", rc);
  rc = bf16 ? broadcast_t<__nv_bfloat16>(s, g, assign, out, stream)
            : broadcast_t<float>(s, g, assign, out, stream);
  return error_in("broadcast", rc);
}

}  // extern "C"
