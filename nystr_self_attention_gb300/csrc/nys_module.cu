// The multi-head attention module around the Nyström attention op: the
// projections in and out that the "Nyströmformer" review page's model wraps
// around it (abstract; Proposed method, bullet 6: Nyström self-attention in
// place of softmax attention in a Transformer layer):
//   [Q | K | V] = X W_qkv + b_qkv        X [B][n][D], D = H d
//   Q, K, V    -> heads [B][H][n][d]      (columns h d .. h d + d - 1 of each)
//   O_h        = Nyström attention of head h (include/nystrom.h)
//   Y          = [O_1 | ... | O_H] W_o + b_o
// The two projections are plain dense GEMMs and run in cuBLAS (fp32
// accumulation, fp32 output into the workspace); the bias, the head split
// and merge (layout changes that HBM bounds) and the attention run in this
// library's kernels.
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "nys_internal.h"

namespace nys {
namespace {

constexpr int kMaxDevices = 64;

template <typename T>
__device__ __forceinline__ void store4(T* p, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float a, float b, float c,
                                                      float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// qkv [B*n][3][H][d] fp32 (+ bias [3][H][d]) -> q, k, v [B][H][n][d] in T.
// One thread per 4 consecutive elements of a head row (coalesced both ways).
template <typename T>
__global__ void __launch_bounds__(256)
split_heads(const float* __restrict__ qkv, const float* __restrict__ bias, T* __restrict__ q,
            T* __restrict__ k, T* __restrict__ v, int n, int H, int d, long long total4) {
  const long long e = (long long)blockIdx.x * 256 + threadIdx.x;  // float4 index of [B*n][3D]
  if (e >= total4) return;
  const int D = H * d, D4 = 3 * D / 4;
  const long long row = e / D4;  // b * n + t
  const int c = (int)(e - row * D4) * 4;  // column of [3D]
  const int which = c / D, h = (c - which * D) / d, j = c - which * D - h * d;
  const long long b = row / n, t = row - b * n;
  float4 x = *reinterpret_cast<const float4*>(qkv + row * 3 * D + c);
  if (bias) {
    const float4 bb = *reinterpret_cast<const float4*>(bias + c);
    x = make_float4(x.x + bb.x, x.y + bb.y, x.z + bb.z, x.w + bb.w);
  }
  T* dst = which == 0 ? q : (which == 1 ? k : v);
  store4<T>(dst + (((size_t)b * H + h) * n + t) * d + j, x.x, x.y, x.z, x.w);
}

// o [B][H][n][d] -> merged [B*n][H*d] (head h in columns h d ..).
template <typename T>
__global__ void __launch_bounds__(256)
merge_heads(const T* __restrict__ o, T* __restrict__ merged, int n, int H, int d,
            long long total4) {
  const long long e = (long long)blockIdx.x * 256 + threadIdx.x;  // 4-element group of merged
  if (e >= total4) return;
  const int D = H * d, D4 = D / 4;
  const long long row = e / D4;
  const int c = (int)(e - row * D4) * 4;
  const int h = c / d, j = c - h * d;
  const long long b = row / n, t = row - b * n;
  const float4 x = load4<T>(o + (((size_t)b * H + h) * n + t) * d + j);
  store4<T>(merged + row * D + c, x.x, x.y, x.z, x.w);
}

// y = y32 + bias, in T. [rows][D].
template <typename T>
__global__ void __launch_bounds__(256)
add_bias(const float* __restrict__ y32, const float* __restrict__ bias, T* __restrict__ y, int D,
         long long total4) {
  const long long e = (long long)blockIdx.x * 256 + threadIdx.x;
  if (e >= total4) return;
  const int c = (int)(e % (D / 4)) * 4;
  float4 x = reinterpret_cast<const float4*>(y32)[e];
  if (bias) {
    const float4 bb = *reinterpret_cast<const float4*>(bias + c);
    x = make_float4(x.x + bb.x, x.y + bb.y, x.z + bb.z, x.w + bb.w);
  }
  store4<T>(y + e * 4, x.x, x.y, x.z, x.w);
}

struct Blas {
  std::mutex mu;
  cublasHandle_t h = nullptr;
};
Blas g_blas[kMaxDevices];

// C[M][N] (fp32, row-major) = A[M][K] B[K][N] (row-major, element type of
// dtype), fp32 accumulation (no reduced-precision math for fp32 inputs).
int gemm_rm(int dev, cudaStream_t stream, const void* A, const void* B, float* C, long long M,
            long long N, long long K, int dtype) {
  Blas& bl = g_blas[dev];
  std::lock_guard<std::mutex> lk(bl.mu);
  if (!bl.h && cublasCreate(&bl.h) != CUBLAS_STATUS_SUCCESS) {
    bl.h = nullptr;
    return set_cuda_error(cudaErrorUnknown);
  }
  if (cublasSetStream(bl.h, stream) != CUBLAS_STATUS_SUCCESS) return set_cuda_error(cudaErrorUnknown);
  const float one = 1.f, zero = 0.f;
  const cudaDataType_t t = dtype == NYS_BF16 ? CUDA_R_16BF : CUDA_R_32F;
  // row-major C = A B is column-major C^T = B^T A^T
  const cublasStatus_t st = cublasGemmEx(bl.h, CUBLAS_OP_N, CUBLAS_OP_N, (int)N, (int)M, (int)K, &one,
                                         B, t, (int)N, A, t, (int)K, &zero, C, CUDA_R_32F, (int)N,
                                         CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  if (st != CUBLAS_STATUS_SUCCESS) {
    cudaGetLastError();
    return set_cuda_error(cudaErrorLaunchFailure);
  }
  return NYS_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct MhaLayout {
  size_t y32, q, k, v, o, merged, attn, total;
};

MhaLayout mha_layout(const Shape& s) {
  MhaLayout L{};
  const size_t rows = (size_t)s.B * s.n, D = (size_t)s.H * s.d;
  const size_t esz = s.dtype == NYS_FP32 ? 4 : 2;
  const size_t heads = (size_t)s.bh() * s.n * s.d * esz;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
  L.y32 = take(rows * 3 * D * 4);  // X W_qkv; later [O] W_o (fp32)
  L.q = take(heads);
  L.k = take(heads);
  L.v = take(heads);
  L.o = take(heads);
  L.merged = take(rows * D * esz);
  L.attn = take(make_layout(s).total);
  L.total = off;
  return L;
}

template <typename T>
int launch_split(const Shape& s, const float* qkv, const float* bias, void* q, void* k, void* v,
                 cudaStream_t st) {
  const long long total4 = (long long)s.B * s.n * 3 * s.H * s.d / 4;
  KernelScope scope("split_heads", st);
  split_heads<T><<<(unsigned)((total4 + 255) / 256), 256, 0, st>>>(
      qkv, bias, static_cast<T*>(q), static_cast<T*>(k), static_cast<T*>(v), s.n, s.H, s.d, total4);
  return launch_status();
}

template <typename T>
int launch_merge(const Shape& s, const void* o, void* merged, cudaStream_t st) {
  const long long total4 = (long long)s.B * s.n * s.H * s.d / 4;
  KernelScope scope("merge_heads", st);
  merge_heads<T><<<(unsigned)((total4 + 255) / 256), 256, 0, st>>>(
      static_cast<const T*>(o), static_cast<T*>(merged), s.n, s.H, s.d, total4);
  return launch_status();
}

template <typename T>
int launch_bias(const Shape& s, const float* y32, const float* bias, void* y, cudaStream_t st) {
  const long long total4 = (long long)s.B * s.n * s.H * s.d / 4;
  KernelScope scope("add_bias", st);
  add_bias<T><<<(unsigned)((total4 + 255) / 256), 256, 0, st>>>(y32, bias, static_cast<T*>(y),
                                                                s.H * s.d, total4);
  return launch_status();
}

std::mutex g_cache_mu;
void* g_cache[kMaxDevices] = {};
size_t g_cache_bytes[kMaxDevices] = {};

}  // namespace

}  // namespace nys

using namespace nys;

extern "C" {

size_t nystrom_mha_workspace_bytes(int B, int n, int H, int d, int m, int dtype) {
  if (check_shape(B, H, n, d, m, 0, 0, dtype) != NYS_OK) return 0;
  return mha_layout(Shape{B, H, n, d, m, 0, 0, dtype}).total;
}

int nystrom_mha_fwd(const void* x, const void* w_qkv, const float* b_qkv, const void* w_o,
                    const float* b_o, const float* conv_w, void* y, int B, int n, int H, int d,
                    int m, int iters, int conv_ks, int dtype, void* workspace, size_t ws_bytes,
                    nys_stream_t stream) {
  if (!x || !w_qkv || !w_o || !y) return NYS_ERR_ARG;
  if (conv_ks > 0 && !conv_w) return NYS_ERR_ARG;
  int rc = check_shape(B, H, n, d, m, iters, conv_ks, dtype);
  if (rc != NYS_OK) return rc;
  const uintptr_t a = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_qkv) |
                      reinterpret_cast<uintptr_t>(w_o) | reinterpret_cast<uintptr_t>(y) |
                      reinterpret_cast<uintptr_t>(b_qkv) | reinterpret_cast<uintptr_t>(b_o);
  if (a & 15u) return NYS_ERR_ALIGN;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return NYS_ERR_ALIGN;
  const Shape s{B, H, n, d, m, iters, conv_ks, dtype};
  const MhaLayout L = mha_layout(s);
  if (workspace && ws_bytes < L.total) return NYS_ERR_NOMEM;
  int dev = 0;
  rc = check_device(&dev);
  if (rc != NYS_OK) return rc;
  char* ws = static_cast<char*>(workspace);
  std::unique_lock<std::mutex> cache_lk(g_cache_mu, std::defer_lock);
  if (!ws) {
    cache_lk.lock();
    if (g_cache_bytes[dev] < L.total) {
      if (g_cache[dev]) cudaFree(g_cache[dev]);
      g_cache[dev] = nullptr;
      g_cache_bytes[dev] = 0;
      if (cudaMalloc(&g_cache[dev], L.total) != cudaSuccess) {
        cudaGetLastError();
        g_cache[dev] = nullptr;
        return NYS_ERR_NOMEM;
      }
      g_cache_bytes[dev] = L.total;
    }
    ws = static_cast<char*>(g_cache[dev]);
  }
  const long long rows = (long long)B * n, D = (long long)H * d;
  float* y32 = reinterpret_cast<float*>(ws + L.y32);
  void *q = ws + L.q, *k = ws + L.k, *v = ws + L.v, *o = ws + L.o, *merged = ws + L.merged;
  const bool bf16 = dtype == NYS_BF16;
  rc = error_in("QKV projection", gemm_rm(dev, stream, x, w_qkv, y32, rows, 3 * D, D, dtype));
  if (rc != NYS_OK) return rc;
  rc = bf16 ? launch_split<__nv_bfloat16>(s, y32, b_qkv, q, k, v, stream)
            : launch_split<float>(s, y32, b_qkv, q, k, v, stream);
  if (rc != NYS_OK) return error_in("head split", rc);
  rc = run(s, q, k, v, conv_w, o, ws + L.attn, stream, dev);
  if (rc != NYS_OK) return rc;
  rc = bf16 ? launch_merge<__nv_bfloat16>(s, o, merged, stream) : launch_merge<float>(s, o, merged, stream);
  if (rc != NYS_OK) return error_in("head merge", rc);
  rc = error_in("output projection", gemm_rm(dev, stream, merged, w_o, y32, rows, D, D, dtype));
  if (rc != NYS_OK) return rc;
  rc = bf16 ? launch_bias<__nv_bfloat16>(s, y32, b_o, y, stream) : launch_bias<float>(s, y32, b_o, y, stream);
  return error_in("output bias", rc);
}

}  // extern "C"
