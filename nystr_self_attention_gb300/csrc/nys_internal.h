// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "nystrom.h"

namespace nys {

// One forward call's shape, validated.
struct Shape {
  int B, H, n, d, m, iters, ks, dtype;
  long long bh() const { return (long long)B * H; }
  int seg() const { return n / m; }
};

// Byte offsets of the workspace regions (all 256-byte aligned). Every
// region is per head, head-major (b*H + h).
struct Layout {
  size_t status;   // int32 status word (+ padding)
  size_t q_tilde;  // f32 [m][d]
  size_t k_tilde;  // f32 [m][d]
  size_t g_part;   // f32 [splits][m][d]  unnormalised partial sums
  size_t g_ml;     // f32 [splits][m][2]  (running max, running sum)
  size_t g;        // f32 [m][d]          softmax(Q~ K^T s) V
  size_t a_s;      // f32 [m][m]
  size_t z;        // f32 [m][m]
  size_t w;        // f32 [m][d]          Z G
  size_t scratch;  // f32 [3][m][m]       pseudo-inverse temporaries
  size_t total;
  int splits;      // key splits of the landmark-row pass
};

Layout make_layout(const Shape& s);

// Brackets one kernel launch: counts it and, while profiling is on, records
// CUDA events before and after it on `stream`.
class KernelScope {
 public:
  KernelScope(const char* name, cudaStream_t stream);
  ~KernelScope();
  KernelScope(const KernelScope&) = delete;
  KernelScope& operator=(const KernelScope&) = delete;

 private:
  const char* name_;
  cudaStream_t stream_;
  cudaEvent_t begin_ = nullptr;
};

// Host helpers of the C ABI (nys_api.cu).
int set_cuda_error(cudaError_t e);  // remembers the message, returns NYS_ERR_CUDA
int check_shape(int B, int H, int n, int d, int m, int iters, int ks, int dtype);
int check_args(const void* q, const void* k, const void* v, const float* conv_w, const void* out,
               int B, int H, int n, int d, int m, int iters, int ks, int dtype);
int check_device(int* dev_out);  // current device, must be compute capability 10.3
// Clears the status word and enqueues the forward pass with workspace `ws`.
int run(const Shape& s, const void* q, const void* k, const void* v, const float* conv_w,
        void* out, char* ws, cudaStream_t stream, int dev);

// Enqueue the whole forward pass. Pointers are device pointers; ws has
// Layout::total bytes. Returns NYS_OK or NYS_ERR_CUDA (launch failure).
int launch_forward(const Shape& s, const void* q, const void* k, const void* v,
                   const float* conv_w, void* out, char* ws, const Layout& L,
                   cudaStream_t stream);

}  // namespace nys
