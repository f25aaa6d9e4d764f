// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <string>

#include "nystrom.h"

namespace nys {

// One forward call's shape, validated.
struct Shape {
  int B, H, n, d, m, iters, ks, dtype;
  // variants (nystrom_attn_fwd_ex): per batch entry number of real tokens
  // (device int32 [B], null: every row is a token), conv filter layout
  const int* lengths = nullptr;
  int conv_layout = NYS_CONV_PER_HEAD;
  // the fused token kernels cover per-head filters on unpadded inputs; the
  // variants run the token kernels for the attention term alone and add the
  // convolution (and zero the padding rows) in a pass of their own
  bool separate_conv() const { return lengths != nullptr || conv_layout != NYS_CONV_PER_HEAD; }
  long long bh() const { return (long long)B * H; }
  int seg_max() const { return (int)(((long long)n + m - 1) / m); }  // rows of the longest segment
  int m64() const { return ((m + 63) / 64) * 64; }  // m rounded up to 64
  int dpad() const { return d <= 64 ? 64 : 128; }   // d rounded up to a 64-column chunk
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
  size_t scratch;  // f32 [scratch_mats][m][m]  pseudo-inverse temporaries
  size_t qt_bf16;  // bf16 [m64][dpad]    Q~, zero padded (tensor-core operand)
  size_t kt_bf16;  // bf16 [m64][dpad]    K~, zero padded (tensor-core operand)
  size_t wt_bf16;  // bf16 [dpad][m64]    W^T, zero padded (tensor-core operand)
  size_t lengths;  // int32 [B]           tokens per batch entry (padded-sequence variant)
  size_t total;
  int splits;      // key splits of the landmark-row pass
  int tiles_per_split;  // 128-key tiles per split (tensor-core landmark-row pass)
};

Layout make_layout(const Shape& s);

// m x m fp32 temporaries per head in Layout::scratch: 5 for the clustered
// tensor-core pseudo-inverse (m > 128), else 3.
int scratch_mats(const Shape& s);

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

// Timeout test switch (nystrom_debug_stall_pinv): > 0 makes the tensor-core
// pseudo-inverse kernel (m <= 128) wait that many ns on a phase nothing
// completes before its first product. 0 (the default): off.
uint32_t debug_stall_ns();

// Host helpers of the C ABI (nys_api.cu).
int set_cuda_error(cudaError_t e);  // remembers the message, returns NYS_ERR_CUDA
// rc unchanged; a CUDA error's message gets the failing step's name in front.
int error_in(const char* step, int rc);
// A tensor map the driver would not encode: NYS_ERR_CUDA, message names the site.
int tensor_map_error(const char* file, int line);
// After a launch: NYS_OK, or NYS_ERR_CUDA with the launch error's message kept.
inline int launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? NYS_OK : set_cuda_error(e);
}
int check_shape(int B, int H, int n, int d, int m, int iters, int ks, int dtype);
int check_args(const void* q, const void* k, const void* v, const float* conv_w, const void* out,
               int B, int H, int n, int d, int m, int iters, int ks, int dtype);
int check_device(int* dev_out);  // current device, must be compute capability 10.3
// Makes `ws` the workspace nystrom_get_status reads for this device and
// clears its status word on `stream` (unless told not to).
int begin_call(char* ws, const Layout& L, cudaStream_t stream, int dev, bool clear_status = true);
// The library's cached workspace of this device, grown to `bytes` (NULL and
// *rc < 0 on failure).
void* cached_workspace(int dev, size_t bytes, cudaStream_t stream, int* rc);
// Clears the status word (unless told not to) and enqueues the forward
// pass with workspace `ws`.
int run(const Shape& s, const void* q, const void* k, const void* v, const float* conv_w,
        void* out, char* ws, cudaStream_t stream, int dev, bool clear_status = true);

// SM count the forward-pass plan and the workspace layout are made for:
// the current device's, or 152 (GB300) when no device can be queried
// (host-only queries on a machine without a GPU).
int plan_sms();

// Tensor-core token kernel (nys_tokens_tc.cu): shared memory it needs for
// this shape, 0 if the shape is outside what it handles.
size_t tokens_tc_smem(const Shape& s);
int launch_tokens_tc(const Shape& s, const void* q, const void* v, const void* kt_bf16,
                     const void* wt_bf16, const float* conv_w, void* out, int* status,
                     int num_sms, cudaStream_t stream);

// Tensor-core token kernel for d = 128 and large m (nys_tokens_big.cu), used
// where the pipelined token kernel's operands do not fit.
bool tokens_big_supported(const Shape& s);
int launch_tokens_big(const Shape& s, const void* q, const void* v, const void* kt_bf16,
                      const void* wt_bf16, const float* conv_w, void* out, int* status,
                      int num_sms, cudaStream_t stream);

// fp32 landmark-row and token-row passes on the tensor cores in three tf32
// products (nys_x3.cu): fp32, d <= 64 with d % 4 == 0, m <= 128. The
// landmark-row pass splits each head's 128-key tiles into `splits` ranges
// of `tiles_per_split` (x3_rows_split); the token pass adds the
// convolution of V (per-head taps) when s.ks > 0, else writes the attention
// term alone.
bool x3_supported(const Shape& s);
void x3_rows_split(const Shape& s, int* splits, int* tiles_per_split);
int launch_rows_x3(const Shape& s, const float* qt, const void* k, const void* v, float* gpart,
                   float* gml, int splits, int tiles_per_split, int* status, cudaStream_t stream);
int launch_tokens_x3(const Shape& s, const void* q, const void* v, const float* kt, const float* w,
                     const float* conv_w, void* out, int* status, cudaStream_t stream);

// Tensor-core landmark-row kernel (nys_rows_tc.cu), bf16 inputs. `s` may be
// a group of heads of the full problem: splits / tiles_per_split come from
// the full problem's layout.
void rows_tc_split(const Shape& s, int ctas, int* splits, int* tiles_per_split);

// Forward-pass plan (nys_forward.cu), a function of the shape alone so that
// the workspace layout matches the launches: whether the pseudo-inverse runs
// beside the landmark-row pass, and the CTAs the tensor-core landmark-row
// pass spreads its tiles over.
bool z_beside_rows(const Shape& s);
int rows_tc_ctas(const Shape& s);
int launch_rows_tc(const Shape& s, const void* qt_bf16, const void* k, const void* v, float* gpart,
                   float* gml, int splits, int tiles_per_split, int* status, cudaStream_t stream);

// CUDA-core steps (nys_simt.cu); `s` may be a group of heads.
// Segment-mean kernel for a shape: landmarks_small (a warp per 32/VPR short
// segments), landmarks_vec (a warp per segment) or landmarks_simt (a thread
// per landmark element, head sizes whose 16-byte row vectors do not divide 32).
enum class LandmarkKernel { Small, Vec, Simt };
LandmarkKernel landmark_kernel(const Shape& s);
// k == nullptr: the means of Q alone (kt, kt_b unused)
int launch_landmarks(const Shape& s, const void* q, const void* k, float* qt, float* kt,
                     __nv_bfloat16* qt_b, __nv_bfloat16* kt_b, cudaStream_t stream);
int launch_rows_simt(const Shape& s, const float* qt, const void* k, const void* v, float* gp,
                     float* gml, int splits, cudaStream_t stream);
int launch_pinv_simt(const Shape& s, const float* qt, const float* kt, const float* gp,
                     const float* gml, float* g, float* a, float* z, float* w, float* scratch,
                     __nv_bfloat16* wt_b, int splits, cudaStream_t stream);
int launch_tokens_simt(const Shape& s, const void* q, const void* v, const float* kt,
                       const float* w, const float* conv_w, void* out, cudaStream_t stream);
// out += DWConv(V) for per-channel filters and/or padded sequences (zeros the
// padding rows; with s.ks == 0 only that). out holds the attention term.
int launch_conv_mask(const Shape& s, const void* v, const float* conv_w, void* out,
                     cudaStream_t stream);
// G = merge of the key-split partials (CUDA cores, one thread per 4
// elements of G), for the plan that computes Z beside the landmark rows.
int launch_merge_g(const Shape& s, const float* gp, const float* gml, float* g, int splits,
                   cudaStream_t stream);

// K-means rounds of clustered attention on the tensor cores (bf16, d in {64,
// 128}, C = s.m <= 128). Workspace per call: the bf16 split of the centroids
// (hi, mid, lo), their squared norms, and the per-CTA members' sums and
// counts of one round.
struct KmWorkspace {
  int S, C_pad;
  size_t mu3_bytes, norm_bytes, part_bytes, cnt_bytes;
};
bool kmeans_tc_supported(const Shape& s);
KmWorkspace kmeans_tc_workspace(const Shape& s);
// split and squared norms of the centroids mu (fp32 [B*H][C][d])
int launch_kmeans_prep(const Shape& s, const float* mu, void* mu3, float* norms, cudaStream_t st);
// one round: assignment with mu3 / norms (the split of mu_old), members'
// sums, then mu_new and, in place in mu3 / norms, the split of mu_new
int launch_kmeans_round_tc(const Shape& s, const void* q, const void* mu3, const float* norms,
                           int* assign, float* part, int* cnt, const float* mu_old, float* mu_new,
                           float* norms_next, void* mu3_next, int* status, cudaStream_t st);

// Most pseudo-inverse updates the tensor-core kernels run: their products
// take tf32 operands, whose rounding the iteration amplifies by cond(A_S) as
// it inverts more of A_S's small singular values. Up to 8 updates (the
// page's "about 6"; 8 in the long-context workload) this stays well inside
// the bf16 parity bar; with more (12 can give 6e-2, 24-64 can diverge) the
// bf16 path runs the pseudo-inverse in fp32 on the CUDA cores instead.
constexpr int kTf32MaxIters = 8;
// fp32 inputs: the tensor-core pseudo-inverse (three tf32 products per
// product, close to fp32 rounding) up to this many updates; the CUDA-core
// kernel beyond.
constexpr int kX3MaxIters = 12;

// Tensor-core pseudo-inverse (nys_pinv_tc.cu): bf16 path, m <= 128; fp32
// path (three tf32 products per product), m <= 64, d 32 or 64.
// Z -> z [B*H][m][m] fp32 when z is set. With gpart == nullptr, Z only: no
// merge of the partials, no W (gml, g, w and wt_bf16 unused; z required).
bool pinv_tc_supported(const Shape& s);
int pinv_tc_ctas(const Shape& s);  // CTAs of one launch over all of s's heads
int launch_pinv_tc(const Shape& s, const float* qt, const float* kt, const float* gpart,
                   const float* gml, float* g, float* a_s, float* z, float* w, void* wt_bf16,
                   int splits, int* status, cudaStream_t stream);
// W = Z G on the tensor cores from Z and the merged G, for the plan that
// computes Z beside the landmark-row pass; d % 16 == 0. Writes W (stage
// export) and W^T bf16.
int launch_w_tc(const Shape& s, const float* z, const float* g, float* w, void* wt_bf16,
                int* status, cudaStream_t stream);

// Clustered tensor-core pseudo-inverse (nys_pinv_big.cu), bf16 path,
// 128 < m <= 256. `scratch` is the group's block of Layout::scratch.
bool pinv_big_supported(const Shape& s);
int launch_pinv_big(const Shape& s, const float* qt, const float* kt, const float* gpart,
                    const float* gml, float* g, float* a_s, float* z, float* scratch, float* w,
                    void* wt_bf16, int splits, int* status, cudaStream_t stream);

// One line naming the kernels a forward call of this shape launches, in
// order, with the plan's host-side sizes (nys_forward.cu). Host only.
std::string describe_plan(const Shape& s);

// Enqueue the whole forward pass (nys_forward.cu). Pointers are device
// pointers; ws has Layout::total bytes; dev is the current device. Returns
// NYS_OK or NYS_ERR_CUDA (a failed launch).
int launch_forward(const Shape& s, const void* q, const void* k, const void* v,
                   const float* conv_w, void* out, char* ws, const Layout& L,
                   cudaStream_t stream, int dev);

}  // namespace nys
