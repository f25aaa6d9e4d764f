// Forward-pass orchestration: which kernel runs each step, and the split of
// the batch into head groups that run concurrently on library streams.
//
// Per head the steps are landmarks -> landmark rows -> pseudo-inverse ->
// token rows (each depends on the previous one). The pseudo-inverse is a
// serial chain of small dependent products and leaves most of the GPU idle,
// while the other steps stream the inputs. Splitting the batch into groups
// of whole batch entries and running each group's four steps on its own
// stream lets one group's pseudo-inverse overlap the other groups' streaming
// steps. The groups share the workspace arrays (each at its own head
// offset), so the workspace layout does not depend on the grouping.
//
// Where the batch stays in one group and the tensor-core pseudo-inverse
// needs at most half of the SMs (few heads, long sequences), its chain of
// products runs on a second stream beside the landmark-row pass instead of
// after it: Z depends only on the landmarks. The landmark-row pass is then
// spread over the SMs the pseudo-inverse leaves free, G is merged from its
// partials while Z is still being formed, and W = Z G is formed by a short
// kernel once both are done.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "nys_internal.h"

namespace nys {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxGroups = 8;

struct DeviceStreams {
  std::mutex mu;
  std::mutex enqueue;  // one multi-stream enqueue at a time (shared events)
  bool ready = false;
  cudaStream_t aux[kMaxGroups] = {};
  cudaEvent_t fork = nullptr;
  cudaEvent_t join[kMaxGroups] = {};
};
DeviceStreams g_streams[kMaxDevices];

int ensure_streams(int dev) {
  DeviceStreams& d = g_streams[dev];
  std::lock_guard<std::mutex> lk(d.mu);
  if (d.ready) return NYS_OK;
  cudaError_t e = cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming);
  for (int i = 1; i < kMaxGroups && e == cudaSuccess; ++i) {
    e = cudaStreamCreateWithFlags(&d.aux[i], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.join[i], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) return set_cuda_error(e);
  d.ready = true;
  return NYS_OK;
}

// SMs the landmark-row pass keeps at least when the pseudo-inverse runs
// beside it
constexpr int kMinRowSms = 48;

// SMs the pseudo-inverse's CTAs take beside the landmark rows: one CTA per
// SM while they fit in half of the GPU, else two per SM (m <= 64: two
// CTAs' shared memory and TMEM fit one SM); 0 if the plan does not apply.
int pinv_beside_sms(const Shape& s) {
  if (s.dtype != NYS_BF16 || !pinv_tc_supported(s) || s.d % 16 != 0) return 0;
  const int sms = plan_sms();
  const int ctas = pinv_tc_ctas(s);
  if (2 * ctas <= sms) return ctas;
  if (s.m <= 64 && (ctas + 1) / 2 <= sms - kMinRowSms) return (ctas + 1) / 2;
  return 0;
}

// Number of head groups: only for the tensor-core path with short
// sequences, where the pseudo-inverse dominates and does not run beside the
// landmark rows; whole batch entries per group.
int choose_groups(const Shape& s) {
  int g = 1;
  if (s.dtype == NYS_BF16 && s.n <= 2048 && s.bh() >= 256 && pinv_beside_sms(s) == 0) g = 2;
  if (g > kMaxGroups) g = kMaxGroups;
  if (g > s.B) g = s.B;
  while (g > 1 && s.B % g != 0) --g;
  return g;
}

template <typename T>
T* at(char* ws, size_t off) { return reinterpret_cast<T*>(ws + off); }

// The four steps for heads [bh0, bh0 + sg.bh()) of the full problem (whole
// batch entries: bh0 is a multiple of H).
int run_group(const Shape& full, const Shape& sg_in, long long bh0, const void* q, const void* k,
              const void* v, const float* conv_w, void* out, char* ws, const Layout& L,
              cudaStream_t st, DeviceStreams* beside) {
  Shape sg = sg_in;
  if (full.lengths) sg.lengths = full.lengths + bh0 / full.H;
  const size_t esz = full.dtype == NYS_FP32 ? 4 : 2;
  const size_t tok = (size_t)bh0 * full.n * full.d * esz;
  const void* qg = static_cast<const char*>(q) + tok;
  const void* kg = static_cast<const char*>(k) + tok;
  const void* vg = static_cast<const char*>(v) + tok;
  void* og = static_cast<char*>(out) + tok;
  const size_t md = (size_t)full.m * full.d, mm = (size_t)full.m * full.m;
  const size_t pad = (size_t)full.m64() * full.dpad();
  float* qt = at<float>(ws, L.q_tilde) + bh0 * md;
  float* kt = at<float>(ws, L.k_tilde) + bh0 * md;
  float* gp = at<float>(ws, L.g_part) + bh0 * L.splits * md;
  float* gml = at<float>(ws, L.g_ml) + bh0 * L.splits * full.m * 2;
  float* g = at<float>(ws, L.g) + bh0 * md;
  float* a = at<float>(ws, L.a_s) + bh0 * mm;
  float* z = at<float>(ws, L.z) + bh0 * mm;
  float* w = at<float>(ws, L.w) + bh0 * md;
  float* scr = at<float>(ws, L.scratch) + bh0 * scratch_mats(full) * mm;
  int* status = at<int>(ws, L.status);
  const bool bf16 = full.dtype == NYS_BF16;
  const bool tc_tokens = tokens_tc_smem(full) > 0;
  const bool big_tokens = !tc_tokens && tokens_big_supported(full);
  const bool bf16_ops = tc_tokens || big_tokens;  // token step reads K~, W^T as bf16
  const bool x3 = x3_supported(full);  // fp32 on the tensor cores
  __nv_bfloat16* qt_b = bf16 ? at<__nv_bfloat16>(ws, L.qt_bf16) + bh0 * pad : nullptr;
  __nv_bfloat16* kt_b = (bf16 && bf16_ops) ? at<__nv_bfloat16>(ws, L.kt_bf16) + bh0 * pad : nullptr;
  __nv_bfloat16* wt_b = bf16 ? at<__nv_bfloat16>(ws, L.wt_bf16) + bh0 * pad : nullptr;

  int rc = launch_landmarks(sg, qg, kg, qt, kt, qt_b, kt_b, st);
  if (rc != NYS_OK) return error_in("landmarks", rc);
  if (beside) {  // Z on the second stream while the landmark rows stream K, V
    cudaStream_t aux = beside->aux[1];
    cudaError_t e = cudaEventRecord(beside->fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(aux, beside->fork, 0);
    if (e != cudaSuccess) return set_cuda_error(e);
    rc = launch_rows_tc(sg, qt_b, kg, vg, gp, gml, L.splits, L.tiles_per_split, status, st);
    if (rc != NYS_OK) return error_in("landmark rows", rc);
    rc = launch_pinv_tc(sg, qt, kt, nullptr, nullptr, nullptr, a, z, nullptr, nullptr, L.splits,
                        status, aux);
    if (rc != NYS_OK) return error_in("pseudo-inverse", rc);
    rc = launch_merge_g(sg, gp, gml, g, L.splits, st);  // while Z is still being formed
    if (rc != NYS_OK) return error_in("merge of G", rc);
    e = cudaEventRecord(beside->join[1], aux);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, beside->join[1], 0);
    if (e != cudaSuccess) return set_cuda_error(e);
    rc = error_in("W = Z G", launch_w_tc(sg, z, g, w, wt_b, status, st));
  } else {
  rc = bf16 ? launch_rows_tc(sg, qt_b, kg, vg, gp, gml, L.splits, L.tiles_per_split, status, st)
       : x3 ? launch_rows_x3(sg, qt, kg, vg, gp, gml, L.splits, L.tiles_per_split, status, st)
            : launch_rows_simt(sg, qt, kg, vg, gp, gml, L.splits, st);
  if (rc != NYS_OK) return error_in("landmark rows", rc);
  rc = pinv_tc_supported(full)
           ? launch_pinv_tc(sg, qt, kt, gp, gml, g, a, z, w, wt_b, L.splits, status, st)
       : pinv_big_supported(full)
           ? launch_pinv_big(sg, qt, kt, gp, gml, g, a, z, scr, w, wt_b, L.splits, status, st)
           : launch_pinv_simt(sg, qt, kt, gp, gml, g, a, z, w, scr, bf16_ops ? wt_b : nullptr,
                              L.splits, st);
    rc = error_in("pseudo-inverse", rc);
  }
  if (rc != NYS_OK) return rc;
  Shape stok = sg;  // the token pass: with the variants, the attention term alone
  if (full.separate_conv()) stok.ks = 0;
  if (tc_tokens)
    rc = launch_tokens_tc(stok, qg, vg, kt_b, wt_b, conv_w, og, status, plan_sms(), st);
  else if (big_tokens)
    rc = launch_tokens_big(stok, qg, vg, kt_b, wt_b, conv_w, og, status, plan_sms(), st);
  else if (x3)
    rc = launch_tokens_x3(stok, qg, vg, kt, w, stok.ks > 0 ? conv_w : nullptr, og, status, st);
  else
    rc = launch_tokens_simt(stok, qg, vg, kt, w, stok.ks > 0 ? conv_w : nullptr, og, st);
  rc = error_in("token rows", rc);
  if (rc == NYS_OK && full.separate_conv())
    rc = error_in("convolution", launch_conv_mask(sg, vg, conv_w, og, st));
  return rc;
}

}  // namespace

bool z_beside_rows(const Shape& s) { return pinv_beside_sms(s) > 0 && choose_groups(s) == 1; }

int rows_tc_ctas(const Shape& s) {
  const int sms = plan_sms();
  return z_beside_rows(s) ? sms - pinv_beside_sms(s) : sms;
}

int launch_forward(const Shape& s, const void* q, const void* k, const void* v,
                   const float* conv_w, void* out, char* ws, const Layout& L,
                   cudaStream_t stream, int dev) {
  const int groups = choose_groups(s);
  const bool beside = groups <= 1 && z_beside_rows(s);
  if (groups <= 1 && !beside) return run_group(s, s, 0, q, k, v, conv_w, out, ws, L, stream, nullptr);
  int rc = ensure_streams(dev);
  if (rc != NYS_OK) return rc;
  DeviceStreams& d = g_streams[dev];
  std::lock_guard<std::mutex> lk(d.enqueue);
  if (beside) return run_group(s, s, 0, q, k, v, conv_w, out, ws, L, stream, &d);
  cudaError_t e = cudaEventRecord(d.fork, stream);
  for (int i = 1; i < groups && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(d.aux[i], d.fork, 0);
  if (e != cudaSuccess) return set_cuda_error(e);
  Shape sg = s;
  sg.B = s.B / groups;
  for (int i = 0; i < groups; ++i) {
    rc = run_group(s, sg, (long long)i * sg.bh(), q, k, v, conv_w, out, ws, L,
                   i == 0 ? stream : d.aux[i], nullptr);
    if (rc != NYS_OK) return rc;
  }
  for (int i = 1; i < groups && e == cudaSuccess; ++i) {
    e = cudaEventRecord(d.join[i], d.aux[i]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, d.join[i], 0);
  }
  return e == cudaSuccess ? NYS_OK : set_cuda_error(e);
}

std::string describe_plan(const Shape& s) {
  const Layout L = make_layout(s);
  const int groups = choose_groups(s);
  const bool beside = groups <= 1 && z_beside_rows(s);
  Shape sg = s;
  sg.B = s.B / groups;
  const bool bf16 = s.dtype == NYS_BF16;
  const bool tc_tokens = tokens_tc_smem(s) > 0;
  const bool big_tokens = !tc_tokens && tokens_big_supported(s);
  std::string out = beside ? "plan=z-beside-rows" : groups > 1 ? "plan=head-groups" : "plan=serial";
  out += " groups=" + std::to_string(groups);
  const LandmarkKernel lk = landmark_kernel(sg);
  out += std::string(" landmarks=") + (lk == LandmarkKernel::Small ? "landmarks_small"
                                       : lk == LandmarkKernel::Vec ? "landmarks_vec"
                                                                   : "landmarks_simt");
  if (bf16) {
    const long long total = (long long)((s.n + 127) / 128) * sg.bh();
    const long long ctas = (total + L.tiles_per_split - 1) / L.tiles_per_split;
    out += " rows=rows_tc[ctas=" + std::to_string(ctas) + ",parts=" + std::to_string(L.splits) +
           ",tiles_per_cta=" + std::to_string(L.tiles_per_split) + "]";
  } else if (x3_supported(s)) {
    out += " rows=rows_x3[splits=" + std::to_string(L.splits) +
           ",tiles_per_split=" + std::to_string(L.tiles_per_split) + "]";
  } else {
    out += " rows=rows_simt[splits=" + std::to_string(L.splits) + "]";
  }
  if (beside) {
    out += " pinv=pinv_tc[z-only,ctas=" + std::to_string(pinv_tc_ctas(sg)) +
           ",sms=" + std::to_string(pinv_beside_sms(s)) + "]";
    out += " merge=merge_g w=w_tc";
  } else if (pinv_tc_supported(s)) {
    out += " pinv=pinv_tc[ctas=" + std::to_string(pinv_tc_ctas(sg)) + "]";
  } else if (pinv_big_supported(s)) {
    out += " pinv=pinv_big[clusters=" + std::to_string(sg.bh()) + "]";
  } else {
    out += " pinv=pinv_simt";
  }
  out += tc_tokens    ? " tokens=tokens_tc"
         : big_tokens ? " tokens=tokens_big"
         : x3_supported(s) ? " tokens=tokens_x3"
                           : " tokens=tokens_simt";
  if (s.separate_conv()) out += " conv=conv_mask";
  return out;
}

}  // namespace nys
