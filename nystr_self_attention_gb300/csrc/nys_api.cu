// C ABI of libnystrom.so: argument checks, workspace layout and caching,
// status word, host-buffer entry point. Declared in include/nystrom.h.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "nys_internal.h"

namespace nys {

namespace {

constexpr int kMaxDevices = 64;
std::atomic<uint32_t> g_stall_ns{0};
thread_local std::string g_last_error;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

uint32_t debug_stall_ns() { return g_stall_ns.load(); }

int set_cuda_error(cudaError_t e) {
  g_last_error = cudaGetErrorString(e);
  return NYS_ERR_CUDA;
}

int error_in(const char* step, int rc) {
  if (rc == NYS_ERR_CUDA) g_last_error = std::string(step) + ": " + g_last_error;
  return rc;
}

int tensor_map_error(const char* file, int line) {
  char msg[160];
  const char* base = std::strrchr(file, '/');
  std::snprintf(msg, sizeof msg, "tensor map encoding failed (%s:%d)", base ? base + 1 : file, line);
  g_last_error = msg;
  return NYS_ERR_CUDA;
}

namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

// Shape rules of include/nystrom.h. Pure host arithmetic.
int check_shape(int B, int H, int n, int d, int m, int iters, int ks, int dtype) {
  if (dtype != NYS_FP32 && dtype != NYS_BF16) return NYS_ERR_ARG;
  if (B < 1 || H < 1 || n < 1 || d < 1 || m < 1) return NYS_ERR_SHAPE;
  if (m > n || m > 256) return NYS_ERR_SHAPE;
  if (d % 8 != 0 || d > 128) return NYS_ERR_SHAPE;
  if (dtype == NYS_BF16 && d != 32 && d != 64 && d != 128) return NYS_ERR_SHAPE;
  if (iters < 0 || iters > 64) return NYS_ERR_SHAPE;
  if (ks < 0 || ks > 127 || (ks > 0 && ks % 2 == 0)) return NYS_ERR_SHAPE;
  const long long total = (long long)B * H * (long long)n * d;
  if (total >= (1ll << 40)) return NYS_ERR_SHAPE;
  return NYS_OK;
}

int check_args(const void* q, const void* k, const void* v, const float* conv_w, const void* out,
               int B, int H, int n, int d, int m, int iters, int ks, int dtype) {
  if (!q || !k || !v || !out) return NYS_ERR_ARG;
  if (ks > 0 && !conv_w) return NYS_ERR_ARG;
  const int rc = check_shape(B, H, n, d, m, iters, ks, dtype);
  if (rc != NYS_OK) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return NYS_ERR_ALIGN;
  if (ks > 0 && (reinterpret_cast<uintptr_t>(conv_w) & 3u)) return NYS_ERR_ALIGN;
  return NYS_OK;
}

int plan_sms() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 152;
  }
  if (cache[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
      cudaGetLastError();
      return 152;
    }
    cache[dev] = v;
  }
  return cache[dev];
}

// The current device must be compute capability 10.3 (GB300).
int check_device(int* dev_out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { set_cuda_error(e); return NYS_ERR_UNSUPPORTED; }
  static int cc_cache[kMaxDevices] = {0};
  if (dev < 0 || dev >= kMaxDevices) return NYS_ERR_UNSUPPORTED;
  if (cc_cache[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return NYS_ERR_UNSUPPORTED;
    cc_cache[dev] = major * 10 + minor;
  }
  if (cc_cache[dev] != 103) return NYS_ERR_UNSUPPORTED;
  *dev_out = dev;
  return NYS_OK;
}

namespace {
constexpr int kHostChunks = 8;  // chunks (head ranges) of the pipelined host entry

struct DeviceCache {
  std::mutex mu;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  void* last_ws = nullptr;  // status word of the most recent call
  void* stage = nullptr;    // host-entry staging buffers
  size_t stage_bytes = 0;
  // host entry: one call at a time per device (it owns the staging buffers);
  // copy streams and events of its pipeline, created on first use
  std::mutex host_mu;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev_start = nullptr, ev_done = nullptr;
  cudaEvent_t ev_in[kHostChunks] = {}, ev_comp[kHostChunks] = {};
};
DeviceCache g_dev[kMaxDevices];

// Grows a cached device buffer to `need` bytes. The old buffer is freed
// with cudaFree, which waits for all work on the device, so no earlier call
// still uses it; the new one is zeroed on `stream`, ahead of the work the
// caller enqueues there next (a memset on the legacy stream would not be
// ordered before work on a non-blocking stream).
int ensure_buffer(void** ptr, size_t* have, size_t need, cudaStream_t stream) {
  if (*have >= need) return NYS_OK;
  if (*ptr) {
    cudaFree(*ptr);
    *ptr = nullptr;
    *have = 0;
  }
  cudaError_t e = cudaMalloc(ptr, need);
  if (e != cudaSuccess) {
    *ptr = nullptr;
    g_last_error = cudaGetErrorString(e);
    cudaGetLastError();
    return NYS_ERR_NOMEM;
  }
  e = cudaMemsetAsync(*ptr, 0, need, stream);
  if (e != cudaSuccess) return set_cuda_error(e);
  *have = need;
  return NYS_OK;
}

}  // namespace

int begin_call(char* ws, const Layout& L, cudaStream_t stream, int dev, bool clear_status) {
  {
    std::lock_guard<std::mutex> lk(g_dev[dev].mu);
    g_dev[dev].last_ws = ws;
  }
  // each call starts with a clear status word (kernels only ever set it)
  if (clear_status) {
    cudaError_t e = cudaMemsetAsync(ws + L.status, 0, sizeof(int), stream);
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  return NYS_OK;
}

void* cached_workspace(int dev, size_t bytes, cudaStream_t stream, int* rc) {
  std::lock_guard<std::mutex> lk(g_dev[dev].mu);
  *rc = ensure_buffer(&g_dev[dev].ws, &g_dev[dev].ws_bytes, bytes, stream);
  return *rc == NYS_OK ? g_dev[dev].ws : nullptr;
}

int run(const Shape& s, const void* q, const void* k, const void* v, const float* conv_w,
        void* out, char* ws, cudaStream_t stream, int dev, bool clear_status) {
  const Layout L = make_layout(s);
  const int rc = begin_call(ws, L, stream, dev, clear_status);
  if (rc != NYS_OK) return rc;
  return launch_forward(s, q, k, v, conv_w, out, ws, L, stream, dev);
}

int scratch_mats(const Shape& s) { return pinv_big_supported(s) ? 5 : 3; }

Layout make_layout(const Shape& s) {
  Layout L{};
  const size_t bh = (size_t)s.bh(), md = (size_t)s.m * s.d, mm = (size_t)s.m * s.m;
  // Key splits of the landmark-row pass: enough CTAs to fill the GPU a few
  // times over (CUDA-core path: at least 32 keys per split; tensor-core
  // path: whole 128-key tiles).
  L.tiles_per_split = 0;
  if (s.dtype == NYS_BF16) {
    rows_tc_split(s, rows_tc_ctas(s), &L.splits, &L.tiles_per_split);
  } else if (x3_supported(s)) {
    x3_rows_split(s, &L.splits, &L.tiles_per_split);
  } else {
    const long long rb = (s.m + 7) / 8;
    const long long sms = plan_sms();
    long long want = (4 * sms + rb * (long long)bh - 1) / (rb * (long long)bh);
    long long cap = s.n / 32 > 0 ? s.n / 32 : 1;
    if (want > cap) want = cap;
    if (want < 1) want = 1;
    if (want > 1024) want = 1024;
    L.splits = (int)want;
  }
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
  L.status = take(256);
  L.q_tilde = take(bh * md * 4);
  L.k_tilde = take(bh * md * 4);
  L.g_part = take(bh * L.splits * md * 4);
  L.g_ml = take(bh * L.splits * s.m * 2 * 4);
  L.g = take(bh * md * 4);
  L.a_s = take(bh * mm * 4);
  L.z = take(bh * mm * 4);
  L.w = take(bh * md * 4);
  L.scratch = take(bh * scratch_mats(s) * mm * 4);
  const size_t pad_bf16 = s.dtype == NYS_BF16 ? bh * (size_t)s.m64() * s.dpad() * 2 : 0;
  L.qt_bf16 = take(pad_bf16);
  L.kt_bf16 = take(pad_bf16);
  L.wt_bf16 = take(pad_bf16);
  L.lengths = take((size_t)s.B * 4);
  L.total = off;
  return L;
}

}  // namespace nys

using namespace nys;

extern "C" {

size_t nystrom_attn_workspace_bytes(int B, int H, int n, int d, int m, int dtype) {
  if (check_shape(B, H, n, d, m, 0, 0, dtype) != NYS_OK) return 0;
  Shape s{B, H, n, d, m, 0, 0, dtype};
  return make_layout(s).total;
}

long long nystrom_attn_stage_offset(int B, int H, int n, int d, int m, int dtype, int stage) {
  if (check_shape(B, H, n, d, m, 0, 0, dtype) != NYS_OK) return -1;
  Shape s{B, H, n, d, m, 0, 0, dtype};
  const Layout L = make_layout(s);
  switch (stage) {
    case NYS_STAGE_Q_TILDE: return (long long)L.q_tilde;
    case NYS_STAGE_K_TILDE: return (long long)L.k_tilde;
    case NYS_STAGE_G: return (long long)L.g;
    case NYS_STAGE_A_S: return (long long)L.a_s;
    case NYS_STAGE_W: return (long long)L.w;
    case NYS_STAGE_Z: return (long long)L.z;
    default: return -1;
  }
}

int nystrom_plan_describe(int B, int H, int n, int d, int m, int iters, int conv_ks, int dtype,
                          char* buf, int len) {
  const int rc = check_shape(B, H, n, d, m, iters, conv_ks, dtype);
  if (rc != NYS_OK) return rc;
  if (len < 0 || (len > 0 && !buf)) return NYS_ERR_ARG;
  const std::string text = describe_plan(Shape{B, H, n, d, m, iters, conv_ks, dtype});
  if (len > 0) {
    const size_t c = text.size() < (size_t)len - 1 ? text.size() : (size_t)len - 1;
    memcpy(buf, text.data(), c);
    buf[c] = '\0';
  }
  return (int)text.size();
}

int nystrom_attn_fwd_ws(const void* q, const void* k, const void* v, const float* conv_w,
                        void* out, int B, int H, int n, int d, int m, int iters, int conv_ks,
                        int dtype, void* workspace, size_t ws_bytes, nys_stream_t stream) {
  int rc = check_args(q, k, v, conv_w, out, B, H, n, d, m, iters, conv_ks, dtype);
  if (rc != NYS_OK) return rc;
  if (!workspace) return NYS_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return NYS_ERR_ALIGN;
  Shape s{B, H, n, d, m, iters, conv_ks, dtype};
  if (ws_bytes < make_layout(s).total) return NYS_ERR_NOMEM;
  int dev = 0;
  rc = check_device(&dev);
  if (rc != NYS_OK) return rc;
  return run(s, q, k, v, conv_w, out, static_cast<char*>(workspace), stream, dev);
}

int nystrom_attn_fwd(const void* q, const void* k, const void* v, const float* conv_w, void* out,
                     int B, int H, int n, int d, int m, int iters, int conv_ks, int dtype,
                     nys_stream_t stream) {
  int rc = check_args(q, k, v, conv_w, out, B, H, n, d, m, iters, conv_ks, dtype);
  if (rc != NYS_OK) return rc;
  int dev = 0;
  rc = check_device(&dev);
  if (rc != NYS_OK) return rc;
  Shape s{B, H, n, d, m, iters, conv_ks, dtype};
  const Layout L = make_layout(s);
  char* ws = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_dev[dev].mu);
    rc = ensure_buffer(&g_dev[dev].ws, &g_dev[dev].ws_bytes, L.total, stream);
    if (rc != NYS_OK) return rc;
    ws = static_cast<char*>(g_dev[dev].ws);
  }
  return run(s, q, k, v, conv_w, out, ws, stream, dev);
}

int nystrom_attn_fwd_ex(const void* q, const void* k, const void* v, const float* conv_w,
                        void* out, int B, int H, int n, int d, int m, int iters, int conv_ks,
                        int dtype, int conv_layout, const int* lengths_host, void* workspace,
                        size_t ws_bytes, nys_stream_t stream) {
  int rc = check_args(q, k, v, conv_w, out, B, H, n, d, m, iters, conv_ks, dtype);
  if (rc != NYS_OK) return rc;
  if (conv_layout != NYS_CONV_PER_HEAD && conv_layout != NYS_CONV_PER_CHANNEL) return NYS_ERR_ARG;
  if (lengths_host)
    for (int b = 0; b < B; ++b)
      if (lengths_host[b] < m || lengths_host[b] > n) return NYS_ERR_SHAPE;
  Shape s{B, H, n, d, m, iters, conv_ks, dtype};
  s.conv_layout = conv_layout;
  const Layout L = make_layout(s);
  if (workspace) {
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return NYS_ERR_ALIGN;
    if (ws_bytes < L.total) return NYS_ERR_NOMEM;
  }
  int dev = 0;
  rc = check_device(&dev);
  if (rc != NYS_OK) return rc;
  char* ws = static_cast<char*>(workspace);
  if (!ws) {
    std::lock_guard<std::mutex> lk(g_dev[dev].mu);
    rc = ensure_buffer(&g_dev[dev].ws, &g_dev[dev].ws_bytes, L.total, stream);
    if (rc != NYS_OK) return rc;
    ws = static_cast<char*>(g_dev[dev].ws);
  }
  if (lengths_host) {
    // ordered on the stream before the kernels that read it; the host array
    // may be reused as soon as the call returns
    const cudaError_t e = cudaMemcpyAsync(ws + L.lengths, lengths_host, (size_t)B * sizeof(int),
                                          cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return set_cuda_error(e);
    s.lengths = reinterpret_cast<const int*>(ws + L.lengths);
  }
  return run(s, q, k, v, conv_w, out, ws, stream, dev);
}

int nystrom_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                          const float* conv_w_host, void* out_host, int B, int H, int n, int d,
                          int m, int iters, int conv_ks, int dtype, nys_stream_t stream) {
  if (!q_host || !k_host || !v_host || !out_host || (conv_ks > 0 && !conv_w_host))
    return NYS_ERR_ARG;
  int rc = check_shape(B, H, n, d, m, iters, conv_ks, dtype);
  if (rc != NYS_OK) return rc;
  int dev = 0;
  rc = check_device(&dev);
  if (rc != NYS_OK) return rc;
  DeviceCache& dc = g_dev[dev];
  std::lock_guard<std::mutex> host_lk(dc.host_mu);
  const size_t esz = dtype == NYS_FP32 ? 4 : 2;
  const size_t elems = (size_t)B * H * n * d;
  const size_t tb = align256(elems * esz);
  const size_t wb = align256((size_t)H * (conv_ks > 0 ? conv_ks : 1) * 4);
  char* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(dc.mu);
    rc = ensure_buffer(&dc.stage, &dc.stage_bytes, 4 * tb + wb, stream);
    if (rc != NYS_OK) return rc;
    base = static_cast<char*>(dc.stage);
  }
  char *dq = base, *dk = base + tb, *dv = base + 2 * tb, *dout = base + 3 * tb;
  float* dw = reinterpret_cast<float*>(base + 4 * tb);
  cudaError_t e = cudaSuccess;
  if (!dc.h2d) {
    e = cudaStreamCreateWithFlags(&dc.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&dc.d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&dc.ev_start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&dc.ev_done, cudaEventDisableTiming);
    for (int c = 0; c < kHostChunks && e == cudaSuccess; ++c) {
      e = cudaEventCreateWithFlags(&dc.ev_in[c], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&dc.ev_comp[c], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  // Pipeline over chunks: chunk c's inputs go up on the h2d stream while
  // chunk c - 1 is computed on `stream` and chunk c - 2's output comes back
  // on the d2h stream (the two copy directions overlap; uploading q, k and v
  // on separate streams was slower). A chunk is a range of heads that are
  // contiguous in [B][H] (whole batch entries when B is large, else an
  // equal split of each entry's heads), so that the last chunk's compute
  // and download, which nothing overlaps, are short.
  int per_b = 1;  // chunks per batch entry (a divisor of H)
  if (B < kHostChunks) {
    per_b = (kHostChunks + B - 1) / B;
    while (per_b > 1 && H % per_b != 0) --per_b;
  }
  int bc = 1;  // batch entries per chunk (when per_b == 1)
  if (per_b == 1) {
    int chunks_b = B < kHostChunks ? B : kHostChunks;
    while (B % chunks_b != 0) --chunks_b;
    bc = B / chunks_b;
  }
  const int hc = H / per_b;  // heads per chunk (per_b > 1)
  const int chunks = per_b > 1 ? B * per_b : B / bc;
  const size_t cbytes = (per_b > 1 ? (size_t)hc : (size_t)bc * H) * n * d * esz;
  const Shape sc = per_b > 1 ? Shape{1, hc, n, d, m, iters, conv_ks, dtype}
                             : Shape{bc, H, n, d, m, iters, conv_ks, dtype};
  char* ws = nullptr;
  {
    std::lock_guard<std::mutex> lk(dc.mu);
    rc = ensure_buffer(&dc.ws, &dc.ws_bytes, make_layout(sc).total, stream);
    if (rc != NYS_OK) return rc;
    ws = static_cast<char*>(dc.ws);
  }
  if ((e = cudaEventRecord(dc.ev_start, stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(dc.h2d, dc.ev_start, 0)) != cudaSuccess)
    return set_cuda_error(e);
  if (conv_ks > 0 &&
      (e = cudaMemcpyAsync(dw, conv_w_host, (size_t)H * conv_ks * 4, cudaMemcpyHostToDevice,
                           dc.h2d)) != cudaSuccess)
    return set_cuda_error(e);
  for (int c = 0; c < chunks; ++c) {
    const size_t off = (size_t)c * cbytes;
    if ((e = cudaMemcpyAsync(dq + off, static_cast<const char*>(q_host) + off, cbytes,
                             cudaMemcpyHostToDevice, dc.h2d)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dk + off, static_cast<const char*>(k_host) + off, cbytes,
                             cudaMemcpyHostToDevice, dc.h2d)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dv + off, static_cast<const char*>(v_host) + off, cbytes,
                             cudaMemcpyHostToDevice, dc.h2d)) != cudaSuccess ||
        (e = cudaEventRecord(dc.ev_in[c], dc.h2d)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, dc.ev_in[c], 0)) != cudaSuccess)
      return set_cuda_error(e);
    // the chunks share the library workspace (in stream order) and its
    // status word, which only the first clears
    // a head-range chunk's conv filters: rows h0 .. of [H][ks]
    const int h0 = per_b > 1 ? (c % per_b) * hc : 0;
    rc = run(sc, dq + off, dk + off, dv + off, conv_ks > 0 ? dw + (size_t)h0 * conv_ks : nullptr,
             dout + off, ws, stream, dev, c == 0);
    if (rc != NYS_OK) return rc;
    if ((e = cudaEventRecord(dc.ev_comp[c], stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(dc.d2h, dc.ev_comp[c], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(static_cast<char*>(out_host) + off, dout + off, cbytes,
                             cudaMemcpyDeviceToHost, dc.d2h)) != cudaSuccess)
      return set_cuda_error(e);
  }
  if ((e = cudaEventRecord(dc.ev_done, dc.d2h)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(stream, dc.ev_done, 0)) != cudaSuccess ||
      (e = cudaStreamSynchronize(stream)) != cudaSuccess)
    return set_cuda_error(e);
  return NYS_OK;
}

int nystrom_get_status(nys_stream_t stream) {
  int dev = 0;
  int rc = check_device(&dev);
  if (rc != NYS_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return set_cuda_error(e);
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_dev[dev].mu);
    ws = g_dev[dev].last_ws;
  }
  if (!ws) return NYS_OK;
  int status = 0;
  if ((e = cudaMemcpy(&status, ws, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return set_cuda_error(e);
  if (status != 0 && (e = cudaMemset(ws, 0, sizeof(int))) != cudaSuccess) return set_cuda_error(e);
  return status;
}

const char* nystrom_strerror(int code) {
  switch (code) {
    case NYS_OK: return "ok";
    case NYS_ERR_ARG: return "invalid argument (NULL pointer, bad dtype)";
    case NYS_ERR_SHAPE: return "shape outside the supported set";
    case NYS_ERR_ALIGN: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case NYS_ERR_UNSUPPORTED: return "no compute capability 10.3 GPU is current";
    case NYS_ERR_NOMEM: return "workspace allocation failed or too small";
    case NYS_ERR_CUDA: return "CUDA runtime error";
    case NYS_ERR_TIMEOUT: return "a device-side bounded wait ran out";
    default: return "unknown status code";
  }
}

const char* nystrom_last_error_string(void) { return g_last_error.c_str(); }

int nystrom_debug_stall_pinv(int on) {
  if (on != 0 && on != 1) return NYS_ERR_ARG;
  g_stall_ns.store(on ? 1000000u : 0u);  // 1 ms
  return NYS_OK;
}

}  // extern "C"
