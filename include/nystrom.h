/*
 * nystrom.h - C ABI of the Nyström self-attention forward library
 * (libnystrom.so, CUDA, sm_103a).
 *
 * What it computes, per head (b, h) of q, k, v in [B, H, n, d]:
 *
 *   Q~, K~ = segment means of Q and K over m contiguous segments; segment
 *            i is rows [floor(i n/m), floor((i+1) n/m)), i.e. n/m rows each
 *            when m divides n, else floor(n/m) or ceil(n/m) rows
 *            ("Nyströmformer" review page, Proposed method, bullet 4)
 *   A_S    = softmax(Q~ K~^T / sqrt(d))                       (bullet 2)
 *   Z      = iterative Moore-Penrose inverse of A_S, `iters` updates of
 *            Z <- 1/4 Z (13I - A_S Z (15I - A_S Z (7I - A_S Z)))
 *            from Z_0 = A_S^T / (||A_S||_1 ||A_S||_inf)       (bullet 5)
 *   out    = softmax(Q K~^T / sqrt(d)) Z softmax(Q~ K^T / sqrt(d)) V
 *            + DWConv(V)                                      (bullets 3, 6)
 *
 * DWConv is a depthwise convolution along the sequence: one odd-width filter
 * of conv_ks taps per head, shared by the d channels, cross-correlation with
 * (conv_ks-1)/2 zero rows of padding on each side, no bias:
 *   conv[t] = sum_{j<conv_ks} conv_w[h][j] * V[t + j - (conv_ks-1)/2].
 * conv_ks = 0 drops the term (the output is then the attention alone).
 *
 * Conventions shared by every entry point below:
 *  - Device pointers unless a name says "host". The caller owns every
 *    buffer; the library never frees or keeps a caller pointer.
 *  - q, k, v, out: [B][H][n][d] contiguous, d innermost, element type
 *    `dtype` (NYS_FP32: float; NYS_BF16: bfloat16 bit patterns). Each base
 *    address 16-byte aligned. out is fully overwritten; it may not alias
 *    q, k or v.
 *  - conv_w: [H][conv_ks] float32 (for both dtypes); may be NULL when
 *    conv_ks == 0.
 *  - Shape rules (else NYS_ERR_SHAPE, nothing launched): B, H, n, d, m >= 1;
 *    m <= n; m <= 256; d % 8 == 0 and d <= 128; for NYS_BF16 also
 *    d in {32, 64, 128}; 0 <= iters <= 64; conv_ks == 0 or odd and <= 127;
 *    B*H*n*d < 2^40.
 *  - Scale: every softmax uses 1/sqrt(d).
 *  - Asynchrony: compute entry points enqueue work on `stream` (0 = the
 *    legacy default stream) and return without waiting. A negative return
 *    means nothing was enqueued (argument errors) or that a launch failed
 *    (NYS_ERR_CUDA; see nystrom_last_error_string). Device-side failures
 *    (a bounded wait that ran out) are reported by nystrom_get_status after
 *    the stream has finished.
 *  - Thread safety: calls may come from several host threads; the cached
 *    workspace of nystrom_attn_fwd is shared per device, so concurrent calls
 *    on different streams of one device must use nystrom_attn_fwd_ws with
 *    their own workspaces.
 */
#ifndef NYSTROM_H_
#define NYSTROM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t. */
typedef struct CUstream_st* nys_stream_t;

typedef enum { NYS_FP32 = 0, NYS_BF16 = 1 } nys_dtype_t;

typedef enum {
  NYS_OK = 0,
  NYS_ERR_ARG = -1,         /* NULL pointer, bad dtype, negative size      */
  NYS_ERR_SHAPE = -2,       /* shape outside the rules above               */
  NYS_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned            */
  NYS_ERR_UNSUPPORTED = -4, /* no GPU of compute capability 10.3 current   */
  NYS_ERR_NOMEM = -5,       /* workspace allocation failed / too small     */
  NYS_ERR_CUDA = -6,        /* a CUDA runtime call or launch failed        */
  NYS_ERR_TIMEOUT = -7      /* a device-side bounded wait ran out          */
} nys_status_t;

/*
 * nystrom_attn_fwd - the forward pass (see the top of this file).
 * Uses a workspace the library allocates and caches per device (grown with
 * cudaMalloc when a call needs more; growing synchronises the device).
 * iters: number of pseudo-inverse updates ("about 6", Proposed method,
 * bullet 5); run exactly, no early exit. For NYS_BF16 inputs up to 8 updates
 * run on the tensor cores (tf32 products, fp32 storage); with more, the
 * pseudo-inverse runs in fp32 on the CUDA cores, since the iteration
 * amplifies tf32 rounding by the condition number of A_S as it inverts more
 * of its small singular values (slower, same result bar).
 * Returns NYS_OK or a negative nys_status_t.
 */
int nystrom_attn_fwd(const void* q, const void* k, const void* v,
                     const float* conv_w, void* out, int B, int H, int n,
                     int d, int m, int iters, int conv_ks, int dtype,
                     nys_stream_t stream);

/*
 * nystrom_attn_workspace_bytes - bytes of device workspace that
 * nystrom_attn_fwd_ws needs for this shape (0 if the shape is invalid).
 * Host arithmetic only; launches nothing. The size depends on the SM count
 * of the current device (the plan spreads work over its SMs; 152, a GB300,
 * when no device can be queried), so ask with the device current that will
 * run the call.
 */
size_t nystrom_attn_workspace_bytes(int B, int H, int n, int d, int m,
                                    int dtype);

/*
 * nystrom_attn_fwd_ws - as nystrom_attn_fwd, with a caller-owned device
 * workspace of ws_bytes >= nystrom_attn_workspace_bytes(...) bytes,
 * 256-byte aligned. The library allocates nothing. The workspace must stay
 * valid and unused by others until the stream has finished the call.
 * Returns NYS_ERR_NOMEM if ws_bytes is too small.
 */
int nystrom_attn_fwd_ws(const void* q, const void* k, const void* v,
                        const float* conv_w, void* out, int B, int H, int n,
                        int d, int m, int iters, int conv_ks, int dtype,
                        void* workspace, size_t ws_bytes, nys_stream_t stream);

/*
 * nystrom_attn_fwd_noalloc - as nystrom_attn_fwd, but allocates nothing:
 * no cudaMalloc, cudaFree or allocating library call. The paper has no
 * counterpart; this entry point exists for callers that cannot allocate
 * device memory at call time, such as plugins inside a host application that
 * owns all device memory through its own allocator, or latency-critical
 * loops where a cudaMalloc/cudaFree would synchronise the device.
 * Its scratch is a fixed 32 MiB device array inside the library, reserved on
 * every GPU that loads the library until the process exits. Shapes whose
 * workspace (nystrom_attn_workspace_bytes) exceeds 32 MiB are rejected with
 * NYS_ERR_NOMEM before anything is enqueued.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture. The first call on a device of a shape whose plan runs on more
 * than one stream (see nystrom_plan_describe) also creates the library's
 * auxiliary streams and events for that device, as every entry point does;
 * they hold no device memory of the caller's and live until exit. All calls
 * share the one array and it keeps the previous call's
 * contents; the library clears what must start at zero on every call. Calls
 * that overlap on the GPU (different streams, or different host threads,
 * same device) race on the array: serialise them.
 */
int nystrom_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                             const float* conv_w, void* out, int B, int H,
                             int n, int d, int m, int iters, int conv_ks,
                             int dtype, nys_stream_t stream);

/*
 * nystrom_attn_fwd_ex - the forward pass with the two variants the page
 * leaves open (Proposed method, bullets 4 and 6), as readings of it:
 *  - conv_layout NYS_CONV_PER_HEAD: conv_w is [H][conv_ks], one filter per
 *    head shared by its d channels (as nystrom_attn_fwd);
 *    NYS_CONV_PER_CHANNEL: conv_w is [H][d][conv_ks] float32, channel c of
 *    head h has its own taps conv_w[h][c][.] ("depthwise": one filter per
 *    channel).
 *  - lengths_host: HOST int32 [B], or NULL. Batch entry b holds
 *    lengths_host[b] real tokens in rows [0, lengths_host[b]) of its n rows,
 *    the rest is padding, which takes part in nothing: the landmarks are the
 *    segment means of the real tokens (segments over lengths_host[b] rows),
 *    padded keys are masked out of softmax(Q~ K^T / sqrt(d)), padded rows of
 *    V read as zero in the convolution, and the output rows of padding are
 *    zero. The real rows' result equals that of the unpadded sequence. Each
 *    length must satisfy m <= lengths_host[b] <= n (else NYS_ERR_SHAPE).
 *    Padded rows of q, k, v must hold finite values (they are read, then
 *    masked). The array is copied to the device inside the call.
 * workspace: caller-owned device workspace of ws_bytes >=
 * nystrom_attn_workspace_bytes(...) bytes, 256-byte aligned, as for
 * nystrom_attn_fwd_ws; or NULL to use the library's cached workspace (as
 * nystrom_attn_fwd does).
 * With NYS_CONV_PER_HEAD and no lengths the result is that of
 * nystrom_attn_fwd. The variants run the token pass for the attention term
 * alone and add the convolution (and zero the padding rows) in a pass of
 * their own, on the CUDA cores.
 * Returns NYS_OK or a negative nys_status_t (NYS_ERR_ARG for an unknown
 * conv_layout).
 */
typedef enum { NYS_CONV_PER_HEAD = 0, NYS_CONV_PER_CHANNEL = 1 } nys_conv_layout_t;
int nystrom_attn_fwd_ex(const void* q, const void* k, const void* v,
                        const float* conv_w, void* out, int B, int H, int n,
                        int d, int m, int iters, int conv_ks, int dtype,
                        int conv_layout, const int* lengths_host,
                        void* workspace, size_t ws_bytes, nys_stream_t stream);

/*
 * nystrom_mha_fwd - the multi-head attention module around the op (the
 * page's model uses Nyström self-attention in place of softmax attention,
 * abstract and Proposed method bullet 6): with D = H*d,
 *   [Q | K | V] = x w_qkv + b_qkv,  Q, K, V split into H heads of d columns
 *   (head h = columns [h*d, (h+1)*d) of each), O_h = the forward pass of the
 *   top of this file on head h (m landmarks, iters updates, conv_w [H][conv_ks]),
 *   y = [O_1 | ... | O_H] w_o + b_o.
 * x, y: [B][n][D], w_qkv: [D][3D] (columns: the Q block, then K, then V),
 * w_o: [D][D], all row-major in `dtype` (device); b_qkv [3D] and b_o [D]
 * float32 device arrays, or NULL for no bias. Pointers 16-byte aligned.
 * The projections run in cuBLAS (fp32 accumulation into the workspace); the
 * head split and merge, the biases and the attention in this library's
 * kernels. No residual connection, normalisation or dropout: those belong to
 * the layer around the module.
 * workspace: device, 256-byte aligned, ws_bytes >= nystrom_mha_workspace_bytes,
 * or NULL to use a buffer the library allocates and caches per device.
 * Returns NYS_OK or a negative nys_status_t (shape rules as the top of this
 * file, with n, H, d, m of the attention).
 */
size_t nystrom_mha_workspace_bytes(int B, int n, int H, int d, int m, int dtype);
int nystrom_mha_fwd(const void* x, const void* w_qkv, const float* b_qkv,
                    const void* w_o, const float* b_o, const float* conv_w,
                    void* y, int B, int n, int H, int d, int m, int iters,
                    int conv_ks, int dtype, void* workspace, size_t ws_bytes,
                    nys_stream_t stream);

/*
 * Clustered attention, centroid path ("Fast Transformers with Clustered
 * Attention" review page, Proposed method, bullets 1, 2 and 4): per head
 * (b, h) the queries Q [n, d] are grouped into C clusters by K-means and
 * attention is computed once per centroid:
 *   mu      = segment means of Q over C contiguous segments (as Q~ above)
 *   iters x:  a(i) = argmin_c |q_i - mu_c|^2 (ties: the lowest c), then
 *             mu_c = mean of the queries with a(i) = c (none: unchanged)
 *   out[i]  = softmax(mu_{a(i)} K^T / sqrt(d)) V
 * K-means: for NYS_BF16 with d in {64, 128} and C <= 128 on the tensor
 * cores (distances to fp32 accuracy: the centroids split into three bf16
 * terms; the members' sums as a one-hot product with fp32 accumulation,
 * added across CTAs in a fixed order: deterministic), otherwise in fp32 on
 * the CUDA cores (the update sums a cluster's queries in index order). The
 * centroid rows run in the landmark-row kernels of the forward pass (bf16
 * tensor cores for NYS_BF16, with the centroids rounded to bf16; fp32 CUDA
 * cores for NYS_FP32).
 * q, k, v, out: [B][H][n][d] in `dtype`, device, 16-byte aligned; shape rules
 * as the top of this file with C in place of m; 1 <= iters <= 64.
 * workspace: device, 256-byte aligned, ws_bytes >=
 * nystrom_clustered_workspace_bytes(...), or NULL for the library's cached
 * workspace. Asynchronous on `stream`; nystrom_get_status reports bounded
 * waits that ran out.
 * nystrom_clustered_stage_offset: byte offset in the workspace, after a
 * call with these sizes has finished, of NYS_CSTAGE_ASSIGN (int32
 * [B*H][n], the last assignment), NYS_CSTAGE_CENTROIDS_PREV (float32
 * [B*H][C][d], the centroids that assignment used), NYS_CSTAGE_CENTROIDS
 * (float32 [B*H][C][d], after the last update), NYS_CSTAGE_G (float32
 * [B*H][C][d], the centroid rows); -1 for invalid sizes or stage.
 */
typedef enum {
  NYS_CSTAGE_ASSIGN = 0,
  NYS_CSTAGE_CENTROIDS_PREV = 1,
  NYS_CSTAGE_CENTROIDS = 2,
  NYS_CSTAGE_G = 3
} nys_cstage_t;
size_t nystrom_clustered_workspace_bytes(int B, int H, int n, int d, int C,
                                         int dtype);
long long nystrom_clustered_stage_offset(int B, int H, int n, int d, int C,
                                         int iters, int dtype, int stage);
int nystrom_clustered_attn_fwd(const void* q, const void* k, const void* v,
                               void* out, int B, int H, int n, int d, int C,
                               int iters, int dtype, void* workspace,
                               size_t ws_bytes, nys_stream_t stream);

/*
 * nystrom_attn_fwd_host - the whole forward pass from and to HOST memory:
 * copies q, k, v, conv_w to the device, runs the forward pass on `stream`,
 * copies out back and waits for the stream. The batch is processed in up
 * to four chunks of whole batch entries, pipelined: a chunk's inputs are
 * copied up (on a library stream) while the previous chunk is computed on
 * `stream` and the one before it is copied back (on another library
 * stream). Host buffers should be pinned (page-locked) for full copy speed;
 * pageable memory works but is slower. Device staging buffers are
 * allocated and cached per device (grown with cudaMalloc when needed); one
 * host-entry call per device runs at a time. Synchronous: out_host is
 * complete on return; nystrom_get_status then reports the status of all
 * chunks.
 */
int nystrom_attn_fwd_host(const void* q_host, const void* k_host,
                          const void* v_host, const float* conv_w_host,
                          void* out_host, int B, int H, int n, int d, int m,
                          int iters, int conv_ks, int dtype,
                          nys_stream_t stream);

/*
 * Stage export, for testing the intermediate results against a reference.
 * After a nystrom_attn_fwd_ws call has finished, the workspace holds, as
 * float32 arrays per head (b*H + h major):
 *   NYS_STAGE_Q_TILDE [m][d], NYS_STAGE_K_TILDE [m][d], NYS_STAGE_G [m][d]
 *   (= softmax(Q~ K^T/sqrt d) V), NYS_STAGE_A_S [m][m], NYS_STAGE_W [m][d]
 *   (= Z G), NYS_STAGE_Z [m][m] (Z after `iters` updates).
 * nystrom_attn_stage_offset returns the byte offset of `stage` in the
 * workspace for this shape, or -1 for an invalid shape or stage.
 */
typedef enum {
  NYS_STAGE_Q_TILDE = 0,
  NYS_STAGE_K_TILDE = 1,
  NYS_STAGE_G = 2,
  NYS_STAGE_A_S = 3,
  NYS_STAGE_W = 4,
  NYS_STAGE_Z = 5
} nys_stage_t;
long long nystrom_attn_stage_offset(int B, int H, int n, int d, int m,
                                    int dtype, int stage);

/*
 * nystrom_plan_describe - the kernels a forward call of this shape
 * launches, in order, as one line of text: the plan ("serial": each step
 * after the previous one; "z-beside-rows": the pseudo-inverse's chain of
 * products on a second stream beside the landmark-row pass, then the merge
 * of G and W = Z G; "head-groups": the batch split into groups of whole
 * batch entries, each group's steps on its own stream), the number of head
 * groups, and per step the kernel with its host-side sizes (the landmark-row
 * pass's CTAs, key ranges per head and 128-key tiles per CTA; the
 * pseudo-inverse's CTAs and, beside the rows, the SMs they take). The plan is
 * a function of the shape and of the current device's SM count (152, a
 * GB300, when no device can be queried).
 * Host only: launches nothing.
 * buf: host memory of `len` bytes (may be NULL when len == 0); receives at
 * most len - 1 characters and a terminating NUL.
 * Returns the length of the full description (without the NUL), or a
 * negative nys_status_t: NYS_ERR_SHAPE / NYS_ERR_ARG for a shape the forward
 * call would reject, NYS_ERR_ARG for len < 0 or a NULL buf with len > 0.
 */
int nystrom_plan_describe(int B, int H, int n, int d, int m, int iters,
                          int conv_ks, int dtype, char* buf, int len);

/*
 * nystrom_get_status - waits for `stream`, then returns and clears the
 * device-side status word of the most recent call on the current device
 * (NYS_OK, or NYS_ERR_TIMEOUT if a bounded wait inside a kernel ran out).
 * Returns NYS_ERR_CUDA if the stream reports an error.
 */
int nystrom_get_status(nys_stream_t stream);

/*
 * Launch accounting and per-kernel timing, for benchmarks.
 * nystrom_launch_count: kernels this library has launched in this process
 * (all devices, all threads).
 * nystrom_profile_enable(1): from now on every kernel launch is bracketed
 * by two CUDA events recorded on the launch's own stream (adds two event
 * records per launch). nystrom_profile_enable(0) stops recording.
 * nystrom_profile_read: waits for the recorded events, returns the number of
 * distinct kernels seen since the last read (at most max_kernels are
 * written), and for kernel i writes its name to names + i*name_len
 * (NUL-terminated, truncated), its summed duration in ms to total_ms[i] and
 * its launch count to launches[i]; then forgets the records. Returns
 * NYS_ERR_CUDA if an event query fails.
 */
unsigned long long nystrom_launch_count(void);
int nystrom_profile_enable(int on);
int nystrom_profile_read(int max_kernels, char* names, int name_len,
                         double* total_ms, long long* launches);

/*
 * nystrom_debug_stall_pinv - testing the device-side timeout path. With
 * on = 1, every later forward call whose pseudo-inverse runs in the
 * tensor-core kernel for m <= 128 (bf16 inputs) makes that kernel wait, at
 * its start and before any copy or product is in flight, on a barrier phase
 * that nothing completes; the bounded wait runs out after 1 ms, the kernel
 * records NYS_ERR_TIMEOUT in the status word and skips its remaining work
 * (its outputs, and the call's output, are then undefined), and
 * nystrom_get_status reports NYS_ERR_TIMEOUT with the CUDA context intact.
 * on = 0 (the default) turns it off. Process-wide; not for production use.
 * Returns NYS_OK, or NYS_ERR_ARG for on other than 0 or 1.
 */
int nystrom_debug_stall_pinv(int on);

/* Static description of a status code. Never NULL. */
const char* nystrom_strerror(int code);

/* Text of the last CUDA error seen by this host thread ("" if none). */
const char* nystrom_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* NYSTROM_H_ */
