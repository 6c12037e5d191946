/*
 * dit_attn — dense, non-causal, multi-head softmax attention forward for the
 * joint text+image token sequence of a diffusion transformer, on NVIDIA B300
 * (sm_103a).
 *
 * The operation is standard attention, the dense BF16 attention that "Speed Up
 * Image Generation with FLUX 3 Image Klein on NVIDIA Blackwell GPUs" (Key
 * takeaways, second item) and the diegocecato.dcsolution.it article
 * "flux-3-blackwell-denoising-latenza-pipeline" (section "NVFP4, attention e
 * caching") put at about 60% of DiT kernel time at 2048x2048.  For every
 * batch b, head h and query row i:
 *
 *     s_ij = scale * sum_c q[b,h,i,c] * k[b,h,j,c]        (j < Lk, no mask)
 *     o[b,h,i,:] = sum_j softmax_j(s_ij) * v[b,h,j,:]
 *
 * The text, image and reference-image tokens of a DiT block form one
 * sequence; every query sees every key.
 *
 * Tensors (all owned by the caller; the library never allocates):
 *   q   : device pointer, bf16, contiguous [B, H, Lq, d]
 *   k, v: device pointers, bf16, contiguous [B, H, Lk, d]
 *   out : device pointer, bf16, contiguous [B, H, Lq, d]; written, never read
 * Every pointer must be 16-byte aligned; out must not overlap q, k or v.
 * (The e4m3 entry points below take one-byte e4m3 codes for q and k, or for
 * q, k and v, with per-tensor scales.)
 * d must be 64 or 128.  Arithmetic: bf16 tensor-core products with fp32
 * accumulation, fp32 online softmax, probabilities rounded to bf16 before the
 * P.V product, output rounded to nearest-even bf16.
 *
 * Streams: work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 * default stream).  No call synchronises, except dit_attn_get_device_error.
 * The forward calls keep no per-call device state of their own (the split
 * tail's workspace belongs to the caller), so calls on different streams may
 * overlap; dit_attn_forward_noalloc is the exception (its scratch is shared).
 *
 * Errors: every entry point returns a dit_attn_status.  Argument checks run
 * before any CUDA call, so an invalid call has no side effect.
 */
#ifndef DIT_ATTN_H
#define DIT_ATTN_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dit_attn_status {
  DIT_ATTN_OK = 0,
  DIT_ATTN_ERR_INVALID_ARG = 1,     /* null / misaligned pointer, size < 1, unusable scale, overlap */
  DIT_ATTN_ERR_UNSUPPORTED = 2,     /* head dim other than 64 or 128; sizes beyond the limits */
  DIT_ATTN_ERR_NOT_INITIALIZED = 3, /* dit_attn_create() not called for the current device */
  DIT_ATTN_ERR_NO_DEVICE = 4,       /* no CUDA device, or the current device is not sm_103 */
  DIT_ATTN_ERR_CUDA = 5,            /* a CUDA runtime/driver call failed; see dit_attn_last_cuda_error */
  DIT_ATTN_ERR_TIMEOUT = 6          /* a kernel gave up a bounded wait (reported by get_device_error) */
} dit_attn_status;

/* Library version, e.g. 100 for 0.1.0. */
int dit_attn_version(void);

/*
 * Prepare the current CUDA device: checks that it is compute capability 10.3,
 * reads its SM count, raises the kernels' dynamic shared-memory limit and
 * resolves the CUDA driver's tensor-map encoder.  Idempotent and thread-safe; call
 * once per device before dit_attn_forward.  Returns NO_DEVICE when no usable
 * device is present.
 */
int dit_attn_create(void);

/*
 * out = softmax(q k^T * scale) v for every (batch, head), enqueued on stream.
 *   B, H, Lq, Lk >= 1; B*H < 2^31; Lq, Lk <= 2^31 - 513;
 *   B*H*ceil(Lq/256) < 2^31 (else UNSUPPORTED).
 *   d in {64, 128}.
 *   scale finite, of either sign (1/sqrt(d) for a standard transformer), with
 *   |scale| * log2(e) within fp32 range, i.e. |scale| <= 2.35e38 (else
 *   INVALID_ARG).  The kernels form scale * log2(e) * (q . k) in fp32; logits
 *   beyond fp32 range (only possible with extreme scales or inputs) give
 *   unspecified outputs.
 * Asynchronous: returns after the launch.  A launch failure returns
 * DIT_ATTN_ERR_CUDA; a device-side wait that gave up is reported later by
 * dit_attn_get_device_error.
 */
int dit_attn_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int Lq,
                     int Lk, int d, float scale, void* stream);

/*
 * dit_attn_forward with a caller-owned workspace for the split tail.  A
 * persistent launch runs the 512-row work units in waves of one unit per CTA
 * pair; when the last wave is partial, its units are cut into key ranges
 * whose unnormalised partial results (output, running max, row sum) go to the
 * workspace and are merged by a second kernel on the same stream, so the last
 * wave fills the GPU.  The result equals dit_attn_forward's within rounding
 * (not bit for bit: the partial sums are added in another order).
 *   workspace: device pointer, 16-byte aligned, must not overlap q, k, v or
 *              out; NULL with workspace_bytes 0 runs without splitting.
 *   workspace_bytes: its size; when smaller than dit_attn_workspace_size
 *              reports, the call runs without splitting.
 * The workspace is scratch for this call only: calls that may overlap (other
 * streams) need separate workspaces.  Otherwise as dit_attn_forward.
 */
int dit_attn_forward_ws(const void* q, const void* k, const void* v, void* out, int B, int H,
                        int Lq, int Lk, int d, float scale, void* workspace,
                        long long workspace_bytes, void* stream);

/*
 * dit_attn_forward for callers that cannot allocate device memory while they
 * run: an inference engine that reserves all device memory up front and
 * forbids later allocations, code running inside a memory allocator's own
 * callback, or a latency-bound loop that must not enter cudaMalloc (which can
 * synchronise the device).  The pages have no counterpart of this entry
 * point; it exists for embedding.  The split tail's scratch is a file-scope
 * device array of the library, 80 key-range chunks of 512 x 130 fp32
 * (21.3 MB), resident on every device from when the library's device code is
 * loaded there (at the latest, its first kernel launch or dit_attn_create)
 * until the process exits.
 * dit_attn_create() takes the array's device address for the current device;
 * the call itself allocates nothing (no cudaMalloc, no library allocator) and
 * takes no workspace argument.
 *   Every call on a device shares the one array and leaves its contents
 *   behind; each call writes every scratch word it later reads, so nothing
 *   needs clearing.  Calls through this entry point that overlap on the GPU
 *   (unordered streams) race on the scratch and give wrong results: keep
 *   them on one stream, or order the streams.
 *   A split plan needs at most one chunk per CTA pair (74 on a 148-SM B300);
 *   a plan beyond the 80 chunks returns UNSUPPORTED.
 *   Before dit_attn_create() on the current device: NOT_INITIALIZED.
 * Arguments, results and other errors as dit_attn_forward_ws.
 */
int dit_attn_forward_noalloc(const void* q, const void* k, const void* v, void* out, int B, int H,
                             int Lq, int Lk, int d, float scale, void* stream);

/*
 * Workspace bytes that dit_attn_forward_ws (variant 0), dit_attn_forward_qk8_ws
 * (variant 1) or dit_attn_forward_fp8_ws (variant 2) uses for these sizes on
 * the current device; 0 when no split applies (d = 64, or the last wave is
 * full or its units too short).  Another variant is INVALID_ARG.  Size
 * arguments as for the forward calls; requires dit_attn_create().
 */
int dit_attn_workspace_size(int B, int H, int Lq, int Lk, int d, int variant, long long* bytes);

/*
 * The same attention with e4m3 queries and keys ("cuDNN FP8 attention" is the
 * FP8 attention that "Speed Up Image Generation with FLUX 3 Image Klein on
 * NVIDIA Blackwell GPUs" (Key takeaways, fourth item) and the sns.style
 * article on TensorRT LLM VisualGen and FLUX 3 Image Klein (third paragraph)
 * compare against dense BF16 attention; the pages print no FP8 recipe):
 *
 *     s_ij = scale * q_scale * k_scale * sum_c e4m3(q8[b,h,i,c]) * e4m3(k8[b,h,j,c])
 *     o[b,h,i,:] = sum_j softmax_j(s_ij) * v[b,h,j,:]
 *
 * q8 : device pointer, e4m3 codes (1 byte; OCP FP8 E4M3, bias 7, no
 *      infinities), contiguous [B, H, Lq, d], dequantised value = code value
 *      * q_scale
 * k8 : the same for keys, [B, H, Lk, d], with k_scale
 * v, out: bf16, as in dit_attn_forward.
 * d must be 128 (else UNSUPPORTED).  q_scale, k_scale finite and >= 0, and
 * the logit scale scale*q_scale*k_scale (either sign) within the bound that
 * dit_attn_forward sets for scale (else INVALID_ARG); the product is folded
 * into the softmax scale once.  Arithmetic: e4m3 tensor-core products
 * with exact fp32 accumulation for S; the softmax, P (bf16), P.V and the
 * output as in dit_attn_forward.  Sizes, alignment, overlap, stream and error
 * behaviour as in dit_attn_forward (q8, k8 sizes counted in bytes).
 * The NaN codes 0x7F and 0xFF are not valid inputs; rows that meet them
 * have unspecified values.
 */
int dit_attn_forward_qk8(const void* q8, const void* k8, const void* v, void* out, int B, int H,
                         int Lq, int Lk, int d, float scale, float q_scale, float k_scale,
                         void* stream);

/* dit_attn_forward_qk8 with a workspace, as dit_attn_forward_ws. */
int dit_attn_forward_qk8_ws(const void* q8, const void* k8, const void* v, void* out, int B,
                            int H, int Lq, int Lk, int d, float scale, float q_scale,
                            float k_scale, void* workspace, long long workspace_bytes,
                            void* stream);

/*
 * The same attention with e4m3 queries, keys and values, P rounded to e4m3
 * before P.V (the FP8 attention the two pages above compare with BF16; the
 * pages print no recipe, so this follows the plainest reading: per-tensor
 * scales for Q, K and V):
 *
 *     s_ij = scale * q_scale * k_scale * sum_c e4m3(q8[b,h,i,c]) * e4m3(k8[b,h,j,c])
 *     p_ij = e4m3( 2^(s_ij * log2(e) - m_i + 3) ),  m_i a running row max (log2 units)
 *     o[b,h,i,:] = v_scale * sum_j p_ij * e4m3(v8[b,h,j,:]) / sum_j p_ij
 *
 * q8, k8 as in dit_attn_forward_qk8; v8: device pointer, e4m3 codes,
 * contiguous [B, H, Lk, d], dequantised value = code value * v_scale.  out:
 * bf16 [B, H, Lq, d].  d must be 128 (else UNSUPPORTED).  q_scale, k_scale
 * finite and >= 0, v_scale finite and > 0 with a finite reciprocal, and the
 * logit scale scale*q_scale*k_scale as in dit_attn_forward_qk8 (else
 * INVALID_ARG).  Arithmetic: both
 * products on e4m3 tensor cores with exact fp32 accumulation; every p is
 * rounded to e4m3 for P.V (relative error at most 2^-4 where p >= 2^-6, i.e.
 * for every key within 2^-9 of the row's largest weight) while the row sum
 * adds the fp32 p, so each weight carries only its own rounding error.
 * Sizes (q8, k8, v8 counted in bytes), alignment, overlap, stream and error
 * behaviour as in dit_attn_forward; NaN codes as in dit_attn_forward_qk8.
 */
int dit_attn_forward_fp8(const void* q8, const void* k8, const void* v8, void* out, int B, int H,
                         int Lq, int Lk, int d, float scale, float q_scale, float k_scale,
                         float v_scale, void* stream);

/* dit_attn_forward_fp8 with a workspace, as dit_attn_forward_ws. */
int dit_attn_forward_fp8_ws(const void* q8, const void* k8, const void* v8, void* out, int B,
                            int H, int Lq, int Lk, int d, float scale, float q_scale,
                            float k_scale, float v_scale, void* workspace,
                            long long workspace_bytes, void* stream);

/*
 * Per-tensor e4m3 quantisation (the prologue that gives dit_attn_forward_fp8
 * its values, or e4m3 queries and keys that are not RMS-normalised):
 *
 *     y8[i] = e4m3( x[i] * out_scale ),  i < n
 *
 * the product in fp32; e4m3() as in dit_attn_rmsnorm_e4m3 (nearest even,
 * saturating at +-448; NaN stays NaN).  out_scale is the reciprocal of the
 * dequantisation scale handed to the forward (for example 448 / max|x|).
 * x: device bf16 [n]; y8: device [n] bytes, not overlapping x; both 16-byte
 * aligned; n >= 1; out_scale finite and > 0 (else INVALID_ARG).  Enqueued on
 * `stream`; requires dit_attn_create().
 */
int dit_attn_quantize_e4m3(const void* x, void* y8, long long n, float out_scale, void* stream);

/*
 * RMS normalisation of queries or keys over the head dimension, per token and
 * head (the normalisation the 1024x1024 and 2048x2048 workloads apply to Q
 * and K before attention; the pages do not print it, so no weight is implied):
 *
 *     y[r, :] = bf16( x[r, :] / sqrt(mean_c x[r, c]^2 + eps) * weight[:] )
 *
 * computed in fp32, rounded to nearest-even bf16.  x and y: device pointers,
 * bf16, contiguous [rows, d] (a [B, H, L, d] tensor is rows = B*H*L); y may
 * equal x (in place) but must not otherwise overlap it.  weight: NULL (all
 * ones) or a device bf16 [d].  d in {64, 128}; rows >= 1; eps finite, >= 0.
 * Pointers 16-byte aligned.  Enqueued on `stream`; requires dit_attn_create().
 */
int dit_attn_rmsnorm(const void* x, void* y, const void* weight, long long rows, int d, float eps,
                     void* stream);

/*
 * The quantising prologue of dit_attn_forward_qk8: RMS normalisation as in
 * dit_attn_rmsnorm, multiplied by out_scale (the reciprocal of the tensor's
 * dequantisation scale) and rounded to e4m3, all in fp32:
 *
 *     y8[r, c] = e4m3( x[r, c] / sqrt(mean_c' x[r, c']^2 + eps) * weight[c] * out_scale )
 *
 * e4m3(): round to nearest, ties to even; magnitudes beyond 448 saturate to
 * +-448.  With eps = 0 and no weight every |value| is at most sqrt(d), so
 * out_scale = 448 / sqrt(d) never saturates.  x: device bf16 [rows, d];
 * y8: device [rows, d] bytes, must not overlap x or weight; weight as in
 * dit_attn_rmsnorm.  out_scale finite and > 0.  Otherwise as dit_attn_rmsnorm.
 */
int dit_attn_rmsnorm_e4m3(const void* x, void* y8, const void* weight, long long rows, int d,
                          float eps, float out_scale, void* stream);

/* Forget the current device's state; forward then returns NOT_INITIALIZED. */
int dit_attn_destroy(void);

/* Static, human-readable name of a status code. */
const char* dit_attn_status_string(int status);

/*
 * Synchronise `stream`, then read and clear the device error word that the
 * kernels set when a bounded wait gives up.  The read and the clear are one
 * atomic exchange on the device (a one-thread kernel on `stream`), so a
 * TIMEOUT recorded meanwhile by a kernel on another stream is kept for the
 * next call, never lost; concurrent callers are serialised.  Returns OK or
 * TIMEOUT (or CUDA if a CUDA call failed).  A test and debugging aid.
 */
int dit_attn_get_device_error(void* stream);

/*
 * Self-test of failure detection: enqueue a one-thread kernel that waits on a
 * barrier nothing ever completes, gives up after limit_us microseconds
 * (1 .. 1000000, else INVALID_ARG) and sets the device error word exactly as
 * an attention kernel does when a bounded wait gives up.  A following
 * dit_attn_get_device_error then returns TIMEOUT, and the context stays
 * usable.  Nothing faults or hangs.  Requires dit_attn_create().
 */
int dit_attn_check_wait_timeout(int limit_us, void* stream);

/*
 * Self-test of the exponential the softmax evaluates on the FMA pipe for part
 * of its probabilities (a Cody-Waite reduction and a minimax polynomial; the
 * pages specify no exponential, so this is an implementation check, not a
 * step of the method):
 *
 *     y_fma[i]  = the FMA-pipe 2^x[i] of the given degree (2: the e4m3-P
 *                 softmax, 3: the bf16-P softmax), x clamped to [-125, 127]
 *     y_mufu[i] = ex2.approx.ftz(x[i]), the MUFU instruction it stands in for
 *
 * x, y_fma, y_mufu: device fp32 [n], 4-byte aligned, not overlapping;
 * 1 <= n <= 2^40; degree 2 or 3 (else INVALID_ARG).  Enqueued on `stream`;
 * requires dit_attn_create().
 */
int dit_attn_check_exp2(const void* x, void* y_fma, void* y_mufu, long long n, int degree,
                        void* stream);

/* The cudaError_t behind the most recent DIT_ATTN_ERR_CUDA on this thread. */
int dit_attn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DIT_ATTN_H */
