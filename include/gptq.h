/*
 * gptq.h — C ABI of libgptq: GPTQ per-layer weight quantization on one GB300 (sm_103a).
 *
 * One layer pass, in the order the GPTQ guide page's "Source code" (`gptq`,
 * `_hessian_inverse_chol`) takes its steps:
 *
 *   gptq_hessian_accumulate   S += X_b^T X_b over token batches          (H = 2 S / n)
 *   gptq_hessian_finalize     H = 2 S / n, diag(X^T X)
 *   gptq_prepare              dead fix, damping, act_order permutation, U = upper chol(H^-1)
 *   gptq_quantize             the fixed-order column loop -> codes, scales, zeros, g_idx,
 *                             dequantised W, packed codes
 *   gptq_prune                the same loop pruning instead of rounding (SparseGPT-style)
 *   rtn_quantize              round-to-nearest on the same grid (the baseline)
 *   gptq_pack                 codes -> LSB-first bitstream of b-bit unsigned codes
 *   gptq_dequant_matmul       Y = X Wq^T read straight from the packed codes, scales,
 *                             zeros and g_idx (the consumer of the stored form)
 *   gptq_set_status_mode,     device-side errors reported by each call (synchronising)
 *   gptq_status_sync          or deferred to one check (calls only enqueue work)
 *
 * Conventions shared by every entry point
 *   - Pointers named as device pointers must be CUDA device (or managed) memory of the
 *     current device; the caller owns every buffer it passes. The library allocates
 *     device memory only inside a gptq_hessian object (its accumulator and tile list).
 *   - Matrices are row-major. W is (rows = out, cols = in); X is (n_tokens, d) with a row
 *     stride of `ld` elements.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is enqueued on it
 *     and runs asynchronously unless an entry point says it synchronises.
 *   - Every entry point returns a gptq_status. Arguments are validated on the host before
 *     any launch; on a validation error nothing is enqueued. GPTQ_ERR_CUDA reports a failed
 *     CUDA call (the CUDA error is cleared with cudaGetLastError()).
 *   - Nothing here falls back to the CPU.
 */
#ifndef GPTQ_H_
#define GPTQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gptq_status {
    GPTQ_OK = 0,
    GPTQ_ERR_INVALID_ARG = 1,   /* null pointer, bad size, stride or alignment */
    GPTQ_ERR_UNSUPPORTED = 2,   /* bits not in {2,3,4}; group neither a divisor nor a multiple of 128 */
    GPTQ_ERR_NOT_SPD = 3,       /* a Cholesky pivot was <= 0 or not finite */
    GPTQ_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    GPTQ_ERR_TIMEOUT = 5,       /* a bounded on-device wait gave up; results are invalid */
    GPTQ_ERR_WORKSPACE = 6,     /* ws_bytes smaller than the matching *_workspace_bytes() */
    GPTQ_ERR_NONFINITE = 7      /* an input held a NaN or an infinity; results are invalid */
} gptq_status;

typedef enum gptq_dtype { GPTQ_F32 = 0, GPTQ_BF16 = 1 } gptq_dtype;

/* Quantizer: bits in {2,3,4}; group = 0 for one scale per output row (from the starting
 * weights), otherwise the group size in columns (a divisor of 128 or a multiple of 128),
 * each group's scale taken at its start from the already-updated weights; sym = 1 for
 * the symmetric grid clip(round(w/s), -qmax, qmax), qmax = 2^(bits-1) - 1, sym = 0 for the
 * min/max + zero-point grid clamp(round(w/s + z), 0, 2^bits - 1) (GPTQ in plain code page,
 * "quantize_weight": s = (max - min) / (2^bits - 1), z = round(-min / s) clamped).
 * zero_in_range = 1 selects the variant of that grid whose range is first widened to
 * contain 0 (min <- min(min, 0), max <- max(max, 0)), so 0 is always a grid point; the
 * pages take the raw min/max (zero_in_range = 0). Ignored by the symmetric grid. */
typedef struct gptq_qconfig {
    int32_t bits;
    int32_t group;
    int32_t sym;
    int32_t zero_in_range;
} gptq_qconfig;

/* ------------------------------------------------------------------------------------
 * Hessian accumulator.  GPTQ guide page, "How it works" and "Source code"
 * (`_hessian_inverse_chol`, first line): H = 2 X^T X / n over the n calibration rows.
 * ------------------------------------------------------------------------------------ */
typedef struct gptq_hessian gptq_hessian;

/* Creates an accumulator for d input channels on the current device (S = 0, n = 0).
 * Allocates S (d*d fp32, upper triangle used) and a small tile list; *out receives the
 * handle. Errors: INVALID_ARG (d < 1, out NULL), CUDA (allocation). */
int gptq_hessian_create(int64_t d, gptq_hessian** out);

/* S = 0, n = 0 (stream-ordered). */
int gptq_hessian_reset(gptq_hessian* h, void* stream);

/* S += X^T X over n_tokens rows of X (device pointer), n += n_tokens. X is (n_tokens, d)
 * row-major with row stride ld >= d elements; dtype GPTQ_BF16 or GPTQ_F32.
 * bf16 runs on the tensor cores (fp32 accumulation) and needs ld*2 % 16 == 0 and a
 * 16-byte-aligned X; fp32 runs on the FP32 pipes (exact fp32 products, fp32 sums).
 * Asynchronous. n_tokens == 0 is a no-op. Errors: INVALID_ARG, CUDA. */
int gptq_hessian_accumulate(gptq_hessian* h, const void* X, int dtype, int64_t n_tokens,
                            int64_t ld, void* stream);

/* H = 2 S / n written to H (device, d*d fp32, both triangles), diag_xtx[j] = S[j][j]
 * (device, d fp32, the raw diag(X^T X) act_order sorts on; may be NULL), *n_tokens = n
 * (host; may be NULL). Synchronises `stream` to report a device-side error (not in the
 * deferred status mode, below). A NaN or infinity anywhere in the accumulated X makes its
 * channel's S[j][j] non-finite, which is reported as NONFINITE (kept until the next reset).
 * Errors: INVALID_ARG (n == 0), TIMEOUT, NONFINITE, CUDA. */
int gptq_hessian_finalize(gptq_hessian* h, float* H, float* diag_xtx, int64_t* n_tokens,
                          void* stream);

/* Releases the accumulator (synchronises the device's pending work on it first). */
int gptq_hessian_destroy(gptq_hessian* h);

/* ------------------------------------------------------------------------------------
 * Preparation.  GPTQ guide page, "Source code" (`_hessian_inverse_chol`, and `gptq`'s
 * act_order branch), "The code, line by line", "How it works" (Damping, trick 2).
 *   dead[j]  = (H[j][j] == 0); H[j][j] = 1 for dead j
 *   H       += damp * mean(diag H) * I          (mean after the dead fix)
 *   perm     = stable descending argsort of diag_xtx if act_order, else identity
 *   U        = upper Cholesky factor of (H[perm][:, perm])^-1, i.e. U^T U = H_perm^-1
 * Inputs: H (device, d*d fp32; only the upper triangle i <= j is read), diag_xtx (device,
 * d fp32; read only when act_order, may then not be NULL).
 * Outputs (device): U (d*d fp32, upper triangular in the loop's column order, zeros below
 * the diagonal), perm (d int32: loop position k quantises original column perm[k]),
 * dead (d uint8, original column order).
 * ws: device workspace of at least gptq_prepare_workspace_bytes(d, act_order) bytes.
 * Synchronises `stream` at the end to report a failed factorisation (not in the deferred
 * status mode, below: the status is then kept for gptq_status_sync). An entry of H's upper
 * triangle that is NaN or infinite is reported as NONFINITE (before any pivot check).
 * For d > 128 the factorisation runs on two library-owned streams forked from and joined
 * back to `stream`: one set per caller stream (up to 8 per device), so calls on different
 * caller streams, with different workspaces, can run side by side on the GPU. The chain
 * stream has the device's greatest priority, the other the caller stream's priority. A
 * caller running many such calls at once should raise CUDA_DEVICE_MAX_CONNECTIONS (up to
 * 32) before its CUDA context is created: with the default 8 hardware queues, unrelated
 * streams share queues and their work serialises.
 * Errors: INVALID_ARG, WORKSPACE, NONFINITE, NOT_SPD, CUDA. */
size_t gptq_prepare_workspace_bytes(int64_t d, int act_order);
int gptq_prepare(const float* H, const float* diag_xtx, int64_t d, float damp, int act_order,
                 float* U, int32_t* perm, uint8_t* dead, void* ws, size_t ws_bytes, void* stream);

/* gptq_prepare without a caller workspace, for callers that cannot allocate device
 * memory (a host framework that owns all device memory through its own pool, or a path
 * that cannot take cudaMalloc's implicit synchronisation). No counterpart on the pages.
 * Same arguments, outputs, synchronisation and errors as gptq_prepare, minus ws/ws_bytes.
 * The scratch is a fixed array compiled into the library (about 14 MiB, held on every
 * GPU that loads the library until the process exits), so d is limited to 1024:
 * d > 1024 returns GPTQ_ERR_UNSUPPORTED. Allocates nothing (no cudaMalloc/cudaFree).
 * The first call in each CUDA context (one per device for the runtime's primary contexts;
 * again after a device reset) looks up that context's copy of the array
 * (cudaGetSymbolAddress); make that first call before any stream capture. All calls share
 * the one array, so calls that overlap on the GPU (other streams, other threads) race;
 * serialise them. Errors: INVALID_ARG, UNSUPPORTED, NONFINITE, NOT_SPD, CUDA. */
int gptq_prepare_noalloc(const float* H, const float* diag_xtx, int64_t d, float damp,
                         int act_order, float* U, int32_t* perm, uint8_t* dead, void* stream);

/* ------------------------------------------------------------------------------------
 * Quantisation.  GPTQ's error-compensation loop page (the four steps); GPTQ guide page,
 * "Source code" (`gptq`), "When it breaks" (clipping; g_idx); AutoGPTQ page
 * (`quantize_weight`, `dequantize_weight`, group-start min/max and zero point).
 * W (device, rows*cols fp32) is read only; columns with dead[c] != 0 are zeroed; the loop
 * runs over loop positions k = 0..cols-1 on column perm[k] (perm NULL = identity) with
 * U in loop order:  q = quantise(w_k);  err = (w_k - q) / U[k][k];
 * W[:, k+1:] -= err * U[k][k+1:].
 * Outputs (device; original column order unless stated):
 *   codes   rows*cols int8: sym code in [-qmax, qmax]; asym code in [0, 2^bits - 1]
 *   scales  rows*G fp32, G = ceil(cols/group) (1 if group == 0); group gi covers loop
 *           positions [gi*group, (gi+1)*group)
 *   zeros   rows*G uint8: asym zero point; sym 2^(bits-1) (the unsigned offset)
 *   g_idx   cols int32 (may be NULL): group of each original column
 *   Wq      rows*cols fp32 (may be NULL): scale * (code) or scale * (code - zero)
 *   packed  rows*gptq_packed_words_per_row(cols,bits) uint32 (may be NULL): per row the
 *           LSB-first bitstream of unsigned codes u (sym u = code + 2^(bits-1))
 *   row_loss rows fp32 (may be NULL): sum_k err_k^2 per row
 * ws: device workspace of at least gptq_quantize_workspace_bytes(rows, cols, q) bytes.
 * Synchronises `stream` at the end to report a device-side error (not in the deferred
 * status mode, below). A NaN or infinity in W (outside dead columns, which are not read) or
 * on U's diagonal is reported as NONFINITE.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, TIMEOUT, NONFINITE, CUDA. */
size_t gptq_quantize_workspace_bytes(int64_t rows, int64_t cols, gptq_qconfig q);
int gptq_quantize(const float* W, int64_t rows, int64_t cols, const float* U,
                  const int32_t* perm, const uint8_t* dead, gptq_qconfig q,
                  int8_t* codes, float* scales, uint8_t* zeros, int32_t* g_idx, float* Wq,
                  uint32_t* packed, float* row_loss, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Pruning with GPTQ's update.  GPTQ guide page, "Going further" (SparseGPT reuses the same
 * error-compensation update for pruning); the loop is the one above with the rounding
 * replaced by pruning. The pages give the update, not the mask rule; the rule here:
 * at the start of each 128-column block of loop positions, each row prunes the
 * round(sparsity * width) weights (ties to even, computed in double from the float
 * sparsity) of smallest saliency (w_k / U[k][k])^2 of its updated weights (the loss the
 * guide page's "How it works" assigns to removing w_k alone, e^2 / (2 H_F^-1[k][k]) with
 * H_F^-1[k][k] = U[k][k]^2, factor 1/2 dropped), ties broken by the lower loop position;
 * then for every k: q = 0 where pruned, q = w_k elsewhere, err = (w_k - q) / U[k][k],
 * W[:, k+1:] -= err * U[k][k+1:].
 * Inputs as gptq_quantize (W read only; dead columns zeroed; perm NULL = identity);
 * sparsity in [0, 1].
 * Outputs (device, original column order): Wp rows*cols fp32, the pruned and compensated
 * weights (exactly 0 where pruned); mask rows*cols uint8 (may be NULL), 1 where pruned;
 * row_loss rows fp32 (may be NULL), sum_k err_k^2 per row.
 * ws: device workspace of at least gptq_prune_workspace_bytes(rows, cols) bytes.
 * Synchronises `stream` at the end to report a device-side error (not in the deferred
 * status mode, below).
 * Errors: INVALID_ARG (sizes, NULL, sparsity outside [0, 1]), WORKSPACE, TIMEOUT, NONFINITE,
 * CUDA. */
size_t gptq_prune_workspace_bytes(int64_t rows, int64_t cols);
int gptq_prune(const float* W, int64_t rows, int64_t cols, const float* U, const int32_t* perm,
               const uint8_t* dead, float sparsity, float* Wp, uint8_t* mask, float* row_loss,
               void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Round-to-nearest baseline (GPTQ's error-compensation loop page, first paragraph; guide
 * page, "The idea"): the same grid with scales from W itself, no error feedback.
 * Same output conventions as gptq_quantize (contiguous groups, no permutation); dead may
 * be NULL. Synchronises `stream` at the end to report a NaN or infinity in W (outside dead
 * columns) as NONFINITE (not in the deferred status mode, below). Allocates nothing (the
 * call's status word is one of a ring of words in static device memory).
 * Errors: INVALID_ARG, UNSUPPORTED, NONFINITE, CUDA. */
int rtn_quantize(const float* W, int64_t rows, int64_t cols, const uint8_t* dead,
                 gptq_qconfig q, int8_t* codes, float* scales, uint8_t* zeros, float* Wq,
                 uint32_t* packed, void* stream);

/* ------------------------------------------------------------------------------------
 * Packing (no counterpart on the pages beyond INT4 memory = fp16 / 4): codes (device,
 * rows*cols int8, as gptq_quantize returns them) -> packed (device,
 * rows*gptq_packed_words_per_row(cols,bits) uint32); code c of a row occupies stream
 * bits [c*bits, (c+1)*bits); stream bit p is bit p%32 of word p/32; rows are padded with
 * zero bits. Asynchronous. Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
int64_t gptq_packed_words_per_row(int64_t cols, int bits);
int gptq_pack(const int8_t* codes, int64_t rows, int64_t cols, int bits, int sym,
              uint32_t* packed, void* stream);

/* ------------------------------------------------------------------------------------
 * Consumer of the stored form.  GPTQ guide page, "When it breaks" (with act_order the
 * groups are scattered over the columns, so a kernel that uses the quantised weights needs
 * the stored column-to-group index g_idx); AutoGPTQ page, `dequantize_weight`
 * (scale * (code - zero)).
 *
 * Y[t][o] = sum_k X[t][k] * Wq[o][k],  Wq[o][k] = scales[o][g] * (u[o][k] - zeros[o][g]),
 * g = g_idx[k], u[o][k] = the k-th bits-wide field of row o of `packed` (the layout of
 * gptq_pack; symmetric codes are stored with zero point 2^(bits-1), so the same formula
 * gives scale * code).
 *   X       device, bf16, (T, K) row-major, row stride ldx elements (ldx % 8 == 0, X 16-byte
 *           aligned), K % 64 == 0
 *   packed  device, uint32, (N, gptq_packed_words_per_row(K, bits))
 *   scales  device, fp32, (N, G); zeros device, uint8, (N, G); g_idx device, int32, (K),
 *           16-byte aligned, values in [0, G) (others record INVALID_ARG and read group 0)
 *   flags   GPTQ_DQ_RELU: Y = max(., 0) (the hidden layers of an MLP forward);
 *           GPTQ_DQ_BF16_OUT: Y is bf16 (rounded to nearest even), else fp32
 *   Y       device, (T, N) row-major, row stride ldy elements
 * The weights are expanded to bf16 on chip (rounding each to 8 significant bits) and
 * multiplied on the tensor cores with fp32 accumulation. Allocates nothing (the call's
 * status word is one of a ring of words in static device memory). Synchronises the stream
 * and returns the device status (in the deferred status mode, below, neither).
 * Errors: INVALID_ARG, UNSUPPORTED (bits not 2-4, K % 64, alignment, K or G too large for
 * the shared-memory plan), TIMEOUT, CUDA. */
enum { GPTQ_DQ_RELU = 1, GPTQ_DQ_BF16_OUT = 2 };
int gptq_dequant_matmul(const void* X, int64_t T, int64_t K, int64_t ldx, const uint32_t* packed,
                        const float* scales, const uint8_t* zeros, const int32_t* g_idx, int64_t N,
                        int64_t G, int bits, int flags, void* Y, int64_t ldy, void* stream);

/* Static text for a status code. */
const char* gptq_status_string(int status);

/* ------------------------------------------------------------------------------------
 * Status reporting (no counterpart on the pages). Errors found on the host (arguments,
 * workspace, CUDA calls) are always returned at once. Errors found on the device (a
 * timed-out wait, a non-positive-definite block) are reported, in the default mode
 * GPTQ_STATUS_SYNC, by the call itself, which synchronises its stream before returning.
 * In mode GPTQ_STATUS_DEFERRED the calls that say "Synchronises" do not: they return
 * GPTQ_OK once their work is enqueued, and a final one-thread kernel of each call folds
 * its device status into one sticky status word per device (the first error is kept).
 * gptq_status_sync then reports it. The mode is process-wide. In deferred mode the
 * calls only enqueue work, so a sequence of them can be captured into a CUDA graph and
 * replayed (make one call of each kind before capturing: the first gptq_prepare on a
 * caller stream creates the streams and events its two-stream schedule uses).
 * ------------------------------------------------------------------------------------ */
enum { GPTQ_STATUS_SYNC = 0, GPTQ_STATUS_DEFERRED = 1 };
/* Errors: INVALID_ARG (unknown mode). Host only. */
int gptq_set_status_mode(int mode);
int gptq_status_mode(void);
/* Synchronises `stream`, returns the current device's sticky status (GPTQ_OK if no call
 * enqueued in deferred mode on this device since the last gptq_status_sync failed) and
 * clears it. Calls made on other streams must be ordered before `stream` by the caller.
 * Errors: CUDA. */
int gptq_status_sync(void* stream);

/* ------------------------------------------------------------------------------------
 * Instrumentation (no counterpart on the pages). Every kernel the library launches is
 * counted; while profiling is enabled each launch is also bracketed by two CUDA events on
 * its stream. Kernel classes are numbered 0 .. gptq_profile_kernel_count()-1.
 * ------------------------------------------------------------------------------------ */
/* Kernel launches since the library was loaded (all devices, all threads). */
unsigned long long gptq_launch_count(void);
/* on != 0 starts recording per-launch events; 0 stops (already recorded ones are kept). */
void gptq_profile_enable(int on);
/* Waits for every recorded event, writes per-class totals (ms[i] milliseconds, launches[i]
 * launches; either may be NULL; n entries at most) and clears the record. Host arrays.
 * Errors: INVALID_ARG (n < 0), CUDA. */
int gptq_profile_read(double* ms, unsigned long long* launches, int n);
int gptq_profile_kernel_count(void);
/* Static name of kernel class `id`. */
const char* gptq_profile_kernel_name(int id);

#ifdef __cplusplus
}
#endif
#endif /* GPTQ_H_ */
