/*
 * sq.h -- C ABI of the SmoothQuant W8A8 INT8 linear block for NVIDIA GB300
 * (sm_103a).
 *
 * The operation is the linear block of BERT-family encoder inference analysed
 * in "Efficient INT8 Inference of Small NLP Models on Server CPUs with PyTorch
 * Native Stack" (Xia, Cui, Cao): SmoothQuant smoothing, dynamic per-token
 * activation quantisation (Table 10, "Smooth-Dynamic"), an int8 x int8 -> int32
 * GEMM, and the GEMM's fused post-operations -- bias, activation, residual
 * addition (Table 3 caption).  The smoothing factor follows SmoothQuant (cited
 * in the pages' reference list), with the migration strength alpha that
 * Table 15 sets per model; GELU is the erf form ("Gaussian Error Linear Units",
 * same reference list).
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers (cudaMalloc'd or equivalent), owned
 *    by the caller, row-major and densely packed, and must be 16-byte aligned
 *    unless stated otherwise.  No entry point allocates device memory
 *    (sq_linear_i8_static_ws uses a static array of the library's module).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously; no entry point synchronises except
 *    sq_device_status().  Kernels are launched with programmatic dependent
 *    launch: their set-up may overlap the end of the previous kernel on the
 *    stream, but every memory access waits for that kernel to complete, so the
 *    stream's ordering holds for all data, as with an ordinary launch.  The
 *    calls may be captured into CUDA graphs once each has run once eagerly on
 *    the device (their one-time set-up is not capturable).
 *  - Arguments are checked on the host before anything is enqueued; a non-OK
 *    status means nothing was launched.  A failed launch returns SQ_ERR_CUDA.
 *    No entry point aborts, traps or throws.
 *  - Sizes are int64_t.  A zero row count (M or N = 0) is a valid empty call:
 *    once the sizes and mode are valid it returns SQ_OK without looking at
 *    the pointers (which may be NULL) and without launching.  K must be a
 *    positive multiple of 16.
 *  - Inputs must be finite; results for NaN or Inf inputs are unspecified.
 *  - Per-device state (function attributes, cluster occupancy, the static
 *    scratch's address) is set up on a device's first call and kept: a
 *    cudaDeviceReset while the library is loaded is not supported.
 */
#ifndef SQ_GB300_H
#define SQ_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SQ_OK = 0,
    SQ_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad mode/alpha      */
    SQ_ERR_ALIGNMENT = 2,   /* K not a multiple of 16 or pointer not 16-B aligned */
    SQ_ERR_UNSUPPORTED = 3, /* size beyond a documented limit, or no sm_103 GPU */
    SQ_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed      */
    SQ_ERR_TIMEOUT = 5      /* a kernel's bounded wait ran out (device status)  */
} sq_status;

/* Epilogue of sq_linear_i8 (the linear block's fused post-operations,
 * Table 3 caption).  With d = acc[m][n] * x_scale[m] * w_scale[n]:
 *   SQ_EPI_NONE          Y = d
 *   SQ_EPI_BIAS          Y = d + bias[n]
 *   SQ_EPI_BIAS_GELU     Y = GELU(d + bias[n]),  GELU(t) = 0.5 t (1 + erf(t/sqrt 2))
 *   SQ_EPI_BIAS_RESIDUAL Y = d + bias[n] + residual[m][n]
 *   SQ_EPI_RAW_I32       Y = acc (int32; the scales, bias and residual are unused)
 * Y is fp32 [M][N] for the first four modes and int32 [M][N] for the last. */
typedef enum {
    SQ_EPI_NONE = 0,
    SQ_EPI_BIAS = 1,
    SQ_EPI_BIAS_GELU = 2,
    SQ_EPI_BIAS_RESIDUAL = 3,
    SQ_EPI_RAW_I32 = 4
} sq_epilogue;

/* Human-readable name of a status code (static string, never NULL). */
const char *sq_status_string(int status);

/* ABI version of this library: (major << 16) | minor. */
int sq_version(void);

/* Bytes of a GEMM-operand buffer for a rows x K matrix of int8 codes.
 * The operand format is the tensor-core operand of sq_linear_i8: each int8
 * code stored as the bf16 number of the same integer value (exact: every
 * integer in [-127, 127] is a bf16), row-major [rows][K], K contiguous.
 * Returns 0 for negative sizes. */
size_t sq_operand_bytes(int64_t rows, int64_t K);

/* Bytes of the packed weight operand of an N x K weight (the Wop buffer of
 * sq_pack_weight): sq_operand_bytes(N, K). */
size_t sq_packed_weight_bytes(int64_t N, int64_t K);

/* ---- Smoothing factor (SmoothQuant; alpha per model in Table 15) ---------- */

/* Running channel maxima for the smoothing factor:
 *   amax[j] = max(amax[j], max_i |A[i][j]|),   A fp32 [rows][cols].
 * The caller initialises amax (zeros for a fresh statistic); calling it once
 * per calibration batch accumulates the maximum over all batches.  Use it on
 * activations X [tokens][K] for max|X_j| and on weights W [N][K] for max|W_j|.
 * amax need only be 4-byte aligned.  cols > 0 required; rows = 0 is a no-op. */
sq_status sq_channel_absmax(const float *A, int64_t rows, int64_t cols, float *amax,
                            void *stream);

/* Smoothing factor per input channel:
 *   s[j] = x_amax[j]^alpha / w_amax[j]^(1 - alpha),
 * computed in double and rounded once to fp32; s[j] = 1 where either maximum
 * is 0.  0 <= alpha <= 1.  Pointers need only be 4-byte aligned. */
sq_status sq_smooth_factor(const float *x_amax, const float *w_amax, int64_t K, float alpha,
                           float *s, void *stream);

/* ---- Weight packing (once per layer, offline) ----------------------------- */

/* Folds the smoothing factor into the weights and quantises each output
 * channel symmetrically (per-channel int8 weights):
 *   W'[n][j]   = W[n][j] * s[j]                                  (fp32)
 *   w_scale[n] = max_j |W'[n][j]| / 127   (IEEE fp32 division; 1 if the row is 0)
 *   Wq[n][j]   = clamp(round_half_even(W'[n][j] / w_scale[n]), -127, 127)
 * W fp32 [N][K] (nn.Linear layout), s fp32 [K].  Outputs: w_scale fp32 [N]
 * (required, 4-byte aligned), Wq int8 [N][K] (may be NULL), Wop GEMM operand
 * of sq_operand_bytes(N, K) bytes (may be NULL); at least one of Wq / Wop;
 * w_row_l1 int32 [N] (may be NULL): sum_j |Wq[n][j]| per row, which lets
 * sq_linear_i8 prove single-pass exactness (see there). */
sq_status sq_pack_weight(const float *W, const float *s, int64_t N, int64_t K, int8_t *Wq,
                         float *w_scale, void *Wop, int32_t *w_row_l1, void *stream);

/* ---- Activation smoothing + dynamic per-token quantisation (Table 10) ----- */

/* Per token (row) m of X fp32 [M][K]:
 *   v[j]       = X[m][j] / s[j]                                  (IEEE fp32 division)
 *   x_scale[m] = max_j |v[j]| / 127       (IEEE fp32 division; 1 if the row is 0)
 *   Xq[m][j]   = clamp(round_half_even(v[j] / x_scale[m]), -127, 127)
 * Outputs: x_scale fp32 [M] (required, 4-byte aligned), Xq int8 [M][K] (may be
 * NULL), Xop GEMM operand of sq_operand_bytes(M, K) bytes (may be NULL); at
 * least one of Xq / Xop; x_row_l1 int32 [M] (may be NULL): sum_j |Xq[m][j]|
 * per token, for sq_linear_i8.  Any K that is a positive multiple of 16 works;
 * rows of up to 8192 elements are held in registers (one HBM read), longer
 * rows are read twice. */
sq_status sq_quantize_act(const float *X, const float *s, int64_t M, int64_t K, int8_t *Xq,
                          float *x_scale, void *Xop, int32_t *x_row_l1, void *stream);

/* ---- Smooth-Static: per-tensor activation scale fixed offline (Table 10) --- */

/* Calibration statistic for Smooth-Static:
 *   *amax = max(*amax, max_{m,j} |X[m][j] / s[j]|)     (IEEE fp32 division)
 * X fp32 [M][K], s fp32 [K]; amax one float (4-byte aligned), initialised by
 * the caller (0 for a fresh statistic) and accumulated over calibration
 * batches.  The static scale then comes from sq_static_scale. */
sq_status sq_act_absmax(const float *X, const float *s, int64_t M, int64_t K, float *amax,
                        void *stream);

/* Smooth-Static per-tensor scale from the calibration statistic:
 *   *scale = fl32(*amax / 127)   (IEEE fp32 division; 1 if *amax is 0),
 * the same rule as the dynamic per-token scale applied to the whole
 * calibration set.  amax and scale: one float each in device memory, 4-byte
 * aligned (they may be the same float).  The result is the `scale` argument
 * of sq_quantize_act_static / sq_linear_i8_requant (read it back once,
 * offline). */
sq_status sq_static_scale(const float *amax, float *scale, void *stream);

/* Smooth-Static quantisation with one per-tensor scale `scale` (> 0, finite):
 *   Xq[m][j] = clamp(round_half_even(fl(fl(X[m][j] / s[j]) / scale)), -127, 127)
 * (values beyond the calibrated range saturate).  Outputs as sq_quantize_act;
 * x_scale[m] is set to `scale` for every token, so sq_linear_i8 applies the
 * per-tensor dequantisation unchanged. */
sq_status sq_quantize_act_static(const float *X, const float *s, int64_t M, int64_t K,
                                 float scale, int8_t *Xq, float *x_scale, void *Xop,
                                 int32_t *x_row_l1, void *stream);

/* ---- LayerNorm with the next linear's quantiser fused in ------------------ */

/* The encoder's LayerNorm (Table 3 lists it among BERT-large's operators),
 * emitting the next linear's smoothed int8 codes directly, as SmoothQuant's
 * folding of the smoothing factor into the normalisation implies:
 *   y[m][j] = fma((H[m][j] - mean_m) * rstd_m, gamma[j], beta[j]),
 *   mean_m = fl(sum_j H[m][j] / K), var_m = fl(sum_j (H[m][j] - mean_m)^2 / K)
 *   (fp32 sums in a tree), rstd_m = RN(1 / sqrt(fl(var_m + eps))),
 * then the codes of y exactly as sq_quantize_act (static_scale == 0: dynamic
 * per-token scale) or sq_quantize_act_static (static_scale > 0, finite) would
 * write them for X = y.  H fp32 [M][K]; gamma, beta fp32 [K] (16-byte
 * aligned); eps >= 0; Y fp32 [M][K] (nullable): y itself; other outputs as
 * sq_quantize_act.  K <= 8192 (SQ_ERR_UNSUPPORTED otherwise). */
sq_status sq_layernorm_quant(const float *H, const float *gamma, const float *beta, float eps,
                             const float *s, int64_t M, int64_t K, float static_scale, float *Y,
                             int8_t *Xq, float *x_scale, void *Xop, int32_t *x_row_l1,
                             void *stream);

/* ---- INT8 GEMM + fused dequantising epilogue ------------------------------ */

/* acc[m][n] = sum_k Xq[m][k] * Wq[n][k], exact in int32, then the epilogue
 * `mode` (sq_epilogue) writes Y.  Operands are GEMM-operand buffers written by
 * sq_quantize_act (Xop, [M][K]) and sq_pack_weight (Wop, [N][K]).  Runs on the
 * tcgen05 tensor cores: the integer codes are multiplied exactly as bf16 and
 * summed exactly in fp32 over chunks of at most 1024 of K (every partial sum
 * stays below 2^24), the chunks being added in int32.  x_row_l1 [M] and
 * w_row_l1 [N] (int32, each may be NULL) are the row sums of |code| written by
 * sq_quantize_act / sq_pack_weight: if 127 * max(row L1) < 2^24 for either
 * operand, no partial sum can reach 2^24 and all of K is summed in one pass
 * (faster for K > 1024, same exact result).  x_scale fp32 [M], w_scale fp32
 * [N], bias fp32 [N] (modes 1-3), residual fp32 [M][N] (mode 3); Y fp32 or
 * int32 [M][N].  Y must not overlap any input; residual may equal Y only if it
 * is exactly the same buffer.  Requires K <= 133144 (so that |acc| < 2^31 for
 * any codes) and a GB300-class (sm_103) device. */
sq_status sq_linear_i8(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                       const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                       const float *bias, const float *residual, int64_t M, int64_t N, int64_t K,
                       int mode, void *Y, void *stream);

/* sq_linear_i8 on the int8 activation codes Xq [M][K] (as sq_quantize_act
 * writes them) instead of the GEMM-operand buffer: the per-token x per-channel
 * INT8 recipe's own input format.  sm_103a's tensor cores take no int8
 * operands, so the codes are first widened, exactly, into the bf16 operand in
 * `workspace` (one streaming pass: M*K bytes read, 2*M*K written), and the
 * tcgen05 GEMM then runs as sq_linear_i8 on it: results bit for bit those of
 * sq_linear_i8 on sq_quantize_act's Xop.  (The pair kernel cannot widen inside
 * its operand path without a per-stage handshake between its two CTAs; the
 * quantiser writes the bf16 operand in the time it writes the codes, so
 * sq_quantize_act + sq_linear_i8 stays the faster pair.)
 * sq_linear_codes_workspace_bytes: *bytes = the workspace an M x K call needs
 * (2*M*K rounded up to 256).  Xq and workspace 16-byte aligned, the workspace
 * overlapping no other argument; workspace_bytes below the requirement:
 * SQ_ERR_INVALID_ARG.  Other arguments, limits and statuses as sq_linear_i8. */
sq_status sq_linear_codes_workspace_bytes(int64_t M, int64_t K, size_t *bytes);
sq_status sq_linear_i8_codes(const int8_t *Xq, const float *x_scale, const int32_t *x_row_l1,
                             const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                             const float *bias, const float *residual, int64_t M, int64_t N,
                             int64_t K, int mode, void *Y, void *workspace, size_t workspace_bytes,
                             void *stream);

/* ---- Producer-fused Smooth-Static quantisation ------------------------------ */

/* sq_linear_i8 whose epilogue hands its results straight to the NEXT linear
 * layer's Smooth-Static quantiser (Table 10), the GPU counterpart of the
 * pages' INT8 subgraph fusion: no fp32 output is written.  For every element
 * the epilogue forms y[m][n], bit for bit the value sq_linear_i8 stores for
 * the same inputs and mode (modes 0-3; not SQ_EPI_RAW_I32), then
 *   code[m][n] = clamp(round_half_even(fl(fl(y[m][n] / s_next[n]) / scale)), -127, 127)
 * (IEEE fp32 divisions), i.e. sq_quantize_act_static applied to Y with the
 * next layer's smoothing factor s_next fp32 [N] and per-tensor scale
 * (> 0, finite).  Outputs: Yop [M][N] codes as exact bf16 values (the next
 * sq_linear_i8's activation operand; 2-byte aligned) and/or Yq int8 [M][N] --
 * at least one; x_scale_next fp32 [M] (nullable) is set to `scale` for every
 * token.  Rows of N a multiple of 16 and 16-byte aligned code arrays take
 * vector stores.  Other arguments, limits and statuses as sq_linear_i8. */
sq_status sq_linear_i8_requant(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                               const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                               const float *bias, const float *residual, int64_t M, int64_t N,
                               int64_t K, int mode, const float *s_next, float scale, int8_t *Yq,
                               void *Yop, float *x_scale_next, void *stream);

/* ---- Producer-fused Smooth-Dynamic quantisation ----------------------------- */

/* Division table of a smoothing factor, for sq_linear_i8_rowmax (offline, once
 * per layer, like the packed weights):
 *   table[2j] = -s[j],  table[2j+1] = RN(1/s[j])  (NaN when |s[j]| is outside
 *   [2^-20, 2^20]; such columns then take IEEE divisions).
 * s fp32 [K] (4-byte aligned); table fp32 [K][2] (16-byte aligned). */
sq_status sq_division_table(const float *s, int64_t K, float *table, void *stream);

/* sq_linear_i8 whose epilogue also produces the NEXT linear's Smooth-Dynamic
 * statistic (Table 10; the pages' INT8 subgraph fusion, with the per-token
 * maximum across the output's column tiles):
 *   Y as sq_linear_i8 writes it (bit for bit), and
 *   row_amax[m] = max(row_amax[m], max_n |fl(Y[m][n] / s_next[n])|)
 * (IEEE fp32 quotients), merged across tiles with integer atomics on the bit
 * patterns.  next_table: sq_division_table of s_next [N].  row_amax fp32 [M]
 * (4-byte aligned), zero-filled by the caller before the call (or holding a
 * running maximum).  sq_quantize_act_rowmax(Y, s_next, row_amax, ...) then
 * writes the next linear's codes without its own row reduction.  Modes 0-3
 * (not SQ_EPI_RAW_I32); other arguments, limits and statuses as sq_linear_i8. */
sq_status sq_linear_i8_rowmax(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                              const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                              const float *bias, const float *residual, int64_t M, int64_t N,
                              int64_t K, int mode, void *Y, const float *next_table,
                              float *row_amax, void *stream);

/* sq_quantize_act with the per-token maxima given: row_amax[m] must be
 *   max_j |fl(X[m][j] / s[j])|
 * (as sq_linear_i8_rowmax leaves it); then x_scale, Xq, Xop and x_row_l1 are
 * bit for bit those of sq_quantize_act(X, s, ...), and no row reduction runs.
 * A maximum below the true one only saturates codes at +-127 (results are then
 * unspecified, but stay in range).  row_amax fp32 [M] (4-byte aligned); other
 * arguments as sq_quantize_act. */
sq_status sq_quantize_act_rowmax(const float *X, const float *s, const float *row_amax,
                                 int64_t M, int64_t K, int8_t *Xq, float *x_scale, void *Xop,
                                 int32_t *x_row_l1, void *stream);

/* Table 10's Smooth-Dynamic run-time step again: sq_quantize_act (row_amax
 * NULL) or sq_quantize_act_rowmax (row_amax given) with s's division table
 * beside s: s_table = sq_division_table(s), computed
 * offline with the packed weights.  Outputs bit for bit those of the call
 * without the table; where the rows are held in registers the kernel reads -s
 * and RN(1/s) from the table instead of forming the reciprocals in every
 * block.  A table that is not sq_division_table(s) gives unspecified codes
 * (in range).  s_table fp32 [K][2] (16-byte aligned); other arguments as
 * sq_quantize_act / sq_quantize_act_rowmax. */
sq_status sq_quantize_act_table(const float *X, const float *s, const float *s_table,
                                const float *row_amax, int64_t M, int64_t K, int8_t *Xq,
                                float *x_scale, void *Xop, int32_t *x_row_l1, void *stream);

/* ---- Encoder self-attention (Table 3, beside the linear block) -------------- */

/* Scaled dot-product attention per sequence b and head h on the fused QKV
 * projection's output:
 *   O[b*S + i][h*D + d] = sum_j P[i][j] V[b*S + j][h*D + d],
 *   P[i][j] = exp(scale q_i.k_j - m_i) / sum_j' exp(scale q_i.k_j' - m_i),
 * m_i the row maximum, every token attending to every token of its sequence
 * (no mask).  QKV fp32 [B*S][3*H*D]: the Q, K and V blocks of H*D columns
 * each, head h at columns h*D of a block (sq_linear_i8's output with
 * N = 3*H*D); O fp32 [B*S][H*D]; both 16-byte aligned, not overlapping.
 * scale finite (1/sqrt(D) for BERT).  D = 64; S a multiple of 64, at most 448;
 * B*S below 2^31 and H at most 65536 (SQ_ERR_UNSUPPORTED otherwise).  The contractions run on the tensor cores in
 * split tf32 (each operand as an exact pair of tf32 numbers, products within
 * about 2^-21 relative), the softmax in fp32: O agrees with the exact
 * definition to about 1e-6 of max |O|. */
sq_status sq_attention(const float *QKV, int64_t B, int64_t S, int64_t H, int64_t D,
                       float scale, float *O, void *stream);

/* ---- Split K over several SMs (caller workspace) ---------------------------- */

/* An output of fewer 128 x 256 tiles than the GPU has SMs keeps most SMs idle
 * while each busy SM runs the whole K.  With a workspace, sq_linear_i8_ws /
 * sq_linear_i8_requant_ws cut each tile's K range into min(4, SMs / tiles)
 * equal pieces when K >= 2048, one per SM: each SM sums its piece exactly
 * (int32), all but the last SM to finish a tile write their partial sums to
 * the workspace, and that last SM adds them and runs the epilogue.  Integer
 * addition is exact and order-free, so the outputs are bit for bit those of
 * sq_linear_i8 / sq_linear_i8_requant.  Other shapes run the whole-tile
 * schedule (their workspace size is 0): measured on GB300, the partial sums'
 * round trip costs more than a split saves there.
 *
 * sq_linear_workspace_bytes: *bytes = the workspace an M x N x K launch needs
 * on the current device (0 when it is not split; at most SMs x (256 KB + 64
 * bytes), 38 MiB on 152 SMs).  A workspace sized for the largest of several
 * shapes serves them all.
 * Workspace rules: device memory, 16-byte aligned, zero-filled once before its
 * first use (cudaMemset); every launch that completes leaves its counters at
 * zero again, so it is reused as it is (the partial slots need no clearing).
 * A workspace serves one launch at a time: launches that share it
 * must be ordered (one stream, or events), or they race on its counters.  After
 * sq_device_status has reported SQ_ERR_TIMEOUT, zero-fill it again.  NULL
 * workspace: the whole-tile schedule of sq_linear_i8.  workspace_bytes below
 * the requirement: SQ_ERR_INVALID_ARG.  Other arguments, limits and statuses
 * as sq_linear_i8 / sq_linear_i8_requant. */
sq_status sq_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t *bytes);
sq_status sq_linear_i8_ws(const void *Xop, const float *x_scale, const int32_t *x_row_l1,
                          const void *Wop, const float *w_scale, const int32_t *w_row_l1,
                          const float *bias, const float *residual, int64_t M, int64_t N,
                          int64_t K, int mode, void *Y, void *workspace, size_t workspace_bytes,
                          void *stream);
sq_status sq_linear_i8_requant_ws(const void *Xop, const float *x_scale,
                                  const int32_t *x_row_l1, const void *Wop, const float *w_scale,
                                  const int32_t *w_row_l1, const float *bias,
                                  const float *residual, int64_t M, int64_t N, int64_t K,
                                  int mode, const float *s_next, float scale, int8_t *Yq,
                                  void *Yop, float *x_scale_next, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* sq_linear_i8_ws on scratch the library holds itself, for callers that
 * allocate no device memory: a file-scope static device array of
 * SQ_STATIC_WORKSPACE_BYTES (40 MiB; a GPU of up to 159 SMs), zero-filled at
 * module load.  Its address is looked up once per device (cudaGetSymbolAddress)
 * on that device's first call; make that first call outside any stream capture,
 * after which a call only launches.  The address is kept for the life of the
 * process: a cudaDeviceReset while the library is loaded is not supported by
 * this entry point.  Nothing is allocated: a shape whose split needs more than
 * the array (sq_linear_workspace_bytes) returns SQ_ERR_UNSUPPORTED.  The
 * scratch is one per device and process: calls whose launches may overlap
 * (different streams without ordering, several host threads) race on it and
 * must be serialised by the caller.  Arguments are checked first, exactly as
 * in sq_linear_i8_ws (same statuses); outputs as sq_linear_i8_ws.  A launch
 * whose bounded wait ran out (SQ_ERR_TIMEOUT) may leave split-K counters in the
 * scratch: sq_device_status clears them when it reports the timeout, and
 * sq_static_workspace_reset clears them on demand; a static call made before
 * either may compute wrong outputs. */
#define SQ_STATIC_WORKSPACE_BYTES (40u * 1024u * 1024u)
sq_status sq_linear_i8_static_ws(const void *Xop, const float *x_scale,
                                 const int32_t *x_row_l1, const void *Wop, const float *w_scale,
                                 const int32_t *w_row_l1, const float *bias,
                                 const float *residual, int64_t M, int64_t N, int64_t K,
                                 int mode, void *Y, void *stream);

/* Zero-fills the split-K counters of the static scratch on the current device
 * (cudaMemsetAsync on `stream`, then a synchronisation; nothing allocated).
 * SQ_OK without doing anything if the scratch has not been used there. */
sq_status sq_static_workspace_reset(void *stream);

/* The static scratch of the current device: *ptr = its device address (looked
 * up as by sq_linear_i8_static_ws), *bytes = SQ_STATIC_WORKSPACE_BYTES.  For
 * inspection and tests; the library's next static call assumes the counter
 * block at its start is zero. */
sq_status sq_static_workspace(void **ptr, size_t *bytes);

/* The same GEMM + epilogue on the legacy warp-level integer MMA path
 * (mma.sync m16n8k32 s8 x s8 -> s32), reading int8 codes directly:
 * Xq int8 [M][K] and Wq int8 [N][K] from sq_quantize_act / sq_pack_weight.
 * Exact by construction; kept as the comparison point for sq_linear_i8.
 * K <= 133144 (|acc| < 2^31 for any codes). */
sq_status sq_linear_i8_mma_sync(const int8_t *Xq, const float *x_scale, const int8_t *Wq,
                                const float *w_scale, const float *bias, const float *residual,
                                int64_t M, int64_t N, int64_t K, int mode, void *Y,
                                void *stream);

/* ---- Self-check of the epilogue's division --------------------------------- */

/* sq_linear_i8_requant divides its results by the next layer's smoothing
 * factor (y / s_next[n], Table 10) with a per-column reciprocal
 * y = RN(1/s) and one fused correction,
 *   q0 = RN(x y),  r = RN(x - s q0),  q = RN(q0 + r y),
 * which is the IEEE quotient RN(x / s) in the range it is used.  Scaling x or
 * s by a power of two scales every step exactly, so correctness is a property
 * of the 2^46 significand pairs.  This entry point runs the kernel's own
 * routine against IEEE division on the pairs a = 1 + af 2^-23,
 * b = 1 + bf 2^-23 with bf in [b_first, b_first + b_count) and af in
 * [a_first, a_first + a_count) (fraction fields, each range within [0, 2^23)).
 * corrected = 0 checks the uncorrected RN(x RN(1/s)) instead (a control that
 * does differ on some pairs).  out: two unsigned 64-bit words in device
 * memory (8-byte aligned), zeroed by the caller: out[0] += the number of pairs
 * that differ; out[1] = 1 + (af << 32 | bf) of one differing pair (unchanged if
 * none).  One thread per b; a call costs about b_count * a_count / 2e12 s. */
sq_status sq_check_division(uint32_t b_first, uint32_t b_count, uint32_t a_first,
                            uint32_t a_count, int corrected, unsigned long long *out,
                            void *stream);

/* ---- The linear block on host buffers -------------------------------------- */

/* One linear layer for sq_linear_block_host.  Device pointers as for
 * sq_quantize_act / sq_quantize_act_table / sq_quantize_act_static and
 * sq_linear_i8; static_scale > 0 selects Smooth-Static with that per-tensor
 * scale, 0 Smooth-Dynamic (then s_table, if not NULL, is sq_division_table(s)). */
typedef struct {
    int64_t K, N;             /* input and output features (K a multiple of 16) */
    int mode;                 /* epilogue: SQ_EPI_NONE .. SQ_EPI_BIAS_RESIDUAL */
    float static_scale;       /* > 0: Smooth-Static scale; 0: Smooth-Dynamic */
    const float *s;           /* smoothing factor [K] */
    const float *s_table;     /* [K][2] division table of s, or NULL */
    const void *Wop;          /* packed weight operand [N][K] (sq_pack_weight) */
    const float *w_scale;     /* [N] */
    const int32_t *w_row_l1;  /* [N] row L1 norms of the weight codes, or NULL */
    const float *bias;        /* [N] or NULL */
    const float *residual;    /* [M][N] or NULL (mode SQ_EPI_BIAS_RESIDUAL) */
} sq_linear_layer;

/* Device scratch that sq_linear_block_host needs for layers of at most max_K
 * inputs and max_N outputs at M tokens: two input slots (M x max_K fp32), two
 * output slots (M x max_N fp32), the operand (M x max_K bf16 codes) and the
 * per-token scales, each 256-byte aligned. */
sq_status sq_linear_block_host_scratch_bytes(int64_t M, int64_t max_K, int64_t max_N,
                                             size_t *bytes);

/* The INT8 linear block (Table 3's linear-block share: quantise, GEMM, fused
 * post-operations) on activations in host memory:
 * Y_host[i] = the linear block of layers[i] on X_host[i] for every i < count
 * (fp32 [M][K_i] in, fp32 [M][N_i] out, host memory; pinned memory makes the
 * copies asynchronous and lets them overlap): per layer the input is copied to
 * the device on stream_h2d, quantised and multiplied (the layer's quantiser,
 * then sq_linear_i8 with its epilogue) on stream_compute, and the output copied
 * back on stream_d2h, through two device slots for inputs and two for outputs
 * in `scratch` (sq_linear_block_host_scratch_bytes over the layers' largest K
 * and N), so that layer i's kernels overlap the copies of layers i + 1 and
 * i - 1.  The streams may coincide (no overlap then).  Returns once everything
 * is enqueued; the outputs are complete when stream_d2h is (synchronise it
 * before reading Y_host).  The call orders its own work through CUDA events
 * it creates and releases; ordering with other work on the device (e.g. the
 * producers of the weights) is the caller's.  scratch 256-byte aligned.
 * Errors: SQ_ERR_INVALID_ARG (NULL arrays or pointers, count or M < 0, K or N
 * <= 0, a mode outside 0..3, scratch too small), SQ_ERR_ALIGNMENT (K % 16,
 * scratch), and the statuses of the calls it makes (checked for every layer
 * before anything is enqueued). */
sq_status sq_linear_block_host(const sq_linear_layer *layers, int64_t count, int64_t M,
                               const float *const *X_host, float *const *Y_host, void *scratch,
                               size_t scratch_bytes, void *stream_h2d, void *stream_compute,
                               void *stream_d2h);

/* ---- Device status --------------------------------------------------------- */

/* Synchronises `stream`, then reports and clears the library's device error
 * word for the current device: SQ_ERR_TIMEOUT if a kernel's bounded
 * pipeline wait ran out since the last call (that kernel's output is then
 * incomplete), SQ_ERR_CUDA if the stream reported an error, else SQ_OK. */
sq_status sq_device_status(void *stream);

/* The same as sq_device_status (the name under which the device error word's
 * report is also known). */
sq_status sq_get_device_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SQ_GB300_H */
