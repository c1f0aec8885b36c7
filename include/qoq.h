/*
 * qoq.h -- C ABI of the GB300 (sm_103a) W4A8 linear layer of QServe's QoQ
 * scheme (g128, and the other group sizes below): progressive group
 * quantization of the weights, per-token int8 activations, and the integer
 * GEMM with an fp16 epilogue.
 *
 * Sources (web pages on W4A8 serving):
 *  [QS]  QServe talk write-up (greptalks.ai, MLSys'25), "Technical Deep Dive":
 *        sections "Progressive Group Quantization for W4A8 GEMM", "Precision
 *        Data Flow and Activation Quantization Fusion", "Quantized Matrix
 *        Multiplication (GEMM) Kernel on GPUs" and "Challenges and Design
 *        Details of QServe GEMM Kernel".
 *  [L15] Lecture 15 notes (cs2680), section 15.6 "QServe: W4A8KV4, and paying
 *        for dequant once", and section 15.5 "The kernel trap".
 *  [QF]  QFactory notes (papercache.org), section 2 (dequantization
 *        w = (w_quant - zero) * scale) and Fig. 3.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers on the current CUDA device; the
 *    caller allocates and owns every buffer (including the workspace).  The
 *    library allocates no device memory and keeps no state beyond a cached
 *    per-device attribute lookup, the debug settings below, and the fixed
 *    device array behind qoq_w4a8_gemm_no_alloc.
 *  - Host buffers at the two ends of the path: X_f16 (qoq_quant_act,
 *    qoq_norm_quant_act) and Y_f16 (qoq_w4a8_gemm, qoq_w4a8_gemm_no_alloc)
 *    may instead point to page-locked host memory that the device can address
 *    (cudaHostAlloc / cudaHostRegister; with unified addressing the host
 *    pointer is the device pointer).  The kernels then read X, or write Y,
 *    directly across the host link, with no staging copy; Y is in host
 *    memory once the call's work on `stream` has completed.  Any other host
 *    pointer there is undefined behaviour: the library cannot tell the two
 *    kinds apart.
 *  - fp16 values cross the ABI as their IEEE binary16 bit patterns (uint16_t).
 *  - Matrices are dense row-major.  W is [N][K] (row n = output channel),
 *    X / Xq are [M][K] (row m = token), Y is [M][N]: Y = X * W^T.
 *  - Every compute call is asynchronous on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  Only qoq_last_device_status synchronizes.
 *  - Argument checks happen on the host before any launch and return an error
 *    code without touching the device; launch failures return QOQ_ERR_CUDA.
 *    The library never aborts, prints or throws across this boundary.
 *  - Requirements shared by the compute calls: N % 128 == 0 and K % 128 == 0
 *    (else QOQ_ERR_SHAPE); the level-2 group size g is 32, 64, or a multiple
 *    of 128 that divides K (128 is the pages' g128; g = K is one group per
 *    output channel) (else QOQ_ERR_UNSUPPORTED);
 *    1 <= M <= 2^24, 128 <= N <= 2^24, 128 <= K <= 131072 (the int32
 *    accumulator bound 127 * 127 * K < 2^31); pointers 16-byte aligned
 *    (else QOQ_ERR_MISALIGNED); a compute capability 10.3 device (else
 *    QOQ_ERR_ARCH).
 */
#ifndef QOQ_H
#define QOQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t. */
typedef struct CUstream_st* qoq_stream_t;

typedef enum {
  QOQ_OK = 0,
  QOQ_ERR_NULL = 1,          /* a required pointer is NULL */
  QOQ_ERR_SHAPE = 2,         /* M, N or K out of range or not a multiple of 128 */
  QOQ_ERR_UNSUPPORTED = 3,   /* group size g not 32, 64 or a multiple of 128 dividing K; bad norm kind or eps */
  QOQ_ERR_MISALIGNED = 4,    /* a pointer is not 16-byte aligned */
  QOQ_ERR_WORKSPACE = 5,     /* workspace NULL or smaller than qoq_gemm_workspace_bytes */
  QOQ_ERR_CUDA = 6,          /* a CUDA runtime call or kernel launch failed */
  QOQ_ERR_DEVICE_TIMEOUT = 7, /* a device-side pipeline wait ran out (see qoq_last_device_status) */
  QOQ_ERR_ARCH = 8           /* current device is not compute capability 10.3 (GB300) */
} qoq_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* qoq_status_str(int status);

/* ABI version of this library (major * 100 + minor). */
int qoq_version(void);

/*
 * Bytes of the packed weight blob for an [N][K] weight at group size g
 * (host-only, no device access).  Returns 0 for an unsupported shape.
 *
 * Layout ([QS] "compute-aware weight reordering": weights are stored in the
 * order the GEMM consumes them, so one contiguous copy serves one pipeline
 * stage): (N/128) x (K/128) k-tiles of T = 256 * S + 8192 bytes, where
 * S = 128 / g scale sets for g = 32 or 64 and S = 1 for g >= 128 (T = 8448
 * for g >= 128, 8704 for g = 64, 9216 for g = 32).  Tile (nt, j) sits at
 * offset (nt * (K/128) + j) * T and holds output rows 128*nt .. 128*nt+127
 * and input channels 128*j .. 128*j+127:
 *   bytes 256u ..      256u + 127 : s2[r] of scale set u (1..16), u < S
 *   bytes 256u + 128 .. 256u + 255 : z[r]  of scale set u (0..15)
 *     (scale set u covers channels 128*j + u*g .. +g-1 when g < 128; for
 *     g >= 128 the one set repeats the scales of the group the tile lies in)
 *   bytes 256S .. T-1 : four 2048-byte chunks c = 0..3 (k = 32c .. 32c+31);
 *                     chunk c holds row r's 16 bytes at offset 16 r; inside,
 *                     32-bit word w (k = 32c + 8w .. +7) carries the code of
 *                     k = 32c + 8w + 2i in bits 4i..4i+3 and that of
 *                     k = 32c + 8w + 2i + 1 in bits 16+4i..16+4i+3 (i = 0..3).
 * That is 4 + 16 S/128 bits per weight plus the fp16 s1 per row.
 */
size_t qoq_packed_weight_bytes(int N, int K, int g);

/*
 * Bytes of device workspace that qoq_w4a8_gemm needs for (M, N, K, g)
 * (host-only; 0 for an unsupported shape).  It holds a status header and
 * the split-K state: for M <= 64 one slot per CTA of partial sums, each
 * tagged with an epoch that the kernel keeps in the header and advances at
 * the end of every launch (BN x 128 x 8 bytes, BN = 16, 32 or 64 as M needs,
 * 160 slots); for M > 64 tile counters and int32 partial sums, and an fp16
 * copy of Xq laid out for the tensor-core B operand; and, for
 * qoq_w4a8_gemm_zero_folded, int32 row sums of Xq per 128-channel k-tile.
 * The caller zero-fills the workspace once after allocating it (e.g.
 * cudaMemsetAsync); every call that completes leaves it fit for the next
 * call of any shape that it is large enough for, so no per-call clearing is
 * needed.  This holds for launches replayed from a captured CUDA graph too:
 * the hand-off tag comes from the device, not from the launch parameters.
 * After a call that reported QOQ_ERR_DEVICE_TIMEOUT, zero-fill it again
 * before reuse.  Two calls in flight at the same time must not share one
 * workspace.
 */
size_t qoq_gemm_workspace_bytes(int M, int N, int K, int g);

/*
 * Offline weight preparation ([QS] "Progressive Group Quantization for W4A8
 * GEMM"; [L15] 15.6), one call per layer:
 *   level 1, per output channel n (symmetric, protective range):
 *     s1[n] = fp16_rn(fp32(max_k |W[n,k]|) / 119)   (IEEE fp32 divide),
 *     Q8[n,k] = clamp(rint(W[n,k] / s1[n]), -119, 119) (fp32 divide, ties even);
 *     an all-zero row, or one whose s1 underflows to 0, gets s1 = 0, Q8 = 0;
 *   level 2, per group of g input channels (asymmetric uint4):
 *     lo = min(0, min Q8), hi = max(0, max Q8),
 *     s2 = max(1, ceil((hi - lo) / 15)), z = rne(-lo / s2),
 *     q4 = clamp(rne(Q8 / s2) + z, 0, 15)   (exact integer, ties to even),
 *   so that w8 = (q4 - z) * s2 ([QF] dequantization) lies in [-127, 127].
 * In:  W_f16 [N][K] fp16 bits.
 * Out: packed, qoq_packed_weight_bytes(N, K, g) bytes in the layout above;
 *      s1_f16 [N] fp16 bits.
 */
qoq_status qoq_pack_weights(int N, int K, int g, const uint16_t* W_f16, uint8_t* packed,
                            uint16_t* s1_f16, qoq_stream_t stream);

/*
 * Per-token symmetric int8 activation quantization ([QS] "Precision Data
 * Flow": every linear layer takes 8-bit activations):
 *   s_x[m] = fp16_rn(fp32(max_k |X[m,k]|) / 127),
 *   Xq[m,k] = clamp(rint(X[m,k] / s_x[m]), -127, 127) (fp32 divide, ties even);
 *   an all-zero row gets s_x = 0, Xq = 0.
 * In:  X_f16 [M][K] fp16 bits.  Out: Xq [M][K] int8, sx_f16 [M] fp16 bits.
 * Shape rules as above except that N and g are not involved.
 * Launched with programmatic dependent launch: it may become resident while
 * the preceding kernel runs and waits for that kernel to complete before it
 * reads X or writes Xq and s_x.
 */
qoq_status qoq_quant_act(int M, int K, const uint16_t* X_f16, int8_t* Xq, uint16_t* sx_f16,
                         qoq_stream_t stream);

/* Norm kinds of qoq_norm_quant_act. */
typedef enum { QOQ_NORM_RMS = 0, QOQ_NORM_LAYER = 1 } qoq_norm_kind;

/*
 * The preceding norm fused with the per-token int8 quantizer ([QS] "Precision
 * Data Flow and Activation Quantization Fusion": activation quantization is
 * fused into the preceding layer, such as LayerNorm, whose output is
 * quantized to 8 bits directly, without writing the normalized fp16 rows).
 * Per token row x (K fp16 values), with exact row statistics
 * S1 = sum_k x_k, S2 = sum_k x_k^2 (integers in units of 2^-24 and 2^-48),
 * each rounded once to fp32 (fl32), and every fp32 operation below rounded
 * to nearest:
 *   QOQ_NORM_RMS:   r = 1 / sqrt(fl32(S2) / K + eps),
 *                   y_k = fp16_rn(fl32(fl32(x_k * r) * gamma_k));
 *   QOQ_NORM_LAYER: mu = fl32(S1) / K,
 *                   r = 1 / sqrt(fl32(K S2 - S1^2) / K^2 + eps),
 *                   y_k = fp16_rn(fl32(fl32(fl32(fl32(x_k - mu) * r) * gamma_k) + beta_k));
 * then s_x and Xq of the rows y exactly as qoq_quant_act computes them.
 * In:  X_f16 [M][K] fp16 bits (finite values), gamma_f16 [K], beta_f16 [K]
 *      (LayerNorm only; may be NULL for RMSNorm), eps > 0 and finite.
 * Out: Xq [M][K] int8, sx_f16 [M] fp16 bits.
 * Errors: QOQ_ERR_UNSUPPORTED for an unknown kind or eps <= 0; otherwise as
 * qoq_quant_act.  Launched like qoq_quant_act (programmatic dependent launch:
 * it waits for the preceding kernel before reading X or writing its outputs).
 */
qoq_status qoq_norm_quant_act(int M, int K, int kind, float eps, const uint16_t* X_f16,
                              const uint16_t* gamma_f16, const uint16_t* beta_f16, int8_t* Xq,
                              uint16_t* sx_f16, qoq_stream_t stream);

/*
 * The W4A8 GEMM ([QS] "Quantized Matrix Multiplication (GEMM) Kernel on
 * GPUs": 4-bit weights are dequantized to 8 bits before the tensor cores,
 * the per-channel scales are applied in the epilogue):
 *   acc[m,n] = sum_k Xq[m,k] * ((q4[n,k] - z[n,k/g]) * s2[n,k/g])  (exact int32),
 *   Y[m,n]   = fp16_rn(float(acc[m,n]) * (float(s_x[m]) * float(s1[n]))).
 * In:  Xq [M][K] int8 and sx_f16 [M] (from qoq_quant_act); packed and s1_f16
 *      (from qoq_pack_weights).
 * Out: Y_f16 [M][N] fp16 bits; acc_debug [M][N] int32 when not NULL.
 * workspace: ws_bytes >= qoq_gemm_workspace_bytes(M, N, K, g), 16-byte
 *      aligned, zero-filled once by the caller (see above), used by one call
 *      at a time.
 * The kernels are launched with programmatic dependent launch: the GEMM
 * starts streaming weights while the preceding kernel on the stream (e.g.
 * qoq_quant_act) finishes, and waits for it before reading Xq and s_x and
 * before touching Y, acc_debug or the workspace.  packed and s1_f16 are read
 * before that wait, so they must not be written by a kernel that can still be
 * running when this call starts (pack weights once, at load time).  For
 * M <= 64 the GEMM in turn lets the next kernel on the stream launch as soon
 * as it starts; that kernel (qoq_quant_act, another qoq_w4a8_gemm) waits for
 * the GEMM to complete before it reads or writes anything the GEMM uses.
 * A device-side pipeline stall that exceeds the wait limit ends the kernel
 * early, leaves Y undefined and records QOQ_ERR_DEVICE_TIMEOUT in the
 * workspace header, which qoq_last_device_status returns.
 */
qoq_status qoq_w4a8_gemm(int M, int N, int K, int g, const int8_t* Xq, const uint16_t* sx_f16,
                         const uint8_t* packed, const uint16_t* s1_f16, uint16_t* Y_f16,
                         int32_t* acc_debug, void* workspace, size_t ws_bytes,
                         qoq_stream_t stream);

/*
 * The same GEMM with the zero points folded out of the main loop (QFactory
 * notes, papercache.org, section 4.3 "mapping function transformation",
 * Table 2: a matmul whose operand carries an offset becomes the offset-free
 * product plus a product with the all-ones matrix J, whose rows are sums
 * over the reduction).  With zs = z * s2 per (row, group) and the per-group
 * row sums RS[m, j] = sum of Xq[m, k] over the channels k of group j:
 *   acc[m,n] = sum_k Xq[m,k] * (q4[n,k] * s2[n,k/g])  -  sum_j zs[n,j] * RS[m,j],
 * which equals qoq_w4a8_gemm's acc exactly (integer distributivity); Y as
 * there.  The tensor cores see q4 * s2 (no zero point per weight); a
 * pre-pass kernel writes RS into the workspace, and the epilogue subtracts
 * the zs * RS terms.
 * Arguments, results, workspace (qoq_gemm_workspace_bytes covers it) and
 * errors as qoq_w4a8_gemm, except that the group size must be a multiple of
 * 128 (g = 32 or 64 return QOQ_ERR_UNSUPPORTED).  Launches: the row-sum
 * pre-pass, then (M > 64) the B-operand copy, then the GEMM, all with
 * programmatic dependent launch.
 */
qoq_status qoq_w4a8_gemm_zero_folded(int M, int N, int K, int g, const int8_t* Xq,
                                     const uint16_t* sx_f16, const uint8_t* packed,
                                     const uint16_t* s1_f16, uint16_t* Y_f16, int32_t* acc_debug,
                                     void* workspace, size_t ws_bytes, qoq_stream_t stream);

/*
 * W4Ax: 4-bit activation blocks with 8-bit outlier blocks (COMET explainer,
 * bookshelf: FMPQ quantizes activations in blocks of 128 channels, the size
 * of the tensor-core tile, keeping the blocks that hold the outlier channels
 * at 8 bits and the rest at 4 bits; a channel permutation clusters the
 * outlier channels into few blocks, and the W4Ax kernel scales each block's
 * partial sums on the general-purpose cores).  Here the permutation is
 * applied upstream (to this layer's weight columns and to the producer of
 * its activations) so that the outlier blocks come first: the n8 leading
 * blocks are 8-bit.
 *
 * Activation row layout ("Xa"): per token row, blocks in order; an 8-bit
 * block is 128 int8 codes; a 4-bit block is 64 bytes, byte i holding the code
 * of channel 2i in its low nibble and that of channel 2i + 1 in its high
 * nibble, two's complement.  Row stride 128 n8 + 64 (K/128 - n8) bytes;
 * qoq_w4ax_act_bytes(M, K, n8) is M times that (0 for bad arguments).
 */
size_t qoq_w4ax_act_bytes(int M, int K, int n8);

/*
 * Per-(token, block) symmetric quantization for W4Ax:
 *   q = 127 for blocks b < n8, 7 otherwise,
 *   sxb[m][b] = fp16_rn(fp32(max over the block |X[m,k]|) / q) (IEEE fp32 divide),
 *   code = clamp(rint(X[m,k] / sxb[m][b]), -q, q)  (fp32 divide, ties even);
 *   an all-zero block gets scale 0 and codes 0.
 * In:  X_f16 [M][K] fp16 bits; 0 <= n8 <= K/128 (else QOQ_ERR_UNSUPPORTED).
 * Out: Xa (qoq_w4ax_act_bytes(M, K, n8) bytes, the layout above),
 *      sxb_f16 [M][K/128] fp16 bits.
 * Shape and pointer rules as qoq_quant_act; launched the same way
 * (programmatic dependent launch).
 */
qoq_status qoq_quant_act_w4ax(int M, int K, int n8, const uint16_t* X_f16, uint8_t* Xa,
                              uint16_t* sxb_f16, qoq_stream_t stream);

/* Bytes of workspace qoq_w4ax_gemm needs (host-only; 0 for a bad shape);
 * zero-filled once by the caller, like qoq_w4a8_gemm's. */
size_t qoq_w4ax_workspace_bytes(int M, int N, int K, int g);

/*
 * The W4Ax GEMM with the progressively quantized 4-bit weights of
 * qoq_pack_weights (w8 = (q4 - z) * s2):
 *   acc_b[m,n] = sum over the channels k of block b of code[m,k] * w8[n,k]  (exact),
 *   Y[m,n] = fp16_rn(s1[n] * sum_b sxb[m][b] * acc_b[m,n]),
 * the sum over blocks in fp32 on the GPU (the oracle takes it in double; the
 * two agree within the parity tolerance).  For a tile whose K range is split
 * over two or more CTAs the fp32 partial sums meet through atomic additions,
 * so Y may differ between calls by the rounding of the last fp32 bit.
 * acc_debug (nullable): sum_b acc_b as int32, written by a second launch of
 * the W4A8 kernel on the same operand copy.
 * Every M runs on the 128-token-tile kernel (COMET's kernel targets the
 * compute-bound, large-batch regime).  Errors as qoq_w4a8_gemm, plus
 * QOQ_ERR_UNSUPPORTED for n8 outside [0, K/128]; workspace:
 * qoq_w4ax_workspace_bytes.
 */
qoq_status qoq_w4ax_gemm(int M, int N, int K, int g, int n8, const uint8_t* Xa, const uint16_t* sxb_f16,
                         const uint8_t* packed, const uint16_t* s1_f16, uint16_t* Y_f16, int32_t* acc_debug,
                         void* workspace, size_t ws_bytes, qoq_stream_t stream);

/*
 * qoq_w4a8_gemm without a caller-supplied workspace.  The paper has no
 * counterpart: this is a service for callers that cannot allocate device
 * memory.  Examples are a plugin given only its input and output buffers by a
 * host program that does not share its allocator, a serving process that
 * reserved nearly all device memory for its caches at start-up, and a step
 * that must not synchronise the device as cudaMalloc/cudaFree may.
 *
 * Arguments, results and argument errors are those of qoq_w4a8_gemm, with no
 * workspace.  The workspace lives in a static device array of
 * QOQ_NO_ALLOC_SCRATCH_BYTES (16 MiB), which every GPU that loads the library's
 * device code holds until the process exits.  This entry point allocates
 * nothing and calls no allocating routine.
 *
 * Limit: a shape whose qoq_gemm_workspace_bytes(M, N, K, g) exceeds
 * QOQ_NO_ALLOC_SCRATCH_BYTES returns QOQ_ERR_WORKSPACE before any device
 * access.  Every shape with M <= 64 fits (2.5 MiB for M <= 16, 5 MiB for
 * M <= 32, 10 MiB for M <= 64, whatever N and K).  Larger M fits only for
 * small problems.
 *
 * The first call on a device (with that device current) looks up the array's
 * device address once and checks the architecture.  Make that first call
 * before any stream capture on that device.  A failed look-up returns
 * QOQ_ERR_CUDA and is not retried.
 *
 * Every call shares the one array per device.  Each call first clears, on
 * `stream`, the part that must start at zero (a small extra kernel), then
 * runs the GEMM in it.  Calls that can overlap on the GPU (other streams,
 * other host threads) race on the array and give wrong results: serialise
 * them.  A device-side wait timeout leaves Y undefined; the next call still
 * starts from a cleared array, and qoq_no_alloc_last_status reports it.
 */
#define QOQ_NO_ALLOC_SCRATCH_BYTES ((size_t)16 << 20)
qoq_status qoq_w4a8_gemm_no_alloc(int M, int N, int K, int g, const int8_t* Xq,
                                  const uint16_t* sx_f16, const uint8_t* packed,
                                  const uint16_t* s1_f16, uint16_t* Y_f16, int32_t* acc_debug,
                                  qoq_stream_t stream);

/*
 * The device status of the qoq_w4a8_gemm_no_alloc calls on the current
 * device since the previous read: synchronizes `stream` (the stream those
 * calls ran on), returns QOQ_OK, QOQ_ERR_DEVICE_TIMEOUT if any of them ran out
 * of a device-side wait limit (sticky: each call's clearing step keeps its
 * predecessor's status), or QOQ_ERR_CUDA (a CUDA error, e.g. one surfaced by
 * the synchronization), and resets the status.  Like the calls themselves,
 * not safe against no-alloc calls running concurrently.
 */
qoq_status qoq_no_alloc_last_status(qoq_stream_t stream);

/*
 * Inverse of the packing layout, for testing: recovers the logical codes.
 * Out: q4 [N][K] (one code per byte), s2 [N][K/g], z [N][K/g].
 */
qoq_status qoq_unpack_weights_debug(int N, int K, int g, const uint8_t* packed, uint8_t* q4,
                                    uint8_t* s2, uint8_t* z, qoq_stream_t stream);

/*
 * Synchronizes `stream`, then reads and clears the device status recorded in
 * `workspace` by the qoq_w4a8_gemm calls since the previous read (the status
 * is sticky: any timeout among them is reported).  Returns QOQ_OK,
 * QOQ_ERR_DEVICE_TIMEOUT, or QOQ_ERR_CUDA (a CUDA error surfaced by the
 * synchronization, e.g. a failed kernel).
 */
qoq_status qoq_last_device_status(void* workspace, qoq_stream_t stream);

/*
 * Test hooks (process-wide, not thread-safe; leave at defaults in production).
 * wait_timeout_ns: limit of every device-side pipeline wait (0 = default, 2 s).
 * fault: 0 = none; 1 = the GEMM's copy producer skips one pipeline stage, so
 * that the waits downstream of it run out and the kernel returns with
 * QOQ_ERR_DEVICE_TIMEOUT recorded (no trap, no invalid access).
 */
qoq_status qoq_set_debug(uint64_t wait_timeout_ns, int fault);

#ifdef __cplusplus
}
#endif

#endif /* QOQ_H */
