/*
 * fa.h - C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * The operation (per batch b and head h, for every query row i):
 *
 *     O[b,h,i,:] = sum_{j in J(i)} softmax_j(scale * q_i . k_j) * v_j
 *     LSE[b,h,i] = ln sum_{j in J(i)} exp(scale * q_i . k_j)
 *
 * with J(i) = {0..N-1}, or {0..i} when causal. It is the flash-attention
 * forward pass: scores are produced tile by tile with an online softmax, so
 * the N x N score matrix never reaches HBM. Sources:
 *   - "TCA 51%, MFU below 8%" (zhihu), section on Flash Attention 2 and the
 *     online softmax (O is softmax(QK^T) V accumulated block by block);
 *   - "TMA + Warp Specialization" (CUDA book ch. 17), sections 17.3-17.5
 *     (TMA descriptors, producer / consumer loop, final O / row_sum);
 *   - "Flash Attention CUDA Kernel: 56 to 986 TFLOPS on B300, G4" (hjcheng0602
 *     blog), versions V14-V16 (TMA + tcgen05 with accumulators in TMEM).
 *   The causal mask and the logsumexp output are part of this library's
 *   specification; the pages do not define them.
 *
 * All entry points are plain C: pointers and sizes, no framework types.
 */
#ifndef FA_SM103_H
#define FA_SM103_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size, bad scale or dtype */
  FA_ERR_UNSUPPORTED = 2, /* head dim not 64 or 128, or sizes beyond the 32-bit limits */
  FA_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed (launch, attribute, encode) */
  FA_ERR_ARCH = 4,        /* the current device is not compute capability 10.3 */
  FA_ERR_TIMEOUT = 5      /* a kernel wait ran past its limit (reported by fa_check) */
} fa_status;

typedef enum fa_dtype {
  FA_DTYPE_FP16 = 0, /* IEEE binary16 */
  FA_DTYPE_BF16 = 1  /* bfloat16 */
} fa_dtype;

/* Element strides of one tensor viewed as [B][H][N][d] (the d stride is 1):
 * element (b, h, n, t) is at base + b*b_stride + h*h_stride + n*n_stride + t. */
typedef struct fa_strides {
  long long b; /* batch stride */
  long long h; /* head stride */
  long long n; /* row (sequence position) stride */
} fa_strides;

/*
 * fa_fwd - enqueue one fused attention forward on `stream`.
 *
 * q, k, v : device pointers, contiguous [B][H][N][d] of `dtype` (16-bit
 *           elements, row i of head (b,h) at ((b*H + h)*N + i)*d).
 *           Caller-owned, read only. 16-byte aligned.
 * o       : device pointer, contiguous [B][H][N][d] of `dtype`, written.
 *           Rounded to nearest even from the fp32 result. 16-byte aligned.
 * lse     : device pointer, contiguous [B][H][N] float32, written: the
 *           natural-log logsumexp of the scaled scores of each row.
 * B, H, N : batch, heads, sequence length (queries = keys = N), each >= 1,
 *           N <= 2^30, B*H*ceil(N/256) <= 2^31-1. Any N is accepted: the last
 *           key tile is masked and rows past N are neither read nor written.
 * d       : head dimension, 64 or 128.
 * causal  : 0 = full attention, nonzero = query i attends keys 0..i.
 * scale   : score scale (usually 1/sqrt(d)); finite and > 0.
 * dtype   : FA_DTYPE_FP16 or FA_DTYPE_BF16 (both inputs and O).
 * stream  : cudaStream_t to enqueue on (NULL = legacy default stream).
 *
 * Asynchronous: returns after the launch is enqueued; O and LSE are valid
 * once the stream reaches that point. Arguments are checked before anything
 * is enqueued; on any error nothing is launched and nothing is written.
 * Head dimension 128 runs on CTA pairs (fa_fwd_pair) when the problem fills
 * the GPU and is not causal, or causal with N >= 16384 (see fa_query_launch);
 * the results do not depend on it.
 * The first call on a device allocates a small device status word for that
 * device (kept until process exit); later calls allocate nothing.
 * A kernel whose internal waits run past their limit stops early and records
 * the failure in that status word: call fa_check to read it.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, int causal, float scale,
                 fa_dtype dtype, void* stream);

/*
 * fa_fwd_pair - fa_fwd computed by pairs of CTAs on neighbouring SMs that
 * share each tensor-core product (tcgen05.mma cta_group::2, M = 256 query
 * rows): the CTA pair of "TMA + Warp Specialization" (CUDA book ch. 17),
 * section 17.9, item 3. Each SM holds two 128-row query tiles and loads and
 * keeps only half of every K and V tile (64 keys of K, 64 columns of V); the
 * per-tile arithmetic is fa_fwd's, and so are the results, bit for bit.
 *
 * Same arguments, layout, errors, asynchrony and status word as fa_fwd, but
 * d must be 128 (else FA_ERR_UNSUPPORTED). Launches clusters of 2 CTAs, one
 * per pair of SMs, each unit 512 query rows of one (batch, head).
 */
fa_status fa_fwd_pair(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H, int N, int d, int causal, float scale,
                      fa_dtype dtype, void* stream);

/*
 * fa_fwd_strided - fa_fwd on tensors in any [B][H][N][d] view with unit d
 * stride: e.g. the [B][N][H][d] layout of a fused projection output
 * (strides {N*H*d, d, H*d}), or rows padded to a longer pitch. This is the
 * layout extension of the seq-major tensor maps of the B300 walkthrough
 * (V14, TMA descriptor section); the pages use contiguous tensors only.
 *
 * strides : host pointer to 4 fa_strides, for q, k, v and o in that order,
 *           in elements. Every stride must be a positive multiple of 8
 *           elements (16 bytes: tensor-map rows and 16-byte output stores)
 *           and every n stride at least d (else FA_ERR_INVALID_ARG); strides
 *           of 2^38 elements or more return FA_ERR_UNSUPPORTED. Read during
 *           the call only.
 * o       : written rows must not overlap one another or q, k, v (not
 *           checked; overlapping outputs give undefined results).
 * lse     : contiguous [B][H][N] float32, as in fa_fwd.
 * Everything else (arguments, errors, asynchrony, status word) is as in
 * fa_fwd; a bad stride returns FA_ERR_INVALID_ARG before anything is
 * enqueued.
 */
fa_status fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, const fa_strides* strides, int causal,
                         float scale, fa_dtype dtype, void* stream);

/*
 * fa_fwd_fp8 - the forward on 8-bit inputs: FP8 E4M3 (OCP 8-bit floating
 * point, "fn" variant: bias 7, 3 fraction bits, no infinities, largest finite
 * 448), after the FP8 path of "TMA + Warp Specialization" (section 17.7):
 * one scale per 128-key block of K, the softmax weights P rounded to 8 bits
 * before the P V product, fp32 accumulation.
 *
 * q, k     : device, contiguous [B][H][N][128] e4m3 codes (one byte each).
 * vt       : device, V transposed: [B][H][128][ldv] e4m3 codes, byte
 *            (b, h, t, n) holding V[b][h][n][t]; bytes n >= N of a row are
 *            not read.
 * ldv      : row length of vt in bytes: ldv >= N and a multiple of 16.
 * k_scales : device float32 [B][H][ceil(N / 128)]: the scale of each 128-key
 *            block of K (finite and > 0; not checked, it is device memory).
 * q_scale, v_scale : scales of Q and V, finite and > 0.
 *            The values are q = q_scale * q8, k_n = k_scales[b][h][n/128] *
 *            k8_n and v = v_scale * v8.
 * o        : device, contiguous [B][H][N][128] bfloat16, written.
 * lse      : as fa_fwd (natural-log logsumexp of the scaled scores).
 * d        : must be 128 (else FA_ERR_UNSUPPORTED).
 * All pointers 16-byte aligned (k_scales 4-byte aligned). Other arguments,
 * errors, asynchrony and the status word are as in fa_fwd.
 *
 * Precision: each weight p of a row (largest weight in [1, 256] on the
 * kernel's scale) is rounded to e4m3, O is normalised by the unrounded sum;
 * per element |O - O_exact| <= sum_j (2^-4 p_j + 2^-10) |v_j| / sum_j p_j with
 * p_j = exp(s_j - max s) (plus fp32 and bf16 output rounding). The LSE is
 * computed from the unrounded weights.
 */
fa_status fa_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse,
                     int B, int H, int N, int d, int ldv, float q_scale,
                     const float* k_scales, float v_scale, int causal, float scale,
                     void* stream);

/*
 * fa_fwd_fp8_pair - fa_fwd_fp8 computed by pairs of CTAs sharing each
 * tensor-core product (tcgen05.mma cta_group::2, M = 256 query rows), as
 * fa_fwd_pair does for 16-bit inputs: each SM keeps half of every K and V^T
 * tile, and the 8-bit weights P go through shared memory to the P V product.
 * Same arguments, layout, precision, errors, asynchrony and status word as
 * fa_fwd_fp8, whose results it reproduces bit for bit.
 */
fa_status fa_fwd_fp8_pair(const void* q, const void* k, const void* vt, void* o, float* lse,
                          int B, int H, int N, int d, int ldv, float q_scale,
                          const float* k_scales, float v_scale, int causal, float scale,
                          void* stream);

/*
 * fa_bwd - enqueue the backward pass of fa_fwd: gradients dq, dk, dv of a
 * loss whose gradient at O is dout. The backward recomputes the scores
 * instead of storing them ("TCA 51%, MFU below 8%", section "MFU is always a
 * little below TCA"); here the softmax weights are recomputed from the
 * forward's lse, which is why the forward emits it (this library's reading):
 *     P_ij = exp(scale q_i.k_j - lse_i),  D_i = dout_i . o_i
 *     dv_j = sum_i P_ij dout_i,           dS_ij = P_ij (dout_i . v_j - D_i)
 *     dq_i = scale sum_j dS_ij k_j,       dk_j = scale sum_i dS_ij q_i
 * with j in J(i) as in fa_fwd.
 *
 * q, k, v, o, dout : device, contiguous [B][H][N][d] of `dtype` (o is the
 *            forward's output for these q, k, v), read only.
 * lse      : device, [B][H][N] float32, the forward's logsumexp.
 * dq, dk, dv : device, contiguous [B][H][N][d] of `dtype`, written (fp32
 *            accumulation, rounded to nearest even).
 * workspace : device scratch of fa_bwd_workspace_size bytes, caller-owned; its
 *            contents are overwritten (row logsumexps and D); it must not be
 *            used by another call on another stream at the same time.
 * All pointers 16-byte aligned. B, H, N, d, causal, scale, dtype, stream and
 * the errors are as in fa_fwd, and B*H*ceil(N/128) >= 2^31 returns
 * FA_ERR_UNSUPPORTED. Three launches on `stream` (a pass forming D,
 * one for dk / dv, one for dq); no atomics, bitwise reproducible. Tolerance
 * of the 16-bit P and dS: see the library's tests.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o,
                 const void* dout, const float* lse, void* dq, void* dk, void* dv,
                 void* workspace, int B, int H, int N, int d, int causal, float scale,
                 fa_dtype dtype, void* stream);

/*
 * fa_bwd_workspace_size - bytes of the workspace fa_bwd needs for these sizes
 * (2 * B * H * ceil(N / 128) * 128 * 4). Host only; same size checks as fa_fwd.
 */
fa_status fa_bwd_workspace_size(int B, int H, int N, int d, size_t* bytes);

/*
 * fa_fwd_noalloc - fa_fwd for callers that cannot allocate device memory.
 * (A library convenience: the pages have no counterpart.)
 *
 * Some callers own all of the GPU's memory through their own allocator (for
 * example a serving process that carves HBM into a pool at start-up), or must
 * not call cudaMalloc / cudaFree at all once running (both can synchronise the
 * device). fa_fwd allocates a small status word on its first call on a
 * device; this entry point never allocates: it takes the same arguments and
 * always runs the one-CTA kernel (fa_fwd's results bit for bit, whichever
 * kernel fa_fwd picks), with its scratch (one status word per launch) in a
 * fixed 256-byte array inside this library that every device loading the
 * library holds until process exit. The scratch need does not grow with the
 * problem, so the size limits are fa_fwd's: larger sizes return
 * FA_ERR_UNSUPPORTED, bad arguments FA_ERR_INVALID_ARG, as fa_fwd.
 *
 * The first call on each device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress; make that first call
 * before any stream capture. Each call clears the status word on `stream`
 * before its launch (an asynchronous memset, not an allocation). All calls
 * share the one array, so calls that overlap on the GPU (different streams
 * without ordering between them) race on it. A launch whose bounded waits
 * gave up leaves O / LSE incomplete and sets that status word, which fa_check
 * reads and clears like fa_fwd's: since each call clears it first, fa_check
 * reports the most recent allocation-free launch on the device (with
 * overlapping calls, any one of them).
 */
fa_status fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, int causal, float scale,
                         fa_dtype dtype, void* stream);

/*
 * fa_fwd_host - fa_fwd on HOST buffers: copies Q, K, V in, runs the forward
 * and copies O and LSE out, the three overlapped across chunks of heads (the
 * method's only serial dependency runs along the keys of one query row, "TCA
 * 51%, MFU below 8%", section "Flash Attention 2 inflates TCA", so (b, h)
 * slices are independent).
 * Chunk c+1 is copied in while chunk c computes and chunk c-1 is copied out,
 * on three internal non-blocking streams of the device (created on the first
 * call, kept until process exit) that fork from and join back to `stream`.
 * The heads are cut into at most 9 chunks: n (at most 8) chunks that each
 * keep at least one wave of the forward's persistent grid busy, with the
 * first and last split to half that size so the exposed copy-in at the start
 * and forward plus copy-out at the end are short (one chunk for small
 * problems).
 *
 * q, k, v   : HOST pointers, contiguous [B][H][N][d] of `dtype`, read.
 * o, lse    : HOST pointers, contiguous [B][H][N][d] of `dtype` and
 *             [B][H][N] float32, written. Page-locked host memory
 *             (cudaHostAlloc / cudaHostRegister) lets the copies overlap;
 *             pageable memory gives the same results without the overlap.
 * workspace : DEVICE pointer, 16-byte aligned, of at least the size
 *             fa_fwd_host_workspace_size returns; caller-owned, not to be
 *             touched until `stream` has passed this call.
 * Everything else (arguments, numerics, status word) is as in fa_fwd. All
 * arguments are checked before anything is enqueued. Asynchronous: O and LSE
 * hold the result once `stream` reaches the point after this call (e.g.
 * after cudaStreamSynchronize(stream)); the host buffers must stay valid
 * until then.
 */
fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H, int N, int d, int causal, float scale, fa_dtype dtype,
                      void* workspace, size_t workspace_size, void* stream);

/*
 * fa_fwd_host_workspace_size - bytes of device workspace fa_fwd_host needs:
 * 4 B H N d 2-byte elements (Q, K, V, O) plus B H N float32 and 144 bytes of
 * alignment padding (16 for each of up to 9 chunks' LSE blocks). Host only.
 */
fa_status fa_fwd_host_workspace_size(int B, int H, int N, int d, size_t* bytes);

/*
 * fa_check - synchronise `stream`, then read and clear the current device's
 * status words (fa_fwd's, shared by every entry point but fa_fwd_noalloc, and
 * fa_fwd_noalloc's). Returns FA_OK, FA_ERR_TIMEOUT if a launch since the last
 * check stopped on a wait limit (for fa_fwd_noalloc: its most recent launch),
 * or FA_ERR_CUDA if the stream reports an error.
 */
fa_status fa_check(void* stream);

/*
 * fa_sm_clock_read - the SM clock the forward and backward kernels actually
 * ran at. Every CTA of a launch through fa_fwd, fa_fwd_strided, fa_fwd_fp8,
 * fa_fwd_host or fa_bwd adds its elapsed clock64 cycles and %globaltimer
 * nanoseconds to a record on the device; this call synchronises `stream`,
 * returns *sm_mhz = 1000 * cycles / ns over the launches since the previous
 * read (the CTAs' clock, weighted by their run time; 0 if none ran) and
 * *ctas = the number of CTAs recorded (ctas may be NULL), and clears the
 * record. Launches still running on other streams may be partly counted.
 * The pages measure a power-capped board whose SM clock falls below its
 * maximum ("TCA 51%, MFU below 8%", measurement section, clock64 readings):
 * a utilisation figure corrected for the clock divides by this, not by the
 * maximum clock. fa_fwd_noalloc launches are not recorded.
 */
fa_status fa_sm_clock_read(void* stream, double* sm_mhz, unsigned long long* ctas);

/*
 * fa_query_launch - launch shape fa_fwd would use on the current device for
 * these sizes: grid (persistent CTAs), threads per CTA, dynamic shared memory
 * bytes per CTA, the number of work units (256 query rows of one head, or 512
 * for the CTA-pair kernel) and the cluster size (1: one CTA per unit; 2: the
 * CTA-pair kernel, which fa_fwd runs for head dimension 128 without a causal
 * mask, or with one when N >= 16384, when there are at least as many 512-row
 * units as SM pairs; its results are the one-CTA kernel's bit for bit). Any output pointer may be NULL. Host
 * memory only; enqueues nothing.
 */
fa_status fa_query_launch(int B, int H, int N, int d, int causal, int* grid, int* threads,
                          int* smem_bytes, int* units, int* cluster);

/*
 * fa_sm_clock_probe - measure the SM clock: one CTA spins for `cycles`
 * clock64 ticks and writes out[0] = clock64 ticks elapsed and
 * out[1] = %globaltimer nanoseconds elapsed (MHz = 1000 * out[0] / out[1]).
 * out: device pointer to 2 uint64. Enqueued on `stream`.
 */
fa_status fa_sm_clock_probe(uint64_t* out, long long cycles, void* stream);

/* Human-readable name of a status code (static string). */
const char* fa_status_string(fa_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_SM103_H */
