/*
 * qgemv — fused dequantize-and-multiply for 4-bit block-quantized weights on
 * GB300 (sm_103a).  C ABI; all pointers are plain device (or, where stated,
 * host) addresses, all sizes are element counts, and every entry point
 * returns a status instead of aborting.
 *
 * The operation (reflex-llm "docs/kernels.md", K-quant GEMV and batched
 * K-quant GEMM sections; TandemLLM "Kernels", NVFP4 matrix products):
 *
 *     y[N x M] = x[N x K] . W^T,   y[n][m] = sum_k w[m][k] * x[n][k]
 *
 * where W[M][K] is stored block-quantized (GGML Q4_K, Q5_K, Q6_K super-blocks
 * of 256 weights, or NVFP4 W4A16: e2m1 codes, one e4m3 scale per 16 weights
 * and one fp32 per-tensor scale), x is fp16 and the accumulation is fp32.
 * The weights are decoded in registers and never written back.  y is stored
 * token-outer, y[n * M + m] (batched K-quant GEMM section).
 *
 * Row invariance (TandemLLM "Kernels", Row invariance and Verify twins):
 * the bits of y[n][:] depend only on x[n] and W, never on N or on the other
 * rows of x.  Every reduction order is fixed by (type, M, K); there are no
 * atomics.
 *
 * Layouts (little-endian; the pages give the sizes and fields, the bit
 * positions follow the GGML K-quant layout):
 *   Q4_K, 144 B / 256 weights: fp16 d, fp16 dmin, scales[12] (eight 6-bit
 *         scales and eight 6-bit mins), qs[128] (two nibbles per byte).
 *   Q5_K, 176 B: d, dmin, scales[12], qh[32] (fifth bits), qs[128].
 *   Q6_K, 210 B: ql[128], qh[64], int8 scales[16], fp16 d.
 *   NVFP4: codes uint8[M][K/2] (element 2i low nibble of byte i), e4m3
 *         scales uint8[M][K/16], fp32 global scale.
 *   FP8:  e4m3 codes uint8[M][K] (one per weight), bf16 scales
 *         [ceil(M/128)][K/128] row-major; w = e4m3 * scale[m/128][k/128].
 * A row of a K-quant matrix is K/256 consecutive blocks; rows are contiguous.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight formats.  12 (Q4_K) and 14 (Q6_K) are the GGML type ids used as
 * template arguments on reflex-llm "docs/performance.md", Path C; 13 follows
 * GGML's order; the NVFP4 id is this library's own. */
typedef enum {
    QG_Q4_K = 12,
    QG_Q5_K = 13,
    QG_Q6_K = 14,
    QG_NVFP4_W4A16 = 256,
    QG_FP8_E4M3 = 257  /* block-scaled e4m3, one bf16 scale per 128 x 128 block
                          (TandemLLM "Kernels", FP8 matrix products); id ours */
} qg_type;

typedef enum {
    QG_OK = 0,
    QG_EINVAL = -1,          /* bad argument (null pointer, size, mismatch) */
    QG_EUNSUPPORTED = -2,    /* valid request this library does not serve   */
    QG_EALIGN = -3,          /* pointer not aligned as required              */
    QG_ECUDA = -4,           /* a CUDA call failed; see qgemv_last_error()  */
    QG_ENOMEM = -5,          /* device allocation failed                     */
    QG_EFAULT_INJECTED = -6  /* failure forced by QGEMV_FAULT_INJECT         */
} qg_status;

/* Output element type of y. */
typedef enum { QG_OUT_F16 = 0, QG_OUT_F32 = 1 } qg_out;

/* Option flags. */
enum {
    QG_FLAG_FORCE_REFERENCE = 1u << 0, /* always use the simple reference kernel */
    QG_FLAG_DEBUG_SYNC = 1u << 1,      /* synchronize the stream after each call and
                                          report asynchronous errors              */
    QG_FLAG_NO_FALLBACK = 1u << 2,     /* return the fast path's launch error instead
                                          of retrying on the reference kernel      */
    QG_FLAG_MMA_SYNC_PREFILL = 1u << 3 /* Q4_K calls with N >= 33 (prefill chunks)
                                          run on the mma.sync kernels, whose rows
                                          keep the bits of N <= 32 calls, instead of
                                          the default tcgen05 / tensor-memory engine
                                          (128 rows x up to 64 tokens per MMA; within
                                          the tolerance, not bit-identical to N <= 32
                                          rows; measured 1.1-1.5x faster at N = 33,
                                          64 and 128 on the decode-layer shapes).   */
};

typedef struct {
    uint32_t flags;      /* QG_FLAG_* */
    int32_t max_tokens;  /* largest N staged at once (<= 0: 128).  Larger N is
                            processed in chunks of this many rows. */
} qg_opts;

typedef struct qg_handle qg_handle;

/* Create a handle for one weight matrix and fix its launch plan.
 * Defining passages: TandemLLM "Kernels", Row invariance (the tile table is
 * keyed by the weight's shape, never by the row count: here the K split and
 * rows per CTA are a function of (t, M, K) only) and NVFP4 matrix products (a
 * tile table per shape); reflex-llm "docs/kernels.md", K-quant GEMV (the
 * dispatcher selects the kernel by GGML tensor type).
 *   t            format
 *   M, K         rows (outputs) and columns (reduction length); M >= 1,
 *                K >= 256 and K % 256 == 0 for every format (NVFP4 too: the
 *                pages' 32-element granularity is not served; every workload
 *                here has K % 256 == 0); M up to 2^30 rows with
 *                ceil(M / 64) <= 65535, K up to 2^24
 *   w_dev        device pointer to the packed matrix (row-major rows of
 *                qgemv_row_bytes(t, K) bytes), 16-byte aligned.  (Inside a
 *                Q6_K matrix the 210-byte blocks are not aligned; they are
 *                staged through 16-byte aligned supersets and no byte outside
 *                the matrix is read.)
 *   scales_dev   NVFP4: e4m3 scales [M][K/16]; FP8: bf16 block scales
 *                [ceil(M/128)][K/128] (K up to 57,344); 16-byte aligned; else
 *                NULL
 *   global_scale NVFP4 only: per-tensor fp32 scale; ignored otherwise
 *   opts         nullable
 * Ownership: w_dev and scales_dev are borrowed and must outlive the handle and
 * stay unchanged while calls are in flight.  The handle owns its plan and a
 * small device staging buffer for x (max_tokens * K * 2.25 bytes per layout).
 * Errors: QG_EINVAL, QG_EALIGN, QG_EUNSUPPORTED, QG_ENOMEM, QG_ECUDA. */
qg_status qgemv_create(qg_handle **h, qg_type t, int64_t M, int64_t K,
                       const void *w_dev, const void *scales_dev, float global_scale,
                       const qg_opts *opts);

/* y = x . W^T (reflex-llm "docs/kernels.md", K-quant GEMV for N = 1 and the
 * batched K-quant GEMM section for N > 1, output token-outer; TandemLLM
 * "Kernels", NVFP4 matrix products).  N = 1..32 rows are row-invariant
 * (TandemLLM "Kernels", Verify twins); N >= 33 Q4_K calls run on the tcgen05
 * prefill engine unless QG_FLAG_MMA_SYNC_PREFILL (TandemLLM "Kernels",
 * Prefill kernels: prompt chunks have no twin contract).
 * x: fp16 [N][K] device, 16-byte aligned; y: [N][M] device of
 * type ydt (fp16 rounded to nearest-even, or fp32), 4-byte aligned.
 * N >= 1.  Work is enqueued on stream (a cudaStream_t; NULL = legacy default
 * stream); the call does not synchronize unless QG_FLAG_DEBUG_SYNC is set.
 * Calls on one handle must be ordered on one stream (they share the staging
 * buffer).  Errors: QG_EINVAL, QG_EALIGN, QG_ECUDA. */
qg_status qgemv_run(qg_handle *h, const void *x, int64_t N, void *y, qg_out ydt,
                    void *stream);

/* y = residual + x . W^T, added in fp32 before one rounding to fp16
 * (reflex-llm "docs/kernels.md", uint32-loads section: the residual-fused Wo
 * kernel gemv_quant_add; "docs/performance.md", Path C, PR #25).
 * residual, y: fp16 [N][M] device; y may equal residual (in place). */
qg_status qgemv_run_add(qg_handle *h, const void *x, int64_t N, const void *residual,
                        void *y, void *stream);

/* Two matrices with the same K sharing x (gate/up pair), one launch
 * (reflex-llm "docs/kernels.md", uint32-loads section: gemv_quant_pair, the
 * gate/up pair, ~44 % of decode).  ya is [N][Ma], yb is [N][Mb]; the handles'
 * checks and errors are those of qgemv_run, plus QG_EINVAL when K differs or
 * ya == yb.  Each matrix's rows have the bits of its own qgemv_run call. */
qg_status qgemv_pair_run(qg_handle *a, qg_handle *b, const void *x, int64_t N,
                         void *ya, void *yb, qg_out ydt, void *stream);

/* Three matrices with the same K sharing x (QKV triple); formats may differ
 * (e.g. Q4_K, Q4_K, Q6_K) (reflex-llm "docs/kernels.md", uint32-loads
 * section: gemv_quant_triple_uint32_q4k_q4k_q6k, the QKV triple of
 * Qwen3-4B).  One staging pass and one product launch where one kernel serves
 * the formats.  QG_EINVAL when the Ks differ or two outputs are equal. */
qg_status qgemv_triple_run(qg_handle *a, qg_handle *b, qg_handle *c, const void *x,
                           int64_t N, void *ya, void *yb, void *yc, qg_out ydt,
                           void *stream);

/* Fused gate/up pair with the SwiGLU epilogue: h = silu(x . Wg^T) * (x . Wu^T),
 * silu(v) = v / (1 + exp(-v)), written once to h without the two products
 * ever reaching memory (reflex-llm "docs/kernels.md", SwiGLU section:
 * output = silu(gate) x up, fusing avoids writing the intermediate;
 * "docs/performance.md", Path B PR #15: batched gate/up + SwiGLU).
 *   gate, up  handles of the same shape (M, K) and weight format
 *   x         fp16 [N][K] device, 16-byte aligned
 *   h         [N][M] device of type hdt (fp16 rounded to nearest-even, or
 *             fp32), 4-byte aligned
 * g and u are the fp32 values a plain qgemv_pair_run returns for the same x
 * (bit for bit); silu and the product are evaluated in fp32 (expf) and
 * rounded once to hdt.  Rows are row-invariant for every N (an elementwise
 * epilogue on row-invariant products).  Q4_K calls with N >= 33 stay on the
 * mma.sync kernels.  Errors: QG_EINVAL (null, shape mismatch, gate == up),
 * QG_EUNSUPPORTED (different formats), QG_EALIGN, QG_ECUDA. */
qg_status qgemv_pair_swiglu_run(qg_handle *gate, qg_handle *up, const void *x, int64_t N,
                                void *h, qg_out hdt, void *stream);

/* Host-buffer form of qgemv_run (the same operation as qgemv_run; the pages
 * time kernels with their inputs resident, TandemLLM "Kernels", How a kernel
 * gets in -- this entry times the whole round trip).
 * x_host (fp16 [N][K]) and y_host ([N][M] of
 * ydt) are host memory (pinned memory gives the fastest copies).  Copies x to
 * the device, runs, copies y back and synchronizes the stream before
 * returning.  The device buffers are owned by the handle and grow on demand. */
qg_status qgemv_run_host(qg_handle *h, const void *x_host, int64_t N, void *y_host,
                         qg_out ydt, void *stream);

/* Dequantize the whole matrix to fp32 w_out[M][K] (device, 4-byte aligned):
 * w = d * sc * q - dmin * m (Q4_K/Q5_K), d * sc * (q - 32) (Q6_K), e2m1 *
 * e4m3 * global scale (NVFP4), each rounded once to fp32 (reflex-llm
 * "docs/performance.md", Path E "What worked": the Q4_K weight formula;
 * TandemLLM "Kernels", NVFP4 matrix products).  It runs the product kernels'
 * own decoder functions on their thread mapping, with the product's rounding
 * steps for a one-hot x, so its output checks those decoders bit for bit;
 * with QG_FLAG_FORCE_REFERENCE it uses the simple per-element reference
 * decoder instead.  A test path, not a hot path (the product never writes
 * weights back: reflex-llm "docs/kernels.md", K-quant GEMV).
 * Errors: QG_EINVAL (null), QG_EALIGN, QG_ECUDA. */
qg_status qgemv_dequantize(qg_handle *h, float *w_out, void *stream);

/* Free the handle and the device buffers it owns (staging buffer, error word,
 * the host-entry buffers); the borrowed weights are not freed, as the pages'
 * kernels read weights where the caller keeps them (reflex-llm
 * "docs/kernels.md", K-quant GEMV: weights stay in the caller's mapping).
 * NULL is a no-op.  No call on h may be in flight. */
void qgemv_destroy(qg_handle *h);

/* Message of the last error on the calling thread ("" if none); also the
 * note left when a fast-path launch failure fell back to the reference
 * kernel (reflex-llm "docs/kernels.md", uint32-loads section: any cudaError
 * falls through to the typed byte-load kernel). */
const char *qgemv_last_error(void);

/* Bytes per row of the packed matrix (codes only for NVFP4); -1 if K is not
 * supported for the format.  Pure host function.  Block sizes: Q4_K 144 and
 * Q6_K 210 bytes (reflex-llm "docs/kernels.md", uint32-loads section), Q5_K
 * 176, NVFP4 K/2 code bytes (TandemLLM "Kernels", NVFP4 matrix products). */
int64_t qgemv_row_bytes(qg_type t, int64_t K);

/* Read (and with clear != 0, reset) the handle's device error word; with
 * h == NULL, the error word of qgemv_run_noalloc on the current device.  The
 * kernels never trap: a bounded wait that runs out (a pipeline that stopped
 * making progress) sets bit 1 (consumer side) or bit 2 (producer side) and
 * the kernel returns with undefined results (reflex-llm "docs/kernels.md",
 * uint32-loads section: a fault must never crash generation;
 * "docs/performance.md", Path C #29: a faulting kernel leaves the context
 * sticky).  Synchronous (a device-to-host copy of 4 bytes).  *flags_out == 0
 * means no kernel reported a problem.  Errors: QG_ECUDA. */
qg_status qgemv_device_status(qg_handle *h, uint32_t *flags_out, int clear);

/* Launch plan of a handle, for tests and profiling: number of K-split ranks
 * (a cluster of CTAs per row tile, combined in rank order: TandemLLM
 * "Kernels", Row invariance, partial sums added in a fixed order), rows per
 * CTA for the given N, and how many kernels one qgemv_run launches.  Pure
 * host.  Errors: QG_EINVAL (null h, N < 1). */
qg_status qgemv_plan_info(const qg_handle *h, int64_t N, int32_t *ksplit,
                          int32_t *rows_per_cta, int32_t *launches);

/* Allocation-free form of qgemv_run, for callers that may not allocate device
 * memory while they run (for example a serving runtime that hands all device
 * memory to its own pool at start-up, so any cudaMalloc behind its back can
 * fail or fragment that pool, or a library that must keep its host process's
 * device footprint fixed).  The pages have no counterpart: this is a
 * library-usage variant of the staging + product path.  It needs no handle:
 * the weights are described by the same arguments as qgemv_create (t, M, K,
 * w_dev, scales_dev, global_scale; checked the same way), x and y as in
 * qgemv_run; every argument is checked before the device is touched.
 * Scratch: one 2 MiB array in the library's device memory (held by every GPU
 * that loads the library until exit) holds the staged x and the kernels'
 * error word; N is processed in chunks of min(32, about 2 MiB / (K/256 * 576))
 * tokens and K above 931,840 is rejected with QG_EUNSUPPORTED.  It never calls
 * cudaMalloc or cudaFree.  All calls on a device share the array and it keeps
 * the last call's contents; every staged byte a call reads it has written
 * first, and the error word starts at zero, so nothing needs clearing, but
 * calls that overlap on the GPU (unordered streams) race and must be ordered.
 * The error word is read (and cleared) with qgemv_device_status(NULL, ..).
 * The first call on a device looks up the array's address
 * (cudaGetSymbolAddress) with that device current; make it before any stream
 * capture.  Results equal qgemv_run's bit for bit for N <= 32, and for every
 * N those of a handle created with QG_FLAG_MMA_SYNC_PREFILL (Q4_K calls with
 * N >= 33 under default flags run on the tcgen05 engine and agree only within
 * the tolerance).  Errors: QG_EINVAL, QG_EALIGN, QG_EUNSUPPORTED, QG_ECUDA. */
qg_status qgemv_run_noalloc(qg_type t, int64_t M, int64_t K, const void *w_dev,
                            const void *scales_dev, float global_scale, const void *x,
                            int64_t N, void *y, qg_out ydt, void *stream);

/* ------------------------------------------------------------------------
 * Decode chains: the calls of a transformer layer (QKV triple, Wo + residual,
 * gate/up pair, down) in one persistent launch that stays resident on the
 * SMs, so the weight stream does not drain and refill at every call boundary
 * (reflex-llm "docs/performance.md", Level 4: persistent kernels that stay
 * resident on the SM; Path C: the per-call launch and tail costs of small
 * matrices).
 * ------------------------------------------------------------------------ */

/* Kinds of chain calls; each is the operation of the named entry point. */
typedef enum {
    QG_CALL_RUN = 0,     /* y[0] = x . W0^T                     (qgemv_run)        */
    QG_CALL_RUN_ADD = 1, /* y[0] = residual + x . W0^T, fp16    (qgemv_run_add)    */
    QG_CALL_PAIR = 2,    /* y[i] = x . Wi^T, i < 2              (qgemv_pair_run)   */
    QG_CALL_TRIPLE = 3   /* y[i] = x . Wi^T, i < 3              (qgemv_triple_run) */
} qg_call_kind;

/* One call of a chain; the arguments have the meaning, layout and checks of
 * the named entry point. */
typedef struct qg_call {
    int32_t kind;          /* qg_call_kind */
    int32_t out_dtype;     /* qg_out of y (QG_CALL_RUN_ADD: must be QG_OUT_F16) */
    int64_t N;             /* tokens */
    qg_handle *h[3];       /* 1, 1, 2 or 3 handles by kind (equal K); the rest ignored */
    const void *x;         /* fp16 [N][K] device, 16-byte aligned */
    const void *residual;  /* QG_CALL_RUN_ADD: fp16 [N][M] device (may equal y[0]) */
    void *y[3];            /* outputs, device, one per handle */
} qg_call;

typedef struct qg_chain qg_chain;

/* qgemv_chain_create flags. */
enum {
    QG_CHAIN_PERSISTENT = 1u << 0  /* run eligible calls in one persistent launch
                                      (default: one launch per call, each
                                      chained to the previous one by
                                      programmatic dependent launch) */
};

/* Create a chain on the current device: the state of the persistent launch
 * (reflex-llm "docs/performance.md", Level 4): a pair of device counters and
 * an error word (16 bytes of device memory, zeroed).  flags: QG_CHAIN_*.
 * Errors: QG_EINVAL (null out, unknown flag), QG_ENOMEM, QG_ECUDA. */
qg_status qgemv_chain_create(qg_chain **out, uint32_t flags);

/* Run calls[0 .. ncalls-1] in order on `stream` (reflex-llm
 * "docs/performance.md", Level 4 persistent kernels; the calls are those of
 * "docs/kernels.md", uint32-loads section).  Results: those of issuing
 * the same calls one by one through their entry points on the same stream,
 * bit for bit; in particular call c reads its x and residual only after
 * calls 0 .. c-1 have written all their outputs, so a call may consume an
 * earlier call's output.  By default each call runs through its entry point
 * (one launch per call, chained by programmatic dependent launch: measured
 * the faster form on GB300).  With QG_CHAIN_PERSISTENT, up to four
 * consecutive calls run in one persistent launch when each has N <= 8, x of
 * at most 48 KB (N * K/256 * 576 bytes), Q4_K or Q6_K handles on the chain's
 * device and no QG_FLAG_FORCE_REFERENCE / QG_FLAG_DEBUG_SYNC; the other calls
 * run through their entry points, in order.  The persistent form puts one CTA
 * on every SM and its CTAs wait for one another: kernels of other streams that
 * hold SMs meanwhile can delay some CTAs past the waits' limit (reported by
 * qgemv_chain_status, bit 4).  Every call is checked (as its entry point
 * checks it) before anything is launched.  Launches of one chain must be
 * ordered (one stream, or streams ordered by events): they share its
 * counters.  The call does not synchronize.  Errors: QG_EINVAL (null c or
 * calls, ncalls < 1, bad kind, a call's own argument errors), QG_EALIGN,
 * QG_EUNSUPPORTED, QG_ECUDA. */
qg_status qgemv_chain_run(qg_chain *c, const qg_call *calls, int32_t ncalls, void *stream);

/* One decode step with its inputs and outputs in host memory (the pages
 * time kernels with their inputs resident, TandemLLM "Kernels", How a kernel
 * gets in -- this entry times the whole round trip): copies in_bytes from
 * in_host to in_dev, runs calls[0 .. ncalls-1] as qgemv_chain_run does (their
 * x, residuals and outputs are device buffers, typically inside in_dev and
 * out_dev), copies out_bytes from out_dev to out_host and synchronizes the
 * stream.  When a host buffer is page-locked and mapped (cudaHostAlloc, or
 * registered as mapped), the copy is whole 16-byte units and every address is
 * 16-byte aligned, the SMs copy it through the mapped buffer (a small kernel
 * chained to the calls); otherwise the copy engine does.  Errors: those of
 * qgemv_chain_run, QG_EINVAL (null buffer with a nonzero size), QG_ECUDA. */
qg_status qgemv_chain_run_host(qg_chain *c, const qg_call *calls, int32_t ncalls,
                               const void *in_host, void *in_dev, size_t in_bytes,
                               const void *out_dev, void *out_host, size_t out_bytes,
                               void *stream);

/* Read (and with clear != 0, reset) the chain's device error word: bits 1
 * and 2 as for qgemv_device_status, bit 4: a wait for the earlier calls'
 * outputs ran out (results undefined); the kernel never traps (reflex-llm
 * "docs/kernels.md", uint32-loads section: a fault must never crash
 * generation).  Synchronous.  Errors: QG_EINVAL (null c), QG_ECUDA. */
qg_status qgemv_chain_status(qg_chain *c, uint32_t *flags_out, int clear);

/* Free the chain's state (NULL is a no-op); the pages have no counterpart
 * (library housekeeping).  No launch of it may be in flight. */
void qgemv_chain_destroy(qg_chain *c);

/* Human-readable description of the options in effect (flags, environment
 * overrides QGEMV_FORCE_REFERENCE, QGEMV_DEBUG_SYNC, QGEMV_FAULT_INJECT)
 * (TandemLLM "Kernels", Knobs: every switch and the values in effect can be
 * printed).  Never fails; the string is owned by the library. */
const char *qgemv_describe(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
