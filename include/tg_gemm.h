/*
 * tg_gemm — fp16 tiled tensor-core GEMM with an optional fused bias + GELU
 * epilogue, for one GB300 (sm_103a) GPU. C ABI.
 *
 * The operation (the problem statement of "TileLang: writing LLM GPU kernels by
 * thinking in tiles", sections 2 and 3, with the epilogue of "Designing
 * high-performance GPU kernels with TileLang ...", section 3 "Epilogue Fusion
 * and Memory Efficiency"):
 *
 *     C[i,j] = epi( sum_k A[i,k] * B[k,j] + bias[j] )
 *
 *   A      M x K, IEEE binary16, row-major (leading dimension K)
 *   B      K x N, IEEE binary16, row-major (leading dimension N)
 *   bias   N binary16 values, added to column j of every row; NULL means no bias
 *   C      M x N, IEEE binary16, row-major (leading dimension N)
 *   epi    identity (TG_EPI_NONE) or GELU(x) = 0.5 x (1 + erf(x / sqrt 2))
 *          (TG_EPI_GELU, the exact-erf form)
 *
 * Products are accumulated in fp32 by the tensor core; bias and GELU are
 * applied in fp32 to the unrounded sum while the tile is still on chip; the
 * result is rounded once to binary16 (to nearest, ties to even; overflow gives
 * +-inf). GELU's erf is evaluated in fp32 to within 1.5e-7 (Abramowitz &
 * Stegun 7.1.26, in the form x (1 - erfc/2), x erfc/2 without cancellation):
 * on every finite binary16 input the rounded GELU is within one ulp of the
 * correctly rounded value. The order of the fp32 accumulation is not specified: results agree
 * with an exact computation to within fp32 accumulation error plus one final
 * binary16 rounding, and are bit-identical from run to run on the same GPU.
 *
 * Pointers and ownership. Unless a function says otherwise, A, B, bias and C
 * are DEVICE pointers on the current CUDA device, owned by the caller; the
 * library never frees or keeps them past the call. C must not overlap A, B or
 * bias (checked). Any alignment is accepted; 16-byte-aligned base pointers with
 * K and N multiples of 8 take the fast (TMA) path, anything else a slower path
 * with ordinary loads.
 *
 * Streams. `stream` is a cudaStream_t (NULL = the legacy default stream). Each
 * call only enqueues work and returns without synchronising. Calls are
 * stream-ordered; the library keeps a separate scratch buffer per stream, so
 * concurrent calls on different streams are safe.
 *
 * Errors. Every function returns a tg_status; TG_OK is 0. Argument errors are
 * detected on the host before anything is enqueued. tg_last_error() gives a
 * human-readable message for the last failure on the calling thread.
 */
#ifndef TG_GEMM_H
#define TG_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Binary-compatible with cudaStream_t / CUstream. */
typedef struct CUstream_st* tg_stream_t;

typedef enum {
    TG_EPI_NONE = 0, /* C = A@B (+ bias) */
    TG_EPI_GELU = 1  /* C = GELU(A@B (+ bias)), exact erf */
} tg_epilogue;

typedef enum {
    TG_OK = 0,
    TG_ERR_INVALID_ARG = 1,        /* bad pointer, size, epilogue, kernel choice or overlap */
    TG_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not compute capability 10.3 */
    TG_ERR_CUDA = 3,               /* a CUDA runtime/driver call or a launch failed */
    TG_ERR_TIMEOUT = 4,            /* a kernel's bounded wait expired (see tg_device_status) */
    TG_ERR_NO_MEMORY = 5,          /* the library could not allocate its scratch buffer */
    TG_ERR_BOUNDS = 6              /* a device-side bounds check failed (debug builds only,
                                      see tg_debug_build) */
} tg_status;

/* Kernel selection for tg_gemm_ex (tg_gemm always uses TG_KERNEL_AUTO). */
typedef enum {
    TG_KERNEL_AUTO = 0,      /* choose by shape and alignment (below) */
    TG_KERNEL_TILED_TMA = 1, /* persistent 128x256 tiles, TMA loads, tcgen05 MMA into TMEM;
                                K split over slices when the tiles leave SMs idle.
                                Needs K % 8 == 0, N % 8 == 0, A and B 16-byte aligned. */
    TG_KERNEL_TILED_LSU = 2, /* the same tiles with operands staged by ordinary loads;
                                any shape and alignment */
    TG_KERNEL_SPLITK = 3,    /* skinny M <= 128: computes C^T = B^T A^T so N fills the
                                128-row MMA, with K split across CTAs; same TMA needs
                                as TG_KERNEL_TILED_TMA */
    TG_KERNEL_TILED_PAIR = 4 /* 256x256 tiles on pairs of SMs (two-CTA clusters sharing
                                one tensor-core MMA); same TMA needs as
                                TG_KERNEL_TILED_TMA */
} tg_kernel;

/*
 * C = epi(A @ B + bias) on `stream`.
 *
 * M, N, K >= 0 and each < 2^31. M == 0 or N == 0: nothing is done. K == 0: the
 * empty sum is 0, so C = epi(bias) (or epi(0) without bias). `epilogue` is a
 * tg_epilogue value. A, B may be NULL only when the product is empty.
 *
 * Kernel choice (TMA-compatible means K % 8 == 0, N % 8 == 0 and 16-byte
 * aligned A and B): not TMA-compatible and (M <= 128 or 2 M N K < 2^32) ->
 * TG_KERNEL_TILED_LSU; not TMA-compatible, M > 128 and 2 M N K >= 2^32 ->
 * each operand TMA cannot describe is first
 * copied (on `stream`) into a library-owned buffer with its row stride rounded
 * up to 8 elements (one buffer per stream, grown as needed, freed by
 * tg_shutdown; TG_ERR_NO_MEMORY if it cannot be allocated), then the TMA
 * kernels below run on the copy; M <= 16, or M <= 128 where the skinny kernel
 * measured faster -> TG_KERNEL_SPLITK; other M <= 128 -> TG_KERNEL_TILED_TMA.
 * "Measured faster" means M <= 64 when K >= 2048; for shorter K, fewer
 * 64-column tiles than SMs with (K / 64) * SMs / tiles >= 1.5 M, or M <= 64
 * with 2 K N >= 256 MiB of B.
 * M > 128: when the 128 x 256 tiles fill at least a wave of SMs and the
 * 256x256 pair tiles fewer than eight waves of SM pairs, the kernel a time
 * model of their waves (with the last wave's cost: pairs' half-width units,
 * or the single-CTA kernel's split tail) predicts faster; with more pair
 * tiles TG_KERNEL_TILED_PAIR; below a wave, at least one 256x256 tile per
 * pair of SMs, or with K >= 8192 at least 0.3 of one -> TG_KERNEL_TILED_PAIR;
 * else TG_KERNEL_TILED_TMA.
 * TG_KERNEL_TILED_TMA (and TG_KERNEL_TILED_LSU) split K when their tiles leave
 * SMs idle and a cost model of the slices and their summation predicts a gain
 * (see tg_gemm_ex). When TG_KERNEL_TILED_TMA's tiles fill whole waves plus a
 * short last one, with split_k 0 the last wave's tiles may run K-split in a
 * second launch (clusters summing on chip) after the whole waves.
 */
tg_status tg_gemm(const void* A, const void* B, const void* bias, void* C,
                  int64_t M, int64_t N, int64_t K, int epilogue, tg_stream_t stream);

/*
 * The choice tg_gemm makes for these operands, without running anything:
 * *kernel receives the tg_kernel value it runs, *split_k the number of K slices
 * that kernel takes (1 = K is not split; always 1 for TG_KERNEL_TILED_PAIR; for
 * TG_KERNEL_TILED_TMA with whole waves of tiles and a split last wave, that
 * wave's slices),
 * and *aligned_copy (may be NULL) 1 when A or B is first copied to an aligned
 * row stride. A and B are only tested for 16-byte alignment, never read; the
 * answer is for the current device. For K == 0 tg_gemm runs only its
 * epilogue pass, and for M or N == 0 nothing, whatever is reported.
 * TG_ERR_INVALID_ARG for sizes outside [0, 2^31) or a NULL kernel / split_k.
 */
tg_status tg_gemm_plan(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                       int* kernel, int* split_k, int* aligned_copy);

/*
 * tg_gemm with an explicit kernel (a tg_kernel value) and an explicit number
 * of K slices `split_k` (0 = automatic, otherwise 1..64; more slices than
 * ceil(K / 64) K blocks are reduced to one per K block). split_k applies to
 * TG_KERNEL_SPLITK and to the single-CTA tiled kernels (TG_KERNEL_TILED_TMA,
 * TG_KERNEL_TILED_LSU); with TG_KERNEL_TILED_PAIR it is TG_ERR_INVALID_ARG, and
 * with TG_KERNEL_AUTO it is used only when the choice is TG_KERNEL_SPLITK.
 * The tiled kernels' automatic count splits only problems whose 128 x 256
 * tiles number fewer than the SMs. With TG_KERNEL_TILED_TMA and 2..8 slices
 * whose clusters (one per tile, one CTA per slice) all fit on the device at
 * once, the slices are summed on chip through distributed shared memory.
 * Otherwise each slice's fp32 partial tile goes to the stream's scratch
 * (splits * N * M rounded up to 16, fp32; allocated as for TG_KERNEL_SPLITK)
 * and a second kernel on `stream` sums the slices (this form needs
 * M <= 1048560). TG_KERNEL_SPLITK sums its slices the same two ways (on chip
 * for 2..8 slices whose clusters, one per 256-column unit, all fit at once).
 * Both ways add the slices in order, so they give the same bits, and the
 * epilogue follows the full sum. A kernel whose requirements the
 * arguments do not meet is TG_ERR_INVALID_ARG. Results of all kernels agree
 * within the accumulation-order tolerance stated above; on inputs whose
 * products and partial sums are exact in fp32 they are bit-identical.
 */
tg_status tg_gemm_ex(const void* A, const void* B, const void* bias, void* C,
                     int64_t M, int64_t N, int64_t K, int epilogue, int kernel, int split_k,
                     tg_stream_t stream);

/*
 * End-to-end form with HOST operands: copies hA, hB, hbias (host, preferably
 * pinned) into the caller's device buffers dA, dB, dbias, runs tg_gemm on
 * them, and copies the result dC back into host hC, all enqueued on `stream`
 * (returns without synchronising; hC is valid after the stream completes).
 * hbias and dbias are both NULL or both non-NULL. Device buffers must hold
 * M*K, K*N, N and M*N binary16 values; they are owned by the caller.
 */
tg_status tg_gemm_staged(const void* hA, const void* hB, const void* hbias, void* hC,
                         void* dA, void* dB, void* dbias, void* dC,
                         int64_t M, int64_t N, int64_t K, int epilogue, tg_stream_t stream);

/*
 * The epilogue alone, in place: C[i,j] = epi(C[i,j] + bias[j]) on an M x N
 * row-major binary16 DEVICE matrix (bias NULL = no bias; epilogue a
 * tg_epilogue value), computed in fp32 and rounded once more to binary16.
 * This is the unfused comparator for the fused epilogue described in
 * "Designing high-performance GPU kernels with TileLang ...", section 3
 * ("Epilogue Fusion and Memory Efficiency"): tg_gemm with TG_EPI_NONE and no
 * bias, then this pass, computes the same function with the product rounded
 * to binary16 in between and two extra HBM passes over C. Any alignment;
 * stream-ordered; allocates nothing.
 */
tg_status tg_bias_gelu(void* C, const void* bias, int64_t M, int64_t N, int epilogue, tg_stream_t stream);

/* Size of the fixed scratch array behind tg_gemm_splitk_noalloc (8 MiB). */
#define TG_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * The skinny split-K GEMM (TG_KERNEL_SPLITK) for callers that must not have the
 * library allocate device memory during a call. Examples: a process that hands
 * nearly all device memory to its own pool allocator at start-up, where a
 * cudaMalloc from inside a library fails or fragments that pool; and a
 * latency-bound serving loop, where cudaMalloc/cudaFree would synchronise the
 * device and stall unrelated streams. The TileLang pages have no counterpart
 * to this entry point: it changes only where the scratch memory comes from,
 * not what is computed.
 *
 * Same arguments and result as tg_gemm_ex(..., TG_KERNEL_SPLITK, split_k, ...):
 * M <= 128, K % 8 == 0, N % 8 == 0, A and B 16-byte aligned; split_k 0 picks
 * the number of K slices automatically, never more than fit in the fixed
 * array (one slice needs none, so an automatic call is never refused for
 * size), 1..64 fixes it. The caller still
 * passes A, B, bias and C (device pointers it owns). With 2..8 K slices whose
 * clusters (one per 256-column unit, one CTA per slice) all fit on the device
 * at once, the slices are summed on chip and no scratch is used, as in
 * tg_gemm_ex. Otherwise, with more than one slice, the partial sums live in
 * one fixed array of TG_NOALLOC_SCRATCH_BYTES compiled into the library's
 * device image: every device that loads the library holds it until the
 * process exits. A call whose partials go through the array and need more
 * (4 * slices * N * Mp bytes, Mp = M rounded up to a multiple of 16, plus a
 * reserved head of 4 bytes per 256-column slice of N, rounded up to 256)
 * returns TG_ERR_INVALID_ARG and enqueues nothing. Nothing is allocated or
 * freed by any call.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture begins. Every call that uses the array writes the
 * partials before a second kernel on `stream` sums them, so nothing carries
 * over between calls. All calls share the one array, so calls whose work can
 * overlap on the GPU (for example on two streams without ordering between
 * them) race and give wrong results; order them on one stream or with events.
 */
tg_status tg_gemm_splitk_noalloc(const void* A, const void* B, const void* bias, void* C,
                                 int64_t M, int64_t N, int64_t K, int epilogue, int split_k,
                                 tg_stream_t stream);

/*
 * Weight-only 4-bit GEMM (decode shapes): C = epi(A @ W + bias) with W
 * dequantized on chip, never written to memory. The form of the operation is
 * that of "TileLang: writing LLM GPU kernels by thinking in tiles", section
 * "Quantized LLM inference" (packed weights converted in a tile that feeds
 * the tensor-core product); the pages fix no storage format, this is the
 * library's:
 *
 *   A       M x K binary16, row-major, DEVICE, 16-byte aligned
 *   Bq      N rows of K/2 bytes, DEVICE, 16-byte aligned: byte j of row n
 *           holds q[2j][n] in bits 0-3 and q[2j+1][n] in bits 4-7, each a
 *           two's-complement integer in [-8, 7] (the weight of a linear layer,
 *           out x in, two values per byte along the input dimension)
 *   scales  K/128 rows of N binary16 values, DEVICE, 16-byte aligned; q[k][n]
 *           uses scales[k/128][n]
 *   W       W[k][n] = q[k][n] * scales[k/128][n], rounded once to binary16
 *   bias, C, epilogue, stream: as for tg_gemm.
 *
 * Needs M <= 128, K % 128 == 0 and N % 8 == 0 (TG_ERR_INVALID_ARG
 * otherwise); M > 64 runs as row blocks of 64, each reading the weights once.
 * M == 0 or N == 0 does nothing; K == 0 gives C = epi(bias).
 * split_k: 0 = automatic, else the number of K slices (1..64, at most
 * ceil(K / 256)); with more than one slice the library's per-stream scratch
 * holds fp32 partial sums, reduced in slice order (deterministic). The
 * tolerance is tg_gemm's, with W in place of B.
 */
tg_status tg_gemm_w4(const void* A, const void* Bq, const void* scales, const void* bias, void* C,
                     int64_t M, int64_t N, int64_t K, int epilogue, int split_k, tg_stream_t stream);

/* Weight formats of the 4-bit GEMM. */
typedef enum {
    TG_W4_INT4 = 0,     /* two's-complement integers in [-8, 7] */
    TG_W4_FP4_E2M1 = 1  /* FP4 E2M1: bit 3 sign, bits 2-1 exponent (bias 1), bit 0 mantissa;
                           values +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}, no infinities or NaN */
} tg_w4_format;

/*
 * tg_gemm_w4 with the format of the 4-bit fields given: the same section
 * ("Quantized LLM inference") names INT4 and FP4 weights. `weight_format` is a
 * tg_w4_format value; storage, scales, W[k][n] = value(q[k][n]) *
 * scales[k/128][n] rounded once to binary16, sizes, splits, errors and
 * tolerance are those of tg_gemm_w4 (which is this call with TG_W4_INT4).
 * An unknown format is TG_ERR_INVALID_ARG.
 */
tg_status tg_gemm_w4_ex(const void* A, const void* Bq, const void* scales, const void* bias, void* C,
                        int64_t M, int64_t N, int64_t K, int epilogue, int weight_format, int split_k,
                        tg_stream_t stream);

/* Kernels of the 4-bit GEMM (tg_gemm_w4_kernel). */
typedef enum {
    TG_W4_KERNEL_AUTO = 0, /* TG_W4_KERNEL_REG when M <= 16, split_k is 0 or 1 and N has at
                              least one 64-column block per SM; otherwise TG_W4_KERNEL_TMEM */
    TG_W4_KERNEL_TMEM = 1, /* weights converted into shared memory, tcgen05 MMAs into tensor
                              memory (64-row MMAs: M > 64 runs as row blocks); split K */
    TG_W4_KERNEL_REG = 2   /* weights converted in registers into the operands of warp-level
                              m16n8k16 MMAs (16 weight columns x 8 tokens each, two per 16
                              tokens); M <= 16; one CTA per 64 output columns over the whole
                              K (no K slices) */
} tg_w4_kernel;

/*
 * tg_gemm_w4_ex with the kernel chosen by the caller (`kernel`, a tg_w4_kernel
 * value): the same product, storage, sizes, errors and tolerance. Both
 * kernels round W to binary16 once per weight and accumulate in fp32; on
 * integer-valued inputs with power-of-two scales their results are identical.
 * TG_W4_KERNEL_REG with M > 16 or split_k > 1, or an unknown kernel, is
 * TG_ERR_INVALID_ARG. tg_gemm_w4_ex is this call with TG_W4_KERNEL_AUTO.
 */
tg_status tg_gemm_w4_kernel(const void* A, const void* Bq, const void* scales, const void* bias, void* C,
                            int64_t M, int64_t N, int64_t K, int epilogue, int weight_format, int kernel,
                            int split_k, tg_stream_t stream);

/*
 * Attention forward (FlashAttention), the fused attention kernel of
 * "TileLang: writing LLM GPU kernels by thinking in tiles", section 5, with
 * the causal option of "Designing high-performance GPU kernels with TileLang
 * ...", section 5:
 *
 *     S = Q K^T / sqrt(D),  P = softmax(S) along each query row,  O = P V
 *
 *   Q, K, V, O  B x S x H x D binary16, row-major in that order (batch,
 *               sequence, head, dim: the bshd layout), DEVICE, 16-byte aligned
 *   causal      0: every query sees every key; 1: query position i sees key
 *               positions 0..i
 *
 * D must be 128 (TG_ERR_INVALID_ARG otherwise). B, S or H == 0 does nothing.
 * Scores, the softmax and the accumulation are fp32 (the exponentials in base
 * 2 with log2(e) folded into the scale; P is rounded to binary16 for the P V
 * product); O is rounded once to binary16. Results agree with the exact
 * definition within |O - ref| <= 1e-2 + 1e-2 |ref| per element, and are
 * bit-identical from run to run. O must not overlap Q, K or V.
 * Stream-ordered. Without the causal mask, when the last round of 128-query
 * blocks would leave at least half of the GPU idle, those blocks are computed
 * in two key halves whose partial results are merged; their fp32 partials use
 * the library's per-stream scratch buffer (allocated on first need, grown as
 * needed, freed by tg_shutdown; TG_ERR_NO_MEMORY if it cannot be allocated).
 */
tg_status tg_attention_fwd(const void* Q, const void* K, const void* V, void* O, int64_t B, int64_t S,
                           int64_t H, int64_t D, int causal, tg_stream_t stream);

/*
 * Row softmax, the reduction kernel of "Designing high-performance GPU kernels
 * with TileLang ...", section 4: for every row i of the M x N row-major
 * binary16 DEVICE matrix X,
 *
 *     Y[i,j] = exp(X[i,j] - max_j X[i,:]) / sum_j exp(X[i,j] - max_j X[i,:])
 *
 * computed in fp32 (the exponentials in base 2) and rounded once to binary16.
 * Entries of -inf give 0; a row that is entirely -inf gives NaN. Y may be X
 * itself (in place) but must not otherwise overlap it. Any alignment; rows
 * that start 16-byte aligned with N <= 32768 and N % 8 == 0 take the
 * register-resident path (one HBM read and one write per element).
 * Stream-ordered; allocates nothing.
 */
tg_status tg_softmax_rows(const void* X, void* Y, int64_t M, int64_t N, tg_stream_t stream);

/*
 * Synchronises `stream`, then reports (and clears) the device-side status word
 * that kernels set when one of their bounded waits expires: TG_OK or
 * TG_ERR_TIMEOUT (or, in debug builds, TG_ERR_BOUNDS for a failed bounds check). `*where` (if not NULL) receives the code of the wait that
 * expired first (0 if none). Every wait inside the kernels gives up after the
 * watchdog limit (tg_set_watchdog_ns) instead of spinning forever; the kernel
 * then drains its in-flight copies, frees its tensor memory and exits, leaving
 * C unspecified.
 */
tg_status tg_device_status(tg_stream_t stream, int* where);

/* tg_device_status(stream, NULL): the same synchronising check, for callers
 * that need only the status. */
tg_status tg_debug_status(tg_stream_t stream);

/* Watchdog limit for every bounded wait, in ns (default 2e9; 0 restores it). */
tg_status tg_set_watchdog_ns(uint64_t ns);

/*
 * Test hook for the watchdog: while `on` is non-zero, the TMA producers of the
 * tiled kernels (TG_KERNEL_TILED_TMA, TG_KERNEL_TILED_PAIR) and of the 4-bit
 * register kernel (TG_W4_KERNEL_REG) skip the first pipeline stage of every
 * CTA (every CTA pair for the pair kernel), so the consumers' bounded waits
 * expire and the call ends with TG_ERR_TIMEOUT from tg_device_status. Off by
 * default; has no effect on other kernels.
 */
tg_status tg_debug_skip_first_arrive(int on);

/*
 * 1 if this library was compiled with TG_DEBUG=1, else 0. Debug builds check,
 * on the device, that every scratch-buffer, arrival-counter and TMA-store
 * coordinate a kernel computes lies inside its buffer (and, for stores, on a
 * 16-byte boundary and not negative); a failed check is recorded in the status
 * word that tg_device_status reads (TG_ERR_BOUNDS) and the access is skipped,
 * so nothing faults. In normal builds the checks are compiled away.
 */
int tg_debug_build(void);

/*
 * Test hook for the bounds checks of debug builds: while `floats` > 0, kernels
 * are told that their scratch holds at most that many floats (the buffer itself
 * is unchanged), so a check fails as soon as a kernel's partial sums reach
 * beyond it. 0 restores the real sizes. No effect in normal builds.
 */
tg_status tg_debug_bounds_limit(int64_t floats);

/* Static description of a status code. */
const char* tg_status_string(int status);

/* Message for the last failure on the calling thread ("" if none). */
const char* tg_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int tg_version(void);

/*
 * Shared memory (bytes per CTA) that a kernel configuration uses for its
 * operand ring: stages * (BM*BK + BK*BN) * 2. Returns -1 for an unknown kernel.
 * For TG_KERNEL_SPLITK the M-side tile is the padded M of a 16-row problem.
 */
int64_t tg_ring_bytes(int kernel);

/*
 * Frees the library's per-device scratch buffers and forgets its per-device
 * caches (tensor maps, device addresses of its own arrays, kernel attributes).
 * Call with no work in flight. After a cudaDeviceReset, call tg_shutdown before
 * the next library call: the caches would otherwise refer to the old context.
 */
void tg_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* TG_GEMM_H */
