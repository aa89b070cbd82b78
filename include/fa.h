/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention forward library, libfa_gb300.so.
 *
 * The operation is the attention forward pass that the tile-programming guide
 * ("Guia Prático de Programação de GPU com Tiles", section 6, flash attention) builds
 * toward, with the FlashAttention-4 features named in "Como Domar o Blackwell Sem
 * Enlouquecer com CUDA" (two MMA stages, online softmax, grouped-query attention):
 *
 *   for every batch b, query head h and query row i:
 *     kvh       = h / (Hq / Hkv)                      (consecutive query heads share a KV head)
 *     J         = { j < Sk : causal == 0,  or j <= i (causal == 1, top-left),
 *                   or j <= i + Sk - Sq (causal == 2, bottom-right) }
 *     s_j       = scale * sum_d q[b,h,i,d] * k[b,kvh,j,d]
 *     o[b,h,i,:]= sum_{j in J} exp(s_j - m) v[b,kvh,j,:] / sum_{j in J} exp(s_j - m),  m = max s_j
 *     lse[b,h,i]= m + ln sum_{j in J} exp(s_j - m)    (natural log, float32)
 *
 * computed tile by tile with an online softmax; the Sq x Sk score matrix is never stored.
 * A row with no allowed key (only possible with causal == 2 and Sq > Sk) gets the empty-sum
 * result: o = 0 and lse = -inf.  The pages name causal masking without an alignment; the
 * bottom-right form serves queries appended after Sk - Sq cached keys.
 *
 * Layout (all tensors dense, row-major, no strides in the ABI):
 *   q   [B, Hq,  Sq, D]  16-bit (bf16 for fa_fwd, fp16 for fa_fwd_fp16)
 *   k   [B, Hkv, Sk, D]  same type
 *   v   [B, Hkv, Sk, D]  same type
 *   o   [B, Hq,  Sq, D]  same type, round-to-nearest-even from the fp32 accumulator
 *   lse [B, Hq,  Sq]     float32
 *
 * Ownership: every pointer is a DEVICE pointer on the current CUDA device, allocated and
 * owned by the caller; the library allocates no device memory and keeps no pointer after
 * the call returns.  o and lse must not overlap q, k, v or each other.
 *
 * Asynchrony: the kernel is enqueued on `stream` (0 = the legacy default stream) and the
 * call returns without synchronising.  Argument errors are returned before any CUDA call
 * is made.  The call never aborts, exits or traps; a device-side watchdog failure is
 * reported later through fa_device_status() and leaves NaN in the affected rows of o and lse.
 *
 * Thread safety: calls may be made from several host threads; the only shared mutable
 * state is the per-device watchdog status word and read-only caches of device properties.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle (binary-compatible with cudaStream_t / CUstream). */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_NULL_PTR = 1,        /* q, k, v, o or lse is NULL for a non-empty problem        */
    FA_ERR_BAD_DIM = 2,         /* B, Sq, Sk < 0, or Sk == 0 while B*Hq*Sq > 0, or too large */
    FA_ERR_HEADS = 3,           /* Hq < 1, Hkv < 1, or Hq % Hkv != 0                         */
    FA_ERR_UNSUPPORTED_D = 4,   /* D not in {64, 128, 256} (or not supported by the chosen kernel) */
    FA_ERR_ALIGN = 5,           /* q/k/v/o not 16-byte aligned, or lse not 4-byte aligned    */
    FA_ERR_ALIAS = 6,           /* o or lse overlaps an input or each other                  */
    FA_ERR_SCALE = 7,           /* scale is NaN or infinite                                  */
    FA_ERR_NO_DEVICE = 8,       /* no CUDA device / runtime error querying it                */
    FA_ERR_ARCH = 9,            /* current device is not compute capability 10.3 (sm_103)    */
    FA_ERR_TENSORMAP = 10,      /* cuTensorMapEncodeTiled unavailable or rejected the layout */
    FA_ERR_LAUNCH = 11,         /* the kernel launch failed (cudaGetLastError)               */
    FA_ERR_DEVICE_TIMEOUT = 12, /* (fa_device_status) a bounded device-side wait expired     */
    FA_ERR_CAUSAL = 13,         /* causal not in {0, 1, 2}                                   */
    FA_ERR_SHAPE = 14,          /* (fa_gemm) K or N not a multiple of 8 (16-byte rows)       */
    FA_ERR_ARG = 15,            /* an enum-like argument (dtype, output type, epilogue) is out of range */
    FA_ERR_TOO_LARGE = 16       /* (fa_fwd_host_noalloc) the problem needs more than FA_HOST_NOALLOC_MAX_BYTES of staging */
} fa_status_t;

/*
 * fa_fwd -- bf16 attention forward.  Writes o and lse as described above.
 *   B, Hq, Hkv, Sq, Sk, D : sizes (D in {64, 128, 256}; Hq % Hkv == 0)
 *   causal                : 0 = full attention, 1 = key j allowed iff j <= i (top-left),
 *                           2 = key j allowed iff j <= i + Sk - Sq (bottom-right)
 *   scale                 : multiplies q.k before the softmax (usually 1/sqrt(D))
 *   stream                : CUDA stream to enqueue on
 * B == 0 or Sq == 0 is a valid empty problem and returns FA_OK without touching memory.
 * Returns FA_OK or one of the fa_status_t codes.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
           fa_stream_t stream);

/*
 * fa_fwd_select -- fa_fwd (dtype 0, bf16) / fa_fwd_fp16 (dtype 1) with an explicit kernel
 * variant, for tuning sweeps (the course's lesson 10: a search space of meta-parameters
 * measured per workload).  Same results up to rounding order.
 *   kernel 0: automatic -- 1 for D <= 128, 2 for D = 256 (what fa_fwd does)
 *   kernel 1: two 128-row query tiles per CTA sharing 128-key steps (D 64 or 128)
 *   kernel 2: one 128-row query tile per CTA, 64-key steps, double-buffered scores (D 64, 128 or
 *             256; the block-size trade of the guide's troubleshooting item, and the only
 *             layout that fits D = 256 in tensor memory; at D = 64 two CTAs share an SM and
 *             every query tile gets its own CTA, heaviest first)
 *   kernel 3: one 128-row query tile per CTA, 128-key steps, double-buffered scores (D 128)
 * An unsupported (kernel, D) pair returns FA_ERR_UNSUPPORTED_D; kernel or dtype out of range
 * returns FA_ERR_ARG.
 */
int fa_fwd_select(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                  fa_stream_t stream, int dtype, int kernel);

/* fa_fwd_fp16 -- identical to fa_fwd with IEEE fp16 q, k, v and o. */
int fa_fwd_fp16(const void *q, const void *k, const void *v, void *o, float *lse,
                int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                fa_stream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char *fa_strerror(int status);

/*
 * fa_device_status -- synchronises `stream`, then reads and clears the current device's
 * watchdog word.  Returns FA_OK if no kernel since the last read gave up on a wait,
 * FA_ERR_DEVICE_TIMEOUT if one did, or FA_ERR_NO_DEVICE on a CUDA error.  A wait gives up
 * only after its limit (2 s by default) without progress, e.g. when the GPU is preempted for
 * that long.  The attention kernels then leave the call's outputs visibly invalid: every
 * query row of every CTA that gave up holds NaN in o and in lse (rows of other CTAs hold
 * their results), so a caller that does not poll this word still sees NaN, never a stale or
 * partial value that looks like a result.  (fa_gemm and fa_softmax_rows outputs of such a
 * call are unspecified.)
 * *detail (if non-NULL) receives the raw word: bit 0 = timeout, bits 8..15 = the wait
 * site that expired first.
 */
int fa_device_status(fa_stream_t stream, uint32_t *detail);

/*
 * fa_fwd_debug -- test hook: fa_fwd / fa_fwd_fp16 (is_fp16 selects) with an explicit
 * watchdog limit per wait (timeout_ns, 0 = the default of 2 s), a fault-injection mask
 * (inject bit 0: the load warp of every CTA skips its first V tile, so the MMA warp's wait for
 * it expires; bit 1: only CTA 0 does; the kernel then records FA_ERR_DEVICE_TIMEOUT, the CTAs
 * that gave up leave NaN in their rows of o and lse and every CTA returns normally),
 * the kernel variant (as fa_fwd_select) and the lazy-rescale threshold tau in log2 units
 * (O and l are rescaled only when the running row maximum grows by more than tau; 0 rescales
 * at every new maximum; negative = the default 12; above 15 -- where an unnormalised P could
 * leave the fp16 range -- or NaN returns FA_ERR_ARG).
 * With inject == 0, timeout_ns == 0, kernel == 0 and tau < 0 it is exactly fa_fwd / fa_fwd_fp16.
 */
int fa_fwd_debug(const void *q, const void *k, const void *v, void *o, float *lse,
                 int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                 fa_stream_t stream, int is_fp16, uint64_t timeout_ns, uint32_t inject,
                 int kernel, float tau);

/*
 * fa_gemm -- tiled matrix product with an optional fused epilogue, the tutorial's building
 * block for both attention products ("Guia Prático de Programação de GPU com Tiles", section 5:
 * K-loop tiling with an fp32 accumulator; section 3 and the course's lesson 9: bias and
 * tanh-GELU fused into the same pass):
 *     epilogue 0: C = A B
 *     epilogue 1: C = A B + bias            (bias broadcast over rows)
 *     epilogue 2: C = gelu_tanh(A B + bias), gelu_tanh(h) = 0.5 h (1 + tanh(sqrt(2/pi)(h + 0.044715 h^3)))
 *   a     [M, K] row-major, b [K, N] row-major: bf16 (dtype 0) or fp16 (dtype 1), device pointers
 *   c     [M, N] row-major: the input type (out_fp32 0, round to nearest even) or float32 (1)
 *   bias  [N] float32 device pointer; required for epilogues 1 and 2, ignored for 0
 * K and N must be multiples of 8 (16-byte rows for TMA); a, b, c 16-byte aligned.  M, N or K
 * need not be tile multiples.  M == 0 or N == 0 is an empty no-op.  c must not overlap a, b
 * or bias.  Asynchronous on `stream`; returns FA_OK or a status code (no CUDA call is made
 * for invalid arguments).
 */
int fa_gemm(const void *a, const void *b, void *c, const float *bias, int M, int N, int K,
            int dtype, int out_fp32, int epilogue, fa_stream_t stream);

/*
 * fa_fwd_host -- the attention forward of fa_fwd / fa_fwd_fp16 for q, k, v in HOST memory,
 * with o and lse written back to host memory: the copies in, the kernels and the copies
 * back are overlapped chunk by chunk.  The pages define no host-memory entry point; this is
 * the host-side wrapper that the tile course's lesson 5 asks for (launch, memory safety,
 * input checks) with the overlap of data movement and computation that its "real use
 * cases" list names, applied to the host<->device link.
 *   q_h, k_h, v_h   host inputs, same layout as fa_fwd's q, k, v; read only.  Pinned
 *                   (page-locked) memory gives the overlap; pageable memory is accepted but
 *                   each copy then blocks the host.
 *   o_h, lse_h      host outputs, layout of o and lse
 *   q_d .. lse_d    caller-owned DEVICE buffers of the same sizes on the current device: the
 *                   staging area that the copies fill (q_d, k_d, v_d) and the kernels write
 *                   (o_d, lse_d); on return of the work they hold the inputs and results.
 *   B .. scale      as for fa_fwd;  dtype 0 = bf16, 1 = fp16
 *   chunks          pipeline depth: the flat (batch, KV head) axis is cut into this many
 *                   runs (0 = automatic, 4; capped at B * Hkv; at most 64)
 *   stream          the work starts after what is already enqueued on `stream`, and `stream`
 *                   waits for the last copy back: synchronise it before reading o_h / lse_h.
 * The call is asynchronous and uses three internal streams per device, created on its first
 * call for that device.  Calls for one device are enqueued one at a time (a lock); two calls
 * on different caller streams that share buffers race, as any two kernels would.
 * Results are bit-identical to fa_fwd on the same inputs (each output row is computed by the
 * same kernel in the same order).  Argument errors (fa_fwd's checks on the device buffers,
 * NULL host pointers, any overlap between a written range and another range, dtype or chunks
 * out of range) are returned before any CUDA call; a CUDA error after the first copy was
 * enqueued returns FA_ERR_LAUNCH, leaves the outputs unspecified and still orders `stream`
 * after the enqueued work.
 */
int fa_fwd_host(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                void *q_d, void *k_d, void *v_d, void *o_d, float *lse_d,
                int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                int dtype, int chunks, fa_stream_t stream);

/*
 * fa_softmax_rows -- numerically stable softmax of every row of x ("Guia Prático de
 * Programação de GPU com Tiles", section 4): y[r, :] = exp(x[r, :] - max) / sum exp(x[r, :] - max).
 *   x, y  [rows, cols] row-major device arrays, float32 (dtype 0) or bf16 (dtype 1)
 * y may be x (in place) but may not partially overlap it.  rows == 0 is a no-op; cols must
 * be >= 1.  Asynchronous on `stream`.
 */
int fa_softmax_rows(const void *x, void *y, int rows, int cols, int dtype, fa_stream_t stream);

/* Size of the fixed device staging area of fa_fwd_host_noalloc: 64 MiB. */
#define FA_HOST_NOALLOC_MAX_BYTES (64ull << 20)

/*
 * fa_fwd_host_noalloc -- fa_fwd_host for callers that cannot allocate device memory.  The pages
 * have no counterpart to it: it exists for callers that hold q, k, v, o and lse in host memory
 * and may not call cudaMalloc themselves -- for instance a plug-in whose host application owns
 * every device allocation and caps it, or a caller that must not pay for the implicit device
 * synchronisation an allocation can bring.  fa_fwd_host needs five device buffers from its
 * caller as the staging area of its copies; this variant takes them instead from one
 * FA_HOST_NOALLOC_MAX_BYTES array of device memory that is part of the library's device image.
 * Each GPU on which that image is loaded keeps the array until the process exits.
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *   q_h .. lse_h, B .. scale, dtype, chunks, stream : as for fa_fwd_host, with the same results
 *                   (bit-identical: the same kernels run on the same values)
 * Staging needs |q| + |k| + |v| + |o| + |lse| bytes, each rounded up to 256 bytes
 * (2 B Hq Sq D + 2 B Hkv Sk D twice + 4 B Hq Sq before rounding); a larger problem returns
 * FA_ERR_TOO_LARGE.  That check and every argument check are made before any CUDA call.
 * The first call on a device (with that device current) looks up the array's device address
 * once (cudaGetSymbolAddress) and keeps it: make that first call before any stream capture
 * starts.  A failed look-up returns FA_ERR_NO_DEVICE.  The kept address belongs to the device's
 * primary context as it was at that first call: do not call this entry point again on a device
 * after cudaDeviceReset() (or any other reset of its primary context) in the same process.
 * Every call on a device shares the one array, and a call leaves its inputs and results
 * there.  Nothing in it has to start at zero: each call writes every byte it reads.  Calls
 * that run at the same time on the GPU race on the array: two calls on one stream run in
 * order, but calls on different streams must be ordered by the caller (an event, a
 * synchronise).  In particular, fa_fwd_host_noalloc calls kept in flight on two streams at
 * once, as fa_fwd_host calls with their own buffers may be, give wrong results.
 */
int fa_fwd_host_noalloc(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                        int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                        int dtype, int chunks, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
