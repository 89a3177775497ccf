/*
 * flash_attn.h -- C ABI of an exact, IO-aware attention library for NVIDIA
 * GB300 (sm_103a): forward and backward of
 *
 *     O = softmax(scale * Q K^T + mask) V
 *
 * computed tile by tile with an online softmax, never storing the N x N score
 * matrix (FlashAttention milestone page (nlp-lineage), "The notation" and
 * "The idea"; FlashAttention proof-of-work page, "SRAM Block Tiling",
 * "Online Softmax Computation", "Activation Gradient Recomputation").
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensors are row-major, contiguous, one (batch, head) after another:
 *      Q, K, V, O, dO, dQ, dK, dV : bfloat16 [B, H, N, d] (fp16 through the
 *                                   *_ex calls)
 *      LSE                         : float32  [B, H, N]
 *    N is the sequence length of both queries and keys. d is a multiple of
 *    8 from 8 to 128: 64 and 128 run on kernels of exactly that width; any
 *    other d runs on the 64- (d < 64) or 128-column (d > 64) kernel over
 *    tiles whose columns past d are zero (the arithmetic of the padded
 *    width is spent, the result is that of width d).
 *  - Every pointer named here is a DEVICE pointer of the current CUDA device,
 *    16-byte aligned, owned by the caller (the library keeps no reference
 *    after the call returns and allocates no device memory).
 *  - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *    default stream). Argument errors are returned before anything is
 *    launched; launch errors are returned as FA_ERR_CUDA. Errors that arise
 *    on the device (a bounded wait that ran out) are recorded in a device
 *    error word read by flash_attn_get_device_error() after the stream has
 *    been synchronised.
 *  - Masks combine by AND. Key j takes part in query row i's softmax when
 *      (causal == 0 || j <= i)  and  j < kv_len[b]  and
 *      block_mask[(i / 128) * nT + (j / 128)] != 0,       nT = ceil(N / 128).
 *    kv_len (device int32 [B], values clamped to [0, N]) and block_mask
 *    (device uint8 [nT, nT], shared by all batches and heads; the block-sparse
 *    pattern whose empty blocks are skipped -- milestone page, "The idea")
 *    may each be NULL, meaning "no such mask". Tiles with no allowed pair
 *    are skipped entirely.
 *  - A query row with no allowed key gets O = 0, LSE = -inf and dQ = 0.
 *  - Every output element is written; outputs need no initialisation.
 */
#ifndef FLASH_ATTN_H
#define FLASH_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,      /* null/misaligned pointer, bad size, non-finite scale */
  FA_ERR_UNSUPPORTED = 2,      /* d not a multiple of 8 in [8, 128], N > 131072, no sm_103a device */
  FA_ERR_WORKSPACE = 3,        /* workspace missing, misaligned or too small */
  FA_ERR_CUDA = 4,             /* a CUDA runtime call or a launch failed */
  FA_ERR_DEVICE_TIMEOUT = 5,   /* a kernel's bounded wait ran out (device error word) */
  FA_ERR_DEVICE_INTERNAL = 6,  /* a kernel found an internal inconsistency (misaligned shared memory,
                                  a work item out of range) */
  FA_ERR_SCRATCH_LIMIT = 7     /* flash_attn_bwd_noalloc: shape needs more than its fixed scratch */
} fa_status;

/*
 * Options of the *_ex calls (no counterpart on the pages; the pages name
 * FP16 and BF16 as the formats the method is meant for -- Flash Attention
 * glossary, "Tensor Cores"; pixelation.org article, "Actionable Next Steps").
 * size must be set to sizeof(fa_options) by the caller; fields past the size
 * a caller declares keep their defaults, so the struct can grow without
 * breaking older callers. Passing NULL for the options selects all defaults.
 *   dtype:  element type of Q, K, V, O, dO, dQ, dK, dV: FA_DTYPE_BF16
 *           (default) or FA_DTYPE_F16. LSE stays fp32.
 *   p_drop: dropout probability applied to P between the two products, as
 *           in the method's fused kernel (milestone page, "The idea");
 *           0 (default) = none, otherwise in (0, 1) and used in steps of
 *           1/256: t = round(256 p_drop) must be <= 255.
 *   seed:   key of the dropout generator. Element (i, j) of batch-head
 *           bh = b * H + h is kept when byte 4 (i mod 4) + (j mod 4) of
 *           Philox4x32-10 with counter (i / 4, j / 4, bh, 0) and key
 *           (seed mod 2^32, seed / 2^32) is >= t; kept values are scaled by
 *           256 / (256 - t). The softmax statistics (LSE) use the undropped
 *           P. The backward call regenerates the same mask from the same
 *           p_drop and seed; nothing of the mask is stored.
 *   tile_record: NULL (default), or a device uint8 [B, H, nT, nT] array that
 *           the caller has zeroed. The kernels then record the tiles they
 *           actually compute: for every (b, h, query tile qi, key tile kj)
 *           that a kernel processes it adds 1 to byte
 *           ((b * H + h) * nT + qi) * nT + kj when the tile needs no element
 *           mask and 2 when it applies one; skipped tiles stay 0. A correct
 *           run therefore reproduces flash_attn_tile_map's states per head,
 *           and a tile computed twice would read 2 or 4. The forward and the
 *           backward call each record into the array they are given (the
 *           block-sparse skipping of the milestone page, "The idea", as the
 *           kernels ran it). Costs one byte update per computed tile.
 *   wait_limit_us: bound of every wait of a kernel on an on-chip barrier,
 *           in microseconds; 0 (default) = 2 s. A wait that runs out makes
 *           the kernel stop, free its on-chip resources and record
 *           FA_ERR_DEVICE_TIMEOUT in the device error word.
 *   test_stall: 0 (default). 1 is for testing the timeout path only: the
 *           kernels' tile loader stops after its first tile, so that a
 *           bounded wait runs out (after wait_limit_us) and the call's
 *           outputs are unspecified; flash_attn_get_device_error then
 *           returns FA_ERR_DEVICE_TIMEOUT. Nothing faults; the device stays
 *           usable.
 */
typedef enum { FA_DTYPE_BF16 = 0, FA_DTYPE_F16 = 1 } fa_dtype;

typedef struct {
  uint32_t size;      /* sizeof(fa_options) */
  int32_t dtype;
  float p_drop;
  uint32_t reserved;  /* 0 */
  uint64_t seed;
  uint8_t* tile_record;
  uint32_t wait_limit_us;
  uint32_t test_stall;
} fa_options;

/*
 * Forward pass. Computes, for every (b, h) and query row i,
 *   O[b,h,i,:]  = sum_j P_ij V[b,h,j,:],  P_ij = exp(S_ij - LSE[b,h,i]),
 *   LSE[b,h,i]  = ln sum_j exp(S_ij),     S_ij = scale * Q[b,h,i,:] . K[b,h,j,:]
 * over the allowed keys j (natural logarithm, scaled scores). Only O and LSE
 * are written (milestone page, "The idea -- Recomputation": the output and the
 * softmax statistics are all the backward pass needs).
 *   Q, K, V : in,  bf16 [B, H, N, d]
 *   O       : out, bf16 [B, H, N, d]
 *   LSE     : out, fp32 [B, H, N]
 *   B, H >= 1; 1 <= N <= 131072; d a multiple of 8 in [8, 128]; scale finite;
 *   causal 0 or 1; kv_len, block_mask as above (may be NULL).
 */
fa_status flash_attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                         int B, int H, int N, int d, float scale, int causal,
                         const int32_t* kv_len, const uint8_t* block_mask, void* stream);

/* flash_attn_fwd with options (see fa_options); flash_attn_fwd is this call
 * with options = NULL. */
fa_status flash_attn_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            int B, int H, int N, int d, float scale, int causal,
                            const int32_t* kv_len, const uint8_t* block_mask,
                            const fa_options* options, void* stream);

/*
 * Bytes of device workspace flash_attn_bwd needs for this shape (fp32 dQ
 * accumulator [B, H, nT*128, d], two fp32 row vectors [B, H, nT*128] and a
 * 256-byte block holding the work counter of the persistent kernel; each
 * section 256-byte aligned). Returns 0 for an invalid shape.
 */
size_t flash_attn_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass by recomputation: given the forward's inputs, its outputs O
 * and LSE, and the output gradient dO, writes
 *   dV = P^T dO,  dQ = scale * dS K,  dK = scale * dS^T Q,
 *   dS = P * (dP - D),  dP = dO V^T,  D_i = sum_c dO_ic O_ic,
 * recomputing S and P block by block on chip (milestone page, "The idea --
 * Recomputation"; the gradient formulas are the textbook derivative of
 * L = sum(dO * O), which the pages do not spell out).
 *   Q, K, V, O, dO : in,  bf16 [B, H, N, d];  LSE : in, fp32 [B, H, N]
 *   dQ, dK, dV     : out, bf16 [B, H, N, d]
 *   workspace      : device scratch of at least
 *                    flash_attn_bwd_workspace_size(B, H, N, d) bytes,
 *                    256-byte aligned, owned by the caller; its contents on
 *                    entry do not matter and on exit are unspecified.
 *   Other arguments as in flash_attn_fwd; they must match the forward call
 *   that produced O and LSE.
 */
fa_status flash_attn_bwd(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                         int B, int H, int N, int d, float scale, int causal,
                         const int32_t* kv_len, const uint8_t* block_mask,
                         void* workspace, size_t workspace_bytes, void* stream);

/* flash_attn_bwd with options (see fa_options); the options must match the
 * forward call that produced O and LSE. flash_attn_bwd is this call with
 * options = NULL. */
fa_status flash_attn_bwd_ex(const void* Q, const void* K, const void* V, const void* O,
                            const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                            int B, int H, int N, int d, float scale, int causal,
                            const int32_t* kv_len, const uint8_t* block_mask,
                            const fa_options* options, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * Backward pass for callers that cannot allocate device memory. (The pages
 * describing the method have no counterpart of this call; it is an interface
 * convenience.) Some callers cannot provide the workspace flash_attn_bwd
 * needs: a plug-in running inside another runtime's execute callback, where
 * allocating device memory is not allowed; a serving loop that must never
 * call cudaMalloc on the request path, because it synchronises the device
 * and can stall every stream; a program whose device memory belongs to a
 * pool that hands out no raw buffers. This call computes exactly what
 * flash_attn_bwd computes (same arguments, minus the workspace) and takes
 * its scratch from a fixed array of FA_BWD_NOALLOC_SCRATCH_BYTES (64 MiB)
 * that the library keeps on every device that loads it, until the process
 * exits. This call allocates nothing (the baseline of standard_attn.h, which
 * creates a cuBLAS handle, is another matter).
 *   - Shapes whose flash_attn_bwd_workspace_size exceeds
 *     FA_BWD_NOALLOC_SCRATCH_BYTES are rejected with FA_ERR_SCRATCH_LIMIT
 *     before anything is launched.
 *   - All calls on a device share the one array. Calls ordered on one stream
 *     are safe; calls whose kernels may overlap on the GPU (several streams,
 *     or several host threads without ordering) race on it and give wrong
 *     results. Each call rewrites whatever it reads from the array, so what a
 *     previous call left there does not matter.
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture
 *     starts. Under CUDA's default lazy module loading that first call is
 *     also when the array is reserved on the device, so make it where
 *     allocation is still allowed (a call refused with FA_ERR_SCRATCH_LIMIT
 *     does as a warm-up, since the lookup comes before the size check), or
 *     set CUDA_MODULE_LOADING=EAGER.
 *   - Profile events set with flash_attn_set_profile_events apply to this
 *     call as to flash_attn_bwd (around the backward main kernel).
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

fa_status flash_attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                 const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                                 int B, int H, int N, int d, float scale, int causal,
                                 const int32_t* kv_len, const uint8_t* block_mask, void* stream);

/*
 * The tile classifier the kernels use to decide which 128 x 128 tiles to
 * compute: writes out[b, qi, kj] (device uint8 [B, nT, nT]) as
 *   0 = skipped (no allowed pair), 1 = full (every pair allowed),
 *   2 = partial (computed with element masking).
 * Rows past N do not count; keys past N count as masked.
 */
fa_status flash_attn_tile_map(int B, int N, int causal, const int32_t* kv_len,
                              const uint8_t* block_mask, uint8_t* out, void* stream);

/*
 * Reads and clears the device error word of the current device. Call after
 * synchronising the streams used. Returns FA_OK when no kernel reported an
 * error. If detail is not NULL it receives 4 host uint32 values:
 * {code, site, block, thread} of the first error recorded.
 */
fa_status flash_attn_get_device_error(uint32_t* detail);

/*
 * Profiling hook (no counterpart on the pages; for timing the kernels with
 * CUDA events on the stream they run on). start_event and stop_event are
 * cudaEvent_t handles created by the caller. Once set, the next
 * flash_attn_fwd or flash_attn_bwd call made by this host thread records
 * start_event on its stream immediately before its dominant kernel (the
 * forward kernel, or the backward main kernel) and stop_event immediately
 * after it, then forgets both. Passing NULL, NULL clears a pending setting.
 * Returns FA_ERR_INVALID_ARG if exactly one handle is NULL.
 */
fa_status flash_attn_set_profile_events(void* start_event, void* stop_event);

/* Human-readable name of a status code (static storage). */
const char* flash_attn_status_string(fa_status status);

/* Library ABI version: 100 * major + minor. */
int flash_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FLASH_ATTN_H */
