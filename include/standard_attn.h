/*
 * standard_attn.h -- C ABI of standard (materialising) attention, the
 * baseline the method is compared against: S = scale * Q K^T is written to
 * device memory, P = softmax(S) is written to device memory and kept for the
 * backward pass, O = P V (FlashAttention milestone page (nlp-lineage),
 * "The notation": standard attention computes S = QK^T, P = softmax(S),
 * O = PV and needs Theta(Nd + N^2) HBM accesses; "What it showed": the
 * memory-traffic comparison on one GPT-2 medium attention layer).
 *
 * It exists to re-measure that comparison (HBM bytes, run time, memory
 * footprint) and the numerical-stability claim against the same oracle; it
 * is not on the path of flash_attn.h and shares none of its kernels. The
 * four matrix products of the backward pass and the two of the forward pass
 * are cuBLAS strided-batched GEMMs (bf16/fp16 inputs, fp32 accumulation); the
 * masked softmax and dS = P * (dP - rowsum(P * dP)) are row kernels of this
 * library.
 *
 * Conventions are those of flash_attn.h (row-major [B, H, N, d] tensors,
 * device pointers owned by the caller, calls asynchronous on `stream`,
 * argument errors returned before any launch, masks combining by AND, a
 * fully masked row giving O = 0, LSE = -inf, dQ = 0), except:
 *  - d may be any multiple of 8 from 8 to 256;
 *  - the workspace holds the materialised matrices and carries P from
 *    standard_attn_fwd to standard_attn_bwd:
 *      S (fp32 [B, H, N, N], or 16-bit with STANDARD_ATTN_S16; reused for dP
 *      in the backward pass), then
 *      P (16-bit [B, H, N, N]; overwritten in place by dS in the backward
 *      pass, so a second backward call needs a new forward call);
 *  - cuBLAS may allocate its own workspace when the library creates its
 *    handle for a device (the first call on that device).
 */
#ifndef STANDARD_ATTN_H
#define STANDARD_ATTN_H

#include "flash_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of workspace for this shape (fp32 S plus 16-bit P, each section
 * 256-byte aligned; enough for either flag setting); 0 for an invalid shape
 * or one whose size overflows. */
size_t standard_attn_workspace_size(int B, int H, int N);

/*
 * flags of standard_attn_fwd / standard_attn_bwd:
 *   STANDARD_ATTN_S16: S = scale * Q K^T and dP = dO V^T are stored in the
 *   16-bit element type of the inputs (as a framework's 16-bit matmul
 *   returns them) instead of fp32; the softmax and dS still compute in fp32
 *   from the stored values. This is the low-precision standard attention the
 *   pages' stability remark is about (FlashAttention proof-of-work page, the
 *   question whether the method is an approximation: with its online softmax
 *   and high-precision accumulators it is often numerically more stable than
 *   standard PyTorch attention). fwd and bwd must use the same flags.
 */
#define STANDARD_ATTN_S16 1

/*
 * Forward pass: writes S and P to the workspace, then O and LSE.
 *   Q, K, V : in,  [B, H, N, d], bf16 (fp16 with options->dtype)
 *   O       : out, [B, H, N, d];  LSE : out, fp32 [B, H, N] (natural log of
 *             the row sum of exp(S) over the allowed keys)
 *   B, H >= 1; 1 <= N <= 65536; d a multiple of 8 in [8, 256]; scale finite;
 *   causal 0 or 1; kv_len, block_mask as in flash_attn.h (may be NULL).
 *   options: NULL or an fa_options; only dtype is used; p_drop must be 0,
 *            tile_record NULL and test_stall 0 (FA_ERR_UNSUPPORTED otherwise).
 *   flags:   0 or STANDARD_ATTN_S16 (FA_ERR_INVALID_ARG otherwise).
 *   workspace: at least standard_attn_workspace_size(B, H, N) bytes,
 *            256-byte aligned (FA_ERR_WORKSPACE otherwise).
 */
fa_status standard_attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            int B, int H, int N, int d, float scale, int causal,
                            const int32_t* kv_len, const uint8_t* block_mask,
                            const fa_options* options, int flags, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * Backward pass from the P that standard_attn_fwd left in the workspace:
 *   dV = P^T dO;  dP = dO V^T (into the S section);
 *   dS = P * (dP - D) with D_i = sum_j P_ij dP_ij (over P, in place);
 *   dQ = scale * dS K;  dK = scale * dS^T Q.
 *   Q, K, V, dO : in,  [B, H, N, d];  dQ, dK, dV : out, [B, H, N, d]
 *   The shape, scale, dtype and workspace must be those of the forward call.
 */
fa_status standard_attn_bwd(const void* Q, const void* K, const void* V, const void* dO,
                            void* dQ, void* dK, void* dV, int B, int H, int N, int d, float scale,
                            const fa_options* options, int flags, void* workspace,
                            size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* STANDARD_ATTN_H */
