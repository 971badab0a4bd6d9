/*
 * attn_bwd.h -- C ABI of the dense BF16 attention backward pass for GB300 (sm_103a).
 *
 * The notes on the method name the backward pass and recomputation as part of it
 * ("FlashAttention'ı Anlamak Bölüm 1", section 0 Giriş) without giving formulas; what it
 * computes is the gradient of the forward of attn_fwd.h (S = scale * Q K^T,
 * P = softmax_row(S), O = P V) for an upstream gradient dO:
 *
 *   D_i = sum_c dO[i,c] O[i,c]                     (= sum_j P_ij dP_ij)
 *   P   = exp(scale * Q K^T - LSE)                  recomputed from the forward's LSE
 *   dV  = P^T dO,   dP = dO V^T,   dS = P * (dP - D)
 *   dQ  = scale * dS K,   dK = scale * dS^T Q
 *
 * S and P are recomputed tile by tile on the tensor cores and never reach HBM.
 *
 * Return values: the ATTN_* codes of attn_fwd.h.
 */
#ifndef ATTN_BWD_H
#define ATTN_BWD_H

#include "attn_fwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_bwd -- gradients of the non-causal forward (no bias).
 *
 *   q, k, v   device, BF16, [B, H, Nq | Nk | Nk, d] contiguous, read only (the forward's inputs)
 *   o         device, BF16, [B, H, Nq, d], the forward's output
 *   dout      device, BF16, [B, H, Nq, d], the upstream gradient dO
 *   lse       device, FP32, [B, H, Nq], the forward's log-sum-exp (natural log)
 *   dq        device, BF16, [B, H, Nq, d], written
 *   dk, dv    device, BF16, [B, H, Nk, d], written
 *   scale     the forward's scale (finite)
 *   stream    cudaStream_t (0 = legacy default stream)
 *
 * Sizes and alignment follow attn_fwd: d must be 128 (else ATTN_ERR_UNSUPPORTED), every
 * BF16 pointer 16-byte aligned and lse 4-byte aligned (else ATTN_ERR_MISALIGNED), null
 * pointers or negative sizes give ATTN_ERR_INVALID_ARG; B*H*Nq = 0 with Nk >= 0 is a no-op
 * (dk and dv are then left unwritten); Nk = 0 with rows is invalid. Outputs must not alias
 * inputs. All checks happen before the GPU is touched.
 *
 * Work: three kernels on `stream` -- a row pass that forms D and the LSE in log2 units
 * (into a workspace of B*H*ceil(Nq/128)*128*8 bytes that the library allocates with
 * cudaMallocAsync on the stream the first time it is needed and keeps per (device,
 * stream)), a pass over key tiles that forms dK and dV, and a pass over query tiles that
 * forms dQ. Calls on one stream are ordered by the stream; calls on different streams
 * use different workspaces. Every wait inside the kernels is bounded; a wait that gives
 * up ends its block and sets a status word read by attn_bwd_status.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, void* stream);

/*
 * attn_bwd_causal -- gradients of the causal forward (attn_fwd_causal: query i sees keys
 * 0 .. i + Nk - Nq, the mask aligned to the bottom-right corner). Arguments, layouts,
 * rules and work are those of attn_bwd, with o and lse from attn_fwd_causal, plus
 * Nq <= Nk (else ATTN_ERR_INVALID_ARG). Blocks visit only the tiles their rows or keys
 * can see.
 */
int attn_bwd_causal(const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                    float scale, void* stream);

/*
 * attn_bwd_bias -- gradients dQ, dK, dV of the biased forward (attn_fwd_bias: S = scale Q K^T
 * + B, the definition's optional B, "FlashAttention'ı Anlamak Bölüm 1", section 0.2), the bias
 * held fixed: it enters only through the recomputed P = exp(scale q.k + B - LSE), and its
 * own gradient (dB = dS) is not formed. bias and its strides as in attn_fwd_bias (with its
 * argument rules: non-null, non-negative strides whose last offset fits 64 bits, 16-byte
 * aligned, strides multiples of 8 elements); o and lse from attn_fwd_bias with the same bias.
 * Other arguments, layouts and return values are those of attn_bwd. Each block reads the
 * bias of its tile pairs once per kernel (the dK/dV kernel by keys, the dQ kernel by rows).
 * Not with the causal mask (a causal bias carries one).
 */
int attn_bwd_bias(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, const void* bias, long long bias_stride_b, long long bias_stride_h,
                  long long bias_stride_q, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                  float scale, void* stream);

/* Synchronises `stream`, then reads and clears the backward kernels' timeout status:
 * ATTN_OK, ATTN_ERR_TIMEOUT or ATTN_ERR_CUDA. */
int attn_bwd_status(void* stream);

/*
 * Test hook for the failure path (mirrors attn_fwd_set_wait_limit): `cycles` sets the
 * per-wait time limit of later backward launches in SM clock cycles (0 restores the
 * default of 2^31); `withhold_tile` != 0 makes the dK/dV kernel's loader stop before the
 * second query tile of every block, so the waits for it run out and the call reports
 * ATTN_ERR_TIMEOUT through attn_bwd_status. Not for production use.
 */
int attn_bwd_set_wait_limit(unsigned long long cycles, int withhold_tile);

/* Kernel launches made by attn_bwd in this process (three per call that does work). */
unsigned long long attn_bwd_kernel_count(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BWD_H */
