/*
 * attn_fwd.h -- C ABI of the GB300 (sm_103a) dense attention forward library.
 *
 * The operation is scaled-dot-product attention for one head at a time,
 *
 *     S = scale * Q K^T,   P = softmax_row(S),   O = P V,
 *
 * as written in "FlashAttention'ı Anlamak Bölüm 1", section 0.2 Notasyon (with the
 * optional mask/bias taken as zero), and computed the FlashAttention way: Q, K, V
 * and O cut into 128x128 tiles, each output tile owned by one thread block, which
 * loads its Q tile once and streams K/V tile pairs through an online softmax, so
 * that neither S nor P is ever written to device memory ("Sıfırdan yazılan CUDA
 * attention kerneli...", section "Kernel işini nasıl bölümlendiriyor"; the online
 * update of "Flash Attention на 5090 в CUDA C++", v1). The notes state that the
 * result is exact attention, not an approximation, up to floating-point order.
 *
 * Besides O the call writes, per query row, the natural log-sum-exp of its scaled
 * scores, lse = log(sum_j exp(S_ij)). The pages do not define this output; it is
 * the softmax denominator in log form, the quantity a backward pass needs.
 *
 * Conventions shared by every entry point below:
 *   - Tensors are dense, C-ordered, [B, H, N, d] (batch, heads, sequence, head dim)
 *     with d = 128 (attn_fwd, attn_fwd_causal, attn_fwd_bias, attn_fwd_noalloc and the
 *     attn_fwd_fp8qk and attn_fwd_fp8 families also take 192 and 256), in device
 *     memory reachable from the current CUDA device.
 *   - BF16 is IEEE-style bfloat16 (1 sign, 8 exponent, 7 mantissa bits), passed as
 *     raw 16-bit storage (void*).
 *   - The caller owns every buffer it passes; the library keeps no pointer to them
 *     after a call returns. When a call's work does not divide evenly over the SMs,
 *     the kernel splits the key range of some query tiles between thread blocks and
 *     merges the pieces; it then needs a workspace (under 300 KB per SM) that the
 *     library allocates with cudaMallocAsync on the call's stream the first time it
 *     is needed, grows when a later call needs more, and keeps per (device, stream)
 *     for the life of the process, so calls on different streams never share one.
 *   - Calls are asynchronous: work is enqueued on `stream` (a cudaStream_t; NULL
 *     means the legacy default stream) and the call returns at once. Only argument
 *     and launch errors are reported by the return value.
 *   - No C++ exception crosses this interface. Calls are thread-safe.
 */
#ifndef ATTN_FWD_H
#define ATTN_FWD_H

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define ATTN_OK               0
#define ATTN_ERR_INVALID_ARG (-1) /* null pointer, negative size, Nk == 0 with rows to compute, non-finite scale, size overflow */
#define ATTN_ERR_UNSUPPORTED (-2) /* a head dimension the entry point does not take, or sizes beyond the kernel's index range */
#define ATTN_ERR_MISALIGNED  (-3) /* q, k, v or o not 16-byte aligned, or lse not 4-byte aligned */
#define ATTN_ERR_CUDA        (-4) /* a CUDA runtime or driver call failed (no device, launch failure, ...) */
#define ATTN_ERR_TIMEOUT     (-5) /* a kernel gave up a pipeline wait after its time limit (see attn_fwd_status) */

/*
 * attn_fwd -- dense, non-causal attention forward.
 *
 *   q    device, BF16 [B, H, Nq, d], read
 *   k    device, BF16 [B, H, Nk, d], read
 *   v    device, BF16 [B, H, Nk, d], read
 *   o    device, BF16 [B, H, Nq, d], written: O = softmax(scale * Q K^T) V,
 *        each element rounded to nearest-even from FP32
 *   lse  device, FP32 [B, H, Nq],    written: log(sum_j exp(scale * q_i . k_j))
 *   B, H, Nq, Nk   sizes, >= 0. B*H*Nq == 0 is an empty call: nothing is read or
 *        written and ATTN_OK is returned. Otherwise Nk must be >= 1. Any Nq and Nk
 *        are accepted; a sequence that is not a multiple of 128 ends in a partial
 *        tile that the kernel masks.
 *   d    head dimension: 128, 192 or 256. Head dimensions above 128 ("Flash Attention на
 *        5090 в CUDA C++", section "Что дальше") run a kernel that gives each thread block
 *        one 128-row query tile (TMEM holds its S twice and its O) and whole key ranges,
 *        so they need no workspace.
 *   scale  any finite float, applied to the scores (1/sqrt(d) for standard attention).
 *   stream a cudaStream_t, or NULL.
 *
 * o must not overlap q, k, v or lse (not checked). The call writes o, lse and, when it
 * splits work between blocks, its own workspace (see above).
 *
 * Returns ATTN_OK once the kernel is enqueued; ATTN_ERR_INVALID_ARG,
 * ATTN_ERR_UNSUPPORTED or ATTN_ERR_MISALIGNED without touching the GPU when an
 * argument is rejected; ATTN_ERR_CUDA when the launch or the workspace allocation fails.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int Nq, int Nk, int d, float scale, void* stream);

/*
 * attn_fwd_causal -- causal attention forward.
 *
 * The optional mask B of the definition ("FlashAttention'ı Anlamak Bölüm 1", section 0.2)
 * taken as the causal mask: B_ij = 0 when j <= i + (Nk - Nq) and -inf otherwise, i.e.
 * query i sees keys 0 .. i + Nk - Nq. The mask is aligned to the bottom-right corner of
 * the score matrix, so the last query sees every key (a block of Nq queries that follows
 * Nk - Nq earlier positions). The pages do not fix the alignment; this is the reading
 * under which a square problem is the usual lower-triangular mask.
 *
 * Arguments, layouts and return values are those of attn_fwd, plus:
 *   - Nq <= Nk is required (every query row sees at least one key); Nq > Nk returns
 *     ATTN_ERR_INVALID_ARG without touching the GPU.
 *   - lse is the log-sum-exp over the visible keys only.
 *   - The call allocates nothing: each block processes whole (b, h, 256-row) groups,
 *     longest first, over only the key tiles its rows can see.
 *   - d = 192 and 256 are taken too (the kernel of attn_fwd at those head dimensions, with
 *     whole 128-row query tiles, longest first).
 */
int attn_fwd_causal(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int Nq, int Nk, int d, float scale, void* stream);

/*
 * attn_fwd_bias -- attention forward with an additive bias.
 *
 * S = scale * Q K^T + B, P = softmax_row(S), O = P V: the definition's optional bias B
 * ("FlashAttention'ı Anlamak Bölüm 1", section 0.2 Notasyon), one Nq x Nk matrix per head,
 * with the caller's scale in place of 1/sqrt(d) as in attn_fwd.
 *
 *   bias   device, BF16, read only. B_ij of head (b, h) is
 *          bias[b * bias_stride_b + h * bias_stride_h + i * bias_stride_q + j]
 *          (strides in elements, keys contiguous). A stride of 0 shares the values:
 *          (0, 0, Nk) is one Nq x Nk matrix for every head, (0, 0, 0) one bias per key
 *          (e.g. a key padding mask). The caller owns it; it must not alias o or lse.
 *
 * Arguments, layouts and return values are otherwise those of attn_fwd, plus:
 *   - ATTN_ERR_INVALID_ARG: bias is NULL, a stride is negative, or the offset of the
 *     last element overflows a 64-bit byte offset.
 *   - ATTN_ERR_MISALIGNED: bias is not 16-byte aligned or a stride is not a multiple
 *     of 8 elements (each row is read in 16-byte pieces).
 *   - Entries must be finite or -inf; -inf removes the key from that row. A row whose
 *     entries are all -inf has no softmax: its O and LSE are unspecified (NaN or inf).
 *     NaN or +inf entries give unspecified results for their row.
 *   - lse is the log-sum-exp of the biased scores, in natural-log units.
 *   - The work split and workspace are those of attn_fwd (the bias adds no state). The
 *     bias is read once per (query row, key), from L2 when it is shared across heads.
 *   - d = 192 and 256 are taken too: attn_fwd's one-query-tile kernel at those head
 *     dimensions, each thread adding its own row's bias; no workspace.
 */
int attn_fwd_bias(const void* q, const void* k, const void* v, const void* bias,
                  long long bias_stride_b, long long bias_stride_h, long long bias_stride_q,
                  void* o, float* lse, int B, int H, int Nq, int Nk, int d, float scale, void* stream);

/*
 * attn_fwd_fp8qk -- attention forward with the scores computed from 8-bit floating point.
 *
 * The low-precision MMA that "Flash Attention на 5090 в CUDA C++" (section "Что дальше")
 * lists as the next step, applied to S: Q and K arrive as FP8 E4M3 codes (the OCP 8-bit
 * floating point format: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, S.1111.111 = NaN, largest finite value 448) with one positive descale factor
 * per tensor, so the real inputs are q_descale * Q8 and k_descale * K8, and
 *
 *     S = scale * q_descale * k_descale * (Q8 K8^T),   P = softmax_row(S),   O = P V
 *
 * with V, P and O in BF16 as in attn_fwd. The products of two E4M3 values are exact in
 * the FP32 accumulators of the tensor cores (kind::f8f6f4); scale * q_descale * k_descale
 * is rounded once to FP32 on the host.
 *
 *   q8     device, [B, H, Nq, d] bytes (E4M3 codes), read only
 *   k8     device, [B, H, Nk, d] bytes (E4M3 codes), read only
 *   v      device, BF16, [B, H, Nk, d], read only
 *   q_descale, k_descale   finite and > 0 (else ATTN_ERR_INVALID_ARG); a combined scale
 *          whose magnitude exceeds FLT_MAX is ATTN_ERR_INVALID_ARG too
 *
 * Arguments, layouts, alignment rules (q8 and k8 16-byte aligned), the work split,
 * workspace and return values are otherwise those of attn_fwd. NaN codes give
 * unspecified results for the rows they reach. d = 192 and 256 run attn_fwd's
 * one-query-tile kernel with Q K^T on kind::f8f6f4 (so do attn_fwd_fp8qk_causal and
 * attn_fwd_fp8qk_bias, and the attn_fwd_fp8 family with P V on kind::f8f6f4 too); the
 * MXFP8 entry points take d = 128 only.
 */
int attn_fwd_fp8qk(const void* q8, const void* k8, const void* v, void* o, float* lse,
                   int B, int H, int Nq, int Nk, int d, float scale, float q_descale, float k_descale,
                   void* stream);

/*
 * attn_fwd_fp8 -- attention forward with both products in 8-bit floating point.
 *
 * As attn_fwd_fp8qk, and V arrives as E4M3 codes too, with its own positive descale factor:
 *
 *     O = v_descale * (P8 V8) / l,   P8 = the weights p_j rounded to E4M3,
 *
 * where l sums the unrounded weights (plus the rounding error of each tile's largest one),
 * so the LSE is exactly that of attn_fwd_fp8qk. Rounding P to E4M3 (3 mantissa bits;
 * weights below 2^-6 of the running maximum lose precision, below 2^-10 they vanish) is
 * the price of the FP8 P V product: O is close to the definition only to within a few
 * 1e-2 on N(0,1) inputs and about 1e-1 on sharply peaked rows, versus 1e-2 for the BF16
 * path.
 *
 *   vt8    device, V^T as E4M3 codes: [B, H, d, ldv] bytes, keys innermost; key j of row c
 *          of head (b, h) at vt8[((b * H + h) * d + c) * ldv + j]. Bytes from Nk to ldv of
 *          each row are not read.
 *   ldv    row stride of vt8 in bytes: ldv >= Nk (else ATTN_ERR_INVALID_ARG), a multiple
 *          of 16 (else ATTN_ERR_MISALIGNED); the tensor cores read V with keys contiguous
 *   v_descale   finite and > 0 (else ATTN_ERR_INVALID_ARG)
 *
 * Everything else (q8, k8, their descale factors, o, lse, sizes, alignment, work split,
 * workspace, return values) is as attn_fwd_fp8qk.
 */
int attn_fwd_fp8(const void* q8, const void* k8, const void* vt8, long long ldv, void* o, float* lse,
                 int B, int H, int Nq, int Nk, int d, float scale, float q_descale, float k_descale,
                 float v_descale, void* stream);

/*
 * attn_fwd_fp8qk_causal, attn_fwd_fp8_causal -- attn_fwd_fp8qk and attn_fwd_fp8 under the
 * causal mask of attn_fwd_causal (query i sees keys 0 .. i + Nk - Nq).
 *
 * Arguments, layouts, accuracy and return values are those of the FP8 entry point of the
 * same name, plus attn_fwd_causal's rules: Nq <= Nk is required (Nq > Nk returns
 * ATTN_ERR_INVALID_ARG without touching the GPU), lse sums over the visible keys only, and
 * the call allocates nothing (whole 256-row groups per block, longest first). d = 128.
 */
int attn_fwd_fp8qk_causal(const void* q8, const void* k8, const void* v, void* o, float* lse,
                          int B, int H, int Nq, int Nk, int d, float scale, float q_descale,
                          float k_descale, void* stream);
int attn_fwd_fp8_causal(const void* q8, const void* k8, const void* vt8, long long ldv, void* o,
                        float* lse, int B, int H, int Nq, int Nk, int d, float scale, float q_descale,
                        float k_descale, float v_descale, void* stream);

/*
 * attn_fwd_fp8qk_bias, attn_fwd_fp8_bias -- the two FP8 entry points with attn_fwd_bias's
 * additive bias: S = scale * q_descale * k_descale * (Q8 K8^T) + B, the bias added after the
 * scale as in attn_fwd_bias (the definition's optional B, "FlashAttention'ı Anlamak Bölüm 1",
 * section 0.2 Notasyon). Arguments, layouts, accuracy and return values are those of
 * attn_fwd_fp8qk / attn_fwd_fp8, with bias and its three strides as in attn_fwd_bias (and its
 * argument checks). Not with the causal mask (a causal bias carries one).
 */
int attn_fwd_fp8qk_bias(const void* q8, const void* k8, const void* v, const void* bias,
                        long long bias_stride_b, long long bias_stride_h, long long bias_stride_q,
                        void* o, float* lse, int B, int H, int Nq, int Nk, int d, float scale,
                        float q_descale, float k_descale, void* stream);
int attn_fwd_fp8_bias(const void* q8, const void* k8, const void* vt8, long long ldv, const void* bias,
                      long long bias_stride_b, long long bias_stride_h, long long bias_stride_q,
                      void* o, float* lse, int B, int H, int Nq, int Nk, int d, float scale,
                      float q_descale, float k_descale, float v_descale, void* stream);

/*
 * attn_fwd_mxfp8 -- attention forward from MXFP8 inputs, both products block-scaled.
 *
 * The "MXFP8 MMA" that "Flash Attention на 5090 в CUDA C++" (section "Что дальше") names as
 * the next step: each input is given as OCP microscaling FP8, E4M3 codes (the format of
 * attn_fwd_fp8qk) with one E8M0 scale 2^(e - 127) per block of 32 elements along the
 * dimension its product contracts over: along d for Q and K, along the keys for V. So
 *
 *     S = scale * Q K^T,   Q[i][c] = 2^(sq[i][c/32] - 127) * E4M3(q8[i][c]),   likewise K,
 *     O = P V,   V[j][c] = 2^(svt[c][j/32] - 127) * E4M3(vt8[c][j]),
 *
 * and the tensor cores apply every scale (kind::mxf8f6f4 with scale factors in tensor
 * memory). P is rounded to E4M3 with a block scale of 2^0 for the P V product, so O carries
 * the E4M3 rounding of P described under attn_fwd_fp8; the row sums, and so the LSE, use the
 * unrounded weights.
 *
 *   q8, k8  device, [B, H, Nq|Nk, d] bytes (E4M3 codes), 16-byte aligned
 *   sq, sk  device, [B, H, Nq|Nk, d/32] bytes (E8M0 scales), 4-byte aligned
 *   vt8     device, V^T as E4M3 codes, [B, H, d, ldv] bytes, keys innermost; ldv >= Nk, a
 *           multiple of 16; bytes from Nk on are not used
 *   svt     device, V^T's scales, [B, H, d, ldsv] bytes: byte t of row c scales keys
 *           32t .. 32t+31 of column c; ldsv a multiple of 16 and at least 4 * ceil(Nk/128)
 *           (whole 128-key tiles are read; bytes past ceil(Nk/32) are read and replaced by
 *           2^0); 4-byte aligned
 *
 * d must be 128. A scale byte of 255 (NaN in E8M0) gives unspecified results for the rows it
 * reaches. Returns ATTN_ERR_INVALID_ARG for a null pointer, ldv < Nk or ldsv too short,
 * ATTN_ERR_MISALIGNED for the alignment rules above; everything else (o, lse, the work split,
 * workspace, return values) as attn_fwd.
 */
int attn_fwd_mxfp8(const void* q8, const void* sq, const void* k8, const void* sk, const void* vt8, long long ldv,
                   const void* svt, long long ldsv, void* o, float* lse, int B, int H, int Nq, int Nk, int d,
                   float scale, void* stream);

/*
 * attn_fwd_mxfp8_causal -- attn_fwd_mxfp8 under the causal mask of attn_fwd_causal (query i
 * sees keys 0 .. i + Nk - Nq). Arguments, layouts, accuracy and return values are those of
 * attn_fwd_mxfp8, plus attn_fwd_causal's rules (Nq <= Nk, LSE over the visible keys only, no
 * allocation).
 */
int attn_fwd_mxfp8_causal(const void* q8, const void* sq, const void* k8, const void* sk, const void* vt8,
                          long long ldv, const void* svt, long long ldsv, void* o, float* lse, int B, int H,
                          int Nq, int Nk, int d, float scale, void* stream);

/*
 * attn_fwd_o32 -- attn_fwd with O written in FP32, before its rounding to BF16.
 *
 * A diagnostic of the computation itself. The notes state that the tiled computation
 * reaches exact attention, not an approximation ("FlashAttention'ı Anlamak Bölüm 1",
 * section 0.1): its only errors are rounding. With a BF16 output, half a BF16 ulp of O
 * (up to 1/64 for |O| in [4, 8)) can exceed an error bound of 1e-2 by itself, so a test
 * of the kernel's own arithmetic against such a bound needs O before that last rounding.
 * This call runs the same kernel code as attn_fwd (same tiles, same online softmax,
 * same work split and merge) and differs only in the store of O.
 *
 *   o32  device, FP32 [B, H, Nq, d], written; 16-byte aligned (else ATTN_ERR_MISALIGNED).
 *        attn_fwd's o is this array rounded to nearest-even BF16.
 *
 * Everything else (q, k, v, lse, sizes, scale, workspace, return values) is as attn_fwd.
 */
int attn_fwd_o32(const void* q, const void* k, const void* v, float* o32, float* lse,
                 int B, int H, int Nq, int Nk, int d, float scale, void* stream);

/*
 * attn_fwd_noalloc -- attn_fwd for callers that cannot allocate device memory.
 *
 * There is no counterpart on the pages: this is a service of the library. Some callers
 * must not allocate once they are running: applications that budget all of the GPU's
 * memory up front (an extra allocation could fail or evict something else), loops where
 * an allocation may synchronise the device, and programs whose own allocator owns every
 * byte of device memory. attn_fwd may allocate a workspace (see the conventions above);
 * this entry point never calls cudaMalloc, cudaMallocAsync, cudaFree or any allocating
 * routine. It computes the same result with the same kernel, keeping the workspace for
 * split work in a fixed 48 MiB array inside the library, which every GPU that loads the
 * library holds until the process exits.
 *
 * Arguments, layouts and return values are those of attn_fwd, plus:
 *   - ATTN_ERR_UNSUPPORTED when the call would need more than the fixed 48 MiB (only on
 *     a device with more than 186 SMs).
 *   - d = 192 and 256 run attn_fwd's one-query-tile kernel, which splits no work and
 *     uses no workspace: the array below is not touched.
 *   - The first call in each CUDA context (on each device, and again after
 *     cudaDeviceReset or in another context made current by the caller) looks up the
 *     array's device address (cudaGetSymbolAddress, which allocates nothing) with that
 *     context current; make that first call before any stream capture on the device.
 *   - Every call on a device uses the same array, which keeps the previous call's
 *     contents; each call clears the part that must start at zero on its own stream.
 *     Calls whose kernels overlap on the GPU (different streams, no ordering between
 *     them) race on the array and may return wrong results: order them.
 */
int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int Nq, int Nk, int d, float scale, void* stream);

/*
 * attn_fwd_status -- synchronises `stream`, then reads and clears the device status
 * word that kernels of this library set when a pipeline wait runs past its time
 * limit (every wait inside the kernel is bounded; on expiry the block stops its work,
 * waits for its own copies and matrix operations in flight, frees its tensor memory
 * and exits, leaving o and lse undefined). The word is per device and shared by all
 * calls on that device since the last attn_fwd_status.
 *
 * Returns ATTN_OK, ATTN_ERR_TIMEOUT, or ATTN_ERR_CUDA if synchronising failed.
 * No counterpart on the pages: this is the library's error channel.
 */
int attn_fwd_status(void* stream);

/*
 * attn_status_string -- a static, human-readable name for a status code.
 */
const char* attn_status_string(int status);

/*
 * attn_fwd_set_wait_limit -- test hook for the failure path. Sets, process-wide and for
 * launches enqueued after the call, the time limit of every in-kernel wait in SM clock
 * cycles (0 restores the default of 2^31 cycles, about one second) and whether launches
 * withhold one K/V tile load (withhold_tile != 0; at d = 192 and 256 the first V unit of
 * each block), so that the consumer's wait for it runs out and the kernel takes its
 * timeout exit. No GPU fault is involved: the kernel
 * returns normally and attn_fwd_status reports ATTN_ERR_TIMEOUT. Returns ATTN_OK.
 * No counterpart on the pages.
 */
int attn_fwd_set_wait_limit(unsigned long long cycles, int withhold_tile);

/*
 * attn_fwd_kernel_count -- number of kernel launches this library has made in this
 * process (all devices), for launch accounting by callers.
 */
unsigned long long attn_fwd_kernel_count(void);

/*
 * attn_fwd_plan -- the work plan attn_fwd would use for n_groups groups (B*H*ceil(Nq/256)) of
 * n_kv key steps (ceil(Nk/128)) on sms SMs, for inspection (host only, no device call):
 * dp_groups groups processed whole, then the split region's key steps cut into grid shares,
 * block c taking steps [cuts[c], cuts[c+1]); cuts must hold 161 values (unused ones are 0);
 * has_split is 1 when a share boundary falls inside a group. Returns ATTN_OK, or
 * ATTN_ERR_INVALID_ARG for a null pointer or a count below 1.
 */
int attn_fwd_plan(long long n_groups, int n_kv, int sms, long long* dp_groups, long long* cuts, int* grid,
                  int* has_split);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_H */
