// attn_wide.h -- internal interface between the C ABI (attn_fwd.cu) and the forward kernel
// for head dimensions above 128 (attn_fwd_wide.cu). Not part of the public headers.
#pragma once

#include <cuda_runtime.h>

namespace attn_wide {

// Head dimensions this kernel serves.
constexpr bool supported(int d) { return d == 192 || d == 256; }

// An additive bias as attn_fwd_bias takes it (BF16, element strides, already validated:
// 16-byte aligned base, strides multiples of 8, offsets within 64 bits).
struct Bias {
  const void* ptr;
  long long sb, sh, sq;
};

// O = softmax(scale Q K^T) V and the natural-log LSE for BF16 [B, H, N, d] tensors, d in
// {192, 256}; arguments as attn_fwd (already validated by the caller: non-null, 16-byte
// aligned, B*H, Nq, Nk >= 1, finite scale). causal: query i sees keys 0 .. i + Nk - Nq only
// (the caller has checked Nq <= Nk). wait_limit: clock64 budget of each of the kernel's
// waits. bias (or null): S = scale Q K^T + B as attn_fwd_bias (not with causal). f8 >= 1: q
// and k hold FP8 E4M3 codes [B, H, N, d] (one byte each), Q K^T runs on kind::f8f6f4 and
// `scale` already includes both descale factors. f8 == 2: v holds V^T as E4M3 codes
// [B, H, d, ldv] (keys innermost, ldv >= Nk a multiple of 16, checked by the caller), P is
// rounded to E4M3 for a kind::f8f6f4 P V and O is scaled by v_scale. withhold (a test
// hook): each block skips the load of its first V unit, so that the wait for it runs out
// and the launch takes its timeout exit. Returns an attn_status code; ATTN_OK once the
// kernel is enqueued.
int forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
            int d, float scale, bool causal, cudaStream_t stream, unsigned long long wait_limit,
            const Bias* bias = nullptr, int f8 = 0, long long ldv = 0, float v_scale = 1.0f, int withhold = 0);

// Reads and clears the kernel's device status word on `stream` (synchronising it): 1 if a
// wait of a launch gave up since the last call, 0 if not, negative on a CUDA error.
int take_status(cudaStream_t stream);

}  // namespace attn_wide
