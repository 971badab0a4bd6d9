// attn_bwd.cu -- dense BF16 attention backward for GB300 (sm_103a).
//
// Gradients of O = softmax(scale * Q K^T) V for an upstream gradient dO, head_dim 128,
// with P recomputed from the forward's log-sum-exp ("FlashAttention'ı Anlamak Bölüm 1",
// section 0 Giriş: recomputation instead of storing S or P):
//
//   D_i = dO_i . O_i,  P = 2^(s * scale * log2 e - LSE_i * log2 e),  dP = dO V^T,
//   dS = P * (dP - D),  dV = P^T dO,  dK = scale * dS^T Q,  dQ = scale * dS K.
//
// attn_bwd_causal: the gradient of the causal forward (query i sees keys 0 .. i + Nk - Nq):
// a dK/dV block starts at the first query tile whose rows see its first key, a dQ block
// stops at the key tile of its last row's diagonal, and the tiles that cross the
// diagonal mask P (hence dS) to zero past it.
//
// Three kernels, all on the caller's stream:
//
//   bwd_rows_kernel  one warp per query row: -D_i and -LSE_i * log2 e, written planar per
//                    128-row tile into a workspace padded to whole tiles (pad rows get
//                    -LSE = -inf, -D = -0, so their P is exactly 0).
//   bwd_dkdv_kernel  one block per (b, h, 128-key tile). K and V are loaded once; then per
//                    128-query tile j (Q_j, dO_j and the tile's row values by TMA, in
//                    rings): S^T = K Q_j^T and dP^T = V dO_j^T on tcgen05 into TMEM; the
//                    compute warps (thread = key) form P^T and write it back over S^T as
//                    BF16 pairs, then dS^T over dP^T; dV += P^T dO_j and dK += dS^T Q_j take
//                    them straight from TMEM (the A operand) with dO_j and Q_j as MN-major B
//                    operands. The MMA thread issues the next tile's S^T as soon as P^T has
//                    been handed over (its columns are then free) and the next dP^T after
//                    dK, so the tensor cores compute tile j+1's scores while the compute
//                    warps work on tile j's dS^T.
//   bwd_dq_kernel    one block per (b, h, 128-query tile). Q and dO are loaded once; per
//                    key tile j (double-buffered K_j, V_j): S = Q K_j^T, dP = dO V_j^T; the
//                    compute warps (thread = query) form dS and write it over S; then
//                    dQ += dS K_j. S is double-buffered in TMEM, so the next tile's S and
//                    dP run on the tensor cores while the compute warps work on this one.
//
// TMEM: dK/dV block: S^T | dP^T | dV | dK (4 x 128 columns); dQ block: S0 | dP | dQ | S1.
// Warp roles: warp 0 lane 0 issues TMA, warp 1 lane 0 issues MMAs (and owns TMEM),
// warps 4-11 compute in two groups: group g (warps 4 + 4g ..) takes score columns
// 64g .. 64g + 63, warp 4 + 4g + q the TMEM lanes 32q .. 32q + 31. Each group writes its
// packed BF16 half over the first 32 of its own 64 columns, so the groups never touch
// each other's columns, and hands it to the MMA thread at once, which runs that half of
// the accumulating products while the other group finishes. Ragged tails are
// zero-filled by TMA and masked. Every mbarrier wait is bounded: on
// expiry the block raises an abort flag, sets the status word and winds down.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "attn_bwd.h"
#include "tc_sm103.cuh"

namespace {

constexpr int kD = 128;
constexpr int kT = 128;                         // rows of a tile (queries or keys)
constexpr int kTileBytes = kT * kD * 2;         // 32 KB of BF16
constexpr int kBoxBytes = kTileBytes / 2;       // one TMA box: 64 columns (128 B) x 128 rows
constexpr int kThreads = 384;                   // warps 0-3 control, 4-11 compute
constexpr int kTmemCols = 512;
constexpr int kStageWarpBytes = 32 * 64 * 2;    // epilogue staging per compute warp
constexpr unsigned long long kDefaultWaitLimit = 1ull << 31;
constexpr float kLog2e = 1.4426950408889634f;

// Both main kernels hold two fixed tiles and stream two tiles per step through two rings.
// The step's first operand (Q_j in the dK/dV block, K_j in the dQ block) is read by a score
// product and again by the step's last product (dK += dS^T Q_j, dQ += dS K_j); the second
// (dO_j, V_j) only by products early in the step. The first ring has three slots, the
// second two: both request every tile more than a step before its first product needs it.
// In the dK/dV block the query rows' (-LSE, -D) travel with dO_j. The compute warps free the
// slots there: each of them, on seeing S^T_{j+1} complete (hence dV_j, the last reader of
// dO_j), has also finished its own work on tile j's rows, and frees dO_j's slot with one
// arrival of eight; one of them, on seeing dP^T_{j+1} complete (hence dK_j), frees Q_j's.
// Seven 32 KB tiles and the rows fill the dK/dV block's shared memory, with no room to
// realign its base: that kernel declares it 1024-aligned (the 128-byte swizzle's atom) and
// checks the alignment before touching it. The dQ block has no rows: its barriers follow
// the tiles, and it realigns its base itself.
constexpr int kSlotsA = 3, kSlotsB = 2;
constexpr int kRowsBytes = kT * 8;                             // a query tile's 128 (-LSE log2 e) and 128 (-D)
constexpr int kOffFixed0 = 0;                                  // K (dK/dV block) or Q (dQ block)
constexpr int kOffFixed1 = kTileBytes;                         // V or dO
constexpr int kOffRingA = 2 * kTileBytes;                      // Q_j or K_j
constexpr int kOffRingB = kOffRingA + kSlotsA * kTileBytes;    // dO_j or V_j
constexpr int kOffRows = kOffRingB + kSlotsB * kTileBytes;     // dK/dV block: rows of dO_j's tile
constexpr int kOffBar = kOffRows + kSlotsB * kRowsBytes;      // dK/dV block
constexpr int kOffBarQ = kOffRows;                             // dQ block

// barriers (both kernels)
constexpr int kBarFixed = 0;        // the block's fixed tiles (K, V or Q, dO) have landed
constexpr int kBarFullA = 1;        // [3] ring A slot landed
constexpr int kBarEmptyA = 4;       // [3] ring A slot read by its last product
constexpr int kBarFullB = 7;        // [2] ring B slot landed
constexpr int kBarEmptyB = 9;       // [2] ring B slot read by its product (dK/dV block: and its rows)
constexpr int kBarSdP = 11;         // S and dP complete in TMEM (dK/dV block: S^T alone)
// hand-overs from the compute warps (one arrival per compute warp)
constexpr int kBarPAll = 12;        // dK/dV block: P^T is in TMEM
constexpr int kBarDSAll = 13;       // dK/dV block: dS^T is in TMEM
constexpr int kBarDS = 12;          // dQ block: [step parity] dS is in TMEM (steps alternate
                                    // between two barriers: the compute warps may finish step
                                    // j + 1 before the MMA thread waits for step j)
constexpr int kBarAcc = 14;         // accumulators complete
constexpr int kBarDPFree = 15;      // dQ block: every compute warp holds dP of the step in registers
constexpr int kBarDPReady = 16;     // dK/dV block: dP^T complete in TMEM
constexpr int kNumBars = 17;
constexpr int kFlagsBytes = kNumBars * 8 + 16;   // barriers, TMEM slot, abort flag

constexpr int kSmemKV = kOffBar + kFlagsBytes;
constexpr int kSmemQ = kOffBarQ + kFlagsBytes + 1024;   // + realignment of the base
static_assert(kTileBytes % 1024 == 0, "tiles need 1024-byte alignment");
static_assert(kSmemKV <= 232448 && kSmemQ <= 232448, "exceeds the 227 KB shared memory of one block");
static_assert(8 * kStageWarpBytes <= kTileBytes, "epilogue staging reuses one tile");

__device__ unsigned int g_bwd_status;   // bit 0: a wait timed out; bit 1: shared memory misaligned

// ---------------------------------------------------------------------------------
// PTX wrappers. The ones every kernel of the library uses (mbarrier, TMA tile loads,
// tcgen05.mma / commit / fences, ex2, max3, BF16 packing, the shared-memory descriptor)
// are in tc_sm103.cuh; this file's own follow.
// ---------------------------------------------------------------------------------
using tc::ex2;
using tc::mbar_arrive;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_try_wait;
using tc::mma_ss;
using tc::mma_ts;
using tc::pack_bf16;
using tc::sdesc_sw128;
using tc::smem_u32;
using tc::tc_commit;
using tc::tc_fence_after;
using tc::tc_fence_before;
using tc::tma_load_3d;

// contiguous global -> shared copy (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&x)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]),
        "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15]),
        "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]),
        "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&x)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]), "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15]), "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]), "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31]), "=r"(x[32]), "=r"(x[33]), "=r"(x[34]), "=r"(x[35]), "=r"(x[36]), "=r"(x[37]), "=r"(x[38]), "=r"(x[39]), "=r"(x[40]), "=r"(x[41]), "=r"(x[42]), "=r"(x[43]), "=r"(x[44]), "=r"(x[45]), "=r"(x[46]), "=r"(x[47]), "=r"(x[48]), "=r"(x[49]), "=r"(x[50]), "=r"(x[51]), "=r"(x[52]), "=r"(x[53]), "=r"(x[54]), "=r"(x[55]), "=r"(x[56]), "=r"(x[57]), "=r"(x[58]), "=r"(x[59]), "=r"(x[60]), "=r"(x[61]), "=r"(x[62]), "=r"(x[63])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&x)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]), "r"(x[8]), "r"(x[9]), "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]), "r"(x[15]), "r"(x[16]), "r"(x[17]), "r"(x[18]), "r"(x[19]), "r"(x[20]), "r"(x[21]), "r"(x[22]), "r"(x[23]), "r"(x[24]), "r"(x[25]), "r"(x[26]), "r"(x[27]), "r"(x[28]), "r"(x[29]), "r"(x[30]), "r"(x[31])
      : "memory");
}
// Packed FP32x2 arithmetic: each lane of the pair is rounded exactly as the scalar
// operation would round it (fma / add / mul, round to nearest, no flush of denormals).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {   // a * b + c
  float2 d;
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 f2(uint32_t lo, uint32_t hi) { return make_float2(__uint_as_float(lo), __uint_as_float(hi)); }

// BF16 x BF16 -> FP32, M = N = 128, A K-major, B K-major or MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16(bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(kT >> 3) << 17) |
         (static_cast<uint32_t>(kT >> 4) << 24);
}
// D = A B^T over d = 128 with both tiles row-major [128][d] in smem (two 64-column
// boxes each, 128B swizzle): S^T = K Q^T, dP^T = V dO^T, S = Q K^T, dP = dO V^T.
__device__ __forceinline__ void mma_rows_by_rows(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
  constexpr uint32_t idesc = idesc_bf16(false);
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>((kk >> 2) * kBoxBytes + (kk & 3) * 32);
    mma_ss(d_tmem, sdesc_sw128(a_smem + off, 16, 1024), sdesc_sw128(b_smem + off, 16, 1024), idesc, kk > 0);
  }
}
// D (+)= A B over K = 64h .. 64h + 63 (one half of K = 128) with A in TMEM as packed BF16
// pairs (8 columns per 16 of K, the half's 32 columns starting at a_half) and B a
// row-major [128][d] tile in smem (K along rows: MN-major): dV += P^T dO, dK += dS^T Q,
// dQ += dS K.
__device__ __forceinline__ void mma_tmem_by_rows_half(uint32_t d_tmem, uint32_t a_half, uint32_t b_smem, int h,
                                                      bool acc) {
  constexpr uint32_t idesc = idesc_bf16(true);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ts(d_tmem, a_half + kk * 8, sdesc_sw128(b_smem + (4 * h + kk) * 16 * 128, kBoxBytes, 1024), idesc,
           acc || kk > 0);
}

// ---------------------------------------------------------------------------------
// Bounded waits
// ---------------------------------------------------------------------------------
struct Ctl {
  uint32_t bars;
  volatile uint32_t* abort;
  unsigned long long limit;
  __device__ __forceinline__ uint32_t bar(int i) const { return bars + 8u * static_cast<uint32_t>(i); }
};
__device__ __forceinline__ bool wait_phase(const Ctl& c, int idx, uint32_t parity, bool watch_abort) {
  const uint32_t b = c.bar(idx);
  if (mbar_try_wait(b, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(b, parity)) return true;
    if (watch_abort && *c.abort) return false;
    if (static_cast<unsigned long long>(clock64() - t0) > c.limit) {
      *c.abort = 1u;
      atomicOr(&g_bwd_status, 1u);
      return false;
    }
  }
}
// warp-uniform result (the callers' next step is a .sync.aligned TMEM access)
__device__ __forceinline__ bool wait_warp(const Ctl& c, int idx, uint32_t parity) {
  const bool ok = wait_phase(c, idx, parity, true);
  return __all_sync(0xffffffffu, ok);
}

struct BwdParams {
  uint16_t* dq;
  uint16_t* dk;
  uint16_t* dv;
  // [BH, q_pad / 128, 2, 128]: per 128-row query tile, -LSE * log2 e of its rows, then -D
  const float* rows;
  int Nq, Nk, q_tiles, k_tiles, q_pad;
  int causal;   // query i sees keys 0 .. i + off only (off = Nk - Nq >= 0)
  int off;
  int withhold;   // test hook: the dK/dV producer stops before its second query tile
  float scale, scale_log2;
  unsigned long long wait_limit;
  // attn_bwd_bias: the forward's additive bias, B_ij of head (b, h) = bias[b * bias_sb + h * bias_sh
  // + i * bias_sq + j] (BF16, strides in elements), H heads per batch
  const uint16_t* bias;
  long long bias_sb, bias_sh, bias_sq;
  int H;
};

// The bias of head bh at query row `row` (nullptr-free: callers check the ranges).
__device__ __forceinline__ const uint16_t* bias_row(const BwdParams& p, int bh, int row) {
  return p.bias + static_cast<long long>(bh / p.H) * p.bias_sb + static_cast<long long>(bh % p.H) * p.bias_sh +
         static_cast<long long>(row) * p.bias_sq;
}

// Stores one 64-column half of this warp's 32 rows (pk: the thread's own row, packed
// BF16 pairs) through the warp's staging tile so that each global store instruction
// covers four whole 128-byte lines. Rows from valid_rows on are not stored.
__device__ __forceinline__ void store_half_rows(uint8_t* stage, const uint32_t (&pk)[32], uint16_t* row0,
                                                int valid_rows, int half) {
  const int lane = threadIdx.x & 31;
  uint4* st = reinterpret_cast<uint4*>(stage);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    st[lane * 8 + (k ^ (lane & 7))] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = i * 4 + (lane >> 3), cc = lane & 7;
    const uint4 v = st[rr * 8 + (cc ^ (rr & 7))];
    if (rr < valid_rows) reinterpret_cast<uint4*>(row0 + static_cast<size_t>(rr) * kD + half * 64)[cc] = v;
  }
  __syncwarp();
}

// Writes columns 64h .. 64h + 63 of this thread's accumulator row (FP32 TMEM columns at
// t_acc) times `mul` as BF16 to the warp's 32 rows starting at row0.
__device__ __forceinline__ void store_acc_half(uint32_t t_acc, int h, float mul, uint8_t* stage, uint16_t* row0,
                                               int valid_rows) {
  uint32_t pk[32];
#pragma unroll
  for (int c2 = 0; c2 < 2; ++c2) {
    uint32_t x[32];
    tmem_ld32(t_acc + h * 64 + c2 * 32, x);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[c2 * 16 + i] = pack_bf16(__uint_as_float(x[2 * i]) * mul, __uint_as_float(x[2 * i + 1]) * mul);
  }
  store_half_rows(stage, pk, row0, valid_rows, h);
}

// Block setup shared by both kernels: barrier init, TMEM allocation. Returns the TMEM base.
__device__ __forceinline__ uint32_t block_setup(const Ctl& c, uint8_t* flags, uint32_t flags_u32, int warp,
                                                bool dkdv) {
  if (threadIdx.x == 0) {
    for (int b = kBarFixed; b <= kBarSdP; ++b) mbar_init(c.bar(b), 1);   // fixed tiles, rings, S
    // one arrival per compute warp
    if (dkdv)
      for (int b = 0; b < kSlotsB; ++b) mbar_init(c.bar(kBarEmptyB + b), 8);
    mbar_init(c.bar(kBarPAll), 8);
    mbar_init(c.bar(kBarDSAll), 8);
    mbar_init(c.bar(kBarAcc), 1);
    mbar_init(c.bar(kBarDPFree), 8);    // one arrival per compute warp
    mbar_init(c.bar(kBarDPReady), 1);
    *c.abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(flags_u32 + kNumBars * 8),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return *reinterpret_cast<volatile uint32_t*>(flags + kNumBars * 8);
}

__device__ __forceinline__ void block_teardown(uint32_t tmem, int warp) {
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------------
// Row pass: -LSE_i log2 e and -D_i (D_i = dO_i . O_i) per query row, stored planar per
// 128-row tile (the tile's 128 values of -LSE log2 e, then its 128 of -D), so the dK/dV
// block reads four consecutive query columns with one shared-memory load. Both are kept
// negated so that the kernels add them: s * c + (-LSE) and dP + (-D) round exactly as
// s * c - LSE and dP - D. Pad rows: (-inf, -0), so their P is exactly 0.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) bwd_rows_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                                       const float* __restrict__ lse, float* __restrict__ rows,
                                                       long long bh_count, int Nq, int q_pad) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= bh_count * q_pad) return;
  const long long bh = row / q_pad;
  const int i = static_cast<int>(row - bh * q_pad);
  float* nl = rows + 2 * row - (i & (kT - 1));   // the tile's first float is 2 * (row - i % 128)
  if (i >= Nq) {
    if (lane == 0) {
      nl[0] = -INFINITY;
      nl[kT] = -0.0f;
    }
    return;
  }
  const size_t base = (static_cast<size_t>(bh) * Nq + i) * kD + lane * 4;
  const uint2 a = *reinterpret_cast<const uint2*>(o + base);
  const uint2 b = *reinterpret_cast<const uint2*>(dout + base);
  float acc = __uint_as_float(a.x << 16) * __uint_as_float(b.x << 16) +
              __uint_as_float(a.x & 0xffff0000u) * __uint_as_float(b.x & 0xffff0000u) +
              __uint_as_float(a.y << 16) * __uint_as_float(b.y << 16) +
              __uint_as_float(a.y & 0xffff0000u) * __uint_as_float(b.y & 0xffff0000u);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    nl[0] = -(lse[static_cast<size_t>(bh) * Nq + i] * kLog2e);
    nl[kT] = -acc;
  }
}

// ---------------------------------------------------------------------------------
// dK / dV: one block per (b, h, key tile)
// ---------------------------------------------------------------------------------
template <bool kCausal, bool kBias>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const BwdParams p) {
  // With a bias the Q ring keeps two of its three slots: the third holds each compute warp's
  // 4 KB bias staging tile (below).
  constexpr int kSlotsQ = kBias ? 2 : kSlotsA;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = smem_u32(smem);
  if (base & 1023u) {   // every thread leaves before any barrier, copy or TMEM allocation
    if (threadIdx.x == 0) atomicOr(&g_bwd_status, 2u);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x % p.k_tiles;
  const int bh = blockIdx.x / p.k_tiles;
  Ctl c;
  c.bars = base + kOffBar;
  c.abort = reinterpret_cast<volatile uint32_t*>(smem + kOffBar + kNumBars * 8 + 4);
  c.limit = p.wait_limit;
  const uint32_t tmem = block_setup(c, smem + kOffBar, base + kOffBar, warp, true);
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
  const uint32_t sK = base + kOffFixed0, sV = base + kOffFixed1;
  // query tiles q0 .. q_tiles - 1; causal: from the first tile whose rows see this tile's
  // first key (query i sees key r when i >= r - off). Step t of the loops is tile q0 + t.
  int q0 = 0;
  if (kCausal) {
    const int first_row = kt * kT - p.off;
    q0 = first_row > 0 ? first_row / kT : 0;
  }
  const int nq = p.q_tiles - q0;
  auto sQ = [&](int j) { return base + kOffRingA + (j % kSlotsQ) * kTileBytes; };
  auto sDO = [&](int j) { return base + kOffRingB + (j % kSlotsB) * kTileBytes; };

  if (warp == 0) {
    if (lane == 0) {
      // K and V of this tile, then per query tile Q_j, and dO_j with the rows' (LSE, D)
      mbar_arrive_expect_tx(c.bar(kBarFixed), 2 * kTileBytes);
      for (int h = 0; h < 2; ++h) {
        tma_load_3d(sK + h * kBoxBytes, &tmK, c.bar(kBarFixed), h * 64, kt * kT, bh);
        tma_load_3d(sV + h * kBoxBytes, &tmV, c.bar(kBarFixed), h * 64, kt * kT, bh);
      }
      int issued = 0;   // query tiles whose Q and dO were both requested
      for (int j = 0; j < nq; ++j, ++issued) {
        const int a = j % kSlotsQ, b = j % kSlotsB;
        if (j >= kSlotsQ && !wait_phase(c, kBarEmptyA + a, (j / kSlotsQ - 1) & 1, true)) break;
        if (p.withhold && j == 1) break;   // test hook: the consumers' waits for this tile run out
        mbar_arrive_expect_tx(c.bar(kBarFullA + a), kTileBytes);
        for (int h = 0; h < 2; ++h) tma_load_3d(sQ(j) + h * kBoxBytes, &tmQ, c.bar(kBarFullA + a), h * 64, (q0 + j) * kT, bh);
        // dO_j's slot held dO_{j-2} and its rows
        if (j >= kSlotsB && !wait_phase(c, kBarEmptyB + b, (j / kSlotsB - 1) & 1, true)) {
          wait_phase(c, kBarFullA + a, (j / kSlotsQ) & 1, false);   // that Q copy is in flight
          break;
        }
        mbar_arrive_expect_tx(c.bar(kBarFullB + b), kTileBytes + kRowsBytes);
        for (int h = 0; h < 2; ++h) tma_load_3d(sDO(j) + h * kBoxBytes, &tmDO, c.bar(kBarFullB + b), h * 64, (q0 + j) * kT, bh);
        bulk_load(base + kOffRows + b * kRowsBytes,
                  p.rows + 2 * (static_cast<size_t>(bh) * p.q_pad + static_cast<size_t>(q0 + j) * kT), kRowsBytes,
                  c.bar(kBarFullB + b));
      }
      // no copy into shared memory may be in flight when the block exits
      wait_phase(c, kBarFixed, 0, false);
      for (int j = issued - kSlotsQ < 0 ? 0 : issued - kSlotsQ; j < issued; ++j)
        wait_phase(c, kBarFullA + j % kSlotsQ, (j / kSlotsQ) & 1, false);
      for (int j = issued - kSlotsB < 0 ? 0 : issued - kSlotsB; j < issued; ++j)
        wait_phase(c, kBarFullB + j % kSlotsB, (j / kSlotsB) & 1, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // Per query tile j: dV += P^T dO_j once the compute warps have handed P^T over, then
      // S^T of tile j+1 into the columns P^T leaves (the compute warps hold S^T_j in
      // registers by then), then dK += dS^T Q_j once dS^T is handed over, then dP^T of tile
      // j+1 into the columns dS^T leaves. The next tile's scores thus run on the tensor cores
      // while the compute warps work on this tile's dS^T, and its dP^T while they compute
      // its P^T. Per step this thread waits twice and commits twice: every other operation
      // of it idles the tensor core (the MMA queue is shallow), so the compute warps check
      // that Q_{j+1} and dO_{j+1} have landed before their hand-overs of step j, and free
      // the ring slots themselves.
      bool ok = wait_phase(c, kBarFixed, 0, true);
      if (ok && nq > 0) ok = wait_phase(c, kBarFullA, 0, true) && wait_phase(c, kBarFullB, 0, true);
      if (ok && nq > 0) {
        tc_fence_after();
        mma_rows_by_rows(tS, sK, sQ(0));                                  // S^T = K Q_0^T
        tc_commit(c.bar(kBarSdP));
        mma_rows_by_rows(tdP, sV, sDO(0));                                // dP^T = V dO_0^T
        tc_commit(c.bar(kBarDPReady));
      }
      for (int j = 0; ok && j < nq; ++j) {
        const int j1 = j + 1;
        const bool more = j1 < nq;
        if (!wait_phase(c, kBarPAll, j & 1, true)) break;
        tc_fence_after();
        for (int h = 0; h < 2; ++h)   // queries 64h .. 64h + 63
          mma_tmem_by_rows_half(tdV, tS + 64 * h, sDO(j), h, j > 0 || h > 0);     // dV += P^T dO_j
        if (more) {
          mma_rows_by_rows(tS, sK, sQ(j1));                               // S^T = K Q_{j+1}^T
          tc_commit(c.bar(kBarSdP));
        }
        if (!wait_phase(c, kBarDSAll, j & 1, true)) break;
        tc_fence_after();
        for (int h = 0; h < 2; ++h)
          mma_tmem_by_rows_half(tdK, tdP + 64 * h, sQ(j), h, j > 0 || h > 0);     // dK += dS^T Q_j
        if (more) {
          mma_rows_by_rows(tdP, sV, sDO(j1));                             // dP^T = V dO_{j+1}^T
          tc_commit(c.bar(kBarDPReady));
        }
      }
      tc_commit(c.bar(kBarAcc));   // also: every MMA this thread issued is done before TMEM is freed
      wait_phase(c, kBarAcc, 0, false);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int quarter = warp & 3;
    const int grp = (warp - 4) >> 2;   // query columns 64 grp .. 64 grp + 63
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // One thread checks, before the hand-overs of step j, that the ring tiles the MMA
    // thread reads next (Q_{j+1} after P^T, dO_{j+1} after dS^T) have landed; another frees
    // Q_j's slot once it sees dP^T_{j+1} complete.
    const bool ringer = warp == 4 && lane == 0, releaser = warp == 8 && lane == 0;
    bool ok = true;
    // Hands the step's P^T (or dS^T) over; false (warp-uniform) if the ring check gave up.
    auto hand_over = [&](int bar, int ring_bar, uint32_t ring_parity, bool check) {
      tc_fence_before();
      __syncwarp();
      bool landed = true;
      if (ringer && check) landed = wait_phase(c, ring_bar, ring_parity, true);
      landed = __shfl_sync(0xffffffffu, landed, 0);
      if (landed && lane == 0) mbar_arrive(c.bar(bar));
      __syncwarp();
      return landed;
    };
    for (int j = 0; j < nq; ++j) {
      // the rows (-LSE, -D) arrive with dO_j; S^T once its MMA is done
      const int b = j % kSlotsB;
      const int j1 = j + 1;
      const bool more = j1 < nq;
      // bias: the warp's 64 query rows x 32 keys (4 KB), requested before the waits as eight
      // 16-byte pieces per thread (load i: row 8i + lane/4, keys 8 (lane%4) .. + 7 of the
      // warp's 32; rows past Nq and keys past Nk read nothing), held as loaded until S^T is
      // in registers, then passed through the warp's staging tile so that each thread reads
      // its own key's column
      uint4 braw[kBias ? 8 : 1];
      if constexpr (kBias) {
        const int kc = kt * kT + quarter * 32 + 8 * (lane & 3);   // the piece's first key
        const int row0 = (q0 + j) * kT + 64 * grp + (lane >> 2);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int row = row0 + 8 * i;
          braw[i] = make_uint4(0u, 0u, 0u, 0u);
          if (row < p.Nq) {
            const uint16_t* src = bias_row(p, bh, row) + kc;
            if (kc + 8 <= p.Nk) {
              braw[i] = __ldg(reinterpret_cast<const uint4*>(src));
            } else {
              uint32_t w[4] = {0u, 0u, 0u, 0u};
              for (int e = 0; e < 8 && kc + e < p.Nk; ++e) w[e >> 1] |= static_cast<uint32_t>(__ldg(src + e)) << (16 * (e & 1));
              braw[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
      if (!wait_warp(c, kBarFullB + b, (j / kSlotsB) & 1) || !wait_warp(c, kBarSdP, j & 1)) {
        ok = false;
        break;
      }
      // S^T_j complete: so is dV_{j-1}, the last reader of dO_{j-1}, and this warp is done
      // with tile j-1's rows
      if (j > 0 && lane == 0) mbar_arrive(c.bar(kBarEmptyB + (j - 1) % kSlotsB));
      __syncwarp();
      tc_fence_after();
      // the tile's -LSE log2 e and -D, 128 query columns each (every lane reads the same words)
      const float* nl = reinterpret_cast<const float*>(smem + kOffRows + b * kRowsBytes) + 64 * grp;
      const float* nd = nl + kT;
      // causal: this thread's key r is seen by query columns c >= r - off - (q0 + j) * 128
      const int key = kt * kT + quarter * 32 + lane;
      const int c_lo = kCausal ? key - p.off - (q0 + j) * kT - 64 * grp : -1;   // in group columns
      const bool mask_warp = kCausal && (kt * kT + quarter * 32 + 31 - p.off - (q0 + j) * kT) > 64 * grp;
      // P^T of the group's 64 query columns, kept in registers for dS^T; written over the
      // first 32 of the group's S^T columns as BF16 pairs and handed over first
      const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
      const float2 lg2 = make_float2(1.4426950408889634f, 1.4426950408889634f);
      float pv[64];
      {
        uint32_t xs[64];
        tmem_ld64(tS + lane_off + 64 * grp, xs);
        // the bias tile: rows of 32 keys (64 bytes), row-major; thread `lane` reads column lane
        const uint16_t* bst = reinterpret_cast<const uint16_t*>(smem + kOffRingA + 2 * kTileBytes + (warp - 4) * 4096);
        if constexpr (kBias) {
          uint4* dst = reinterpret_cast<uint4*>(smem + kOffRingA + 2 * kTileBytes + (warp - 4) * 4096);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[(8 * i + (lane >> 2)) * 4 + (lane & 3)] = braw[i];
          __syncwarp();
        }
        uint32_t pw[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {   // query columns 4i .. 4i + 3 of the group
          const float4 l4 = *reinterpret_cast<const float4*>(nl + 4 * i);
          float2 n0 = make_float2(l4.x, l4.y), n1 = make_float2(l4.z, l4.w);
          if constexpr (kBias) {   // + B log2 e: the biased scores' exponent
            const uint32_t b0 = bst[(4 * i) * 32 + lane], b1 = bst[(4 * i + 1) * 32 + lane];
            const uint32_t b2 = bst[(4 * i + 2) * 32 + lane], b3 = bst[(4 * i + 3) * 32 + lane];
            n0 = ffma2(f2(b0 << 16, b1 << 16), lg2, n0);
            n1 = ffma2(f2(b2 << 16, b3 << 16), lg2, n1);
          }
          const float2 a0 = ffma2(f2(xs[4 * i], xs[4 * i + 1]), c2, n0);
          const float2 a1 = ffma2(f2(xs[4 * i + 2], xs[4 * i + 3]), c2, n1);
          float q[4] = {ex2(a0.x), ex2(a0.y), ex2(a1.x), ex2(a1.y)};
          if (mask_warp) {
#pragma unroll
            for (int t = 0; t < 4; ++t) q[t] = 4 * i + t >= c_lo ? q[t] : 0.0f;
          }
#pragma unroll
          for (int t = 0; t < 4; ++t) pv[4 * i + t] = q[t];
          pw[2 * i] = pack_bf16(q[0], q[1]);
          pw[2 * i + 1] = pack_bf16(q[2], q[3]);
        }
        tmem_st32(tS + lane_off + 64 * grp, pw);
      }
      if (!hand_over(kBarPAll, kBarFullA + j1 % kSlotsQ, (j1 / kSlotsQ) & 1, more) ||
          !wait_warp(c, kBarDPReady, j & 1)) {
        ok = false;
        break;
      }
      // dP^T_j complete: so is dK_{j-1}, the last reader of Q_{j-1}
      if (j > 0 && releaser) mbar_arrive(c.bar(kBarEmptyA + (j - 1) % kSlotsQ));
      __syncwarp();
      tc_fence_after();
      {
        // dS^T = P^T (dP^T - D), written over the first 32 of the group's dP^T columns
        uint32_t xd[64];
        tmem_ld64(tdP + lane_off + 64 * grp, xd);
        uint32_t dw[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 d4 = *reinterpret_cast<const float4*>(nd + 4 * i);
          const float2 t0 = fmul2(make_float2(pv[4 * i], pv[4 * i + 1]), fadd2(f2(xd[4 * i], xd[4 * i + 1]), make_float2(d4.x, d4.y)));
          const float2 t1 = fmul2(make_float2(pv[4 * i + 2], pv[4 * i + 3]), fadd2(f2(xd[4 * i + 2], xd[4 * i + 3]), make_float2(d4.z, d4.w)));
          dw[2 * i] = pack_bf16(t0.x, t0.y);
          dw[2 * i + 1] = pack_bf16(t1.x, t1.y);
        }
        tmem_st32(tdP + lane_off + 64 * grp, dw);
      }
      if (!hand_over(kBarDSAll, kBarFullB + j1 % kSlotsB, (j1 / kSlotsB) & 1, more)) {
        ok = false;
        break;
      }
    }
    if (ok && wait_warp(c, kBarAcc, 0)) {
      tc_fence_after();
      const int row0 = kt * kT + quarter * 32;   // the warp's first key
      const int valid = p.Nk - row0;
      uint8_t* st = smem + kOffFixed0 + (warp - 4) * kStageWarpBytes;   // K is no longer read
      const size_t off = (static_cast<size_t>(bh) * p.Nk + row0) * kD;
      store_acc_half(tdV + lane_off, grp, 1.0f, st, p.dv + off, valid);      // d columns 64 grp ..
      store_acc_half(tdK + lane_off, grp, p.scale, st, p.dk + off, valid);
    }
  }
  block_teardown(tmem, warp);
}

// ---------------------------------------------------------------------------------
// dQ: one block per (b, h, query tile)
// ---------------------------------------------------------------------------------
template <bool kCausal, bool kBias>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // causal: the longest blocks (last query tiles) are launched first
  const int qt = kCausal ? p.q_tiles - 1 - static_cast<int>(blockIdx.x % p.q_tiles)
                          : static_cast<int>(blockIdx.x % p.q_tiles);
  const int bh = blockIdx.x / p.q_tiles;
  Ctl c;
  c.bars = base + kOffBarQ;
  c.abort = reinterpret_cast<volatile uint32_t*>(smem + kOffBarQ + kNumBars * 8 + 4);
  c.limit = p.wait_limit;
  const uint32_t tmem = block_setup(c, smem + kOffBarQ, base + kOffBarQ, warp, false);
  const uint32_t sQ = base + kOffFixed0, sDO = base + kOffFixed1;
  // S is double-buffered (the fourth 128 columns), so S and dP of the next key tile are
  // computed while the compute warps work on this one; dP has one buffer, which the
  // compute warps release as soon as they hold their columns of it in registers.
  const uint32_t tS0 = tmem, tdP = tmem + 128, tdQ = tmem + 256, tS1 = tmem + 384;
  // key tiles 0 .. nk - 1; causal: up to the diagonal of this tile's last row
  const int nk = kCausal ? (min(p.Nq, (qt + 1) * kT) + p.off + kT - 1) / kT : p.k_tiles;
  auto kslot = [&](int j) { return base + kOffRingA + (j % kSlotsA) * kTileBytes; };
  auto vslot = [&](int j) { return base + kOffRingB + (j % kSlotsB) * kTileBytes; };

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(c.bar(kBarFixed), 2 * kTileBytes);
      for (int h = 0; h < 2; ++h) {
        tma_load_3d(sQ + h * kBoxBytes, &tmQ, c.bar(kBarFixed), h * 64, qt * kT, bh);
        tma_load_3d(sDO + h * kBoxBytes, &tmDO, c.bar(kBarFixed), h * 64, qt * kT, bh);
      }
      int issued = 0;   // key tiles whose K and V were both requested
      for (int j = 0; j < nk; ++j, ++issued) {
        const int ks = j % kSlotsA, vs = j % kSlotsB;
        if (j >= kSlotsA && !wait_phase(c, kBarEmptyA + ks, (j / kSlotsA - 1) & 1, true)) break;
        mbar_arrive_expect_tx(c.bar(kBarFullA + ks), kTileBytes);
        for (int h = 0; h < 2; ++h) tma_load_3d(kslot(j) + h * kBoxBytes, &tmK, c.bar(kBarFullA + ks), h * 64, j * kT, bh);
        if (j >= kSlotsB && !wait_phase(c, kBarEmptyB + vs, (j / kSlotsB - 1) & 1, true)) {
          wait_phase(c, kBarFullA + ks, (j / kSlotsA) & 1, false);   // that K copy is in flight
          break;
        }
        mbar_arrive_expect_tx(c.bar(kBarFullB + vs), kTileBytes);
        for (int h = 0; h < 2; ++h) tma_load_3d(vslot(j) + h * kBoxBytes, &tmV, c.bar(kBarFullB + vs), h * 64, j * kT, bh);
      }
      // no copy into shared memory may be in flight when the block exits
      wait_phase(c, kBarFixed, 0, false);
      for (int j = issued - kSlotsA < 0 ? 0 : issued - kSlotsA; j < issued; ++j)
        wait_phase(c, kBarFullA + j % kSlotsA, (j / kSlotsA) & 1, false);
      for (int j = issued - kSlotsB < 0 ? 0 : issued - kSlotsB; j < issued; ++j)
        wait_phase(c, kBarFullB + j % kSlotsB, (j / kSlotsB) & 1, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // Per key tile j: S(j+1) into the other S buffer (its dS(j-1) was read by the dQ MMAs
      // issued before) and dP(j+1) once every compute warp holds dP(j) in registers, then
      // dQ += dS K_j once dS is handed over. This thread waits twice and commits twice per
      // step: the compute warps check that K_{j+1} and V_{j+1} have landed before their
      // dP hand-over of step j, and free V_j's slot themselves (on seeing dP(j) complete).
      bool ok = wait_phase(c, kBarFixed, 0, true) && wait_phase(c, kBarFullA, 0, true) &&
                wait_phase(c, kBarFullB, 0, true);
      if (ok) {
        tc_fence_after();
        mma_rows_by_rows(tS0, sQ, kslot(0));                   // S(0) = Q K_0^T
        mma_rows_by_rows(tdP, sDO, vslot(0));                  // dP(0) = dO V_0^T
        tc_commit(c.bar(kBarSdP));
      }
      for (int j = 0; ok && j < nk; ++j) {
        const int s = j & 1;
        const uint32_t tSj = s ? tS1 : tS0;
        if (j + 1 < nk) {
          const int j1 = j + 1;
          if (!wait_phase(c, kBarDPFree, j & 1, true)) break;
          tc_fence_after();
          mma_rows_by_rows(s ? tS0 : tS1, sQ, kslot(j1));      // S(j+1) = Q K_{j+1}^T
          mma_rows_by_rows(tdP, sDO, vslot(j1));               // dP(j+1) = dO V_{j+1}^T
          tc_commit(c.bar(kBarSdP));
        }
        if (!wait_phase(c, kBarDS + s, (j >> 1) & 1, true)) break;
        tc_fence_after();
        for (int h = 0; h < 2; ++h)   // keys 64h .. 64h + 63
          mma_tmem_by_rows_half(tdQ, tSj + 64 * h, kslot(j), h, j > 0 || h > 0);   // dQ += dS K_j
        tc_commit(c.bar(kBarEmptyA + j % kSlotsA));   // K_j is free once dQ(j) is done
      }
      tc_commit(c.bar(kBarAcc));
      wait_phase(c, kBarAcc, 0, false);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int quarter = warp & 3;
    const int grp = (warp - 4) >> 2;   // key columns 64 grp .. 64 grp + 63
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int qrow = qt * kT + quarter * 32 + lane;
    // this row's -LSE log2 e and -D; rows past Nq: any finite values (never stored)
    float nl = 0.0f, nd = 0.0f;
    if (qrow < p.Nq) {
      const float* rt = p.rows + 2 * (static_cast<size_t>(bh) * p.q_pad + static_cast<size_t>(qt) * kT);
      nl = rt[quarter * 32 + lane];
      nd = rt[kT + quarter * 32 + lane];
    }
    const float2 c2 = make_float2(p.scale_log2, p.scale_log2), nl2 = make_float2(nl, nl), nd2 = make_float2(nd, nd);
    // One thread checks, before the dP hand-over of step j, that K_{j+1} and V_{j+1} (read
    // by the MMAs that hand-over releases) have landed; another frees V_j's slot.
    const bool ringer = warp == 4 && lane == 0, releaser = warp == 8 && lane == 0;
    bool ok = true;
    const float2 lg2 = make_float2(1.4426950408889634f, 1.4426950408889634f);
    for (int j = 0; j < nk; ++j) {
      const int j1 = j + 1;
      // bias: this thread's row over the group's 64 key columns, as BF16 pairs, requested
      // before the waits: eight 16-byte loads when all 64 keys are inside Nk (strides are
      // multiples of 8 elements), else key by key; nothing past Nq or Nk is read. (Staging
      // them through shared memory, for loads that cover whole row pieces, needs one of the
      // K ring's three slots: measured slower, 1.12 against 0.92 ms on square-4k.)
      uint32_t bw[kBias ? 32 : 1];
      if constexpr (kBias) {
        const int k0 = j * kT + 64 * grp;
        const int nvalid = p.Nk - k0;
        if (qrow < p.Nq && nvalid >= 64) {
          const uint4* src = reinterpret_cast<const uint4*>(bias_row(p, bh, qrow) + k0);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint4 t = __ldg(src + g);
            bw[4 * g] = t.x;
            bw[4 * g + 1] = t.y;
            bw[4 * g + 2] = t.z;
            bw[4 * g + 3] = t.w;
          }
        } else {
          const uint16_t* src = qrow < p.Nq ? bias_row(p, bh, qrow) + k0 : nullptr;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint32_t lo = src != nullptr && 2 * i < nvalid ? __ldg(src + 2 * i) : 0u;
            const uint32_t hi = src != nullptr && 2 * i + 1 < nvalid ? __ldg(src + 2 * i + 1) : 0u;
            bw[i] = lo | (hi << 16);
          }
        }
      }
      if (!wait_warp(c, kBarSdP, j & 1)) {
        ok = false;
        break;
      }
      if (releaser) mbar_arrive(c.bar(kBarEmptyB + j % kSlotsB));   // dP(j) complete: V_j is free
      __syncwarp();
      tc_fence_after();
      const uint32_t tSj = (j & 1) ? tS1 : tS0;
      // keys of this tile inside the sequence: columns < valid; causal: also <= c_hi
      const int valid = p.Nk - j * kT - 64 * grp;   // in group columns
      const int c_hi = kCausal ? qrow + p.off - j * kT - 64 * grp : kT;
      const bool mask_warp = kCausal && (qt * kT + quarter * 32 + p.off - j * kT) < 64 * grp + 63;
      const bool full = valid >= 64 && !mask_warp;   // warp-uniform: no column of the group is masked
      uint32_t xd[64];
      tmem_ld64(tdP + lane_off + 64 * grp, xd);
      tc_fence_before();
      __syncwarp();
      bool landed = true;
      if (ringer && j1 < nk)
        landed = wait_phase(c, kBarFullA + j1 % kSlotsA, (j1 / kSlotsA) & 1, true) &&
                 wait_phase(c, kBarFullB + j1 % kSlotsB, (j1 / kSlotsB) & 1, true);
      if (!__shfl_sync(0xffffffffu, landed, 0)) {
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive(c.bar(kBarDPFree));   // dP may be overwritten now
      __syncwarp();
      {
        // dS = P (dP - D) over the group's 64 key columns, written over the first 32 of them
        uint32_t xs[64];
        tmem_ld64(tSj + lane_off + 64 * grp, xs);
        uint32_t dw[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float2 n = nl2;
          if constexpr (kBias) n = ffma2(f2(bw[i] << 16, bw[i] & 0xffff0000u), lg2, nl2);   // + B log2 e
          const float2 a = ffma2(f2(xs[2 * i], xs[2 * i + 1]), c2, n);
          float p0 = ex2(a.x), p1 = ex2(a.y);
          if (!full) {
            p0 = 2 * i < valid ? p0 : 0.0f;
            p1 = 2 * i + 1 < valid ? p1 : 0.0f;
            if (mask_warp) {
              p0 = 2 * i <= c_hi ? p0 : 0.0f;
              p1 = 2 * i + 1 <= c_hi ? p1 : 0.0f;
            }
          }
          const float2 d = fmul2(make_float2(p0, p1), fadd2(f2(xd[2 * i], xd[2 * i + 1]), nd2));
          dw[i] = pack_bf16(d.x, d.y);
        }
        tmem_st32(tSj + lane_off + 64 * grp, dw);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(kBarDS + (j & 1)));
      __syncwarp();
    }
    if (ok && wait_warp(c, kBarAcc, 0)) {
      tc_fence_after();
      const int row0 = qt * kT + quarter * 32;
      uint8_t* st = smem + kOffFixed0 + (warp - 4) * kStageWarpBytes;   // Q is no longer read
      store_acc_half(tdQ + lane_off, grp, p.scale, st, p.dq + (static_cast<size_t>(bh) * p.Nq + row0) * kD,
                     p.Nq - row0);
    }
  }
  block_teardown(tmem, warp);
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
std::atomic<unsigned long long> g_bwd_launches{0};
std::atomic<unsigned long long> g_bwd_wait_limit{kDefaultWaitLimit};
std::atomic<int> g_bwd_withhold{0};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// [BH, rows, 128] BF16 viewed as a 3-D tensor (d innermost); box = 64 columns x 128 rows x 1.
bool make_map(CUtensorMap* map, const void* ptr, int rows, long long bh) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(rows) * kD * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kT), 1};
  cuuint32_t elem[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Workspace of the row pass, per (device, stream); calls on one stream are ordered.
std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, std::pair<void*, size_t>> g_ws;

int get_rows_workspace(int dev, cudaStream_t stream, size_t bytes, float** out) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  auto& ws = g_ws[std::make_pair(dev, reinterpret_cast<uintptr_t>(stream))];
  if (ws.second < bytes) {
    if (ws.first) cudaFreeAsync(ws.first, stream);
    ws.first = nullptr;
    ws.second = 0;
    if (cudaMallocAsync(&ws.first, bytes, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    ws.second = bytes;
  }
  *out = static_cast<float*>(ws.first);
  return ATTN_OK;
}

std::atomic<int> g_attr_done[3] = {{0}, {0}, {0}};   // per instantiation (plain, causal, bias)

template <bool kCausal, bool kBias = false>
int launch_bwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
               const BwdParams& p, long long bh, long long k_tiles, long long q_tiles, cudaStream_t s) {
  constexpr int kInst = kBias ? 2 : (kCausal ? 1 : 0);
  if (!g_attr_done[kInst].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(bwd_dkdv_kernel<kCausal, kBias>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemKV) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_dq_kernel<kCausal, kBias>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemQ) !=
            cudaSuccess)
      return ATTN_ERR_CUDA;
    g_attr_done[kInst].store(1, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cfg.gridDim = dim3(static_cast<unsigned>(bh * k_tiles));
  cfg.dynamicSmemBytes = kSmemKV;
  if (cudaLaunchKernelEx(&cfg, bwd_dkdv_kernel<kCausal, kBias>, mq, mk, mv, mdo, p) != cudaSuccess)
    return ATTN_ERR_CUDA;
  g_bwd_launches.fetch_add(1, std::memory_order_relaxed);
  cfg.gridDim = dim3(static_cast<unsigned>(bh * q_tiles));
  cfg.dynamicSmemBytes = kSmemQ;
  if (cudaLaunchKernelEx(&cfg, bwd_dq_kernel<kCausal, kBias>, mq, mk, mv, mdo, p) != cudaSuccess)
    return ATTN_ERR_CUDA;
  g_bwd_launches.fetch_add(1, std::memory_order_relaxed);
  return ATTN_OK;
}

struct BwdBias {
  const void* ptr;
  long long sb, sh, sq;
};

int backward(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, void* stream,
             bool causal, const BwdBias* bias = nullptr) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (d != kD) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  if (bh == 0 || Nq == 0) return ATTN_OK;
  if (Nk == 0 || (causal && Nq > Nk)) return ATTN_ERR_INVALID_ARG;
  if (causal && Nk > INT_MAX - 1024) return ATTN_ERR_UNSUPPORTED;   // row + off + 2 * kT stays in int
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                        reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                        reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv);
  if ((a16 & 15u) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_MISALIGNED;
  const long long q_tiles = (static_cast<long long>(Nq) + kT - 1) / kT;
  const long long k_tiles = (static_cast<long long>(Nk) + kT - 1) / kT;
  if (bh * q_tiles > INT_MAX || bh * k_tiles > INT_MAX || q_tiles * kT > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  if ((bh * q_tiles * kT + 7) / 8 > INT_MAX) return ATTN_ERR_UNSUPPORTED;   // the row pass's grid
  const long long max_rows = static_cast<long long>(Nq > Nk ? Nq : Nk);
  if (bh > (LLONG_MAX / 256) / max_rows) return ATTN_ERR_INVALID_ARG;
  if (bias != nullptr) {   // the rules of attn_fwd_bias
    if (!bias->ptr || bias->sb < 0 || bias->sh < 0 || bias->sq < 0) return ATTN_ERR_INVALID_ARG;
    constexpr long long kCap = LLONG_MAX / 8;
    const long long ext[3] = {B - 1LL, H - 1LL, Nq - 1LL};
    const long long str[3] = {bias->sb, bias->sh, bias->sq};
    for (int i = 0; i < 3; ++i)
      if (str[i] > 0 && ext[i] > kCap / str[i]) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(bias->ptr) & 15u) || ((bias->sb | bias->sh | bias->sq) & 7))
      return ATTN_ERR_MISALIGNED;
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map(&mq, q, Nq, bh) || !make_map(&mk, k, Nk, bh) || !make_map(&mv, v, Nk, bh) ||
      !make_map(&mdo, dout, Nq, bh))
    return ATTN_ERR_CUDA;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  BwdParams p;
  p.dq = static_cast<uint16_t*>(dq);
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  p.Nq = Nq;
  p.Nk = Nk;
  p.q_tiles = static_cast<int>(q_tiles);
  p.k_tiles = static_cast<int>(k_tiles);
  p.q_pad = static_cast<int>(q_tiles * kT);
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.wait_limit = g_bwd_wait_limit.load(std::memory_order_relaxed);
  p.causal = causal ? 1 : 0;
  p.off = causal ? Nk - Nq : 0;
  p.withhold = g_bwd_withhold.load(std::memory_order_relaxed);
  p.bias = bias ? static_cast<const uint16_t*>(bias->ptr) : nullptr;
  p.bias_sb = bias ? bias->sb : 0;
  p.bias_sh = bias ? bias->sh : 0;
  p.bias_sq = bias ? bias->sq : 0;
  p.H = H;
  float* rows = nullptr;
  {
    const int rc = get_rows_workspace(dev, s, static_cast<size_t>(bh) * p.q_pad * 2 * sizeof(float), &rows);
    if (rc != ATTN_OK) return rc;
  }
  p.rows = rows;

  const long long n_rows = bh * p.q_pad;
  bwd_rows_kernel<<<static_cast<unsigned>((n_rows + 7) / 8), 256, 0, s>>>(
      static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), lse, rows, bh, Nq, p.q_pad);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  g_bwd_launches.fetch_add(1, std::memory_order_relaxed);

  if (bias != nullptr) return launch_bwd<false, true>(mq, mk, mv, mdo, p, bh, k_tiles, q_tiles, s);
  return causal ? launch_bwd<true>(mq, mk, mv, mdo, p, bh, k_tiles, q_tiles, s)
                : launch_bwd<false>(mq, mk, mv, mdo, p, bh, k_tiles, q_tiles, s);
}

}  // namespace

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                        float scale, void* stream) {
  return backward(q, k, v, o, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, stream, false);
}

extern "C" int attn_bwd_causal(const void* q, const void* k, const void* v, const void* o, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                               float scale, void* stream) {
  return backward(q, k, v, o, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, stream, true);
}

extern "C" int attn_bwd_bias(const void* q, const void* k, const void* v, const void* o, const void* dout,
                             const float* lse, const void* bias, long long bias_stride_b, long long bias_stride_h,
                             long long bias_stride_q, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk,
                             int d, float scale, void* stream) {
  const BwdBias ba = {bias, bias_stride_b, bias_stride_h, bias_stride_q};
  return backward(q, k, v, o, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, stream, false, &ba);
}

extern "C" int attn_bwd_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int h = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_bwd_status, sizeof h, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  if (h == 0) return ATTN_OK;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_bwd_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return (h & 2u) ? ATTN_ERR_CUDA : ATTN_ERR_TIMEOUT;
}

extern "C" unsigned long long attn_bwd_kernel_count(void) { return g_bwd_launches.load(std::memory_order_relaxed); }

extern "C" int attn_bwd_set_wait_limit(unsigned long long cycles, int withhold_tile) {
  g_bwd_wait_limit.store(cycles ? cycles : kDefaultWaitLimit, std::memory_order_relaxed);
  g_bwd_withhold.store(withhold_tile ? 1 : 0, std::memory_order_relaxed);
  return ATTN_OK;
}
