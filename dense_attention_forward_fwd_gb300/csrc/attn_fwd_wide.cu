// attn_fwd_wide.cu -- dense BF16 attention forward for head dimensions above 128 (192, 256)
// on GB300 (sm_103a).
//
// The same computation as the d = 128 kernel (O = softmax(scale Q K^T) V with an online
// softmax, "FlashAttention'ı Anlamak Bölüm 1", section 0.1; head dimensions above 128 are
// what "Flash Attention на 5090 в CUDA C++" lists next, section "Что дальше"), laid out for
// the larger d. TMEM holds 512 columns of 128 lanes: two Q tiles' S and O, as in the d = 128
// kernel, would need 2 x (128 + d) columns, so a block here owns one 128-row Q tile, with
// S double-buffered (2 x 128 columns) beside O (d columns). The next key tile's scores are
// computed while the softmax works on this one, and P V of a step (d / 128 times the work
// at d = 128) overlaps the next softmax: per 128-key step the tensor cores do 2 d / 128
// times the work of one d = 128 tile step while the softmax's work is unchanged.
//
// Shared memory (224 KB at d = 256): Q as d / 64 boxes of 64 columns x 128 rows (16 KB
// each); one key tile of K in the same boxes, a ring whose box c holds box c of successive
// key tiles and is freed by a commit after the four K16 steps of Q K^T that read it; V in
// a ring of three 64-key half tiles, each freed by a commit after the half of P V that
// read it. Those early releases are what let the next tiles land a whole product ahead of
// their use: with V as one 128-key tile, V_{j+1} could only be requested once all of
// P_j V_j was done, and the first half of P_{j+1} waited for it every step.
//
// Roles (256 threads): warp 0 lane 0 issues TMA, warp 1 lane 0 issues tcgen05.mma and owns
// TMEM, warps 4-7 run the softmax and the epilogue with one thread per query row (TMEM lane).
// Per 128-key step j the MMA thread waits for each 64-key half of P_j and issues its half
// of O += P_j V_j, then S_{j+2} = Q K_{j+2}^T into the S buffer P_j leaves. The softmax
// thread that hands a half of P over has first checked that its V half has landed, so the
// MMA thread waits only for P and for K_{j+2}'s boxes. Whole query tiles per block, no split
// of the key range.
//
// Every wait is bounded (clock64 budget): on expiry the block raises an abort flag, sets
// the status word and winds down; no trap, no fault.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_fwd.h"
#include "attn_wide.h"
#include "tc_sm103.cuh"

namespace attn_wide {
namespace {

using namespace tc;

constexpr int kBM = 128;                  // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;                  // keys per step
constexpr int kBoxCols = 64;              // one TMA box: 64 BF16 columns (128 B) x 128 rows
constexpr int kBoxBytes = kBoxCols * 2 * 128;
constexpr int kMaxVSlots = 3;             // V ring, in 64-key half tiles (2 at d = 256 with a bias)
constexpr int kStageWarpBytes = 32 * kBN * 2;   // a softmax warp's 32 bias rows of one step
constexpr int kThreads = 256;
constexpr float kRescaleLog2 = 32.0f;     // the running maximum moves when a tile's exceeds it by this
constexpr int kTmemCols = 512;
constexpr int kMaxChunks = 4;             // d <= 256
// K boxes that share one full and one free barrier. Each barrier operation of the MMA
// thread leaves the tensor pipe idle for about 95 cycles, which sets the pace at d = 256,
// where the tensor work of a step exceeds the softmax's: there boxes go in pairs (measured
// +7 to +10 %; the whole tile at once loses on short key ranges). At d = 192 the softmax
// sets the pace and each box keeps its own barriers, so the first Q K^T steps start early.
template <int D>
constexpr int kKGroupBoxesFor = D == 256 ? 2 : 1;

// kind::f8f6f4 instruction descriptor: E4M3 x E4M3 -> FP32 (format code 0 for A and B),
// M = 128, N = 128, both K-major (S = Q K^T from FP8 codes)
constexpr uint32_t kIdQK8 =
    (1u << 4) | (static_cast<uint32_t>(128 >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
// D (TMEM) (+)= A (shared memory) * B (shared memory), 8-bit floating-point operands
__device__ __forceinline__ void mma_ss_e4m3(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc))
      : "memory");
}
// D (TMEM) (+)= A (TMEM) * B (shared memory), 8-bit floating-point operands
__device__ __forceinline__ void mma_ts_e4m3(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc))
      : "memory");
}
// kind::f8f6f4 descriptor for O += P V with V as E4M3 codes: M = 128, N = d, A (P, in TMEM)
// and B (V^T: d rows of keys) both K-major
template <int D>
constexpr uint32_t kIdPV8 =
    (1u << 4) | (static_cast<uint32_t>(D >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
// 16 columns of this warp's 32 TMEM lanes
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&x)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]), "r"(x[8]), "r"(x[9]),
      "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]), "r"(x[15])
      : "memory");
}
// Four values rounded to E4M3 (nearest even, saturating), the first in the lowest byte
// (cvt puts its first source in the upper half of its 16-bit result).
__device__ __forceinline__ uint32_t pack_e4m3x4(float a0, float a1, float a2, float a3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(a1), "f"(a0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(a3), "f"(a2));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}
// x rounded to E4M3 as pack_e4m3x4 rounds it, widened back exactly (through FP16) to FP32
__device__ __forceinline__ float round_e4m3(float x) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(0.0f), "f"(x));
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  float r;
  asm("cvt.f32.f16 %0, %1;" : "=f"(r) : "h"(static_cast<uint16_t>(h2 & 0xffffu)));
  return r;
}

// barriers
constexpr int kBarQFull = 0;
constexpr int kBarQEmpty = 1;                     // the tile's last Q K^T is done with Q
constexpr int kBarKFull = 2;                      // [box group]
constexpr int kBarKFree = kBarKFull + kMaxChunks; // [box group]: the Q K^T steps that read it are done
constexpr int kBarVFull = kBarKFree + kMaxChunks; // [V slot]
constexpr int kBarVFree = kBarVFull + kMaxVSlots; // [V slot]: the P V products that read it are done
constexpr int kBarSFull = kBarVFree + kMaxVSlots; // [2 buffers]
constexpr int kBarPFull = kBarSFull + 2;          // [step parity][half], one arrival per softmax warp
constexpr int kBarOFull = kBarPFull + 4;
constexpr int kBarOEmpty = kBarOFull + 1;         // the epilogue has read O out of TMEM
constexpr int kBarDrain = kBarOEmpty + 1;
constexpr int kNumBars = kBarDrain + 1;
constexpr int kFlagsBytes = kNumBars * 8 + 8;     // barriers, TMEM slot, abort flag

// With a bias, each softmax warp stages its rows' bias in shared memory; at d = 256 that
// room comes from one V slot. kF8 >= 1: Q and K as FP8 codes, a box holding 128 columns
// (128 bytes) of the head dimension: two boxes per tile at d = 192 and 256 (at d = 192 the
// second box's upper half lies past the tensor and is filled with zeros). kF8 == 2: V too,
// given as V^T codes (d rows of keys); a V slot then holds a whole key tile (d rows of 128
// bytes), else one 64-key half of V.
template <int D, bool kBias, int kF8 = 0>
struct Layout {
  static constexpr int kChunks = D / kBoxCols;             // V boxes: 64 BF16 columns
  static constexpr int kQKChunks = kF8 >= 1 ? (D + 127) / 128 : kChunks;   // boxes per Q or K tile
  static constexpr int kTileBytes = kQKChunks * kBoxBytes;  // one Q or K tile
  static constexpr int kHalfBytes = kChunks * kBoxBytes / 2;   // V: 64 keys x d
  static constexpr int kVUnitBytes = kF8 == 2 ? D * kBN : kHalfBytes;   // one V slot
  static constexpr int kVSlots = (kBias && D == 256 && kF8 == 0) ? 2 : kMaxVSlots;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffStage = kOffV + kVSlots * kVUnitBytes;
  static constexpr int kOffBar = kOffStage + (kBias ? 4 * kStageWarpBytes : 0);
  static constexpr int kSmem = kOffBar + kFlagsBytes + 1024;   // + realignment of the base to 1024
  static_assert(D % kBoxCols == 0 && kChunks <= kMaxChunks, "head dimension in whole boxes");
  static_assert(kSmem <= 232448, "exceeds the 227 KB shared memory of one block");
  static_assert(2 * kBN + D <= kTmemCols, "two S buffers and O must fit TMEM");
};

__device__ unsigned int g_wide_status;   // bit 0: a wait timed out

struct Params {
  uint16_t* o;
  float* lse;
  int Nq, Nk;
  int q_tiles;        // 128-row query tiles per head
  int n_kv;           // 128-key steps
  int kv_tail;        // keys in the last step (1 .. 128)
  int groups;         // B * H * q_tiles
  int bh_count;       // B * H
  int causal;         // query i sees keys 0 .. i + causal_off only
  int causal_off;     // Nk - Nq
  float scale_log2;   // scale * log2(e)
  unsigned long long wait_limit;
  // additive bias (kBias): B_ij of head (b, h) = bias[b * bias_sb + h * bias_sh + i * bias_sq + j],
  // BF16, strides in elements (multiples of 8), H heads per batch; scores become scale q.k + B
  const uint16_t* bias;
  long long bias_sb, bias_sh, bias_sq;
  int H;
  float scale;
  float v_scale;   // V's descale factor (V as FP8 codes), applied with 1 / l
  int withhold;    // test hook: never load a block's first V unit, so that a wait for it runs out
};

// The query tiles a block runs, in order; every role walks the same sequence. Plain: tile
// g = blockIdx.x + r * gridDim.x of the list (bh, qt) with qt fastest (a head's tiles on
// neighbouring blocks share its K and V in L2). Causal: the list sorted longest first (a
// tile's key range ends at its last row's diagonal), every head's longest tile before any
// head's second longest, dealt to the blocks in a snake (odd rounds in reverse block order)
// to even out the rounds.
struct TileIter {
  const Params& p;
  int r = 0;
  __device__ explicit TileIter(const Params& pp) : p(pp) {}
  __device__ bool next(int& bh, int& qt, int& n) {
    const int grid = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
    const long long pos = static_cast<long long>(r) * grid + ((p.causal && (r & 1)) ? grid - 1 - b : b);
    ++r;
    if (pos >= p.groups) return false;
    if (p.causal) {
      qt = p.q_tiles - 1 - static_cast<int>(pos / p.bh_count);
      bh = static_cast<int>(pos % p.bh_count);
      const int last_row = min(p.Nq, (qt + 1) * kBM) - 1;
      n = (last_row + p.causal_off) / kBN + 1;   // key tiles up to its last row's diagonal
    } else {
      bh = static_cast<int>(pos / p.q_tiles);
      qt = static_cast<int>(pos % p.q_tiles);
      n = p.n_kv;
    }
    return true;
  }
};

struct Ctl {
  uint32_t bars;
  volatile uint32_t* abort;
  unsigned long long limit;
  __device__ __forceinline__ uint32_t bar(int i) const { return bars + 8u * static_cast<uint32_t>(i); }
};

// true once the phase with this parity has completed; false on timeout, or (when
// watch_abort) as soon as another role of the block has given up.
__device__ __forceinline__ bool wait_phase(const Ctl& c, int idx, uint32_t parity, bool watch_abort) {
  const uint32_t b = c.bar(idx);
  if (mbar_try_wait(b, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(b, parity)) return true;
    if (watch_abort && *c.abort) return false;
    if (static_cast<unsigned long long>(clock64() - t0) > c.limit) {
      *c.abort = 1u;
      atomicOr(&g_wide_status, 1u);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_warp(const Ctl& c, int idx, uint32_t parity) {
  const bool ok = wait_phase(c, idx, parity, true);
  return __all_sync(0xffffffffu, ok);
}

// 16 bytes global -> shared without passing through registers; the bytes past src_bytes
// (0 .. 16) are written as zeros and not read
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Global counters (every role keeps them alike): step gs of the block's key stream (all its
// query tiles' key tiles, in order) uses S buffer gs & 1 and K tile gs (box c in K slot c);
// its V halves are half tiles 2 gs and 2 gs + 1, in V slots (2 gs + h) % kVSlots. A ring
// barrier completes once per use of its slot, so the k-th use waits for parity k & 1.
template <int D, bool kPos, bool kBias, int kF8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Params p) {
  using L = Layout<D, kBias, kF8>;
  constexpr bool kQK8 = kF8 >= 1, kV8 = kF8 == 2;
  constexpr int kVSlots = L::kVSlots;
  constexpr int kChunks = L::kQKChunks;   // Q and K boxes
  constexpr int kVChunks = L::kChunks;    // V boxes
  constexpr int kQKBoxCols = kQK8 ? 128 : kBoxCols;   // head-dimension columns per Q or K box
  constexpr int kKGroupBoxes = kQK8 ? 1 : kKGroupBoxesFor<D>;
  constexpr int kVUnits = kV8 ? 1 : 2;   // V slots per key tile
  constexpr int kKGroups = (kChunks + kKGroupBoxes - 1) / kKGroupBoxes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctl c;
  c.bars = base + L::kOffBar;
  c.abort = reinterpret_cast<volatile uint32_t*>(smem + L::kOffBar + kNumBars * 8 + 4);
  c.limit = p.wait_limit;
  const uint32_t sQ = base + L::kOffQ, sK = base + L::kOffK, sV = base + L::kOffV;
  auto vslot = [&](int vi) { return sV + static_cast<uint32_t>(vi % kVSlots) * L::kVUnitBytes; };

  if (threadIdx.x == 0) {
    for (int b = 0; b < kNumBars; ++b) mbar_init(c.bar(b), 1);
    for (int b = 0; b < 4; ++b) mbar_init(c.bar(kBarPFull + b), 4);   // one arrival per softmax warp
    mbar_init(c.bar(kBarOEmpty), 4);
    *c.abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(c.bars + kNumBars * 8),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kOffBar + kNumBars * 8);

  if (warp == 0) {
    if (lane == 0) {
      // -------- TMA producer: per query tile Q, then K_0, and per step K_{t+1}, V_t --------
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmV)) : "memory");
      int u = 0, gj = 0;           // query tiles started, steps of earlier tiles
      int k_loads[kMaxChunks] = {0, 0, 0, 0};   // loads requested into each K box group
      int v_halves = 0;                          // V halves requested
      bool ok = true;
      auto load_k = [&](int t, int bh) {   // key tile t of this query tile (global step gj + t)
        const int gt = gj + t;
        for (int g = 0; ok && g < kKGroups; ++g) {
          if (gt > 0 && !wait_phase(c, kBarKFree + g, static_cast<uint32_t>(gt - 1) & 1u, true)) {
            ok = false;
            break;
          }
          const int c0 = g * kKGroupBoxes, c1 = min(kChunks, c0 + kKGroupBoxes);
          mbar_arrive_expect_tx(c.bar(kBarKFull + g), (c1 - c0) * kBoxBytes);
          for (int cc = c0; cc < c1; ++cc)
            tma_load_3d(sK + cc * kBoxBytes, &tmK, c.bar(kBarKFull + g), cc * kQKBoxCols, t * kBN, bh);
          k_loads[g] = gt + 1;
        }
      };
      auto load_v = [&](int t, int bh) {   // both 64-key halves of V_t, or the V^T tile of step t
        for (int h = 0; ok && h < kVUnits; ++h) {
          const int vi = kVUnits * (gj + t) + h, slot = vi % kVSlots;
          if (p.withhold && vi == 0) {   // (the test hook) the unit is never requested
            v_halves = vi + 1;
            continue;
          }
          if (vi >= kVSlots && !wait_phase(c, kBarVFree + slot, static_cast<uint32_t>(vi / kVSlots - 1) & 1u, true)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(c.bar(kBarVFull + slot), L::kVUnitBytes);
          if constexpr (kV8) {   // keys t*128 .. t*128+127 of all d rows of V^T
            tma_load_3d(vslot(vi), &tmV, c.bar(kBarVFull + slot), t * kBN, 0, bh);
          } else {
            for (int cc = 0; cc < kVChunks; ++cc)
              tma_load_3d(vslot(vi) + cc * (kBoxBytes / 2), &tmV, c.bar(kBarVFull + slot), cc * kBoxCols,
                          t * kBN + h * (kBN / 2), bh);
          }
          v_halves = vi + 1;
        }
      };
      TileIter it(p);
      int bh, qt, n;
      while (ok && it.next(bh, qt, n)) {
        if (u > 0 && !wait_phase(c, kBarQEmpty, (u - 1) & 1, true)) break;
        mbar_arrive_expect_tx(c.bar(kBarQFull), L::kTileBytes);
        for (int cc = 0; cc < kChunks; ++cc)
          tma_load_3d(sQ + cc * kBoxBytes, &tmQ, c.bar(kBarQFull), cc * kQKBoxCols, qt * kBM, bh);
        ++u;
        load_k(0, bh);
        for (int t = 0; ok && t < n; ++t) {
          if (t + 1 < n) load_k(t + 1, bh);
          load_v(t, bh);
        }
        gj += n;
      }
      // no copy into shared memory may be in flight when the block exits
      if (u > 0) wait_phase(c, kBarQFull, (u - 1) & 1, false);
      for (int g = 0; g < kKGroups; ++g)
        if (k_loads[g] > 0) wait_phase(c, kBarKFull + g, static_cast<uint32_t>(k_loads[g] - 1) & 1u, false);
      for (int vi = v_halves > kVSlots ? v_halves - kVSlots : 0; vi < v_halves; ++vi)
        wait_phase(c, kBarVFull + vi % kVSlots, static_cast<uint32_t>(vi / kVSlots) & 1u, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // -------- MMA issuer --------
      const uint32_t tS[2] = {tmem, tmem + kBN};
      const uint32_t tO = tmem + 2 * kBN;
      constexpr uint32_t kIdQK = idesc_bf16(kBM, kBN, false);
      constexpr uint32_t kIdPV = idesc_bf16(kBM, D, true);
      bool ok = true;
      // S = Q K^T for the key tile of global step gt, group by group of boxes; each group
      // is released as soon as the K16 steps that read it are done
      auto qk = [&](uint32_t d_tmem, int gt) {
        for (int g = 0; g < kKGroups; ++g) {
          if (!wait_phase(c, kBarKFull + g, static_cast<uint32_t>(gt) & 1u, true)) {
            ok = false;
            return;
          }
          tc_fence_after();
          const int c0 = g * kKGroupBoxes, c1 = min(kChunks, c0 + kKGroupBoxes);
          for (int cc = c0; cc < c1; ++cc) {
            // 32 bytes of each 128-byte row per MMA: 16 BF16 columns, or 32 FP8 columns (at
            // d = 192 the second FP8 box holds 64 columns: two MMAs)
            const int steps = kQK8 ? min(4, (D - cc * 128) / 32) : 4;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              if (k4 >= steps) break;
              const uint32_t off = static_cast<uint32_t>(cc * kBoxBytes + k4 * 32);
              if constexpr (kQK8)
                mma_ss_e4m3(d_tmem, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), kIdQK8,
                            cc > 0 || k4 > 0);
              else
                mma_ss(d_tmem, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), kIdQK,
                       cc > 0 || k4 > 0);
            }
          }
          tc_commit(c.bar(kBarKFree + g));
        }
      };
      int u = 0, gj = 0;
      TileIter it(p);
      int bh, qt, n;
      while (ok && it.next(bh, qt, n)) {
        if (!wait_phase(c, kBarQFull, u & 1, true)) break;
        tc_fence_after();
        // the first two key tiles' scores; later ones follow each step's P V
        for (int t = 0; ok && t < 2 && t < n; ++t) {
          qk(tS[(gj + t) & 1], gj + t);
          tc_commit(c.bar(kBarSFull + ((gj + t) & 1)));
        }
        if (!ok) break;
        if (n <= 2) tc_commit(c.bar(kBarQEmpty));
        // the first P V overwrites O: the previous tile's epilogue must have read it
        if (u > 0 && !wait_phase(c, kBarOEmpty, (u - 1) & 1, true)) break;
        for (int j = 0; ok && j < n; ++j) {
          const int gs = gj + j, buf = gs & 1;
          const uint32_t ph = static_cast<uint32_t>(gs >> 1) & 1u;
          for (int h = 0; h < 2; ++h) {   // keys 64h .. 64h + 63: P columns 32h .., V half 2 gs + h
            if (!wait_phase(c, kBarPFull + 2 * (gs & 1) + h, ph, true)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if constexpr (kV8) {
              // P as E4M3 (four keys per TMEM column: 32 keys = 8 columns per MMA) times V^T
              // (d rows of the tile's 128 keys, K-major like K): 32 bytes of each row per MMA
#pragma unroll
              for (int kk = 2 * h; kk < 2 * h + 2; ++kk)
                mma_ts_e4m3(tO, tS[buf] + kk * 8, sdesc_sw128(vslot(gs) + kk * 32, 16, 1024), kIdPV8<D>,
                            j > 0 || kk > 0);
              if (h == 1) tc_commit(c.bar(kBarVFree + gs % kVSlots));
            } else {
              const int vi = 2 * gs + h;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)   // 16 keys per MMA: 8 columns of packed P
                mma_ts(tO, tS[buf] + (4 * h + kk) * 8, sdesc_sw128(vslot(vi) + kk * 16 * 128, kBoxBytes / 2, 1024),
                       kIdPV, j > 0 || h > 0 || kk > 0);
              tc_commit(c.bar(kBarVFree + vi % kVSlots));
            }
          }
          if (!ok) break;
          if (j + 2 < n) {
            qk(tS[buf], gs + 2);
            if (!ok) break;
            tc_commit(c.bar(kBarSFull + buf));
            if (j + 2 == n - 1) tc_commit(c.bar(kBarQEmpty));
          }
        }
        if (!ok) break;
        tc_commit(c.bar(kBarOFull));
        gj += n;
        ++u;
      }
      // every MMA this thread issued must finish before TMEM and shared memory are released
      tc_commit(c.bar(kBarDrain));
      wait_phase(c, kBarDrain, 0, false);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // -------- softmax and epilogue: thread = query row --------
    const int quarter = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS[2] = {tmem + lane_off, tmem + lane_off + kBN};
    const uint32_t tO = tmem + lane_off + 2 * kBN;
    // the factor still to apply to a score: with a bias, s already holds scale q.k + B (natural units)
    const float cs = kBias ? 1.4426950408889634f : (kPos ? p.scale_log2 : 1.0f);
    const bool ringer = warp == 4 && lane == 0;
    int u = 0, gj = 0;
    TileIter it(p);
    int bh, qt, n;
    while (it.next(bh, qt, n)) {
      float m_used = -INFINITY, l = 0.0f, corr = 0.0f;
      bool ok = true;
      // bias: the warp's 32 rows x 128 keys of a step, staged in its own shared memory by
      // 16-byte copies issued one step ahead. Copy i puts rows 2i and 2i + 1 (16 lanes each,
      // 256 contiguous bytes per row, so four 128-byte lines per instruction); 16-byte chunk
      // ch of staged row r sits at chunk ch ^ (r & 15), so neither the copies nor the
      // row-per-lane reads meet a bank conflict. Rows past Nq and keys past Nk read nothing
      // and are staged as 0 (those scores are never stored, or masked).
      const int row0 = qt * kBM + quarter * 32;
      const uint16_t* bbase = nullptr;
      if constexpr (kBias)
        bbase = p.bias + static_cast<long long>(bh / p.H) * p.bias_sb + static_cast<long long>(bh % p.H) * p.bias_sh;
      const uint32_t stage = base + L::kOffStage + static_cast<uint32_t>(quarter * kStageWarpBytes);
      auto stage_bias = [&](int j) {
        const int k0 = j * kBN, ch = lane & 15;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = 2 * i + (lane >> 4), row = row0 + r, key = k0 + 8 * ch;
          const int valid = row < p.Nq ? max(0, min(8, p.Nk - key)) : 0;
          const uint16_t* src = valid > 0 ? bbase + static_cast<long long>(row) * p.bias_sq + key : p.bias;
          cp_async16(stage + static_cast<uint32_t>((r * 16 + (ch ^ (r & 15))) * 16), src, 2 * valid);
        }
        cp_async_commit();
      };
      if constexpr (kBias) stage_bias(0);
      for (int j = 0; j < n; ++j) {
        const int gs = gj + j, buf = gs & 1;
        if (!wait_warp(c, kBarSFull + buf, static_cast<uint32_t>(gs >> 1) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[128];
        {
          uint32_t x[128];
          tmem_ld<128>(tS[buf], x);
          if constexpr (kBias) {   // scale q.k + B, B from the staged row
            cp_async_wait_all();
            __syncwarp();
            const float2 sc2 = make_float2(p.scale, p.scale);
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
              uint4 b;
              asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                           : "r"(stage + static_cast<uint32_t>((lane * 16 + (cc ^ (lane & 15))) * 16)));
              const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = 4 * cc + e;
                const float2 t = ffma2(f2(x[2 * i], x[2 * i + 1]), sc2, f2(bw[e] << 16, bw[e] & 0xffff0000u));
                s[2 * i] = t.x;
                s[2 * i + 1] = t.y;
              }
            }
            __syncwarp();   // every lane has read the stage before the next step's copies land
            if (j + 1 < n) stage_bias(j + 1);
          } else {
#pragma unroll
            for (int i = 0; i < 128; ++i) s[i] = kPos ? __uint_as_float(x[i]) : __uint_as_float(x[i]) * p.scale_log2;
          }
        }
        if (j == p.n_kv - 1 && p.kv_tail < kBN) {   // keys past the sequence
          const int valid = p.kv_tail;
#pragma unroll
          for (int i = 0; i < 128; ++i) s[i] = i < valid ? s[i] : -INFINITY;
        }
        if (p.causal) {
          // key j * 128 + i is visible to this row iff it is <= row + causal_off
          const int lim_warp = qt * kBM + quarter * 32 + p.causal_off - j * kBN;   // the warp's first row
          if (lim_warp < kBN - 1) {   // warp-uniform: some row of this warp has keys masked here
            const int lim = lim_warp + lane;
#pragma unroll
            for (int i = 0; i < 128; ++i) s[i] = i <= lim ? s[i] : -INFINITY;
          }
        }
        // row max: eight independent three-input max chains
        float mx[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) mx[t] = fmaxf(s[t], s[t + 8]);
#pragma unroll
        for (int i = 16; i < 128; i += 16) {
#pragma unroll
          for (int t = 0; t < 8; ++t) mx[t] = max3(mx[t], s[i + t], s[i + 8 + t]);
        }
        const float m_raw =
            fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float m_tile = m_raw * cs;
        bool rescale = false;
        float alpha = 1.0f;
        // (P as E4M3 must stay below its largest finite value, 448: tau = 8)
        if (m_tile > m_used + (kV8 ? 8.0f : kRescaleLog2)) {
          alpha = ex2(m_used - m_tile);   // 0 on a tile's first step
          l *= alpha;
          corr *= alpha;
          m_used = m_tile;
          rescale = j > 0;
        }
        if (__any_sync(0xffffffffu, rescale)) {
          // O must hold the previous step's P V before it is rescaled (S_j's product was
          // issued before that one), and be rescaled before this step's accumulates: wait
          // for the commit of the previous step's second half (V half 2 gs - 1)
          const int vi = kV8 ? gs - 1 : 2 * gs - 1;
          if (!wait_warp(c, kBarVFree + vi % kVSlots, static_cast<uint32_t>(vi / kVSlots) & 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float a = rescale ? alpha : 1.0f;
#pragma unroll 1
          for (int ch = 0; ch < D / 8; ++ch) {
            uint32_t ov[8];
            tmem_ld<8>(tO + ch * 8, ov);
#pragma unroll
            for (int i = 0; i < 8; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * a);
            tmem_st<8>(tO + ch * 8, ov);
          }
        }
        // (with a bias a row may have seen only -inf so far: its weights are all 0 then)
        const float neg_m = (kBias && m_used == -INFINITY) ? 0.0f : -m_used;
        {
          // the BF16 rounding error of the tile's largest weight, with the arithmetic that
          // forms it below: l + corr is then the sum of the weights the tensor cores apply
          const float pm = (kBias && m_tile == -INFINITY) ? 0.0f : ex2(fmaf(m_raw, cs, neg_m));
          if constexpr (kV8)
            corr += round_e4m3(pm) - pm;
          else
            corr += __uint_as_float(pack_bf16(pm, 0.0f) << 16) - pm;
        }
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const float2 cs2 = make_float2(cs, cs), nm2 = make_float2(neg_m, neg_m);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if constexpr (kV8) {   // 64 keys = 16 columns of four E4M3 values
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int e = half * 64 + 4 * i;
              const float2 a2 = ffma2(make_float2(s[e], s[e + 1]), cs2, nm2);
              const float2 b2 = ffma2(make_float2(s[e + 2], s[e + 3]), cs2, nm2);
              const float e0 = ex2(a2.x), e1 = ex2(a2.y), e2 = ex2(b2.x), e3 = ex2(b2.y);
              pk[i] = pack_e4m3x4(e0, e1, e2, e3);
              const int r = 2 * (i & 1);
              const float2 t2 = fadd2(make_float2(acc[2 * r], acc[2 * r + 1]), make_float2(e0, e1));
              const float2 t3 = fadd2(make_float2(acc[2 * r + 2], acc[2 * r + 3]), make_float2(e2, e3));
              acc[2 * r] = t2.x;
              acc[2 * r + 1] = t2.y;
              acc[2 * r + 2] = t3.x;
              acc[2 * r + 3] = t3.y;
            }
            tmem_st16(tS[buf] + half * 16, pk);
          } else {
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int e = half * 64 + 2 * i;
              const float2 a2 = ffma2(make_float2(s[e], s[e + 1]), cs2, nm2);
              const float e0 = ex2(a2.x), e1 = ex2(a2.y);
              pk[i] = pack_bf16(e0, e1);
              const float2 t2 = fadd2(make_float2(acc[2 * (i & 3)], acc[2 * (i & 3) + 1]), make_float2(e0, e1));
              acc[2 * (i & 3)] = t2.x;
              acc[2 * (i & 3) + 1] = t2.y;
            }
            tmem_st<32>(tS[buf] + half * 32, pk);
          }
          tc_fence_before();
          __syncwarp();
          // the MMAs this hand-over releases read this half's V (the step's V^T tile)
          bool landed = true;
          if (ringer) {
            const int vi = kV8 ? gs : 2 * gs + half;
            landed = wait_phase(c, kBarVFull + vi % kVSlots, static_cast<uint32_t>(vi / kVSlots) & 1u, true);
          }
          if (!__shfl_sync(0xffffffffu, landed, 0)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive(c.bar(kBarPFull + 2 * (gs & 1) + half));
          __syncwarp();
        }
        if (!ok) break;
        l += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      }
      if (!ok || !wait_warp(c, kBarOFull, static_cast<uint32_t>(u) & 1u)) break;
      tc_fence_after();
      // epilogue: O / (l + corr) as BF16, each thread its own row; the natural-log LSE
      const int row = qt * kBM + quarter * 32 + lane;
      const bool live = row < p.Nq;
      const float inv_l = (kV8 ? p.v_scale : 1.0f) / (l + corr);
      uint4* orow = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(bh) * p.Nq + (live ? row : 0)) * D);
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t x[32];
        tmem_ld<32>(tO + ch * 32, x);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16(__uint_as_float(x[2 * i]) * inv_l, __uint_as_float(x[2 * i + 1]) * inv_l);
        if (live) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            orow[ch * 4 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(kBarOEmpty));
      __syncwarp();
      if (live) p.lse[static_cast<size_t>(bh) * p.Nq + row] = (m_used + log2f(l)) * 0.69314718055994531f;
      gj += n;
      ++u;
    }
    if constexpr (kBias) cp_async_wait_all();   // (after an abort) no copy still lands in shared memory
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
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

// [BH, rows, d] BF16 as a 3-D tensor (d innermost); box = 64 columns x box_rows rows x 1.
// f8: E4M3 codes, one byte per element, boxes of 128 columns (128 bytes as for BF16).
bool make_map(CUtensorMap* map, const void* ptr, int rows, long long bh, int d, int box_rows, bool f8 = false) {
  auto enc = encoder();
  if (!enc) return false;
  const cuuint64_t es = f8 ? 1 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * es, static_cast<cuuint64_t>(rows) * d * es};
  cuuint32_t box[3] = {f8 ? 128u : static_cast<cuuint32_t>(kBoxCols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t elem[3] = {1, 1, 1};
  return enc(map, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr),
             dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
// V^T as E4M3 codes, [BH, d, ldv] with keys innermost (Nk of each row of ldv used); box =
// 128 keys x d rows x 1, one 128-byte swizzle span per row.
bool make_map_vt(CUtensorMap* map, const void* ptr, int Nk, long long ldv, long long bh, int d) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(Nk), static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldv), static_cast<cuuint64_t>(ldv) * d};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kBN), static_cast<cuuint32_t>(d), 1};
  cuuint32_t elem[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// per instantiation (d, sign of the scale or bias, 8-bit inputs) and device
std::atomic<int> g_attr_done[18][kMaxDevices];

template <int D, bool kPos, bool kBias, int kF8>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const Params& p, int grid, int dev,
           cudaStream_t stream) {
  auto kern = attn_fwd_wide_kernel<D, kPos, kBias, kF8>;
  constexpr int kInst = 3 * ((D == 256 ? 3 : 0) + (kBias ? 2 : (kPos ? 1 : 0))) + kF8;
  constexpr int kSmem = Layout<D, kBias, kF8>::kSmem;
  if (dev < 0 || dev >= kMaxDevices || !g_attr_done[kInst][dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) g_attr_done[kInst][dev].store(1, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, p) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

// One head dimension, scale sign, bias and input format.
template <int D, int kF8>
int launch_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const Params& p, int grid, int dev,
             cudaStream_t stream, bool bias, float scale) {
  // with a bias the scale is applied before the row max: one instantiation serves any sign
  if (bias) return launch<D, true, true, kF8>(mq, mk, mv, p, grid, dev, stream);
  return scale > 0.0f ? launch<D, true, false, kF8>(mq, mk, mv, p, grid, dev, stream)
                      : launch<D, false, false, kF8>(mq, mk, mv, p, grid, dev, stream);
}

int forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk, int d,
            float scale, bool causal, cudaStream_t stream, unsigned long long wait_limit, const Bias* bias, int f8,
            long long ldv, float v_scale, int withhold) {
  if (!supported(d)) return ATTN_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  const long long q_tiles = (static_cast<long long>(Nq) + kBM - 1) / kBM;
  if (bh > INT_MAX || bh * q_tiles > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return ATTN_ERR_CUDA;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, Nq, bh, d, kBM, f8 >= 1) || !make_map(&mk, k, Nk, bh, d, kBN, f8 >= 1) ||
      !(f8 == 2 ? make_map_vt(&mv, v, Nk, ldv, bh, d) : make_map(&mv, v, Nk, bh, d, kBN / 2)))
    return ATTN_ERR_CUDA;
  Params p;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.Nq = Nq;
  p.Nk = Nk;
  p.q_tiles = static_cast<int>(q_tiles);
  p.n_kv = (Nk + kBN - 1) / kBN;
  p.kv_tail = Nk - (p.n_kv - 1) * kBN;
  p.groups = static_cast<int>(bh * q_tiles);
  p.bh_count = static_cast<int>(bh);
  p.causal = causal ? 1 : 0;
  p.causal_off = causal ? Nk - Nq : 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.wait_limit = wait_limit;
  p.bias = bias ? static_cast<const uint16_t*>(bias->ptr) : nullptr;
  p.bias_sb = bias ? bias->sb : 0;
  p.bias_sh = bias ? bias->sh : 0;
  p.bias_sq = bias ? bias->sq : 0;
  p.H = H;
  p.scale = scale;
  p.v_scale = v_scale;
  p.withhold = withhold;
  const int grid = std::min(sms, p.groups);
  const bool b = bias != nullptr;
  if (d == 256)
    return f8 == 2   ? launch_d<256, 2>(mq, mk, mv, p, grid, dev, stream, b, scale)
           : f8 == 1 ? launch_d<256, 1>(mq, mk, mv, p, grid, dev, stream, b, scale)
                     : launch_d<256, 0>(mq, mk, mv, p, grid, dev, stream, b, scale);
  return f8 == 2   ? launch_d<192, 2>(mq, mk, mv, p, grid, dev, stream, b, scale)
         : f8 == 1 ? launch_d<192, 1>(mq, mk, mv, p, grid, dev, stream, b, scale)
                   : launch_d<192, 0>(mq, mk, mv, p, grid, dev, stream, b, scale);
}

int take_status(cudaStream_t stream) {
  unsigned int h = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_wide_status, sizeof h, 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return -1;
  if (h == 0) return 0;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_wide_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return -1;
  return 1;
}

}  // namespace attn_wide
