// attn_fwd.cu -- dense BF16 attention forward for GB300 (sm_103a): non-causal, causal
// (attn_fwd_causal), with an additive bias (attn_fwd_bias, its own instantiation) and with
// 8-bit inputs: Q and K as FP8 E4M3 codes (attn_fwd_fp8qk: the producer loads one 128-byte
// box per Q or K tile and S = Q K^T is issued as kind::f8f6f4 MMAs), or Q, K and V
// (attn_fwd_fp8: V^T tiles as one box each, P rounded to E4M3 in TMEM, four keys per
// column, and O += P V issued as kind::f8f6f4 MMAs with P read from TMEM).
//
// O = softmax(scale * Q K^T) V and the per-row log-sum-exp, head_dim 128, computed
// FlashAttention-style: Q tiles of 128 query rows are loaded once and 128-key K/V
// tiles are streamed through an online softmax, so S and P stay on chip ("Sıfırdan
// yazılan CUDA attention kerneli...", section "Kernel işini nasıl bölümlendiriyor";
// the running max / running sum / rescale recurrence of "Flash Attention на 5090 в
// CUDA C++", v1).
//
// Blackwell mapping (one persistent block per SM, 12 warps):
//   warp 0        TMA producer: the two Q tiles of each work segment, then per step the
//                 K/V unit {V_j, K_j+1} into one of two pairs of 128B-swizzled
//                 shared-memory slots (one full and one empty mbarrier per pair).
//   warp 1        MMA issuer (one thread): tcgen05.mma S_i = Q_i K_j^T into TMEM, and
//                 O_i += P_i V_j with P_i read from TMEM; owns the TMEM allocation. Its
//                 queue is shallow, so anything else it does idles the tensor core: it
//                 only waits for P and commits S, and softmax threads look after the ring
//                 (one thread of tile 0 checks each unit before handing over P, one of
//                 tile 1 releases it once S_1 of its step is complete).
//   warps 4-7     softmax + epilogue for Q tile 0 (thread = query row = TMEM lane).
//   warps 8-11    softmax + epilogue for Q tile 1.
//   warps 2-3     idle.
// setmaxnreg gives warps 0-3 120 registers per thread and the softmax warps 192.
// Two Q tiles per block let one tile's softmax run while the tensor core works on
// the other tile's two GEMMs (the two-query-tile schedule that the FlashAttention-4
// summary in "Hacker News Digest" describes). TMEM holds S0, S1, O0, O1 (4 x 128
// columns of FP32); P_i is written as BF16 over the first 64 columns of S_i.
//
// Work is a list of groups (two Q tiles of one (b, h)) times K/V steps. Each block
// walks a list of segments (group, key-step range): whole groups dealt round-robin in
// waves (neighbouring blocks share heads, so K/V stay in L2), then, for the last one
// or two waves' worth of groups, an even split of their key steps over all blocks, so
// no SM idles at the end. A group split between blocks is finished by whichever block
// completes its share last: every share leaves its unnormalised O, running max and
// sums in a workspace, and the last one merges them in share order (so results do not
// depend on which block finished last). No block waits for another. Causal launches
// take whole groups only, each over the key steps up to its last row's diagonal,
// longest first in snake order across blocks; the softmax masks keys past each row's
// diagonal on the steps that cross it. Bias launches add the bias to the scaled scores
// before the row max; each softmax warp reads its rows' bias with coalesced loads and
// transposes it through its staging tile.
//
// The softmax keeps, per row, m (running max of scale*s in log2 units) and l (running
// sum of 2^(scale*s*log2e - m)). O is accumulated unnormalised and divided once at the
// end ("normalised once the loop ends, then written", same write-up). The running max
// only moves when it grows by more than kRescaleLog2 (log2 units; 8 when P is rounded to
// E4M3, whose largest value is 448): the exponentials
// are then bounded by 2^kRescaleLog2 and O and l keep sharing one m, so the result is
// unchanged; skipping the move avoids reading and rewriting O in TMEM. P is BF16 (range
// to 2^127) and every sum is FP32, so the bound can be generous: with weights up to 2^32,
// |V| up to 2^20 and 2^24 keys the accumulators stay below 2^76, far from FP32's 2^128,
// while a row's running max practically never moves after its first tile.
//
// Every wait is bounded (clock64 budget). On expiry a block raises a flag in shared
// memory, the others stop at their next wait, the producer and the MMA thread wait
// (bounded) for their own copies and MMAs in flight, TMEM is freed and the block
// exits; the host learns of it through attn_fwd_status().

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <vector>
#include <utility>

#include "attn_fwd.h"
#include "attn_wide.h"
#include "tc_sm103.cuh"

namespace {

// ---------------------------------------------------------------------------------
// Tiling constants
// ---------------------------------------------------------------------------------
constexpr int kD = 128;                        // head dimension
constexpr int kBM = 128;                       // query rows per Q tile (= TMEM lanes)
constexpr int kBN = 128;                       // keys per K/V tile
constexpr int kQTiles = 2;                     // Q tiles per block
constexpr int kSlots = 4;                      // K/V ring depth, one 128x128 tile per slot
constexpr int kPairs = kSlots / 2;             // the ring hands over units of two slots
constexpr int kTileBytes = kBM * kD * 2;       // 32 KB of BF16
constexpr int kBoxBytes = kTileBytes / 2;      // one TMA box: 64 columns (128 B) x 128 rows
constexpr int kTile8Bytes = kBM * kD;          // 16 KB of FP8 codes: one box of 128 columns (128 B)
constexpr int kThreads = 384;
// Register split between the warpgroups. setmaxnreg.inc draws only on registers that
// the block holds: 128 * kRegsCtl + 256 * kRegsSoftmax must equal 384 * kRegsLaunch,
// the per-thread count the kernel is compiled to (checked on the host before the first
// launch), or the increase would wait forever.
constexpr int kRegsLaunch = 168;
constexpr int kRegsCtl = 120;
constexpr int kRegsSoftmax = 192;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax == kThreads * kRegsLaunch, "register split must balance");
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 32.0f;
constexpr unsigned long long kDefaultWaitLimit = 1ull << 31;

// shared memory map (byte offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kQTiles * kTileBytes;
constexpr int kOffBar = kOffKV + kSlots * kTileBytes;
constexpr int kBarQFull = 0;
constexpr int kBarQEmpty = 1;                      // the Q tiles may be overwritten
constexpr int kBarKVFull = 2;                      // [pair]
constexpr int kBarKVEmpty = kBarKVFull + kPairs;   // [pair]
constexpr int kBarSFull = kBarKVEmpty + kPairs;
constexpr int kBarPFull = kBarSFull + kQTiles;     // [tile][half]: one barrier per 64-key half of P
constexpr int kBarOFull = kBarPFull + 2 * kQTiles;
constexpr int kBarOEmpty = kBarOFull + kQTiles;    // the epilogue has read O_i out of TMEM
constexpr int kBarDrain = kBarOEmpty + kQTiles;
constexpr int kBarSfReady = kBarDrain + 1;         // [tile]: the scale factors of S_tile's next product are in TMEM (MXFP8)
constexpr int kNumBars = kBarSfReady + kQTiles;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
// Per softmax warp, a staging tile for its 32 rows x 64 columns of BF16 output.
constexpr int kStageBytes = 32 * 64 * 2;
constexpr int kOffStage = (kOffAbort + 4 + 127) & ~127;
constexpr int kSmemUsed = kOffStage + kQTiles * 4 * kStageBytes;   // one stage per softmax warp
constexpr int kSmemBytes = kSmemUsed + 1024;   // slack to align the dynamic base to 1024

static_assert(kOffKV % 1024 == 0 && kOffBar % 8 == 0, "swizzle atoms need 1024-byte alignment");
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB shared memory of one block");

// Workspace of split groups: per block two partial records (its first and its last
// split segment), each holding per Q tile the unnormalised O in groups of four columns
// (columns 4g..4g+3 of row r at (g * kBM + r) * 4, so that a warp's 32 rows of one
// group are 512 contiguous bytes and each thread moves 16-byte vectors), then m (log2
// units), l and corr, kBM floats each.
constexpr int kPartFloatsPerTile = kD * kBM + 3 * kBM;
constexpr size_t kPartBytesPerBlock = size_t(2) * kQTiles * kPartFloatsPerTile * sizeof(float);
static_assert(kPartFloatsPerTile % 4 == 0, "each tile record must start on a 16-byte boundary");
constexpr int kMinSegSteps = 8;   // smallest share of a group worth a block of its own
constexpr int kMaxGrid = 160;     // blocks of a launch at most (one per SM)

struct Params {
  uint16_t* o;            // BF16 bits [BH, Nq, 128]
  float* lse;             // [BH, Nq]
  int Nq, Nk;
  int q_groups;           // ceil(Nq / (kQTiles * kBM)): groups per (b, h)
  int n_kv;               // ceil(Nk / kBN)
  int kv_tail;            // valid keys in the last K/V tile, 1..128
  int dp_groups;          // groups [0, dp_groups) are processed whole, group g by block g % grid
  long long sk_steps;     // key steps of groups [dp_groups, n_groups), shared out over the blocks
  long long cuts[kMaxGrid + 1];   // block c's share of them: steps [cuts[c], cuts[c + 1])
  float* part;            // partial records, kPartBytesPerBlock per block (split groups only)
  unsigned int* cnt;      // [n_groups - dp_groups][kQTiles][4] arrival counters, zero at launch
  unsigned int* cnt_next; // the other bank: this launch zeroes it for the next one (or null)
  int cnt_len;            // counters per bank (the whole allocated bank, not only this launch's)
  float scale_log2;       // scale * log2(e)
  unsigned long long wait_limit;
  int withhold_tile;      // test hook: never load the second K/V unit of a block (V of step 0, K of step 1)
  int causal;             // query i sees keys 0 .. i + causal_off only (causal_off = Nk - Nq >= 0)
  int causal_off;
  int bh_count;           // B * H
  // additive bias (kernels instantiated with kBias): B_ij of head (b, h) is
  // bias[b * bias_sb + h * bias_sh + i * bias_sq + j], BF16, strides in elements
  const uint16_t* bias;
  long long bias_sb, bias_sh, bias_sq;
  int H;                  // heads per batch (splits b*H + h)
  float scale;            // the caller's scale (the bias path scales before adding B)
  float v_scale = 1.0f;   // V's descale factor (V as FP8 codes), applied with 1 / l
  float* o32 = nullptr;   // FP32 [BH, Nq, 128]: O before rounding (kernels instantiated with kO32)
  // MXFP8 inputs (kF8 == 3): E8M0 block scales, byte b of a word for elements 32b .. 32b+31
  const uint32_t* sfq = nullptr;   // [BH, Nq]: a query row's four scales along d
  const uint32_t* sfk = nullptr;   // [BH, Nk]: a key row's four scales along d
  const uint8_t* sfv = nullptr;    // [BH, 128, ldsv]: row c of V^T, byte t = keys 32t .. 32t+31
  long long ldsv = 0;
};

// floor(a / b) for a >= 0, b > 0. On the device a 64-bit division is a long dependent
// sequence; operands that fit 32 bits (all but enormous problems) take the short one.
__host__ __device__ __forceinline__ long long div_floor(long long a, long long b) {
#ifdef __CUDA_ARCH__
  if (((static_cast<unsigned long long>(a) | static_cast<unsigned long long>(b)) >> 32) == 0)
    return static_cast<long long>(static_cast<unsigned>(a) / static_cast<unsigned>(b));
#endif
  return a / b;
}

// First key step (counted over the split region) of block c's share.
__host__ __device__ __forceinline__ long long sk_share_start(long long c, long long sk_steps, long long grid) {
  return div_floor(c * sk_steps, grid);
}

struct Segment {
  int group;      // b*H*q_groups + h*q_groups + q-group
  int kv0, kv1;   // key steps [kv0, kv1) of the group
  int which;      // 0: first segment of this block's split share, 1: its last
  bool split;     // other blocks hold other key steps of this group
  // split-region numbering (split groups only): the group's first key step, its number of
  // key steps, and its index among the split region's groups (its merge counters)
  long long x0;
  int glen, cidx;
};

// The segments of one block, in processing order; every role of the block walks the
// same sequence.
//
// Causal launches: a group needs only the keys up to its last row's diagonal, so groups
// differ in length. List position x holds diagonal position q_groups - 1 - x / (B*H) of
// head x % (B*H) (longest first). With many groups they are processed whole: block b takes
// position b of even waves and grid - 1 - b of odd ones, which evens out the waves. With
// few (sk_steps > 0) the list's key steps are concatenated and cut into equal shares, as
// the split region of a non-causal launch: a long group is then split between blocks and
// merged like one.
struct SegIter {
  int n_kv, dp_groups, grid, next_dp;
  long long sk_begin, sk_end, sk_pos;
  int causal, causal_off, q_groups, bh_count, Nq, wave;
  __device__ explicit SegIter(const Params& p) {
    n_kv = p.n_kv;
    dp_groups = p.dp_groups;
    grid = static_cast<int>(gridDim.x);
    next_dp = static_cast<int>(blockIdx.x);
    sk_begin = p.cuts[blockIdx.x];
    sk_end = p.cuts[blockIdx.x + 1];
    sk_pos = sk_begin;
    causal = p.causal;
    causal_off = p.causal_off;
    q_groups = p.q_groups;
    bh_count = p.bh_count;
    Nq = p.Nq;
    wave = 0;
  }
  // causal split shares: the list level (diagonal position) holding sk_pos and its first step
  int lvl = 0;
  long long lvl_start = 0;
  __device__ int level_len(int level) const {   // key steps of each group of a list level
    const int qg = q_groups - 1 - level;
    const int row_end = min(Nq, (qg + 1) * (kQTiles * kBM));
    return (row_end + causal_off + kBN - 1) / kBN;
  }
  __device__ bool next(Segment& sg) {
    if (causal && sk_end > 0) {
      if (sk_pos >= sk_end) return false;
      int len = level_len(lvl);
      while (sk_pos >= lvl_start + static_cast<long long>(bh_count) * len) {
        lvl_start += static_cast<long long>(bh_count) * len;
        len = level_len(++lvl);
      }
      const long long in_lvl = sk_pos - lvl_start;
      const int h = static_cast<int>(div_floor(in_lvl, len));
      const int kv0 = static_cast<int>(in_lvl - static_cast<long long>(h) * len);
      const long long left = sk_end - sk_pos;
      const int kv1 = left < len - kv0 ? kv0 + static_cast<int>(left) : len;
      sg.group = h * q_groups + (q_groups - 1 - lvl);
      sg.kv0 = kv0;
      sg.kv1 = kv1;
      sg.which = sk_pos == sk_begin ? 0 : 1;
      sg.split = !(kv0 == 0 && kv1 == len);
      sg.x0 = lvl_start + static_cast<long long>(h) * len;
      sg.glen = len;
      sg.cidx = lvl * bh_count + h;
      sk_pos = sg.x0 + kv1;
      return true;
    }
    if (causal) {
      const int pos = (wave & 1) ? grid - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
      const long long x = static_cast<long long>(wave) * grid + pos;
      if (x >= static_cast<long long>(bh_count) * q_groups) return false;
      ++wave;
      const int xi = static_cast<int>(x);
      const int qg = q_groups - 1 - xi / bh_count;
      sg.group = (xi % bh_count) * q_groups + qg;
      const int row_end = min(Nq, (qg + 1) * (kQTiles * kBM));   // one past the group's last row
      sg.kv0 = 0;
      sg.kv1 = (row_end + causal_off + kBN - 1) / kBN;
      sg.which = 0;
      sg.split = false;
      return true;
    }
    if (next_dp < dp_groups) {
      sg.group = next_dp;
      sg.kv0 = 0;
      sg.kv1 = n_kv;
      sg.which = 0;
      sg.split = false;
      next_dp += grid;
      return true;
    }
    if (sk_pos < sk_end) {
      const long long g_rel = div_floor(sk_pos, n_kv);
      const int kv0 = static_cast<int>(sk_pos - g_rel * n_kv);
      const long long left = sk_end - sk_pos;
      const int kv1 = left < n_kv - kv0 ? kv0 + static_cast<int>(left) : n_kv;
      sg.group = dp_groups + static_cast<int>(g_rel);
      sg.kv0 = kv0;
      sg.kv1 = kv1;
      sg.which = sk_pos == sk_begin ? 0 : 1;
      sg.split = !(kv0 == 0 && kv1 == n_kv);
      sg.x0 = g_rel * n_kv;
      sg.glen = n_kv;
      sg.cidx = static_cast<int>(g_rel);
      sk_pos = g_rel * n_kv + kv1;
      return true;
    }
    return false;
  }
};

// The block whose share contains split-region key step x (every share is non-empty).
__device__ __forceinline__ int sk_block_of(long long x, const Params& p, int grid) {
  int lo = 0, hi = grid - 1;   // the last c with cuts[c] <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cuts[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ unsigned int g_attn_status;   // per device; bit 0 = a wait timed out

// ---------------------------------------------------------------------------------
// PTX wrappers. The ones every kernel of the library uses (mbarrier, TMA tile loads,
// tcgen05.mma / commit / fences, ex2, max3, BF16 packing, the shared-memory descriptor)
// are in tc_sm103.cuh; this file's own follow.
// ---------------------------------------------------------------------------------
using tc::ex2;
using tc::max3;
using tc::mbar_arrive;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_test_wait;
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


__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* ptr) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

// D(tmem) (+)= A(smem desc) * B(smem desc), 8-bit floating-point operands
__device__ __forceinline__ void mma_ss_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc))
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem desc), 8-bit floating-point operands
__device__ __forceinline__ void mma_ts_f8(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc))
      : "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc), E4M3 operands scaled per 32 elements of K by E8M0
// factors read from TMEM (sfa for the rows of A, sfb for the rows of B)
__device__ __forceinline__ void mma_ss_mx(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                          bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(static_cast<uint32_t>(acc))
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem desc), scaled as mma_ss_mx
__device__ __forceinline__ void mma_ts_mx(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                          bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(static_cast<uint32_t>(acc))
      : "memory");
}

// 128 consecutive FP32 columns of this thread's TMEM lane (32x32b shape), waited on.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&x)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]),
        "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15]),
        "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]),
        "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31]),
        "=r"(x[32]), "=r"(x[33]), "=r"(x[34]), "=r"(x[35]), "=r"(x[36]), "=r"(x[37]), "=r"(x[38]), "=r"(x[39]),
        "=r"(x[40]), "=r"(x[41]), "=r"(x[42]), "=r"(x[43]), "=r"(x[44]), "=r"(x[45]), "=r"(x[46]), "=r"(x[47]),
        "=r"(x[48]), "=r"(x[49]), "=r"(x[50]), "=r"(x[51]), "=r"(x[52]), "=r"(x[53]), "=r"(x[54]), "=r"(x[55]),
        "=r"(x[56]), "=r"(x[57]), "=r"(x[58]), "=r"(x[59]), "=r"(x[60]), "=r"(x[61]), "=r"(x[62]), "=r"(x[63]),
        "=r"(x[64]), "=r"(x[65]), "=r"(x[66]), "=r"(x[67]), "=r"(x[68]), "=r"(x[69]), "=r"(x[70]), "=r"(x[71]),
        "=r"(x[72]), "=r"(x[73]), "=r"(x[74]), "=r"(x[75]), "=r"(x[76]), "=r"(x[77]), "=r"(x[78]), "=r"(x[79]),
        "=r"(x[80]), "=r"(x[81]), "=r"(x[82]), "=r"(x[83]), "=r"(x[84]), "=r"(x[85]), "=r"(x[86]), "=r"(x[87]),
        "=r"(x[88]), "=r"(x[89]), "=r"(x[90]), "=r"(x[91]), "=r"(x[92]), "=r"(x[93]), "=r"(x[94]), "=r"(x[95]),
        "=r"(x[96]), "=r"(x[97]), "=r"(x[98]), "=r"(x[99]), "=r"(x[100]), "=r"(x[101]), "=r"(x[102]), "=r"(x[103]),
        "=r"(x[104]), "=r"(x[105]), "=r"(x[106]), "=r"(x[107]), "=r"(x[108]), "=r"(x[109]), "=r"(x[110]), "=r"(x[111]),
        "=r"(x[112]), "=r"(x[113]), "=r"(x[114]), "=r"(x[115]), "=r"(x[116]), "=r"(x[117]), "=r"(x[118]), "=r"(x[119]),
        "=r"(x[120]), "=r"(x[121]), "=r"(x[122]), "=r"(x[123]), "=r"(x[124]), "=r"(x[125]), "=r"(x[126]), "=r"(x[127])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&x)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]),
        "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15]),
        "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]),
        "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&x)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&x)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&x)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]),
        "r"(x[8]), "r"(x[9]), "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]), "r"(x[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&x)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]),
        "r"(x[8]), "r"(x[9]), "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]), "r"(x[15]),
        "r"(x[16]), "r"(x[17]), "r"(x[18]), "r"(x[19]), "r"(x[20]), "r"(x[21]), "r"(x[22]), "r"(x[23]),
        "r"(x[24]), "r"(x[25]), "r"(x[26]), "r"(x[27]), "r"(x[28]), "r"(x[29]), "r"(x[30]), "r"(x[31])
      : "memory");
}

// (y0, y1) = (x0 * a + b, x1 * a + b) as one packed FP32x2 FMA
__device__ __forceinline__ void fma2(float& y0, float& y1, float x0, float x1, float a, float b) {
  asm("{\n\t.reg .b64 x, a, b, y;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 a, {%4, %4};\n\t"
      "mov.b64 b, {%5, %5};\n\t"
      "fma.rn.f32x2 y, x, a, b;\n\t"
      "mov.b64 {%0, %1}, y;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(a), "f"(b));
}
// (y0, y1) = (x0, x1) * a + (b0, b1) as one packed FP32x2 FMA
__device__ __forceinline__ void fma2v(float& y0, float& y1, float x0, float x1, float a, float b0, float b1) {
  asm("{\n\t.reg .b64 x, a, b, y;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 a, {%4, %4};\n\t"
      "mov.b64 b, {%5, %6};\n\t"
      "fma.rn.f32x2 y, x, a, b;\n\t"
      "mov.b64 {%0, %1}, y;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(a), "f"(b0), "f"(b1));
}
// 16 bytes of read-only data, not kept in L1 (little of it is left beside shared memory)
__device__ __forceinline__ uint4 ld_nc_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}
// The bias of a warp's 32 query rows for keys k0 .. k0 + 127, read with coalesced
// 16-byte loads: load i of half h covers rows 4i .. 4i + 3 of the warp, eight lanes per
// row, each lane 8 keys (lane >> 3 picks the row, lane & 7 the 8 keys), so one load
// instruction touches four 128-byte lines. g[32h + 4i .. 32h + 4i + 3] receives the
// lane's piece. BiasRows holds what stays fixed over a segment: `piece` points at the
// lane's first piece (row row0 + (lane >> 3), keys from 8 (lane & 7)), `s4` is four rows.
struct BiasRows {
  const uint16_t* piece;
  const uint16_t* own_row;   // this lane's row (row0 + lane), for the L2 prefetch of the next step
  bool own_in;               // that row lies inside the sequence
  long long sq, s4;
  int row0;
  bool rows_full;   // all 32 rows of the warp lie inside the sequence (warp-uniform)
};
// Rows at or past Nq and keys at or past Nk read nothing and get 0 (those scores are
// masked or never stored); a piece that straddles Nk is read key by key.
__device__ __forceinline__ void load_bias_pieces(uint32_t (&g)[64], const BiasRows& br, int Nq, int k0, int Nk) {
  if (br.rows_full && k0 + kBN <= Nk) {   // warp-uniform: every piece is in range
    const uint16_t* src = br.piece + k0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 t0 = ld_nc_v4(src + i * br.s4);
      const uint4 t1 = ld_nc_v4(src + i * br.s4 + 64);
      g[4 * i] = t0.x;
      g[4 * i + 1] = t0.y;
      g[4 * i + 2] = t0.z;
      g[4 * i + 3] = t0.w;
      g[32 + 4 * i] = t1.x;
      g[32 + 4 * i + 1] = t1.y;
      g[32 + 4 * i + 2] = t1.z;
      g[32 + 4 * i + 3] = t1.w;
    }
    return;
  }
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3, cc = lane & 7;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = br.row0 + 4 * i + sub;
      const int key = k0 + 64 * h + 8 * cc;
      uint4 t = make_uint4(0u, 0u, 0u, 0u);
      if (row < Nq) {
        const uint16_t* src = br.piece + i * br.s4 + k0 + 64 * h;
        if (key + 8 <= Nk) {
          t = ld_nc_v4(src);
        } else if (key < Nk) {
          uint32_t w[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t lo = key + 2 * m < Nk ? src[2 * m] : 0u;
            const uint32_t hi = key + 2 * m + 1 < Nk ? src[2 * m + 1] : 0u;
            w[m] = lo | (hi << 16);
          }
          t = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      g[32 * h + 4 * i] = t.x;
      g[32 * h + 4 * i + 1] = t.y;
      g[32 * h + 4 * i + 2] = t.z;
      g[32 * h + 4 * i + 3] = t.w;
    }
  }
}
// Half h of the pieces above, transposed through the warp's 4 KB staging tile: b[w]
// receives this lane's row, keys 64h + 2w (low half) and 64h + 2w + 1. The 16-byte
// chunks are swizzled by row, so both the writes and the reads are free of bank conflicts.
__device__ __forceinline__ void bias_half_to_row(uint8_t* stage, const uint32_t (&g)[64], int h, uint32_t (&b)[32]) {
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3, cc = lane & 7;
  uint4* st = reinterpret_cast<uint4*>(stage);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = 4 * i + sub;
    st[rr * 8 + (cc ^ (rr & 7))] =
        make_uint4(g[32 * h + 4 * i], g[32 * h + 4 * i + 1], g[32 * h + 4 * i + 2], g[32 * h + 4 * i + 3]);
  }
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 v = st[lane * 8 + (c ^ (lane & 7))];
    b[4 * c] = v.x;
    b[4 * c + 1] = v.y;
    b[4 * c + 2] = v.z;
    b[4 * c + 3] = v.w;
  }
  __syncwarp();   // the tile is written again by the next half
}
// (a0, a1) += (x0, x1) as one packed FP32x2 add
__device__ __forceinline__ void add2(float& a0, float& a1, float x0, float x1) {
  asm("{\n\t.reg .b64 a, x;\n\t"
      "mov.b64 a, {%0, %1};\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "add.rn.f32x2 a, a, x;\n\t"
      "mov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(x0), "f"(x1));
}
// Four values rounded to E4M3 (nearest even, saturating), the first in the lowest byte.
// As with the BF16 pair, cvt puts its first source in the upper half of the result.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a0, float a1, float a2, float a3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(a1), "f"(a0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(a3), "f"(a2));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}
// x rounded to E4M3 and widened back (exactly, through FP16) to FP32.
__device__ __forceinline__ float round_e4m3(float x) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(0.0f), "f"(x));
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  float r;
  asm("cvt.f32.f16 %0, %1;" : "=f"(r) : "h"(static_cast<uint16_t>(h2 & 0xffffu)));
  return r;
}

// ---------------------------------------------------------------------------------
// Instruction descriptors (kind::f16, kind::f8f6f4, kind::mxf8f6f4; field layouts per the
// PTX ISA)
// ---------------------------------------------------------------------------------
// BF16 x BF16 -> FP32, M = 128, N = 128, A K-major, B K-major (S = Q K^T) or
// MN-major (O += P V, V stored key-major with d contiguous).
__host__ __device__ constexpr uint32_t idesc_bf16(bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(kBN >> 3) << 17) | (static_cast<uint32_t>(kBM >> 4) << 24);
}
// kind::f8f6f4: E4M3 x E4M3 -> FP32 (format code 0 for A and B), M = 128, N = 128, both
// K-major (S = Q K^T from FP8 codes).
__host__ __device__ constexpr uint32_t idesc_e4m3() {
  return (1u << 4) | (static_cast<uint32_t>(kBN >> 3) << 17) | (static_cast<uint32_t>(kBM >> 4) << 24);
}

// kind::mxf8f6f4 with block scaling: E4M3 x E4M3 -> FP32, M = 128, N = 128, both K-major, E8M0
// scale factors (bit 23), the scale byte of A's and B's rows chosen by sf (bits 29-30 and
// 4-5): byte sf of each 32-bit scale column holds the factor of K block sf.
__host__ __device__ constexpr uint32_t idesc_mx(uint32_t sf) {
  return (sf << 4) | (static_cast<uint32_t>(kBN >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(kBM >> 4) << 24) |
         (sf << 29);
}

// ---------------------------------------------------------------------------------
// Bounded waits
// ---------------------------------------------------------------------------------
struct Ctl {
  uint32_t bars;                 // shared address of barrier 0
  volatile uint32_t* abort;      // shared flag: some wait of this block gave up
  unsigned long long limit;      // clock64 budget per wait
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
      atomicOr(&g_attn_status, 1u);
      return false;
    }
  }
}
// warp-uniform variant for roles whose next step is a .sync.aligned TMEM access
__device__ __forceinline__ bool wait_warp(const Ctl& c, int idx, uint32_t parity) {
  const bool ok = wait_phase(c, idx, parity, true);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------------
// Roles
// ---------------------------------------------------------------------------------
// kF8 >= 1: Q and K are FP8 codes, one 128-byte box per tile in the first half of its
// slot; kF8 == 2: V too, transposed (keys innermost), one box in the first half of its slot.
template <int kF8>
__device__ void run_producer(const Ctl& c, uint32_t base, const CUtensorMap* tmQ,
                             const CUtensorMap* tmK, const CUtensorMap* tmV, const Params& p) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmQ)) : "memory");
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmK)) : "memory");
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmV)) : "memory");

  int last_unit[kPairs];
#pragma unroll
  for (int q = 0; q < kPairs; ++q) last_unit[q] = -1;

  int unit = 0;   // K/V units of every segment issued or skipped
  int u = 0;      // segments whose Q load was issued
  bool ok = true;
  SegIter si(p);
  Segment sg;
  while (ok && si.next(sg)) {
    const int bh = sg.group / p.q_groups;
    const int q_row0 = (sg.group % p.q_groups) * (kQTiles * kBM);
    // the previous segment's S MMAs must be done with the Q tiles
    if (u > 0 && !wait_phase(c, kBarQEmpty, (u - 1) & 1, true)) break;
    constexpr bool kQK8 = kF8 >= 1, kV8 = kF8 >= 2;
    mbar_arrive_expect_tx(c.bar(kBarQFull), kQTiles * (kQK8 ? kTile8Bytes : kTileBytes));
    for (int i = 0; i < kQTiles; ++i)
      for (int h = 0; h < (kQK8 ? 1 : 2); ++h)
        tma_load_3d(base + kOffQ + i * kTileBytes + h * kBoxBytes, tmQ, c.bar(kBarQFull), h * 64,
                    q_row0 + i * kBM, bh);
    ++u;
    // A segment of n steps streams n + 1 units: {K_0}, {V_0, K_1}, ..., {V_{n-2}, K_{n-1}},
    // {V_{n-1}}. Unit i is what the MMA thread consumes in one step (V for the P V
    // products, K for the next S); one softmax thread checks it has landed, another
    // releases it. Units alternate between the two slot pairs; the first tile of a unit
    // takes the pair's first slot.
    const int n = sg.kv1 - sg.kv0;
    for (int i = 0; ok && i <= n; ++i, ++unit) {
      const int pr = unit % kPairs, use = unit / kPairs;
      if (use > 0 && !wait_phase(c, kBarKVEmpty + pr, (use - 1) & 1, true)) {
        ok = false;
        break;
      }
      if (p.withhold_tile && unit == 1) continue;
      const bool has_v = i > 0, has_k = i < n;
      const uint32_t fb = c.bar(kBarKVFull + pr);
      mbar_arrive_expect_tx(fb, (has_v ? (kV8 ? kTile8Bytes : kTileBytes) : 0) +
                                    (has_k ? (kQK8 ? kTile8Bytes : kTileBytes) : 0));
      uint32_t dst = base + kOffKV + 2 * pr * kTileBytes;
      if (has_v) {
        if constexpr (kV8) {   // V^T: keys are the innermost coordinate
          tma_load_3d(dst, tmV, fb, (sg.kv0 + i - 1) * kBN, 0, bh);
        } else {
          for (int h = 0; h < 2; ++h)
            tma_load_3d(dst + h * kBoxBytes, tmV, fb, h * 64, (sg.kv0 + i - 1) * kBN, bh);
        }
        dst += kTileBytes;
      }
      if (has_k) {
        for (int h = 0; h < (kQK8 ? 1 : 2); ++h)
          tma_load_3d(dst + h * kBoxBytes, tmK, fb, h * 64, (sg.kv0 + i) * kBN, bh);
      }
      last_unit[pr] = unit;
    }
  }
  // Leave no copy in flight into shared memory that the block is about to release
  // (on the normal path these phases have completed or are about to).
  if (u > 0) wait_phase(c, kBarQFull, (u - 1) & 1, false);
  for (int q = 0; q < kPairs; ++q)
    if (last_unit[q] >= 0) wait_phase(c, kBarKVFull + q, (last_unit[q] / kPairs) & 1, false);
}

template <bool kQK8>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  if constexpr (kQK8) {
    // FP8 codes: the whole head dimension is one 128-byte row of the box; 32 columns
    // (32 bytes) per MMA.
    constexpr uint32_t idesc = idesc_e4m3();
#pragma unroll
    for (int kk = 0; kk < kD / 32; ++kk) {
      const uint32_t off = static_cast<uint32_t>(kk * 32);
      mma_ss_f8(d_tmem, sdesc_sw128(q_smem + off, 16, 1024), sdesc_sw128(k_smem + off, 16, 1024), idesc,
                kk > 0);
    }
    return;
  }
  constexpr uint32_t idesc = idesc_bf16(false);
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    // K-major, 128B swizzle: 16 columns = 32 bytes inside a 128-byte row; the second
    // 64-column half of the head dimension is the second TMA box.
    const uint32_t off = static_cast<uint32_t>((kk >> 2) * kBoxBytes + (kk & 3) * 32);
    mma_ss(d_tmem, sdesc_sw128(q_smem + off, 16, 1024), sdesc_sw128(k_smem + off, 16, 1024), idesc,
           kk > 0);
  }
}

// S = Q K^T from MXFP8 codes: four K32 blocks of the head dimension, block kk scaled by byte kk
// of the scale columns at sfa (rows of Q) and sfb (rows of K).
__device__ __forceinline__ void issue_qk_mx(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem, uint32_t sfa, uint32_t sfb) {
#pragma unroll
  for (int kk = 0; kk < kD / 32; ++kk) {
    const uint32_t off = static_cast<uint32_t>(kk * 32);
    mma_ss_mx(d_tmem, sdesc_sw128(q_smem + off, 16, 1024), sdesc_sw128(k_smem + off, 16, 1024),
              idesc_mx(static_cast<uint32_t>(kk)), sfa, sfb, kk > 0);
  }
}
// keys [64*half, 64*half + 64) of O += P V with P and V^T as MXFP8 (key blocks 2*half, 2*half + 1)
__device__ __forceinline__ void issue_pv_half_mx(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem, int half, bool acc,
                                                 uint32_t sfa, uint32_t sfb) {
#pragma unroll
  for (int kk = 2 * half; kk < 2 * half + 2; ++kk)
    mma_ts_mx(d_tmem, p_tmem + kk * 8, sdesc_sw128(v_smem + kk * 32, 16, 1024), idesc_mx(static_cast<uint32_t>(kk)),
              sfa, sfb, acc || kk > 0);
}

// keys [64*half, 64*half + 64) of O += P V
template <bool kPV8>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem, int half, bool acc) {
  if constexpr (kPV8) {
    // P as E4M3 in TMEM (four keys per column: 32 keys = 8 columns per MMA) times V^T as
    // E4M3 codes in shared memory (d rows of 128 keys, K-major like K for S): 32 keys
    // (32 bytes of each V^T row) per MMA.
    constexpr uint32_t idesc = idesc_e4m3();
#pragma unroll
    for (int kk = 2 * half; kk < 2 * half + 2; ++kk)
      mma_ts_f8(d_tmem, p_tmem + kk * 8, sdesc_sw128(v_smem + kk * 32, 16, 1024), idesc, acc || kk > 0);
    return;
  }
  constexpr uint32_t idesc = idesc_bf16(true);
#pragma unroll
  for (int kk = 4 * half; kk < 4 * half + 4; ++kk) {
    // MN-major, 128B swizzle: 16 keys = 16 rows of 128 bytes; the two 64-column
    // halves of d sit one box (kBoxBytes) apart, 8-row groups 1024 bytes apart.
    mma_ts(d_tmem, p_tmem + kk * 8, sdesc_sw128(v_smem + kk * 16 * 128, kBoxBytes, 1024), idesc,
           acc || kk > 0);
  }
}

// One K/V step of the MMA issuer: O_i += P_i V_j for both Q tiles and, when another
// step follows (kMore), S_i = Q_i K_{j+1}^T; otherwise the commits that hand O to the
// epilogue. `unit` is the step's K/V unit ({V_j, K_{j+1}}, or {V_j} on the last step).
// Every operation of this thread that is not an MMA leaves the tensor core idle for
// about a hundred cycles (its queue is shallow), so a step does only the four P waits
// and two commits: softmax threads check and release the ring slots.
// Returns false when a wait gave up.
// MXFP8 (kF8 == 3): the scale factors of S_i's next product sit in the other tile's S
// columns 96..103 (written by the other tile's softmax once it holds its own scores), those
// of P_i V in S_i's columns 32..39 (written with P_i); see run_softmax.
__device__ __forceinline__ uint32_t mx_sf_qk(const uint32_t (&tS)[2], int i) { return tS[1 - i] + 96; }

template <bool kMore, int kF8>
__device__ __forceinline__ bool mma_step(const Ctl& c, uint32_t base, const uint32_t (&tS)[2],
                                         const uint32_t (&tO)[2], const uint32_t (&sQ)[2], int unit,
                                         uint32_t ph, bool first) {
  const int pr = unit % kPairs;
  const uint32_t sV = base + kOffKV + 2 * pr * kTileBytes;
  const uint32_t sK = sV + kTileBytes;
  constexpr bool kQK8 = kF8 >= 1, kPV8 = kF8 >= 2, kMX = kF8 == 3;
#pragma unroll
  for (int i = 0; i < kQTiles; ++i) {
    // tile i: O_i += P_i V_j, then S_i = Q_i K_{j+1}^T. The first half of P_0 is handed over
    // only after a softmax thread has seen the unit loaded, so that wait covers the unit too.
    if (!wait_phase(c, kBarPFull + 2 * i, ph, true)) return false;
    tc_fence_after();
    if constexpr (kMX)
      issue_pv_half_mx(tO[i], tS[i], sV, 0, !first, tS[i] + 32, tS[i] + 36);
    else
      issue_pv_half<kPV8>(tO[i], tS[i], sV, 0, !first);
    if (!wait_phase(c, kBarPFull + 2 * i + 1, ph, true)) return false;
    tc_fence_after();
    if constexpr (kMX)
      issue_pv_half_mx(tO[i], tS[i], sV, 1, true, tS[i] + 32, tS[i] + 36);
    else
      issue_pv_half<kPV8>(tO[i], tS[i], sV, 1, true);
    if (kMore) {
      if constexpr (kMX) {
        if (!wait_phase(c, kBarSfReady + i, ph ^ 1u, true)) return false;
        tc_fence_after();
        issue_qk_mx(tS[i], sQ[i], sK, mx_sf_qk(tS, i), mx_sf_qk(tS, i) + 4);
      } else {
        issue_qk<kQK8>(tS[i], sQ[i], sK);
      }
      tc_commit(c.bar(kBarSFull + i));
    } else {
      tc_commit(c.bar(kBarOFull + i));
    }
  }
  return true;
}

template <int kF8>
__device__ void run_mma(const Ctl& c, uint32_t base, uint32_t tmem, const Params& p) {
  const uint32_t tS[2] = {tmem, tmem + 128};
  const uint32_t tO[2] = {tmem + 256, tmem + 384};
  const uint32_t sQ[2] = {base + kOffQ, base + kOffQ + kTileBytes};
  int unit = 0;         // K/V units consumed
  uint32_t gstep = 0;   // K/V steps of all previous segments: phase of s_full / p_full
  int u = 0;            // segments started
  SegIter si(p);
  Segment sg;
  while (si.next(sg)) {
    const int n = sg.kv1 - sg.kv0;
    if (!wait_phase(c, kBarQFull, u & 1, true) ||
        !wait_phase(c, kBarKVFull + unit % kPairs, (unit / kPairs) & 1, true))
      break;
    tc_fence_after();
    const uint32_t sK = base + kOffKV + 2 * (unit % kPairs) * kTileBytes;   // unit {K_0}
    bool sf_ok = true;
    for (int i = 0; i < kQTiles && sf_ok; ++i) {
      if constexpr (kF8 == 3) {
        sf_ok = wait_phase(c, kBarSfReady + i, gstep & 1u, true);
        if (!sf_ok) break;
        tc_fence_after();
        issue_qk_mx(tS[i], sQ[i], sK, mx_sf_qk(tS, i), mx_sf_qk(tS, i) + 4);
      } else {
        issue_qk<(kF8 >= 1)>(tS[i], sQ[i], sK);
      }
      tc_commit(c.bar(kBarSFull + i));
    }
    if (!sf_ok) break;
    if (n == 1) tc_commit(c.bar(kBarQEmpty));   // the segment's last S MMA is issued
    // The segment's first P V products overwrite O: the previous segment's epilogue must
    // have read both accumulators out of TMEM.
    if (u > 0 && (!wait_phase(c, kBarOEmpty + 0, (u - 1) & 1, true) ||
                  !wait_phase(c, kBarOEmpty + 1, (u - 1) & 1, true)))
      break;
    bool ok = true;
    int j = 0;
    for (; j + 1 < n; ++j) {
      if (!mma_step<true, kF8>(c, base, tS, tO, sQ, unit + 1 + j, (gstep + j) & 1u, j == 0)) {
        ok = false;
        break;
      }
    }
    if (!ok) break;
    if (n > 1) tc_commit(c.bar(kBarQEmpty));   // the last S MMA (step n-2) is issued
    if (!mma_step<false, kF8>(c, base, tS, tO, sQ, unit + 1 + j, (gstep + j) & 1u, j == 0)) break;
    unit += n + 1;
    gstep += static_cast<uint32_t>(n);
    ++u;
  }
  // Every MMA this thread issued must finish before TMEM and shared memory are released.
  tc_commit(c.bar(kBarDrain));
  wait_phase(c, kBarDrain, 0, false);
}

// Stores one 64-column half of this warp's 32 output rows (pk: the calling thread's own
// row, packed BF16 pairs). The rows go through the warp's staging tile in shared memory
// (16-byte chunks swizzled by row) so that each global store instruction covers four
// whole 128-byte lines instead of touching 32 lines with 16 bytes each. Rows from
// valid_rows on are not stored.
__device__ __forceinline__ void store_half_rows(uint8_t* stage, const uint32_t (&pk)[32], uint16_t* o_row0,
                                                int valid_rows, int half) {
  const int lane = threadIdx.x & 31;
  uint4* st = reinterpret_cast<uint4*>(stage);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    st[lane * 8 + (k ^ (lane & 7))] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = i * 4 + (lane >> 3), cc = lane & 7;   // row within the warp, 16-byte chunk
    const uint4 v = st[rr * 8 + (cc ^ (rr & 7))];
    if (rr < valid_rows) reinterpret_cast<uint4*>(o_row0 + static_cast<size_t>(rr) * kD + half * 64)[cc] = v;
  }
  __syncwarp();
}

// Merges the partial records of one split group for this thread's query row (the
// calling warp was the last of the group's shares to finish these 32 rows). With
// m_s, l_s, corr_s, O_s the running max, sums and unnormalised output of share s and
// M = max m_s, w_s = 2^(m_s - M): O = sum w_s O_s / sum w_s (l_s + corr_s) and
// LSE = (M + log2 sum w_s l_s) * ln 2. Shares are visited in block order, so the
// result does not depend on which share finished last.
// When own_tO is non-zero the calling block's own share is still in TMEM (O at own_tO,
// its max and sums in own_m, own_l, own_corr) and its record is not read. O is also
// multiplied by o_scale (V's descale factor when V is given as FP8 codes, else 1).
// kO32: the row goes to o32_row in FP32 (null for rows past the sequence) instead of BF16.
template <bool kO32 = false>
__device__ void merge_split_row(const Params& p, int tile, int r, int c_first, int c_last, long long x0,
                                uint8_t* stage, uint16_t* o_row0, int valid_rows, float* lse_out, uint32_t own_tO,
                                float own_m, float own_l, float own_corr, float o_scale, float* o32_row) {
  const int self = own_tO != 0 ? static_cast<int>(blockIdx.x) : -1;
  // share cs's record: its first segment's slot when its share starts inside this group,
  // else its last segment's
  auto record = [&](int cs) -> const float* {
    const int which = p.cuts[cs] >= x0 ? 0 : 1;
    return p.part + (static_cast<size_t>(cs) * 2 + which) * kQTiles * kPartFloatsPerTile +
           static_cast<size_t>(tile) * kPartFloatsPerTile;
  };
  constexpr int kM = kD * kBM, kL = kM + kBM, kC = kL + kBM;
  // Every sum runs over the shares in share order, the merging block's own share in its
  // place, so the result does not depend on which block happened to finish last.
  float M = -INFINITY;
  for (int cs = c_first; cs <= c_last; ++cs) M = fmaxf(M, cs == self ? own_m : __ldcg(record(cs) + kM + r));
  float L = 0.0f, Lr = 0.0f;
  for (int cs = c_first; cs <= c_last; ++cs) {
    float m_s = own_m, l_s = own_l, c_s = own_corr;
    if (cs != self) {
      const float* rec = record(cs);
      m_s = __ldcg(rec + kM + r);
      l_s = __ldcg(rec + kL + r);
      c_s = __ldcg(rec + kC + r);
    }
    const float w = ex2(m_s - M);
    L += l_s * w;
    Lr += (l_s + c_s) * w;
  }
  const float inv = o_scale / Lr;   // o_scale: V's descale factor, else 1
  // Two 64-column halves; per half and share, the share's max and its 64 values are
  // requested together, so each share costs one round trip to L2 per half.
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    float acc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
    for (int cs = c_first; cs <= c_last; ++cs) {
      float v[64];
      float m_s = own_m;
      if (cs == self) {   // warp-uniform: the TMEM loads below are .sync.aligned
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t ov[32];
          tmem_ld32(own_tO + (2 * h + cc) * 32, ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * cc + i] = __uint_as_float(ov[i]);
        }
      } else {
        const float* rec = record(cs);
        m_s = __ldcg(rec + kM + r);
        const float4* rec4 = reinterpret_cast<const float4*>(rec);
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          const float4 t = __ldcg(rec4 + (h * 16 + g) * kBM + r);
          v[4 * g] = t.x;
          v[4 * g + 1] = t.y;
          v[4 * g + 2] = t.z;
          v[4 * g + 3] = t.w;
        }
      }
      const float w = ex2(m_s - M);
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = fmaf(v[i], w, acc[i]);
    }
    if constexpr (kO32) {
      if (o32_row != nullptr) {
        float4* dst = reinterpret_cast<float4*>(o32_row + h * 64);
#pragma unroll
        for (int g = 0; g < 16; ++g)
          dst[g] = make_float4(acc[4 * g] * inv, acc[4 * g + 1] * inv, acc[4 * g + 2] * inv, acc[4 * g + 3] * inv);
      }
    } else {
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) pk[i] = pack_bf16(acc[2 * i] * inv, acc[2 * i + 1] * inv);
      store_half_rows(stage, pk, o_row0, valid_rows, h);
    }
  }
  if (lse_out != nullptr) *lse_out = (M + log2f(L)) * 0.69314718055994531f;
}

// kP8: P is rounded to E4M3 (four keys per TMEM column) for an FP8 P V product; the
// running max then moves once it grows by 8 (log2 units), so that every p <= 2^8 stays
// below E4M3's largest value 448, and O is scaled by V's descale factor with 1 / l.
// kO32: O is written in FP32 to p.o32 (the value the BF16 output is rounded from).
// kMX (with kP8): Q, K and V are MXFP8; each tile's softmax warps also write scale factors
// into TMEM, in the layout the block-scaled MMA reads (each 32-lane quarter holds the same
// 4 columns: lane l, column c = the 4 scale bytes of operand row l + 32c, byte t for K block
// t): those of its own P V product (P's, all 2^0, and V^T's) at S columns 32..39 with P, and
// those of the other tile's next Q K^T (the other tile's Q rows and the key tile's K rows) at
// S columns 96..103, right after it has read its own scores out of those columns.
template <bool kPosScale, bool kBias, bool kP8 = false, bool kO32 = false, bool kMX = false>
__device__ void run_softmax(const Ctl& c, uint32_t tmem, uint8_t* stage, const Params& p, int tile) {
  constexpr float kTau = kP8 ? 8.0f : kRescaleLog2;
  const int quarter = (threadIdx.x >> 5) & 3;   // TMEM lanes this warp may access
  const int lane = threadIdx.x & 31;
  const int r = quarter * 32 + lane;            // query row within the tile
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tS = tmem + lane_off + tile * 128;
  const uint32_t tO = tmem + lane_off + 256 + tile * 128;
  // factor still to apply to s: with a bias, s already holds scale * q.k + B in natural units
  const float cs = kBias ? 1.4426950408889634f : (kPosScale ? p.scale_log2 : 1.0f);

  uint32_t gstep = 0;   // K/V steps of all previous segments: phase of s_full / p_full
  int u = 0;            // segments finished
  int unit = 0;         // K/V units of all previous segments
  // One thread of tile 1 releases the K/V ring: once S_1 of step j is complete, every MMA
  // issued before it (all readers of unit j: S_0 and S_1 of step j, the P V products of
  // step j - 1) has finished, and once O_1 is complete the segment's last unit is free.
  const bool releaser = tile == 1 && quarter == 0 && lane == 0;
  // One thread of tile 0 checks the ring for the MMA thread: before its first P arrival of
  // step j it has seen unit j + 1 ({V_j, K_j+1}) loaded, so the MMA thread's wait for that
  // P also covers the unit (the MMA thread's waits are what idle the tensor core). The
  // check is a non-blocking test issued when the step starts and read before the arrival,
  // so its latency hides behind the exponentials; a blocking wait follows only if the
  // unit was not there yet.
  const bool ringer = tile == 0 && quarter == 0 && lane == 0;
  SegIter si(p);
  Segment sg;
  while (si.next(sg)) {
    const int n = sg.kv1 - sg.kv0;
    // this warp's first query row (causal masking)
    const int seg_row0 = (sg.group % p.q_groups) * (kQTiles * kBM) + tile * kBM + quarter * 32;
    float m_used = -INFINITY;   // log2 units
    float l = 0.0f;             // sum of 2^(s*cs - m_used) in FP32
    float corr = 0.0f;          // BF16 rounding error of the largest term of each tile
    // bias of this warp's rows: each step's tile is loaded before the wait for its scores,
    // so the loads overlap that wait
    BiasRows br;
    uint32_t bg[kBias ? 64 : 1];
    if constexpr (kBias) {
      const int bh = sg.group / p.q_groups;
      br.row0 = seg_row0;
      br.rows_full = seg_row0 + 32 <= p.Nq;
      br.sq = p.bias_sq;
      br.s4 = 4 * p.bias_sq;
      br.piece = p.bias + static_cast<long long>(bh / p.H) * p.bias_sb + static_cast<long long>(bh % p.H) * p.bias_sh +
                 static_cast<long long>(seg_row0 + (lane >> 3)) * p.bias_sq + 8 * (lane & 7);
      br.own_row = p.bias + static_cast<long long>(bh / p.H) * p.bias_sb + static_cast<long long>(bh % p.H) * p.bias_sh +
                   static_cast<long long>(seg_row0 + lane) * p.bias_sq;
      br.own_in = seg_row0 + lane < p.Nq;
    }
    // MXFP8: the other tile's query scales for the whole segment; per step, the scales of
    // the key tile whose Q K^T the other tile computes next and of this step's V^T tile
    uint32_t sf_qo[kMX ? 4 : 1], sf_k[kMX ? 4 : 1], sf_v[kMX ? 4 : 1];
    const int bh_mx = sg.group / p.q_groups;
    auto mx_load_k = [&](int kt) {   // key tile kt: rows kt*128 + lane + 32c
      if constexpr (kMX) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int key = kt * kBN + lane + 32 * cc;
          sf_k[cc] = key < p.Nk ? __ldg(p.sfk + static_cast<size_t>(bh_mx) * p.Nk + key) : 0x7F7F7F7Fu;
        }
      }
    };
    auto mx_load_v = [&](int kt) {   // V^T rows lane + 32c, key blocks 4kt .. 4kt+3 (past the keys: 2^0)
      if constexpr (kMX) {
        const int nkb = (p.Nk + 31) / 32;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(
              p.sfv + (static_cast<size_t>(bh_mx) * kD + lane + 32 * cc) * static_cast<size_t>(p.ldsv) + 4 * kt));
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (4 * kt + t >= nkb) w = (w & ~(0xFFu << (8 * t))) | (0x7Fu << (8 * t));
          sf_v[cc] = w;
        }
      }
    };
    auto mx_store_qk = [&]() {   // the other tile's next Q K^T: its Q rows, then the key rows
      if constexpr (kMX) {
        const uint32_t w[8] = {sf_qo[0], sf_qo[1], sf_qo[2], sf_qo[3], sf_k[0], sf_k[1], sf_k[2], sf_k[3]};
        tmem_st8(tS + 96, w);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(c.bar(kBarSfReady + (1 - tile)));
        __syncwarp();
      }
    };
    if constexpr (kMX) {
      const int orow0 = (sg.group % p.q_groups) * (kQTiles * kBM) + (1 - tile) * kBM;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int row = orow0 + lane + 32 * cc;
        sf_qo[cc] = row < p.Nq ? __ldg(p.sfq + static_cast<size_t>(bh_mx) * p.Nq + row) : 0x7F7F7F7Fu;
      }
      if (tile == 1) {   // the segment's first S_0: S_1's columns are free once the last segment ended
        mx_load_k(sg.kv0);
        mx_store_qk();
      }
    }
    for (int j = 0; j < n; ++j) {
      if constexpr (kBias) {
        load_bias_pieces(bg, br, p.Nq, (sg.kv0 + j) * kBN, p.Nk);
        // the next step's bias of this lane's row (two 128-byte lines) into L2 meanwhile
        const int k1 = (sg.kv0 + j + 1) * kBN;
        if (j + 1 < n && br.own_in && k1 + kBN <= p.Nk) {
          asm volatile("prefetch.global.L2 [%0];" ::"l"(br.own_row + k1));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(br.own_row + k1 + 64));
        }
      }
      if constexpr (kMX) {   // loads in flight while the step's scores are awaited
        mx_load_v(sg.kv0 + j);
        if (tile == 0 || j + 1 < n) mx_load_k(sg.kv0 + j + tile);
      }
      if (!wait_warp(c, kBarSFull + tile, (gstep + static_cast<uint32_t>(j)) & 1u)) return;
      if (releaser) mbar_arrive(c.bar(kBarKVEmpty + (unit + j) % kPairs));
      const int ring_unit = unit + j + 1;
      const bool ring_seen = ringer && mbar_test_wait(c.bar(kBarKVFull + ring_unit % kPairs), (ring_unit / kPairs) & 1);
      __syncwarp();   // lane 0 alone may have run the two lines above; tcgen05.ld is .sync.aligned
      tc_fence_after();
      float s[128];
      if constexpr (kBias) {
        // s = scale * q.k + B, one 64-key half at a time
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t b[32];
          bias_half_to_row(stage, bg, h, b);
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            uint32_t x[32];
            tmem_ld32(tS + h * 64 + q2 * 32, x);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t b2 = b[q2 * 16 + i];
              fma2v(s[h * 64 + q2 * 32 + 2 * i], s[h * 64 + q2 * 32 + 2 * i + 1], __uint_as_float(x[2 * i]),
                    __uint_as_float(x[2 * i + 1]), p.scale, __uint_as_float(b2 << 16),
                    __uint_as_float(b2 & 0xffff0000u));
            }
          }
        }
      } else {
        uint32_t x[128];
        tmem_ld128(tS, x);
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(x[i]);
        if (!kPosScale) {
#pragma unroll
          for (int i = 0; i < 128; ++i) s[i] *= p.scale_log2;
        }
      }
      if constexpr (kMX) {
        // the scores are in registers: this step's P V scales go next to P (P's own are 2^0),
        // and the other tile's next Q K^T scales into columns 96..103
        const uint32_t wv[8] = {0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, sf_v[0], sf_v[1], sf_v[2], sf_v[3]};
        tmem_st8(tS + 32, wv);
        if (tile == 0 || j + 1 < n) mx_store_qk();
      }
      if (sg.kv0 + j == p.n_kv - 1 && p.kv_tail < kBN) {
        const int valid = p.kv_tail;
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = (i < valid) ? s[i] : -INFINITY;
      }
      if (p.causal) {
        // key (kv0 + j) * 128 + i is visible to this row iff it is <= row + causal_off
        const int lim_warp = seg_row0 + p.causal_off - (sg.kv0 + j) * kBN;   // the warp's first row
        if (lim_warp < kBN - 1) {   // warp-uniform: some row of this warp has keys masked here
          const int lim = lim_warp + lane;
#pragma unroll
          for (int i = 0; i < 128; ++i) s[i] = (i <= lim) ? s[i] : -INFINITY;
        }
      }
      // row max: eight independent three-input max chains over s[0..127]
      // (chain t covers s[t], s[t + 8], s[t + 16], ..., s[t + 120])
      float mx[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) mx[t] = fmaxf(s[t], s[t + 8]);             // s[0..15]
#pragma unroll
      for (int i = 16; i < 128; i += 16) {                                    // i = 16, 32, ..., 112
#pragma unroll
        for (int t = 0; t < 8; ++t) mx[t] = max3(mx[t], s[i + t], s[i + 8 + t]);  // s[i..i+15]
      }
      const float m_raw =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float m_tile = m_raw * cs;
      bool rescale = false;
      float alpha = 1.0f;
      if (m_tile > m_used + kTau) {
        alpha = ex2(m_used - m_tile);   // 0 on the first step of a segment
        l *= alpha;
        corr *= alpha;
        m_used = m_tile;
        rescale = j > 0;
      }
      // O must be rescaled before this step's first P V MMA accumulates into it.
      if (__any_sync(0xffffffffu, rescale)) {
        const float a = rescale ? alpha : 1.0f;
#pragma unroll 1
        for (int ch = 0; ch < 16; ++ch) {   // small chunks: s[] is still live here
          uint32_t ov[8];
          tmem_ld8(tO + ch * 8, ov);
#pragma unroll
          for (int i = 0; i < 8; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * a);
          tmem_st8(tO + ch * 8, ov);
        }
      }
      // every p is 0 then: a row that has seen only -inf (a bias, or keys past its diagonal
      // in a causal share that starts after them)
      const float neg_m = ((kBias || p.causal) && m_used == -INFINITY) ? 0.0f : -m_used;
      // The BF16 rounding of P matters most for the tile's largest term, which the stale
      // running max leaves anywhere in [1, 2^kRescaleLog2]. corr accumulates that term's
      // rounding error, so that l + corr is the sum of the weights the tensor core
      // actually applies to V (up to the far smaller errors of the other terms). The term
      // is recomputed with exactly the arithmetic that produces it below (one FMA of the
      // raw maximum score, then ex2): a value computed another way can differ in its last
      // bit and round to the other BF16 neighbour, which would put a whole BF16 ulp of the
      // row's dominant weight into the sum.
      {
        // (with a bias a row may have seen only -inf so far: its largest term is then 0)
        const float pm = (kBias && m_tile == -INFINITY) ? 0.0f : ex2(fmaf(m_raw, cs, neg_m));
        if constexpr (kP8)
          corr += round_e4m3(pm) - pm;
        else
          corr += __uint_as_float(pack_bf16(pm, 0.0f) << 16) - pm;
      }
      // p = 2^(s*cs - m) in two halves of 64 keys; each half is rounded to BF16, stored
      // over S in TMEM and handed to the MMA warp at once, so the first half of the
      // P V product runs while the second half is computed.
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if constexpr (kP8) {   // 64 keys = 16 columns of four E4M3 values
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int e = half * 64 + 4 * i;
            float e0, e1, e2, e3;
            fma2(e0, e1, s[e], s[e + 1], cs, neg_m);
            fma2(e2, e3, s[e + 2], s[e + 3], cs, neg_m);
            e0 = ex2(e0);
            e1 = ex2(e1);
            e2 = ex2(e2);
            e3 = ex2(e3);
            pk[i] = pack_e4m3x4(e0, e1, e2, e3);
            add2(acc[2 * (i & 3)], acc[2 * (i & 3) + 1], e0, e1);
            add2(acc[2 * ((i + 2) & 3)], acc[2 * ((i + 2) & 3) + 1], e2, e3);
          }
          tmem_st16(tS + half * 16, pk);
        } else {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int e = half * 64 + 2 * i;
            float e0, e1;
            fma2(e0, e1, s[e], s[e + 1], cs, neg_m);
            e0 = ex2(e0);
            e1 = ex2(e1);
            pk[i] = pack_bf16(e0, e1);
            add2(acc[2 * (i & 3)], acc[2 * (i & 3) + 1], e0, e1);
          }
          tmem_st32(tS + half * 32, pk);
        }
        tc_fence_before();
        __syncwarp();
        // (on expiry the abort flag is set and the block winds down; arriving is harmless)
        if (half == 0 && ringer && !ring_seen)
          wait_phase(c, kBarKVFull + ring_unit % kPairs, (ring_unit / kPairs) & 1, true);
        if (lane == 0) mbar_arrive(c.bar(kBarPFull + 2 * tile + half));
        __syncwarp();   // reconverge before the next .sync.aligned TMEM access
      }

      l += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    }

    if (!wait_warp(c, kBarOFull + tile, u & 1)) return;
    if (releaser) mbar_arrive(c.bar(kBarKVEmpty + (unit + n) % kPairs));
    __syncwarp();
    unit += n + 1;
    tc_fence_after();
    const int bh = sg.group / p.q_groups;
    const int qrow_w0 = (sg.group % p.q_groups) * (kQTiles * kBM) + tile * kBM + quarter * 32;   // warp's first row
    const int qrow = qrow_w0 + lane;
    const bool live = qrow < p.Nq;
    const int valid_rows = p.Nq - qrow_w0;   // rows of this warp inside the sequence (may be <= 0)
    const size_t row_id = static_cast<size_t>(bh) * static_cast<size_t>(p.Nq) + static_cast<size_t>(qrow);
    uint16_t* o_row0 = p.o + (static_cast<size_t>(bh) * static_cast<size_t>(p.Nq) + static_cast<size_t>(qrow_w0)) * kD;
    if (!sg.split) {
      const float inv_l = kP8 ? p.v_scale / (l + corr) : 1.0f / (l + corr);
      // O in one TMEM load; the accumulator is handed back to the MMA thread at once, so
      // the next segment's first P V products can run while this one's rows are stored.
      uint32_t ov[128];
      tmem_ld128(tO, ov);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(kBarOEmpty + tile));
      __syncwarp();
      if constexpr (kO32) {
        if (live) {
          float4* dst = reinterpret_cast<float4*>(p.o32 + row_id * kD);
#pragma unroll
          for (int g = 0; g < kD / 4; ++g)
            dst[g] = make_float4(__uint_as_float(ov[4 * g]) * inv_l, __uint_as_float(ov[4 * g + 1]) * inv_l,
                                 __uint_as_float(ov[4 * g + 2]) * inv_l, __uint_as_float(ov[4 * g + 3]) * inv_l);
        }
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            pk[i] = pack_bf16(__uint_as_float(ov[64 * h + 2 * i]) * inv_l, __uint_as_float(ov[64 * h + 2 * i + 1]) * inv_l);
          store_half_rows(stage, pk, o_row0, valid_rows, h);
        }
      }
      if (live) p.lse[row_id] = (m_used + log2f(l)) * 0.69314718055994531f;
    } else {
      // This block holds only some key steps of the group. Counters count, per 32 rows,
      // the shares that have left their record; the last share to finish merges.
      const long long x0 = sg.x0;
      const int grid = static_cast<int>(gridDim.x);
      const int c_first = sk_block_of(x0, p, grid);
      const int c_last = sk_block_of(x0 + sg.glen - 1, p, grid);
      unsigned int* ctr = p.cnt + (static_cast<long long>(sg.cidx) * kQTiles + tile) * 4 + quarter;
      unsigned int arrived = 0;
      if (lane == 0) arrived = ld_acquire(ctr);
      __syncwarp();
      arrived = __shfl_sync(0xffffffffu, arrived, 0);
      if (static_cast<int>(arrived) == c_last - c_first) {
        // Every other share has left its record: merge with this share's O straight
        // from TMEM, without writing a record of its own.
        __threadfence();
        merge_split_row<kO32>(p, tile, r, c_first, c_last, x0, stage, o_row0, valid_rows,
                              live ? p.lse + row_id : nullptr, tO, m_used, l, corr, kP8 ? p.v_scale : 1.0f,
                              kO32 && live ? p.o32 + row_id * kD : nullptr);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(c.bar(kBarOEmpty + tile));
      } else {
        float* rec = p.part + (static_cast<size_t>(blockIdx.x) * 2 + sg.which) * kQTiles * kPartFloatsPerTile +
                     static_cast<size_t>(tile) * kPartFloatsPerTile;
        {
          uint32_t ov[128];
          tmem_ld128(tO, ov);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(c.bar(kBarOEmpty + tile));   // O_tile may be overwritten now
          __syncwarp();
          float4* rec4 = reinterpret_cast<float4*>(rec);
#pragma unroll
          for (int g = 0; g < kD / 4; ++g)   // 512 contiguous bytes per warp
            rec4[g * kBM + r] = make_float4(__uint_as_float(ov[4 * g]), __uint_as_float(ov[4 * g + 1]),
                                            __uint_as_float(ov[4 * g + 2]), __uint_as_float(ov[4 * g + 3]));
        }
        rec[kD * kBM + r] = m_used;
        rec[kD * kBM + kBM + r] = l;
        rec[kD * kBM + 2 * kBM + r] = corr;
        __threadfence();
        __syncwarp();
        unsigned int before = 0;
        if (lane == 0) before = atomicAdd(ctr, 1u);
        before = __shfl_sync(0xffffffffu, before, 0);
        if (static_cast<int>(before) == c_last - c_first) {
          __threadfence();
          merge_split_row<kO32>(p, tile, r, c_first, c_last, x0, stage, o_row0, valid_rows,
                                live ? p.lse + row_id : nullptr, 0u, 0.0f, 0.0f, 0.0f, kP8 ? p.v_scale : 1.0f,
                                kO32 && live ? p.o32 + row_id * kD : nullptr);
        }
      }
    }
    gstep += static_cast<uint32_t>(n);
    ++u;
  }
}

// ---------------------------------------------------------------------------------
// Kernel
// ---------------------------------------------------------------------------------
template <bool kPosScale, bool kBias, int kF8 = 0, bool kO32 = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  Ctl c;
  c.bars = base + kOffBar;
  c.abort = reinterpret_cast<volatile uint32_t*>(smem + kOffAbort);
  c.limit = p.wait_limit;

  // Counters of the next launch that shares this workspace: zero this block's slice now,
  // before any wait, so that it happens even if this launch gives up later.
  if (p.cnt_next != nullptr) {
    const int lo = static_cast<int>(static_cast<long long>(blockIdx.x) * p.cnt_len / gridDim.x);
    const int hi = static_cast<int>((static_cast<long long>(blockIdx.x) + 1) * p.cnt_len / gridDim.x);
    for (int i = lo + static_cast<int>(threadIdx.x); i < hi; i += kThreads) p.cnt_next[i] = 0u;
  }
  if (threadIdx.x == 0) {
    mbar_init(c.bar(kBarQFull), 1);
    mbar_init(c.bar(kBarQEmpty), 1);
    for (int q = 0; q < kPairs; ++q) {
      mbar_init(c.bar(kBarKVFull + q), 1);
      mbar_init(c.bar(kBarKVEmpty + q), 1);   // released by one softmax thread of tile 1
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(c.bar(kBarSFull + t), 1);
      mbar_init(c.bar(kBarPFull + 2 * t), 4);       // one arrival per softmax warp
      mbar_init(c.bar(kBarPFull + 2 * t + 1), 4);
      mbar_init(c.bar(kBarOFull + t), 1);
      mbar_init(c.bar(kBarOEmpty + t), 4);          // one arrival per softmax warp
    }
    mbar_init(c.bar(kBarDrain), 1);
    for (int t = 0; t < kQTiles; ++t) mbar_init(c.bar(kBarSfReady + t), 4);   // one arrival per softmax warp
    *c.abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + kOffTmemSlot),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);

  // Whole warpgroups: warps 0-3 give registers back, warps 4-11 take them.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (warp == 0) {
      if (lane == 0) run_producer<kF8>(c, base, &tmQ, &tmK, &tmV, p);
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) run_mma<kF8>(c, base, tmem, p);
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    run_softmax<kPosScale, kBias, kF8 >= 2, kO32, kF8 == 3>(c, tmem, smem + kOffStage + (warp - 4) * kStageBytes, p, (warp >> 2) - 1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}


// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
std::atomic<unsigned long long> g_wait_limit{kDefaultWaitLimit};
std::atomic<int> g_withhold{0};
std::atomic<unsigned long long> g_launches{0};

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

// [BH, rows, 128] viewed as a 3-D tensor (d innermost). BF16: box = 64 columns x 128 rows x 1;
// 8-bit codes (codes8): box = 128 columns x 128 rows x 1. Either way one box row is 128 bytes,
// the span of the 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* ptr, int rows, long long bh, bool codes8 = false) {
  auto enc = encoder();
  if (!enc) return false;
  const cuuint64_t esize = codes8 ? 1 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * esize, static_cast<cuuint64_t>(rows) * kD * esize};
  cuuint32_t box[3] = {codes8 ? 128u : 64u, static_cast<cuuint32_t>(kBM), 1};
  cuuint32_t elem[3] = {1, 1, 1};
  return enc(map, codes8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void*>(ptr), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// V^T as 8-bit codes, [BH, 128, ldv] with keys innermost (Nk of each row of ldv used); box =
// 128 keys x 128 rows of d x 1, one 128-byte swizzle span per row.
bool make_map_vt(CUtensorMap* map, const void* ptr, int Nk, long long ldv, long long bh) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(Nk), static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldv), static_cast<cuuint64_t>(ldv) * kD};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kBN), static_cast<cuuint32_t>(kD), 1};
  cuuint32_t elem[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_attr_done[18][kMaxDevices];   // per instantiation (kPos + 2 * kBias + 4 * kF8, 16 + kPos for kO32)
std::atomic<int> g_sm_count[kMaxDevices];

int sm_count(int dev) {
  if (dev >= 0 && dev < kMaxDevices) {
    const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
    if (cached > 0) return cached;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return -1;
  if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

// How the groups are spread over the persistent blocks (see the kernel's header).
struct Plan {
  int grid = 1;
  long long dp_groups = 0;   // processed whole, round-robin
  long long sk_groups = 0;   // their key steps shared out over the blocks
  long long sk_steps = 0;
  std::vector<long long> cuts;   // grid + 1 share boundaries over the sk_steps
  bool has_split = false;    // some group's key steps end up in two or more blocks
};

// Share boundaries of a split region whose groups end at `bounds` (ascending, the last the
// region's total): block c takes steps [floor(cT/G), floor((c+1)T/G)). (Shares balanced on a
// cost that charges each further group a share enters about three steps, the start-up and
// merge a per-block timeline measured, came out 2-3 % slower on rect-4k-8k: the grid shrank
// and the shares that stay in one group grew.)
std::vector<long long> share_cuts(const std::vector<long long>& bounds, int grid) {
  const long long total = bounds.back();
  std::vector<long long> cuts;
  for (int c = 0; c <= grid; ++c) cuts.push_back(sk_share_start(c, total, grid));
  return cuts;
}

bool cuts_split_a_group(const std::vector<long long>& cuts, const std::vector<long long>& bounds) {
  for (size_t c = 1; c + 1 < cuts.size(); ++c)
    if (!std::binary_search(bounds.begin(), bounds.end(), cuts[c])) return true;
  return false;
}

Plan make_plan(long long n_groups, int n_kv, int sms) {
  Plan pl;
  sms = std::min(sms, kMaxGrid);
  if (n_groups >= sms) {
    pl.grid = sms;
    const long long waves = n_groups / sms, rem = n_groups % sms;
    // Whole waves of whole groups; the remainder plus one full wave is split, which gives
    // every block between one and two groups' worth of key steps in the split part.
    pl.dp_groups = rem == 0 ? n_groups : (waves - 1) * sms;
  } else {
    const long long steps = n_groups * n_kv;
    long long g = steps / kMinSegSteps;
    pl.grid = static_cast<int>(g < 1 ? 1 : (g > sms ? sms : g));
    pl.dp_groups = 0;
  }
  pl.sk_groups = n_groups - pl.dp_groups;
  pl.sk_steps = pl.sk_groups * n_kv;
  if (pl.sk_steps > 0) {
    std::vector<long long> bounds;
    for (long long g = 1; g <= pl.sk_groups; ++g) bounds.push_back(g * n_kv);
    pl.cuts = share_cuts(bounds, pl.grid);
    pl.has_split = cuts_split_a_group(pl.cuts, bounds);
  }
  return pl;
}

// the plan's share boundaries into the launch parameters
void set_cuts(Params& p, const std::vector<long long>& cuts) {
  for (int c = 0; c <= kMaxGrid; ++c) p.cuts[c] = c < static_cast<int>(cuts.size()) ? cuts[c] : 0;
}

// Workspace for split groups, cached per (device, stream) so that calls on different
// streams never share one; calls on one stream are ordered by the stream.
struct Workspace {
  float* part = nullptr;
  unsigned int* cnt = nullptr;   // two banks of counters
  size_t part_bytes = 0, cnt_bytes = 0;   // cnt_bytes: one bank
  int bank = 0;                  // the bank the next launch uses; it is all zero
};
std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, Workspace> g_ws;

// Returns ATTN_OK and fills part and the two counter banks (current, next), or ATTN_ERR_CUDA.
int get_workspace(int dev, cudaStream_t stream, size_t part_bytes, size_t cnt_bytes, float** part,
                  unsigned int** cnt, unsigned int** cnt_next, int* bank_len) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  Workspace& ws = g_ws[std::make_pair(dev, reinterpret_cast<uintptr_t>(stream))];
  if (ws.part_bytes < part_bytes) {
    if (ws.part) cudaFreeAsync(ws.part, stream);
    ws.part = nullptr;
    ws.part_bytes = 0;
    if (cudaMallocAsync(reinterpret_cast<void**>(&ws.part), part_bytes, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    ws.part_bytes = part_bytes;
  }
  if (ws.cnt_bytes < cnt_bytes) {
    if (ws.cnt) cudaFreeAsync(ws.cnt, stream);
    ws.cnt = nullptr;
    ws.cnt_bytes = 0;
    if (cudaMallocAsync(reinterpret_cast<void**>(&ws.cnt), 2 * cnt_bytes, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemsetAsync(ws.cnt, 0, 2 * cnt_bytes, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    ws.cnt_bytes = cnt_bytes;
    ws.bank = 0;
  }
  const size_t bank_words = ws.cnt_bytes / sizeof(unsigned int);
  *part = ws.part;
  *cnt = ws.cnt + ws.bank * bank_words;
  *cnt_next = ws.cnt + (ws.bank ^ 1) * bank_words;
  *bank_len = static_cast<int>(bank_words);
  ws.bank ^= 1;
  return ATTN_OK;
}

template <bool kPos, bool kBias = false, int kF8 = 0, bool kO32 = false>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const Params& p, int grid,
           int dev, cudaStream_t stream) {
  auto kern = attn_fwd_kernel<kPos, kBias, kF8, kO32>;
  constexpr int kInst = kO32 ? 16 + (kPos ? 1 : 0) : (kPos ? 1 : 0) + (kBias ? 2 : 0) + 4 * kF8;
  if (dev < 0 || dev >= kMaxDevices || !g_attr_done[kInst][dev].load(std::memory_order_acquire)) {
    // The in-kernel register split (setmaxnreg) balances only at kRegsLaunch registers
    // per thread; at any other count the increase would never be granted. Refuse.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.numRegs != kRegsLaunch) return ATTN_ERR_CUDA;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) g_attr_done[kInst][dev].store(1, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  if (cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, p) != cudaSuccess) return ATTN_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return ATTN_OK;
}

struct BiasArg {
  const void* ptr;
  long long sb, sh, sq;
};

// MXFP8 block scales (attn_fwd_mxfp8)
struct MxArg {
  const void* sq;   // [BH, Nq, 4] bytes
  const void* sk;   // [BH, Nk, 4] bytes
  const void* svt;  // [BH, 128, ldsv] bytes
  long long ldsv;
};

// attn_fwd_bias's rules for its bias argument.
int check_bias(const BiasArg& bias, int B, int H, int Nq) {
  if (!bias.ptr || bias.sb < 0 || bias.sh < 0 || bias.sq < 0) return ATTN_ERR_INVALID_ARG;
  // the last element's offset, (B-1) sb + (H-1) sh + (Nq-1) sq + Nk - 1, in bytes must fit int64
  constexpr long long kCap = LLONG_MAX / 8;
  const long long ext[3] = {B - 1LL, H - 1LL, Nq - 1LL};
  const long long str[3] = {bias.sb, bias.sh, bias.sq};
  for (int i = 0; i < 3; ++i)
    if (str[i] > 0 && ext[i] > kCap / str[i]) return ATTN_ERR_INVALID_ARG;
  // 16-byte vector loads of each row's 8-key chunks
  if ((reinterpret_cast<uintptr_t>(bias.ptr) & 15u) || ((bias.sb | bias.sh | bias.sq) & 7)) return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

// The 8-bit entry points' own argument rules (f8 as forward's).
int check_f8_args(int f8, long long ldv, const MxArg* mx, int Nk, long long bh) {
  if (f8 >= 2) {
    // V^T rows of ldv bytes: at least Nk, 16-byte multiples (TMA strides), and the last
    // byte's offset, bh * 128 * ldv, must fit a signed 64-bit offset
    if (ldv < Nk) return ATTN_ERR_INVALID_ARG;
    if (ldv % 16 != 0) return ATTN_ERR_MISALIGNED;
    if (bh > (LLONG_MAX / kD) / ldv) return ATTN_ERR_INVALID_ARG;
  }
  if (f8 == 3) {
    // scale rows: 4 bytes per Q or K row (read as words); V^T scale rows of ldsv bytes, a
    // word per key tile of 128, so at least 4 * ceil(Nk / 128) bytes (those past the last
    // key block are read and replaced by 2^0)
    if (mx == nullptr || !mx->sq || !mx->sk || !mx->svt) return ATTN_ERR_INVALID_ARG;
    const long long n_kv = (static_cast<long long>(Nk) + kBN - 1) / kBN;
    if (mx->ldsv < 4 * n_kv) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(mx->sq) | reinterpret_cast<uintptr_t>(mx->sk) |
         reinterpret_cast<uintptr_t>(mx->svt)) & 3u || mx->ldsv % 16 != 0)
      return ATTN_ERR_MISALIGNED;
    if (bh > (LLONG_MAX / kD) / mx->ldsv) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

// attn_fwd, attn_fwd_bias (bias != nullptr), attn_fwd_fp8qk (f8 = 1: q and k hold FP8 E4M3
// codes), attn_fwd_fp8 (f8 = 2: v too, as V^T with row stride ldv, descaled by v_scale) and
// attn_fwd_o32 (o32 != nullptr: O in FP32 there, o unused): the argument rules, the plan,
// the launch.
int forward(const void* q, const void* k, const void* v, const BiasArg* bias, void* o, float* lse, int B, int H,
            int Nq, int Nk, int d, float scale, void* stream, int f8 = 0, long long ldv = 0, float v_scale = 1.0f,
            float* o32 = nullptr, const MxArg* mx = nullptr) {
  const bool qk8 = f8 >= 1;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (d != kD) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  if (bh == 0 || Nq == 0) return ATTN_OK;   // nothing to compute
  if (Nk == 0) return ATTN_ERR_INVALID_ARG;  // softmax over an empty key set
  if (o32 != nullptr) o = o32;               // the output, whichever type it has
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(o)) & 15u)
    return ATTN_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return ATTN_ERR_MISALIGNED;
  // index ranges: TMA coordinates and group indices are 32-bit
  const long long q_groups = (static_cast<long long>(Nq) + kQTiles * kBM - 1) / (kQTiles * kBM);
  if (bh > INT_MAX || bh * q_groups > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  // element counts must fit a signed 64-bit byte offset
  const long long max_rows = static_cast<long long>(Nq > Nk ? Nq : Nk);
  if (bh > (LLONG_MAX / 256) / max_rows) return ATTN_ERR_INVALID_ARG;
  if (const int rc = check_f8_args(f8, ldv, mx, Nk, bh); rc != ATTN_OK) return rc;
  if (bias != nullptr)
    if (const int rc = check_bias(*bias, B, H, Nq); rc != ATTN_OK) return rc;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  const int sms = sm_count(dev);
  if (sms <= 0) return ATTN_ERR_CUDA;

  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, Nq, bh, qk8) || !make_map(&mk, k, Nk, bh, qk8) ||
      !(f8 >= 2 ? make_map_vt(&mv, v, Nk, ldv, bh) : make_map(&mv, v, Nk, bh)))
    return ATTN_ERR_CUDA;

  Params p;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.Nq = Nq;
  p.Nk = Nk;
  p.q_groups = static_cast<int>(q_groups);
  p.n_kv = (Nk + kBN - 1) / kBN;
  p.kv_tail = Nk - (p.n_kv - 1) * kBN;
  const Plan pl = make_plan(bh * q_groups, p.n_kv, sms);
  p.dp_groups = static_cast<int>(pl.dp_groups);
  p.sk_steps = pl.sk_steps;
  set_cuts(p, pl.cuts);
  p.part = nullptr;
  p.cnt = nullptr;
  p.cnt_next = nullptr;
  p.cnt_len = 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  p.withhold_tile = g_withhold.load(std::memory_order_relaxed);
  p.causal = 0;
  p.causal_off = 0;
  p.bh_count = static_cast<int>(bh);
  p.bias = bias ? static_cast<const uint16_t*>(bias->ptr) : nullptr;
  p.bias_sb = bias ? bias->sb : 0;
  p.bias_sh = bias ? bias->sh : 0;
  p.bias_sq = bias ? bias->sq : 0;
  p.H = H;
  p.scale = scale;
  p.v_scale = v_scale;
  p.o32 = o32;
  if (mx != nullptr) {
    p.sfq = static_cast<const uint32_t*>(mx->sq);
    p.sfk = static_cast<const uint32_t*>(mx->sk);
    p.sfv = static_cast<const uint8_t*>(mx->svt);
    p.ldsv = mx->ldsv;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pl.has_split) {
    const size_t part_bytes = static_cast<size_t>(pl.grid) * kPartBytesPerBlock;
    const size_t cnt_bytes = static_cast<size_t>(pl.sk_groups) * kQTiles * 4 * sizeof(unsigned int);
    // a later launch may use more counters than this one: it zeroes the whole other bank
    const int rc = get_workspace(dev, s, part_bytes, cnt_bytes, &p.part, &p.cnt, &p.cnt_next, &p.cnt_len);
    if (rc != ATTN_OK) return rc;
  }
  if (o32 != nullptr)
    return scale > 0.0f ? launch<true, false, 0, true>(mq, mk, mv, p, pl.grid, dev, s)
                        : launch<false, false, 0, true>(mq, mk, mv, p, pl.grid, dev, s);
  // with a bias the scale is applied before the row max, so one instantiation serves any sign
  if (bias != nullptr) {
    if (f8 == 2) return launch<true, true, 2>(mq, mk, mv, p, pl.grid, dev, s);
    if (f8 == 1) return launch<true, true, 1>(mq, mk, mv, p, pl.grid, dev, s);
    if (f8 != 0) return ATTN_ERR_UNSUPPORTED;
    return launch<true, true>(mq, mk, mv, p, pl.grid, dev, s);
  }
  if (f8 == 3)
    return scale > 0.0f ? launch<true, false, 3>(mq, mk, mv, p, pl.grid, dev, s)
                        : launch<false, false, 3>(mq, mk, mv, p, pl.grid, dev, s);
  if (f8 == 2)
    return scale > 0.0f ? launch<true, false, 2>(mq, mk, mv, p, pl.grid, dev, s)
                        : launch<false, false, 2>(mq, mk, mv, p, pl.grid, dev, s);
  if (qk8)
    return scale > 0.0f ? launch<true, false, 1>(mq, mk, mv, p, pl.grid, dev, s)
                        : launch<false, false, 1>(mq, mk, mv, p, pl.grid, dev, s);
  return scale > 0.0f ? launch<true>(mq, mk, mv, p, pl.grid, dev, s) : launch<false>(mq, mk, mv, p, pl.grid, dev, s);
}

}  // namespace

namespace {
// Head dimensions above 128: the one-Q-tile kernel (attn_fwd_wide.cu), after the argument
// checks of the d = 128 entry points (causal: also Nq <= Nk).
int forward_wide(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                 int d, float scale, bool causal, void* stream, const BiasArg* bias = nullptr, int f8 = 0,
                 long long ldv = 0, float v_scale = 1.0f) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H == 0 || Nq == 0) return ATTN_OK;
  if (Nk == 0 || (causal && Nq > Nk) || !q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (causal && Nk > INT_MAX - 1024) return ATTN_ERR_UNSUPPORTED;   // row + causal_off + 2 * 128 stays in int
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(o)) & 15u)
    return ATTN_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return ATTN_ERR_MISALIGNED;
  const long long max_rows = static_cast<long long>(Nq > Nk ? Nq : Nk);
  if (static_cast<long long>(B) * H > (LLONG_MAX / (2 * d)) / max_rows) return ATTN_ERR_INVALID_ARG;
  if (f8 == 2) {
    // V^T rows of ldv bytes: at least Nk, 16-byte multiples (TMA strides), and the last
    // byte's offset, B * H * d * ldv, must fit a signed 64-bit offset
    if (ldv < Nk) return ATTN_ERR_INVALID_ARG;
    if (ldv % 16 != 0) return ATTN_ERR_MISALIGNED;
    if (static_cast<long long>(B) * H > (LLONG_MAX / d) / ldv) return ATTN_ERR_INVALID_ARG;
  }
  attn_wide::Bias wb{};
  if (bias != nullptr) {
    if (const int rc = check_bias(*bias, B, H, Nq); rc != ATTN_OK) return rc;
    wb = {bias->ptr, bias->sb, bias->sh, bias->sq};
  }
  const int rc = attn_wide::forward(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, static_cast<cudaStream_t>(stream),
                                    g_wait_limit.load(std::memory_order_relaxed), bias != nullptr ? &wb : nullptr, f8,
                                    ldv, v_scale, g_withhold.load(std::memory_order_relaxed));
  if (rc == ATTN_OK) g_launches.fetch_add(1, std::memory_order_relaxed);
  return rc;
}
}  // namespace

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                        int Nk, int d, float scale, void* stream) {
  if (attn_wide::supported(d)) return forward_wide(q, k, v, o, lse, B, H, Nq, Nk, d, scale, false, stream);
  return forward(q, k, v, nullptr, o, lse, B, H, Nq, Nk, d, scale, stream);
}

extern "C" int attn_fwd_o32(const void* q, const void* k, const void* v, float* o32, float* lse, int B, int H,
                            int Nq, int Nk, int d, float scale, void* stream) {
  return forward(q, k, v, nullptr, nullptr, lse, B, H, Nq, Nk, d, scale, stream, 0, 0, 1.0f, o32);
}

extern "C" int attn_fwd_bias(const void* q, const void* k, const void* v, const void* bias, long long bias_stride_b,
                             long long bias_stride_h, long long bias_stride_q, void* o, float* lse, int B, int H,
                             int Nq, int Nk, int d, float scale, void* stream) {
  const BiasArg ba = {bias, bias_stride_b, bias_stride_h, bias_stride_q};
  if (attn_wide::supported(d)) return forward_wide(q, k, v, o, lse, B, H, Nq, Nk, d, scale, false, stream, &ba);
  return forward(q, k, v, &ba, o, lse, B, H, Nq, Nk, d, scale, stream);
}

extern "C" int attn_fwd_fp8qk(const void* q8, const void* k8, const void* v, void* o, float* lse, int B, int H,
                              int Nq, int Nk, int d, float scale, float q_descale, float k_descale,
                              void* stream) {
  // S = scale * q_descale * k_descale * (Q8 K8^T): the three factors are folded into one FP32
  // scale on the host; the codes' products are exact in the FP32 accumulators.
  if (!std::isfinite(scale) || !std::isfinite(q_descale) || !std::isfinite(k_descale) || !(q_descale > 0.0f) ||
      !(k_descale > 0.0f))
    return ATTN_ERR_INVALID_ARG;
  const double eff = static_cast<double>(scale) * q_descale * k_descale;
  if (!(std::fabs(eff) <= static_cast<double>(FLT_MAX))) return ATTN_ERR_INVALID_ARG;
  if (attn_wide::supported(d))
    return forward_wide(q8, k8, v, o, lse, B, H, Nq, Nk, d, static_cast<float>(eff), false, stream, nullptr, 1);
  return forward(q8, k8, v, nullptr, o, lse, B, H, Nq, Nk, d, static_cast<float>(eff), stream, 1);
}

extern "C" int attn_fwd_fp8(const void* q8, const void* k8, const void* vt8, long long ldv, void* o, float* lse,
                            int B, int H, int Nq, int Nk, int d, float scale, float q_descale, float k_descale,
                            float v_descale, void* stream) {
  // S = scale * q_descale * k_descale * (Q8 K8^T) as in attn_fwd_fp8qk; O = v_descale * P8 V8
  // with P rounded to E4M3 and the sum l of the unrounded weights.
  if (!std::isfinite(scale) || !std::isfinite(q_descale) || !std::isfinite(k_descale) ||
      !std::isfinite(v_descale) || !(q_descale > 0.0f) || !(k_descale > 0.0f) || !(v_descale > 0.0f))
    return ATTN_ERR_INVALID_ARG;
  const double eff = static_cast<double>(scale) * q_descale * k_descale;
  if (!(std::fabs(eff) <= static_cast<double>(FLT_MAX))) return ATTN_ERR_INVALID_ARG;
  if (attn_wide::supported(d))
    return forward_wide(q8, k8, vt8, o, lse, B, H, Nq, Nk, d, static_cast<float>(eff), false, stream, nullptr, 2,
                        ldv, v_descale);
  return forward(q8, k8, vt8, nullptr, o, lse, B, H, Nq, Nk, d, static_cast<float>(eff), stream, 2, ldv, v_descale);
}

extern "C" int attn_fwd_mxfp8(const void* q8, const void* sq, const void* k8, const void* sk, const void* vt8,
                              long long ldv, const void* svt, long long ldsv, void* o, float* lse, int B, int H, int Nq,
                              int Nk, int d, float scale, void* stream) {
  // S = scale * (Q K^T) from block-scaled E4M3 codes, O = P V with P rounded to E4M3 (scale
  // 2^0 per block) and V^T block-scaled per 32 keys; the tensor cores apply every scale.
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  const MxArg mx = {sq, sk, svt, ldsv};
  return forward(q8, k8, vt8, nullptr, o, lse, B, H, Nq, Nk, d, scale, stream, 3, ldv, 1.0f, nullptr, &mx);
}

namespace {
// The causal launches: whole (b, h, 256-row) groups, longest first, each over the key tiles
// its rows can see (the causal order of SegIter): no workspace, no merge. f8: 0 BF16 inputs,
// 1 Q and K as E4M3 codes, 2 V too (V^T rows of ldv bytes, v_scale its descale factor),
// 3 MXFP8 (mx: the block scales); scale already holds any Q and K descale factors.
int forward_causal(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                   int d, float scale, void* stream, int f8 = 0, long long ldv = 0, float v_scale = 1.0f,
                   const MxArg* mx = nullptr) {
  // the argument rules of attn_fwd, plus Nq <= Nk (every query row sees at least one key)
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (d != kD) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  if (bh == 0 || Nq == 0) return ATTN_OK;
  if (Nk == 0 || Nq > Nk) return ATTN_ERR_INVALID_ARG;
  if (Nk > INT_MAX - 1024) return ATTN_ERR_UNSUPPORTED;   // row + causal_off + 2 * kBN stays in int
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(o)) & 15u)
    return ATTN_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return ATTN_ERR_MISALIGNED;
  const long long q_groups = (static_cast<long long>(Nq) + kQTiles * kBM - 1) / (kQTiles * kBM);
  if (bh > INT_MAX || bh * q_groups > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  const long long max_rows = static_cast<long long>(Nk);
  if (bh > (LLONG_MAX / 256) / max_rows) return ATTN_ERR_INVALID_ARG;
  if (const int rc = check_f8_args(f8, ldv, mx, Nk, bh); rc != ATTN_OK) return rc;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  const int sms = sm_count(dev);
  if (sms <= 0) return ATTN_ERR_CUDA;

  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, Nq, bh, f8 >= 1) || !make_map(&mk, k, Nk, bh, f8 >= 1) ||
      !(f8 >= 2 ? make_map_vt(&mv, v, Nk, ldv, bh) : make_map(&mv, v, Nk, bh)))
    return ATTN_ERR_CUDA;

  const long long n_groups = bh * q_groups;
  Params p;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.Nq = Nq;
  p.Nk = Nk;
  p.q_groups = static_cast<int>(q_groups);
  p.n_kv = (Nk + kBN - 1) / kBN;
  p.kv_tail = Nk - (p.n_kv - 1) * kBN;
  p.dp_groups = 0;
  p.sk_steps = 0;
  set_cuts(p, {});
  p.part = nullptr;
  p.cnt = nullptr;
  p.cnt_next = nullptr;
  p.cnt_len = 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  p.withhold_tile = g_withhold.load(std::memory_order_relaxed);
  p.causal = 1;
  p.causal_off = Nk - Nq;
  p.bh_count = static_cast<int>(bh);
  p.bias = nullptr;
  p.bias_sb = p.bias_sh = p.bias_sq = 0;
  p.H = H;
  p.scale = scale;
  p.v_scale = v_scale;
  if (mx != nullptr) {
    p.sfq = static_cast<const uint32_t*>(mx->sq);
    p.sfk = static_cast<const uint32_t*>(mx->sk);
    p.sfv = static_cast<const uint8_t*>(mx->svt);
    p.ldsv = mx->ldsv;
  }
  // Few groups (under two waves): the list's key steps are shared out evenly and long
  // groups are split and merged (SegIter); otherwise whole groups in balanced waves.
  const int max_grid = std::min(sms, kMaxGrid);
  int grid = static_cast<int>(n_groups < max_grid ? n_groups : max_grid);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n_groups < 2LL * sms) {
    // the list's group boundaries: level l (diagonal position q_groups - 1 - l) holds bh
    // groups of len(l) steps
    std::vector<long long> bounds;
    long long total = 0;
    for (long long l = 0; l < q_groups; ++l) {
      const long long row_end = std::min<long long>(Nq, (q_groups - l) * (kQTiles * kBM));
      const long long len = (row_end + p.causal_off + kBN - 1) / kBN;
      for (long long h = 0; h < bh; ++h) bounds.push_back(total += len);
    }
    const long long g = total / kMinSegSteps;
    grid = static_cast<int>(g < 1 ? 1 : (g > max_grid ? max_grid : g));
    const std::vector<long long> cuts = share_cuts(bounds, grid);
    p.sk_steps = total;
    set_cuts(p, cuts);
    // a share boundary inside a group needs the merge workspace
    if (cuts_split_a_group(cuts, bounds)) {
      const size_t part_bytes = static_cast<size_t>(grid) * kPartBytesPerBlock;
      const size_t cnt_bytes = static_cast<size_t>(n_groups) * kQTiles * 4 * sizeof(unsigned int);
      const int rc = get_workspace(dev, s, part_bytes, cnt_bytes, &p.part, &p.cnt, &p.cnt_next, &p.cnt_len);
      if (rc != ATTN_OK) return rc;
    }
  }
  if (f8 == 3)
    return scale > 0.0f ? launch<true, false, 3>(mq, mk, mv, p, grid, dev, s)
                        : launch<false, false, 3>(mq, mk, mv, p, grid, dev, s);
  if (f8 == 2)
    return scale > 0.0f ? launch<true, false, 2>(mq, mk, mv, p, grid, dev, s)
                        : launch<false, false, 2>(mq, mk, mv, p, grid, dev, s);
  if (f8 == 1)
    return scale > 0.0f ? launch<true, false, 1>(mq, mk, mv, p, grid, dev, s)
                        : launch<false, false, 1>(mq, mk, mv, p, grid, dev, s);
  return scale > 0.0f ? launch<true>(mq, mk, mv, p, grid, dev, s) : launch<false>(mq, mk, mv, p, grid, dev, s);
}

// The FP8 entry points' factor checks: the effective score scale, or 0 with *rc set.
float fp8_scale(float scale, float q_descale, float k_descale, float v_descale, int* rc) {
  *rc = ATTN_OK;
  if (!std::isfinite(scale) || !std::isfinite(q_descale) || !std::isfinite(k_descale) ||
      !std::isfinite(v_descale) || !(q_descale > 0.0f) || !(k_descale > 0.0f) || !(v_descale > 0.0f)) {
    *rc = ATTN_ERR_INVALID_ARG;
    return 0.0f;
  }
  const double eff = static_cast<double>(scale) * q_descale * k_descale;
  if (!(std::fabs(eff) <= static_cast<double>(FLT_MAX))) *rc = ATTN_ERR_INVALID_ARG;
  return static_cast<float>(eff);
}
}  // namespace

extern "C" int attn_fwd_causal(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                               int Nq, int Nk, int d, float scale, void* stream) {
  if (attn_wide::supported(d)) return forward_wide(q, k, v, o, lse, B, H, Nq, Nk, d, scale, true, stream);
  return forward_causal(q, k, v, o, lse, B, H, Nq, Nk, d, scale, stream);
}
extern "C" int attn_fwd_fp8qk_causal(const void* q8, const void* k8, const void* v, void* o, float* lse, int B,
                                     int H, int Nq, int Nk, int d, float scale, float q_descale, float k_descale,
                                     void* stream) {
  int rc = ATTN_OK;
  const float eff = fp8_scale(scale, q_descale, k_descale, 1.0f, &rc);
  if (rc != ATTN_OK) return rc;
  if (attn_wide::supported(d)) return forward_wide(q8, k8, v, o, lse, B, H, Nq, Nk, d, eff, true, stream, nullptr, 1);
  return forward_causal(q8, k8, v, o, lse, B, H, Nq, Nk, d, eff, stream, 1);
}
extern "C" int attn_fwd_fp8_causal(const void* q8, const void* k8, const void* vt8, long long ldv, void* o,
                                   float* lse, int B, int H, int Nq, int Nk, int d, float scale, float q_descale,
                                   float k_descale, float v_descale, void* stream) {
  int rc = ATTN_OK;
  const float eff = fp8_scale(scale, q_descale, k_descale, v_descale, &rc);
  if (rc != ATTN_OK) return rc;
  if (attn_wide::supported(d))
    return forward_wide(q8, k8, vt8, o, lse, B, H, Nq, Nk, d, eff, true, stream, nullptr, 2, ldv, v_descale);
  return forward_causal(q8, k8, vt8, o, lse, B, H, Nq, Nk, d, eff, stream, 2, ldv, v_descale);
}
extern "C" int attn_fwd_fp8qk_bias(const void* q8, const void* k8, const void* v, const void* bias,
                                   long long bias_stride_b, long long bias_stride_h, long long bias_stride_q, void* o,
                                   float* lse, int B, int H, int Nq, int Nk, int d, float scale, float q_descale,
                                   float k_descale, void* stream) {
  // S = scale * q_descale * k_descale * (Q8 K8^T) + B: attn_fwd_fp8qk's scores with
  // attn_fwd_bias's bias, added after the (folded) scale
  int rc = ATTN_OK;
  const float eff = fp8_scale(scale, q_descale, k_descale, 1.0f, &rc);
  if (rc != ATTN_OK) return rc;
  const BiasArg ba = {bias, bias_stride_b, bias_stride_h, bias_stride_q};
  if (attn_wide::supported(d)) return forward_wide(q8, k8, v, o, lse, B, H, Nq, Nk, d, eff, false, stream, &ba, 1);
  return forward(q8, k8, v, &ba, o, lse, B, H, Nq, Nk, d, eff, stream, 1);
}
extern "C" int attn_fwd_fp8_bias(const void* q8, const void* k8, const void* vt8, long long ldv, const void* bias,
                                 long long bias_stride_b, long long bias_stride_h, long long bias_stride_q, void* o,
                                 float* lse, int B, int H, int Nq, int Nk, int d, float scale, float q_descale,
                                 float k_descale, float v_descale, void* stream) {
  int rc = ATTN_OK;
  const float eff = fp8_scale(scale, q_descale, k_descale, v_descale, &rc);
  if (rc != ATTN_OK) return rc;
  const BiasArg ba = {bias, bias_stride_b, bias_stride_h, bias_stride_q};
  if (attn_wide::supported(d))
    return forward_wide(q8, k8, vt8, o, lse, B, H, Nq, Nk, d, eff, false, stream, &ba, 2, ldv, v_descale);
  return forward(q8, k8, vt8, &ba, o, lse, B, H, Nq, Nk, d, eff, stream, 2, ldv, v_descale);
}
extern "C" int attn_fwd_mxfp8_causal(const void* q8, const void* sq, const void* k8, const void* sk,
                                     const void* vt8, long long ldv, const void* svt, long long ldsv, void* o,
                                     float* lse, int B, int H, int Nq, int Nk, int d, float scale, void* stream) {
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  const MxArg mx = {sq, sk, svt, ldsv};
  return forward_causal(q8, k8, vt8, o, lse, B, H, Nq, Nk, d, scale, stream, 3, ldv, 1.0f, &mx);
}

extern "C" int attn_fwd_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int h = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_attn_status, sizeof h, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  const int wide = attn_wide::take_status(s);   // the d > 128 kernel's own status word
  if (wide < 0) return ATTN_ERR_CUDA;
  if (h == 0) return wide ? ATTN_ERR_TIMEOUT : ATTN_OK;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_attn_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_ERR_TIMEOUT;
}

extern "C" const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

extern "C" int attn_fwd_set_wait_limit(unsigned long long cycles, int withhold_tile) {
  g_wait_limit.store(cycles ? cycles : kDefaultWaitLimit, std::memory_order_relaxed);
  g_withhold.store(withhold_tile ? 1 : 0, std::memory_order_relaxed);
  return ATTN_OK;
}

extern "C" unsigned long long attn_fwd_kernel_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int attn_fwd_plan(long long n_groups, int n_kv, int sms, long long* dp_groups, long long* cuts, int* grid,
                             int* has_split) {
  if (n_groups < 1 || n_kv < 1 || sms < 1 || !dp_groups || !cuts || !grid || !has_split) return ATTN_ERR_INVALID_ARG;
  const Plan pl = make_plan(n_groups, n_kv, sms);
  *dp_groups = pl.dp_groups;
  *grid = pl.grid;
  *has_split = pl.has_split ? 1 : 0;
  for (int c = 0; c <= kMaxGrid; ++c) cuts[c] = c < static_cast<int>(pl.cuts.size()) ? pl.cuts[c] : 0;
  return ATTN_OK;
}

// ---------------------------------------------------------------------------------
// Entry point that allocates nothing
// ---------------------------------------------------------------------------------
// Some callers must not allocate device memory once they are running: applications
// that budget all of the GPU's memory up front (an extra allocation could fail or push
// something else out), loops where an allocation may synchronise the device and stall
// the pipeline, and programs whose own allocator owns every byte of device memory. For
// them attn_fwd_noalloc runs the same kernel with its split-merge workspace in the
// fixed array below instead of a cudaMallocAsync allocation. The array belongs to this
// library's module: every GPU that loads the library holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;   // 48 MiB: the records of up to 186 SMs
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// The array's device address differs between CUDA contexts (the library's module is loaded
// into each context on its own, again after cudaDeviceReset), so it is cached per context,
// keyed by the context's process-unique id.
std::mutex g_noalloc_mu;
std::map<unsigned long long, void*> g_noalloc_addr;
using PFN_ctxGetCurrent = CUresult (*)(CUcontext*);
using PFN_ctxGetId = CUresult (*)(CUcontext, unsigned long long*);
PFN_ctxGetCurrent g_ctx_current = nullptr;
PFN_ctxGetId g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// The id of the calling thread's current context, or 0 when there is none yet.
unsigned long long current_context_id() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_ctxGetCurrent>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_ctxGetId>(fn);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current == nullptr || g_ctx_id == nullptr || g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      g_ctx_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}
}  // namespace

extern "C" int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                int Nq, int Nk, int d, float scale, void* stream) {
  // d = 192 / 256: the one-query-tile kernel, which never needs a workspace
  if (attn_wide::supported(d)) return forward_wide(q, k, v, o, lse, B, H, Nq, Nk, d, scale, false, stream);
  // the same argument rules as attn_fwd
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (d != kD) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  if (bh == 0 || Nq == 0) return ATTN_OK;
  if (Nk == 0) return ATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(o)) & 15u)
    return ATTN_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return ATTN_ERR_MISALIGNED;
  const long long q_groups = (static_cast<long long>(Nq) + kQTiles * kBM - 1) / (kQTiles * kBM);
  if (bh > INT_MAX || bh * q_groups > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  const long long max_rows = static_cast<long long>(Nq > Nk ? Nq : Nk);
  if (bh > (LLONG_MAX / 256) / max_rows) return ATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  const int sms = sm_count(dev);
  if (sms <= 0) return ATTN_ERR_CUDA;

  // In host code g_noalloc_scratch only stands for the array: its device address has to
  // be asked for, with this device current. The first call in each context does that (a
  // lookup, no allocation); later calls in the same context reuse the address.
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    unsigned long long ctx = current_context_id();
    auto it = ctx != 0 ? g_noalloc_addr.find(ctx) : g_noalloc_addr.end();
    if (it != g_noalloc_addr.end()) {
      scratch = it->second;
    } else {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return ATTN_ERR_CUDA;
      scratch = ptr;
      ctx = current_context_id();   // the lookup makes the device's primary context current if none was
      if (ctx != 0) g_noalloc_addr[ctx] = ptr;
    }
  }

  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, Nq, bh) || !make_map(&mk, k, Nk, bh) || !make_map(&mv, v, Nk, bh))
    return ATTN_ERR_CUDA;

  Params p;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.Nq = Nq;
  p.Nk = Nk;
  p.q_groups = static_cast<int>(q_groups);
  p.n_kv = (Nk + kBN - 1) / kBN;
  p.kv_tail = Nk - (p.n_kv - 1) * kBN;
  const Plan pl = make_plan(bh * q_groups, p.n_kv, sms);
  p.dp_groups = static_cast<int>(pl.dp_groups);
  p.sk_steps = pl.sk_steps;
  set_cuts(p, pl.cuts);
  p.part = nullptr;
  p.cnt = nullptr;
  p.cnt_next = nullptr;   // the counters are cleared on the stream before each launch
  p.cnt_len = 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  p.withhold_tile = g_withhold.load(std::memory_order_relaxed);
  p.causal = 0;
  p.causal_off = 0;
  p.bh_count = static_cast<int>(bh);
  p.bias = nullptr;
  p.bias_sb = p.bias_sh = p.bias_sq = 0;
  p.H = H;
  p.scale = scale;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pl.has_split) {
    const size_t part_bytes = static_cast<size_t>(pl.grid) * kPartBytesPerBlock;
    const size_t cnt_off = (part_bytes + 255) & ~static_cast<size_t>(255);
    const size_t cnt_bytes = static_cast<size_t>(pl.sk_groups) * kQTiles * 4 * sizeof(unsigned int);
    if (cnt_off + cnt_bytes > kNoAllocScratchBytes) return ATTN_ERR_UNSUPPORTED;   // beyond the fixed maximum
    p.part = static_cast<float*>(scratch);
    p.cnt = reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(scratch) + cnt_off);
    // The array keeps whatever the previous call left; the arrival counters must start
    // at zero, so they are cleared on the call's stream before the kernel runs.
    if (cudaMemsetAsync(p.cnt, 0, cnt_bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return scale > 0.0f ? launch<true>(mq, mk, mv, p, pl.grid, dev, s) : launch<false>(mq, mk, mv, p, pl.grid, dev, s);
}
