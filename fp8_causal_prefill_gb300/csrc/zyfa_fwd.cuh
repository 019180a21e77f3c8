// Causal forward (prefill) attention for sm_103a: FP8 e4m3 with the ZYFA numerics, and a BF16 twin
// on the same schedule.
//
// What is computed (ZYFA: Speed and Accuracy of FP8 FlashAttention on AMD CDNA4, abstract,
// techniques (1)-(3); spbcomputers.ru ZYFA article, section "Три приёма"; captivela ZYFA article,
// section "Tiga Trik"): for every (batch b, head h, query row i),
//   S_ij = q8_i . k8_j (raw e4m3 values, fp32 tensor-core accumulation), keys j <= i only;
//   u_ij = S_ij * a,  a = fl32(fl32(fl32(scale*dq)*dk) * fl32(8 log2 e))   (1/8-binade units);
//   keys form blocks of 64 aligned at key 0; per (row, block) e = ceil(max u / 8);
//   Lean P: code_ij = clamp(rne(fl32(u_ij + 55.625 - 8e)), 0, 126)  -- one FMA and one conversion;
//   the block's codes are e4m3 probabilities scaled up by 2^-e; the PV product removes the scale
//   with an e8m0 block scale factor 2^(e - M) (M: the row's integer reference exponent);
//   out_i = dv * sum_j w_ij v8_j / sum_j w_ij with the same rounded weights w: the row sum comes from
//   the same block-scaled PV MMA, widened by 16 columns whose B operand is a tile of ones (the pages'
//   "one extra matrix instruction per block", +16/DV of the PV work).
// BF16 twin: p_ij = bf16(2^(S_ij*a' - M)), a' = fl32(scale*log2 e), normalised by the fp32 sum of the
// rounded p (accumulated by the softmax threads), no block scaling.
//
// Schedule (one persistent CTA per SM; one work unit = (b, h, 256 query rows) = two 128-row tiles
// Q0, Q1 that share every K/V tile of BN keys; a launch covers the query blocks of a given range):
//   warp 0      TMA producer: Q tiles and K tiles (and V tiles, when K and V share one ring)
//   warp 1      MMA issuer (the whole warp runs the loop, one elected lane issues) and TMEM owner
//   warp 2      TMA producer of V tiles when K and V have rings of their own (three slots or fewer:
//               BF16 at D=128, both types at D=192)
//   warps 4..7  softmax warpgroup of Q0, warps 8..11 softmax warpgroup of Q1
// The two score tiles share one TMEM buffer, filled in the order S0(0), S1(0), S0(1), S1(1), ...: a
// softmax warpgroup copies its scores to registers and releases the buffer at once, and the next
// score MMA is issued as soon as that release is seen.  The release also tells the MMA warp that
// the warpgroup's previous P is in TMEM, so PV_t(j-1) is issued right after the score MMA that follows
// the read of S_t(j): score MMAs never wait for a softmax computation, and the PV of one tile keeps
// the tensor core busy while the other tile's scores are handed over (the pages' ping-pong, here
// between two query tiles with mbarrier completion tracking).  Every PV commits to its tile's
// pv_done barrier; a warpgroup stores P_t(j) (and rescales O_t) once PV_t(j-1) has completed.
// The MMA warp's own instruction stream is on the critical path, so the middle of every unit (both
// query tiles active) runs as a fixed, branch-free sequence.
// Every tcgen05 instruction costs the issuing warp tens of cycles, so score MMAs are 128 keys wide.
//
// Tensor memory (512 columns x 128 lanes; lane = query row of a tile):
//   [  0,128)            S: fp32 scores of the tile being handed to a softmax warpgroup
//   [128,128+NO)         O0 (fp32, DV output columns; FP8: then 16 columns of the rounded row sum)
//   [128+NO,128+2NO)     O1
//   [416,480)            FP8: P0 | P1, e4m3 codes, BN/4 columns each;  BF16: [384,448) P0, [448,512) P1
//   [480,484) [488,492)  e8m0 scale factors of P0, P1 (FP8)   [496,504) scale factors of V (all 1.0)
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace zyfa {

// Status bits a kernel may set in the library's status word.
enum : int { kStatusTimeout = 1 };

constexpr int kBlockM = 128;         // query rows per tile
constexpr int kUnitRows = 2 * kBlockM;
constexpr int kScaleBlock = 64;      // keys per power-of-two scale block
constexpr int kThreads = 384;
// Register split (per thread): the kernel is built for 168 registers x 384 threads; the producer /
// MMA warpgroup gives registers back so the two softmax warpgroups can hold a 128-key score row.
// 128 x 72 + 256 x 208 <= 384 x 168: the split never asks for more than the launch allotted.
constexpr int kRegsLaunch = 168;
constexpr int kRegsControl = 72;
constexpr int kRegsSoftmax = 208;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");
// Lazy reference: a row's reference exponent moves (and O and l are rescaled by the exact power of two)
// only when a tile's largest block exponent exceeds it by more than p.rescale_binades.  Where the
// probabilities themselves are formed against the reference (BF16, and FP8 without block scaling) it
// must keep them inside the format: 8 binades.  With per-block scaling the codes are formed against
// their own block (largest weight at most 1) and the scale factors carry the difference, so the host
// allows the widest lag the fp32 accumulators bear for the launch's sequence length (see zyfa_api.cu).
constexpr int kRescaleBinades = 8;
constexpr float kLeanPC0 = 55.625f;  // Lean-P constant: code(2^x) = rne(8x + 55.625)
constexpr long long kWaitLimit = 1ll << 31;  // ~1 s of SM clocks before a wait gives up
constexpr int kNoExp = -2147483647;  // block exponent of a fully masked block

template <bool FP8, int DQK, int DV, int BN>
struct Cfg {
  static_assert(BN == 64 || BN == 128, "K/V tile of 64 or 128 keys");
  static constexpr int kElem = FP8 ? 1 : 2;
  // K / Q rows: 128-byte chunks (128-byte swizzle) and at most one 64-byte chunk (64-byte swizzle)
  static constexpr int kRowBytesK = DQK * kElem;
  static constexpr int kChunks128K = kRowBytesK / 128;
  static constexpr bool kTail64K = (kRowBytesK % 128) == 64;
  static_assert(kRowBytesK % 64 == 0, "head dim must give whole 64-byte chunks");
  static constexpr int kKStageBytes = BN * kRowBytesK;
  static constexpr int kQTileBytes = kBlockM * kRowBytesK;
  // V rows (MN-major B operand): atoms of 128-byte (or 64-byte) rows
  static constexpr int kRowBytesV = DV * kElem;
  static constexpr int kVAtomRow = kRowBytesV >= 128 ? 128 : 64;
  static constexpr int kVAtoms = kRowBytesV / kVAtomRow;
  static constexpr int kVAtomBytes = BN * kVAtomRow;
  static constexpr int kVStageBytes = BN * kRowBytesV;
  static constexpr bool kOnes = FP8;  // FP8: row sum from the widened PV MMA
  static_assert(!kOnes || kVAtoms == 1, "the shared ones atom needs a single V atom");
  static constexpr int kOnesBytes = kOnes ? kVAtomBytes : 0;
  static constexpr int kNO = kOnes ? DV + 16 : DV;  // PV MMA width
  static constexpr int kKSteps = kRowBytesK / 32;  // 32 bytes of K per MMA
  static constexpr int kKeysPerStep = FP8 ? 32 : 16;
  static constexpr int kPVSteps = BN / kKeysPerStep;
  static constexpr int kPCols = BN * kElem / 4;    // TMEM columns of one P tile
  // shared memory
  static constexpr int kSmemBudget = 220 * 1024;
  static constexpr int kStageBytes = kKStageBytes + kVStageBytes;
  static constexpr int kFixedBytes = 2 * kQTileBytes + kOnesBytes + 1024 /*align slack*/;
  static constexpr int kStagesRaw = (kSmemBudget - kFixedBytes) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static_assert(kStages >= 2, "not enough shared memory for two K/V stages");
  // epilogue: each softmax warp stages 32 rows x kEpiCols bf16 of its output (64- or 32-byte rows,
  // swizzled) for a TMA store; 64-byte rows where the shared memory allows
  static constexpr int kSmemMax = 232448;  // opt-in limit per block on sm_103
  static constexpr int kEpiCols = kFixedBytes + kStages * kStageBytes + 8 * 2048 <= kSmemMax ? 32 : 16;
  static constexpr int kEpiWarpBytes = 32 * kEpiCols * 2;
  static_assert(DV % kEpiCols == 0, "whole epilogue boxes");
  // two tiles per warp where they fit: a box is staged while the previous one is still being stored
  static constexpr int kEpiBufs =
      kFixedBytes + kStages * kStageBytes + 2 * 8 * kEpiWarpBytes <= kSmemMax ? 2 : 1;
  static constexpr int kSmemBytes = kFixedBytes + kStages * kStageBytes + kEpiBufs * 8 * kEpiWarpBytes;
  static_assert(kSmemBytes <= kSmemMax, "shared memory");
  // tensor memory columns
  static constexpr uint32_t kColS = 0;
  __device__ static constexpr uint32_t col_o(int t) { return 128u + static_cast<uint32_t>(kNO) * t; }
  // P tiles: FP8 [416,448) [448,480) below the scale factors; BF16 [384,448) [448,512)
  static constexpr uint32_t kColP = FP8 ? 416u : 384u;
  __device__ static constexpr uint32_t col_p(int t) { return kColP + static_cast<uint32_t>(kPCols) * t; }
  __device__ static constexpr uint32_t col_sfa(int t) { return 480u + 8u * t; }
  static constexpr uint32_t kColSFB = 496;
  static_assert(128 + 2 * kNO <= static_cast<int>(kColP), "O accumulators overlap the P tiles");
  static_assert(kColP + 2 * kPCols <= (FP8 ? 480u : 512u), "P tiles overlap the scale factors");
  // K and V tiles sit in two rings of kStages slots.  With a short ring (three slots or fewer) K and V
  // have their own barriers and producers: a K slot is free once the last score MMA of its tile
  // completed, a V slot once the last PV did, so a score MMA never waits for a PV.  A longer ring
  // (whose stages are always ready in time) keeps one barrier per K/V pair, released after the later
  // PV, which spares the MMA warp a wait and a commit per tile.
  static constexpr bool kSplitKV = kStages <= 3;
  // With one barrier per K/V pair, the last PV of query tile 0 waits for the end of the unit while
  // tile 1 may still need up to kBlockM / BN more tiles: the ring must hold them.
  static_assert(kSplitKV || kStages > kBlockM / BN, "K/V ring too short for the PV lag");
  static_assert(kNO % 16 == 0 && kNO <= 256, "PV MMA width");
};

struct Params {
  __nv_bfloat16* out;  // [B,S,H,DV]
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  int B, S, H, H_kv;
  float softmax_scale;
  int num_units;  // B*H*(qb_end - qb_begin)
  int qb_end;     // query blocks (256 rows) [qb_end - num_units/(B*H), qb_end) are processed
  int* status;    // device status word (timeouts)
  int stall_loads;  // self-test of the timeout path: the producer withholds every load
  float* lse;       // optional [B,H,S] natural-log sum of exp of the scores (nullptr: not written)
  int desc_per_head;  // descales are arrays [B][H_kv] (1) or single values (0)
  int no_block_scale; // exact P only: every block rounds against the row reference (scale factor 1)
  int rescale_binades;  // block-scaled FP8: lag of the row reference before O and l are rescaled
};

struct __align__(8) SharedCtl {
  uint64_t k_full[8], k_empty[8], v_full[8], v_empty[8];
  uint64_t q_full[2], q_empty[2], s_full[2], p_full[2], pv_done[2];
  uint64_t s_free, drain;
  uint32_t tmem_base;
  int abort_;
};

struct Unit {
  int b, h, r0;
};

// Units in longest-first order, dealt to CTAs in a snake (boustrophedon) so the per-CTA causal
// work is balanced without any shared counter: round r gives CTA c the unit r*G + c (r even) or
// r*G + G-1-c (r odd).  Units of one round share query-block length and run concurrently, and
// neighbouring heads share a KV head (L2 reuse of K/V under GQA).
__device__ __forceinline__ bool unit_at(const Params& p, int round, Unit& u) {
  const int G = gridDim.x;
  const int c = blockIdx.x;
  const int idx = round * G + ((round & 1) ? (G - 1 - c) : c);
  if (idx >= p.num_units) return false;
  const int bh = p.B * p.H;
  const int qb = p.qb_end - 1 - idx / bh;
  const int rest = idx % bh;
  u.b = rest / p.H;
  u.h = rest % p.H;
  u.r0 = qb * kUnitRows;
  return true;
}

// Number of BN-key tiles query tile t of a unit needs (0 if the tile has no rows).
template <int BN>
__device__ __forceinline__ int tiles_for(const Params& p, int r0, int t) {
  const int first = r0 + t * kBlockM;
  if (first >= p.S) return 0;
  const int end = min(first + kBlockM, p.S);
  return (end + BN - 1) / BN;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// max over 64 consecutive values, as a tree of 3-input maxima (short dependency chains)
__device__ __forceinline__ float max64(const float* s) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    m[i] = fmax3(fmax3(s[8 * i], s[8 * i + 1], s[8 * i + 2]), fmax3(s[8 * i + 3], s[8 * i + 4], s[8 * i + 5]),
                 fmaxf(s[8 * i + 6], s[8 * i + 7]));
  return fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// Two fp32 -> packed f16x2 with negative values clamped to +0; the upper half takes `hi`.
__device__ __forceinline__ uint32_t cvt_relu_f16x2(float hi, float lo) {
  uint32_t r;
  asm("cvt.rn.relu.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t cvt_bf16x2(float hi, float lo) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^d for an integer d, exactly (0 below the normal range).
__device__ __forceinline__ float exp2i(int d) {
  return d < -126 ? 0.0f : __int_as_float((127 + d) << 23);
}

// Two fp32 lanes in one 64-bit register, for the packed multiply-add.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ void unpack2(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
// lo += the low bf16 of w, hi += its high bf16 (each widened exactly, one fp32 rounding per add)
__device__ __forceinline__ void add_bf16x2(uint32_t w, float& lo, float& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %0;\n\t"
      "add.rn.f32.bf16 %1, h, %1;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "r"(w));
}
__device__ __forceinline__ uint32_t cvt_relu_f16x2_pair(uint64_t t) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(t));
  return cvt_relu_f16x2(hi, lo);
}

// Lean-P codes of the 64 scores of one scale block with exponent e: t = fma(s, a, 55.625 - 8e) scaled
// by 2^-24 (two scores per packed fp32 multiply-add, each lane rounded as a scalar fma), so the f16
// subnormal that the rounding conversion produces carries the integer code in its low byte
// (negative values clamp to 0).  Four codes per 32-bit word, key order = byte order.
__device__ __forceinline__ void leanp_block(const float* s, float a24, int e, uint32_t (&pw)[16]) {
  const float c24 = __fmul_rn(kLeanPC0 - 8.0f * static_cast<float>(e), 0x1p-24f);
  const uint64_t a2 = pack2(a24, a24), c2 = pack2(c24, c24);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t t01 = ffma2(pack2(s[4 * i + 0], s[4 * i + 1]), a2, c2);
    const uint64_t t23 = ffma2(pack2(s[4 * i + 2], s[4 * i + 3]), a2, c2);
    pw[i] = prmt(cvt_relu_f16x2_pair(t01), cvt_relu_f16x2_pair(t23), 0x6420u);
  }
}

template <bool FP8, int DV>
__device__ __forceinline__ void rescale_o(uint32_t tO, float f) {
  using namespace ptx;
#pragma unroll
  for (int c = 0; c < DV / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(tO + 32 * c, r);
    tmem_wait_ld();
    tmem_ld_fence(r);
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
    tmem_st32(tO + 32 * c, r);
  }
  if constexpr (FP8) {
    uint32_t lv[1];
    tmem_ld1(tO + DV, lv[0]);
    tmem_wait_ld();
    tmem_ld_fence(lv);
    tmem_st1(tO + DV, __float_as_uint(__uint_as_float(lv[0]) * f));
  }
}

// Two fp32 -> e4m3 codes (round to nearest even, saturating), the upper byte takes `hi`.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Exact-P codes of the 64 scores of one scale block with exponent e: the probability
// 2^(s*a/8 - e) from the hardware exponential, rounded to e4m3.  The comparison point for Lean P
// (one exponential per probability, exactly rounded).
__device__ __forceinline__ void exactp_block(const float* s, float a8, int e, uint32_t (&pw)[16]) {
  const float ne = -static_cast<float>(e);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float p0 = ex2(__fmaf_rn(s[4 * i + 0], a8, ne));
    const float p1 = ex2(__fmaf_rn(s[4 * i + 1], a8, ne));
    const float p2 = ex2(__fmaf_rn(s[4 * i + 2], a8, ne));
    const float p3 = ex2(__fmaf_rn(s[4 * i + 3], a8, ne));
    pw[i] = cvt_e4m3x2(p1, p0) | (cvt_e4m3x2(p3, p2) << 16);
  }
}

template <bool FP8, int DQK, int DV, int BN, bool EXACT>
__global__ void __launch_bounds__(kThreads, 1)
    zyfa_fwd_kernel(const __grid_constant__ Params p, const __grid_constant__ Maps maps) {
  using C = Cfg<FP8, DQK, DV, BN>;
  using namespace ptx;
  extern __shared__ uint8_t smem_raw[];
  __shared__ SharedCtl ctl;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- shared memory: [Q0 | Q1 | K/V slots | ones atom | epilogue tiles], 1024-byte aligned ----
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t s_q = base;
  const uint32_t s_stages = s_q + 2 * C::kQTileBytes;
  // FP8: one atom of e4m3 1.0 above every V stage; the PV descriptor reaches it through its
  // leading-dimension offset (a positive distance from each stage)
  // split rings: all K slots, then all V slots; one ring: each slot holds a K tile and its V tile
  const uint32_t s_ones = s_stages + C::kStages * C::kStageBytes;
  const uint32_t s_epi = s_ones + C::kOnesBytes;  // 8 softmax warps x kEpiWarpBytes
  auto k_stage = [&](int s) { return s_stages + s * (C::kSplitKV ? C::kKStageBytes : C::kStageBytes); };
  auto v_stage = [&](int s) {
    return C::kSplitKV ? s_stages + C::kStages * C::kKStageBytes + s * C::kVStageBytes
                       : s_stages + s * C::kStageBytes + C::kKStageBytes;
  };

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&ctl.k_full[s]), 1);
      mbar_init(smem_u32(&ctl.k_empty[s]), 1);
      mbar_init(smem_u32(&ctl.v_full[s]), 1);
      mbar_init(smem_u32(&ctl.v_empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&ctl.q_full[t]), 1);
      mbar_init(smem_u32(&ctl.q_empty[t]), 1);
      mbar_init(smem_u32(&ctl.s_full[t]), 1);
      mbar_init(smem_u32(&ctl.p_full[t]), 4);
      mbar_init(smem_u32(&ctl.pv_done[t]), 1);
    }
    mbar_init(smem_u32(&ctl.s_free), 4);
    mbar_init(smem_u32(&ctl.drain), 1);
    ctl.abort_ = 0;
    fence_mbar_init();
  }
  if constexpr (C::kOnes) {
    uint32_t* o32 = reinterpret_cast<uint32_t*>(base_ptr + (s_ones - base));
    for (int i = tid; i < C::kOnesBytes / 4; i += kThreads) o32[i] = 0x38383838u;  // e4m3 1.0
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort_;
  auto give_up = [&]() {
    *abort_flag = 1;
    atomicOr(p.status, kStatusTimeout);
  };
  const int hgroup = p.H / p.H_kv;

  if (warp == 0) {
    // =========================== TMA producer: Q and K (and V with a long ring) ===========================
    regs_dec<kRegsControl>();
    if (!p.stall_loads) {
      const bool leader = elect_one();
      if (leader) {
        tma_prefetch_desc(&maps.k0);
        tma_prefetch_desc(&maps.v);
        tma_prefetch_desc(&maps.q0);
      }
      uint32_t kv_cnt = 0;
      uint32_t q_cnt[2] = {0, 0};
      bool ok = true;
      Unit u;
      for (int round = 0; ok && unit_at(p, round, u); ++round) {
        const int hk = u.h / hgroup;
        const int n0 = tiles_for<BN>(p, u.r0, 0), n1 = tiles_for<BN>(p, u.r0, 1);
        const int nkv = n1 > n0 ? n1 : n0;
        for (int t = 0; t < 2 && ok; ++t) {
          if ((t == 0 ? n0 : n1) == 0) continue;
          ok = mbar_wait(smem_u32(&ctl.q_empty[t]), (q_cnt[t] & 1) ^ 1, abort_flag, kWaitLimit);
          if (!ok) break;
          const uint32_t bar = smem_u32(&ctl.q_full[t]);
          const uint32_t dst = s_q + t * C::kQTileBytes;
          if (leader) {
            mbar_arrive_expect_tx(bar, C::kQTileBytes);
            for (int c = 0; c < C::kChunks128K; ++c)
              tma_load_4d(dst + c * (kBlockM * 128), &maps.q0, bar, c * (128 / C::kElem), u.h, u.r0 + t * kBlockM,
                          u.b);
            if (C::kTail64K)
              tma_load_4d(dst + C::kChunks128K * (kBlockM * 128), &maps.q1, bar, C::kChunks128K * (128 / C::kElem),
                          u.h, u.r0 + t * kBlockM, u.b);
          }
          ++q_cnt[t];
        }
        for (int j = 0; j < nkv && ok; ++j) {
          const int st = kv_cnt % C::kStages;
          ok = mbar_wait(smem_u32(&ctl.k_empty[st]), ((kv_cnt / C::kStages) & 1) ^ 1, abort_flag, kWaitLimit);
          if (!ok) break;
          const uint32_t bar = smem_u32(&ctl.k_full[st]);
          if (leader) {
            mbar_arrive_expect_tx(bar, C::kKStageBytes + (C::kSplitKV ? 0 : C::kVStageBytes));
            for (int c = 0; c < C::kChunks128K; ++c)
              tma_load_4d(k_stage(st) + c * (BN * 128), &maps.k0, bar, c * (128 / C::kElem), hk, j * BN, u.b);
            if (C::kTail64K)
              tma_load_4d(k_stage(st) + C::kChunks128K * (BN * 128), &maps.k1, bar,
                          C::kChunks128K * (128 / C::kElem), hk, j * BN, u.b);
            if (!C::kSplitKV)  // V on the same barrier
              for (int c = 0; c < C::kVAtoms; ++c)
                tma_load_4d(v_stage(st) + c * C::kVAtomBytes, &maps.v, bar, c * (C::kVAtomRow / C::kElem), hk,
                            j * BN, u.b);
          }
          ++kv_cnt;
        }
      }
      if (!ok) {
        if (leader) give_up();
        // every load already issued lands before the CTA may exit (its shared memory is released then)
        const int never = 0;
        const uint32_t ns = C::kStages;
        for (uint32_t i = (kv_cnt > ns ? kv_cnt - ns : 0); i < kv_cnt; ++i)
          mbar_wait(smem_u32(&ctl.k_full[i % ns]), (i / ns) & 1, &never, kWaitLimit);
        for (int t = 0; t < 2; ++t)
          if (q_cnt[t] > 0) mbar_wait(smem_u32(&ctl.q_full[t]), (q_cnt[t] - 1) & 1, &never, kWaitLimit);
      }
    }
  } else if (warp == 1) {
    // =========================== MMA issuer ===========================
    regs_dec<kRegsControl>();
    {
      const bool leader = elect_one();
      const uint32_t fmt = FP8 ? kFmtE4M3 : kFmtBF16;
      const uint32_t idesc_s = idesc_dense(fmt, fmt, false, false, kBlockM, BN);
      // shared-memory descriptors of the first K step of each operand; a K step of 32 bytes moves the
      // start address by 2 (16-byte units), a 128-byte chunk by rows * 8
      const uint64_t q_desc0 = smem_desc(s_q, 16, 1024, kSwizzle128B);
      const uint64_t q_tail0 = smem_desc(s_q + C::kChunks128K * (kBlockM * 128), 16, 512, kSwizzle64B);
      const uint64_t k_desc0 = smem_desc(k_stage(0), 16, 1024, kSwizzle128B);
      const uint64_t k_tail0 = smem_desc(k_stage(0) + C::kChunks128K * (BN * 128), 16, 512, kSwizzle64B);
      constexpr uint32_t kQTile16 = C::kQTileBytes >> 4;
      constexpr uint32_t kStage16 = (C::kSplitKV ? C::kKStageBytes : C::kStageBytes) >> 4;
      uint32_t kv_cnt = 0, s_seq = 0;
      uint32_t q_cnt[2] = {0, 0}, p_cnt[2] = {0, 0};
      bool ok = true;
      // the score tile issued last, while its reader has not yet been seen to copy it out
      bool read_pending = false;
      int last_t = 0, last_j = 0;

      // S = Q_t K^T for the K tile in stage st (both operands K-major in shared memory)
      auto issue_s = [&](int t, uint32_t st) {
        const uint64_t qd = q_desc0 + t * kQTile16, kd = k_desc0 + st * kStage16;
        const uint64_t qt = q_tail0 + t * kQTile16, kt = k_tail0 + st * kStage16;
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          const int off = ks * 32;
          uint64_t ad, bd;
          if (off < C::kChunks128K * 128) {
            ad = qd + (off / 128) * (kBlockM * 8) + (off % 128) / 16;
            bd = kd + (off / 128) * (BN * 8) + (off % 128) / 16;
          } else {
            ad = qt + (off - C::kChunks128K * 128) / 16;
            bd = kt + (off - C::kChunks128K * 128) / 16;
          }
          if constexpr (FP8) mma_f8_ss(tmem + C::kColS, ad, bd, idesc_s, ks > 0);
          else mma_f16_ss(tmem + C::kColS, ad, bd, idesc_s, ks > 0);
        }
        tc_commit(smem_u32(&ctl.s_full[t]));
      };
      // O_t (| l_t) += P_t x [V | 1]
      auto issue_pv = [&](int t, uint32_t st, bool first) {
        const uint32_t o = tmem + C::col_o(t), pa = tmem + C::col_p(t), vb = v_stage(st);
        const uint32_t lbo = C::kOnes ? (s_ones - vb) : static_cast<uint32_t>(C::kVAtomBytes);
        const uint64_t vd = C::kVAtomRow == 128 ? smem_desc(vb, lbo, 1024, kSwizzle128B)
                                                : smem_desc(vb, lbo, 512, kSwizzle64B);
#pragma unroll
        for (int ks = 0; ks < C::kPVSteps; ++ks) {
          const uint64_t vdk = vd + (ks * C::kKeysPerStep * C::kVAtomRow) / 16;
          const uint32_t acc = (!first || ks > 0) ? 1u : 0u;
          if constexpr (FP8) {
            // K step ks covers keys [32ks, 32ks+32): its e8m0 scale is byte ks of the scale word
            mma_mxf8_ts(o, pa + ks * 8, vdk, idesc_block_scaled(kFmtE4M3, kFmtE4M3, true, kBlockM, C::kNO, ks, 0),
                        tmem + C::col_sfa(t), tmem + C::kColSFB, acc);
          } else {
            mma_f16_ts(o, pa + ks * 8, vdk, idesc_dense(kFmtBF16, kFmtBF16, false, true, kBlockM, C::kNO), acc);
          }
        }
      };

      // PV_t(j) of a unit whose K/V tiles start at ring position kvb and whose query tiles have n0_ /
      // n1_ K/V tiles, announced on pv_done.  A K/V stage is released after the later of its (at most
      // two) PVs.
      auto do_pv_at = [&](int t, int j, uint32_t kvb, int n0_, int n1_) -> bool {
        const uint32_t st = (kvb + j) % C::kStages;
        if constexpr (C::kSplitKV) {
          if (!mbar_wait_warp(smem_u32(&ctl.v_full[st]), ((kvb + j) / C::kStages) & 1, abort_flag, kWaitLimit))
            return false;
          tc_fence_after();
        }
        issue_pv(t, st, j == 0);
        tc_commit(smem_u32(&ctl.pv_done[t]));
        const bool pv0_last = n1_ == 0 || (j == n0_ - 1 && n1_ > n0_);
        if ((t == 0) == pv0_last)
          tc_commit(smem_u32(C::kSplitKV ? &ctl.v_empty[st] : &ctl.k_empty[st]));
        return true;
      };
      // The last PV of each query tile waits for that tile's final P (p_full).  It is issued after
      // the next unit's first score MMA, so that score tile is not held behind the slower warpgroup's
      // last softmax; per tile the PVs stay in order.
      // the pending last PVs all belong to one unit: its K/V ring base and tile counts
      int tail_n[2] = {0, 0};
      uint32_t tail_kvb = 0;
      auto issue_tails = [&]() -> bool {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (tail_n[t] == 0) continue;
          if (!mbar_wait_warp(smem_u32(&ctl.p_full[t]), p_cnt[t] & 1, abort_flag, kWaitLimit)) return false;
          ++p_cnt[t];
          tc_fence_after();
          if (!do_pv_at(t, tail_n[t] - 1, tail_kvb, tail_n[0], tail_n[1])) return false;
        }
        tail_n[0] = tail_n[1] = 0;
        return true;
      };

      Unit u;
      for (int round = 0; ok && unit_at(p, round, u); ++round) {
        const int n0 = tiles_for<BN>(p, u.r0, 0), n1 = tiles_for<BN>(p, u.r0, 1);
        const int nkv = n1 > n0 ? n1 : n0;
        if (n0 > 0) {
          ok = mbar_wait_warp(smem_u32(&ctl.q_full[0]), q_cnt[0] & 1, abort_flag, kWaitLimit);
          ++q_cnt[0];
        }
        if (ok && n1 > 0) {
          ok = mbar_wait_warp(smem_u32(&ctl.q_full[1]), q_cnt[1] & 1, abort_flag, kWaitLimit);
          ++q_cnt[1];
        }
        if (!ok) break;

        auto do_pv = [&](int t, int j) -> bool { return do_pv_at(t, j, kv_cnt, n0, n1); };
        // Waits until the last score tile issued has been copied out of the shared S buffer.  Its
        // reader stored P of its previous tile before that, so the PV of that tile may follow; that
        // tile is returned in rt / rj (rj < 0: nothing to unlock).
        int rt = 0, rj = -1;
        auto wait_read = [&]() -> bool {
          rj = -1;
          if (!read_pending) return true;
          if (!mbar_wait_warp(smem_u32(&ctl.s_free), (s_seq - 1) & 1, abort_flag, kWaitLimit)) return false;
          read_pending = false;
          tc_fence_after();
          if (last_j >= 1) {
            rt = last_t;
            rj = last_j - 1;
          }
          return true;
        };

        // score tiles in the order S0(0), S1(0), S0(1), S1(1), ...; each one waits until the previous
        // was read, and the PV that read unlocks is issued next to it: after the score MMA when that
        // belongs to the other query tile, before it when it belongs to the same one (so a score tile
        // always follows the previous PV of its own query tile)
        for (int j = 0; j < nkv && ok; ++j) {
          if (j >= 1 && j < n0 && n1 > 0) {
            // steady state (both query tiles active): S0(j), PV1(j-2), S1(j), PV0(j-1)
            const uint32_t st = (kv_cnt + j) % C::kStages;
            // K first: it is normally in place long before the read, so checking it while the read is
            // outstanding keeps the check off the path from the read to the next score MMA
            if (!(ok = mbar_wait_warp(smem_u32(&ctl.k_full[st]), ((kv_cnt + j) / C::kStages) & 1, abort_flag,
                                 kWaitLimit)))
              break;
            if (!(ok = mbar_wait_warp(smem_u32(&ctl.s_free), (s_seq - 1) & 1, abort_flag, kWaitLimit))) break;
            tc_fence_after();
            issue_s(0, st);
            if (j == n0 - 1) tc_commit(smem_u32(&ctl.q_empty[0]));
            if (j >= 2) {
              const uint32_t st2 = (kv_cnt + j - 2) % C::kStages;
              if constexpr (C::kSplitKV) {
                if (!(ok = mbar_wait_warp(smem_u32(&ctl.v_full[st2]), ((kv_cnt + j - 2) / C::kStages) & 1, abort_flag,
                                     kWaitLimit)))
                  break;
                tc_fence_after();
              }
              issue_pv(1, st2, j == 2);
              tc_commit(smem_u32(&ctl.pv_done[1]));
              tc_commit(smem_u32(C::kSplitKV ? &ctl.v_empty[st2] : &ctl.k_empty[st2]));
            }
            if (!(ok = mbar_wait_warp(smem_u32(&ctl.s_free), s_seq & 1, abort_flag, kWaitLimit))) break;
            tc_fence_after();
            issue_s(1, st);
            // query tile 1 normally has one more K/V tile than tile 0 and ends after this block; a
            // unit whose two tiles end together ends tile 1 here
            if (j == n1 - 1) tc_commit(smem_u32(&ctl.q_empty[1]));
            if (C::kSplitKV) tc_commit(smem_u32(&ctl.k_empty[st]));  // S1(j): last reader of K tile j
            const uint32_t st1 = (kv_cnt + j - 1) % C::kStages;
            if constexpr (C::kSplitKV) {
              if (!(ok = mbar_wait_warp(smem_u32(&ctl.v_full[st1]), ((kv_cnt + j - 1) / C::kStages) & 1, abort_flag,
                                   kWaitLimit)))
                break;
              tc_fence_after();
            }
            issue_pv(0, st1, j == 1);
            tc_commit(smem_u32(&ctl.pv_done[0]));
            s_seq += 2;
            last_t = 1;
            last_j = j;
            read_pending = true;
            continue;
          }
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (j >= (t ? n1 : n0)) continue;
            if (t == 0 || j >= n0) {  // first score tile of K tile j
              if (!(ok = mbar_wait_warp(smem_u32(&ctl.k_full[(kv_cnt + j) % C::kStages]),
                                   ((kv_cnt + j) / C::kStages) & 1, abort_flag, kWaitLimit)))
                break;
              tc_fence_after();
            }
            if (!(ok = wait_read())) break;
            // a PV of the same query tile goes before its next score MMA, one of the other tile after it
            const bool pv_first = rj >= 0 && rt == t;
            if (pv_first && !(ok = do_pv(rt, rj))) break;
            issue_s(t, (kv_cnt + j) % C::kStages);
            ++s_seq;
            read_pending = true;
            last_t = t;
            last_j = j;
            if (j == (t ? n1 : n0) - 1) tc_commit(smem_u32(&ctl.q_empty[t]));
            // the last score MMA reading K tile j: S1(j), or S0(j) when query tile 1 has no tile j
            if (C::kSplitKV && (t == 1 || j >= n1))
              tc_commit(smem_u32(&ctl.k_empty[(kv_cnt + j) % C::kStages]));
            if (rj >= 0 && !pv_first && !(ok = do_pv(rt, rj))) break;
            if (t == 0 && j == 0 && !(ok = issue_tails())) break;
          }
        }
        if (!ok) break;
        // unit end: the read of the last score tile unlocks one more PV; the last PV of each query
        // tile (which waits for its final P) goes with the next unit's first score MMA
        if (!(ok = wait_read())) break;
        if (rj >= 0 && !(ok = do_pv(rt, rj))) break;
        tail_n[0] = n0;
        tail_n[1] = n1;
        tail_kvb = kv_cnt;
        kv_cnt += nkv;
      }
      if (ok) ok = issue_tails();
      if (!ok && leader) give_up();
      // drain: all MMAs issued by this warp complete before TMEM is released
      const int never = 0;
      tc_commit(smem_u32(&ctl.drain));
      mbar_wait_warp(smem_u32(&ctl.drain), 0, &never, kWaitLimit);
    }
  } else if (warp == 2) {
    // =========================== TMA producer: V (short rings) ===========================
    regs_dec<kRegsControl>();
    if (C::kSplitKV && !p.stall_loads) {
      const bool leader = elect_one();
      uint32_t v_cnt = 0;
      bool ok = true;
      Unit u;
      for (int round = 0; ok && unit_at(p, round, u); ++round) {
        const int hk = u.h / hgroup;
        const int n0 = tiles_for<BN>(p, u.r0, 0), n1 = tiles_for<BN>(p, u.r0, 1);
        const int nkv = n1 > n0 ? n1 : n0;
        for (int j = 0; j < nkv && ok; ++j) {
          const int st = v_cnt % C::kStages;
          ok = mbar_wait(smem_u32(&ctl.v_empty[st]), ((v_cnt / C::kStages) & 1) ^ 1, abort_flag, kWaitLimit);
          if (!ok) break;
          const uint32_t bar = smem_u32(&ctl.v_full[st]);
          if (leader) {
            mbar_arrive_expect_tx(bar, C::kVStageBytes);
            for (int c = 0; c < C::kVAtoms; ++c)
              tma_load_4d(v_stage(st) + c * C::kVAtomBytes, &maps.v, bar, c * (C::kVAtomRow / C::kElem), hk,
                          j * BN, u.b);
          }
          ++v_cnt;
        }
      }
      if (!ok) {
        if (leader) give_up();
        const int never = 0;
        const uint32_t ns = C::kStages;
        for (uint32_t i = (v_cnt > ns ? v_cnt - ns : 0); i < v_cnt; ++i)
          mbar_wait(smem_u32(&ctl.v_full[i % ns]), (i / ns) & 1, &never, kWaitLimit);
      }
    }
  } else if (warp < 4) {
    regs_dec<kRegsControl>();  // warp 3: idle member of the control warpgroup
  } else {
    // =========================== softmax warpgroups ===========================
    regs_inc<kRegsSoftmax>();
    const int t = (warp - 4) >> 2;         // query tile of this warpgroup
    const int quarter = warp & 3;          // TMEM lane quarter of this warp
    const int rloc = quarter * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::kColS;
    const uint32_t tO = tmem + lane_addr + C::col_o(t);
    const uint32_t tP = tmem + lane_addr + C::col_p(t);
    const uint32_t epi_tile = s_epi + (warp - 4) * C::kEpiBufs * C::kEpiWarpBytes;  // 1024-byte aligned

    // score scale a (FP8: 1/8-binade units, with the descales; BF16: binades) and output scale dv,
    // per unit when the descales are per (batch, KV head)
    auto unit_scales = [&](const Unit& un, float& a_, float& out_) {
      if constexpr (FP8) {
        const int di = p.desc_per_head ? un.b * p.H_kv + un.h / (p.H / p.H_kv) : 0;
        const float dq = p.q_descale ? p.q_descale[di] : 1.0f;
        const float dk = p.k_descale ? p.k_descale[di] : 1.0f;
        a_ = __fmul_rn(__fmul_rn(__fmul_rn(p.softmax_scale, dq), dk), 11.541560327111707f);
        out_ = p.v_descale ? p.v_descale[di] : 1.0f;
      } else {
        a_ = __fmul_rn(p.softmax_scale, 1.4426950408889634f);
        out_ = 1.0f;
      }
    };
    if constexpr (FP8) {
      if (t == 0) {
        // e8m0 scale factors of V (all 1.0), written once; every PV is issued after an arrival of
        // this warpgroup (query tile 0 of a unit always has rows), which releases these stores
        tmem_st4(tmem + lane_addr + C::kColSFB, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        tmem_st4(tmem + lane_addr + C::kColSFB + 4, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        tmem_wait_st();
      }
    }

    uint32_t s_cnt = 0;
    uint32_t pv_ph = 0;  // pv_done phases of this query tile seen so far
    bool ok = true;
    Unit u;
    for (int round = 0; ok && unit_at(p, round, u); ++round) {
      const int n0 = tiles_for<BN>(p, u.r0, 0), n1 = tiles_for<BN>(p, u.r0, 1);
      const int ntiles = t == 0 ? n0 : n1;
      if (ntiles == 0) continue;
      const int row0 = u.r0 + t * kBlockM;  // first row of the tile
      const int row = row0 + rloc;
      const bool row_ok = row < p.S;
      float a, out_scale;
      unit_scales(u, a, out_scale);
      const float a24 = a * 0x1p-24f;  // exact: scales Lean-P values into f16 subnormal units
      const float a8 = a * 0.125f;     // exact: binade units for the exact-P exponential

      int m_ref = 0;
      const int rescale_binades =
          FP8 && !(EXACT && p.no_block_scale) ? p.rescale_binades : kRescaleBinades;
      float l_bf16 = 0.0f;  // BF16: fp32 sum of the rounded probabilities of this row
      // Iteration j copies score tile j out of the shared S buffer and releases it (the release also
      // tells the MMA warp that P of tile j-1, stored before, is in place), computes P of tile j and
      // stores it as soon as PV_t(j-1), which reads the same TMEM buffer, has completed (pv_done).
      constexpr int kNB = BN / kScaleBlock;
      constexpr int kPW = BN * C::kElem / 4;  // 32-bit words of P per row
      for (int j = 0; j < ntiles; ++j) {
        ok = mbar_wait(smem_u32(&ctl.s_full[t]), s_cnt & 1, abort_flag, kWaitLimit);
        ++s_cnt;
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        float s[BN];
        {
          uint32_t r[BN];
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
          tmem_wait_ld();
          tmem_ld_fence(r);
#pragma unroll
          for (int i = 0; i < BN; ++i) s[i] = __uint_as_float(r[i]);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl.s_free));

        const int key0 = j * BN;
        if (key0 + BN - 1 > row0) {  // tile touches the diagonal: mask keys after the row
#pragma unroll
          for (int i = 0; i < BN; ++i)
            if (key0 + i > row) s[i] = -INFINITY;
        }
        int e[kNB];
        int e_top = kNoExp;
#pragma unroll
        for (int b = 0; b < kNB; ++b) {
          // block exponent (FP8: ceil(max u / 8); BF16: ceil(max log2-score))
          const float mx = max64(s + 64 * b);
          const bool empty = mx == -INFINITY;
          if constexpr (FP8) e[b] = empty ? kNoExp : static_cast<int>(ceilf(__fmul_rn(mx, a) * 0.125f));
          else e[b] = empty ? kNoExp : static_cast<int>(ceilf(__fmul_rn(mx, a)));
          e_top = max(e_top, e[b]);
        }
        const bool need = j > 0 && e_top > m_ref + rescale_binades;
        const float f = need ? exp2i(m_ref - e_top) : 1.0f;
        if (j == 0 || need) m_ref = e_top;

        uint32_t pw[kPW];
        uint32_t sfw = 0;
        float lsum = 0.0f;
        if constexpr (FP8) {
#pragma unroll
          for (int b = 0; b < kNB; ++b) {
            int eb = e[b] == kNoExp ? m_ref : e[b];
            // the ablation of the block scaling: the row's running reference for every block
            if constexpr (EXACT) eb = p.no_block_scale ? m_ref : eb;
            if constexpr (EXACT) exactp_block(s + 64 * b, a8, eb, *reinterpret_cast<uint32_t(*)[16]>(pw + 16 * b));
            else leanp_block(s + 64 * b, a24, eb, *reinterpret_cast<uint32_t(*)[16]>(pw + 16 * b));
            int sf = 127 + eb - m_ref;
            sf = sf < 0 ? 0 : (sf > 254 ? 254 : sf);
            sfw |= static_cast<uint32_t>(sf) * (0x0101u << (16 * b));
          }
          if (kNB == 1) sfw |= sfw << 16;
        } else {
          // the softmax warps are issue-bound: the multiply-add takes one packed instruction per two
          // keys, and the row sum adds each rounded bf16 probability straight into an fp32
          // accumulator (four of them: even / odd keys of even / odd words)
          const float negm = -static_cast<float>(m_ref);
          const uint64_t a2 = pack2(a, a), m2 = pack2(negm, negm);
          float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
          for (int i = 0; i < kPW; ++i) {
            float x0, x1;
            unpack2(ffma2(pack2(s[2 * i], s[2 * i + 1]), a2, m2), x0, x1);
            pw[i] = cvt_bf16x2(ex2(x1), ex2(x0));
            if (i & 1) add_bf16x2(pw[i], l2, l3);
            else add_bf16x2(pw[i], l0, l1);
          }
          lsum = (l0 + l2) + (l1 + l3);
        }
        if (j > 0) {
          ok = mbar_wait(smem_u32(&ctl.pv_done[t]), pv_ph & 1, abort_flag, kWaitLimit);
          ++pv_ph;
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          if (__any_sync(0xffffffffu, need)) rescale_o<FP8, DV>(tO, f);
        }
        l_bf16 = l_bf16 * f + lsum;
#pragma unroll
        for (int c = 0; c < kPW / 16; ++c)
          tmem_st16(tP + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(pw + 16 * c));
        if constexpr (FP8) tmem_st4(tmem + lane_addr + C::col_sfa(t), sfw, sfw, sfw, sfw);
        if (j + 1 == ntiles) {
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl.p_full[t]));
        }
      }
      if (!ok) break;

      // epilogue: out = O * (dv / l) -> bf16, once the last PV of this tile completed
      ok = mbar_wait(smem_u32(&ctl.pv_done[t]), pv_ph & 1, abort_flag, kWaitLimit);
      ++pv_ph;
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      // all of O (and the FP8 row sum) in one round trip
      uint32_t o[DV];
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) tmem_ld32(tO + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(o + 32 * c));
      float l;
      if constexpr (FP8) {
        uint32_t lv[1];
        tmem_ld1(tO + DV, lv[0]);
        tmem_wait_ld();
        tmem_ld_fence(lv);
        l = __uint_as_float(lv[0]);
      } else {
        tmem_wait_ld();
        l = l_bf16;
      }
      tmem_ld_fence(o);
      const float inv = __fdiv_rn(out_scale, l);
      if (p.lse != nullptr && row_ok) {
        // ln sum_j exp(s_ij) = (M + log2 l) ln 2: l sums the rounded weights relative to 2^M
        p.lse[(static_cast<size_t>(u.b) * p.H + u.h) * p.S + row] =
            (static_cast<float>(m_ref) + __log2f(l)) * 0.6931471805599453f;
      }
      // The warp's 32 rows go out through its staging tile, kEpiCols columns at a time, as TMA
      // stores (each row is contiguous in global memory only within itself, so stores straight from
      // the row-per-lane registers would touch 32 lines per instruction); rows past S are clipped.
      constexpr int kCW = C::kEpiCols, kPieces = kCW * 2 / 16;  // 16-byte pieces per staged row
#pragma unroll
      for (int c = 0; c < DV / kCW; ++c) {
        const uint32_t* r = o + c * kCW;
        uint32_t packed[kCW / 2];
#pragma unroll
        for (int i = 0; i < kCW / 2; ++i)
          packed[i] = cvt_bf16x2(__uint_as_float(r[2 * i + 1]) * inv, __uint_as_float(r[2 * i]) * inv);
        // the store that last used this tile has finished reading it
        const uint32_t tile = epi_tile + (c % C::kEpiBufs) * C::kEpiWarpBytes;
        if (lane == 0) {
          if constexpr (C::kEpiBufs == 2) bulk_wait_read_but1();
          else bulk_wait_read_all();
        }
        __syncwarp();
        // row `lane` at lane * kCW * 2 bytes; 16-byte piece i at (i ^ swz), the TMA swizzle of the
        // map (64-byte rows: piece ^= (row >> 1) & 3; 32-byte rows: piece ^= (row >> 2) & 1)
        const int swz = kPieces == 4 ? (lane >> 1) & 3 : (lane >> 2) & 1;
#pragma unroll
        for (int i = 0; i < kPieces; ++i)
          st_shared_v4(tile + lane * (kCW * 2) + ((i ^ swz) << 4), packed[4 * i], packed[4 * i + 1],
                       packed[4 * i + 2], packed[4 * i + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_4d(&maps.o, tile, c * kCW, u.h, row0 + quarter * 32, u.b);
          bulk_commit();
        }
      }
      tc_fence_before();
    }
    if (!ok && lane == 0) give_up();
    if (lane == 0) bulk_wait_all();  // the output stores are complete before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace zyfa
