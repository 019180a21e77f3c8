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
//   out_i = dv * sum_j w_ij v8_j / sum_j w_ij with the same rounded weights w (the row sum is an
//   same block-scaled PV MMA, widened by 16 columns whose B operand is a tile of ones: the pages'
//   "one extra matrix instruction per block", +16/DV of the PV work).
// BF16 twin: p_ij = bf16(2^(S_ij*a' - M)), a' = fl32(scale*log2 e), normalised by the sum of the
// rounded p (same widened PV MMA), no block scaling.
//
// Schedule (one persistent CTA per SM, one work unit = (b, h, 256 query rows) = two 128-row tiles):
//   warp 0      TMA producer: K/V tiles of 64 keys into a ring of shared-memory stages (BF16: Q too)
//   warp 1      MMA issuer (one thread) and TMEM owner
//   warps 4..7  softmax warpgroup 0 (query tile 0), warps 8..11 softmax warpgroup 1 (query tile 1)
// The MMA thread interleaves the tiles, S0(j+1) between PV0(j) and PV1(j), so one warpgroup computes
// probabilities while the tensor core works on the other tile (the pages' ping-pong, here between
// two query tiles with mbarrier completion tracking instead of instruction order).
//
// Tensor memory (512 columns x 128 lanes, lane = query row of the tile):
//   [  0, 64) S0 (fp32 scores); after the softmax reads it: P0 at 0 (fp8: 16 cols, bf16: 32 cols),
//             FP8 scale factors of P0 at 32..35, of V (all 1.0) at 48..55
//   [ 64,128) S1, P1, scale factors of tile 1
//   [128,128+DV+16) O0 | l0, then O1 | l1   (fp32 accumulators: DV output columns followed by 16
//             identical columns holding the rounded row sum)
//   [416,512) Q0, Q1 (FP8 only: e4m3 query rows, DQK/4 columns each)
// Shared memory per pipeline stage: the K tile, then the V tile (MN-major, 1-2 swizzle atoms) followed
// by one atom of ones, so the widened PV MMA reads [V | 1] with a single descriptor.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace zyfa {

// Status bits a kernel may set in the library's status word.
enum : int { kStatusTimeout = 1 };

constexpr int kBlockN = 64;          // keys per K/V tile = keys per scale block
constexpr int kBlockM = 128;         // query rows per tile
constexpr int kUnitRows = 2 * kBlockM;
constexpr int kThreads = 384;
constexpr int kRescaleBinades = 8;   // lazy reference update threshold (binades)
constexpr float kLeanPC0 = 55.625f;  // Lean-P constant: code(2^x) = rne(8x + 55.625)
constexpr long long kWaitLimit = 1ll << 31;  // ~1 s of SM clocks before a wait gives up

template <bool FP8, int DQK, int DV>
struct Cfg {
  static constexpr int kElem = FP8 ? 1 : 2;
  static constexpr int kRowBytesK = DQK * kElem;
  static constexpr int kChunks128K = kRowBytesK / 128;                 // 128-byte K-major chunks
  static constexpr bool kTail64K = (kRowBytesK % 128) == 64;           // one 64-byte chunk
  static_assert(kRowBytesK % 64 == 0, "head dim must give whole 64-byte chunks");
  static constexpr int kKStageBytes = kBlockN * kRowBytesK;
  static constexpr int kRowBytesV = DV * kElem;
  static_assert(kRowBytesV == 64 || kRowBytesV % 128 == 0, "value row must be 64 or k*128 bytes");
  static constexpr int kVAtoms = kRowBytesV >= 128 ? kRowBytesV / 128 : 1;
  static constexpr int kVAtomBytes = kBlockN * (kRowBytesV >= 128 ? 128 : 64);
  static constexpr int kVStageBytes = kBlockN * kRowBytesV;                // bytes TMA writes
  static constexpr int kVRegionBytes = (kVAtoms + 1) * kVAtomBytes;        // + the ones atom
  static constexpr int kNO = DV + 16;                                      // PV MMA width
  static constexpr int kQTileBytes = FP8 ? 0 : kBlockM * kRowBytesK;  // BF16 keeps Q in smem
  static constexpr int kKSteps = kRowBytesK / 32;                      // 32 bytes of K per MMA
  static constexpr int kKeysPerStep = FP8 ? 32 : 16;
  static constexpr int kPVSteps = kBlockN / kKeysPerStep;
  static constexpr int kSmemBudget = 220 * 1024;
  static constexpr int kFixedBytes = 2 * kQTileBytes + 1024 /*align slack*/;
  static constexpr int kStageBytes = kKStageBytes + kVRegionBytes;
  static constexpr int kStagesRaw = (kSmemBudget - kFixedBytes) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static_assert(kStages >= 2, "not enough shared memory for two K/V stages");
  static constexpr int kSmemBytes = kFixedBytes + kStages * kStageBytes;
  // TMEM columns of query tile t
  __device__ static constexpr uint32_t col_s(int t) { return 64u * t; }
  __device__ static constexpr uint32_t col_o(int t) { return 128u + static_cast<uint32_t>(kNO) * t; }
  __device__ static constexpr uint32_t col_l(int t) { return col_o(t) + DV; }
  __device__ static constexpr uint32_t col_q(int t) { return 416u + (DQK / 4) * t; }
  static_assert(128 + 2 * kNO <= 416, "O accumulators overlap the Q columns");
  static_assert(!FP8 || 416 + 2 * (DQK / 4) <= 512, "TMEM overflow");
  static_assert(DV <= 128 && kNO % 16 == 0, "PV MMA width must be a multiple of 16, at most 144");
  static constexpr uint32_t kColSFA = 32, kColSFB = 48;
};

struct Params {
  const uint8_t* q;  // [B,S,H,DQK] e4m3 or bf16
  __nv_bfloat16* out;  // [B,S,H,DV]
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  int B, S, H, H_kv;
  float softmax_scale;
  int num_units;     // B*H*ceil(S/256)
  int* status;       // device status word (timeouts)
};

struct __align__(8) SharedCtl {
  uint64_t k_full[8], k_empty[8], v_full[8], v_empty[8];
  uint64_t q_full[2], q_empty[2], s_full[2], p_full[2], o_done[2];
  uint64_t drain;
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
  const int nqb = (p.S + kUnitRows - 1) / kUnitRows;
  const int qb = nqb - 1 - idx / bh;
  const int rest = idx % bh;
  u.b = rest / p.H;
  u.h = rest % p.H;
  u.r0 = qb * kUnitRows;
  return true;
}

// Number of 64-key tiles tile t of a unit needs (0 if it has no rows).
__device__ __forceinline__ int tiles_for(const Params& p, int r0, int t) {
  const int first = r0 + t * kBlockM;
  if (first >= p.S) return 0;
  const int end = min(first + kBlockM, p.S);
  return (end + kBlockN - 1) / kBlockN;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
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

template <bool FP8, int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    zyfa_fwd_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k0, const __grid_constant__ CUtensorMap tm_k1,
                    const __grid_constant__ CUtensorMap tm_v) {
  using C = Cfg<FP8, DQK, DV>;
  using namespace ptx;
  extern __shared__ uint8_t smem_raw[];
  __shared__ SharedCtl ctl;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- shared memory carve-up (1024-byte aligned for the 128-byte swizzle) ----
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t s_q = base;                          // BF16: two Q tiles
  const uint32_t s_stages = s_q + 2 * C::kQTileBytes; // K/V ring
  auto k_stage = [&](int s) { return s_stages + s * C::kStageBytes; };
  auto v_stage = [&](int s) { return s_stages + s * C::kStageBytes + C::kKStageBytes; };  // 1024-aligned

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&ctl.k_full[s]), 1);
      mbar_init(smem_u32(&ctl.k_empty[s]), 1);
      mbar_init(smem_u32(&ctl.v_full[s]), 1);
      mbar_init(smem_u32(&ctl.v_empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&ctl.q_full[t]), FP8 ? 4 : 1);
      mbar_init(smem_u32(&ctl.q_empty[t]), 1);
      mbar_init(smem_u32(&ctl.s_full[t]), 1);
      mbar_init(smem_u32(&ctl.p_full[t]), 4);
      mbar_init(smem_u32(&ctl.o_done[t]), 1);
    }
    mbar_init(smem_u32(&ctl.drain), 1);
    ctl.abort_ = 0;
    fence_mbar_init();
  }
  {
    // the ones atom after every V tile: e4m3 1.0 = 0x38, bf16 1.0 = 0x3F80
    const uint32_t one = FP8 ? 0x38383838u : 0x3F803F80u;
    for (int st = 0; st < C::kStages; ++st) {
      uint32_t* o32 = reinterpret_cast<uint32_t*>(base_ptr + (v_stage(st) - base) + C::kVAtoms * C::kVAtomBytes);
      for (int i = tid; i < C::kVAtomBytes / 4; i += kThreads) o32[i] = one;
    }
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
    // =========================== TMA producer ===========================
    if (lane == 0) {
      tma_prefetch_desc(&tm_k0);
      tma_prefetch_desc(&tm_v);
      if (C::kTail64K) tma_prefetch_desc(&tm_k1);
      if (!FP8) tma_prefetch_desc(&tm_q);
      uint32_t k_cnt = 0, v_cnt = 0;  // K / V tiles issued
      uint32_t q_cnt[2] = {0, 0};      // BF16 Q tiles issued
      bool ok = true;
      Unit u;
      for (int round = 0; ok && unit_at(p, round, u); ++round) {
        const int hk = u.h / hgroup;
        const int n0 = tiles_for(p, u.r0, 0), n1 = tiles_for(p, u.r0, 1);
        const int nkv = n1 > n0 ? n1 : n0;
        if (!FP8) {
          for (int t = 0; t < 2 && ok; ++t) {
            if ((t == 0 ? n0 : n1) == 0) continue;
            ok = mbar_wait(smem_u32(&ctl.q_empty[t]), (q_cnt[t] & 1) ^ 1, abort_flag, kWaitLimit);
            if (!ok) break;
            const uint32_t bar = smem_u32(&ctl.q_full[t]);
            mbar_arrive_expect_tx(bar, C::kQTileBytes);
            for (int c = 0; c < C::kChunks128K; ++c)
              tma_load_4d(s_q + t * C::kQTileBytes + c * (kBlockM * 128), &tm_q, bar, c * (128 / C::kElem),
                          u.h, u.r0 + t * kBlockM, u.b);
            ++q_cnt[t];
          }
        }
        for (int j = 0; j < nkv && ok; ++j) {
          const int st = k_cnt % C::kStages;
          const uint32_t ph = ((k_cnt / C::kStages) & 1) ^ 1;
          ok = mbar_wait(smem_u32(&ctl.k_empty[st]), ph, abort_flag, kWaitLimit);
          if (!ok) break;
          const uint32_t kb = smem_u32(&ctl.k_full[st]);
          mbar_arrive_expect_tx(kb, C::kKStageBytes);
          for (int c = 0; c < C::kChunks128K; ++c)
            tma_load_4d(k_stage(st) + c * (kBlockN * 128), &tm_k0, kb, c * (128 / C::kElem), hk, j * kBlockN, u.b);
          if (C::kTail64K)
            tma_load_4d(k_stage(st) + C::kChunks128K * (kBlockN * 128), &tm_k1, kb,
                        C::kChunks128K * (128 / C::kElem), hk, j * kBlockN, u.b);
          ++k_cnt;
          ok = mbar_wait(smem_u32(&ctl.v_empty[st]), ph, abort_flag, kWaitLimit);
          if (!ok) break;
          const uint32_t vb = smem_u32(&ctl.v_full[st]);
          mbar_arrive_expect_tx(vb, C::kVStageBytes);
          for (int c = 0; c < C::kVAtoms; ++c)
            tma_load_4d(v_stage(st) + c * C::kVAtomBytes, &tm_v, vb, c * (128 / C::kElem), hk, j * kBlockN, u.b);
          ++v_cnt;
        }
      }
      if (!ok) {
        give_up();
        // every load already issued lands before the CTA may exit (its shared memory is released then)
        const int never = 0;
        const uint32_t ns = C::kStages;
        for (uint32_t i = (k_cnt > ns ? k_cnt - ns : 0); i < k_cnt; ++i)
          mbar_wait(smem_u32(&ctl.k_full[i % ns]), (i / ns) & 1, &never, kWaitLimit);
        for (uint32_t i = (v_cnt > ns ? v_cnt - ns : 0); i < v_cnt; ++i)
          mbar_wait(smem_u32(&ctl.v_full[i % ns]), (i / ns) & 1, &never, kWaitLimit);
        for (int t = 0; t < 2; ++t)
          if (q_cnt[t] > 0) mbar_wait(smem_u32(&ctl.q_full[t]), (q_cnt[t] - 1) & 1, &never, kWaitLimit);
      }
    }
  } else if (warp == 1) {
    // =========================== MMA issuer ===========================
    if (lane == 0) {
      const uint32_t idesc_s = idesc_dense(FP8 ? kFmtE4M3 : kFmtBF16, FP8 ? kFmtE4M3 : kFmtBF16, false, false,
                                           kBlockM, kBlockN);
      uint32_t kv_cnt = 0;
      uint32_t q_cnt[2] = {0, 0}, p_cnt[2] = {0, 0};
      bool ok = true;

      auto k_desc = [&](int st, int ks) -> uint64_t {
        const int off = ks * 32;
        if (off < C::kChunks128K * 128)
          return smem_desc(k_stage(st) + (off / 128) * (kBlockN * 128) + (off % 128), 16, 1024, kSwizzle128B);
        return smem_desc(k_stage(st) + C::kChunks128K * (kBlockN * 128) + (off - C::kChunks128K * 128), 16, 512,
                         kSwizzle64B);
      };
      auto issue_s = [&](int t, int st) {
        const uint32_t d = tmem + C::col_s(t);
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          if constexpr (FP8) {
            mma_f8_ts(d, tmem + C::col_q(t) + ks * 8, k_desc(st, ks), idesc_s, ks > 0);
          } else {
            const int off = ks * 32;
            const uint64_t qd = smem_desc(s_q + t * C::kQTileBytes + (off / 128) * (kBlockM * 128) + (off % 128), 16,
                                          1024, kSwizzle128B);
            mma_f16_ss(d, qd, k_desc(st, ks), idesc_s, ks > 0);
          }
        }
        tc_commit(smem_u32(&ctl.s_full[t]));
      };
      // O|l += P x [V | 1]: one MMA per K step, DV + 16 columns wide
      auto issue_pv = [&](int t, int st, bool first) {
        const uint32_t o = tmem + C::col_o(t), pa = tmem + C::col_s(t);
        for (int ks = 0; ks < C::kPVSteps; ++ks) {
          const uint32_t vaddr = v_stage(st) + ks * C::kKeysPerStep * (C::kRowBytesV >= 128 ? 128 : 64);
          const uint64_t vd = C::kRowBytesV >= 128 ? smem_desc(vaddr, C::kVAtomBytes, 1024, kSwizzle128B)
                                                   : smem_desc(vaddr, C::kVAtomBytes, 512, kSwizzle64B);
          const uint32_t acc = (!first || ks > 0) ? 1u : 0u;
          if constexpr (FP8) {
            const uint32_t sfa = tmem + C::col_s(t) + C::kColSFA, sfb = tmem + C::col_s(t) + C::kColSFB;
            mma_mxf8_ts(o, pa + ks * 8, vd, idesc_block_scaled(kFmtE4M3, kFmtE4M3, true, kBlockM, C::kNO, ks, 0), sfa,
                        sfb, acc);
          } else {
            mma_f16_ts(o, pa + ks * 8, vd, idesc_dense(kFmtBF16, kFmtBF16, false, true, kBlockM, C::kNO), acc);
          }
        }
        tc_commit(smem_u32(&ctl.o_done[t]));
      };
      auto wait_k = [&](uint32_t cnt) {
        return mbar_wait(smem_u32(&ctl.k_full[cnt % C::kStages]), (cnt / C::kStages) & 1, abort_flag, kWaitLimit);
      };
      auto wait_v = [&](uint32_t cnt) {
        return mbar_wait(smem_u32(&ctl.v_full[cnt % C::kStages]), (cnt / C::kStages) & 1, abort_flag, kWaitLimit);
      };

      Unit u;
      for (int round = 0; ok && unit_at(p, round, u); ++round) {
        const int n[2] = {tiles_for(p, u.r0, 0), tiles_for(p, u.r0, 1)};
        const int nkv = n[1] > n[0] ? n[1] : n[0];
        for (int t = 0; t < 2 && ok; ++t) {
          if (n[t] == 0) continue;
          ok = mbar_wait(smem_u32(&ctl.q_full[t]), q_cnt[t] & 1, abort_flag, kWaitLimit);
          ++q_cnt[t];
        }
        if (!ok) break;
        tc_fence_after();
        // prologue: S0(0), S1(0)
        ok = wait_k(kv_cnt);
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; t < 2; ++t)
          if (n[t] > 0) {
            issue_s(t, kv_cnt % C::kStages);
            if (!FP8 && n[t] == 1) tc_commit(smem_u32(&ctl.q_empty[t]));
          }
        tc_commit(smem_u32(&ctl.k_empty[kv_cnt % C::kStages]));
        for (int j = 0; j < nkv && ok; ++j) {
          const uint32_t cur = kv_cnt + j, nxt = cur + 1;
          const bool more = j + 1 < nkv;
          ok = wait_v(cur);
          if (!ok) break;
          bool k_ready = false;
          for (int t = 0; t < 2 && ok; ++t) {
            if (j < n[t]) {
              ok = mbar_wait(smem_u32(&ctl.p_full[t]), p_cnt[t] & 1, abort_flag, kWaitLimit);
              if (!ok) break;
              ++p_cnt[t];
              tc_fence_after();
              issue_pv(t, cur % C::kStages, j == 0);
            }
            if (t == 1) tc_commit(smem_u32(&ctl.v_empty[cur % C::kStages]));
            if (more && j + 1 < n[t]) {
              if (!k_ready) {
                ok = wait_k(nxt);
                if (!ok) break;
                tc_fence_after();
                k_ready = true;
              }
              issue_s(t, nxt % C::kStages);
              // BF16: last S MMA of this tile issued; its Q tile may be refilled once it completes
              if (!FP8 && j + 2 == n[t]) tc_commit(smem_u32(&ctl.q_empty[t]));
            }
          }
          if (ok && more) tc_commit(smem_u32(&ctl.k_empty[nxt % C::kStages]));
        }
        kv_cnt += nkv;
      }
      if (!ok) give_up();
      // drain: all MMAs issued by this thread complete before TMEM is released
      const int never = 0;
      tc_commit(smem_u32(&ctl.drain));
      mbar_wait(smem_u32(&ctl.drain), 0, &never, kWaitLimit);
    }
  } else if (warp >= 4) {
    // =========================== softmax warpgroups ===========================
    const int t = (warp - 4) >> 2;            // query tile of this warpgroup
    const int quarter = warp & 3;             // TMEM lane quarter of this warp
    const int rloc = quarter * 32 + lane;     // row within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::col_s(t);
    const uint32_t tO = tmem + lane_addr + C::col_o(t);
    const uint32_t tL = tmem + lane_addr + C::col_l(t);

    float a;
    if constexpr (FP8) {
      const float dq = p.q_descale ? *p.q_descale : 1.0f;
      const float dk = p.k_descale ? *p.k_descale : 1.0f;
      a = __fmul_rn(__fmul_rn(__fmul_rn(p.softmax_scale, dq), dk), 11.541560327111707f);
    } else {
      a = __fmul_rn(p.softmax_scale, 1.4426950408889634f);
    }
    const float out_scale = (FP8 && p.v_descale) ? *p.v_descale : 1.0f;
    const float a24 = a * 0x1p-24f;  // exact: scales the Lean-P result into f16 subnormal units

    uint32_t s_cnt = 0, p_cnt = 0;
    bool ok = true;
    Unit u;
    for (int round = 0; ok && unit_at(p, round, u); ++round) {
      const int ntiles = tiles_for(p, u.r0, t);
      if (ntiles == 0) continue;
      const int row0 = u.r0 + t * kBlockM;   // first row of the tile
      const int row = row0 + rloc;
      const bool row_ok = row < p.S;
      if constexpr (FP8) {
        // Q row -> TMEM (zeros past the end of the sequence)
        uint32_t w[32];
        const uint4* qrow = reinterpret_cast<const uint4*>(
            p.q + ((static_cast<size_t>(u.b) * p.S + (row_ok ? row : 0)) * p.H + u.h) * DQK);
        constexpr int kVec = DQK / 16;
        constexpr int kFirst = kVec < 8 ? kVec : 8;
#pragma unroll
        for (int i = 0; i < kFirst; ++i) {
          uint4 x = row_ok ? __ldg(qrow + i) : make_uint4(0, 0, 0, 0);
          w[4 * i] = x.x; w[4 * i + 1] = x.y; w[4 * i + 2] = x.z; w[4 * i + 3] = x.w;
        }
        if constexpr (DQK == 64) {
          uint32_t w16[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w16[i] = w[i];
          tmem_st16(tmem + lane_addr + C::col_q(t), w16);
        } else {
          tmem_st32(tmem + lane_addr + C::col_q(t), w);
          if constexpr (DQK == 192) {
            uint32_t w16[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 x = row_ok ? __ldg(qrow + 8 + i) : make_uint4(0, 0, 0, 0);
              w16[4 * i] = x.x; w16[4 * i + 1] = x.y; w16[4 * i + 2] = x.z; w16[4 * i + 3] = x.w;
            }
            tmem_st16(tmem + lane_addr + C::col_q(t) + 32, w16);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl.q_full[t]));
      }

      int m_ref = 0;
      for (int j = 0; j < ntiles; ++j) {
        ok = mbar_wait(smem_u32(&ctl.s_full[t]), s_cnt & 1, abort_flag, kWaitLimit);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        ++s_cnt;
        tc_fence_after();
        float s[64];
        {
          uint32_t r[32];
          tmem_ld32(tS, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(r[i]);
          tmem_ld32(tS + 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) s[32 + i] = __uint_as_float(r[i]);
        }
        const int key0 = j * kBlockN;
        if (key0 + kBlockN - 1 > row0) {  // tile touches the diagonal: mask keys after the row
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (key0 + i > row) s[i] = -INFINITY;
        }
        float mx = fmax3(s[0], s[1], s[2]);
#pragma unroll
        for (int i = 3; i < 63; i += 2) mx = fmax3(mx, s[i], s[i + 1]);
        mx = fmaxf(mx, s[63]);

        // block exponent (FP8: ceil(max u / 8); BF16: ceil(max log2-score)) and lazy reference update
        const bool empty = mx == -INFINITY;
        int e;
        if constexpr (FP8) e = empty ? 0 : static_cast<int>(ceilf(__fmul_rn(mx, a) * 0.125f));
        else e = empty ? 0 : static_cast<int>(ceilf(__fmul_rn(mx, a)));
        if (j == 0) {
          m_ref = e;
        } else {
          const bool need = !empty && e > m_ref + kRescaleBinades;
          if (__any_sync(0xffffffffu, need)) {
            // the previous PV into this tile's accumulators must be complete before rescaling
            ok = mbar_wait(smem_u32(&ctl.o_done[t]), (p_cnt - 1) & 1, abort_flag, kWaitLimit);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const float f = need ? exp2i(m_ref - e) : 1.0f;
            uint32_t r[32];
#pragma unroll
            for (int c = 0; c < DV / 32; ++c) {
              tmem_ld32(tO + 32 * c, r);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
              tmem_st32(tO + 32 * c, r);
            }
            uint32_t lv;
            tmem_ld1(tL, lv);
            tmem_wait_ld();
            tmem_st1(tL, __float_as_uint(__uint_as_float(lv) * f));
            tmem_wait_st();
            if (need) m_ref = e;
          }
        }

        if constexpr (FP8) {
          // Lean P: t = fma(s, a, 55.625 - 8e) in units of 2^-24, so the f16 subnormal produced by
          // the rounding conversion carries the integer code in its low byte (negative -> 0).
          const float c24 = __fmul_rn(kLeanPC0 - 8.0f * static_cast<float>(e), 0x1p-24f);
          uint32_t pw[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float t0 = __fmaf_rn(s[4 * i + 0], a24, c24);
            const float t1 = __fmaf_rn(s[4 * i + 1], a24, c24);
            const float t2 = __fmaf_rn(s[4 * i + 2], a24, c24);
            const float t3 = __fmaf_rn(s[4 * i + 3], a24, c24);
            pw[i] = prmt(cvt_relu_f16x2(t1, t0), cvt_relu_f16x2(t3, t2), 0x6420u);
          }
          int sf = 127 + e - m_ref;
          sf = sf < 0 ? 0 : (sf > 254 ? 254 : sf);
          const uint32_t sfw = static_cast<uint32_t>(sf) * 0x01010101u;
          tmem_st16(tS, pw);
          tmem_st4(tS + C::kColSFA, sfw, sfw, sfw, sfw);
          tmem_st4(tS + C::kColSFB, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
          tmem_st4(tS + C::kColSFB + 4, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        } else {
          const float negm = -static_cast<float>(m_ref);
          uint32_t pw[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            pw[i] = cvt_bf16x2(ex2(__fmaf_rn(s[2 * i + 1], a, negm)), ex2(__fmaf_rn(s[2 * i], a, negm)));
          tmem_st32(tS, pw);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl.p_full[t]));
        ++p_cnt;
      }
      if (!ok) break;

      // epilogue: out = O * (dv / l) -> bf16
      ok = mbar_wait(smem_u32(&ctl.o_done[t]), (p_cnt - 1) & 1, abort_flag, kWaitLimit);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t lv;
      tmem_ld1(tL, lv);
      tmem_wait_ld();
      const float inv = __fdiv_rn(out_scale, __uint_as_float(lv));
      __nv_bfloat16* orow = p.out + ((static_cast<size_t>(u.b) * p.S + (row_ok ? row : 0)) * p.H + u.h) * DV;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + 32 * c, r);
        tmem_wait_ld();
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          packed[i] = cvt_bf16x2(__uint_as_float(r[2 * i + 1]) * inv, __uint_as_float(r[2 * i]) * inv);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
      }
      tc_fence_before();
    }
    if (!ok && lane == 0) give_up();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace zyfa
