// C ABI of libzyfa.so: argument checks, TMA tensor maps, per-device status word, dispatch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/zyfa.h"
#include "launch.h"

namespace {

// Set by a kernel that gave up on a pipeline wait; read and cleared by zyfa_check_errors.
__device__ int g_zyfa_status;

constexpr int kMaxDevices = 64;
constexpr int kUnitRows = 256;  // query rows per work unit (two 128-row tiles)

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int*> g_status_ptr[kMaxDevices];

// Copy streams of the host-buffer entry point, one pair per device, created on first use and kept
// for the life of the process (uploads and downloads run beside the caller's compute stream).
constexpr int kMaxHostChunks = 64;
std::mutex g_stream_mutex;
cudaStream_t g_up[kMaxDevices], g_down[kMaxDevices];

bool copy_streams(int dev, cudaStream_t* up, cudaStream_t* down) {
  std::lock_guard<std::mutex> lock(g_stream_mutex);
  if (!g_up[dev]) {
    cudaStream_t a = nullptr, b = nullptr;
    if (cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking) != cudaSuccess) {
      cudaStreamDestroy(a);
      return false;
    }
    g_up[dev] = a;
    g_down[dev] = b;
  }
  *up = g_up[dev];
  *down = g_down[dev];
  return true;
}

// Events of one host-buffer call; destroying a recorded event is safe (its resources go once it fired).
struct EventSet {
  cudaEvent_t e[2 * kMaxHostChunks + 2] = {};
  int n = 0;
  bool create(int count) {
    for (; n < count; ++n)
      if (cudaEventCreateWithFlags(&e[n], cudaEventDisableTiming) != cudaSuccess) return false;
    return true;
  }
  ~EventSet() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(e[i]);
  }
};

// Device-side address of the status word for the current device (looked up once per device).
int* status_ptr(int dev) {
  int* p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_zyfa_status) != cudaSuccess) return nullptr;
  g_status_ptr[dev].store(static_cast<int*>(addr), std::memory_order_release);
  return static_cast<int*>(addr);
}

int sm_count(int dev) {
  int n = g_sm_count[dev].load(std::memory_order_acquire);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
  g_sm_count[dev].store(n, std::memory_order_release);
  return n;
}

// 4-D map over a [B][S][heads][D] tensor: box = {box_inner elements of D, 1 head, box_rows rows, 1}.
bool make_map(CUtensorMap* m, const void* base, bool fp8, int D, int heads, int S, int B, int box_inner,
              int box_rows, CUtensorMapSwizzle sw) {
  const int es = fp8 ? 1 : 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * es, static_cast<cuuint64_t>(heads) * D * es,
                           static_cast<cuuint64_t>(S) * heads * D * es};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_inner), 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FP8, int DQK, int DV, bool EXACT>
zyfa_status_t run(zyfa::LaunchArgs& a, const void* q, const void* k, const void* v) {
  constexpr int es = FP8 ? 1 : 2;
  constexpr int kRowK = DQK * es, kRowV = DV * es;
  constexpr int kChunk = 128 / es;  // elements per 128-byte chunk
  constexpr int BN = zyfa::tile_keys<FP8, DQK, DV>();
  constexpr int kRowsQ = 128;
  bool ok = true;
  zyfa::Maps& m = a.maps;
  // Q and K rows: 128-byte chunks with the 128-byte swizzle, a 64-byte tail chunk with the 64-byte one
  if (kRowK >= 128) {
    ok &= make_map(&m.q0, q, FP8, DQK, a.H, a.S, a.B, kChunk, kRowsQ, CU_TENSOR_MAP_SWIZZLE_128B);
    ok &= make_map(&m.k0, k, FP8, DQK, a.H_kv, a.S, a.B, kChunk, BN, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (kRowK % 128 == 64) {
    ok &= make_map(&m.q1, q, FP8, DQK, a.H, a.S, a.B, 64 / es, kRowsQ, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= make_map(&m.k1, k, FP8, DQK, a.H_kv, a.S, a.B, 64 / es, BN, CU_TENSOR_MAP_SWIZZLE_64B);
  }
  // V: MN-major tiles, one swizzle atom per 128 bytes (or the whole 64-byte row) of the value row
  ok &= make_map(&m.v, v, FP8, DV, a.H_kv, a.S, a.B, kRowV >= 128 ? kChunk : DV, BN,
                 kRowV >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
  // output: per-warp boxes of 32 rows x kEpiCols bf16 columns, swizzled like the staging tile
  const int epi_cols = zyfa::epi_cols<FP8, DQK, DV>();
  ok &= make_map(&m.o, a.out, false, DV, a.H, a.S, a.B, epi_cols, 32,
                 epi_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  if (!ok) return ZYFA_ERR_CUDA;
  // maps the instantiation never touches are copies of valid ones
  if (kRowK < 128) { m.q0 = m.q1; m.k0 = m.k1; }
  if (kRowK % 128 != 64) { m.q1 = m.q0; m.k1 = m.k0; }
  return zyfa::launch_fwd<FP8, DQK, DV, EXACT>(a) == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* zyfa_status_string(zyfa_status_t s) {
  switch (s) {
    case ZYFA_OK: return "ZYFA_OK";
    case ZYFA_ERR_INVALID_ARG: return "ZYFA_ERR_INVALID_ARG";
    case ZYFA_ERR_UNSUPPORTED: return "ZYFA_ERR_UNSUPPORTED";
    case ZYFA_ERR_MISALIGNED: return "ZYFA_ERR_MISALIGNED";
    case ZYFA_ERR_CUDA: return "ZYFA_ERR_CUDA";
    case ZYFA_ERR_TIMEOUT: return "ZYFA_ERR_TIMEOUT";
  }
  return "ZYFA_ERR_UNKNOWN";
}

int zyfa_kernel_launches(int B, int S, int H) { return (B > 0 && S > 0 && H > 0) ? 1 : 0; }

}  // extern "C"

namespace {

// Shared body of the entry points: validation, tensor maps, launch.  stall_loads != 0 makes the
// kernel's producer withhold every load (the self-test of the timeout path).
zyfa_status_t attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int S, int H, int H_kv,
                       int D_qk, int D_v, float softmax_scale, zyfa_dtype_t dtype, const float* q_descale,
                       const float* k_descale, const float* v_descale, const zyfa_fwd_options_t* opts,
                       cudaStream_t stream, int stall_loads, long long qb_begin = 0, long long qb_end = -1) {
  if (B < 1 || H < 1 || H_kv < 1 || S < 0 || H % H_kv != 0) return ZYFA_ERR_INVALID_ARG;
  if (dtype != ZYFA_DTYPE_E4M3 && dtype != ZYFA_DTYPE_BF16) return ZYFA_ERR_INVALID_ARG;
  zyfa_fwd_options_t o = {ZYFA_P_LEAN, 0, nullptr};
  if (opts) o = *opts;
  if (o.p_mode != ZYFA_P_LEAN && o.p_mode != ZYFA_P_EXACT && o.p_mode != ZYFA_P_EXACT_NO_BLOCK_SCALE)
    return ZYFA_ERR_INVALID_ARG;
  if (o.descale_per_kv_head != 0 && o.descale_per_kv_head != 1) return ZYFA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(o.lse) & 3u) != 0) return ZYFA_ERR_MISALIGNED;
  if (!std::isfinite(softmax_scale) || softmax_scale < 0.0f) return ZYFA_ERR_INVALID_ARG;
  const bool shape_ok = (D_qk == 64 && D_v == 64) || (D_qk == 128 && D_v == 128) || (D_qk == 192 && D_v == 128);
  if (!shape_ok) return ZYFA_ERR_UNSUPPORTED;
  if (S == 0) return ZYFA_OK;
  if (!q || !k || !v || !out) return ZYFA_ERR_INVALID_ARG;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out)) return ZYFA_ERR_MISALIGNED;
  const long long nqb = (static_cast<long long>(S) + kUnitRows - 1) / kUnitRows;
  if (nqb * B * H > (1ll << 30) || static_cast<long long>(S) > (1ll << 30)) return ZYFA_ERR_UNSUPPORTED;
  if (qb_end < 0) qb_end = nqb;
  if (qb_begin < 0 || qb_begin >= qb_end || qb_end > nqb) return ZYFA_ERR_INVALID_ARG;
  const long long units = (qb_end - qb_begin) * B * H;
  if (softmax_scale == 0.0f) softmax_scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D_qk)));
  if (!get_encode()) return ZYFA_ERR_CUDA;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ZYFA_ERR_CUDA;
  const int nsm = sm_count(dev);
  int* status = status_ptr(dev);
  if (nsm <= 0 || !status) return ZYFA_ERR_CUDA;

  zyfa::LaunchArgs a;
  std::memset(&a, 0, sizeof(a));
  a.out = out;
  const bool fp8 = dtype == ZYFA_DTYPE_E4M3;
  a.q_descale = fp8 ? q_descale : nullptr;
  a.k_descale = fp8 ? k_descale : nullptr;
  a.v_descale = fp8 ? v_descale : nullptr;
  a.B = B;
  a.S = S;
  a.H = H;
  a.H_kv = H_kv;
  a.softmax_scale = softmax_scale;
  a.num_units = static_cast<int>(units);
  a.qb_end = static_cast<int>(qb_end);
  a.status = status;
  a.grid = static_cast<int>(units < nsm ? units : nsm);
  a.stream = stream;
  a.stall_loads = stall_loads;
  a.lse = o.lse;
  a.desc_per_head = fp8 ? o.descale_per_kv_head : 0;
  a.no_block_scale = fp8 && o.p_mode == ZYFA_P_EXACT_NO_BLOCK_SCALE ? 1 : 0;
  // Block-scaled FP8: a block's largest weight is at most 1 and |v| at most 448, so with the row
  // reference lagging the row's largest block exponent by at most L binades each key adds at most
  // 448 * 2^L to O (and 2^L to l): over S keys below 2^(8.8 + L + log2 S), which fp32 holds while
  // L + log2 S < 118.  96 binades up to 2^21 keys, 64 beyond; the e8m0 scale factors hold either.
  a.rescale_binades = S <= (1 << 21) ? 96 : 64;
  if (fp8 && (o.p_mode == ZYFA_P_EXACT || o.p_mode == ZYFA_P_EXACT_NO_BLOCK_SCALE)) {
    if (D_qk == 64) return run<true, 64, 64, true>(a, q, k, v);
    if (D_qk == 128) return run<true, 128, 128, true>(a, q, k, v);
    return run<true, 192, 128, true>(a, q, k, v);
  }
  if (fp8) {
    if (D_qk == 64) return run<true, 64, 64, false>(a, q, k, v);
    if (D_qk == 128) return run<true, 128, 128, false>(a, q, k, v);
    return run<true, 192, 128, false>(a, q, k, v);
  }
  if (D_qk == 64) return run<false, 64, 64, false>(a, q, k, v);
  if (D_qk == 128) return run<false, 128, 128, false>(a, q, k, v);
  return run<false, 192, 128, false>(a, q, k, v);
}

}  // namespace

extern "C" {

zyfa_status_t zyfa_attn_fwd_causal(const void* q, const void* k, const void* v, void* out, int B, int S, int H,
                                   int H_kv, int D_qk, int D_v, float softmax_scale, zyfa_dtype_t dtype,
                                   const float* q_descale, const float* k_descale, const float* v_descale,
                                   cudaStream_t stream) {
  return attn_fwd(q, k, v, out, B, S, H, H_kv, D_qk, D_v, softmax_scale, dtype, q_descale, k_descale, v_descale,
                  nullptr, stream, 0);
}

zyfa_status_t zyfa_attn_fwd_causal_ex(const void* q, const void* k, const void* v, void* out, int B, int S, int H,
                                      int H_kv, int D_qk, int D_v, float softmax_scale, zyfa_dtype_t dtype,
                                      const float* q_descale, const float* k_descale, const float* v_descale,
                                      const zyfa_fwd_options_t* options, cudaStream_t stream) {
  return attn_fwd(q, k, v, out, B, S, H, H_kv, D_qk, D_v, softmax_scale, dtype, q_descale, k_descale, v_descale,
                  options, stream, 0);
}

zyfa_status_t zyfa_attn_fwd_causal_host(const void* q_host, const void* k_host, const void* v_host, void* out_host,
                                        void* q_dev, void* k_dev, void* v_dev, void* out_dev, int B, int S, int H,
                                        int H_kv, int D_qk, int D_v, float softmax_scale, zyfa_dtype_t dtype,
                                        const float* q_descale, const float* k_descale, const float* v_descale,
                                        int chunks, cudaStream_t stream) {
  if (B < 1 || H < 1 || H_kv < 1 || S < 0 || H % H_kv != 0 || chunks < 0) return ZYFA_ERR_INVALID_ARG;
  if (dtype != ZYFA_DTYPE_E4M3 && dtype != ZYFA_DTYPE_BF16) return ZYFA_ERR_INVALID_ARG;
  const bool shape_ok = (D_qk == 64 && D_v == 64) || (D_qk == 128 && D_v == 128) || (D_qk == 192 && D_v == 128);
  if (!shape_ok) return ZYFA_ERR_UNSUPPORTED;
  if (S == 0) return ZYFA_OK;
  if (!q_host || !k_host || !v_host || !out_host) return ZYFA_ERR_INVALID_ARG;
  // the checks the kernel launches would make, before any copy is enqueued: an argument error
  // leaves every buffer and stream untouched
  if (!q_dev || !k_dev || !v_dev || !out_dev) return ZYFA_ERR_INVALID_ARG;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (misaligned(q_dev) || misaligned(k_dev) || misaligned(v_dev) || misaligned(out_dev)) return ZYFA_ERR_MISALIGNED;
  if (!std::isfinite(softmax_scale) || softmax_scale < 0.0f) return ZYFA_ERR_INVALID_ARG;
  const long long nqb = (static_cast<long long>(S) + kUnitRows - 1) / kUnitRows;
  if (nqb * B * H > (1ll << 30) || static_cast<long long>(S) > (1ll << 30)) return ZYFA_ERR_UNSUPPORTED;
  // chunk boundaries in query blocks: `chunks` equal chunks, or for chunks == 0 the library's plan.
  // Every row's output waits for its chunk's download, and the last chunk's download follows the last
  // kernel with nothing left to hide it behind; causal work grows with the row, so the plan ends with
  // two short chunks of nqb/16 query blocks each (short downloads, kernels still long enough to fill
  // the GPU) after four equal chunks.  Below 32 query blocks (8K rows) those tails would be a block
  // or two and the plan is four equal chunks.
  long long bound[kMaxHostChunks + 1];
  if (chunks == 0 && nqb >= 32) {
    const long long tail = (nqb + 8) / 16, body = nqb - 2 * tail;
    chunks = 6;
    for (int c = 0; c <= 4; ++c) bound[c] = body * c / 4;
    bound[5] = body + tail;
    bound[6] = nqb;
  } else {
    if (chunks == 0) chunks = 4;
    if (chunks > nqb) chunks = static_cast<int>(nqb);
    if (chunks > kMaxHostChunks) chunks = kMaxHostChunks;
    for (int c = 0; c <= chunks; ++c) bound[c] = nqb * c / chunks;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ZYFA_ERR_CUDA;
  cudaStream_t up = nullptr, down = nullptr;
  if (!copy_streams(dev, &up, &down)) return ZYFA_ERR_CUDA;

  const size_t es = dtype == ZYFA_DTYPE_E4M3 ? 1 : 2;
  const size_t row_q = static_cast<size_t>(H) * D_qk * es, row_k = static_cast<size_t>(H_kv) * D_qk * es;
  const size_t row_v = static_cast<size_t>(H_kv) * D_v * es, row_o = static_cast<size_t>(H) * D_v * 2;
  // rows [r0, r1) of every batch of a [B][S][row] tensor: one pitched copy of B pieces
  auto copy_rows = [&](void* dst, const void* src, size_t row, long long r0, long long r1, cudaMemcpyKind kind,
                       cudaStream_t st) {
    const size_t off = static_cast<size_t>(r0) * row, pitch = static_cast<size_t>(S) * row;
    return cudaMemcpy2DAsync(static_cast<char*>(dst) + off, pitch, static_cast<const char*>(src) + off, pitch,
                             static_cast<size_t>(r1 - r0) * row, static_cast<size_t>(B), kind, st) == cudaSuccess;
  };
  EventSet ev;
  if (!ev.create(2 * chunks + 2)) return ZYFA_ERR_CUDA;
  bool ok = cudaEventRecord(ev.e[0], stream) == cudaSuccess && cudaStreamWaitEvent(up, ev.e[0], 0) == cudaSuccess;
  zyfa_status_t st = ZYFA_OK;
  for (int c = 0; ok && c < chunks; ++c) {
    const long long qb0 = bound[c], qb1 = bound[c + 1];
    const long long r0 = qb0 * kUnitRows, r1 = std::min<long long>(qb1 * kUnitRows, S);
    ok = copy_rows(q_dev, q_host, row_q, r0, r1, cudaMemcpyHostToDevice, up) &&
         copy_rows(k_dev, k_host, row_k, r0, r1, cudaMemcpyHostToDevice, up) &&
         copy_rows(v_dev, v_host, row_v, r0, r1, cudaMemcpyHostToDevice, up) &&
         cudaEventRecord(ev.e[1 + 2 * c], up) == cudaSuccess &&
         cudaStreamWaitEvent(stream, ev.e[1 + 2 * c], 0) == cudaSuccess;
    if (!ok) break;
    // query blocks [qb0, qb1) read keys [0, r1): every one of them arrived with this or an earlier chunk
    st = attn_fwd(q_dev, k_dev, v_dev, out_dev, B, S, H, H_kv, D_qk, D_v, softmax_scale, dtype, q_descale, k_descale,
                  v_descale, nullptr, stream, 0, qb0, qb1);
    if (st != ZYFA_OK) break;
    ok = cudaEventRecord(ev.e[2 + 2 * c], stream) == cudaSuccess &&
         cudaStreamWaitEvent(down, ev.e[2 + 2 * c], 0) == cudaSuccess &&
         copy_rows(out_host, out_dev, row_o, r0, r1, cudaMemcpyDeviceToHost, down);
  }
  // the caller's stream resumes once the last output rows are back on the host
  const bool tail = cudaEventRecord(ev.e[2 * chunks + 1], down) == cudaSuccess &&
                    cudaStreamWaitEvent(stream, ev.e[2 * chunks + 1], 0) == cudaSuccess;
  if (st != ZYFA_OK) return st;
  return ok && tail ? ZYFA_OK : ZYFA_ERR_CUDA;
}

zyfa_status_t zyfa_selftest_stalled_pipeline(const void* q, const void* k, const void* v, void* out, int B, int S,
                                             int H, int H_kv, int D_qk, int D_v, zyfa_dtype_t dtype,
                                             cudaStream_t stream) {
  return attn_fwd(q, k, v, out, B, S, H, H_kv, D_qk, D_v, 0.0f, dtype, nullptr, nullptr, nullptr, nullptr, stream,
                  1);
}

zyfa_status_t zyfa_check_errors(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ZYFA_ERR_CUDA;
  int value = 0;
  if (cudaMemcpyFromSymbol(&value, g_zyfa_status, sizeof(int)) != cudaSuccess) return ZYFA_ERR_CUDA;
  if (value != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_zyfa_status, &zero, sizeof(int)) != cudaSuccess) return ZYFA_ERR_CUDA;
    return ZYFA_ERR_TIMEOUT;
  }
  return ZYFA_OK;
}

}  // extern "C"
