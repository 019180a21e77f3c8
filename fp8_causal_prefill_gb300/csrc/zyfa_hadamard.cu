// Hadamard rotation of Q or K followed by per-tensor FP8 e4m3 quantisation: the pre-pass that
// roughly halves the error input quantisation adds to attention (spbcomputers.ru ZYFA article, FAQ
// "Что даёт поворот Адамара?"; captivela ZYFA article, "Angka Nyata").
//
// x [rows][D] bf16 -> y = x R with R block-diagonal, normalised Walsh-Hadamard blocks of n = 128
// (D = 128) or 64 (D = 64, 192); the usual FP8 scale pair scale = fl32(448 / max|y|),
// descale = fl32(max|y| / 448) (both 1 if the maximum is 0); codes =
// rne_e4m3_satfinite(fl32(y * scale)).  y is computed in fp32 by the radix-2 transform, stages
// h = 1, 2, 4, ... with the butterflies (a + b, a - b), then one multiply by fl32(1/sqrt(n)).
//
// The per-tensor maximum needs a pass over the whole tensor before any code can be written, so the
// work is two launches over the same rows: pass 1 rotates and writes one partial maximum per block of
// 128 rows into scratch memory, pass 2 reduces those partials to the descale, rotates again and
// writes the codes.  One launch of each pass can cover two tensors (Q and K, which share the head
// dimension): their 128-row blocks are numbered one after the other, each tensor keeps its own
// maximum, and the grid's single wave of resident CTAs is shared by both (separate launches left the
// smaller tensor's last wave partly empty).  The scratch is caller-provided workspace
// (zyfa_hadamard_quantize_e4m3, zyfa_hadamard_quantize_qk_e4m3) or a fixed array inside this
// library (zyfa_hadamard_quantize_e4m3_noalloc).
//
// HBM-bound: per element 2 bytes read twice and 1 byte written.  Each thread rotates whole Hadamard
// blocks of one row in registers (no cross-lane traffic); a CTA of 128 threads covers 128 rows.  A
// thread's next row is copied into shared memory (cp.async, a padded slot per thread) while it
// rotates the current one, which keeps the loads of the next rows in flight behind the arithmetic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "zyfa.h"

namespace {

constexpr int kRowsPerPartial = 128;  // rows per partial maximum = threads per CTA (one row each)
constexpr int kThreads = 128;
constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed fp32 pairs: each lane rounded as its scalar operation.
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// One N-wide Hadamard block held by one thread, transformed in place: stages h = 1, 2, 4, ...,
// butterflies (a + b, a - b), then one multiply by fl32(1/sqrt(N)).  From h = 2 on, the butterflies
// of neighbouring elements go through packed pairs.
template <int N>
__device__ __forceinline__ void fwht(float (&v)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float a = v[i], b = v[i + 1];
    v[i] = __fadd_rn(a, b);
    v[i + 1] = __fsub_rn(a, b);
  }
#pragma unroll
  for (int h = 2; h < N; h *= 2) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      if ((i & h) == 0) {
        const uint64_t a = pk(v[i], v[i + 1]), b = pk(v[i + h], v[i + h + 1]);
        upk(add2(a, b), v[i], v[i + 1]);
        upk(sub2(a, b), v[i + h], v[i + h + 1]);
      }
    }
  }
  const float c = N == 128 ? 0.088388347648318440550f : 0.125f;  // fl32(1/sqrt(N))
  const uint64_t c2 = pk(c, c);
#pragma unroll
  for (int i = 0; i < N; i += 2) upk(mul2(pk(v[i], v[i + 1]), c2), v[i], v[i + 1]);
}

// A thread's row slot in shared memory: the row's D bf16 values, padded by 16 bytes so that the
// slots of 8 consecutive threads fall on 8 different 16-byte bank groups.
template <int D>
struct Slots {
  static constexpr int kPitch = D * 2 + 16;
  static constexpr int kBytes = 2 * kThreads * kPitch;  // two rows per thread: current and next
};

// The tensors of one launch: blocks [0, np[0]) are tensor 0's, [np[0], np[0] + np[1]) tensor 1's
// (np[1] = 0 for a single tensor).  A block's partial maximum sits at its global block number.
struct Pair {
  const __nv_bfloat16* x[2];
  uint8_t* x8[2];
  float* descale[2];
  long long rows[2];
  long long np[2];
};

// Tensor and first row of global block pb (blocks past the end map to tensor 1 beyond its rows,
// which fetch_rows and the row checks skip).
__device__ __forceinline__ int block_tensor(const Pair& t, long long pb, long long& r0) {
  const int k = pb >= t.np[0] ? 1 : 0;
  r0 = (pb - (k ? t.np[0] : 0)) * 128;
  return k;
}

// Start copying the warp's 32 rows [r0, r0 + 32) (those below `rows`) into their threads' slots
// (slots are kPitch apart from `slots`): each copy instruction moves 32 consecutive 16-byte pieces,
// 512 contiguous bytes of the tensor.  One commit group per call, empty or not.
template <int D>
__device__ __forceinline__ void fetch_rows(const __nv_bfloat16* x, long long r0, long long rows, uint32_t slots) {
  constexpr int kPieces = D * 2 / 16;  // 16-byte pieces per row
  const int lane = threadIdx.x & 31;
  const char* base = reinterpret_cast<const char*>(x + r0 * D);
#pragma unroll
  for (int i = 0; i < kPieces; ++i) {
    const int q = i * 32 + lane;  // piece of the warp's rows
    const int row = q / kPieces, piece = q % kPieces;
    if (r0 + row < rows)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(slots + row * Slots<D>::kPitch + 16 * piece),
                   "l"(base + 16 * q)
                   : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// All but the most recent commit group of every lane have landed and are visible to the whole warp.
__device__ __forceinline__ void fetch_wait_prev() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
  __syncwarp();
}

// Block of N bf16 values from shared memory (16-byte loads) as fp32.
template <int N>
__device__ __forceinline__ void load_block(uint32_t src, float (&v)[N]) {
#pragma unroll
  for (int i = 0; i < N / 8; ++i) {
    uint4 w;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                 : "r"(src + 16 * i));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[8 * i + 2 * k] = __uint_as_float(u[k] << 16);
      v[8 * i + 2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ float block_max(float m, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red[] may still be read from a previous use
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, red[w]);
  return m;
}

// Pass 1: partial[p] = max |y| over the rows of global block p; thread t rotates the block's row t.
template <int D, int N>
__global__ void __launch_bounds__(kThreads) hadamard_amax_kernel(const __grid_constant__ Pair t,
                                                                 float* __restrict__ partial) {
  __shared__ float red[kThreads / 32];
  extern __shared__ __align__(16) uint8_t slots_raw[];
  const uint32_t slot0 = static_cast<uint32_t>(__cvta_generic_to_shared(slots_raw)) + threadIdx.x * Slots<D>::kPitch;
  const uint32_t warp_slots = slot0 - (threadIdx.x & 31) * Slots<D>::kPitch;
  const int wrow = threadIdx.x & ~31;                        // the warp's first row in a 128-row block
  constexpr uint32_t kOther = kThreads * Slots<D>::kPitch;  // offset of the second slot
  const long long nparts = t.np[0] + t.np[1];
  int cur = 0;
  long long r0;
  int k = block_tensor(t, blockIdx.x, r0);
  fetch_rows<D>(t.x[k], r0 + wrow, t.rows[k], warp_slots);
  for (long long pb = blockIdx.x; pb < nparts; pb += gridDim.x) {
    const int kc = block_tensor(t, pb, r0);
    const long long r = r0 + threadIdx.x;
    long long rn;
    const int kn = block_tensor(t, pb + gridDim.x, rn);
    fetch_rows<D>(t.x[kn], rn + wrow, t.rows[kn], warp_slots + (cur ^ 1) * kOther);
    fetch_wait_prev();
    const uint32_t slot = slot0 + cur * kOther;
    float m = 0.0f;
    if (r < t.rows[kc]) {
#pragma unroll 1
      for (int c = 0; c < D / N; ++c) {
        float v[N];
        load_block<N>(slot + c * N * 2, v);
        fwht<N>(v);
#pragma unroll
        for (int i = 0; i < N; ++i) m = fmaxf(m, fabsf(v[i]));
      }
    }
    m = block_max(m, red);
    if (threadIdx.x == 0) partial[pb] = m;
    cur ^= 1;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Pass 2: each tensor's descale from its partial maxima, then the codes of every row.
template <int D, int N>
__global__ void __launch_bounds__(kThreads) hadamard_quant_kernel(const __grid_constant__ Pair t,
                                                                  const float* __restrict__ partial) {
  __shared__ float red[kThreads / 32];
  float sc[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const long long p0 = k ? t.np[0] : 0;
    float m = 0.0f;
    for (long long i = threadIdx.x; i < t.np[k]; i += kThreads) m = fmaxf(m, partial[p0 + i]);
    const float amax = block_max(m, red);
    const float ds = amax > 0.0f ? __fdiv_rn(amax, kE4M3Max) : 1.0f;
    sc[k] = amax > 0.0f ? __fdiv_rn(kE4M3Max, amax) : 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0 && t.np[k] > 0) *t.descale[k] = ds;
  }
  extern __shared__ __align__(16) uint8_t slots_raw[];
  const uint32_t slot0 = static_cast<uint32_t>(__cvta_generic_to_shared(slots_raw)) + threadIdx.x * Slots<D>::kPitch;
  const uint32_t warp_slots = slot0 - (threadIdx.x & 31) * Slots<D>::kPitch;
  const int wrow = threadIdx.x & ~31;
  constexpr uint32_t kOther = kThreads * Slots<D>::kPitch;
  const long long nparts = t.np[0] + t.np[1];
  int cur = 0;
  long long r0;
  int k = block_tensor(t, blockIdx.x, r0);
  fetch_rows<D>(t.x[k], r0 + wrow, t.rows[k], warp_slots);
  for (long long pb = blockIdx.x; pb < nparts; pb += gridDim.x, cur ^= 1) {
    const int kc = block_tensor(t, pb, r0);
    const long long r = r0 + threadIdx.x;
    const long long rows = t.rows[kc];
    const float scale = kc ? sc[1] : sc[0];
    const uint64_t scale2 = pk(scale, scale);
    __syncwarp();  // every lane has read the slots the next copies overwrite
    long long rn;
    const int kn = block_tensor(t, pb + gridDim.x, rn);
    fetch_rows<D>(t.x[kn], rn + wrow, t.rows[kn], warp_slots + (cur ^ 1) * kOther);
    fetch_wait_prev();
    const uint32_t slot = slot0 + cur * kOther;
    if (r < rows) {
#pragma unroll 1
      for (int c = 0; c < D / N; ++c) {
        float v[N];
        load_block<N>(slot + c * N * 2, v);
        fwht<N>(v);
        // the codes of block c go to bytes [c N, (c + 1) N) of the slot, below the bf16 values of
        // the blocks still to be read
#pragma unroll
        for (int i = 0; i < N / 16; ++i) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float* e = v + 16 * i + 4 * q;
            float y0, y1, y2, y3;
            upk(mul2(pk(e[0], e[1]), scale2), y0, y1);
            upk(mul2(pk(e[2], e[3]), scale2), y2, y3);
            w[q] = cvt_e4m3x2(y1, y0) | (cvt_e4m3x2(y3, y2) << 16);
          }
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(slot + c * N + 16 * i), "r"(w[0]),
                       "r"(w[1]), "r"(w[2]), "r"(w[3])
                       : "memory");
        }
      }
    }
    __syncwarp();
    // the warp's 32 rows of codes are contiguous in global memory: 512 bytes per store instruction
    {
      constexpr int kPieces = D / 16;  // 16-byte pieces of codes per row
      const int lane = threadIdx.x & 31;
      const long long w0 = r0 + wrow;
      uint8_t* base = t.x8[kc] + w0 * D;
#pragma unroll
      for (int i = 0; i < kPieces; ++i) {
        const int q = i * 32 + lane;
        const int row = q / kPieces, piece = q % kPieces;
        if (w0 + row < rows) {
          uint4 w;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                       : "r"(warp_slots + cur * kOther + row * Slots<D>::kPitch + 16 * piece));
          reinterpret_cast<uint4*>(base)[q] = w;
        }
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_nsm[kMaxDevices];

// Scratch of the allocation-free entry point: the partial maxima (one float per 128 rows) live in
// this fixed array, which every GPU that loads the library holds until the process exits.  128 KiB
// covers 32768 partials, i.e. at most 4,194,304 rows per call.
constexpr long long kNoAllocMaxPartials = 32768;
constexpr long long kNoAllocMaxRows = kNoAllocMaxPartials * kRowsPerPartial;
static __device__ __align__(256) float g_noalloc_partials[kNoAllocMaxPartials];
// Device address of g_noalloc_partials per device, looked up once (in host code the array's name
// is only a host-side stand-in, not a device address).
std::atomic<float*> g_noalloc_ptr[kMaxDevices];

float* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  float* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_noalloc_partials) != cudaSuccess || !addr) return nullptr;
  g_noalloc_ptr[dev].store(static_cast<float*>(addr), std::memory_order_release);
  return static_cast<float*>(addr);
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = g_nsm[dev].load(std::memory_order_acquire);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
  g_nsm[dev].store(n, std::memory_order_release);
  return n;
}

long long num_partials(long long rows) { return (rows + kRowsPerPartial - 1) / kRowsPerPartial; }

template <int D, int N>
zyfa_status_t launch_both(const Pair& t, float* partial, cudaStream_t stream) {
  const long long np = t.np[0] + t.np[1];
  const int nsm = sm_count();
  if (nsm <= 0) return ZYFA_ERR_CUDA;
  constexpr int kSmem = Slots<D>::kBytes;
  auto k1 = hadamard_amax_kernel<D, N>;
  auto k2 = hadamard_quant_kernel<D, N>;
  if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess ||
      cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return ZYFA_ERR_CUDA;
  // one wave of resident CTAs; each walks its rows with the next row's copy in flight
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k2, kThreads, kSmem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const long long cap = static_cast<long long>(per_sm) * nsm;
  const int grid = static_cast<int>(np < cap ? np : cap);
  k1<<<grid, kThreads, kSmem, stream>>>(t, partial);
  if (cudaGetLastError() != cudaSuccess) return ZYFA_ERR_CUDA;
  k2<<<grid, kThreads, kSmem, stream>>>(t, partial);
  return cudaGetLastError() == cudaSuccess ? ZYFA_OK : ZYFA_ERR_CUDA;
}

// Argument checks shared by both entry points; ZYFA_OK means "launch".
zyfa_status_t check_args(const void* x, const void* x8, const float* descale, long long rows, int D) {
  if (rows < 0) return ZYFA_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 192) return ZYFA_ERR_UNSUPPORTED;
  if (rows > (1ll << 40) / D) return ZYFA_ERR_UNSUPPORTED;
  if (rows == 0) return ZYFA_OK;
  if (!x || !x8 || !descale) return ZYFA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x8) & 15u) ||
      (reinterpret_cast<uintptr_t>(descale) & 3u))
    return ZYFA_ERR_MISALIGNED;
  return ZYFA_OK;
}

zyfa_status_t dispatch(const Pair& t, int D, float* partial, cudaStream_t stream) {
  if (D == 128) return launch_both<128, 128>(t, partial, stream);
  if (D == 64) return launch_both<64, 64>(t, partial, stream);
  return launch_both<192, 64>(t, partial, stream);
}

Pair make_pair(const void* x, void* x8, float* descale, long long rows) {
  Pair t = {};
  t.x[0] = t.x[1] = static_cast<const __nv_bfloat16*>(x);
  t.x8[0] = t.x8[1] = static_cast<uint8_t*>(x8);
  t.descale[0] = t.descale[1] = descale;
  t.rows[0] = rows;
  t.np[0] = num_partials(rows);
  return t;
}

}  // namespace

extern "C" {

size_t zyfa_hadamard_workspace_bytes(long long rows) {
  return rows > 0 ? static_cast<size_t>(num_partials(rows)) * sizeof(float) : 0;
}

zyfa_status_t zyfa_hadamard_quantize_e4m3(const void* x, void* x8, float* descale, long long rows, int D,
                                          void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const zyfa_status_t st = check_args(x, x8, descale, rows, D);
  if (st != ZYFA_OK || rows == 0) return st;
  if (!workspace || workspace_bytes < zyfa_hadamard_workspace_bytes(rows)) return ZYFA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 3u) return ZYFA_ERR_MISALIGNED;
  return dispatch(make_pair(x, x8, descale, rows), D, static_cast<float*>(workspace), stream);
}

// Q and K in one launch per pass: the partial maxima of K follow those of Q in the workspace.
zyfa_status_t zyfa_hadamard_quantize_qk_e4m3(const void* q, void* q8, float* q_descale, long long q_rows,
                                             const void* k, void* k8, float* k_descale, long long k_rows, int D,
                                             void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  zyfa_status_t st = check_args(q, q8, q_descale, q_rows, D);
  if (st == ZYFA_OK) st = check_args(k, k8, k_descale, k_rows, D);
  if (st != ZYFA_OK) return st;
  if (q_rows == 0 && k_rows == 0) return ZYFA_OK;
  if (q_rows == 0) return zyfa_hadamard_quantize_e4m3(k, k8, k_descale, k_rows, D, workspace, workspace_bytes, stream);
  if (k_rows == 0) return zyfa_hadamard_quantize_e4m3(q, q8, q_descale, q_rows, D, workspace, workspace_bytes, stream);
  if (!workspace || workspace_bytes < zyfa_hadamard_workspace_bytes(q_rows) + zyfa_hadamard_workspace_bytes(k_rows))
    return ZYFA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 3u) return ZYFA_ERR_MISALIGNED;
  Pair t = make_pair(q, q8, q_descale, q_rows);
  t.x[1] = static_cast<const __nv_bfloat16*>(k);
  t.x8[1] = static_cast<uint8_t*>(k8);
  t.descale[1] = k_descale;
  t.rows[1] = k_rows;
  t.np[1] = num_partials(k_rows);
  return dispatch(t, D, static_cast<float*>(workspace), stream);
}

// The allocation-free variant: the same two kernels, with the partial maxima in the library's own
// fixed device array instead of caller workspace.  Every slot the second kernel reads is written by
// the first kernel of the same call, so nothing needs clearing between calls.
zyfa_status_t zyfa_hadamard_quantize_e4m3_noalloc(const void* x, void* x8, float* descale, long long rows, int D,
                                                  cudaStream_t stream) {
  const zyfa_status_t st = check_args(x, x8, descale, rows, D);
  if (st != ZYFA_OK || rows == 0) return st;
  if (rows > kNoAllocMaxRows) return ZYFA_ERR_UNSUPPORTED;
  float* scratch = noalloc_scratch();
  if (!scratch) return ZYFA_ERR_CUDA;
  return dispatch(make_pair(x, x8, descale, rows), D, scratch, stream);
}

}  // extern "C"
