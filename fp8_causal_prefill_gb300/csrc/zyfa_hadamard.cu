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
// writes the codes.  The scratch is caller-provided workspace (zyfa_hadamard_quantize_e4m3) or a
// fixed array inside this library (zyfa_hadamard_quantize_e4m3_noalloc).
//
// HBM-bound: per element 2 bytes read twice and 1 byte written.  Each thread rotates whole Hadamard
// blocks of one row in registers (no cross-lane traffic); a CTA of 128 threads covers 128 rows.
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

// One N-wide Hadamard block held by one thread, transformed in place: stages h = 1, 2, 4, ...,
// butterflies (a + b, a - b), then one multiply by fl32(1/sqrt(N)).
template <int N>
__device__ __forceinline__ void fwht(float (&v)[N]) {
#pragma unroll
  for (int h = 1; h < N; h *= 2) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
  const float c = N == 128 ? 0.088388347648318440550f : 0.125f;  // fl32(1/sqrt(N))
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = __fmul_rn(v[i], c);
}

// Block c of row r (N bf16 values, 16-byte loads) as fp32.
template <int N>
__device__ __forceinline__ void load_block(const __nv_bfloat16* src, float (&v)[N]) {
#pragma unroll
  for (int i = 0; i < N / 8; ++i) {
    const uint4 w = reinterpret_cast<const uint4*>(src)[i];
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

// Pass 1: partial[p] = max |y| over rows [128p, 128p + 128); thread t rotates row 128p + t.
template <int D, int N>
__global__ void __launch_bounds__(kThreads) hadamard_amax_kernel(const __nv_bfloat16* __restrict__ x,
                                                                 long long rows, float* __restrict__ partial,
                                                                 long long nparts) {
  __shared__ float red[kThreads / 32];
  for (long long pb = blockIdx.x; pb < nparts; pb += gridDim.x) {
    const long long r = pb * kRowsPerPartial + threadIdx.x;
    float m = 0.0f;
    if (r < rows) {
#pragma unroll 1
      for (int c = 0; c < D / N; ++c) {
        float v[N];
        load_block<N>(x + r * D + c * N, v);
        fwht<N>(v);
#pragma unroll
        for (int i = 0; i < N; ++i) m = fmaxf(m, fabsf(v[i]));
      }
    }
    m = block_max(m, red);
    if (threadIdx.x == 0) partial[pb] = m;
  }
}

// Pass 2: descale from the partial maxima, then the codes of every row.
template <int D, int N>
__global__ void __launch_bounds__(kThreads) hadamard_quant_kernel(const __nv_bfloat16* __restrict__ x,
                                                                  long long rows, const float* __restrict__ partial,
                                                                  long long nparts, uint8_t* __restrict__ x8,
                                                                  float* __restrict__ descale_out) {
  __shared__ float red[kThreads / 32];
  float m = 0.0f;
  for (long long i = threadIdx.x; i < nparts; i += kThreads) m = fmaxf(m, partial[i]);
  const float amax = block_max(m, red);
  const float ds = amax > 0.0f ? __fdiv_rn(amax, kE4M3Max) : 1.0f;
  const float sc = amax > 0.0f ? __fdiv_rn(kE4M3Max, amax) : 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0) *descale_out = ds;
  for (long long pb = blockIdx.x; pb < nparts; pb += gridDim.x) {
    const long long r = pb * kRowsPerPartial + threadIdx.x;
    if (r >= rows) continue;
#pragma unroll 1
    for (int c = 0; c < D / N; ++c) {
      float v[N];
      load_block<N>(x + r * D + c * N, v);
      fwht<N>(v);
      uint4* dst = reinterpret_cast<uint4*>(x8 + r * D + c * N);
#pragma unroll
      for (int i = 0; i < N / 16; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float* e = v + 16 * i + 4 * k;
          w[k] = cvt_e4m3x2(__fmul_rn(e[1], sc), __fmul_rn(e[0], sc)) |
                 (cvt_e4m3x2(__fmul_rn(e[3], sc), __fmul_rn(e[2], sc)) << 16);
        }
        dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
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
zyfa_status_t launch_both(const void* x, void* x8, float* descale, long long rows, float* partial,
                          cudaStream_t stream) {
  const long long np = num_partials(rows);
  const int nsm = sm_count();
  if (nsm <= 0) return ZYFA_ERR_CUDA;
  const long long cap = 16ll * nsm;
  const int grid = static_cast<int>(np < cap ? np : cap);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  hadamard_amax_kernel<D, N><<<grid, kThreads, 0, stream>>>(xb, rows, partial, np);
  if (cudaGetLastError() != cudaSuccess) return ZYFA_ERR_CUDA;
  hadamard_quant_kernel<D, N><<<grid, kThreads, 0, stream>>>(xb, rows, partial, np, static_cast<uint8_t*>(x8),
                                                             descale);
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

zyfa_status_t dispatch(const void* x, void* x8, float* descale, long long rows, int D, float* partial,
                       cudaStream_t stream) {
  if (D == 128) return launch_both<128, 128>(x, x8, descale, rows, partial, stream);
  if (D == 64) return launch_both<64, 64>(x, x8, descale, rows, partial, stream);
  return launch_both<192, 64>(x, x8, descale, rows, partial, stream);
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
  return dispatch(x, x8, descale, rows, D, static_cast<float*>(workspace), stream);
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
  return dispatch(x, x8, descale, rows, D, scratch, stream);
}

}  // extern "C"
