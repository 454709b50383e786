// Backward pass of exact attention on sm_103a (recompute-based).
//
// The pages describe the backward only as recomputing S and P on chip from the
// saved inputs instead of storing P ("为什么Flash Attention能将注意力计算提速数倍
// 而不损失精度", section "反向传播中的重计算策略").  The gradients are the calculus
// of the forward definition:
//   dV = P^T dO, dP = dO V^T, D_i = sum_c dO_ic O_ic, dS = P o (dP - D),
//   dQ = scale dS K, dK = scale dS^T Q,
// with P recomputed as exp(scale q.k - LSE) from the forward's log-sum-exp.
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <cmath>

namespace fa {
namespace {

__device__ unsigned int g_status_bwd = 0;

// ---------------------------------------------------------------------------
// Step 1: D_i = sum_c dO_ic O_ic.  HBM-bound: 16-byte loads, d/8 threads per
// row reduce with shuffles, four rows in flight per thread.
// ---------------------------------------------------------------------------

constexpr int kPreThreads = 256;
constexpr int kPreUnroll = 4;

__device__ __forceinline__ float dot8_bf16(const uint4& a, const uint4& b) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fx = __bfloat1622float2(x[i]);
    const float2 fy = __bfloat1622float2(y[i]);
    s = fmaf(fx.x, fy.x, s);
    s = fmaf(fx.y, fy.y, s);
  }
  return s;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int D>
__global__ void __launch_bounds__(kPreThreads) fa_bwd_preprocess_kernel(const uint8_t* __restrict__ o,
                                                                       const uint8_t* __restrict__ dO,
                                                                       float* __restrict__ Dvec, long long rows) {
  constexpr int kTpr = D / 8;                 // threads per row, one 16-byte chunk each
  constexpr int kRows = kPreThreads / kTpr;   // rows per block per step
  const int sub = threadIdx.x % kTpr;
  const long long stride = static_cast<long long>(gridDim.x) * kRows * kPreUnroll;
  for (long long base = static_cast<long long>(blockIdx.x) * kRows * kPreUnroll + threadIdx.x / kTpr;
       base < rows; base += stride) {
    uint4 a[kPreUnroll], b[kPreUnroll];
#pragma unroll
    for (int u = 0; u < kPreUnroll; ++u) {
      const long long row = base + static_cast<long long>(u) * kRows;
      if (row < rows) {
        const size_t off = (static_cast<size_t>(row) * D + sub * 8) * 2;
        a[u] = ldg_stream(o + off);
        b[u] = ldg_stream(dO + off);
      }
    }
#pragma unroll
    for (int u = 0; u < kPreUnroll; ++u) {
      const long long row = base + static_cast<long long>(u) * kRows;
      float s = row < rows ? dot8_bf16(a[u], b[u]) : 0.f;
#pragma unroll
      for (int w = kTpr / 2; w > 0; w /= 2) s += __shfl_xor_sync(0xffffffffu, s, w);
      if (sub == 0 && row < rows) Dvec[row] = s;
    }
  }
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void* o, const void* dO, float* Dvec, const Shape& s, cudaStream_t st) {
  const long long rows = static_cast<long long>(s.B) * s.H * s.N;
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int rows_per_block = (kPreThreads / (s.d / 8)) * kPreUnroll;
  const long long want = (rows + rows_per_block - 1) / rows_per_block;
  const int grid = static_cast<int>(want < 8LL * sms ? want : 8LL * sms);
  if (s.d == 128)
    fa_bwd_preprocess_kernel<128><<<grid, kPreThreads, 0, st>>>(static_cast<const uint8_t*>(o),
                                                                 static_cast<const uint8_t*>(dO), Dvec, rows);
  else
    fa_bwd_preprocess_kernel<64><<<grid, kPreThreads, 0, st>>>(static_cast<const uint8_t*>(o),
                                                                static_cast<const uint8_t*>(dO), Dvec, rows);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                            const CUtensorMap&, const CUtensorMap&, const float*, const float*, const Shape&,
                            cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t launch_bwd_dq(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                          const CUtensorMap&, const float*, const float*, const Shape&, cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t bwd_status(uint32_t* out, bool reset) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_status_bwd, sizeof(v));
  if (e != cudaSuccess) return e;
  *out = v;
  if (reset && v != 0) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_status_bwd, &z, sizeof(z));
  }
  return e;
}

}  // namespace fa
