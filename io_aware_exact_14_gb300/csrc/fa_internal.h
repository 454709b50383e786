// Host-side interface between the C-ABI layer (fa_api.cu) and the kernel
// translation units.  Not part of the public header.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Problem shape shared by every launcher.  Tensors are [B, H, N, d]
// contiguous bf16; row statistics (LSE, D) are [B, H, N] contiguous fp32.
struct Shape {
  int B, H, N, d;
  float scale;   // softmax scale, > 0
  int causal;    // 0 or 1
};

// Forward: O and LSE from Q, K, V (TMA maps are 3-D {d, N, B*H}, box {64, 128, 1}).
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, float* lse, const Shape& s, cudaStream_t st);

// Backward, step 1: D_i = sum_c dO_ic O_ic (fp32).
cudaError_t launch_bwd_preprocess(const void* o, const void* dO, float* Dvec, const Shape& s,
                                  cudaStream_t st);

// Backward, step 2: dK, dV for each 128-key tile, looping over query tiles.
cudaError_t launch_bwd_dkdv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const float* lse, const float* Dvec, const Shape& s, cudaStream_t st);

// Backward, step 3: dQ for each 128-query tile, looping over key tiles.
cudaError_t launch_bwd_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq, const float* lse,
                          const float* Dvec, const Shape& s, cudaStream_t st);

// Fixed device scratch for callers that cannot allocate: room for the fp32
// row term of up to kNoAllocRows rows (B*H*N), in a file-scope device array of
// fa_bwd.cu.  Returns its device address for the current device, looking it up
// (cudaGetSymbolAddress) on the first call made with that device current.
constexpr size_t kNoAllocRows = size_t(1) << 21;  // 8 MiB of fp32
cudaError_t noalloc_scratch(float** out);

// Heads per scheduling band: the band's K and V (2 * N * d bf16 per head)
// stay within ~48 MB of L2, at most 16 heads.
inline int head_band(int N, int d) {
  const long long per_head = 4ll * N * d;
  long long b = (48ll << 20) / (per_head > 0 ? per_head : 1);
  return static_cast<int>(b < 1 ? 1 : (b > 16 ? 16 : b));
}

// Device status words (0 = no kernel gave up on a wait).  `reset` clears them.
// Synchronous: copies from the device.
cudaError_t fwd_status(uint32_t* out, bool reset);
cudaError_t bwd_status(uint32_t* out, bool reset);

}  // namespace fa
