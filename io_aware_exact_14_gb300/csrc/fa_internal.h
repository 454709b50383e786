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

// Dropout on the probabilities: Philox4x32-10 with key (k0, k1) = the seed's
// low and high words (rk0[r] = k0 + r * 0x9E3779B9, rk1[r] = k1 + r *
// 0xBB67AE85: the key of round r), counter word 3 = offset.  t (0..255) is
// the keep threshold: t4 holds it in every byte, tlo4 its low 7 bits in every
// byte and maj is ~0 when t < 128, else 0 (the two cases of the byte compare).
// Kept probabilities are multiplied by scale = 256 / (256 - t).  t == 0 (t4 ==
// 0) means no dropout.
struct DropArgs {
  uint32_t rk0[10], rk1[10];
  uint32_t offset, t4, tlo4, maj;
  float scale;
};

inline DropArgs make_drop_args(uint64_t seed, uint32_t offset, int t) {
  DropArgs a{};
  const uint32_t k0 = static_cast<uint32_t>(seed & 0xffffffffull), k1 = static_cast<uint32_t>(seed >> 32);
  for (uint32_t r = 0; r < 10; ++r) {
    a.rk0[r] = k0 + r * 0x9E3779B9u;
    a.rk1[r] = k1 + r * 0xBB67AE85u;
  }
  a.offset = offset;
  a.t4 = 0x01010101u * static_cast<uint32_t>(t);
  a.tlo4 = 0x01010101u * static_cast<uint32_t>(t & 0x7f);
  a.maj = t < 128 ? 0xffffffffu : 0u;
  a.scale = static_cast<float>(256.0 / (256.0 - t));
  return a;
}
inline DropArgs no_drop_args() { return make_drop_args(0, 0, 0); }

// Bounded waits of one launch.  Every pipeline wait of a kernel gives up after
// limit_us microseconds: the CTA records a site in the kernel family's status
// word (first failure wins, kept until read with reset) and writes `epoch` to
// the family's abort word, which ends the waits of every other CTA of the same
// launch.  epoch is unique per launch (never 0), so a launch that gave up never
// cuts short a later one.  withhold >= 0 is a test hook of the forward: its
// producer issues no copy for K/V group `withhold` (nor any later one), so a
// consumer's wait on that group runs into the limit; < 0 in every normal call.
struct WaitCfg {
  uint32_t epoch;
  uint32_t limit_us;
  int32_t withhold;
};
constexpr uint32_t kDefaultWaitLimitUs = 4000000;   // 4 s
// The next launch's configuration: a fresh epoch, the default limit, no hook.
WaitCfg next_wait_cfg();

// Host-side launch preparation, done once instead of on every call (a call
// right after a synchronisation otherwise paid tens of microseconds of it):
//   prepare_kernel: the opt-in dynamic shared-memory size, and the check that
//     the launch's register allocation covers the warpgroups' setmaxnreg
//     split (regs_needed = 0: no split), once per kernel and CUDA context;
//     failures are not remembered;
//   sm_count: the current device's SM count, looked up once per device;
//   current_context_id: the current CUDA context's unique id (cuCtxGetCurrent
//     and cuCtxGetId, fetched through the runtime so nothing links libcuda),
//     0 when no context is current or the driver cannot say.
cudaError_t prepare_kernel(const void* kern, uint32_t smem_bytes, int threads, uint32_t regs_needed);
cudaError_t sm_count(int* out);
unsigned long long current_context_id();

// Head dims: any multiple of 8 from 8 to 256 runs in the kernel built for
// D = 64 (d <= 64), D = 128 (d <= 128) or D = 256.  The tensor maps carry the
// true extent d, so TMA loads fill columns d .. D-1 of every tile with zeros
// (they add nothing to Q K^T, and P V gives zeros there) and TMA stores clip
// them.
inline int kernel_dim(int d) { return d > 128 ? 256 : (d > 64 ? 128 : 64); }
constexpr int kMaxHeadDim = 256;
// Products that contract over the head dim (Q K^T, dO V^T and their
// transposes) issue only the ceil(d / 16) steps of 16 columns that hold data.
inline int score_ksteps(int d) { return (d + 15) / 16; }
// Products whose output columns are the head dim (P V, dV, dK, dQ) run with
// N = ceil(d / 16) * 16 (the tensor core's step for M = 128), not the
// kernel's D: the accumulator columns from N to D are never written and the
// stores clip them.
inline int out_cols(int d) { return (d + 15) / 16 * 16; }

// Element strides of a [B, H, N, d] bf16 view (d contiguous).
struct Strides {
  long long b, h, n;
};
inline Strides contiguous_strides(const Shape& s) {
  return Strides{static_cast<long long>(s.H) * s.N * s.d, static_cast<long long>(s.N) * s.d, s.d};
}

// Forward: O and LSE from Q, K, V (TMA maps are 4-D {d, N, H, B}, box
// {64, 128, 1, 1}, with each tensor's own strides).
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, float* lse, const Shape& s, const DropArgs& drop, const WaitCfg& wc,
                       cudaStream_t st);

// Forward for wide heads (128 < d <= 256): one query tile per CTA, K/V
// d-halves through a ring (fa_fwd_d256.cu).  Same maps as launch_fwd.
cudaError_t launch_fwd_d256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, float* lse, const Shape& s, const DropArgs& drop,
                            const WaitCfg& wc, cudaStream_t st);

// Forward for narrow heads (d <= 64, no dropout): four query tiles per CTA,
// 64-key steps (fa_fwd_q4.cu).  Q and O maps with 128-row boxes, K and V maps
// with 64-row boxes.
cudaError_t launch_fwd_q4(const CUtensorMap& tq, const CUtensorMap& tk64, const CUtensorMap& tv64,
                          const CUtensorMap& to, float* lse, const Shape& s, const WaitCfg& wc, cudaStream_t st);

// Split-KV forward for short query blocks against long key sequences
// (s.causal: the block is the last Nq positions of the keys' sequence): Q
// maps {d, Nq, H, B} (s.N = Nq; 32-row boxes with replicated rows), K/V maps
// {d, Nk, H, B}; each chunk of key tiles writes its normalised O (fp32, map
// `top` {D, Nq, R*n_splits*B*H}, 32-column boxes of 128 rows, or 32 with
// replicated rows) and its LSE (lse_part, fp32 [R*n_splits, B*H, Nq]; R =
// splitkv_replicas); the merge then writes o (bf16 [B, H, Nq, d]) and lse
// (fp32 [B, H, Nq]).  n_splits and kt_per_split come from splitkv_chunks.
cudaError_t launch_fwd_splitkv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& top, const float* o_part, float* lse_part, void* o, float* lse,
                               const Shape& s, int Nk, int n_splits, int kt_per_split, const WaitCfg& wc,
                               cudaStream_t st);

// Split-KV calls with at most kRepRows query rows whose key tiles carry 32 KB
// of K and V (e4m3 codes of d <= 128, or bf16 of d <= 64) replicate those rows over the four
// 32-row quarters of the query tile, each quarter taking a quarter of every
// key tile's keys: the per-tile softmax is what bounds those calls (measured:
// d = 64 decode 87% -> 97% of the copy rate, e4m3 d = 128 80% -> 87%); with
// 64 KB or more per key tile the stream already hides it.  Each chunk then
// writes splitkv_replicas(...) partial results: the Q map and the
// partial-output map have 32-row boxes, and the merge sees replicas *
// n_splits chunks.
constexpr int kRepRows = 32;
inline int splitkv_replicas(int Nq, int d, bool e4m3) {
  return Nq <= kRepRows && kernel_dim(d) <= (e4m3 ? 128 : 64) ? 4 : 1;
}

// The split-KV chunks (fa_fwd_d256.cu's one-query-tile kernel at the
// kernel head width D = kernel_dim(d)): the fp32 partial outputs through
// `top` (the 32-column boxes at or past d unwritten) and the partial LSE, as
// launch_fwd_splitkv describes; launch_fwd_splitkv calls it and then merges.
cudaError_t launch_fwd_onetile_split(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                     const CUtensorMap& top, float* lse_part, const Shape& s, int Nk, int n_splits,
                                     int kt_per_split, const WaitCfg& wc, cudaStream_t st);

// FP8 split-KV chunks: the one-query-tile kernel's e4m3 variant (kernel
// width 128 for d <= 128, else 256) on e4m3 Q, K (maps {d, Nq or Nk, H, B}, 128 x 128-byte
// boxes) and V^T (map {Nk, d, H, B}, row pitch fp8 ldv), descales per (b, h);
// partial outputs as launch_fwd_onetile_split at that width.
cudaError_t launch_fwd_fp8_split(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                                 const CUtensorMap& top, const float* dsq, const float* dsk, const float* dsv,
                                 float* lse_part, const Shape& s, int Nk, int n_splits, int kt_per_split,
                                 const WaitCfg& wc, cudaStream_t st);

// FP8 forward for 128 < d <= 256 (fa_fwd_d256.cu, the e4m3 variant at width
// 256): maps as launch_fwd_fp8_split's with 128-row Q boxes, bf16 O map as
// fa_fwd's; one query tile per CTA, causal or not.
cudaError_t launch_fwd_fp8_wide(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                                const CUtensorMap& to, const float* dsq, const float* dsk, const float* dsv,
                                float* lse, const Shape& s, const WaitCfg& wc, cudaStream_t st);

// The split-KV merge (fa_fwd.cu): n_splits chunks' fp32 partial outputs
// (rows D wide) and LSE -> o (bf16 [B, H, Nq, d]) and lse; n_splits == 0
// writes O = 0, LSE = -inf.
cudaError_t launch_fwd_merge(const float* o_part, const float* lse_part, void* o, float* lse, const Shape& s,
                             int n_splits, int D, cudaStream_t st);

// Split-KV chunking: `want` splits (<= 0: chosen from the SM count) of the
// ceil(Nk/128) key tiles into chunks of kt_per_split whole tiles; n_splits is
// the number of non-empty chunks (0 when Nk == 0).
inline void splitkv_chunks(int B, int H, int Nq, int Nk, int want, int sm_count, int& kt_per_split,
                           int& n_splits) {
  const int n_kt = (Nk + 127) / 128;
  if (n_kt <= 0) {
    kt_per_split = 0;
    n_splits = 0;
    return;
  }
  if (want <= 0) {
    // One CTA per SM at a time; the chunks stream K/V from HBM.  Cost model
    // (hundredths of the time one tile takes when every SM streams at once,
    // fitted to GB300 measurements of decode shapes): a full wave costs
    // per-chunk tiles x 100 plus a fixed 120 (load latency, epilogue, launch
    // gap); a partial wave of m CTAs streams at the shared rate 100 m / SMs
    // per tile but no faster than one CTA's own limit, 83.
    const long long units = static_cast<long long>(B) * H * ((Nq + 127) / 128);
    const long long sms = sm_count > 0 ? sm_count : 1;
    long long best = -1;
    want = 1;
    for (int s = 1; s <= n_kt && s <= 256; ++s) {
      const long long per = (n_kt + s - 1) / s;
      if (s > 1 && per == (n_kt + s - 2) / (s - 1)) continue;   // same chunks as s - 1
      const long long ctas = units * s, full = ctas / sms, m = ctas % sms;
      long long cost = full * (per * 100 + 120);
      if (m > 0) {
        const long long rate = 100 * m / sms > 83 ? 100 * m / sms : 83;
        cost += per * rate + 120;
      }
      if (best < 0 || cost < best) {
        best = cost;
        want = s;
      }
    }
  }
  const int w = want < n_kt ? want : n_kt;
  kt_per_split = (n_kt + w - 1) / w;
  n_splits = (n_kt + kt_per_split - 1) / kt_per_split;
}

// Backward, step 1: D_i = sum_c dO_ic O_ic (fp32).
cudaError_t launch_bwd_preprocess(const void* o, const Strides& so, const void* dO, const Strides& sdo, float* Dvec,
                                  const Shape& s, cudaStream_t st);

// Backward, step 2: dK, dV for each 128-key tile, looping over query tiles.
cudaError_t launch_bwd_dkdv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const float* lse, const float* Dvec, const Shape& s, const DropArgs& drop,
                            const WaitCfg& wc, cudaStream_t st);

// Backward, step 3: dQ for each 128-query tile, looping over key tiles.
cudaError_t launch_bwd_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq, const float* lse,
                          const float* Dvec, const Shape& s, const DropArgs& drop, const WaitCfg& wc,
                          cudaStream_t st);

// Backward for wide heads (128 < d <= 256, fa_bwd_d256.cu): three launches
// (dV, dK, dQ), each with resident 128-row tiles and streamed 64-row tiles,
// so every tensor is mapped with 128-row boxes and, where it streams, 64-row
// boxes.  wide_dkdv runs the dV and dK launches, wide_dq the dQ launch.
struct WideBwdMaps {
  CUtensorMap q128, q64, k128, k64, v128, v64, do128, do64, dq128, dk128, dv128;
};
cudaError_t launch_bwd_d256_dkdv(const WideBwdMaps& m, const float* lse, const float* Dvec, const Shape& s,
                                 const DropArgs& drop, cudaStream_t st);
cudaError_t launch_bwd_d256_dq(const WideBwdMaps& m, const float* lse, const float* Dvec, const Shape& s,
                               const DropArgs& drop, cudaStream_t st);

// FP8 (e4m3): per-(b, h) quantisation of a contiguous bf16 [B, H, N, d] tensor
// into codes [B, H, N, d] (or, transposed, [B, H, d, ldv]) with descale[b*H + h]
// = amax / 448, optionally rotated along d by the random-sign Hadamard
// transform of `seed` (d = 64 or 128); and the forward on such codes (Q, K
// [B, H, N, d], V transposed [B, H, d, ldv]; maps of 1-byte elements with
// 128 x 128 boxes), writing bf16 O and fp32 LSE.
cudaError_t launch_fp8_quantize(const void* x, void* out, float* descale, const Shape& s, bool transpose,
                                long long ldv, bool rotate, uint64_t seed, cudaStream_t st);
cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const CUtensorMap& to, const float* dq, const float* dk, const float* dv, float* lse,
                           const Shape& s, const WaitCfg& wc, cudaStream_t st);

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

// Device status words (0 = no kernel gave up on a wait).  `reset` clears them
// (and the abort words).
// Synchronous: copies from the device.
cudaError_t fwd_status(uint32_t* out, bool reset);
cudaError_t bwd_status(uint32_t* out, bool reset);
cudaError_t fp8_status(uint32_t* out, bool reset);
cudaError_t fwd_d256_status(uint32_t* out, bool reset);
cudaError_t bwd_d256_status(uint32_t* out, bool reset);
cudaError_t fwd_q4_status(uint32_t* out, bool reset);

}  // namespace fa
