// Backward pass for wide heads (128 < d <= 256, kernels built for D = 256) on
// sm_103a.  The same recompute-based method as fa_bwd.cu ("为什么Flash Attention
// 能将注意力计算提速数倍而不损失精度", section "反向传播中的重计算策略"): P is
// recomputed on chip from the forward's log-sum-exp, and
//   dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q,
// with D_i = sum_c dO_ic O_ic from the preprocess kernel.
//
// Why kernels of their own: at D = 256 an accumulator takes 256 of the 512
// TMEM columns, so dK and dV no longer fit one CTA's tensor memory together,
// and a 128-row tile of Q, K, V or dO is 64 KB, so two resident tiles leave
// room for only 96 KB of streamed ones.  One kernel template, three modes:
//   DQ: unit = 128-query tile i (Q_i, dO_i resident); key tiles of 64 rows
//       stream: S = Q_i K_j^T, dP = dO_i V_j^T, dS = P o (dP - D_row),
//       dQ_i += dS K_j;
//   DK: unit = 128-key tile j (K_j, V_j resident); query tiles of 64 rows
//       stream: S^T = K_j Q_i^T, dP^T = V_j dO_i^T, dS^T = P^T o (dP^T - D_col),
//       dK_j += dS^T Q_i;
//   DV: unit = 128-key tile j (K_j resident): S^T, P^T, dV_j += P^T dO_i.
// (DK and DV recompute S^T each; that is the price of the TMEM budget.)
//
// GB300 design (one CTA per SM, 192 threads):
//   warps 0-3  compute (thread = resident row = TMEM lane)
//   warp  4    producer (lane 0 issues the TMA copies; in DK / DV the whole
//              warp writes the streamed tiles' row vectors -lse*log2(e), -D)
//   warp  5    TMEM owner and tcgen05.mma issuer (elect.sync in a converged warp)
// TMEM: S buffers [0,64) and [64,128) (step j uses buffer j & 1, so S(j+1)
// runs while the compute warps work on step j), dP [128,192), accumulator
// [256,512).  The bf16 operand of the accumulating product (dS, dS^T or P^T)
// overwrites the first 32 columns of the tile it was computed from and is
// read from TMEM.
// MMA order (DQ, DK): S(0) dP(0) S(1) | acc(0) dP(1) S(2) | acc(1) dP(2) S(3) ...
// (DV: S(0) S(1) | acc(0) S(2) | acc(1) S(3) ...).
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <cmath>

namespace fa {
namespace {

__device__ unsigned int g_status_bwd256[2] = {0, 0};   // status, abort epoch (see CtaGuard)

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kSiteBwd256 = 0x500;
enum { kModeDQ = 0, kModeDK = 1, kModeDV = 2 };

template <int MODE>
struct B256 {
  static constexpr bool kHasDP = MODE != kModeDV;        // dP product and a second resident tile
  static constexpr bool kColVecs = MODE != kModeDQ;      // row vectors travel with the streamed tiles
  static constexpr uint32_t kResBox = 128u * 128u;       // 128 rows x 128 B
  static constexpr uint32_t kResTile = 4 * kResBox;      // 128 x 256 bf16
  static constexpr uint32_t kStrBox = 64u * 128u;        // 64 rows x 128 B
  static constexpr uint32_t kStrTile = 4 * kStrBox;      // 64 x 256 bf16
  static constexpr int kT1Slots = 2;
  static constexpr int kT2Slots = kHasDP ? 1 : 2;
  // Full and empty barriers, and row-vector slots, go by step parity (two of
  // each per stream) whatever the number of tile slots: a barrier then never
  // runs two phases ahead of a waiter, and a step's vectors are rewritten only
  // two steps later, after the compute warps have passed that step.
  static constexpr uint32_t kR1Off = 0;
  static constexpr uint32_t kR2Off = kResTile;
  static constexpr uint32_t kT1Off = (kHasDP ? 2 : 1) * kResTile;
  static constexpr uint32_t kT2Off = kT1Off + kT1Slots * kStrTile;
  static constexpr uint32_t kVecOff = kT2Off + kT2Slots * kStrTile;     // 64 fp32 per streamed slot
  static constexpr uint32_t kBarOff = kVecOff + 4 * 256;
  // r_full, t1_full[2], t1_empty[2], t2_full[2], t2_empty[2], s_full[2],
  // dp_full, ds_full[2], acc_done, staged, drain, a_ready
  static constexpr int kBars = 1 + 8 + 9;
  static constexpr uint32_t kMiscOff = kBarOff + kBars * 8;   // tmem holder, abort flag
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared-memory budget");
  static constexpr int kThreads = 192;
  static constexpr uint32_t kColDP = 128, kColAcc = 256;
  // DV (no dP product): the resident tile (K_j) is copied into the dP
  // columns and its score products take A from TMEM (TS form): a 64-row
  // streamed B operand from shared memory alone keeps the tensor core at
  // full rate, where an N = 64 product with both operands in shared memory
  // runs at 2/3 of it (the operand reads hit the 128 bytes per clock limit).
  static constexpr bool kTmemA = MODE == kModeDV;
  __host__ __device__ static constexpr uint32_t t1_off(int s) { return kT1Off + s * kStrTile; }
  __host__ __device__ static constexpr uint32_t t2_off(int s) { return kT2Off + s * kStrTile; }
  __host__ __device__ static constexpr uint32_t t1_vec(int j) { return kVecOff + (j & 1) * 256; }
  __host__ __device__ static constexpr uint32_t t2_vec(int j) { return kVecOff + (2 + (j & 1)) * 256; }
};

// A CTA's unit: head bh, resident tile u (128 rows), streamed tiles
// first .. first + n - 1 (64 rows each).
struct U256 {
  int bh, u, first, n;
  HeadCoord hc;
};

template <int MODE, bool CAUSAL>
__device__ __forceinline__ U256 unit256(int N, int n_res, int BH, int H, int band) {
  U256 w;
  int rank;
  banded_order(blockIdx.x, n_res, BH, band, w.bh, rank);
  w.hc = head_coord(w.bh, H);
  const int n_str = (N + 63) / 64;
  if (MODE == kModeDQ) {
    w.u = CAUSAL ? n_res - 1 - rank : rank;           // causal: long query rows first
    w.first = 0;
    w.n = CAUSAL ? min(2 * w.u + 2, n_str) : n_str;   // key tiles starting at or before the last row
  } else {
    w.u = rank;                                       // causal: key tile 0 (most queries) first
    w.first = CAUSAL ? 2 * w.u : 0;                   // query tiles ending at or after the first key
    w.n = n_str - w.first;
  }
  return w;
}

template <int MODE>
__device__ void b256_producer(const U256& w, uint8_t* smem, uint64_t* r_full, uint64_t* t1_full, uint64_t* t1_empty,
                              uint64_t* t2_full, uint64_t* t2_empty, const CUtensorMap* tmR1,
                              const CUtensorMap* tmR2, const CUtensorMap* tmT1, const CUtensorMap* tmT2,
                              const float* __restrict__ lse, const float* __restrict__ Dg, int N,
                              const CtaGuard& g) {
  using C = B256<MODE>;
  const int lane = threadIdx.x & 31;
  const size_t row_base = static_cast<size_t>(w.bh) * N;
  if (lane == 0) {
    mbar_arrive_expect_tx(r_full, (C::kHasDP ? 2u : 1u) * C::kResTile);
    for (int b = 0; b < 4; ++b) {
      tma_load_hd(smem + C::kR1Off + b * C::kResBox, tmR1, r_full, 64 * b, 128 * w.u, w.hc);
      if (C::kHasDP) tma_load_hd(smem + C::kR2Off + b * C::kResBox, tmR2, r_full, 64 * b, 128 * w.u, w.hc);
    }
  }
  int issued1 = 0, issued2 = 0;
  bool ok = true;
  for (int j = 0; j < w.n && ok; ++j) {
    const int row0 = 64 * (w.first + j);
    for (int which = 0; which < 2; ++which) {
      const int slots = which ? C::kT2Slots : C::kT1Slots;
      const int s = j % slots;
      uint64_t* full = which ? &t2_full[j & 1] : &t1_full[j & 1];
      if (j >= slots) {   // the slot's previous step (j - slots) has released it
        const int pj = j - slots;
        uint64_t* empty = which ? &t2_empty[pj & 1] : &t1_empty[pj & 1];
        if (!(ok = mbar_wait_w(empty, (pj >> 1) & 1, g, kSiteBwd256 | 1u))) break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(full, C::kStrTile);
        uint8_t* dst = smem + (which ? C::t2_off(s) : C::t1_off(s));
        for (int b = 0; b < 4; ++b)
          tma_load_hd(dst + b * C::kStrBox, which ? tmT2 : tmT1, full, 64 * b, row0, w.hc);
      }
      if (C::kColVecs && (which == 0 || MODE == kModeDK)) {
        // -lse * log2(e) with Q_i (-inf past N: P = 0 there), -D with dO_i (0 past N)
        float* vec = reinterpret_cast<float*>(smem + (which ? C::t2_vec(j) : C::t1_vec(j)));
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int q = row0 + lane + 32 * k;
          float x = which ? 0.f : -INFINITY;
          if (q < N) {
            const float v = which ? Dg[row_base + q] : lse[row_base + q];
            x = which ? -v : ((v == -INFINITY) ? -INFINITY : -v * kLog2e);
          }
          vec[lane + 32 * k] = x;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(full);
      }
      if (which) issued2 = j + 1;
      else issued1 = j + 1;
    }
  }
  if (!ok && lane == 0) {   // unwinding: let the copies in flight land before shared memory is released
    mbar_drain(r_full, 0);
    for (int j = max(0, issued1 - C::kT1Slots); j < issued1; ++j) mbar_drain(&t1_full[j & 1], (j >> 1) & 1);
    for (int j = max(0, issued2 - C::kT2Slots); j < issued2; ++j) mbar_drain(&t2_full[j & 1], (j >> 1) & 1);
  }
}

// Score product D(128 x 64) = A(128 x d) B(64 x d)^T: A a resident tile
// (boxes 16 KB apart), B a streamed one (boxes 8 KB apart), both K-major;
// ks = ceil(d / 16) steps of 16 columns.
template <int MODE, bool FD>
__device__ __forceinline__ void b256_score(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc, int ks) {
  using C = B256<MODE>;
  constexpr uint32_t idesc = idesc_bf16(128, 64, false, false);
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) {
    const uint64_t oa = ((kk / 4) * C::kResBox + (kk % 4) * 32) >> 4;
    const uint64_t ob = ((kk / 4) * C::kStrBox + (kk % 4) * 32) >> 4;
    if constexpr (FD)
      tc_mma_ss_w(tmem_d, a_desc + oa, b_desc + ob, idesc, kk > 0 ? 1u : 0u);
    else
      tc_mma_ss_w_if(tmem_d, a_desc + oa, b_desc + ob, idesc, kk > 0 ? 1u : 0u, kk < ks ? 1u : 0u);
  }
}

// The same with A (128 x d, bf16) in TMEM: K step kk at column a_tmem + 8 kk.
template <int MODE, bool FD>
__device__ __forceinline__ void b256_score_ts(uint32_t tmem_d, uint32_t a_tmem, uint64_t b_desc, int ks) {
  using C = B256<MODE>;
  constexpr uint32_t idesc = idesc_bf16(128, 64, false, false);
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) {
    const uint64_t ob = ((kk / 4) * C::kStrBox + (kk % 4) * 32) >> 4;
    if constexpr (FD)
      tc_mma_ts_w(tmem_d, a_tmem + kk * 8, b_desc + ob, idesc, kk > 0 ? 1u : 0u);
    else
      tc_mma_ts_w_if(tmem_d, a_tmem + kk * 8, b_desc + ob, idesc, kk > 0 ? 1u : 0u, kk < ks ? 1u : 0u);
  }
}

// Accumulating product acc(128 x d) += A(128 x 64, bf16 in TMEM) * B(64 x d),
// B a streamed tile read MN-major (64-column blocks 8 KB apart); idesc has
// N = ceil(d / 16) * 16.
template <int MODE, bool FD>
__device__ __forceinline__ void b256_acc(uint32_t tmem_acc, uint32_t a_tmem, uint64_t b_desc, bool acc,
                                         uint32_t idesc_rt) {
  const uint32_t idesc = FD ? idesc_bf16(128, 256, false, true) : idesc_rt;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)   // 64 rows, 16 per MMA; A packs 2 per TMEM column
    tc_mma_ts_w(tmem_acc, a_tmem + kk * 8, b_desc + ((kk * 2048) >> 4), idesc, (acc || kk > 0) ? 1u : 0u);
}

template <int MODE, bool FD>
__device__ void b256_mma(const U256& w, uint32_t tmem, uint32_t sbase, uint64_t* r_full, uint64_t* t1_full,
                         uint64_t* t1_empty, uint64_t* t2_full, uint64_t* t2_empty, uint64_t* s_full,
                         uint64_t* dp_full, uint64_t* ds_full, uint64_t* acc_done, uint64_t* a_ready, int ks,
                         uint32_t idesc_acc, const CtaGuard& g) {
  using C = B256<MODE>;
  const uint64_t r1 = sdesc_sw128(sbase + C::kR1Off, 16, 1024);
  const uint64_t r2 = sdesc_sw128(sbase + C::kR2Off, 16, 1024);
  auto t1k = [&](int s) { return sdesc_sw128(sbase + C::t1_off(s), 16, 1024); };
  auto t2k = [&](int s) { return sdesc_sw128(sbase + C::t2_off(s), 16, 1024); };
  auto t1m = [&](int s) { return sdesc_sw128(sbase + C::t1_off(s), C::kStrBox, 1024); };
  auto t2m = [&](int s) { return sdesc_sw128(sbase + C::t2_off(s), C::kStrBox, 1024); };
  auto w1 = [&](int j) { return mbar_wait_w(&t1_full[j & 1], (j >> 1) & 1, g, kSiteBwd256 | 2u); };
  auto w2 = [&](int j) { return mbar_wait_w(&t2_full[j & 1], (j >> 1) & 1, g, kSiteBwd256 | 3u); };
  auto issue_s = [&](int j) -> bool {   // S(j) into buffer j & 1
    if (!w1(j)) return false;
    if constexpr (C::kTmemA)
      b256_score_ts<MODE, FD>(tmem + 64u * (j & 1), tmem + C::kColDP, t1k(j % C::kT1Slots), ks);
    else
      b256_score<MODE, FD>(tmem + 64u * (j & 1), r1, t1k(j % C::kT1Slots), ks);
    tc_commit_w(&s_full[j & 1]);
    return true;
  };
  auto issue_dp = [&](int j) -> bool {   // dP(j)
    if (!w2(j)) return false;
    b256_score<MODE, FD>(tmem + C::kColDP, r2, t2k(j % C::kT2Slots), ks);
    tc_commit_w(dp_full);
    tc_commit_w(&t2_empty[j & 1]);   // V_j / dO_i: its only reader (its -D is read before dP(j + 1))
    return true;
  };
  if (!mbar_wait_w(r_full, 0, g, kSiteBwd256 | 4u)) return;
  if (C::kTmemA) {   // the resident tile is in TMEM (copied by the compute warps)
    if (!mbar_wait_w(a_ready, 0, g, kSiteBwd256 | 12u)) return;
    tc_fence_after();
  }
  if (!issue_s(0)) return;
  if (C::kHasDP && !issue_dp(0)) return;
  if (w.n > 1 && !issue_s(1)) return;
  for (int j = 0; j < w.n; ++j) {
    if (!C::kHasDP && !w2(j)) return;   // DV: dO_i
    // ds_full by step parity: without a dP product (DV) the compute warps can
    // finish step j + 1 before this wait, but not step j + 2 (S(j + 2) goes
    // out below)
    if (!mbar_wait_w(&ds_full[j & 1], (j >> 1) & 1, g, kSiteBwd256 | 5u)) return;
    tc_fence_after();
    if (C::kHasDP) {
      b256_acc<MODE, FD>(tmem + C::kColAcc, tmem + C::kColDP, t1m(j % C::kT1Slots), j > 0, idesc_acc);   // += dS K_j / dS^T Q_i
      tc_commit_w(&t1_empty[j & 1]);   // last reader of the tile; its -lse was read before ds_full
      if (j + 1 < w.n && !issue_dp(j + 1)) return;   // after acc(j) has read dS(j) from the dP columns
    } else {
      b256_acc<MODE, FD>(tmem + C::kColAcc, tmem + 64u * (j & 1), t2m(j % C::kT2Slots), j > 0, idesc_acc);   // += P^T dO_i
      tc_commit_w(&t2_empty[j & 1]);
      tc_commit_w(&t1_empty[j & 1]);   // Q_i was read by S(j), its -lse before ds_full
    }
    if (j + 2 < w.n && !issue_s(j + 2)) return;      // buffer j & 1: step j's scores have been read
  }
  tc_commit_w(acc_done);
}

// DROPOUT: the keep mask of the forward, redrawn on chip: dV takes (P o M)^T
// (x 1/(1-p) in the epilogue), dS = P o (M~ o dP - D) with M~ = M / (1-p).
template <int MODE, bool CAUSAL, bool DROPOUT>
__device__ void b256_compute(const U256& w, uint32_t tmem, uint8_t* smem, uint64_t* r_full, uint64_t* t1_full,
                             uint64_t* t2_full, uint64_t* s_full, uint64_t* dp_full, uint64_t* ds_full,
                             uint64_t* acc_done, uint64_t* a_ready, uint64_t* staged, const CUtensorMap* tmOut,
                             const float* __restrict__ lse, const float* __restrict__ Dg, int N, int d, float scale,
                             float scale_log2, const DropArgs& drop, const CtaGuard& g) {
  using C = B256<MODE>;
  const int r = threadIdx.x & 127;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) * 32u << 16;
  const uint32_t sbase = smem_u32(smem);
  if constexpr (C::kTmemA) {
    // row r of the resident tile (swizzled boxes of 64 columns) into TMEM lane
    // r: box b's 128 bytes fill columns kColDP + 32b .. + 32 (two bf16 each)
    if (!mbar_wait(r_full, 0, g, kSiteBwd256 | 13u)) return;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint32_t v[32];
      const uint32_t row = sbase + C::kR1Off + b * C::kResBox + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 x = ld_shared_f4(row + ((c ^ (r & 7)) << 4));
        v[4 * c] = __float_as_uint(x.x);
        v[4 * c + 1] = __float_as_uint(x.y);
        v[4 * c + 2] = __float_as_uint(x.z);
        v[4 * c + 3] = __float_as_uint(x.w);
      }
      tmem_st32(tmem + lane_base + C::kColDP + 32 * b, v);
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(a_ready);
  }
  const int res_row = 128 * w.u + r;   // DQ: query row; DK, DV: key row
  // DQ: this row's terms (-inf / 0 past N, so P = dS = 0 there)
  float nl = -INFINITY, nd = 0.f;
  if (MODE == kModeDQ && res_row < N) {
    const float l = lse[static_cast<size_t>(w.bh) * N + res_row];
    nl = (l == -INFINITY) ? -INFINITY : -l * kLog2e;
    nd = -Dg[static_cast<size_t>(w.bh) * N + res_row];
  }
  const float2 sc2 = make_float2(scale_log2, scale_log2);
  for (int j = 0; j < w.n; ++j) {
    const int col0 = 64 * (w.first + j);   // first streamed row of this step
    const uint32_t tS = tmem + lane_base + 64u * (j & 1);
    // keep words of this row against the step's 64 streamed rows, drawn before
    // the scores land: column c in byte c % 4 of ge[c / 4]
    uint32_t ge[DROPOUT ? 16 : 1];
    if constexpr (DROPOUT) {
      if constexpr (MODE == kModeDQ)
        dropout_rows<4>(drop, w.bh, res_row, col0, ge);   // query row against keys
      else
        dropout_cols<4>(drop, w.bh, res_row, col0, ge);   // key row against queries
    }
    if (C::kColVecs && !mbar_wait(&t1_full[j & 1], (j >> 1) & 1, g, kSiteBwd256 | 6u)) return;
    if (!mbar_wait(&s_full[j & 1], (j >> 1) & 1, g, kSiteBwd256 | 7u)) return;
    __syncwarp();
    tc_fence_after();
    uint32_t sr[2][32];
    tmem_ld32(tS, sr[0]);
    tmem_ld32(tS + 32, sr[1]);
    tmem_ld_wait(sr[0]);
    tmem_ld_fence(sr[1]);
    float p[64];
    if (C::kColVecs) {
      const uint32_t va = sbase + C::t1_vec(j);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 l4 = ld_shared_f4(va + 16 * i);
        const int c = 4 * i;
        const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sr[c / 32][c % 32]),
                                                 __uint_as_float(sr[c / 32][c % 32 + 1])),
                                     sc2, make_float2(l4.x, l4.y));
        const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sr[c / 32][c % 32 + 2]),
                                                 __uint_as_float(sr[c / 32][c % 32 + 3])),
                                     sc2, make_float2(l4.z, l4.w));
        p[c] = ex2_approx(x0.x);
        p[c + 1] = ex2_approx(x0.y);
        p[c + 2] = ex2_approx(x1.x);
        p[c + 3] = ex2_approx(x1.y);
      }
      if (CAUSAL && col0 < 128 * w.u + 127) {   // query col0 + c precedes key res_row: masked
        const int lim = res_row - col0;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < lim) p[c] = 0.f;
      }
    } else {
      const float2 nl2 = make_float2(nl, nl);
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[c / 32][c % 32]),
                                                __uint_as_float(sr[c / 32][c % 32 + 1])),
                                    sc2, nl2);
        p[c] = ex2_approx(x.x);
        p[c + 1] = ex2_approx(x.y);
      }
      // keys past N, and (causal) keys after this query row: masked
      int lim = N - col0;
      if (CAUSAL) lim = min(lim, res_row - col0 + 1);
      if (lim < 64) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= lim) p[c] = 0.f;
      }
    }
    if (!C::kHasDP) {   // DV: P^T (bf16) into the first 32 columns of its score buffer
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        pk[i] = pack_bf16x2(p[2 * i], p[2 * i + 1]);
        if constexpr (DROPOUT) pk[i] &= keep_mask_pair(ge[i / 2], 2 * (i % 2));   // (P o M)^T
      }
      tmem_st32(tS, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ds_full[j & 1]);
      continue;
    }
    if (MODE == kModeDK && !mbar_wait(&t2_full[j & 1], (j >> 1) & 1, g, kSiteBwd256 | 8u)) return;
    if (!mbar_wait(dp_full, j & 1, g, kSiteBwd256 | 9u)) return;
    __syncwarp();
    tc_fence_after();
    const uint32_t tDP = tmem + lane_base + C::kColDP;
    uint32_t dr[2][32];
    tmem_ld32(tDP, dr[0]);
    tmem_ld32(tDP + 32, dr[1]);
    tmem_ld_wait(dr[0]);
    tmem_ld_fence(dr[1]);
    uint32_t pk[32];
    if (MODE == kModeDK) {
      const uint32_t vd = sbase + C::t2_vec(j);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 d4 = ld_shared_f4(vd + 16 * i);
        const int c = 4 * i;
        const float2 dr01 = make_float2(__uint_as_float(dr[c / 32][c % 32]), __uint_as_float(dr[c / 32][c % 32 + 1]));
        const float2 dr23 = make_float2(__uint_as_float(dr[c / 32][c % 32 + 2]),
                                        __uint_as_float(dr[c / 32][c % 32 + 3]));
        float2 a, b;
        if constexpr (DROPOUT) {   // M~ o dP - D
          const float2 ds2 = make_float2(drop.scale, drop.scale);
          a = __ffma2_rn(keep_pair_f(dr01, ge, c), ds2, make_float2(d4.x, d4.y));
          b = __ffma2_rn(keep_pair_f(dr23, ge, c + 2), ds2, make_float2(d4.z, d4.w));
        } else {
          a = __fadd2_rn(dr01, make_float2(d4.x, d4.y));
          b = __fadd2_rn(dr23, make_float2(d4.z, d4.w));
        }
        const float2 s0 = __fmul2_rn(make_float2(p[c], p[c + 1]), a);
        const float2 s1 = __fmul2_rn(make_float2(p[c + 2], p[c + 3]), b);
        pk[2 * i] = pack_bf16x2(s0.x, s0.y);
        pk[2 * i + 1] = pack_bf16x2(s1.x, s1.y);
      }
    } else {
      const float2 nd2 = make_float2(nd, nd);
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float2 dr01 = make_float2(__uint_as_float(dr[c / 32][c % 32]), __uint_as_float(dr[c / 32][c % 32 + 1]));
        float2 a;
        if constexpr (DROPOUT)   // M~ o dP - D
          a = __ffma2_rn(keep_pair_f(dr01, ge, c), make_float2(drop.scale, drop.scale), nd2);
        else
          a = __fadd2_rn(dr01, nd2);
        const float2 s0 = __fmul2_rn(make_float2(p[c], p[c + 1]), a);
        pk[c / 2] = pack_bf16x2(s0.x, s0.y);
      }
    }
    tmem_st32(tDP, pk);   // dS (or dS^T) over the first 32 dP columns
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&ds_full[j & 1]);
  }

  // epilogue: acc * mult -> bf16 -> swizzled staging in the first resident
  // tile (its last reader has completed with acc_done) -> TMA store
  if (!mbar_wait(acc_done, 0, g, kSiteBwd256 | 10u)) return;
  __syncwarp();
  tc_fence_after();
  const float mult = MODE == kModeDV ? (DROPOUT ? drop.scale : 1.f) : scale;
  const uint32_t tAcc = tmem + lane_base + C::kColAcc;
#pragma unroll 1
  for (int c = 0; c < 256; c += 32) {
    uint32_t o[32];
    tmem_ld32(tAcc + c, o);
    tmem_ld_wait(o);
    const uint32_t box = sbase + C::kR1Off + (c / 64) * C::kResBox + r * 128;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int chunk = (c % 64) / 8 + q;
      float f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[8 * q + e]) * mult;
      st_shared_v4(box + ((chunk ^ (r & 7)) << 4), pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                   pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
    }
  }
  fence_proxy_async_smem();
  mbar_arrive(staged);
  if (r == 0 && mbar_wait(staged, 0, g, kSiteBwd256 | 11u)) {
    for (int b = 0; b < 4; ++b)
      if (64 * b < d) tma_store_hd(tmOut, smem + C::kR1Off + b * C::kResBox, 64 * b, 128 * w.u, w.hc);
    tma_store_commit();
    tma_store_wait_read_all();
  }
}

// FD: d = 256 (compile-time K steps and output width of the products).
template <int MODE, bool CAUSAL, bool FD, bool DROPOUT>
__global__ void __launch_bounds__(192, 1)
    fa_bwd_d256_kernel(const __grid_constant__ CUtensorMap tmR1, const __grid_constant__ CUtensorMap tmR2,
                       const __grid_constant__ CUtensorMap tmT1, const __grid_constant__ CUtensorMap tmT2,
                       const __grid_constant__ CUtensorMap tmOut, const float* __restrict__ lse,
                       const float* __restrict__ Dg, int N, int d, int n_res, int BH, int H, int band, float scale,
                       float scale_log2, int ks, uint32_t idesc_acc, const __grid_constant__ DropArgs drop,
                       const WaitCfg wc) {
  using C = B256<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* r_full = bars;
  uint64_t* t1_full = r_full + 1;     // [2], by step parity
  uint64_t* t1_empty = t1_full + 2;   // [2]
  uint64_t* t2_full = t1_empty + 2;   // [2]
  uint64_t* t2_empty = t2_full + 2;   // [2]
  uint64_t* s_full = t2_empty + 2;    // [2]
  uint64_t* dp_full = s_full + 2;
  uint64_t* ds_full = dp_full + 1;    // [2], by step parity
  uint64_t* acc_done = ds_full + 2;
  uint64_t* staged = acc_done + 1;
  uint64_t* drain = staged + 1;
  uint64_t* a_ready = drain + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const U256 w = unit256<MODE, CAUSAL>(N, n_res, BH, H, band);

  if (threadIdx.x == 0) {
    mbar_init(r_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&t1_full[i], C::kColVecs ? 2 : 1);   // TMA bytes (+ the producer warp's vector writes)
      mbar_init(&t1_empty[i], 1);
      mbar_init(&t2_full[i], MODE == kModeDK ? 2 : 1);
      mbar_init(&t2_empty[i], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(dp_full, 1);
    mbar_init(&ds_full[0], 128);
    mbar_init(&ds_full[1], 128);
    mbar_init(acc_done, 1);
    mbar_init(staged, 128);
    mbar_init(drain, 1);
    mbar_init(a_ready, 128);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmR1);
    if (C::kHasDP) tma_prefetch_desc(&tmR2);
    tma_prefetch_desc(&tmT1);
    tma_prefetch_desc(&tmT2);
    tma_prefetch_desc(&tmOut);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const CtaGuard g{abort_flag, g_status_bwd256, wc.epoch, wc.limit_us};

  if (warp == 4) {
    b256_producer<MODE>(w, smem, r_full, t1_full, t1_empty, t2_full, t2_empty, &tmR1, &tmR2, &tmT1, &tmT2, lse, Dg,
                        N, g);
  } else if (warp == 5) {
    b256_mma<MODE, FD>(w, tmem, smem_u32(smem), r_full, t1_full, t1_empty, t2_full, t2_empty, s_full, dp_full, ds_full,
                       acc_done, a_ready, ks, idesc_acc, g);
    tc_commit_w(drain);   // every MMA issued above has finished before TMEM is released
    mbar_drain(drain, 0);
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, 160);
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  } else {
    b256_compute<MODE, CAUSAL, DROPOUT>(w, tmem, smem, r_full, t1_full, t2_full, s_full, dp_full, ds_full, acc_done,
                                        a_ready, staged, &tmOut, lse, Dg, N, d, scale, scale_log2, drop, g);
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, 160);
  }
}

template <int MODE, bool CAUSAL, bool DROPOUT>
cudaError_t launch_t(const CUtensorMap& r1, const CUtensorMap& r2, const CUtensorMap& t1, const CUtensorMap& t2,
                     const CUtensorMap& out, const float* lse, const float* Dvec, const Shape& s,
                     const DropArgs& drop, const WaitCfg& wc, cudaStream_t st) {
  using C = B256<MODE>;
  auto kern = s.d == 256 ? fa_bwd_d256_kernel<MODE, CAUSAL, true, DROPOUT>
                         : fa_bwd_d256_kernel<MODE, CAUSAL, false, DROPOUT>;
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads, 0);
  if (e != cudaSuccess) return e;
  const int n_res = (s.N + 127) / 128;
  const float scale_log2 = static_cast<float>(static_cast<double>(s.scale) * 1.4426950408889634);
  const dim3 grid(static_cast<unsigned>(s.B) * s.H * n_res);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(r1, r2, t1, t2, out, lse, Dvec, s.N, s.d, n_res, s.B * s.H, s.H,
                                                 head_band(s.N, s.d), s.scale, scale_log2, score_ksteps(s.d),
                                                 idesc_bf16(128, out_cols(s.d), false, true), drop, wc);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_m(const CUtensorMap& r1, const CUtensorMap& r2, const CUtensorMap& t1, const CUtensorMap& t2,
                     const CUtensorMap& out, const float* lse, const float* Dvec, const Shape& s,
                     const DropArgs& drop, const WaitCfg& wc, cudaStream_t st) {
  if (drop.t4 != 0)
    return s.causal ? launch_t<MODE, true, true>(r1, r2, t1, t2, out, lse, Dvec, s, drop, wc, st)
                    : launch_t<MODE, false, true>(r1, r2, t1, t2, out, lse, Dvec, s, drop, wc, st);
  return s.causal ? launch_t<MODE, true, false>(r1, r2, t1, t2, out, lse, Dvec, s, drop, wc, st)
                  : launch_t<MODE, false, false>(r1, r2, t1, t2, out, lse, Dvec, s, drop, wc, st);
}

}  // namespace

cudaError_t launch_bwd_d256_dkdv(const WideBwdMaps& m, const float* lse, const float* Dvec, const Shape& s,
                                 const DropArgs& drop, cudaStream_t st) {
  const cudaError_t e =
      launch_m<kModeDV>(m.k128, m.k128, m.q64, m.do64, m.dv128, lse, Dvec, s, drop, next_wait_cfg(), st);
  if (e != cudaSuccess) return e;
  return launch_m<kModeDK>(m.k128, m.v128, m.q64, m.do64, m.dk128, lse, Dvec, s, drop, next_wait_cfg(), st);
}

cudaError_t launch_bwd_d256_dq(const WideBwdMaps& m, const float* lse, const float* Dvec, const Shape& s,
                               const DropArgs& drop, cudaStream_t st) {
  return launch_m<kModeDQ>(m.q128, m.do128, m.k64, m.v64, m.dq128, lse, Dvec, s, drop, next_wait_cfg(), st);
}

cudaError_t bwd_d256_status(uint32_t* out, bool reset) {
  unsigned int v[2] = {0, 0};
  cudaError_t e = cudaMemcpyFromSymbol(v, g_status_bwd256, sizeof(v));
  if (e != cudaSuccess) return e;
  *out = v[0];
  if (reset && (v[0] | v[1]) != 0) {
    const unsigned int z[2] = {0, 0};
    e = cudaMemcpyToSymbol(g_status_bwd256, z, sizeof(z));
  }
  return e;
}

}  // namespace fa
