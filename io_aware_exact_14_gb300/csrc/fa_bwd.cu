// Backward pass of exact attention on sm_103a (recompute-based).
//
// The pages describe the backward only as recomputing S and P on chip from the
// saved inputs instead of storing P ("为什么Flash Attention能将注意力计算提速数倍
// 而不损失精度", section "反向传播中的重计算策略").  The gradients are the calculus
// of the forward definition:
//   dV = P^T dO, dP = dO V^T, D_i = sum_c dO_ic O_ic, dS = P o (dP - D),
//   dQ = scale dS K, dK = scale dS^T Q,
// with P recomputed as exp(scale q.k - LSE) from the forward's log-sum-exp.
// With dropout on the probabilities (mask M~ = keep / (1 - p), regenerated
// from the same counter-based Philox stream as the forward), dV = (P o M~)^T dO
// and dS = P o (M~ o dP - D), D taken from the dropped O.
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <cmath>
#include <mutex>

namespace fa {
namespace {

__device__ unsigned int g_status_bwd[2] = {0, 0};   // status, abort epoch (see CtaGuard)
constexpr int kMaxDevices = 64;

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

// Byte offset of row `row` (= (b H + h) N + n) of a strided [B, H, N, d] bf16
// view; `contig` takes the contiguous layout's plain row * d.
__device__ __forceinline__ size_t pre_row_offset(long long row, bool contig, int d, int H, int N,
                                                 const Strides& st) {
  if (contig) return static_cast<size_t>(row) * d * 2;
  const long long t = row / N, n = row - t * N, b = t / H, h = t - b * H;
  return static_cast<size_t>(b * st.b + h * st.h + n * st.n) * 2;
}

template <int D, bool FULL>
__global__ void __launch_bounds__(kPreThreads) fa_bwd_preprocess_kernel(const uint8_t* __restrict__ o,
                                                                       const uint8_t* __restrict__ dO,
                                                                       float* __restrict__ Dvec, long long rows,
                                                                       int H, int N, int d, Strides so,
                                                                       Strides sdo, bool contig) {
  // D = 64, 128 or 256 covers d <= D: chunks at or past d count as zero.  FULL
  // (d == D) keeps the row length a compile-time constant, and the loads
  // unconditional, on the common path.
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
      if constexpr (FULL) {
        if (row < rows) {
          a[u] = ldg_stream(o + pre_row_offset(row, contig, D, H, N, so) + sub * 16);
          b[u] = ldg_stream(dO + pre_row_offset(row, contig, D, H, N, sdo) + sub * 16);
        }
      } else {
        a[u] = make_uint4(0u, 0u, 0u, 0u);
        b[u] = a[u];
        if (row < rows && sub * 8 < d) {
          a[u] = ldg_stream(o + pre_row_offset(row, contig, d, H, N, so) + sub * 16);
          b[u] = ldg_stream(dO + pre_row_offset(row, contig, d, H, N, sdo) + sub * 16);
        }
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

// ---------------------------------------------------------------------------
// Steps 2 and 3: the two tensor-core kernels.
//
// Shared layout: one CTA per SM, 384 threads.
//   warps 0-3  compute warpgroup 0: columns [0, 64) of each 128 x 128 tile
//   warps 4-7  compute warpgroup 1: columns [64, 128)
//   warp  8    producer (TMA tiles, the work-unit sequence and the epilogue
//              stores; in dK/dV the whole warp also writes the row vectors)
//   warp  9    TMEM owner and tcgen05.mma issuer (elect.sync in a converged warp)
//   warp  10   dQ: loads each unit's dO
//   others     idle
// TMEM (512 columns): scores, dP, then accumulators (dQ double-buffers its
// scores in the columns its single accumulator leaves free).  bf16 operands
// made by the compute warps (P^T, dS^T, dS) overwrite the first 32 columns of
// their own half of the score / dP tile and feed the next MMA from TMEM.
// ---------------------------------------------------------------------------

constexpr float kLog2e = 1.4426950408889634f;
// L2 prefetch: the dQ producer warms the first kL2Ahead key tiles of its next
// unit.  Per-tile prefetches in the steady loops, and the dK/dV producer's
// prefetch of its next unit, measured slower: the prefetches queue on the
// SM's copy engine ahead of the loads that need it, and the streamed tiles of
// a head are L2 hits anyway (heads run in small bands).
constexpr int kL2Ahead = 4;

// Tile geometry shared by both kernels: a 128-row tile of d bf16 columns is
// d/64 swizzled boxes of 128 rows x 128 bytes.
template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kBoxes = D / 64;
  static constexpr uint32_t kBoxBytes = 128u * 128u;
  static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;
  static constexpr uint32_t kMaxSmem = 232448;   // per-CTA opt-in limit
};

// S-like product: D(128 x 128) = A(128 x d) * B(128 x d)^T, both K-major
// tiles; only the ks = ceil(d / 16) steps of 16 columns that hold data.  FD
// (d == D): all D / 16 steps as a straight run of MMAs; otherwise each
// step's issue is predicated (a branch per MMA measured 11% slower).
template <int D, bool FD>
__device__ __forceinline__ void mma_nt(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc, int ks) {
  using C = BwdCfg<D>;
  constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = ((kk / 4) * C::kBoxBytes + (kk % 4) * 32) >> 4;   // descriptor address units
    if constexpr (FD)
      tc_mma_ss_w(tmem_d, a_desc + off, b_desc + off, idesc, kk > 0 ? 1u : 0u);
    else
      tc_mma_ss_w_if(tmem_d, a_desc + off, b_desc + off, idesc, kk > 0 ? 1u : 0u, kk < ks ? 1u : 0u);
  }
}

// Accumulating product: D(128 x d) += A(128 x 128, TMEM bf16) * B(128 x d, MN-major tile).
// A's 128 K columns live as two 64-wide halves at a_tmem and a_tmem + 64.
// idesc: M = 128, N = ceil(d / 16) * 16, B MN-major (a compile-time constant
// when d == D).
template <int D, bool FD>
__device__ __forceinline__ void mma_tn_acc(uint32_t tmem_d, uint32_t a_tmem, uint64_t b_desc, bool acc,
                                           uint32_t idesc_rt) {
  const uint32_t idesc = FD ? idesc_bf16(128, D, false, true) : idesc_rt;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t a = a_tmem + (kk / 4) * 64 + (kk % 4) * 8;
    tc_mma_ts_w(tmem_d, a, b_desc + ((kk * 2048) >> 4), idesc, (acc || kk > 0) ? 1u : 0u);
  }
}

// K-major (kmaj) and MN-major (mnmaj) descriptors of a 128-row tile at `addr`.
template <int D>
__device__ __forceinline__ uint64_t kmaj(uint32_t addr) { return sdesc_sw128(addr, 16, 1024); }
template <int D>
__device__ __forceinline__ uint64_t mnmaj(uint32_t addr) { return sdesc_sw128(addr, BwdCfg<D>::kBoxBytes, 1024); }

// Pack 32 fp32 values (in two 16-value halves) into 16 bf16x2 words and store
// them to 16 TMEM columns.
__device__ __forceinline__ void st_bf16_16cols(uint32_t taddr, const float* v) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  tmem_st16(taddr, w);
}

// The same for v o M (0/1): column c is zeroed unless kept, its keep bit in
// byte c % 4 of ge[c / 4] (byte-MSB form).
__device__ __forceinline__ void st_bf16_16cols_dropped(uint32_t taddr, const float* v, const uint32_t* ge) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]) & keep_mask_pair(ge[i / 2], 2 * (i % 2));
  tmem_st16(taddr, w);
}

// Epilogue staging for one 128 x d accumulator: TMEM -> * mult -> bf16 ->
// swizzled tile (the layout a TMA store reads) at shared address `stage`;
// thread r writes row r.
template <int D>
__device__ __forceinline__ void bwd_stage_acc(uint32_t tacc, uint32_t stage, float mult, int r) {
  using C = BwdCfg<D>;
#pragma unroll
  for (int c = 0; c < D; c += 32) {
    uint32_t o[32];
    tmem_ld32(tacc + c, o);
    tmem_ld_wait(o);
    const uint32_t box = stage + (c / 64) * C::kBoxBytes + r * 128;
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
}

// Row vectors for a query tile, stored negated so the compute warps add them
// with packed FMAs: -lse * log2(e) (-inf past N, so P = 0 there) and -D
// (0 past N).  The whole producer warp handles them, four columns per lane:
// fetched into registers one tile ahead (so the global-load latency hides
// behind the wait for a free stage), then written to the stage.
struct RowVecs {
  float a[4], d[4];
};

__device__ __forceinline__ RowVecs fetch_row_vectors(const float* __restrict__ lse, const float* __restrict__ Dg,
                                                     size_t row_base, int q0, int N, int lane) {
  RowVecs r;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int q = q0 + lane + 32 * k;
    r.a[k] = -INFINITY;
    r.d[k] = 0.f;
    if (q < N) {
      const float l = lse[row_base + q];
      r.a[k] = (l == -INFINITY) ? -INFINITY : -l * kLog2e;
      r.d[k] = -Dg[row_base + q];
    }
  }
  return r;
}

// ---------------------------------------------------------------------------
// dK / dV: one work unit per (b, h, 128-key tile j); loop over query tiles i.
//   S^T = K_j Q_i^T, P^T = exp2(S^T * scale * log2e - lse2_i)
//   dP^T = V_j dO_i^T, dS^T = P^T o (dP^T - D_i)
//   dV_j += P^T dO_i,  dK_j += dS^T Q_i,  finally dK_j *= scale
// K_j and V_j are resident per unit; Q_i (with -lse) streams through a 3-deep
// ring and dO_i (with -D) through a 2-deep ring, so the next query tile is
// loaded well before S^T(i+1) needs it.
// MMA order S(i) dP(i) dV(i) {S(i+1), dK(i)} dP(i+1) ...: the exponentials of
// tile i run under dP(i), the dS products under dV(i); S^T(i+1) and dK(i)
// touch different TMEM columns and go in whichever order their inputs land.
// TMEM: T0 = S^T, T1 = dP^T, acc0 = dV, acc1 = dK.
// Persistent CTAs (cluster launch control, as in dQ below): a running CTA
// takes over the next not-yet-started CTA's unit, so barriers, TMEM and the
// rings carry on across units (global query-tile count).  The next unit's
// first Q tile loads as soon as the unit is known, its K_j once this unit's
// last S^T has read the old one and its V_j once the last dP^T has, so its
// first S^T and dP^T run while the compute warps drain this unit's
// accumulators.  Epilogue: the compute warps stage dV in the dO slot
// and dK in the Q slot of the unit's last query tile L (both free once dK(L)
// is done); the producer stores them with TMA and reloads those slots (with
// dO(L+2) and Q(L+3)) only after the stores have read them.
// ---------------------------------------------------------------------------

template <int D>
struct DkdvCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kBoxes = D / 64;
  static constexpr uint32_t kBoxBytes = 128u * 128u;
  static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kQStages = 3, kDOStages = 2;
  static constexpr uint32_t kKOff = 0, kVOff = kTileBytes;
  static constexpr uint32_t kQOff = 2 * kTileBytes;
  static constexpr uint32_t kDOOff = kQOff + kQStages * kTileBytes;
  static constexpr uint32_t kLseOff = kDOOff + kDOStages * kTileBytes;   // 128 fp32 per Q stage
  static constexpr uint32_t kDVecOff = kLseOff + kQStages * 512;          // 128 fp32 per dO stage
  static constexpr uint32_t kBarOff = kDVecOff + kDOStages * 512;
  // k_full[2], v_full[2], k_free, v_free, q_full[3], q_empty[3], do_full[2],
  // s_full, dp_full, p_full, ds_full, acc_done, acc_free, drain, staged[2],
  // sched.  A dO slot has no empty barrier of its own: dO_i's last reader
  // (dV(i)) finishes before dK(i), whose commit already releases Q_i's slot.
  // k_full, v_full and staged go by unit parity, so none of them runs two
  // phases ahead of a waiter.
  static constexpr int kBars = 6 + 2 * kQStages + kDOStages + 10;
  static constexpr uint32_t kMiscOff = kBarOff + kBars * 8;   // tmem holder, abort flag, unit ids [2]
  static constexpr uint32_t kRespOff = (kMiscOff + 16 + 15) / 16 * 16;   // 16-byte work-steal response
  static constexpr uint32_t kLayoutBytes = kRespOff + 16;
  static constexpr uint32_t kMaxSmem = BwdCfg<D>::kMaxSmem;
  // room for the 1024-byte alignment of the base when it fits, else all there is
  static constexpr uint32_t kSmemBytes = kLayoutBytes + 1024 <= kMaxSmem ? kLayoutBytes + 1024 : kMaxSmem;
  static_assert(kLayoutBytes <= kMaxSmem, "dK/dV shared-memory layout too large");
  static constexpr int kThreads = 384;
  static constexpr int kRequestAhead = 3;   // query tiles before a unit's end at which the next is requested
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  __host__ __device__ static constexpr uint32_t q_off(int s) { return kQOff + s * kTileBytes; }
  __host__ __device__ static constexpr uint32_t do_off(int s) { return kDOOff + s * kTileBytes; }
  __host__ __device__ static constexpr uint32_t lse_off(int s) { return kLseOff + s * 512; }
  __host__ __device__ static constexpr uint32_t dvec_off(int s) { return kDVecOff + s * 512; }
};

// Work unit u (a CTA index of the launch grid) -> head, key tile, query tiles.
struct DkdvUnit {
  int bh, kt, i0, cnt;
};
template <bool CAUSAL>
__device__ __forceinline__ DkdvUnit dkdv_unit(int u, int n_tiles, int BH, int band) {
  DkdvUnit w;
  banded_order(u, n_tiles, BH, band, w.bh, w.kt);   // causal: small kt is heavy, rank 0 -> kt 0
  w.i0 = CAUSAL ? w.kt : 0;                          // first query tile
  w.cnt = n_tiles - w.i0;                            // query tiles visited (>= 1)
  return w;
}

// FD: d == D (compile-time K steps and output width of the products).
template <int D, bool CAUSAL, bool DROPOUT, bool FD>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
                       const float* __restrict__ lse, const float* __restrict__ Dg, int N, int n_tiles,
                       int BH, int H, int band, float scale, float scale_log2, int ks, uint32_t idesc_acc,
                       const __grid_constant__ DropArgs drop, const WaitCfg wc) {
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (static_cast<uint32_t>(smem - smem_raw) + C::kLayoutBytes > C::kSmemBytes) {
    // the aligned layout does not fit this launch's shared memory: report, touch nothing
    if (threadIdx.x == 0) atomicCAS(&g_status_bwd[0], 0u, kSiteDkdv | 0xFFu);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* k_full = bars;                  // [2], by unit parity; also publishes the unit id
  uint64_t* v_full = k_full + 2;            // [2], by unit parity
  uint64_t* k_free = v_full + 2;
  uint64_t* v_free = k_free + 1;
  uint64_t* q_full = v_free + 1;
  uint64_t* q_empty = q_full + C::kQStages;
  uint64_t* do_full = q_empty + C::kQStages;
  uint64_t* s_full = do_full + C::kDOStages;
  uint64_t* dp_full = s_full + 1;
  uint64_t* p_full = dp_full + 1;
  uint64_t* ds_full = p_full + 1;
  uint64_t* acc_done = ds_full + 1;
  uint64_t* acc_free = acc_done + 1;
  uint64_t* drain = acc_free + 1;
  uint64_t* staged = drain + 1;             // [2], by unit parity
  uint64_t* sched = staged + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff + 4);
  // unit ids by unit parity: unit k + 2's id is written only after unit k + 1's
  // S^T have all been issued, by which time every reader has taken k's
  volatile int* unit_id = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 8);
  uint8_t* resp = smem + C::kRespOff;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);     // the producer's expect-tx arrival (plain arrival when no unit is left)
      mbar_init(&v_full[i], 1);
      mbar_init(&staged[i], 256);   // every compute thread, after staging its rows
    }
    mbar_init(k_free, 1);
    mbar_init(v_free, 1);
    for (int i = 0; i < C::kQStages; ++i) {
      mbar_init(&q_full[i], 2);     // TMA bytes + the producer warp's -lse writes
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < C::kDOStages; ++i) {
      mbar_init(&do_full[i], 2);    // TMA bytes + the producer warp's -D writes
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, 256);
    mbar_init(ds_full, 256);
    mbar_init(acc_done, 1);
    mbar_init(acc_free, 256);
    mbar_init(drain, 1);
    mbar_init(sched, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const CtaGuard g{abort_flag, g_status_bwd, wc.epoch, wc.limit_us};
  const uint32_t sbase = smem_u32(smem);

  if (warp >= 8) {
    if (warp == 8) {
      // Producer: per unit K_j, V_j; per query tile Q_i and dO_i (+ row
      // vectors); the next unit; the epilogue stores.  The whole warp runs the
      // loop (it writes the row vectors), lane 0 issues every copy.
      //
      // Pending epilogue stores, oldest first: unit `pend_su` and the next.  A
      // unit ending at query tile L is stored just before dO(L+2) reuses its dV
      // slot; its dK store may still be reading when that load goes out and is
      // waited for before the next Q load (Q(L+3) is the first to reuse it).
      int p0_bh = 0, p0_kt = 0, p0_last = 0, p1_bh = 0, p1_kt = 0, p1_last = 0;
      int n_pend = 0, pend_su = 0;
      bool dk_reading = false;
      auto store_front = [&]() -> bool {   // lane 0
        if (!mbar_wait(&staged[pend_su & 1], (pend_su >> 1) & 1, g, kSiteDkdv | 16u)) return false;
        const HeadCoord phc = head_coord(p0_bh, H);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_store_hd(&tmDV, smem + C::do_off(p0_last % C::kDOStages) + b * C::kBoxBytes, 64 * b, 128 * p0_kt, phc);
        tma_store_commit();
        for (int b = 0; b < C::kBoxes; ++b)
          tma_store_hd(&tmDK, smem + C::q_off(p0_last % C::kQStages) + b * C::kBoxBytes, 64 * b, 128 * p0_kt, phc);
        tma_store_commit();
        tma_store_wait_read_but_one();   // dV has been read out of the dO slot
        dk_reading = true;
        p0_bh = p1_bh;
        p0_kt = p1_kt;
        p0_last = p1_last;
        --n_pend;
        ++pend_su;
        return true;
      };
      int u = static_cast<int>(blockIdx.x);
      int gi = 0;   // global query-tile count (ring index)
      bool ok = true;
      for (int su = 0; ok; ++su) {
        int okl = 1;
        if (u < 0) {   // no work left: release the consumers (published like a unit id)
          if (lane == 0 && (su == 0 || mbar_wait(k_free, (su - 1) & 1, g, kSiteDkdv | 15u))) {
            unit_id[su & 1] = -1;
            mbar_arrive(&k_full[su & 1]);
          }
          break;
        }
        const DkdvUnit w = dkdv_unit<CAUSAL>(u, n_tiles, BH, band);
        const HeadCoord hc = head_coord(w.bh, H);
        const size_t row_base = static_cast<size_t>(w.bh) * N;
        RowVecs rv = fetch_row_vectors(lse, Dg, row_base, 128 * w.i0, N, lane);
        for (int it = 0; it < w.cnt; ++it, ++gi) {
          const int qt = w.i0 + it;
          const int qs = gi % C::kQStages, ds = gi % C::kDOStages;
          if (lane == 0) {
            if (it == max(0, w.cnt - C::kRequestAhead)) {   // ask for the next unit
              mbar_arrive_expect_tx(sched, 16);
              clc_try_cancel(resp, sched);
            }
            okl = mbar_wait(&q_empty[qs], ((gi / C::kQStages) & 1u) ^ 1u, g, kSiteDkdv | 1u);
            if (okl && dk_reading) {   // a staged dK may still be read from this slot
              tma_store_wait_read_all();
              dk_reading = false;
            }
          }
          if (!__shfl_sync(0xffffffffu, okl, 0)) { ok = false; break; }
          if (lane == 0) {
            mbar_arrive_expect_tx(&q_full[qs], C::kTileBytes);
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_hd(smem + C::q_off(qs) + b * C::kBoxBytes, &tmQ, &q_full[qs], 64 * b, 128 * qt, hc);
          }
          if (it == 0) {
            // the unit's K_j replaces the previous unit's once its last S^T is
            // done (and goes out with the unit id), V_j once its last dP^T is;
            // both before this tile's row vector, whose global loads may still
            // be in flight
            if (lane == 0) {
              if (su > 0) okl = mbar_wait(k_free, (su - 1) & 1, g, kSiteDkdv | 15u);
              if (okl) {
                unit_id[su & 1] = u;
                mbar_arrive_expect_tx(&k_full[su & 1], C::kTileBytes);
                for (int b = 0; b < C::kBoxes; ++b)
                  tma_load_hd(smem + C::kKOff + b * C::kBoxBytes, &tmK, &k_full[su & 1], 64 * b, 128 * w.kt, hc);
                if (su > 0) okl = mbar_wait(v_free, (su - 1) & 1, g, kSiteDkdv | 20u);
              }
              if (okl) {
                mbar_arrive_expect_tx(&v_full[su & 1], C::kTileBytes);
                for (int b = 0; b < C::kBoxes; ++b)
                  tma_load_hd(smem + C::kVOff + b * C::kBoxBytes, &tmV, &v_full[su & 1], 64 * b, 128 * w.kt, hc);
              }
            }
            if (!__shfl_sync(0xffffffffu, okl, 0)) { ok = false; break; }
          }
          float* nl = reinterpret_cast<float*>(smem + C::lse_off(qs));
#pragma unroll
          for (int k = 0; k < 4; ++k) nl[lane + 32 * k] = rv.a[k];
          __syncwarp();
          if (lane == 0) mbar_arrive(&q_full[qs]);
          // dO slot reuse: tile gi - 2's dK (after its dV) has completed, which
          // the q_empty commit of that tile signals; a unit that ended there
          // is stored first (its dV is staged in this slot)
          if (lane == 0) {
            if (gi >= C::kDOStages) {
              const int pt = gi - C::kDOStages;
              okl = mbar_wait(&q_empty[pt % C::kQStages], (pt / C::kQStages) & 1u, g, kSiteDkdv | 12u);
            }
            if (okl && n_pend > 0 && p0_last + C::kDOStages == gi) okl = store_front();
          }
          if (!__shfl_sync(0xffffffffu, okl, 0)) { ok = false; break; }
          if (lane == 0) {
            mbar_arrive_expect_tx(&do_full[ds], C::kTileBytes);
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_hd(smem + C::do_off(ds) + b * C::kBoxBytes, &tmDO, &do_full[ds], 64 * b, 128 * qt, hc);
          }
          float* nd = reinterpret_cast<float*>(smem + C::dvec_off(ds));
#pragma unroll
          for (int k = 0; k < 4; ++k) nd[lane + 32 * k] = rv.d[k];
          __syncwarp();
          if (lane == 0) mbar_arrive(&do_full[ds]);
          if (it + 1 < w.cnt) rv = fetch_row_vectors(lse, Dg, row_base, 128 * (qt + 1), N, lane);
        }
        if (!ok) break;
        int nu = -1;
        if (lane == 0) {
          if (n_pend == 0) {   // at most one older store is still pending here
            p0_bh = w.bh;
            p0_kt = w.kt;
            p0_last = gi - 1;
          } else {
            p1_bh = w.bh;
            p1_kt = w.kt;
            p1_last = gi - 1;
          }
          ++n_pend;
          okl = mbar_wait(sched, su & 1, g, kSiteDkdv | 19u);
          if (okl) nu = clc_decode(resp);
        }
        if (!__shfl_sync(0xffffffffu, okl, 0)) break;
        u = __shfl_sync(0xffffffffu, nu, 0);
      }
      if (lane == 0) {   // the remaining epilogue stores; all of them land before the CTA retires
        bool sok = true;
        while (sok && n_pend > 0) sok = store_front();
        tma_store_wait_all();
      }
    } else if (warp == 9) {  // MMA issuer: the whole warp runs the loop, one lane issues
      const uint32_t tS = tmem + C::kColS, tDP = tmem + C::kColDP;
      const uint32_t tDV = tmem + C::kColDV, tDK = tmem + C::kColDK;
      const uint64_t kK = kmaj<D>(sbase + C::kKOff), kV = kmaj<D>(sbase + C::kVOff);
      // Q and dO stages as K-major B operands (S^T, dP^T) and MN-major B operands (dK, dV)
      auto kQ = [&](int s) { return kmaj<D>(sbase + C::q_off(s)); };
      auto mQ = [&](int s) { return mnmaj<D>(sbase + C::q_off(s)); };
      auto kDO = [&](int s) { return kmaj<D>(sbase + C::do_off(s)); };
      auto mDO = [&](int s) { return mnmaj<D>(sbase + C::do_off(s)); };
      auto qpar = [](int i) { return static_cast<uint32_t>((i / C::kQStages) & 1); };
      auto dpar = [](int i) { return static_cast<uint32_t>((i / C::kDOStages) & 1); };
      bool ok = true;
      int gi = 0;
      for (int su = 0; ok; ++su) {
        if (!(ok = mbar_wait_w(&k_full[su & 1], (su >> 1) & 1, g, kSiteDkdv | 2u))) break;
        const int u = unit_id[su & 1];
        if (u < 0) break;
        const int cnt = dkdv_unit<CAUSAL>(u, n_tiles, BH, band).cnt;
        const int g0 = gi;
        // S^T(0), dP^T(0): the previous unit's readers of these columns (its
        // last dV and dK) were issued before
        if (!(ok = mbar_wait_w(&q_full[g0 % C::kQStages], qpar(g0), g, kSiteDkdv | 3u))) break;
        mma_nt<D, FD>(tS, kK, kQ(g0 % C::kQStages), ks);
        tc_commit_w(s_full);
        if (cnt == 1) tc_commit_w(k_free);    // K_j: last reader issued
        if (!(ok = mbar_wait_w(&v_full[su & 1], (su >> 1) & 1, g, kSiteDkdv | 3u))) break;
        if (!(ok = mbar_wait_w(&do_full[g0 % C::kDOStages], dpar(g0), g, kSiteDkdv | 3u))) break;
        mma_nt<D, FD>(tDP, kV, kDO(g0 % C::kDOStages), ks);
        tc_commit_w(dp_full);
        if (cnt == 1) tc_commit_w(v_free);    // V_j: last reader issued
        for (int it = 0; ok && it < cnt; ++it) {
          const int i = g0 + it;
          const int qs = i % C::kQStages, ds = i % C::kDOStages;
          const int qs1 = (i + 1) % C::kQStages, ds1 = (i + 1) % C::kDOStages;
          const uint32_t par = i & 1;
          const bool next = it + 1 < cnt;
          if (!(ok = mbar_wait_w(p_full, par, g, kSiteDkdv | 4u))) break;
          // the unit's first dV overwrites the accumulator: the previous
          // unit's epilogue must have read both accumulators out
          if (it == 0 && su > 0 && !(ok = mbar_wait_w(acc_free, (su - 1) & 1, g, kSiteDkdv | 18u))) break;
          tc_fence_after();
          mma_tn_acc<D, FD>(tDV, tS, mDO(ds), it > 0, idesc_acc);          // dV += P^T dO_i
          bool s_done = !next, k_done = false;
          while (ok && !(s_done && k_done)) {
            int which;
            if (!s_done && !k_done)
              which = mbar_wait_either_w(&q_full[qs1], qpar(i + 1), ds_full, par, g, kSiteDkdv | 5u);
            else if (!s_done)
              which = mbar_wait_w(&q_full[qs1], qpar(i + 1), g, kSiteDkdv | 5u) ? 0 : -1;
            else
              which = mbar_wait_w(ds_full, par, g, kSiteDkdv | 6u) ? 1 : -1;
            if (which < 0) {
              ok = false;
            } else if (which == 0) {
              mma_nt<D, FD>(tS, kK, kQ(qs1), ks);                     // S^T(i+1)
              tc_commit_w(s_full);
              if (it + 2 == cnt) tc_commit_w(k_free);       // K_j: last reader issued
              s_done = true;
            } else {
              tc_fence_after();
              mma_tn_acc<D, FD>(tDK, tDP, mQ(qs), it > 0, idesc_acc);        // dK += dS^T Q_i
              tc_commit_w(&q_empty[qs]);                     // Q_i, -lse_i, and dO_i, -D_i: last readers done
              k_done = true;
            }
          }
          if (!ok) break;
          if (next) {
            if (!(ok = mbar_wait_w(&do_full[ds1], dpar(i + 1), g, kSiteDkdv | 13u))) break;
            mma_nt<D, FD>(tDP, kV, kDO(ds1), ks);                     // dP^T(i+1), after dK(i) has read dS^T(i)
            tc_commit_w(dp_full);
            if (it + 2 == cnt) tc_commit_w(v_free);         // V_j: last reader issued
          }
        }
        if (!ok) break;
        tc_commit_w(acc_done);
        gi = g0 + cnt;
      }
      tc_commit_w(drain);
      mbar_drain(drain, 0);
      __syncwarp();
      tc_fence_before();
      named_bar_sync(1, 288);
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
    return;
  }

  // compute warpgroups: key row t = TMEM lane; half h owns query columns [64h, 64h+64)
  const int h = warp >> 2;
  const int t = threadIdx.x & 127;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_base + C::kColS + 64 * h;
  const uint32_t tDP = tmem + lane_base + C::kColDP + 64 * h;
  const float2 sc2 = make_float2(scale_log2, scale_log2);
  bool ok = true;
  int gi = 0;
  for (int su = 0; ok; ++su) {
    if (!(ok = mbar_wait(&k_full[su & 1], (su >> 1) & 1, g, kSiteDkdv | 17u))) break;
    const int u = unit_id[su & 1];
    if (u < 0) break;
    const DkdvUnit w = dkdv_unit<CAUSAL>(u, n_tiles, BH, band);
    for (int it = 0; ok && it < w.cnt; ++it, ++gi) {
      const int qs = gi % C::kQStages, ds = gi % C::kDOStages;
      const uint32_t par = gi & 1;
      const int qt = w.i0 + it;
      // dropout keep words of key 128 kt + t against this half's 64 queries,
      // drawn before S^T lands: query column c in byte c % 4 of ge[c / 4]
      uint32_t ge[DROPOUT ? 16 : 1];
      if constexpr (DROPOUT) dropout_cols<4>(drop, w.bh, 128 * w.kt + t, 128 * qt + 64 * h, ge);
      // -lse arrived with Q_i (q_full), -D with dO_i (do_full)
      if (!(ok = mbar_wait(&q_full[qs], (gi / C::kQStages) & 1u, g, kSiteDkdv | 7u))) break;
      if (!(ok = mbar_wait(s_full, par, g, kSiteDkdv | 8u))) break;
      __syncwarp();
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld32(tS, sr[0]);
      tmem_ld32(tS + 32, sr[1]);
      tmem_ld_wait(sr[0]);
      tmem_ld_fence(sr[1]);
      float p[64];
      const uint32_t lse_addr = sbase + C::lse_off(qs) + 256 * h;   // -lse * log2(e) of this half's columns
#pragma unroll
      for (int b8 = 0; b8 < 2; ++b8) {   // 32 columns at a time: their loads go out before the math
        float4 l4[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) l4[i] = ld_shared_f4(lse_addr + (8 * b8 + i) * 16);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int c = 32 * b8 + 4 * i + e;
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[c / 32][c % 32]),
                                                    __uint_as_float(sr[(c + 1) / 32][(c + 1) % 32])),
                                        sc2, e ? make_float2(l4[i].z, l4[i].w) : make_float2(l4[i].x, l4[i].y));
            p[c] = ex2_approx(x.x);
            p[c + 1] = ex2_approx(x.y);
          }
        }
      }
      if (CAUSAL && qt == w.kt) {
        // diagonal tile: query column 64h + c precedes key t (and is masked) when c < t - 64h
        const int lim = t - 64 * h;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < lim) p[c] = 0.f;
      }
      if constexpr (DROPOUT) {   // dV takes (P o M)^T (x 1/(1-p) at the end); dS below still needs P
#pragma unroll
        for (int c = 0; c < 64; c += 32) st_bf16_16cols_dropped(tS + c / 2, p + c, ge + c / 4);
      } else {
#pragma unroll
        for (int c = 0; c < 64; c += 32) st_bf16_16cols(tS + c / 2, p + c);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full);

      if (!(ok = mbar_wait(&do_full[ds], (gi / C::kDOStages) & 1u, g, kSiteDkdv | 14u))) break;
      if (!(ok = mbar_wait(dp_full, par, g, kSiteDkdv | 9u))) break;
      __syncwarp();
      tc_fence_after();
      uint32_t dr[2][32];
      tmem_ld32(tDP, dr[0]);
      tmem_ld32(tDP + 32, dr[1]);
      tmem_ld_wait(dr[0]);
      tmem_ld_fence(dr[1]);
      const uint32_t d_addr = sbase + C::dvec_off(ds) + 256 * h;   // -D of this half's columns
#pragma unroll
      for (int b8 = 0; b8 < 2; ++b8) {
        float4 d4[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) d4[i] = ld_shared_f4(d_addr + (8 * b8 + i) * 16);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int c = 32 * b8 + 4 * i + e;
            const float2 dr2 = make_float2(__uint_as_float(dr[c / 32][c % 32]),
                                           __uint_as_float(dr[(c + 1) / 32][(c + 1) % 32]));
            const float2 nd = e ? make_float2(d4[i].z, d4[i].w) : make_float2(d4[i].x, d4[i].y);
            float2 dp;
            if constexpr (DROPOUT)
              dp = __ffma2_rn(keep_pair_f(dr2, ge, c), make_float2(drop.scale, drop.scale), nd);   // M~ o dP - D
            else
              dp = __fadd2_rn(dr2, nd);
            const float2 dsv = __fmul2_rn(make_float2(p[c], p[c + 1]), dp);
            p[c] = dsv.x;
            p[c + 1] = dsv.y;
          }
        }
      }
#pragma unroll
      for (int c = 0; c < 64; c += 32) st_bf16_16cols(tDP + c / 2, p + c);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    if (!ok || !(ok = mbar_wait(acc_done, su & 1, g, kSiteDkdv | 10u))) break;
    __syncwarp();
    tc_fence_after();
    // warpgroup 0 stages dV in the dO slot, warpgroup 1 dK (x scale) in the Q
    // slot of the unit's last query tile; the producer stores both
    const int last = gi - 1;
    bwd_stage_acc<D>(tmem + lane_base + (h ? C::kColDK : C::kColDV),
                     sbase + (h ? C::q_off(last % C::kQStages) : C::do_off(last % C::kDOStages)),
                     h ? scale : (DROPOUT ? drop.scale : 1.f), t);
    tc_fence_before();
    mbar_arrive(acc_free);   // both accumulators may be overwritten
    fence_proxy_async_smem();
    mbar_arrive(&staged[su & 1]);
  }
  __syncwarp();
  tc_fence_before();
  named_bar_sync(1, 288);
}

// ---------------------------------------------------------------------------
// dQ: one work unit per (b, h, 128-query tile i); loop over key tiles j.
//   S = Q_i K_j^T, P = exp2(S * scale * log2e - lse2_row)
//   dP = dO_i V_j^T, dS = P o (dP - D_row),  dQ_i += dS K_j,  finally dQ_i *= scale
// Persistent CTAs: the grid has one CTA per unit, but a running CTA takes the
// next not-yet-started CTA's unit over (cluster launch control) instead of
// exiting, so TMEM, barriers and pipelines carry on and the next unit's loads
// and first products overlap this unit's tail and epilogue.  The request goes
// out a few tiles before the unit ends, so units still start in launch order
// (heaviest first) on whichever CTA frees up first; the next unit's id is
// published as soon as it is known, so the compute warps fetch its row terms
// (-lse, -D) before this unit's epilogue.
// Q_i and dO_i are resident per unit; K_j streams through a 3-deep ring (read
// by S(j) and dQ(j)) and V_j through a 2-deep ring (read by dP(j) only); the
// rings and the per-tile barriers run on across units (global tile count).
// The epilogue stages dQ in the K slot of the unit's last key tile L (free
// once dQ(L) is done); the producer stores it with TMA and reloads that slot
// (with K(L+3)) only after the store has read it.  The next unit's Q loads
// once this unit's last S is done, its dO once the last dP is.
// MMA order S(j) dP(j) S(j+1) dQ(j) dP(j+1) ...: the exponentials of tile j
// run under dP(j), the dS products under S(j+1).
// TMEM: T0 = S, T1 = dP, acc = dQ.
// ---------------------------------------------------------------------------

template <int D>
struct DqCfg {
  static constexpr int kKStages = 3, kVStages = 2;
  static constexpr uint32_t kTileBytes = BwdCfg<D>::kTileBytes;
  static constexpr uint32_t kQOff = 0, kDOOff = kTileBytes;
  static constexpr uint32_t kKOff = 2 * kTileBytes;
  static constexpr uint32_t kVOff = kKOff + kKStages * kTileBytes;
  static constexpr uint32_t kBarOff = kVOff + kVStages * kTileBytes;
  // q_full, q_empty, do_full, do_empty, k_full[3], k_empty[3], v_full[2],
  // s_full[2], dp_full, ds_full, acc_done, acc_free, drain, sched, id_taken,
  // id_full[2], staged[4].  A V slot has no empty barrier of its own: dP(j) is
  // issued before dQ(j), whose commit releases K_j.  One s_full per S buffer:
  // its next phase (tile j+2) needs this tile's dS(j) first, so no barrier
  // runs two phases ahead of a compute warp's wait.  id_full goes by unit
  // parity, staged by unit index mod 4 (a unit's store waits for K(L+3), by
  // which time at most three later units can have staged theirs).
  static constexpr int kBars = 4 + 2 * kKStages + kVStages + 15;
  // readers of a unit id: the MMA warp, the eight compute warps, the dO loader
  static constexpr uint32_t kIdReaders = 10;
  static constexpr uint32_t kMiscOff = kBarOff + kBars * 8;   // tmem holder, abort flag, unit ids [2]
  static constexpr uint32_t kRespOff = (kMiscOff + 16 + 15) / 16 * 16;   // 16-byte work-steal response
  static constexpr uint32_t kLayoutBytes = kRespOff + 16;
  static constexpr uint32_t kMaxSmem = BwdCfg<D>::kMaxSmem;
  static constexpr uint32_t kSmemBytes = kLayoutBytes + 1024 <= kMaxSmem ? kLayoutBytes + 1024 : kMaxSmem;
  static_assert(kLayoutBytes <= kMaxSmem, "dQ shared-memory layout too large");
  static constexpr int kThreads = 384;
  static constexpr int kRequestAhead = 5;   // key tiles before a unit's end at which the next is requested
  // TMEM: S double-buffered (tile j in buffer j & 1), dP, dQ accumulator.  S(j+1)
  // never overwrites the S the compute warps are reading, and S(j+2) is issued
  // only after the MMA warp has seen dS(j) (so S(j) was read long before): no
  // "S read" barrier is needed.
  static constexpr uint32_t kColS0 = 0, kColDP = 128, kColAcc = 256, kColS1 = 384;
  static_assert(kColAcc + D <= kColS1, "TMEM layout");
  __host__ __device__ static constexpr uint32_t col_s(int j) { return (j & 1) ? kColS1 : kColS0; }
  __host__ __device__ static constexpr uint32_t k_off(int s) { return kKOff + s * kTileBytes; }
  __host__ __device__ static constexpr uint32_t v_off(int s) { return kVOff + s * kTileBytes; }
};

// Work unit u (a CTA index of the launch grid) -> head and query tile.
struct DqUnit {
  int bh, qt, cnt;
};
template <bool CAUSAL>
__device__ __forceinline__ DqUnit dq_unit(int u, int n_tiles, int BH, int band) {
  DqUnit w;
  int rank;
  banded_order(u, n_tiles, BH, band, w.bh, rank);
  w.qt = n_tiles - 1 - rank;                 // causal: large qt is heavy, rank 0 first
  w.cnt = CAUSAL ? w.qt + 1 : n_tiles;       // key tiles visited
  return w;
}

// A compute thread's row terms for unit u: -lse * log2(e) and -D of its query row.
template <bool CAUSAL>
__device__ __forceinline__ float2 dq_row_terms(int u, int n_tiles, int BH, int band, int N, int r,
                                               const float* __restrict__ lse, const float* __restrict__ Dg) {
  const DqUnit w = dq_unit<CAUSAL>(u, n_tiles, BH, band);
  const int row = 128 * w.qt + r;
  float2 t = make_float2(-INFINITY, 0.f);
  if (row < N) {
    const size_t idx = static_cast<size_t>(w.bh) * N + row;
    const float l = lse[idx];
    t.x = (l == -INFINITY) ? -INFINITY : -l * kLog2e;
    t.y = -Dg[idx];
  }
  return t;
}

template <int D, bool CAUSAL, bool DROPOUT, bool FD>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                     const __grid_constant__ CUtensorMap tmDQ, const float* __restrict__ lse,
                     const float* __restrict__ Dg, int N, int n_tiles, int BH, int H, int band, float scale,
                     float scale_log2, int ks, uint32_t idesc_acc, const __grid_constant__ DropArgs drop,
                     const WaitCfg wc) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (static_cast<uint32_t>(smem - smem_raw) + C::kLayoutBytes > C::kSmemBytes) {
    // the aligned layout does not fit this launch's shared memory: report, touch nothing
    if (threadIdx.x == 0) atomicCAS(&g_status_bwd[0], 0u, kSiteDq | 0xFFu);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* do_full = bars + 2;
  uint64_t* do_empty = bars + 3;
  uint64_t* k_full = bars + 4;
  uint64_t* k_empty = k_full + C::kKStages;
  uint64_t* v_full = k_empty + C::kKStages;
  uint64_t* s_full = v_full + C::kVStages;
  uint64_t* dp_full = s_full + 2;   // s_full[2], by S buffer
  uint64_t* ds_full = dp_full + 1;
  uint64_t* acc_done = ds_full + 1;
  uint64_t* acc_free = acc_done + 1;
  uint64_t* drain = acc_free + 1;
  uint64_t* sched = drain + 1;
  uint64_t* id_taken = sched + 1;
  uint64_t* id_full = id_taken + 1;   // [2], by unit parity
  uint64_t* staged = id_full + 2;     // [4], by unit index mod 4
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff + 4);
  // Unit ids, by unit parity.  The producer publishes unit k+1's id (id_full)
  // only after every reader has taken unit k's (id_taken), so no id is
  // overwritten unread and no id_full phase runs two ahead of a reader.
  volatile int* unit_id = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 8);
  uint8_t* resp = smem + C::kRespOff;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(do_full, 1);
    mbar_init(do_empty, 1);
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < C::kVStages; ++i) mbar_init(&v_full[i], 1);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 256);
    mbar_init(acc_done, 1);
    mbar_init(acc_free, 256);
    mbar_init(drain, 1);
    mbar_init(sched, 1);
    mbar_init(id_taken, C::kIdReaders);
    for (int i = 0; i < 2; ++i) mbar_init(&id_full[i], 1);
    for (int i = 0; i < 4; ++i) mbar_init(&staged[i], 256);
    unit_id[0] = static_cast<int>(blockIdx.x);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const CtaGuard g{abort_flag, g_status_bwd, wc.epoch, wc.limit_us};
  const uint32_t sbase = smem_u32(smem);
  auto kpar = [](int j) { return static_cast<uint32_t>((j / C::kKStages) & 1); };
  auto vpar = [](int j) { return static_cast<uint32_t>((j / C::kVStages) & 1); };

  if (warp >= 8) {
    if (warp == 8) {  // producer: unit ids; per unit Q_i; K_j and V_j through their rings; dQ stores
      if (lane == 0) {
        // Pending dQ stores, oldest first (a ring of 4, by unit index): unit p
        // ended at key tile last[p & 3] and staged dQ in that tile's K slot,
        // which K(last + 3) reuses; the store goes out just before that load.
        int pend_bh[4] = {}, pend_qt[4] = {}, pend_last[4] = {};
        int pend_head = 0, pend_tail = 0;   // unit indices: [head, tail) pending
        auto store_front = [&]() -> bool {
          const int p = pend_head & 3;
          if (!mbar_wait(&staged[p], (pend_head >> 2) & 1, g, kSiteDq | 18u)) return false;
          const HeadCoord phc = head_coord(pend_bh[p], H);
          for (int b = 0; b < BwdCfg<D>::kBoxes; ++b)
            tma_store_hd(&tmDQ, smem + C::k_off(pend_last[p] % C::kKStages) + b * BwdCfg<D>::kBoxBytes, 64 * b,
                         128 * pend_qt[p], phc);
          tma_store_commit();
          tma_store_wait_read_all();
          ++pend_head;
          return true;
        };
        mbar_arrive(&id_full[0]);   // unit 0: this CTA's own (its id was written before the start)
        int u = static_cast<int>(blockIdx.x);
        int gk = 0;   // global key-tile count (ring index)
        bool ok = true;
        for (int su = 0; ok; ++su) {
          const DqUnit w = dq_unit<CAUSAL>(u, n_tiles, BH, band);
          const HeadCoord hc = head_coord(w.bh, H);
          // Q_i: the previous unit's last S product has read the buffer
          if (su > 0 && !(ok = mbar_wait(q_empty, (su - 1) & 1, g, kSiteDq | 14u))) break;
          mbar_arrive_expect_tx(q_full, C::kTileBytes);
          for (int b = 0; b < BwdCfg<D>::kBoxes; ++b)
            tma_load_hd(smem + C::kQOff + b * BwdCfg<D>::kBoxBytes, &tmQ, q_full, 64 * b, 128 * w.qt, hc);
          for (int it = 0; it < w.cnt; ++it, ++gk) {
            const int ks = gk % C::kKStages, vs = gk % C::kVStages;
            if (it == max(0, w.cnt - C::kRequestAhead)) {   // ask for the next unit
              mbar_arrive_expect_tx(sched, 16);
              clc_try_cancel(resp, sched);
            }
            if (!(ok = mbar_wait(&k_empty[ks], kpar(gk) ^ 1u, g, kSiteDq | 1u))) break;
            // a unit that ended at key tile gk - 3 staged its dQ in this slot
            if (pend_head < pend_tail && pend_last[pend_head & 3] + C::kKStages == gk && !(ok = store_front())) break;
            mbar_arrive_expect_tx(&k_full[ks], C::kTileBytes);
            for (int b = 0; b < BwdCfg<D>::kBoxes; ++b)
              tma_load_hd(smem + C::k_off(ks) + b * BwdCfg<D>::kBoxBytes, &tmK, &k_full[ks], 64 * b, 128 * it,
                          hc);
            // V slot reuse: the dQ of key tile gk - 2 (issued after that tile's
            // dP) has completed, which its k_empty commit signals
            if (gk >= C::kVStages &&
                !(ok = mbar_wait(&k_empty[(gk - C::kVStages) % C::kKStages], kpar(gk - C::kVStages), g,
                                 kSiteDq | 11u)))
              break;
            mbar_arrive_expect_tx(&v_full[vs], C::kTileBytes);
            for (int b = 0; b < BwdCfg<D>::kBoxes; ++b)
              tma_load_hd(smem + C::v_off(vs) + b * BwdCfg<D>::kBoxBytes, &tmV, &v_full[vs], 64 * b, 128 * it,
                          hc);
          }
          if (!ok) break;
          const int p = pend_tail & 3;   // at most three older stores are still pending here
          pend_bh[p] = w.bh;
          pend_qt[p] = w.qt;
          pend_last[p] = gk - 1;
          ++pend_tail;
          if (!(ok = mbar_wait(sched, su & 1, g, kSiteDq | 13u))) break;
          u = clc_decode(resp);
          if (u >= 0) {   // the next unit's first tiles into L2 while this unit finishes
            const DqUnit w1 = dq_unit<CAUSAL>(u, n_tiles, BH, band);
            const HeadCoord hc1 = head_coord(w1.bh, H);
            for (int b = 0; b < BwdCfg<D>::kBoxes; ++b) {
              tma_prefetch_l2_hd(&tmQ, 64 * b, 128 * w1.qt, hc1);
              tma_prefetch_l2_hd(&tmDO, 64 * b, 128 * w1.qt, hc1);
              for (int t = 0; t < kL2Ahead && t < w1.cnt; ++t) {
                tma_prefetch_l2_hd(&tmK, 64 * b, 128 * t, hc1);
                tma_prefetch_l2_hd(&tmV, 64 * b, 128 * t, hc1);
              }
            }
          }
          // publish the next unit's id once every reader has taken this one's
          if (!(ok = mbar_wait(id_taken, su & 1, g, kSiteDq | 20u))) break;
          unit_id[(su + 1) & 1] = u;
          mbar_arrive(&id_full[(su + 1) & 1]);
          if (u < 0) {   // no work left: release the MMA warp with an empty Q phase
            if (mbar_wait(q_empty, su & 1, g, kSiteDq | 14u)) mbar_arrive(q_full);
            break;
          }
        }
        while (ok && pend_head < pend_tail) ok = store_front();   // the remaining stores
        tma_store_wait_all();   // every store has landed before the CTA retires
      }
    } else if (warp == 10) {  // dO loader: each unit's dO once the previous unit's last dP is done
      if (lane == 0) {
        for (int su = 0;; ++su) {
          if (!mbar_wait_backoff(&id_full[su & 1], (su >> 1) & 1, g, kSiteDq | 17u)) break;
          const int u = unit_id[su & 1];
          if (u < 0) break;
          mbar_arrive(id_taken);
          if (su > 0 && !mbar_wait_backoff(do_empty, (su - 1) & 1, g, kSiteDq | 19u)) break;
          const DqUnit w = dq_unit<CAUSAL>(u, n_tiles, BH, band);
          mbar_arrive_expect_tx(do_full, C::kTileBytes);
          for (int b = 0; b < BwdCfg<D>::kBoxes; ++b)
            tma_load_hd(smem + C::kDOOff + b * BwdCfg<D>::kBoxBytes, &tmDO, do_full, 64 * b, 128 * w.qt,
                        head_coord(w.bh, H));
        }
      }
    } else if (warp == 9) {  // MMA issuer: the whole warp runs the loop, one lane issues
      const uint32_t tDP = tmem + C::kColDP, tDQ = tmem + C::kColAcc;
      const uint64_t kQ = kmaj<D>(sbase + C::kQOff), kDO = kmaj<D>(sbase + C::kDOOff);
      // K stages as K-major B operands (S) and MN-major B operands (dQ); V stages K-major (dP)
      auto kK = [&](int s) { return kmaj<D>(sbase + C::k_off(s)); };
      auto mK = [&](int s) { return mnmaj<D>(sbase + C::k_off(s)); };
      auto kV = [&](int s) { return kmaj<D>(sbase + C::v_off(s)); };
      bool ok = true;
      int gk = 0;
      // One unit: S(0) dP(0) | S(1) dQ(0) dP(1) | ... | S(c-1) dQ(c-2) dP(c-1) | dQ(c-1).
      // The first and last tile are peeled so the steady loop carries no
      // per-unit conditions: this warp's issue time bounds the tensor core.
      for (int su = 0; ok; ++su) {
        if (!(ok = mbar_wait_w(q_full, su & 1, g, kSiteDq | 2u))) break;
        const int u = unit_id[su & 1];
        if (u < 0) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(id_taken);
        const int cnt = dq_unit<CAUSAL>(u, n_tiles, BH, band).cnt;
        const int g0 = gk;   // this unit's first global key tile
        // S(0): its K tile (its S buffer was read before the dS the previous
        // unit's last dQ waited for)
        if (!(ok = mbar_wait_w(&k_full[g0 % C::kKStages], kpar(g0), g, kSiteDq | 3u))) break;
        tc_fence_after();
        mma_nt<D, FD>(tmem + C::col_s(g0), kQ, kK(g0 % C::kKStages), ks);
        tc_commit_w(&s_full[g0 & 1]);
        if (!(ok = mbar_wait_w(&v_full[g0 % C::kVStages], vpar(g0), g, kSiteDq | 3u))) break;
        if (!(ok = mbar_wait_w(do_full, su & 1, g, kSiteDq | 19u))) break;
        mma_nt<D, FD>(tDP, kDO, kV(g0 % C::kVStages), ks);
        tc_commit_w(dp_full);
        if (cnt == 1) tc_commit_w(do_empty);   // dO_i: last reader issued
        for (int it = 0; it < cnt; ++it) {
          const int j = g0 + it;   // global index of key tile it
          const uint32_t par = j & 1;
          const bool next = it + 1 < cnt;
          if (next) {   // S(j+1), into the other S buffer
            if (!(ok = mbar_wait_w(&k_full[(j + 1) % C::kKStages], kpar(j + 1), g, kSiteDq | 4u))) break;
            tc_fence_after();
            mma_nt<D, FD>(tmem + C::col_s(j + 1), kQ, kK((j + 1) % C::kKStages), ks);
            tc_commit_w(&s_full[(j + 1) & 1]);
          } else {
            tc_commit_w(q_empty);   // every reader of Q_i has been issued
          }
          if (!(ok = mbar_wait_w(ds_full, par, g, kSiteDq | 6u))) break;
          if (it == 0) {
            // the unit's first dQ overwrites the accumulator: the previous
            // unit's epilogue must have read it out
            if (su > 0 && !(ok = mbar_wait_w(acc_free, (su - 1) & 1, g, kSiteDq | 15u))) break;
            tc_fence_after();
            mma_tn_acc<D, FD>(tDQ, tDP, mK(j % C::kKStages), false, idesc_acc);
          } else {
            tc_fence_after();
            mma_tn_acc<D, FD>(tDQ, tDP, mK(j % C::kKStages), true, idesc_acc);   // dQ += dS K_j
          }
          tc_commit_w(&k_empty[j % C::kKStages]);                 // K_j: last reader done
          if (!next) {
            tc_commit_w(acc_done);
            break;
          }
          // dP(j+1), after dQ(j) has read dS(j) from the same columns
          if (!(ok = mbar_wait_w(&v_full[(j + 1) % C::kVStages], vpar(j + 1), g, kSiteDq | 12u))) break;
          mma_nt<D, FD>(tDP, kDO, kV((j + 1) % C::kVStages), ks);
          tc_commit_w(dp_full);
          if (it + 2 == cnt) tc_commit_w(do_empty);   // dO_i: last reader issued
        }
        gk = g0 + cnt;
      }
      tc_commit_w(drain);
      mbar_drain(drain, 0);
      __syncwarp();
      tc_fence_before();
      named_bar_sync(1, 288);
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
    return;
  }

  // compute warpgroups: query row r = TMEM lane; half h owns key columns [64h, 64h+64)
  const int h = warp >> 2;
  const int r = threadIdx.x & 127;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tDP = tmem + lane_base + C::kColDP + 64 * h;
  const float2 sc2 = make_float2(scale_log2, scale_log2);
  bool ok = mbar_wait(&id_full[0], 0, g, kSiteDq | 16u);
  int u = unit_id[0];
  __syncwarp();
  if (ok && lane == 0) mbar_arrive(id_taken);
  float2 terms = dq_row_terms<CAUSAL>(u, n_tiles, BH, band, N, r, lse, Dg);
  int gk = 0;
  for (int su = 0; ok && u >= 0; ++su) {
    const DqUnit w = dq_unit<CAUSAL>(u, n_tiles, BH, band);
    const int row = 128 * w.qt + r;
    const float2 nl2 = make_float2(terms.x, terms.x), nd2 = make_float2(terms.y, terms.y);
    for (int it = 0; ok && it < w.cnt; ++it, ++gk) {
      const uint32_t par = gk & 1;
      // dropout keep words of this row against this half's 64 keys, drawn
      // before S lands: key column c in byte c % 4 of ge[c / 4]
      uint32_t ge[DROPOUT ? 16 : 1];
      if constexpr (DROPOUT) dropout_rows<4>(drop, w.bh, row, 128 * it + 64 * h, ge);
      if (!(ok = mbar_wait(&s_full[gk & 1], (gk >> 1) & 1, g, kSiteDq | 7u))) break;
      __syncwarp();
      tc_fence_after();
      const uint32_t tS = tmem + lane_base + C::col_s(gk) + 64 * h;
      uint32_t sr[2][32];
      tmem_ld32(tS, sr[0]);
      tmem_ld32(tS + 32, sr[1]);
      tmem_ld_wait(sr[0]);
      tmem_ld_fence(sr[1]);
      // keys k0 .. k0+lim-1 of this half are visible to the row
      const int k0 = 128 * it + 64 * h;
      int lim = N - k0;
      if (CAUSAL) lim = min(lim, row - k0 + 1);
      float p[64];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[c / 32][c % 32]),
                                                __uint_as_float(sr[(c + 1) / 32][(c + 1) % 32])),
                                    sc2, nl2);
        p[c] = ex2_approx(x.x);
        p[c + 1] = ex2_approx(x.y);
      }
      if (lim < 64) {  // diagonal or ragged-tail tile only
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= lim) p[c] = 0.f;
      }
      if (!(ok = mbar_wait(dp_full, par, g, kSiteDq | 8u))) break;
      __syncwarp();
      tc_fence_after();
      uint32_t dr[2][32];
      tmem_ld32(tDP, dr[0]);
      tmem_ld32(tDP + 32, dr[1]);
      tmem_ld_wait(dr[0]);
      tmem_ld_fence(dr[1]);
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float2 dr2 = make_float2(__uint_as_float(dr[c / 32][c % 32]),
                                       __uint_as_float(dr[(c + 1) / 32][(c + 1) % 32]));
        float2 dp;
        if constexpr (DROPOUT)
          dp = __ffma2_rn(keep_pair_f(dr2, ge, c), make_float2(drop.scale, drop.scale), nd2);   // M~ o dP - D
        else
          dp = __fadd2_rn(dr2, nd2);
        const float2 ds = __fmul2_rn(make_float2(p[c], p[c + 1]), dp);
        p[c] = ds.x;
        p[c + 1] = ds.y;
      }
#pragma unroll
      for (int c = 0; c < 64; c += 32) st_bf16_16cols(tDP + c / 2, p + c);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    if (!ok) break;
    // the next unit's id and row terms: their loads overlap this epilogue
    if (!(ok = mbar_wait(&id_full[(su + 1) & 1], ((su + 1) >> 1) & 1, g, kSiteDq | 16u))) break;
    const int u_next = unit_id[(su + 1) & 1];
    __syncwarp();
    if (u_next >= 0 && lane == 0) mbar_arrive(id_taken);
    if (u_next >= 0) terms = dq_row_terms<CAUSAL>(u_next, n_tiles, BH, band, N, r, lse, Dg);
    if (!(ok = mbar_wait(acc_done, su & 1, g, kSiteDq | 9u))) break;
    __syncwarp();
    tc_fence_after();
    // epilogue: both warpgroups stage dQ (x scale, bf16) in the K slot of the
    // unit's last key tile (its last reader, dQ, finished before acc_done);
    // the producer stores it with TMA before that slot is reloaded
    {
      const uint32_t stage = sbase + C::k_off((gk - 1) % C::kKStages);
#pragma unroll
      for (int c = h * (D / 2); c < (h + 1) * (D / 2); c += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + C::kColAcc + c, o);
        tmem_ld_wait(o);
        const uint32_t box = stage + (c / 64) * BwdCfg<D>::kBoxBytes + r * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = (c % 64) / 8 + q;
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[8 * q + e]) * scale;
          st_shared_v4(box + ((chunk ^ (r & 7)) << 4), pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                       pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
        }
      }
      tc_fence_before();
      mbar_arrive(acc_free);   // the accumulator may be overwritten
      fence_proxy_async_smem();
      mbar_arrive(&staged[su & 3]);
    }
    u = u_next;
  }
  __syncwarp();
  tc_fence_before();
  named_bar_sync(1, 288);
}

template <int D, bool CAUSAL, bool DROPOUT>
cudaError_t launch_dkdv_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv, const float* lse,
                          const float* Dvec, const Shape& s, const DropArgs& drop, const WaitCfg& wc,
                          cudaStream_t st) {
  using C = DkdvCfg<D>;
  auto kern = s.d == D ? fa_bwd_dkdv_kernel<D, CAUSAL, DROPOUT, true> : fa_bwd_dkdv_kernel<D, CAUSAL, DROPOUT, false>;
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads, 0);
  if (e != cudaSuccess) return e;
  const int n_tiles = (s.N + 127) / 128;
  const float scale_log2 = static_cast<float>(static_cast<double>(s.scale) * 1.4426950408889634);
  const dim3 grid(static_cast<unsigned>(s.B) * s.H * n_tiles);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, s.N, n_tiles, s.B * s.H, s.H,
                                                 head_band(s.N, s.d), s.scale, scale_log2, score_ksteps(s.d),
                                                 idesc_bf16(128, out_cols(s.d), false, true), drop, wc);
  return cudaGetLastError();
}

template <int D, bool CAUSAL, bool DROPOUT>
cudaError_t launch_dq_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tdo, const CUtensorMap& tdq, const float* lse, const float* Dvec,
                        const Shape& s, const DropArgs& drop, const WaitCfg& wc, cudaStream_t st) {
  using C = DqCfg<D>;
  auto kern = s.d == D ? fa_bwd_dq_kernel<D, CAUSAL, DROPOUT, true> : fa_bwd_dq_kernel<D, CAUSAL, DROPOUT, false>;
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads, 0);
  if (e != cudaSuccess) return e;
  const int n_tiles = (s.N + 127) / 128;
  const float scale_log2 = static_cast<float>(static_cast<double>(s.scale) * 1.4426950408889634);
  const dim3 grid(static_cast<unsigned>(s.B) * s.H * n_tiles);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tv, tdo, tdq, lse, Dvec, s.N, n_tiles, s.B * s.H, s.H,
                                                 head_band(s.N, s.d), s.scale, scale_log2, score_ksteps(s.d),
                                                 idesc_bf16(128, out_cols(s.d), false, true), drop, wc);
  return cudaGetLastError();
}


template <int D>
cudaError_t launch_dkdv_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv, const float* lse,
                          const float* Dvec, const Shape& s, const DropArgs& drop, const WaitCfg& wc,
                          cudaStream_t st) {
  if (drop.t4 != 0)
    return s.causal ? launch_dkdv_t<D, true, true>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, s, drop, wc, st)
                    : launch_dkdv_t<D, false, true>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, s, drop, wc, st);
  return s.causal ? launch_dkdv_t<D, true, false>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, s, drop, wc, st)
                  : launch_dkdv_t<D, false, false>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, s, drop, wc, st);
}

template <int D>
cudaError_t launch_dq_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tdo, const CUtensorMap& tdq, const float* lse, const float* Dvec,
                        const Shape& s, const DropArgs& drop, const WaitCfg& wc, cudaStream_t st) {
  if (drop.t4 != 0)
    return s.causal ? launch_dq_t<D, true, true>(tq, tk, tv, tdo, tdq, lse, Dvec, s, drop, wc, st)
                    : launch_dq_t<D, false, true>(tq, tk, tv, tdo, tdq, lse, Dvec, s, drop, wc, st);
  return s.causal ? launch_dq_t<D, true, false>(tq, tk, tv, tdo, tdq, lse, Dvec, s, drop, wc, st)
                  : launch_dq_t<D, false, false>(tq, tk, tv, tdo, tdq, lse, Dvec, s, drop, wc, st);
}

}  // namespace

cudaError_t launch_bwd_dkdv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const float* lse, const float* Dvec, const Shape& s, const DropArgs& drop,
                            const WaitCfg& wc, cudaStream_t st) {
  return kernel_dim(s.d) == 128 ? launch_dkdv_d<128>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, s, drop, wc, st)
                    : launch_dkdv_d<64>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, s, drop, wc, st);
}

cudaError_t launch_bwd_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq, const float* lse, const float* Dvec,
                          const Shape& s, const DropArgs& drop, const WaitCfg& wc, cudaStream_t st) {
  return kernel_dim(s.d) == 128 ? launch_dq_d<128>(tq, tk, tv, tdo, tdq, lse, Dvec, s, drop, wc, st)
                    : launch_dq_d<64>(tq, tk, tv, tdo, tdq, lse, Dvec, s, drop, wc, st);
}

cudaError_t launch_bwd_preprocess(const void* o, const Strides& so, const void* dO, const Strides& sdo, float* Dvec,
                                  const Shape& s, cudaStream_t st) {
  const long long rows = static_cast<long long>(s.B) * s.H * s.N;
  int sms = 148;
  const cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int rows_per_block = (kPreThreads / (kernel_dim(s.d) / 8)) * kPreUnroll;
  const long long want = (rows + rows_per_block - 1) / rows_per_block;
  const int grid = static_cast<int>(want < 8LL * sms ? want : 8LL * sms);
  const Strides c = contiguous_strides(s);
  const bool contig = so.b == c.b && so.h == c.h && so.n == c.n && sdo.b == c.b && sdo.h == c.h && sdo.n == c.n;
  const auto* po = static_cast<const uint8_t*>(o);
  const auto* pdo = static_cast<const uint8_t*>(dO);
  if (s.d == 256)
    fa_bwd_preprocess_kernel<256, true><<<grid, kPreThreads, 0, st>>>(po, pdo, Dvec, rows, s.H, s.N, s.d, so, sdo, contig);
  else if (kernel_dim(s.d) == 256)
    fa_bwd_preprocess_kernel<256, false><<<grid, kPreThreads, 0, st>>>(po, pdo, Dvec, rows, s.H, s.N, s.d, so, sdo,
                                                                       contig);
  else if (s.d == 128)
    fa_bwd_preprocess_kernel<128, true><<<grid, kPreThreads, 0, st>>>(po, pdo, Dvec, rows, s.H, s.N, s.d, so, sdo, contig);
  else if (s.d == 64)
    fa_bwd_preprocess_kernel<64, true><<<grid, kPreThreads, 0, st>>>(po, pdo, Dvec, rows, s.H, s.N, s.d, so, sdo, contig);
  else if (kernel_dim(s.d) == 128)
    fa_bwd_preprocess_kernel<128, false><<<grid, kPreThreads, 0, st>>>(po, pdo, Dvec, rows, s.H, s.N, s.d, so, sdo,
                                                                       contig);
  else
    fa_bwd_preprocess_kernel<64, false><<<grid, kPreThreads, 0, st>>>(po, pdo, Dvec, rows, s.H, s.N, s.d, so, sdo,
                                                                      contig);
  return cudaGetLastError();
}

// Scratch for fa_bwd_noalloc: the row term D lives here instead of in a
// caller-provided workspace.  Every GPU that loads the library holds these
// 8 MiB until the process exits; all calls share them.
static __device__ __align__(256) float g_noalloc_rows[kNoAllocRows];

// A symbol's host-side name is not a device address, and the address belongs
// to one context: it is looked up (cudaGetSymbolAddress, which allocates
// nothing) on the first call with a device current and again whenever the
// current context is not the one it was looked up in (after cudaDeviceReset,
// say, or on a thread with no context bound yet).
cudaError_t noalloc_scratch(float** out) {
  static std::mutex mu;
  static float* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || ctx == 0 || ctx_of[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_rows);   // binds the device's context if none was current
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<float*>(p);
    ctx_of[dev] = current_context_id();
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t bwd_status(uint32_t* out, bool reset) {
  unsigned int v[2] = {0, 0};
  cudaError_t e = cudaMemcpyFromSymbol(v, g_status_bwd, sizeof(v));
  if (e != cudaSuccess) return e;
  *out = v[0];
  if (reset && (v[0] | v[1]) != 0) {
    const unsigned int z[2] = {0, 0};
    e = cudaMemcpyToSymbol(g_status_bwd, z, sizeof(z));
  }
  return e;
}

}  // namespace fa
