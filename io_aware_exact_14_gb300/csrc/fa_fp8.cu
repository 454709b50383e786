// FP8 (e4m3) forward of exact attention on sm_103a, and the quantiser that
// feeds it.
//
// The pages say only that FlashAttention-3 runs the forward on FP8 tensor
// cores and reduces the quantisation error with "incoherent processing"
// ("为什么Flash Attention能将注意力计算提速数倍而不损失精度", section
// "Flash Attention 3：拥抱Hopper架构").  The contract here:
//   * e4m3 is OCP FP8 E4M3FN; conversions round to nearest even and saturate
//     to +-448 (cvt.rn.satfinite);
//   * quantisation is per (batch, head): x * (448 / amax) in fp32, and the
//     dequantisation factor (descale) is amax / 448 (1 for an all-zero head);
//   * incoherent processing rotates Q and K along d by diag(sigma) H_d /
//     sqrt(d) (Sylvester-Hadamard, random signs from Philox4x32-10), which
//     leaves Q K^T unchanged and spreads outliers before quantisation;
//   * the forward takes Q and K as [B, H, N, d] codes and V transposed,
//     [B, H, d, ldv] (ldv = N rounded up to 16), so both products read
//     K-major operands; S = scale (dq Q)(dk K)^T in fp32, the unnormalised
//     probabilities are rounded to e4m3 for O = (P V) dv / l, with l the fp32
//     sum of the unrounded ones; O is bf16, LSE fp32.
//
// GB300 design: the bf16 forward's pipeline (one CTA per SM, two 128-row
// query tiles whose softmax alternates with the other tile's products, a TMA
// producer warp, one MMA-issuing warp) with 1-byte tiles: a 128 x 128 tile is
// 128 rows of 128 bytes, one 128-byte-swizzled box, so Q, K and V^T all use
// the plain K-major descriptor, and each product is four kind::f8f6f4 MMAs
// (K = 32).  P (e4m3, four keys per 32-bit column) overwrites the first 32
// columns of its S tile in TMEM and feeds P V from there, as in the bf16
// forward (measured 2.6% faster than staging P through shared memory).
#include "fa_internal.h"
// the softmax and MMA warps change their register budgets (setmaxnreg)
#define FA_INLINE_WAITS 1
#include "fa_ptx.cuh"

#include <cmath>

namespace fa {
namespace {

__device__ unsigned int g_status_fp8[2] = {0, 0};   // status, abort epoch (see CtaGuard)
constexpr uint32_t kSiteFp8 = 0x700u;
constexpr float kRescaleThreshold8 = 8.0f;   // log2 units; P~ stays <= 256 < 448
constexpr float kLn2f = 0.6931471805599453f;
constexpr float kE4m3Max = 448.0f;

struct Fp8Cfg {
  static constexpr uint32_t kTileBytes = 128u * 128u;   // 128 rows x 128 B
  static constexpr int kSlots = 8;                      // K / V^T ring
  static constexpr int kGroups = kSlots / 2;
  // Q_t at 2t tiles, a second 16 KB right after it: the epilogue stages the
  // 128 x 128 bf16 O of tile t (two 64-column boxes, 32 KB) across both
  __host__ __device__ static constexpr uint32_t q_off(int t) { return 2u * t * kTileBytes; }
  static constexpr uint32_t kSlotOff = 4 * kTileBytes;
  static constexpr uint32_t kBarOff = kSlotOff + kSlots * kTileBytes;
  // gfull[G], release[G], q_full, s_full[2], p_full[2], o_done[2], drain, staged[2]
  static constexpr int kBars = 2 * kGroups + 10;
  static constexpr uint32_t kMiscOff = kBarOff + kBars * 8;
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;
  static constexpr int kThreads = 384;
  static constexpr uint32_t kRegsSoftmax = 216;
  static constexpr uint32_t kRegsOther = 56;
  static constexpr uint32_t kRegsNeeded = 256 * kRegsSoftmax + 128 * kRegsOther;
  __host__ __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return t ? 384u : 256u; }
};
static_assert(Fp8Cfg::kSmemBytes <= 227u * 1024u, "shared memory");

// One 128 x 128 product: four K = 32 steps, 32 bytes apart inside the
// 128-byte swizzle rows (descriptor start address is in 16-byte units).
__device__ __forceinline__ void fp8_issue(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc, bool acc) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    tc_mma_f8_ss_w(tmem_d, a_desc + 2 * kk, b_desc + 2 * kk, (acc || kk > 0) ? 1u : 0u);
}

// O (+)= P V with P in TMEM (32 keys = 8 columns per K step) and V^T in shared memory.
__device__ __forceinline__ void fp8_issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t vt_desc, bool acc) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    tc_mma_f8_ts_w(tmem_o, tmem_p + 8 * kk, vt_desc + 2 * kk, (acc || kk > 0) ? 1u : 0u);
}

struct Fp8Work {
  int bh, qt0, n0, n1, n;
  HeadCoord hc;
};

__device__ __forceinline__ Fp8Work fp8_work(int N, int n_pairs, int BH, int H, int band, bool causal) {
  Fp8Work w;
  int rank;
  banded_order(blockIdx.x, n_pairs, BH, band, w.bh, rank);
  w.hc = head_coord(w.bh, H);
  const int pair = n_pairs - 1 - rank;   // heavy (causal) pairs first
  const int n_qt = (N + 127) / 128;
  w.qt0 = 2 * pair;
  const int qt1 = w.qt0 + 1;
  w.n0 = causal ? min(w.qt0 + 1, n_qt) : n_qt;
  w.n1 = qt1 < n_qt ? (causal ? min(qt1 + 1, n_qt) : n_qt) : 0;
  w.n = max(w.n0, w.n1);
  return w;
}

// Producer (one lane): Q0 (and Q1), then K_j and V^T_j through the ring in
// groups (group 0 = K_0, group j+1 = {V^T_j, K_{j+1}}), one full barrier per group.
__device__ __forceinline__ void fp8_producer(const Fp8Work& w, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                             uint64_t* q_full, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                             const CUtensorMap* tmVt, const CtaGuard& g) {
  using C = Fp8Cfg;
  mbar_arrive_expect_tx(q_full, (w.n1 > 0 ? 2u : 1u) * C::kTileBytes);
  tma_load_hd(smem + C::q_off(0), tmQ, q_full, 0, 128 * w.qt0, w.hc);
  if (w.n1 > 0) tma_load_hd(smem + C::q_off(1), tmQ, q_full, 0, 128 * (w.qt0 + 1), w.hc);
  int issued = 0;
  bool ok = true;
  for (int j = 0; j < w.n && ok; ++j) {
    for (int kind = 0; kind < 2; ++kind) {   // K_j (group j), then V^T_j (group j+1)
      const int idx = 2 * j + kind;
      const int grp = (idx + 1) >> 1;
      if (kind == 1 || j == 0) {
        if (grp >= C::kGroups &&
            !mbar_wait(&empty[grp % C::kGroups], ((grp / C::kGroups) - 1) & 1u, g, kSiteFp8 | 1u)) {
          ok = false;
          break;
        }
        const bool pair = grp > 0 && grp < w.n;   // group n holds V^T_{n-1} alone
        mbar_arrive_expect_tx(&full[grp % C::kGroups], (pair ? 2u : 1u) * C::kTileBytes);
      }
      uint8_t* dst = smem + C::kSlotOff + (idx % C::kSlots) * C::kTileBytes;
      if (kind == 0)
        tma_load_hd(dst, tmK, &full[grp % C::kGroups], 0, 128 * j, w.hc);        // keys 128j.. x d
      else
        tma_load_hd(dst, tmVt, &full[grp % C::kGroups], 128 * j, 0, w.hc);       // d x keys 128j..
      issued = idx + 1;
    }
  }
  if (!ok) {   // unwinding: let issued copies land before shared memory is released (bounded waits)
    mbar_drain(q_full, 0);
    for (int q = max(0, ((issued + 1) >> 1) - C::kGroups); q <= (issued >> 1); ++q)
      if (2 * q - 1 < issued || q == 0) mbar_drain(&full[q % C::kGroups], (q / C::kGroups) & 1);
  }
}

// One issuing warp for both tiles: S0(0) S1(0) | PV0(0) S0(1) PV1(0) S1(1) | ...
// S_t = Q_t K^T: A = Q_t, B = K (both rows of 128 key/query bytes over d).
// O_t += P_t V: A = P_t in TMEM (queries x keys), B = V^T (d x keys).
__device__ __forceinline__ void fp8_mma(const Fp8Work& w, uint32_t tmem, uint32_t smem_base, uint64_t* full,
                                        uint64_t* empty, uint64_t* q_full, uint64_t* s_full, uint64_t* p_full,
                                        uint64_t* o_done, const CtaGuard& g) {
  using C = Fp8Cfg;
  const uint64_t q_desc[2] = {sdesc_sw128(smem_base + C::q_off(0), 16, 1024),
                              sdesc_sw128(smem_base + C::q_off(1), 16, 1024)};
  const uint64_t slot0 = sdesc_sw128(smem_base + C::kSlotOff, 16, 1024);
  auto slot_off = [&](int idx) { return static_cast<uint64_t>((idx % C::kSlots) * (C::kTileBytes >> 4)); };
  auto group_wait = [&](int grp) {
    return mbar_wait_w(&full[grp % C::kGroups], (grp / C::kGroups) & 1, g, kSiteFp8 | 2u);
  };
  if (!mbar_wait_w(q_full, 0, g, kSiteFp8 | 3u)) return;
  if (!group_wait(0)) return;
  if (w.n0 > 0) {
    fp8_issue(tmem + C::col_s(0), q_desc[0], slot0 + slot_off(0), false);
    tc_commit_w(&s_full[0]);
  }
  if (w.n1 > 0) {
    fp8_issue(tmem + C::col_s(1), q_desc[1], slot0 + slot_off(0), false);
    tc_commit_w(&s_full[1]);
  }
  tc_commit_w(&empty[0]);
  for (int j = 0; j < w.n; ++j) {
    const int iv = 2 * j + 1, ik = 2 * j + 2;
    const bool next = j + 1 < w.n;
    if (!group_wait(j + 1)) return;
    const uint64_t vd = slot0 + slot_off(iv), kd = slot0 + slot_off(ik);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int n_t = t ? w.n1 : w.n0;
      if (j < n_t) {
        if (!mbar_wait_w(&p_full[t], j & 1, g, kSiteFp8 | (4u + t))) return;
        tc_fence_after();
        fp8_issue_pv(tmem + C::col_o(t), tmem + C::col_s(t), vd, j > 0);
        if (next && j + 1 < n_t) fp8_issue(tmem + C::col_s(t), q_desc[t], kd, false);
        if (j == n_t - 1) tc_commit_w(&o_done[t]);
        if (next && j + 1 < n_t) tc_commit_w(&s_full[t]);
      }
    }
    tc_commit_w(&empty[(j + 1) % C::kGroups]);
  }
}

// Softmax of one query tile (thread = query row = TMEM lane).  scale_log2
// already carries dq * dk; P~ goes back to TMEM as e4m3 (the first 32
// columns of the row's S); O is scaled by dv / l at the end.
template <bool CAUSAL>
__device__ __forceinline__ void fp8_softmax(const Fp8Work& w, int tile, uint32_t tmem, uint8_t* smem,
                                            uint64_t* s_full, uint64_t* p_full, uint64_t* o_done, uint64_t* staged,
                                            const CUtensorMap* tmO, float* __restrict__ lse, int N, int BH,
                                            float scale_log2, float out_mult, const CtaGuard& g) {
  using C = Fp8Cfg;
  const int n_i = tile ? w.n1 : w.n0;
  if (n_i == 0) return;
  const int r = threadIdx.x & 127;
  const int qt = w.qt0 + tile;
  const int row = qt * 128 + r;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) * 32u << 16;
  const uint32_t tS = tmem + lane_base + C::col_s(tile);
  const uint32_t tO = tmem + lane_base + C::col_o(tile);
  float m_use = -INFINITY;
  float l = 0.f;
  for (int j = 0; j < n_i; ++j) {
    if (!mbar_wait(&s_full[tile], j & 1, g, kSiteFp8 | 6u)) return;
    __syncwarp();
    tc_fence_after();
    uint32_t s[4][32];
    tmem_ld32(tS + 0, s[0]);
    tmem_ld32(tS + 32, s[1]);
    tmem_ld32(tS + 64, s[2]);
    tmem_ld32(tS + 96, s[3]);
    tmem_ld_wait(s[0]);
    tmem_ld_fence(s[1]);
    tmem_ld_fence(s[2]);
    tmem_ld_fence(s[3]);
    const int kv0 = j * 128;
    int lim = N - kv0;
    if (CAUSAL) lim = min(lim, row - kv0 + 1);
    if (lim < 128) {
#pragma unroll
      for (int c = 0; c < 128; ++c)
        if (c >= lim) s[c / 32][c % 32] = __float_as_uint(-INFINITY);
    }
    float mx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
    for (int c = 0; c < 128; c += 2)
      mx[(c / 2) % 8] = max3f(mx[(c / 2) % 8], __uint_as_float(s[c / 32][c % 32]),
                              __uint_as_float(s[(c + 1) / 32][(c + 1) % 32]));
    const float row_max =
        fmaxf(max3f(mx[0], mx[1], mx[2]), max3f(max3f(mx[3], mx[4], mx[5]), mx[6], mx[7])) * scale_log2;
    if (j == 0) {
      m_use = row_max;
    } else {
      const bool need = row_max > m_use + kRescaleThreshold8;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? row_max : m_use;
        const float corr = (m_use == -INFINITY) ? 0.f : ex2_approx(m_use - m_new);
        l *= corr;
        m_use = m_new;
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
          tmem_st32(tO + c, o);
        }
        tmem_st_wait();
      }
    }
    __syncwarp();
    const float m_off = (m_use == -INFINITY) ? 0.f : m_use;
    const float2 sc2 = make_float2(scale_log2, scale_log2), mo2 = make_float2(-m_off, -m_off);
    float2 sum[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sum[i] = make_float2(0.f, 0.f);
    uint32_t pk[32];   // P~ as e4m3, four keys per word, into the first 32 columns of S
#pragma unroll
    for (int q = 0; q < 8; ++q) {   // 16 keys at a time
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        const int c = 16 * q + e;
        const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(s[c / 32][c % 32]),
                                                 __uint_as_float(s[(c + 1) / 32][(c + 1) % 32])),
                                     sc2, mo2);
        const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(s[(c + 2) / 32][(c + 2) % 32]),
                                                 __uint_as_float(s[(c + 3) / 32][(c + 3) % 32])),
                                     sc2, mo2);
        const float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
        const float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
        sum[(c / 4) % 4] = __fadd2_rn(sum[(c / 4) % 4], __fadd2_rn(p0, p1));
        pk[4 * q + e / 4] = e4m3x4(p0.x, p0.y, p1.x, p1.y);
      }
    }
    tmem_st32(tS, pk);
    const float2 s01 = __fadd2_rn(sum[0], sum[1]), s23 = __fadd2_rn(sum[2], sum[3]);
    const float2 s0123 = __fadd2_rn(s01, s23);
    l += s0123.x + s0123.y;
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&p_full[tile]);
  }

  // epilogue: O = acc * dv / l -> bf16 -> swizzled staging across Q_t and P_t -> TMA store
  if (!mbar_wait(&o_done[tile], 0, g, kSiteFp8 | 7u)) return;
  __syncwarp();
  tc_fence_after();
  const float mult = l > 0.f ? out_mult / l : 0.f;
  const uint32_t stage = smem_u32(smem + C::q_off(tile));
#pragma unroll
  for (int c = 0; c < 128; c += 32) {
    uint32_t o[32];
    tmem_ld32(tO + c, o);
    tmem_ld_wait(o);
    const uint32_t box = stage + (c / 64) * C::kTileBytes + r * 128;
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
  mbar_arrive(&staged[tile]);
  if (r == 0 && mbar_wait(&staged[tile], 0, g, kSiteFp8 | 8u)) {
    tma_store_hd(tmO, smem + C::q_off(tile), 0, qt * 128, w.hc);
    tma_store_hd(tmO, smem + C::q_off(tile) + C::kTileBytes, 64, qt * 128, w.hc);
    tma_store_commit();
    tma_store_wait_read_all();
  }
  if (row < N)
    lse[static_cast<size_t>(w.bh) * N + row] = l > 0.f ? (m_use + __log2f(l)) * kLn2f : -INFINITY;
}

template <bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmVt, const __grid_constant__ CUtensorMap tmO,
                      const float* __restrict__ dq, const float* __restrict__ dk, const float* __restrict__ dv,
                      float* __restrict__ lse, int N, int n_pairs, int BH, int H, int band, float scale_log2,
                      const WaitCfg wc) {
  using C = Fp8Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kGroups;
  uint64_t* q_full = empty + C::kGroups;
  uint64_t* s_full = q_full + 1;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 2;
  uint64_t* staged = drain + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Fp8Work w = fp8_work(N, n_pairs, BH, H, band, CAUSAL);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kGroups; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
      mbar_init(&staged[i], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
    tma_prefetch_desc(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const CtaGuard g{abort_flag, g_status_fp8, wc.epoch, wc.limit_us};

  if (warp >= 8) {
    regs_dec<C::kRegsOther>();
    if (warp == 8) {
      if (lane == 0) fp8_producer(w, smem, full, empty, q_full, &tmQ, &tmK, &tmVt, g);
    } else if (warp == 9) {
      fp8_mma(w, tmem, smem_u32(smem), full, empty, q_full, s_full, p_full, o_done, g);
      tc_commit_w(drain);   // every MMA issued above has finished before TMEM is released
      mbar_drain(drain, 0);
      __syncwarp();
      tc_fence_before();
      named_bar_sync(1, 256 + 32);
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
  } else {
    regs_inc<C::kRegsSoftmax>();
    const float sl = scale_log2 * dq[w.bh] * dk[w.bh];
    fp8_softmax<CAUSAL>(w, warp >> 2, tmem, smem, s_full, p_full, o_done, staged, &tmO, lse, N, BH, sl, dv[w.bh],
                        g);
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, 256 + 32);
  }
}

// ---------------------------------------------------------------------------
// Quantiser: per-(b, h) amax, then codes, then descale = amax / 448.  A row's
// d elements are held by d/8 consecutive lanes (8 each, 16-byte loads); the
// optional rotation is the Walsh-Hadamard butterfly (a, b) -> (a + b, a - b)
// with strides 1, 2, 4 inside a thread and 8, 16, ... across lanes, on
// sign-flipped inputs, then x 1/sqrt(d).  Every step is an explicit fp32
// operation (no contraction), so the codes are an exact function of x.
// ---------------------------------------------------------------------------

constexpr int kQThreads = 256;

struct QuantArgs {
  DropArgs key;     // Philox round keys of the rotation's signs (seed)
  float inv_sqrt_d;
  int rotate;
};

// A row's 8 bf16 values of lane `sub` as raw bits (0 past d), and their fp32
// values.  Callers load all rows of a tile first, so the loads are in flight
// together before the rotations' shuffles.
__device__ __forceinline__ uint4 load_raw8(const uint8_t* __restrict__ x, long long row, int d, int sub) {
  uint4 u = make_uint4(0u, 0u, 0u, 0u);
  if (sub * 8 < d) u = *reinterpret_cast<const uint4*>(x + (static_cast<size_t>(row) * d + sub * 8) * 2);
  return u;
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&v)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

// The lane's 8 sign flips as a mask on its raw bf16 words (bit 15 of each
// half): flipping a bf16's sign bit before the exact widening to fp32 flips
// the fp32 value's sign, as multiplying by -1 would.
__device__ __forceinline__ uint4 sign_mask8(uint32_t signs8) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = (((signs8 >> (2 * i)) & 1u) << 15) | (((signs8 >> (2 * i + 1)) & 1u) << 31);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint4 xor4(const uint4& a, const uint4& b) {
  return make_uint4(a.x ^ b.x, a.y ^ b.y, a.z ^ b.z, a.w ^ b.w);
}

// The butterfly of one sign-flipped row, in place (all D/8 lanes of the row
// take part); the caller multiplies by 1/sqrt(d).
template <int D>
__device__ __forceinline__ void butterfly_row8(float (&v)[8], int sub) {
#pragma unroll
  for (int h = 1; h < 8; h *= 2) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int m = 1; m < D / 8; m *= 2) {   // lane partner sub ^ m holds columns 8m further on (or back)
    // the lower lane keeps v + o, the upper one o - v: o + sg v with sg = +-1
    // is exact in the product, so one fused multiply-add rounds once, as the
    // add or the subtract would
    const float sg = (sub & m) != 0 ? -1.f : 1.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
      v[i] = __fmaf_rn(v[i], sg, o);
    }
  }
}

// Columns 8 sub .. 8 sub + 7: bits of counter block sub / 16 (128 signs a
// block), word (sub % 16) / 4, byte sub % 4.
template <int D>
__device__ __forceinline__ uint32_t row_signs8(const QuantArgs& a, int sub) {
  if (!a.rotate) return 0u;
  const uint4 x = philox4x32_10(static_cast<uint32_t>(sub / 16), 0u, 0u, 0u, a.key);
  const int wi = (sub % 16) / 4;
  const uint32_t word = wi == 0 ? x.x : (wi == 1 ? x.y : (wi == 2 ? x.z : x.w));
  return (word >> (8 * (sub % 4))) & 0xFFu;
}

// Thread-block cluster helpers: a barrier over the cluster's CTAs (release /
// acquire, so shared-memory writes before it are visible after it) and a
// load from another CTA's shared memory.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(const void* local, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// The codes of one 128-row tile (rows n0 ..) of head bh with scale s: out[row,
// c], or out[(bh * d + c) * ldv + n] transposed, staged through shared memory
// so that each 16-byte store holds 16 keys of one row of V^T.  In the staging
// tile, row r's 8-byte column blocks are XOR-swizzled by (r / 16) mod 8: the
// gather reads one column of rows 16 apart, which would otherwise all fall
// in one shared-memory bank.
template <int D, bool TRANSPOSE>
__device__ __forceinline__ void quant_tile(const uint8_t* __restrict__ x, uint8_t* __restrict__ out, int bh, int n0,
                                           int N, int d, long long ldv, float s, uint4 smask,
                                           const QuantArgs& qa, uint8_t (*tile)[D + 16]) {
  constexpr int kTpr = D / 8, kRows = kQThreads / kTpr;
  const int sub = threadIdx.x % kTpr;
  uint4 raw[128 / kRows];
#pragma unroll
  for (int it = 0; it < 128 / kRows; ++it) {   // all the tile's loads go out first
    const int n = n0 + threadIdx.x / kTpr + it * kRows;
    raw[it] = load_raw8(x, static_cast<long long>(bh) * N + (n < N ? n : N - 1), d, sub);
  }
#pragma unroll
  for (int it = 0; it < 128 / kRows; ++it) {
    const int rr = threadIdx.x / kTpr + it * kRows;
    const int n = n0 + rr;
    float v[8];
    if (qa.rotate) {
      unpack8(xor4(raw[it], smask), v);
      butterfly_row8<D>(v, sub);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], qa.inv_sqrt_d);
    } else {
      unpack8(raw[it], v);
    }
    uint2 c;
    c.x = e4m3x4(__fmul_rn(v[0], s), __fmul_rn(v[1], s), __fmul_rn(v[2], s), __fmul_rn(v[3], s));
    c.y = e4m3x4(__fmul_rn(v[4], s), __fmul_rn(v[5], s), __fmul_rn(v[6], s), __fmul_rn(v[7], s));
    if (n >= N) c = make_uint2(0u, 0u);
    if constexpr (TRANSPOSE) {
      if (sub * 8 < D) *reinterpret_cast<uint2*>(&tile[rr][(sub * 8) ^ (((rr >> 4) & 7) * 8)]) = c;
    } else {
      if (n < N && sub * 8 < d) *reinterpret_cast<uint2*>(out + (static_cast<size_t>(bh) * N + n) * d + sub * 8) = c;
    }
  }
  if constexpr (TRANSPOSE) {
    __syncthreads();
    // row c of V^T gets keys n0 .. n0 + 127 (those below ldv), 16 per store
    for (int i = threadIdx.x; i < d * 8; i += kQThreads) {
      const int c = i / 8, k16 = (i % 8) * 16;
      if (n0 + k16 >= ldv) continue;
      const int cs = c ^ ((k16 >> 4) * 8);   // rows k16 .. k16 + 15 share one swizzle
      uint32_t wv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        wv[q] = tile[k16 + 4 * q][cs] | (tile[k16 + 4 * q + 1][cs] << 8) | (tile[k16 + 4 * q + 2][cs] << 16) |
                (static_cast<uint32_t>(tile[k16 + 4 * q + 3][cs]) << 24);
      *reinterpret_cast<uint4*>(out + (static_cast<size_t>(bh) * d + c) * ldv + n0 + k16) =
          make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
    __syncthreads();
  }
}

// One cluster of kQCluster CTAs per head (b, h): CTA r takes the head's
// 128-row tiles r * per, .. (per = ceil(tiles / kQCluster)).  Pass 1: each CTA
// reduces max |x| (after the optional rotation) over its rows; the cluster
// combines the partial maxima through distributed shared memory.  Pass 2:
// each CTA reads its rows again -- L2 hits, since only the heads of the
// clusters in flight (about SMs / kQCluster of them) are being read -- and
// writes their codes with s = 448 / amax; rank 0 writes descale = amax / 448
// (1 for an all-zero head).  One launch, each input byte read once from HBM.
constexpr int kQCluster = 8;

template <int D, bool TRANSPOSE>
__global__ void __launch_bounds__(kQThreads) fa_fp8_quant_cluster_kernel(const uint8_t* __restrict__ x,
                                                                        uint8_t* __restrict__ out,
                                                                        float* __restrict__ descale, int N, int d,
                                                                        long long ldv, QuantArgs qa) {
  constexpr int kTpr = D / 8, kRows = kQThreads / kTpr;
  __shared__ __align__(16) uint8_t tile[128][D + 16];   // transposed path: 128 rows (keys) x d codes
  __shared__ float wmax[kQThreads / 32];
  __shared__ float cta_max;
  const int bh = static_cast<int>(blockIdx.x / kQCluster);
  const int rank = static_cast<int>(blockIdx.x % kQCluster);   // the CTA's rank in its cluster (clusters along x)
  const int sub = threadIdx.x % kTpr;
  const uint4 smask = sign_mask8(row_signs8<D>(qa, sub));
  const int n_tiles = (N + 127) / 128;
  const int per = (n_tiles + kQCluster - 1) / kQCluster;
  const int t0 = rank * per, t1 = min(n_tiles, t0 + per);
  float m = 0.f;
  for (int t = t0; t < t1; ++t) {
    uint4 raw[128 / kRows];
#pragma unroll
    for (int it = 0; it < 128 / kRows; ++it) {   // all the tile's loads go out first
      const int n = t * 128 + threadIdx.x / kTpr + it * kRows;
      raw[it] = load_raw8(x, static_cast<long long>(bh) * N + (n < N ? n : N - 1), d, sub);
    }
#pragma unroll
    for (int it = 0; it < 128 / kRows; ++it) {
      const int n = t * 128 + threadIdx.x / kTpr + it * kRows;
      float v[8];
      if (qa.rotate) {   // (the 1/sqrt(d) factor is applied to the maximum below)
        unpack8(xor4(raw[it], smask), v);
        butterfly_row8<D>(v, sub);
      } else {
        unpack8(raw[it], v);
      }
      if (n < N) {
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
      }
    }
  }
  // rounding a product with a positive constant is monotone and odd, so the
  // largest |fl(v c)| is fl(c max |v|): one multiply instead of one per value
  if (qa.rotate) m = __fmul_rn(m, qa.inv_sqrt_d);
#pragma unroll
  for (int o = 16; o > 0; o /= 2) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float c = 0.f;
#pragma unroll
    for (int i = 0; i < kQThreads / 32; ++i) c = fmaxf(c, wmax[i]);
    cta_max = c;
  }
  cluster_sync();   // every CTA's partial maximum is written
  float am = 0.f;
#pragma unroll
  for (int r = 0; r < kQCluster; ++r) am = fmaxf(am, ld_cluster_f32(&cta_max, static_cast<uint32_t>(r)));
  cluster_sync();   // no CTA leaves while another may still read its partial
  if (rank == 0 && threadIdx.x == 0) descale[bh] = am > 0.f ? __fdiv_rn(am, kE4m3Max) : 1.f;
  const float s = am > 0.f ? __fdiv_rn(kE4m3Max, am) : 1.f;
  for (int t = t0; t < t1; ++t) quant_tile<D, TRANSPOSE>(x, out, bh, t * 128, N, d, ldv, s, smask, qa, tile);
}

template <int D>
cudaError_t launch_quant_d(const void* x, void* out, float* descale, int B, int H, int N, int d, bool transpose,
                           long long ldv, const QuantArgs& qa, cudaStream_t st) {
  const long long ctas = static_cast<long long>(B) * H * kQCluster;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kQCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const auto* xb = static_cast<const uint8_t*>(x);
  auto* ob = static_cast<uint8_t*>(out);
  return transpose ? cudaLaunchKernelEx(&cfg, fa_fp8_quant_cluster_kernel<D, true>, xb, ob, descale, N, d, ldv, qa)
                   : cudaLaunchKernelEx(&cfg, fa_fp8_quant_cluster_kernel<D, false>, xb, ob, descale, N, d, ldv, qa);
}

template <bool CAUSAL>
cudaError_t launch_fwd_fp8_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                             const CUtensorMap& to, const float* dq, const float* dk, const float* dv, float* lse,
                             const Shape& s, const WaitCfg& wc, cudaStream_t st) {
  using C = Fp8Cfg;
  auto kern = fa_fwd_fp8_kernel<CAUSAL>;
  // opt-in shared memory; the softmax warpgroups' setmaxnreg split must fit the launch allocation
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads, C::kRegsNeeded);
  if (e != cudaSuccess) return e;
  const int n_qt = (s.N + 127) / 128;
  const int n_pairs = (n_qt + 1) / 2;
  const float scale_log2 = static_cast<float>(static_cast<double>(s.scale) * 1.4426950408889634);
  const dim3 grid(static_cast<unsigned>(s.B) * s.H * n_pairs);
  // L2 band: e4m3 K and V of a head take 2 N d bytes
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tvt, to, dq, dk, dv, lse, s.N, n_pairs, s.B * s.H, s.H,
                                                 head_band(s.N, (s.d + 1) / 2), scale_log2, wc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_quantize(const void* x, void* out, float* descale, const Shape& s, bool transpose,
                                long long ldv, bool rotate, uint64_t seed, cudaStream_t st) {
  QuantArgs qa;
  qa.key = make_drop_args(seed, 0, 0);
  qa.inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(s.d)));
  qa.rotate = rotate ? 1 : 0;
  switch (kernel_dim(s.d)) {
    case 256: return launch_quant_d<256>(x, out, descale, s.B, s.H, s.N, s.d, transpose, ldv, qa, st);
    case 128: return launch_quant_d<128>(x, out, descale, s.B, s.H, s.N, s.d, transpose, ldv, qa, st);
    default: return launch_quant_d<64>(x, out, descale, s.B, s.H, s.N, s.d, transpose, ldv, qa, st);
  }
}

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const CUtensorMap& to, const float* dq, const float* dk, const float* dv, float* lse,
                           const Shape& s, const WaitCfg& wc, cudaStream_t st) {
  return s.causal ? launch_fwd_fp8_t<true>(tq, tk, tvt, to, dq, dk, dv, lse, s, wc, st)
                  : launch_fwd_fp8_t<false>(tq, tk, tvt, to, dq, dk, dv, lse, s, wc, st);
}

cudaError_t fp8_status(uint32_t* out, bool reset) {
  unsigned int v[2] = {0, 0};
  cudaError_t e = cudaMemcpyFromSymbol(v, g_status_fp8, sizeof(v));
  if (e != cudaSuccess) return e;
  *out = v[0];
  if (reset && (v[0] | v[1]) != 0) {
    const unsigned int z[2] = {0, 0};
    e = cudaMemcpyToSymbol(g_status_fp8, z, sizeof(z));
  }
  return e;
}

}  // namespace fa
