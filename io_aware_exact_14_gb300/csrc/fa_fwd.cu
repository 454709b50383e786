// Forward pass of exact attention on sm_103a: tiled over 128-row query tiles
// and 128-key tiles with running softmax statistics, so the N x N score and
// probability matrices never leave the SM.
//
// Method (cited by page title and section):
//   * tiling with the query tile held on chip and K/V tiles streamed in the
//     inner loop: "FlashAttention的Triton实现：IO-aware注意力机制底层原理",
//     sections "分块策略：SRAM容量限制下的精打细算" and "FA1 vs FA2：循环顺序的工程权衡";
//   * the running (m, l, acc) update and final division by l:
//     "为什么Flash Attention能将注意力计算提速数倍而不损失精度", section
//     "在线Softmax技巧" (two-block merge), and "GPU Kernel 入门：Triton /
//     FlashAttention", section "FlashAttention 与在线 softmax：难点与解法";
//   * one fused kernel (scores -> mask -> softmax -> PV, one read of Q/K/V, one
//     write of O): same page, section "核函数融合（Kernel Fusion）";
//   * asynchronous tensor cores fed by TMA with a producer/consumer pipeline
//     and two query tiles whose softmax alternates with the other tile's
//     matrix products: same page, section "Flash Attention 3：拥抱Hopper架构".
//
// GB300 design (one CTA per SM, 384 threads = 3 warpgroups):
//   warps 0-3  softmax for query tile 0 (thread = query row = TMEM lane)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q0/Q1 once, then K_j, V_j through a ring of slots
//              (tiles grouped per key step, one barrier per group)
//   warp  9    TMEM owner and tcgen05.mma issuer (elect.sync in a converged warp)
//   warp  10   second issuer for long rows (d = 128): tile 1's products
//   warp  11   idle
// The third warpgroup gives registers to the softmax warpgroups (setmaxnreg):
// each softmax thread holds a full 128-score row in registers.
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [256+d,256+2d).
// P (bf16) overwrites the first 64 columns of its S tile and feeds O += P V
// straight from TMEM.  Scores live in base-2 units: x = s * scale * log2(e).
//
// Lazy rescaling: the merge identity holds for any common reference value, so
// a row keeps its reference max until a new block exceeds it by more than
// 2^8; P values stay <= 256, and O is rescaled in TMEM only when some row of
// the warp moved its reference.  The final O = acc / l is unchanged.
#include "fa_internal.h"
// the softmax and MMA warps change their register budgets (setmaxnreg)
#define FA_INLINE_WAITS 1
#include "fa_ptx.cuh"

#include <cmath>

namespace fa {
namespace {

__device__ unsigned int g_status_fwd[2] = {0, 0};   // status, abort epoch (see CtaGuard)
constexpr int kL2Ahead = 4;   // key/value tiles the producer prefetches into L2 ahead of its loads

constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kBoxes = D / 64;                     // 128-byte boxes per row
  static constexpr uint32_t kBoxBytes = 128u * 128u;        // 128 rows x 128 B
  static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kSlots = (D == 128) ? 4 : 8;         // K/V ring
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kSlotOff = 2 * kTileBytes;
  static constexpr uint32_t kBarOff = kSlotOff + kSlots * kTileBytes;
  // Ring tiles travel in groups: group 0 is K_0, group j+1 is {V_j, K_{j+1}},
  // the tiles key step j needs beyond those it already has.  A group lands on
  // one full barrier and is released by one commit, so a key step costs the
  // issuing warp one wait and one commit for its operands; group q uses
  // gfull[q % kGroups] and release[q % kGroups].
  static constexpr int kGroups = kSlots / 2;
  // gfull[G], release[G], q_full, s_full[2], p_full[2], o_done[2], drain, staged[2]
  static constexpr int kBars = 2 * kGroups + 10;
  static constexpr uint32_t kMiscOff = kBarOff + kBars * 8;
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
  static constexpr int kThreads = 384;
  static constexpr uint32_t kRegsSoftmax = 216;  // per thread, warpgroups 0-1
  static constexpr uint32_t kRegsOther = 56;     // per thread, warpgroup 2
  static constexpr uint32_t kRegsNeeded = 256 * kRegsSoftmax + 128 * kRegsOther;

  __host__ __device__ static constexpr uint32_t col_s(int tile) { return tile ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t col_o(int tile) { return tile ? 256u + D : 256u; }
};

// A CTA's work: head bh, query tiles qt0 (and qt0 + 1 when n1 > 0), key
// tiles 0 .. n - 1 (n0 / n1 of them for tile 0 / 1).
struct FwdWork {
  int bh, qt0, n0, n1, n;
  HeadCoord hc;   // bh as (h, b) for the 4-D tensor maps
};

__device__ __forceinline__ FwdWork fwd_work(int N, int n_pairs, int BH, int H, int band, bool causal) {
  FwdWork w;
  int rank;
  banded_order(blockIdx.x, n_pairs, BH, band, w.bh, rank);
  w.hc = head_coord(w.bh, H);
  const int pair = n_pairs - 1 - rank;  // heavy (causal) pairs first
  const int n_qt = (N + 127) / 128;
  w.qt0 = 2 * pair;
  const int qt1 = w.qt0 + 1;
  w.n0 = causal ? min(w.qt0 + 1, n_qt) : n_qt;
  w.n1 = qt1 < n_qt ? (causal ? min(qt1 + 1, n_qt) : n_qt) : 0;
  w.n = max(w.n0, w.n1);
  return w;
}

template <int D>
__device__ __forceinline__ void fwd_producer(const FwdWork& w, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                             uint64_t* q_full, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                             const CUtensorMap* tmV, int withhold, const CtaGuard& g) {
  using C = FwdCfg<D>;
  mbar_arrive_expect_tx(q_full, (w.n1 > 0 ? 2u : 1u) * C::kTileBytes);
#pragma unroll
  for (int b = 0; b < C::kBoxes; ++b)
    tma_load_hd(smem + C::kQOff + b * C::kBoxBytes, tmQ, q_full, 64 * b, 128 * w.qt0, w.hc);
  if (w.n1 > 0) {
#pragma unroll
    for (int b = 0; b < C::kBoxes; ++b)
      tma_load_hd(smem + C::kQOff + C::kTileBytes + b * C::kBoxBytes, tmQ, q_full, 64 * b, 128 * (w.qt0 + 1),
                  w.hc);
  }
  int issued = 0;   // tiles whose load was issued
  bool ok = true;
  for (int j = 0; j < w.n && ok; ++j) {
    for (int kind = 0; kind < 2; ++kind) {   // K_j (group j), then V_j (group j+1)
      const int idx = 2 * j + kind;
      const int grp = (idx + 1) >> 1;
      if (kind == 1 || j == 0) {
        if (grp == withhold) {   // test hook: this group (and every later one) never arrives
          ok = false;
          break;
        }
        // first tile of its group: wait until the group that last used these
        // two slots (grp - kGroups) is released, then expect the whole group
        if (grp >= C::kGroups &&
            !mbar_wait(&empty[grp % C::kGroups], ((grp / C::kGroups) - 1) & 1u, g, kSiteFwd | 1u)) {
          ok = false;
          break;
        }
        const bool pair = grp > 0 && grp < w.n;   // group n holds V_{n-1} alone
        mbar_arrive_expect_tx(&full[grp % C::kGroups], (pair ? 2u : 1u) * C::kTileBytes);
      }
      if (j + kL2Ahead < w.n) {   // the same tile kL2Ahead steps on, into L2 while this one lands
#pragma unroll
        for (int b = 0; b < C::kBoxes; ++b)
          tma_prefetch_l2_hd(kind ? tmV : tmK, 64 * b, 128 * (j + kL2Ahead), w.hc);
      }
      uint8_t* dst = smem + C::kSlotOff + (idx % C::kSlots) * C::kTileBytes;
#pragma unroll
      for (int b = 0; b < C::kBoxes; ++b)
        tma_load_hd(dst + b * C::kBoxBytes, kind ? tmV : tmK, &full[grp % C::kGroups], 64 * b, 128 * j,
                    w.hc);
      issued = idx + 1;
    }
  }
  if (!ok) {  // unwinding: let copies already issued land before smem is released (bounded waits)
    mbar_drain(q_full, 0);
    for (int q = max(0, ((issued + 1) >> 1) - C::kGroups); q <= (issued >> 1); ++q)
      if (2 * q - 1 < issued || q == 0) mbar_drain(&full[q % C::kGroups], (q / C::kGroups) & 1);
  }
}

// Descriptor arithmetic: the start-address field is the low 14 bits of a
// descriptor (address >> 4), so advancing an operand inside shared memory is a
// plain add on the descriptor; every call site below adds compile-time
// constants to a base descriptor, keeping the issuing thread's work per MMA
// to a few instructions (the tensor core's queue is shallow, so a slow issuer
// starves it).
// The score product contracts over the true head dim: ks = ceil(d / 16) steps
// of 16 columns (the zero-filled columns past d would add nothing).  FD (d ==
// D): all D / 16 steps, a straight run of MMAs; otherwise each step's issue is
// predicated on kk < ks (a branch per MMA measured 11% slower on the
// backward kernels, the predicate alone a few percent).
template <int D, bool FD>
__device__ __forceinline__ void fwd_issue_s(uint32_t tmem_d, uint64_t q_desc, uint64_t k_desc, int ks) {
  using C = FwdCfg<D>;
  constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = ((kk / 4) * C::kBoxBytes + (kk % 4) * 32) >> 4;
    if constexpr (FD)
      tc_mma_ss_w(tmem_d, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
    else
      tc_mma_ss_w_if(tmem_d, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u, kk < ks ? 1u : 0u);
  }
}

// idesc: M = 128, N = ceil(d / 16) * 16, B (V) MN-major (a compile-time
// constant when d == D).
template <int D, bool FD>
__device__ __forceinline__ void fwd_issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t v_desc, bool acc,
                                             uint32_t idesc_rt) {
  const uint32_t idesc = FD ? idesc_bf16(128, D, false, true) : idesc_rt;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)  // 128 keys, 16 per MMA; P packs 2 keys per TMEM column
    tc_mma_ts_w(tmem_o, tmem_p + kk * 8, v_desc + ((kk * 2048) >> 4), idesc, (acc || kk > 0) ? 1u : 0u);
}

// One issuing warp per query tile (warp 9: tile 0, warp 10: tile 1), so the
// waits, commits and issue of the two tiles' products proceed side by side;
// each warp issues S_t(0) | PV_t(0) S_t(1) | PV_t(1) S_t(2) | ... and the
// tensor core interleaves the two streams, so one tile's products run while
// the other tile's softmax works.  Both warps walk every key step (a tile
// with fewer steps just stops issuing) and both release each K/V slot.
// Runs converged: waits and descriptors are warp-uniform and `elect.sync`
// picks the issuing lane inside each MMA and commit.
template <int D, bool FD>
__device__ __forceinline__ void fwd_mma(const FwdWork& w, int tile, uint32_t tmem, uint32_t smem_base,
                                        uint64_t* full, uint64_t* empty, uint64_t* q_full, uint64_t* s_full,
                                        uint64_t* p_full, uint64_t* o_done, int ks, uint32_t idesc_pv,
                                        const CtaGuard& g) {
  using C = FwdCfg<D>;
  const int n_t = tile ? w.n1 : w.n0;
  const uint64_t q_desc = sdesc_sw128(smem_base + C::kQOff + tile * C::kTileBytes, 16, 1024);
  // K-major (S = Q K^T) and MN-major (O += P V) descriptors of ring slot 0;
  // slot s is `s * kTileBytes` further on
  const uint64_t k_desc0 = sdesc_sw128(smem_base + C::kSlotOff, 16, 1024);
  const uint64_t v_desc0 = sdesc_sw128(smem_base + C::kSlotOff, C::kBoxBytes, 1024);
  const uint32_t t_s = tmem + C::col_s(tile), t_o = tmem + C::col_o(tile);
  auto slot_off = [&](int idx) { return static_cast<uint64_t>((idx % C::kSlots) * (C::kTileBytes >> 4)); };
  auto group_wait = [&](int grp) {   // group 0: K_0; group j+1: V_j and K_{j+1}
    return mbar_wait_w(&full[grp % C::kGroups], (grp / C::kGroups) & 1, g, kSiteFwd | 2u);
  };
  if (!mbar_wait_w(q_full, 0, g, kSiteFwd | 3u)) return;
  if (!group_wait(0)) return;
  if (n_t > 0) {
    fwd_issue_s<D, FD>(t_s, q_desc, k_desc0 + slot_off(0), ks);
    tc_commit_w(&s_full[tile]);
  }
  tc_commit_w(&empty[0]);   // group 0: K_0
  for (int j = 0; j < w.n; ++j) {
    const int iv = 2 * j + 1, ik = 2 * j + 2;   // ring indices of V_j and K_{j+1}
    if (!group_wait(j + 1)) return;
    if (j < n_t) {
      if (!mbar_wait_w(&p_full[tile], j & 1, g, tile ? (kSiteFwd | 5u) : (kSiteFwd | 4u))) return;
      tc_fence_after();
      fwd_issue_pv<D, FD>(t_o, t_s, v_desc0 + slot_off(iv), j > 0, idesc_pv);
      if (j + 1 < n_t) {
        fwd_issue_s<D, FD>(t_s, q_desc, k_desc0 + slot_off(ik), ks);
        tc_commit_w(&s_full[tile]);
      } else {
        tc_commit_w(&o_done[tile]);
      }
    }
    tc_commit_w(&empty[(j + 1) % C::kGroups]);   // group j+1: V_j and K_{j+1}
  }
}

// One issuing warp for both tiles (d = 64).
// Issue order S0(0) S1(0) | PV0(0) S0(1) PV1(0) S1(1) | PV0(1) ...: while one
// tile's softmax runs, the tensor core works on the other tile.  All slot
// waits of an iteration happen before the first P wait, so once P is ready a
// PV product and the next S product go out back to back.  Run by the whole
// warp: waits and descriptors are warp-uniform and `elect.sync` picks the
// issuing lane inside each MMA and commit.
template <int D, bool FD>
__device__ __forceinline__ void fwd_mma_both(const FwdWork& w, uint32_t tmem, uint32_t smem_base, uint64_t* full,
                                        uint64_t* empty, uint64_t* q_full, uint64_t* s_full, uint64_t* p_full,
                                        uint64_t* o_done, int ks, uint32_t idesc_pv, const CtaGuard& g) {
  using C = FwdCfg<D>;
  const uint64_t q_desc[2] = {sdesc_sw128(smem_base + C::kQOff, 16, 1024),
                              sdesc_sw128(smem_base + C::kQOff + C::kTileBytes, 16, 1024)};
  // K-major (S = Q K^T) and MN-major (O += P V) descriptors of ring slot 0;
  // slot s is `s * kTileBytes` further on
  const uint64_t k_desc0 = sdesc_sw128(smem_base + C::kSlotOff, 16, 1024);
  const uint64_t v_desc0 = sdesc_sw128(smem_base + C::kSlotOff, C::kBoxBytes, 1024);
  auto slot_off = [&](int idx) { return static_cast<uint64_t>((idx % C::kSlots) * (C::kTileBytes >> 4)); };
  auto group_wait = [&](int grp) {   // group 0: K_0; group j+1: V_j and K_{j+1}
    return mbar_wait_w(&full[grp % C::kGroups], (grp / C::kGroups) & 1, g, kSiteFwd | 2u);
  };
  if (!mbar_wait_w(q_full, 0, g, kSiteFwd | 3u)) return;
  if (!group_wait(0)) return;
  if (w.n0 > 0) {
    fwd_issue_s<D, FD>(tmem + C::col_s(0), q_desc[0], k_desc0 + slot_off(0), ks);
    tc_commit_w(&s_full[0]);
  }
  if (w.n1 > 0) {
    fwd_issue_s<D, FD>(tmem + C::col_s(1), q_desc[1], k_desc0 + slot_off(0), ks);
    tc_commit_w(&s_full[1]);
  }
  tc_commit_w(&empty[0]);   // group 0: K_0
  for (int j = 0; j < w.n; ++j) {
    const int iv = 2 * j + 1, ik = 2 * j + 2;
    const bool next = j + 1 < w.n;
    if (!group_wait(j + 1)) return;
    const uint64_t vd = v_desc0 + slot_off(iv), kd = k_desc0 + slot_off(ik);
    if (j < w.n0) {
      if (!mbar_wait_w(&p_full[0], j & 1, g, kSiteFwd | 4u)) return;
      tc_fence_after();
      fwd_issue_pv<D, FD>(tmem + C::col_o(0), tmem + C::col_s(0), vd, j > 0, idesc_pv);
      if (next && j + 1 < w.n0) fwd_issue_s<D, FD>(tmem + C::col_s(0), q_desc[0], kd, ks);
      if (j == w.n0 - 1) tc_commit_w(&o_done[0]);
      if (next && j + 1 < w.n0) tc_commit_w(&s_full[0]);
    }
    if (j < w.n1) {
      if (!mbar_wait_w(&p_full[1], j & 1, g, kSiteFwd | 5u)) return;
      tc_fence_after();
      fwd_issue_pv<D, FD>(tmem + C::col_o(1), tmem + C::col_s(1), vd, j > 0, idesc_pv);
      if (next && j + 1 < w.n1) fwd_issue_s<D, FD>(tmem + C::col_s(1), q_desc[1], kd, ks);
      if (j == w.n1 - 1) tc_commit_w(&o_done[1]);
      if (next && j + 1 < w.n1) tc_commit_w(&s_full[1]);
    }
    tc_commit_w(&empty[(j + 1) % C::kGroups]);   // group j+1: V_j and K_{j+1}
  }
}

// DROPOUT: the probabilities that feed O += P V are multiplied by the keep
// mask and the scale (the row sum l, hence LSE, uses the plain ones).
template <int D, bool CAUSAL, bool DROPOUT>
__device__ __forceinline__ void fwd_softmax(const FwdWork& w, int tile, uint32_t tmem, uint8_t* smem,
                                            uint64_t* s_full, uint64_t* p_full, uint64_t* o_done,
                                            uint64_t* staged, const CUtensorMap* tmO, float* __restrict__ lse, int N,
                                            float scale_log2, const DropArgs& drop, const CtaGuard& g) {
  using C = FwdCfg<D>;
  const int n_i = tile ? w.n1 : w.n0;
  if (n_i == 0) return;
  const int r = threadIdx.x & 127;                 // row within the tile = TMEM lane
  const int qt = w.qt0 + tile;
  const int row = qt * 128 + r;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) * 32u << 16;
  const uint32_t tS = tmem + lane_base + C::col_s(tile);
  const uint32_t tO = tmem + lane_base + C::col_o(tile);

  float m_use = -INFINITY;  // reference max, base-2 units
  float l = 0.f;
  for (int j = 0; j < n_i; ++j) {
    // dropout keep words of this row's 128 keys, drawn before S lands (they
    // depend only on the row and the key tile): key c in byte c % 4 of ge[c / 4]
    // (four words per register: key c in byte c % 4 of word (c / 4) % 4 of kp[c / 16])
    uint32_t kp[DROPOUT ? 8 : 1];
    if constexpr (DROPOUT) {
      uint32_t ge[32];
      dropout_rows<8>(drop, w.bh, row, j * 128, ge);
#pragma unroll
      for (int g = 0; g < 8; ++g) kp[g] = pack_keep4(ge[4 * g], ge[4 * g + 1], ge[4 * g + 2], ge[4 * g + 3]);
    }
    if (!mbar_wait(&s_full[tile], j & 1, g, kSiteFwd | 6u)) return;
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

    // keys kv0 .. kv0+lim-1 are visible to this row
    const int kv0 = j * 128;
    int lim = N - kv0;
    if (CAUSAL) lim = min(lim, row - kv0 + 1);
    if (lim < 128) {
#pragma unroll
      for (int c = 0; c < 128; ++c)
        if (c >= lim) s[c / 32][c % 32] = __float_as_uint(-INFINITY);
    }
    // row max: 3-input maxes over 8 independent chains
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
      m_use = row_max;  // O is overwritten by the first P V product
    } else {
      const bool need = row_max > m_use + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? row_max : m_use;
        const float corr = (m_use == -INFINITY) ? 0.f : ex2_approx(m_use - m_new);
        l *= corr;
        m_use = m_new;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
          tmem_st32(tO + c, o);
        }
      }
    }
    __syncwarp();
    const float m_off = (m_use == -INFINITY) ? 0.f : m_use;
    // x = s * scale * log2(e) - m and the row sums, two columns per packed instruction
    const float2 sc2 = make_float2(scale_log2, scale_log2), mo2 = make_float2(-m_off, -m_off);
    float2 sum[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sum[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // keys [64h, 64h+64) -> P columns [32h, 32h+32)
      uint32_t pk[32];
#pragma unroll
      for (int c = 64 * h; c < 64 * h + 64; c += 2) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[c / 32][c % 32]),
                                                __uint_as_float(s[(c + 1) / 32][(c + 1) % 32])),
                                    sc2, mo2);
        const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        sum[(c / 2) % 4] = __fadd2_rn(sum[(c / 2) % 4], pp);
        if constexpr (DROPOUT) {   // P o M (0/1); the 1/(1-p) scale goes into the epilogue
          pk[(c / 2) % 32] = pack_bf16x2(pp.x, pp.y) & keep_mask_pair(unpack_keep4(kp[c / 16], (c / 4) % 4), c % 4);
        } else {
          pk[(c / 2) % 32] = pack_bf16x2(pp.x, pp.y);
        }
      }
      tmem_st32(tS + 32 * h, pk);
    }
    const float2 s01 = __fadd2_rn(sum[0], sum[1]), s23 = __fadd2_rn(sum[2], sum[3]);
    const float2 s0123 = __fadd2_rn(s01, s23);
    l += s0123.x + s0123.y;
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&p_full[tile]);
  }

  // epilogue: O = acc / l -> bf16 -> swizzled staging (this tile's Q buffer) -> TMA store
  if (!mbar_wait(&o_done[tile], 0, g, kSiteFwd | 7u)) return;
  __syncwarp();
  tc_fence_after();
  const float inv_l = l > 0.f ? (DROPOUT ? drop.scale : 1.f) / l : 0.f;
  const uint32_t stage = smem_u32(smem + C::kQOff + tile * C::kTileBytes);
#pragma unroll
  for (int c = 0; c < D; c += 32) {
    uint32_t o[32];
    tmem_ld32(tO + c, o);
    tmem_ld_wait(o);
    const uint32_t box = stage + (c / 64) * C::kBoxBytes + r * 128;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int chunk = (c % 64) / 8 + q;
      float f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[8 * q + e]) * inv_l;
      st_shared_v4(box + ((chunk ^ (r & 7)) << 4), pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                   pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
    }
  }
  fence_proxy_async_smem();
  mbar_arrive(&staged[tile]);
  if (r == 0 && mbar_wait(&staged[tile], 0, g, kSiteFwd | 8u)) {
#pragma unroll
    for (int b = 0; b < C::kBoxes; ++b)
      tma_store_hd(tmO, smem + C::kQOff + tile * C::kTileBytes + b * C::kBoxBytes, 64 * b, qt * 128, w.hc);
    tma_store_commit();
    tma_store_wait_read_all();
  }
  if (row < N) lse[static_cast<size_t>(w.bh) * N + row] = l > 0.f ? (m_use + __log2f(l)) * kLn2 : -INFINITY;
}

// ISSUERS: MMA-issuing warps, 1 (warp 9 issues both tiles) or 2 (one per tile).
// DROPOUT: dropout on the probabilities (mask from `drop`, see fwd_softmax).
// FD: d == D (compile-time K steps and output width of the products).
template <int D, bool CAUSAL, int ISSUERS, bool DROPOUT, bool FD>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  float* __restrict__ lse, int N, int n_pairs, int BH, int H, int band, float scale_log2, int ks,
                  uint32_t idesc_pv, const __grid_constant__ DropArgs drop, const WaitCfg wc) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* full = bars;                   // gfull[kGroups]
  uint64_t* empty = bars + C::kGroups;     // release[kGroups]
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
  const FwdWork w = fwd_work(N, n_pairs, BH, H, band, CAUSAL);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kGroups; ++i) {
      mbar_init(&full[i], 1);          // one expect-tx arrival per group
      mbar_init(&empty[i], ISSUERS);   // one commit per issuing warp
    }
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
      mbar_init(&staged[i], 128);
    }
    mbar_init(drain, ISSUERS);   // one commit per issuing warp
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
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const CtaGuard g{abort_flag, g_status_fwd, wc.epoch, wc.limit_us};

  // Roles.  Each branch ends the kernel on its own (no shared tail), so the
  // register budget set by setmaxnreg holds for the whole branch.  The MMA
  // warp frees TMEM after every TMEM user has passed the end barrier.
  if (warp >= 8) {
    regs_dec<C::kRegsOther>();
    if (warp == 8) {
      if (lane == 0) fwd_producer<D>(w, smem, full, empty, q_full, &tmQ, &tmK, &tmV, wc.withhold, g);
    } else if (warp == 9 || (ISSUERS == 2 && warp == 10)) {
      // issuing warps (warp 9 also owns TMEM): whole-warp loops, one elected lane issues
      if (ISSUERS == 2)
        fwd_mma<D, FD>(w, warp - 9, tmem, smem_u32(smem), full, empty, q_full, s_full, p_full, o_done, ks, idesc_pv, g);
      else
        fwd_mma_both<D, FD>(w, tmem, smem_u32(smem), full, empty, q_full, s_full, p_full, o_done, ks, idesc_pv, g);
      tc_commit_w(drain);  // every MMA issued above has finished before TMEM is released
      mbar_drain(drain, 0);
      __syncwarp();
      tc_fence_before();
      named_bar_sync(1, 256 + 32 * ISSUERS);
      tc_fence_after();
      if (warp == 9) tmem_dealloc(tmem, 512);
    }
  } else {
    regs_inc<C::kRegsSoftmax>();
    fwd_softmax<D, CAUSAL, DROPOUT>(w, warp >> 2, tmem, smem, s_full, p_full, o_done, staged, &tmO, lse, N,
                                    scale_log2, drop, g);
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, 256 + 32 * ISSUERS);
  }
}

template <int D, bool CAUSAL, int ISSUERS, bool DROPOUT>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, float* lse, const Shape& s, const DropArgs& drop,
                         const WaitCfg& wc, cudaStream_t st) {
  using C = FwdCfg<D>;
  // d == D: the compile-time instantiation; two issuing warps only there
  auto kern = s.d == D ? fa_fwd_kernel<D, CAUSAL, ISSUERS, DROPOUT, true> : fa_fwd_kernel<D, CAUSAL, 1, DROPOUT, false>;
  // opt-in shared memory; the softmax warpgroups' setmaxnreg split must fit the launch allocation
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads, C::kRegsNeeded);
  if (e != cudaSuccess) return e;
  const int n_qt = (s.N + 127) / 128;
  const int n_pairs = (n_qt + 1) / 2;
  const float scale_log2 = static_cast<float>(static_cast<double>(s.scale) * 1.4426950408889634);
  const dim3 grid(static_cast<unsigned>(s.B) * s.H * n_pairs);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tv, to, lse, s.N, n_pairs, s.B * s.H, s.H,
                                                 head_band(s.N, s.d), scale_log2, score_ksteps(s.d),
                                                 idesc_bf16(128, out_cols(s.d), false, true), drop, wc);
  return cudaGetLastError();
}

// Split-KV merge: for each query row, the chunks' (O_s, LSE_s) combine by the
// two-block merge identity of [WHY-FAST] "在线Softmax技巧" applied to all
// chunks at once: LSE = log sum_s e^{LSE_s}, O = sum_s e^{LSE_s - LSE} O_s
// (each O_s is its chunk's normalised output).  HBM-bound: one warp per row,
// each lane D/32 consecutive floats of every chunk; a row whose chunks are
// all empty (or that has none) gets O = 0, LSE = -inf.
template <int D>
__global__ void __launch_bounds__(256) fa_fwd_merge_kernel(const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part,
                                                           __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                           long long rows, int n_splits, int d) {
  constexpr int kPer = D / 32;
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;   // whole warps: one row each
  float m = -INFINITY;
  for (int s = lane; s < n_splits; s += 32) m = fmaxf(m, lse_part[static_cast<long long>(s) * rows + row]);
#pragma unroll
  for (int w = 16; w > 0; w /= 2) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, w));
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (m != -INFINITY) {
    // chunks in order s = 0, 1, ...; the loads of kBatch chunks go out
    // together (independent of the sums), the sums then run in order
    constexpr int kBatch = 4;
    for (int s0 = 0; s0 < n_splits; s0 += kBatch) {
      float ls[kBatch];
      float x[kBatch][kPer];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        ls[u] = -INFINITY;
#pragma unroll
        for (int e = 0; e < kPer; ++e) x[u][e] = 0.f;
        if (s0 + u < n_splits) {
          const long long idx = static_cast<long long>(s0 + u) * rows + row;
          ls[u] = lse_part[idx];
          const float* src = o_part + idx * D + lane * kPer;
#pragma unroll
          for (int e = 0; e < kPer; e += (kPer >= 4 ? 4 : 2)) {
            if constexpr (kPer >= 4) {
              const float4 v = *reinterpret_cast<const float4*>(src + e);
              x[u][e] = v.x;
              x[u][e + 1] = v.y;
              x[u][e + 2] = v.z;
              x[u][e + 3] = v.w;
            } else {
              const float2 v = *reinterpret_cast<const float2*>(src + e);
              x[u][e] = v.x;
              x[u][e + 1] = v.y;
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (s0 + u >= n_splits) break;
        const float wgt = ls[u] == -INFINITY ? 0.f : __expf(ls[u] - m);
        wsum += wgt;
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[e] = fmaf(wgt, x[u][e], acc[e]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  // partial rows are D wide (padded with zeros); O rows are d wide
  __nv_bfloat16* dst = o + row * d + lane * kPer;
  if (lane * kPer < d) {
#pragma unroll
    for (int e = 0; e < kPer; e += 2)
      *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  }
  if (lane == 0) lse[row] = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
}

template <int D>
cudaError_t launch_merge_t(const float* o_part, const float* lse_part, void* o, float* lse, const Shape& s,
                           int n_splits, cudaStream_t st) {
  const long long rows = static_cast<long long>(s.B) * s.H * s.N;
  const long long blocks = (rows + 7) / 8;   // 8 warps (rows) per block
  fa_fwd_merge_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      o_part, lse_part, static_cast<__nv_bfloat16*>(o), lse, rows, n_splits, s.d);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_merge(const float* o_part, const float* lse_part, void* o, float* lse, const Shape& s,
                             int n_splits, int D, cudaStream_t st) {
  switch (D) {
    case 256: return launch_merge_t<256>(o_part, lse_part, o, lse, s, n_splits, st);
    case 128: return launch_merge_t<128>(o_part, lse_part, o, lse, s, n_splits, st);
    default: return launch_merge_t<64>(o_part, lse_part, o, lse, s, n_splits, st);
  }
}

cudaError_t launch_fwd_splitkv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& top, const float* o_part, float* lse_part, void* o, float* lse,
                               const Shape& s, int Nk, int n_splits, int kt_per_split, const WaitCfg& wc,
                               cudaStream_t st) {
  if (n_splits > 0) {   // the chunks: the one-query-tile kernel's split mode
    const cudaError_t e = launch_fwd_onetile_split(tq, tk, tv, top, lse_part, s, Nk, n_splits, kt_per_split, wc, st);
    if (e != cudaSuccess) return e;
  }
  return launch_fwd_merge(o_part, lse_part, o, lse, s, n_splits * splitkv_replicas(s.N, s.d, false), kernel_dim(s.d), st);
}

// Issue strategy (measured on GB300): at d = 128 one warp's issue loop (two
// tiles' waits, commits and 32 MMAs per key step) cannot keep the tensor core
// fed once CTAs run long, so long rows get one issuing warp per tile; short
// CTAs (few key steps, where prologue and epilogue weigh more) and d = 64
// (half-length products, softmax-bound) keep one issuer.
constexpr int kTwoIssuerMinSteps = 24;   // average key steps per CTA

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, float* lse, const Shape& s, const DropArgs& drop, const WaitCfg& wc,
                       cudaStream_t st) {
  if (drop.t4 != 0) {   // dropout launches keep one issuing warp
    if (kernel_dim(s.d) == 128)
      return s.causal ? launch_fwd_t<128, true, 1, true>(tq, tk, tv, to, lse, s, drop, wc, st)
                      : launch_fwd_t<128, false, 1, true>(tq, tk, tv, to, lse, s, drop, wc, st);
    return s.causal ? launch_fwd_t<64, true, 1, true>(tq, tk, tv, to, lse, s, drop, wc, st)
                    : launch_fwd_t<64, false, 1, true>(tq, tk, tv, to, lse, s, drop, wc, st);
  }
  if (kernel_dim(s.d) == 128) {
    const int n_qt = (s.N + 127) / 128;
    const int avg_steps = s.causal ? (n_qt + 1) / 2 : n_qt;
    if (avg_steps >= kTwoIssuerMinSteps)
      return s.causal ? launch_fwd_t<128, true, 2, false>(tq, tk, tv, to, lse, s, drop, wc, st)
                      : launch_fwd_t<128, false, 2, false>(tq, tk, tv, to, lse, s, drop, wc, st);
    return s.causal ? launch_fwd_t<128, true, 1, false>(tq, tk, tv, to, lse, s, drop, wc, st)
                    : launch_fwd_t<128, false, 1, false>(tq, tk, tv, to, lse, s, drop, wc, st);
  }
  return s.causal ? launch_fwd_t<64, true, 1, false>(tq, tk, tv, to, lse, s, drop, wc, st)
                  : launch_fwd_t<64, false, 1, false>(tq, tk, tv, to, lse, s, drop, wc, st);
}

cudaError_t fwd_status(uint32_t* out, bool reset) {
  unsigned int v[2] = {0, 0};
  cudaError_t e = cudaMemcpyFromSymbol(v, g_status_fwd, sizeof(v));
  if (e != cudaSuccess) return e;
  *out = v[0];
  if (reset && (v[0] | v[1]) != 0) {
    const unsigned int z[2] = {0, 0};
    e = cudaMemcpyToSymbol(g_status_fwd, z, sizeof(z));
  }
  return e;
}

}  // namespace fa
