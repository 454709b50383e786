// One-query-tile forward on sm_103a: wide heads (128 < d <= 256, kernel
// width DK = 256) and every split-KV launch (DK = 64, 128 or 256, the
// kernel width of d).  The same method as fa_fwd.cu -- query tile on chip, K/V tiles
// streamed, running (m, l, acc) with one division by l at the end
// ("为什么Flash Attention能将注意力计算提速数倍而不损失精度", sections
// "分块计算（Tiling）" and "在线Softmax技巧"; "FlashAttention的Triton实现：
// IO-aware注意力机制底层原理", section "分块策略：SRAM容量限制下的精打细算", which
// sizes the blocks from the on-chip budget and the head dim).
//
// Why a kernel of its own: at DK = 256 one query tile's O accumulator takes
// 256 of the 512 TMEM columns, so a CTA holds one query tile (not two), and a
// 128 x 256 bf16 K or V tile is 64 KB, so the ring moves d-halves.
//
// GB300 design (one CTA per SM, 192 threads):
//   warps 0-3  softmax (thread = query row = TMEM lane)
//   warp  4    TMA producer: Q once (DK / 64 boxes), then K/V "units"
//              (DK = 256: d-halves of 128 rows x 128 columns = 32 KB; else
//              whole tiles) through the ring
//   warp  5    TMEM owner and tcgen05.mma issuer (elect.sync in a converged warp)
// TMEM: S buffers [0,128) and [128,256) (key step j uses buffer j & 1, so
// S(j+1) is computed while the softmax works on S(j)); O [256, 256 + DK).
// P (bf16) overwrites the first 64 columns of its S buffer and feeds
// O += P V from TMEM, one 128-column part of O per V unit.
// Tiles stream in the order the products need them: K_0 K_1 V_0 K_2 V_1 ...
// K_{n-1} V_{n-2} V_{n-1}; each unit lands on its slot's barrier, and one
// commit per tile releases its units.
// Lazy rescaling as in fa_fwd.cu: a row keeps its reference max until a block
// exceeds it by more than 2^8; O is rescaled in TMEM only when some row of
// the warp moves, after the previous P V product has completed.
// Split-KV launches (non-causal): a CTA takes one query tile and one chunk of
// key tiles and writes the chunk's normalised O in fp32 (staged across the
// then idle Q buffer and ring) and its LSE; fa_fwd.cu's merge combines them.
// For a decode-shaped call (a few query rows against many keys) this layout
// streams K/V best: S is double-buffered, so the next tile's scores overlap
// the softmax, and the ring holds every byte shared memory leaves beside Q
// (DK = 64: 13 tiles of 16 KB; DK = 128: 6 of 32 KB; DK = 256: 5 d-halves).
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <cmath>

namespace fa {
namespace {

__device__ unsigned int g_status_fwd256[2] = {0, 0};   // status, abort epoch (see CtaGuard)

constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kSiteFwd256 = 0x400;

// DK: the kernel's head width (256 for wide heads; split-KV launches also
// run it at 64 and 128).  A K or V tile moves as kHalves units of
// kUnitBoxes 64-column boxes; the ring takes what shared memory leaves
// beside Q.  Each tile's release is one commit on empty[tile % kTileBars],
// and kTileBars * kHalves >= kSlots, so a release barrier is never reused
// before the producer has waited on it.
// F8: e4m3 Q, K and V^T (DK = 128 or 256): a K tile is DK / 128 boxes of
// 128 rows x 128 bytes side by side, a V^T tile (d rows x key columns) DK /
// 128 boxes stacked by rows, moved as one unit; the products are
// kind::f8f6f4 (K = 32 per MMA) on K-major operands, and P goes back to TMEM
// as e4m3, four keys per column.
template <int DK, bool F8 = false>
struct F256 {
  static_assert(DK == 64 || DK == 128 || DK == 256, "kernel head width");
  static_assert(!F8 || DK >= 128, "e4m3 tiles are 128 bytes wide");
  static constexpr int kHalves = (DK == 256 && !F8) ? 2 : 1;      // units per tile
  static constexpr int kUnitBoxes = F8 ? DK / 128 : (DK == 64 ? 1 : 2);   // boxes per unit
  static constexpr int kUnitSteps = 4 * kUnitBoxes;                // 32-byte K steps per unit
  static constexpr uint32_t kBoxBytes = 128u * 128u;       // 128 rows x 128 B (swizzled)
  static constexpr uint32_t kUnitBytes = kUnitBoxes * kBoxBytes;
  static constexpr int kQBoxes = F8 ? DK / 128 : DK / 64;
  static constexpr int kSlots = kUnitBytes == 32768u ? (DK == 256 && !F8 ? 5 : 6) : 13;
  static constexpr int kTileBars = kHalves == 2 ? 4 : 16;
  static_assert(kTileBars * kHalves >= kSlots, "release barriers outlast the ring");
  static constexpr uint32_t kQOff = 0;                     // Q boxes; O staging at the end
  static constexpr uint32_t kSlotOff = kQBoxes * kBoxBytes;
  static constexpr uint32_t kBarOff = kSlotOff + kSlots * kUnitBytes;
  // full[kSlots], empty[kTileBars], q_full, s_full[2], p_full, o_ready, staged, drain
  static constexpr int kBars = kSlots + kTileBars + 7;
  static constexpr uint32_t kMiscOff = kBarOff + kBars * 8;   // tmem holder, abort flag
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;   // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared-memory budget");
  static_assert(kBarOff >= 128u * DK * 4u, "fp32 staging of O fits the Q buffer and the ring");
  static constexpr int kThreads = 192;
  static constexpr uint32_t kColO = 256;
};

// Stream position t (0 .. 2n-1) -> (K or V, key tile j): K_0 K_1 V_0 K_2 V_1 ...
// K_{n-1} V_{n-2} V_{n-1}; and the positions of K_j and V_j.
__device__ __forceinline__ void stream_tile(int t, int n, bool& is_v, int& j) {
  if (t == 0) {
    is_v = false;
    j = 0;
  } else if (t == 2 * n - 1) {
    is_v = true;
    j = n - 1;
  } else if (t & 1) {
    is_v = false;
    j = (t + 1) >> 1;
  } else {
    is_v = true;
    j = (t - 2) >> 1;
  }
}
__device__ __forceinline__ int pos_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int pos_v(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }

// A CTA's work: head bh (hc for the 4-D maps), query tile qt, key tiles
// kt0 .. kt0 + n - 1; split is the key chunk of a split-KV launch (else 0).
struct W256 {
  int bh, qt, n, kt0, split;
  HeadCoord hc;
};

__device__ __forceinline__ W256 w256_work(int n_qt, int BH, int H, int band, bool causal) {
  W256 w;
  int rank;
  banded_order(blockIdx.x, n_qt, BH, band, w.bh, rank);
  w.hc = head_coord(w.bh, H);
  w.qt = causal ? n_qt - 1 - rank : rank;   // causal: heavy (long-row) tiles first
  w.n = causal ? w.qt + 1 : n_qt;
  w.kt0 = 0;
  w.split = 0;
  return w;
}

// Split-KV: CTA u takes query tile u % n_qt of one head and one chunk of
// kt_per_split key tiles (the last chunk may be shorter, never empty); CTAs
// of one (head, chunk) are adjacent, so they share the chunk's K/V in L2.
// Causal (query i at position Nk - Nq + i): the CTA stops at the last key
// tile its rows can see, but keeps one tile where it sees none, so that it
// still writes its (empty) partial result.
__device__ __forceinline__ W256 w256_split_work(int n_qt, int n_splits, int kt_per_split, int n_kt, int H,
                                                bool causal, int Nq, int Nk) {
  W256 w;
  const int u = static_cast<int>(blockIdx.x);
  w.qt = u % n_qt;
  const int rest = u / n_qt;
  w.split = rest % n_splits;
  w.bh = rest / n_splits;
  w.hc = head_coord(w.bh, H);
  w.kt0 = w.split * kt_per_split;
  w.n = min(kt_per_split, n_kt - w.kt0);
  if (causal) {
    const long long last_key = static_cast<long long>(w.qt) * 128 + 127 + (Nk - Nq);
    const long long tiles = last_key < 0 ? 0 : last_key / 128 + 1;   // key tiles the rows can see
    const long long seen = (tiles < n_kt ? tiles : n_kt) - w.kt0;
    if (seen < w.n) w.n = seen < 1 ? 1 : static_cast<int>(seen);
  }
  return w;
}

template <int DK, bool F8, bool REP>
__device__ void f256_producer(const W256& w, uint8_t* smem, uint64_t* full, uint64_t* empty, uint64_t* q_full,
                              const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                              const CtaGuard& g) {
  using C = F256<DK, F8>;
  mbar_arrive_expect_tx(q_full, C::kQBoxes * C::kBoxBytes);
  constexpr int kBoxCols = F8 ? 128 : 64;   // elements per 128-byte box row
  if constexpr (REP) {   // rows 0-31 (a 32-row box map) into each 32-row quarter of the tile
#pragma unroll
    for (int b = 0; b < C::kQBoxes; ++b)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        tma_load_hd(smem + C::kQOff + b * C::kBoxBytes + q * 4096u, tmQ, q_full, kBoxCols * b, 0, w.hc);
  } else {
#pragma unroll
    for (int b = 0; b < C::kQBoxes; ++b)
      tma_load_hd(smem + C::kQOff + b * C::kBoxBytes, tmQ, q_full, kBoxCols * b, 128 * w.qt, w.hc);
  }
  const int units = 2 * C::kHalves * w.n;
  int issued = 0;
  for (int u = 0; u < units; ++u) {
    const int t = u / C::kHalves, h = u % C::kHalves, slot = u % C::kSlots;
    if (u >= C::kSlots) {   // the slot's previous unit belongs to tile (u - kSlots) / kHalves: wait for its release
      const int pt = (u - C::kSlots) / C::kHalves;
      if (!mbar_wait(&empty[pt % C::kTileBars], (pt / C::kTileBars) & 1, g, kSiteFwd256 | 1u)) break;
    }
    bool is_v;
    int j;
    stream_tile(t, w.n, is_v, j);
    uint8_t* dst = smem + C::kSlotOff + slot * C::kUnitBytes;
    mbar_arrive_expect_tx(&full[slot], C::kUnitBytes);
    if (F8 && is_v) {   // V^T: d rows x keys, boxes stacked by rows
#pragma unroll
      for (int b = 0; b < C::kUnitBoxes; ++b)
        tma_load_hd(dst + b * C::kBoxBytes, tmV, &full[slot], 128 * (w.kt0 + j), 128 * b, w.hc);
    } else if (F8) {    // K: keys x d, boxes side by side
#pragma unroll
      for (int b = 0; b < C::kUnitBoxes; ++b)
        tma_load_hd(dst + b * C::kBoxBytes, tmK, &full[slot], 128 * b, 128 * (w.kt0 + j), w.hc);
    } else {
#pragma unroll
      for (int b = 0; b < C::kUnitBoxes; ++b)
        tma_load_hd(dst + b * C::kBoxBytes, is_v ? tmV : tmK, &full[slot], 128 * h + 64 * b, 128 * (w.kt0 + j),
                    w.hc);
    }
    issued = u + 1;
  }
  if (issued < units) {   // unwinding: let the copies in flight land before shared memory is released
    mbar_drain(q_full, 0);
    for (int u = (issued > C::kSlots ? issued - C::kSlots : 0); u < issued; ++u)
      mbar_drain(&full[u % C::kSlots], (u / C::kSlots) & 1);
  }
}

// Descriptor offset of K step kk (16 columns) inside a unit (K-major).
__device__ __forceinline__ uint64_t kstep_off(int kk) {
  return static_cast<uint64_t>(((kk / 4) * (128u * 128u) + (kk % 4) * 32) >> 4);
}

// The MMA warp: S(0) S(1) | PV(0) S(2) | PV(1) S(3) | ... | PV(n-1).
// ks = ceil(d / 16) steps of 16 columns hold data; the last unit's part of O
// is idesc_pvl wide (N = ceil(d / 16) * 16 - 128 (kHalves - 1)).  FD
// (d = DK): compile-time steps and widths; otherwise the steps are
// predicated.
template <int DK, bool FD, bool F8>
__device__ void f256_mma(const W256& w, uint32_t tmem, uint32_t sbase, uint64_t* full, uint64_t* empty,
                         uint64_t* q_full, uint64_t* s_full, uint64_t* p_full, uint64_t* o_ready, int ks,
                         uint32_t idesc_pvl, const CtaGuard& g) {
  using C = F256<DK, F8>;
  constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
  constexpr uint32_t idesc_pv = idesc_bf16(128, 64 * C::kUnitBoxes, false, true);
  const uint64_t qd0 = sdesc_sw128(sbase + C::kQOff, 16, 1024);
  const uint64_t kd0 = sdesc_sw128(sbase + C::kSlotOff, 16, 1024);            // slot 0, K-major
  const uint64_t vd0 = sdesc_sw128(sbase + C::kSlotOff, C::kBoxBytes, 1024);  // slot 0, MN-major
  auto slot_off = [](int u) { return static_cast<uint64_t>((u % C::kSlots) * (C::kUnitBytes >> 4)); };
  auto unit_wait = [&](int u) {
    return mbar_wait_w(&full[u % C::kSlots], (u / C::kSlots) & 1, g, kSiteFwd256 | 2u);
  };
  auto issue_s = [&](int buf, int t) -> bool {   // S into buffer `buf` from the K tile at stream position t
    const uint32_t ts = tmem + 128u * buf;
    for (int h = 0; h < C::kHalves; ++h) {
      if (!unit_wait(C::kHalves * t + h)) return false;
      const uint64_t q = qd0 + static_cast<uint64_t>((h * C::kUnitBytes) >> 4);
      const uint64_t k = kd0 + slot_off(C::kHalves * t + h);
#pragma unroll
      for (int kk = 0; kk < C::kUnitSteps; ++kk)
        if constexpr (F8)   // e4m3: 32 bytes = 32 columns per step; columns past d are zero
          tc_mma_f8_ss_w(ts, q + kstep_off(kk), k + kstep_off(kk), kk ? 1u : 0u);
        else if constexpr (FD)
          tc_mma_ss_w(ts, q + kstep_off(kk), k + kstep_off(kk), idesc_s, (h | kk) ? 1u : 0u);
        else
          tc_mma_ss_w_if(ts, q + kstep_off(kk), k + kstep_off(kk), idesc_s, (h | kk) ? 1u : 0u,
                         C::kUnitSteps * h + kk < ks ? 1u : 0u);
    }
    tc_commit_w(&s_full[buf]);
    tc_commit_w(&empty[t % C::kTileBars]);
    return true;
  };
  if (!mbar_wait_w(q_full, 0, g, kSiteFwd256 | 3u)) return;
  if (!issue_s(0, pos_k(0))) return;
  if (w.n > 1 && !issue_s(1, pos_k(1))) return;
  for (int j = 0; j < w.n; ++j) {
    const int t = pos_v(j, w.n), buf = j & 1;
    for (int h = 0; h < C::kHalves; ++h)
      if (!unit_wait(C::kHalves * t + h)) return;
    if (!mbar_wait_w(p_full, j & 1, g, kSiteFwd256 | 4u)) return;
    tc_fence_after();
    const uint32_t tp = tmem + 128u * buf;
    if constexpr (F8) {   // 128 keys, 32 per MMA; P packs 4 keys per TMEM column; V^T K-major,
                          // one 128-row box per 128 columns of O
#pragma unroll
      for (int b = 0; b < C::kUnitBoxes; ++b) {
        const uint64_t vt = kd0 + slot_off(t) + static_cast<uint64_t>((b * C::kBoxBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_f8_ts_w(tmem + C::kColO + 128u * b, tp + kk * 8, vt + kstep_off(kk), (j > 0 || kk > 0) ? 1u : 0u);
      }
    } else {
#pragma unroll
      for (int h = 0; h < C::kHalves; ++h) {
        const uint64_t v = vd0 + slot_off(C::kHalves * t + h);
        const uint32_t idesc = (h == C::kHalves - 1 && !FD) ? idesc_pvl : idesc_pv;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // 128 keys, 16 per MMA; P packs 2 keys per TMEM column
          tc_mma_ts_w(tmem + C::kColO + 128u * h, tp + kk * 8, v + ((kk * 2048) >> 4), idesc,
                      (j > 0 || kk > 0) ? 1u : 0u);
      }
    }
    tc_commit_w(o_ready);
    tc_commit_w(&empty[t % C::kTileBars]);
    if (j + 2 < w.n && !issue_s(buf, pos_k(j + 2))) return;
  }
}

// DROPOUT: dropout on the probabilities that feed O += P V (the keep mask of
// the shared counter-based contract, drawn on chip; the row sum l, hence
// LSE, uses the plain ones, and 1/(1-p) goes into the epilogue).
// SPLIT: O goes out in fp32 through the partial-output map (z = split * BH +
// bh) and the LSE to lse[(split * BH + bh) * N + row].  N is the query
// length, Nk the key length.
template <int DK, bool CAUSAL, bool SPLIT, bool DROPOUT, bool F8>
__device__ void f256_softmax(const W256& w, uint32_t tmem, uint8_t* smem, uint64_t* s_full, uint64_t* p_full,
                             uint64_t* o_ready, uint64_t* staged, const CUtensorMap* tmO, float* __restrict__ lse,
                             int N, int Nk, int BH, int d, float scale_log2, const DropArgs& drop,
                             float out_mult, const CtaGuard& g) {
  using C = F256<DK, F8>;
  const int r = threadIdx.x & 127;
  const int row = w.qt * 128 + r;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) * 32u << 16;
  const uint32_t tO = tmem + lane_base + C::kColO;

  float m_use = -INFINITY;  // reference max, base-2 units
  float l = 0.f;
  for (int j = 0; j < w.n; ++j) {
    const int buf = j & 1;
    const uint32_t tS = tmem + lane_base + 128u * buf;
    // keep words of this row's 128 keys, drawn before S lands (key c in byte
    // c % 4 of word (c / 4) % 4 of kp[c / 16])
    uint32_t kp[DROPOUT ? 8 : 1];
    if constexpr (DROPOUT) {
      uint32_t ge[32];
      dropout_rows<8>(drop, w.bh, row, j * 128, ge);
#pragma unroll
      for (int q = 0; q < 8; ++q) kp[q] = pack_keep4(ge[4 * q], ge[4 * q + 1], ge[4 * q + 2], ge[4 * q + 3]);
    }
    if (!mbar_wait(&s_full[buf], (j >> 1) & 1, g, kSiteFwd256 | 6u)) return;
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

    const int kv0 = (w.kt0 + j) * 128;
    int lim = Nk - kv0;
    if (CAUSAL) lim = min(lim, row + (Nk - N) - kv0 + 1);   // query row at position Nk - N + row
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

    bool rescale = false;
    float corr = 1.f;
    if (j == 0) {
      m_use = row_max;   // O is overwritten by the first P V product
    } else {
      const bool need = row_max > m_use + kRescaleThreshold;
      rescale = __any_sync(0xffffffffu, need);
      if (rescale) {
        const float m_new = need ? row_max : m_use;
        corr = (m_use == -INFINITY) ? 0.f : ex2_approx(m_use - m_new);
        l *= corr;
        m_use = m_new;
      }
    }
    const float m_off = (m_use == -INFINITY) ? 0.f : m_use;
    const float2 sc2 = make_float2(scale_log2, scale_log2), mo2 = make_float2(-m_off, -m_off);
    float2 sum[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sum[i] = make_float2(0.f, 0.f);
    if constexpr (F8) {   // P~ as e4m3, four keys per column, into the first 32 columns of S
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 128; c += 4) {
        const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(s[c / 32][c % 32]),
                                                 __uint_as_float(s[(c + 1) / 32][(c + 1) % 32])),
                                     sc2, mo2);
        const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(s[(c + 2) / 32][(c + 2) % 32]),
                                                 __uint_as_float(s[(c + 3) / 32][(c + 3) % 32])),
                                     sc2, mo2);
        const float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
        const float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
        sum[(c / 4) % 4] = __fadd2_rn(sum[(c / 4) % 4], __fadd2_rn(p0, p1));
        pk[c / 4] = e4m3x4(p0.x, p0.y, p1.x, p1.y);
      }
      tmem_st32(tS, pk);
    } else {
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
          if constexpr (DROPOUT)   // P o M (0/1); the 1/(1-p) scale goes into the epilogue
            pk[(c / 2) % 32] = pack_bf16x2(pp.x, pp.y) & keep_mask_pair(unpack_keep4(kp[c / 16], (c / 4) % 4), c % 4);
          else
            pk[(c / 2) % 32] = pack_bf16x2(pp.x, pp.y);
        }
        tmem_st32(tS + 32 * h, pk);
      }
    }
    const float2 s01 = __fadd2_rn(sum[0], sum[1]), s23 = __fadd2_rn(sum[2], sum[3]);
    const float2 s0123 = __fadd2_rn(s01, s23);
    l += s0123.x + s0123.y;
    if (j > 0) {
      // O may be touched only once the previous P V product has completed
      if (!mbar_wait(o_ready, (j - 1) & 1, g, kSiteFwd256 | 5u)) return;
      __syncwarp();
      tc_fence_after();
      if (rescale) {
#pragma unroll 1
        for (int c = 0; c < DK; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
          tmem_st32(tO + c, o);
        }
      }
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(p_full);
  }

  // epilogue: O = acc / l -> bf16 -> swizzled staging in the Q buffer (its last
  // reader, S(n-1), has completed) -> TMA store of the boxes holding columns < d
  if (!mbar_wait(o_ready, (w.n - 1) & 1, g, kSiteFwd256 | 7u)) return;
  __syncwarp();
  tc_fence_after();
  const float inv_l = l > 0.f ? out_mult / l : 0.f;
  const uint32_t stage = smem_u32(smem + C::kQOff);
  if constexpr (SPLIT) {
    // fp32 staging: DK / 32 boxes of 128 rows x 32 floats (128-byte rows,
    // swizzled) over the Q buffer and the ring, whose last readers (S(n-1)
    // and P V(n-1)) have completed and which no copy refills
#pragma unroll 1
    for (int c = 0; c < DK; c += 32) {
      if (c >= d) break;   // the columns past d are not stored
      uint32_t o[32];
      tmem_ld32(tO + c, o);
      tmem_ld_wait(o);
      const uint32_t box = stage + (c / 32) * 16384u + r * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_shared_v4(box + ((q ^ (r & 7)) << 4), __float_as_uint(__uint_as_float(o[4 * q]) * inv_l),
                     __float_as_uint(__uint_as_float(o[4 * q + 1]) * inv_l),
                     __float_as_uint(__uint_as_float(o[4 * q + 2]) * inv_l),
                     __float_as_uint(__uint_as_float(o[4 * q + 3]) * inv_l));
    }
    fence_proxy_async_smem();
    mbar_arrive(staged);
    if (r == 0 && mbar_wait(staged, 0, g, kSiteFwd256 | 8u)) {
      for (int b = 0; b < DK / 32; ++b)
        if (32 * b < d) tma_store_3d(tmO, smem + C::kQOff + b * 16384u, 32 * b, w.qt * 128, w.split * BH + w.bh);
      tma_store_commit();
      tma_store_wait_read_all();
    }
    if (row < N)
      lse[static_cast<size_t>(w.split * BH + w.bh) * N + row] = l > 0.f ? (m_use + __log2f(l)) * kLn2 : -INFINITY;
  } else {
#pragma unroll 1
    for (int c = 0; c < DK; c += 32) {
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
    mbar_arrive(staged);
    if (r == 0 && mbar_wait(staged, 0, g, kSiteFwd256 | 8u)) {
      for (int b = 0; b < DK / 64; ++b)   // bf16 O: 64-column boxes
        if (64 * b < d) tma_store_hd(tmO, smem + C::kQOff + b * C::kBoxBytes, 64 * b, w.qt * 128, w.hc);
      tma_store_commit();
      tma_store_wait_read_all();
    }
    if (row < N) lse[static_cast<size_t>(w.bh) * N + row] = l > 0.f ? (m_use + __log2f(l)) * kLn2 : -INFINITY;
  }
}

// Split-KV with at most 32 query rows (REP): the producer loads Q's rows
// 0-31 into all four 32-row quarters of the tile, and softmax warp q works on
// keys [32q, 32q + 32) of every key tile for those rows, with P = 0 for the
// other keys: four independent chunks of each key tile's softmax, a quarter
// of the exponentials and registers per row each.  O row 32q + i then holds
// query row i over warp q's keys; each quarter is stored as its own partial
// result (z = (4 split + q) BH + bh, rows 0-31 through a 32-row box map), so
// the merge, given 4 n_splits chunks, combines them like any other chunks.
template <int DK, bool CAUSAL, bool F8>
__device__ void f256_softmax_rep(const W256& w, uint32_t tmem, uint8_t* smem, uint64_t* s_full, uint64_t* p_full,
                                 uint64_t* o_ready, uint64_t* staged, const CUtensorMap* tmO,
                                 float* __restrict__ lse, int N, int Nk, int BH, int d, float scale_log2,
                                 float out_mult, const CtaGuard& g) {
  using C = F256<DK, F8>;
  const int r = threadIdx.x & 127;
  const int wq = r >> 5;            // this warp's quarter of the keys (and of the TMEM lanes)
  const int row = r & 31;           // query row (the tile is query tile 0)
  const uint32_t lane_base = static_cast<uint32_t>(wq) * 32u << 16;
  const uint32_t tO = tmem + lane_base + C::kColO;
  float m_use = -INFINITY;  // reference max, base-2 units
  float l = 0.f;
  for (int j = 0; j < w.n; ++j) {
    const int buf = j & 1;
    const uint32_t tS = tmem + lane_base + 128u * buf;
    if (!mbar_wait(&s_full[buf], (j >> 1) & 1, g, kSiteFwd256 | 6u)) return;
    __syncwarp();
    tc_fence_after();
    uint32_t s[32];
    tmem_ld32(tS + 32 * wq, s);
    tmem_ld_wait(s);
    const int kq0 = (w.kt0 + j) * 128 + 32 * wq;   // first key of this quarter
    int lim = Nk - kq0;                            // visible keys of this quarter
    if (CAUSAL) lim = min(lim, row + (Nk - N) - kq0 + 1);   // query row at position Nk - N + row
    if (lim < 32) {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c >= lim) s[c] = __float_as_uint(-INFINITY);
    }
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int c = 0; c < 32; c += 2)
      mx[(c / 2) % 4] = max3f(mx[(c / 2) % 4], __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
    const float row_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
    bool rescale = false;
    float corr = 1.f;
    if (j == 0) {
      m_use = row_max;
    } else {
      const bool need = row_max > m_use + kRescaleThreshold;
      rescale = __any_sync(0xffffffffu, need);
      if (rescale) {
        const float m_new = need ? row_max : m_use;
        corr = (m_use == -INFINITY) ? 0.f : ex2_approx(m_use - m_new);
        l *= corr;
        m_use = m_new;
      }
    }
    const float m_off = (m_use == -INFINITY) ? 0.f : m_use;
    const float2 sc2 = make_float2(scale_log2, scale_log2), mo2 = make_float2(-m_off, -m_off);
    float2 sum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float p[32];
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
      const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sc2, mo2);
      p[c] = ex2_approx(x.x);
      p[c + 1] = ex2_approx(x.y);
      sum[(c / 2) % 2] = __fadd2_rn(sum[(c / 2) % 2], make_float2(p[c], p[c + 1]));
    }
    uint32_t pk[32];
    if constexpr (F8) {   // e4m3, four keys per column: this quarter is columns [8 wq, 8 wq + 8)
#pragma unroll
      for (int i = 0; i < 32; ++i) pk[i] = 0u;
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (q == wq) pk[8 * q + i] = e4m3x4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
      tmem_st32(tS, pk);
    } else {              // bf16 pairs: this quarter is columns [16 wq, 16 wq + 16) of the 64
#pragma unroll
      for (int i = 0; i < 32; ++i) pk[i] = (i / 16 == (wq & 1)) ? pack_bf16x2(p[2 * (i % 16)], p[2 * (i % 16) + 1]) : 0u;
      tmem_st32(tS + 32 * (wq >> 1), pk);
#pragma unroll
      for (int i = 0; i < 32; ++i) pk[i] = 0u;
      tmem_st32(tS + 32 * (1 - (wq >> 1)), pk);
    }
    const float2 s01 = __fadd2_rn(sum[0], sum[1]);
    l += s01.x + s01.y;
    if (j > 0) {
      // O may be touched only once the previous P V product has completed
      if (!mbar_wait(o_ready, (j - 1) & 1, g, kSiteFwd256 | 5u)) return;
      __syncwarp();
      tc_fence_after();
      if (rescale) {
#pragma unroll 1
        for (int c = 0; c < DK; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
          tmem_st32(tO + c, o);
        }
      }
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(p_full);
  }

  // epilogue: fp32 staging of the whole tile (as the split epilogue), then
  // each quarter's 32 rows to its own partial result
  if (!mbar_wait(o_ready, (w.n - 1) & 1, g, kSiteFwd256 | 7u)) return;
  __syncwarp();
  tc_fence_after();
  const float inv_l = l > 0.f ? out_mult / l : 0.f;
  const uint32_t stage = smem_u32(smem + C::kQOff);
#pragma unroll 1
  for (int c = 0; c < DK; c += 32) {
    if (c >= d) break;   // the columns past d are not stored
    uint32_t o[32];
    tmem_ld32(tO + c, o);
    tmem_ld_wait(o);
    const uint32_t box = stage + (c / 32) * 16384u + r * 128;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      st_shared_v4(box + ((q ^ (r & 7)) << 4), __float_as_uint(__uint_as_float(o[4 * q]) * inv_l),
                   __float_as_uint(__uint_as_float(o[4 * q + 1]) * inv_l),
                   __float_as_uint(__uint_as_float(o[4 * q + 2]) * inv_l),
                   __float_as_uint(__uint_as_float(o[4 * q + 3]) * inv_l));
  }
  fence_proxy_async_smem();
  mbar_arrive(staged);
  if (r == 0 && mbar_wait(staged, 0, g, kSiteFwd256 | 8u)) {
    for (int b = 0; b < DK / 32; ++b)
      if (32 * b < d)
        for (int q = 0; q < 4; ++q)
          tma_store_3d(tmO, smem + C::kQOff + b * 16384u + q * 4096u, 32 * b, 0, (4 * w.split + q) * BH + w.bh);
    tma_store_commit();
    tma_store_wait_read_all();
  }
  if (row < N)
    lse[static_cast<size_t>((4 * w.split + wq) * BH + w.bh) * N + row] =
        l > 0.f ? (m_use + __log2f(l)) * kLn2 : -INFINITY;
}

// SPLIT: a split-KV launch (non-causal, no dropout): n_kt key tiles in
// n_splits chunks of kt_per_split; tmO is then the fp32 partial-output map
// and lse the partial LSE.  N is the query length and Nk the key length
// (equal outside split-KV launches).  F8: e4m3 inputs (tmV maps V^T) with
// per-(b, h) descales dsq, dsk, dsv (unused otherwise): S carries dsq dsk,
// O is multiplied by dsv.
template <int DK, bool CAUSAL, bool FD, bool DROPOUT, bool SPLIT, bool F8 = false, bool REP = false>
__global__ void __launch_bounds__(192, 1)
    fa_fwd_d256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                       float* __restrict__ lse, int N, int Nk, int d, int n_qt, int BH, int H, int band,
                       float scale_log2, int ks, uint32_t idesc_pvl, int n_kt, int n_splits, int kt_per_split,
                       const float* __restrict__ dsq, const float* __restrict__ dsk, const float* __restrict__ dsv,
                       const __grid_constant__ DropArgs drop, const WaitCfg wc) {
  static_assert(!SPLIT || !DROPOUT, "split-KV launches have no dropout");
  static_assert(SPLIT || DK == 256, "below d = 256 only split-KV launches run this kernel");
  static_assert(!REP || SPLIT, "row replication serves split-KV launches");
  using C = F256<DK, F8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* full = bars;                     // [kSlots]
  uint64_t* empty = full + C::kSlots;        // [kTileBars]
  uint64_t* q_full = empty + C::kTileBars;
  uint64_t* s_full = q_full + 1;             // [2]
  uint64_t* p_full = s_full + 2;
  uint64_t* o_ready = p_full + 1;
  uint64_t* staged = o_ready + 1;
  uint64_t* drain = staged + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const W256 w = SPLIT ? w256_split_work(n_qt, n_splits, kt_per_split, n_kt, H, CAUSAL, N, Nk)
                       : w256_work(n_qt, BH, H, band, CAUSAL);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kSlots; ++i) mbar_init(&full[i], 1);
    for (int i = 0; i < C::kTileBars; ++i) mbar_init(&empty[i], 1);
    mbar_init(q_full, 1);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 128);
    mbar_init(o_ready, 1);
    mbar_init(staged, 128);
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const CtaGuard g{abort_flag, g_status_fwd256, wc.epoch, wc.limit_us};

  if (warp == 4) {
    if (lane == 0) f256_producer<DK, F8, REP>(w, smem, full, empty, q_full, &tmQ, &tmK, &tmV, g);
  } else if (warp == 5) {
    f256_mma<DK, FD, F8>(w, tmem, smem_u32(smem), full, empty, q_full, s_full, p_full, o_ready, ks, idesc_pvl, g);
    tc_commit_w(drain);   // every MMA issued above has finished before TMEM is released
    mbar_drain(drain, 0);
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, 160);
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  } else {
    float sl = scale_log2, out_mult = DROPOUT ? drop.scale : 1.f;
    if constexpr (F8) {
      sl *= dsq[w.bh] * dsk[w.bh];
      out_mult = dsv[w.bh];
    }
    if constexpr (REP)
      f256_softmax_rep<DK, CAUSAL, F8>(w, tmem, smem, s_full, p_full, o_ready, staged, &tmO, lse, N, Nk, BH, d, sl,
                                       out_mult, g);
    else
      f256_softmax<DK, CAUSAL, SPLIT, DROPOUT, F8>(w, tmem, smem, s_full, p_full, o_ready, staged, &tmO, lse, N, Nk,
                                                   BH, d, sl, drop, out_mult, g);
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, 160);
  }
}

template <bool CAUSAL, bool DROPOUT>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                     float* lse, const Shape& s, const DropArgs& drop, const WaitCfg& wc, cudaStream_t st) {
  using C = F256<256>;
  auto kern = s.d == 256 ? fa_fwd_d256_kernel<256, CAUSAL, true, DROPOUT, false>
                         : fa_fwd_d256_kernel<256, CAUSAL, false, DROPOUT, false>;
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads, 0);
  if (e != cudaSuccess) return e;
  const int n_qt = (s.N + 127) / 128;
  const float scale_log2 = static_cast<float>(static_cast<double>(s.scale) * 1.4426950408889634);
  const dim3 grid(static_cast<unsigned>(s.B) * s.H * n_qt);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tv, to, lse, s.N, s.N, s.d, n_qt, s.B * s.H, s.H,
                                                 head_band(s.N, s.d), scale_log2, score_ksteps(s.d),
                                                 idesc_bf16(128, out_cols(s.d) - 128, false, true), n_qt, 1, n_qt,
                                                 nullptr, nullptr, nullptr, drop, wc);
  return cudaGetLastError();
}

// The e4m3 variant at width DK: a split-KV launch (SPLIT; REP: row
// replication) or a plain forward (grid B H n_qt, causal or not).
template <int DK, bool CAUSAL, bool SPLIT, bool REP>
cudaError_t launch_f8_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                        const CUtensorMap& to, const float* dsq, const float* dsk, const float* dsv, float* lse,
                        const Shape& s, int Nk, int n_splits, int kt_per_split, const WaitCfg& wc, cudaStream_t st) {
  using C = F256<DK, true>;
  auto kern = fa_fwd_d256_kernel<DK, CAUSAL, true, false, SPLIT, true, REP>;
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads, 0);
  if (e != cudaSuccess) return e;
  const int n_qt = (s.N + 127) / 128, n_kt = (Nk + 127) / 128;
  const float scale_log2 = static_cast<float>(static_cast<double>(s.scale) * 1.4426950408889634);
  const dim3 grid(static_cast<unsigned>(s.B) * s.H * (SPLIT ? n_splits : 1) * n_qt);
  // L2 band: e4m3 K and V of a head take 2 N d bytes, as bf16 ones of d / 2 columns
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tvt, to, lse, s.N, Nk, s.d, n_qt, s.B * s.H, s.H,
                                                 head_band(s.N, (s.d + 1) / 2), scale_log2, 0, 0u, n_kt,
                                                 n_splits, kt_per_split, dsq, dsk, dsv, no_drop_args(), wc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_d256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, float* lse, const Shape& s, const DropArgs& drop,
                            const WaitCfg& wc, cudaStream_t st) {
  if (drop.t4 != 0)
    return s.causal ? launch_t<true, true>(tq, tk, tv, to, lse, s, drop, wc, st)
                    : launch_t<false, true>(tq, tk, tv, to, lse, s, drop, wc, st);
  return s.causal ? launch_t<true, false>(tq, tk, tv, to, lse, s, drop, wc, st)
                  : launch_t<false, false>(tq, tk, tv, to, lse, s, drop, wc, st);
}

template <int DK, bool CAUSAL>
cudaError_t launch_split_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& top, float* lse_part, const Shape& s, int Nk, int n_splits,
                           int kt_per_split, const WaitCfg& wc, cudaStream_t st) {
  using C = F256<DK>;
  auto kern = s.d == DK ? fa_fwd_d256_kernel<DK, CAUSAL, true, false, true>
                        : fa_fwd_d256_kernel<DK, CAUSAL, false, false, true>;
  if constexpr (DK == 64) {   // row replication (splitkv_replicas) applies at width 64 only
    if (splitkv_replicas(s.N, s.d, false) > 1)
      kern = s.d == DK ? fa_fwd_d256_kernel<DK, CAUSAL, true, false, true, false, true>
                       : fa_fwd_d256_kernel<DK, CAUSAL, false, false, true, false, true>;
  }
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads, 0);
  if (e != cudaSuccess) return e;
  const int n_qt = (s.N + 127) / 128, n_kt = (Nk + 127) / 128;
  const float scale_log2 = static_cast<float>(static_cast<double>(s.scale) * 1.4426950408889634);
  const dim3 grid(static_cast<unsigned>(s.B) * s.H * n_splits * n_qt);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tv, top, lse_part, s.N, Nk, s.d, n_qt, s.B * s.H, s.H, 1,
                                                 scale_log2, score_ksteps(s.d),
                                                 idesc_bf16(128, out_cols(s.d) - 128 * (C::kHalves - 1), false, true),
                                                 n_kt, n_splits, kt_per_split, nullptr, nullptr, nullptr,
                                                 no_drop_args(), wc);
  return cudaGetLastError();
}

cudaError_t launch_fwd_onetile_split(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                     const CUtensorMap& top, float* lse_part, const Shape& s, int Nk, int n_splits,
                                     int kt_per_split, const WaitCfg& wc, cudaStream_t st) {
  if (s.causal) {
    switch (kernel_dim(s.d)) {
      case 256: return launch_split_t<256, true>(tq, tk, tv, top, lse_part, s, Nk, n_splits, kt_per_split, wc, st);
      case 128: return launch_split_t<128, true>(tq, tk, tv, top, lse_part, s, Nk, n_splits, kt_per_split, wc, st);
      default: return launch_split_t<64, true>(tq, tk, tv, top, lse_part, s, Nk, n_splits, kt_per_split, wc, st);
    }
  }
  switch (kernel_dim(s.d)) {
    case 256: return launch_split_t<256, false>(tq, tk, tv, top, lse_part, s, Nk, n_splits, kt_per_split, wc, st);
    case 128: return launch_split_t<128, false>(tq, tk, tv, top, lse_part, s, Nk, n_splits, kt_per_split, wc, st);
    default: return launch_split_t<64, false>(tq, tk, tv, top, lse_part, s, Nk, n_splits, kt_per_split, wc, st);
  }
}

cudaError_t launch_fwd_fp8_split(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                                 const CUtensorMap& top, const float* dsq, const float* dsk, const float* dsv,
                                 float* lse_part, const Shape& s, int Nk, int n_splits, int kt_per_split,
                                 const WaitCfg& wc, cudaStream_t st) {
  const bool rep = splitkv_replicas(s.N, s.d, true) > 1;
  if (s.causal) {
    if (s.d > 128)
      return launch_f8_t<256, true, true, false>(tq, tk, tvt, top, dsq, dsk, dsv, lse_part, s, Nk, n_splits,
                                                 kt_per_split, wc, st);
    return rep ? launch_f8_t<128, true, true, true>(tq, tk, tvt, top, dsq, dsk, dsv, lse_part, s, Nk, n_splits,
                                                    kt_per_split, wc, st)
               : launch_f8_t<128, true, true, false>(tq, tk, tvt, top, dsq, dsk, dsv, lse_part, s, Nk, n_splits,
                                                     kt_per_split, wc, st);
  }
  if (s.d > 128)
    return launch_f8_t<256, false, true, false>(tq, tk, tvt, top, dsq, dsk, dsv, lse_part, s, Nk, n_splits,
                                                kt_per_split, wc, st);
  return rep ? launch_f8_t<128, false, true, true>(tq, tk, tvt, top, dsq, dsk, dsv, lse_part, s, Nk, n_splits,
                                                   kt_per_split, wc, st)
             : launch_f8_t<128, false, true, false>(tq, tk, tvt, top, dsq, dsk, dsv, lse_part, s, Nk, n_splits,
                                                    kt_per_split, wc, st);
}

cudaError_t launch_fwd_fp8_wide(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                                const CUtensorMap& to, const float* dsq, const float* dsk, const float* dsv,
                                float* lse, const Shape& s, const WaitCfg& wc, cudaStream_t st) {
  return s.causal ? launch_f8_t<256, true, false, false>(tq, tk, tvt, to, dsq, dsk, dsv, lse, s, s.N, 1, 0, wc, st)
                  : launch_f8_t<256, false, false, false>(tq, tk, tvt, to, dsq, dsk, dsv, lse, s, s.N, 1, 0, wc, st);
}

cudaError_t fwd_d256_status(uint32_t* out, bool reset) {
  unsigned int v[2] = {0, 0};
  cudaError_t e = cudaMemcpyFromSymbol(v, g_status_fwd256, sizeof(v));
  if (e != cudaSuccess) return e;
  *out = v[0];
  if (reset && (v[0] | v[1]) != 0) {
    const unsigned int z[2] = {0, 0};
    e = cudaMemcpyToSymbol(g_status_fwd256, z, sizeof(z));
  }
  return e;
}

}  // namespace fa
