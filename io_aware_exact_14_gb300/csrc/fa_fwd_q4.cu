// Forward pass for narrow heads (d <= 64) on sm_103a: four query tiles per
// CTA and 64-key steps.  The method is fa_fwd.cu's (tiles of Q on chip, K/V
// streamed, running (m, l, acc), one division by l at the end:
// "为什么Flash Attention能将注意力计算提速数倍而不损失精度", sections "分块计算
// （Tiling）" and "在线Softmax技巧"; the softmax of some tiles overlapping the
// matrix products of others: same page, "Flash Attention 3：拥抱Hopper架构").
//
// Why a kernel of its own: at d = 64 the products are half as long as at
// d = 128 while each score still costs one exponential, so with two query
// tiles per CTA a tile's own chain -- softmax, then its P V and next S
// products -- sets the pace and the tensor core idles half the time.  Four
// query tiles keep four such chains in flight; with 64-key steps each tile
// needs 64 TMEM columns of scores and 64 of output, so four fit the 512.
//
// GB300 design (one CTA per SM, 640 threads):
//   warps 0-15  softmax, four warpgroups: warpgroup t serves query tile t
//               (thread = query row = TMEM lane)
//   warp  16    TMA producer: Q once (four 128-row tiles), then K_j, V_j
//               (64-key tiles, 8 KB) through a ring of slots in per-step
//               groups (K_0, then {V_j, K_{j+1}}), one barrier per group
//   warps 17-18 tcgen05.mma issuers (elect.sync in converged warps): warp
//               17 issues tiles 0 and 1, warp 18 tiles 2 and 3, each in the
//               order S_a(0) S_b(0) | PV_a(0) S_a(1) PV_b(0) S_b(1) | ...
//               (issuing whichever tile's P is ready first measured 3-4%
//               slower: the two-barrier poll costs more than it saves);
//               warp 17 also owns TMEM
//   warp  19    idle
// TMEM: tile t has S at columns [128t, 128t + 64) and O at [128t + 64,
// 128t + 128).  P (bf16, two keys per column) overwrites the first 32 columns
// of its S and feeds O += P V from TMEM.  Lazy rescaling as in fa_fwd.cu.
#include "fa_internal.h"
// the polling loops inline at each wait: measured 2-4% faster here than the
// shared out-of-line copies
#define FA_INLINE_WAITS 1
#include "fa_ptx.cuh"

#include <cmath>

namespace fa {
namespace {

__device__ unsigned int g_status_q4[2] = {0, 0};   // status, abort epoch (see CtaGuard)

constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kSiteQ4 = 0x600;

struct Q4 {
  static constexpr int kTiles = 4;
  static constexpr uint32_t kQBytes = 128u * 128u;          // a query tile: 128 rows x 64 bf16 (one box)
  static constexpr uint32_t kKVBytes = 64u * 128u;          // a key/value tile: 64 rows x 64 bf16
  static constexpr int kSlots = 16;                         // ring slots (8 groups)
  static constexpr int kGroups = kSlots / 2;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kSlotOff = kTiles * kQBytes;
  static constexpr uint32_t kBarOff = kSlotOff + kSlots * kKVBytes;
  // gfull[G], release[G], q_full, s_full[4], p_full[4], o_done[4], staged[4], drain
  static constexpr int kBars = 2 * kGroups + 1 + 4 * kTiles + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kBars * 8;   // tmem holder, abort flag
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared-memory budget");
  // 96 registers a thread (65536 / 640, in steps of 8) serve every role
  // without spilling: the softmax holds 64 scores, and rescales O (rarely)
  // only after P is out, when the scores are dead.
  static constexpr int kThreads = 640;
  __host__ __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 128u * t + 64u; }
};

// A CTA's work: head bh, query tiles 4u .. 4u + 3 (n_t 64-key steps each, 0
// past the last tile), n = the largest n_t.
struct WQ4 {
  int bh, qt0, n;
  int nt[4];
  HeadCoord hc;
};

// n_t of tile t, by selects (a run-time index into nt[] would put it on the stack).
__device__ __forceinline__ int tile_steps(const WQ4& w, int t) {
  return t == 0 ? w.nt[0] : (t == 1 ? w.nt[1] : (t == 2 ? w.nt[2] : w.nt[3]));
}

__device__ __forceinline__ WQ4 q4_work(int n_qt, int n_units, int n_kt, int BH, int H, int band, bool causal) {
  WQ4 w;
  int rank;
  banded_order(blockIdx.x, n_units, BH, band, w.bh, rank);
  w.hc = head_coord(w.bh, H);
  const int unit = causal ? n_units - 1 - rank : rank;   // causal: long rows first
  w.qt0 = 4 * unit;
  w.n = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int qt = w.qt0 + t;
    w.nt[t] = qt < n_qt ? (causal ? min(2 * qt + 2, n_kt) : n_kt) : 0;
    w.n = max(w.n, w.nt[t]);
  }
  return w;
}

__device__ void q4_producer(const WQ4& w, uint8_t* smem, uint64_t* full, uint64_t* empty, uint64_t* q_full,
                            const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV, const CtaGuard& g) {
  using C = Q4;
  int nq = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) nq += w.nt[t] > 0 ? 1 : 0;
  mbar_arrive_expect_tx(q_full, nq * C::kQBytes);
#pragma unroll
  for (int t = 0; t < 4; ++t)
    if (w.nt[t] > 0) tma_load_hd(smem + C::kQOff + t * C::kQBytes, tmQ, q_full, 0, 128 * (w.qt0 + t), w.hc);
  int issued = 0;
  bool ok = true;
  for (int j = 0; j < w.n && ok; ++j) {
    for (int kind = 0; kind < 2; ++kind) {   // K_j (group j), then V_j (group j + 1)
      const int idx = 2 * j + kind;
      const int grp = (idx + 1) >> 1;
      if (kind == 1 || j == 0) {
        // first tile of its group: wait until the group that last used these
        // two slots is released, then expect the whole group
        if (grp >= C::kGroups &&
            !mbar_wait(&empty[grp % C::kGroups], ((grp / C::kGroups) - 1) & 1u, g, kSiteQ4 | 1u)) {
          ok = false;
          break;
        }
        const bool pair = grp > 0 && grp < w.n;   // group n holds V_{n-1} alone
        mbar_arrive_expect_tx(&full[grp % C::kGroups], (pair ? 2u : 1u) * C::kKVBytes);
      }
      tma_load_hd(smem + C::kSlotOff + (idx % C::kSlots) * C::kKVBytes, kind ? tmV : tmK,
                  &full[grp % C::kGroups], 0, 64 * j, w.hc);
      issued = idx + 1;
    }
  }
  if (!ok) {   // unwinding: let copies already issued land before shared memory is released
    mbar_drain(q_full, 0);
    for (int q = max(0, ((issued + 1) >> 1) - C::kGroups); q <= (issued >> 1); ++q)
      if (2 * q - 1 < issued || q == 0) mbar_drain(&full[q % C::kGroups], (q / C::kGroups) & 1);
  }
}

// S_t = Q_t K^T (M = 128, N = 64 keys, K = d: ks steps of 16) and O_t (+)= P_t V
// (M = 128, N = d, K = 64 keys: 4 steps, P from TMEM, V MN-major).
template <bool FD>
__device__ __forceinline__ void q4_issue_s(uint32_t tmem_s, uint64_t q_desc, uint64_t k_desc, int ks) {
  constexpr uint32_t idesc = idesc_bf16(128, 64, false, false);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
    if constexpr (FD)
      tc_mma_ss_w(tmem_s, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
    else
      tc_mma_ss_w_if(tmem_s, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u, kk < ks ? 1u : 0u);
  }
}

template <bool FD>
__device__ __forceinline__ void q4_issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t v_desc, bool acc,
                                            uint32_t idesc_rt) {
  const uint32_t idesc = FD ? idesc_bf16(128, 64, false, true) : idesc_rt;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)   // 64 keys, 16 per MMA; P packs 2 keys per TMEM column
    tc_mma_ts_w(tmem_o, tmem_p + kk * 8, v_desc + ((kk * 2048) >> 4), idesc, (acc || kk > 0) ? 1u : 0u);
}

// Issuer for tiles a = 2w and b = 2w + 1 (w = 0 or 1).  Both issuers walk
// every key step and release each group (release barriers count two commits).
template <bool FD>
__device__ void q4_mma(const WQ4& w, int wi, uint32_t tmem, uint32_t smem_base, uint64_t* full, uint64_t* empty,
                       uint64_t* q_full, uint64_t* s_full, uint64_t* p_full, uint64_t* o_done, int ks,
                       uint32_t idesc_pv, const CtaGuard& g) {
  using C = Q4;
  const int ta = 2 * wi, tb = 2 * wi + 1;
  const int na = tile_steps(w, ta), nb = tile_steps(w, tb);
  const uint64_t qa = sdesc_sw128(smem_base + C::kQOff + ta * C::kQBytes, 16, 1024);
  const uint64_t qb = sdesc_sw128(smem_base + C::kQOff + tb * C::kQBytes, 16, 1024);
  const uint64_t k0 = sdesc_sw128(smem_base + C::kSlotOff, 16, 1024);           // K-major (S = Q K^T)
  const uint64_t v0 = sdesc_sw128(smem_base + C::kSlotOff, C::kKVBytes, 1024);  // MN-major (O += P V)
  auto slot_off = [&](int idx) { return static_cast<uint64_t>((idx % C::kSlots) * (C::kKVBytes >> 4)); };
  auto group_wait = [&](int grp) {   // group 0: K_0; group j+1: V_j and K_{j+1}
    return mbar_wait_w(&full[grp % C::kGroups], (grp / C::kGroups) & 1, g, kSiteQ4 | 2u);
  };
  if (!mbar_wait_w(q_full, 0, g, kSiteQ4 | 3u)) return;
  if (!group_wait(0)) return;
  if (na > 0) {
    q4_issue_s<FD>(tmem + C::col_s(ta), qa, k0 + slot_off(0), ks);
    tc_commit_w(&s_full[ta]);
  }
  if (nb > 0) {
    q4_issue_s<FD>(tmem + C::col_s(tb), qb, k0 + slot_off(0), ks);
    tc_commit_w(&s_full[tb]);
  }
  tc_commit_w(&empty[0]);   // group 0: K_0
  for (int j = 0; j < w.n; ++j) {
    const int iv = 2 * j + 1, ik = 2 * j + 2;   // ring indices of V_j and K_{j+1}
    if (!group_wait(j + 1)) return;
    const uint64_t vd = v0 + slot_off(iv), kd = k0 + slot_off(ik);
    if (j < na) {
      if (!mbar_wait_w(&p_full[ta], j & 1, g, kSiteQ4 | 4u)) return;
      tc_fence_after();
      q4_issue_pv<FD>(tmem + C::col_o(ta), tmem + C::col_s(ta), vd, j > 0, idesc_pv);
      if (j + 1 < na) q4_issue_s<FD>(tmem + C::col_s(ta), qa, kd, ks);
      if (j == na - 1) tc_commit_w(&o_done[ta]);
      if (j + 1 < na) tc_commit_w(&s_full[ta]);
    }
    if (j < nb) {
      if (!mbar_wait_w(&p_full[tb], j & 1, g, kSiteQ4 | 5u)) return;
      tc_fence_after();
      q4_issue_pv<FD>(tmem + C::col_o(tb), tmem + C::col_s(tb), vd, j > 0, idesc_pv);
      if (j + 1 < nb) q4_issue_s<FD>(tmem + C::col_s(tb), qb, kd, ks);
      if (j == nb - 1) tc_commit_w(&o_done[tb]);
      if (j + 1 < nb) tc_commit_w(&s_full[tb]);
    }
    tc_commit_w(&empty[(j + 1) % C::kGroups]);   // group j+1: V_j and K_{j+1}
  }
}

template <bool CAUSAL>
__device__ void q4_softmax(const WQ4& w, int t, uint32_t tmem, uint8_t* smem, uint64_t* s_full, uint64_t* p_full,
                           uint64_t* o_done, uint64_t* staged, const CUtensorMap* tmO, float* __restrict__ lse,
                           int N, float scale_log2, const CtaGuard& g) {
  using C = Q4;
  const int n_t = tile_steps(w, t);
  if (n_t == 0) return;
  const int r = threadIdx.x & 127;
  const int qt = w.qt0 + t;
  const int row = qt * 128 + r;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) * 32u << 16;
  const uint32_t tS = tmem + lane_base + C::col_s(t);
  const uint32_t tO = tmem + lane_base + C::col_o(t);

  float m_use = -INFINITY;  // reference max, base-2 units
  float l = 0.f;
  for (int j = 0; j < n_t; ++j) {
    if (!mbar_wait(&s_full[t], j & 1, g, kSiteQ4 | 6u)) return;
    __syncwarp();
    tc_fence_after();
    uint32_t s[2][32];
    tmem_ld32(tS + 0, s[0]);
    tmem_ld32(tS + 32, s[1]);
    tmem_ld_wait(s[0]);
    tmem_ld_fence(s[1]);

    // keys kv0 .. kv0 + lim - 1 are visible to this row
    const int kv0 = j * 64;
    int lim = N - kv0;
    if (CAUSAL) lim = min(lim, row - kv0 + 1);
    if (lim < 64) {
#pragma unroll
      for (int c = 0; c < 64; ++c)
        if (c >= lim) s[c / 32][c % 32] = __float_as_uint(-INFINITY);
    }
    float mx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
    for (int c = 0; c < 64; c += 2)
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
#pragma unroll
    for (int h = 0; h < 2; ++h) {   // keys [32h, 32h + 32) -> P columns [16h, 16h + 16)
      uint32_t pk[16];
#pragma unroll
      for (int c = 32 * h; c < 32 * h + 32; c += 2) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[h][c % 32]), __uint_as_float(s[h][c % 32 + 1])),
                                    sc2, mo2);
        const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        sum[(c / 2) % 4] = __fadd2_rn(sum[(c / 2) % 4], pp);
        pk[(c / 2) % 16] = pack_bf16x2(pp.x, pp.y);
      }
      tmem_st16(tS + 16 * h, pk);
    }
    const float2 s01 = __fadd2_rn(sum[0], sum[1]), s23 = __fadd2_rn(sum[2], sum[3]);
    const float2 s0123 = __fadd2_rn(s01, s23);
    l += s0123.x + s0123.y;
    if (rescale) {
      // after P, so the scores are no longer live; before p_full, so PV(j)
      // adds to the rescaled O.  O holds the P V products of earlier steps,
      // all completed: S(j) was issued after PV(j - 1) and has completed.
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t o[32];
        tmem_ld32(tO + c, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
        tmem_st32(tO + c, o);
      }
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&p_full[t]);
  }

  // epilogue: O = acc / l -> bf16 -> swizzled staging (this tile's Q buffer,
  // whose last reader S_t(n_t - 1) has completed) -> TMA store
  if (!mbar_wait(&o_done[t], 0, g, kSiteQ4 | 7u)) return;
  __syncwarp();
  tc_fence_after();
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
  const uint32_t stage = smem_u32(smem + C::kQOff + t * C::kQBytes);
#pragma unroll
  for (int c = 0; c < 64; c += 32) {
    uint32_t o[32];
    tmem_ld32(tO + c, o);
    tmem_ld_wait(o);
    const uint32_t box = stage + r * 128;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int chunk = c / 8 + q;
      float f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[8 * q + e]) * inv_l;
      st_shared_v4(box + ((chunk ^ (r & 7)) << 4), pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                   pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
    }
  }
  fence_proxy_async_smem();
  mbar_arrive(&staged[t]);
  if (r == 0 && mbar_wait(&staged[t], 0, g, kSiteQ4 | 8u)) {
    tma_store_hd(tmO, smem + C::kQOff + t * C::kQBytes, 0, qt * 128, w.hc);
    tma_store_commit();
    tma_store_wait_read_all();
  }
  if (row < N) lse[static_cast<size_t>(w.bh) * N + row] = l > 0.f ? (m_use + __log2f(l)) * kLn2 : -INFINITY;
}

// FD: d == 64 (compile-time K steps and output width of the products).
template <bool CAUSAL, bool FD>
__global__ void __launch_bounds__(640, 1)
    fa_fwd_q4_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     float* __restrict__ lse, int N, int n_qt, int n_units, int n_kt, int BH, int H, int band,
                     float scale_log2, int ks, uint32_t idesc_pv, const WaitCfg wc) {
  using C = Q4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* full = bars;                   // gfull[kGroups]
  uint64_t* empty = bars + C::kGroups;     // release[kGroups]
  uint64_t* q_full = empty + C::kGroups;
  uint64_t* s_full = q_full + 1;           // [4]
  uint64_t* p_full = s_full + 4;           // [4]
  uint64_t* o_done = p_full + 4;           // [4]
  uint64_t* staged = o_done + 4;           // [4]
  uint64_t* drain = staged + 4;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WQ4 w = q4_work(n_qt, n_units, n_kt, BH, H, band, CAUSAL);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kGroups; ++i) {
      mbar_init(&full[i], 1);    // one expect-tx arrival per group
      mbar_init(&empty[i], 2);   // one commit per issuing warp
    }
    mbar_init(q_full, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
      mbar_init(&staged[i], 128);
    }
    mbar_init(drain, 2);         // one commit per issuing warp
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 17) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  if (warp == 16 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const CtaGuard g{abort_flag, g_status_q4, wc.epoch, wc.limit_us};

  // Roles.  Warp 17 frees TMEM after every TMEM user has passed the end barrier.
  if (warp >= 16) {
    if (warp == 16) {
      if (lane == 0) q4_producer(w, smem, full, empty, q_full, &tmQ, &tmK, &tmV, g);
    } else if (warp == 17 || warp == 18) {
      q4_mma<FD>(w, warp - 17, tmem, smem_u32(smem), full, empty, q_full, s_full, p_full, o_done, ks, idesc_pv, g);
      tc_commit_w(drain);   // every MMA issued above has finished before TMEM is released
      mbar_drain(drain, 0);
      __syncwarp();
      tc_fence_before();
      named_bar_sync(1, 512 + 64);
      tc_fence_after();
      if (warp == 17) tmem_dealloc(tmem, 512);
    }
  } else {
    q4_softmax<CAUSAL>(w, warp >> 2, tmem, smem, s_full, p_full, o_done, staged, &tmO, lse, N, scale_log2, g);
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, 512 + 64);
  }
}

template <bool CAUSAL>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk64, const CUtensorMap& tv64, const CUtensorMap& to,
                     float* lse, const Shape& s, const WaitCfg& wc, cudaStream_t st) {
  using C = Q4;
  auto kern = s.d == 64 ? fa_fwd_q4_kernel<CAUSAL, true> : fa_fwd_q4_kernel<CAUSAL, false>;
  const cudaError_t e =
      prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, C::kThreads, 0);
  if (e != cudaSuccess) return e;
  const int n_qt = (s.N + 127) / 128;
  const int n_units = (n_qt + 3) / 4;
  const int n_kt = (s.N + 63) / 64;
  const float scale_log2 = static_cast<float>(static_cast<double>(s.scale) * 1.4426950408889634);
  const dim3 grid(static_cast<unsigned>(s.B) * s.H * n_units);
  kern<<<grid, C::kThreads, C::kSmemBytes, st>>>(tq, tk64, tv64, to, lse, s.N, n_qt, n_units, n_kt, s.B * s.H, s.H,
                                                 head_band(s.N, s.d), scale_log2, score_ksteps(s.d),
                                                 idesc_bf16(128, out_cols(s.d), false, true), wc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_q4(const CUtensorMap& tq, const CUtensorMap& tk64, const CUtensorMap& tv64,
                          const CUtensorMap& to, float* lse, const Shape& s, const WaitCfg& wc, cudaStream_t st) {
  return s.causal ? launch_t<true>(tq, tk64, tv64, to, lse, s, wc, st)
                  : launch_t<false>(tq, tk64, tv64, to, lse, s, wc, st);
}

cudaError_t fwd_q4_status(uint32_t* out, bool reset) {
  unsigned int v[2] = {0, 0};
  cudaError_t e = cudaMemcpyFromSymbol(v, g_status_q4, sizeof(v));
  if (e != cudaSuccess) return e;
  *out = v[0];
  if (reset && (v[0] | v[1]) != 0) {
    const unsigned int z[2] = {0, 0};
    e = cudaMemcpyToSymbol(g_status_q4, z, sizeof(z));
  }
  return e;
}

}  // namespace fa
