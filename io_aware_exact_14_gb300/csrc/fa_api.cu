// C-ABI layer of libfa.so: argument checks, TMA tensor-map encoding and
// dispatch to the kernels.  Every device step runs in the kernels of
// fa_fwd.cu / fa_bwd.cu; nothing here touches tensor data.
#include "fa.h"
#include "fa_internal.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

namespace fa {

// Launch ids start at 1 and skip 0 when the counter wraps (after 2^32 - 1
// launches): 0 is the abort word's "no launch gave up".
WaitCfg next_wait_cfg() {
  static std::atomic<uint32_t> counter{0};
  uint32_t e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  if (e == 0) e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  return WaitCfg{e, kDefaultWaitLimitUs, -1};
}

unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(fn);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

cudaError_t prepare_kernel(const void* kern, uint32_t smem_bytes, int threads, uint32_t regs_needed) {
  struct Entry {
    unsigned long long ctx;
    const void* kern;
  };
  static std::mutex mu;
  static Entry done[256];
  static int n_done = 0;
  const unsigned long long ctx = current_context_id();
  if (ctx != 0) {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
      if (done[i].ctx == ctx && done[i].kern == kern) return cudaSuccess;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes));
  if (e != cudaSuccess) return e;
  if (regs_needed > 0) {
    // the warpgroups' register split must fit the launch allocation, or the
    // warpgroups asking for more would wait forever in setmaxnreg.inc
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    if (static_cast<uint32_t>(attr.numRegs) * static_cast<uint32_t>(threads) < regs_needed)
      return cudaErrorInvalidConfiguration;
  }
  const unsigned long long ctx_now = ctx != 0 ? ctx : current_context_id();   // the calls above bind one
  if (ctx_now != 0) {
    std::lock_guard<std::mutex> lock(mu);
    bool seen = false;
    for (int i = 0; i < n_done && !seen; ++i) seen = done[i].ctx == ctx_now && done[i].kern == kern;
    if (!seen) {
      if (n_done == 256) n_done = 0;   // more kernels x contexts than ever expected: start over
      done[n_done++] = Entry{ctx_now, kern};
    }
  }
  return cudaSuccess;
}

cudaError_t sm_count(int* out) {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *out = c;
      return cudaSuccess;
    }
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cached[dev].store(sms, std::memory_order_relaxed);
  *out = sms;
  return cudaSuccess;
}

}  // namespace fa

namespace {

using fa::Shape;
using fa::Strides;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
unsigned int g_last_site = 0;
thread_local char g_detail[256] = "no error";

fa_status fail(const char* what, int code, const char* text) {
  std::snprintf(g_detail, sizeof(g_detail), "%s failed: %s (code %d)", what, text ? text : "?", code);
  return FA_ERR_CUDA;
}

bool load_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr) fail("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", 0, "not found");
  return g_encode != nullptr;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Span {
  const void* p;
  size_t bytes;
};

bool overlaps(const Span& a, const Span& b) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a.bytes && b.bytes && a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Sizes: B, H >= 1, N >= 0, d a multiple of 8 in [8, max_d], grid-size limits.
// The forward takes d up to 256; the other entry points up to 128.
fa_status check_sizes(int B, int H, int N, int d, int max_d = 128) {
  if (B < 1 || H < 1 || N < 0) return FA_ERR_INVALID_ARG;
  if (d < 8 || d > max_d || d % 8 != 0) return FA_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  const long long tiles = bh * ((static_cast<long long>(N) + 127) / 128);
  if (bh > INT32_MAX || tiles > INT32_MAX || bh * N > (1ll << 40)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status check_scale(float scale) {
  return (std::isfinite(scale) && scale > 0.f) ? FA_OK : FA_ERR_INVALID_ARG;
}

// Every tensor pointer non-null and 16-byte aligned; fp32 vectors 4-byte aligned.
fa_status check_ptrs(std::initializer_list<const void*> tensors, std::initializer_list<const void*> vecs) {
  for (const void* p : tensors)
    if (p == nullptr || !aligned(p, 16)) return FA_ERR_INVALID_ARG;
  for (const void* p : vecs)
    if (p == nullptr || !aligned(p, 4)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// No output may overlap an input or another output.
fa_status check_disjoint(std::initializer_list<Span> outs, std::initializer_list<Span> ins) {
  for (auto o = outs.begin(); o != outs.end(); ++o) {
    for (const Span& i : ins)
      if (overlaps(*o, i)) return FA_ERR_INVALID_ARG;
    for (auto o2 = o + 1; o2 != outs.end(); ++o2)
      if (overlaps(*o, *o2)) return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

// Encoded tensor maps, per thread: a map is a pure function of the base
// address, sizes, strides and box, so a call that repeats an earlier one's
// buffers reuses its maps instead of encoding them again.  Direct-mapped.
struct MapKey {
  const void* base;
  long long d, N, H, B, sn, sh, sb;
  unsigned box_rows;
  bool operator==(const MapKey& o) const {
    return base == o.base && d == o.d && N == o.N && H == o.H && B == o.B && sn == o.sn && sh == o.sh &&
           sb == o.sb && box_rows == o.box_rows;
  }
};
struct MapSlot {
  bool valid;
  MapKey key;
  CUtensorMap map;
};
constexpr int kMapSlots = 64;
thread_local MapSlot t_maps[kMapSlots];

size_t map_slot(const MapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
  for (long long v : {k.d, k.N, k.H, k.B, k.sn, k.sh, k.sb, static_cast<long long>(k.box_rows)})
    h = (h ^ static_cast<uint64_t>(v)) * 0x100000001B3ull;
  return static_cast<size_t>(h >> 40) % kMapSlots;
}

// 4-D view {d, N, H, B} of a [B, H, N, d] bf16 tensor with element strides
// `st` (d contiguous); boxes of 64 x 128 rows with the 128-byte swizzle the
// tensor-core descriptors expect.  Rows past N and columns past d read as
// zero and are clipped on store.
fa_status make_map(CUtensorMap* m, const void* base, const Shape& s, const Strides& st, unsigned box_rows = 128) {
  const MapKey key{base, s.d, s.N, s.H, s.B, st.n, st.h, st.b, box_rows};
  MapSlot& slot = t_maps[map_slot(key)];
  if (slot.valid && slot.key == key) {
    *m = slot.map;
    return FA_OK;
  }
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(s.d), static_cast<cuuint64_t>(s.N),
                              static_cast<cuuint64_t>(s.H), static_cast<cuuint64_t>(s.B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n) * 2, static_cast<cuuint64_t>(st.h) * 2,
                                 static_cast<cuuint64_t>(st.b) * 2};
  const cuuint32_t box[4] = {64, box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail("cuTensorMapEncodeTiled", static_cast<int>(r), "invalid tensor map");
  slot.valid = true;
  slot.key = key;
  slot.map = *m;
  return FA_OK;
}

fa_status make_map(CUtensorMap* m, const void* base, const Shape& s) {
  return make_map(m, base, s, fa::contiguous_strides(s));
}

// A caller's strides (NULL: contiguous [B, H, N, d]).  Each stride must be a
// positive multiple of 8 elements (16 bytes, the copy engine's rule) below
// 2^37, with rows at least d apart.
fa_status read_strides(const fa_strides* in, const Shape& s, Strides& out) {
  if (in == nullptr) {
    out = fa::contiguous_strides(s);
    return FA_OK;
  }
  out = Strides{in->b, in->h, in->n};
  for (long long x : {out.b, out.h, out.n})
    if (x <= 0 || (x & 7) != 0 || x >= (1ll << 37)) return FA_ERR_INVALID_ARG;
  if (out.n < s.d) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Element span [0, extent) covered by a strided [B, H, N, d] view.
long long view_extent(const Shape& s, const Strides& st) {
  return (s.B - 1) * st.b + (s.H - 1) * st.h + (s.N - 1) * st.n + s.d;
}

// Can some element of view a equal one of view b?  Both views have the same
// sizes.  When they also share strides that nest (each stride at least the
// span of the dimensions with smaller strides), a common element exists iff
// the base offset (in elements) is sum_k delta_k stride_k + delta_c with
// |delta_k| < size_k and |delta_c| < d, which a short search decides (packed
// layouts such as [B, N, 3, H, d] pass); otherwise overlapping spans count as
// overlap.
bool views_overlap(const void* a, const Strides& sa, const void* b, const Strides& sb, const Shape& s) {
  const long long ea = view_extent(s, sa) * 2, eb = view_extent(s, sb) * 2;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  if (!(a0 < b0 + eb && b0 < a0 + ea)) return false;
  if (!(sa.b == sb.b && sa.h == sb.h && sa.n == sb.n)) return true;
  long long diff = static_cast<long long>(b0 > a0 ? b0 - a0 : a0 - b0);
  if (diff & 1) return true;
  diff /= 2;
  struct Dim { long long stride, size; };
  Dim dims[3] = {{sa.b, s.B}, {sa.h, s.H}, {sa.n, s.N}};
  for (int i = 0; i < 3; ++i)   // by decreasing stride
    for (int j = i + 1; j < 3; ++j)
      if (dims[j].stride > dims[i].stride) { const Dim t = dims[i]; dims[i] = dims[j]; dims[j] = t; }
  long long inner = s.d;   // span of the dimensions below the current one
  for (int i = 2; i >= 0; --i) {
    if (dims[i].stride < inner) return true;   // not nested: stay conservative
    inner += (dims[i].size - 1) * dims[i].stride;
  }
  // search delta_k in {floor(r / stride), floor(r / stride) + 1} level by level
  struct Frame { int level; long long r; };
  Frame stack[16];
  int top = 0;
  stack[top++] = {0, diff};
  while (top > 0) {
    const Frame f = stack[--top];
    if (f.level == 3) {
      if (f.r > -s.d && f.r < s.d) return true;
      continue;
    }
    const long long st = dims[f.level].stride, sz = dims[f.level].size;
    long long q = f.r >= 0 ? f.r / st : -((-f.r + st - 1) / st);
    for (long long dq = q; dq <= q + 1; ++dq)
      if (dq > -sz && dq < sz && top < 16) stack[top++] = {f.level + 1, f.r - dq * st};
  }
  return false;
}

struct TView {
  const void* p;
  Strides st;
};

// No output view may overlap an input view or another output view.
fa_status check_views_disjoint(std::initializer_list<TView> outs, std::initializer_list<TView> ins,
                               const Shape& s) {
  for (auto o = outs.begin(); o != outs.end(); ++o) {
    for (const TView& i : ins)
      if (views_overlap(o->p, o->st, i.p, i.st, s)) return FA_ERR_INVALID_ARG;
    for (auto o2 = o + 1; o2 != outs.end(); ++o2)
      if (views_overlap(o->p, o->st, o2->p, o2->st, s)) return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

size_t tensor_bytes(const Shape& s) { return static_cast<size_t>(s.B) * s.H * s.N * s.d * 2; }
size_t vec_bytes(const Shape& s) { return static_cast<size_t>(s.B) * s.H * s.N * 4; }
size_t workspace_need(const Shape& s) { return (vec_bytes(s) + 255) & ~size_t(255); }

#define FA_TRY(expr)                      \
  do {                                    \
    const fa_status st_ = (expr);         \
    if (st_ != FA_OK) return st_;         \
  } while (0)

fa_status cuda_status(cudaError_t e, const char* what) {
  return e == cudaSuccess ? FA_OK : fail(what, static_cast<int>(e), cudaGetErrorString(e));
}

// 3-D view {D, Nq, Z} of fp32 rows (split-KV partial outputs, Z = splits *
// B*H, D the kernel's padded head dim); boxes of 32 floats (128 bytes) x 128
// rows, 128-byte swizzle.
fa_status make_map_f32(CUtensorMap* m, const void* base, int d, int Nq, long long Z, unsigned box_rows = 128) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Nq), static_cast<cuuint64_t>(Z)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(Nq) * d * 4};
  const cuuint32_t box[3] = {32, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : fail("cuTensorMapEncodeTiled", static_cast<int>(r), "invalid tensor map");
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// FP8: sizes (d a multiple of 16 in [16, 256], the copy engine's 16-byte row
// rule for 1-byte elements), the transposed-V row pitch, and 4-D maps of
// e4m3 codes with 128 x 128 boxes.
fa_status check_sizes_fp8(int B, int H, int N, int d) {
  FA_TRY(check_sizes(B, H, N, d, fa::kMaxHeadDim));
  return d % 16 == 0 ? FA_OK : FA_ERR_UNSUPPORTED;
}

long long fp8_vt_ld(int N) { return (static_cast<long long>(N) + 15) / 16 * 16; }

fa_status make_map_u8(CUtensorMap* m, const void* base, const cuuint64_t (&dims)[4], const cuuint64_t (&strides)[3],
                      unsigned box_rows = 128) {
  const cuuint32_t box[4] = {128, box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : fail("cuTensorMapEncodeTiled", static_cast<int>(r), "invalid tensor map");
}

// Split-KV workspace: fp32 partial O [n, B*H, Nq, D] (D = kernel_dim(d): the
// kernel writes its padded columns, zeros), then fp32 partial LSE [n, B*H, Nq].
struct SplitPlan {
  int kt_per_split, n_splits;
  size_t o_bytes, lse_bytes;
};

// width: the partial rows' floats (the kernel width of d; 128 for e4m3);
// each chunk writes `reps` partial results (fa::splitkv_replicas).
fa_status split_plan(int B, int H, int Nq, int Nk, int width, int reps, int want, SplitPlan& p) {
  int sms = 0;
  if (want <= 0) FA_TRY(cuda_status(fa::sm_count(&sms), "reading the SM count"));
  fa::splitkv_chunks(B, H, Nq, Nk, want, sms, p.kt_per_split, p.n_splits);
  const size_t rows = static_cast<size_t>(B) * H * Nq * p.n_splits * reps;
  p.o_bytes = round256(rows * width * 4);
  p.lse_bytes = round256(rows * 4);
  return FA_OK;
}

// Strides of every tensor of a backward call: q, k, v, o, dO, dq, dk, dv.
struct BwdStrides {
  Strides q, k, v, o, dO, dq, dk, dv;
};

BwdStrides contiguous_bwd(const Shape& s) {
  const Strides c = fa::contiguous_strides(s);
  return BwdStrides{c, c, c, c, c, c, c, c};
}

// No dropout: threshold 0 selects the plain kernels.
const fa::DropArgs kNoDrop = fa::no_drop_args();

// The dropout contract of fa.h: t = round(256 p) (p in [0, 1)), clamped to
// 255; kept entries scaled by 256 / (256 - t).
fa_status read_dropout(const fa_dropout* in, fa::DropArgs& out) {
  if (in == nullptr) return FA_ERR_INVALID_ARG;
  const float p = in->p;
  if (!(p >= 0.f && p < 1.f)) return FA_ERR_INVALID_ARG;   // also rejects NaN
  int t = static_cast<int>(std::floor(256.0 * static_cast<double>(p) + 0.5));
  t = t < 0 ? 0 : (t > 255 ? 255 : t);
  out = fa::make_drop_args(in->seed, in->offset, t);
  return FA_OK;
}

// Wide heads (d > 128): every map the three launches use; `which` = 0 for
// the dK/dV maps, 1 for the dQ maps (outputs not in use stay unencoded).
fa_status wide_maps(fa::WideBwdMaps& m, const void* q, const void* k, const void* v, const void* dO, void* dq,
                    void* dk, void* dv, const Shape& s, const BwdStrides& t, int which) {
  if (which == 0) {
    FA_TRY(make_map(&m.k128, k, s, t.k));
    FA_TRY(make_map(&m.v128, v, s, t.v));
    FA_TRY(make_map(&m.q64, q, s, t.q, 64));
    FA_TRY(make_map(&m.do64, dO, s, t.dO, 64));
    FA_TRY(make_map(&m.dk128, dk, s, t.dk));
    FA_TRY(make_map(&m.dv128, dv, s, t.dv));
  } else {
    FA_TRY(make_map(&m.q128, q, s, t.q));
    FA_TRY(make_map(&m.do128, dO, s, t.dO));
    FA_TRY(make_map(&m.k64, k, s, t.k, 64));
    FA_TRY(make_map(&m.v64, v, s, t.v, 64));
    FA_TRY(make_map(&m.dq128, dq, s, t.dq));
  }
  return FA_OK;
}

fa_status dkdv_checked(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                       const float* Dvec, void* dk, void* dv, const Shape& s, const BwdStrides& t,
                       cudaStream_t st, const fa::DropArgs& drop = kNoDrop) {
  if (!load_encoder()) return FA_ERR_CUDA;
  if (s.d > 128) {
    fa::WideBwdMaps m;
    FA_TRY(wide_maps(m, q, k, v, dO, nullptr, dk, dv, s, t, 0));
    return cuda_status(fa::launch_bwd_d256_dkdv(m, lse, Dvec, s, drop, st), "wide-head dK/dV kernel launch");
  }
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  FA_TRY(make_map(&tq, q, s, t.q));
  FA_TRY(make_map(&tk, k, s, t.k));
  FA_TRY(make_map(&tv, v, s, t.v));
  FA_TRY(make_map(&tdo, dO, s, t.dO));
  FA_TRY(make_map(&tdk, dk, s, t.dk));
  FA_TRY(make_map(&tdv, dv, s, t.dv));
  return cuda_status(fa::launch_bwd_dkdv(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, s, drop, fa::next_wait_cfg(), st),
                     "dK/dV kernel launch");
}

fa_status dq_checked(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                     const float* Dvec, void* dq, const Shape& s, const BwdStrides& t, cudaStream_t st,
                     const fa::DropArgs& drop = kNoDrop) {
  if (!load_encoder()) return FA_ERR_CUDA;
  if (s.d > 128) {
    fa::WideBwdMaps m;
    FA_TRY(wide_maps(m, q, k, v, dO, dq, nullptr, nullptr, s, t, 1));
    return cuda_status(fa::launch_bwd_d256_dq(m, lse, Dvec, s, drop, st), "wide-head dQ kernel launch");
  }
  CUtensorMap tq, tk, tv, tdo, tdq;
  FA_TRY(make_map(&tq, q, s, t.q));
  FA_TRY(make_map(&tk, k, s, t.k));
  FA_TRY(make_map(&tv, v, s, t.v));
  FA_TRY(make_map(&tdo, dO, s, t.dO));
  FA_TRY(make_map(&tdq, dq, s, t.dq));
  return cuda_status(fa::launch_bwd_dq(tq, tk, tv, tdo, tdq, lse, Dvec, s, drop, fa::next_wait_cfg(), st),
                     "dQ kernel launch");
}

Span view_span(const void* p, const Shape& s, const Strides& st) {
  return Span{p, static_cast<size_t>(view_extent(s, st)) * 2};
}

fa_status fwd_impl(const void* q, const fa_strides* qs, const void* k, const fa_strides* ks, const void* v,
                   const fa_strides* vs, void* o, const fa_strides* os, float* lse, int B, int H, int N, int d,
                   float scale, int causal, cudaStream_t stream, const fa::DropArgs& drop = kNoDrop,
                   const fa::WaitCfg* wait = nullptr) {
  FA_TRY(check_sizes(B, H, N, d, wait == nullptr ? fa::kMaxHeadDim : 128));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({q, k, v, o}, {lse}));
  FA_TRY(check_scale(scale));
  const Shape s{B, H, N, d, scale, causal ? 1 : 0};
  Strides Sq, Sk, Sv, So;
  FA_TRY(read_strides(qs, s, Sq));
  FA_TRY(read_strides(ks, s, Sk));
  FA_TRY(read_strides(vs, s, Sv));
  FA_TRY(read_strides(os, s, So));
  FA_TRY(check_views_disjoint({{o, So}}, {{q, Sq}, {k, Sk}, {v, Sv}}, s));
  FA_TRY(check_disjoint({{lse, vec_bytes(s)}}, {view_span(q, s, Sq), view_span(k, s, Sk), view_span(v, s, Sv),
                                                 view_span(o, s, So)}));
  if (!load_encoder()) return FA_ERR_CUDA;
  CUtensorMap tq, tk, tv, to;
  FA_TRY(make_map(&tq, q, s, Sq));
  FA_TRY(make_map(&tk, k, s, Sk));
  FA_TRY(make_map(&tv, v, s, Sv));
  FA_TRY(make_map(&to, o, s, So));
  if (d > 128)
    return cuda_status(fa::launch_fwd_d256(tq, tk, tv, to, lse, s, drop, fa::next_wait_cfg(), stream),
                       "forward kernel launch");
  if (d <= 64 && drop.t4 == 0 && wait == nullptr) {   // narrow heads: four query tiles per CTA
    CUtensorMap tk64, tv64;
    FA_TRY(make_map(&tk64, k, s, Sk, 64));
    FA_TRY(make_map(&tv64, v, s, Sv, 64));
    return cuda_status(fa::launch_fwd_q4(tq, tk64, tv64, to, lse, s, fa::next_wait_cfg(), stream),
                       "forward kernel launch");
  }
  return cuda_status(fa::launch_fwd(tq, tk, tv, to, lse, s, drop, wait ? *wait : fa::next_wait_cfg(), stream),
                     "forward kernel launch");
}

fa_status bwd_impl(const void* q, const fa_strides* qs, const void* k, const fa_strides* ks, const void* v,
                   const fa_strides* vs, const void* o, const fa_strides* os, const float* lse, const void* dO,
                   const fa_strides* dos, void* dq, const fa_strides* dqs, void* dk, const fa_strides* dks,
                   void* dv, const fa_strides* dvs, int B, int H, int N, int d, float scale, int causal,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream,
                   const fa::DropArgs& drop = kNoDrop) {
  FA_TRY(check_sizes(B, H, N, d, fa::kMaxHeadDim));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({q, k, v, o, dO, dq, dk, dv}, {lse}));
  FA_TRY(check_scale(scale));
  const Shape s{B, H, N, d, scale, causal ? 1 : 0};
  BwdStrides t;
  FA_TRY(read_strides(qs, s, t.q));
  FA_TRY(read_strides(ks, s, t.k));
  FA_TRY(read_strides(vs, s, t.v));
  FA_TRY(read_strides(os, s, t.o));
  FA_TRY(read_strides(dos, s, t.dO));
  FA_TRY(read_strides(dqs, s, t.dq));
  FA_TRY(read_strides(dks, s, t.dk));
  FA_TRY(read_strides(dvs, s, t.dv));
  const size_t need = workspace_need(s);
  if (workspace == nullptr || !aligned(workspace, 16) || workspace_bytes < need) return FA_ERR_WORKSPACE;
  FA_TRY(check_views_disjoint({{dq, t.dq}, {dk, t.dk}, {dv, t.dv}},
                              {{q, t.q}, {k, t.k}, {v, t.v}, {o, t.o}, {dO, t.dO}}, s));
  const size_t vb = vec_bytes(s);
  FA_TRY(check_disjoint({{workspace, need}},
                        {view_span(q, s, t.q), view_span(k, s, t.k), view_span(v, s, t.v), view_span(o, s, t.o),
                         view_span(dO, s, t.dO), view_span(dq, s, t.dq), view_span(dk, s, t.dk),
                         view_span(dv, s, t.dv), {lse, vb}}));
  FA_TRY(check_disjoint({{lse, vb}}, {view_span(dq, s, t.dq), view_span(dk, s, t.dk), view_span(dv, s, t.dv)}));
  float* Dvec = static_cast<float*>(workspace);
  FA_TRY(cuda_status(fa::launch_bwd_preprocess(o, t.o, dO, t.dO, Dvec, s, stream), "preprocess kernel launch"));
  FA_TRY(dkdv_checked(q, k, v, lse, dO, Dvec, dk, dv, s, t, stream, drop));
  return dq_checked(q, k, v, lse, dO, Dvec, dq, s, t, stream, drop);
}

}  // namespace

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, struct CUstream_st* stream) {
  return fwd_impl(q, nullptr, k, nullptr, v, nullptr, o, nullptr, lse, B, H, N, d, scale, causal, stream);
}

fa_status fa_fwd_strided(const void* q, const fa_strides* q_st, const void* k, const fa_strides* k_st,
                         const void* v, const fa_strides* v_st, void* o, const fa_strides* o_st, float* lse,
                         int B, int H, int N, int d, float scale, int causal, struct CUstream_st* stream) {
  return fwd_impl(q, q_st, k, k_st, v, v_st, o, o_st, lse, B, H, N, d, scale, causal, stream);
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                         int Nk, int d, float scale, int causal, int num_splits, void* workspace,
                         size_t workspace_bytes, struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, Nq, d, fa::kMaxHeadDim));
  FA_TRY(check_sizes(B, H, Nk, d, fa::kMaxHeadDim));
  if (Nq == 0) return FA_OK;
  FA_TRY(check_ptrs({q, o}, {lse}));
  if (Nk > 0) FA_TRY(check_ptrs({k, v}, {}));   // never read when there are no keys
  FA_TRY(check_scale(scale));
  SplitPlan p;
  const int reps = fa::splitkv_replicas(Nq, d, false);
  FA_TRY(split_plan(B, H, Nq, Nk, fa::kernel_dim(d), reps, num_splits, p));
  if (static_cast<long long>(B) * H * p.n_splits * std::max((Nq + 127) / 128, reps) > INT32_MAX)
    return FA_ERR_UNSUPPORTED;   // the grid, and the partial results' z coordinate
  const size_t need = p.n_splits > 0 ? p.o_bytes + p.lse_bytes : 0;
  if (need > 0 && (workspace == nullptr || !aligned(workspace, 16) || workspace_bytes < need)) return FA_ERR_WORKSPACE;
  const Shape sq{B, H, Nq, d, scale, causal ? 1 : 0}, sk{B, H, Nk, d, scale, 0};
  const size_t qb = tensor_bytes(sq), kb = tensor_bytes(sk);
  FA_TRY(check_disjoint({{o, qb}, {lse, vec_bytes(sq)}, {workspace, need}}, {{q, qb}, {k, kb}, {v, kb}}));
  if (!load_encoder()) return FA_ERR_CUDA;
  CUtensorMap tq, tk, tv, top;
  const unsigned rows_box = reps > 1 ? fa::kRepRows : 128;
  FA_TRY(make_map(&tq, q, sq, fa::contiguous_strides(sq), rows_box));
  if (p.n_splits > 0) {
    FA_TRY(make_map(&tk, k, sk));
    FA_TRY(make_map(&tv, v, sk));
    FA_TRY(make_map_f32(&top, workspace, fa::kernel_dim(d), Nq, static_cast<long long>(p.n_splits) * reps * B * H,
                        rows_box));
  } else {
    tk = tq;
    tv = tq;
    top = tq;
  }
  const float* o_part = static_cast<const float*>(workspace);
  float* lse_part = p.n_splits > 0 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + p.o_bytes) : nullptr;
  return cuda_status(fa::launch_fwd_splitkv(tq, tk, tv, top, o_part, lse_part, o, lse, sq, Nk, p.n_splits,
                                            p.kt_per_split, fa::next_wait_cfg(), stream),
                     "split-KV forward launch");
}

size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (check_sizes(B, H, Nq, d, fa::kMaxHeadDim) != FA_OK || check_sizes(B, H, Nk, d, fa::kMaxHeadDim) != FA_OK ||
      Nq <= 0 || Nk <= 0)
    return 0;
  SplitPlan p;
  if (split_plan(B, H, Nq, Nk, fa::kernel_dim(d), fa::splitkv_replicas(Nq, d, false), num_splits, p) != FA_OK ||
      p.n_splits == 0)
    return 0;
  return p.o_bytes + p.lse_bytes;
}

fa_status fa_fwd_fp8_splitkv(const void* q8, const void* k8, const void* vt8, const float* descale_q,
                             const float* descale_k, const float* descale_v, void* o, float* lse, int B, int H,
                             int Nq, int Nk, int d, float scale, int causal, int num_splits, void* workspace,
                             size_t workspace_bytes, struct CUstream_st* stream) {
  FA_TRY(check_sizes_fp8(B, H, Nq, d));
  FA_TRY(check_sizes_fp8(B, H, Nk, d));
  if (Nq == 0) return FA_OK;
  FA_TRY(check_ptrs({q8, o}, {descale_q, descale_k, descale_v, lse}));
  if (Nk > 0) FA_TRY(check_ptrs({k8, vt8}, {}));   // never read when there are no keys
  FA_TRY(check_scale(scale));
  SplitPlan p;
  const int reps = fa::splitkv_replicas(Nq, d, true);
  const int width = d > 128 ? 256 : 128;   // partial rows: the e4m3 kernel's width
  FA_TRY(split_plan(B, H, Nq, Nk, width, reps, num_splits, p));
  if (static_cast<long long>(B) * H * p.n_splits * std::max((Nq + 127) / 128, reps) > INT32_MAX)
    return FA_ERR_UNSUPPORTED;   // the grid, and the partial results' z coordinate
  const size_t need = p.n_splits > 0 ? p.o_bytes + p.lse_bytes : 0;
  if (need > 0 && (workspace == nullptr || !aligned(workspace, 16) || workspace_bytes < need)) return FA_ERR_WORKSPACE;
  const Shape sq{B, H, Nq, d, scale, causal ? 1 : 0};
  const size_t q_bytes = tensor_bytes(sq) / 2, k_bytes = static_cast<size_t>(B) * H * Nk * d;
  const size_t vt_bytes = static_cast<size_t>(B) * H * d * fp8_vt_ld(Nk), ds_bytes = static_cast<size_t>(B) * H * 4;
  FA_TRY(check_disjoint({{o, tensor_bytes(sq)}, {lse, vec_bytes(sq)}, {workspace, need}},
                        {{q8, q_bytes}, {k8, k_bytes}, {vt8, vt_bytes}, {descale_q, ds_bytes}, {descale_k, ds_bytes},
                         {descale_v, ds_bytes}}));
  const float* o_part = static_cast<const float*>(workspace);
  float* lse_part = p.n_splits > 0 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + p.o_bytes) : nullptr;
  if (p.n_splits > 0) {
    if (!load_encoder()) return FA_ERR_CUDA;
    const cuuint64_t dB = B, dH = H, dQ = Nq, dK = Nk, dd = d, ld = static_cast<cuuint64_t>(fp8_vt_ld(Nk));
    const cuuint64_t q_dims[4] = {dd, dQ, dH, dB}, q_str[3] = {dd, dQ * dd, dH * dQ * dd};
    const cuuint64_t k_dims[4] = {dd, dK, dH, dB}, k_str[3] = {dd, dK * dd, dH * dK * dd};
    const cuuint64_t vt_dims[4] = {dK, dd, dH, dB}, vt_str[3] = {ld, dd * ld, dH * dd * ld};
    CUtensorMap tq, tk, tvt, top;
    const unsigned rows_box = reps > 1 ? fa::kRepRows : 128;
    FA_TRY(make_map_u8(&tq, q8, q_dims, q_str, rows_box));
    FA_TRY(make_map_u8(&tk, k8, k_dims, k_str));
    FA_TRY(make_map_u8(&tvt, vt8, vt_dims, vt_str));
    FA_TRY(make_map_f32(&top, workspace, width, Nq, static_cast<long long>(p.n_splits) * reps * B * H, rows_box));
    FA_TRY(cuda_status(fa::launch_fwd_fp8_split(tq, tk, tvt, top, descale_q, descale_k, descale_v, lse_part, sq, Nk,
                                                p.n_splits, p.kt_per_split, fa::next_wait_cfg(), stream),
                       "FP8 split-KV forward launch"));
  }
  return cuda_status(fa::launch_fwd_merge(o_part, lse_part, o, lse, sq, p.n_splits * reps, width, stream),
                     "split-KV merge launch");
}

size_t fa_fwd_fp8_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (check_sizes_fp8(B, H, Nq, d) != FA_OK || check_sizes_fp8(B, H, Nk, d) != FA_OK || Nq <= 0 || Nk <= 0) return 0;
  SplitPlan p;
  if (split_plan(B, H, Nq, Nk, d > 128 ? 256 : 128, fa::splitkv_replicas(Nq, d, true), num_splits, p) != FA_OK ||
      p.n_splits == 0)
    return 0;
  return p.o_bytes + p.lse_bytes;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_sizes(B, H, N, d, fa::kMaxHeadDim) != FA_OK || N <= 0) return 0;
  return workspace_need(Shape{B, H, N, d, 1.f, 0});
}

fa_status fa_bwd_preprocess(const void* o, const void* dO, float* Dvec, int B, int H, int N, int d,
                            struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, N, d, fa::kMaxHeadDim));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({o, dO}, {Dvec}));
  const Shape s{B, H, N, d, 1.f, 0};
  const size_t tb = tensor_bytes(s);
  FA_TRY(check_disjoint({{Dvec, vec_bytes(s)}}, {{o, tb}, {dO, tb}}));
  return cuda_status(fa::launch_bwd_preprocess(o, fa::contiguous_strides(s), dO, fa::contiguous_strides(s), Dvec, s, stream), "preprocess kernel launch");
}

fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                      const float* Dvec, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                      struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, N, d, fa::kMaxHeadDim));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({q, k, v, dO, dk, dv}, {lse, Dvec}));
  FA_TRY(check_scale(scale));
  const Shape s{B, H, N, d, scale, causal ? 1 : 0};
  const size_t tb = tensor_bytes(s), vb = vec_bytes(s);
  FA_TRY(check_disjoint({{dk, tb}, {dv, tb}}, {{q, tb}, {k, tb}, {v, tb}, {dO, tb}, {lse, vb}, {Dvec, vb}}));
  return dkdv_checked(q, k, v, lse, dO, Dvec, dk, dv, s, contiguous_bwd(s), stream);
}

fa_status fa_bwd_dq(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                    const float* Dvec, void* dq, int B, int H, int N, int d, float scale, int causal,
                    struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, N, d, fa::kMaxHeadDim));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({q, k, v, dO, dq}, {lse, Dvec}));
  FA_TRY(check_scale(scale));
  const Shape s{B, H, N, d, scale, causal ? 1 : 0};
  const size_t tb = tensor_bytes(s), vb = vec_bytes(s);
  FA_TRY(check_disjoint({{dq, tb}}, {{q, tb}, {k, tb}, {v, tb}, {dO, tb}, {lse, vb}, {Dvec, vb}}));
  return dq_checked(q, k, v, lse, dO, Dvec, dq, s, contiguous_bwd(s), stream);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                 void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  return bwd_impl(q, nullptr, k, nullptr, v, nullptr, o, nullptr, lse, dO, nullptr, dq, nullptr, dk, nullptr, dv,
                  nullptr, B, H, N, d, scale, causal, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_strided(const void* q, const fa_strides* q_st, const void* k, const fa_strides* k_st,
                         const void* v, const fa_strides* v_st, const void* o, const fa_strides* o_st,
                         const float* lse, const void* dO, const fa_strides* dO_st, void* dq,
                         const fa_strides* dq_st, void* dk, const fa_strides* dk_st, void* dv,
                         const fa_strides* dv_st, int B, int H, int N, int d, float scale, int causal,
                         void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  return bwd_impl(q, q_st, k, k_st, v, v_st, o, o_st, lse, dO, dO_st, dq, dq_st, dk, dk_st, dv, dv_st, B, H, N, d,
                  scale, causal, workspace, workspace_bytes, stream);
}

fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                         int d, float scale, int causal, const fa_dropout* dropout, struct CUstream_st* stream) {
  fa::DropArgs drop;
  FA_TRY(read_dropout(dropout, drop));
  return fwd_impl(q, nullptr, k, nullptr, v, nullptr, o, nullptr, lse, B, H, N, d, scale, causal, stream, drop);
}

fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, const fa_dropout* dropout, void* workspace, size_t workspace_bytes,
                         struct CUstream_st* stream) {
  fa::DropArgs drop;
  FA_TRY(read_dropout(dropout, drop));
  return bwd_impl(q, nullptr, k, nullptr, v, nullptr, o, nullptr, lse, dO, nullptr, dq, nullptr, dk, nullptr, dv,
                  nullptr, B, H, N, d, scale, causal, workspace, workspace_bytes, stream, drop);
}

size_t fa_fp8_vt_ld(int N) { return N > 0 ? static_cast<size_t>(fp8_vt_ld(N)) : 0; }

fa_status fa_fp8_quantize(const void* x, void* out, float* descale, int B, int H, int N, int d, int transpose,
                          int rotate, unsigned long long seed, struct CUstream_st* stream) {
  FA_TRY(check_sizes_fp8(B, H, N, d));
  if (rotate && d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({x, out}, {descale}));
  const Shape s{B, H, N, d, 1.f, 0};
  const size_t out_bytes = transpose ? static_cast<size_t>(B) * H * d * fp8_vt_ld(N) : tensor_bytes(s) / 2;
  FA_TRY(check_disjoint({{out, out_bytes}, {descale, static_cast<size_t>(B) * H * 4}}, {{x, tensor_bytes(s)}}));
  FA_TRY(check_disjoint({{out, out_bytes}}, {{descale, static_cast<size_t>(B) * H * 4}}));
  return cuda_status(fa::launch_fp8_quantize(x, out, descale, s, transpose != 0, fp8_vt_ld(N), rotate != 0, seed,
                                             stream),
                     "FP8 quantise launch");
}

fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* descale_q,
                     const float* descale_k, const float* descale_v, void* o, float* lse, int B, int H, int N, int d,
                     float scale, int causal, struct CUstream_st* stream) {
  FA_TRY(check_sizes_fp8(B, H, N, d));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({q8, k8, vt8, o}, {descale_q, descale_k, descale_v, lse}));
  FA_TRY(check_scale(scale));
  const Shape s{B, H, N, d, scale, causal ? 1 : 0};
  const size_t qk_bytes = tensor_bytes(s) / 2, vt_bytes = static_cast<size_t>(B) * H * d * fp8_vt_ld(N);
  const size_t ds_bytes = static_cast<size_t>(B) * H * 4;
  FA_TRY(check_disjoint({{o, tensor_bytes(s)}, {lse, vec_bytes(s)}},
                        {{q8, qk_bytes}, {k8, qk_bytes}, {vt8, vt_bytes}, {descale_q, ds_bytes},
                         {descale_k, ds_bytes}, {descale_v, ds_bytes}}));
  FA_TRY(check_disjoint({{o, tensor_bytes(s)}}, {{lse, vec_bytes(s)}}));
  if (!load_encoder()) return FA_ERR_CUDA;
  const cuuint64_t dB = B, dH = H, dN = N, dd = d, ld = static_cast<cuuint64_t>(fp8_vt_ld(N));
  CUtensorMap tq, tk, tvt, to;
  const cuuint64_t qk_dims[4] = {dd, dN, dH, dB}, qk_str[3] = {dd, dN * dd, dH * dN * dd};
  const cuuint64_t vt_dims[4] = {dN, dd, dH, dB}, vt_str[3] = {ld, dd * ld, dH * dd * ld};
  FA_TRY(make_map_u8(&tq, q8, qk_dims, qk_str));
  FA_TRY(make_map_u8(&tk, k8, qk_dims, qk_str));
  FA_TRY(make_map_u8(&tvt, vt8, vt_dims, vt_str));
  FA_TRY(make_map(&to, o, s));
  if (d > 128)   // wide heads: the one-query-tile kernel's e4m3 variant
    return cuda_status(fa::launch_fwd_fp8_wide(tq, tk, tvt, to, descale_q, descale_k, descale_v, lse, s,
                                               fa::next_wait_cfg(), stream),
                       "FP8 forward launch");
  return cuda_status(fa::launch_fwd_fp8(tq, tk, tvt, to, descale_q, descale_k, descale_v, lse, s,
                                        fa::next_wait_cfg(), stream),
                     "FP8 forward launch");
}

fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, N, d, fa::kMaxHeadDim));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({q, k, v, o, dO, dq, dk, dv}, {lse}));
  FA_TRY(check_scale(scale));
  const Shape s{B, H, N, d, scale, causal ? 1 : 0};
  if (static_cast<size_t>(B) * H * N > fa::kNoAllocRows) {
    std::snprintf(g_detail, sizeof(g_detail),
                  "fa_bwd_noalloc: B*H*N = %lld rows exceeds the built-in scratch of %zu rows; use fa_bwd",
                  static_cast<long long>(B) * H * N, fa::kNoAllocRows);
    return FA_ERR_WORKSPACE;
  }
  const size_t tb = tensor_bytes(s), vb = vec_bytes(s);
  FA_TRY(check_disjoint({{dq, tb}, {dk, tb}, {dv, tb}}, {{q, tb}, {k, tb}, {v, tb}, {o, tb}, {dO, tb}, {lse, vb}}));
  float* Dvec = nullptr;
  FA_TRY(cuda_status(fa::noalloc_scratch(&Dvec), "locating the built-in scratch (cudaGetSymbolAddress)"));
  FA_TRY(cuda_status(fa::launch_bwd_preprocess(o, fa::contiguous_strides(s), dO, fa::contiguous_strides(s), Dvec, s, stream), "preprocess kernel launch"));
  FA_TRY(dkdv_checked(q, k, v, lse, dO, Dvec, dk, dv, s, contiguous_bwd(s), stream));
  return dq_checked(q, k, v, lse, dO, Dvec, dq, s, contiguous_bwd(s), stream);
}

fa_status fa_debug_fwd_withhold(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                int N, int d, float scale, int causal, int withhold_group,
                                unsigned int wait_limit_us, struct CUstream_st* stream) {
  if (withhold_group < 0 || wait_limit_us == 0) return FA_ERR_INVALID_ARG;
  fa::WaitCfg wc = fa::next_wait_cfg();
  wc.limit_us = wait_limit_us;
  wc.withhold = withhold_group;
  return fwd_impl(q, nullptr, k, nullptr, v, nullptr, o, nullptr, lse, B, H, N, d, scale, causal, stream, kNoDrop,
                  &wc);
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK: success";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null, misaligned or overlapping pointer, or bad size/scale";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dim not a multiple of 8 in the entry point's range, or sizes exceed the limits";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call or kernel launch failed";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel gave up on a pipeline wait";
  }
  return "unknown fa_status";
}

fa_status fa_debug_status(int reset) {
  uint32_t a = 0, b = 0;
  cudaError_t e = fa::fwd_status(&a, reset != 0);
  if (e != cudaSuccess) return fail("reading the forward status word", e, cudaGetErrorString(e));
  e = fa::bwd_status(&b, reset != 0);
  if (e != cudaSuccess) return fail("reading the backward status word", e, cudaGetErrorString(e));
  uint32_t c = 0;
  e = fa::fp8_status(&c, reset != 0);
  if (e != cudaSuccess) return fail("reading the FP8 status word", e, cudaGetErrorString(e));
  uint32_t w = 0;
  e = fa::fwd_d256_status(&w, reset != 0);
  if (e != cudaSuccess) return fail("reading the wide-head forward status word", e, cudaGetErrorString(e));
  uint32_t x = 0;
  e = fa::bwd_d256_status(&x, reset != 0);
  if (e != cudaSuccess) return fail("reading the wide-head backward status word", e, cudaGetErrorString(e));
  uint32_t y = 0;
  e = fa::fwd_q4_status(&y, reset != 0);
  if (e != cudaSuccess) return fail("reading the narrow-head forward status word", e, cudaGetErrorString(e));
  g_last_site = a ? a : (b ? b : (c ? c : (w ? w : (x ? x : y))));
  return (a | b | c | w | x | y) ? FA_ERR_TIMEOUT : FA_OK;
}

unsigned int fa_debug_site(void) { return g_last_site; }

const char* fa_last_error_detail(void) { return g_detail; }

}  // extern "C"
