// C-ABI layer of libfa.so: argument checks, TMA tensor-map encoding and
// dispatch to the kernels.  Every device step runs in the kernels of
// fa_fwd.cu / fa_bwd.cu; nothing here touches tensor data.
#include "fa.h"
#include "fa_internal.h"

#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

namespace {

using fa::Shape;

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

// Sizes: B, H >= 1, N >= 0, d in {64, 128}, grid-size limits.
fa_status check_sizes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
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

// 3-D view {d, N, B*H} of a [B, H, N, d] bf16 tensor; boxes of 64 x 128 rows
// with the 128-byte swizzle the tensor-core descriptors expect.  Rows past N
// read as zero and are clipped on store.
fa_status make_map(CUtensorMap* m, const void* base, const Shape& s) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(s.d), static_cast<cuuint64_t>(s.N),
                              static_cast<cuuint64_t>(s.B) * s.H};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(s.d) * 2, static_cast<cuuint64_t>(s.N) * s.d * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : fail("cuTensorMapEncodeTiled", static_cast<int>(r), "invalid tensor map");
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

// 3-D view {d, Nq, Z} of fp32 rows (split-KV partial outputs, Z = splits *
// B*H); boxes of 32 floats (128 bytes) x 128 rows, 128-byte swizzle.
fa_status make_map_f32(CUtensorMap* m, const void* base, int d, int Nq, long long Z) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Nq), static_cast<cuuint64_t>(Z)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(Nq) * d * 4};
  const cuuint32_t box[3] = {32, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : fail("cuTensorMapEncodeTiled", static_cast<int>(r), "invalid tensor map");
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Split-KV workspace: fp32 partial O [n, B*H, Nq, d], then fp32 partial LSE [n, B*H, Nq].
struct SplitPlan {
  int kt_per_split, n_splits;
  size_t o_bytes, lse_bytes;
};

fa_status split_plan(int B, int H, int Nq, int Nk, int d, int want, SplitPlan& p) {
  int sms = 0;
  if (want <= 0) {
    int dev = 0;
    FA_TRY(cuda_status(cudaGetDevice(&dev), "cudaGetDevice"));
    FA_TRY(cuda_status(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute"));
  }
  fa::splitkv_chunks(B, H, Nq, Nk, want, sms, p.kt_per_split, p.n_splits);
  const size_t rows = static_cast<size_t>(B) * H * Nq * p.n_splits;
  p.o_bytes = round256(rows * d * 4);
  p.lse_bytes = round256(rows * 4);
  return FA_OK;
}

fa_status dkdv_checked(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                       const float* Dvec, void* dk, void* dv, const Shape& s, cudaStream_t st) {
  if (!load_encoder()) return FA_ERR_CUDA;
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  FA_TRY(make_map(&tq, q, s));
  FA_TRY(make_map(&tk, k, s));
  FA_TRY(make_map(&tv, v, s));
  FA_TRY(make_map(&tdo, dO, s));
  FA_TRY(make_map(&tdk, dk, s));
  FA_TRY(make_map(&tdv, dv, s));
  return cuda_status(fa::launch_bwd_dkdv(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, s, st), "dK/dV kernel launch");
}

fa_status dq_checked(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                     const float* Dvec, void* dq, const Shape& s, cudaStream_t st) {
  if (!load_encoder()) return FA_ERR_CUDA;
  CUtensorMap tq, tk, tv, tdo, tdq;
  FA_TRY(make_map(&tq, q, s));
  FA_TRY(make_map(&tk, k, s));
  FA_TRY(make_map(&tv, v, s));
  FA_TRY(make_map(&tdo, dO, s));
  FA_TRY(make_map(&tdq, dq, s));
  return cuda_status(fa::launch_bwd_dq(tq, tk, tv, tdo, tdq, lse, Dvec, s, st), "dQ kernel launch");
}

}  // namespace

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, N, d));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({q, k, v, o}, {lse}));
  FA_TRY(check_scale(scale));
  const Shape s{B, H, N, d, scale, causal ? 1 : 0};
  const size_t tb = tensor_bytes(s), vb = vec_bytes(s);
  FA_TRY(check_disjoint({{o, tb}, {lse, vb}}, {{q, tb}, {k, tb}, {v, tb}}));
  if (!load_encoder()) return FA_ERR_CUDA;
  CUtensorMap tq, tk, tv, to;
  FA_TRY(make_map(&tq, q, s));
  FA_TRY(make_map(&tk, k, s));
  FA_TRY(make_map(&tv, v, s));
  FA_TRY(make_map(&to, o, s));
  return cuda_status(fa::launch_fwd(tq, tk, tv, to, lse, s, stream), "forward kernel launch");
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                         int Nk, int d, float scale, int num_splits, void* workspace, size_t workspace_bytes,
                         struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, Nq, d));
  FA_TRY(check_sizes(B, H, Nk, d));
  if (Nq == 0) return FA_OK;
  FA_TRY(check_ptrs({q, o}, {lse}));
  if (Nk > 0) FA_TRY(check_ptrs({k, v}, {}));   // never read when there are no keys
  FA_TRY(check_scale(scale));
  SplitPlan p;
  FA_TRY(split_plan(B, H, Nq, Nk, d, num_splits, p));
  if (static_cast<long long>(B) * H * p.n_splits * ((Nq + 127) / 128) > INT32_MAX) return FA_ERR_UNSUPPORTED;
  const size_t need = p.n_splits > 0 ? p.o_bytes + p.lse_bytes : 0;
  if (need > 0 && (workspace == nullptr || !aligned(workspace, 16) || workspace_bytes < need)) return FA_ERR_WORKSPACE;
  const Shape sq{B, H, Nq, d, scale, 0}, sk{B, H, Nk, d, scale, 0};
  const size_t qb = tensor_bytes(sq), kb = tensor_bytes(sk);
  FA_TRY(check_disjoint({{o, qb}, {lse, vec_bytes(sq)}, {workspace, need}}, {{q, qb}, {k, kb}, {v, kb}}));
  if (!load_encoder()) return FA_ERR_CUDA;
  CUtensorMap tq, tk, tv, top;
  FA_TRY(make_map(&tq, q, sq));
  if (p.n_splits > 0) {
    FA_TRY(make_map(&tk, k, sk));
    FA_TRY(make_map(&tv, v, sk));
    FA_TRY(make_map_f32(&top, workspace, d, Nq, static_cast<long long>(p.n_splits) * B * H));
  } else {
    tk = tq;
    tv = tq;
    top = tq;
  }
  const float* o_part = static_cast<const float*>(workspace);
  float* lse_part = p.n_splits > 0 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + p.o_bytes) : nullptr;
  return cuda_status(fa::launch_fwd_splitkv(tq, tk, tv, top, o_part, lse_part, o, lse, sq, Nk, p.n_splits,
                                            p.kt_per_split, stream),
                     "split-KV forward launch");
}

size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (check_sizes(B, H, Nq, d) != FA_OK || check_sizes(B, H, Nk, d) != FA_OK || Nq <= 0 || Nk <= 0) return 0;
  SplitPlan p;
  if (split_plan(B, H, Nq, Nk, d, num_splits, p) != FA_OK || p.n_splits == 0) return 0;
  return p.o_bytes + p.lse_bytes;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_sizes(B, H, N, d) != FA_OK || N <= 0) return 0;
  return workspace_need(Shape{B, H, N, d, 1.f, 0});
}

fa_status fa_bwd_preprocess(const void* o, const void* dO, float* Dvec, int B, int H, int N, int d,
                            struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, N, d));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({o, dO}, {Dvec}));
  const Shape s{B, H, N, d, 1.f, 0};
  const size_t tb = tensor_bytes(s);
  FA_TRY(check_disjoint({{Dvec, vec_bytes(s)}}, {{o, tb}, {dO, tb}}));
  return cuda_status(fa::launch_bwd_preprocess(o, dO, Dvec, s, stream), "preprocess kernel launch");
}

fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                      const float* Dvec, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                      struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, N, d));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({q, k, v, dO, dk, dv}, {lse, Dvec}));
  FA_TRY(check_scale(scale));
  const Shape s{B, H, N, d, scale, causal ? 1 : 0};
  const size_t tb = tensor_bytes(s), vb = vec_bytes(s);
  FA_TRY(check_disjoint({{dk, tb}, {dv, tb}}, {{q, tb}, {k, tb}, {v, tb}, {dO, tb}, {lse, vb}, {Dvec, vb}}));
  return dkdv_checked(q, k, v, lse, dO, Dvec, dk, dv, s, stream);
}

fa_status fa_bwd_dq(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                    const float* Dvec, void* dq, int B, int H, int N, int d, float scale, int causal,
                    struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, N, d));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({q, k, v, dO, dq}, {lse, Dvec}));
  FA_TRY(check_scale(scale));
  const Shape s{B, H, N, d, scale, causal ? 1 : 0};
  const size_t tb = tensor_bytes(s), vb = vec_bytes(s);
  FA_TRY(check_disjoint({{dq, tb}}, {{q, tb}, {k, tb}, {v, tb}, {dO, tb}, {lse, vb}, {Dvec, vb}}));
  return dq_checked(q, k, v, lse, dO, Dvec, dq, s, stream);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                 void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, N, d));
  if (N == 0) return FA_OK;
  FA_TRY(check_ptrs({q, k, v, o, dO, dq, dk, dv}, {lse}));
  FA_TRY(check_scale(scale));
  const Shape s{B, H, N, d, scale, causal ? 1 : 0};
  const size_t need = workspace_need(s);
  if (workspace == nullptr || !aligned(workspace, 16) || workspace_bytes < need) return FA_ERR_WORKSPACE;
  const size_t tb = tensor_bytes(s), vb = vec_bytes(s);
  FA_TRY(check_disjoint({{dq, tb}, {dk, tb}, {dv, tb}, {workspace, need}},
                        {{q, tb}, {k, tb}, {v, tb}, {o, tb}, {dO, tb}, {lse, vb}}));
  float* Dvec = static_cast<float*>(workspace);
  FA_TRY(cuda_status(fa::launch_bwd_preprocess(o, dO, Dvec, s, stream), "preprocess kernel launch"));
  FA_TRY(dkdv_checked(q, k, v, lse, dO, Dvec, dk, dv, s, stream));
  return dq_checked(q, k, v, lse, dO, Dvec, dq, s, stream);
}

fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, struct CUstream_st* stream) {
  FA_TRY(check_sizes(B, H, N, d));
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
  FA_TRY(cuda_status(fa::launch_bwd_preprocess(o, dO, Dvec, s, stream), "preprocess kernel launch"));
  FA_TRY(dkdv_checked(q, k, v, lse, dO, Dvec, dk, dv, s, stream));
  return dq_checked(q, k, v, lse, dO, Dvec, dq, s, stream);
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK: success";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null, misaligned or overlapping pointer, or bad size/scale";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dim must be 64 or 128, or sizes exceed the limits";
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
  g_last_site = a ? a : b;
  return (a | b) ? FA_ERR_TIMEOUT : FA_OK;
}

unsigned int fa_debug_site(void) { return g_last_site; }

const char* fa_last_error_detail(void) { return g_detail; }

}  // extern "C"
