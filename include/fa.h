/*
 * fa.h -- C ABI of libfa.so: exact scaled-dot-product attention on one
 * NVIDIA GB300 (sm_103a), forward and backward, computed tile by tile with
 * running softmax statistics so that no N x N matrix is ever written to HBM.
 *
 * Sources (cited by page title and section):
 *   [TRITON-IO]  "FlashAttention的Triton实现：IO-aware注意力机制底层原理"
 *   [WHY-FAST]   "为什么Flash Attention能将注意力计算提速数倍而不损失精度"
 *   [KERNEL-101] "GPU Kernel 入门：Triton / FlashAttention"
 *
 * Conventions shared by every entry point
 *   - Tensors are row-major, contiguous, [B, H, N, d] bf16 (d innermost);
 *     row statistics (LSE, D) are [B, H, N] fp32.  Q, K, V share one N.
 *   - d must be a multiple of 8 from 8 to 256 for every entry point but
 *     the FP8 ones (a multiple of 16) and the deadlock-guard test hook (d up
 *     to 128, see there); else FA_ERR_UNSUPPORTED.  d <= 64 runs the d = 64 kernels,
 *     64 < d <= 128 the d = 128 ones and 128 < d <= 256 the wide-head
 *     (d = 256) ones: the missing columns are zero-filled on chip, never
 *     read from or written to memory, and the products that contract over d
 *     skip the all-zero 16-column steps.  N >= 0; N == 0 is a no-op that returns
 *     FA_OK.  B, H >= 1.  B*H*ceil(N/128) must fit in 2^31 - 1.
 *   - Every device pointer must be 16-byte aligned (fp32 vectors: 4-byte),
 *     outputs must not overlap inputs or each other; otherwise
 *     FA_ERR_INVALID_ARG.  The library never writes its inputs.
 *   - scale is the softmax scale applied to Q K^T; it must be finite and > 0
 *     (FA_ERR_INVALID_ARG otherwise).  The pages never write the scale; the
 *     usual choice is 1/sqrt(d).
 *   - causal != 0 keeps key j only for query rows i >= j.
 *   - Ownership: the caller allocates and frees every buffer, including the
 *     backward workspace.  The library holds no device allocation between
 *     calls and keeps no pointer after a call returns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t / CUstream; NULL
 *     is the legacy default stream).  The return value reports argument
 *     checks and launch errors (FA_ERR_CUDA: the launch failed; the CUDA
 *     error is left in the runtime's last-error slot).  Faults inside a
 *     kernel surface at the caller's next synchronisation.
 *   - No exception ever crosses this interface.
 *   - Stream capture: the kernels take their tensor maps and wait settings as
 *     launch parameters, so calls may be captured into a CUDA graph and
 *     replayed on the same buffers.  Make one call of each kind (same
 *     entry point, head-dim class and mask) before capturing: the first
 *     sets kernel attributes, which capture does not record.  A replayed
 *     launch reuses the wait epoch it was captured with, so after a kernel
 *     of that graph has given up on a wait (FA_ERR_TIMEOUT), reset the
 *     status (fa_debug_status(1)) before replaying it again.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t and CUstream are both `struct CUstream_st *` */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null/misaligned/overlapping pointer, bad size or scale */
  FA_ERR_UNSUPPORTED = 2,  /* head dim not a multiple of 8 in the entry point's range, or sizes beyond the limits */
  FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or a launch failed */
  FA_ERR_WORKSPACE = 4,    /* workspace missing, misaligned or too small */
  FA_ERR_TIMEOUT = 5       /* a kernel gave up on a wait (see fa_debug_status) */
} fa_status;

/*
 * Forward pass: O = softmax(scale * Q K^T [+ causal mask]) V, and
 * LSE_i = log(sum_j exp(scale * q_i . k_j)) over the unmasked keys (natural
 * log, fp32).  The pages' "exact attention": tiling plus the online softmax
 * reach the plain result up to rounding ([WHY-FAST] "分块计算（Tiling）",
 * "在线Softmax技巧"; [KERNEL-101] "FlashAttention 与在线 softmax：难点与解法").
 * LSE replaces the pages' separately saved (m, l) ([WHY-FAST] "分块计算（Tiling）"
 * saves both): LSE = m + ln l.
 *   q, k, v  in : bf16 [B, H, N, d]
 *   o        out: bf16 [B, H, N, d]
 *   lse      out: fp32 [B, H, N]
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int causal,
                 struct CUstream_st* stream);

/*
 * Split-KV forward for short query blocks against long key sequences, e.g.
 * decoding or a prefill chunk: the keys are cut into num_splits chunks of whole
 * 128-key tiles, each chunk's (O_s, LSE_s) is computed as in fa_fwd and the
 * chunks are merged with the two-block merge identity of [WHY-FAST]
 * "在线Softmax技巧" (LSE = log sum_s e^{LSE_s}, O = sum_s e^{LSE_s - LSE} O_s),
 * which reaches the same exact result.
 *   q          in : bf16 [B, H, Nq, d]
 *   k, v       in : bf16 [B, H, Nk, d]
 *   o          out: bf16 [B, H, Nq, d]
 *   lse        out: fp32 [B, H, Nq]  (Nk == 0: O = 0, LSE = -inf)
 *   causal     0: every query sees every key.  1: the query block is the
 *              last Nq positions of the Nk-long sequence (query i at
 *              position Nk - Nq + i, aligned to the end of the keys), and
 *              sees keys 0 .. Nk - Nq + i; a query with no such key (Nq >
 *              Nk) gets O = 0, LSE = -inf.  Nq == Nk is fa_fwd's causal mask.
 *              (The library's reading: the pages define the mask only for
 *              equal lengths.)
 *   num_splits  chunks wanted (<= 0: chosen from the SM count); the count
 *               used is at most ceil(Nk / 128), every chunk non-empty
 *   workspace   scratch for the chunks' fp32 (O_s, LSE_s), owned by the
 *               caller, 16-byte aligned, at least
 *               fa_fwd_splitkv_workspace_bytes(...) bytes (may be NULL when
 *               that is 0); FA_ERR_WORKSPACE otherwise
 * Nq == 0 is a no-op; k and v may be NULL when Nk == 0.  Sizes, alignment
 * and overlap rules as for fa_fwd, with Nq and Nk each in place of N.
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int Nq, int Nk, int d, float scale, int causal, int num_splits,
                         void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/*
 * Workspace bytes fa_fwd_splitkv needs for these arguments (the same
 * num_splits rule, on the current device): R * n_used * B*H*Nq*D fp32
 * partial outputs (D = 64 for d <= 64, 128 for d <= 128, else 256) plus
 * R * n_used * B*H*Nq fp32 partial LSE, each rounded up to 256 bytes, with
 * R = 4 for Nq <= 32 and d <= 64 (each chunk then writes one partial result
 * per quarter of its keys) and 1 otherwise.  0 for invalid sizes, Nq == 0
 * or Nk == 0.
 */
size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits);

/*
 * Element strides of a [B, H, N, d] bf16 view whose d elements are
 * contiguous, so any layout that permutes B, H and N (for example
 * [B, N, H, d], or q, k, v packed as [B, N, 3, H, d]) can be passed without a
 * copy: element (b, h, n, c) sits at base + b*b + h*h + n*n + c (in
 * elements).  Each stride is a positive multiple of 8 elements (the copy
 * engine's 16-byte rule) below 2^37, and n >= d; FA_ERR_INVALID_ARG
 * otherwise.  A NULL fa_strides pointer means the contiguous layout.  The row
 * statistics (LSE, D) stay contiguous fp32 [B, H, N].
 */
typedef struct {
  long long b, h, n;
} fa_strides;

/*
 * fa_fwd on strided views (see fa_strides).  Outputs must not share an
 * element with an input or with each other: views with identical strides are
 * checked element-exactly (so interleaved outputs are accepted), others by
 * their address spans.
 */
fa_status fa_fwd_strided(const void* q, const fa_strides* q_st, const void* k, const fa_strides* k_st,
                         const void* v, const fa_strides* v_st, void* o, const fa_strides* o_st, float* lse,
                         int B, int H, int N, int d, float scale, int causal, struct CUstream_st* stream);

/*
 * Bytes of device workspace fa_bwd needs: the fp32 row term D [B, H, N],
 * rounded up to 256 bytes.  Returns 0 for N <= 0 or invalid sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass of L(q, k, v) with upstream gradient dO = dL/dO, recomputing
 * the probabilities from the saved LSE instead of storing them
 * ([WHY-FAST] "反向传播中的重计算策略").  The gradients are the calculus of
 * the forward definition (the pages give none):
 *   dV = P^T dO, dP = dO V^T, D_i = sum_c dO_ic O_ic,
 *   dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
 * Runs fa_bwd_preprocess, fa_bwd_dkdv and fa_bwd_dq in that order on `stream`
 * (for d > 128, fa_bwd_dkdv is two launches, dV then dK: one CTA's tensor
 * memory holds one 128 x 256 fp32 accumulator next to its score tiles, so
 * the dK launch recomputes the scores the dV launch used).
 *   q, k, v, o, dO in : bf16 [B, H, N, d]; o and lse from fa_fwd
 *   lse            in : fp32 [B, H, N]
 *   dq, dk, dv     out: bf16 [B, H, N, d]
 *   workspace      scratch, >= fa_bwd_workspace_bytes(B, H, N, d) bytes,
 *                  16-byte aligned, owned by the caller; its contents on
 *                  return are the row term D (fp32 [B, H, N]).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, float scale, int causal,
                 void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/*
 * fa_bwd on strided views (see fa_strides and fa_fwd_strided); dq, dk, dv may
 * be interleaved (for example one [B, N, 3, H, d] buffer).
 */
fa_status fa_bwd_strided(const void* q, const fa_strides* q_st, const void* k, const fa_strides* k_st,
                         const void* v, const fa_strides* v_st, const void* o, const fa_strides* o_st,
                         const float* lse, const void* dO, const fa_strides* dO_st, void* dq,
                         const fa_strides* dq_st, void* dk, const fa_strides* dk_st, void* dv,
                         const fa_strides* dv_st, int B, int H, int N, int d, float scale, int causal,
                         void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/*
 * Dropout on the attention probabilities, fused into the kernels ([WHY-FAST]
 * "标准注意力机制的内存困局" names dropout among the steps a fused kernel
 * does on chip; the random-number contract is this library's):
 *   p       drop probability, 0 <= p < 1 (FA_ERR_INVALID_ARG otherwise); it is
 *           quantised to t = round(256 p) clamped to 255, and t = 0 runs the
 *           plain kernels
 *   seed    Philox4x32-10 key: (seed mod 2^32, seed div 2^32)
 *   offset  fourth counter word, so one seed gives independent masks per call
 * Element (b, h, i, j) uses byte j mod 4 (least significant first) of word
 * i mod 4 of Philox(counter = (j div 4, i div 4, b*H + h, offset)); it is kept
 * when that byte is >= t, and kept probabilities are scaled by 256 / (256 - t).
 * The same (seed, offset) in forward and backward gives the same mask.
 */
typedef struct {
  float p;
  unsigned long long seed;
  unsigned int offset;
} fa_dropout;

/*
 * fa_fwd with dropout: O = (P o M~) V, M~ = keep * 256 / (256 - t), P the
 * softmax of the scores; lse is the plain log-sum-exp (dropout acts after
 * normalisation).  dropout must not be NULL (FA_ERR_INVALID_ARG).  Other
 * arguments, layout and errors as fa_fwd.
 */
fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, float scale, int causal,
                         const fa_dropout* dropout, struct CUstream_st* stream);

/*
 * fa_bwd for fa_fwd_dropout (same dropout parameters, so the same mask):
 *   dV = (P o M~)^T dO, dP = dO V^T, D_i = sum_c dO_ic O_ic (O with dropout),
 *   dS = P o (M~ o dP - D), dQ = scale dS K, dK = scale dS^T Q.
 * Other arguments, layout, workspace and errors as fa_bwd.
 */
fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, float scale, int causal, const fa_dropout* dropout,
                         void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/*
 * FP8 (e4m3) forward.  [WHY-FAST] "Flash Attention 3：拥抱Hopper架构" names FP8
 * tensor cores and "incoherent processing" (a random orthogonal rotation of
 * Q and K before quantisation); the format and rounding contract is this
 * library's: OCP FP8 E4M3FN codes (1 byte, largest 448), conversions round
 * to nearest even and saturate, one dequantisation factor (descale) per
 * (batch, head).
 *
 * fa_fp8_quantize: codes of a contiguous bf16 [B, H, N, d] tensor x.  Per
 * (b, h): amax = max |x| (after the optional rotation), each element becomes
 * e4m3(x * (448 / amax)) (fp32 arithmetic), descale[b*H + h] = amax / 448
 * (1 for an all-zero head).
 *   transpose 0: out is e4m3 [B, H, N, d]; 1: out is e4m3 [B, H, d, ldv],
 *                ldv = fa_fp8_vt_ld(N) (the layout fa_fwd_fp8 takes for V;
 *                entries past N are written as 0)
 *   rotate != 0: x is first multiplied along d by diag(sigma) H_d / sqrt(d)
 *                (Sylvester-Hadamard; sigma_c = +-1 from bit c of
 *                Philox4x32-10(counter 0, key = seed)); apply it to Q and to
 *                K with the same seed (Q K^T is unchanged).  d must be 64,
 *                128 or 256 (FA_ERR_UNSUPPORTED otherwise); sigma_c for
 *                c >= 128 comes from counter block c / 128 (bit c mod 128).
 * d must be a multiple of 16 in [16, 256] (FA_ERR_UNSUPPORTED).  descale is
 * fp32 [B, H] device memory; x, out 16-byte aligned.  One kernel on
 * `stream` (a cluster launch: one 8-CTA cluster per (b, h)).
 */
fa_status fa_fp8_quantize(const void* x, void* out, float* descale, int B, int H, int N, int d,
                          int transpose, int rotate, unsigned long long seed, struct CUstream_st* stream);

/* Row pitch (elements = bytes) of the transposed V codes: N rounded up to 16. */
size_t fa_fp8_vt_ld(int N);

/*
 * Forward on e4m3 codes: q8, k8 [B, H, N, d], vt8 [B, H, d, fa_fp8_vt_ld(N)]
 * (V transposed, from fa_fp8_quantize with transpose = 1), descales fp32
 * [B, H].  S = scale (descale_q Q)(descale_k K)^T in fp32; the unnormalised
 * probabilities P~ = exp(S - m) are rounded to e4m3 before P~ V;
 * O = (P~ V) descale_v / l (l the fp32 sum of the unrounded P~), bf16
 * [B, H, N, d]; lse fp32 [B, H, N] of S.  Error contract (derived, not on
 * the pages): against the exact attention of the dequantised inputs,
 * |O - O_exact| <= sum_j max(2^-4 P~_ij, 2^-10) |V_jc| / l_i plus fp32
 * and bf16 output rounding.  d a multiple of 16 in [16, 256] (d > 128 runs
 * the one-query-tile kernel's e4m3 variant); causal as in fa_fwd; other
 * errors as fa_fwd.
 */
fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* descale_q,
                     const float* descale_k, const float* descale_v, void* o, float* lse,
                     int B, int H, int N, int d, float scale, int causal, struct CUstream_st* stream);

/*
 * Split-KV forward on e4m3 codes (causal as in fa_fwd_splitkv), e.g.
 * decoding against an e4m3 key/value cache: q8 [B, H, Nq, d], k8 [B, H, Nk, d], vt8
 * [B, H, d, fa_fp8_vt_ld(Nk)] (from fa_fp8_quantize; V with transpose = 1),
 * descales fp32 [B, H].  The keys are cut into chunks as in fa_fwd_splitkv;
 * each chunk computes fa_fwd_fp8's arithmetic (its own reference maximum,
 * P~ rounded to e4m3) into fp32 partials, merged by their LSE as in
 * fa_fwd_splitkv.  The error contract of fa_fwd_fp8 holds unchanged: a
 * chunk's P~ is the row's P~ times e^{m - m_chunk} >= 1, so its rounding is
 * no larger relative to the row's.  o bf16 [B, H, Nq, d], lse fp32
 * [B, H, Nq] (Nk == 0: O = 0, LSE = -inf).  workspace: at least
 * fa_fwd_fp8_splitkv_workspace_bytes(...) bytes, 16-byte aligned (may be
 * NULL when that is 0), else FA_ERR_WORKSPACE.  d a multiple of 16 in
 * [16, 256]; Nq == 0 is a no-op; k8, vt8 may be NULL when Nk == 0; other
 * errors as fa_fwd_splitkv.
 */
fa_status fa_fwd_fp8_splitkv(const void* q8, const void* k8, const void* vt8, const float* descale_q,
                             const float* descale_k, const float* descale_v, void* o, float* lse,
                             int B, int H, int Nq, int Nk, int d, float scale, int causal, int num_splits,
                             void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/*
 * Workspace bytes fa_fwd_fp8_splitkv needs: R * n_used * B*H*Nq*W fp32
 * partial outputs (W = 128 for d <= 128, else 256) plus R * n_used * B*H*Nq
 * fp32 partial LSE, each rounded up to 256 bytes, with R = 4 for Nq <= 32
 * and d <= 128 (one partial result per quarter of a chunk's keys) and 1
 * otherwise, n_used as in
 * fa_fwd_splitkv_workspace_bytes.  0 for invalid sizes, Nq == 0 or Nk == 0.
 */
size_t fa_fwd_fp8_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits);

/*
 * Backward step 1: D_i = sum_c dO_ic O_ic (fp32 [B, H, N]), the row term of
 * the softmax Jacobian (derived; not on the pages).  Memory-bound.
 */
fa_status fa_bwd_preprocess(const void* o, const void* dO, float* Dvec,
                            int B, int H, int N, int d, struct CUstream_st* stream);

/*
 * Backward step 2: dK and dV.  For each 128-key tile, loops over the query
 * tiles, recomputing P^T = exp(scale K Q^T - LSE) on chip.
 *   Dvec in: fp32 [B, H, N] from fa_bwd_preprocess.
 */
fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const float* lse,
                      const void* dO, const float* Dvec, void* dk, void* dv,
                      int B, int H, int N, int d, float scale, int causal,
                      struct CUstream_st* stream);

/*
 * Backward step 3: dQ.  For each 128-query tile, loops over the key tiles,
 * recomputing P = exp(scale Q K^T - LSE) on chip.
 */
fa_status fa_bwd_dq(const void* q, const void* k, const void* v, const float* lse,
                    const void* dO, const float* Dvec, void* dq,
                    int B, int H, int N, int d, float scale, int causal,
                    struct CUstream_st* stream);

/*
 * fa_bwd without a workspace argument, for callers that cannot allocate
 * device memory themselves: code whose device memory belongs to a framework
 * allocator or to a fixed budget (where a raw cudaMalloc may fail or break the
 * owner's accounting), and code on latency-critical paths that cannot accept
 * cudaMalloc's implicit device synchronisation.  The pages have no
 * counterpart: this is a deployment convenience of this library.
 *
 * Same arguments, results and rules as fa_bwd.  The row term D is kept in a
 * scratch array built into the library (8 MiB of device memory, reserved on
 * every GPU that loads the library until the process exits), so
 * B*H*N may be at most 2^21 = 2097152 rows; larger problems return
 * FA_ERR_WORKSPACE (see fa_last_error_detail) and must use fa_bwd.  This entry
 * point allocates nothing and calls no allocating routine.
 *   - The first call with a given device current looks up the scratch's
 *     device address (and again when that device's CUDA context changes, for
 *     example after cudaDeviceReset); make that first call before any stream
 *     capture.
 *   - All calls share the one scratch array: two calls whose kernels overlap
 *     on the GPU (for example on different streams) race on it.  Calls
 *     ordered on one stream are safe; each call overwrites the rows it uses.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, float scale, int causal,
                         struct CUstream_st* stream);

/*
 * Test hook of the deadlock guard; not for production use.  fa_fwd's
 * two-query-tile kernel (d <= 128, whatever kernel fa_fwd would pick for d)
 * with every pipeline wait bounded by wait_limit_us (>= 1) instead of the
 * built-in 4 s, and with the copy producer of every CTA withholding K/V group
 * withhold_group (>= 0) and all later ones: group 0 is K_0, group j+1 holds
 * V_j and K_{j+1}.  The tensor-core warp's wait for that group then runs into
 * the limit; the CTA records FA_ERR_TIMEOUT (fa_debug_status; fa_debug_site()
 * == 0x102, the forward's K/V-group wait, unless another wait of the same
 * launch gave up first), ends the waits of the launch's other CTAs, lets the
 * copies and products already issued complete, frees its tensor memory and
 * returns.  O and LSE are then incomplete.  Launches made before or after are
 * unaffected: a launch that gives up ends only its own waits.  A group index
 * past the last group withholds nothing (the call computes what fa_fwd
 * does).  FA_ERR_INVALID_ARG for withhold_group < 0 or wait_limit_us == 0;
 * FA_ERR_UNSUPPORTED for d > 128; other arguments and errors as fa_fwd.
 */
fa_status fa_debug_fwd_withhold(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int N, int d, float scale, int causal, int withhold_group,
                                unsigned int wait_limit_us, struct CUstream_st* stream);

/* Static description of a status code (never NULL). */
const char* fa_status_string(fa_status s);

/*
 * Device-side status of the kernels: FA_OK, or FA_ERR_TIMEOUT if some kernel
 * gave up on a pipeline wait (a deadlock guard; each wait is bounded, 4 s,
 * and the kernel unwinds instead of hanging, leaving that launch's outputs
 * incomplete).  The first failure's site is kept until a call with
 * reset != 0 clears it; a failure ends only the waits of its own launch, so
 * later calls run normally whether or not the state was cleared.
 * Synchronous: reads device memory.  FA_ERR_CUDA if the read fails.
 */
fa_status fa_debug_status(int reset);

/*
 * Site code of the first recorded timeout (0 if none); valid after
 * fa_debug_status.  The high byte names the kernel: 0x1 forward (d <= 128,
 * two query tiles per CTA), 0x2 dK/dV, 0x3 dQ (d <= 128), 0x4 wide-head
 * forward, 0x5 wide-head backward (its dV, dK and dQ launches), 0x6
 * narrow-head forward (d <= 64, four query tiles per CTA), 0x7 FP8 forward;
 * the low byte names the wait inside that kernel.
 */
unsigned int fa_debug_site(void);

/*
 * Text describing the last FA_ERR_CUDA returned on the calling thread: which
 * call failed and the CUDA error string.  Static storage, never NULL.
 */
const char* fa_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
