/*
 * spec_verify.h — C ABI of the GB300 (sm_103a) speculative-decoding verify library.
 *
 * The library runs the target model's side of one speculative-decoding round:
 * the verify pass that scores all gamma+1 positions of B sequences in ONE
 * forward pass (every weight byte read once for M = sum_b (gamma_b + 1) rows),
 * and the rejection-sampling step that accepts a prefix of the drafts and
 * emits a correction or bonus token.
 *
 * Sources (web pages describing the method):
 *   [P1] "Speculative Decoding Spends Arithmetic You May Not Have" — section
 *        "What one iteration actually does" (Algorithm 1) and "The speedup is
 *        borrowed, and there is a lender".
 *   [P3] "How Speculative Decoding Works (and When It Doesn't)" — "Prefill and
 *        Decode", "How speculative decoding works", "Why the output doesn't
 *        change".
 *   [P5] "Speculative Decoding Is a Bet on How Predictable Your Traffic Is" —
 *        "What it looks like in code" (score_parallel, sample_residual).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or copies host memory for them.
 *   - spec_bf16 is a bf16 bit pattern; matrices are row-major with the given
 *     leading dimension (elements).  bf16 matrices must start on a 16-byte
 *     boundary and have a leading dimension that is a multiple of 8.
 *   - Packed ragged rows: sequence b owns verify rows cu_rows[b] ..
 *     cu_rows[b+1]-1 (gamma_b + 1 >= 1 rows).  Row 0 of a sequence is its last
 *     committed token, rows 1..gamma_b are its drafts x_1..x_gamma.  Per-draft
 *     arrays (Q, draft_tok) hold sum_b gamma_b rows; sequence b's start at
 *     cu_rows[b] - b.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and may be captured in a CUDA graph.  Arguments are
 *     checked on the host before anything is launched; on error nothing is
 *     launched and a non-zero code is returned.  spec_last_error() gives the
 *     message (per host thread).
 *   - Workspace: ops with a *_workspace_bytes query need a caller-provided
 *     device buffer of at least that size, zero-filled before its FIRST use.
 *     Its first 64 KiB hold arrival counters that the kernels return to zero
 *     themselves; scratch follows.  So one workspace, sized for the largest
 *     call, can serve any sequence of calls on one stream without clearing.
 *     Calls that may run concurrently must not share a workspace.
 *   - Device-side waits (TMA/MMA pipelines) are bounded; a wait that runs out
 *     sets a status word read by spec_device_status().
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

typedef uint16_t spec_bf16;
typedef void* spec_stream;

enum {
  SPEC_OK = 0,
  SPEC_EINVAL = 1,        /* bad argument (null pointer, size, alignment) */
  SPEC_EUNSUPPORTED = 2,  /* valid but outside what the kernels implement */
  SPEC_ECUDA = 3,         /* a CUDA runtime / driver call or launch failed */
  SPEC_ETIMEOUT = 4       /* a bounded device wait ran out (spec_device_status) */
};

/* Message of the last failing call on this host thread ("" if none). */
SPEC_API const char* spec_last_error(void);

/* Number of library kernels the last call on this host thread enqueued (0 after
 * a failing call): spec_verify_linear enqueues one, or two when the GEMM split
 * some tiles' k-steps between CTAs (the second sums their pieces);
 * spec_lmhead_softmax two; the other compute calls one.  For launch accounting. */
SPEC_API int spec_launches(void);

/* Library ABI version (increments on any signature change). */
SPEC_API int spec_version(void);

/* Tuning knobs (process-wide): "gemv_max_m" (0..4, default 0): largest M
 * that takes the CUDA-core path of spec_verify_linear (by default every M runs
 * on the tensor cores, which stream the weights faster even at M = 1); "persistent_grid" (0..4096,
 * default 0 = one CTA per SM): CTAs of the persistent tensor-core GEMM and
 * attention kernels;
 * "attention_impl" (1 = tcgen05 kernel, default; 0 = mma.sync kernel);
 * "attention_pair_cost" (0..64, default 12): work the tcgen05 attention kernel
 * charges for starting a (sequence, kv head) pair, in quarters of a 128-key
 * tile, when it splits the key tiles evenly between CTAs;
 * "linear_nsub" (2, default: one tensor-core tile covers up to 384 rows; 1: up
 * to 256); "linear_cluster" (1 default, 0 off): layers with few weight
 * tiles split each tile's k-steps between the CTAs of a thread-block cluster
 * and sum the pieces on chip; "linear_split_rows" (1 default, 0 off): such a
 * product at 257..384 rows may take two tiles of half the rows on clusters of
 * half the size when a cost model says the smaller on-chip exchange pays
 * (the O projection at 368 rows); "lmhead_nsub" (2 default, or 1): the LM head's
 * tensor-core tiles cover up to 384 or 256 rows; "lmhead_pair" (1 default,
 * 0 off): the LM head (64+ rows) runs 256-row vocabulary tiles on CTA pairs
 * (the tcgen05 2-SM MMA: each CTA of a pair stages half of the token rows),
 * a persistent kernel on every pair taking whole tiles round-robin;
 * "linear_pair" (1 default, 0 off): verify linears of 64+ rows with more
 * 128-row weight tiles than SMs run 256-row tiles on CTA pairs, whole pair
 * tiles first (one launch), the rest split between the pairs of a cluster
 * (a second launch), no workspace; "linear_pair_persistent" (0 default, 1,
 * 2): instead the persistent pair kernel takes the whole pair tiles, then
 * with 1 cuts the rest into stream-K pieces that a second kernel sums
 * (workspace: 4 fp32 token tiles per pair), with 2 runs the rest split
 * between the pairs of a cluster; "linear_pair_few" (0
 * default, 1): the pair kernel also for products with fewer tiles (split-K
 * on pairs; measured slower than the one-SM cluster kernel at 368 rows);
 * "weight_l2_promotion" / "kv_l2_promotion" (0..3: none, 64, 128, 256 bytes;
 * default 3 for both): the L2 promotion of the TMA loads of weight tiles and of
 * the attention kernels' K/V tiles;
 * "weight_prefetch" (1 default, 0 off): the cluster split-K kernel issues its
 * first ring stages' weight-tile loads before waiting for the kernel ahead of
 * it on the stream; the library never writes a weight matrix, and a caller
 * whose own kernel, launched just before with programmatic dependent launch,
 * writes W must set 0;
 * "pdl" (1 default, 0 off):
 * kernels are launched with programmatic dependent launch, so each one's
 * launch and on-chip setup overlap the end of the kernel before it on the
 * stream (every kernel still waits for that kernel before touching memory).
 * Changing a knob can change the workspace queries.  Returns SPEC_EINVAL for
 * an unknown name or value. */
SPEC_API int spec_set_option(const char* name, int value);

/* Synchronizes `stream`, then reads and clears the current device's status
 * word (the first problem any kernel recorded since the last read).  Returns
 * SPEC_OK; SPEC_ETIMEOUT when a bounded wait ran out; SPEC_EINVAL when a
 * kernel met invalid device-side input (ragged arrays past max_rows or the
 * cache capacity, draft tokens outside the vocabulary); or SPEC_ECUDA.
 * *detail (may be NULL) gets the kernel's site code. */
SPEC_API int spec_device_status(spec_stream stream, int* detail);

/* Failure-detection probe of the bounded device wait that every TMA / MMA
 * pipeline of the library waits with (no counterpart on the pages: it tests
 * the library's own error path, the way a failing wait would surface).  One
 * CTA waits on an mbarrier that expects one arrival.  arrive = 0: nothing
 * arrives, the wait gives up after limit_us microseconds (1..2000000) and
 * records site SPEC_PROBE_WAIT_SITE, so the next spec_device_status returns
 * SPEC_ETIMEOUT with that detail and clears it; the kernel returns and the
 * context stays usable.  arrive = 1: a second warp arrives after about
 * limit_us / 4 and the wait succeeds (status stays clear).  Asynchronous on
 * `stream`; no workspace. */
#define SPEC_PROBE_WAIT_SITE 0x1E1
SPEC_API int spec_probe_bounded_wait(int limit_us, int arrive, spec_stream stream);

/* ------------------------------------------------------------------------ */
/* Verify linear: Y = X W^T (+ residual)                                     */
/* ------------------------------------------------------------------------ */
/* One weight read serves all M verify rows ([P1] "The speedup is borrowed";
 * [P3] "Prefill and Decode": intensity ~ M FLOP/byte in bf16).
 *   X        [M x K] bf16, leading dim ldx          (activations)
 *   W        [N x K] bf16, leading dim ldw           (nn.Linear weight)
 *   Y        [M x N] bf16, leading dim ldy           (output, fp32 accumulate)
 *   residual [M x N] bf16, leading dim ldr, or NULL  (added before rounding;
 *            may alias Y exactly: same pointer and leading dimension)
 * Requires N >= 1, K % 8 == 0; M = 0 is a no-op.  Runs on tcgen05 tensor
 * cores with TMA-staged 128 x 64 weight tiles (M <= "gemv_max_m", off by
 * default, takes a CUDA-core weight stream instead).  Workspace:
 * spec_linear_workspace_bytes (0 when no K split is needed; the pointer may
 * then be NULL). */
SPEC_API size_t spec_linear_workspace_bytes(int M, int N, int K);
SPEC_API int spec_verify_linear(const spec_bf16* X, int M, int K, int ldx,
                       const spec_bf16* W, int N, int ldw,
                       spec_bf16* Y, int ldy,
                       const spec_bf16* residual, int ldr,
                       void* workspace, size_t workspace_bytes, spec_stream stream);

/* Allocation-free variant of spec_verify_linear.  The pages have no
 * counterpart: this exists for callers that cannot allocate device memory or
 * pass a workspace — e.g. an op embedded in a host runtime whose allocator
 * already owns the whole GPU, or a plugin interface that hands the op only its
 * input and output buffers.  The caller still passes X, W, Y (and residual).
 * Scratch comes from a library-owned static device array of
 * SPEC_NOALLOC_SCRATCH_BYTES (16 MiB), which every GPU that loads the library
 * holds until the process exits.  Calls whose K split needs more scratch than
 * that return SPEC_EUNSUPPORTED and launch nothing (use spec_verify_linear with
 * a workspace instead; small verify passes need none or a few MiB).  Where a
 * shape has several plans, the first one whose scratch fits in the array is
 * taken (the optional persistent pair plan's stream-K pieces, "linear_pair_
 * persistent" 1, do not fit at a few hundred rows), so the plan, and the
 * rounding of the result, can differ from spec_verify_linear's under the same
 * options.
 * The first call in each CUDA context looks up the array's device address
 * (cudaGetSymbolAddress) and caches it for that context (a device reset gives
 * a new context, so the next call looks it up again); make that first call
 * outside any stream capture.  All argument checks run before the stream or
 * the array is touched: a rejected call enqueues nothing.
 * Each call clears the counters it needs (an async memset on `stream`); all
 * calls share the array, so calls that may overlap on the GPU (other streams,
 * other host threads) race.  No cudaMalloc, cudaFree or other allocating call
 * is made. */
#define SPEC_NOALLOC_SCRATCH_BYTES (16u << 20)
SPEC_API int spec_verify_linear_noalloc(const spec_bf16* X, int M, int K, int ldx,
                                        const spec_bf16* W, int N, int ldw,
                                        spec_bf16* Y, int ldy,
                                        const spec_bf16* residual, int ldr, spec_stream stream);

/* ------------------------------------------------------------------------ */
/* RMSNorm folded into the verify linears                                    */
/* ------------------------------------------------------------------------ */
/* A pre-norm layer computes h = RMSNorm(x) = x / sqrt(mean(x^2) + eps) * w and
 * then h W^T.  With w folded into W once (W' = W diag(w)), that is
 * (x W'^T) / rms(x): the product can take x itself and scale its rows in the
 * epilogue, and the product that stores x can leave the sums of squares of the
 * values it stored, so no separate normalisation pass over x is needed.
 *   in_ssq   [M x in_tiles] fp32 or NULL: partial sums of squares of X's
 *            rows (their sum over the in_tiles entries, in order, is
 *            sum_k X[m][k]^2); row m of the product is scaled by
 *            1 / sqrt(sum / K + eps)
 *   out_ssq  [M x ceil(Nout / 128)] fp32 or NULL: per row and 128-column tile
 *            of the output (Nout = N; I for SwiGLU), the sum of squares of
 *            the bf16 values stored
 * Plans whose epilogue cannot do this (tiles not split between CTAs) run a
 * small normalisation / sum-of-squares kernel instead (same results within
 * the chain tolerance); the _norm workspace query covers that case. */
typedef struct {
  const float* in_ssq;
  int in_tiles;
  float eps;
  float* out_ssq;
} spec_rownorm;

/* out[m][t] = sum of squares of X[m][128 t .. 128 t + 127] (bf16 values): the
 * partial sums of a tensor no product stored (e.g. the first layer's input). */
SPEC_API int spec_row_ssq(const spec_bf16* X, int M, int N, int ldx, float* out, spec_stream stream);

/* spec_verify_linear / _swiglu / _rope with a folded RMSNorm (norm may be NULL). */
SPEC_API size_t spec_linear_norm_workspace_bytes(int M, int N, int K, int swiglu);
SPEC_API int spec_verify_linear_norm(const spec_bf16* X, int M, int K, int ldx,
                                     const spec_bf16* W, int N, int ldw, spec_bf16* Y, int ldy,
                                     const spec_bf16* residual, int ldr, const spec_rownorm* norm,
                                     void* workspace, size_t workspace_bytes, spec_stream stream);
SPEC_API int spec_verify_linear_swiglu_norm(const spec_bf16* X, int M, int K, int ldx,
                                            const spec_bf16* Wgu, int ldw, int I, spec_bf16* A, int lda,
                                            const spec_rownorm* norm, void* workspace,
                                            size_t workspace_bytes, spec_stream stream);
SPEC_API int spec_verify_linear_rope_norm(const spec_bf16* X, int M, int K, int ldx,
                                          const spec_bf16* W, int N, int ldw, spec_bf16* Y, int ldy,
                                          const float* cs, int rope_heads, const spec_rownorm* norm,
                                          void* workspace, size_t workspace_bytes, spec_stream stream);

/* ------------------------------------------------------------------------ */
/* Chain of verify linears for a handful of rows (weight-streaming path)     */
/* ------------------------------------------------------------------------ */
/* One product of a chain: Y = X W^T (+ residual), or with swiglu = 1 the
 * fused SwiGLU form of spec_verify_linear_swiglu (W = [2I x K] gate|up rows
 * interleaved in blocks of 16, N = 2I, Y = A [M x I], no residual).  Same
 * layouts and alignment rules as spec_verify_linear. */
typedef struct {
  const spec_bf16* X; int ldx;
  const spec_bf16* W; int ldw;
  spec_bf16* Y; int ldy;
  const spec_bf16* residual; int ldr;   /* NULL or [M x N]; may alias Y exactly */
  int N, K;
  int swiglu;
} spec_linear_op;

/* Runs n_ops products over the same M (1..64) verify rows, in order: the
 * result is that of calling spec_verify_linear / spec_verify_linear_swiglu
 * for each in turn.  At small M the verify pass is a weight stream ([P1] "The
 * speedup is borrowed, and there is a lender": one weight read serves all
 * rows; [P3] "Prefill and Decode": bound by memory bandwidth), and one launch
 * per product pays a pipeline fill and drain each time.  Here one persistent
 * launch (up to 48 products; longer chains take several) streams the weights
 * of product j+1 while product j drains: weights never depend on
 * activations.  Token loads, residual reads and output writes wait on device
 * flags of the products they depend on, which the library derives from the
 * buffers' address ranges (read-after-write per 128-column tile where the
 * regions line up, whole products otherwise).  Putting independent products
 * between a producer and its consumer (e.g. the next layer's QKV projection
 * between gate|up and down) hides the wait.  Per 128 x 64 weight tile, the
 * k-steps are split evenly between CTAs and the pieces summed on chip in CTA
 * order (deterministic).  X of a product must not overlap its own Y.
 * Workspace: spec_linear_chain_workspace_bytes (the first 64 KiB are the
 * shared counter region and are left untouched; the call clears its own
 * flags after it with an async memset). */
SPEC_API size_t spec_linear_chain_workspace_bytes(const spec_linear_op* ops, int n_ops, int M);
SPEC_API int spec_verify_linear_chain(const spec_linear_op* ops, int n_ops, int M,
                                      void* workspace, size_t workspace_bytes, spec_stream stream);

/* Fused QKV projection and rotary embedding: Y = X W^T, then the first
 * rope_heads 128-column heads of Y (the query and key heads of a fused QKV
 * output) rotated as spec_rope does (rotate-half pairs (i, i + 64)), with the
 * rotation of row r taken from cs (spec_rope_table).  When the projection has
 * few weight tiles (the cluster split-K plan) the rotation happens on the
 * fp32 sums before the single rounding to bf16 and no extra kernel runs;
 * otherwise Y is rounded, then rotated by a second kernel (one more bf16
 * rounding of q and k, within the linear tolerance).
 *   X, W, Y as spec_verify_linear (no residual); cs [M x 64] pairs of fp32
 *   (cos, sin), 16-byte aligned.  Requires rope_heads * 128 <= N.
 * Workspace: spec_linear_workspace_bytes(M, N, K). */
SPEC_API int spec_verify_linear_rope(const spec_bf16* X, int M, int K, int ldx, const spec_bf16* W, int N,
                                     int ldw, spec_bf16* Y, int ldy, const float* cs, int rope_heads,
                                     void* workspace, size_t workspace_bytes, spec_stream stream);
/* The rotation table of a verify pass: cs[r][i] = (cos, sin) of p_r * theta^(-2i/D),
 * i < D/2, p_r = ctx_len[b] + (r - cu_rows[b]) the position of row r; the angle is
 * formed and reduced mod 2 pi in fp64, then one fp32 sincos (as spec_rope).
 *   cs [M x D/2] pairs of fp32 out.  Requires D even, D <= 256, theta > 0. */
SPEC_API int spec_rope_table(const int32_t* cu_rows, const int32_t* ctx_len, int B, int M, int D, float theta,
                             float* cs, spec_stream stream);

/* Fused gate|up projection and SwiGLU activation of the MLP:
 *   A[r, i] = silu(gate[r, i]) * up[r, i],  gate = X Wg^T, up = X Wu^T,
 * silu(g) = g / (1 + e^-g), fp32 from the fp32 accumulators, one bf16 rounding.
 *   X    [M x K] bf16, leading dim ldx
 *   Wgu  [2I x K] bf16, leading dim ldw: gate and up rows interleaved in blocks
 *        of 16, i.e. rows 32 j .. 32 j + 15 are gate rows 16 j .. 16 j + 15
 *        and rows 32 j + 16 .. 32 j + 31 the matching up rows
 *   A    [M x I] bf16, leading dim lda (output)
 * Same result as spec_verify_linear into a [M x 2I] scratch followed by
 * spec_silu_mul, except that gate and up are not rounded to bf16 first; the
 * [M x 2I] intermediate never reaches HBM on the tensor-core path.  Requires
 * I % 64 == 0, K % 8 == 0, leading dimensions multiples of 8, 16-byte aligned
 * pointers.  Workspace: spec_swiglu_linear_workspace_bytes (may be 0). */
SPEC_API size_t spec_swiglu_linear_workspace_bytes(int M, int I, int K);
SPEC_API int spec_verify_linear_swiglu(const spec_bf16* X, int M, int K, int ldx,
                                       const spec_bf16* Wgu, int ldw, int I,
                                       spec_bf16* A, int lda,
                                       void* workspace, size_t workspace_bytes, spec_stream stream);

/* ------------------------------------------------------------------------ */
/* n-gram prompt-lookup drafter (the weightless drafter)                     */
/* ------------------------------------------------------------------------ */
/* [P2] "Under the Hood" (N-gram: match the recent context against earlier
 * text, copy what followed) and "Cheat Sheet" (num_speculative_tokens k,
 * prompt_lookup_min / prompt_lookup_max).  Per sequence with history
 * h[0 .. L-1]: for n = n_max down to n_min, the latest start j with
 * h[j .. j+n-1] == h[L-n .. L-1] and j + n <= L - 1; the first n that has one
 * wins and the drafts are h[j+n .. min(j+n+k, L) - 1]; no match, no drafts.
 *   tokens  [sum L] int32, history b at tokens[cu_len[b] .. cu_len[b+1] - 1]
 *   cu_len  [B + 1] int32 device array (non-decreasing; a negative length is
 *           flagged in the status word and gives no drafts)
 *   drafts  [B x k] int32 out, -1 after the n_drafts[b] proposed tokens
 *   n_drafts [B] int32 out
 * Requires 1 <= k <= 4096, 1 <= n_min <= n_max <= 64.  One kernel, no
 * workspace. */
SPEC_API int spec_ngram_propose(const int32_t* tokens, const int32_t* cu_len, int B, int k, int n_min,
                                int n_max, int32_t* drafts, int32_t* n_drafts, spec_stream stream);

/* ------------------------------------------------------------------------ */
/* Verify attention (causal GQA over the KV cache + the new block)           */
/* ------------------------------------------------------------------------ */
/* Row j of sequence b sits at position ctx_len[b] + j and attends the
 * ctx_len[b] committed keys plus new keys 0..j of its own block, which is
 * what gamma_b + 1 sequential decode steps would see ([P1] Algorithm 1,
 * parallel line; "the cache read serves every query position").  The new
 * keys/values are written into the cache at positions ctx_len[b] ..
 * ctx_len[b] + gamma_b (the caller advances ctx_len by n_acc + 1 afterwards;
 * entries past that are overwritten next round).
 *   Q       row r, query head h  at Q + r*ldq + h*D         (bf16, RoPE applied)
 *   Knew    row r, kv head g     at Knew + r*ldkv + g*D      (bf16, RoPE applied)
 *   Vnew    row r, kv head g     at Vnew + r*ldkv + g*D
 *   Kcache, Vcache [B][Hkv][cap][D] bf16 (in/out)
 *   cu_rows [B+1], ctx_len [B] int32 device arrays; max_rows >= max_b (gamma_b+1)
 *   O       row r, query head h  at O + r*ldo + h*D          (bf16 out)
 *   scale   softmax scale (1/sqrt(D) for the standard model)
 * Query head h reads kv head h / (Hq / Hkv).  Requires D == 128,
 * Hq % Hkv == 0, (Hq / Hkv) * max_rows <= 64, ctx_len[b] + gamma_b + 1 <= cap.
 * The last two are checked on the device: a sequence that breaks them is
 * skipped and the status word is set (spec_device_status).
 * Workspace: spec_attention_workspace_bytes. */
SPEC_API size_t spec_attention_workspace_bytes(int B, int max_rows, int Hq, int Hkv, int D, int cap);
SPEC_API int spec_verify_attention(const spec_bf16* Q, int ldq,
                          const spec_bf16* Knew, const spec_bf16* Vnew, int ldkv,
                          const int32_t* cu_rows, const int32_t* ctx_len, int B, int max_rows,
                          spec_bf16* Kcache, spec_bf16* Vcache, int cap,
                          int Hq, int Hkv, int D, float scale,
                          spec_bf16* O, int ldo,
                          void* workspace, size_t workspace_bytes, spec_stream stream);

/* Same pass over a paged cache: Kpool, Vpool [Hkv][num_pages][128][D] bf16
 * (in/out; one pool per kv head, page ids shared across heads, so pages
 * handed out in order give each head one unbroken run of keys) and
 * block_table [B x max_pages] int32 (device): keys
 * 128 t .. 128 t + 127 of sequence b live in page block_table[b * max_pages + t]
 * (one page = one 128-key tile of the kernel).  ctx_len[b] + gamma_b + 1 <=
 * 128 * max_pages is checked on the device as for cap; a page id outside
 * [0, num_pages) is flagged in the status word (page 0 is read instead).  The
 * new keys / values go into their pages.  Pages need not be distinct across
 * sequences for reading (shared prefixes), but pages that receive new rows
 * must belong to one sequence.  Needs the tcgen05 kernel (attention_impl 1).
 * Workspace: spec_attention_paged_workspace_bytes. */
SPEC_API size_t spec_attention_paged_workspace_bytes(int B, int max_rows, int Hq, int Hkv, int D, int max_pages);
SPEC_API int spec_verify_attention_paged(const spec_bf16* Q, int ldq, const spec_bf16* Knew,
                                         const spec_bf16* Vnew, int ldkv, const int32_t* cu_rows,
                                         const int32_t* ctx_len, int B, int max_rows,
                                         spec_bf16* Kpool, spec_bf16* Vpool, int num_pages,
                                         const int32_t* block_table, int max_pages,
                                         int Hq, int Hkv, int D, float scale,
                                         spec_bf16* O, int ldo, void* workspace, size_t workspace_bytes,
                                         spec_stream stream);

/* ------------------------------------------------------------------------ */
/* LM head + softmax: P = softmax((H W_lm^T) / T); T == 0 -> one-hot argmax  */
/* ------------------------------------------------------------------------ */
/* Produces p_1 .. p_{gamma+1} for every verify row from the same pass
 * ([P1] Algorithm 1).  Greedy ties go to the lowest token index.
 *   H   [M x K] bf16 (final-normed hidden states), W_lm [V x K] bf16
 *   P   [M x V] fp32 out
 * Requires V % 4 == 0, K % 8 == 0, temperature >= 0; H row-major with leading
 * dimension K.  Workspace: spec_lmhead_workspace_bytes. */
SPEC_API size_t spec_lmhead_workspace_bytes(int M, int K, int V);
SPEC_API int spec_lmhead_softmax(const spec_bf16* H, int M, int K, const spec_bf16* Wlm, int V,
                        float temperature, float* P,
                        void* workspace, size_t workspace_bytes, spec_stream stream);
/* Same, writing row m of P at P + m*ldp (ldp >= V, a multiple of 4): lets a
 * decode step put its rows straight into a larger packed array (the draft
 * side writes step i of sequence b at row b*gamma + i of the verify pass's q). */
SPEC_API int spec_lmhead_softmax_ld(const spec_bf16* H, int M, int K, const spec_bf16* Wlm, int V,
                                    float temperature, float* P, long long ldp,
                                    void* workspace, size_t workspace_bytes, spec_stream stream);

/* ------------------------------------------------------------------------ */
/* Rejection sampler (one CTA per sequence)                                  */
/* ------------------------------------------------------------------------ */
/* [P1] Algorithm 1 in order: accept x_i iff U_i * q_i(x_i) <= p_i(x_i)
 * (exact product; q = 0 accepts), stop at the first rejection n; draw t from
 * max(0, p_{n+1} - q_{n+1}) (falling back to p_{n+1} if that is all zero) when
 * n < gamma, else from p_{gamma+1} (bonus).  t is the smallest token x with
 * sum_{y<=x} w(y) > u * sum_y w(y), u = U[row gamma_b]; the weights are formed
 * in fp32 (exact sign) and summed with fp64 tile and warp prefixes, ~1e-7
 * relative error, inside the near-tie band below.
 *   P [M x V] fp32, Q [sum gamma x V] fp32, draft_tok [sum gamma] int32,
 *   U [M] fp32 in (0,1): rows 0..gamma_b-1 = acceptance draws, row gamma_b =
 *   the draw for t.
 *   n_acc [B] out: accepted drafts n_b in 0..gamma_b
 *   out_tok [M] out: sequence b emits out_tok[cu_rows[b] .. cu_rows[b]+n_b]
 *                    (x_1..x_n, t); later slots are set to -1
 *   near_tie [B] out: decisions with |u*q - p| < tie_eps plus a final pick
 *                    whose CDF boundary is within tie_eps * sum(w) of u*sum(w)
 * Requires 1 <= V <= 1048576, draft tokens in [0, V) (an out-of-range token
 * is clamped and flagged in the status word). */
SPEC_API int spec_reject_sample(const float* P, const float* Q, const int32_t* draft_tok,
                       const float* U, const int32_t* cu_rows, int B, int V,
                       float tie_eps, int32_t* n_acc, int32_t* out_tok, int32_t* near_tie,
                       spec_stream stream);

/* One token per row: out_tok[r] = the smallest x with sum_{y<=x} p_r(y) >
 * U[r] * sum_y p_r(y) (the sampler's inverse CDF, fp64 prefixes), p_r at
 * P + r*ldp.  The draft side's sampling step; rows of zero mass give V - 1.
 * Requires ldp >= V, 1 <= V <= 1048576. */
SPEC_API int spec_sample_rows(const float* P, long long ldp, int M, int V, const float* U, int32_t* out_tok,
                              spec_stream stream);

/* Typical acceptance, the lossy accept rule ([P3] "Exactness is a choice"):
 * keep draft x_i iff p_i(x_i) > max(epsilon, delta * exp(-H_i)), H_i =
 * -sum_x p_i(x) ln p_i(x) the entropy of the target row (epsilon the floor of
 * the bar, delta its entropy slope; the page's formula is lost, this is the
 * reading of its words), stopping at the first draft that fails (n_b); the
 * token after the kept prefix is drawn from the target row p_{n+1} itself by
 * the same inverse CDF as spec_reject_sample (no residual, so Q is not an
 * argument).  The output is no longer distributed as p; at temperature 0
 * (one-hot rows) it equals the exact rule's.  Entropies are summed from fp32
 * terms with fp64 across warps; near_tie counts tests with
 * |p_i(x_i) - threshold| < tie_eps and final picks as for spec_reject_sample.
 *   P, draft_tok, U, cu_rows, n_acc, out_tok, near_tie: as spec_reject_sample
 *   (U rows 0 .. gamma_b - 1 are not used).
 * Requires epsilon, delta finite and >= 0, 1 <= V <= 1048576. */
SPEC_API int spec_typical_sample(const float* P, const int32_t* draft_tok, const float* U,
                                 const int32_t* cu_rows, int B, int V, float epsilon, float delta,
                                 float tie_eps, int32_t* n_acc, int32_t* out_tok, int32_t* near_tie,
                                 spec_stream stream);

/* Fused LM head -> sampler: the same n_acc / out_tok / near_tie as
 * spec_lmhead_softmax followed by spec_reject_sample on the same inputs (bit
 * for bit), without materialising p.  The acceptance test needs p_i(x_i) only
 * at the draft token and the row's softmax normaliser ([P1] Algorithm 1, the
 * accept step), and only the final row's full distribution is read; so the
 * GEMM writes z / T and per-tile (max, sum e^z) statistics into the workspace,
 * and the sampler evaluates p_x = e^(z_x - max) / sum for the entries it reads
 * (a one-hot at the argmax when temperature == 0, where no logits are stored).
 * The normalisation pass and the M x V probability write / read go away.
 *   H [M x K] bf16, W_lm [V x K] bf16; the M verify rows are the rows that
 *   cu_rows [B + 1] packs (cu_rows[B] <= M is checked on the device: a
 *   sequence outside the M rows is skipped and the status word set);
 *   Q, draft_tok, U, tie_eps, n_acc, out_tok, near_tie as for
 *   spec_reject_sample.
 * Requires K % 8 == 0, V % 4 == 0, V <= 1048576, temperature >= 0, M >= B.
 * Workspace: spec_lmhead_sample_workspace_bytes (the logits, M x V x 4 bytes,
 * plus statistics; statistics only when temperature == 0). */
SPEC_API size_t spec_lmhead_sample_workspace_bytes(int M, int K, int V, float temperature);
SPEC_API int spec_lmhead_reject_sample(const spec_bf16* H, int M, int K, const spec_bf16* Wlm, int V,
                                       float temperature, const float* Q, const int32_t* draft_tok,
                                       const float* U, const int32_t* cu_rows, int B, float tie_eps,
                                       int32_t* n_acc, int32_t* out_tok, int32_t* near_tie,
                                       void* workspace, size_t workspace_bytes, spec_stream stream);
/* The same with the final RMSNorm folded in: H is the residual stream x itself
 * (W_lm carrying the norm weight) and norm->in_ssq its rows' partial sums of
 * squares (see spec_rownorm; out_ssq unused).  Same workspace query. */
SPEC_API int spec_lmhead_reject_sample_norm(const spec_bf16* H, int M, int K, const spec_bf16* Wlm, int V,
                                            float temperature, const float* Q, const int32_t* draft_tok,
                                            const float* U, const int32_t* cu_rows, int B, float tie_eps,
                                            int32_t* n_acc, int32_t* out_tok, int32_t* near_tie,
                                            const spec_rownorm* norm, void* workspace, size_t workspace_bytes,
                                            spec_stream stream);

/* ------------------------------------------------------------------------ */
/* Layer glue of the decoder stack (not on the pages: the stack's layout is  */
/* the builder's reading of a Qwen3-8B-shaped decoder)                      */
/* ------------------------------------------------------------------------ */
/* Y = X / sqrt(mean(X^2) + eps) * w per row; X [M x N], w [N] bf16.
 * Y may alias X.  Requires N % 8 == 0, N <= 16384. */
SPEC_API int spec_rmsnorm(const spec_bf16* X, int M, int N, int ldx, const spec_bf16* w, float eps,
                 spec_bf16* Y, int ldy, spec_stream stream);

/* X[r] = table[ids[r]] (token-embedding rows feeding a decode step), d bf16
 * per row; ids outside [0, V) are flagged in the status word and read row 0.
 * Requires d, ldt, ldx multiples of 8, ldt, ldx >= d, 16-byte aligned. */
SPEC_API int spec_embed(const int32_t* ids, int M, const spec_bf16* table, int V, int d, int ldt,
               spec_bf16* X, int ldx, spec_stream stream);

/* In-place rotary embedding (rotate-half pairs (i, i + D/2), frequency
 * theta^(-2i/D)) on Hq query heads at Q + r*ldq + h*D and Hkv key heads at
 * K + r*ldk + g*D; row r of sequence b is at position ctx_len[b] + (r - cu_rows[b]).
 * Requires D even, D <= 256. */
SPEC_API int spec_rope(spec_bf16* Q, int ldq, int Hq, spec_bf16* K, int ldk, int Hkv, int D,
              const int32_t* cu_rows, const int32_t* ctx_len, int B, int M, float theta,
              spec_stream stream);

/* A[r, i] = silu(GU[r, i]) * GU[r, I + i] for i < I (gate columns then up
 * columns).  Requires I % 8 == 0. */
SPEC_API int spec_silu_mul(const spec_bf16* GU, int M, int I, int ldgu, spec_bf16* A, int lda,
                  spec_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
