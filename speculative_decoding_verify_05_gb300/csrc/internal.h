// Host-side launchers shared between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "linear_tc.cuh"

namespace spec {

// 1: kernels are launched with programmatic stream serialization (see pdl_wait); knob "pdl".
bool pdl_enabled();

// Launch with the library's launch attributes (programmatic dependent launch when enabled).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Same, as clusters of `cluster` CTAs along x when cluster > 1 (grid counts CTAs).
template <typename... KArgs, typename... Args>
cudaError_t launch_kc(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                      int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.numAttrs = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cfg.attrs = attr;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- tcgen05 GEMM: NSUB sub-tiles of BN verify rows per CTA tile
//      (NSUB = 1: BN = 16..256 step 16; NSUB = 2: BN = 144..256 step 16)
constexpr int kMaxBN = 256;
constexpr int kMaxTN = 384;   // rows of a two-MMA token tile (three 64 KB ring stages)
int linear_tc_smem_bytes(int BN, int NSUB);
bool linear_tc_supported(int BN, int NSUB);
cudaError_t launch_linear_tc_bf16(int BN, int NSUB, const CUtensorMap& tw, const CUtensorMap& tx,
                                  const LinearArgs& a, dim3 grid, cudaStream_t s);
cudaError_t launch_linear_tc_swiglu(int BN, int NSUB, const CUtensorMap& tw, const CUtensorMap& tx,
                                    const LinearArgs& a, dim3 grid, cudaStream_t s);
// Cluster split-K GEMM (few tiles): CTAs that may be resident at once for clusters of S
// (0 when the tile shape has no cluster build or S is out of range), and the launch
// (tiles * S CTAs; no workspace).
int linear_cluster_capacity(int BN, int NSUB, int S);
cudaError_t launch_linear_cluster(int BN, int NSUB, const CUtensorMap& tw, const CUtensorMap& tx,
                                  const LinearArgs& a, int S, int tiles, cudaStream_t s);
// Split-K GEMM on CTA pairs (tcgen05 2-SM MMA, 256-row pair tiles): CTAs resident at once in
// clusters of S pairs (0: no pair build for the tile shape, or S out of range), and the launch of
// pair tiles a.dp_tiles .. + pair_tiles - 1 (2 S CTAs each; no workspace).
int linear_pair_capacity(int BN, int NSUB, int S);
cudaError_t launch_linear_pair(int BN, int NSUB, const CUtensorMap& tw, const CUtensorMap& tx, const LinearArgs& a,
                               int S, int pair_tiles, cudaStream_t s);
// The persistent GEMM on CTA pairs (2-SM MMA, 256-row pair tiles; a.pair = 1, a.grid pairs): the
// tile shapes with a build (BN token rows per MMA, NSUB MMAs per k-step), the pairs resident at
// once (0: no build for the shape), and the launch of `pairs` clusters of 2 CTAs (epilogue epi).
#define SPEC_TC_PAIR_SHAPES(X) \
  X(64, 1) X(96, 1) X(128, 1) X(160, 1) X(192, 1) X(224, 1) X(256, 1) X(144, 2) X(160, 2) X(176, 2) X(192, 2)
int linear_tc_pair_capacity(int BN, int NSUB, bool lmhead);
int linear_tc_pair_capacity_lmhead(int BN, int NSUB);
cudaError_t launch_linear_tc_pair(int BN, int NSUB, int epi, const CUtensorMap& tw, const CUtensorMap& tx,
                                  const LinearArgs& a, int pairs, cudaStream_t s);
cudaError_t launch_linear_tc_pair_lmhead(int BN, int NSUB, bool greedy, const CUtensorMap& tw, const CUtensorMap& tx,
                                         const LinearArgs& a, int pairs, cudaStream_t s);
// Second pass of a split GEMM: sums the fp32 pieces of every split tile (in CTA order), adds the
// residual and writes bf16 Y.  `sms` sizes its grid.
cudaError_t launch_linear_reduce(const LinearArgs& a, int sms, cudaStream_t s);
cudaError_t launch_linear_tc_lmhead(int BN, int NSUB, bool greedy, const CUtensorMap& tw,
                                    const CUtensorMap& tx, const LinearArgs& a, dim3 grid,
                                    cudaStream_t s);

// ---- weight-streaming chain of small-M GEMMs (one persistent launch for a list of products)
constexpr int CH_MAX_OPS = 48;     // products per launch (kernel parameter space)
constexpr int CH_MAX_DEPS = 6;
constexpr int CH_MAX_M = 64;
enum ChainDepKind : int {
  CH_DEP_X = 0,       // X of the product reads Y of `op`: token loads wait (per tile when shift >= 0)
  CH_DEP_RES = 1,     // the residual reads Y of `op`: the epilogue waits (per tile when shift >= 0)
  CH_DEP_WRITE = 2    // Y overwrites what `op` reads or writes: the first write waits for all of `op`
};
struct ChainDep {
  int op, kind;
  int shift;          // >= 0: column c of the consumer's operand is column c + shift of Y_op; -1: whole op
};
struct ChainOp {
  uint16_t* Y;
  const uint16_t* residual;
  int ldy, ldr;
  int N, K, k_tiles, tiles_n;
  int units;          // tiles_n * k_tiles
  int epi;            // EPI_BF16 (+ residual) or EPI_SWIGLU
  int ycols;          // Y columns per weight tile: 128, or 64 with the SwiGLU epilogue
  int flag_base;      // first per-tile flag of this product
  int n_deps;
  ChainDep dep[CH_MAX_DEPS];
};
struct ChainParams {
  CUtensorMap tw[CH_MAX_OPS];
  CUtensorMap tx[CH_MAX_OPS];
  ChainOp op[CH_MAX_OPS];
  int n_ops, M, grid;
  float* pieces;      // [n_ops][grid][BN][128] fp32
  unsigned* arrive;   // per tile: pieces published
  unsigned* done;     // per tile: 1 once Y of the tile is stored
  unsigned* op_done;  // per product: tiles stored
  unsigned* status;
};
int chain_bn(int M);   // token rows per tile for an M-row chain (-1: M too large)
cudaError_t launch_linear_chain(const ChainParams& p, cudaStream_t s);

// ---- CUDA-core skinny GEMM (M <= 4)
struct GemvArgs {
  const uint16_t* X; int ldx;
  const uint16_t* W; int ldw;
  uint16_t* Y; int ldy;
  const uint16_t* residual; int ldr;
  int M, N, K;
  int splits;           // K split count
  int k_per_split;      // multiple of 256 elements
  float* partial;       // [splits][M][N]
  unsigned* counters;   // [ceil(N / rows_per_group)]
};
int gemv_k_slice(int M);   // K elements per split for an M-row pass
cudaError_t launch_gemv(const GemvArgs& a, int grid, cudaStream_t s);

// ---- softmax normalisation of the LM head output
cudaError_t launch_lmhead_normalize(float* P, long long ldp, const float2* stats, int M, int V, int n_tiles,
                                    bool greedy, cudaStream_t s);

// ---- verify attention
struct AttnArgs {
  const uint16_t* Q; int ldq;
  const uint16_t* Knew; const uint16_t* Vnew; int ldkv;
  const int32_t* cu_rows; const int32_t* ctx_len;
  uint16_t* Kc; uint16_t* Vc; int cap;
  int B, Hq, Hkv, G, max_rows;
  float scale_log2;     // softmax scale * log2(e)
  uint16_t* O; int ldo;
  int chunk;            // keys per CTA (multiple of 64)
  int max_chunks;
  float* partial;       // [B*Hkv][max_chunks][64][128 + 2]
  unsigned* counters;   // [B*Hkv]
  unsigned* status;
  int pair_cost;        // tcgen05 kernel: work charged per (sequence, kv head) pair, quarter tiles
  // paged cache (tcgen05 kernel only; nullptr: the contiguous [B][Hkv][cap][D] layout): Kc / Vc are
  // pools [Hkv][num_pages][128][D] and key tile t of sequence b is page block_table[b * max_pages + t]
  const int32_t* block_table;
  int max_pages, num_pages;
  int* pfx;             // tcgen05 kernel: [grid][B + 1] each CTA's copy of the per-sequence unit prefix
};
cudaError_t launch_attention(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a,
                             cudaStream_t s);
// tcgen05 variant (persistent, stream-K over 128-key tiles): K/V tensor maps with
// 128-key boxes; `grid` persistent CTAs, partial slots [grid][2][64][128 + 2], prefix slices
// [grid][B + 1]
int attention_tc_key_tile();
int attention_tc_max_batch();
int attention_tc_rows(int G, int max_rows);   // padded query rows per kv head, -1 if unsupported
cudaError_t launch_attention_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, int grid,
                                cudaStream_t s);

// ---- rejection sampler
cudaError_t launch_reject_sample(const float* P, const float* Q, const int32_t* draft,
                                 const float* U, const int32_t* cu_rows, int B, int V,
                                 float tie_eps, int32_t* n_acc, int32_t* out_tok,
                                 int32_t* near_tie, unsigned* status, cudaStream_t s);
// Fused LM-head path: p from the logits Z = z / T [M x V] and the GEMM's per-tile statistics
// stats [M][n_stats] (or the argmax statistics when greedy; Z unused).
cudaError_t launch_reject_sample_logits(const float* Z, const float2* stats, int n_stats, bool greedy,
                                        const float* Q, const int32_t* draft, const float* U,
                                        const int32_t* cu_rows, int B, int M, int V, float tie_eps,
                                        int32_t* n_acc, int32_t* out_tok, int32_t* near_tie, unsigned* status,
                                        cudaStream_t s);

// One token per row of p (rows at P + r*ldp) by the sampler's inverse CDF with U[r].
cudaError_t launch_sample_rows(const float* P, long long ldp, int M, int V, const float* U, int32_t* out_tok,
                               unsigned* status, cudaStream_t s);
// Typical acceptance (lossy): p [M x V] given; Q not used.
cudaError_t launch_typical_sample(const float* P, const int32_t* draft, const float* U, const int32_t* cu_rows,
                                  int B, int V, float t_eps, float t_delta, float tie_eps, int32_t* n_acc,
                                  int32_t* out_tok, int32_t* near_tie, unsigned* status, cudaStream_t s);

// ---- n-gram prompt-lookup drafter
constexpr int NGRAM_MAX_WINDOW = 64;
cudaError_t launch_ngram_propose(const int32_t* tokens, const int32_t* cu_len, int B, int k, int n_min, int n_max,
                                 int32_t* drafts, int32_t* n_drafts, unsigned* status, cudaStream_t s);

// ---- failure-detection probe: one bounded mbarrier wait that nothing (arrive = 0) or a second
//      warp (arrive = 1) completes
cudaError_t launch_wait_probe(unsigned* status, unsigned site, unsigned long long limit_ns, int arrive,
                              cudaStream_t s);

// ---- folded RMSNorm: per-row, per-128-column-tile sums of squares of a bf16 matrix; and the
//      row normalisation from such sums (the fallback for plans whose epilogue cannot scale rows)
cudaError_t launch_row_ssq(const uint16_t* X, int M, int N, int ldx, float* out, cudaStream_t s);
cudaError_t launch_rownorm_ssq(const uint16_t* X, int M, int K, int ldx, const float* ssq, int tiles, float eps,
                               uint16_t* Y, int ldy, cudaStream_t s);

// ---- glue
cudaError_t launch_rmsnorm(const uint16_t* X, int M, int N, int ldx, const uint16_t* w, float eps,
                           uint16_t* Y, int ldy, cudaStream_t s);
cudaError_t launch_rope(uint16_t* Q, int ldq, int Hq, uint16_t* K, int ldk, int Hkv, int D,
                        const int32_t* cu_rows, const int32_t* ctx_len, int B, int M, float theta,
                        cudaStream_t s);
cudaError_t launch_rope_table(const int32_t* cu_rows, const int32_t* ctx_len, int B, int M, int D, float theta,
                              float2* cs, cudaStream_t s);
cudaError_t launch_rope_apply(uint16_t* Y, int ldy, int heads, int D, const float2* cs, int M, cudaStream_t s);
cudaError_t launch_silu_mul(const uint16_t* GU, int M, int I, int ldgu, uint16_t* A, int lda,
                            cudaStream_t s);
cudaError_t launch_embed(const int32_t* ids, int M, const uint16_t* table, int V, int d, int ldt, uint16_t* X,
                         int ldx, unsigned* status, cudaStream_t s);
cudaError_t launch_swiglu_interleaved(const uint16_t* GU, int M, int I, int ldgu, uint16_t* A, int lda,
                                      cudaStream_t s);

}  // namespace spec
