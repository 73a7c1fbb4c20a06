// Layer glue of the decoder stack between the verify GEMMs and attention:
// RMSNorm, rotary position embedding, SwiGLU.  All bandwidth-trivial (M rows
// of a few thousand elements); fp32 math, bf16 storage, 16-byte accesses.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int RMS_THREADS = 256;
constexpr int RMS_MAX_VEC = 8;          // 8 x 8 bf16 per thread -> N <= 16384

__global__ void __launch_bounds__(RMS_THREADS)
rmsnorm_kernel(const uint16_t* __restrict__ X, int N, int ldx, const uint16_t* __restrict__ w,
               float eps, uint16_t* __restrict__ Y, int ldy) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const uint16_t* x = X + (size_t)r * ldx;
  const int nv = N / 8;
  float v[RMS_MAX_VEC][8];
  uint4 wv[RMS_MAX_VEC];               // weights fetched with the row (one memory round trip)
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < RMS_MAX_VEC; ++k) {
    const int c = threadIdx.x + k * RMS_THREADS;
    if (c < nv) {
      const uint4 u = *reinterpret_cast<const uint4*>(x + c * 8);
      wv[k] = *reinterpret_cast<const uint4*>(w + c * 8);
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[k][2 * e] = bf16lo(w4[e]);
        v[k][2 * e + 1] = bf16hi(w4[e]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) ss += v[k][e] * v[k][e];
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  __shared__ float s_part[RMS_THREADS / 32];
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int k = 0; k < RMS_THREADS / 32; ++k) tot += s_part[k];
  const float rstd = 1.0f / sqrtf(tot / (float)N + eps);
  uint16_t* y = Y + (size_t)r * ldy;
#pragma unroll
  for (int k = 0; k < RMS_MAX_VEC; ++k) {
    const int c = threadIdx.x + k * RMS_THREADS;
    if (c < nv) {
      const uint32_t w4[4] = {wv[k].x, wv[k].y, wv[k].z, wv[k].w};
      uint32_t o4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        o4[e] = pack_bf16x2(v[k][2 * e] * rstd * bf16lo(w4[e]), v[k][2 * e + 1] * rstd * bf16hi(w4[e]));
      *reinterpret_cast<uint4*>(y + c * 8) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
  }
}

constexpr int ROPE_THREADS = 256;

// (cos, sin) of pos * inv: the angle is formed and reduced to [-pi, pi] in fp64, then one fp32
// sincos (an fp32 angle would be off by up to 5e-4 rad at position 8192).
__device__ __forceinline__ float2 rope_cs(int pos, double inv) {
  const double ang = (double)pos * inv;
  const double two_pi = 6.283185307179586476925286766559;
  const double red = ang - two_pi * rint(ang / two_pi);
  float sv, cv;
  sincosf((float)red, &sv, &cv);
  return make_float2(cv, sv);
}
// Position of row r = ctx_len[b] + (r - cu_rows[b]), b the last sequence with cu_rows[b] <= r.
__device__ __forceinline__ int row_position(int r, const int32_t* cu_rows, const int32_t* ctx_len, int B) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_rows[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return ctx_len[lo] + (r - cu_rows[lo]);
}

// Inverse frequencies theta^(-2 i / D), computed once in fp64 on the host.
struct RopeFreq {
  double inv[128];
};
constexpr int ROPE_SMEM_B = 8192;   // sequences whose row offsets are staged in shared memory

__global__ void __launch_bounds__(ROPE_THREADS)
rope_kernel(uint16_t* __restrict__ Q, int ldq, int Hq, uint16_t* __restrict__ K, int ldk, int Hkv,
            int D, const int32_t* __restrict__ cu_rows, const int32_t* __restrict__ ctx_len, int B,
            const __grid_constant__ RopeFreq f, int vec) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int half = D / 2;
  __shared__ float s_cos[128];
  __shared__ float s_sin[128];
  __shared__ int s_cu[ROPE_SMEM_B + 1];
  __shared__ int s_pos;
  // position of row r = ctx_len[b] + (r - cu_rows[b]), b = last sequence with cu_rows[b] <= r
  const bool staged = B <= ROPE_SMEM_B;
  if (staged)
    for (int i = threadIdx.x; i <= B; i += ROPE_THREADS) s_cu[i] = cu_rows[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((staged ? s_cu[mid] : cu_rows[mid]) <= r) lo = mid; else hi = mid - 1;
    }
    s_pos = ctx_len[lo] + (r - (staged ? s_cu[lo] : cu_rows[lo]));
  }
  __syncthreads();
  if (threadIdx.x < half) {
    const float2 cs = rope_cs(s_pos, f.inv[threadIdx.x]);
    s_cos[threadIdx.x] = cs.x;
    s_sin[threadIdx.x] = cs.y;
  }
  __syncthreads();
  const int heads = Hq + Hkv;
  if (vec) {
    // 8 consecutive pairs (i, i + D/2) per thread: two 16-byte loads and stores
    const int chunks = half / 8;
    for (int idx = threadIdx.x; idx < heads * chunks; idx += ROPE_THREADS) {
      const int hd = idx / chunks, i0 = (idx - hd * chunks) * 8;
      uint16_t* base = hd < Hq ? Q + (size_t)r * ldq + (size_t)hd * D
                               : K + (size_t)r * ldk + (size_t)(hd - Hq) * D;
      const uint4 av = *reinterpret_cast<const uint4*>(base + i0);
      const uint4 bv = *reinterpret_cast<const uint4*>(base + half + i0);
      const uint32_t a4[4] = {av.x, av.y, av.z, av.w}, b4[4] = {bv.x, bv.y, bv.z, bv.w};
      uint32_t x4[4], y4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = i0 + 2 * e;
        const float a0 = bf16lo(a4[e]), a1 = bf16hi(a4[e]), b0 = bf16lo(b4[e]), b1 = bf16hi(b4[e]);
        x4[e] = pack_bf16x2(a0 * s_cos[i] - b0 * s_sin[i], a1 * s_cos[i + 1] - b1 * s_sin[i + 1]);
        y4[e] = pack_bf16x2(b0 * s_cos[i] + a0 * s_sin[i], b1 * s_cos[i + 1] + a1 * s_sin[i + 1]);
      }
      *reinterpret_cast<uint4*>(base + i0) = make_uint4(x4[0], x4[1], x4[2], x4[3]);
      *reinterpret_cast<uint4*>(base + half + i0) = make_uint4(y4[0], y4[1], y4[2], y4[3]);
    }
    return;
  }
  for (int idx = threadIdx.x; idx < heads * half; idx += ROPE_THREADS) {
    const int hd = idx / half, i = idx - hd * half;
    uint16_t* base = hd < Hq ? Q + (size_t)r * ldq + (size_t)hd * D
                             : K + (size_t)r * ldk + (size_t)(hd - Hq) * D;
    const float a = bf16f(base[i]);
    const float b = bf16f(base[i + half]);
    const float c = s_cos[i], s = s_sin[i];
    base[i] = f2bf(a * c - b * s);
    base[i + half] = f2bf(b * c + a * s);
  }
}

__global__ void silu_mul_kernel(const uint16_t* __restrict__ GU, int M, int I, int ldgu,
                                uint16_t* __restrict__ A, int lda) {
  pdl_wait();
  pdl_trigger();
  const int per_row = I / 8;
  const size_t total = (size_t)M * per_row;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx / per_row);
    const int c = (int)(idx - (size_t)r * per_row) * 8;
    const uint4 g = *reinterpret_cast<const uint4*>(GU + (size_t)r * ldgu + c);
    const uint4 u = *reinterpret_cast<const uint4*>(GU + (size_t)r * ldgu + I + c);
    const uint32_t g4[4] = {g.x, g.y, g.z, g.w};
    const uint32_t u4[4] = {u.x, u.y, u.z, u.w};
    uint32_t o4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float g0 = bf16lo(g4[e]), g1 = bf16hi(g4[e]);
      const float s0 = silu(g0), s1 = silu(g1);
      o4[e] = pack_bf16x2(s0 * bf16lo(u4[e]), s1 * bf16hi(u4[e]));
    }
    *reinterpret_cast<uint4*>(A + (size_t)r * lda + c) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  }
}

// A[m][16 j + r] = silu(GU[m][32 j + r]) * GU[m][32 j + 16 + r]: gate and up rows interleaved per
// 16 (the layout of the fused SwiGLU linear), 8 outputs per thread.
__global__ void swiglu_interleaved_kernel(const uint16_t* __restrict__ GU, int M, int I, int ldgu,
                                          uint16_t* __restrict__ A, int lda) {
  pdl_wait();
  pdl_trigger();
  const int per_row = I / 8;
  const size_t total = (size_t)M * per_row;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx / per_row);
    const int c = (int)(idx - (size_t)r * per_row) * 8;
    const int gcol = (c / 16) * 32 + (c % 16);
    const uint4 g = *reinterpret_cast<const uint4*>(GU + (size_t)r * ldgu + gcol);
    const uint4 u = *reinterpret_cast<const uint4*>(GU + (size_t)r * ldgu + gcol + 16);
    const uint32_t g4[4] = {g.x, g.y, g.z, g.w};
    const uint32_t u4[4] = {u.x, u.y, u.z, u.w};
    uint32_t o4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float g0 = bf16lo(g4[e]), g1 = bf16hi(g4[e]);
      const float s0 = silu(g0), s1 = silu(g1);
      o4[e] = pack_bf16x2(s0 * bf16lo(u4[e]), s1 * bf16hi(u4[e]));
    }
    *reinterpret_cast<uint4*>(A + (size_t)r * lda + c) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  }
}

// X[r] = table[ids[r]]: the token-embedding row gather that feeds a decode step, 8 bf16 per
// thread (16-byte loads and stores).  An id outside [0, V) is flagged and row 0 is used.
__global__ void embed_kernel(const int32_t* __restrict__ ids, int M, const uint16_t* __restrict__ table, int V,
                             int d, int ldt, uint16_t* __restrict__ X, int ldx, unsigned* status) {
  pdl_wait();
  pdl_trigger();
  const int per_row = d / 8;
  const size_t total = (size_t)M * per_row;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx / per_row);
    const int c = (int)(idx - (size_t)r * per_row) * 8;
    int id = ids[r];
    if (id < 0 || id >= V) {
      if (c == 0) set_status(status, 0x5F0u);
      id = 0;
    }
    *reinterpret_cast<uint4*>(X + (size_t)r * ldx + c) =
        *reinterpret_cast<const uint4*>(table + (size_t)id * ldt + c);
  }
}

// cs[r][i] = (cos, sin) of row r's position times theta^(-2 i / D), i < D / 2: the rotation of a
// verify pass, computed once and read by every layer's fused QKV epilogue (or rope_apply_kernel).
__global__ void rope_table_kernel(const int32_t* __restrict__ cu_rows, const int32_t* __restrict__ ctx_len, int B,
                                  int M, int half, const __grid_constant__ RopeFreq f, float2* __restrict__ cs) {
  pdl_wait();
  pdl_trigger();
  const int total = M * half;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
    const int r = idx / half, i = idx - r * half;
    cs[idx] = rope_cs(row_position(r, cu_rows, ctx_len, B), f.inv[i]);
  }
}

// In-place rotate-half on `heads` heads of D at Y + r*ldy + h*D, angles from the table.
__global__ void __launch_bounds__(ROPE_THREADS)
rope_apply_kernel(uint16_t* __restrict__ Y, int ldy, int heads, int D, const float2* __restrict__ cs) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int half = D / 2;
  const float2* row = cs + (size_t)r * half;
  for (int idx = threadIdx.x; idx < heads * half; idx += ROPE_THREADS) {
    const int hd = idx / half, i = idx - hd * half;
    uint16_t* base = Y + (size_t)r * ldy + (size_t)hd * D;
    const float a = bf16f(base[i]);
    const float b = bf16f(base[i + half]);
    const float2 t = row[i];
    base[i] = f2bf(a * t.x - b * t.y);
    base[i + half] = f2bf(b * t.x + a * t.y);
  }
}

// Failure-detection probe of the bounded wait every pipeline uses: thread 0 waits on an mbarrier
// that expects one arrival.  With arrive = 0 nothing arrives, so the wait runs out after limit_ns
// and records `site`; with arrive = 1 warp 1 arrives after about limit_ns / 4 and the wait succeeds.
// Both ends are bounded: the waiting side by the wait's limit, the arriving side by its own delay.
__global__ void wait_probe_kernel(unsigned* status, unsigned site, unsigned long long limit_ns, int arrive) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_wait(&bar, 0u, status, site, limit_ns);
  } else if (threadIdx.x == 32 && arrive) {
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < limit_ns / 4) {
    }
    mbar_arrive(&bar);
  }
  __syncthreads();
}

// Sums of squares of the bf16 values of X, per row and 128-column tile: one warp per (row, tile),
// 4 columns per lane, a fixed butterfly across the warp.
__global__ void __launch_bounds__(256) row_ssq_kernel(const uint16_t* __restrict__ X, int M, int N, int ldx,
                                                       float* __restrict__ out, int tiles) {
  pdl_wait();
  pdl_trigger();
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (long long)M * tiles) return;
  const int m = (int)(w / tiles), t = (int)(w - (long long)m * tiles);
  float s = 0.f;
  const int c0 = t * 128 + lane * 4;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (c0 + e < N) {
      const float v = bf16f(X[(size_t)m * ldx + c0 + e]);
      s += v * v;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) out[(size_t)m * tiles + t] = s;
}

// Y = X row-scaled by 1 / sqrt(sum_t ssq[m][t] / K + eps) (t in order), rounded to bf16: the
// RMSNorm of a row whose partial sums of squares were written by the product that stored it.
__global__ void __launch_bounds__(256) rownorm_ssq_kernel(const uint16_t* __restrict__ X, int K, int ldx,
                                                           const float* __restrict__ ssq, int tiles, float eps,
                                                           uint16_t* __restrict__ Y, int ldy) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x;
  __shared__ float s_r;
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int t = 0; t < tiles; ++t) s += ssq[(size_t)m * tiles + t];
    s_r = 1.0f / sqrtf(s / (float)K + eps);
  }
  __syncthreads();
  const float r = s_r;
  for (int c = threadIdx.x; c < K; c += blockDim.x)
    Y[(size_t)m * ldy + c] = f2bf(bf16f(X[(size_t)m * ldx + c]) * r);
}

}  // namespace

cudaError_t launch_row_ssq(const uint16_t* X, int M, int N, int ldx, float* out, cudaStream_t s) {
  const int tiles = (N + 127) / 128;
  const long long warps = (long long)M * tiles;
  const long long blocks = (warps + 7) / 8;
  cudaError_t e = launch_k(row_ssq_kernel, dim3((unsigned)(blocks > 0 ? blocks : 1)), dim3(256), 0, s, X, M, N, ldx,
                           out, tiles);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_rownorm_ssq(const uint16_t* X, int M, int K, int ldx, const float* ssq, int tiles, float eps,
                               uint16_t* Y, int ldy, cudaStream_t s) {
  cudaError_t e = launch_k(rownorm_ssq_kernel, dim3(M), dim3(256), 0, s, X, K, ldx, ssq, tiles, eps, Y, ldy);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_wait_probe(unsigned* status, unsigned site, unsigned long long limit_ns, int arrive,
                              cudaStream_t s) {
  cudaError_t e = launch_k(wait_probe_kernel, dim3(1), dim3(64), 0, s, status, site, limit_ns, arrive);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_rmsnorm(const uint16_t* X, int M, int N, int ldx, const uint16_t* w, float eps,
                           uint16_t* Y, int ldy, cudaStream_t s) {
  cudaError_t e = launch_k(rmsnorm_kernel, dim3(M), dim3(RMS_THREADS), 0, s, X, N, ldx, w, eps, Y, ldy);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_rope(uint16_t* Q, int ldq, int Hq, uint16_t* K, int ldk, int Hkv, int D,
                        const int32_t* cu_rows, const int32_t* ctx_len, int B, int M, float theta,
                        cudaStream_t s) {
  RopeFreq f{};
  for (int i = 0; i < D / 2; ++i) f.inv[i] = std::pow((double)theta, -2.0 * (double)i / (double)D);
  const bool vec = D % 16 == 0 && ldq % 8 == 0 && ldk % 8 == 0 &&
                   (reinterpret_cast<uintptr_t>(Q) & 15) == 0 && (reinterpret_cast<uintptr_t>(K) & 15) == 0;
  cudaError_t e = launch_k(rope_kernel, dim3(M), dim3(ROPE_THREADS), 0, s, Q, ldq, Hq, K, ldk, Hkv, D, cu_rows,
                           ctx_len, B, f, vec ? 1 : 0);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_silu_mul(const uint16_t* GU, int M, int I, int ldgu, uint16_t* A, int lda,
                            cudaStream_t s) {
  const size_t total = (size_t)M * (I / 8);
  int grid = (int)((total + 255) / 256);
  if (grid > 152 * 16) grid = 152 * 16;
  if (grid < 1) grid = 1;
  cudaError_t e = launch_k(silu_mul_kernel, dim3(grid), dim3(256), 0, s, GU, M, I, ldgu, A, lda);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_swiglu_interleaved(const uint16_t* GU, int M, int I, int ldgu, uint16_t* A, int lda,
                                      cudaStream_t s) {
  const size_t total = (size_t)M * (I / 8);
  int grid = (int)((total + 255) / 256);
  if (grid > 152 * 16) grid = 152 * 16;
  if (grid < 1) grid = 1;
  cudaError_t e = launch_k(swiglu_interleaved_kernel, dim3(grid), dim3(256), 0, s, GU, M, I, ldgu, A, lda);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_embed(const int32_t* ids, int M, const uint16_t* table, int V, int d, int ldt, uint16_t* X,
                         int ldx, unsigned* status, cudaStream_t s) {
  const size_t total = (size_t)M * (d / 8);
  int grid = (int)((total + 255) / 256);
  if (grid > 152 * 16) grid = 152 * 16;
  if (grid < 1) grid = 1;
  cudaError_t e = launch_k(embed_kernel, dim3(grid), dim3(256), 0, s, ids, M, table, V, d, ldt, X, ldx, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_rope_table(const int32_t* cu_rows, const int32_t* ctx_len, int B, int M, int D, float theta,
                              float2* cs, cudaStream_t s) {
  RopeFreq f{};
  for (int i = 0; i < D / 2; ++i) f.inv[i] = std::pow((double)theta, -2.0 * (double)i / (double)D);
  const int total = M * (D / 2);
  int grid = (total + 255) / 256;
  if (grid > 152 * 8) grid = 152 * 8;
  if (grid < 1) grid = 1;
  cudaError_t e = launch_k(rope_table_kernel, dim3(grid), dim3(256), 0, s, cu_rows, ctx_len, B, M, D / 2, f, cs);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_rope_apply(uint16_t* Y, int ldy, int heads, int D, const float2* cs, int M, cudaStream_t s) {
  cudaError_t e = launch_k(rope_apply_kernel, dim3(M), dim3(ROPE_THREADS), 0, s, Y, ldy, heads, D, cs);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace spec
