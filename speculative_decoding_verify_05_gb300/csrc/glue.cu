// Layer glue of the decoder stack between the verify GEMMs and attention:
// RMSNorm, rotary position embedding, SwiGLU.  All bandwidth-trivial (M rows
// of a few thousand elements); fp32 math, bf16 storage, 16-byte accesses.
#include "common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int RMS_THREADS = 256;
constexpr int RMS_MAX_VEC = 8;          // 8 x 8 bf16 per thread -> N <= 16384

__global__ void __launch_bounds__(RMS_THREADS)
rmsnorm_kernel(const uint16_t* __restrict__ X, int N, int ldx, const uint16_t* __restrict__ w,
               float eps, uint16_t* __restrict__ Y, int ldy) {
  const int r = blockIdx.x;
  const uint16_t* x = X + (size_t)r * ldx;
  const int nv = N / 8;
  float v[RMS_MAX_VEC][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < RMS_MAX_VEC; ++k) {
    const int c = threadIdx.x + k * RMS_THREADS;
    if (c < nv) {
      const uint4 u = *reinterpret_cast<const uint4*>(x + c * 8);
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
      const uint4 wu = *reinterpret_cast<const uint4*>(w + c * 8);
      const uint32_t w4[4] = {wu.x, wu.y, wu.z, wu.w};
      uint32_t o4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        o4[e] = pack_bf16x2(v[k][2 * e] * rstd * bf16lo(w4[e]), v[k][2 * e + 1] * rstd * bf16hi(w4[e]));
      *reinterpret_cast<uint4*>(y + c * 8) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
  }
}

constexpr int ROPE_THREADS = 256;

__global__ void __launch_bounds__(ROPE_THREADS)
rope_kernel(uint16_t* __restrict__ Q, int ldq, int Hq, uint16_t* __restrict__ K, int ldk, int Hkv,
            int D, const int32_t* __restrict__ cu_rows, const int32_t* __restrict__ ctx_len, int B,
            double theta) {
  const int r = blockIdx.x;
  const int half = D / 2;
  __shared__ float s_cos[128];
  __shared__ float s_sin[128];
  __shared__ int s_pos;
  if (threadIdx.x == 0) {
    int lo = 0, hi = B - 1;           // last b with cu_rows[b] <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu_rows[mid] <= r) lo = mid; else hi = mid - 1;
    }
    s_pos = ctx_len[lo] + (r - cu_rows[lo]);
  }
  __syncthreads();
  if (threadIdx.x < half) {
    // angle in fp64, reduced to [-pi, pi] before the fp32 sincos
    const int i = threadIdx.x;
    const double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
    const double ang = (double)s_pos * inv_freq;
    const double two_pi = 6.283185307179586476925286766559;
    const double red = ang - two_pi * rint(ang / two_pi);
    float sv, cv;
    sincosf((float)red, &sv, &cv);
    s_cos[i] = cv;
    s_sin[i] = sv;
  }
  __syncthreads();
  const int heads = Hq + Hkv;
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
      const float s0 = g0 / (1.f + expf(-g0)), s1 = g1 / (1.f + expf(-g1));
      o4[e] = pack_bf16x2(s0 * bf16lo(u4[e]), s1 * bf16hi(u4[e]));
    }
    *reinterpret_cast<uint4*>(A + (size_t)r * lda + c) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const uint16_t* X, int M, int N, int ldx, const uint16_t* w, float eps,
                           uint16_t* Y, int ldy, cudaStream_t s) {
  rmsnorm_kernel<<<M, RMS_THREADS, 0, s>>>(X, N, ldx, w, eps, Y, ldy);
  return cudaGetLastError();
}

cudaError_t launch_rope(uint16_t* Q, int ldq, int Hq, uint16_t* K, int ldk, int Hkv, int D,
                        const int32_t* cu_rows, const int32_t* ctx_len, int B, int M, float theta,
                        cudaStream_t s) {
  rope_kernel<<<M, ROPE_THREADS, 0, s>>>(Q, ldq, Hq, K, ldk, Hkv, D, cu_rows, ctx_len, B,
                                         (double)theta);
  return cudaGetLastError();
}

cudaError_t launch_silu_mul(const uint16_t* GU, int M, int I, int ldgu, uint16_t* A, int lda,
                            cudaStream_t s) {
  const size_t total = (size_t)M * (I / 8);
  int grid = (int)((total + 255) / 256);
  if (grid > 152 * 16) grid = 152 * 16;
  if (grid < 1) grid = 1;
  silu_mul_kernel<<<grid, 256, 0, s>>>(GU, M, I, ldgu, A, lda);
  return cudaGetLastError();
}

}  // namespace spec
