// Block-scaled matmul for any block size, on the CUDA cores
// (jax.nn.scaled_matmul, "Mathematically" and Parameters: the block size is
// K / K_a, K / K_b, whatever it is).
//
// The tensor cores apply scale factors only per 32 (UE8M0) or 16 (UE4M3)
// elements.  Blocks that are multiples of those take the tensor-core path
// with each scale repeated (gemm_tc.cu); every other block size -- e.g. the
// jax cuDNN example's UE8M0 scales per 16 FP8 elements -- is computed here:
// each operand element is decoded and multiplied by its block's scale into an
// FP32 shared-memory tile (both factors have at most 4 significant bits, so
// the product is exact), and the tiles are multiplied with FP32 FMAs.
//
// CTA: 256 threads, a 64 x 64 output tile, K steps of 32; thread (ty, tx)
// owns rows 4ty..4ty+3 and columns 4tx..4tx+3 of the tile.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"

namespace bsmm {
namespace {

constexpr int GT = 64, GK = 32;

// Exact values of the code and scale formats (OCP FP8 / MX definitions).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t s = b >> 7, e = (b >> 3) & 0xFu, m = b & 7u;
  float v;
  if (e == 15 && m == 7) v = __int_as_float(0x7fc00000);              // NaN
  else if (e == 0) v = static_cast<float>(m) * 0.001953125f;          // m * 2^-9
  else v = __uint_as_float(((e + 120u) << 23) | (m << 20));          // 1.m * 2^(e-7)
  return s ? -v : v;
}
__device__ __forceinline__ float e5m2_value(uint32_t b) {
  const uint32_t s = b >> 7, e = (b >> 2) & 0x1Fu, m = b & 3u;
  float v;
  if (e == 31) v = m ? __int_as_float(0x7fc00000) : __int_as_float(0x7f800000);
  else if (e == 0) v = static_cast<float>(m) * 0.0000152587890625f;  // m * 2^-16
  else v = __uint_as_float(((e + 112u) << 23) | (m << 21));          // 1.m * 2^(e-15)
  return s ? -v : v;
}
__device__ __forceinline__ float e2m1_value(uint32_t nib) {
  const uint32_t e = (nib >> 1) & 3u, m = nib & 1u;
  const float v = e == 0 ? 0.5f * static_cast<float>(m) : __uint_as_float(((e + 126u) << 23) | (m << 22));
  return (nib & 8u) ? -v : v;
}
__device__ __forceinline__ float ue8m0_value(uint32_t b) {
  return b == 255 ? __int_as_float(0x7fc00000) : (b == 0 ? 5.877471754111438e-39f : __uint_as_float(b << 23));
}
__device__ __forceinline__ float ue4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  if (e == 15 && m == 7) return __int_as_float(0x7fc00000);
  if (e == 0) return static_cast<float>(m) * 0.001953125f;
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

struct GenParams {
  int B, M, N, K;
  const uint8_t* a;
  const uint8_t* b;
  int a_type, b_type;
  const uint8_t* sa;
  const uint8_t* sb;
  int K_a, K_b, bs_a, bs_b;
  int scale_type;
  void* y;
  int y_bf16;
};

// Decoded, scaled element k of row r of one operand ([B][R][K] codes, E2M1
// packed two per byte with the even element in the low nibble).
__device__ __forceinline__ float operand(const uint8_t* codes, const uint8_t* scales, int type, int scale_type,
                                         int K, int Ks, int bs, int64_t row, int k) {
  float v;
  if (type == BSMM_E2M1) {
    const uint32_t byte = codes[row * (K / 2) + k / 2];
    v = e2m1_value((k & 1) ? (byte >> 4) : (byte & 0xFu));
  } else {
    const uint32_t byte = codes[row * K + k];
    v = type == BSMM_E4M3 ? e4m3_value(byte) : e5m2_value(byte);
  }
  const uint32_t sb = scales[row * Ks + k / bs];
  return v * (scale_type == BSMM_SCALE_UE8M0 ? ue8m0_value(sb) : ue4m3_value(sb));
}

__global__ void __launch_bounds__(256) gemm_generic(GenParams p) {
  __shared__ float As[GK][GT + 4];
  __shared__ float Bs[GK][GT + 4];
  const int t = threadIdx.x, tx = t & 15, ty = t >> 4;
  const int bz = blockIdx.z;
  const int m0 = blockIdx.y * GT, n0 = blockIdx.x * GT;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < p.K; k0 += GK) {
    // 64 rows x 32 K of each operand: thread t loads K offset t % 32 of
    // rows t / 32 + 8i
    const int kk = t & 31;
    const int k = k0 + kk;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = (t >> 5) + 8 * i;
      const int m = m0 + r, n = n0 + r;
      As[kk][r] = (m < p.M && k < p.K)
                      ? operand(p.a, p.sa, p.a_type, p.scale_type, p.K, p.K_a, p.bs_a,
                                static_cast<int64_t>(bz) * p.M + m, k)
                      : 0.f;
      Bs[kk][r] = (n < p.N && k < p.K)
                      ? operand(p.b, p.sb, p.b_type, p.scale_type, p.K, p.K_b, p.bs_b,
                                static_cast<int64_t>(bz) * p.N + n, k)
                      : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int q = 0; q < GK; ++q) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        av[i] = As[q][4 * ty + i];
        bv[i] = Bs[q][4 * tx + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + 4 * ty + i;
    if (m >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + 4 * tx + j;
      if (n >= p.N) continue;
      const int64_t o = (static_cast<int64_t>(bz) * p.M + m) * p.N + n;
      if (p.y_bf16)
        reinterpret_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(acc[i][j]);
      else
        reinterpret_cast<float*>(p.y)[o] = acc[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_mx_gemm_generic(const MxGemmRequest& r, int64_t K_a, int64_t K_b, int scale_type,
                                   cudaStream_t s) {
  GenParams p{};
  p.B = static_cast<int>(r.B);
  p.M = static_cast<int>(r.M);
  p.N = static_cast<int>(r.N);
  p.K = static_cast<int>(r.K);
  p.a = static_cast<const uint8_t*>(r.a);
  p.b = static_cast<const uint8_t*>(r.b);
  p.a_type = r.a_fmt;
  p.b_type = r.b_fmt;
  p.sa = r.a_scales;
  p.sb = r.b_scales;
  p.K_a = static_cast<int>(K_a);
  p.K_b = static_cast<int>(K_b);
  p.bs_a = static_cast<int>(r.K / K_a);
  p.bs_b = static_cast<int>(r.K / K_b);
  p.scale_type = scale_type;
  p.y = r.y;
  p.y_bf16 = r.y_bf16 ? 1 : 0;
  dim3 grid(static_cast<unsigned>(ceil_div(r.N, GT)), static_cast<unsigned>(ceil_div(r.M, GT)),
            static_cast<unsigned>(r.B));
  {
    TraceScope tr("gemm_generic", s);
    gemm_generic<<<grid, 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace bsmm
