// INT8 per-channel symmetric matmul (TensorTonic "Int8 Matmul with Per-Channel
// Scales"): s_x[b] = max_i |x[b,i]|/127, s_w[j] = max_i |w[i,j]|/127 (all-zero
// line -> 1), codes clip(round(v/s), +-127), a = sum_i x_q*w_q exact in int32,
// y = float(a) * s_x[b] * s_w[j].
//
// tcgen05 has no integer MMA kind on sm_103a, and GB300's integer tensor
// rate is far below its 16-bit one.  Codes in [-127, 127] are exact in bf16
// and their products exact in FP32, so the matmul runs on the bf16 tensor
// cores (tc_gemm_pair kPairI8 in gemm_pair.cu): FP32 sums over chunks of
// 1024 products stay below 2^24 in magnitude, hence exact integers, and are
// added in int32.  Kernels here:
//   i8_quant_rows   one CTA per row of x: absmax, scale, codes into x_q and a
//                   zero-padded K-major copy [B, Kp] the matmul reads (bf16,
//                   or int8 for the fallback below).
//   i8_quant_w_strip  all of w in one launch: a cluster of eight CTAs per
//                   strip of 32 columns takes the column maxima (combined
//                   through distributed shared memory), then the codes in the
//                   page's layout [D_in, D_out] and transposed [D_out, Kp].
//   i8_colmax, i8_quant_cols  the same in two launches (maxima by integer
//                   atomicMax on the non-negative float bits; codes through
//                   a shared-memory tile) where D_out % 4 != 0 or w is not
//                   16-byte aligned.
//   i8_gemm         fallback for outputs TMA cannot store (D_out % 4 != 0 or
//                   unaligned y): the warp-level integer MMA (mma.sync
//                   m16n8k32 s8.s8.s32, exact int32), 128x128 CTA tile,
//                   4-stage cp.async pipeline, XOR-swizzled shared memory.
#include <cuda_bf16.h>

#include <cstdlib>
#include <mutex>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "quotient.cuh"

namespace bsmm {
namespace {

constexpr int kKpAlign = 128;  // padded K, elements per operand row (int8: 128-byte rows; bf16: 4 K blocks)

__device__ __forceinline__ float i8_scale(float absmax) {
  return absmax == 0.f ? 1.f : __fdiv_rn(absmax, 127.f);
}
// round(clamp(v / s, -127, 127)), ties to even; y = block_recip(s).
__device__ __forceinline__ int8_t i8_code(float v, float s, float y) {
  const float q = fminf(fmaxf(y != 0.f ? quot_rn(v, s, y) : __fdiv_rn(v, s), -127.f), 127.f);
  return static_cast<int8_t>(__float2int_rn(q));
}

// The same for two elements, kept as floats t = q + 1.5 * 2^23: adding the
// constant rounds the clamped quotient q to the nearest integer k (ties to
// even: the ulp there is 1) and leaves k in the low bits of t's significand,
// so t's low byte is k's two's-complement byte, and t - 1.5 * 2^23 is k as
// an exact float (+0 for k = 0), whose upper 16 bits are k in bfloat16.
// As with the division, a NaN element clamps to -127.
constexpr float kRoundMagic = 12582912.f;  // 1.5 * 2^23
__device__ __forceinline__ float2 i8_round2(float v0, float v1, float s, float y) {
  float2 q = y != 0.f ? quot2_rn_int(make_float2(v0, v1), s, y) : make_float2(__fdiv_rn(v0, s), __fdiv_rn(v1, s));
  q.x = fminf(fmaxf(q.x, -127.f), 127.f);
  q.y = fminf(fmaxf(q.y, -127.f), 127.f);
  return __fadd2_rn(q, make_float2(kRoundMagic, kRoundMagic));
}
// Code bytes of four rounded elements, element a lowest.
__device__ __forceinline__ uint32_t i8_bytes4(float ta, float tb, float tc, float td) {
  return __byte_perm(__byte_perm(__float_as_uint(ta), __float_as_uint(tb), 0x0040),
                     __byte_perm(__float_as_uint(tc), __float_as_uint(td), 0x0040), 0x5410);
}
// bfloat16 copies of two rounded elements, element a in the low half.
__device__ __forceinline__ uint32_t i8_bf16x2(float ta, float tb) {
  const float2 k = __fadd2_rn(make_float2(ta, tb), make_float2(-kRoundMagic, -kRoundMagic));
  return __byte_perm(__float_as_uint(k.x), __float_as_uint(k.y), 0x7632);
}
template <typename Pad>
__device__ __forceinline__ Pad pad_code(int8_t q);
template <>
__device__ __forceinline__ int8_t pad_code<int8_t>(int8_t q) {
  return q;
}
template <>
__device__ __forceinline__ __nv_bfloat16 pad_code<__nv_bfloat16>(int8_t q) {
  return __int2bfloat16_rn(q);  // exact: |q| <= 127 < 2^8
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Pad is int8_t (fallback matmul) or __nv_bfloat16 (tensor-core matmul).
template <typename Pad>
__global__ void __launch_bounds__(256) i8_quant_rows(const float* __restrict__ x, int64_t D, int64_t Kp,
                                                     int8_t* __restrict__ xq, float* __restrict__ xs,
                                                     Pad* __restrict__ xq_pad) {
  __shared__ float wmax[8];
  const int64_t r = blockIdx.x;
  const float* row = x + r * D;
  float m = 0.f;
  for (int64_t c = threadIdx.x; c < D; c += 256) m = fmaxf(m, fabsf(__ldg(row + c)));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = wmax[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, wmax[i]);
  const float s = i8_scale(m), y = block_recip(s);
  if (threadIdx.x == 0) xs[r] = s;
  for (int64_t c = threadIdx.x; c < Kp; c += 256) {
    const int8_t q = c < D ? i8_code(__ldg(row + c), s, y) : int8_t(0);
    if (c < D) xq[r * D + c] = q;
    xq_pad[r * Kp + c] = pad_code<Pad>(q);
  }
}

// The tensor-core path's row quantizer when a row fits in registers (D % 4
// == 0, x 16-byte and x_q 4-byte aligned, D <= 1024 V): each of 256 threads
// keeps V float4 of the row, so x is read once, and the codes leave as
// 4-byte (int8) and 8-byte (bf16) stores.
template <int V>
__global__ void __launch_bounds__(256) i8_quant_rows_reg(const float* __restrict__ x, int64_t D, int64_t Kp,
                                                         int8_t* __restrict__ xq, float* __restrict__ xs,
                                                         __nv_bfloat16* __restrict__ xb) {
  __shared__ float wmax[8];
  const int64_t r = blockIdx.x;
  const float4* row = reinterpret_cast<const float4*>(x + r * D);
  const int n4 = static_cast<int>(D / 4);
  float4 v[V];
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int c4 = threadIdx.x + 256 * i;
    v[i] = c4 < n4 ? __ldg(row + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
  }
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = wmax[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, wmax[i]);
  const float s = i8_scale(m), y = block_recip(s);
  if (threadIdx.x == 0) xs[r] = s;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int c4 = threadIdx.x + 256 * i;
    if (c4 < n4) {
      const float2 t01 = i8_round2(v[i].x, v[i].y, s, y), t23 = i8_round2(v[i].z, v[i].w, s, y);
      *reinterpret_cast<uint32_t*>(xq + r * D + 4 * c4) = i8_bytes4(t01.x, t01.y, t23.x, t23.y);
      *reinterpret_cast<uint2*>(xb + r * Kp + 4 * c4) = make_uint2(i8_bf16x2(t01.x, t01.y), i8_bf16x2(t23.x, t23.y));
    }
  }
  for (int64_t c = D + threadIdx.x; c < Kp; c += 256) xb[r * Kp + c] = __int2bfloat16_rn(0);
}

// Column maxima, four columns per thread (D_out % 4 == 0, w 16-byte
// aligned): grid (ceil(D_out/128), row chunks), 8 warps stride rows with four
// 16-byte loads in flight per thread.
__global__ void __launch_bounds__(256) i8_colmax4(const float* __restrict__ w, int64_t D_in, int64_t D_out,
                                                  int rows_per_cta, unsigned* __restrict__ colmax) {
  __shared__ float4 wm[8][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c4 = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const int64_t n4 = D_out / 4;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_cta;
  const int64_t r1 = (D_in < r0 + rows_per_cta) ? D_in : r0 + rows_per_cta;
  float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c4 < n4) {
    const float4* base = reinterpret_cast<const float4*>(w) + c4;
    int64_t r = r0 + warp;
    for (; r + 24 < r1; r += 32) {
      float4 t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) t[u] = __ldg(base + (r + 8 * u) * n4);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        m.x = fmaxf(m.x, fabsf(t[u].x));
        m.y = fmaxf(m.y, fabsf(t[u].y));
        m.z = fmaxf(m.z, fabsf(t[u].z));
        m.w = fmaxf(m.w, fabsf(t[u].w));
      }
    }
    for (; r < r1; r += 8) {
      const float4 t = __ldg(base + r * n4);
      m.x = fmaxf(m.x, fabsf(t.x));
      m.y = fmaxf(m.y, fabsf(t.y));
      m.z = fmaxf(m.z, fabsf(t.z));
      m.w = fmaxf(m.w, fabsf(t.w));
    }
  }
  wm[warp][lane] = m;
  __syncthreads();
  if (warp == 0 && c4 < n4) {
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      m.x = fmaxf(m.x, wm[i][lane].x);
      m.y = fmaxf(m.y, wm[i][lane].y);
      m.z = fmaxf(m.z, wm[i][lane].z);
      m.w = fmaxf(m.w, wm[i][lane].w);
    }
    unsigned* cm = colmax + 4 * c4;
    atomicMax(cm + 0, __float_as_uint(m.x));  // non-negative floats order like their bits
    atomicMax(cm + 1, __float_as_uint(m.y));
    atomicMax(cm + 2, __float_as_uint(m.z));
    atomicMax(cm + 3, __float_as_uint(m.w));
  }
}

// grid (ceil(D_out/32), row chunks); lane = column, 8 warps stride rows.
__global__ void __launch_bounds__(256) i8_colmax(const float* __restrict__ w, int64_t D_in, int64_t D_out,
                                                 int rows_per_cta, unsigned* __restrict__ colmax) {
  __shared__ float wm[8][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_cta;
  const int64_t r1 = (D_in < r0 + rows_per_cta) ? D_in : r0 + rows_per_cta;
  float m = 0.f;
  if (c < D_out)
    for (int64_t r = r0 + warp; r < r1; r += 8) m = fmaxf(m, fabsf(__ldg(w + r * D_out + c)));
  wm[warp][lane] = m;
  __syncthreads();
  if (warp == 0 && c < D_out) {
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, wm[i][lane]);
    atomicMax(colmax + c, __float_as_uint(m));  // non-negative floats order like their bits
  }
}

// 64 x 64 tiles of w (rows i over Kp, columns j): codes into w_q[i][j] and
// wqT[j][i]; rows i >= D_in give zero codes in wqT (the K padding).
template <typename Pad>
__global__ void __launch_bounds__(256) i8_quant_cols(const float* __restrict__ w, int64_t D_in, int64_t D_out,
                                                     int64_t Kp, const unsigned* __restrict__ colmax,
                                                     int8_t* __restrict__ wq, float* __restrict__ ws,
                                                     Pad* __restrict__ wqT) {
  __shared__ int8_t tile[64][64 + 4];
  const int64_t i0 = static_cast<int64_t>(blockIdx.y) * 64, j0 = static_cast<int64_t>(blockIdx.x) * 64;
  const int t = threadIdx.x;
  const int jj = t & 63, ig = t >> 6;  // column in tile, row group (16 rows each)
  const int64_t j = j0 + jj;
  const float s = j < D_out ? i8_scale(__uint_as_float(colmax[j])) : 1.f, y = block_recip(s);
  if (blockIdx.y == 0 && ig == 0 && j < D_out) ws[j] = s;
  float v[16];  // all sixteen loads in flight before any arithmetic
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int64_t i = i0 + ig * 16 + k;
    v[k] = (i < D_in && j < D_out) ? __ldg(w + i * D_out + j) : 0.f;
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int ii = ig * 16 + k;
    const int64_t i = i0 + ii;
    int8_t q = 0;
    if (i < D_in && j < D_out) {
      q = i8_code(v[k], s, y);
      wq[i * D_out + j] = q;
    }
    tile[ii][jj] = q;
  }
  __syncthreads();
  // transposed write: thread -> (row j of wqT, 16 consecutive i)
  const int jt = t >> 2, part = t & 3;
  const int64_t jrow = j0 + jt;
  if (wqT != nullptr && jrow < D_out) {  // no matmul copy when x has no rows
    const int64_t ibase = i0 + part * 16;
    if (ibase < Kp) {
      if constexpr (sizeof(Pad) == 1) {
        uint32_t word[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          word[g] = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            word[g] |= static_cast<uint32_t>(static_cast<uint8_t>(tile[part * 16 + 4 * g + b][jt])) << (8 * b);
        }
        *reinterpret_cast<uint4*>(wqT + jrow * Kp + ibase) = make_uint4(word[0], word[1], word[2], word[3]);
      } else {
        uint32_t word[8];  // 16 bf16 codes, two per word
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const __nv_bfloat16 lo = __int2bfloat16_rn(tile[part * 16 + 2 * g][jt]);
          const __nv_bfloat16 hi = __int2bfloat16_rn(tile[part * 16 + 2 * g + 1][jt]);
          word[g] = static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
                    (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
        }
        uint4* dst = reinterpret_cast<uint4*>(wqT + jrow * Kp + ibase);
        dst[0] = make_uint4(word[0], word[1], word[2], word[3]);
        dst[1] = make_uint4(word[4], word[5], word[6], word[7]);
      }
    }
  }
}

// All of w's per-column quantization in one kernel.  A strip of 32 columns
// goes to a cluster of eight CTAs, CTA q taking rows q Kp/8 .. (q+1) Kp/8 - 1.
// Thread (warp, lane) owns columns 4 (lane % 8) .. +3 of the strip and, in
// each step of 256 rows, the 8 consecutive rows 8 (4 warp + lane / 8) .. +7.
// Pass 1: column maxima of the CTA's rows; the eight CTAs combine them
// through distributed shared memory.  Up to 512 rows a CTA (D_in <= 4096)
// the rows stay in registers between the passes (RES = 2: 16 x 16-byte
// loads in flight per thread, two CTAs per SM), so w is read once; beyond
// that pass 1 streams them (8 loads in flight) and pass 2 reads them again,
// from L2 when w fits there.
// Pass 2 writes the codes into w_q [D_in, D_out] (32
// bytes a row per strip) and into wqT [D_out, Kp], where a thread's 8 codes
// of one column are 8 consecutive elements of a row (zero codes for rows
// >= D_in).  Needs D_out % 4 == 0, w 16-byte and w_q 4-byte aligned.
// At D = 4096 the eight CTAs a strip make 1024 CTAs, two per SM (3.4
// waves).  Measured there (one launch, cold): 37 us with the rows held in
// registers and 37 streamed twice, 35 with sixteen CTAs a strip, 45 with
// 64-column strips; strip width and split are compile-time constants.
constexpr int kStrip = 32, kStripSplit = 8, kStripResident = 2;
constexpr int kStripCG = kStrip / 4;                  // 16-byte column groups per row
constexpr int kStripRows = 8 * (256 / kStripCG);      // rows per step of 256 threads
template <typename Pad, int RES>
__global__ void __launch_bounds__(256, RES ? 2 : 4) i8_quant_w_strip(const float* __restrict__ w, int64_t D_in,
                                                                  int64_t D_out, int64_t Kp, int8_t* __restrict__ wq,
                                                                  float* __restrict__ ws, Pad* __restrict__ wqT) {
  __shared__ float red[8][kStrip];  // [warp][column]
  __shared__ float part_max[kStrip];
  __shared__ float sc[kStrip], yc[kStrip];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int cg = lane % kStripCG;
  const int rsub = warp * (32 / kStripCG) + lane / kStripCG;  // 8-row group of the step
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kStrip;
  const int64_t jc = j0 + 4 * cg;
  const bool col_ok = jc < D_out;  // D_out % 4 == 0: all four in or all out
  const int64_t n4 = D_out / 4;
  const float4* base = reinterpret_cast<const float4*>(w) + (jc / 4);
  const uint32_t q = cluster_ctarank();
  const int64_t Kq = Kp / kStripSplit;  // a multiple of 16 (Kp % 128 == 0)
  const int64_t rbeg = q * Kq, rend = rbeg + Kq;
  const int64_t dend = D_in < rend ? D_in : rend;
  // pass 1: column maxima of this CTA's rows
  float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 keep[RES ? RES : 1][8];  // RES > 0: all of the CTA's rows, held for pass 2
  if constexpr (RES > 0) {
#pragma unroll
    for (int it = 0; it < RES; ++it)
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t r = rbeg + kStripRows * it + 8 * rsub + u;
        keep[it][u] = (col_ok && r < dend) ? __ldg(base + r * n4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int it = 0; it < RES; ++it)
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        m.x = fmaxf(m.x, fabsf(keep[it][u].x));
        m.y = fmaxf(m.y, fabsf(keep[it][u].y));
        m.z = fmaxf(m.z, fabsf(keep[it][u].z));
        m.w = fmaxf(m.w, fabsf(keep[it][u].w));
      }
  } else if (col_ok) {
    for (int64_t r0 = rbeg; r0 < dend; r0 += kStripRows) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t r = r0 + 8 * rsub + u;
        v[u] = r < dend ? __ldg(base + r * n4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        m.x = fmaxf(m.x, fabsf(v[u].x));
        m.y = fmaxf(m.y, fabsf(v[u].y));
        m.z = fmaxf(m.z, fabsf(v[u].z));
        m.w = fmaxf(m.w, fabsf(v[u].w));
      }
    }
  }
#pragma unroll
  for (int o = kStripCG; o < 32; o <<= 1) {  // over the lanes holding the same columns
    m.x = fmaxf(m.x, __shfl_xor_sync(0xffffffffu, m.x, o));
    m.y = fmaxf(m.y, __shfl_xor_sync(0xffffffffu, m.y, o));
    m.z = fmaxf(m.z, __shfl_xor_sync(0xffffffffu, m.z, o));
    m.w = fmaxf(m.w, __shfl_xor_sync(0xffffffffu, m.w, o));
  }
  if (lane < kStripCG) {
    red[warp][4 * lane + 0] = m.x;
    red[warp][4 * lane + 1] = m.y;
    red[warp][4 * lane + 2] = m.z;
    red[warp][4 * lane + 3] = m.w;
  }
  __syncthreads();
  if (t < kStrip) {
    float mm = red[0][t];
#pragma unroll
    for (int i = 1; i < 8; ++i) mm = fmaxf(mm, red[i][t]);
    part_max[t] = mm;
  }
  cluster_sync();  // the strip's partial maxima are visible
  if (t < kStrip) {
    const uint32_t a = smem_u32(&part_max[t]);
    float mm = 0.f;
#pragma unroll
    for (int c = 0; c < kStripSplit; ++c) mm = fmaxf(mm, ld_shared_cluster_f32(mapa_shared(a, c)));
    const float sv = i8_scale(mm);
    sc[t] = sv;
    yc[t] = block_recip(sv);
    if (q == 0 && j0 + t < D_out) ws[j0 + t] = sv;
  }
  cluster_sync();  // peers have read part_max; sc is visible to the CTA
  float scol[4], ycol[4];  // the thread's four columns
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    scol[c] = sc[4 * cg + c];
    ycol[c] = yc[4 * cg + c];
  }
  // pass 2: codes, 256 rows at a time (rend - i0 is a multiple of 8, so a
  // thread's 8 rows are all below rend or all at or above it)
  const int n_it = RES ? RES : static_cast<int>((rend - rbeg + kStripRows - 1) / kStripRows);
#pragma unroll
  for (int it = 0; it < n_it; ++it) {
    const int64_t ir = rbeg + kStripRows * static_cast<int64_t>(it) + 8 * rsub;
    if (ir >= rend) break;
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if constexpr (RES > 0)
        v[u] = keep[it][u];
      else
        v[u] = (col_ok && ir + u < dend) ? __ldg(base + (ir + u) * n4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float2 t[4][4];  // column c, rows 2g and 2g + 1, rounded (i8_round2)
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      t[0][g] = i8_round2(v[2 * g].x, v[2 * g + 1].x, scol[0], ycol[0]);
      t[1][g] = i8_round2(v[2 * g].y, v[2 * g + 1].y, scol[1], ycol[1]);
      t[2][g] = i8_round2(v[2 * g].z, v[2 * g + 1].z, scol[2], ycol[2]);
      t[3][g] = i8_round2(v[2 * g].w, v[2 * g + 1].w, scol[3], ycol[3]);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {  // row u: the four columns' codes, low byte first
      const int g = u >> 1;
      const uint32_t code = (u & 1) ? i8_bytes4(t[0][g].y, t[1][g].y, t[2][g].y, t[3][g].y)
                                    : i8_bytes4(t[0][g].x, t[1][g].x, t[2][g].x, t[3][g].x);
      if (col_ok && ir + u < dend) *reinterpret_cast<uint32_t*>(wq + (ir + u) * D_out + jc) = code;
    }
    if (wqT != nullptr && col_ok) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // column jc + c: rows ir .. ir+7
        Pad* dst = wqT + (jc + c) * Kp + ir;
        if constexpr (sizeof(Pad) == 1) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(i8_bytes4(t[c][0].x, t[c][0].y, t[c][1].x, t[c][1].y),
                                                      i8_bytes4(t[c][2].x, t[c][2].y, t[c][3].x, t[c][3].y));
        } else {
          *reinterpret_cast<uint4*>(dst) = make_uint4(i8_bf16x2(t[c][0].x, t[c][0].y), i8_bf16x2(t[c][1].x, t[c][1].y),
                                                      i8_bf16x2(t[c][2].x, t[c][2].y), i8_bf16x2(t[c][3].x, t[c][3].y));
        }
      }
    }
  }
}

// A second stream per device, on which w's quantization runs beside x's: it
// forks from the caller's stream after its earlier work and joins back before
// the matmul.  The record / wait pairs are made under a lock, so that calls
// from several host threads never wait on each other's event records.
std::mutex g_side_mutex;
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[64];

cudaError_t side_fork(int dev, cudaStream_t main, cudaStream_t* side) {
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_side_mutex);
  SideStream& ss = g_side[dev];
  if (!ss.s) {
    cudaError_t e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaEventRecord(ss.fork, main);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ss.s, ss.fork, 0);
  *side = ss.s;
  return e;
}

cudaError_t side_join(int dev, cudaStream_t main) {
  std::lock_guard<std::mutex> lock(g_side_mutex);
  SideStream& ss = g_side[dev];
  cudaError_t e = cudaEventRecord(ss.join, ss.s);
  return e == cudaSuccess ? cudaStreamWaitEvent(main, ss.join, 0) : e;
}

template <typename Pad>
cudaError_t launch_w_strip(const Int8Request& r, int64_t Kp, Pad* wqT, cudaStream_t s) {
  // up to 512 rows per CTA stay in registers between the two passes
  const bool resident = Kp / kStripSplit <= kStripRows * kStripResident;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = kStripSplit;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(r.D_out, kStrip)), kStripSplit, 1);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  TraceScope tr("i8_quant_w_strip", s);
  if (resident)
    return cudaLaunchKernelEx(&cfg, i8_quant_w_strip<Pad, kStripResident>, r.w, static_cast<int64_t>(r.D_in),
                              static_cast<int64_t>(r.D_out), Kp, r.w_q, r.w_scales, wqT);
  return cudaLaunchKernelEx(&cfg, i8_quant_w_strip<Pad, 0>, r.w, static_cast<int64_t>(r.D_in),
                            static_cast<int64_t>(r.D_out), Kp, r.w_q, r.w_scales, wqT);
}

// ---------------------------------------------------------------- the matmul
constexpr int GM = 128, GN = 128, GK = 128, GSTAGES = 4;
constexpr int G_STAGE_BYTES = (GM + GN) * GK;

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_s8(int (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// 16-byte chunk `c` of row `r` in a [rows][128 B] tile, XOR-swizzled.
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int c) {
  return base + r * GK + ((c ^ (r & 7)) << 4);
}

__global__ void __launch_bounds__(256) i8_gemm(const int8_t* __restrict__ A, const int8_t* __restrict__ Bt, int M,
                                               int N, int Kp, const float* __restrict__ sx,
                                               const float* __restrict__ sw, float* __restrict__ y,
                                               int32_t* __restrict__ acc_out) {
  extern __shared__ __align__(128) uint8_t gsm[];
  const uint32_t sbase = smem_u32(gsm);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int m0 = blockIdx.y * GM, n0 = blockIdx.x * GN;
  const int ktiles = Kp / GK;

  auto load_stage = [&](int st, int kt) {
    const uint32_t sa = sbase + st * G_STAGE_BYTES, sb = sa + GM * GK;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // 1024 chunks of A, 1024 of B; 4 + 4 per thread
      const int idx = t + 256 * i;
      const int r = idx >> 3, c = idx & 7;
      const int gm = m0 + r, gn = n0 + r;
      const int8_t* pa = A + static_cast<int64_t>(gm < M ? gm : 0) * Kp + kt * GK + c * 16;
      const int8_t* pb = Bt + static_cast<int64_t>(gn < N ? gn : 0) * Kp + kt * GK + c * 16;
      cp_async16(swz(sa, r, c), pa, gm < M ? 16 : 0);
      cp_async16(swz(sb, r, c), pb, gn < N ? 16 : 0);
    }
  };

  int acc[4][4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][b][c] = 0;

#pragma unroll
  for (int st = 0; st < GSTAGES - 1; ++st) {
    if (st < ktiles) load_stage(st, st);
    cp_async_commit();
  }
  const int wm = warp >> 2, wn = warp & 3;  // warp tile rows wm*64, cols wn*32
  for (int kt = 0; kt < ktiles; ++kt) {
    cp_async_wait<GSTAGES - 2>();
    __syncthreads();
    {
      const int nk = kt + GSTAGES - 1;
      if (nk < ktiles) load_stage(nk % GSTAGES, nk);
      cp_async_commit();
    }
    const uint32_t sa = sbase + (kt % GSTAGES) * G_STAGE_BYTES, sb = sa + GM * GK;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {  // 32-byte K steps
      uint32_t af[4][4], bf[4][2];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        const int r = wm * 64 + mi * 16 + (lane & 15);
        const int c = 2 * kk + (lane >> 4);
        ldmatrix_x4(swz(sa, r, c), af[mi][0], af[mi][1], af[mi][2], af[mi][3]);
      }
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        const int r = wn * 32 + nj * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = 2 * kk + ((lane >> 3) & 1);
        ldmatrix_x4(swz(sb, r, c), bf[2 * nj][0], bf[2 * nj][1], bf[2 * nj + 1][0], bf[2 * nj + 1][1]);
      }
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) mma_s8(acc[mi][ni], af[mi], bf[ni][0], bf[ni][1]);
    }
  }
  cp_async_wait<0>();

  const int gr = lane >> 2, tc = lane & 3;
#pragma unroll
  for (int mi = 0; mi < 4; ++mi) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = m0 + wm * 64 + mi * 16 + gr + 8 * h;
      if (row >= M) continue;
      const float srow = sx[row];
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) {
        const int col = n0 + wn * 32 + ni * 8 + 2 * tc;
        const int a0 = acc[mi][ni][2 * h], a1 = acc[mi][ni][2 * h + 1];
        const int64_t o = static_cast<int64_t>(row) * N + col;
        if (col + 1 < N) {
          const float y0 = (static_cast<float>(a0) * srow) * sw[col];
          const float y1 = (static_cast<float>(a1) * srow) * sw[col + 1];
          if ((N & 1) == 0) {
            *reinterpret_cast<float2*>(y + o) = make_float2(y0, y1);
            if (acc_out) *reinterpret_cast<int2*>(acc_out + o) = make_int2(a0, a1);
          } else {
            y[o] = y0;
            y[o + 1] = y1;
            if (acc_out) {
              acc_out[o] = a0;
              acc_out[o + 1] = a1;
            }
          }
        } else if (col < N) {
          y[o] = (static_cast<float>(a0) * srow) * sw[col];
          if (acc_out) acc_out[o] = a0;
        }
      }
    }
  }
}

}  // namespace

// The split matmul's counters (kSplitTilesMax x 32) and int32 partial tiles.
constexpr size_t kSplitCntBytes = static_cast<size_t>(kSplitTilesMax) * 32 * 4;
size_t int8_split_bytes(int64_t B, int64_t D_out) {
  const int64_t tiles = ceil_div(B, 256) * ceil_div(D_out, 256);
  return kSplitCntBytes + static_cast<size_t>(int8_split_units(tiles)) * 256 * 256 * 4;
}

size_t int8_workspace_bytes(int64_t B, int64_t D_in, int64_t D_out) {
  // room for the bf16 operand copies (the fallback's int8 copies fit
  // inside), then the split matmul's counters and partial sums
  const int64_t Kp = ceil_div(D_in, kKpAlign) * kKpAlign;
  return align_up(static_cast<size_t>(D_out) * 4, 256) + align_up(static_cast<size_t>(B) * Kp * 2, 256) +
         align_up(static_cast<size_t>(D_out) * Kp * 2, 256) + int8_split_bytes(B, D_out);
}

cudaError_t launch_int8_channel(const Int8Request& r, cudaStream_t s) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  const int64_t Kp = ceil_div(r.D_in, kKpAlign) * kKpAlign;  // elements
  uint8_t* ws = reinterpret_cast<uint8_t*>(r.workspace);
  unsigned* colmax = reinterpret_cast<unsigned*>(ws);
  uint8_t* xpad = ws + align_up(static_cast<size_t>(r.D_out) * 4, 256);
  uint8_t* wpadT = xpad + align_up(static_cast<size_t>(r.B) * Kp * 2, 256);
  uint8_t* split = wpadT + align_up(static_cast<size_t>(r.D_out) * Kp * 2, 256);  // B > 0 only
  // The tensor-core path stores y (and the int32 sums) through TMA: 16-byte
  // rows and bases.  BSMM_INT8_KERNEL=mma forces the fallback.
  const char* force = std::getenv("BSMM_INT8_KERNEL");
  const bool tc = !(force && std::strcmp(force, "mma") == 0) && (r.D_out * 4) % 16 == 0 &&
                  reinterpret_cast<uintptr_t>(r.y) % 16 == 0 && reinterpret_cast<uintptr_t>(r.acc) % 16 == 0;

  // w's quantization in one pass over strips of columns (16-byte loads)
  const bool w_strip = (r.D_out % 4) == 0 && (reinterpret_cast<uintptr_t>(r.w) & 15) == 0 &&
                       (reinterpret_cast<uintptr_t>(r.w_q) & 3) == 0;
  cudaError_t e = cudaSuccess;
  if (!w_strip) {
    e = cudaMemsetAsync(colmax, 0, static_cast<size_t>(r.D_out) * 4, s);
    if (e != cudaSuccess) return e;
  }
  if (r.B == 0 && w_strip) {  // w alone: codes and scales (no transposed copy)
    return launch_w_strip<int8_t>(r, Kp, nullptr, s);
  }
  if (r.B == 0) {  // w alone: column maxima, then codes and scales (no transposed copy)
    const int rows_per_cta = 256;
    dim3 g1(static_cast<unsigned>(ceil_div(r.D_out, 32)), static_cast<unsigned>(ceil_div(r.D_in, rows_per_cta)));
    {
      TraceScope tr("i8_colmax", s);
      i8_colmax<<<g1, 256, 0, s>>>(r.w, r.D_in, r.D_out, rows_per_cta, colmax);
    }
    dim3 g2(static_cast<unsigned>(ceil_div(r.D_out, 64)), static_cast<unsigned>(Kp / 64));
    {
      TraceScope tr("i8_quant_cols", s);
      i8_quant_cols<int8_t><<<g2, 256, 0, s>>>(r.w, r.D_in, r.D_out, Kp, colmax, r.w_q, r.w_scales, nullptr);
    }
    return cudaGetLastError();
  }
  // w's quantization beside x's on the side stream (tensor-core path)
  const bool side = tc && w_strip;
  if (side) {
    cudaStream_t ss;
    e = side_fork(ctx->device, s, &ss);
    if (e == cudaSuccess) e = launch_w_strip<__nv_bfloat16>(r, Kp, reinterpret_cast<__nv_bfloat16*>(wpadT), ss);
    if (e != cudaSuccess) return e;
  }
  const bool rows_vec = (r.D_in % 4) == 0 && (reinterpret_cast<uintptr_t>(r.x) & 15) == 0 &&
                        (reinterpret_cast<uintptr_t>(r.x_q) & 3) == 0 && r.D_in <= 8192;
  __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(xpad);
  const unsigned nrows = static_cast<unsigned>(r.B);
  if (tc) {  // the split matmul's counters start from zero
    e = cudaMemsetAsync(split, 0, kSplitCntBytes, s);
    if (e != cudaSuccess) return e;
  }
  if (tc && rows_vec) {
    if (r.D_in <= 1024) {
      TraceScope tr("i8_quant_rows_reg", s);
      i8_quant_rows_reg<1><<<nrows, 256, 0, s>>>(r.x, r.D_in, Kp, r.x_q, r.x_scales, xb);
    } else if (r.D_in <= 2048) {
      TraceScope tr("i8_quant_rows_reg", s);
      i8_quant_rows_reg<2><<<nrows, 256, 0, s>>>(r.x, r.D_in, Kp, r.x_q, r.x_scales, xb);
    } else if (r.D_in <= 4096) {
      TraceScope tr("i8_quant_rows_reg", s);
      i8_quant_rows_reg<4><<<nrows, 256, 0, s>>>(r.x, r.D_in, Kp, r.x_q, r.x_scales, xb);
    } else {
      TraceScope tr("i8_quant_rows_reg", s);
      i8_quant_rows_reg<8><<<nrows, 256, 0, s>>>(r.x, r.D_in, Kp, r.x_q, r.x_scales, xb);
    }
  } else if (tc) {
    TraceScope tr("i8_quant_rows", s);
    i8_quant_rows<__nv_bfloat16><<<nrows, 256, 0, s>>>(r.x, r.D_in, Kp, r.x_q, r.x_scales, xb);
  } else {
    TraceScope tr("i8_quant_rows", s);
    i8_quant_rows<int8_t><<<static_cast<unsigned>(r.B), 256, 0, s>>>(r.x, r.D_in, Kp, r.x_q, r.x_scales,
                                                                     reinterpret_cast<int8_t*>(xpad));
  }
  if (side) {
    e = side_join(ctx->device, s);
    if (e != cudaSuccess) return e;
  } else if (w_strip) {
    e = launch_w_strip<int8_t>(r, Kp, reinterpret_cast<int8_t*>(wpadT), s);
    if (e != cudaSuccess) return e;
  } else if ((r.D_out % 4) == 0 && (reinterpret_cast<uintptr_t>(r.w) & 15) == 0) {
    const int rows_per_cta = 256;
    dim3 grid(static_cast<unsigned>(ceil_div(r.D_out, 128)), static_cast<unsigned>(ceil_div(r.D_in, rows_per_cta)));
    {
      TraceScope tr("i8_colmax4", s);
      i8_colmax4<<<grid, 256, 0, s>>>(r.w, r.D_in, r.D_out, rows_per_cta, colmax);
    }
  } else {
    const int rows_per_cta = 256;
    dim3 grid(static_cast<unsigned>(ceil_div(r.D_out, 32)), static_cast<unsigned>(ceil_div(r.D_in, rows_per_cta)));
    {
      TraceScope tr("i8_colmax", s);
      i8_colmax<<<grid, 256, 0, s>>>(r.w, r.D_in, r.D_out, rows_per_cta, colmax);
    }
  }
  if (!w_strip) {
    dim3 grid(static_cast<unsigned>(ceil_div(r.D_out, 64)), static_cast<unsigned>(Kp / 64));
    if (tc) {
      TraceScope tr("i8_quant_cols", s);
      i8_quant_cols<__nv_bfloat16><<<grid, 256, 0, s>>>(r.w, r.D_in, r.D_out, Kp, colmax, r.w_q, r.w_scales,
                                                        reinterpret_cast<__nv_bfloat16*>(wpadT));
    } else {
      TraceScope tr("i8_quant_cols", s);
      i8_quant_cols<int8_t><<<grid, 256, 0, s>>>(r.w, r.D_in, r.D_out, Kp, colmax, r.w_q, r.w_scales,
                                                 reinterpret_cast<int8_t*>(wpadT));
    }
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (tc) {
    std::string why;
    // BSMM_INT8_SPLIT=0 keeps every tile whole
    const char* no_split = std::getenv("BSMM_INT8_SPLIT");
    const bool split_ok = !(no_split && std::strcmp(no_split, "0") == 0);
    e = launch_int8_gemm_pair(r, xpad, wpadT, Kp, split_ok ? reinterpret_cast<int32_t*>(split + kSplitCntBytes) : nullptr,
                              split_ok ? reinterpret_cast<unsigned*>(split) : nullptr, s, &why);
    if (e != cudaSuccess && !why.empty()) set_error(why);
    return e;
  }
  const int smem = GSTAGES * G_STAGE_BYTES;
  e = cudaFuncSetAttribute(i8_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(ceil_div(r.D_out, GN)), static_cast<unsigned>(ceil_div(r.B, GM)));
  {
    TraceScope tr("i8_gemm", s);
    i8_gemm<<<grid, 256, smem, s>>>(reinterpret_cast<const int8_t*>(xpad), reinterpret_cast<const int8_t*>(wpadT),
                                    static_cast<int>(r.B), static_cast<int>(r.D_out), static_cast<int>(Kp), r.x_scales,
                                    r.w_scales, r.y, r.acc);
  }
  return cudaGetLastError();
}

}  // namespace bsmm
