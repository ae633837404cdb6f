// Absmax block quantizer kernels.
//
// Rule (atrex-bench #002 block_scaled_mm, Input Generation; TensorTonic "Int8
// Matmul with Per-Channel Scales", problem statement): per block, absmax =
// largest |x|; scale from absmax (see make_scale); code = round(x / scale)
// with saturation.  All arithmetic is binary32; every quotient is the
// correctly rounded IEEE x / scale (quotient.cuh: a per-block reciprocal and
// two exact-remainder corrections, or a plain division).
//
// Kernels:
//   quant_rows   1 x {16,32,64,128} blocks along the contiguous axis; a
//                thread owns 16-element slices, 1..8 lanes per block, absmax
//                by xor-shuffle; HBM-streaming.
//   quant_cols   {16,32,64,128} x 1 blocks down the columns; a 128 x 64 tile
//                staged in shared memory, codes written as is or transposed.
//   quant_cols_tma, quant_cols_tma2
//                bf16 columns into transposed 8-bit codes with one-byte
//                scales, tiles fed by a TMA ring; tma2 (32 x 1 blocks) also
//                quantizes the same tiles along their rows (DUAL) or a second
//                array in the same launch (PAIR).
//   quant_tile   128 x 128 blocks (one scale per tile); quant_tile_batch:
//                several such quantizations in one launch.
//   quant_wrow   one block per row (1 x cols).
//   quant_wcol   one block per column (rows x 1).
//   quant_any    one thread per block: every other block shape.
#include <cuda_bf16.h>

#include <algorithm>
#include <vector>

#include "internal.h"
#include "ptx.cuh"
#include "quotient.cuh"

namespace bsmm {
namespace {

struct QP {
  const void* x;
  int64_t rows, cols, ld_x;
  int br, bc;
  int code, scale;
  int transpose;
  void* codes;
  int64_t ld_codes;
  void* scales;
  int64_t ld_scales;
  int sf_atoms;
  int64_t sf_rows, sf_rt, sf_ks4;
};

// Where the scale of output row r, block kb goes: [rows][ld_scales], or the
// tensor-core atom layout (512-byte atoms of 128 rows x 4 blocks; row w of
// the tile at byte (w % 32) * 16 + (w / 32) * 4 + kb % 4).
__device__ __forceinline__ int64_t scale_index(const QP& p, int64_t r, int64_t kb) {
  if (!p.sf_atoms) return r * p.ld_scales + kb;
  const int64_t b = r < p.sf_rows ? 0 : r / p.sf_rows, rr = r - b * p.sf_rows;
  const int w = static_cast<int>(rr & 127);
  return ((b * p.sf_rt + (rr >> 7)) * p.sf_ks4 + (kb >> 2)) * 512 + (w & 31) * 16 + (w >> 5) * 4 + (kb & 3);
}

__device__ __forceinline__ float qmax_of(int code) {
  return code == BSMM_E4M3 ? 448.f : code == BSMM_E5M2 ? 57344.f : code == BSMM_E2M1 ? 6.f : 127.f;
}

// Value of an unsigned E4M3 byte, exactly.
__device__ __forceinline__ float ue4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  if (e == 0) return static_cast<float>(m) * 0.001953125f;  // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));     // 1.m * 2^(e-7)
}

struct Scale {
  float s;          // the divisor
  float inv;        // POW2: 1/s (exact); else RN(1/s) for quotient.cuh, or 0 (divide)
  uint32_t stored;  // what is written: binary32 bits or the scale byte
};

__device__ __forceinline__ Scale make_scale(float absmax, int code, int scale) {
  const float r = __fdiv_rn(absmax, qmax_of(code));
  Scale out;
  if (scale == BSMM_SCALE_F32) {
    // INT8 (TensorTonic): absmax/127, an all-zero block gets 1.
    // FP8/FP4 (atrex-bench): max(absmax/qmax, 1e-10).
    const float s = (code == BSMM_INT8) ? (absmax == 0.f ? 1.f : r) : fmaxf(r, 1e-10f);
    out.s = s;
    out.inv = block_recip(s);
    out.stored = __float_as_uint(s);
  } else if (scale == BSMM_SCALE_UE8M0) {
    // Smallest power of two not below r: 2^ceil(log2 r), exponent in [-127,127].
    int e;
    if (absmax == 0.f) {
      e = 0;
    } else if (r == 0.f) {
      e = -127;
    } else {
      const uint32_t bits = __float_as_uint(r);
      const int E = static_cast<int>((bits >> 23) & 0xFFu);
      const uint32_t man = bits & 0x7FFFFFu;
      if (E == 0)
        e = -149 + (32 - __clz(static_cast<int>(man - 1u)));  // subnormal r = man * 2^-149
      else
        e = E - 127 + (man != 0u ? 1 : 0);
      e = max(-127, min(127, e));
    }
    out.stored = static_cast<uint32_t>(e + 127);
    out.s = e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(0x00400000u);
    // 2^-e is exact for e in [-127, 127]; x * 2^-e rounds the same exact
    // value that x / 2^e does, so multiplying is the IEEE quotient.
    out.inv = -e >= -126 ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23) : __uint_as_float(0x00400000u);
  } else {
    // UE4M3: nearest E4M3 value of r; zero block -> 1.0; a scale that rounds
    // to zero -> the smallest subnormal.
    uint32_t b;
    if (absmax == 0.f) {
      b = 0x38u;
    } else {
      b = cvt_e4m3x2(r, 0.f) & 0xFFu;
      if (b == 0u) b = 1u;
    }
    out.stored = b;
    out.s = ue4m3_value(b);
    out.inv = block_recip(out.s);
  }
  return out;
}

__device__ __forceinline__ float clampq(float q, float qmax) { return fminf(fmaxf(q, -qmax), qmax); }

__device__ __forceinline__ uint32_t int8_code(float q) {
  return static_cast<uint32_t>(__float2int_rn(clampq(q, 127.f))) & 0xFFu;
}

// x / s, correctly rounded: a multiply by the exact reciprocal when s is a
// power of two (POW2), else quotient.cuh's corrected product, or a division
// for divisors outside its range.
template <bool POW2>
__device__ __forceinline__ float quot(float x, const Scale& sc) {
  if constexpr (POW2)
    return x * sc.inv;
  else
    return sc.inv != 0.f ? quot_rn(x, sc.s, sc.inv) : __fdiv_rn(x, sc.s);
}

template <bool POW2>
__device__ __forceinline__ float2 quot2(float x0, float x1, const Scale& sc) {
  if constexpr (POW2)
    return make_float2(x0 * sc.inv, x1 * sc.inv);
  else if (sc.inv != 0.f)
    return quot2_rn(make_float2(x0, x1), sc.s, sc.inv);
  else
    return make_float2(__fdiv_rn(x0, sc.s), __fdiv_rn(x1, sc.s));
}

__device__ __forceinline__ uint32_t pack4(float q0, float q1, float q2, float q3, int code) {
  // The float conversions saturate (satfinite): for finite quotients that is
  // clamp(q, +-qmax) followed by nearest-even rounding.  INT8 clamps.
  switch (code) {
    case BSMM_E4M3: return cvt_e4m3x2(q0, q1) | (cvt_e4m3x2(q2, q3) << 16);
    case BSMM_E5M2: return cvt_e5m2x2(q0, q1) | (cvt_e5m2x2(q2, q3) << 16);
    case BSMM_E2M1: return cvt_e2m1x2(q0, q1) | (cvt_e2m1x2(q2, q3) << 8);
    default: return int8_code(q0) | (int8_code(q1) << 8) | (int8_code(q2) << 16) | (int8_code(q3) << 24);
  }
}

// Codes of four consecutive elements: 4 bytes (E4M3/E5M2/INT8, element 0 in
// the low byte) or 2 bytes (E2M1, element 0 in the low nibble).
template <bool POW2>
__device__ __forceinline__ uint32_t encode4(float x0, float x1, float x2, float x3, const Scale& sc, int code) {
  const float2 q01 = quot2<POW2>(x0, x1, sc), q23 = quot2<POW2>(x2, x3, sc);
  return pack4(q01.x, q01.y, q23.x, q23.y, code);
}

// The same where the block's quotients take the corrected product (POW2, or
// sc.inv != 0), with no per-element test.
template <bool POW2>
__device__ __forceinline__ uint32_t encode4_fast(float x0, float x1, float x2, float x3, const Scale& sc, int code) {
  if constexpr (POW2) {
    return pack4(x0 * sc.inv, x1 * sc.inv, x2 * sc.inv, x3 * sc.inv, code);
  } else {
    const float2 q01 = quot2_rn(make_float2(x0, x1), sc.s, sc.inv), q23 = quot2_rn(make_float2(x2, x3), sc.s, sc.inv);
    return pack4(q01.x, q01.y, q23.x, q23.y, code);
  }
}

// One code (8-bit formats) or one nibble (E2M1).
template <bool POW2>
__device__ __forceinline__ uint32_t encode1(float x, const Scale& sc, int code) {
  const float q = clampq(quot<POW2>(x, sc), qmax_of(code));
  switch (code) {
    case BSMM_E4M3: return cvt_e4m3x2(q, 0.f) & 0xFFu;
    case BSMM_E5M2: return cvt_e5m2x2(q, 0.f) & 0xFFu;
    case BSMM_E2M1: return cvt_e2m1x2(q, 0.f) & 0xFu;
    default: return int8_code(q);
  }
}

__device__ __forceinline__ void store_scale(void* scales, int64_t idx, int scale, uint32_t stored) {
  if (scale == BSMM_SCALE_F32)
    reinterpret_cast<uint32_t*>(scales)[idx] = stored;
  else
    reinterpret_cast<uint8_t*>(scales)[idx] = static_cast<uint8_t>(stored);
}

template <typename In>
__device__ __forceinline__ float load1(const void* x, int64_t idx) {
  if constexpr (sizeof(In) == 4) {
    return __ldg(reinterpret_cast<const float*>(x) + idx);
  } else {
    const uint16_t b = __ldg(reinterpret_cast<const unsigned short*>(x) + idx);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
}

// 16-byte vector of 4 (binary32) or 8 (bfloat16) elements, streamed.
template <typename In>
__device__ __forceinline__ void load_vec(const void* p, float (&v)[16 / sizeof(In)]) {
  const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
  if constexpr (sizeof(In) == 4) {
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
  } else {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

// ---------------------------------------------------------------------------
// 1 x bc blocks along rows
// ---------------------------------------------------------------------------
// A thread owns a slice of 16 consecutive elements of one block; G = bc / 16
// lanes (1..8) share a block and combine their maxima by xor-shuffle.  Each
// thread handles two slices per trip (32 elements in flight).
constexpr int kSlice = 16;

template <typename In>
__device__ __forceinline__ void load_slice(const In* p, float (&v)[kSlice]) {
  constexpr int VEC = 16 / sizeof(In);
#pragma unroll
  for (int i = 0; i < kSlice / VEC; ++i) {
    float t[VEC];
    load_vec<In>(p + i * VEC, t);
#pragma unroll
    for (int k = 0; k < VEC; ++k) v[i * VEC + k] = t[k];
  }
}

template <typename In, bool POW2>
__global__ void __launch_bounds__(256) quant_rows(QP p) {
  const int G = p.bc / kSlice;                 // lanes per block: 1, 2, 4 or 8
  const int64_t spr = p.cols / kSlice;         // slices per row
  const int64_t total = p.rows * spr;
  const int lane = threadIdx.x & 31;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const bool fp4 = p.code == BSMM_E2M1;
  // dense: x and codes contiguous; sdense: row-major scales without padding
  const bool dense = p.ld_x == p.cols && p.ld_codes == p.cols;
  const bool sdense = dense && !p.sf_atoms && p.ld_scales * p.bc == p.cols;
  const int g_shift = __ffs(G) - 1;
  const bool spr_pow2 = (spr & (spr - 1)) == 0;
  const int spr_shift = __ffsll(spr) - 1;
  const In* x = reinterpret_cast<const In*>(p.x);
  uint8_t* out = reinterpret_cast<uint8_t*>(p.codes);
  // b0 is warp-uniform, so every shuffle sees the whole warp
  for (int64_t b0 = tid - lane; b0 < total; b0 += 2 * nth) {
    float v[2][kSlice];
    int64_t si[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      si[u] = b0 + u * nth + lane;
      if (si[u] < total) {
        int64_t off = si[u] * kSlice;
        if (!dense) {
          const int64_t r = spr_pow2 ? si[u] >> spr_shift : si[u] / spr;
          off = r * p.ld_x + (si[u] - r * spr) * kSlice;
        }
        load_slice<In>(x + off, v[u]);
      } else {
#pragma unroll
        for (int i = 0; i < kSlice; ++i) v[u][i] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < kSlice; ++i) m = fmaxf(m, fabsf(v[u][i]));
      for (int o = G >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (si[u] >= total) continue;
      const Scale sc = make_scale(m, p.code, p.scale);
      int64_t e = si[u] * kSlice, sidx = si[u] >> g_shift;
      if (!sdense) {
        const int64_t r = spr_pow2 ? si[u] >> spr_shift : si[u] / spr;
        const int64_t c = si[u] - r * spr;
        if (!dense) e = r * p.ld_codes + c * kSlice;
        sidx = scale_index(p, r, c >> g_shift);  // (c * kSlice) / bc
      }
      if ((lane & (G - 1)) == 0) store_scale(p.scales, sidx, p.scale, sc.stored);
      uint32_t w[4];
#pragma unroll
      for (int g = 0; g < 4; ++g)
        w[g] = encode4<POW2>(v[u][4 * g], v[u][4 * g + 1], v[u][4 * g + 2], v[u][4 * g + 3], sc, p.code);
      if (fp4)
        *reinterpret_cast<uint2*>(out + e / 2) = make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
      else
        *reinterpret_cast<uint4*>(out + e) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// ---------------------------------------------------------------------------
// br x 1 blocks down the columns, 128-row x 64-column tiles
// ---------------------------------------------------------------------------
constexpr int kColTileR = 128, kColTileC = 64;

template <typename In, bool POW2>
// Persistent: CTA b takes tiles b, b + gridDim.x, ... (column tiles fastest);
// on the vector path the next tile's raw data is loaded into registers while
// the current one is reduced and encoded.
// The tile keeps the input type: FP32 as words (65 per row), bf16 as
// packed pairs (33 words per row).  Either stride leaves the row-wise vector
// stores and the column reads free of bank conflicts, and bf16 tiles take
// half the shared memory and traffic.
__global__ void __launch_bounds__(256, 3) quant_cols(QP p, int vec_ok, int tiles_c, int64_t n_tiles) {
  constexpr int kRowWords = sizeof(In) == 4 ? kColTileC + 1 : kColTileC / 2 + 1;
  __shared__ __align__(16) uint32_t tile_w[kColTileR * kRowWords];
  __shared__ float pmax[4][kColTileC];
  auto tile_val = [&](int r, int c) -> float {
    if constexpr (sizeof(In) == 4) {
      return __uint_as_float(tile_w[r * kRowWords + c]);
    } else {
      const uint32_t wv = tile_w[r * kRowWords + (c >> 1)];
      return __uint_as_float((c & 1) ? (wv & 0xFFFF0000u) : (wv << 16));
    }
  };
  const int t = threadIdx.x;
  const In* x = reinterpret_cast<const In*>(p.x);
  constexpr int VEC = 16 / sizeof(In);
  constexpr int VPR = kColTileC / VEC;        // vectors per tile row
  constexpr int NV = kColTileR * VPR / 256;   // vectors per thread
  uint4 raw[NV];
  auto fetch = [&](int64_t tt) {  // all loads in flight before any use
    const int64_t fr0 = (tt / tiles_c) * kColTileR, fc0 = (tt % tiles_c) * kColTileC;
    const int fnr = static_cast<int>(p.rows - fr0 < kColTileR ? p.rows - fr0 : kColTileR);
    const int fnc = static_cast<int>(p.cols - fc0 < kColTileC ? p.cols - fc0 : kColTileC);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int i = t + 256 * j;
      const int rr = i / VPR, cv = i % VPR;
      raw[j] = (rr < fnr && cv * VEC < fnc)
                   ? __ldcs(reinterpret_cast<const uint4*>(x + (fr0 + rr) * p.ld_x + fc0 + cv * VEC))
                   : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if (vec_ok && blockIdx.x < n_tiles) fetch(blockIdx.x);
  for (int64_t tt = blockIdx.x; tt < n_tiles; tt += gridDim.x) {
    const int64_t r0 = (tt / tiles_c) * kColTileR;
    const int64_t c0 = (tt % tiles_c) * kColTileC;
    const int nr = static_cast<int>(p.rows - r0 < kColTileR ? p.rows - r0 : kColTileR);
    const int nc = static_cast<int>(p.cols - c0 < kColTileC ? p.cols - c0 : kColTileC);
    __syncthreads();  // every thread is done with the previous tile's shared data
    // Stage the tile (coalesced along columns).
    if (vec_ok) {
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int i = t + 256 * j;
        const int rr = i / VPR, cv = i % VPR;
        const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) tile_w[rr * kRowWords + cv * 4 + k] = w[k];  // 4 floats or 8 bf16
      }
    } else {
      for (int i = t; i < kColTileR * kColTileC; i += 256) {
        const int rr = i / kColTileC, cc = i % kColTileC;
        const float v = (rr < nr && cc < nc) ? load1<In>(x, (r0 + rr) * p.ld_x + c0 + cc) : 0.f;
        if constexpr (sizeof(In) == 4)
          tile_w[rr * kRowWords + cc] = __float_as_uint(v);
        else  // v is a bf16 value: its top 16 bits are the code
          reinterpret_cast<uint16_t*>(tile_w)[rr * 2 * kRowWords + cc] = static_cast<uint16_t>(__float_as_uint(v) >> 16);
      }
    }
    __syncthreads();
    if (vec_ok && tt + gridDim.x < n_tiles) fetch(tt + gridDim.x);
    // Thread (col, part) owns rows 32*part .. 32*part+31 of one column, held in
    // registers from here on.
    const int col = t % kColTileC, part = t / kColTileC;
    const int rbase = part * 32;
    const int br = p.br;
    float v[32];  // read once from shared memory
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = tile_val(rbase + i, col);
    float m0 = 0.f, m1 = 0.f;  // maxima of the two 16-row halves
#pragma unroll
    for (int i = 0; i < 16; ++i) m0 = fmaxf(m0, fabsf(v[i]));
#pragma unroll
    for (int i = 16; i < 32; ++i) m1 = fmaxf(m1, fabsf(v[i]));
    if (br > 32) {
      pmax[part][col] = fmaxf(m0, m1);
      __syncthreads();
    }
    const bool active = rbase < nr && col < nc;
    // Scales of the (one or two) blocks this thread's 32 rows belong to.
    float amax_a, amax_b;
    if (br == 16) {
      amax_a = m0;
      amax_b = m1;
    } else if (br == 32) {
      amax_a = amax_b = fmaxf(m0, m1);
    } else if (br == 64) {
      const int pp = part & ~1;
      amax_a = amax_b = fmaxf(pmax[pp][col], pmax[pp + 1][col]);
    } else {
      amax_a = amax_b = fmaxf(fmaxf(pmax[0][col], pmax[1][col]), fmaxf(pmax[2][col], pmax[3][col]));
    }
    const Scale sa = make_scale(amax_a, p.code, p.scale);
    const Scale sb = (br == 16) ? make_scale(amax_b, p.code, p.scale) : sa;
    if (active) {
      const int64_t gc = c0 + col;
      const int64_t blk0 = (r0 + rbase) / br;
      const bool writes_a = (rbase % br) == 0;
      if (p.transpose) {
        if (writes_a) store_scale(p.scales, scale_index(p, gc, blk0), p.scale, sa.stored);
        if (br == 16) store_scale(p.scales, scale_index(p, gc, blk0 + 1), p.scale, sb.stored);
      } else {
        if (writes_a) store_scale(p.scales, blk0 * p.ld_scales + gc, p.scale, sa.stored);
        if (br == 16) store_scale(p.scales, (blk0 + 1) * p.ld_scales + gc, p.scale, sb.stored);
      }
    }
    uint8_t* out = reinterpret_cast<uint8_t*>(p.codes);
    if (p.transpose) {
      if (!active) continue;
      // 32 consecutive output elements of row `gc` of the transposed array.
      uint32_t w[8];
#pragma unroll
      for (int g = 0; g < 8; ++g)
        w[g] = encode4<POW2>(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3], g < 4 ? sa : sb, p.code);
      const int64_t e = (c0 + col) * p.ld_codes + r0 + rbase;
      const bool full32 = rbase + 32 <= nr;  // else only the first 16 rows exist
      if (p.code == BSMM_E2M1) {
        if (full32)
          *reinterpret_cast<uint4*>(out + e / 2) =
              make_uint4(w[0] | (w[1] << 16), w[2] | (w[3] << 16), w[4] | (w[5] << 16), w[6] | (w[7] << 16));
        else
          *reinterpret_cast<uint2*>(out + e / 2) = make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
      } else {
        *reinterpret_cast<uint4*>(out + e) = make_uint4(w[0], w[1], w[2], w[3]);
        if (full32) *reinterpret_cast<uint4*>(out + e + 16) = make_uint4(w[4], w[5], w[6], w[7]);
      }
    } else {
      // Row-major codes: lanes hold consecutive columns.
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint32_t cval = encode1<POW2>(v[i], i < 16 ? sa : sb, p.code);
        const int64_t e = (r0 + rbase + i) * p.ld_codes + c0 + col;
        const bool ok = active && rbase + i < nr;
        if (p.code == BSMM_E2M1) {
          const uint32_t hi = __shfl_down_sync(0xffffffffu, cval, 1);
          if (ok && (col & 1) == 0) out[e / 2] = static_cast<uint8_t>(cval | (hi << 4));
        } else if (ok) {
          out[e] = static_cast<uint8_t>(cval);
        }
      }
    }
  }  // tiles
}

// ---------------------------------------------------------------------------
// br x 1 blocks down the columns of a bf16 array, transposed output, tiles
// streamed by TMA
// ---------------------------------------------------------------------------
// The same 128-row x 64-column tiles and per-tile arithmetic as quant_cols,
// but the tiles reach shared memory through a ring of kColStages TMA loads
// (16 KB each), so the bytes in flight no longer depend on registers, and the
// output goes out through shared memory as whole 128-byte lines (one-byte
// scale types: UE8M0, UE4M3).
// Persistent CTAs take tiles b, b + gridDim.x, ...; thread 0 refills a stage
// as soon as every thread has read it.  Waits are bounded: the CTA agrees on
// a failure before any barrier, and waits for its own copies in flight
// before it exits.
constexpr int kColStages = 3;
constexpr int kColTileBytes = kColTileR * kColTileC * 2;  // 16 KB of bf16
constexpr int kSiteQuantTile = 21, kSiteQuantDrain = 22;

template <bool POW2>
__global__ void __launch_bounds__(256) quant_cols_tma(const __grid_constant__ CUtensorMap tm, QP p, int tiles_c,
                                                      int64_t n_tiles, int* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t qsm_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsm_raw) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kColStages * kColTileBytes);
  __shared__ float pmax[4][kColTileC];
  // the tile's output staged for whole-line stores: 64 transposed rows of
  // 128 codes (16-byte chunks swizzled by row) and their 128/br scale bytes
  __shared__ __align__(16) uint8_t ostg[kColTileC * kColTileR];
  __shared__ __align__(16) uint8_t sstg[kColTileC][8];
  __shared__ int abort_flag;
  int never_abort_storage = 0;
  volatile int* never_abort = &never_abort_storage;
  const int t = threadIdx.x;
  if (t == 0) {
    for (int st = 0; st < kColStages; ++st) mbar_init(&full[st], 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int64_t my_n = (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x;
  auto issue = [&](int64_t i) {  // this CTA's i-th tile into stage i % kColStages
    const int64_t tt = blockIdx.x + i * gridDim.x;
    const int st = static_cast<int>(i % kColStages);
    mbar_arrive_expect_tx(&full[st], kColTileBytes);
    tma_load_3d(ring + st * kColTileBytes, &tm, &full[st], static_cast<int>((tt % tiles_c) * kColTileC),
                static_cast<int>((tt / tiles_c) * kColTileR), 0);
  };
  int64_t issued = 0;
  if (t == 0)
    for (; issued < my_n && issued < kColStages; ++issued) issue(issued);
  const int col = t % kColTileC, part = t / kColTileC;
  const int rbase = part * 32;
  const int br = p.br;
  int64_t i = 0;
  for (; i < my_n; ++i) {
    const int st = static_cast<int>(i % kColStages);
    const bool ok = mbar_wait(&full[st], static_cast<uint32_t>(i / kColStages) & 1u, timeout_ns, &abort_flag,
                              status, kSiteQuantTile);
    float v[32];  // this thread's column, rows rbase .. rbase + 31
    if (ok) {
      const __nv_bfloat16* tile = reinterpret_cast<const __nv_bfloat16*>(ring + st * kColTileBytes);
#pragma unroll
      for (int r = 0; r < 32; ++r) v[r] = __bfloat162float(tile[(rbase + r) * kColTileC + col]);
    }
    if (__syncthreads_or(!ok)) break;  // every thread has read stage st (or the CTA gives up together)
    if (t == 0 && issued < my_n) issue(issued++);
    const int64_t tt = blockIdx.x + i * gridDim.x;
    const int64_t r0 = (tt / tiles_c) * kColTileR;
    const int64_t c0 = (tt % tiles_c) * kColTileC;
    const int nr = static_cast<int>(p.rows - r0 < kColTileR ? p.rows - r0 : kColTileR);
    const int nc = static_cast<int>(p.cols - c0 < kColTileC ? p.cols - c0 : kColTileC);
    float m0 = 0.f, m1 = 0.f;  // maxima of the two 16-row halves (rows past the array read as zero)
#pragma unroll
    for (int r = 0; r < 16; ++r) m0 = fmaxf(m0, fabsf(v[r]));
#pragma unroll
    for (int r = 16; r < 32; ++r) m1 = fmaxf(m1, fabsf(v[r]));
    if (br > 32) {
      pmax[part][col] = fmaxf(m0, m1);
      __syncthreads();
    }
    float amax_a, amax_b;
    if (br == 16) {
      amax_a = m0;
      amax_b = m1;
    } else if (br == 32) {
      amax_a = amax_b = fmaxf(m0, m1);
    } else if (br == 64) {
      const int pp = part & ~1;
      amax_a = amax_b = fmaxf(pmax[pp][col], pmax[pp + 1][col]);
    } else {
      amax_a = amax_b = fmaxf(fmaxf(pmax[0][col], pmax[1][col]), fmaxf(pmax[2][col], pmax[3][col]));
    }
    if (br > 32) __syncthreads();  // pmax is rewritten by the next tile
    const Scale sa = make_scale(amax_a, p.code, p.scale);
    const Scale sb = (br == 16) ? make_scale(amax_b, p.code, p.scale) : sa;
    {
      uint32_t w[8];
#pragma unroll
      for (int g = 0; g < 8; ++g)
        w[g] = encode4<POW2>(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3], g < 4 ? sa : sb, p.code);
      // row `col` of the staged output, chunks 2*part and 2*part+1 (XOR-swizzled)
      uint8_t* row = ostg + col * kColTileR;
      *reinterpret_cast<uint4*>(row + (((2 * part) ^ (col & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(row + (((2 * part + 1) ^ (col & 7)) * 16)) = make_uint4(w[4], w[5], w[6], w[7]);
      if ((rbase % br) == 0) sstg[col][rbase / br] = static_cast<uint8_t>(sa.stored);
      if (br == 16) sstg[col][rbase / 16 + 1] = static_cast<uint8_t>(sb.stored);
    }
    __syncthreads();
    // whole-line stores: each instruction writes 4 output rows x 128 bytes
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int idx = t + 256 * k;
      const int c = idx >> 3, ch = idx & 7;
      if (c < nc && ch * 16 < nr)
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.codes) + (c0 + c) * p.ld_codes + r0 + ch * 16) =
            *reinterpret_cast<const uint4*>(ostg + c * kColTileR + ((ch ^ (c & 7)) * 16));
    }
    if (t < nc) {  // this column's scale bytes for the tile's rows
      const int nblk = (nr + br - 1) / br;
      // (atom layout: r0 / br is a multiple of 4, so the tile's blocks are the
      // consecutive bytes of one word)
      uint8_t* dst = reinterpret_cast<uint8_t*>(p.scales) + scale_index(p, c0 + t, r0 / br);
      if (nblk == 4 && (reinterpret_cast<uintptr_t>(dst) & 3) == 0)
        *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(&sstg[t][0]);
      else
        for (int k = 0; k < nblk; ++k) dst[k] = sstg[t][k];
    }
  }
  // copies this CTA started and did not consume (only after giving up)
  if (t == 0)
    for (int64_t j = i; j < issued; ++j)
      mbar_wait(&full[j % kColStages], static_cast<uint32_t>(j / kColStages) & 1u, timeout_ns, never_abort, status,
                kSiteQuantDrain);
}

// The same for 32-row blocks (MXFP8) with tiles of 128 x 128: a thread owns
// two adjacent columns of one 32-row block, read as bf16 pairs (half the
// shared-memory loads of one column per thread, which bound the kernel above).
constexpr int kCol2C = 128;
constexpr int kCol2TileBytes = kColTileR * kCol2C * 2;  // 32 KB of bf16

// DUAL: the same tiles are also quantized along their rows (1 x 32 blocks,
// untransposed output described by p2: codes, scales and their layout), so
// an array both GEMMs of the backward read along different axes (dY) is
// read from HBM once.  PAIR: p2 (read through tm2, tiles_c2 tiles a row) is
// a second array quantized like p, its tiles numbered after p's n_a: two
// arrays in one launch pay its start and its last wave once.  CODE (E4M3 or
// E5M2) is fixed at compile time, and block maxima are taken on the bf16
// pairs as loaded (packed max of magnitudes): the kernel is bound by
// instruction issue, not by HBM.
template <bool POW2, bool DUAL, bool PAIR, int CODE>
__global__ void __launch_bounds__(256, 2)
    quant_cols_tma2(const __grid_constant__ CUtensorMap tm, const __grid_constant__ QP p, int tiles_c, int64_t n_tiles,
                    int* status, uint64_t timeout_ns, const __grid_constant__ QP p2,
                    const __grid_constant__ CUtensorMap tm2, int tiles_c2, int64_t n_a) {
  extern __shared__ uint8_t qsm_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsm_raw) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kColStages * kCol2TileBytes);
  // 128 transposed output rows of 128 codes (16-byte chunks swizzled by row)
  // and their four scale bytes
  __shared__ __align__(16) uint8_t ostg[kCol2C * kColTileR];
  __shared__ __align__(16) uint8_t sstg[kCol2C][4];
  __shared__ int abort_flag;
  int never_abort_storage = 0;
  volatile int* never_abort = &never_abort_storage;
  const int t = threadIdx.x;
  if (t == 0) {
    for (int st = 0; st < kColStages; ++st) mbar_init(&full[st], 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int64_t my_n = (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x;
  auto issue = [&](int64_t i) {  // this CTA's i-th tile into stage i % kColStages
    int64_t tt = blockIdx.x + i * gridDim.x;
    const bool b2 = PAIR && tt >= n_a;
    if (b2) tt -= n_a;
    const int tc = b2 ? tiles_c2 : tiles_c;
    const int st = static_cast<int>(i % kColStages);
    mbar_arrive_expect_tx(&full[st], kCol2TileBytes);
    tma_load_3d(ring + st * kCol2TileBytes, b2 ? &tm2 : &tm, &full[st], static_cast<int>((tt % tc) * kCol2C),
                static_cast<int>((tt / tc) * kColTileR), 0);
  };
  int64_t issued = 0;
  if (t == 0)
    for (; issued < my_n && issued < kColStages; ++issued) issue(issued);
  const int cp = t & 63, part = t >> 6;  // columns 2cp, 2cp+1; rows 32 part .. +31 (one block)
  int64_t i = 0;
  for (; i < my_n; ++i) {
    const int st = static_cast<int>(i % kColStages);
    const bool ok = mbar_wait(&full[st], static_cast<uint32_t>(i / kColStages) & 1u, timeout_ns, &abort_flag,
                              status, kSiteQuantTile);
    uint32_t w[32];  // bf16 pairs: rows 32 part + r, columns 2cp (low half) and 2cp+1 (high half)
    int64_t tt = blockIdx.x + i * gridDim.x;
    const bool b2 = PAIR && tt >= n_a;
    if (b2) tt -= n_a;
    const QP& q = b2 ? p2 : p;  // the array this tile belongs to
    const int tc = b2 ? tiles_c2 : tiles_c;
    const int64_t r0 = (tt / tc) * kColTileR;
    const int64_t c0 = (tt % tc) * kCol2C;
    const int nr = static_cast<int>(q.rows - r0 < kColTileR ? q.rows - r0 : kColTileR);
    const int nc = static_cast<int>(q.cols - c0 < kCol2C ? q.cols - c0 : kCol2C);
    if (ok) {
      const uint32_t* tile = reinterpret_cast<const uint32_t*>(ring + st * kCol2TileBytes);
      if constexpr (DUAL) {
        // along the rows: thread t takes 32-column block t % 4 of tile rows
        // t / 4 and t / 4 + 64, so that four lanes cover a row and every code
        // store writes whole 128-byte lines.  Rows are 256 bytes apart (the
        // same banks), so each lane reads its block's four 16-byte chunks in
        // the order rotated by rot: the eight lanes of a load phase (two rows
        // x four blocks) then hit eight different bank groups.
        const int blk = t & 3;
        const int64_t gcol = c0 + 32 * blk;
        constexpr int kScaleType = POW2 ? BSMM_SCALE_UE8M0 : BSMM_SCALE_UE4M3;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          const int rr = (t >> 2) + 64 * pass;
          const int rot = 2 * (rr & 1) + (blk >> 1);
          const uint4* src = reinterpret_cast<const uint4*>(tile + rr * (kCol2C / 2) + 16 * blk);
          uint4 q[4];  // q[j] is the block's 16-byte chunk (j + rot) % 4
#pragma unroll
          for (int j = 0; j < 4; ++j) q[j] = src[(j + rot) & 3];
          uint32_t m = 0u;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            m = bf16x2_max_abs(m, bf16x2_max_abs(bf16x2_max_abs(q[j].x, q[j].y), bf16x2_max_abs(q[j].z, q[j].w)));
          const Scale sc = make_scale(fmaxf(bf16_lo_abs(m), bf16_hi_abs(m)), CODE, kScaleType);
          uint2 v[4];  // codes of chunk (j + rot) % 4
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v[j].x = encode4<POW2>(__uint_as_float(q[j].x << 16), __uint_as_float(q[j].x & 0xFFFF0000u),
                                   __uint_as_float(q[j].y << 16), __uint_as_float(q[j].y & 0xFFFF0000u), sc, CODE);
            v[j].y = encode4<POW2>(__uint_as_float(q[j].z << 16), __uint_as_float(q[j].z & 0xFFFF0000u),
                                   __uint_as_float(q[j].w << 16), __uint_as_float(q[j].w & 0xFFFF0000u), sc, CODE);
          }
          // back into column order: rotate by rot (two conditional steps)
          if (rot & 1) {
            const uint2 l = v[3];
            v[3] = v[2];
            v[2] = v[1];
            v[1] = v[0];
            v[0] = l;
          }
          if (rot & 2) {
            const uint2 a0 = v[0], a1 = v[1];
            v[0] = v[2];
            v[1] = v[3];
            v[2] = a0;
            v[3] = a1;
          }
          const int64_t grow = r0 + rr;
          if (grow < p.rows && gcol < p.cols) {  // cols % 32 == 0: a block is all in or all out
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p2.codes) + grow * p2.ld_codes + gcol);
            dst[0] = make_uint4(v[0].x, v[0].y, v[1].x, v[1].y);
            dst[1] = make_uint4(v[2].x, v[2].y, v[3].x, v[3].y);
            reinterpret_cast<uint8_t*>(p2.scales)[scale_index(p2, grow, gcol / 32)] = static_cast<uint8_t>(sc.stored);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 32; ++r) w[r] = tile[(32 * part + r) * (kCol2C / 2) + cp];
    }
    if (__syncthreads_or(!ok)) break;  // every thread has read stage st (or the CTA gives up together)
    if (t == 0 && issued < my_n) issue(issued++);
    uint32_t mc = 0u;  // packed maxima of the two columns; rows past the array read as zero
#pragma unroll
    for (int r = 0; r < 32; ++r) mc = bf16x2_max_abs(mc, w[r]);
    constexpr int kColScale = POW2 ? BSMM_SCALE_UE8M0 : BSMM_SCALE_UE4M3;
    const Scale s0 = make_scale(bf16_lo_abs(mc), CODE, kColScale);
    const Scale s1 = make_scale(bf16_hi_abs(mc), CODE, kColScale);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int col = 2 * cp + h;
      uint32_t q[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        float f[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          f[j] = __uint_as_float(h ? (w[4 * g + j] & 0xFFFF0000u) : (w[4 * g + j] << 16));
        q[g] = encode4<POW2>(f[0], f[1], f[2], f[3], h ? s1 : s0, CODE);
      }
      uint8_t* row = ostg + col * kColTileR;
      *reinterpret_cast<uint4*>(row + (((2 * part) ^ (col & 7)) * 16)) = make_uint4(q[0], q[1], q[2], q[3]);
      *reinterpret_cast<uint4*>(row + (((2 * part + 1) ^ (col & 7)) * 16)) = make_uint4(q[4], q[5], q[6], q[7]);
      sstg[col][part] = static_cast<uint8_t>((h ? s1 : s0).stored);
    }
    __syncthreads();
    // whole-line stores: each instruction writes 4 output rows x 128 bytes
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = t + 256 * k;
      const int c = idx >> 3, ch = idx & 7;
      if (c < nc && ch * 16 < nr)
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(q.codes) + (c0 + c) * q.ld_codes + r0 + ch * 16) =
            *reinterpret_cast<const uint4*>(ostg + c * kColTileR + ((ch ^ (c & 7)) * 16));
    }
    if (t < nc) {  // this column's scale bytes for the tile's rows (atoms: one word)
      const int nblk = (nr + 31) / 32;
      uint8_t* dst = reinterpret_cast<uint8_t*>(q.scales) + scale_index(q, c0 + t, r0 / 32);
      if (nblk == 4 && (reinterpret_cast<uintptr_t>(dst) & 3) == 0)
        *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(&sstg[t][0]);
      else
        for (int k = 0; k < nblk; ++k) dst[k] = sstg[t][k];
    }
    __syncthreads();  // ostg and sstg are rewritten by the next tile
  }
  // copies this CTA started and did not consume (only after giving up)
  if (t == 0)
    for (int64_t j = i; j < issued; ++j)
      mbar_wait(&full[j % kColStages], static_cast<uint32_t>(j / kColStages) & 1u, timeout_ns, never_abort, status,
                kSiteQuantDrain);
}

// ---------------------------------------------------------------------------
// 128 x 128 blocks
// ---------------------------------------------------------------------------
// 512 threads: lane l of warp w owns columns 4l .. 4l+3 of rows w, w+16, ...,
// w+112, so every load instruction of a warp reads one whole tile row (512
// bytes of FP32, 256 of bf16) and every store writes that row's 128 codes.
// Sixteen warps of 32 values each (rather than eight of 64): two CTAs on an
// SM, so one CTA's loads overlap another's encoding.  One CTA, tile (ty, tx).
template <typename In, bool POW2>
__device__ __forceinline__ void quant_tile_body(const QP& p, int64_t ty, int64_t tx) {
  __shared__ float wmax[16];
  __shared__ Scale tile_sc;
  const int64_t r0 = ty * 128, c0 = tx * 128;
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const In* x = reinterpret_cast<const In*>(p.x) + (r0 + warp) * p.ld_x + c0 + 4 * lane;
  float v[32];  // v[4k + j]: row warp + 16k, column 4 lane + j
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const In* src = x + static_cast<int64_t>(16 * k) * p.ld_x;
    if constexpr (sizeof(In) == 4) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(src));
      v[4 * k] = q.x;
      v[4 * k + 1] = q.y;
      v[4 * k + 2] = q.z;
      v[4 * k + 3] = q.w;
    } else {
      const uint2 q = __ldg(reinterpret_cast<const uint2*>(src));
      v[4 * k] = __uint_as_float(q.x << 16);
      v[4 * k + 1] = __uint_as_float(q.x & 0xFFFF0000u);
      v[4 * k + 2] = __uint_as_float(q.y << 16);
      v[4 * k + 3] = __uint_as_float(q.y & 0xFFFF0000u);
    }
  }
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(v[i]));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  // warp 0 takes the tile's maximum and scale (the divisions once per tile)
  if (warp == 0) {
    m = lane < 16 ? wmax[lane] : 0.f;
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) {
      const Scale s0 = make_scale(m, p.code, p.scale);
      tile_sc = s0;
      store_scale(p.scales, ty * p.ld_scales + tx, p.scale, s0.stored);
    }
  }
  __syncthreads();
  const Scale sc = tile_sc;
  uint8_t* out = reinterpret_cast<uint8_t*>(p.codes);
  auto put = [&](int k, uint32_t w) {
    const int64_t e = (r0 + warp + 16 * k) * p.ld_codes + c0 + 4 * lane;
    if (p.code == BSMM_E2M1)
      *reinterpret_cast<uint16_t*>(out + e / 2) = static_cast<uint16_t>(w);
    else
      *reinterpret_cast<uint32_t*>(out + e) = w;
  };
  if (POW2 || sc.inv != 0.f) {  // the whole tile takes the same path
#pragma unroll
    for (int k = 0; k < 8; ++k) put(k, encode4_fast<POW2>(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3], sc, p.code));
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) put(k, encode4<POW2>(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3], sc, p.code));
  }
}

template <typename In, bool POW2>
__global__ void __launch_bounds__(512) quant_tile(QP p) {
  quant_tile_body<In, POW2>(p, blockIdx.y, blockIdx.x);
}

// Several 128 x 128 quantizations in one launch: CTA t takes the tile of job
// j with first[j] <= t < first[j + 1], row-major over that job's tiles.
constexpr int kTileBatchMax = 16;
struct QTileBatch {
  QP p[kTileBatchMax];
  int64_t first[kTileBatchMax + 1];
  int64_t tiles_c[kTileBatchMax];
  int n;
};

template <typename In, bool POW2>
__global__ void __launch_bounds__(512) quant_tile_batch(const __grid_constant__ QTileBatch b) {
  const int64_t t = blockIdx.x;
  int j = 0;
  while (j + 1 < b.n && t >= b.first[j + 1]) ++j;
  const int64_t local = t - b.first[j];
  quant_tile_body<In, POW2>(b.p[j], local / b.tiles_c[j], local % b.tiles_c[j]);
}

// ---------------------------------------------------------------------------
// Whole-row and whole-column blocks, and the generic fallback
// ---------------------------------------------------------------------------
template <typename In, bool POW2>
__global__ void __launch_bounds__(256) quant_wrow(QP p) {
  __shared__ float wmax[8];
  const int64_t r = blockIdx.x;
  const int t = threadIdx.x;
  const In* x = reinterpret_cast<const In*>(p.x);
  float m = 0.f;
  for (int64_t c = t; c < p.cols; c += 256) m = fmaxf(m, fabsf(load1<In>(x, r * p.ld_x + c)));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((t & 31) == 0) wmax[t >> 5] = m;
  __syncthreads();
  m = wmax[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, wmax[i]);
  const Scale sc = make_scale(m, p.code, p.scale);
  if (t == 0) store_scale(p.scales, scale_index(p, r, 0), p.scale, sc.stored);
  uint8_t* out = reinterpret_cast<uint8_t*>(p.codes);
  if (p.code == BSMM_E2M1) {
    for (int64_t c = 2 * t; c < p.cols; c += 512) {
      const uint32_t lo = encode1<POW2>(load1<In>(x, r * p.ld_x + c), sc, p.code);
      const uint32_t hi = (c + 1 < p.cols) ? encode1<POW2>(load1<In>(x, r * p.ld_x + c + 1), sc, p.code) : 0u;
      out[(r * p.ld_codes + c) / 2] = static_cast<uint8_t>(lo | (hi << 4));
    }
  } else {
    for (int64_t c = t; c < p.cols; c += 256)
      out[r * p.ld_codes + c] = static_cast<uint8_t>(encode1<POW2>(load1<In>(x, r * p.ld_x + c), sc, p.code));
  }
}

// One CTA per 32 columns, 8 warps striding down the rows.
template <typename In, bool POW2>
__global__ void __launch_bounds__(256) quant_wcol(QP p) {
  __shared__ float wmax[8][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const bool cok = c < p.cols;
  const In* x = reinterpret_cast<const In*>(p.x);
  float m = 0.f;
  if (cok)
    for (int64_t r = warp; r < p.rows; r += 8) m = fmaxf(m, fabsf(load1<In>(x, r * p.ld_x + c)));
  wmax[warp][lane] = m;
  __syncthreads();
  m = wmax[0][lane];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, wmax[i][lane]);
  const Scale sc = make_scale(m, p.code, p.scale);
  if (warp == 0 && cok) store_scale(p.scales, p.transpose ? scale_index(p, c, 0) : c, p.scale, sc.stored);
  uint8_t* out = reinterpret_cast<uint8_t*>(p.codes);
  const bool fp4 = p.code == BSMM_E2M1;
  if (p.transpose) {
    // Column c becomes row c of the output; elements along the rows.
    if (!cok) return;
    if (fp4) {
      for (int64_t r = 2 * warp; r < p.rows; r += 16) {
        const uint32_t lo = encode1<POW2>(load1<In>(x, r * p.ld_x + c), sc, p.code);
        const uint32_t hi = (r + 1 < p.rows) ? encode1<POW2>(load1<In>(x, (r + 1) * p.ld_x + c), sc, p.code) : 0u;
        out[(c * p.ld_codes + r) / 2] = static_cast<uint8_t>(lo | (hi << 4));
      }
    } else {
      for (int64_t r = warp; r < p.rows; r += 8)
        out[c * p.ld_codes + r] = static_cast<uint8_t>(encode1<POW2>(load1<In>(x, r * p.ld_x + c), sc, p.code));
    }
  } else {
    for (int64_t r = warp; r < p.rows; r += 8) {
      const uint32_t v = cok ? encode1<POW2>(load1<In>(x, r * p.ld_x + c), sc, p.code) : 0u;
      if (fp4) {
        const uint32_t hi = __shfl_down_sync(0xffffffffu, v, 1);
        if (cok && (lane & 1) == 0) out[(r * p.ld_codes + c) / 2] = static_cast<uint8_t>(v | (hi << 4));
      } else if (cok) {
        out[r * p.ld_codes + c] = static_cast<uint8_t>(v);
      }
    }
  }
}

// One thread per block; any block shape that divides the array (E2M1 needs
// an even block extent along the output's contiguous axis).
template <typename In, bool POW2>
__global__ void __launch_bounds__(256) quant_any(QP p) {
  const int64_t nbr = p.rows / p.br, nbc = p.cols / p.bc;
  const int64_t bid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (bid >= nbr * nbc) return;
  const int64_t bi = bid / nbc, bj = bid % nbc;
  const In* x = reinterpret_cast<const In*>(p.x);
  float m = 0.f;
  for (int i = 0; i < p.br; ++i)
    for (int j = 0; j < p.bc; ++j) m = fmaxf(m, fabsf(load1<In>(x, (bi * p.br + i) * p.ld_x + bj * p.bc + j)));
  const Scale sc = make_scale(m, p.code, p.scale);
  store_scale(p.scales, p.transpose ? scale_index(p, bj, bi) : scale_index(p, bi, bj), p.scale, sc.stored);
  uint8_t* out = reinterpret_cast<uint8_t*>(p.codes);
  for (int i = 0; i < p.br; ++i) {
    for (int j = 0; j < p.bc; ++j) {
      const int64_t r = bi * p.br + i, c = bj * p.bc + j;
      const uint32_t v = encode1<POW2>(load1<In>(x, r * p.ld_x + c), sc, p.code);
      const int64_t e = p.transpose ? c * p.ld_codes + r : r * p.ld_codes + c;
      if (p.code == BSMM_E2M1) {
        uint8_t& byte = out[e / 2];
        byte = (e & 1) ? static_cast<uint8_t>((byte & 0x0Fu) | (v << 4)) : static_cast<uint8_t>((byte & 0xF0u) | v);
      } else {
        out[e] = static_cast<uint8_t>(v);
      }
    }
  }
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// DUAL: p2 is p's row-block output.  PAIR: p2 is a second array, quantized
// like p in the same launch.
template <bool POW2, bool DUAL, bool PAIR, int CODE>
cudaError_t launch_cols_tma2_code(const QP& p, const DeviceCtx* ctx, cudaStream_t s, const QP& p2) {
  CUtensorMap tm, tm2;
  if (!make_tmap_3d(&tm, p.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.cols, p.rows, 1, kCol2C, kColTileR, false))
    return cudaErrorInvalidValue;
  const int tiles_c = static_cast<int>(ceil_div(p.cols, kCol2C));
  const int64_t n_a = static_cast<int64_t>(tiles_c) * ceil_div(p.rows, kColTileR);
  int tiles_c2 = 0;
  int64_t n_tiles = n_a;
  if (PAIR) {
    if (!make_tmap_3d(&tm2, p2.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p2.cols, p2.rows, 1, kCol2C, kColTileR, false))
      return cudaErrorInvalidValue;
    tiles_c2 = static_cast<int>(ceil_div(p2.cols, kCol2C));
    n_tiles += static_cast<int64_t>(tiles_c2) * ceil_div(p2.rows, kColTileR);
  } else {
    tm2 = tm;  // not read
  }
  const int smem = kColStages * kCol2TileBytes + 128 + kColStages * 8;
  cudaError_t e =
      cudaFuncSetAttribute(quant_cols_tma2<POW2, DUAL, PAIR, CODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(n_tiles, static_cast<int64_t>(ctx->num_sms) * 2);
  {
    TraceScope tr(DUAL ? "quant_cols_tma2 (dual)" : (PAIR ? "quant_cols_tma2 (pair)" : "quant_cols_tma2"), s);
    quant_cols_tma2<POW2, DUAL, PAIR, CODE><<<static_cast<unsigned>(std::max<int64_t>(grid, 1)), 256, smem, s>>>(
        tm, p, tiles_c, n_tiles, ctx->status, wait_timeout_ns(), p2, tm2, tiles_c2, n_a);
  }
  return cudaGetLastError();
}

// The 8-bit code formats this kernel takes (E4M3, E5M2), as a template
// parameter.
template <bool POW2, bool DUAL = false, bool PAIR = false>
cudaError_t launch_cols_tma2(const QP& p, const DeviceCtx* ctx, cudaStream_t s, const QP& p2 = QP{}) {
  return p.code == BSMM_E4M3 ? launch_cols_tma2_code<POW2, DUAL, PAIR, BSMM_E4M3>(p, ctx, s, p2)
                             : launch_cols_tma2_code<POW2, DUAL, PAIR, BSMM_E5M2>(p, ctx, s, p2);
}

template <bool POW2>
cudaError_t launch_cols_tma(const QP& p, const DeviceCtx* ctx, cudaStream_t s) {
  CUtensorMap tm;
  if (!make_tmap_3d(&tm, p.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.cols, p.rows, 1, kColTileC, kColTileR, false))
    return cudaErrorInvalidValue;
  const int tiles_c = static_cast<int>(ceil_div(p.cols, kColTileC));
  const int64_t n_tiles = static_cast<int64_t>(tiles_c) * ceil_div(p.rows, kColTileR);
  const int smem = kColStages * kColTileBytes + 128 + kColStages * 8;
  cudaError_t e = cudaFuncSetAttribute(quant_cols_tma<POW2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(n_tiles, static_cast<int64_t>(ctx->num_sms) * 3);
  {
    TraceScope tr("quant_cols_tma", s);
    quant_cols_tma<POW2><<<static_cast<unsigned>(std::max<int64_t>(grid, 1)), 256, smem, s>>>(
        tm, p, tiles_c, n_tiles, ctx->status, wait_timeout_ns());
  }
  return cudaGetLastError();
}

template <typename In, bool POW2>
cudaError_t dispatch(const QP& p, const DeviceCtx* ctx, cudaStream_t s) {
  const int esz = sizeof(In);
  const bool x_vec = aligned(p.x, 16) && (p.ld_x * esz) % 16 == 0 && p.cols % (16 / esz) == 0;
  const bool codes16 = aligned(p.codes, 16) && p.ld_codes % 32 == 0;
  const bool pow2_small = (p.bc == 16 || p.bc == 32 || p.bc == 64 || p.bc == 128);
  const bool pow2_small_r = (p.br == 16 || p.br == 32 || p.br == 64 || p.br == 128);
  // bf16 columns into transposed 8-bit codes (the backward's operands): TMA-fed tiles
  const bool cols_tma = sizeof(In) == 2 && p.transpose && p.bc == 1 && pow2_small_r && p.code != BSMM_E2M1 &&
                        p.scale != BSMM_SCALE_F32 && codes16 && p.ld_codes % 32 == 0 && p.ld_x == p.cols &&
                        p.cols % 8 == 0 && aligned(p.x, 16);
  if (cols_tma) return p.br == 32 ? launch_cols_tma2<POW2>(p, ctx, s) : launch_cols_tma<POW2>(p, ctx, s);
  if (p.br == 1 && pow2_small && !p.transpose && x_vec && codes16) {
    int64_t blocks = ceil_div(p.rows * (p.cols / kSlice), 256 * 2);
    blocks = std::min<int64_t>(blocks, static_cast<int64_t>(ctx->num_sms) * 8);
    {
      TraceScope tr("quant_rows", s);
      quant_rows<In, POW2><<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, s>>>(p);
    }
  } else if (p.bc == 1 && pow2_small_r && (!p.transpose || (codes16 && p.ld_codes % 32 == 0))) {
    const int tiles_c = static_cast<int>(ceil_div(p.cols, kColTileC));
    const int64_t n_tiles = static_cast<int64_t>(tiles_c) * ceil_div(p.rows, kColTileR);
    const int64_t grid = std::min<int64_t>(n_tiles, static_cast<int64_t>(ctx->num_sms) * 3);
    {
      TraceScope tr("quant_cols", s);
      quant_cols<In, POW2><<<static_cast<unsigned>(std::max<int64_t>(grid, 1)), 256, 0, s>>>(p, x_vec ? 1 : 0, tiles_c,
                                                                                        n_tiles);
    }
  } else if (p.br == 128 && p.bc == 128 && !p.transpose && x_vec && codes16) {
    dim3 grid(static_cast<unsigned>(p.cols / 128), static_cast<unsigned>(p.rows / 128));
    {
      TraceScope tr("quant_tile", s);
      quant_tile<In, POW2><<<grid, 512, 0, s>>>(p);
    }
  } else if (p.br == 1 && p.bc == p.cols && !p.transpose) {
    {
      TraceScope tr("quant_wrow", s);
      quant_wrow<In, POW2><<<static_cast<unsigned>(p.rows), 256, 0, s>>>(p);
    }
  } else if (p.bc == 1 && p.br == p.rows) {
    {
      TraceScope tr("quant_wcol", s);
      quant_wcol<In, POW2><<<static_cast<unsigned>(ceil_div(p.cols, 32)), 256, 0, s>>>(p);
    }
  } else {
    const int64_t nblk = (p.rows / p.br) * (p.cols / p.bc);
    {
      TraceScope tr("quant_any", s);
      quant_any<In, POW2><<<static_cast<unsigned>(ceil_div(nblk, 256)), 256, 0, s>>>(p);
    }
  }
  return cudaGetLastError();
}

}  // namespace

namespace {
QP to_qp(const QuantRequest& q) {
  return QP{q.x, q.rows, q.cols, q.ld_x, q.br, q.bc, q.code, q.scale, q.transpose ? 1 : 0,
            q.codes, q.ld_codes, q.scales, q.ld_scales, q.sf_atoms ? 1 : 0, q.sf_rows, q.sf_rt, q.sf_ks4};
}

// Whether dispatch() runs p on quant_tile (the earlier branches all need
// 1-wide blocks or a transposed output).
template <typename In>
bool tile_eligible(const QP& p) {
  const int esz = sizeof(In);
  const bool x_vec = aligned(p.x, 16) && (p.ld_x * esz) % 16 == 0 && p.cols % (16 / esz) == 0;
  const bool codes16 = aligned(p.codes, 16) && p.ld_codes % 32 == 0;
  return p.br == 128 && p.bc == 128 && !p.transpose && x_vec && codes16;
}

// Whether dispatch() runs a bf16 p on quant_cols_tma2 (transposed 32 x 1
// blocks of 8-bit codes with one-byte scales).
bool cols_tma2_eligible(const QuantRequest& q) {
  const QP p = to_qp(q);
  const bool codes16 = aligned(p.codes, 16) && p.ld_codes % 32 == 0;
  return q.x_bf16 && p.transpose && p.bc == 1 && p.br == 32 && p.code != BSMM_E2M1 && p.code != BSMM_INT8 &&
         p.scale != BSMM_SCALE_F32 && codes16 && p.ld_x == p.cols && p.cols % 8 == 0 && aligned(p.x, 16);
}

template <typename In, bool POW2>
cudaError_t launch_tile_batch(const QuantRequest* q, const std::vector<int>& jobs, cudaStream_t s) {
  for (size_t j0 = 0; j0 < jobs.size(); j0 += kTileBatchMax) {
    QTileBatch b{};
    b.n = static_cast<int>(std::min<size_t>(kTileBatchMax, jobs.size() - j0));
    b.first[0] = 0;
    for (int k = 0; k < b.n; ++k) {
      const QuantRequest& r = q[jobs[j0 + k]];
      b.p[k] = to_qp(r);
      b.tiles_c[k] = r.cols / 128;
      b.first[k + 1] = b.first[k] + (r.rows / 128) * (r.cols / 128);
    }
    if (b.first[b.n] > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    TraceScope tr("quant_tile_batch", s);
    quant_tile_batch<In, POW2><<<static_cast<unsigned>(b.first[b.n]), 512, 0, s>>>(b);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_quantize_pair(const QuantRequest& qa, const QuantRequest& qb, cudaStream_t s) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  const bool eligible = cols_tma2_eligible(qa) && cols_tma2_eligible(qb) && qa.code == qb.code &&
                        qa.scale == qb.scale;
  if (!eligible) {
    const cudaError_t e = launch_quantize(qa, s);
    return e != cudaSuccess ? e : launch_quantize(qb, s);
  }
  const QP pa = to_qp(qa), pb = to_qp(qb);
  return qa.scale == BSMM_SCALE_UE8M0 ? launch_cols_tma2<true, false, true>(pa, ctx, s, pb)
                                      : launch_cols_tma2<false, false, true>(pa, ctx, s, pb);
}

cudaError_t launch_quantize_batch(const QuantRequest* q, int n, cudaStream_t s) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  // the 128 x 128 jobs quant_tile takes, by input type and scale kind
  // (f32 / bf16 x divided / power of two); the rest run one launch each
  std::vector<int> tiles[4];
  for (int i = 0; i < n; ++i) {
    const QP p = to_qp(q[i]);
    const bool ok = q[i].x_bf16 ? tile_eligible<__nv_bfloat16>(p) : tile_eligible<float>(p);
    if (ok) {
      tiles[(q[i].x_bf16 ? 2 : 0) + (q[i].scale == BSMM_SCALE_UE8M0 ? 1 : 0)].push_back(i);
    } else {
      const cudaError_t e = launch_quantize(q[i], s);
      if (e != cudaSuccess) return e;
    }
  }
  cudaError_t e = launch_tile_batch<float, false>(q, tiles[0], s);
  if (e == cudaSuccess) e = launch_tile_batch<float, true>(q, tiles[1], s);
  if (e == cudaSuccess) e = launch_tile_batch<__nv_bfloat16, false>(q, tiles[2], s);
  if (e == cudaSuccess) e = launch_tile_batch<__nv_bfloat16, true>(q, tiles[3], s);
  return e;
}

cudaError_t launch_quantize_dual(const QuantRequest& qc, const QuantRequest& qr, cudaStream_t s) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  // One pass over x when both are 8-bit MX quantizations of the same bf16
  // array: qc transposed in 32 x 1 blocks, qr untransposed in 1 x 32.
  const bool one_byte = qc.scale != BSMM_SCALE_F32 && qc.scale == qr.scale;
  const bool eligible = qc.x == qr.x && qc.x_bf16 && qr.x_bf16 && qc.rows == qr.rows && qc.cols == qr.cols &&
                        qc.transpose && qc.br == 32 && qc.bc == 1 && !qr.transpose && qr.br == 1 && qr.bc == 32 &&
                        qc.code == qr.code && qc.code != BSMM_E2M1 && qc.code != BSMM_INT8 && one_byte &&
                        qc.ld_x == qc.cols && qr.ld_x == qr.cols && qc.cols % 32 == 0 && aligned(qc.x, 16) &&
                        aligned(qc.codes, 16) && qc.ld_codes % 32 == 0 && aligned(qr.codes, 16) && qr.ld_codes % 16 == 0;
  if (!eligible) {
    cudaError_t e = launch_quantize(qc, s);
    return e != cudaSuccess ? e : launch_quantize(qr, s);
  }
  const QP pc = to_qp(qc), pr = to_qp(qr);
  return qc.scale == BSMM_SCALE_UE8M0 ? launch_cols_tma2<true, true>(pc, ctx, s, pr)
                                      : launch_cols_tma2<false, true>(pc, ctx, s, pr);
}

namespace {
// ---------------------------------------------------------------------------
// Self-test: quotient.cuh against the hardware's correctly rounded division
// ---------------------------------------------------------------------------
// splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014): pair i draws from the hashes of seed + 2i, +1.
__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// One (x, s) pair: s in [2^-80, 2^126) with a random exponent and a random,
// all-ones or zero significand; x one of
//   0, 1  x = RN(t s) for a random quotient t with |t| in [2^-100, 2^18),
//   2     x = RN(m s) nudged by up to two ulps, m a rounding midpoint
//         (2j + 1) 2^(k-1) of the code grids (k in [-17, 7]): quotients
//         that sit on or next to a tie,
//   3     |x| < 2^-100: subnormals, zeros and tiny normals.
// Counts a pair as bad unless the scalar and the packed forms agree bit for
// bit with __fdiv_rn when neither |x| nor |x / s| is below 2^-100, and
// otherwise give a quotient below 2^-19 with x's sign (as __fdiv_rn does).
__global__ void __launch_bounds__(256) selftest_quotient_kernel(uint64_t pairs, uint64_t seed,
                                                                unsigned long long* bad) {
  unsigned long long nbad = 0;
  for (uint64_t i = blockIdx.x * 256ull + threadIdx.x; i < pairs; i += gridDim.x * 256ull) {
    const uint64_t h1 = splitmix64(seed + 2 * i), h2 = splitmix64(seed + 2 * i + 1);
    const int es = -80 + static_cast<int>(h1 % 206u);
    const uint32_t skind = static_cast<uint32_t>(h1 >> 8) & 7u;
    const uint32_t sman = skind == 0 ? 0x7FFFFFu : (skind == 1 ? 0u : static_cast<uint32_t>(h1 >> 16) & 0x7FFFFFu);
    const float s = __uint_as_float((static_cast<uint32_t>(es + 127) << 23) | sman);
    const uint32_t sign = static_cast<uint32_t>(h2 >> 63) << 31;
    const uint32_t xkind = static_cast<uint32_t>(h2) & 3u;
    float x;
    if (xkind < 2) {
      const int d = -100 + static_cast<int>((h2 >> 2) % 118u);
      const float t = __uint_as_float((static_cast<uint32_t>(d + 127) << 23) | (static_cast<uint32_t>(h2 >> 9) & 0x7FFFFFu));
      x = __fmul_rn(t, s);
    } else if (xkind == 2) {
      const int k = -17 + static_cast<int>((h2 >> 2) % 25u);
      const float m = ldexpf(static_cast<float>(2 * (static_cast<int>(h2 >> 8) & 255) + 1), k - 1);
      const int nudge = static_cast<int>((h2 >> 16) % 5u) - 2;
      x = __uint_as_float(__float_as_uint(__fmul_rn(m, s)) + nudge);
    } else {
      x = __uint_as_float(static_cast<uint32_t>(h2 >> 2) % (27u << 23));  // below 2^-100
    }
    x = __uint_as_float(__float_as_uint(x) | sign);
    if (!(fabsf(x) < 0x1p127f)) continue;  // a nudge or product past the finite range
    const float y = block_recip(s);
    const float r = __fdiv_rn(x, s), nr = __fdiv_rn(-x, s);
    const float q = quot_rn(x, s, y);
    const float2 q2 = quot2_rn(make_float2(x, -x), s, y);
    const float2 qi = quot2_rn_int(make_float2(x, -x), s, y);
    bool ok;
    if (fabsf(x) >= 0x1p-100f && fabsf(r) >= 0x1p-100f) {
      ok = y != 0.f && __float_as_uint(q) == __float_as_uint(r) && __float_as_uint(q2.x) == __float_as_uint(r) &&
           __float_as_uint(q2.y) == __float_as_uint(nr) && qi.x == r && qi.y == nr;
    } else {
      const uint32_t sx = __float_as_uint(x) & 0x80000000u;
      ok = y != 0.f && fabsf(q) < 0x1p-19f && fabsf(q2.x) < 0x1p-19f && fabsf(q2.y) < 0x1p-19f &&
           fabsf(qi.x) < 0x1p-19f && fabsf(qi.y) < 0x1p-19f && (__float_as_uint(q) & 0x80000000u) == sx &&
           (__float_as_uint(q2.x) & 0x80000000u) == sx && (__float_as_uint(q2.y) & 0x80000000u) != sx &&
           fabsf(r) < 0x1p-19f;
    }
    nbad += ok ? 0 : 1;
  }
  if (nbad) atomicAdd(bad, nbad);
}
}  // namespace

cudaError_t launch_selftest_quotient(uint64_t pairs, uint64_t seed, unsigned long long* bad, cudaStream_t s) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  const uint64_t want = (pairs + 255) / 256;
  const unsigned grid = static_cast<unsigned>(std::max<uint64_t>(1, std::min<uint64_t>(want, 8ull * ctx->num_sms)));
  {
    TraceScope tr("selftest_quotient", s);
    selftest_quotient_kernel<<<grid, 256, 0, s>>>(pairs, seed, bad);
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize(const QuantRequest& q, cudaStream_t s) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  QP p = to_qp(q);
  // UE8M0 scales are powers of two: the codes divide by multiplying with the
  // exact reciprocal.
  const bool pow2 = q.scale == BSMM_SCALE_UE8M0;
  if (q.x_bf16) return pow2 ? dispatch<__nv_bfloat16, true>(p, ctx, s) : dispatch<__nv_bfloat16, false>(p, ctx, s);
  return pow2 ? dispatch<float, true>(p, ctx, s) : dispatch<float, false>(p, ctx, s);
}

}  // namespace bsmm
