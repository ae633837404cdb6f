// Block-scaled GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// One persistent, warp-specialised kernel template serves three paths:
//
//   kF32Scale  y[m,n] = sum_kb sa[m,kb] * sb[n/128,kb] * (a . b over K block kb)
//              (atrex-bench #002 block_scaled_mm, Reference Implementation).
//              FP8 x FP8 -> FP32 partial per 128-K block in tensor memory
//              (kind::f8f6f4); the epilogue warps read each partial with
//              tcgen05.ld and promote it into FP32 registers with sa*sb.
//              Partials are double-buffered so the MMA runs a block ahead.
//   kMXF8      y = sum_k a*2^(ea-127) * b*2^(eb-127), UE8M0 scale per 32 K
//              (jax.nn.scaled_matmul, Notes: MXFP8 on Blackwell).  Hardware
//              block scaling (kind::mxf8f6f4.block_scale.block32), scales
//              staged into tensor memory with tcgen05.cp.
//   kNVF4      packed E2M1 operands, UE4M3 scale per 16 K (Notes: NVFP4),
//              kind::mxf4nvf4.block_scale.block16.
//
// CTA: 384 threads.  warp 0 issues TMA loads (A, B and scale-factor atoms)
// into a STAGES-deep shared-memory ring; warp 1 issues the MMAs from one
// thread; warp 2 owns the tensor-memory allocation; warps 4..11 are the
// epilogue (two warpgroups, each owning half of the tile's columns; warp w
// reads TMEM lanes 32*(w%4)..+31 = rows of the tile).  Output tiles leave
// through a swizzled staging buffer and TMA stores.  Tiles are visited in
// groups of kGroupM M-tiles so the operands a wave touches stay in L2.
//
// Every wait is bounded (mbar_wait); on expiry the kernel records the site,
// drains its own copies and MMAs, frees its tensor memory and returns.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace bsmm {
namespace {

enum Mode { kF32Scale = 0, kMXF8 = 1, kNVF4 = 2 };
// Names the trace records give the one-CTA kernel's launches.
constexpr const char* mode_trace_name(int mode, bool split_k) {
  return split_k ? "tc_gemm<F32> split-K"
                 : (mode == kF32Scale ? "tc_gemm<F32>" : (mode == kMXF8 ? "tc_gemm<MXF8>" : "tc_gemm<NVF4>"));
}

constexpr int BM = 128;          // rows per tile (TMEM lanes)
constexpr int BK_BYTES = 128;    // K bytes per stage: 128 FP8 or 256 FP4 elements
constexpr int kThreads = 384;
constexpr int kEpiWarps = 8;
constexpr int kTmemCols = 512;
constexpr int kGroupM = 16;
constexpr int kStagingPerWarp = 2 * 4096;  // two 32-row x 128-byte buffers

enum Site { kSiteProducer = 1, kSiteMmaTmem = 2, kSiteMmaFull = 3, kSiteEpilogue = 4, kSiteDrain = 5,
            kSiteDone = 6, kSiteSelftest = 7, kSiteSplitK = 8 };

constexpr int align1024(int v) { return (v + 1023) / 1024 * 1024; }

template <int MODE, int BN, int STAGES>
struct Cfg {
  static constexpr int A_BYTES = BM * BK_BYTES;
  static constexpr int B_BYTES = BN * BK_BYTES;
  // scale-factor atoms (128 rows x 4 bytes = 512 B) per K-tile per 128 rows
  static constexpr int ATOMS = MODE == kMXF8 ? 1 : (MODE == kNVF4 ? 4 : 0);
  static constexpr int SFA_BYTES = ATOMS * 512;
  static constexpr int SFB_BYTES = ATOMS * 512 * (BN / 128);
  static constexpr int SF_BYTES = SFA_BYTES + SFB_BYTES;
  static constexpr int STAGE_TX = A_BYTES + B_BYTES + SF_BYTES;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_STG = align1024(OFF_SF + STAGES * SF_BYTES);
  static constexpr int OFF_BAR = OFF_STG + kEpiWarps * kStagingPerWarp;
  // full/empty per stage, tfull/tempty per accumulator, done, and (split K)
  // red_full/red_empty per epilogue warp
  static constexpr int N_BARS = 2 * STAGES + 2 * 4 + 1 + 2 * kEpiWarps;
  static constexpr int SMEM = OFF_BAR + N_BARS * 8 + 16 + 1024;  // + alignment slack
  // tensor-memory columns: NACC accumulators of BN columns, then scale factors
  static constexpr int NACC = MODE == kF32Scale ? kTmemCols / BN : 2;
  static constexpr int SF_COL0 = NACC * BN;
  static constexpr int SFA_COLS = ATOMS * 4;
  static constexpr int SFB_COLS = ATOMS * 4 * (BN / 128);
  static constexpr int SF_COLS = SFA_COLS + SFB_COLS;
  static_assert(SF_COL0 + STAGES * SF_COLS <= kTmemCols, "tensor memory budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(BN % 128 == 0 && BN <= 256, "BN");
};

struct Params {
  int M, N, K;  // K in elements
  int m_tiles, n_tiles, k_tiles;
  int num_tiles;  // over all batches
  // block-scaled paths: scale-factor atoms [batch][row tile][K atom] x 512 B
  const uint8_t* sfa;
  const uint8_t* sfb;
  int sfa_rt, sfb_rt, ks4;
  // FP32-scale path
  const float* a_scales;
  const float* b_scales;
  int kb;  // K / 128
  // split K (FP32-scale path): clusters of `splits` CTAs share each tile,
  // CTA rank r taking K tiles r * kpb .. min((r + 1) * kpb, k_tiles) - 1
  int splits, kpb;
  // output
  void* y;
  int y_bf16;
  int tma_store;
  uint32_t idesc;
  int* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ void decode_tile(const Params& p, int t, int& b, int& mb, int& nb) {
  const int per_batch = p.m_tiles * p.n_tiles;
  b = t / per_batch;
  const int r = t - b * per_batch;
  const int span = kGroupM * p.n_tiles;
  const int g = r / span;
  const int within = r - g * span;
  const int rows = min(kGroupM, p.m_tiles - g * kGroupM);
  mb = g * kGroupM + within % rows;
  nb = within / rows;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int MODE, int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmY, const Params p) {
  using C = Cfg<MODE, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* sSF = smem + C::OFF_SF;
  uint8_t* stg = smem + C::OFF_STG;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + C::NACC;
  uint64_t* done = tempty + C::NACC;
  uint64_t* red_full = done + 1;              // split K, in a block's owner: the peers' partials are staged
  uint64_t* red_empty = red_full + kEpiWarps;  // split K, in each peer: the owner has read them
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(red_empty + kEpiWarps);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int never_abort_storage = 0;  // drains ignore the CTA abort flag
  volatile int* never_abort = &never_abort_storage;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < C::NACC; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiWarps);
    }
    mbar_init(done, 1);
    for (int i = 0; i < kEpiWarps; ++i) {
      mbar_init(&red_full[i], p.splits > 1 ? p.splits - 1 : 1);
      mbar_init(&red_empty[i], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 2) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (p.splits > 1) cluster_sync();  // every CTA's barriers are initialized before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // Split K: cluster `cid` of `ncl` works on tiles cid, cid + ncl, ..; this
  // CTA (rank `krank`) on K tiles kbeg .. kend - 1 of each.
  const int krank = p.splits > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cid = blockIdx.x / p.splits, ncl = gridDim.x / p.splits;
  const int kbeg = krank * p.kpb;
  const int kend = min(kbeg + p.kpb, p.k_tiles);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int t = cid; ok && t < p.num_tiles; t += ncl) {
        int b, mb, nb;
        decode_tile(p, t, b, mb, nb);
        for (int kt = kbeg; kt < kend; ++kt) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.status, kSiteProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], C::STAGE_TX);
          tma_load_3d(sA + stage * C::A_BYTES, &tmA, &full[stage], kt * BK_BYTES, mb * BM, b);
          tma_load_3d(sB + stage * C::B_BYTES, &tmB, &full[stage], kt * BK_BYTES, nb * BN, b);
          if constexpr (MODE != kF32Scale) {
            uint8_t* sf = sSF + stage * C::SF_BYTES;
            const uint8_t* ga =
                p.sfa + (static_cast<size_t>(b * p.sfa_rt + mb) * p.ks4 + static_cast<size_t>(kt) * C::ATOMS) * 512;
            bulk_load(sf, ga, C::SFA_BYTES, &full[stage]);
#pragma unroll
            for (int i = 0; i < BN / 128; ++i) {
              const uint8_t* gb = p.sfb + (static_cast<size_t>(b * p.sfb_rt + nb * (BN / 128) + i) * p.ks4 +
                                           static_cast<size_t>(kt) * C::ATOMS) * 512;
              bulk_load(sf + C::SFA_BYTES + i * C::ATOMS * 512, gb, C::ATOMS * 512, &full[stage]);
            }
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // No copy may still target this CTA's shared memory when it exits.
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          mbar_wait(&full[s], (last_par >> s) & 1u, p.timeout_ns, never_abort, p.status, kSiteDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, tb = 0;
      uint32_t phase = 0, tph = 0;
      bool ok = true;
      for (int t = cid; ok && t < p.num_tiles; t += ncl) {
        if constexpr (MODE != kF32Scale) {
          if (!mbar_wait(&tempty[tb], tph ^ 1u, p.timeout_ns, abort_flag, p.status, kSiteMmaTmem)) break;
          tc_fence_after();
        }
        for (int kt = kbeg; kt < kend; ++kt) {
          if constexpr (MODE == kF32Scale) {
            if (!mbar_wait(&tempty[tb], tph ^ 1u, p.timeout_ns, abort_flag, p.status, kSiteMmaTmem)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.status, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * C::B_BYTES);
          const uint32_t d = tmem + static_cast<uint32_t>(tb * BN);
          if constexpr (MODE == kF32Scale) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f8f6f4(d, smem_desc(a_base + 32 * k, 16, 1024, 2), smem_desc(b_base + 32 * k, 16, 1024, 2), p.idesc,
                         k > 0 ? 1u : 0u);
            tc_commit(&empty[stage]);
            tc_commit(&tfull[tb]);
            if (++tb == C::NACC) {
              tb = 0;
              tph ^= 1u;
            }
          } else {
            const uint32_t sf_t = tmem + static_cast<uint32_t>(C::SF_COL0 + stage * C::SF_COLS);
            const uint32_t sfa_t = sf_t, sfb_t = sf_t + C::SFA_COLS;
            const uint32_t sf_s = smem_u32(sSF + stage * C::SF_BYTES);
            // SFA atom i (K sub-block i) -> columns sfa_t + 4i.
#pragma unroll
            for (int i = 0; i < C::ATOMS; ++i) tc_cp_sf(sfa_t + 4 * i, smem_desc(sf_s + 512 * i, 0, 128, 0));
            // SFB atom (row tile r, K sub-block i) -> columns sfb_t + 4*(i*(BN/128) + r).
#pragma unroll
            for (int r = 0; r < BN / 128; ++r)
#pragma unroll
              for (int i = 0; i < C::ATOMS; ++i)
                tc_cp_sf(sfb_t + 4 * (i * (BN / 128) + r),
                         smem_desc(sf_s + C::SFA_BYTES + 512 * (r * C::ATOMS + i), 0, 128, 0));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc(a_base + 32 * k, 16, 1024, 2);
              const uint64_t bd = smem_desc(b_base + 32 * k, 16, 1024, 2);
              const uint32_t acc = (kt > kbeg || k > 0) ? 1u : 0u;
              if constexpr (MODE == kMXF8) {
                // one byte of the 4-byte scale word per 32-K step
                const uint32_t idesc = p.idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
                mma_mxf8(d, ad, bd, idesc, sfa_t, sfb_t, acc);
              } else {
                mma_nvf4(d, ad, bd, p.idesc, sfa_t + 4 * k, sfb_t + 4 * k * (BN / 128), acc);
              }
            }
            tc_commit(&empty[stage]);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if constexpr (MODE != kF32Scale) {
          if (!ok) break;
          tc_commit(&tfull[tb]);
          if (++tb == C::NACC) {
            tb = 0;
            tph ^= 1u;
          }
        }
      }
      // Every MMA and copy this thread issued must finish before TMEM is freed.
      tc_commit(done);
      mbar_wait(done, 0, p.timeout_ns, never_abort, p.status, kSiteDone);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    constexpr int COLS = BN / 2;  // columns per thread
    const int ew = warp - 4;
    const int q = warp & 3;   // TMEM lane quarter
    const int g = ew >> 2;    // column half of the tile
    uint8_t* my_stg = stg + ew * kStagingPerWarp;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int tb = 0, sbuf = 0;
    uint32_t tph = 0, rph = 0;
    for (int t = cid; t < p.num_tiles; t += ncl) {
      int b, mb, nb;
      decode_tile(p, t, b, mb, nb);
      const int row = mb * BM + q * 32 + lane;
      const int col0 = nb * BN + g * COLS;
      float acc[COLS];
      bool ok = true;
      if constexpr (MODE == kF32Scale) {
#pragma unroll
        for (int i = 0; i < COLS; ++i) acc[i] = 0.f;
        const bool row_ok = row < p.M;
        const float* sa_row = p.a_scales + static_cast<size_t>(row_ok ? row : 0) * p.kb;
        const float* sb_row = p.b_scales + static_cast<size_t>(col0 / 128) * p.kb;
        float sa_next = row_ok ? __ldg(sa_row + kbeg) : 0.f;
        float sb_next = __ldg(sb_row + kbeg);
        for (int kt = kbeg; kt < kend; ++kt) {
          const float s = sa_next * sb_next;
          if (kt + 1 < kend) {
            sa_next = row_ok ? __ldg(sa_row + kt + 1) : 0.f;
            sb_next = __ldg(sb_row + kt + 1);
          }
          if (!mbar_wait(&tfull[tb], tph, p.timeout_ns, abort_flag, p.status, kSiteEpilogue)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(tb * BN + g * COLS);
          static_assert(COLS == 64, "promotion epilogue reads two 32-column chunks");
          uint32_t r0[32], r1[32];
          tmem_ld32(taddr, r0);
          tmem_ld32(taddr + 32, r1);
          tmem_wait_ld();
          // packed two-lane FP32 FMAs (each lane an ordinary fmaf): half the
          // instructions of the promotion, which bounds this loop
          const float2 s2 = make_float2(s, s);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 v = __ffma2_rn(make_float2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1])), s2,
                                        make_float2(acc[2 * j], acc[2 * j + 1]));
            acc[2 * j] = v.x;
            acc[2 * j + 1] = v.y;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 v = __ffma2_rn(make_float2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1])), s2,
                                        make_float2(acc[32 + 2 * j], acc[32 + 2 * j + 1]));
            acc[32 + 2 * j] = v.x;
            acc[32 + 2 * j + 1] = v.y;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[tb]);
          if (++tb == C::NACC) {
            tb = 0;
            tph ^= 1u;
          }
        }
      } else {
        if (!mbar_wait(&tfull[tb], tph, p.timeout_ns, abort_flag, p.status, kSiteEpilogue)) {
          ok = false;
        } else {
          tc_fence_after();
          const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(tb * BN + g * COLS);
#pragma unroll
          for (int c = 0; c < COLS / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(taddr + 32 * c, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[32 * c + j] = __uint_as_float(r[j]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[tb]);
          if (++tb == C::NACC) {
            tb = 0;
            tph ^= 1u;
          }
        }
      }
      if (!ok) break;
      if constexpr (MODE == kF32Scale) {
        if (p.splits > 1) {
          // Split K, reduce-scatter: the 32 x 64 block of epilogue warp ew is
          // summed and stored by rank ew % splits.  Every other rank stages
          // its partial of that block (16-byte units rotated by lane) and
          // signals the owner, which adds the partials and hands the staging
          // buffers back.  Each rank reads (splits - 1) x 8 KB per block it
          // owns instead of one rank reading them all.
          const int owner = ew % p.splits;
          const uint32_t part = smem_u32(my_stg);
          if (krank != owner) {
            if (!mbar_spin_acq_cluster(&red_empty[ew], rph ^ 1u, p.timeout_ns, abort_flag, p.status, kSiteSplitK))
              break;
#pragma unroll
            for (int j = 0; j < COLS / 4; ++j)
              *reinterpret_cast<float4*>(my_stg + 16 * (lane * 16 + (j ^ (lane & 15)))) =
                  make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
            __syncwarp();
            if (lane == 0)
              mbar_arrive_release_cluster(mapa_shared(smem_u32(&red_full[ew]), static_cast<uint32_t>(owner)));
            rph ^= 1u;
            continue;
          }
          if (!mbar_spin_acq_cluster(&red_full[ew], rph, p.timeout_ns, abort_flag, p.status, kSiteSplitK)) break;
          // The owner adds the peers' blocks to its own in the fixed order
          // owner + 1, owner + 2, .. (mod splits): deterministic for a given
          // split count.  A peer's whole block is requested at once (16 reads
          // in flight, each a round trip to another SM) before it is added.
          for (int i = 1; i < p.splits; ++i) {
            const int r = owner + i < p.splits ? owner + i : owner + i - p.splits;
            const uint32_t peer = mapa_shared(part, static_cast<uint32_t>(r));
            float4 v[COLS / 4];
#pragma unroll
            for (int j = 0; j < COLS / 4; ++j) v[j] = ld_shared_cluster_v4(peer + 16 * (lane * 16 + (j ^ (lane & 15))));
#pragma unroll
            for (int j = 0; j < COLS / 4; ++j) {
              acc[4 * j] += v[j].x;
              acc[4 * j + 1] += v[j].y;
              acc[4 * j + 2] += v[j].z;
              acc[4 * j + 3] += v[j].w;
            }
          }
          __syncwarp();
          if (lane == 0)
            for (int r = 0; r < p.splits; ++r)
              if (r != owner) mbar_arrive_release_cluster(mapa_shared(smem_u32(&red_empty[ew]), static_cast<uint32_t>(r)));
          rph ^= 1u;
        }
      }
      // ---- store the thread's row segment [col0, col0 + COLS)
      if (p.tma_store) {
        const int y0 = mb * BM + q * 32;
        if (!p.y_bf16) {
#pragma unroll
          for (int c = 0; c < COLS / 32; ++c) {
            uint8_t* buf = my_stg + sbuf * 4096;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float* v = &acc[32 * c + 4 * j];
              const uint32_t off = lane * 128 + ((j ^ (lane & 7)) * 16);
              *reinterpret_cast<uint4*>(buf + off) = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                                                                __float_as_uint(v[2]), __float_as_uint(v[3]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmY, buf, col0 + 32 * c, y0, b);
              bulk_commit();
            }
            sbuf ^= 1;
          }
        } else {
#pragma unroll
          for (int c = 0; c < COLS / 64; ++c) {
            uint8_t* buf = my_stg + sbuf * 4096;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float* v = &acc[64 * c + 8 * j];
              const uint32_t off = lane * 128 + ((j ^ (lane & 7)) * 16);
              *reinterpret_cast<uint4*>(buf + off) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                                pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmY, buf, col0 + 64 * c, y0, b);
              bulk_commit();
            }
            sbuf ^= 1;
          }
        }
      } else if (row < p.M) {
        const size_t base = (static_cast<size_t>(b) * p.M + row) * static_cast<size_t>(p.N);
        if (!p.y_bf16) {
          float* y = reinterpret_cast<float*>(p.y) + base;
#pragma unroll
          for (int j = 0; j < COLS; ++j)
            if (col0 + j < p.N) y[col0 + j] = acc[j];
        } else {
          __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.y) + base;
#pragma unroll
          for (int j = 0; j < COLS; ++j)
            if (col0 + j < p.N) y[col0 + j] = __float2bfloat16_rn(acc[j]);
        }
      }
    }
    if (lane == 0) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (p.splits > 1) cluster_sync();  // no CTA exits while a peer may still touch its shared memory
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Scale bytes [batch][rows][KSu] (row-major, one per user block of `rep`
// hardware blocks) -> atoms of the tensor-core scale-factor layout: atom
// (b, row tile rt, K atom j) is 512 bytes; byte (r%32)*16 + ((r%128)/32)*4 +
// (kb%4) holds the scale of row rt*128 + r for hardware K block 4j + kb%4,
// i.e. user scale (4j + kb%4) / rep.  Missing rows / blocks get `pad`.
// A thread owns word w of eight consecutive atoms j0..j0+7 of one row tile:
// it reads the 32 scale bytes of row rt*128 + (w>>2) + 32*(w&3) for K blocks
// 4*j0 .. 4*j0+31 (two 16-byte loads when in range and aligned) and writes
// one word to each atom; a warp's stores to an atom are 128 contiguous bytes.
// The 16-byte loads need KS % 16 == 0 and a 16-byte aligned base; otherwise
// (and at the K tail) the bytes are read one by one.
__global__ void __launch_bounds__(256) sf_relayout(const uint8_t* __restrict__ src, uint32_t* __restrict__ dst,
                                                   int nb, int R, int KS, int RT, int KS4, uint32_t pad, int KSu,
                                                   int rep) {
  const int groups = (KS4 + 7) / 8;  // groups of eight atoms per row tile
  const int64_t total = static_cast<int64_t>(nb) * RT * groups * 128;
  const uint32_t pad4 = pad * 0x01010101u;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int w = static_cast<int>(idx & 127);
    const int64_t t = idx >> 7;
    const int jg = static_cast<int>(t % groups);
    const int64_t t2 = t / groups;
    const int rt = static_cast<int>(t2 % RT);
    const int64_t b = t2 / RT;
    const int r = rt * 128 + (w >> 2) + 32 * (w & 3);
    const int kb0 = 32 * jg;
    uint32_t word[8];
    if (r >= R) {
#pragma unroll
      for (int i = 0; i < 8; ++i) word[i] = pad4;
    } else {
      const uint8_t* row = src + (b * R + r) * static_cast<int64_t>(KSu);
      if (rep == 1 && kb0 + 32 <= KS && (KS & 15) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(row + kb0));
        const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(row + kb0 + 16));
        word[0] = v0.x; word[1] = v0.y; word[2] = v0.z; word[3] = v0.w;
        word[4] = v1.x; word[5] = v1.y; word[6] = v1.z; word[7] = v1.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t v = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int kb = kb0 + 4 * i + k;
            v |= static_cast<uint32_t>(kb < KS ? row[kb / rep] : pad) << (8 * k);
          }
          word[i] = v;
        }
      }
    }
    uint32_t* out = dst + ((b * RT + rt) * static_cast<int64_t>(KS4) + 8 * jg) * 128 + w;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (8 * jg + i < KS4) out[i * 128] = word[i];
  }
}

// Scale bytes [batch][rows][KSu] -> the CTA-pair kernel's blocks of 512-byte
// slots, one block per (batch, T, K tile kt) holding the scales of K tile kt
// for `tiles` row tiles of 128 (rows 128 * tiles * T ..).  Atom a = tiles * j
// + r holds the scales of row tile tiles * T + r for hardware K blocks
// 4 (kt * atoms + j) .. +3.  Its row 32q + m0 is word q of 16-byte line m0 of
// slot a + q (`skew`), of slot a (neither), or of each of slots 4a .. 4a + 3
// (`replicate`); one byte per hardware block, in K order.  Missing rows and
// blocks past K get `pad`.  Slot positions that no atom fills are never read
// by the GEMM and are left as they are.  With src_rt > 0 the source is the
// plain atom layout instead ([batch][src_rt row tiles][src_ks4 atoms]).
// A thread owns one row (q, m0) of one tile of one block: it reads the row's
// 4 * atoms scale bytes of the K tile and writes its word of every atom.
__global__ void __launch_bounds__(256) sf_relayout_pair(const uint8_t* __restrict__ src, uint32_t* __restrict__ dst,
                                                        int nb, int R, int KS, int NT, int k_tiles, int atoms,
                                                        int tiles, int slots, int skew, int replicate,
                                                        uint32_t pad, int KSu, int rep, int src_rt, int src_ks4) {
  const int64_t total = static_cast<int64_t>(nb) * NT * k_tiles * tiles * 128;
  const uint32_t pad4 = pad * 0x01010101u;
  const bool fast = src_rt == 0 && rep == 1 && (KS & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 3) == 0;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int q = static_cast<int>(idx & 3);
    const int m0 = static_cast<int>((idx >> 2) & 31);
    int64_t t = idx >> 7;
    const int r = static_cast<int>(t % tiles);
    t /= tiles;
    const int kt = static_cast<int>(t % k_tiles);
    t /= k_tiles;
    const int T = static_cast<int>(t % NT);
    const int64_t b = t / NT;
    const int row = (T * tiles + r) * 128 + 32 * q + m0;
    uint32_t* block = dst + ((b * NT + T) * k_tiles + kt) * static_cast<int64_t>(slots) * 128;
    const uint8_t* src_row = src + (src_rt > 0 ? 0 : (b * R + (row < R ? row : 0)) * static_cast<int64_t>(KSu));
    for (int j = 0; j < atoms; ++j) {
      const int hb0 = 4 * (kt * atoms + j);
      uint32_t v;
      if (row >= R) {
        v = pad4;
      } else if (src_rt > 0) {  // word (row % 128) / 32 of line row % 32 of atom hb0 / 4
        const uint32_t* at = reinterpret_cast<const uint32_t*>(src) +
                             ((b * src_rt + (row >> 7)) * static_cast<int64_t>(src_ks4) + (hb0 >> 2)) * 128;
        v = __ldg(at + (row & 31) * 4 + ((row >> 5) & 3));
      } else if (fast && hb0 + 4 <= KS) {
        v = __ldg(reinterpret_cast<const uint32_t*>(src_row + hb0));
      } else {
        v = 0;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
          v |= static_cast<uint32_t>(hb0 + kb < KS ? src_row[(hb0 + kb) / rep] : pad) << (8 * kb);
      }
      const int a = tiles * j + r;
      if (replicate) {
#pragma unroll
        for (int c = 0; c < 4; ++c) block[(4 * a + c) * 128 + m0 * 4 + q] = v;
      } else {
        block[(a + (skew ? q : 0)) * 128 + m0 * 4 + q] = v;
      }
    }
  }
}

__global__ void selftest_wait_kernel(uint64_t timeout_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, timeout_ns, &abort_flag, status, kSiteSelftest);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
int rt_rows(int64_t R) { return static_cast<int>(ceil_div(R, 256) * 2); }  // row tiles, even for BN = 256

template <int MODE, int BN, int STAGES>
cudaError_t launch_kernel(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const Params& p_in,
                          const DeviceCtx* ctx, cudaStream_t s) {
  using C = Cfg<MODE, BN, STAGES>;
  auto kern = tc_gemm<MODE, BN, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  Params p = p_in;
  if (p.splits <= 1) {
    p.splits = 1;
    p.kpb = p.k_tiles;
    const int grid = std::max(1, std::min(p.num_tiles, ctx->num_sms));
    {
      TraceScope tr(mode_trace_name(MODE, false), s);
      kern<<<grid, kThreads, C::SMEM, s>>>(ta, tb, ty, p);
    }
    return cudaGetLastError();
  }
  // split K: clusters of `splits` CTAs, one tile per cluster at a time, as
  // many clusters as fit at once (the GPCs' SM counts need not be multiples
  // of the cluster size)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(p.splits * (ctx->num_sms / p.splits)));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int fit = 0;
  e = cudaOccupancyMaxActiveClusters(&fit, kern, &cfg);
  if (e != cudaSuccess) return e;
  const int ncl = std::max(1, std::min(p.num_tiles, fit));
  cfg.gridDim = dim3(static_cast<unsigned>(ncl * p.splits));
  TraceScope tr(mode_trace_name(MODE, true), s);
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, ty, p);
}

uint32_t f8_fmt(int dtype) { return dtype == BSMM_E5M2 ? 1u : 0u; }

bool make_output_map(CUtensorMap* ty, void* y, bool bf16, int64_t B, int64_t M, int64_t N) {
  const int esz = bf16 ? 2 : 4;
  if ((N * esz) % 16 != 0 || (reinterpret_cast<uintptr_t>(y) % 16) != 0) return false;
  return make_tmap_3d(ty, y, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, esz, N, M, B,
                      bf16 ? 64 : 32, 32, true);
}

}  // namespace

size_t sf_atoms_plain_bytes(int64_t B, int64_t R, int64_t K, int fmt) {
  const int64_t k_tiles = ceil_div(K, fmt == kFmtMXF8 ? 128 : 256);
  const int atoms = fmt == kFmtNVF4 ? 4 : (fmt == kFmtMXF4 ? 2 : 1);
  return static_cast<size_t>(B) * rt_rows(R) * k_tiles * atoms * 512;
}

size_t sf_atoms_bytes(int64_t B, int64_t R, int64_t K, int fmt) {
  // K per 128-byte tile: 128 FP8 or 256 FP4 elements; atoms per tile: one per
  // 4 scales (MXF8 1, NVF4 4, MXF4 2).  The larger of the one-CTA kernel's
  // atoms and the pair kernel's blocks, for either operand.
  const int64_t k_tiles = ceil_div(K, fmt == kFmtMXF8 ? 128 : 256);
  const int atoms = fmt == kFmtNVF4 ? 4 : (fmt == kFmtMXF4 ? 2 : 1);
  const int64_t rt = rt_rows(R);
  const int64_t slots = std::max({rt * atoms, rt * pair_sfa_slots(atoms),
                                  pair_b_replicated(atoms) ? rt / 2 * pair_sfb_slots(atoms) : 0});
  return static_cast<size_t>(B) * k_tiles * slots * 512;
}

cudaError_t launch_mx_gemm(const MxGemmRequest& r, cudaStream_t s, std::string* why) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  constexpr int BN = 128;
  const bool nv = r.fmt == kFmtNVF4, mf4 = r.fmt == kFmtMXF4;
  const int64_t k_tiles = ceil_div(r.K, (nv || mf4) ? 256 : 128);
  const int ks4 = static_cast<int>(k_tiles * (nv ? 4 : (mf4 ? 2 : 1)));
  const int KS = static_cast<int>(r.K / (nv ? 16 : 32));
  uint8_t* ws = reinterpret_cast<uint8_t*>(r.workspace);
  const size_t a_bytes = align_up(sf_atoms_bytes(r.B, r.M, r.K, r.fmt), 256);
  uint8_t* sfa = ws;
  uint8_t* sfb = ws + a_bytes;
  const uint32_t pad = nv ? 0u : 127u;  // scale 1 for UE8M0 blocks past K (their codes are zero)

  // Kernel choice: CTA-pair 256 x 256 tiles when there is a tile for every
  // cluster, else one CTA per 128 x 128 tile.  BSMM_MX_KERNEL=pair|single
  // overrides the choice (pair still needs TMA-storable output rows).
  const char* force = std::getenv("BSMM_MX_KERNEL");
  const bool want_pair = force && std::strcmp(force, "pair") == 0;
  const bool want_single = force && std::strcmp(force, "single") == 0;
  const int esz = r.y_bf16 ? 2 : 4;
  const bool storable = (r.N * esz) % 16 == 0 && reinterpret_cast<uintptr_t>(r.y) % 16 == 0;
  if (mf4 && !storable) {  // MXFP4 has only the pair kernel
    *why = "MXFP4 output rows must be 16-byte aligned (N * element size % 16 == 0)";
    return cudaErrorInvalidValue;
  }
  // Scales given in the plain atom layout (r.sf_atoms) are read in place by
  // every kernel that takes that layout; only the pair kernel's skewed and
  // replicated blocks are rewritten from them.
  // One operand's plain atoms [B][RT][ks4], from row-major scale bytes.
  auto plain_atoms = [&](const uint8_t* src, uint8_t* dst, int64_t R, int64_t KU) {
    const int RT = rt_rows(R);
    const int64_t words = r.B * RT * static_cast<int64_t>((ks4 + 7) / 8) * 128;
    const int blocks = static_cast<int>(std::min<int64_t>(ceil_div(words, 256), ctx->num_sms * 16));
    {
      TraceScope tr("sf_relayout", s);
      sf_relayout<<<blocks, 256, 0, s>>>(src, reinterpret_cast<uint32_t*>(dst), static_cast<int>(r.B),
                                         static_cast<int>(R), KS, RT, ks4, pad, static_cast<int>(KU),
                                         static_cast<int>(KS / KU));
    }
  };
  if (mf4 || (!want_single && (want_pair ? storable : mx_pair_eligible(r, ctx)))) {
    const int atoms = nv ? 4 : (mf4 ? 2 : 1);
    const int RTa = rt_rows(r.M), RTb = rt_rows(r.N);
    const int sa = pair_sfa_slots(atoms), sb = pair_sfb_slots(atoms);
    const int64_t ta_threads = r.B * RTa * k_tiles * 128, tb_threads = r.B * (RTb / 2) * k_tiles * 2 * 128;
    const int ga = static_cast<int>(std::min<int64_t>(ceil_div(ta_threads, 256), ctx->num_sms * 16));
    const int gb = static_cast<int>(std::min<int64_t>(ceil_div(tb_threads, 256), ctx->num_sms * 16));
    const int src_rta = r.sf_atoms ? RTa : 0, src_rtb = r.sf_atoms ? RTb : 0;
    const uint8_t* use_a = sfa;
    const uint8_t* use_b = sfb;
    if (atoms > 1) {
      {
        TraceScope tr("sf_relayout_pair", s);
        sf_relayout_pair<<<ga, 256, 0, s>>>(r.a_scales, reinterpret_cast<uint32_t*>(sfa), static_cast<int>(r.B),
                                            static_cast<int>(r.M), KS, RTa, static_cast<int>(k_tiles), atoms, 1, sa,
                                            1, 0, pad, static_cast<int>(r.K_a),
                                            r.sf_atoms ? 1 : static_cast<int>(KS / r.K_a), src_rta, ks4);
      }
    } else if (r.sf_atoms) {  // one atom per K tile: the pair layout is the plain one
      use_a = r.a_scales;
    } else {
      plain_atoms(r.a_scales, sfa, r.M, r.K_a);
    }
    if (pair_b_replicated(atoms)) {
      {
        TraceScope tr("sf_relayout_pair", s);
        sf_relayout_pair<<<gb, 256, 0, s>>>(r.b_scales, reinterpret_cast<uint32_t*>(sfb), static_cast<int>(r.B),
                                            static_cast<int>(r.N), KS, RTb / 2, static_cast<int>(k_tiles), atoms, 2,
                                            sb, 0, 1, pad, static_cast<int>(r.K_b),
                                            r.sf_atoms ? 1 : static_cast<int>(KS / r.K_b), src_rtb, ks4);
      }
    } else if (r.sf_atoms) {
      use_b = r.b_scales;
    } else {
      plain_atoms(r.b_scales, sfb, r.N, r.K_b);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const MxAtoms at{use_a, use_b, RTa, RTb, ks4, static_cast<int>(k_tiles)};
    return launch_mx_gemm_pair(r, at, s, why);
  }

  const uint8_t* use_a = sfa;
  const uint8_t* use_b = sfb;
  if (r.sf_atoms) {
    use_a = r.a_scales;
    use_b = r.b_scales;
  } else {
    plain_atoms(r.a_scales, sfa, r.M, r.K_a);
    plain_atoms(r.b_scales, sfb, r.N, r.K_b);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int64_t kbytes = nv ? r.K / 2 : r.K;
  CUtensorMap ta, tb, ty;
  if (!make_tmap_3d(&ta, r.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kbytes, r.M, r.B, BK_BYTES, BM, true) ||
      !make_tmap_3d(&tb, r.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kbytes, r.N, r.B, BK_BYTES, BN, true)) {
    *why = "cuTensorMapEncodeTiled failed for an operand";
    return cudaErrorInvalidValue;
  }
  Params p{};
  p.M = static_cast<int>(r.M);
  p.N = static_cast<int>(r.N);
  p.K = static_cast<int>(r.K);
  p.m_tiles = static_cast<int>(ceil_div(r.M, BM));
  p.n_tiles = static_cast<int>(ceil_div(r.N, BN));
  p.k_tiles = static_cast<int>(k_tiles);
  p.num_tiles = static_cast<int>(r.B) * p.m_tiles * p.n_tiles;
  p.sfa = use_a;
  p.sfb = use_b;
  p.sfa_rt = rt_rows(r.M);
  p.sfb_rt = rt_rows(r.N);
  p.ks4 = ks4;
  p.y = r.y;
  p.y_bf16 = r.y_bf16 ? 1 : 0;
  p.tma_store = make_output_map(&ty, r.y, r.y_bf16, r.B, r.M, r.N) ? 1 : 0;
  if (!p.tma_store) std::memset(&ty, 0, sizeof(ty));
  p.status = ctx->status;
  p.timeout_ns = wait_timeout_ns();
  if (nv) {
    // kind::mxf4nvf4: E2M1 = 1 for A and B, UE4M3 scales (bit 23 = 0), M = 128.
    p.idesc = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
    return launch_kernel<kNVF4, BN, 4>(ta, tb, ty, p, ctx, s);
  }
  // kind::mxf8f6f4: E4M3 = 0 / E5M2 = 1, UE8M0 scales (bit 23 = 1), M = 128.
  p.idesc = (f8_fmt(r.a_fmt) << 7) | (f8_fmt(r.b_fmt) << 10) | (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
            (static_cast<uint32_t>(BM >> 4) << 24);
  return launch_kernel<kMXF8, BN, 4>(ta, tb, ty, p, ctx, s);
}

cudaError_t launch_grouped_gemm(const GroupedGemmRequest& r, cudaStream_t s, std::string* why) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  // Kernel choice: CTA-pair 256 x 256 tiles when there is a tile for every
  // cluster, else one CTA per 128 x 128 tile.  BSMM_GROUPED_KERNEL=pair|single
  // overrides the choice (pair still needs N % 128 == 0 and K % 128 == 0).
  const char* force = std::getenv("BSMM_GROUPED_KERNEL");
  const bool want_pair = force && std::strcmp(force, "pair") == 0;
  const bool want_single = force && std::strcmp(force, "single") == 0;
  if (!want_single && (want_pair ? (r.N % 128 == 0 && r.K % 128 == 0) : grouped_pair_eligible(r.M, r.N, r.K, ctx)))
    return launch_grouped_gemm_pair(r, s, why);
  constexpr int BN = 128;
  CUtensorMap ta, tb, ty;
  if (!make_tmap_3d(&ta, r.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, r.K, r.M, 1, BK_BYTES, BM, true) ||
      !make_tmap_3d(&tb, r.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, r.K, r.N, 1, BK_BYTES, BN, true)) {
    *why = "cuTensorMapEncodeTiled failed for an operand";
    return cudaErrorInvalidValue;
  }
  Params p{};
  p.M = static_cast<int>(r.M);
  p.N = static_cast<int>(r.N);
  p.K = static_cast<int>(r.K);
  p.m_tiles = static_cast<int>(ceil_div(r.M, BM));
  p.n_tiles = static_cast<int>(ceil_div(r.N, BN));
  p.k_tiles = static_cast<int>(r.K / 128);
  p.num_tiles = p.m_tiles * p.n_tiles;
  p.a_scales = r.a_scales;
  p.b_scales = r.b_scales;
  p.kb = static_cast<int>(r.K / 128);
  // Split K: double the splits (up to 4) while the clusters still fit on the
  // SMs at once and each split keeps at least 16 K tiles.  Measured (device
  // time, CUDA-graph replay, us for 1 / 2 / 4 splits): m=237 n=k=4096
  // 16.2 / 15.2 / 27.0; m=512 n=2048 k=8192 27.4 / 21.2 / 32.8; m=256 n=1024
  // k=16384 49.2 / 31.2 / 22.6; m=349 n=k=2048 10.2 / 11.7 (8 K tiles a
  // split: the fixed costs of a cluster launch and of the cross-CTA sum
  // outweigh the shorter K loop).  Beyond the SM count, or past 4 splits, the
  // clusters run in more than one round and it is slower again.
  int splits = 1;
  while (splits < 4 && p.num_tiles * 2 * splits <= ctx->num_sms && p.k_tiles >= 32 * splits) splits *= 2;
  if (const char* fs = std::getenv("BSMM_GROUPED_SPLITK")) splits = std::max(1, std::min({8, std::atoi(fs), p.k_tiles}));
  p.kpb = static_cast<int>(ceil_div(p.k_tiles, splits));
  p.splits = static_cast<int>(ceil_div(p.k_tiles, p.kpb));  // no empty split
  p.y = r.y;
  p.y_bf16 = 0;
  p.tma_store = make_output_map(&ty, r.y, false, 1, r.M, r.N) ? 1 : 0;
  if (!p.tma_store) std::memset(&ty, 0, sizeof(ty));
  p.status = ctx->status;
  p.timeout_ns = wait_timeout_ns();
  // kind::f8f6f4: D = F32 (bits 4-5 = 1), A/B E4M3 = 0 / E5M2 = 1, K-major, N >> 3, M >> 4.
  p.idesc = (1u << 4) | (f8_fmt(r.a_fmt) << 7) | (f8_fmt(r.b_fmt) << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
            (static_cast<uint32_t>(BM >> 4) << 24);
  return launch_kernel<kF32Scale, BN, 4>(ta, tb, ty, p, ctx, s);
}

// ---------------------------------------------------------------------------
// Scratch for callers that cannot allocate device memory
// ---------------------------------------------------------------------------
// bsmm_gemm_noalloc keeps the tensor-core scale-factor atoms here instead of
// in a caller-provided workspace.  Every GPU that loads this library holds
// the array until the process exits.  All calls share it: each call rewrites
// every byte it reads (the relayout fills whole atoms), so nothing needs
// clearing, but calls whose kernels overlap on the GPU race on it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[BSMM_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_scratch_mutex;
void* g_scratch_addr[64] = {};
}  // namespace

cudaError_t launch_mx_gemm_noalloc(const MxGemmRequest& r, cudaStream_t s, std::string* why) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) {
    *why = "device ordinal beyond the library's table";
    return cudaErrorInvalidDevice;
  }
  void* scratch = nullptr;
  {
    // Set-up once per device, with that device current: host code only has
    // a stand-in for the array's name, so its device address is looked up.
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) {
        *why = std::string("cudaGetSymbolAddress of the scratch array failed: ") + cudaGetErrorString(e);
        return e;
      }
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  MxGemmRequest rr = r;
  rr.workspace = scratch;
  return launch_mx_gemm(rr, s, why);
}

cudaError_t launch_selftest_wait(uint64_t timeout_ns, cudaStream_t s) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  {
    TraceScope tr("selftest_wait", s);
    selftest_wait_kernel<<<1, 32, 0, s>>>(timeout_ns, ctx->status);
  }
  return cudaGetLastError();
}

}  // namespace bsmm
