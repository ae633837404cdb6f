// Block-scaled GEMMs on a CTA pair (tcgen05 .cta_group::2), 256 x 256 tiles.
//
// Two CTAs of a cluster share one 256 x 256 output tile: CTA r loads rows
// 128r..128r+127 of the A tile and of the B tile, the leader (rank 0) issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256), which reads both CTAs' shared
// memory and writes a 128 x 256 FP32 result into each CTA's tensor memory.
// N = 256 instructions keep the tensor pipe busy (N = 128 ones run it at about
// half rate), and per SM the operands are 32 KB per 128-byte K block for twice
// the FLOPs of a 128 x 128 tile on one CTA.  Five modes:
//
//   kPairF32   y = sum_kb sa[m,kb] * sb[n/128,kb] * (a . b over K block kb)
//              (atrex-bench #002 block_scaled_mm, Reference Implementation):
//              kind::f8f6f4, one FP32 partial per 128-K block in one of two
//              256-column TMEM buffers, promoted into registers by the epilogue.
//   kPairMXF8  jax.nn.scaled_matmul with MXFP8 (Notes, cuDNN on Blackwell):
//              kind::mxf8f6f4.block_scale.block32, UE8M0 scale per 32 K.
//   kPairNVF4  the same with NVFP4: kind::mxf4nvf4.block_scale.block16, packed
//              E2M1 operands, UE4M3 scale per 16 K.
//   kPairMXF4  the same with MXFP4: kind::mxf4nvf4.block_scale.block32, UE8M0.
//   kPairI8    TensorTonic's INT8 per-channel matmul: int8 codes as bf16
//              (exact), kind::f16, FP32 partials of 16 K blocks (exact
//              integers below 2^24) added in int32 by the epilogue, then
//              y = (acc * s_x) * s_w.  The tiles of the last, partial wave
//              are split along K over the clusters that would idle; the
//              parts meet through int32 sums in the workspace.
// In the block-scaled modes the result accumulates over all of K in one
// 256-column TMEM buffer; each stage's scale-factor atoms are copied into TMEM
// with tcgen05.cp.cta_group::2, which moves each CTA's own shared memory into
// its own tensor memory, so each CTA holds the scales of its 128 A rows and of
// all 256 B rows.
//
// Synchronization across the pair:
//   full[s]   in the leader, 2 arrivals (leader with expect_tx for both CTAs'
//             bytes, peer remotely); both CTAs' TMA loads complete on it.
//   empty[s]  in both CTAs; the leader's MMA commit multicasts to both.
//   tfull[i]  in both CTAs; multicast commit when a TMEM buffer is ready.
//   tempty[i] in the leader, 32 arrivals (16 epilogue warps of each CTA).
// Cross-CTA arrivals are relaxed: each follows tcgen05.wait::ld or a TMA issue,
// and a release at cluster scope costs the arriving thread ~1.2k cycles.
// Every wait is bounded; on expiry a CTA records the site and winds down.
//
// Epilogue: 16 warps per CTA (four per TMEM lane quarter).  Warp w reads lanes
// 32*(w%4).. (its 32 rows) and one 64-column quarter of the tile.  In kPairF32
// the per-K-block promotion (packed FP32 FMAs) is this kernel's bound, so the
// epilogue warps do nothing else: at a tile's end each writes its 32 x 64
// result into its own 8 KB of shared memory and moves on to the next tile,
// while the two otherwise idle control warps copy the staged results out with
// coalesced global stores (through the TMA unit those stores delayed the
// operand loads) and warm L2 with the next tile's A-scale rows.  The block-
// scaled modes drain the accumulator once per tile and hand it to the same
// copy warps in 128-byte column chunks.
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>
#include <atomic>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace bsmm {
namespace {

enum PairMode { kPairF32 = 0, kPairMXF8 = 1, kPairNVF4 = 2, kPairI8 = 3, kPairMXF4 = 4 };

constexpr int PM = 256, PN = 256;          // pair tile
constexpr int HALF = 128;                  // A rows and B rows per CTA
constexpr int KB = 128;                    // K bytes per stage
constexpr int THREADS = 640;               // 4 control warps + 16 epilogue warps
constexpr int EPI_WARPS = 16;
constexpr int EPI_COLS = 64;               // columns per epilogue thread
constexpr int TMEM_COLS = 512;
constexpr int GROUP_M = 8;
constexpr int A_BYTES = HALF * KB, B_BYTES = HALF * KB;

template <int MODE>
struct PCfg {
  // scale-factor atoms per K block per 128 rows: MXF8 1 (128 K / 32), NVF4 4
  // (256 K / 16), MXF4 2 (256 K / 32)
  static constexpr int ATOMS = MODE == kPairMXF8 ? 1 : (MODE == kPairNVF4 ? 4 : (MODE == kPairMXF4 ? 2 : 0));
  static constexpr int STAGES = MODE == kPairF32 ? 3 : 4;
  // output staging per epilogue warp: 32 rows x 128 bytes per 32-column chunk
  // (kPairF32 stages both chunks of a tile; kPairI8's TMA stores reuse one;
  // the block-scaled modes stage STG_ROWS rows of one chunk at a time)
  // Rows per staging round in the block-scaled modes: NVFP4's scale blocks
  // leave room for 8 (1 KB per warp), the others stage all 32 at once.
  static constexpr int STG_ROWS = MODE == kPairNVF4 ? 8 : 32;
  static constexpr int STG_PER_WARP = MODE == kPairF32 ? 8192 : (ATOMS > 0 ? STG_ROWS * 128 : 4096);
  // Scale factors per stage, in 512-byte slots: this CTA's 128 A rows, ATOMS
  // atoms skewed by lane quarter over ATOMS + 3 slots (a single atom in one
  // slot); all 256 B rows, 2 ATOMS atoms, for NVFP4 each four times over
  // (every lane quarter reads all of B's scales), which costs shared memory
  // but halves B's copies.
  static constexpr bool B_REPL = ATOMS > 0 && pair_b_replicated(ATOMS);
  static constexpr int SFA_SLOTS = ATOMS == 0 ? 0 : pair_sfa_slots(ATOMS);
  static constexpr int SFB_SLOTS = ATOMS == 0 ? 0 : pair_sfb_slots(ATOMS);
  static constexpr int SFA_BYTES = SFA_SLOTS * 512;
  static constexpr int SFB_BYTES = SFB_SLOTS * 512;
  static constexpr int SF_BYTES = SFA_BYTES + SFB_BYTES;
  static constexpr int STAGE_TX = A_BYTES + B_BYTES + SF_BYTES;  // per CTA
  static constexpr int NACC = (MODE == kPairF32 || MODE == kPairI8) ? 2 : 1;
  static constexpr int SF_COL0 = NACC * PN;
  static constexpr int SFA_COLS = ATOMS * 4;
  static constexpr int SFB_COLS = 2 * ATOMS * 4;
  static constexpr int SF_COLS = SFA_COLS + SFB_COLS;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_STG = (OFF_SF + STAGES * SF_BYTES + 1023) / 1024 * 1024;
  static constexpr int OFF_BAR = OFF_STG + EPI_WARPS * STG_PER_WARP;
  static constexpr int N_BARS = 2 * STAGES + 2 * NACC + 3;
  static constexpr int SMEM = OFF_BAR + N_BARS * 8 + 16 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(SF_COL0 + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
};

enum Site { kSiteProducer = 11, kSiteMmaTmem = 12, kSiteMmaFull = 13, kSiteEpilogue = 14, kSiteDrain = 15,
            kSiteDone = 16, kSiteStore = 17, kSiteStaging = 18 };

struct PairParams {
  int M, N, K;
  int batches;
  int m_tiles, n_tiles, k_tiles;  // tiles of 256 x 256, K blocks of 128 bytes
  int num_tiles;                  // over all batches
  // kPairF32
  const float* a_scales;
  const float* b_scales;
  int kb;  // K / 128
  // block-scaled: atoms [batch][row tile of 128][K atom] of 512 B, read
  // through 2-D tensor maps of 128-byte rows (an atom is 4 rows)
  int sfa_rt, sfb_rt, ks4;
  int y_bf16;
  float* y;  // output [B][M][N] (F32, or bf16 when y_bf16), written by the copy warps
  // kPairI8: per-row and per-column scales, K blocks per exact FP32 chunk,
  // whether the int32 sums are stored (through tmSFA)
  const float* sx;
  const float* sw;
  int chunk;
  int store_acc;
  uint32_t idesc;
  int* status;
  uint64_t timeout_ns;
};

// kPairI8's work units: first each tile from whole_tiles on as `split` K
// ranges of k_split K blocks, then tiles [0, whole_tiles) whole (num_units
// in all).  The parts come first so that the extra work of each part's end
// overlaps a whole tile's MMAs in the other TMEM buffer.  A part leaves its
// int32 sums in split_ws [tile - whole_tiles][part][32 warp slots][2048] and
// counts itself in split_cnt [tile - whole_tiles][32 warp slots]; the last
// part of a warp slot adds the others' sums and writes y.  (The other modes
// keep the plain parameters: a larger parameter block made the FP32-scale
// epilogue spill.)
struct PairSplitParams : PairParams {
  int32_t* split_ws;
  unsigned* split_cnt;
  int whole_tiles, split, k_split, num_units;
};
template <int MODE>
using PairArgs = std::conditional_t<MODE == kPairI8, PairSplitParams, PairParams>;

__device__ __forceinline__ void decode_pair_tile(const PairParams& p, int t, int& b, int& mb, int& nb) {
  const int per_batch = p.m_tiles * p.n_tiles;
  b = t / per_batch;
  const int r = t - b * per_batch;
  const int span = GROUP_M * p.n_tiles;
  const int g = r / span;
  const int within = r - g * span;
  const int rows = min(GROUP_M, p.m_tiles - g * GROUP_M);
  mb = g * GROUP_M + within % rows;
  nb = within / rows;
}

// Work unit u: tile t, K blocks [k0, k1), and the part's index (-1: whole tile).
struct PairUnit {
  int t, k0, k1, part;
};
// Only kPairI8 splits; the other modes' units are their tiles.
template <int MODE>
__device__ __forceinline__ PairUnit pair_unit(const PairArgs<MODE>& p, int u) {
  if constexpr (MODE == kPairI8) {
    const int parts = p.num_units - p.whole_tiles;
    if (u < parts) {
      const int part = u % p.split;
      const int k0 = part * p.k_split;
      return {p.whole_tiles + u / p.split, k0, min(p.k_tiles, k0 + p.k_split), part};
    }
    return {u - parts, 0, p.k_tiles, -1};
  }
  return {u, 0, p.k_tiles, -1};
}
template <int MODE>
__device__ __forceinline__ int pair_units(const PairArgs<MODE>& p) {
  if constexpr (MODE == kPairI8) return p.num_units;
  return p.num_tiles;
}

__device__ __forceinline__ uint32_t pack_bf16x2_pair(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Two int32 sums kept in the bits of a float2, plus two exact FP32 integers.
__device__ __forceinline__ float2 iadd_f2(float2 acc, uint32_t p0, uint32_t p1) {
  return make_float2(__int_as_float(__float_as_int(acc.x) + __float2int_rn(__uint_as_float(p0))),
                     __int_as_float(__float_as_int(acc.y) + __float2int_rn(__uint_as_float(p1))));
}

// A warp's 32 rows x 64 columns of 32-bit values leave through `map` as two
// 32 x 32 TMA stores from the warp's 4 KB staging buffer (128B-swizzled rows).
__device__ __forceinline__ void store_box_f32(const CUtensorMap* map, uint8_t* stg, const float2 (&acc)[EPI_COLS / 2],
                                              int col0, int row0, int z, int lane) {
#pragma unroll
  for (int c = 0; c < EPI_COLS / 32; ++c) {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 v0 = acc[16 * c + 2 * j], v1 = acc[16 * c + 2 * j + 1];
      const uint32_t off = lane * 128 + ((j ^ (lane & 7)) * 16);
      *reinterpret_cast<uint4*>(stg + off) =
          make_uint4(__float_as_uint(v0.x), __float_as_uint(v0.y), __float_as_uint(v1.x), __float_as_uint(v1.y));
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(map, stg, col0 + 32 * c, row0, z);
      bulk_commit();
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmSFA,
                 const __grid_constant__ CUtensorMap tmSFB, const PairArgs<MODE> p) {
  using C = PCfg<MODE>;
  constexpr int STAGES = C::STAGES;
  constexpr int NACC = C::NACC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* sSF = smem + C::OFF_SF;
  uint8_t* stg = smem + C::OFF_STG;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + NACC;
  uint64_t* done = tempty + NACC;
  uint64_t* stg_full = done + 1;   // kPairF32: the 16 epilogue warps staged a tile
  uint64_t* stg_empty = done + 2;  // kPairF32: both copy warps emptied the staging
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int never_abort_storage = 0;
  volatile int* never_abort = &never_abort_storage;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 2);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 2 * EPI_WARPS);
    }
    mbar_init(done, 1);
    mbar_init(stg_full, EPI_WARPS);
    mbar_init(stg_empty, 2);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialized before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // 640 threads launch with 96 registers each (61440); the control warpgroup
  // gives up 40 of its 96, the four epilogue warpgroups take 104 each:
  // 128 x 56 + 512 x 104 = 60416 <= 61440.
  if (warp < 4) {
    setmaxnreg_dec<56>();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------- producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int u = cid; ok && u < pair_units<MODE>(p); u += ncl) {
        const PairUnit w = pair_unit<MODE>(p, u);
        int b, mb, nb;
        decode_pair_tile(p, w.t, b, mb, nb);
        for (int kt = w.k0; kt < w.k1; ++kt) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.status, kSiteProducer)) {
            ok = false;
            break;
          }
          const uint32_t full_leader = mapa_shared(smem_u32(&full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_TX);
          tma_load_3d_pair(sA + stage * A_BYTES, &tmA, full_leader, kt * KB, mb * PM + rank * HALF, b);
          tma_load_3d_pair(sB + stage * B_BYTES, &tmB, full_leader, kt * KB, nb * PN + rank * HALF, b);
          if constexpr (C::ATOMS > 0) {  // block-scaled modes: this stage's scale-factor atoms
            // one block of slots per operand, as rows of 128 bytes: A's for
            // (batch, row tile, K tile), B's for (batch, row-tile pair, K tile)
            uint8_t* sf = sSF + stage * C::SF_BYTES;
            const int a_row = 4 * C::SFA_SLOTS * ((b * p.sfa_rt + 2 * mb + static_cast<int>(rank)) * p.k_tiles + kt);
            tma_load_3d_pair(sf, &tmSFA, full_leader, 0, a_row, 0);
            if constexpr (C::B_REPL) {
              const int b_row = 4 * C::SFB_SLOTS * ((b * (p.sfb_rt / 2) + nb) * p.k_tiles + kt);
              tma_load_3d_pair(sf + C::SFA_BYTES, &tmSFB, full_leader, 0, b_row, 0);
            } else {  // atom j of row tile rt of batch b: rows 4 ((b rt_count + rt) ks4 + j) ..
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                const int b_row = 4 * ((b * p.sfb_rt + 2 * nb + r) * p.ks4 + kt * C::ATOMS);
                tma_load_3d_pair(sf + C::SFA_BYTES + r * C::ATOMS * 512, &tmSFB, full_leader, 0, b_row, 0);
              }
            }
          }
          if (!leader) mbar_arrive_cluster(full_leader);
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every stage this CTA filled must have been released by the leader's
      // MMA (its multicast arrivals on our empty[] have landed) before any
      // CTA of the pair winds down.
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          mbar_wait(&empty[s], (last_par >> s) & 1u, p.timeout_ns, ok ? never_abort : abort_flag, p.status,
                    kSiteDrain);
      if (leader) {
        for (int s = 0; s < STAGES; ++s)
          if ((issued >> s) & 1u)
            mbar_wait(&full[s], (last_par >> s) & 1u, p.timeout_ns, never_abort, p.status, kSiteDrain);
      } else if (!ok) {
        // The peer cannot observe the leader's barrier; after giving up, give
        // its own copies in flight time to land before the CTA winds down.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    } else if (warp == 1 && lane == 0 && leader) {
      // ------------------------------------------------------- MMA issuer (leader)
      if constexpr (C::ATOMS > 0) {
        // Block-scaled: one accumulator over all of K per tile; each stage's
        // scale factors are copied into tensor memory ahead of its MMAs.
        int stage = 0;
        uint32_t phase = 0, tph = 0;
        bool ok = true;
        for (int t = cid; ok && t < p.num_tiles; t += ncl) {
          if (!mbar_wait(&tempty[0], tph ^ 1u, p.timeout_ns, abort_flag, p.status, kSiteMmaTmem)) break;
          tc_fence_after();
          for (int kt = 0; kt < p.k_tiles; ++kt) {
            if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.status, kSiteMmaFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // descriptors for the stage's first bytes, stepped by constants
            const uint64_t a_d = smem_desc(smem_u32(sA + stage * A_BYTES), 16, 1024, 2);
            const uint64_t b_d = smem_desc(smem_u32(sB + stage * B_BYTES), 16, 1024, 2);
            const uint32_t sf_s = smem_u32(sSF + stage * C::SF_BYTES);
            const uint32_t sfa_t = tmem + static_cast<uint32_t>(C::SF_COL0 + stage * C::SF_COLS);
            const uint32_t sfb_t = sfa_t + C::SFA_COLS;
            // A atom i (K sub-block i) -> columns sfa_t + 4i; B atom (row tile
            // r, K sub-block i) -> columns sfb_t + 4*(2i + r).  In each atom's
            // 4 columns, lane 32q + m0 column j holds row 32j + m0's scales.
            // The MMA reads A's rows 32q.. from lane quarter q's column q
            // only, but every quarter reads all 256 of B's rows.  A 128-lane
            // copy of 8 columns (core matrices of 8 rows x 16 bytes, 128
            // bytes apart; second 16 bytes LBO on) fills two atoms at once:
            //  - A: row 32q + m0's words sit at slot a + q, so with LBO one
            //    slot the copy's rows 32q.. read atoms 2c and 2c + 1 from
            //    slots 2c + q and 2c + 1 + q;
            //  - B (NVFP4): each atom is stored four times (slot 4a + q for
            //    quarter q), so with LBO four slots quarter q reads its own.
            // One copy per pair of atoms instead of one per atom.
            if constexpr (C::ATOMS == 1) {  // a single A atom, replicated by the copy
              tc_cp_sf_pair(sfa_t, smem_desc(sf_s, 0, 128, 0));
            } else {
              const uint64_t sfa_d = smem_desc(sf_s, 512, 128, 0);
#pragma unroll
              for (int c = 0; c < C::ATOMS / 2; ++c) tc_cp_sf_pair_x2(sfa_t + 8 * c, desc_add(sfa_d, 1024 * c));
            }
            if constexpr (C::B_REPL) {
              const uint64_t sfb_d = smem_desc(sf_s + C::SFA_BYTES, 2048, 128, 0);
#pragma unroll
              for (int i = 0; i < C::ATOMS; ++i) tc_cp_sf_pair_x2(sfb_t + 8 * i, desc_add(sfb_d, 4096 * i));
            } else {  // one copy per atom, replicated to the four lane quarters by the copy
              const uint64_t sfb_d = smem_desc(sf_s + C::SFA_BYTES, 0, 128, 0);
#pragma unroll
              for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int i = 0; i < C::ATOMS; ++i)
                  tc_cp_sf_pair(sfb_t + 4 * (2 * i + r), desc_add(sfb_d, 512 * (r * C::ATOMS + i)));
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = desc_add(a_d, 32 * k);
              const uint64_t bd = desc_add(b_d, 32 * k);
              const uint32_t acc = (kt > 0 || k > 0) ? 1u : 0u;
              if constexpr (MODE == kPairMXF8) {  // one atom, byte k of each row's word
                const uint32_t idesc = p.idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
                mma_mxf8_pair(tmem, ad, bd, idesc, sfa_t, sfb_t, acc);
              } else if constexpr (MODE == kPairMXF4) {  // atom k/2, bytes 2(k%2) .. 2(k%2)+1
                const uint32_t id = static_cast<uint32_t>(2 * (k & 1));
                mma_mxf4_pair(tmem, ad, bd, p.idesc | (id << 4) | (id << 29), sfa_t + 4 * (k >> 1),
                              sfb_t + 8 * (k >> 1), acc);
              } else {  // one atom per instruction
                mma_nvf4_pair(tmem, ad, bd, p.idesc, sfa_t + 4 * k, sfb_t + 8 * k, acc);
              }
            }
            tc_commit_pair_mc(&empty[stage], 0x3);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit_pair_mc(&tfull[0], 0x3);
          tph ^= 1u;
        }
      } else if constexpr (MODE == kPairI8) {
        // one TMEM buffer per chunk of p.chunk K blocks (exact FP32 integer
        // sums), alternating between the two buffers
        int stage = 0, tb = 0;
        uint32_t phase = 0, tph = 0;
        bool ok = true;
        for (int u = cid; ok && u < pair_units<MODE>(p); u += ncl) {
          const PairUnit w = pair_unit<MODE>(p, u);
          for (int k0 = w.k0; ok && k0 < w.k1; k0 += p.chunk) {
            if (!mbar_wait(&tempty[tb], tph ^ 1u, p.timeout_ns, abort_flag, p.status, kSiteMmaTmem)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem + static_cast<uint32_t>(tb * PN);
            const int k1 = k0 + p.chunk < w.k1 ? k0 + p.chunk : w.k1;
            for (int kt = k0; kt < k1; ++kt) {
              if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.status, kSiteMmaFull)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t a_d = smem_desc(smem_u32(sA + stage * A_BYTES), 16, 1024, 2);
              const uint64_t b_d = smem_desc(smem_u32(sB + stage * B_BYTES), 16, 1024, 2);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f16_pair(d, desc_add(a_d, 32 * k), desc_add(b_d, 32 * k), p.idesc, (kt > k0 || k > 0) ? 1u : 0u);
              tc_commit_pair_mc(&empty[stage], 0x3);
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            tc_commit_pair_mc(&tfull[tb], 0x3);
            if (++tb == NACC) {
              tb = 0;
              tph ^= 1u;
            }
          }
        }
      } else {
        // kPairF32: every K block's partial gets a TMEM buffer of its own
        int stage = 0, tb = 0;
        uint32_t phase = 0, tph = 0;
        bool ok = true;
        for (int t = cid; ok && t < p.num_tiles; t += ncl) {
          for (int kt = 0; kt < p.k_tiles; ++kt) {
            if (!mbar_wait(&tempty[tb], tph ^ 1u, p.timeout_ns, abort_flag, p.status, kSiteMmaTmem) ||
                !mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.status, kSiteMmaFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t a_d = smem_desc(smem_u32(sA + stage * A_BYTES), 16, 1024, 2);
            const uint64_t b_d = smem_desc(smem_u32(sB + stage * B_BYTES), 16, 1024, 2);
            const uint32_t d = tmem + static_cast<uint32_t>(tb * PN);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f8f6f4_pair(d, desc_add(a_d, 32 * k), desc_add(b_d, 32 * k), p.idesc, k > 0 ? 1u : 0u);
            tc_commit_pair_mc(&empty[stage], 0x3);
            tc_commit_pair_mc(&tfull[tb], 0x3);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            if (++tb == NACC) {
              tb = 0;
              tph ^= 1u;
            }
          }
        }
      }
      tc_commit_pair_mc(done, 0x1);
      mbar_wait(done, 0, p.timeout_ns, never_abort, p.status, kSiteDone);
    } else if (C::ATOMS > 0 && warp >= 2) {
      // ------------------------------------------------ output copy (both CTAs)
      // Block-scaled modes: the epilogue stages each tile's result STG_ROWS
      // rows of one 128-byte column chunk at a time (FP32: 2 chunks, bf16: 1,
      // times 32 / STG_ROWS row groups); warp 2 copies epilogue warps 0-7,
      // warp 3 warps 8-15, four whole 128-byte lines per instruction.  The
      // copies trickle out during the next tile.  (Tile-end TMA stores held
      // up the operand loads queued behind them.)
      constexpr int GROUPS = 32 / C::STG_ROWS;
      const int cw = warp - 2;
      const int rounds = (p.y_bf16 ? 1 : 2) * GROUPS;
      uint32_t sph = 0;
      bool ok = true;
      for (int t = cid; ok && t < p.num_tiles; t += ncl) {
        int b, mb, nb;
        decode_pair_tile(p, t, b, mb, nb);
        for (int c = 0; c < rounds; ++c) {
          if (!mbar_wait(stg_full, sph, p.timeout_ns, abort_flag, p.status, kSiteStore)) {
            ok = false;
            break;
          }
          for (int i = 0; i < EPI_WARPS / 2; ++i) {
            const int ew = cw * (EPI_WARPS / 2) + i;
            const int row0 = mb * PM + static_cast<int>(rank) * HALF + (ew & 3) * 32 + C::STG_ROWS * (c % GROUPS);
            const int col0 = nb * PN + (ew >> 2) * EPI_COLS + 32 * (c / GROUPS);
            const uint8_t* src = stg + ew * C::STG_PER_WARP;
            const int u = lane & 7;
            const int col = col0 + (p.y_bf16 ? 8 : 4) * u;  // this lane's 16 bytes
            if (row0 >= p.M || col >= p.N) continue;       // N * size % 16 == 0: all in or all out
#pragma unroll
            for (int j = 0; j < C::STG_ROWS / 4; ++j) {
              const int r = 4 * j + (lane >> 3);
              const uint4 v = *reinterpret_cast<const uint4*>(src + r * 128 + ((u ^ (r & 7)) * 16));
              if (row0 + r < p.M) {
                const size_t e = (static_cast<size_t>(b) * p.M + row0 + r) * p.N + col;
                uint4* dst = p.y_bf16 ? reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.y) + e)
                                      : reinterpret_cast<uint4*>(p.y + e);
                __stcs(dst, v);  // streaming: y is not read again
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(stg_empty);
          sph ^= 1u;
        }
      }
    } else if (MODE == kPairF32 && warp >= 2) {
      // ------------------------------------------------ output copy (both CTAs)
      // Warp 2 copies the staging of epilogue warps 0-7, warp 3 that of 8-15:
      // per 32-column chunk, each instruction moves four rows of 128 bytes
      // (lane l: row 4j + l/8, 16-byte unit l%8), so every global store
      // writes four whole 128-byte lines.
      const int cw = warp - 2;
      uint32_t sph = 0;
      for (int t = cid; t < p.num_tiles; t += ncl) {
        int b, mb, nb;
        decode_pair_tile(p, t, b, mb, nb);
        if (t + ncl < p.num_tiles) {  // the A-scale rows of this CTA's next tile, 64 per warp
          int b2, mb2, nb2;
          decode_pair_tile(p, t + ncl, b2, mb2, nb2);
          for (int i = lane; i < 64; i += 32) {
            const int r = mb2 * PM + static_cast<int>(rank) * HALF + cw * 64 + i;
            if (r < p.M) {
              const char* pa = reinterpret_cast<const char*>(p.a_scales + static_cast<size_t>(r) * p.kb);
              for (int off = 0; off < p.kb * 4; off += 128) prefetch_l2(pa + off);
            }
          }
        }
        if (!mbar_wait(stg_full, sph, p.timeout_ns, abort_flag, p.status, kSiteStore)) break;
        for (int i = 0; i < EPI_WARPS / 2; ++i) {
          const int ew = cw * (EPI_WARPS / 2) + i;
          const int row0 = mb * PM + static_cast<int>(rank) * HALF + (ew & 3) * 32;
          const int col0 = nb * PN + (ew >> 2) * EPI_COLS;
          if (row0 >= p.M || col0 >= p.N) continue;
          const uint8_t* src = stg + ew * C::STG_PER_WARP;
          const int u = lane & 7;
#pragma unroll 1
          for (int j = 0; j < 8; ++j) {
            const int r = 4 * j + (lane >> 3);
            const uint32_t soff = r * 128 + ((u ^ (r & 7)) * 16);
            const uint4 v0 = *reinterpret_cast<const uint4*>(src + soff);
            const uint4 v1 = *reinterpret_cast<const uint4*>(src + 4096 + soff);
            if (row0 + r < p.M) {
              float* dst = p.y + (static_cast<size_t>(b) * p.M + row0 + r) * p.N + col0 + 4 * u;
              *reinterpret_cast<uint4*>(dst) = v0;
              *reinterpret_cast<uint4*>(dst + 32) = v1;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(stg_empty);
        sph ^= 1u;
      }
    }
  } else {
    setmaxnreg_inc<104>();
    // --------------------------------------------------------- epilogue (both CTAs)
    constexpr int COLS = EPI_COLS;
    const int ew = warp - 4;
    const int q = warp & 3;   // TMEM lane quarter = the warp's 32 rows
    const int g = ew >> 2;    // 64-column quarter of the tile
    uint8_t* my_stg = stg + ew * C::STG_PER_WARP;
    uint32_t sph = 0;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int tb = 0;
    uint32_t tph = 0;
    for (int u = cid; u < pair_units<MODE>(p); u += ncl) {
      const PairUnit w = pair_unit<MODE>(p, u);
      int b, mb, nb;
      decode_pair_tile(p, w.t, b, mb, nb);
      const int row0 = mb * PM + static_cast<int>(rank) * HALF + q * 32;
      const int row = row0 + lane;
      const int col0 = nb * PN + g * COLS;
      const bool col_ok = col0 < p.N;
      // column pairs: the promotion runs as packed two-lane FP32 FMAs, each
      // lane an ordinary round-to-nearest fused multiply-add
      float2 acc[COLS / 2];
      bool ok = true;
      if constexpr (MODE == kPairF32) {
        // Rows past M compute values nobody stores: they read row M-1's
        // scales, so no lane needs a predicate or a 64-bit pointer in the loop
        // (the epilogue runs at the edge of its registers; measured 3% faster).
        // M * K / 128 scales fit 32 bits, as M * K bytes of codes fit in memory.
        const uint32_t sa_off = static_cast<uint32_t>(min(row, p.M - 1)) * static_cast<uint32_t>(p.kb);
        const uint32_t sb_off = static_cast<uint32_t>(col_ok ? col0 / 128 : 0) * static_cast<uint32_t>(p.kb);
#pragma unroll
        for (int i = 0; i < COLS / 2; ++i) acc[i] = make_float2(0.f, 0.f);
        float sa_next = __ldg(p.a_scales + sa_off);
        float sb_next = __ldg(p.b_scales + sb_off);
        const uint32_t tad0 = tmem + lane_base + static_cast<uint32_t>(g * COLS);
        // One K block: its scale product (the next block's scales loaded
        // meanwhile), the wait for its partial in TMEM buffer buf, the
        // promotion, and the buffer handed back to the issuer.
        auto promote = [&](int buf, int kt) -> bool {
          const float s = sa_next * sb_next;
          const float2 s2 = make_float2(s, s);
          if (kt + 1 < p.k_tiles) {
            sa_next = __ldg(p.a_scales + sa_off + kt + 1);
            sb_next = __ldg(p.b_scales + sb_off + kt + 1);
          }
          if (!mbar_wait(&tfull[buf], tph, p.timeout_ns, abort_flag, p.status, kSiteEpilogue)) return false;
          tc_fence_after();
          const uint32_t taddr = tad0 + static_cast<uint32_t>(buf * PN);
#pragma unroll
          for (int h = 0; h < COLS / 32; ++h) {  // two loads in flight per wait
            uint32_t r0[16], r1[16];
            tmem_ld16(taddr + 32 * h, r0);
            tmem_ld16(taddr + 32 * h + 16, r1);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              acc[16 * h + j] = __ffma2_rn(make_float2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1])), s2,
                                           acc[16 * h + j]);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              acc[16 * h + 8 + j] = __ffma2_rn(
                  make_float2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1])), s2, acc[16 * h + 8 + j]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[buf]), 0));
          return true;
        };
        if ((p.k_tiles & 1) == 0 && tb == 0) {
          // K blocks in pairs, buffer 0 then buffer 1: the buffer index and
          // its addresses are constants (1-2% faster than the general loop)
          for (int kt = 0; kt < p.k_tiles; kt += 2) {
            if (!promote(0, kt) || !promote(1, kt + 1)) {
              ok = false;
              break;
            }
            tph ^= 1u;
          }
        } else {
          for (int kt = 0; kt < p.k_tiles; ++kt) {
            if (!promote(tb, kt)) {
              ok = false;
              break;
            }
            if (++tb == NACC) {
              tb = 0;
              tph ^= 1u;
            }
          }
        }
      } else if constexpr (MODE == kPairI8) {
        // int32 sums in the bits of acc: each chunk's FP32 partial is an
        // exact integer below 2^24, converted exactly and added
#pragma unroll
        for (int i = 0; i < COLS / 2; ++i) acc[i] = make_float2(0.f, 0.f);  // int 0 has the same bits
        for (int kt = w.k0; kt < w.k1; kt += p.chunk) {
          if (!mbar_wait(&tfull[tb], tph, p.timeout_ns, abort_flag, p.status, kSiteEpilogue)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(tb * PN + g * COLS);
#pragma unroll
          for (int h = 0; h < COLS / 32; ++h) {
            uint32_t r0[16], r1[16];
            tmem_ld16(taddr + 32 * h, r0);
            tmem_ld16(taddr + 32 * h + 16, r1);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              acc[16 * h + j] = iadd_f2(acc[16 * h + j], r0[2 * j], r0[2 * j + 1]);
              acc[16 * h + 8 + j] = iadd_f2(acc[16 * h + 8 + j], r1[2 * j], r1[2 * j + 1]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[tb]), 0));
          if (++tb == NACC) {
            tb = 0;
            tph ^= 1u;
          }
        }
      } else {
        if (!mbar_wait(&tfull[0], tph, p.timeout_ns, abort_flag, p.status, kSiteEpilogue)) {
          ok = false;
        } else {
          tc_fence_after();
          const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(g * COLS);
#pragma unroll
          for (int h = 0; h < COLS / 32; ++h) {
            uint32_t r0[16], r1[16];
            tmem_ld16(taddr + 32 * h, r0);
            tmem_ld16(taddr + 32 * h + 16, r1);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              acc[16 * h + j] = make_float2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1]));
              acc[16 * h + 8 + j] = make_float2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1]));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[0]), 0));
          tph ^= 1u;
        }
      }
      if (!ok) break;
      if constexpr (MODE == kPairF32) {
        // the previous tile's staging has been copied out (a tile ago)
        if (!mbar_wait(stg_empty, sph ^ 1u, p.timeout_ns, abort_flag, p.status, kSiteStaging)) break;
        if (row0 < p.M && col_ok) {
#pragma unroll
          for (int c = 0; c < COLS / 32; ++c)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float2 v0 = acc[16 * c + 2 * j], v1 = acc[16 * c + 2 * j + 1];
              const uint32_t off = c * 4096 + lane * 128 + ((j ^ (lane & 7)) * 16);
              *reinterpret_cast<uint4*>(my_stg + off) = make_uint4(__float_as_uint(v0.x), __float_as_uint(v0.y),
                                                                   __float_as_uint(v1.x), __float_as_uint(v1.y));
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(stg_full);
        sph ^= 1u;
        continue;
      }
      if constexpr (C::ATOMS > 0) {
        // stage the tile's result for the copy warps: per round, the
        // STG_ROWS rows of one row group of one 128-byte column chunk
        // (128 bytes a row, 16-byte units rotated by row)
        constexpr int GROUPS = 32 / C::STG_ROWS;
        const bool in_y = row0 < p.M && col_ok;
        const int rounds = (p.y_bf16 ? 1 : 2) * GROUPS;
        for (int rd = 0; rd < rounds; ++rd) {
          const int c = rd / GROUPS, rg = rd % GROUPS;
          if (!mbar_wait(stg_empty, sph ^ 1u, p.timeout_ns, abort_flag, p.status, kSiteStaging)) {
            ok = false;
            break;
          }
          if (in_y && lane / C::STG_ROWS == rg) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint4 v;
              if (p.y_bf16) {
                const float2* a = &acc[4 * j];
                v = make_uint4(pack_bf16x2_pair(a[0].x, a[0].y), pack_bf16x2_pair(a[1].x, a[1].y),
                               pack_bf16x2_pair(a[2].x, a[2].y), pack_bf16x2_pair(a[3].x, a[3].y));
              } else {
                const float2 a0 = acc[16 * c + 2 * j], a1 = acc[16 * c + 2 * j + 1];
                v = make_uint4(__float_as_uint(a0.x), __float_as_uint(a0.y), __float_as_uint(a1.x),
                               __float_as_uint(a1.y));
              }
              *reinterpret_cast<uint4*>(my_stg + (lane % C::STG_ROWS) * 128 + ((j ^ (lane & 7)) * 16)) = v;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(stg_full);
          sph ^= 1u;
        }
        if (!ok) break;
        continue;
      }
      if (row0 >= p.M || !col_ok) continue;  // this warp's box lies outside y
      if constexpr (MODE == kPairI8) {
        const PairUnit wu = pair_unit<MODE>(p, u);  // recomputed: not live across the K loop
        if (wu.part >= 0) {
          // One K range of a split tile: this warp's 32 x 64 int32 sums go
          // to the part's slot; the part that counts last for this warp slot
          // adds the other parts' sums (integer adds: any order is exact)
          // and writes y.  No part waits for another.  A warp slot's 8 KB
          // hold 16-byte unit i of lane l at (32 i + l), so that every store
          // and load instruction moves 512 contiguous bytes.
          const int tail = wu.t - p.whole_tiles;
          const int slot = static_cast<int>(rank) * EPI_WARPS + ew;
          int32_t* slot_ws = p.split_ws + static_cast<size_t>(tail) * p.split * (PM * PN) + slot * (32 * COLS);
          int4* mine = reinterpret_cast<int4*>(slot_ws + static_cast<size_t>(wu.part) * (PM * PN)) + lane;
#pragma unroll
          for (int i = 0; i < COLS / 4; ++i)
            mine[32 * i] = make_int4(__float_as_int(acc[2 * i].x), __float_as_int(acc[2 * i].y),
                                     __float_as_int(acc[2 * i + 1].x), __float_as_int(acc[2 * i + 1].y));
          __threadfence();
          __syncwarp();
          unsigned before = 0;
          if (lane == 0) before = atomicAdd(p.split_cnt + tail * (2 * EPI_WARPS) + slot, 1u);
          before = __shfl_sync(0xffffffffu, before, 0);
          if (before != static_cast<unsigned>(p.split - 1)) continue;
          __threadfence();
          for (int o = 0; o < p.split; ++o) {
            if (o == wu.part) continue;
            const int4* other = reinterpret_cast<const int4*>(slot_ws + static_cast<size_t>(o) * (PM * PN)) + lane;
#pragma unroll
            for (int i = 0; i < COLS / 4; ++i) {
              const int4 v = __ldcg(other + 32 * i);
              acc[2 * i] = make_float2(__int_as_float(__float_as_int(acc[2 * i].x) + v.x),
                                       __int_as_float(__float_as_int(acc[2 * i].y) + v.y));
              acc[2 * i + 1] = make_float2(__int_as_float(__float_as_int(acc[2 * i + 1].x) + v.z),
                                           __int_as_float(__float_as_int(acc[2 * i + 1].y) + v.w));
            }
          }
        }
        if (p.store_acc) store_box_f32(&tmSFA, my_stg, acc, col0, row0, b, lane);  // int32 bits as they are
        // y = (float(acc) * s_x[row]) * s_w[col], in that order
        const float sxr = row < p.M ? __ldg(p.sx + row) : 0.f;
#pragma unroll
        for (int i = 0; i < COLS / 2; ++i) {
          const int c = col0 + 2 * i;
          const float w0 = c < p.N ? __ldg(p.sw + c) : 0.f;
          const float w1 = c + 1 < p.N ? __ldg(p.sw + c + 1) : 0.f;
          acc[i] = make_float2((static_cast<float>(__float_as_int(acc[i].x)) * sxr) * w0,
                               (static_cast<float>(__float_as_int(acc[i].y)) * sxr) * w1);
        }
        store_box_f32(&tmY, my_stg, acc, col0, row0, b, lane);
        continue;
      }
    }
    if (lane == 0) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no signal may target a CTA that has exited
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// max co-resident clusters per mode and device, found on first use (calls
// from several host threads may race to fill it in; they find the same value)
std::atomic<int> g_pair_clusters[5][64] = {};

template <int MODE>
cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const CUtensorMap& tsa,
                        const CUtensorMap& tsb, const PairArgs<MODE>& p, const DeviceCtx* ctx, cudaStream_t s,
                        std::string* why) {
  using C = PCfg<MODE>;
  auto kern = tc_gemm_pair<MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until the block's launch registers cover the split
  // (control warpgroup 56, four epilogue warpgroups 104): a build whose
  // register count fell below the one the split was sized for would wait
  // forever, so it is refused here instead.
  cudaFuncAttributes fa{};
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * THREADS < 128 * 56 + 32 * EPI_WARPS * 104) {
    *why = "pair GEMM built with " + std::to_string(fa.numRegs) + " registers a thread, fewer than its register split needs";
    return cudaErrorInvalidConfiguration;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (ctx->device < 0 || ctx->device >= 64) {
    *why = "device ordinal beyond the library's table";
    return cudaErrorInvalidDevice;
  }
  int max_clusters = g_pair_clusters[MODE][ctx->device].load(std::memory_order_relaxed);
  if (max_clusters == 0) {
    cfg.gridDim = dim3(2 * (ctx->num_sms / 2));
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) {
      *why = "no cluster of two CTAs fits on this device";
      return cudaErrorInvalidConfiguration;
    }
    max_clusters = n;
    g_pair_clusters[MODE][ctx->device].store(n, std::memory_order_relaxed);
  }
  PairArgs<MODE> q = p;
  int units = q.num_tiles;
  if constexpr (MODE == kPairI8) {
    q.whole_tiles = q.num_units = q.num_tiles;
    q.split = 1;
    q.k_split = q.k_tiles;
    if (q.split_ws && q.split_cnt) {
      // The last wave's tiles (all of them when there are fewer tiles than
      // clusters) split their K blocks over the clusters that would idle:
      // S = clusters / tail parts, at most kSplitMax, each a whole number of
      // exact chunks where K allows.
      const int tail = q.num_tiles % max_clusters;
      int split = tail > 0 ? std::min(kSplitMax, max_clusters / tail) : 1;
      if (split >= 2) {
        int k_split = static_cast<int>(ceil_div(q.k_tiles, split));
        if (k_split > q.chunk) k_split = static_cast<int>(ceil_div(k_split, q.chunk)) * q.chunk;
        split = static_cast<int>(ceil_div(q.k_tiles, k_split));
        if (split >= 2 && tail <= kSplitTilesMax && tail * split <= kSplitUnitsMax) {
          q.whole_tiles = q.num_tiles - tail;
          q.split = split;
          q.k_split = k_split;
          q.num_units = q.whole_tiles + tail * split;
        }
      }
    }
    units = q.num_units;
  }
  const int clusters = std::max(1, std::min(units, max_clusters));
  cfg.gridDim = dim3(2 * clusters);
  {
    constexpr const char* kNames[] = {"tc_gemm_pair<F32>", "tc_gemm_pair<MXF8>", "tc_gemm_pair<NVF4>",
                                      "tc_gemm_pair<I8>", "tc_gemm_pair<MXF4>"};
    TraceScope tr(kNames[MODE], s);
    e = cudaLaunchKernelEx(&cfg, kern, ta, tb, ty, tsa, tsb, q);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

uint32_t f8_code(int dtype) { return dtype == BSMM_E5M2 ? 1u : 0u; }

// Tiles of 256 x 256 over all batches.
int64_t pair_tiles(int64_t B, int64_t M, int64_t N) { return B * ceil_div(M, PM) * ceil_div(N, PN); }

}  // namespace

bool grouped_pair_eligible(int64_t M, int64_t N, int64_t K, const DeviceCtx* ctx) {
  // The pair kernel stores through TMA (N*4 % 16 == 0 holds: N % 128 == 0)
  // and wants at least one 256 x 256 tile per cluster.
  return K % 128 == 0 && N % 128 == 0 && pair_tiles(1, M, N) >= ctx->num_sms / 2;
}

cudaError_t launch_grouped_gemm_pair(const GroupedGemmRequest& r, cudaStream_t s, std::string* why) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  CUtensorMap ta, tb, ty;
  if (!make_tmap_3d(&ta, r.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, r.K, r.M, 1, KB, HALF, true) ||
      !make_tmap_3d(&tb, r.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, r.K, r.N, 1, KB, HALF, true) ||
      !make_tmap_3d(&ty, r.y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, r.N, r.M, 1, 32, 32, true)) {
    *why = "cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  PairParams p{};
  p.M = static_cast<int>(r.M);
  p.N = static_cast<int>(r.N);
  p.K = static_cast<int>(r.K);
  p.batches = 1;
  p.m_tiles = static_cast<int>(ceil_div(r.M, PM));
  p.n_tiles = static_cast<int>(ceil_div(r.N, PN));
  p.k_tiles = static_cast<int>(r.K / 128);
  p.num_tiles = p.m_tiles * p.n_tiles;
  p.a_scales = r.a_scales;
  p.b_scales = r.b_scales;
  p.kb = static_cast<int>(r.K / 128);
  p.y = r.y;
  p.status = ctx->status;
  p.timeout_ns = wait_timeout_ns();
  // kind::f8f6f4: D = F32, A/B E4M3 = 0 / E5M2 = 1, K-major, N = 256, M = 256 (pair).
  p.idesc = (1u << 4) | (f8_code(r.a_fmt) << 7) | (f8_code(r.b_fmt) << 10) | (static_cast<uint32_t>(PN >> 3) << 17) |
            (static_cast<uint32_t>(PM >> 4) << 24);
  // no scale-factor atoms in this mode: the operand maps stand in, unread
  return launch_pair<kPairF32>(ta, tb, ty, ta, tb, p, ctx, s, why);
}

bool mx_pair_eligible(const MxGemmRequest& r, const DeviceCtx* ctx) {
  // TMA output stores need 16-byte rows and base; at least one tile per cluster.
  const int esz = r.y_bf16 ? 2 : 4;
  return (r.N * esz) % 16 == 0 && reinterpret_cast<uintptr_t>(r.y) % 16 == 0 &&
         pair_tiles(r.B, r.M, r.N) >= ctx->num_sms / 2;
}

cudaError_t launch_mx_gemm_pair(const MxGemmRequest& r, const MxAtoms& at, cudaStream_t s, std::string* why) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  const bool nv = r.fmt == kFmtNVF4, mf4 = r.fmt == kFmtMXF4;
  const int atoms = nv ? 4 : (mf4 ? 2 : 1);
  const int64_t kbytes = (nv || mf4) ? r.K / 2 : r.K;
  // scale blocks as 128-byte rows, one TMA box per block
  const int sa_rows = 4 * pair_sfa_slots(atoms), sb_rows = 4 * pair_sfb_slots(atoms);
  const int64_t sfa_rows = r.B * static_cast<int64_t>(at.sfa_rt) * at.k_tiles * sa_rows;
  const bool brep = pair_b_replicated(atoms);
  const int64_t sfb_rows = brep ? r.B * static_cast<int64_t>(at.sfb_rt / 2) * at.k_tiles * sb_rows
                                : r.B * static_cast<int64_t>(at.sfb_rt) * at.ks4 * 4;
  CUtensorMap ta, tb, ty, tsa, tsb;
  const bool ok =
      make_tmap_3d(&ta, r.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kbytes, r.M, r.B, KB, HALF, true) &&
      make_tmap_3d(&tb, r.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kbytes, r.N, r.B, KB, HALF, true) &&
      make_tmap_3d(&ty, r.y, r.y_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                   r.y_bf16 ? 2 : 4, r.N, r.M, r.B, r.y_bf16 ? 64 : 32, 32, true) &&
      make_tmap_3d(&tsa, at.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128, sfa_rows, 1, 128, sa_rows, false) &&
      make_tmap_3d(&tsb, at.sfb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128, sfb_rows, 1, 128, brep ? sb_rows : 4 * atoms,
                   false);
  if (!ok) {
    *why = "cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  PairParams p{};
  p.M = static_cast<int>(r.M);
  p.N = static_cast<int>(r.N);
  p.K = static_cast<int>(r.K);
  p.batches = static_cast<int>(r.B);
  p.m_tiles = static_cast<int>(ceil_div(r.M, PM));
  p.n_tiles = static_cast<int>(ceil_div(r.N, PN));
  p.k_tiles = at.k_tiles;
  p.num_tiles = static_cast<int>(pair_tiles(r.B, r.M, r.N));
  p.sfa_rt = at.sfa_rt;
  p.sfb_rt = at.sfb_rt;
  p.y = static_cast<float*>(r.y);
  p.ks4 = at.ks4;
  p.y_bf16 = r.y_bf16 ? 1 : 0;
  p.status = ctx->status;
  p.timeout_ns = wait_timeout_ns();
  if (nv) {
    // kind::mxf4nvf4: E2M1 = 1 for A and B, UE4M3 scales (bit 23 = 0), N = 256, M = 256 (pair).
    p.idesc = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(PN >> 3) << 17) | (static_cast<uint32_t>(PM >> 4) << 24);
    return launch_pair<kPairNVF4>(ta, tb, ty, tsa, tsb, p, ctx, s, why);
  }
  if (mf4) {
    // kind::mxf4nvf4 .block32: E2M1 = 1 for A and B, UE8M0 scales (bit 23 = 1), N = 256, M = 256 (pair).
    p.idesc = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(PN >> 3) << 17) | (1u << 23) |
              (static_cast<uint32_t>(PM >> 4) << 24);
    return launch_pair<kPairMXF4>(ta, tb, ty, tsa, tsb, p, ctx, s, why);
  }
  // kind::mxf8f6f4: E4M3 = 0 / E5M2 = 1, UE8M0 scales (bit 23 = 1), N = 256, M = 256 (pair).
  p.idesc = (f8_code(r.a_fmt) << 7) | (f8_code(r.b_fmt) << 10) | (static_cast<uint32_t>(PN >> 3) << 17) | (1u << 23) |
            (static_cast<uint32_t>(PM >> 4) << 24);
  return launch_pair<kPairMXF8>(ta, tb, ty, tsa, tsb, p, ctx, s, why);
}

cudaError_t launch_int8_gemm_pair(const Int8Request& r, const void* xb, const void* wbT, int64_t Kp,
                                  int32_t* split_ws, unsigned* split_cnt, cudaStream_t s, std::string* why) {
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return cudaErrorInitializationError;
  // The bf16 operands are moved as bytes: a 128-byte K block is 64 codes.
  CUtensorMap ta, tb, ty, tacc;
  bool ok = make_tmap_3d(&ta, xb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Kp * 2, r.B, 1, KB, HALF, true) &&
            make_tmap_3d(&tb, wbT, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Kp * 2, r.D_out, 1, KB, HALF, true) &&
            make_tmap_3d(&ty, r.y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, r.D_out, r.B, 1, 32, 32, true);
  if (ok && r.acc) ok = make_tmap_3d(&tacc, r.acc, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, r.D_out, r.B, 1, 32, 32, true);
  if (!ok) {
    *why = "cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  if (!r.acc) tacc = ty;  // not read: store_acc = 0
  PairSplitParams p{};
  p.M = static_cast<int>(r.B);
  p.N = static_cast<int>(r.D_out);
  p.K = static_cast<int>(r.D_in);
  p.batches = 1;
  p.m_tiles = static_cast<int>(ceil_div(r.B, PM));
  p.n_tiles = static_cast<int>(ceil_div(r.D_out, PN));
  p.k_tiles = static_cast<int>(Kp / 64);
  p.num_tiles = p.m_tiles * p.n_tiles;
  p.sx = r.x_scales;
  p.sw = r.w_scales;
  // |code product| <= 127^2, so 16 K blocks (1024 products) sum to at most
  // 16,516,096 < 2^24 in magnitude: every FP32 partial is an exact integer.
  p.chunk = 16;
  p.store_acc = r.acc ? 1 : 0;
  p.split_ws = split_ws;
  p.split_cnt = split_cnt;
  p.status = ctx->status;
  p.timeout_ns = wait_timeout_ns();
  // kind::f16: D = F32 (bits 4-5 = 1), A = B = BF16 (bits 7-9, 10-12 = 1), K-major, N = 256, M = 256 (pair).
  p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(PN >> 3) << 17) |
            (static_cast<uint32_t>(PM >> 4) << 24);
  return launch_pair<kPairI8>(ta, tb, ty, tacc, ta, p, ctx, s, why);
}

}  // namespace bsmm
