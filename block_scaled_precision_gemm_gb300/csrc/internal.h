// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "../../include/bsmm.h"

namespace bsmm {

// ---- error reporting (thread-local last error) ---------------------------
void set_error(const std::string& msg);
bsmm_status fail(bsmm_status st, const std::string& msg);
bsmm_status cuda_fail(cudaError_t e, const char* what);

// ---- per-kernel timing (bsmm_trace_*) -------------------------------------
// While tracing is on, every launch of the library's kernels records a CUDA
// event on its stream before and after itself.  A TraceScope placed just
// before a launch statement does both (the second in its destructor, after
// the launch); when tracing is off it costs one relaxed atomic load.
bool trace_on();
int trace_begin(const char* name, cudaStream_t s);  // record index, or -1
void trace_end(int idx, cudaStream_t s);
struct TraceScope {
  TraceScope(const char* name, cudaStream_t s) : s_(s), idx_(trace_on() ? trace_begin(name, s) : -1) {}
  ~TraceScope() {
    if (idx_ >= 0) trace_end(idx_, s_);
  }
  TraceScope(const TraceScope&) = delete;
  TraceScope& operator=(const TraceScope&) = delete;

 private:
  cudaStream_t s_;
  int idx_;
};

// ---- per-device context ---------------------------------------------------
struct DeviceCtx {
  int device = -1;
  int num_sms = 0;
  int* status = nullptr;  // device address of the status word
};
// Context of the current device (sets up on first use).  Returns nullptr and
// sets the last error on failure.
const DeviceCtx* device_ctx();
uint64_t wait_timeout_ns();

// ---- TMA descriptors --------------------------------------------------------
// 3-D tiled tensor map over a row-major [d2][d1][d0] array of `elem_bytes`
// elements, box {b0, b1, 1}, 128-byte swizzle.  Returns false on failure.
bool make_tmap_3d(CUtensorMap* tm, const void* base, CUtensorMapDataType dtype, int elem_bytes, uint64_t d0,
                  uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, bool swizzle128);

// ---- kernel launchers (return cudaSuccess or the launch error) -----------
struct QuantRequest {
  const void* x;
  bool x_bf16;
  int64_t rows, cols, ld_x;
  int br, bc;
  int code;   // bsmm_dtype of the codes
  int scale;  // bsmm_scale_type
  bool transpose;
  void* codes;
  int64_t ld_codes;
  void* scales;
  int64_t ld_scales;
  // Scales in the tensor-core atom layout instead of [rows][blocks]: output
  // row r of batch r / sf_rows, row tile ((r % sf_rows) / 128) of sf_rt per
  // batch, sf_ks4 atoms (4 blocks each) per row tile (gemm_tc.cu, sf_relayout).
  bool sf_atoms = false;
  int64_t sf_rows = 0, sf_rt = 0, sf_ks4 = 0;
};
cudaError_t launch_quantize(const QuantRequest& q, cudaStream_t s);
// Independent quantizations, all on s (bsmm_quantize_batch): the 128 x 128
// ones quant_tile takes run as one launch per input type and scale kind,
// the rest one launch each.
cudaError_t launch_quantize_batch(const QuantRequest* q, int n, cudaStream_t s);
// Two quantizations of one bf16 array (qc: 32 x 1 blocks, transposed; qr:
// 1 x 32 blocks) in a single pass over it where the formats allow, else the
// two launches.
cudaError_t launch_quantize_dual(const QuantRequest& qc, const QuantRequest& qr, cudaStream_t s);
// Two independent quantizations of bf16 arrays into transposed 32 x 1 blocks
// (the backward's W^T and X^T) in one launch where both take the TMA-fed
// column kernel, else the two launches.
cudaError_t launch_quantize_pair(const QuantRequest& qa, const QuantRequest& qb, cudaStream_t s);

// Block-scaled formats of bsmm_gemm.
enum MxFormat { kFmtMXF8 = 0, kFmtNVF4 = 1, kFmtMXF4 = 2 };
// Scale relayout into the tensor-core scale-factor atoms (see gemm_tc.cu).
size_t sf_atoms_bytes(int64_t B, int64_t R, int64_t K, int fmt);

struct MxGemmRequest {
  int64_t B, M, N, K;
  const void* a;
  const void* b;
  int a_fmt, b_fmt;  // bsmm_dtype
  const uint8_t* a_scales;
  const uint8_t* b_scales;
  int fmt;  // MxFormat
  void* y;
  bool y_bf16;
  void* workspace;
  // scales per row as given (K_a, K_b): a user block may span several
  // hardware blocks (32 elements for UE8M0, 16 for UE4M3), which then repeat
  // its scale
  int64_t K_a, K_b;
  // a_scales / b_scales already in the tensor-core atom layout
  // (sf_atoms_plain_bytes): one scale per hardware block, K_a / K_b unused
  bool sf_atoms = false;
};
// Bytes of one operand's scales in the plain atom layout [B][row tiles of
// 128, rounded to pairs][K atoms], 512 each (what bsmm_quantize_atoms writes).
size_t sf_atoms_plain_bytes(int64_t B, int64_t R, int64_t K, int fmt);
// Any block size, CUDA cores (gemm_generic.cu); no workspace.
cudaError_t launch_mx_gemm_generic(const MxGemmRequest& r, int64_t K_a, int64_t K_b, int scale_type,
                                   cudaStream_t s);
cudaError_t launch_mx_gemm(const MxGemmRequest& r, cudaStream_t s, std::string* why);
// Same, with the scale-factor atoms in the library's static device array.
cudaError_t launch_mx_gemm_noalloc(const MxGemmRequest& r, cudaStream_t s, std::string* why);
// Scale factors already laid out by launch_mx_gemm for the CTA-pair kernel,
// in 512-byte slots.  A: [batch][row tile of 128 (sfa_rt)][K tile] x
// pair_sfa_slots, the atoms skewed by lane quarter (one atom: as is).  B, when
// pair_b_replicated: [batch][pair of row tiles (sfb_rt / 2)][K tile] x
// pair_sfb_slots, each atom four times over; otherwise the one-CTA kernel's
// atoms [batch][row tile][K atom (ks4)].  See sf_relayout_pair (gemm_tc.cu).
constexpr int pair_sfa_slots(int atoms) { return atoms == 1 ? 1 : atoms + 3; }
constexpr bool pair_b_replicated(int atoms) { return atoms == 4; }
constexpr int pair_sfb_slots(int atoms) { return pair_b_replicated(atoms) ? 8 * atoms : 2 * atoms; }
struct MxAtoms {
  const uint8_t* sfa;
  const uint8_t* sfb;
  int sfa_rt, sfb_rt, ks4, k_tiles;
};
// 256 x 256 tiles on CTA pairs (gemm_pair.cu); eligible when the output rows
// suit TMA stores and there is at least one tile per cluster.
bool mx_pair_eligible(const MxGemmRequest& r, const DeviceCtx* ctx);
cudaError_t launch_mx_gemm_pair(const MxGemmRequest& r, const MxAtoms& at, cudaStream_t s, std::string* why);

struct GroupedGemmRequest {
  int64_t M, N, K;
  const void* a;
  const void* b;
  int a_fmt, b_fmt;
  const float* a_scales;
  const float* b_scales;
  float* y;
};
cudaError_t launch_grouped_gemm(const GroupedGemmRequest& r, cudaStream_t s, std::string* why);
// 256 x 256 tiles on CTA pairs (gemm_pair.cu); eligible when N and K are
// multiples of 128 and there is at least one tile per cluster.
bool grouped_pair_eligible(int64_t M, int64_t N, int64_t K, const DeviceCtx* ctx);
cudaError_t launch_grouped_gemm_pair(const GroupedGemmRequest& r, cudaStream_t s, std::string* why);

struct Int8Request {
  const float* x;
  const float* w;
  int64_t B, D_in, D_out;
  int8_t* x_q;
  float* x_scales;
  int8_t* w_q;
  float* w_scales;
  float* y;
  int32_t* acc;
  void* workspace;
};
size_t int8_workspace_bytes(int64_t B, int64_t D_in, int64_t D_out);
cudaError_t launch_int8_channel(const Int8Request& r, cudaStream_t s);
// The exact INT8 matmul on bf16 tensor cores (gemm_pair.cu): xb [B, Kp] and
// wbT [D_out, Kp] are bf16 codes, K-major, zero beyond D_in (Kp % 64 == 0);
// writes r.y and, if non-null, r.acc.  The tiles of its last, partial wave
// split their K blocks into up to kSplitMax parts over the clusters that
// would otherwise idle: split_cnt holds kSplitTilesMax x 32 zeroed counters
// and split_ws int32 tiles of 256 x 256 for int8_split_units(tiles) parts
// (no split when either is null).
constexpr int kSplitMax = 4, kSplitTilesMax = 64, kSplitUnitsMax = 128;
inline int64_t int8_split_units(int64_t tiles) { return tiles * kSplitMax < kSplitUnitsMax ? tiles * kSplitMax : kSplitUnitsMax; }
cudaError_t launch_int8_gemm_pair(const Int8Request& r, const void* xb, const void* wbT, int64_t Kp,
                                  int32_t* split_ws, unsigned* split_cnt, cudaStream_t s, std::string* why);

cudaError_t launch_selftest_wait(uint64_t timeout_ns, cudaStream_t s);
cudaError_t launch_selftest_quotient(uint64_t pairs, uint64_t seed, unsigned long long* bad, cudaStream_t s);

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace bsmm
