// C ABI of libbsmm.so: argument validation, per-device state, TMA descriptor
// factory and dispatch to the kernels.  No exception crosses this boundary.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace bsmm {

// One status word per device (per loaded module); kernels record the site
// of the first bounded wait that gave up.
__device__ int g_status_word;

namespace {
thread_local std::string t_last_error;
std::atomic<uint64_t> g_timeout_ns{1000000000ull};

constexpr int kMaxDevices = 64;
DeviceCtx g_ctx[kMaxDevices];
std::once_flag g_ctx_once[kMaxDevices];
bool g_ctx_ok[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void init_ctx(int dev) {
  DeviceCtx& c = g_ctx[dev];
  c.device = dev;
  g_ctx_ok[dev] = false;
  if (cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return;
  c.status = static_cast<int*>(p);
  if (cudaMemset(c.status, 0, sizeof(int)) != cudaSuccess) return;
  g_ctx_ok[dev] = true;
}
}  // namespace

void set_error(const std::string& msg) { t_last_error = msg; }

bsmm_status fail(bsmm_status st, const std::string& msg) {
  set_error(msg);
  return st;
}

bsmm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(BSMM_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

const DeviceCtx* device_ctx() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    set_error("no current CUDA device");
    return nullptr;
  }
  std::call_once(g_ctx_once[dev], init_ctx, dev);
  if (!g_ctx_ok[dev]) {
    set_error("device set-up failed (status word or SM count)");
    return nullptr;
  }
  return &g_ctx[dev];
}

uint64_t wait_timeout_ns() { return g_timeout_ns.load(); }

bool make_tmap_3d(CUtensorMap* tm, const void* base, CUtensorMapDataType dtype, int elem_bytes, uint64_t d0,
                  uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, bool swizzle128) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * elem_bytes, d0 * d1 * elem_bytes};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(tm, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---- per-kernel timing ------------------------------------------------------
namespace {
struct TraceRec {
  const char* name;
  int device;
  cudaEvent_t e0, e1;
  bool ok;
};
std::atomic<bool> g_trace_on{false};
std::mutex g_trace_mu;
std::vector<TraceRec> g_trace;

void trace_clear_locked() {
  for (TraceRec& r : g_trace) {
    if (r.e0) cudaEventDestroy(r.e0);
    if (r.e1) cudaEventDestroy(r.e1);
  }
  g_trace.clear();
}
}  // namespace

bool trace_on() { return g_trace_on.load(std::memory_order_relaxed); }

// Event failures never change what the launch itself returns: the record is
// kept, marked unusable, and the CUDA error state is cleared.
int trace_begin(const char* name, cudaStream_t s) {
  TraceRec r{name, 0, nullptr, nullptr, false};
  r.ok = cudaGetDevice(&r.device) == cudaSuccess && cudaEventCreate(&r.e0) == cudaSuccess &&
         cudaEventCreate(&r.e1) == cudaSuccess && cudaEventRecord(r.e0, s) == cudaSuccess;
  if (!r.ok) cudaGetLastError();
  std::lock_guard<std::mutex> lock(g_trace_mu);
  g_trace.push_back(r);
  return static_cast<int>(g_trace.size()) - 1;
}

void trace_end(int idx, cudaStream_t s) {
  cudaEvent_t e1 = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (idx < 0 || idx >= static_cast<int>(g_trace.size()) || !g_trace[idx].ok) return;
    e1 = g_trace[idx].e1;
  }
  if (cudaEventRecord(e1, s) != cudaSuccess) {
    cudaGetLastError();
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (idx < static_cast<int>(g_trace.size())) g_trace[idx].ok = false;
  }
}

}  // namespace bsmm

using namespace bsmm;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is_code(int t) { return t == BSMM_E4M3 || t == BSMM_E5M2 || t == BSMM_E2M1 || t == BSMM_INT8; }
bool is_scale(int t) { return t == BSMM_SCALE_F32 || t == BSMM_SCALE_UE8M0 || t == BSMM_SCALE_UE4M3; }

bsmm_status launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return cuda_fail(e, what);
  set_error("");
  return BSMM_OK;
}

std::string last_error_text() { return t_last_error; }

static_assert(sizeof(void*) != 8 || sizeof(bsmm_quantize_job) == 96, "bsmm_quantize_job layout (the binding mirrors it)");

// One quantization's arguments checked as bsmm_quantize documents them, and
// turned into a launch request (*empty: a zero-sized job, nothing to do).
bsmm_status quantize_request(const bsmm_quantize_job& j, QuantRequest* q, bool* empty) {
  if (j.x_type != BSMM_F32 && j.x_type != BSMM_BF16) return fail(BSMM_ERR_INVALID_ARG, "x_type must be F32 or BF16");
  if (!is_code(j.code_type)) return fail(BSMM_ERR_INVALID_ARG, "code_type must be E4M3, E5M2, E2M1 or INT8");
  if (!is_scale(j.scale_type)) return fail(BSMM_ERR_INVALID_ARG, "bad scale_type");
  if (j.rows < 0 || j.cols < 0) return fail(BSMM_ERR_INVALID_ARG, "negative size");
  *empty = j.rows == 0 || j.cols == 0;
  if (*empty) return BSMM_OK;
  if (!j.x || !j.codes || !j.scales) return fail(BSMM_ERR_INVALID_ARG, "null pointer");
  if (j.block_rows < 1 || j.block_cols < 1) return fail(BSMM_ERR_INVALID_ARG, "block sizes must be positive");
  if (j.rows % j.block_rows || j.cols % j.block_cols) return fail(BSMM_ERR_SHAPE, "rows/cols not divisible by the block");
  if (j.code_type == BSMM_INT8 && j.scale_type != BSMM_SCALE_F32)
    return fail(BSMM_ERR_UNSUPPORTED, "INT8 codes take F32 scales");
  if (j.transpose_out && j.block_cols != 1) return fail(BSMM_ERR_UNSUPPORTED, "transposed output needs column blocks");
  if (j.ld_x < j.cols) return fail(BSMM_ERR_SHAPE, "ld_x < cols");
  const int64_t out_cols = j.transpose_out ? j.rows : j.cols;
  if (j.ld_codes < out_cols) return fail(BSMM_ERR_SHAPE, "ld_codes too small");
  const int64_t s_cols = j.transpose_out ? j.rows / j.block_rows : j.cols / j.block_cols;
  if (j.ld_scales < s_cols) return fail(BSMM_ERR_SHAPE, "ld_scales too small");
  if (j.code_type == BSMM_E2M1) {
    if (j.ld_codes % 2 || out_cols % 2) return fail(BSMM_ERR_SHAPE, "E2M1 codes need an even contiguous extent");
    // Column blocks written untransposed are packed across lanes by the
    // column kernels; every other layout packs within one block.
    const int br = j.block_rows;
    const bool pow2r = br == 16 || br == 32 || br == 64 || br == 128;
    const bool paired = !j.transpose_out && j.block_cols == 1 && (pow2r || br == j.rows);
    const int ext = j.transpose_out ? j.block_rows : j.block_cols;
    if (ext % 2 && !paired) return fail(BSMM_ERR_UNSUPPORTED, "E2M1 blocks need an even extent along the contiguous axis");
  }
  *q = QuantRequest{j.x,         j.x_type == BSMM_BF16, j.rows,   j.cols,   j.ld_x,   j.block_rows,
                    j.block_cols, j.code_type,          j.scale_type, j.transpose_out != 0, j.codes, j.ld_codes,
                    j.scales,    j.ld_scales};
  return BSMM_OK;
}

// Which kernel a bsmm_gemm problem takes.  The tensor cores scale per 32
// elements (UE8M0: MXFP8, MXFP4) or 16 (UE4M3 with E2M1: NVFP4); a block that
// is a multiple of that repeats its scale there.  Any other block size, and
// FP8 codes with UE4M3 scales, run on the CUDA-core kernel.
struct GemmRoute {
  bool ok, tensor;
  int fmt;  // MxFormat, for the tensor path
  const char* why;
};
GemmRoute route_gemm(int at, int bt, int st, int64_t K, int64_t K_a, int64_t K_b) {
  const bool fp8 = (at == BSMM_E4M3 || at == BSMM_E5M2) && (bt == BSMM_E4M3 || bt == BSMM_E5M2);
  const bool fp4 = at == BSMM_E2M1 && bt == BSMM_E2M1;
  if (!(fp8 || fp4) || (st != BSMM_SCALE_UE8M0 && st != BSMM_SCALE_UE4M3))
    return {false, false, 0, "codes E4M3/E5M2 (both operands) or E2M1 (both), scales UE8M0 or UE4M3"};
  if (fp4 && K % 2) return {false, false, 0, "E2M1 codes need an even K"};
  const int64_t bs_a = K / K_a, bs_b = K / K_b;
  const int64_t hw = (fp4 && st == BSMM_SCALE_UE4M3) ? 16 : 32;
  const bool tensor = (fp4 || st == BSMM_SCALE_UE8M0) && bs_a % hw == 0 && bs_b % hw == 0 && K % 32 == 0;
  const int fmt = fp8 ? kFmtMXF8 : (st == BSMM_SCALE_UE4M3 ? kFmtNVF4 : kFmtMXF4);
  return {true, tensor, fmt, ""};
}

// The format of a GEMM operand quantized with hardware blocks: FP8 codes take
// UE8M0 per 32 (MXFP8); E2M1 takes UE8M0 per 32 (MXFP4) or UE4M3 per 16
// (NVFP4).  -1: no tensor-core format.
int atom_format(int code, int scale) {
  if ((code == BSMM_E4M3 || code == BSMM_E5M2) && scale == BSMM_SCALE_UE8M0) return kFmtMXF8;
  if (code == BSMM_E2M1 && scale == BSMM_SCALE_UE8M0) return kFmtMXF4;
  if (code == BSMM_E2M1 && scale == BSMM_SCALE_UE4M3) return kFmtNVF4;
  return -1;
}

// The request that quantizes a GEMM operand of B x rows x K (contraction K)
// with its scales written straight into the plain atom layout, after filling
// the atoms with the neutral scale (UE8M0 127 = 1.0, UE4M3 0) so that padding
// rows and blocks past K contribute nothing.  transpose_in: x is [K][rows]
// (B == 1).
cudaError_t atoms_request(const void* x, bool bf16, int64_t B, int64_t rows, int64_t K, bool transpose_in, int code,
                          int scale, void* codes, void* atoms, cudaStream_t s, QuantRequest* q) {
  const int fmt = atom_format(code, scale);
  const int bs = fmt == kFmtNVF4 ? 16 : 32;
  const int per_tile = fmt == kFmtNVF4 ? 4 : (fmt == kFmtMXF4 ? 2 : 1);
  const int64_t k_tiles = ceil_div(K, fmt == kFmtMXF8 ? 128 : 256);
  cudaError_t e = cudaMemsetAsync(atoms, scale == BSMM_SCALE_UE4M3 ? 0 : 127, sf_atoms_plain_bytes(B, rows, K, fmt), s);
  if (e != cudaSuccess) return e;
  *q = transpose_in ? QuantRequest{x, bf16, K, rows, rows, bs, 1, code, scale, true, codes, K, atoms, 1}
                    : QuantRequest{x, bf16, B * rows, K, K, 1, bs, code, scale, false, codes, K, atoms, 1};
  q->sf_atoms = true;
  q->sf_rows = rows;
  q->sf_rt = ceil_div(rows, 256) * 2;
  q->sf_ks4 = k_tiles * per_tile;
  return cudaSuccess;
}

cudaError_t quantize_to_atoms(const void* x, bool bf16, int64_t B, int64_t rows, int64_t K, bool transpose_in,
                              int code, int scale, void* codes, void* atoms, cudaStream_t s) {
  QuantRequest q;
  const cudaError_t e = atoms_request(x, bf16, B, rows, K, transpose_in, code, scale, codes, atoms, s, &q);
  return e != cudaSuccess ? e : launch_quantize(q, s);
}

}  // namespace

extern "C" {

int bsmm_version(void) { return 100; }

const char* bsmm_last_error(void) { return t_last_error.c_str(); }

void bsmm_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns == 0 ? 1 : ns); }

bsmm_status bsmm_check_device_status(bsmm_stream_t stream, int* where) {
  if (where) *where = 0;
  const DeviceCtx* ctx = device_ctx();
  if (!ctx) return BSMM_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int v = 0;
  e = cudaMemcpy(&v, ctx->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpy(ctx->status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear status word");
    if (where) *where = v;
    return fail(BSMM_ERR_TIMEOUT, "a bounded in-kernel wait gave up (site " + std::to_string(v) + ")");
  }
  set_error("");
  return BSMM_OK;
}

bsmm_status bsmm_selftest_wait_timeout(uint64_t timeout_ns, bsmm_stream_t stream) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return fail(BSMM_ERR_INVALID_ARG, "timeout_ns out of range");
  return launched(launch_selftest_wait(timeout_ns, reinterpret_cast<cudaStream_t>(stream)), "selftest launch");
}

bsmm_status bsmm_selftest_quotient(uint64_t pairs, uint64_t seed, uint64_t* mismatches, bsmm_stream_t stream) {
  if (!mismatches) return fail(BSMM_ERR_INVALID_ARG, "mismatches is NULL");
  return launched(launch_selftest_quotient(pairs, seed, reinterpret_cast<unsigned long long*>(mismatches),
                                           reinterpret_cast<cudaStream_t>(stream)),
                  "selftest launch");
}

bsmm_status bsmm_trace_start(void) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  trace_clear_locked();
  g_trace_on.store(true);
  return BSMM_OK;
}

bsmm_status bsmm_trace_stop(void) {
  g_trace_on.store(false);
  return BSMM_OK;
}

int bsmm_trace_count(void) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  return static_cast<int>(g_trace.size());
}

bsmm_status bsmm_trace_read(int i, const char** name, float* start_ms, float* ms) {
  TraceRec r, first;
  {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (i < 0 || i >= static_cast<int>(g_trace.size())) return fail(BSMM_ERR_INVALID_ARG, "trace index out of range");
    r = g_trace[i];
    first = g_trace[0];
  }
  if (name) *name = r.name;
  if (!r.ok) return fail(BSMM_ERR_CUDA, "this launch's events could not be recorded");
  int old = 0;
  cudaError_t e = cudaGetDevice(&old);
  if (e == cudaSuccess && old != r.device) e = cudaSetDevice(r.device);
  if (e == cudaSuccess) e = cudaEventSynchronize(r.e1);
  float t = 0.f, t0 = 0.f;
  if (e == cudaSuccess && ms) e = cudaEventElapsedTime(&t, r.e0, r.e1);
  if (e == cudaSuccess && start_ms) {
    if (first.ok && first.device == r.device)
      e = cudaEventElapsedTime(&t0, first.e0, r.e0);
    else
      t0 = 0.f;
  }
  if (old != r.device) cudaSetDevice(old);
  if (e != cudaSuccess) return cuda_fail(e, "trace event");
  if (ms) *ms = t;
  if (start_ms) *start_ms = t0;
  return BSMM_OK;
}

bsmm_status bsmm_quantize(const void* x, bsmm_dtype x_type, int64_t rows, int64_t cols, int64_t ld_x,
                          int block_rows, int block_cols, bsmm_dtype code_type, bsmm_scale_type scale_type,
                          int transpose_out, void* codes, int64_t ld_codes, void* scales, int64_t ld_scales,
                          bsmm_stream_t stream) {
  const bsmm_quantize_job j{x,          x_type,     rows,          cols,  ld_x,     block_rows, block_cols,
                            code_type,  scale_type, transpose_out, codes, ld_codes, scales,     ld_scales};
  QuantRequest q{};
  bool empty = false;
  const bsmm_status st = quantize_request(j, &q, &empty);
  if (st != BSMM_OK) return st;
  if (empty) {
    set_error("");
    return BSMM_OK;
  }
  return launched(launch_quantize(q, reinterpret_cast<cudaStream_t>(stream)), "quantize launch");
}

bsmm_status bsmm_quantize_batch(const bsmm_quantize_job* jobs, int count, bsmm_stream_t stream) {
  if (count < 0) return fail(BSMM_ERR_INVALID_ARG, "negative count");
  if (count > 0 && !jobs) return fail(BSMM_ERR_INVALID_ARG, "null jobs");
  std::vector<QuantRequest> q;
  q.reserve(static_cast<size_t>(count));
  for (int i = 0; i < count; ++i) {  // every job checked before any launch
    QuantRequest r{};
    bool empty = false;
    const bsmm_status st = quantize_request(jobs[i], &r, &empty);
    if (st != BSMM_OK) return fail(st, "job " + std::to_string(i) + ": " + last_error_text());
    if (!empty) q.push_back(r);
  }
  if (q.empty()) {
    set_error("");
    return BSMM_OK;
  }
  return launched(launch_quantize_batch(q.data(), static_cast<int>(q.size()), reinterpret_cast<cudaStream_t>(stream)),
                  "quantize batch launch");
}

size_t bsmm_gemm_workspace_size(int64_t B, int64_t M, int64_t N, int64_t K, bsmm_dtype a_type) {
  if (B <= 0 || M <= 0 || N <= 0 || K <= 0) return 0;
  // E2M1: room for NVFP4's atoms, which covers MXFP4's
  const int fmt = a_type == BSMM_E2M1 ? kFmtNVF4 : kFmtMXF8;
  return align_up(sf_atoms_bytes(B, M, K, fmt), 256) + align_up(sf_atoms_bytes(B, N, K, fmt), 256);
}

bsmm_status bsmm_gemm(int64_t B, int64_t M, int64_t N, int64_t K, const void* a, bsmm_dtype a_type, const void* b,
                      bsmm_dtype b_type, const void* a_scales, int64_t K_a, const void* b_scales, int64_t K_b,
                      bsmm_scale_type scale_type, void* y, bsmm_dtype y_type, void* workspace,
                      size_t workspace_bytes, bsmm_stream_t stream) {
  if (B < 0 || M < 0 || N < 0 || K < 0) return fail(BSMM_ERR_INVALID_ARG, "negative size");
  if (y_type != BSMM_F32 && y_type != BSMM_BF16) return fail(BSMM_ERR_INVALID_ARG, "y_type must be F32 or BF16");
  if (!is_scale(scale_type)) return fail(BSMM_ERR_INVALID_ARG, "bad scale_type");
  if (!is_code(a_type) || !is_code(b_type)) return fail(BSMM_ERR_INVALID_ARG, "bad operand type");
  if (K_a <= 0 || K_b <= 0 || K % K_a || K % K_b)
    return fail(BSMM_ERR_SHAPE, "K must be a multiple of K_a and of K_b");
  if (B == 0 || M == 0 || N == 0) {
    set_error("");
    return BSMM_OK;
  }
  if (K == 0) return fail(BSMM_ERR_UNSUPPORTED, "K == 0");
  const GemmRoute route = route_gemm(a_type, b_type, scale_type, K, K_a, K_b);
  if (!route.ok) return fail(BSMM_ERR_UNSUPPORTED, route.why);
  if (!a || !b || !a_scales || !b_scales || !y) return fail(BSMM_ERR_INVALID_ARG, "null pointer");
  if (!route.tensor) {  // a block size the tensor cores do not scale by
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2 || B > 65535)
      return fail(BSMM_ERR_SHAPE, "size beyond the supported range");
    MxGemmRequest g{B, M, N, K, a, b, a_type, b_type, static_cast<const uint8_t*>(a_scales),
                    static_cast<const uint8_t*>(b_scales), route.fmt, y, y_type == BSMM_BF16, nullptr, K_a, K_b};
    return launched(launch_mx_gemm_generic(g, K_a, K_b, scale_type, reinterpret_cast<cudaStream_t>(stream)),
                    "gemm (generic block) launch");
  }
  if (!aligned16(a) || !aligned16(b) || !aligned16(y)) return fail(BSMM_ERR_ALIGNMENT, "a, b, y must be 16-byte aligned");
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2 || B > 65535)
    return fail(BSMM_ERR_SHAPE, "size beyond the supported range");
  const size_t need = bsmm_gemm_workspace_size(B, M, N, K, a_type);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(BSMM_ERR_WORKSPACE, "workspace must be 256-byte aligned and at least " + std::to_string(need) +
                                        " bytes");
  MxGemmRequest r{B, M, N, K, a, b, a_type, b_type, static_cast<const uint8_t*>(a_scales),
                  static_cast<const uint8_t*>(b_scales), route.fmt, y, y_type == BSMM_BF16, workspace, K_a, K_b};
  std::string why;
  const cudaError_t e = launch_mx_gemm(r, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess && !why.empty()) return fail(BSMM_ERR_CUDA, why);
  return launched(e, "gemm launch");
}

size_t bsmm_scale_atoms_size(int64_t B, int64_t rows, int64_t K, bsmm_dtype code_type, bsmm_scale_type scale_type) {
  const int fmt = atom_format(code_type, scale_type);
  if (fmt < 0 || B <= 0 || rows <= 0 || K <= 0) return 0;
  return sf_atoms_plain_bytes(B, rows, K, fmt);
}

bsmm_status bsmm_quantize_atoms(const void* x, bsmm_dtype x_type, int64_t B, int64_t rows, int64_t K,
                                int transpose_in, bsmm_dtype code_type, bsmm_scale_type scale_type, void* codes,
                                void* atoms, size_t atoms_bytes, bsmm_stream_t stream) {
  if (x_type != BSMM_F32 && x_type != BSMM_BF16) return fail(BSMM_ERR_INVALID_ARG, "x_type must be F32 or BF16");
  const int fmt = atom_format(code_type, scale_type);
  if (fmt < 0)
    return fail(BSMM_ERR_UNSUPPORTED, "atoms take E4M3/E5M2 or E2M1 codes with UE8M0, or E2M1 with UE4M3");
  if (B < 0 || rows < 0 || K < 0) return fail(BSMM_ERR_INVALID_ARG, "negative size");
  if (B == 0 || rows == 0 || K == 0) {
    set_error("");
    return BSMM_OK;
  }
  if (transpose_in && B != 1) return fail(BSMM_ERR_SHAPE, "a transposed input has one batch");
  const int bs = fmt == kFmtNVF4 ? 16 : 32;
  if (K % bs) return fail(BSMM_ERR_SHAPE, "K must be a multiple of the hardware block (32, or 16 for UE4M3)");
  if (!x || !codes || !atoms) return fail(BSMM_ERR_INVALID_ARG, "null pointer");
  const size_t need = sf_atoms_plain_bytes(B, rows, K, fmt);
  if (atoms_bytes < need) return fail(BSMM_ERR_WORKSPACE, "atoms need " + std::to_string(need) + " bytes");
  if (reinterpret_cast<uintptr_t>(atoms) & 3u) return fail(BSMM_ERR_ALIGNMENT, "atoms must be 4-byte aligned");
  return launched(quantize_to_atoms(x, x_type == BSMM_BF16, B, rows, K, transpose_in != 0, code_type, scale_type,
                                    codes, atoms, reinterpret_cast<cudaStream_t>(stream)),
                  "quantize (atoms) launch");
}

bsmm_status bsmm_gemm_atoms(int64_t B, int64_t M, int64_t N, int64_t K, const void* a, bsmm_dtype a_type,
                            const void* b, bsmm_dtype b_type, const void* a_atoms, const void* b_atoms,
                            bsmm_scale_type scale_type, void* y, bsmm_dtype y_type, void* workspace,
                            size_t workspace_bytes, bsmm_stream_t stream) {
  if (B < 0 || M < 0 || N < 0 || K < 0) return fail(BSMM_ERR_INVALID_ARG, "negative size");
  if (y_type != BSMM_F32 && y_type != BSMM_BF16) return fail(BSMM_ERR_INVALID_ARG, "y_type must be F32 or BF16");
  const int fa = atom_format(a_type, scale_type), fb = atom_format(b_type, scale_type);
  if (fa < 0 || fb < 0 || fa != fb)
    return fail(BSMM_ERR_UNSUPPORTED, "both operands MXFP8 (E4M3/E5M2, UE8M0), MXFP4 or NVFP4");
  if (B == 0 || M == 0 || N == 0) {
    set_error("");
    return BSMM_OK;
  }
  if (K == 0 || K % (fa == kFmtNVF4 ? 16 : 32)) return fail(BSMM_ERR_SHAPE, "K must be a positive multiple of the block");
  if (K % 32) return fail(BSMM_ERR_SHAPE, "K must be a multiple of 32");
  if (!a || !b || !a_atoms || !b_atoms || !y) return fail(BSMM_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(a) || !aligned16(b) || !aligned16(y) || !aligned16(a_atoms) || !aligned16(b_atoms))
    return fail(BSMM_ERR_ALIGNMENT, "a, b, y and the atoms must be 16-byte aligned");
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2 || B > 65535)
    return fail(BSMM_ERR_SHAPE, "size beyond the supported range");
  if (fa != kFmtMXF8) {  // the pair kernel's skewed / replicated blocks are written from the atoms
    const size_t need = bsmm_gemm_workspace_size(B, M, N, K, a_type);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return fail(BSMM_ERR_WORKSPACE, "workspace must be 256-byte aligned and at least " + std::to_string(need) +
                                          " bytes");
  }
  const int64_t hw = fa == kFmtNVF4 ? 16 : 32;
  MxGemmRequest r{B, M, N, K, a, b, a_type, b_type, static_cast<const uint8_t*>(a_atoms),
                  static_cast<const uint8_t*>(b_atoms), fa, y, y_type == BSMM_BF16, workspace, K / hw, K / hw};
  r.sf_atoms = true;
  std::string why;
  const cudaError_t e = launch_mx_gemm(r, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess && !why.empty()) return fail(BSMM_ERR_CUDA, why);
  return launched(e, "gemm (atoms) launch");
}

bsmm_status bsmm_gemm_noalloc(int64_t B, int64_t M, int64_t N, int64_t K, const void* a, bsmm_dtype a_type,
                              const void* b, bsmm_dtype b_type, const void* a_scales, int64_t K_a,
                              const void* b_scales, int64_t K_b, bsmm_scale_type scale_type, void* y,
                              bsmm_dtype y_type, bsmm_stream_t stream) {
  if (B < 0 || M < 0 || N < 0 || K < 0) return fail(BSMM_ERR_INVALID_ARG, "negative size");
  if (y_type != BSMM_F32 && y_type != BSMM_BF16) return fail(BSMM_ERR_INVALID_ARG, "y_type must be F32 or BF16");
  if (!is_scale(scale_type)) return fail(BSMM_ERR_INVALID_ARG, "bad scale_type");
  if (!is_code(a_type) || !is_code(b_type)) return fail(BSMM_ERR_INVALID_ARG, "bad operand type");
  if (K_a <= 0 || K_b <= 0 || K % K_a || K % K_b)
    return fail(BSMM_ERR_SHAPE, "K must be a multiple of K_a and of K_b");
  if (B == 0 || M == 0 || N == 0) {
    set_error("");
    return BSMM_OK;
  }
  if (K == 0) return fail(BSMM_ERR_UNSUPPORTED, "K == 0");
  const GemmRoute route = route_gemm(a_type, b_type, scale_type, K, K_a, K_b);
  if (!route.ok) return fail(BSMM_ERR_UNSUPPORTED, route.why);
  if (!a || !b || !a_scales || !b_scales || !y) return fail(BSMM_ERR_INVALID_ARG, "null pointer");
  if (!route.tensor) {  // a block size the tensor cores do not scale by
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2 || B > 65535)
      return fail(BSMM_ERR_SHAPE, "size beyond the supported range");
    MxGemmRequest g{B, M, N, K, a, b, a_type, b_type, static_cast<const uint8_t*>(a_scales),
                    static_cast<const uint8_t*>(b_scales), route.fmt, y, y_type == BSMM_BF16, nullptr, K_a, K_b};
    return launched(launch_mx_gemm_generic(g, K_a, K_b, scale_type, reinterpret_cast<cudaStream_t>(stream)),
                    "gemm (generic block) launch");
  }
  if (!aligned16(a) || !aligned16(b) || !aligned16(y)) return fail(BSMM_ERR_ALIGNMENT, "a, b, y must be 16-byte aligned");
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2 || B > 65535)
    return fail(BSMM_ERR_SHAPE, "size beyond the supported range");
  const size_t need = bsmm_gemm_workspace_size(B, M, N, K, a_type);
  if (need > BSMM_NOALLOC_SCRATCH_BYTES)
    return fail(BSMM_ERR_WORKSPACE, "this problem needs " + std::to_string(need) +
                                        " bytes of scratch; the no-allocation entry point holds at most " +
                                        std::to_string(BSMM_NOALLOC_SCRATCH_BYTES) +
                                        " (use bsmm_gemm with a workspace)");
  MxGemmRequest r{B, M, N, K, a, b, a_type, b_type, static_cast<const uint8_t*>(a_scales),
                  static_cast<const uint8_t*>(b_scales), route.fmt, y, y_type == BSMM_BF16, nullptr, K_a, K_b};
  std::string why;
  const cudaError_t e = launch_mx_gemm_noalloc(r, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess && !why.empty()) return fail(BSMM_ERR_CUDA, why);
  return launched(e, "gemm (no allocation) launch");
}

bsmm_status bsmm_gemm_grouped(int64_t M, int64_t N, int64_t K, const void* a, bsmm_dtype a_type, const void* b,
                              bsmm_dtype b_type, const float* a_scales, const float* b_scales, int group_n,
                              int group_k, float* y, bsmm_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return fail(BSMM_ERR_INVALID_ARG, "negative size");
  if ((a_type != BSMM_E4M3 && a_type != BSMM_E5M2) || (b_type != BSMM_E4M3 && b_type != BSMM_E5M2))
    return fail(BSMM_ERR_INVALID_ARG, "operands must be E4M3 or E5M2");
  if (group_n <= 0 || group_k <= 0) return fail(BSMM_ERR_INVALID_ARG, "group sizes must be positive");
  if (N % group_n || K % group_k) return fail(BSMM_ERR_SHAPE, "N % group_n and K % group_k must be 0");
  if (group_n != 128 || group_k != 128) return fail(BSMM_ERR_UNSUPPORTED, "only group_n = group_k = 128");
  if (M == 0 || N == 0) {
    set_error("");
    return BSMM_OK;
  }
  if (K == 0) return fail(BSMM_ERR_UNSUPPORTED, "K == 0");
  if (!a || !b || !a_scales || !b_scales || !y) return fail(BSMM_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(a) || !aligned16(b) || !aligned16(y)) return fail(BSMM_ERR_ALIGNMENT, "a, b, y must be 16-byte aligned");
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2)
    return fail(BSMM_ERR_SHAPE, "size beyond the supported range");
  GroupedGemmRequest r{M, N, K, a, b, a_type, b_type, a_scales, b_scales, y};
  std::string why;
  const cudaError_t e = launch_grouped_gemm(r, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess && !why.empty()) return fail(BSMM_ERR_CUDA, why);
  return launched(e, "grouped gemm launch");
}

size_t bsmm_int8_channel_workspace_size(int64_t B, int64_t D_in, int64_t D_out) {
  if (B < 0 || D_in <= 0 || D_out <= 0) return 0;
  if (B == 0) return align_up(static_cast<size_t>(D_out) * 4, 256);  // w alone: its column maxima
  return int8_workspace_bytes(B, D_in, D_out);
}

bsmm_status bsmm_int8_channel(const float* x, const float* w, int64_t B, int64_t D_in, int64_t D_out, int8_t* x_q,
                              float* x_scales, int8_t* w_q, float* w_scales, float* y, int32_t* acc,
                              void* workspace, size_t workspace_bytes, bsmm_stream_t stream) {
  if (B < 0 || D_in < 0 || D_out < 0) return fail(BSMM_ERR_INVALID_ARG, "negative size");
  if (D_out == 0) {
    set_error("");
    return BSMM_OK;
  }
  if (D_in == 0) return fail(BSMM_ERR_UNSUPPORTED, "D_in == 0");
  if (B == 0) {  // no rows of x: w_q and w_scales are still outputs
    if (!w || !w_q || !w_scales) return fail(BSMM_ERR_INVALID_ARG, "null pointer");
    const size_t need = bsmm_int8_channel_workspace_size(0, D_in, D_out);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return fail(BSMM_ERR_WORKSPACE, "workspace must be 256-byte aligned and at least " + std::to_string(need) +
                                          " bytes");
    Int8Request r{x, w, 0, D_in, D_out, x_q, x_scales, w_q, w_scales, y, acc, workspace};
    return launched(launch_int8_channel(r, reinterpret_cast<cudaStream_t>(stream)), "int8 launch");
  }
  if (!x || !w || !x_q || !x_scales || !w_q || !w_scales || !y) return fail(BSMM_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(y) || (acc && !aligned16(acc))) return fail(BSMM_ERR_ALIGNMENT, "y and acc must be 16-byte aligned");
  if (B > 65535LL * 128 || D_out > INT32_MAX / 2 || D_in > 1 << 24)
    return fail(BSMM_ERR_SHAPE, "size beyond the supported range");
  const size_t need = bsmm_int8_channel_workspace_size(B, D_in, D_out);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(BSMM_ERR_WORKSPACE, "workspace must be 256-byte aligned and at least " + std::to_string(need) +
                                        " bytes");
  Int8Request r{x, w, B, D_in, D_out, x_q, x_scales, w_q, w_scales, y, acc, workspace};
  return launched(launch_int8_channel(r, reinterpret_cast<cudaStream_t>(stream)), "int8 launch");
}

size_t bsmm_linear_backward_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  // codes: dY along N [M,N], W^T [K,N], dY^T [N,M], X^T [K,M]; the UE8M0
  // scales of each in the tensor-core atom layout, read in place by the GEMMs
  size_t total = 0;
  total += align_up(static_cast<size_t>(M * N), 256) + align_up(sf_atoms_plain_bytes(1, M, N, kFmtMXF8), 256);
  total += align_up(static_cast<size_t>(K * N), 256) + align_up(sf_atoms_plain_bytes(1, K, N, kFmtMXF8), 256);
  total += align_up(static_cast<size_t>(N * M), 256) + align_up(sf_atoms_plain_bytes(1, N, M, kFmtMXF8), 256);
  total += align_up(static_cast<size_t>(K * M), 256) + align_up(sf_atoms_plain_bytes(1, K, M, kFmtMXF8), 256);
  return total;
}

namespace {
// dX = dY . W and dW = dY^T . X from the four quantized operands.
bsmm_status backward_gemms(int64_t M, int64_t N, int64_t K, int ft, const void* dy_n, const void* dy_n_s,
                           const void* wt, const void* wt_s, const void* dyt, const void* dyt_s, const void* xt,
                           const void* xt_s, bool atoms, void* dX, void* dW, void* gws, cudaStream_t s) {
  std::string why;
  // dX [M, K] = dY [M, N] . (W^T [K, N])^T, contraction over N
  MxGemmRequest g1{1, M, K, N, dy_n, wt, ft, ft, static_cast<const uint8_t*>(dy_n_s),
                   static_cast<const uint8_t*>(wt_s), kFmtMXF8, dX, true, gws, N / 32, N / 32};
  g1.sf_atoms = atoms;
  cudaError_t e = launch_mx_gemm(g1, s, &why);
  if (e != cudaSuccess) return why.empty() ? cuda_fail(e, "dX gemm launch") : fail(BSMM_ERR_CUDA, why);
  // dW [N, K] = dY^T [N, M] . (X^T [K, M])^T, contraction over M
  MxGemmRequest g2{1, N, K, M, dyt, xt, ft, ft, static_cast<const uint8_t*>(dyt_s),
                   static_cast<const uint8_t*>(xt_s), kFmtMXF8, dW, true, gws, M / 32, M / 32};
  g2.sf_atoms = atoms;
  e = launch_mx_gemm(g2, s, &why);
  if (e != cudaSuccess) return why.empty() ? cuda_fail(e, "dW gemm launch") : fail(BSMM_ERR_CUDA, why);
  set_error("");
  return BSMM_OK;
}
}  // namespace

bsmm_status bsmm_linear_backward(const void* dY, const void* W, const void* X, int64_t M, int64_t N, int64_t K,
                                 bsmm_dtype fp8_type, void* dX, void* dW, void* workspace, size_t workspace_bytes,
                                 bsmm_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return fail(BSMM_ERR_INVALID_ARG, "negative size");
  if (fp8_type != BSMM_E5M2 && fp8_type != BSMM_E4M3) return fail(BSMM_ERR_INVALID_ARG, "fp8_type must be E5M2 or E4M3");
  if (M == 0 || N == 0 || K == 0) {
    set_error("");
    return BSMM_OK;
  }
  if (!dY || !W || !X || !dX || !dW) return fail(BSMM_ERR_INVALID_ARG, "null pointer");
  if (M % 32 || N % 32 || K % 32) return fail(BSMM_ERR_SHAPE, "M, N and K must be multiples of 32");
  if (!aligned16(dY) || !aligned16(W) || !aligned16(X) || !aligned16(dX) || !aligned16(dW))
    return fail(BSMM_ERR_ALIGNMENT, "pointers must be 16-byte aligned");
  const size_t need = bsmm_linear_backward_workspace_size(M, N, K);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(BSMM_ERR_WORKSPACE, "workspace must be 256-byte aligned and at least " + std::to_string(need) +
                                        " bytes");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* p = static_cast<uint8_t*>(workspace);
  auto take = [&](size_t bytes) {
    uint8_t* r = p;
    p += align_up(bytes, 256);
    return r;
  };
  uint8_t* dy_n = take(M * N);
  uint8_t* dy_n_s = take(sf_atoms_plain_bytes(1, M, N, kFmtMXF8));
  uint8_t* wt = take(K * N);
  uint8_t* wt_s = take(sf_atoms_plain_bytes(1, K, N, kFmtMXF8));
  uint8_t* dyt = take(N * M);
  uint8_t* dyt_s = take(sf_atoms_plain_bytes(1, N, M, kFmtMXF8));
  uint8_t* xt = take(K * M);
  uint8_t* xt_s = take(sf_atoms_plain_bytes(1, K, M, kFmtMXF8));

  // Each operand quantized along its GEMM's contraction axis, scales straight
  // into the tensor-core atom layout (no relayout before the GEMMs); dY's two
  // quantizations in one pass over it.
  const int ft = fp8_type;
  QuantRequest q_dyn, q_dyt;
  cudaError_t e = atoms_request(dY, true, 1, M, N, false, ft, BSMM_SCALE_UE8M0, dy_n, dy_n_s, s, &q_dyn);  // [M, N]
  if (e == cudaSuccess)
    e = atoms_request(dY, true, 1, N, M, true, ft, BSMM_SCALE_UE8M0, dyt, dyt_s, s, &q_dyt);  // dY^T [N, M]
  if (e == cudaSuccess) e = launch_quantize_dual(q_dyt, q_dyn, s);
  // W [N,K] along N -> W^T [K, N] and X [M,K] along M -> X^T [K, M], one launch
  QuantRequest q_wt, q_xt;
  if (e == cudaSuccess) e = atoms_request(W, true, 1, K, N, true, ft, BSMM_SCALE_UE8M0, wt, wt_s, s, &q_wt);
  if (e == cudaSuccess) e = atoms_request(X, true, 1, K, M, true, ft, BSMM_SCALE_UE8M0, xt, xt_s, s, &q_xt);
  if (e == cudaSuccess) e = launch_quantize_pair(q_wt, q_xt, s);
  if (e != cudaSuccess) return cuda_fail(e, "backward quantize launch");
  return backward_gemms(M, N, K, ft, dy_n, dy_n_s, wt, wt_s, dyt, dyt_s, xt, xt_s, true, dX, dW, nullptr, s);
}

size_t bsmm_linear_backward_quantized_workspace_size(int64_t M, int64_t N, int64_t K, int scales_are_atoms) {
  if (M <= 0 || N <= 0 || K <= 0 || scales_are_atoms) return 0;
  const size_t g1 = bsmm_gemm_workspace_size(1, M, K, N, BSMM_E4M3);
  const size_t g2 = bsmm_gemm_workspace_size(1, N, K, M, BSMM_E4M3);
  return g1 > g2 ? g1 : g2;
}

bsmm_status bsmm_linear_backward_quantized(int64_t M, int64_t N, int64_t K, bsmm_dtype fp8_type, const void* dy_n,
                                           const void* dy_n_scales, const void* w_t, const void* w_t_scales,
                                           const void* dy_t, const void* dy_t_scales, const void* x_t,
                                           const void* x_t_scales, int scales_are_atoms, void* dX, void* dW,
                                           void* workspace, size_t workspace_bytes, bsmm_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return fail(BSMM_ERR_INVALID_ARG, "negative size");
  if (fp8_type != BSMM_E5M2 && fp8_type != BSMM_E4M3) return fail(BSMM_ERR_INVALID_ARG, "fp8_type must be E5M2 or E4M3");
  if (M == 0 || N == 0 || K == 0) {
    set_error("");
    return BSMM_OK;
  }
  if (!dy_n || !dy_n_scales || !w_t || !w_t_scales || !dy_t || !dy_t_scales || !x_t || !x_t_scales || !dX || !dW)
    return fail(BSMM_ERR_INVALID_ARG, "null pointer");
  if (M % 32 || N % 32 || K % 32) return fail(BSMM_ERR_SHAPE, "M, N and K must be multiples of 32");
  for (const void* q : {dy_n, w_t, dy_t, x_t, static_cast<const void*>(dX), static_cast<const void*>(dW)})
    if (!aligned16(q)) return fail(BSMM_ERR_ALIGNMENT, "codes and outputs must be 16-byte aligned");
  if (scales_are_atoms)
    for (const void* q : {dy_n_scales, w_t_scales, dy_t_scales, x_t_scales})
      if (!aligned16(q)) return fail(BSMM_ERR_ALIGNMENT, "atoms must be 16-byte aligned");
  const size_t need = bsmm_linear_backward_quantized_workspace_size(M, N, K, scales_are_atoms);
  if (need && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return fail(BSMM_ERR_WORKSPACE, "workspace must be 256-byte aligned and at least " + std::to_string(need) +
                                        " bytes");
  return backward_gemms(M, N, K, fp8_type, dy_n, dy_n_scales, w_t, w_t_scales, dy_t, dy_t_scales, x_t, x_t_scales,
                        scales_are_atoms != 0, dX, dW, workspace, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
