// C ABI of libbsmm.so: argument validation, per-device state, TMA descriptor
// factory and dispatch to the kernels.  No exception crosses this boundary.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

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

bsmm_status bsmm_quantize(const void* x, bsmm_dtype x_type, int64_t rows, int64_t cols, int64_t ld_x,
                          int block_rows, int block_cols, bsmm_dtype code_type, bsmm_scale_type scale_type,
                          int transpose_out, void* codes, int64_t ld_codes, void* scales, int64_t ld_scales,
                          bsmm_stream_t stream) {
  if (x_type != BSMM_F32 && x_type != BSMM_BF16) return fail(BSMM_ERR_INVALID_ARG, "x_type must be F32 or BF16");
  if (!is_code(code_type)) return fail(BSMM_ERR_INVALID_ARG, "code_type must be E4M3, E5M2, E2M1 or INT8");
  if (!is_scale(scale_type)) return fail(BSMM_ERR_INVALID_ARG, "bad scale_type");
  if (rows < 0 || cols < 0) return fail(BSMM_ERR_INVALID_ARG, "negative size");
  if (rows == 0 || cols == 0) {
    set_error("");
    return BSMM_OK;
  }
  if (!x || !codes || !scales) return fail(BSMM_ERR_INVALID_ARG, "null pointer");
  if (block_rows < 1 || block_cols < 1) return fail(BSMM_ERR_INVALID_ARG, "block sizes must be positive");
  if (rows % block_rows || cols % block_cols) return fail(BSMM_ERR_SHAPE, "rows/cols not divisible by the block");
  if (code_type == BSMM_INT8 && scale_type != BSMM_SCALE_F32)
    return fail(BSMM_ERR_UNSUPPORTED, "INT8 codes take F32 scales");
  if (transpose_out && block_cols != 1) return fail(BSMM_ERR_UNSUPPORTED, "transposed output needs column blocks");
  if (ld_x < cols) return fail(BSMM_ERR_SHAPE, "ld_x < cols");
  const int64_t out_cols = transpose_out ? rows : cols, out_rows = transpose_out ? cols : rows;
  if (ld_codes < out_cols) return fail(BSMM_ERR_SHAPE, "ld_codes too small");
  const int64_t s_rows = transpose_out ? cols / block_cols : rows / block_rows;
  const int64_t s_cols = transpose_out ? rows / block_rows : cols / block_cols;
  if (ld_scales < s_cols) return fail(BSMM_ERR_SHAPE, "ld_scales too small");
  (void)s_rows;
  (void)out_rows;
  if (code_type == BSMM_E2M1) {
    if (ld_codes % 2 || out_cols % 2) return fail(BSMM_ERR_SHAPE, "E2M1 codes need an even contiguous extent");
    // Column blocks written untransposed are packed across lanes by the
    // column kernels; every other layout packs within one block.
    const bool pow2r = block_rows == 16 || block_rows == 32 || block_rows == 64 || block_rows == 128;
    const bool paired = !transpose_out && block_cols == 1 && (pow2r || block_rows == rows);
    const int ext = transpose_out ? block_rows : block_cols;
    if (ext % 2 && !paired)
      return fail(BSMM_ERR_UNSUPPORTED, "E2M1 blocks need an even extent along the contiguous axis");
  }
  QuantRequest q{x, x_type == BSMM_BF16, rows, cols, ld_x, block_rows, block_cols, code_type, scale_type,
                 transpose_out != 0, codes, ld_codes, scales, ld_scales};
  return launched(launch_quantize(q, reinterpret_cast<cudaStream_t>(stream)), "quantize launch");
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
  // codes: dY along N [M,N], W^T [K,N], dY^T [N,M], X^T [K,M]; UE8M0 scales of each
  size_t total = 0;
  total += align_up(static_cast<size_t>(M * N), 256) + align_up(static_cast<size_t>(M * (N / 32)), 256);
  total += align_up(static_cast<size_t>(K * N), 256) + align_up(static_cast<size_t>(K * (N / 32)), 256);
  total += align_up(static_cast<size_t>(N * M), 256) + align_up(static_cast<size_t>(N * (M / 32)), 256);
  total += align_up(static_cast<size_t>(K * M), 256) + align_up(static_cast<size_t>(K * (M / 32)), 256);
  const size_t g1 = bsmm_gemm_workspace_size(1, M, K, N, BSMM_E4M3);
  const size_t g2 = bsmm_gemm_workspace_size(1, N, K, M, BSMM_E4M3);
  total += align_up(g1 > g2 ? g1 : g2, 256);
  return total;
}

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
  uint8_t* dy_n_s = take(M * (N / 32));
  uint8_t* wt = take(K * N);
  uint8_t* wt_s = take(K * (N / 32));
  uint8_t* dyt = take(N * M);
  uint8_t* dyt_s = take(N * (M / 32));
  uint8_t* xt = take(K * M);
  uint8_t* xt_s = take(K * (M / 32));
  uint8_t* gws = p;
  const size_t gws_bytes = workspace_bytes - static_cast<size_t>(gws - static_cast<uint8_t*>(workspace));

  const int ft = fp8_type;
  struct Q {
    const void* x;
    int64_t rows, cols;
    int br, bc, tr;
    uint8_t *codes, *scales;
    int64_t ldc, lds;
  } qs[4] = {
      {dY, M, N, 1, 32, 0, dy_n, dy_n_s, N, N / 32},  // dY along N          -> [M, N]
      {W, N, K, 32, 1, 1, wt, wt_s, N, N / 32},       // W along N, transposed -> [K, N]
      {dY, M, N, 32, 1, 1, dyt, dyt_s, M, M / 32},    // dY along M, transposed -> [N, M]
      {X, M, K, 32, 1, 1, xt, xt_s, M, M / 32},       // X along M, transposed  -> [K, M]
  };
  for (const Q& q : qs) {
    QuantRequest r{q.x, true, q.rows, q.cols, q.cols, q.br, q.bc, ft, BSMM_SCALE_UE8M0, q.tr != 0,
                   q.codes, q.ldc, q.scales, q.lds};
    const cudaError_t e = launch_quantize(r, s);
    if (e != cudaSuccess) return cuda_fail(e, "backward quantize launch");
  }
  std::string why;
  // dX [M, K] = dY [M, N] . (W^T [K, N])^T, contraction over N
  MxGemmRequest g1{1, M, K, N, dy_n, wt, ft, ft, dy_n_s, wt_s, kFmtMXF8, dX, true, gws, N / 32, N / 32};
  cudaError_t e = launch_mx_gemm(g1, s, &why);
  if (e != cudaSuccess) return why.empty() ? cuda_fail(e, "dX gemm launch") : fail(BSMM_ERR_CUDA, why);
  // dW [N, K] = dY^T [N, M] . (X^T [K, M])^T, contraction over M
  MxGemmRequest g2{1, N, K, M, dyt, xt, ft, ft, dyt_s, xt_s, kFmtMXF8, dW, true, gws, M / 32, M / 32};
  e = launch_mx_gemm(g2, s, &why);
  if (e != cudaSuccess) return why.empty() ? cuda_fail(e, "dW gemm launch") : fail(BSMM_ERR_CUDA, why);
  (void)gws_bytes;
  set_error("");
  return BSMM_OK;
}

}  // extern "C"
