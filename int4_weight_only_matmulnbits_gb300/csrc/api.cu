// C ABI of the MatMulNBits library (declared in include/mnb.h): argument
// validation, path dispatch and launch-error reporting. Every check happens
// on the host before anything is enqueued; nothing here falls back to a CPU
// computation.
#include <atomic>
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "../../include/mnb.h"
#include "mnb_common.cuh"
#include "mnb_launch.h"

namespace mnb {

namespace {
std::atomic<int> g_pdl{1};
thread_local char g_last_error[256] = "";

mnb_status cuda_fail(cudaError_t e, const char *where) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where,
                cudaGetErrorName(e), cudaGetErrorString(e));
  return MNB_ERR_CUDA;
}

bool valid_block_size(int bs) {
  return bs >= 16 && bs <= 256 && (bs & (bs - 1)) == 0;
}

bool valid_dtype(int d) { return d == MNB_F32 || d == MNB_BF16; }

size_t dtype_size(int d) { return d == MNB_F32 ? 4 : 2; }

bool aligned(const void *p, size_t a) {
  return reinterpret_cast<uintptr_t>(p) % a == 0;
}

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a);
  const uintptr_t y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

struct Sizes {
  size_t b, s, z;
};

// Bytes of the packed codes; packed_b holds them, then the header.
size_t codes_bytes(int64_t N, int64_t K) {
  return size_t(ceil_div(N, kTileN)) * ceil_div(K, kChunkK) * kChunkBytes;
}

Sizes packed_sizes(int64_t N, int64_t K, int bs, int scale_dtype, bool zp) {
  const int64_t N16 = ceil_div(N, kTileN);
  const int64_t nb = ceil_div(K, bs);
  Sizes s;
  s.b = codes_bytes(N, K) + MNB_PACKED_HEADER_BYTES;
  s.s = size_t(N16) * nb * kTileN * dtype_size(scale_dtype);
  s.z = zp ? size_t(N16) * ceil_div(nb, 2) * 2 * 8 : 0;
  return s;
}

// Largest sizes the kernels index with 32-bit arithmetic.
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

mnb_status check_shape(int64_t N, int64_t K, int bs, int scale_dtype) {
  if (N < 1 || K < 1 || N > kMaxDim || K > kMaxDim) return MNB_ERR_SHAPE;
  if (ceil_div(N, kTileN) * ceil_div(K, kChunkK) > (int64_t(1) << 40))
    return MNB_ERR_SHAPE;
  if (!valid_block_size(bs)) return MNB_ERR_BLOCKSIZE;
  if (!valid_dtype(scale_dtype)) return MNB_ERR_DTYPE;
  return MNB_OK;
}

// ---- packed-weight headers and their host-side records ---------------------

static_assert(sizeof(mnb_packed_header) == 80, "mnb_packed_header layout");
static_assert(sizeof(mnb_packed_header) <= MNB_PACKED_HEADER_BYTES, "header room");

uint64_t header_check(const mnb_packed_header &h) {
  const unsigned char *b = reinterpret_cast<const unsigned char *>(&h);
  uint64_t x = 1469598103934665603ull;  // FNV-1a 64
  for (size_t i = 0; i < offsetof(mnb_packed_header, check); ++i) {
    x ^= b[i];
    x *= 1099511628211ull;
  }
  return x;
}

mnb_packed_header make_header(int64_t N, int64_t K, int bs, int scale_dtype, bool zp,
                              int codes) {
  mnb_packed_header h;
  std::memset(&h, 0, sizeof h);
  h.magic = MNB_PACKED_MAGIC;
  h.version = MNB_PACKED_VERSION;
  h.codes = static_cast<uint32_t>(codes);
  h.N = N;
  h.K = K;
  h.block_size = bs;
  h.scale_dtype = scale_dtype;
  h.has_zero_points = zp ? 1 : 0;
  const Sizes z = packed_sizes(N, K, bs, scale_dtype, zp);
  h.packed_b_bytes = z.b;
  h.packed_scales_bytes = z.s;
  h.packed_zp_bytes = z.z;
  h.check = header_check(h);
  return h;
}

// A header some prepack call could have written, with a matching check.
mnb_status header_valid(const mnb_packed_header &h) {
  if (h.magic != MNB_PACKED_MAGIC || h.version != MNB_PACKED_VERSION ||
      h.check != header_check(h)) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "not a packed-weight header of this library (magic, version or check)");
    return MNB_ERR_LAYOUT;
  }
  const bool ok_codes = h.codes == MNB_CODES_AFFINE ||
                        (h.codes == MNB_CODES_CODEBOOK && h.has_zero_points == 0);
  if (!ok_codes || (h.has_zero_points != 0 && h.has_zero_points != 1) || h.reserved != 0 ||
      check_shape(h.N, h.K, h.block_size, h.scale_dtype) != MNB_OK) {
    std::snprintf(g_last_error, sizeof g_last_error, "packed-weight header with invalid fields");
    return MNB_ERR_LAYOUT;
  }
  const Sizes z = packed_sizes(h.N, h.K, h.block_size, h.scale_dtype, h.has_zero_points != 0);
  if (h.packed_b_bytes != z.b || h.packed_scales_bytes != z.s || h.packed_zp_bytes != z.z) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "packed-weight header sizes do not match its shape");
    return MNB_ERR_LAYOUT;
  }
  return MNB_OK;
}

std::mutex g_headers_mu;
std::unordered_map<uintptr_t, mnb_packed_header> g_headers;

void record_header(const void *packed_b, const mnb_packed_header &h) {
  std::lock_guard<std::mutex> lock(g_headers_mu);
  g_headers[reinterpret_cast<uintptr_t>(packed_b)] = h;
}

const char *dtype_name(int d) { return d == MNB_F32 ? "fp32" : "bf16"; }

// The header recorded for packed_b against what a call passes.
mnb_status check_layout(const void *packed_b, int64_t N, int64_t K, int bs, int scale_dtype,
                        bool zp, int codes) {
  mnb_packed_header h;
  {
    std::lock_guard<std::mutex> lock(g_headers_mu);
    const auto it = g_headers.find(reinterpret_cast<uintptr_t>(packed_b));
    if (it == g_headers.end()) {
      std::snprintf(g_last_error, sizeof g_last_error,
                    "no packed-weight header is recorded for %p: pack it with a prepack "
                    "call, or register the header stored with it",
                    packed_b);
      return MNB_ERR_LAYOUT;
    }
    h = it->second;
  }
  const char *field = h.N != N                             ? "N"
                      : h.K != K                           ? "K"
                      : h.block_size != bs                 ? "block_size"
                      : h.scale_dtype != scale_dtype       ? "scale dtype"
                      : (h.has_zero_points != 0) != zp     ? "zero-point presence"
                      : static_cast<int>(h.codes) != codes ? "code form"
                                                           : nullptr;
  if (!field) return MNB_OK;
  std::snprintf(g_last_error, sizeof g_last_error,
                "packed weight %p differs in %s: packed as N=%lld K=%lld bs=%d scales %s, "
                "%s zero points, %s codes; called with N=%lld K=%lld bs=%d scales %s, %s "
                "zero points, %s codes",
                packed_b, field, (long long)h.N, (long long)h.K, h.block_size,
                dtype_name(h.scale_dtype), h.has_zero_points ? "with" : "no",
                h.codes == MNB_CODES_AFFINE ? "affine" : "code-book", (long long)N,
                (long long)K, bs, dtype_name(scale_dtype), zp ? "with" : "no",
                codes == MNB_CODES_AFFINE ? "affine" : "code-book");
  return MNB_ERR_LAYOUT;
}

mnb_status check_device() {
  int dev = 0, major = 0, minor = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess)
    err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (err == cudaSuccess)
    err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (err != cudaSuccess) return cuda_fail(err, "device query");
  if (major != 10 || minor != 3) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "device is sm_%d%d; this library is built for sm_103a",
                  major, minor);
    return MNB_ERR_DEVICE;
  }
  return MNB_OK;
}

mnb_status check_outputs_disjoint(void *const outs[3], const size_t out_n[3],
                                  const void *const ins[3],
                                  const size_t in_n[3]) {
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 3; ++j)
      if (overlap(outs[i], out_n[i], ins[j], in_n[j])) return MNB_ERR_ALIAS;
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i], out_n[i], outs[j], out_n[j])) return MNB_ERR_ALIAS;
  }
  return MNB_OK;
}

// Argument checks of a product (no device query).
mnb_status validate_matmul_args(const void *A, const void *packed_b,
                                const void *scales, const void *zero_points,
                                const float *bias, int64_t M, int64_t N, int64_t K,
                                int block_size, const void *Y, int a_dtype,
                                int scale_dtype, int path) {
  if (!A || !packed_b || !scales || !Y) return MNB_ERR_NULL;
  if (M < 1 || M > kMaxDim) return MNB_ERR_SHAPE;
  mnb_status st = check_shape(N, K, block_size, scale_dtype);
  if (st != MNB_OK) return st;
  if (!valid_dtype(a_dtype)) return MNB_ERR_DTYPE;
  if (path != MNB_PATH_AUTO && path != MNB_PATH_GEMV && path != MNB_PATH_GEMM &&
      path != MNB_PATH_GEMM_STREAMK && path != MNB_PATH_GEMM_PAIR)
    return MNB_ERR_UNSUPPORTED;
  if (path == MNB_PATH_GEMV && M > kGemvMaxM) return MNB_ERR_UNSUPPORTED;
  const size_t es = dtype_size(a_dtype);
  if (!aligned(A, es) || !aligned(Y, es) || !aligned(packed_b, 16) ||
      !aligned(scales, 16) || (zero_points && !aligned(zero_points, 16)) ||
      (bias && !aligned(bias, 4)))
    return MNB_ERR_ALIGN;
  const Sizes in = packed_sizes(N, K, block_size, scale_dtype, zero_points != nullptr);
  const size_t y_bytes = size_t(M) * N * es;
  const void *ins[5] = {A, packed_b, scales, zero_points, bias};
  const size_t in_n[5] = {size_t(M) * K * es, in.b, in.s, in.z,
                          bias ? size_t(N) * 4 : 0};
  for (int j = 0; j < 5; ++j)
    if (overlap(Y, y_bytes, ins[j], in_n[j])) return MNB_ERR_ALIAS;
  return MNB_OK;
}

// Argument checks and the packed weight's recorded header (host only).
mnb_status validate_matmul_host(const void *A, const void *packed_b, const void *scales,
                                const void *zero_points, const float *bias, int64_t M,
                                int64_t N, int64_t K, int block_size, const void *Y,
                                int a_dtype, int scale_dtype, int path,
                                int codes = MNB_CODES_AFFINE) {
  const mnb_status st = validate_matmul_args(A, packed_b, scales, zero_points, bias, M, N, K,
                                             block_size, Y, a_dtype, scale_dtype, path);
  if (st != MNB_OK) return st;
  return check_layout(packed_b, N, K, block_size, scale_dtype, zero_points != nullptr, codes);
}

mnb_status validate_matmul(const void *A, const void *packed_b,
                           const void *scales, const void *zero_points,
                           const float *bias, int64_t M, int64_t N, int64_t K,
                           int block_size, const void *Y, int a_dtype,
                           int scale_dtype, int path, int codes = MNB_CODES_AFFINE) {
  const mnb_status st = validate_matmul_host(A, packed_b, scales, zero_points, bias, M, N, K,
                                             block_size, Y, a_dtype, scale_dtype, path, codes);
  return st != MNB_OK ? st : check_device();
}

mnb_status run_matmul(const void *A, const void *packed_b, const void *scales,
                      const void *zero_points, const float *bias, int64_t M,
                      int64_t N, int64_t K, int block_size, void *Y,
                      int a_dtype, int scale_dtype, int path,
                      cudaStream_t stream, void *ws = nullptr, size_t ws_bytes = 0) {
  MatmulArgs a{A, packed_b, scales, zero_points, bias, Y, M, N, K, block_size,
               a_dtype == MNB_F32, scale_dtype == MNB_F32, g_pdl.load() != 0};
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.sk_only = path == MNB_PATH_GEMM_STREAMK;
  cudaError_t e;
  if (path == MNB_PATH_GEMV || (path == MNB_PATH_AUTO && M <= kGemvMaxM)) {
    e = launch_gemv(a, stream);
  } else if (path == MNB_PATH_GEMM_PAIR) {
    e = launch_gemm_pair(a, stream);
  } else if (path == MNB_PATH_GEMM || path == MNB_PATH_GEMM_STREAMK || gemm_supports(a)) {
    e = launch_gemm(a, stream);
  } else {
    // Activations the tensor-core kernel cannot stage (fp32, or rows that
    // are not 16-byte aligned): the decode kernel over 16-row slices.
    const size_t es = dtype_size(a_dtype);
    e = cudaSuccess;
    for (int64_t m0 = 0; m0 < M && e == cudaSuccess; m0 += kGemvMaxM) {
      MatmulArgs s = a;
      s.A = static_cast<const char *>(A) + size_t(m0) * K * es;
      s.Y = static_cast<char *>(Y) + size_t(m0) * N * es;
      s.M = M - m0 < kGemvMaxM ? M - m0 : kGemvMaxM;
      e = launch_gemv(s, stream);
    }
  }
  if (e == cudaErrorNotSupported) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "no kernel for M=%lld N=%lld K=%lld bs=%d", (long long)M,
                  (long long)N, (long long)K, block_size);
    return MNB_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return cuda_fail(e, "mnb_matmul");
  return MNB_OK;
}

// The Python binding mirrors these two structs field by field.
static_assert(sizeof(mnb_chain_op) == 112, "mnb_chain_op layout");
static_assert(sizeof(mnb_chain_info) == 72, "mnb_chain_info layout");

uint64_t chain_checksum(const mnb_chain_info &i) {
  const int64_t f[] = {static_cast<int64_t>(i.plan_bytes), i.n_ops, i.n_segments, i.grid,
                       i.smem_bytes, i.M, i.block_size, i.a_dtype, i.scale_dtype,
                       i.has_zero_points, i.ring_stages, i.k_max, i.tiles_per_segment,
                       i.ctas_per_sm};
  uint64_t h = 1469598103934665603ull;  // FNV-1a over the fields
  for (int64_t v : f)
    for (int b = 0; b < 8; ++b) {
      h ^= static_cast<uint64_t>(v >> (8 * b)) & 0xFFu;
      h *= 1099511628211ull;
    }
  return h;
}

// Memory ranges an op reads (A, weights, biases) and writes (Y).
struct OpRanges {
  const void *a, *y, *w[8];
  size_t na, ny, nw[8];
};

OpRanges op_ranges(const mnb_chain_op &o, int64_t M, int bs, int a_dtype, int scale_dtype) {
  OpRanges r{};
  const size_t es = dtype_size(a_dtype);
  r.a = o.A;
  r.na = size_t(M) * o.K * es;
  r.y = o.Y;
  r.ny = size_t(M) * o.N * es;
  const Sizes sz = packed_sizes(o.N, o.K, bs, scale_dtype, o.packed_zp != nullptr);
  const void *w[8] = {o.packed_b, o.packed_scales, o.packed_zp, o.bias,
                      o.packed_b_up, o.packed_scales_up, o.packed_zp_up, o.bias_up};
  const size_t nw[8] = {sz.b, sz.s, sz.z, o.bias ? size_t(o.N) * 4 : 0,
                        o.packed_b_up ? sz.b : 0, o.packed_b_up ? sz.s : 0,
                        o.packed_zp_up ? sz.z : 0, o.bias_up ? size_t(o.N) * 4 : 0};
  for (int i = 0; i < 8; ++i) {
    r.w[i] = w[i];
    r.nw[i] = w[i] ? nw[i] : 0;
  }
  return r;
}

}  // namespace

int sm_count() {
  static std::once_flag once;
  static int count = 148;
  std::call_once(once, [] {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev);
  });
  return count;
}

}  // namespace mnb

using namespace mnb;

extern "C" {

const char *mnb_status_string(int status) {
  switch (status) {
    case MNB_OK: return "MNB_OK";
    case MNB_ERR_NULL: return "MNB_ERR_NULL: a required pointer is NULL";
    case MNB_ERR_SHAPE: return "MNB_ERR_SHAPE: M, N or K out of range";
    case MNB_ERR_BLOCKSIZE:
      return "MNB_ERR_BLOCKSIZE: block_size must be a power of two in [16, 256]";
    case MNB_ERR_DTYPE: return "MNB_ERR_DTYPE: unknown or unsupported dtype";
    case MNB_ERR_ALIGN: return "MNB_ERR_ALIGN: a pointer breaks its alignment rule";
    case MNB_ERR_ALIAS: return "MNB_ERR_ALIAS: an output overlaps an input";
    case MNB_ERR_CUDA: return "MNB_ERR_CUDA: a CUDA launch or copy failed";
    case MNB_ERR_UNSUPPORTED:
      return "MNB_ERR_UNSUPPORTED: no kernel serves this combination";
    case MNB_ERR_DEVICE: return "MNB_ERR_DEVICE: current device is not sm_103";
    case MNB_ERR_LAYOUT:
      return "MNB_ERR_LAYOUT: the packed weight does not match the call, or has no header";
    default: return "unknown mnb_status";
  }
}

const char *mnb_last_error_string(void) { return g_last_error; }

int mnb_version(void) { return (1 << 16) | 0; }

void mnb_set_programmatic_launch(int enable) { g_pdl.store(enable ? 1 : 0); }

void mnb_test_wait_fault(int stop_stage) { gemv_set_wait_fault(stop_stage); }

mnb_status mnb_fault_status(unsigned int *fault_bits) {
  if (!fault_bits) return MNB_ERR_NULL;
  unsigned int a = 0, b = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = gemv_take_fault(&a);
  if (e == cudaSuccess) e = gemm_take_fault(&b);
  unsigned int c = 0, d = 0;
  if (e == cudaSuccess) e = chain_take_fault(&c);
  if (e == cudaSuccess) e = pair_take_fault(&d);
  if (e != cudaSuccess) return cuda_fail(e, "mnb_fault_status");
  *fault_bits = a | b | c | d;
  return MNB_OK;
}

mnb_status mnb_packed_header_make(int64_t N, int64_t K, int block_size, mnb_dtype scale_dtype,
                                  int has_zero_points, int codes, mnb_packed_header *out) {
  if (!out) return MNB_ERR_NULL;
  const mnb_status st = check_shape(N, K, block_size, scale_dtype);
  if (st != MNB_OK) return st;
  if ((codes != MNB_CODES_AFFINE && codes != MNB_CODES_CODEBOOK) ||
      (codes == MNB_CODES_CODEBOOK && has_zero_points))
    return MNB_ERR_UNSUPPORTED;
  *out = make_header(N, K, block_size, scale_dtype, has_zero_points != 0, codes);
  return MNB_OK;
}

mnb_status mnb_packed_register(const void *packed_b, const mnb_packed_header *header) {
  if (!packed_b || !header) return MNB_ERR_NULL;
  const mnb_status st = header_valid(*header);
  if (st != MNB_OK) return st;
  record_header(packed_b, *header);
  return MNB_OK;
}

mnb_status mnb_packed_read_header(const void *packed_b, size_t packed_b_bytes,
                                  mnb_packed_header *out, mnb_stream_t stream) {
  if (!packed_b || !out) return MNB_ERR_NULL;
  if (packed_b_bytes < MNB_PACKED_HEADER_BYTES) return MNB_ERR_SHAPE;
  mnb_status st = check_device();
  if (st != MNB_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mnb_packed_header h;
  cudaError_t e = cudaMemcpyAsync(
      &h, static_cast<const char *>(packed_b) + (packed_b_bytes - MNB_PACKED_HEADER_BYTES),
      sizeof h, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "mnb_packed_read_header");
  st = header_valid(h);
  if (st != MNB_OK) return st;
  if (h.packed_b_bytes != packed_b_bytes) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "the header gives packed_b %llu bytes, the call %llu",
                  (unsigned long long)h.packed_b_bytes, (unsigned long long)packed_b_bytes);
    return MNB_ERR_SHAPE;
  }
  *out = h;
  return MNB_OK;
}

mnb_status mnb_packed_forget(const void *packed_b) {
  if (!packed_b) return MNB_ERR_NULL;
  std::lock_guard<std::mutex> lock(g_headers_mu);
  g_headers.erase(reinterpret_cast<uintptr_t>(packed_b));
  return MNB_OK;
}

mnb_status mnb_prepacked_sizes(int64_t N, int64_t K, int block_size,
                               mnb_dtype scale_dtype, int has_zero_points,
                               size_t *packed_b_bytes,
                               size_t *packed_scales_bytes,
                               size_t *packed_zp_bytes) {
  if (!packed_b_bytes || !packed_scales_bytes || !packed_zp_bytes)
    return MNB_ERR_NULL;
  const mnb_status st = check_shape(N, K, block_size, scale_dtype);
  if (st != MNB_OK) return st;
  const Sizes s = packed_sizes(N, K, block_size, scale_dtype, has_zero_points != 0);
  *packed_b_bytes = s.b;
  *packed_scales_bytes = s.s;
  *packed_zp_bytes = s.z;
  return MNB_OK;
}

mnb_status mnb_prepack(const uint8_t *B, const void *scales,
                       const uint8_t *zero_points, int64_t N, int64_t K,
                       int block_size, mnb_dtype scale_dtype, void *packed_b,
                       void *packed_scales, void *packed_zp,
                       mnb_stream_t stream) {
  if (!B || !scales || !packed_b || !packed_scales) return MNB_ERR_NULL;
  if (zero_points && !packed_zp) return MNB_ERR_NULL;
  mnb_status st = check_shape(N, K, block_size, scale_dtype);
  if (st != MNB_OK) return st;
  if (!aligned(packed_b, 16) || !aligned(packed_scales, 16) ||
      (zero_points && !aligned(packed_zp, 16)) ||
      !aligned(scales, dtype_size(scale_dtype)))
    return MNB_ERR_ALIGN;
  const int64_t nb = ceil_div(K, block_size);
  const Sizes out = packed_sizes(N, K, block_size, scale_dtype, zero_points != nullptr);
  const void *const ins[3] = {B, scales, zero_points};
  const size_t in_n[3] = {size_t(N) * nb * (block_size / 2),
                          size_t(N) * nb * dtype_size(scale_dtype),
                          zero_points ? size_t(N) * ((nb + 1) / 2) : 0};
  void *const outs[3] = {packed_b, packed_scales, zero_points ? packed_zp : nullptr};
  const size_t out_n[3] = {out.b, out.s, out.z};
  st = check_outputs_disjoint(outs, out_n, ins, in_n);
  if (st != MNB_OK) return st;
  st = check_device();
  if (st != MNB_OK) return st;
  PrepackArgs a{B, scales, zero_points, N, K, block_size,
                scale_dtype == MNB_F32, packed_b, packed_scales, packed_zp};
  a.header = make_header(N, K, block_size, scale_dtype, zero_points != nullptr,
                         MNB_CODES_AFFINE);
  a.header_dst = static_cast<char *>(packed_b) + codes_bytes(N, K);
  const cudaError_t e = launch_prepack(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mnb_prepack");
  record_header(packed_b, a.header);
  return MNB_OK;
}

mnb_status mnb_prepack_qdq(const uint8_t *B_qdq, const void *scales,
                           const uint8_t *zero_points, int axis, int64_t N, int64_t K,
                           int block_size, mnb_dtype scale_dtype, void *packed_b,
                           void *packed_scales, void *packed_zp, mnb_stream_t stream) {
  if (!B_qdq || !scales || !packed_b || !packed_scales || !packed_zp) return MNB_ERR_NULL;
  if (axis != 0 && axis != 1) return MNB_ERR_SHAPE;
  mnb_status st = check_shape(N, K, block_size, scale_dtype);
  if (st != MNB_OK) return st;
  if (!aligned(packed_b, 16) || !aligned(packed_scales, 16) || !aligned(packed_zp, 16) ||
      !aligned(scales, dtype_size(scale_dtype)))
    return MNB_ERR_ALIGN;
  const int64_t nb = ceil_div(K, block_size);
  const Sizes out = packed_sizes(N, K, block_size, scale_dtype, true);
  const void *const ins[3] = {B_qdq, scales, zero_points};
  const size_t in_n[3] = {size_t((K * N + 1) / 2), size_t(N) * nb * dtype_size(scale_dtype),
                          zero_points ? size_t((nb * N + 1) / 2) : 0};
  void *const outs[3] = {packed_b, packed_scales, packed_zp};
  const size_t out_n[3] = {out.b, out.s, out.z};
  st = check_outputs_disjoint(outs, out_n, ins, in_n);
  if (st != MNB_OK) return st;
  st = check_device();
  if (st != MNB_OK) return st;
  PrepackArgs a{B_qdq, scales, zero_points, N, K, block_size,
                scale_dtype == MNB_F32, packed_b, packed_scales, packed_zp};
  a.qdq_axis = axis;
  a.header = make_header(N, K, block_size, scale_dtype, true, MNB_CODES_AFFINE);
  a.header_dst = static_cast<char *>(packed_b) + codes_bytes(N, K);
  const cudaError_t e = launch_prepack(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mnb_prepack_qdq");
  record_header(packed_b, a.header);
  return MNB_OK;
}

mnb_status mnb_unprepack(const void *packed_b, const void *packed_scales,
                         const void *packed_zp, int64_t N, int64_t K,
                         int block_size, mnb_dtype scale_dtype, uint8_t *B,
                         void *scales, uint8_t *zero_points,
                         mnb_stream_t stream) {
  if (!packed_b || !packed_scales || !B || !scales) return MNB_ERR_NULL;
  if (packed_zp && !zero_points) return MNB_ERR_NULL;
  mnb_status st = check_shape(N, K, block_size, scale_dtype);
  if (st != MNB_OK) return st;
  if (!aligned(packed_b, 16) || !aligned(packed_scales, 16) ||
      (packed_zp && !aligned(packed_zp, 16)) ||
      !aligned(scales, dtype_size(scale_dtype)))
    return MNB_ERR_ALIGN;
  const int64_t nb = ceil_div(K, block_size);
  const Sizes in = packed_sizes(N, K, block_size, scale_dtype, packed_zp != nullptr);
  const void *const ins[3] = {packed_b, packed_scales, packed_zp};
  const size_t in_n[3] = {in.b, in.s, in.z};
  void *const outs[3] = {B, scales, packed_zp ? zero_points : nullptr};
  const size_t out_n[3] = {size_t(N) * nb * (block_size / 2),
                           size_t(N) * nb * dtype_size(scale_dtype),
                           packed_zp ? size_t(N) * ((nb + 1) / 2) : 0};
  st = check_outputs_disjoint(outs, out_n, ins, in_n);
  if (st != MNB_OK) return st;
  st = check_layout(packed_b, N, K, block_size, scale_dtype, packed_zp != nullptr,
                    MNB_CODES_AFFINE);
  if (st == MNB_ERR_LAYOUT && packed_zp == nullptr)  // the bitsandbytes-style plan
    st = check_layout(packed_b, N, K, block_size, scale_dtype, false, MNB_CODES_CODEBOOK);
  if (st != MNB_OK) return st;
  st = check_device();
  if (st != MNB_OK) return st;
  UnprepackArgs a{packed_b, packed_scales, packed_zp, N, K, block_size,
                  scale_dtype == MNB_F32, B, scales, zero_points};
  const cudaError_t e = launch_unprepack(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mnb_unprepack");
  return MNB_OK;
}

mnb_status mnb_matmul_path(const void *A, const void *packed_b,
                           const void *scales, const void *zero_points,
                           const float *bias, int64_t M, int64_t N, int64_t K,
                           int block_size, void *Y, mnb_dtype a_dtype,
                           mnb_dtype scale_dtype, mnb_path path,
                           mnb_stream_t stream) {
  const mnb_status st = validate_matmul(A, packed_b, scales, zero_points, bias,
                                        M, N, K, block_size, Y, a_dtype,
                                        scale_dtype, path);
  if (st != MNB_OK) return st;
  return run_matmul(A, packed_b, scales, zero_points, bias, M, N, K,
                    block_size, Y, a_dtype, scale_dtype, path,
                    reinterpret_cast<cudaStream_t>(stream));
}

static_assert(sizeof(mnb_matmul_plan_info) == 40, "mnb_matmul_plan_info layout");

mnb_status mnb_matmul_plan(int64_t M, int64_t N, int64_t K, int block_size,
                           mnb_dtype a_dtype, mnb_dtype scale_dtype, int has_zero_points,
                           mnb_path path, size_t workspace_bytes, int sm_count_in,
                           mnb_matmul_plan_info *out) {
  if (!out) return MNB_ERR_NULL;
  if (M < 1 || M > kMaxDim) return MNB_ERR_SHAPE;
  mnb_status st = check_shape(N, K, block_size, scale_dtype);
  if (st != MNB_OK) return st;
  if (!valid_dtype(a_dtype)) return MNB_ERR_DTYPE;
  if (path != MNB_PATH_AUTO && path != MNB_PATH_GEMV && path != MNB_PATH_GEMM &&
      path != MNB_PATH_GEMM_STREAMK && path != MNB_PATH_GEMM_PAIR)
    return MNB_ERR_UNSUPPORTED;
  if (path == MNB_PATH_GEMV && M > kGemvMaxM) return MNB_ERR_UNSUPPORTED;
  int sms = sm_count_in;
  if (sms <= 0) {
    st = check_device();
    if (st != MNB_OK) return st;
    sms = sm_count();
  }
  // The arguments run_matmul builds; null A and Y count as aligned, and the
  // planner only tests the zero points and the workspace for presence.
  alignas(256) static unsigned char present[1];
  MatmulArgs a{nullptr, nullptr, nullptr, has_zero_points ? present : nullptr,
               nullptr, nullptr, M, N, K, block_size, a_dtype == MNB_F32,
               scale_dtype == MNB_F32, false};
  a.ws = workspace_bytes ? present : nullptr;
  a.ws_bytes = workspace_bytes;
  a.sk_only = path == MNB_PATH_GEMM_STREAMK;
  mnb_matmul_plan_info r{};
  if (path == MNB_PATH_GEMV || (path == MNB_PATH_AUTO && M <= kGemvMaxM)) {
    r.path = MNB_PATH_GEMV;
  } else if (path == MNB_PATH_GEMM_PAIR) {
    if (!pair_supports(a)) return MNB_ERR_UNSUPPORTED;
    const PairPlan pp = plan_pair(a, sm_count_in > 0 ? sms / 2 : pair_slots());
    if (pp.nt == 0) return MNB_ERR_UNSUPPORTED;
    r.path = MNB_PATH_GEMM;
    r.tile_rows = 256;
    r.k_split = 1;
    r.pair_cols = 32 * pp.nt;
    r.ctas = 2 * int64_t(pp.pairs);
  } else if (path == MNB_PATH_GEMM || path == MNB_PATH_GEMM_STREAMK || gemm_supports(a)) {
    if (!gemm_supports(a) || (a.sk_only && (a.a_f32 || !a.ws))) return MNB_ERR_UNSUPPORTED;
    const GemmPlanInfo g = gemm_plan_info(a, sms);
    if (a.sk_only && !g.stream_k) return MNB_ERR_UNSUPPORTED;
    r.path = MNB_PATH_GEMM;
    r.tile_rows = g.tile_rows;
    r.k_split = g.k_split;
    r.stream_k = g.stream_k;
    r.tf32 = g.tf32;
    r.tma_store = g.tma_store;
    r.ctas = g.ctas;
  } else {
    r.path = MNB_PATH_GEMV;
    r.m_slices = static_cast<int32_t>((M + kGemvMaxM - 1) / kGemvMaxM);
  }
  *out = r;
  return MNB_OK;
}

size_t mnb_matmul_workspace_size(void) {
  if (check_device() != MNB_OK) return 0;
  return gemm_workspace_bytes();
}

mnb_status mnb_matmul_ws(const void *A, const void *packed_b, const void *scales,
                         const void *zero_points, const float *bias, int64_t M,
                         int64_t N, int64_t K, int block_size, void *Y,
                         mnb_dtype a_dtype, mnb_dtype scale_dtype, mnb_path path,
                         void *workspace, size_t workspace_bytes, mnb_stream_t stream) {
  mnb_status st = validate_matmul_args(A, packed_b, scales, zero_points, bias, M, N, K,
                                       block_size, Y, a_dtype, scale_dtype, path);
  if (st != MNB_OK) return st;
  if (workspace) {
    if (!aligned(workspace, 256)) return MNB_ERR_ALIGN;
    const size_t es = dtype_size(a_dtype);
    const Sizes in = packed_sizes(N, K, block_size, scale_dtype, zero_points != nullptr);
    const void *others[6] = {A, packed_b, scales, zero_points, bias, Y};
    const size_t on[6] = {size_t(M) * K * es, in.b, in.s, in.z, bias ? size_t(N) * 4 : 0,
                          size_t(M) * N * es};
    for (int j = 0; j < 6; ++j)
      if (overlap(workspace, workspace_bytes, others[j], on[j])) return MNB_ERR_ALIAS;
  }
  st = check_layout(packed_b, N, K, block_size, scale_dtype, zero_points != nullptr,
                    MNB_CODES_AFFINE);
  if (st != MNB_OK) return st;
  st = check_device();
  if (st != MNB_OK) return st;
  return run_matmul(A, packed_b, scales, zero_points, bias, M, N, K, block_size, Y,
                    a_dtype, scale_dtype, path, reinterpret_cast<cudaStream_t>(stream),
                    workspace, workspace ? workspace_bytes : 0);
}

mnb_status mnb_matmul(const void *A, const void *packed_b, const void *scales,
                      const void *zero_points, const float *bias, int64_t M,
                      int64_t N, int64_t K, int block_size, void *Y,
                      mnb_dtype a_dtype, mnb_dtype scale_dtype,
                      mnb_stream_t stream) {
  return mnb_matmul_path(A, packed_b, scales, zero_points, bias, M, N, K,
                         block_size, Y, a_dtype, scale_dtype, MNB_PATH_AUTO,
                         stream);
}

mnb_status mnb_matmul_grouped(const void *A, int count,
                              const void *const *packed_b,
                              const void *const *scales,
                              const void *const *zero_points,
                              const float *const *bias, const int64_t *N,
                              void *const *Y, int64_t M, int64_t K,
                              int block_size, mnb_dtype a_dtype,
                              mnb_dtype scale_dtype, mnb_stream_t stream) {
  if (!packed_b || !scales || !N || !Y) return MNB_ERR_NULL;
  if (count < 1 || count > kMaxGroup) return MNB_ERR_SHAPE;
  const bool has_zp = zero_points && zero_points[0];
  for (int i = 0; i < count; ++i) {
    if (zero_points && ((zero_points[i] != nullptr) != has_zp)) return MNB_ERR_NULL;
    const mnb_status st = validate_matmul_host(
        A, packed_b[i], scales[i], has_zp ? zero_points[i] : nullptr,
        bias ? bias[i] : nullptr, M, N[i], K, block_size, Y[i], a_dtype,
        scale_dtype, MNB_PATH_AUTO);
    if (st != MNB_OK) return st;
    const size_t es = dtype_size(a_dtype);
    for (int j = 0; j < count; ++j) {
      if (j == i) continue;
      const Sizes in = packed_sizes(N[j], K, block_size, scale_dtype, has_zp);
      const void *others[5] = {packed_b[j], scales[j], has_zp ? zero_points[j] : nullptr,
                               bias ? bias[j] : nullptr, Y[j]};
      const size_t on[5] = {in.b, in.s, in.z, (bias && bias[j]) ? size_t(N[j]) * 4 : 0,
                            size_t(M) * N[j] * es};
      for (int k = 0; k < 5; ++k)
        if (overlap(Y[i], size_t(M) * N[i] * es, others[k], on[k])) return MNB_ERR_ALIAS;
    }
  }
  if (const mnb_status st = check_device(); st != MNB_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M > kGemvMaxM) {
    for (int i = 0; i < count; ++i) {
      const mnb_status st = run_matmul(A, packed_b[i], scales[i],
                                       has_zp ? zero_points[i] : nullptr,
                                       bias ? bias[i] : nullptr, M, N[i], K,
                                       block_size, Y[i], a_dtype, scale_dtype,
                                       MNB_PATH_AUTO, s);
      if (st != MNB_OK) return st;
    }
    return MNB_OK;
  }
  GroupArgs g{};
  g.A = A;
  g.count = count;
  for (int i = 0; i < count; ++i) {
    g.packed_b[i] = packed_b[i];
    g.scales[i] = scales[i];
    g.zp[i] = has_zp ? zero_points[i] : nullptr;
    g.bias[i] = bias ? bias[i] : nullptr;
    g.Y[i] = Y[i];
    g.N[i] = N[i];
  }
  g.M = M;
  g.K = K;
  g.bs = block_size;
  g.a_f32 = a_dtype == MNB_F32;
  g.scale_f32 = scale_dtype == MNB_F32;
  g.has_zp = has_zp;
  g.pdl = g_pdl.load() != 0;
  const cudaError_t e = launch_gemv_group(g, s);
  if (e == cudaErrorNotSupported) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "no grouped kernel for M=%lld K=%lld bs=%d", (long long)M,
                  (long long)K, block_size);
    return MNB_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return cuda_fail(e, "mnb_matmul_grouped");
  return MNB_OK;
}

mnb_status mnb_matmul_gate_up(const void *A, const void *packed_gate,
                              const void *scales_gate, const void *zp_gate,
                              const float *bias_gate, const void *packed_up,
                              const void *scales_up, const void *zp_up,
                              const float *bias_up, int64_t M, int64_t N, int64_t K,
                              int block_size, void *Y, mnb_dtype a_dtype,
                              mnb_dtype scale_dtype, mnb_stream_t stream) {
  if ((zp_gate != nullptr) != (zp_up != nullptr)) return MNB_ERR_NULL;
  mnb_status st = validate_matmul_host(A, packed_gate, scales_gate, zp_gate, bias_gate, M, N,
                                       K, block_size, Y, a_dtype, scale_dtype, MNB_PATH_AUTO);
  if (st != MNB_OK) return st;
  st = validate_matmul_host(A, packed_up, scales_up, zp_up, bias_up, M, N, K, block_size, Y,
                            a_dtype, scale_dtype, MNB_PATH_AUTO);
  if (st != MNB_OK) return st;
  st = check_device();
  if (st != MNB_OK) return st;
  const size_t es = dtype_size(a_dtype);
  GroupArgs g{};
  g.count = 2;
  g.paired = true;
  g.packed_b[0] = packed_gate;
  g.packed_b[1] = packed_up;
  g.scales[0] = scales_gate;
  g.scales[1] = scales_up;
  g.zp[0] = zp_gate;
  g.zp[1] = zp_up;
  g.bias[0] = bias_gate;
  g.bias[1] = bias_up;
  g.N[0] = g.N[1] = N;
  g.K = K;
  g.bs = block_size;
  g.a_f32 = a_dtype == MNB_F32;
  g.scale_f32 = scale_dtype == MNB_F32;
  g.has_zp = zp_gate != nullptr;
  g.pdl = g_pdl.load() != 0;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M > kGemvMaxM) {
    // The tensor-core kernel's paired mode, when it takes these activations.
    MatmulArgs t{A, packed_gate, scales_gate, zp_gate, bias_gate, Y, M, N, K, block_size,
                 a_dtype == MNB_F32, scale_dtype == MNB_F32, g_pdl.load() != 0};
    t.paired = true;
    t.packed_b2 = packed_up;
    t.scales2 = scales_up;
    t.zp2 = zp_up;
    t.bias2 = bias_up;
    if (gemm_supports(t)) {
      const cudaError_t e = launch_gemm(t, s);
      if (e != cudaSuccess) return cuda_fail(e, "mnb_matmul_gate_up");
      return MNB_OK;
    }
  }
  // The decode kernel takes up to 16 rows per launch.
  for (int64_t m0 = 0; m0 < M; m0 += kGemvMaxM) {
    g.M = std::min<int64_t>(kGemvMaxM, M - m0);
    g.A = static_cast<const char *>(A) + m0 * K * es;
    g.Y[0] = static_cast<char *>(Y) + m0 * N * es;
    const cudaError_t e = launch_gemv_group(g, s);
    if (e == cudaErrorNotSupported) {
      std::snprintf(g_last_error, sizeof g_last_error,
                    "no gate/up kernel for K=%lld bs=%d", (long long)K, block_size);
      return MNB_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return cuda_fail(e, "mnb_matmul_gate_up");
  }
  return MNB_OK;
}

mnb_status mnb_matmul_from_host(const void *A_host, void *A_dev,
                                const void *packed_b, const void *scales,
                                const void *zero_points, const float *bias,
                                int64_t M, int64_t N, int64_t K,
                                int block_size, void *Y_dev, void *Y_host,
                                mnb_dtype a_dtype, mnb_dtype scale_dtype,
                                mnb_stream_t stream) {
  if (!A_host || !Y_host) return MNB_ERR_NULL;
  const mnb_status st = validate_matmul(A_dev, packed_b, scales, zero_points,
                                        bias, M, N, K, block_size, Y_dev,
                                        a_dtype, scale_dtype, MNB_PATH_AUTO);
  if (st != MNB_OK) return st;
  const size_t es = dtype_size(a_dtype);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(A_dev, A_host, size_t(M) * K * es,
                                  cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "mnb_matmul_from_host (A copy)");
  const mnb_status rs = run_matmul(A_dev, packed_b, scales, zero_points, bias,
                                   M, N, K, block_size, Y_dev, a_dtype,
                                   scale_dtype, MNB_PATH_AUTO, s);
  if (rs != MNB_OK) return rs;
  e = cudaMemcpyAsync(Y_host, Y_dev, size_t(M) * N * es, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "mnb_matmul_from_host (Y copy)");
  return MNB_OK;
}

mnb_status mnb_matmul_rmsnorm(const void *A, int normalize, const float *gamma,
                              float epsilon, const void *packed_b, const void *scales,
                              const void *zero_points, const float *bias, int64_t M, int64_t N,
                              int64_t K, int block_size, void *Y, int64_t *argmax,
                              mnb_dtype a_dtype, mnb_dtype scale_dtype, mnb_stream_t stream) {
  if (!A || !packed_b || !scales || (!Y && !argmax)) return MNB_ERR_NULL;
  if (normalize != 0 && normalize != 1) return MNB_ERR_SHAPE;
  if (M < 1 || M > kMaxDim) return MNB_ERR_SHAPE;
  mnb_status st = check_shape(N, K, block_size, scale_dtype);
  if (st != MNB_OK) return st;
  if (!valid_dtype(a_dtype)) return MNB_ERR_DTYPE;
  if (normalize && !(epsilon >= 0.f && epsilon <= 3.0e38f)) return MNB_ERR_SHAPE;
  const size_t es = dtype_size(a_dtype);
  if (!aligned(A, es) || (Y && !aligned(Y, es)) || !aligned(packed_b, 16) ||
      !aligned(scales, 16) || (zero_points && !aligned(zero_points, 16)) ||
      (bias && !aligned(bias, 4)) || (gamma && !aligned(gamma, 4)) ||
      (argmax && !aligned(argmax, 8)))
    return MNB_ERR_ALIGN;
  const Sizes in = packed_sizes(N, K, block_size, scale_dtype, zero_points != nullptr);
  const void *ins[6] = {A, packed_b, scales, zero_points, bias, normalize ? gamma : nullptr};
  const size_t in_n[6] = {size_t(M) * K * es, in.b, in.s, in.z, bias ? size_t(N) * 4 : 0,
                          (normalize && gamma) ? size_t(K) * 4 : 0};
  const size_t y_bytes = Y ? size_t(M) * N * es : 0, k_bytes = argmax ? size_t(M) * 8 : 0;
  for (int j = 0; j < 6; ++j)
    if (overlap(Y, y_bytes, ins[j], in_n[j]) || overlap(argmax, k_bytes, ins[j], in_n[j]))
      return MNB_ERR_ALIAS;
  if (overlap(Y, y_bytes, argmax, k_bytes)) return MNB_ERR_ALIAS;
  st = check_layout(packed_b, N, K, block_size, scale_dtype, zero_points != nullptr,
                    MNB_CODES_AFFINE);
  if (st != MNB_OK) return st;
  st = check_device();
  if (st != MNB_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (M > kGemvMaxM && !argmax && Y) {
    // Prefill rows: the tensor-core kernel normalizes each staged A tile
    // and scales its output rows, when it can stage these activations.
    MatmulArgs t{A, packed_b, scales, zero_points, bias, Y, M, N, K, block_size,
                 a_dtype == MNB_F32, scale_dtype == MNB_F32, g_pdl.load() != 0};
    t.norm = normalize != 0;
    t.gamma = normalize ? gamma : nullptr;
    t.eps = epsilon;
    if (!t.a_f32 && gemm_supports(t)) {
      e = launch_gemm(t, s);
      if (e != cudaSuccess) return cuda_fail(e, "mnb_matmul_rmsnorm");
      return MNB_OK;
    }
  }
  if (argmax)
    e = launch_argmax_init(reinterpret_cast<unsigned long long *>(argmax), static_cast<int>(M),
                           s);
  if (e != cudaSuccess) return cuda_fail(e, "mnb_matmul_rmsnorm (ArgMax keys)");
  // The decode kernel, over 16-row slices beyond 16 rows (fp32 rows, rows the
  // tensor core cannot stage, or with the ArgMax): each slice normalizes
  // its own rows over the whole of K.
  GroupArgs g{};
  g.count = 1;
  g.packed_b[0] = packed_b;
  g.scales[0] = scales;
  g.zp[0] = zero_points;
  g.bias[0] = bias;
  g.N[0] = N;
  g.K = K;
  g.bs = block_size;
  g.a_f32 = a_dtype == MNB_F32;
  g.scale_f32 = scale_dtype == MNB_F32;
  g.has_zp = zero_points != nullptr;
  g.pdl = g_pdl.load() != 0;
  g.norm = normalize != 0;
  g.gamma = normalize ? gamma : nullptr;
  g.eps = epsilon;
  for (int64_t m0 = 0; m0 < M && e == cudaSuccess; m0 += kGemvMaxM) {
    g.M = std::min<int64_t>(kGemvMaxM, M - m0);
    g.A = static_cast<const char *>(A) + size_t(m0) * K * es;
    g.Y[0] = Y ? static_cast<char *>(Y) + size_t(m0) * N * es : nullptr;
    g.amax = argmax ? reinterpret_cast<unsigned long long *>(argmax) + m0 : nullptr;
    e = launch_gemv_group(g, s);
  }
  if (e == cudaErrorNotSupported) {
    std::snprintf(g_last_error, sizeof g_last_error, "no kernel for M=%lld N=%lld K=%lld bs=%d",
                  (long long)M, (long long)N, (long long)K, block_size);
    return MNB_ERR_UNSUPPORTED;
  }
  if (e == cudaSuccess && argmax)
    e = launch_argmax_finalize(reinterpret_cast<unsigned long long *>(argmax),
                               static_cast<int>(M), g.pdl, s);
  if (e != cudaSuccess) return cuda_fail(e, "mnb_matmul_rmsnorm");
  return MNB_OK;
}

mnb_status mnb_prepack_bnb4(const uint8_t *B, const void *absmax, int64_t N, int64_t K,
                            int block_size, mnb_dtype absmax_dtype, void *packed_b,
                            void *packed_scales, mnb_stream_t stream) {
  if (!B || !absmax || !packed_b || !packed_scales) return MNB_ERR_NULL;
  mnb_status st = check_shape(N, K, block_size, absmax_dtype);
  if (st != MNB_OK) return st;
  if (K % block_size != 0) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "mnb_prepack_bnb4: K=%lld is not a multiple of block_size=%d (blocks "
                  "would straddle rows)",
                  (long long)K, block_size);
    return MNB_ERR_UNSUPPORTED;
  }
  if (!aligned(packed_b, 16) || !aligned(packed_scales, 16) ||
      !aligned(absmax, dtype_size(absmax_dtype)))
    return MNB_ERR_ALIGN;
  const int64_t nb = K / block_size;
  const Sizes out = packed_sizes(N, K, block_size, absmax_dtype, false);
  const void *const ins[3] = {B, absmax, nullptr};
  const size_t in_n[3] = {size_t((N * K + 1) / 2), size_t(N) * nb * dtype_size(absmax_dtype),
                          0};
  void *const outs[3] = {packed_b, packed_scales, nullptr};
  const size_t out_n[3] = {out.b, out.s, 0};
  st = check_outputs_disjoint(outs, out_n, ins, in_n);
  if (st != MNB_OK) return st;
  st = check_device();
  if (st != MNB_OK) return st;
  PrepackArgs a{B, absmax, nullptr, N, K, block_size, absmax_dtype == MNB_F32, packed_b,
                packed_scales, nullptr};
  a.bnb4 = true;
  a.header = make_header(N, K, block_size, absmax_dtype, false, MNB_CODES_CODEBOOK);
  a.header_dst = static_cast<char *>(packed_b) + codes_bytes(N, K);
  const cudaError_t e = launch_prepack(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mnb_prepack_bnb4");
  record_header(packed_b, a.header);
  return MNB_OK;
}

mnb_status mnb_matmul_bnb4(const void *A, const void *packed_b, const void *packed_scales,
                           const float *code, const float *bias, int64_t M, int64_t N,
                           int64_t K, int block_size, void *Y, mnb_dtype a_dtype,
                           mnb_dtype absmax_dtype, mnb_stream_t stream) {
  if (!code) return MNB_ERR_NULL;
  if (!aligned(code, 4)) return MNB_ERR_ALIGN;
  mnb_status st = validate_matmul(A, packed_b, packed_scales, nullptr, bias, M, N, K,
                                  block_size, Y, a_dtype, absmax_dtype, MNB_PATH_AUTO,
                                  MNB_CODES_CODEBOOK);
  if (st != MNB_OK) return st;
  if (overlap(Y, size_t(M) * N * dtype_size(a_dtype), code, 64)) return MNB_ERR_ALIAS;
  const size_t es = dtype_size(a_dtype);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M > kGemvMaxM) {
    // Prefill rows: the tensor-core kernel's code-book mode, when it can
    // stage these activations (bf16 rows, 16-byte aligned).
    MatmulArgs t{A, packed_b, packed_scales, nullptr, bias, Y, M, N, K, block_size,
                 a_dtype == MNB_F32, absmax_dtype == MNB_F32, g_pdl.load() != 0};
    t.code = code;
    if (!t.a_f32 && gemm_supports(t)) {
      const cudaError_t e = launch_gemm(t, s);
      if (e != cudaSuccess) return cuda_fail(e, "mnb_matmul_bnb4");
      return MNB_OK;
    }
  }
  // The decode kernel in code-book mode, over 8-row slices.
  constexpr int64_t kRows = kGemvMaxM / 2;
  for (int64_t m0 = 0; m0 < M; m0 += kRows) {
    GroupArgs g{};
    g.A = static_cast<const char *>(A) + size_t(m0) * K * es;
    g.count = 1;
    g.packed_b[0] = packed_b;
    g.scales[0] = packed_scales;
    g.bias[0] = bias;
    g.Y[0] = static_cast<char *>(Y) + size_t(m0) * N * es;
    g.N[0] = N;
    g.M = std::min<int64_t>(kRows, M - m0);
    g.K = K;
    g.bs = block_size;
    g.a_f32 = a_dtype == MNB_F32;
    g.scale_f32 = absmax_dtype == MNB_F32;
    g.has_zp = false;
    g.pdl = g_pdl.load() != 0;
    g.code = code;
    const cudaError_t e = launch_gemv_group(g, s);
    if (e == cudaErrorNotSupported) {
      std::snprintf(g_last_error, sizeof g_last_error,
                    "no code-book kernel for N=%lld K=%lld bs=%d", (long long)N, (long long)K,
                    block_size);
      return MNB_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return cuda_fail(e, "mnb_matmul_bnb4");
  }
  return MNB_OK;
}

mnb_status mnb_chain_build(const mnb_chain_op *ops, int32_t n_ops, int64_t M,
                           int block_size, mnb_dtype a_dtype, mnb_dtype scale_dtype,
                           void *plan, size_t plan_bytes, mnb_chain_info *info,
                           mnb_stream_t stream) {
  if (!ops || !info) return MNB_ERR_NULL;
  if (n_ops < 1 || n_ops > kChainMaxOps || M < 1 || M > kChainMaxM) return MNB_ERR_SHAPE;
  if (!valid_block_size(block_size)) return MNB_ERR_BLOCKSIZE;
  if (!valid_dtype(a_dtype) || !valid_dtype(scale_dtype)) return MNB_ERR_DTYPE;
  const bool has_zp = ops[0].packed_zp != nullptr;
  const size_t es = dtype_size(a_dtype);
  std::vector<ChainOp> cops(n_ops);
  std::vector<OpRanges> rg(n_ops);
  for (int j = 0; j < n_ops; ++j) {
    const mnb_chain_op &o = ops[j];
    if (!o.A || !o.Y || !o.packed_b || !o.packed_scales) return MNB_ERR_NULL;
    if ((o.packed_zp != nullptr) != has_zp) return MNB_ERR_NULL;
    const bool paired = o.packed_b_up != nullptr;
    if (paired && (!o.packed_scales_up || (o.packed_zp_up != nullptr) != has_zp))
      return MNB_ERR_NULL;
    if (!paired && (o.packed_scales_up || o.packed_zp_up || o.bias_up)) return MNB_ERR_NULL;
    mnb_status st = check_shape(o.N, o.K, block_size, scale_dtype);
    if (st != MNB_OK) return st;
    const void *al16[6] = {o.packed_b, o.packed_scales, o.packed_zp,
                           o.packed_b_up, o.packed_scales_up, o.packed_zp_up};
    for (const void *q : al16)
      if (q && !aligned(q, 16)) return MNB_ERR_ALIGN;
    if (!aligned(o.A, es) || !aligned(o.Y, es) || (o.bias && !aligned(o.bias, 4)) ||
        (o.bias_up && !aligned(o.bias_up, 4)))
      return MNB_ERR_ALIGN;
    for (int k = 0; k < kChainMaxDeps; ++k)
      if (o.deps[k] < -1 || o.deps[k] >= j) return MNB_ERR_SHAPE;
    rg[j] = op_ranges(o, M, block_size, a_dtype, scale_dtype);
    ChainOp &c = cops[j];
    c.A = o.A;
    c.Y = o.Y;
    c.b[0] = o.packed_b;
    c.s[0] = o.packed_scales;
    c.z[0] = o.packed_zp;
    c.bias[0] = o.bias;
    c.b[1] = o.packed_b_up;
    c.s[1] = o.packed_scales_up;
    c.z[1] = o.packed_zp_up;
    c.bias[1] = o.bias_up;
    c.N = o.N;
    c.K = o.K;
    c.paired = paired;
    for (int k = 0; k < kChainMaxDeps; ++k) c.dep[k] = o.deps[k];
  }
  // Hazards: transitive dependencies as bit sets.
  const int words = (n_ops + 63) / 64;
  std::vector<uint64_t> reach(size_t(n_ops) * words, 0);
  for (int j = 0; j < n_ops; ++j) {
    uint64_t *rj = reach.data() + size_t(j) * words;
    for (int k = 0; k < kChainMaxDeps; ++k) {
      const int d = ops[j].deps[k];
      if (d < 0) continue;
      const uint64_t *rd = reach.data() + size_t(d) * words;
      for (int w = 0; w < words; ++w) rj[w] |= rd[w];
      rj[d / 64] |= uint64_t(1) << (d % 64);
    }
  }
  for (int j = 0; j < n_ops; ++j) {
    const OpRanges &a = rg[j];
    if (overlap(a.y, a.ny, a.a, a.na)) return MNB_ERR_ALIAS;
    for (int i = 0; i < n_ops; ++i)
      for (int w = 0; w < 8; ++w)
        if (overlap(a.y, a.ny, rg[i].w[w], rg[i].nw[w])) return MNB_ERR_ALIAS;
    const uint64_t *rj = reach.data() + size_t(j) * words;
    for (int i = 0; i < j; ++i) {
      const bool ordered = (rj[i / 64] >> (i % 64)) & 1u;
      if (ordered) continue;
      if (overlap(rg[i].y, rg[i].ny, a.a, a.na) || overlap(a.y, a.ny, rg[i].a, rg[i].na) ||
          overlap(a.y, a.ny, rg[i].y, rg[i].ny))
        return MNB_ERR_ALIAS;
    }
  }
  // The weights' headers, after the argument and hazard checks.
  for (int j = 0; j < n_ops; ++j) {
    const mnb_chain_op &o = ops[j];
    mnb_status ls = check_layout(o.packed_b, o.N, o.K, block_size, scale_dtype, has_zp,
                                 MNB_CODES_AFFINE);
    if (ls == MNB_OK && o.packed_b_up)
      ls = check_layout(o.packed_b_up, o.N, o.K, block_size, scale_dtype, has_zp,
                        MNB_CODES_AFFINE);
    if (ls != MNB_OK) return ls;
  }
  mnb_status st = check_device();
  if (st != MNB_OK) return st;
  const ChainShape sh{static_cast<int>(M), block_size, a_dtype == MNB_F32,
                      scale_dtype == MNB_F32, has_zp};
  ChainGeom g{};
  std::vector<unsigned char> image;
  cudaError_t e = chain_plan(cops.data(), n_ops, sh, g, plan ? &image : nullptr);
  if (e == cudaErrorNotSupported) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "no chain layout for M=%lld, largest K=%d, bs=%d", (long long)M, g.kmax,
                  block_size);
    return MNB_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return cuda_fail(e, "mnb_chain_build (plan)");
  mnb_chain_info inf{};
  inf.plan_bytes = g.plan_bytes;
  inf.n_ops = n_ops;
  inf.n_segments = g.n_segs;
  inf.grid = g.grid;
  inf.smem_bytes = g.smem;
  inf.M = static_cast<int32_t>(M);
  inf.block_size = block_size;
  inf.a_dtype = a_dtype;
  inf.scale_dtype = scale_dtype;
  inf.has_zero_points = has_zp ? 1 : 0;
  inf.ring_stages = g.nst;
  inf.k_max = g.kmax;
  inf.tiles_per_segment = g.tmax;
  inf.ctas_per_sm = g.per_sm;
  inf.check = chain_checksum(inf);
  if (plan) {
    if (!aligned(plan, 256)) return MNB_ERR_ALIGN;
    if (plan_bytes < g.plan_bytes) return MNB_ERR_SHAPE;
    for (int j = 0; j < n_ops; ++j) {
      const OpRanges &a = rg[j];
      bool hit = overlap(plan, plan_bytes, a.a, a.na) || overlap(plan, plan_bytes, a.y, a.ny);
      for (int w = 0; w < 8; ++w) hit = hit || overlap(plan, plan_bytes, a.w[w], a.nw[w]);
      if (hit) return MNB_ERR_ALIAS;
    }
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = cudaMemcpyAsync(plan, image.data(), g.plan_bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "mnb_chain_build (plan copy)");
  }
  *info = inf;
  return MNB_OK;
}

mnb_status mnb_chain_run(const void *plan, const mnb_chain_info *info, mnb_stream_t stream) {
  if (!plan || !info) return MNB_ERR_NULL;
  if (chain_checksum(*info) != info->check) return MNB_ERR_SHAPE;
  if (!aligned(plan, 256)) return MNB_ERR_ALIGN;
  const ChainShape sh{info->M, info->block_size, info->a_dtype == MNB_F32,
                      info->scale_dtype == MNB_F32, info->has_zero_points != 0};
  ChainGeom g{};
  if (!chain_geom(sh, info->n_ops, info->k_max, info->grid, info->ctas_per_sm,
                  info->ring_stages, info->n_segments, g) ||
      g.plan_bytes != info->plan_bytes || g.smem != info->smem_bytes ||
      g.tmax != info->tiles_per_segment)
    return MNB_ERR_SHAPE;
  mnb_status st = check_device();
  if (st != MNB_OK) return st;
  const cudaError_t e = chain_launch(plan, sh, g, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mnb_chain_run");
  return MNB_OK;
}

mnb_status mnb_chain_run_noalloc(const mnb_chain_op *ops, int32_t n_ops, int64_t M,
                                 int block_size, mnb_dtype a_dtype, mnb_dtype scale_dtype,
                                 mnb_stream_t stream) {
  // Plan (query only), check it fits the library's fixed array, plan into
  // the array, run: the two public chain calls with library-owned storage.
  mnb_chain_info info{};
  mnb_status st = mnb_chain_build(ops, n_ops, M, block_size, a_dtype, scale_dtype, nullptr, 0,
                                  &info, stream);
  if (st != MNB_OK) return st;
  void *scratch = nullptr;
  size_t cap = 0;
  const cudaError_t e = chain_scratch(&scratch, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "mnb_chain_run_noalloc (scratch address)");
  if (info.plan_bytes > cap) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "mnb_chain_run_noalloc: this chain's plan needs %llu bytes, the library's "
                  "fixed plan array holds %zu; pass a buffer to mnb_chain_build instead",
                  (unsigned long long)info.plan_bytes, cap);
    return MNB_ERR_UNSUPPORTED;
  }
  st = mnb_chain_build(ops, n_ops, M, block_size, a_dtype, scale_dtype, scratch, cap, &info,
                       stream);
  if (st != MNB_OK) return st;
  return mnb_chain_run(scratch, &info, stream);
}

}  // extern "C"
