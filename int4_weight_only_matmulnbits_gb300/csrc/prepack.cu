// Offline re-layout of MatMulNBits weights into the prepacked form, and its
// inverse; also the re-layout of the standard QDQ INT4 encoding (logical
// UINT4 matrix + DequantizeLinear) into the same form. The layout is defined
// in mnb_common.cuh.
#include "mnb_common.cuh"
#include "mnb_launch.h"

namespace mnb {
namespace {

// Code q[n,k] of the MatMulNBits storage: byte (k mod bs)/2 of block k/bs,
// low nibble for even k. Zero outside the logical N x K matrix.
__device__ __forceinline__ uint32_t source_code(const uint8_t *B, int64_t n,
                                                int64_t k, int64_t N, int64_t K,
                                                int64_t nb, int bs) {
  if (n >= N || k >= K) return 0;
  const int64_t within = k % bs;
  const uint8_t byte = B[(n * nb + k / bs) * (bs / 2) + within / 2];
  return (within & 1) ? (byte >> 4) : (byte & 0x0F);
}

// Code source for the MatMulNBits storage.
struct NBitsCodes {
  const uint8_t *B;
  int64_t N, K, nb;
  int bs;
  __device__ __forceinline__ uint32_t operator()(int64_t n, int64_t k) const {
    return source_code(B, n, k, N, K, nb, bs);
  }
};

// Code source for a logical UINT4 matrix in ONNX row-major, low-nibble-first
// storage (page "Qwen3 CPU Inference Critical Path", section
// "qwen3-int4-qdq"): element i of the flattened matrix is nibble i of the
// byte stream, low nibble first. axis 0: the matrix is [K, N] (projections,
// DequantizeLinear along K); axis 1: [N, K] (the tied LM-head weight).
struct QdqCodes {
  const uint8_t *B;
  int64_t N, K;
  int axis;
  __device__ __forceinline__ uint32_t operator()(int64_t n, int64_t k) const {
    if (n >= N || k >= K) return 0;
    const int64_t i = axis == 0 ? k * N + n : n * K + k;
    const uint8_t byte = B[i >> 1];
    return (i & 1) ? (byte >> 4) : (byte & 0x0F);
  }
};

// Code source for the bitsandbytes-style 4-bit matrix (page "Qwen3 CPU
// Inference Critical Path", MatMulBnb4 row; the storage is this library's
// reading): the N x K weight flattened row-major, two codes per byte, the
// first of a pair in the high nibble.
struct Bnb4Codes {
  const uint8_t *B;
  int64_t N, K;
  __device__ __forceinline__ uint32_t operator()(int64_t n, int64_t k) const {
    if (n >= N || k >= K) return 0;
    const int64_t i = n * K + k;
    const uint8_t byte = B[i >> 1];
    return (i & 1) ? (byte & 0x0F) : (byte >> 4);
  }
};

template <typename Src>
__global__ void pack_codes_kernel(Src src, uint32_t *__restrict__ out, int64_t K64,
                                  int64_t words) {
  for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < words;
       w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t chunk = w >> 7;
    const int idx = static_cast<int>(w & 127);
    const int lane = idx >> 2, j = idx & 3, g = lane >> 2, t = lane & 3;
    const int64_t tile = chunk / K64, c = chunk % K64;
    const int64_t r0 = tile * kTileN + g;
    const int64_t k0 = c * kChunkK + 16 * j + 4 * t;
    uint32_t word = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        word |= src(r0 + 8 * h, k0 + e) << code_shift(e, h);
    out[w] = word;
  }
}

// Scales s[n, b] stored [N, nb] (k_major false) or [nb, N] (true).
template <typename T>
__global__ void pack_scales_kernel(const T *__restrict__ s, T *__restrict__ out,
                                   int64_t N, int64_t nb, bool k_major, int64_t total) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int r = static_cast<int>(i & 15);
    const int64_t tb = i >> 4;
    const int64_t tile = tb / nb, b = tb % nb;
    const int64_t n = tile * kTileN + r;
    out[i] = n < N ? s[k_major ? b * N + n : n * nb + b] : T(0);
  }
}

// Zero-point sources: MatMulNBits [N, ceil(nb/2)] bytes, even block low;
// QDQ UINT4 [nb, N] (axis 0) or [N, nb] (axis 1) flattened low-nibble-first;
// QDQ without zero points: 0 (the DequantizeLinear default).
struct NBitsZp {
  const uint8_t *zp;
  int64_t nb;
  __device__ __forceinline__ uint32_t operator()(int64_t n, int64_t b) const {
    const uint8_t byte = zp[n * ((nb + 1) / 2) + b / 2];
    return (b & 1) ? (byte >> 4) : (byte & 0x0F);
  }
};
struct QdqZp {
  const uint8_t *zp;
  int64_t N, nb;
  int axis;
  __device__ __forceinline__ uint32_t operator()(int64_t n, int64_t b) const {
    if (zp == nullptr) return 0;
    const int64_t i = axis == 0 ? b * N + n : n * nb + b;
    const uint8_t byte = zp[i >> 1];
    return (i & 1) ? (byte >> 4) : (byte & 0x0F);
  }
};

template <typename Src>
__global__ void pack_zp_kernel(Src src, uint64_t *__restrict__ out, int64_t N,
                               int64_t nb, int64_t nbz, int64_t total) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = i / nbz, b = i % nbz;
    uint64_t word = 0;
    for (int r = 0; r < kTileN && b < nb; ++r) {
      const int64_t n = tile * kTileN + r;
      if (n >= N) break;
      word |= static_cast<uint64_t>(src(n, b)) << (4 * r);
    }
    out[i] = word;
  }
}

// Inverse of pack_codes_kernel: one thread per byte of B [N, nb, bs/2].
__global__ void unpack_codes_kernel(const uint32_t *__restrict__ packed,
                                    uint8_t *__restrict__ B, int64_t N,
                                    int64_t K, int64_t nb, int bs, int64_t K64,
                                    int64_t total) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t half = bs / 2;
    const int64_t n = i / (nb * half);
    const int64_t rem = i % (nb * half);
    const int64_t kk = (rem / half) * bs + (rem % half) * 2;  // even k
    uint32_t byte = 0;
    for (int o = 0; o < 2; ++o) {
      const int64_t k = kk + o;
      if (k >= K) continue;
      const int64_t tile = n / kTileN;
      const int r = static_cast<int>(n % kTileN);
      const int64_t c = k / kChunkK;
      const int kin = static_cast<int>(k % kChunkK);
      const int j = kin >> 4, t = (kin >> 2) & 3, e = kin & 3;
      const int g = r & 7, h = r >> 3;
      const int lane = g * 4 + t;
      const uint32_t word = packed[(tile * K64 + c) * 128 + lane * 4 + j];
      byte |= ((word >> code_shift(e, h)) & 0xF) << (4 * o);
    }
    B[i] = static_cast<uint8_t>(byte);
  }
}

template <typename T>
__global__ void unpack_scales_kernel(const T *__restrict__ packed,
                                     T *__restrict__ s, int64_t nb,
                                     int64_t total) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i / nb, b = i % nb;
    s[i] = packed[((n / kTileN) * nb + b) * kTileN + (n % kTileN)];
  }
}

__global__ void unpack_zp_kernel(const uint64_t *__restrict__ packed,
                                 uint8_t *__restrict__ zp, int64_t nb,
                                 int64_t nbz, int64_t total) {
  const int64_t zbytes = (nb + 1) / 2;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i / zbytes, zb = i % zbytes;
    const int64_t tile = n / kTileN;
    const int r = static_cast<int>(n % kTileN);
    uint32_t byte = 0;
    for (int o = 0; o < 2; ++o) {
      const int64_t b = zb * 2 + o;
      if (b >= nb) continue;
      byte |= static_cast<uint32_t>((packed[tile * nbz + b] >> (4 * r)) & 0xF)
              << (4 * o);
    }
    zp[i] = static_cast<uint8_t>(byte);
  }
}

// Launched last by every prepack call: writes the packed-weight header at
// the end of packed_b. Matmul kernels launched with programmatic dependent
// launch may start loading their packed weights as soon as the kernel before
// them on the stream begins to exit; ending the prepack with this kernel,
// which writes nothing the matmul kernels read, puts a full kernel boundary
// between the writes of the packed weights and any such early load.
// The header fills the first 80 of its 256 bytes; the rest are zeros, so
// the packed bytes of a weight are fully determined by its contents.
__global__ void prepack_fence_kernel(const mnb_packed_header h, uint64_t *dst) {
  static_assert(sizeof(mnb_packed_header) % 8 == 0 && MNB_PACKED_HEADER_BYTES == 32 * 8,
                "one 8-byte word per thread");
  const int i = threadIdx.x;
  if (!dst || i >= 32) return;
  uint64_t w = 0;
  if (i < static_cast<int>(sizeof(h) / 8)) w = reinterpret_cast<const uint64_t *>(&h)[i];
  dst[i] = w;
}

inline unsigned grid_for(int64_t total) {
  int64_t blocks = ceil_div(total, 256);
  if (blocks > (1 << 20)) blocks = 1 << 20;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

}  // namespace

cudaError_t launch_prepack(const PrepackArgs &a, cudaStream_t stream) {
  const int64_t nb = ceil_div(a.K, a.bs);
  const int64_t N16 = ceil_div(a.N, kTileN), K64 = ceil_div(a.K, kChunkK);
  const int64_t words = N16 * K64 * (kChunkBytes / 4);
  const bool qdq = a.qdq_axis >= 0;
  if (a.bnb4)
    pack_codes_kernel<<<grid_for(words), 256, 0, stream>>>(
        Bnb4Codes{a.B, a.N, a.K}, static_cast<uint32_t *>(a.packed_b), K64, words);
  else if (qdq)
    pack_codes_kernel<<<grid_for(words), 256, 0, stream>>>(
        QdqCodes{a.B, a.N, a.K, a.qdq_axis}, static_cast<uint32_t *>(a.packed_b), K64, words);
  else
    pack_codes_kernel<<<grid_for(words), 256, 0, stream>>>(
        NBitsCodes{a.B, a.N, a.K, nb, a.bs}, static_cast<uint32_t *>(a.packed_b), K64, words);
  const int64_t ns = N16 * nb * kTileN;
  const bool k_major = a.qdq_axis == 0;
  if (a.scale_f32)
    pack_scales_kernel<float><<<grid_for(ns), 256, 0, stream>>>(
        static_cast<const float *>(a.scales),
        static_cast<float *>(a.packed_scales), a.N, nb, k_major, ns);
  else
    pack_scales_kernel<uint16_t><<<grid_for(ns), 256, 0, stream>>>(
        static_cast<const uint16_t *>(a.scales),
        static_cast<uint16_t *>(a.packed_scales), a.N, nb, k_major, ns);
  const int64_t nbz = ceil_div(nb, 2) * 2;
  if (qdq)  // always packed: QDQ zero points default to 0, not 8
    pack_zp_kernel<<<grid_for(N16 * nbz), 256, 0, stream>>>(
        QdqZp{a.zp, a.N, nb, a.qdq_axis}, static_cast<uint64_t *>(a.packed_zp), a.N, nb, nbz,
        N16 * nbz);
  else if (a.zp != nullptr)
    pack_zp_kernel<<<grid_for(N16 * nbz), 256, 0, stream>>>(
        NBitsZp{a.zp, nb}, static_cast<uint64_t *>(a.packed_zp), a.N, nb, nbz, N16 * nbz);
  prepack_fence_kernel<<<1, 32, 0, stream>>>(a.header, static_cast<uint64_t *>(a.header_dst));
  return cudaGetLastError();
}

cudaError_t launch_unprepack(const UnprepackArgs &a, cudaStream_t stream) {
  const int64_t nb = ceil_div(a.K, a.bs);
  const int64_t K64 = ceil_div(a.K, kChunkK);
  const int64_t nbytes = a.N * nb * (a.bs / 2);
  unpack_codes_kernel<<<grid_for(nbytes), 256, 0, stream>>>(
      static_cast<const uint32_t *>(a.packed_b), a.B, a.N, a.K, nb, a.bs, K64,
      nbytes);
  const int64_t ns = a.N * nb;
  if (a.scale_f32)
    unpack_scales_kernel<float><<<grid_for(ns), 256, 0, stream>>>(
        static_cast<const float *>(a.packed_scales),
        static_cast<float *>(a.scales), nb, ns);
  else
    unpack_scales_kernel<uint16_t><<<grid_for(ns), 256, 0, stream>>>(
        static_cast<const uint16_t *>(a.packed_scales),
        static_cast<uint16_t *>(a.scales), nb, ns);
  if (a.packed_zp != nullptr) {
    const int64_t nz = a.N * ((nb + 1) / 2);
    unpack_zp_kernel<<<grid_for(nz), 256, 0, stream>>>(
        static_cast<const uint64_t *>(a.packed_zp), a.zp, nb, ceil_div(nb, 2) * 2, nz);
  }
  return cudaGetLastError();
}

}  // namespace mnb
