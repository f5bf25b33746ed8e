/*
 * mnb.h — C ABI of the GB300 (sm_103a) weight-only INT4 blockwise MatMul in
 * the ONNX com.microsoft::MatMulNBits form.
 *
 * Operation (page "Qwen3 CPU Inference Critical Path", section "Exact kernel
 * inventory", row com.microsoft::MatMulNBits v1; section "Prepared weight-only
 * plan"):
 *
 *   Y[m,n] = sum_k A[m,k] * (q[n,k] - z[n,k/bs]) * s[n,k/bs] + bias[n]
 *
 * for 0 <= m < M, 0 <= n < N, 0 <= k < K, bs = block_size, with the 4-bit
 * codes q and zero points z unsigned (0..15) and z = 8 when no zero points
 * are given. Weights stay compressed: no call expands them to a dense matrix.
 *
 * Conventions for every call:
 *  - Every pointer argument is a DEVICE pointer unless its comment says HOST.
 *    The caller owns and allocates every buffer; the library allocates no
 *    device memory in any call.
 *  - Calls that take a stream are asynchronous on it (NULL = legacy default
 *    stream). A returned MNB_OK means the work was validated and enqueued.
 *  - Arguments are validated on the host before anything is enqueued; a
 *    rejected call enqueues nothing and touches no buffer. No call ever falls
 *    back to a CPU path. MNB_ERR_CUDA reports a failed launch or copy;
 *    mnb_last_error_string() then describes it (per calling thread).
 *  - No exception crosses this boundary.
 */
#ifndef MNB_H
#define MNB_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MNB_API __attribute__((visibility("default")))
#else
#define MNB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *mnb_stream_t;

typedef enum {
  MNB_OK = 0,
  MNB_ERR_NULL = -1,        /* a required pointer is NULL                 */
  MNB_ERR_SHAPE = -2,       /* M, N or K out of range                     */
  MNB_ERR_BLOCKSIZE = -3,   /* block_size not a power of two in [16, 256] */
  MNB_ERR_DTYPE = -4,       /* unknown dtype or unsupported combination   */
  MNB_ERR_ALIGN = -5,       /* a pointer breaks its alignment rule        */
  MNB_ERR_ALIAS = -6,       /* the output overlaps an input               */
  MNB_ERR_CUDA = -7,        /* a CUDA launch or copy failed               */
  MNB_ERR_UNSUPPORTED = -8, /* valid request the library cannot serve     */
  MNB_ERR_DEVICE = -9,      /* current device is not an sm_103 GPU        */
  MNB_ERR_LAYOUT = -10      /* a packed weight does not match the call, or
                               the library holds no header for it         */
} mnb_status;

typedef enum { MNB_F32 = 0, MNB_BF16 = 1 } mnb_dtype;

/* Path selection for mnb_matmul_path (the crossover sweep forces a path). */
typedef enum {
  MNB_PATH_AUTO = 0, /* small-M kernel for M <= 16, tensor-core GEMM above */
  MNB_PATH_GEMV = 1, /* split-K decode kernel (M <= 16)                    */
  MNB_PATH_GEMM = 2, /* TMA + tcgen05/TMEM prefill kernel (any M)          */
  MNB_PATH_GEMM_STREAMK = 3, /* the same kernel's stream-K schedule: bf16
                               activations, a single weight and a workspace
                               (mnb_matmul_ws), else MNB_ERR_UNSUPPORTED     */
  MNB_PATH_GEMM_PAIR = 4 /* persistent CTA-pair tensor-core kernel
                            (tcgen05.mma.cta_group::2, 256-row tiles): bf16
                            activations and a single weight, else
                            MNB_ERR_UNSUPPORTED                           */
} mnb_path;

/* Human-readable name of a status code (static string, never NULL). */
MNB_API const char *mnb_status_string(int status);

/* Description of the last failing call on the calling thread (static buffer
 * owned by the library, valid until the thread's next failing call). */
MNB_API const char *mnb_last_error_string(void);

/* Library ABI version: (major << 16) | minor. */
MNB_API int mnb_version(void);

/*
 * Packed-weight header (page "Qwen3 CPU Inference Critical Path", section
 * "Prepared weight-only plan": the plan captures K, N, the nibble order and
 * the block size, and packed weights are reused by every token).
 *
 * Every prepack call writes one into the last MNB_PACKED_HEADER_BYTES bytes
 * of packed_b, so a packed weight saved with its three buffers carries its
 * own description, and records it on the host, keyed by packed_b's device
 * address. Every call that reads a packed weight (the matmul entry points,
 * mnb_unprepack, mnb_chain_build, mnb_chain_run_noalloc) first compares the
 * header recorded for its packed_b with the call's N, K, block_size, scale
 * dtype, zero-point presence (a zero_points pointer given or not) and code
 * form, on the host, after the argument checks and before anything is
 * enqueued: a mismatch, or a packed_b for which the library holds no
 * header, returns MNB_ERR_LAYOUT with the differing field in
 * mnb_last_error_string(). A weight restored from storage into new device
 * buffers is made known with mnb_packed_read_header + mnb_packed_register.
 */
#define MNB_PACKED_MAGIC 0x4B43415034424E4DULL /* the bytes "MNB4PACK" */
#define MNB_PACKED_VERSION 1u
#define MNB_PACKED_HEADER_BYTES 256

typedef enum {
  MNB_CODES_AFFINE = 0,  /* w = (q - z) * s: mnb_prepack, mnb_prepack_qdq */
  MNB_CODES_CODEBOOK = 1 /* w = code[q] * absmax: mnb_prepack_bnb4        */
} mnb_codes;

typedef struct {
  uint64_t magic;          /* MNB_PACKED_MAGIC                              */
  uint32_t version;        /* MNB_PACKED_VERSION                            */
  uint32_t codes;          /* mnb_codes                                     */
  int64_t N, K;
  int32_t block_size;
  int32_t scale_dtype;     /* mnb_dtype of the scales (absmax)              */
  int32_t has_zero_points; /* 0 or 1                                        */
  int32_t reserved;        /* 0                                             */
  uint64_t packed_b_bytes, packed_scales_bytes, packed_zp_bytes;
  uint64_t check;          /* FNV-1a 64 of the 72 bytes before this field   */
} mnb_packed_header;

/* The header a prepack call writes for these arguments (pure host
 * arithmetic). Errors: MNB_ERR_NULL, MNB_ERR_SHAPE, MNB_ERR_BLOCKSIZE,
 * MNB_ERR_DTYPE, MNB_ERR_UNSUPPORTED (codes not an mnb_codes value, or a
 * code-book weight with zero points). */
MNB_API mnb_status mnb_packed_header_make(int64_t N, int64_t K, int block_size,
                                          mnb_dtype scale_dtype, int has_zero_points,
                                          int codes, mnb_packed_header *out);

/* Records `header` (HOST) for the packed weight whose codes start at
 * packed_b (DEVICE address; not dereferenced), replacing any earlier record
 * for that address. Errors: MNB_ERR_NULL, MNB_ERR_LAYOUT (wrong magic or
 * version, a check that does not match, or fields no prepack call writes). */
MNB_API mnb_status mnb_packed_register(const void *packed_b, const mnb_packed_header *header);

/* Copies the header stored in the last MNB_PACKED_HEADER_BYTES bytes of
 * packed_b (DEVICE, packed_b_bytes long) into *out (HOST) and validates it
 * as mnb_packed_register does; waits for the copy (synchronous with respect
 * to the host, ordered on `stream`). Nothing is recorded. Errors:
 * MNB_ERR_NULL, MNB_ERR_SHAPE (packed_b_bytes too small or not the size the
 * header gives), MNB_ERR_LAYOUT, MNB_ERR_DEVICE, MNB_ERR_CUDA. */
MNB_API mnb_status mnb_packed_read_header(const void *packed_b, size_t packed_b_bytes,
                                          mnb_packed_header *out, mnb_stream_t stream);

/* Drops the record for packed_b (before its buffer is freed or reused for
 * something else). MNB_OK whether or not there was one; MNB_ERR_NULL. */
MNB_API mnb_status mnb_packed_forget(const void *packed_b);

/*
 * Sizes in bytes of the three prepacked buffers for an N x K weight
 * (section "Prepared weight-only plan": packed constant storage aligned for
 * the selected kernel). HOST outputs; zp_bytes is 0 when has_zero_points is
 * 0. The packed layout pads N up to a multiple of 16 and K up to a multiple
 * of 64 with zero codes; for N % 16 == 0 and K % 64 == 0 the packed codes
 * take exactly the N*K/2 bytes of the input, and packed_b holds them
 * followed by the MNB_PACKED_HEADER_BYTES-byte header. Zero points take 4
 * bits per (row, block), with rows padded to 16 and blocks to an even count.
 * Errors: MNB_ERR_NULL (an output pointer), MNB_ERR_SHAPE (N or K < 1),
 * MNB_ERR_BLOCKSIZE, MNB_ERR_DTYPE.
 */
MNB_API mnb_status mnb_prepacked_sizes(int64_t N, int64_t K, int block_size,
                                       mnb_dtype scale_dtype,
                                       int has_zero_points,
                                       size_t *packed_b_bytes,
                                       size_t *packed_scales_bytes,
                                       size_t *packed_zp_bytes);

/*
 * Offline re-layout of one MatMulNBits weight into the prepacked form the
 * kernels stream with 128-bit loads (run once per weight; section "Prepared
 * weight-only plan" and section "Phase Q1", item "plan-owned packed weights
 * reused by every token").
 *
 *  B            uint8 [N, nb, bs/2], nb = ceil(K/bs): element k of row n is
 *               byte (k mod bs)/2 of block k/bs, even k in the low nibble
 *               (the MatMulNBits "packed UINT8 storage").
 *  scales       [N, nb] in scale_dtype (fp32, or bf16 as raw 16-bit words).
 *  zero_points  uint8 [N, ceil(nb/2)], even block in the low nibble, or NULL
 *               (every zero point is 8; packed_zp is then not written).
 *  packed_b, packed_scales, packed_zp: outputs of the sizes given by
 *               mnb_prepacked_sizes, 16-byte aligned.
 * The re-layout is lossless for every code with k < K; the storage padding
 * nibbles past K in the last block are not kept. Inputs need only byte
 * (B, zero_points) or element (scales) alignment. The last kernel it
 * enqueues writes the packed-weight header into packed_b and nothing else
 * (see mnb_set_programmatic_launch); the header is also recorded on the
 * host for packed_b (affine codes).
 * Errors: MNB_ERR_NULL, MNB_ERR_SHAPE, MNB_ERR_BLOCKSIZE, MNB_ERR_DTYPE,
 * MNB_ERR_ALIGN (a packed output not 16-byte aligned), MNB_ERR_ALIAS (an
 * output overlaps an input or another output), MNB_ERR_CUDA.
 */
MNB_API mnb_status mnb_prepack(const uint8_t *B, const void *scales,
                               const uint8_t *zero_points, int64_t N,
                               int64_t K, int block_size,
                               mnb_dtype scale_dtype, void *packed_b,
                               void *packed_scales, void *packed_zp,
                               mnb_stream_t stream);

/*
 * Offline re-layout of one weight in the standard QDQ INT4 encoding into the
 * same prepacked form (page "Qwen3 CPU Inference Critical Path", section
 * "qwen3-int4-qdq": a logical UINT4 initializer in ONNX row-major,
 * low-nibble-first storage, DequantizeLinear with block_size along one axis,
 * then MatMul). The packed weight then runs through mnb_matmul like any
 * other, computing Y[m,n] = sum_k A[m,k] (q - z) s + bias[n] with
 *   axis 0 (projections):   q = Bq[k, n] of a logical [K, N] matrix,
 *                           s = scales[k / bs, n], z = zero_points[k / bs, n];
 *   axis 1 (tied LM head):  q = Bq[n, k] of a logical [N, K] matrix,
 *                           s = scales[n, k / bs], z = zero_points[n, k / bs].
 *  B_qdq        uint8, ceil(K*N / 2) bytes: element i of the flattened
 *               logical matrix is nibble i, low nibble first.
 *  scales       [ceil(K/bs), N] (axis 0) or [N, ceil(K/bs)] (axis 1), in
 *               scale_dtype (fp32, or bf16 as raw 16-bit words).
 *  zero_points  UINT4 of the scales' shape, flattened low-nibble-first
 *               (ceil(nb*N / 2) bytes), or NULL: every zero point is 0, the
 *               DequantizeLinear default. packed_zp is always written.
 *  packed_b, packed_scales, packed_zp: outputs of the sizes given by
 *               mnb_prepacked_sizes(..., has_zero_points = 1), 16-byte
 *               aligned.
 * Use the packed weight with zero points (pass packed_zp to mnb_matmul).
 * Errors: as mnb_prepack, and MNB_ERR_SHAPE for an axis other than 0 or 1.
 */
MNB_API mnb_status mnb_prepack_qdq(const uint8_t *B_qdq, const void *scales,
                                   const uint8_t *zero_points, int axis,
                                   int64_t N, int64_t K, int block_size,
                                   mnb_dtype scale_dtype, void *packed_b,
                                   void *packed_scales, void *packed_zp,
                                   mnb_stream_t stream);

/*
 * Inverse of mnb_prepack: writes B [N, nb, bs/2] (padding nibbles past K set
 * to 0), scales [N, nb] and, when packed_zp is not NULL, zero_points
 * [N, ceil(nb/2)] (an unused high nibble of an odd nb set to 0). Used to
 * prove the re-layout lossless. Same error rules as mnb_prepack.
 */
MNB_API mnb_status mnb_unprepack(const void *packed_b,
                                 const void *packed_scales,
                                 const void *packed_zp, int64_t N, int64_t K,
                                 int block_size, mnb_dtype scale_dtype,
                                 uint8_t *B, void *scales,
                                 uint8_t *zero_points, mnb_stream_t stream);

/*
 * Y = A * dequant(B)^T + bias on the prepacked weight.
 *
 *  A            [M, K] row-major in a_dtype (fp32 or bf16), element-aligned.
 *  packed_b     prepacked codes from mnb_prepack (16-byte aligned).
 *  scales       prepacked scales from mnb_prepack, in scale_dtype.
 *  zero_points  prepacked zero points from mnb_prepack, or NULL for the
 *               default zero point 8 (must match how the weight was packed).
 *  bias         fp32 [N] or NULL.
 *  Y            [M, N] row-major in a_dtype; bf16 results are rounded to
 *               nearest even from the fp32 accumulator. Must not overlap
 *               any input.
 *  M >= 1, N >= 1, K >= 1, each below 2^31; block_size a power of two in
 *  [16, 256], matching the prepacked weight.
 * Accumulation is fp32. Results are bitwise reproducible for a given device,
 * shape and path (every split-K reduction runs in a fixed order).
 * Errors: MNB_ERR_NULL, MNB_ERR_SHAPE, MNB_ERR_BLOCKSIZE, MNB_ERR_DTYPE,
 * MNB_ERR_ALIGN, MNB_ERR_ALIAS, MNB_ERR_LAYOUT (the header recorded for
 * packed_b differs from N, K, block_size, scale_dtype, zero-point presence
 * or the affine code form, or there is none), MNB_ERR_UNSUPPORTED (no kernel
 * for this combination), MNB_ERR_DEVICE, MNB_ERR_CUDA. Every other call that
 * reads a packed weight checks its header the same way.
 */
MNB_API mnb_status mnb_matmul(const void *A, const void *packed_b,
                              const void *scales, const void *zero_points,
                              const float *bias, int64_t M, int64_t N,
                              int64_t K, int block_size, void *Y,
                              mnb_dtype a_dtype, mnb_dtype scale_dtype,
                              mnb_stream_t stream);

/* mnb_matmul with the kernel path forced (MNB_PATH_GEMV needs M <= 16,
 * else MNB_ERR_UNSUPPORTED). */
MNB_API mnb_status mnb_matmul_path(const void *A, const void *packed_b,
                                   const void *scales, const void *zero_points,
                                   const float *bias, int64_t M, int64_t N,
                                   int64_t K, int block_size, void *Y,
                                   mnb_dtype a_dtype, mnb_dtype scale_dtype,
                                   mnb_path path, mnb_stream_t stream);

/*
 * Bytes of workspace that let mnb_matmul_ws run its stream-K schedule on the
 * current device (0 when no usable device is current): a 4096-byte page of
 * counters, then two 256 x 128 fp32 partial tiles (256 KiB) for each CTA of
 * the grid, two CTAs per SM.
 */
MNB_API size_t mnb_matmul_workspace_size(void);

/*
 * mnb_matmul with the path chosen as in mnb_matmul_path and a caller-owned
 * device workspace. With M > 16 and bf16 activations on a single weight, the
 * tensor-core path may then split the product's (output tile, 64-wide k
 * stage) units evenly over two CTAs per SM instead of giving each CTA a
 * whole tile, where its cost model expects that to be faster: shapes whose
 * 256 x 128 tiles leave SMs idle (few output tiles, or just more than the
 * resident CTAs can take at once). A tile that several CTAs share is
 * completed by whichever of them finishes last, adding the fp32 partial sums
 * in the order of their k stages; no CTA waits for another. Results are
 * bitwise reproducible for a given device and shape, and within the same
 * bound as mnb_matmul. The pages
 * describe no such schedule (their kernels run on CPU cores); the operation
 * computed is unchanged.
 *  workspace: NULL (then exactly mnb_matmul_path), or device memory of
 *    workspace_bytes bytes, 256-byte aligned, overlapping no input or output.
 *    Its first 4096 bytes (the counters) must be zero before the first call
 *    that uses it; every call leaves them zero again, unless
 *    mnb_fault_status reports a fault, after which the caller zeroes them
 *    before the next call. One workspace serves calls that are ordered one
 *    after another (one stream, or a CUDA graph); concurrent calls need
 *    their own. A workspace smaller than mnb_matmul_workspace_size() limits
 *    the grid (one CTA per 256 KiB); one of 4096 bytes or less is not used.
 * Errors: as mnb_matmul_path; MNB_ERR_ALIGN (workspace alignment),
 * MNB_ERR_ALIAS (workspace overlaps an input or Y).
 */
MNB_API mnb_status mnb_matmul_ws(const void *A, const void *packed_b,
                                 const void *scales, const void *zero_points,
                                 const float *bias, int64_t M, int64_t N,
                                 int64_t K, int block_size, void *Y,
                                 mnb_dtype a_dtype, mnb_dtype scale_dtype,
                                 mnb_path path, void *workspace,
                                 size_t workspace_bytes, mnb_stream_t stream);

/*
 * What mnb_matmul_ws would launch for a product: the kernel and, on the
 * tensor-core path, its tile height, K split, schedule and epilogue. Pure
 * host arithmetic (the same cost models the launch uses), for a GPU with
 * sm_count SMs (0: the current device's). Activations and Y are taken to be
 * 16-byte aligned, a workspace of workspace_bytes present when it is not 0.
 * No counterpart in the pages; it reports, it computes nothing.
 *  out: filled on MNB_OK.
 * Errors: MNB_ERR_NULL (out), the argument errors of mnb_matmul_path,
 * MNB_ERR_UNSUPPORTED (a forced path that cannot serve the product),
 * MNB_ERR_DEVICE / MNB_ERR_CUDA (sm_count 0 without a usable device).
 */
typedef struct {
  int32_t path;      /* MNB_PATH_GEMV (the decode kernel) or MNB_PATH_GEMM  */
  int32_t m_slices;  /* decode kernel over 16-row slices of A (activations
                        the tensor-core kernel cannot stage): how many; else 0 */
  int32_t tile_rows; /* tensor-core kernel: output rows per tile (128, 256)  */
  int32_t k_split;   /* tensor-core kernel: CTAs of a cluster sharing a
                        tile's k range (1, 2, 4, 8)                          */
  int32_t stream_k;  /* 1: the stream-K schedule                             */
  int32_t tf32;      /* 1: the tf32 kernel (fp32 activations)                */
  int32_t tma_store; /* 1: the output tile goes out through TMA stores      */
  int32_t pair_cols; /* persistent CTA-pair kernel: output columns per
                        256-row tile (128 .. 256); 0: another kernel        */
  int64_t ctas;      /* CTAs of the tensor-core launch                       */
} mnb_matmul_plan_info;

MNB_API mnb_status mnb_matmul_plan(int64_t M, int64_t N, int64_t K,
                                   int block_size, mnb_dtype a_dtype,
                                   mnb_dtype scale_dtype, int has_zero_points,
                                   mnb_path path, size_t workspace_bytes,
                                   int sm_count, mnb_matmul_plan_info *out);

/*
 * Fused-N projections: Y_i = A * dequant(B_i)^T + bias_i for i < count
 * (1 <= count <= 4), for weights that read the same activations, such as
 * the q/k/v or the gate/up projections of a decoder layer (page "Qwen3 CPU
 * Inference Critical Path", section "Exact kernel inventory": the artifact's
 * fused 1024x4096 QKV projection and its Split row; section "Phase Q5":
 * fusions that remove measured memory traffic). One launch streams every
 * weight of the group; A is read once.
 *  packed_b, scales, zero_points, bias, N, Y: HOST arrays of count entries
 *  (device pointers inside, except N). zero_points is NULL or holds count
 *  entries that are all NULL or all non-NULL; bias may be NULL or hold NULL
 *  entries. Every weight shares K, block_size and the dtypes.
 * M <= 16 runs the decode kernel once for the whole group; larger M runs
 * one product per weight. Errors: as mnb_matmul, for every entry; Y_i must
 * not overlap any input or any other output.
 */
MNB_API mnb_status mnb_matmul_grouped(const void *A, int count,
                                      const void *const *packed_b,
                                      const void *const *scales,
                                      const void *const *zero_points,
                                      const float *const *bias,
                                      const int64_t *N, void *const *Y,
                                      int64_t M, int64_t K, int block_size,
                                      mnb_dtype a_dtype, mnb_dtype scale_dtype,
                                      mnb_stream_t stream);

/*
 * mnb_matmul for callers whose activations and results live in HOST memory:
 * copies A_host [M, K] into the caller's device buffer A_dev, runs the
 * product into Y_dev, and copies Y_dev back into Y_host [M, N], all
 * enqueued on stream (page-locked host buffers make the copies
 * asynchronous; pageable ones make them synchronous with the host). The
 * host buffers must stay valid until the stream reaches this point.
 * Errors: as mnb_matmul; MNB_ERR_NULL also for the host buffers.
 */
MNB_API mnb_status mnb_matmul_from_host(const void *A_host, void *A_dev,
                                        const void *packed_b,
                                        const void *scales,
                                        const void *zero_points,
                                        const float *bias, int64_t M,
                                        int64_t N, int64_t K, int block_size,
                                        void *Y_dev, void *Y_host,
                                        mnb_dtype a_dtype,
                                        mnb_dtype scale_dtype,
                                        mnb_stream_t stream);

/*
 * Gated-MLP projection pair in one call (page "Qwen3 CPU Inference Critical
 * Path": the graph-level fusion "gate projection, SiLU, and gate/up
 * multiplication", with SiLU computed as x * Sigmoid(x) in FP32 as in the
 * audited graph):
 *   g = A * dequant(gate)^T + bias_gate,  u = A * dequant(up)^T + bias_up,
 *   Y[m,n] = g * sigmoid(g) * u  (fp32, then A's dtype; bf16 to nearest even).
 * gate and up are two prepacked weights of the same N, K, block_size, scale
 * dtype and zero-point presence; each CTA streams matching rows of both, so
 * neither projection is written to memory (M <= 16: the decode kernel; more
 * rows: the tensor-core kernel for bf16 activations with 16-byte-aligned
 * rows, else the decode kernel over 16-row slices). All pointers DEVICE;
 * Y [M, N].
 * Arguments and errors as mnb_matmul (both zero-point pointers set, or both
 * NULL: MNB_ERR_NULL otherwise); Y must not overlap any input.
 */
MNB_API mnb_status mnb_matmul_gate_up(const void *A, const void *packed_gate,
                                      const void *scales_gate, const void *zp_gate,
                                      const float *bias_gate, const void *packed_up,
                                      const void *scales_up, const void *zp_up,
                                      const float *bias_up, int64_t M, int64_t N,
                                      int64_t K, int block_size, void *Y,
                                      mnb_dtype a_dtype, mnb_dtype scale_dtype,
                                      mnb_stream_t stream);

/*
 * Programmatic dependent launch (on by default): each matmul kernel lets the
 * next kernel on the stream launch early and starts streaming its own
 * (constant) prepacked weights before the previous kernel has finished; it
 * reads A, and writes Y, only after that kernel's results are visible. The
 * packed buffers must therefore have been written before the previous
 * kernel on the stream started; mnb_prepack guarantees this by ending with
 * an empty kernel. Pass 0 to launch every kernel in plain stream order.
 * Process-wide setting.
 */
MNB_API void mnb_set_programmatic_launch(int enable);

/*
 * Failure detection. Every wait inside a kernel (on a bulk copy's mbarrier)
 * has an iteration cap far above any legitimate wait; a kernel whose wait
 * runs out records a bit in a device fault word, abandons its tile and
 * exits instead of hanging. This call waits for the current device to be
 * idle, returns the fault bits seen since the last call in *fault_bits
 * (HOST; 0 = none; 1 = decode kernel, 2 = a tensor-core kernel, 4 = decode
 * chain) and clears
 * them. Errors: MNB_ERR_NULL, MNB_ERR_CUDA.
 */
MNB_API mnb_status mnb_fault_status(unsigned int *fault_bits);

/*
 * Test-only failure injection for the decode kernel (off by default), so that
 * the bounded waits above can be exercised without faulting a GPU. While
 * stop_stage >= 0, decode-kernel launches of one configuration (bf16
 * activations and scales, block_size 128, no zero points, M <= 8) whose
 * CTAs work without a cluster run a separate instantiation of the kernel
 * whose waits give up after 2^16 iterations and whose CTA 0 producer issues
 * weight stages 0 .. stop_stage - 1 and then stops. CTA 0's consumers, having
 * consumed every copy issued, wait for stage stop_stage, give up, record
 * fault bit 1 and end the launch (the CTA's outputs are then wrong; nothing
 * is left in flight and the context stays usable). Every other launch, and
 * every launch while stop_stage < 0, is unaffected (the normal kernels hold
 * none of this). Process-wide; launches recorded into a CUDA graph keep the
 * setting of their recording.
 */
MNB_API void mnb_test_wait_fault(int stop_stage);

/*
 * Projection of an RMS-normalized row, optionally followed by greedy ArgMax
 * (page "Qwen3 CPU Inference Critical Path": the fusions "RMSNorm into packed
 * projection input" and "final RMSNorm, LM-head GEMV, and greedy ArgMax";
 * the normalization is the inventory's SimplifiedLayerNormalization, FP32
 * RMS-style normalization over the last axis, epsilon 1e-6 in the audited
 * graph):
 *
 *   a'[m,k] = A[m,k] / sqrt(mean_k A[m,k]^2 + epsilon) * gamma[k]   (normalize = 1)
 *   a'      = A                                                     (normalize = 0)
 *   Y[m,n]  = sum_k a'[m,k] * dequant(B)[n,k] + bias[n]
 *   argmax[m] = the smallest n with the largest Y[m,n]
 *
 * in one decode-kernel launch for M <= 16 (plus a one-block finishing kernel
 * for the ArgMax). Prefill rows (M > 16, bf16 activations whose rows TMA
 * can stage, no ArgMax) run the tensor-core kernel in one launch: each
 * staged A tile is multiplied by gamma in place and every output row scaled
 * by its r[m], summed over the whole K (no K split); other rows (fp32, rows
 * not 16-byte aligned, or with the ArgMax) run the decode kernel over
 * 16-row slices, each normalizing its own rows. gamma: fp32 [K] DEVICE or
 * NULL (1); the sum of squares and the scale are fp32; a normalized bf16
 * row is rounded to bf16 once before the products (as the unfused graph
 * rounds the normalization's output). Y [M, N] in A's dtype, or NULL when
 * only argmax is wanted (the logits are then never written). argmax: int64
 * [M] DEVICE or NULL; the comparison uses the fp32 value of each output
 * before it is rounded to A's dtype. Other arguments as mnb_matmul.
 * Errors: as mnb_matmul; MNB_ERR_NULL if Y and argmax are both NULL;
 * MNB_ERR_SHAPE for normalize not 0/1 or a negative or non-finite epsilon;
 * MNB_ERR_ALIGN for gamma (4 bytes) or argmax (8 bytes); MNB_ERR_ALIAS if Y
 * or argmax overlaps an input or each other.
 */
MNB_API mnb_status mnb_matmul_rmsnorm(const void *A, int normalize, const float *gamma,
                                      float epsilon, const void *packed_b,
                                      const void *scales, const void *zero_points,
                                      const float *bias, int64_t M, int64_t N, int64_t K,
                                      int block_size, void *Y, int64_t *argmax,
                                      mnb_dtype a_dtype, mnb_dtype scale_dtype,
                                      mnb_stream_t stream);

/*
 * The bitsandbytes-style 4-bit matrix (page "Qwen3 CPU Inference Critical
 * Path", com.microsoft operator inventory, row MatMulBnb4: an alternative
 * bitsandbytes-style 4-bit matrix format, adapted into the same weight-only
 * plan). The pages name the format only; this library reads it as:
 *   B       uint8 [(N*K + 1) / 2] DEVICE: the N x K weight (row n = output
 *           n) flattened row-major, two codes per byte, the first of each
 *           pair in the HIGH nibble;
 *   absmax  [N*K / block_size] DEVICE, fp32 or bf16 (absmax_dtype): one
 *           scale per block_size consecutive flattened elements;
 *   code    fp32 [16] DEVICE: the code book (NF4, FP4 or any other);
 *   w[n,k]  = code[q] * absmax[(n*K + k) / block_size]
 *   Y[m,n]  = sum_k A[m,k] w[n,k] + bias[n]
 * K must be a multiple of block_size (a block may not straddle two rows of
 * the plan), and block_size a power of two in [16, 256].
 *
 * mnb_prepack_bnb4 re-lays out B and absmax into the packed plan (codes as
 * mnb_prepack's, absmax as its scales; sizes from mnb_prepacked_sizes with
 * no zero points). Errors: as mnb_prepack; MNB_ERR_UNSUPPORTED when K is
 * not a multiple of block_size.
 *
 * mnb_matmul_bnb4 runs the decode kernel with the code book for M <= 16
 * (8-row launches): each CTA turns the 16 values into a table of bf16 pairs,
 * each value c held as hi = bf16(c) and lo = bf16(c - hi) and both
 * multiplied by the activations, so every weight is within 2^-16 |c| of
 * code[q], times the fp32 or bf16 absmax applied in fp32. Above 16 rows,
 * bf16 activations with 16-byte-aligned rows run the tensor-core kernel's
 * code-book mode (w = code[q] * absmax formed in fp32 and fed as an exact
 * hi + lo bf16 pair); other activations run 8-row decode launches.
 * Errors: as mnb_matmul;
 * MNB_ERR_NULL for code; MNB_ERR_ALIAS if Y overlaps code.
 */
MNB_API mnb_status mnb_prepack_bnb4(const uint8_t *B, const void *absmax, int64_t N,
                                    int64_t K, int block_size, mnb_dtype absmax_dtype,
                                    void *packed_b, void *packed_scales, mnb_stream_t stream);
MNB_API mnb_status mnb_matmul_bnb4(const void *A, const void *packed_b,
                                   const void *packed_scales, const float *code,
                                   const float *bias, int64_t M, int64_t N, int64_t K,
                                   int block_size, void *Y, mnb_dtype a_dtype,
                                   mnb_dtype absmax_dtype, mnb_stream_t stream);

/*
 * Decode chain: a sequence of MatMulNBits projections with declared data
 * dependencies, run as ONE persistent cooperative kernel launch.
 *
 * The page "Qwen3 CPU Inference Critical Path" (section "Prepared
 * weight-only plan") describes one operator call per projection; a decode
 * step of a transformer runs hundreds of them back to back (per layer
 * q/k/v, o, gate/up and down, then the LM head), each small enough that a
 * kernel launch's fixed start and drain cost rivals its weight streaming.
 * This entry point has no counterpart in the pages: it is the GB300
 * executor for such a sequence. Every op computes exactly what
 * mnb_matmul (or, for a gated-MLP pair, mnb_matmul_gate_up) computes for
 * its arguments; results are bitwise identical from run to run.
 *
 * Execution: one CTA per resident slot of every SM (cooperative launch, so
 * all CTAs run at once). Each CTA streams the packed weights of its share
 * of every op, in op order, through a ring of shared-memory stages, across
 * op boundaries; an op's activations are read only after every op listed in
 * its deps[] has stored all of its Y (device-scope release/acquire on a
 * per-op completion counter in the plan buffer). Every wait is bounded: a
 * wait that runs out records fault bit 4 (mnb_fault_status), makes every
 * other wait of the launch give up at once, and the launch ends with the
 * plan's counters reset.
 */
typedef struct {
  const void *A;         /* [M, K] activations, a_dtype                      */
  void *Y;               /* [M, N] output, a_dtype                           */
  const void *packed_b;  /* prepacked weight (mnb_prepack / mnb_prepack_qdq) */
  const void *packed_scales;
  const void *packed_zp; /* NULL: zero point 8                               */
  const float *bias;     /* [N] fp32 or NULL                                 */
  /* Gated-MLP pair: the up weight (same N, K), else all four NULL; then
   * Y = silu(A gate^T + bias) * (A up^T + bias_up), silu(x) = x sigmoid(x). */
  const void *packed_b_up;
  const void *packed_scales_up;
  const void *packed_zp_up;
  const float *bias_up;
  int64_t N, K;
  /* Indices of EARLIER ops whose Y must be complete before this op reads
   * A; -1 = unused slot. */
  int32_t deps[4];
} mnb_chain_op;

/* Launch description filled by mnb_chain_build (HOST struct; pass it
 * unchanged to mnb_chain_run together with the plan buffer it was built
 * for). */
typedef struct {
  uint64_t plan_bytes;  /* device bytes the plan buffer needs             */
  int32_t n_ops, n_segments, grid, smem_bytes;
  int32_t M, block_size, a_dtype, scale_dtype, has_zero_points;
  int32_t ring_stages, k_max, tiles_per_segment, ctas_per_sm;
  uint64_t check;       /* checksum of the fields above                   */
} mnb_chain_info;

/*
 * Plans a chain. ops: HOST array of n_ops (1..4096) op descriptors, all with
 * the same block_size, activation dtype, scale dtype and zero-point presence
 * (DEVICE pointers inside). M: activation rows, 1..8.
 *
 * With plan == NULL only *info is filled (info->plan_bytes tells how large
 * the plan buffer must be). Otherwise plan is a caller-owned DEVICE buffer
 * of plan_bytes >= info->plan_bytes bytes, 256-byte aligned; the schedule
 * (which CTA streams which 16-row tiles of which op), the op table and the
 * completion counters are written into it with a copy on `stream`, and the
 * call returns after that copy finished (the host image it copies from is
 * freed on return). The plan holds the op descriptors' device pointers: the
 * buffers must stay allocated while the plan is used. A plan runs on one
 * stream at a time.
 *
 * Hazards are checked: op j may read an earlier op's Y, overwrite an
 * earlier op's A or Y, only if that op is among j's (transitive) deps;
 * no Y may overlap any packed weight or bias of the chain, nor its own A.
 * Errors: MNB_ERR_NULL, MNB_ERR_SHAPE (M, N, K, n_ops, a deps entry not an
 * earlier op), MNB_ERR_BLOCKSIZE, MNB_ERR_DTYPE, MNB_ERR_ALIGN (as
 * mnb_matmul; plan not 256-byte aligned), MNB_ERR_ALIAS (a hazard above,
 * or the plan overlaps a buffer of an op), MNB_ERR_SHAPE also for
 * plan_bytes too small, MNB_ERR_UNSUPPORTED (the shared-memory layout
 * does not fit: M or K too large), MNB_ERR_DEVICE, MNB_ERR_CUDA.
 */
MNB_API mnb_status mnb_chain_build(const mnb_chain_op *ops, int32_t n_ops,
                                   int64_t M, int block_size,
                                   mnb_dtype a_dtype, mnb_dtype scale_dtype,
                                   void *plan, size_t plan_bytes,
                                   mnb_chain_info *info, mnb_stream_t stream);

/*
 * Runs a built chain: one cooperative launch on `stream`. plan: DEVICE
 * buffer written by mnb_chain_build; info: HOST, from the same build.
 * Errors: MNB_ERR_NULL, MNB_ERR_SHAPE (info altered: checksum mismatch),
 * MNB_ERR_DEVICE, MNB_ERR_CUDA (the launch failed, e.g. the device cannot
 * hold every CTA at once).
 */
MNB_API mnb_status mnb_chain_run(const void *plan, const mnb_chain_info *info,
                                 mnb_stream_t stream);

/*
 * Decode chain without a caller-provided plan buffer. The paper has no
 * counterpart for this call: it exists for callers that cannot call
 * cudaMalloc, for example a plugin whose host runtime owns every device
 * allocation through its own pool and forbids direct allocation, or a
 * process whose device memory is fully reserved up front (weights, KV
 * cache) so that no allocation may happen while it serves.
 *
 * Same ops, rules and errors as mnb_chain_build followed by mnb_chain_run,
 * with the plan written into a fixed array inside the library (1 MiB on
 * every GPU that loads the library, held until the process exits) instead
 * of a caller buffer; the library allocates no device memory. Each call
 * plans again (host work), copies the plan into the array, waits on the
 * host until that copy has finished on `stream` (so every call
 * synchronises `stream` and none can be recorded by a stream capture: a
 * capturing stream cannot be synchronised, and the capture would be
 * invalidated), then launches; the copy also clears the
 * completion counters the launch starts from. A chain whose plan exceeds
 * the array is rejected with MNB_ERR_UNSUPPORTED and a message giving both
 * sizes (the Qwen3-4B decode step needs about 0.6 MB).
 *
 * Every call shares the one array: calls whose work overlaps on the GPU
 * (two streams, or two host threads) race and must be serialised by the
 * caller. The first call on a device looks up the array's device address
 * (once per device, with that device current) and keeps it for the life of
 * the process; do not use this entry point on a device after
 * cudaDeviceReset (the kept address would no longer map the array).
 */
MNB_API mnb_status mnb_chain_run_noalloc(const mnb_chain_op *ops, int32_t n_ops,
                                         int64_t M, int block_size,
                                         mnb_dtype a_dtype, mnb_dtype scale_dtype,
                                         mnb_stream_t stream);

/*
 * A sequence of projections as one CUDA graph: the GPU form of the page's
 * session executor around one operator call per projection (page "Qwen3 CPU
 * Inference Critical Path", section "Prepared weight-only plan"). The library
 * records its own launches for the whole sequence once and then runs the
 * sequence with one graph launch per step; no counterpart exists in the
 * pages for the graph itself.
 *
 * mnb_graph_build: ops is a HOST array of n_ops (1..65536) descriptors, run
 * in array order (deps is ignored: each op starts after the one before it
 * on the stream). Consecutive ops without an up weight that read the same A
 * with the same K form one fused-N call (mnb_matmul_grouped, up to 4 ops,
 * M <= 16); an op with an up weight is one gated-MLP call
 * (mnb_matmul_gate_up); any other op is one mnb_matmul call. Every call is
 * validated as that entry point validates it (headers included) while it is
 * recorded; the first failure ends the build with that call's status and
 * message. The graph keeps the descriptors' device pointers: the buffers
 * must stay allocated, and their contents are read (A, weights) and
 * written (Y) each time the graph runs. The graph belongs to the device
 * current at build time; the build records on a private stream and runs
 * nothing. Host memory only (the graph objects); the library allocates no
 * device memory.
 * Errors: MNB_ERR_NULL, MNB_ERR_SHAPE, the recorded calls' errors,
 * MNB_ERR_CUDA (capture or instantiation failed).
 */
typedef struct mnb_graph_st *mnb_graph;
MNB_API mnb_status mnb_graph_build(const mnb_chain_op *ops, int32_t n_ops, int64_t M,
                                   int block_size, mnb_dtype a_dtype, mnb_dtype scale_dtype,
                                   mnb_graph *out);

/* Library calls recorded and kernel nodes in the graph (HOST outputs, each
 * may be NULL). Errors: MNB_ERR_NULL. */
MNB_API mnb_status mnb_graph_info(mnb_graph graph, int32_t *calls, int32_t *kernels);

/* One run of the graph on `stream` (asynchronous). Errors: MNB_ERR_NULL,
 * MNB_ERR_DEVICE (another device is current), MNB_ERR_CUDA. */
MNB_API mnb_status mnb_graph_run(mnb_graph graph, mnb_stream_t stream);

/* One run framed by host copies, all on `stream`: in_bytes from in_host
 * (HOST) to in_dev (DEVICE), the graph, then out_bytes from out_dev (DEVICE)
 * to out_host (HOST). Page-locked host buffers make the copies asynchronous;
 * the host buffers must stay valid until the stream reaches the end of the
 * run. A zero byte count skips that copy. Errors: as mnb_graph_run;
 * MNB_ERR_NULL for a missing buffer of a copy. */
MNB_API mnb_status mnb_graph_run_from_host(mnb_graph graph, const void *in_host,
                                           void *in_dev, size_t in_bytes,
                                           const void *out_dev, void *out_host,
                                           size_t out_bytes, mnb_stream_t stream);

/* Frees the graph (host objects). Errors: MNB_ERR_NULL. */
MNB_API mnb_status mnb_graph_destroy(mnb_graph graph);

#ifdef __cplusplus
}
#endif

#endif /* MNB_H */
