/*
 * mhr_gemm.h -- C ABI of the GB300 (sm_103a) dense matrix-multiply library
 * libmhr_gemm.so.
 *
 * Operation (every gemm_* entry point):
 *
 *     C[i*ldc + j] = sum over k < K of A[i*lda + k] * B[k*ldb + j]
 *     for 0 <= i < M, 0 <= j < N
 *
 * This is the product the pages compute -- "矩阵乘法 tiling:把分块搬进 shared
 * memory,让 GFLOPS 翻百倍", sections 一 and 二 (C = A x B, row-major floats,
 * each output tile built from a row strip of A and a column strip of B);
 * "CUDA 深入浅出（二）：为什么分块可以减少 Global Memory 访问", section
 * "naive kernel 怎么读数据" -- generalised from N x N to M x N x K with leading
 * dimensions.  As on the pages, K-tiles of A and B are staged on chip so that
 * each element read from HBM is reused across a whole output tile.
 *
 * Layout: all three matrices are row-major.  lda >= K, ldb >= N, ldc >= N
 * (elements, not bytes).  C is overwritten (no accumulation into prior
 * contents).  Elements of C outside the logical M x N block (the ld padding)
 * are never written.  K == 0 writes zeros to C (the empty sum); M == 0 or
 * N == 0 is a no-op.  Sizes that are not tile multiples are handled: inputs
 * outside the matrix count as zero, outputs outside it are not written
 * ("矩阵乘法 tiling", section 六; "CUDA 编程系列之三", section 7).
 *
 * Pointers: A, B and C are DEVICE pointers on the current CUDA device.  The
 * caller owns them; the library never frees or retains them.  C must not
 * overlap A or B (rejected with MHR_ERR_INVALID_ARG).
 *
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 * default stream).  Calls enqueue their work on it and return without
 * waiting.  A launch-time failure is returned at once; a device-side failure
 * (a bounded wait that ran out) is recorded in a per-device status word that
 * gemm_check() reads.
 *
 * Scratch: gemm_f32_3xtf32 (normally) and gemm_bf16_f32acc (only when an
 * operand's address or leading dimension is not 16-byte aligned) need a
 * device workspace.  The library owns it: one buffer per (device, stream),
 * grown with cudaMalloc on demand and kept until gemm_release(), for at most
 * four streams per device -- a call on a fifth stream first frees the least
 * recently used stream's buffer, after waiting for that stream's last call
 * to finish.  Each call makes its stream wait for the previous call that used
 * the same buffer, so a stream handle that comes back after cudaStreamDestroy
 * (with the destroyed stream's work still running) is safe.  When the 3xTF32
 * workspace cannot be allocated, gemm_f32_3xtf32 splits its operands inside
 * the kernel instead (same result bit for bit, slower, no workspace).
 *
 * Errors: every entry point returns an int status (mhr_status below); none
 * throws, none traps on the device.  Thread safety: calls from several host
 * threads are serialised on an internal lock.
 */
#ifndef MHR_GEMM_H
#define MHR_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mhr_status {
  MHR_OK = 0,
  MHR_ERR_INVALID_ARG = 1, /* NULL pointer with nonzero size, negative size,
                              ld too small, size overflow, C overlapping A/B */
  MHR_ERR_UNSUPPORTED = 2, /* current device is not sm_103 (GB300) */
  MHR_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch,
                              allocation, tensor-map encode) */
  MHR_ERR_TIMEOUT = 4      /* a device-side bounded wait ran out; the kernel
                              stopped early and C is not valid */
} mhr_status;

/*
 * Strict-FP32 path: a register-tiled SIMT kernel (fp32 FMA, fp32
 * accumulation).  128 x 128 output tile per block, K staged through a
 * double-buffered shared-memory ring, each thread accumulating an 8 x 8
 * register block ("矩阵乘法 tiling", sections 四 and 五: thread coarsening,
 * accumulator in registers; "CUDA 编程系列之三", section 6: register tiling).
 * Aligned problems whose sizes are multiples of 128 x 256 x 8 use 128 x 256
 * tiles with 8 x 16 register blocks where that shortens the deepest queue of
 * blocks on one SM; problems with few tiles give each tile a cluster of CTAs
 * that split K and sum their partial tiles in distributed shared memory.
 * Loads of B and stores of C are as wide as their alignment allows (16, 8
 * or 4 bytes).  Every output is summed in one fixed
 * order per shape: results are bitwise repeatable.  Any alignment and any
 * leading dimension are accepted.
 */
int gemm_f32(const float* A, const float* B, float* C, int64_t M, int64_t N, int64_t K,
             int64_t lda, int64_t ldb, int64_t ldc, void* stream);

/*
 * FP32-accurate path on the tensor cores: each operand is split as
 * x = big + small, where big keeps the top 11 significant bits of x
 * (truncated, which is what the tensor core reads from an fp32 operand) and
 * small = tf32(x - big) (round to nearest even), and C accumulates
 * small*big + big*small + big*big with tcgen05.mma kind::tf32 into a TMEM
 * accumulator (the small*small term is dropped).  A split pre-pass writes
 * the tf32 operands into the library's workspace (B transposed to K-major;
 * A's big part is A itself when A is 16-byte aligned with lda a multiple of
 * 4; the workspace takes 8 (M + N) K bytes in all), then a TMA + mbarrier
 * ring feeds the tensor cores.  Small problems (M N <= 2^18 and K <= 2048,
 * with A 16-byte aligned and lda a multiple of 4) skip the pre-pass: one
 * launch of the single-CTA kernel stages A by TMA and splits on chip, with
 * clusters of CTAs splitting K (no workspace).  If the workspace cannot be
 * allocated, converter warps of the CTA-pair kernel load A and B directly
 * and split them on chip instead: the same MMAs in the same order, so the
 * same C bit for bit, at about 60 % of the speed on GB300.  Any alignment and
 * leading dimension are accepted.
 */
int gemm_f32_3xtf32(const float* A, const float* B, float* C, int64_t M, int64_t N,
                    int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void* stream);

/*
 * bf16 tensor-core path: A and B hold bfloat16 bit patterns (uint16_t), C is
 * fp32; products are accumulated in fp32 in TMEM (tcgen05.mma kind::f16).
 * Fast path: A, B 16-byte aligned with lda, ldb multiples of 8 elements;
 * otherwise the operands are first packed into the workspace.  C written with
 * TMA stores when C is 16-byte aligned and ldc is a multiple of 4, else with
 * masked vector stores.
 */
int gemm_bf16_f32acc(const uint16_t* A, const uint16_t* B, float* C, int64_t M, int64_t N,
                     int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void* stream);

/*
 * The 3xTF32 GEMM without any device allocation.  The pages have no
 * counterpart: this entry point exists for callers that must not allocate
 * device memory inside a library call -- programs whose device memory is
 * owned by their own pool allocator (an outside cudaMalloc may fail or
 * fragment it), latency-critical loops (cudaMalloc and cudaFree synchronise
 * the device), and programs in which only one owner thread allocates.
 *
 * Same arguments, result and numerics as gemm_f32_3xtf32 (same kernels; the
 * small problems that gemm_f32_3xtf32 runs as one launch with the split
 * inside run the same way here).  The split operands of the pre-pass live in
 * a 64 MiB static device array inside the library instead of the allocated
 * workspace:
 *   - problems for which 8 * Kp * (M + N) bytes exceed 64 MiB, Kp = K
 *     rounded up to a multiple of 4 (e.g. larger than M = N = K = 2048), are
 *     rejected with MHR_ERR_INVALID_ARG before any work is enqueued;
 *   - every GPU on which the library is loaded holds those 64 MiB until exit;
 *   - all calls on a device share the one array.  Calls whose work overlaps
 *     on the GPU (streams with no ordering between them) race on it and give
 *     wrong results: order them on one stream or with events.  The array
 *     keeps the last call's contents; nothing in it needs to start at zero;
 *   - the first call on each device looks up the array's device address;
 *     make that first call before any stream capture begins.
 * The caller still passes (and owns) A, B and C.
 */
int gemm_f32_3xtf32_noalloc(const float* A, const float* B, float* C, int64_t M, int64_t N,
                            int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void* stream);

/*
 * The pages' optimisation ladder, kept for measuring their claims on this
 * GPU (fp32 FMA, fp32 accumulation, one output per thread):
 *   rung 0  one thread per output reading a row of A and a column of B from
 *           global memory: 2MNK element loads ("矩阵乘法 tiling", section 一;
 *           "CUDA 深入浅出（二）", section "naive kernel 怎么读数据");
 *   rung 1  16 x 16 blocks staging 16 x 16 tiles of A and B in shared memory
 *           with two barriers per K step: 2MNK/16 loads ("矩阵乘法 tiling",
 *           sections 二-四; "CUDA 编程系列之三", section 6);
 *   rung 2  the same with 32 x 32 tiles: 2MNK/32 loads.
 * Edges are zero-filled (inputs) and masked (outputs), which the pages'
 * listings omit.  Same arguments and contract as gemm_f32, plus `rung`;
 * MHR_ERR_INVALID_ARG for another rung or for M > 65535 * T.
 */
int gemm_f32_ladder(int rung, const float* A, const float* B, float* C, int64_t M, int64_t N,
                    int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void* stream);

/*
 * Reads and clears the current device's status word in stream order on
 * `stream`, then waits for `stream` alone (other streams keep running).
 * Returns MHR_OK, MHR_ERR_TIMEOUT (some kernel that finished before this
 * point hit a wait limit since the last check) or MHR_ERR_CUDA (the launch,
 * copy or synchronisation failed).
 */
int gemm_check(void* stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char* gemm_status_string(int status);

/*
 * Frees every workspace the library holds (all devices, all streams), each
 * after the last call that used it has finished.
 */
void gemm_release(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MHR_GEMM_H */
