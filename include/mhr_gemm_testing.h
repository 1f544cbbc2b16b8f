/*
 * mhr_gemm_testing.h -- test hooks of libmhr_gemm.so.  Not for production use.
 *
 * The pages have no counterpart: these hooks exist so the failure path of the
 * tensor-core kernels (a bounded wait that runs out) can be exercised without
 * faulting, trapping or hanging a GPU.
 */
#ifndef MHR_GEMM_TESTING_H
#define MHR_GEMM_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Sets the limit, in nanoseconds, of every bounded wait inside the
 * tensor-core kernels launched afterwards (process-wide; default 2 s).
 * Values below 1 ms are raised to 1 ms.  Returns the previous limit.
 */
uint64_t gemm_testing_set_wait_limit_ns(uint64_t limit_ns);

/*
 * When `enable` is nonzero, the next tensor-core launches run with an
 * injected stall: block 0 leaves its first ring stage incomplete (the TMA
 * producer arms it for a load it never issues; the on-chip split's converter
 * warps fill it without arriving), so that stage never fills.  Its consumers'
 * waits then run out, the kernel records MHR_ERR_TIMEOUT in the device status
 * word, frees its TMEM and exits; gemm_check() reports the timeout.  No GPU
 * fault occurs and the CUDA context stays usable.  Returns the previous
 * setting.
 */
int gemm_testing_set_inject_stall(int enable);

/*
 * Synchronises `stream` and returns the raw bits of the current device's
 * status word without clearing it (1: producer timeout, 2: MMA-issuer
 * timeout, 4: epilogue timeout, 8: drain timeout).  Negative on a CUDA error.
 */
int64_t gemm_testing_peek_status(void* stream);

/*
 * Chooses the tensor-core kernel variant of the following calls
 * (process-wide): 0 = automatic (the CTA-pair kernel when its 256 x 256
 * tiles fill half of its clusters -- for bf16 only with K >= 1536 or at
 * least two tiles per cluster -- or, for 3xTF32, when tiles of 256, 192 or
 * 128 columns -- split into two K halves each where twice the tiles fit --
 * keep at least 80 % of them busy, else the single-CTA kernel), 1 = always the single-CTA
 * kernel, 2 = always the CTA-pair kernel.  Other values mean 0.  Returns the
 * previous mode.
 */
int gemm_testing_set_cta_pair_mode(int mode);

/*
 * Chooses where gemm_f32_3xtf32 splits its operands into tf32 big and small
 * parts (process-wide): 0 = automatic (the single-CTA kernel's one-launch
 * form for small problems -- M N <= 2^18, K <= 2048, A 16-byte aligned with
 * lda a multiple of 4, unless the CTA-pair mode is 2 --, else a pre-pass
 * into the workspace, or inside the CTA-pair kernel when the workspace
 * cannot be allocated), 1 = always a pre-pass, 2 = always inside a kernel:
 * the single-CTA kernel's one-launch form when the CTA-pair mode is 1 and A
 * is aligned as above, else the CTA-pair kernel's (used whatever the
 * CTA-pair mode says).  Other values mean 0.  Pre-pass and in-kernel split
 * give bit-identical results for the same kernel and tile schedule.
 * Returns the previous mode.
 */
int gemm_testing_set_split_mode(int mode);

/*
 * When `enable` is nonzero, gemm_f32_3xtf32 calls that split in a pre-pass
 * (split mode 1, or 0 where it takes the pre-pass) clear A's small part after the split,
 * so the main kernel accumulates A_big * (B_big + B_small) only.  With B the
 * identity that exposes what the tensor core reads from an fp32 A operand
 * under kind::tf32 -- the library relies on it being A with the low 13 bits
 * of each value cleared, so that A itself can serve as A's big part.  Test
 * use only; returns the previous setting.
 */
int gemm_testing_set_zero_a_small(int enable);

/*
 * Caps the bytes the library's workspace may grow to (process-wide), so that
 * a larger request fails as an allocation failure would.  UINT64_MAX (the
 * initial value) removes the cap.  Returns the previous cap.
 */
uint64_t gemm_testing_set_workspace_limit(uint64_t bytes);

/*
 * Tuning hook: the number of tile rows per raster group of the tensor-core
 * kernels' tile schedule (consecutive work units sweep that many tile rows
 * column by column, so co-resident CTAs share A and B panels in L2).  0
 * restores the default (8).  Returns the previous setting.
 */
int gemm_testing_set_raster_group(int tile_rows);

/*
 * Number of kernels the most recent gemm_* call launched: its pre-passes
 * (split, repack, zero fills) and its main kernel.  Meaningful when calls do
 * not overlap in time from several host threads.
 */
int gemm_testing_last_launches(void);

/*
 * Name, grid size and tile count of the main kernel that the most recent
 * gemm_* call launched, e.g. "tc_gemm_pair_kernel<3xtf32> grid=148
 * tiles=256" ("none" before the first launch).  Static storage, overwritten
 * by the next call.
 */
const char* gemm_testing_last_main_kernel(void);

/*
 * Profiling hook.  When `start` and `stop` are both non-NULL cudaEvent_t
 * handles, every following gemm_* call records `start` on its stream just
 * before it launches its main GEMM kernel (after any split or pack pre-pass
 * and any kernel zeroing C for a K-split schedule) and `stop` just after, so
 * the caller can time that kernel alone with
 * cudaEventElapsedTime.  Passing NULL for either turns the hook off.  The
 * events stay owned by the caller.
 */
void gemm_testing_set_main_kernel_events(void* start, void* stop);

/*
 * Forces the width of the CTA-pair kernel's 3xTF32 output tiles (256 rows x
 * `columns`) for the following calls (process-wide): a multiple of 16 in
 * [128, 256]; any other value, 0 included, restores the planner's choice.  A
 * width that is not a multiple of 32 writes C with register stores even where
 * C could take TMA stores.  The single-CTA kernel and the bf16 path ignore
 * it.  Returns the previous setting.
 */
int gemm_testing_set_pair_tile_n(int columns);

/*
 * The planner's choice of those tile columns for an M x N x K 3xTF32 problem
 * on `clusters` co-resident CTA pairs, with C written by TMA stores when
 * c_tma is nonzero (a multiple of 32 then) or by register stores.  Host
 * arithmetic only: it needs no GPU.  It weighs the tile-size trade-off of
 * "矩阵乘法 tiling", section 五 (a wider tile reuses each staged B element over
 * more columns; fewer, wider tiles fill the SMs in fewer, coarser rounds):
 * rounds of tiles over the clusters against the shared-memory bytes per
 * tensor cycle that narrower tiles need.
 */
int gemm_testing_plan_pair_tile_n(int64_t M, int64_t N, int64_t K, int clusters, int c_tma);

/*
 * Forces the width of the single-CTA kernel's output tiles (128 rows x
 * `columns`) for the following calls (process-wide): 3xTF32 takes 128, 96, 64
 * or 32, bf16 256 or 128; a width the kind lacks leaves that kind's automatic
 * choice, and any other value, 0 included, restores the automatic choice for
 * both.  3xTF32 calls with a pre-pass that take the cluster split plan 128
 * and take any forced width; the one-launch form (split inside) takes 128, 64 or 32 and splits K over
 * clusters at any of them; bf16 takes the cluster split at either width.
 * Automatically, bf16 takes 128 columns when those tiles, split as the kernel
 * splits them (a cluster per tile, or two K halves), put more CTAs to work in
 * a single round of tiles.  Returns the previous setting.
 */
int gemm_testing_set_single_tile_n(int columns);

/*
 * The planner's choice of those columns for an M x N x K 3xTF32 problem on
 * `sms` SMs, C written by TMA stores when c_tma is nonzero.  Host arithmetic
 * only, as for gemm_testing_plan_pair_tile_n: smaller tiles spread a small
 * problem over more SMs ("矩阵乘法 tiling", section 五, on the tile size).
 */
int gemm_testing_plan_single_tile_n(int64_t M, int64_t N, int64_t K, int sms, int c_tma);

/*
 * Chooses between gemm_f32's two SIMT kernels for the following calls
 * (process-wide), where A, B and C are 16-byte aligned with leading
 * dimensions multiples of 4 and M, N, K multiples of 128, 256 and 8:
 * 0 = automatic (gemm_testing_plan_simt_wide), 1 = always the 128 x 128
 * kernel, 2 = always the 128 x 256 kernel (on two K halves when that
 * shortens its queue of blocks).  Other values mean 0.  Other problems take
 * the 128 x 128 kernel whatever the mode.  Returns the previous mode.
 */
int gemm_testing_set_simt_wide_mode(int mode);

/*
 * The automatic choice for such a problem on `sms` SMs: 0 = the 128 x 128
 * kernel, 1 = the 128 x 256 kernel, 2 = the 128 x 256 kernel on two K halves
 * added into a zeroed C; 0 too for sizes that are not multiples of
 * 128 x 256 x 8.  Host arithmetic only.  The estimate: a kernel's time
 * follows the deepest queue of blocks on one SM, and a 128 x 256 block takes
 * 11/6 of a 128 x 128 block's time (register tiling, "矩阵乘法 tiling",
 * section 五: the wider block reuses each A value twice as often).
 */
int gemm_testing_plan_simt_wide(int64_t M, int64_t N, int64_t K, int sms);

#ifdef __cplusplus
}
#endif

#endif /* MHR_GEMM_TESTING_H */
