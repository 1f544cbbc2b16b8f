// The 3xTF32 split done inside the tensor-core kernels: converter warps that
// read fp32 operand boxes, split them into tf32 big and small parts and store
// the parts into a ring stage in the layout TMA gives the pre-split operands
// (128-row x 128-byte K-major boxes, 128-byte swizzle).  Used by the CTA-pair
// kernel (tc_gemm_pair.cu) and the single-CTA kernel (tc_gemm_1cta.cu); each
// stage holds A_big, A_small, B_big^T and B_small^T boxes, in that order, for
// A rows m0 .. m0+127 and B columns nb0 .. nb0+cols-1 (cols = 128, or the
// single-CTA kernel's narrower tile width: the B boxes are then cols x 128
// bytes).
#pragma once

#include <cstdint>

#include "tc_common.cuh"
#include "tf32_split.cuh"

namespace mhr {
namespace tc {

constexpr int SPLIT_BOX_ROWS = 128;                     // rows of A, columns of B per box
constexpr int SPLIT_BOX_BYTES = SPLIT_BOX_ROWS * 32 * 4;  // x 32 k fp32 = 16 KB

// ------------------------------------------------------------------ in-kernel split
//
// KIND_3XTF32_SPLIT (CTA-pair kernel) replaces the TMA producer by SPLIT_WARPS
// converter warps per CTA.  They read the fp32 operands straight from global
// memory, split
// each value into tf32 big + small in registers, and store the four parts
// into the ring stage in exactly the layout the TMA loads of the pre-split
// operands produce: 128-row x 128-byte K-major boxes with the 128-byte swizzle,
// 16-byte chunk c of row r at r * 128 + ((c ^ (r % 8)) * 16).  Compared with
// the split pre-pass, the split operands never exist in HBM, and the kernel
// needs no workspace.
//
// The big part is stored as the fp32 value itself: the tensor core reads an
// fp32 operand of kind::tf32 as its top 19 bits, which is the truncated big
// part.  Only the small part takes arithmetic: small = tf32_rn(x - x with its
// low 13 bits cleared), three instructions per element (finite inputs; an
// infinite one gives a NaN small part).
//
// Thread ct (0..255) of the converter warps, with w = ct % 8, owns per
// K-block:
//   A (this CTA's 128 rows x 32 k): the 16-byte chunks (row ct/8 + 32j,
//     k-chunk w), j = 0..3 -- a warp reads 4 rows x 128 contiguous bytes;
//   B (32 k x this CTA's 128 columns): a 4 x 4 block, k-rows 4w .. 4w+3 of
//     columns 4nb .. 4nb+3, nb = (ct % 32) / 8 + 4 (ct / 32) -- four 16-byte
//     row pieces (a warp reads 8 k-rows x 64 contiguous bytes per load),
//     transposed in registers: column 4nb + i is the 16-byte chunk w of row
//     4nb + i of the K-major box.  The 8 lanes sharing nb write 8 different
//     chunk positions w ^ (row % 8).
// Both store patterns write 8 distinct 16-byte slots per 8 lanes: no bank
// conflicts.  When A or B is not 16-byte aligned with a leading dimension
// that is a multiple of 4, its pieces are read element by element.
//
// Latency: a thread keeps two K-blocks of loads in flight in two register
// sets used in turn, issuing a block's loads after the proxy fence of the
// block before, so that no fence has the thread's own loads outstanding to
// order.  A third stream of prefetches pulls the K-block SPLIT_PREFETCH ahead
// of the loads from HBM into L2, so that the register loads hit there.
constexpr int SPLIT_WARPS = 8;
constexpr int SPLIT_THREADS = 32 * SPLIT_WARPS;
constexpr int SPLIT_CHUNKS = 4;    // per thread, per operand, per K-block
constexpr int SPLIT_PREFETCH = 4;  // K-blocks between the L2 prefetches and the loads

struct SplitRegs {
  float4 a[SPLIT_CHUNKS];  // A chunk j
  float4 b[SPLIT_CHUNKS];  // B k-row 4w + j, columns 4nb .. 4nb+3
};

// The next K-block whose loads a converter thread issues: pointers to its A
// chunk 0 and its B row 4w at that K-block, and whether the unit's boxes lie
// inside the matrices in M and N (only K is then checked, per block).  WALK
// maps a work unit to this CTA's boxes (A rows m0.., 128 of them, B columns
// nb0.., walk.cols() of them) and K-block range: bool box(p, u, m0, nb0, kb0,
// kb1).  has_b: the thread's 4 B columns lie inside the box (all threads when
// it is 128 wide).
template <class WALK>
struct LoadCursor {
  const float* a;
  const float* b;
  int arow, bcol, u, kb, kb1;
  bool valid, interior, has_b;

  __device__ __forceinline__ void seek(const TcParams& p, const WALK& walk, int unit, int ct) {
    int m0, nb0;
    valid = walk.box(p, unit, m0, nb0, kb, kb1);
    if (!valid) return;
    u = unit;
    const int w = ct & 7, nb = ((ct & 31) >> 3) + 4 * (ct >> 5);
    arow = m0 + (ct >> 3);
    bcol = nb0 + 4 * nb;
    has_b = 4 * nb < walk.cols();
    interior = m0 + SPLIT_BOX_ROWS <= p.M && nb0 + walk.cols() <= p.N;
    a = p.A + static_cast<int64_t>(arow) * p.lda + 32 * kb + 4 * w;
    b = p.B + static_cast<int64_t>(32 * kb + 4 * w) * p.ldb + bcol;
  }
  // The first unit from `unit` on (step `stride`) with a K-block, if any.
  __device__ __forceinline__ void seek_work(const TcParams& p, const WALK& walk, int unit,
                                            int stride, int ct) {
    seek(p, walk, unit, ct);
    while (valid && kb == kb1) seek(p, walk, u + stride, ct);
  }
  __device__ __forceinline__ void advance(const TcParams& p, const WALK& walk, int stride,
                                          int ct) {
    if (!valid) return;
    if (++kb == kb1) {
      seek_work(p, walk, u + stride, stride, ct);
    } else {
      a += 32;
      b += 32 * p.ldb;
    }
  }
};

template <class WALK>
struct PrefetchCursor {
  int m0, nb0, u, kb, kb1, cols;
  bool valid;

  __device__ __forceinline__ void seek(const TcParams& p, const WALK& walk, int unit) {
    valid = walk.box(p, unit, m0, nb0, kb, kb1);
    u = unit;
    cols = walk.cols();
  }
  __device__ __forceinline__ void seek_work(const TcParams& p, const WALK& walk, int unit,
                                            int stride) {
    seek(p, walk, unit);
    while (valid && kb == kb1) seek(p, walk, u + stride);
  }
  __device__ __forceinline__ void advance(const TcParams& p, const WALK& walk, int stride) {
    if (valid && ++kb == kb1) seek_work(p, walk, u + stride, stride);
  }
};

template <bool VEC>
__device__ __forceinline__ float4 load4(const float* src) {
  if constexpr (VEC) {
    return __ldg(reinterpret_cast<const float4*>(src));
  } else {
    return make_float4(__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3));
  }
}

// The first `n` (0..3) of 4 consecutive elements, the rest zero.
__device__ __forceinline__ float4 load_partial(const float* src, int n, int64_t stride) {
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (n > 0) v.x = __ldg(src);
  if (n > 1) v.y = __ldg(src + stride);
  if (n > 2) v.z = __ldg(src + 2 * stride);
  return v;
}

// Loads of K-block c.kb into r; elements outside the matrices read as zero.
template <bool VA, bool VB, class CURSOR>
__device__ __forceinline__ void split_load(SplitRegs& r, const TcParams& p, const CURSOR& c,
                                           int ct) {
  const int64_t lda32 = 32 * p.lda;
  const int k0 = c.kb * 32;
  if (c.interior && k0 + 32 <= p.K) {  // the whole box is inside: no checks
#pragma unroll
    for (int j = 0; j < SPLIT_CHUNKS; ++j) r.a[j] = load4<VA>(c.a + j * lda32);
#pragma unroll
    for (int j = 0; j < SPLIT_CHUNKS; ++j) r.b[j] = load4<VB>(c.b + j * p.ldb);
    return;
  }
  const int ka = k0 + 4 * (ct & 7);  // first k of the thread's A chunks and B rows
#pragma unroll
  for (int j = 0; j < SPLIT_CHUNKS; ++j) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c.arow + 32 * j < p.M) {
      const float* src = c.a + j * lda32;
      if (ka + 4 <= p.K)
        v = load4<VA>(src);
      else if (ka < p.K)
        v = load_partial(src, p.K - ka, 1);
    }
    r.a[j] = v;
  }
#pragma unroll
  for (int j = 0; j < SPLIT_CHUNKS; ++j) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ka + j < p.K) {
      const float* src = c.b + j * p.ldb;
      if (c.bcol + 4 <= p.N)
        v = load4<VB>(src);
      else if (c.bcol < p.N)
        v = load_partial(src, p.N - c.bcol, 1);
    }
    r.b[j] = v;
  }
}

// Pull one future K-block of this CTA's boxes into L2: each of the first 128
// converter threads takes one row of the A box (128 bytes), each of the others
// one 128-byte quarter of a row of the B box (32 rows x up to 512 bytes).
// Both ends of each piece are touched, in case it straddles two lines.
// Addresses outside the matrices (or the box) are skipped.
__device__ __forceinline__ void prefetch_l2(const float* a) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

template <class CURSOR>
__device__ __forceinline__ void split_prefetch_l2(const TcParams& p, int ct, const CURSOR& c) {
  if (!c.valid) return;
  const int k0 = c.kb * 32;
  if (ct < 128) {
    const int row = c.m0 + ct;
    if (row >= p.M || k0 >= p.K) return;
    const float* a = p.A + static_cast<int64_t>(row) * p.lda + k0;
    prefetch_l2(a);
    prefetch_l2(a + (min(k0 + 31, p.K - 1) - k0));
  } else {
    const int q = ct - 128, k = k0 + (q >> 2), col = c.nb0 + 32 * (q & 3);
    if (k >= p.K || col >= p.N || 32 * (q & 3) >= c.cols) return;
    const float* b = p.B + static_cast<int64_t>(k) * p.ldb + col;
    prefetch_l2(b);
    prefetch_l2(b + (min(col + 31, p.N - 1) - col));
  }
}

// A converter thread's fixed store offsets within a stage's boxes: its A
// chunk 0 (chunk j is 4 KB further: 32 rows) and its four B columns' chunks.
struct StoreOffsets {
  uint32_t a;
  uint32_t b[4];
  __device__ __forceinline__ explicit StoreOffsets(int ct) {
    const int w = ct & 7, row = ct >> 3;
    a = row * 128 + ((w ^ (row & 7)) << 4);
    const int nb = ((ct & 31) >> 3) + 4 * (ct >> 5);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = 4 * nb + i;
      b[i] = n * 128 + ((w ^ (n & 7)) << 4);
    }
  }
};

// Split the registers of one K-block into ring stage `st`: A_big, A_small,
// B_big^T, B_small^T boxes of 16 KB each, in that order; the big parts are the
// values themselves (see above).
__device__ __forceinline__ void split_store(const SplitRegs& r, uint32_t st,
                                            const StoreOffsets& o) {
#pragma unroll
  for (int j = 0; j < SPLIT_CHUNKS; ++j) {
    const uint32_t off = o.a + j * 4096;
    st_shared_v4(st + off, r.a[j]);
    st_shared_v4(st + SPLIT_BOX_BYTES + off, small4_tf32_trunc(r.a[j]));
  }
  const float4 col[4] = {make_float4(r.b[0].x, r.b[1].x, r.b[2].x, r.b[3].x),
                         make_float4(r.b[0].y, r.b[1].y, r.b[2].y, r.b[3].y),
                         make_float4(r.b[0].z, r.b[1].z, r.b[2].z, r.b[3].z),
                         make_float4(r.b[0].w, r.b[1].w, r.b[2].w, r.b[3].w)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    st_shared_v4(st + 2 * SPLIT_BOX_BYTES + o.b[i], col[i]);
    st_shared_v4(st + 2 * SPLIT_BOX_BYTES + SPLIT_BOX_BYTES + o.b[i], small4_tf32_trunc(col[i]));
  }
}

// ------------------------------------------------- in-kernel split, A staged by TMA
//
// KIND_3XTF32_SPLIT_TMA_A (both kernels): when A is 16-byte aligned with lda a
// multiple of 4, each CTA's producer warp TMA-loads A's box (128 rows x 32 k)
// into the stage's A_big box, completing on a barrier of its own CTA; the
// tensor core reads it there as A's truncated big part.  The converter warps read
// their A chunks back from that box (the positions they would have stored
// to), write A_small, and take B through registers as in KIND_3XTF32_SPLIT.
//
// Two groups of SPLIT_WARPS converter warps take the K-blocks in turn (even
// and odd).  A thread issues the B loads of its group's next K-block right
// after handing over the current one, so they have two K-block times to land,
// and it never has loads outstanding when it executes its proxy fence: on
// GB300 that fence also waits for the thread's outstanding global loads,
// which made one group with several register sets no faster than one load
// round trip per K-block (1.7 us against 0.8 us of MMAs, measured).
// Shared memory carries per stage TMA's 16 KB of A, the converters' 16 KB of
// A reads and 48 KB of stores, and the MMAs' 96 KB of operand reads.
struct BRegs {
  float4 b[SPLIT_CHUNKS];  // B k-row 4w + j, columns 4nb .. 4nb+3
};

template <bool VB, class CURSOR>
__device__ __forceinline__ void load_b(BRegs& r, const TcParams& p, const CURSOR& c, int ct) {
  if (!c.has_b) return;  // columns beyond a narrow box: nothing to load or store
  const int k0 = c.kb * 32;
  if (c.bcol + 4 <= p.N && k0 + 32 <= p.K) {
#pragma unroll
    for (int j = 0; j < SPLIT_CHUNKS; ++j) r.b[j] = load4<VB>(c.b + j * p.ldb);
    return;
  }
  const int kb_row = k0 + 4 * (ct & 7);
#pragma unroll
  for (int j = 0; j < SPLIT_CHUNKS; ++j) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (kb_row + j < p.K) {
      const float* src = c.b + j * p.ldb;
      if (c.bcol + 4 <= p.N)
        v = load4<VB>(src);
      else if (c.bcol < p.N)
        v = load_partial(src, p.N - c.bcol, 1);
    }
    r.b[j] = v;
  }
}

// A_small from the staged A box, and B_big^T, B_small^T from registers (the
// B_small^T box b_small_off bytes after B_big^T's: cols x 128; has_b as in
// LoadCursor).
__device__ __forceinline__ void split_store_tma_a(const BRegs& r, uint32_t st,
                                                  const StoreOffsets& o, uint32_t b_small_off,
                                                  bool has_b) {
#pragma unroll
  for (int j = 0; j < SPLIT_CHUNKS; ++j) {
    const uint32_t off = o.a + j * 4096;
    st_shared_v4(st + SPLIT_BOX_BYTES + off, small4_tf32_trunc(ld_shared_v4(st + off)));
  }
  if (!has_b) return;
  const float4 col[4] = {make_float4(r.b[0].x, r.b[1].x, r.b[2].x, r.b[3].x),
                         make_float4(r.b[0].y, r.b[1].y, r.b[2].y, r.b[3].y),
                         make_float4(r.b[0].z, r.b[1].z, r.b[2].z, r.b[3].z),
                         make_float4(r.b[0].w, r.b[1].w, r.b[2].w, r.b[3].w)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    st_shared_v4(st + 2 * SPLIT_BOX_BYTES + o.b[i], col[i]);
    st_shared_v4(st + 2 * SPLIT_BOX_BYTES + b_small_off + o.b[i], small4_tf32_trunc(col[i]));
  }
}

}  // namespace tc
}  // namespace mhr
