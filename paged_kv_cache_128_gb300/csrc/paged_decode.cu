// Single-query (decode) paged attention with GQA, split-K and LSE merge.
//
// What is computed ("MiniPaged-Qwen: Paged KV Cache 与 KV Block Manager"
// §13 decode attention through block tables, §14 GQA head mapping, §16.6
// seq_lens boundary, §17.3 online softmax):
//   out[b, qh] = sum_{j < L_b} softmax_j(scale * q[b, qh] . K_j) V_j,
//   kvh = qh / (Hq / Hkv),  K_j = k_cache[table[b][j / bs]][j % bs][kvh].
//
// Kernels (the host plan picks one per call):
//  * decode_sk_kernel, the default for fp16/bf16 caches at head_dim
//    64/128/256 and fp8 (E4M3) caches at head_dim 128, block_size 16/32,
//    G = Hq / Hkv <= 16: stream-K
//    over the ordered tiles (sequence, kv head, 32 or 64 tokens) in one
//    cooperative wave of persistent CTAs, each CTA a TMA producer warp, four
//    mma.sync consumer warps and a writer warp; units cut by range
//    boundaries are combined by their owner CTA (see "Stream-K tensor-core
//    kernel" below).  It also runs the fused decode step: its writer warps
//    scatter the step's new K/V rows into the caches.
//  * decode_split_kernel, the same shapes where the stream-K shared memory
//    does not fit or a split size is forced: one CTA per (split, kv head,
//    sequence) over blocks_per_split blocks, serving all G query heads of
//    its kv head so each K/V byte is read once.  Its producer warp walks the
//    block table (entries fetched 32 at a time and shuffled) and issues TMA
//    loads of each block's K and V slices into a ring of shared-memory
//    stages; four consumer warps compute S^T = K Q^T (tokens in M, query
//    heads in N, m16n8k16 mma.sync, fp32 accumulation), an fp32 online
//    softmax in the exp2 domain, and O^T += V^T P^T (P^T turned into the B
//    operand with movmatrix, V^T from ldmatrix.trans).
//  * decode_simt_kernel, any dtype, head_dim a multiple of 4 up to 256, any
//    block size and group: one warp per block, lane-parallel dot products
//    reduced with shuffles, the same online softmax.
// Split partials (acc, m, l) of the split and SIMT kernels are combined by
// lse_merge_kernel (log-sum-exp, flash-decoding style split-K).
//
// Tail handling: only ceil(L / bs) table entries are read.  Positions >= L
// in the last block are excluded by selection (score = -inf), and their V
// rows are zeroed in shared memory before the PV product, so whatever those
// slots hold (stale data, NaN) never reaches the output.

#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <atomic>
#include <chrono>
#include <mutex>
#include <random>
#include <type_traits>

#include "common.cuh"

namespace pagedkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  int32_t num_seqs, num_heads, num_kv_heads, group, head_dim, block_size;
  int64_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t blocks_per_split, num_splits;
  float scale_log2;  // scale * log2(e): scores live in the exp2 domain
  int32_t num_ctas;  // stream-K grid size P
  float* ws_o;       // split: [B][Hq][S][D]; stream-K: [P][2][G][D] unnormalised partial outputs
  float* ws_ml;      // split: [B][Hq][S][2]; stream-K: [P][2][G][2] (running max, running sum)
  uint64_t* ws_flags;  // stream-K: [P] "partial in slot 0 ready" flags, holding the call's epoch
  uint64_t epoch;      // stream-K: tag unique to this call (flags from other calls never match)
  int32_t seg_cost;    // stream-K: extra tiles charged per unit when ranges are drawn
  uint64_t wait_limit_ns;   // stream-K: longest one bounded wait may take
  int32_t test_skip_tile;   // stream-K test control (-1: off): CTA 0 never loads this tile of its range
  // Fused step (stream-K only; new_k == nullptr otherwise): the step's new
  // tokens' rows [num_new][Hkv][D] are scattered into the caches by
  // slot_mapping, and sequence b's newest position seq_lens[b] - 1 is taken
  // from row new_row[b] of new_k / new_v (-1: none) instead of the cache.
  const void* new_k;
  const void* new_v;
  const int32_t* slot_mapping;
  const int32_t* new_row;
  int64_t num_new;
  int64_t new_k_stride, new_v_stride;  // bytes between consecutive tokens' rows
  // fp8 caches: float32 scales [num_blocks][num_kv_heads][block_size]
  const float* k_scales;
  const float* v_scales;
};

// Sequence length after bounds checks: at most what the table row and the
// split partition cover.  A violation is recorded and the length clamped.
__device__ __forceinline__ int checked_len(const DecodeParams& p, int b) {
  int L = __ldg(p.seq_lens + b);
  const int64_t cap = min(static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size,
                          static_cast<int64_t>(p.num_splits) * p.blocks_per_split * p.block_size);
  if (L < 0 || L > cap) {
    record_error(KV_ERR_DEVICE_BOUNDS);
    L = L < 0 ? 0 : static_cast<int>(cap);
  }
  return L;
}

// Combine per-warp states (m, l, acc) held in shared memory and write either
// the final output (single split for this sequence) or this split's partial.
// Ms/Ls: [nw][gstride], Os: [nw][gstride][dstride].  Threads tid..nthreads.
template <typename T>
__device__ __forceinline__ void combine_and_store(const DecodeParams& p, const float* Ms, const float* Ls,
                                                  const float* Os, int nw, int gstride, int dstride, int D, int b,
                                                  int qh0, int gn, int split, bool single, int tid, int nthreads) {
  for (int idx = tid; idx < gn * D; idx += nthreads) {
    const int g = idx / D, d = idx - g * D;
    float mx = -INFINITY;
    for (int w = 0; w < nw; ++w) mx = fmaxf(mx, Ms[w * gstride + g]);
    float num = 0.f, den = 0.f;
    if (mx != -INFINITY) {
      for (int w = 0; w < nw; ++w) {
        const float mw = Ms[w * gstride + g];
        if (mw == -INFINITY) continue;
        const float sc = fast_exp2(mw - mx);
        num += sc * Os[(w * gstride + g) * dstride + d];
        den += sc * Ls[w * gstride + g];
      }
    }
    const int qh = qh0 + g;
    if (single) {
      T* o = static_cast<T*>(p.out) + (static_cast<int64_t>(b) * p.num_heads + qh) * D + d;
      *o = DType<T>::from_float(den > 0.f ? num / den : 0.f);
    } else {
      const int64_t row = (static_cast<int64_t>(b) * p.num_heads + qh) * p.num_splits + split;
      p.ws_o[row * D + d] = num;
      if (d == 0) {
        p.ws_ml[row * 2 + 0] = mx;
        p.ws_ml[row * 2 + 1] = den;
      }
    }
  }
}

template <typename T>
__device__ __forceinline__ void store_zero_rows(const DecodeParams& p, int b, int qh0, int gn, int D, int tid,
                                                int nthreads) {
  T* o = static_cast<T*>(p.out) + (static_cast<int64_t>(b) * p.num_heads + qh0) * D;
  for (int idx = tid; idx < gn * D; idx += nthreads) o[idx] = DType<T>::from_float(0.f);
}

// =========================================================================
// Tensor-core path: shared consumer math.
//
// Each consumer warp owns whole tiles (one physical block of one kv head,
// BS tokens) and keeps its own online-softmax state for the current unit
// (sequence, kv head).  Per 16-token sub-tile:
//   S^T[16 tok x 8*NG heads] = K[16 x D] Q^T          (mma m16n8k16, fp32 acc)
//   softmax update in the exp2 domain, P^T packed to the MMA type,
//   movmatrix turns the P^T accumulator fragment into a B operand,
//   O^T[D x 8*NG] += V^T[D x 16] P^T                   (V^T via ldmatrix.trans)
// =========================================================================

template <int D, int BS>
struct Tile {
  static constexpr int kSub = D / 64;              // 128-byte column slabs per row
  static constexpr int kSlabBytes = BS * 128;      // one slab of one tile
  static constexpr int kTileBytes = BS * D * 2;    // K or V of one block, one kv head
  static constexpr int kStageBytes = 2 * kTileBytes;
  static_assert(D % 64 == 0, "head_dim must be a multiple of 64");
  static_assert(BS % 16 == 0, "block_size must be a multiple of 16");
  static_assert(kSlabBytes % 1024 == 0, "slabs must keep 1024-byte swizzle alignment");
};

// Byte offset of element (row t, column d) inside a tile written by TMA with
// 128-byte swizzle.  The tile holds whole physical blocks of PB rows, block
// by block; inside a block, 64-column slab by slab (PB rows of 128 bytes
// each); inside a row, 16-byte chunk (d%64)/8 XOR (t%8) (PB is a multiple of
// 8, so a row's swizzle phase is t % 8 wherever its block sits).
template <int D, int PB>
__device__ __forceinline__ uint32_t swz(int t, int d) {
  return static_cast<uint32_t>(((t / PB) * (D / 64) + (d >> 6)) * (PB * 128) + (t % PB) * 128 +
                               ((((d & 63) >> 3) ^ (t & 7)) << 4));
}

template <int D, int NG>
struct WarpState {
  static constexpr int KS = D / 16;  // k-steps of S^T = K Q^T, and m-tiles of O^T
  uint32_t qf[KS][NG][2];            // Q^T as B operand
  float acc[KS][NG][4];              // O^T accumulator fragments
  float m[NG][2], l[NG][2];          // running max (exp2 domain) and sum, 2 heads per lane
};

// B operand of S^T = K Q^T: b0 = Q[g][kk*16 + 2*(lane%4) + {0,1}], b1 at d + 8,
// g = ng*8 + lane/4; heads past G are zero.
template <typename T, int D, int NG>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[D / 16][NG][2], const T* qb, int G, int lane) {
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
    const int g = ng * 8 + (lane >> 2);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int d = kk * 16 + (lane & 3) * 2;
      if (g < G) {
        qf[kk][ng][0] = __ldg(reinterpret_cast<const uint32_t*>(qb + g * D + d));
        qf[kk][ng][1] = __ldg(reinterpret_cast<const uint32_t*>(qb + g * D + d + 8));
      } else {
        qf[kk][ng][0] = 0u;
        qf[kk][ng][1] = 0u;
      }
    }
  }
}

template <typename T, int D, int NG>
__device__ __forceinline__ void load_q(WarpState<D, NG>& st, const T* qb, int G, int lane) {
  load_q_frags<T, D, NG>(st.qf, qb, G, lane);
}

template <int D, int NG>
__device__ __forceinline__ void reset_state(WarpState<D, NG>& st) {
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.acc[mt][ng][e] = 0.f;
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
    st.m[ng][0] = st.m[ng][1] = -INFINITY;
    st.l[ng][0] = st.l[ng][1] = 0.f;
  }
}

// Accumulate NS 16-token sub-tiles (tokens tok0 .. tok0 + 16 * NS - 1) of
// one tile held in shared memory at kt_a (K) and vt_a (V) as one step of the
// online softmax: the score chains of the sub-tiles are interleaved, and
// the running max, the rescale of the accumulator and l are updated once.
template <typename T, int D, int PB, int NG, int NS>
__device__ __forceinline__ void consume_subtiles(WarpState<D, NG>& st, uint32_t kt_a, uint32_t vt_a, int tok0, int L,
                                                 float sl2, int lane) {
  using M = Mma<T>;
  constexpr int KS = D / 16;
  // ldmatrix lane -> (row, column) of the 8x8 matrix it addresses
  const int k_row = (lane & 7) + ((lane >> 3) & 1) * 8, k_col = (lane >> 4) * 8;  // A = K (non-trans)
  const int v_row = (lane & 7) + (lane >> 4) * 8, v_col = ((lane >> 3) & 1) * 8;  // A = V^T (trans)
  float sc[NS][NG][4];
#pragma unroll
  for (int u = 0; u < NS; ++u)
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) sc[u][ng][0] = sc[u][ng][1] = sc[u][ng][2] = sc[u][ng][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    uint32_t a[NS][4];
#pragma unroll
    for (int u = 0; u < NS; ++u)
      ldmatrix_x4(kt_a + swz<D, PB>(u * 16 + k_row, kk * 16 + k_col), a[u][0], a[u][1], a[u][2], a[u][3]);
#pragma unroll
    for (int u = 0; u < NS; ++u)
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) M::run(sc[u][ng], a[u], st.qf[kk][ng][0], st.qf[kk][ng][1]);
  }
  uint32_t pb[NS][NG][2];
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
    // scores in the exp2 domain; rows past the sequence end are -inf
    float x[NS][4];
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int u = 0; u < NS; ++u) {
      const int t_lo = tok0 + u * 16 + (lane >> 2);
      const bool in_lo = t_lo < L, in_hi = t_lo + 8 < L;
      x[u][0] = in_lo ? sc[u][ng][0] * sl2 : -INFINITY;
      x[u][1] = in_lo ? sc[u][ng][1] * sl2 : -INFINITY;
      x[u][2] = in_hi ? sc[u][ng][2] * sl2 : -INFINITY;
      x[u][3] = in_hi ? sc[u][ng][3] * sl2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(x[u][0], x[u][2]));
      mx1 = fmaxf(mx1, fmaxf(x[u][1], x[u][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(st.m[ng][0], mx0), mn1 = fmaxf(st.m[ng][1], mx1);
    const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0, mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
    const float al0 = fast_exp2(st.m[ng][0] - mu0), al1 = fast_exp2(st.m[ng][1] - mu1);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int u = 0; u < NS; ++u) {
      // l sums the probabilities as rounded for the PV product
      const uint32_t lo = M::pack(fast_exp2(x[u][0] - mu0), fast_exp2(x[u][1] - mu1));
      const uint32_t hi = M::pack(fast_exp2(x[u][2] - mu0), fast_exp2(x[u][3] - mu1));
      const float2 flo = M::unpack(lo), fhi = M::unpack(hi);
      s0 += flo.x + fhi.x;
      s1 += flo.y + fhi.y;
      pb[u][ng][0] = movmatrix_trans(lo);
      pb[u][ng][1] = movmatrix_trans(hi);
    }
    st.l[ng][0] = st.l[ng][0] * al0 + s0;
    st.l[ng][1] = st.l[ng][1] * al1 + s1;
    st.m[ng][0] = mn0;
    st.m[ng][1] = mn1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      st.acc[mt][ng][0] *= al0;
      st.acc[mt][ng][1] *= al1;
      st.acc[mt][ng][2] *= al0;
      st.acc[mt][ng][3] *= al1;
    }
  }
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    uint32_t a[NS][4];
#pragma unroll
    for (int u = 0; u < NS; ++u)
      ldmatrix_x4_trans(vt_a + swz<D, PB>(u * 16 + v_row, mt * 16 + v_col), a[u][0], a[u][1], a[u][2], a[u][3]);
#pragma unroll
    for (int u = 0; u < NS; ++u)
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) M::run(st.acc[mt][ng], a[u], pb[u][ng][0], pb[u][ng][1]);
  }
}

// Accumulate one tile (tokens tok0 .. tok0 + BS - 1 of a sequence of length
// L) held in shared memory at kt (K) and vt (V).  Sub-tiles wholly past the
// sequence end are skipped.
// BS: tokens of the tile; PB: rows of each physical block in it (the tile's
// layout, see swz).
template <typename T, int D, int BS, int NG, int PB = BS>
__device__ __forceinline__ void consume_tile(WarpState<D, NG>& st, uint8_t* kt, uint8_t* vt, int tok0, int L,
                                             float sl2, int lane) {
  const int valid = min(BS, L - tok0);
  if (valid < BS) {
    // zero the V rows past the sequence end: P is 0 there, but 0 * NaN is not
    const int chunks = (BS - valid) * (D / 8);
    for (int c = lane; c < chunks; c += 32) {
      const int t = valid + c / (D / 8), d = (c % (D / 8)) * 8;
      *reinterpret_cast<uint4*>(vt + swz<D, PB>(t, d)) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();  // these bytes are TMA-written again later
    __syncwarp();
  }
  const uint32_t kt_a = smem_u32(kt), vt_a = smem_u32(vt);
  if constexpr (BS == 32) {
    if (valid > 16) consume_subtiles<T, D, PB, NG, 2>(st, kt_a, vt_a, tok0, L, sl2, lane);
    else consume_subtiles<T, D, PB, NG, 1>(st, kt_a, vt_a, tok0, L, sl2, lane);
  } else {
    static_assert(BS == 16, "tiles are 16 or 32 tokens");
    consume_subtiles<T, D, PB, NG, 1>(st, kt_a, vt_a, tok0, L, sl2, lane);
  }
}

// Row stride of a head's accumulator in the warp-merge buffer: padded by 4
// floats so that both the fragment stores below and float4 reads of
// consecutive d are free of bank conflicts.
template <int D>
__host__ __device__ constexpr int merge_row() { return D + 4; }

// Reduce l across the lanes that share a head, then store this warp's
// state: Os[cw][g][DP], Ms[cw][GP], Ls[cw][GP] (GP = 8 * NG, DP = D + 4).
template <int D, int NG>
__device__ __forceinline__ void store_state(WarpState<D, NG>& st, float* Os, float* Ms, float* Ls, int cw,
                                            int lane) {
  constexpr int GP = 8 * NG;
#pragma unroll
  for (int ng = 0; ng < NG; ++ng)
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) st.l[ng][c] += __shfl_xor_sync(0xffffffffu, st.l[ng][c], off);
  constexpr int DP = merge_row<D>();
  float* o = Os + cw * GP * DP;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      const int d0 = mt * 16 + (lane >> 2), g0 = ng * 8 + (lane & 3) * 2;
      o[g0 * DP + d0] = st.acc[mt][ng][0];
      o[(g0 + 1) * DP + d0] = st.acc[mt][ng][1];
      o[g0 * DP + d0 + 8] = st.acc[mt][ng][2];
      o[(g0 + 1) * DP + d0 + 8] = st.acc[mt][ng][3];
    }
  if (lane < 4) {
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        Ms[cw * GP + ng * 8 + lane * 2 + c] = st.m[ng][c];
        Ls[cw * GP + ng * 8 + lane * 2 + c] = st.l[ng][c];
      }
  }
}

// =========================================================================
// fp8 (E4M3) cache tiles ("paged-attention-impl-detail", 实践建议 4: the KV
// cache inside a block quantised on its own).  A tile holds TT tokens of
// one kv head: TMA writes each 128-byte row (128 dims) with the 128-byte
// swizzle, and the tokens' float32 scales (one per token for K, one for V)
// sit in a small separate array.  The consumer builds the mma operands from
// byte loads: E4M3 pairs convert exactly to f16 (cvt.rn.f16x2.e4m3x2), and
// from there exactly to bf16.  A token's K scale multiplies its scores; its
// V scale multiplies its softmax weights before the PV product (the softmax
// sum uses the unscaled weights).
// =========================================================================

template <int D, int TT>
struct Tile8 {
  static constexpr int kSub = D / 128;          // 128-byte column slabs per row
  static constexpr int kSlabBytes = TT * 128;
  static constexpr int kTileBytes = TT * D;     // K or V codes of one tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static_assert(D % 128 == 0, "fp8 tiles need head_dim a multiple of 128");
  static_assert(kSlabBytes % 1024 == 0, "slabs must keep 1024-byte swizzle alignment");
};

template <int TT>
__device__ __forceinline__ uint32_t swz8(int t, int d) {
  return static_cast<uint32_t>((d >> 7) * (TT * 128) + t * 128 + ((((d & 127) >> 4) ^ (t & 7)) << 4) + (d & 15));
}

// Two E4M3 codes (low byte first) -> f16x2, exactly.
__device__ __forceinline__ uint32_t e4m3x2_f16(uint32_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(two & 0xffffu)));
  return h;
}

// The fp8 path multiplies in f16 whatever the q/out type: E4M3 -> f16 is
// exact, and so is bf16 -> f16 for |q| in f16's normal range.
//
// Operands come from the byte tiles through ldmatrix, which moves 16-bit
// elements: to it a 128-byte row of 128 codes is 64 "elements" of two
// codes.  For S^T = K Q^T, ldmatrix (no transpose) gives a lane 4
// consecutive codes of one token, dims 4t..4t+3 of a 16-dim k-step; the
// k-step takes them as its columns 2t, 2t+1 (dims 4t, 4t+1) and 2t+8,
// 2t+9 (dims 4t+2, 4t+3), and the Q^T fragments are loaded in the same dim
// order, so the contraction is unchanged.  For O^T += V^T P^T, ldmatrix
// with transpose gives a lane codes (token 2t, dims 2g, 2g+1) and (token
// 2t+1, dims 2g, 2g+1); one byte permute pairs them by dim, which makes
// dim 2g row g and dim 2g+1 row g + 8 of the m-tile.  The accumulator's
// rows are then permuted within each 16-dim group, and store_state_f8
// writes them back to their dims.

// Q^T fragments in the fp8 k-step dim order, converted to f16: b0 = Q[g][4t,
// 4t+1], b1 = Q[g][4t+2, 4t+3] of each k-step, g = ng*8 + lane/4.
template <typename T, int D, int NG>
__device__ __forceinline__ void load_q_frags_f8(uint32_t (&qf)[D / 16][NG][2], const T* qb, int G, int lane) {
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
    const int g = ng * 8 + (lane >> 2);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int d = kk * 16 + (lane & 3) * 4;
      if (g < G) {
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>(qb + g * D + d));
        if constexpr (std::is_same<T, __half>::value) {
          qf[kk][ng][0] = raw.x;
          qf[kk][ng][1] = raw.y;
        } else {
          const float2 a = Mma<__nv_bfloat16>::unpack(raw.x), b = Mma<__nv_bfloat16>::unpack(raw.y);
          qf[kk][ng][0] = Mma<__half>::pack(a.x, a.y);
          qf[kk][ng][1] = Mma<__half>::pack(b.x, b.y);
        }
      } else {
        qf[kk][ng][0] = 0u;
        qf[kk][ng][1] = 0u;
      }
    }
  }
}

// store_state for the fp8 path: accumulator row g of m-tile mt is dim
// mt*16 + 2g, row g + 8 is dim mt*16 + 2g + 1.
template <int D, int NG>
__device__ __forceinline__ void store_state_f8(WarpState<D, NG>& st, float* Os, float* Ms, float* Ls, int cw,
                                               int lane) {
  constexpr int GP = 8 * NG;
#pragma unroll
  for (int ng = 0; ng < NG; ++ng)
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) st.l[ng][c] += __shfl_xor_sync(0xffffffffu, st.l[ng][c], off);
  constexpr int DP = merge_row<D>();
  float* o = Os + cw * GP * DP;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      const int d0 = mt * 16 + (lane >> 2) * 2, g0 = ng * 8 + (lane & 3) * 2;
      o[g0 * DP + d0] = st.acc[mt][ng][0];
      o[(g0 + 1) * DP + d0] = st.acc[mt][ng][1];
      o[g0 * DP + d0 + 1] = st.acc[mt][ng][2];
      o[(g0 + 1) * DP + d0 + 1] = st.acc[mt][ng][3];
    }
  if (lane < 4) {
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        Ms[cw * GP + ng * 8 + lane * 2 + c] = st.m[ng][c];
        Ls[cw * GP + ng * 8 + lane * 2 + c] = st.l[ng][c];
      }
  }
}

// One fp8 tile as one online-softmax step (as consume_subtiles, with the
// operands taken from E4M3 codes and the per-token scales applied).
template <int D, int TT, int NG, int NS>
__device__ __forceinline__ void consume_subtiles_f8(WarpState<D, NG>& st, uint32_t kt_a, uint32_t vt_a,
                                                    const float* ks, const float* vs, int tok0, int L, float sl2,
                                                    int lane) {
  using M = Mma<__half>;
  constexpr int KS = D / 16;
  const int g = lane >> 2;
  // ldmatrix x4 lane -> (token within the sub-tile, 16-byte column chunk offset)
  const int lm_tok = (lane & 7) + ((lane >> 3) & 1) * 8, lm_chunk = lane >> 4;
  float sc[NS][NG][4];
#pragma unroll
  for (int u = 0; u < NS; ++u)
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) sc[u][ng][0] = sc[u][ng][1] = sc[u][ng][2] = sc[u][ng][3] = 0.f;
#pragma unroll
  for (int kp = 0; kp < KS / 2; ++kp) {  // 32 dims: two k-steps per ldmatrix.x4
    uint32_t r[NS][4];
#pragma unroll
    for (int u = 0; u < NS; ++u)
      ldmatrix_x4(kt_a + swz8<TT>(u * 16 + lm_tok, (2 * kp + lm_chunk) * 16), r[u][0], r[u][1], r[u][2], r[u][3]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // k-step 2kp + h from registers 2h (tokens g) and 2h + 1 (tokens g + 8)
      uint32_t a[NS][4];
#pragma unroll
      for (int u = 0; u < NS; ++u) {
        a[u][0] = e4m3x2_f16(r[u][2 * h]);
        a[u][1] = e4m3x2_f16(r[u][2 * h + 1]);
        a[u][2] = e4m3x2_f16(r[u][2 * h] >> 16);
        a[u][3] = e4m3x2_f16(r[u][2 * h + 1] >> 16);
      }
#pragma unroll
      for (int u = 0; u < NS; ++u)
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) M::run(sc[u][ng], a[u], st.qf[2 * kp + h][ng][0], st.qf[2 * kp + h][ng][1]);
    }
  }
  // per-token scales of this lane's two rows per sub-tile; V's are 0 past the end
  float kslo[NS], kshi[NS], vslo[NS], vshi[NS];
#pragma unroll
  for (int u = 0; u < NS; ++u) {
    const int rr = u * 16 + g;
    kslo[u] = ks[rr];
    kshi[u] = ks[rr + 8];
    vslo[u] = tok0 + rr < L ? vs[rr] : 0.f;
    vshi[u] = tok0 + rr + 8 < L ? vs[rr + 8] : 0.f;
  }
  uint32_t pb[NS][NG][2];
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
    float x[NS][4];
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int u = 0; u < NS; ++u) {
      const int t_lo = tok0 + u * 16 + g;
      const bool in_lo = t_lo < L, in_hi = t_lo + 8 < L;
      x[u][0] = in_lo ? sc[u][ng][0] * kslo[u] * sl2 : -INFINITY;
      x[u][1] = in_lo ? sc[u][ng][1] * kslo[u] * sl2 : -INFINITY;
      x[u][2] = in_hi ? sc[u][ng][2] * kshi[u] * sl2 : -INFINITY;
      x[u][3] = in_hi ? sc[u][ng][3] * kshi[u] * sl2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(x[u][0], x[u][2]));
      mx1 = fmaxf(mx1, fmaxf(x[u][1], x[u][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(st.m[ng][0], mx0), mn1 = fmaxf(st.m[ng][1], mx1);
    const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0, mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
    const float al0 = fast_exp2(st.m[ng][0] - mu0), al1 = fast_exp2(st.m[ng][1] - mu1);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int u = 0; u < NS; ++u) {
      const float p0 = fast_exp2(x[u][0] - mu0), p1 = fast_exp2(x[u][1] - mu1);
      const float p2 = fast_exp2(x[u][2] - mu0), p3 = fast_exp2(x[u][3] - mu1);
      s0 += p0 + p2;
      s1 += p1 + p3;
      pb[u][ng][0] = movmatrix_trans(M::pack(p0 * vslo[u], p1 * vslo[u]));
      pb[u][ng][1] = movmatrix_trans(M::pack(p2 * vshi[u], p3 * vshi[u]));
    }
    st.l[ng][0] = st.l[ng][0] * al0 + s0;
    st.l[ng][1] = st.l[ng][1] * al1 + s1;
    st.m[ng][0] = mn0;
    st.m[ng][1] = mn1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      st.acc[mt][ng][0] *= al0;
      st.acc[mt][ng][1] *= al1;
      st.acc[mt][ng][2] *= al0;
      st.acc[mt][ng][3] *= al1;
    }
  }
  // O^T += V^T P^T, two m-tiles (32 dims) per ldmatrix.x4.trans
#pragma unroll
  for (int mp = 0; mp < KS / 2; ++mp) {
    uint32_t r[NS][4];
#pragma unroll
    for (int u = 0; u < NS; ++u)
      ldmatrix_x4_trans(vt_a + swz8<TT>(u * 16 + lm_tok, (2 * mp + lm_chunk) * 16), r[u][0], r[u][1], r[u][2],
                        r[u][3]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // m-tile 2mp + h: registers 2h (tokens 2t, 2t+1) and 2h + 1 (tokens + 8)
      uint32_t a[NS][4];
#pragma unroll
      for (int u = 0; u < NS; ++u) {
        // bytes (tok 2t: dim 2g, 2g+1; tok 2t+1: dim 2g, 2g+1) -> (dim 2g: both tokens | dim 2g+1: both)
        const uint32_t lo = __byte_perm(r[u][2 * h], 0u, 0x3120), hi = __byte_perm(r[u][2 * h + 1], 0u, 0x3120);
        a[u][0] = e4m3x2_f16(lo);        // row g = dim 2g, tokens 2t, 2t+1
        a[u][1] = e4m3x2_f16(lo >> 16);  // row g + 8 = dim 2g + 1
        a[u][2] = e4m3x2_f16(hi);        // dim 2g, tokens 2t + 8, 2t + 9
        a[u][3] = e4m3x2_f16(hi >> 16);
      }
#pragma unroll
      for (int u = 0; u < NS; ++u)
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) M::run(st.acc[2 * mp + h][ng], a[u], pb[u][ng][0], pb[u][ng][1]);
    }
  }
}

template <int D, int TT, int NG>
__device__ __forceinline__ void consume_tile_f8(WarpState<D, NG>& st, uint8_t* kt, uint8_t* vt, const float* ks,
                                                const float* vs, int tok0, int L, float sl2, int lane) {
  const int valid = min(TT, L - tok0);
  if (valid < TT) {
    // zero the V code rows past the sequence end: their weight is 0, but a
    // stale code may be the NaN pattern and 0 * NaN is not 0
    constexpr int kRowChunks = D / 16;
    for (int c = lane; c < (TT - valid) * kRowChunks; c += 32) {
      const int t = valid + c / kRowChunks, d = (c % kRowChunks) * 16;
      *reinterpret_cast<uint4*>(vt + swz8<TT>(t, d)) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();  // these bytes are TMA-written again later
    __syncwarp();
  }
  const uint32_t kt_a = smem_u32(kt), vt_a = smem_u32(vt);
  static_assert(TT == 32 || TT == 64, "fp8 tiles are 32 or 64 tokens");
  if (TT == 64 && valid > 48) consume_subtiles_f8<D, TT, NG, TT / 16>(st, kt_a, vt_a, ks, vs, tok0, L, sl2, lane);
  else if (TT == 64 && valid > 32) consume_subtiles_f8<D, TT, NG, 3>(st, kt_a, vt_a, ks, vs, tok0, L, sl2, lane);
  else if (valid > 16) consume_subtiles_f8<D, TT, NG, 2>(st, kt_a, vt_a, ks, vs, tok0, L, sl2, lane);
  else consume_subtiles_f8<D, TT, NG, 1>(st, kt_a, vt_a, ks, vs, tok0, L, sl2, lane);
}

constexpr int kConsumers = 4;
constexpr int kTcThreads = 32 * (kConsumers + 1);
// Stream-K kernel: the producer warp, the consumer warps, and a writer warp
// that does the fused step's cache write while the others stream tiles (the
// writes belong to no tile of the launch, so their order does not matter)
constexpr int kSkWriterWarp = kConsumers + 1;
constexpr int kSkThreads = 32 * (kConsumers + 2);

template <int D, int NG>
struct MergeArea {
  static constexpr int kGP = 8 * NG;
  static constexpr int kBytes = kConsumers * (merge_row<D>() * kGP + 2 * kGP) * 4;
};

// Output (g, d) of the consumer warps' states stored by store_state:
// running max, unnormalised numerator and denominator after rescaling every
// warp to the common max (all -inf: no token seen, zeros).
template <int D, int GP>
__device__ __forceinline__ void warp_merge(const float* Os, const float* Ms, const float* Ls, int g, int d, float& mx,
                                           float& num, float& den) {
  mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kConsumers; ++w) mx = fmaxf(mx, Ms[w * GP + g]);
  num = den = 0.f;
  if (mx == -INFINITY) return;
#pragma unroll
  for (int w = 0; w < kConsumers; ++w) {
    const float mw = Ms[w * GP + g];
    if (mw == -INFINITY) continue;
    const float sc = fast_exp2(mw - mx);
    num += sc * Os[(w * GP + g) * merge_row<D>() + d];
    den += sc * Ls[w * GP + g];
  }
}

// =========================================================================
// Stream-K tensor-core kernel (the default for fp16/bf16).
//
// The work is the ordered list of tiles (sequence b, kv head, 32 tokens),
// W = Hkv * sum_b ceil(L_b / 32) of them.  The grid is one wave of
// persistent CTAs; CTA p takes the tiles whose positions in a cost space
// (tiles plus a fixed charge per unit) fall in [p*Wc/P, (p+1)*Wc/P), so
// every CTA moves about the same number of bytes whatever the length mix.
// A unit (b, kv head) whose tiles all fall in one CTA is finished there and
// written to `out`.  A unit cut by range boundaries is finished by its
// owner, the CTA holding its first tiles (the end of the owner's range):
// every later CTA holding a piece of it writes an unnormalised partial
// (acc, m, l) to the workspace and releases a ready flag.  Once the owner's
// producer warp has issued its last tile it waits for those flags and
// bulk-copies the partials into the stage that frees up next, so the
// owner's combine, right after its last tile, reads them from shared memory
// and its own piece from the warp-merge buffer.  Every CTA first rebuilds
// the per-sequence prefixes of tile counts and costs in shared memory from
// seq_lens.
//
// Warps: a producer (TMA), four consumers (tile j goes to consumer j % 4),
// and a writer that does a fused step's cache write while the others stream
// tiles.  At the end of a unit's segment each consumer stores its softmax
// state into one of two merge buffers and counts itself in; the last of the
// four merges the segment (output or partial) while the others go on with
// their next tiles, then frees the buffer for the segment two later.
// =========================================================================

// Fused step, cache write ("MiniPaged-Qwen" §12): warp gw of nw copies the
// K and V rows of tokens gw, gw + nw, ... to cache[slot / bs][slot % bs],
// slot = slot_mapping[t] (-1: padded token, skipped; outside the pool:
// recorded and skipped).  A lane fetches the slots of 32 of the warp's
// tokens at once; each row is loaded whole (16-byte vectors) before it is
// stored.
template <typename T>
__device__ __forceinline__ void scatter_new_rows(const DecodeParams& p, int64_t gw, int64_t nw, int lane) {
  const int row_vecs = p.num_kv_heads * p.head_dim * static_cast<int>(sizeof(T)) / 16;
  const int64_t row_bytes = static_cast<int64_t>(row_vecs) * 16;
  const int64_t num_slots = p.num_blocks * p.block_size;
  constexpr int kVec = 4;
  for (int64_t base = gw; base < p.num_new; base += 32 * nw) {
    const int64_t mine = base + lane * nw;
    const int32_t my_slot = mine < p.num_new ? __ldg(p.slot_mapping + mine) : -1;
    for (int i = 0; i < 32; ++i) {
      const int64_t t = base + i * nw;
      if (t >= p.num_new) break;
      const int32_t slot = __shfl_sync(0xffffffffu, my_slot, i);
      if (slot == -1) continue;
      if (slot < 0 || slot >= num_slots) {
        if (lane == 0) record_error(KV_ERR_DEVICE_BOUNDS);
        continue;
      }
      const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const char*>(p.new_k) + t * p.new_k_stride);
      const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const char*>(p.new_v) + t * p.new_v_stride);
      uint4* kd = reinterpret_cast<uint4*>(static_cast<char*>(const_cast<void*>(p.k_cache)) + slot * row_bytes);
      uint4* vd = reinterpret_cast<uint4*>(static_cast<char*>(const_cast<void*>(p.v_cache)) + slot * row_bytes);
      for (int v0 = lane; v0 < row_vecs; v0 += 32 * kVec) {
        uint4 kr[kVec], vr[kVec];
#pragma unroll
        for (int u = 0; u < kVec; ++u)
          if (v0 + 32 * u < row_vecs) {
            kr[u] = __ldg(ks + v0 + 32 * u);
            vr[u] = __ldg(vs + v0 + 32 * u);
          }
#pragma unroll
        for (int u = 0; u < kVec; ++u)
          if (v0 + 32 * u < row_vecs) {
            kd[v0 + 32 * u] = kr[u];
            vd[v0 + 32 * u] = vr[u];
          }
      }
    }
  }
}

// fp8 (E4M3) quantisation of one (token, kv head) row of 128 values held 4
// per lane across a warp: scale = amax / 448 (1 for a zero row), values
// divided by it with one correct rounding and rounded to E4M3 nearest-even,
// saturating -- the steps of paged_reshape_and_cache_fp8, so the codes and
// scale are bit-identical.  Returns the lane's 4 codes (lowest dim first).
template <typename T>
__device__ __forceinline__ uint32_t quantize4_e4m3(uint2 raw, float& scale) {
  const T* v = reinterpret_cast<const T*>(&raw);
  float x[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = DType<T>::to_float(v[e]);
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(__fdiv_rn(x[1], scale)), "f"(__fdiv_rn(x[0], scale)));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(__fdiv_rn(x[3], scale)), "f"(__fdiv_rn(x[2], scale)));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Fused fp8 step, cache write: as scatter_new_rows, each (token, kv head)
// row quantised into the E4M3 caches and its scale into the scale arrays
// (head_dim 128).
template <typename T>
__device__ __forceinline__ void scatter_new_rows_f8(const DecodeParams& p, int64_t gw, int64_t nw, int lane) {
  const int64_t num_slots = p.num_blocks * p.block_size;
  const int Hkv = p.num_kv_heads, BS = p.block_size;
  for (int64_t base = gw; base < p.num_new; base += 32 * nw) {
    const int64_t mine = base + lane * nw;
    const int32_t my_slot = mine < p.num_new ? __ldg(p.slot_mapping + mine) : -1;
    for (int i = 0; i < 32; ++i) {
      const int64_t t = base + i * nw;
      if (t >= p.num_new) break;
      const int32_t slot = __shfl_sync(0xffffffffu, my_slot, i);
      if (slot == -1) continue;
      if (slot < 0 || slot >= num_slots) {
        if (lane == 0) record_error(KV_ERR_DEVICE_BOUNDS);
        continue;
      }
      const int64_t blk = slot / BS, off = slot % BS;
      for (int h = 0; h < Hkv; ++h) {
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const char* src = static_cast<const char*>(which ? p.new_v : p.new_k) +
                            t * (which ? p.new_v_stride : p.new_k_stride) +
                            (static_cast<int64_t>(h) * 128 + lane * 4) * static_cast<int64_t>(sizeof(T));
          float scale;
          const uint32_t codes = quantize4_e4m3<T>(__ldg(reinterpret_cast<const uint2*>(src)), scale);
          uint8_t* dst = static_cast<uint8_t*>(const_cast<void*>(which ? p.v_cache : p.k_cache)) +
                         (static_cast<int64_t>(slot) * Hkv + h) * 128 + lane * 4;
          *reinterpret_cast<uint32_t*>(dst) = codes;
          if (lane == 0) const_cast<float*>(which ? p.v_scales : p.k_scales)[(blk * Hkv + h) * BS + off] = scale;
        }
      }
    }
  }
}

// Grid cap: an owner CTA indexes up to kMaxSkCtas pieces in shared memory.
constexpr int kMaxSkCtas = 640;
// An owner's producer warp waits for the later pieces and copies them into
// stages as the consumers free them on their last tiles (else the consumers
// wait and read every piece from global memory after the last tile).
constexpr bool kPrefetchParts = true;

// Tokens a stream-K tile aims at: 32 for 16-bit caches (one block of 32, or
// two consecutive blocks of 16: fewer, larger pipeline transactions; 16-token
// tiles were measured slower, a consumer's fixed cost per tile outweighing
// the second stage per warp they allow).  fp8: 64 tokens for up to 8 query
// heads per kv head, so a stage carries as many bytes as a 16-bit one (more
// heads: 32, to fit registers).
constexpr int sk_want_tokens(int D, int NG, bool F8) { return F8 ? (NG == 1 ? 64 : 32) : 32; }

template <typename T, int D, int BS, int NG, int NST, bool F8 = false>
struct SkCfg {
  // A stream-K tile is sk_want_tokens tokens: one block, or consecutive
  // blocks of the same sequence.
  static constexpr int kWantTokens = sk_want_tokens(D, NG, F8);
  static constexpr int kBlocksPerTile = BS >= kWantTokens ? 1 : kWantTokens / BS;
  static constexpr int kTileTokens = BS * kBlocksPerTile;
  // fp8 caches: E4M3 code tiles, and per stage the tile's K and V scales.
  // A tile of 2 or 4 blocks gets each of its K and V scale rows with one
  // TMA gather of four table rows (a 2-block tile repeats its last block),
  // so a scale slot holds 4 blocks' rows; otherwise one bulk copy per block.
  using TL = typename std::conditional<F8, Tile8<D, kTileTokens>, Tile<D, kTileTokens>>::type;
  static constexpr bool kGatherScales = F8 && (kBlocksPerTile == 2 || kBlocksPerTile == 4);
  static constexpr int kScaleSlot = kGatherScales ? 4 * BS : kTileTokens;  // floats per (stage, K or V)
  static constexpr int kStages = NST * TL::kStageBytes;
  static constexpr int kScales = F8 ? NST * 2 * kScaleSlot * 4 : 0;
  static constexpr int kMerge = 2 * MergeArea<D, NG>::kBytes;  // double-buffered per segment
  static constexpr int kPartRows = kMaxSkCtas + 8;  // row index per part of a combined unit
  static constexpr int kFixed = 1024 + kStages + kScales + kMerge + 2 * NST * 8 + 16 + 32 + kPartRows * 4;
  static int smem_bytes(int B) { return kFixed + (2 * (B + 1) * 4 + 15) / 16 * 16; }
};

// cta_of(x): the CTA whose range [p*W/P, (p+1)*W/P) holds position x.
__device__ __forceinline__ int sk_cta_of(int64_t t, int64_t W, int P) {
  return static_cast<int>(((t + 1) * P + W - 1) / W - 1);
}


template <typename T, int D, int BS, int NG, int NST, bool F8 = false>
__global__ void __launch_bounds__(kSkThreads, D <= 128 ? 2 : 1)  // two CTAs per SM where shared memory allows
decode_sk_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKS,
                 const __grid_constant__ CUtensorMap tmVS) {
  using C = SkCfg<T, D, BS, NG, NST, F8>;
  using TL = typename C::TL;
  constexpr int TPB = C::kBlocksPerTile, TT = C::kTileTokens;
  // TMA copies per block of a tile: 16-bit caches one each for K and V (a
  // 4-D box covers all of a block's 64-column slabs); fp8 caches K and V
  // slabs, and the K and V scales unless two gathers per tile bring them
  constexpr bool kGather = C::kGatherScales;
  constexpr int kPerBlock = F8 ? 2 * TL::kSub + (kGather ? 0 : 2) : 2;
  constexpr int kCopies = kPerBlock * TPB + (kGather ? 2 : 0);
  static_assert(kCopies <= 32, "one copy per producer lane");
  // bytes one block of a tile brings into its stage (scales by gather: per tile)
  constexpr int kBlockTx = F8 ? 2 * BS * D + (kGather ? 0 : 2 * BS * 4) : TL::kStageBytes / TPB;
  constexpr int kTileTx = kGather ? 2 * 4 * BS * 4 : 0;
  constexpr int kScaleSlot = C::kScaleSlot;
  constexpr int GP = 8 * NG;
  static_assert(NST % kConsumers == 0, "stage s must always be drained by consumer s % kConsumers");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* scales = reinterpret_cast<float*>(smem + C::kStages);  // fp8: [NST][2][kScaleSlot] K, V scales
  float* merge_base = reinterpret_cast<float*>(smem + C::kStages + C::kScales);
  constexpr int kMergeFloats = MergeArea<D, NG>::kBytes / 4;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages + C::kScales + C::kMerge);
  uint64_t* empty = full + NST;
  uint64_t* pre_bar = empty + NST;                       // owner: later pieces copied in
  uint64_t* seg_free = pre_bar + 2;                      // [2] merge buffer read by its merge
  int* seg_cnt = reinterpret_cast<int*>(seg_free + 2);   // [2] warps that stored into the buffer
  int* part_row = seg_cnt + 4;                           // [kPartRows]
  int* CB = part_row + C::kPartRows;  // CB[b] = sum_{b' < b} ceil(L_b' / TT) (tiles)

  const int B = p.num_seqs, Hkv = p.num_kv_heads, G = p.group;
  int* CC = CB + (B + 1);  // CC[b] = sum_{b' < b} cost_b' (tiles + seg_cost, 0 if empty)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- prefixes of block counts and costs over the batch (block-wide scans) ----
  {
    const int per = (B + kSkThreads - 1) / kSkThreads;
    const int beg = min(B, tid * per), end = min(B, beg + per);
    int local = 0, local_c = 0;
    for (int i = beg; i < end; ++i) {
      const int nb = (checked_len(p, i) + TT - 1) / TT;
      CB[i + 1] = nb;
      local += nb;
      local_c += nb > 0 ? nb + p.seg_cost : 0;
    }
    int incl = local, incl_c = local_c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      const int yc = __shfl_up_sync(0xffffffffu, incl_c, off);
      if (lane >= off) {
        incl += y;
        incl_c += yc;
      }
    }
    __shared__ int warp_tot[kConsumers + 2], warp_tot_c[kConsumers + 2];
    if (lane == 31) {
      warp_tot[warp] = incl;
      warp_tot_c[warp] = incl_c;
    }
    if (tid == 0) CB[0] = CC[0] = 0;
    __syncthreads();
    int base = 0, base_c = 0;
    for (int w = 0; w < warp; ++w) {
      base += warp_tot[w];
      base_c += warp_tot_c[w];
    }
    int run = base + incl - local, run_c = base_c + incl_c - local_c;
    for (int i = beg; i < end; ++i) {
      const int nb = CB[i + 1];
      run += nb;
      run_c += nb > 0 ? nb + p.seg_cost : 0;
      CB[i + 1] = run;
      CC[i + 1] = run_c;
    }
    if (tid == 0) {
      for (int s = 0; s < NST; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      mbar_init(pre_bar, 1);
      mbar_init(&seg_free[0], 1);
      mbar_init(&seg_free[1], 1);
      seg_cnt[0] = seg_cnt[1] = 0;
      fence_mbar_init();
    }
    __syncthreads();
  }
  // sequences with no tokens get zero rows (no tile covers them)
  for (int bz = blockIdx.x; bz < B; bz += gridDim.x)
    if (CB[bz + 1] == CB[bz]) {
      T* o = static_cast<T*>(p.out) + static_cast<int64_t>(bz) * p.num_heads * D;
      for (int i = tid; i < p.num_heads * D; i += kSkThreads) o[i] = DType<T>::from_float(0.f);
    }

  // CTA ranges are drawn in cost space, where unit (b, kvh) occupies
  // seg_cost virtual positions followed by its ceil(L_b / BS) tiles, so a
  // CTA whose range holds many short units (each paying a merge) gets fewer
  // tiles.  Tile range of CTA p: the tiles whose positions fall in
  // [p * Wc / P, (p + 1) * Wc / P).
  const int64_t W = static_cast<int64_t>(Hkv) * CB[B];
  const int64_t Wc = static_cast<int64_t>(Hkv) * CC[B];
  const int P = gridDim.x, pid = blockIdx.x;
  auto tiles_before = [&](int64_t x) -> int64_t {  // tiles at cost positions < x
    if (x >= Wc) return W;
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<int64_t>(Hkv) * CC[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const int cs = CC[lo + 1] - CC[lo], nb = CB[lo + 1] - CB[lo];
    const int64_t rel = x - static_cast<int64_t>(Hkv) * CC[lo];
    const int kvh = static_cast<int>(rel / cs), r = static_cast<int>(rel % cs);
    return static_cast<int64_t>(Hkv) * CB[lo] + static_cast<int64_t>(kvh) * nb + max(0, r - p.seg_cost);
  };
  const int64_t t0 = tiles_before(static_cast<int64_t>(pid) * Wc / P);
  const int64_t t1 = tiles_before(static_cast<int64_t>(pid + 1) * Wc / P);
  // Fused step: the writer warps of all CTAs copy the step's new rows into
  // the caches, CTA p's warp rows p, p + P, ... (a CTA with no tiles as well)
  if (warp == kSkWriterWarp) {
    if (p.new_k != nullptr) {
      if constexpr (F8) scatter_new_rows_f8<T>(p, pid, P, lane);
      else scatter_new_rows<T>(p, pid, P, lane);
    }
    return;
  }
  if (t0 >= t1) return;
  const int n = static_cast<int>(t1 - t0);

  // Tile cursor shared by producer and consumers: advances (blk, kvh, b).
  struct Cursor {
    int b, kvh, blk, nb;
  };
  auto advance = [&](Cursor& c) {
    if (++c.blk == c.nb) {
      c.blk = 0;
      if (++c.kvh == Hkv) {
        c.kvh = 0;
        do {
          ++c.b;
        } while (c.b < B && CB[c.b + 1] == CB[c.b]);
        c.nb = c.b < B ? CB[c.b + 1] - CB[c.b] : 0;
      }
    }
  };
  // cursor of tile t < W: the largest b with Hkv * CB[b] <= t is never empty
  auto locate = [&](int64_t t) -> Cursor {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<int64_t>(Hkv) * CB[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int nb = CB[lo + 1] - CB[lo];
    const int rel = static_cast<int>(t - static_cast<int64_t>(Hkv) * CB[lo]);
    return Cursor{lo, rel / nb, rel % nb, nb};
  };

  // ---- the unit cut at the range end, if any: this CTA (its owner)
  // combines it with the pieces later CTAs hold ----
  // Given the cursor of the range's last tile: the unit started inside the
  // range and goes on after it.  Its other pieces are the later CTAs up to
  // `last` (the one holding the unit's last tile) whose cost ranges are not
  // empty: their ranges lie inside the unit's tiles.
  auto owner_of = [&](const Cursor& lc, int& last) -> bool {
    const bool own = lc.blk <= n - 1 && lc.blk + 1 < lc.nb;
    last = pid;
    if (own) {
      const int cs = CC[lc.b + 1] - CC[lc.b];
      last = sk_cta_of(
          static_cast<int64_t>(Hkv) * CC[lc.b] + static_cast<int64_t>(lc.kvh) * cs + p.seg_cost + lc.nb - 1, Wc, P);
    }
    return own;
  };
  // The first pieces (up to the capacity of one stage) are copied into the
  // stage that frees up after the last tile, so the owner's combine reads
  // them from shared memory; further pieces are read from global memory.
  // Piece i goes to the stage virtual tile n + i / per_stage would use,
  // which frees up once tile n + i / per_stage - NST is consumed.
  const int part_o = G * D * 4, part_ml = (G * 8 + 15) & ~15, part_bytes = part_o + part_ml;
  const int per_stage = TL::kStageBytes / part_bytes;  // 0: pieces too large for a stage, none copied
  auto npre_of = [&](int last) {
    return kPrefetchParts && Wc >= P && per_stage > 0 ? min(min(NST * per_stage, 32), last - pid) : 0;
  };
  auto pre_part = [&](int i) {
    return smem + ((n + i / per_stage) % NST) * TL::kStageBytes + (i % per_stage) * part_bytes;
  };
  const Cursor c_first = locate(t0);

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      if constexpr (kGather) {
        prefetch_tensormap(&tmKS);
        prefetch_tensormap(&tmVS);
      }
    }
    Cursor c = c_first;  // c.blk counts tiles of TPB blocks
    // Block-table entries are fetched 32 at a time (one per lane; entries
    // past the sequence are fetched but never used) and the chunk the walk
    // needs next is fetched while the current one is used.
    auto fetch = [&](int b, int chunk) -> int {
      const int e = (chunk << 5) + lane;
      return e < p.max_blocks_per_seq ? __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq + e)
                                      : 0;
    };
    auto nblocks = [&](int b) { return (checked_len(p, b) + BS - 1) / BS; };
    int cache_b = -1, cache_chunk = -1, cache_nblk = 0, mine = 0;
    int next_b = -1, next_chunk = -1, nxt = 0;
    int ok = 1, issued = 0;
    for (int j = 0; j < n && ok; ++j) {
      const int blk = c.blk * TPB;  // first block of this tile
      if (c.b != cache_b || (blk >> 5) != cache_chunk) {
        mine = (c.b == next_b && (blk >> 5) == next_chunk) ? nxt : fetch(c.b, blk >> 5);
        if (c.b != cache_b) cache_nblk = nblocks(c.b);
        cache_b = c.b;
        cache_chunk = blk >> 5;
        // the chunk after this one in walk order: next chunk of the row, the
        // row's first chunk again for the next kv head, or the next sequence
        int nbk = c.b, nck = cache_chunk + 1;
        if (nck * 32 >= cache_nblk) {
          nck = 0;
          if (c.kvh + 1 >= Hkv) {
            do {
              ++nbk;
            } while (nbk < B && CB[nbk + 1] == CB[nbk]);
          }
        }
        if (nbk < B && !(nbk == cache_b && nck == cache_chunk)) {
          nxt = fetch(nbk, nck);
          next_b = nbk;
          next_chunk = nck;
        } else {
          next_b = -1;
        }
      }
      // One copy per lane: lane l < kCopies loads block r = l / kPerBlock of
      // the tile.  16-bit caches: w = l % 2 is K (0) or V (1), all of the
      // block's column slabs in one 4-D tensor copy into the block's place
      // in the tile (block-major, see swz).  fp8: w < 2 kSub is column slab
      // w / 2 of K (even w) or V (odd w), and w = 2 kSub, 2 kSub + 1 the
      // block's K and V scales, bs contiguous floats each (a bulk copy:
      // 16-byte aligned source and destination, bs * 4 bytes).  Tensor-copy
      // destinations are 1024-byte aligned.
      const int cr = lane / kPerBlock, cw8 = lane % kPerBlock, csl = (cw8 >> 1) % TL::kSub;
      int pb = __shfl_sync(0xffffffffu, mine, (blk + min(cr, TPB - 1)) & 31);
      const int here = min(TPB, cache_nblk - blk);  // blocks of this tile inside the sequence (>= 1)
      // scale gathers: the table rows (block, kv head) of the tile's blocks,
      // blocks past the sequence's end repeating its last one
      int srow[4] = {0, 0, 0, 0};
      if constexpr (kGather) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          int b4 = __shfl_sync(0xffffffffu, mine, (blk + min(r, here - 1)) & 31);
          if (b4 < 0 || b4 >= p.num_blocks) b4 = 0;  // recorded by the code copy of that block
          srow[r] = b4 * Hkv + c.kvh;
        }
      }
      const int s = j % NST;
      if (lane == 0) {
        if (j >= NST) ok = mbar_wait_for(&empty[s], ((j / NST) - 1) & 1, p.wait_limit_ns);
        if (ok) mbar_arrive_expect_tx(&full[s], here * kBlockTx + kTileTx);
      }
      __syncwarp();
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // test control: CTA 0 never loads its tile test_skip_tile, so the wait
      // for it runs out (the timeout path, exercised without a fault)
      const bool skip = p.test_skip_tile >= 0 && pid == 0 && j == p.test_skip_tile;
      const bool gather_lane = kGather && lane >= kPerBlock * TPB && lane < kCopies;
      if (ok && !skip && gather_lane) {
        const int which = lane - kPerBlock * TPB;  // 0: K scales, 1: V scales
        tma_gather4(scales + (s * 2 + which) * kScaleSlot, which ? &tmVS : &tmKS, &full[s], 0, srow[0], srow[1],
                    srow[2], srow[3]);
      } else if (ok && !skip && lane < kPerBlock * TPB && cr < here) {
        if (pb < 0 || pb >= p.num_blocks) {
          record_error(KV_ERR_DEVICE_BOUNDS);
          pb = 0;
        }
        if constexpr (!F8) {
          uint8_t* dst = smem + s * TL::kStageBytes + cw8 * TL::kTileBytes + cr * (TL::kSub * BS * 128);
          tma_load_4d(dst, cw8 ? &tmV : &tmK, &full[s], 0, pb * BS, 0, c.kvh);
        } else if (cw8 < 2 * TL::kSub) {
          uint8_t* dst = smem + s * TL::kStageBytes + (cw8 & 1) * TL::kTileBytes + csl * TL::kSlabBytes + cr * BS * 128;
          tma_load_3d(dst, (cw8 & 1) ? &tmV : &tmK, &full[s], csl * 128, c.kvh, pb * BS);
        } else {
          const int which = cw8 - 2 * TL::kSub;  // 0: K scales, 1: V scales
          float* dst = scales + (s * 2 + which) * kScaleSlot + cr * BS;
          const float* src = (which ? p.v_scales : p.k_scales) + (static_cast<int64_t>(pb) * Hkv + c.kvh) * BS;
          bulk_load(dst, src, BS * 4, &full[s]);
        }
      }
      if (ok) ++issued;
      if (j + 1 < n) advance(c);
    }
    int last;
    const bool owner = owner_of(c, last);
    const int npre = npre_of(last);
    if (kPrefetchParts && owner) {
      // Wait (bounded) for every later piece's ready flag; each flag has
      // this one reader, which clears it, so flags are zero between calls
      // even when a replayed launch reuses its epoch.  Those CTAs publish
      // their first piece before they wait on anyone: no cycle.
      for (int q0 = pid + 1; q0 <= last; q0 += 32) {
        const int q = q0 + lane;
        if (q <= last && static_cast<int64_t>(q) * Wc / P != static_cast<int64_t>(q + 1) * Wc / P) {
          const uint64_t t_start = globaltimer_ns();
          while (ok && ld_acquire_gpu(p.ws_flags + q) != p.epoch) {
            if (globaltimer_ns() - t_start > p.wait_limit_ns) {
              record_error(KV_ERR_DEVICE_TIMEOUT);
              ok = 0;
            }
            __nanosleep(32);
          }
          p.ws_flags[q] = 0;
        }
      }
      fence_proxy_async_global();  // the partials acquired above, before the bulk copies read them
      // Every lane's flags are seen before lane 0 signals pre_bar: with no
      // piece to copy its arrive alone releases the consumers, who then read
      // all pieces from global memory.
      __syncwarp();
      if (lane == 0) {
        if (npre > 0) {
          mbar_arrive_expect_tx(pre_bar, npre * (part_o + part_ml));
          // the stages the pieces go to (virtual tiles n, n + 1, ...) must be free
          for (int v = n; (v - n) * per_stage < npre; ++v)
            if (v >= NST) mbar_wait_for(&empty[v % NST], ((v / NST) - 1) & 1, p.wait_limit_ns);
        } else {
          mbar_arrive(pre_bar);
        }
      }
      __syncwarp();
      if (lane < npre) {  // lane i acquired piece i's flag above and copies it (npre <= 32)
        const int64_t row = static_cast<int64_t>(pid + 1 + lane) * 2 * G;  // slot 0 of CTA pid + 1 + lane
        bulk_load(pre_part(lane), p.ws_o + row * D, part_o, pre_bar);
        bulk_load(pre_part(lane) + part_o, p.ws_ml + row * 2, part_ml, pre_bar);
      }
    }
    if (lane == 0) {  // keep the CTA alive until every issued copy has landed (bounded)
      for (int s = 0; s < NST && s < issued; ++s) {
        const int lst = s + ((issued - 1 - s) / NST) * NST;
        mbar_wait_for(&full[s], (lst / NST) & 1, p.wait_limit_ns);
      }
      if (kPrefetchParts && owner && npre > 0) mbar_wait_for(pre_bar, 0, p.wait_limit_ns);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int cw = warp - 1, ctid = tid - 32;
  WarpState<D, NG> st;
  Cursor c = c_first;
  const float sl2 = p.scale_log2;
  int ok = 1;
  int64_t unit_start = static_cast<int64_t>(Hkv) * CB[c.b] + static_cast<int64_t>(c.kvh) * c.nb;
  int L = checked_len(p, c.b);
  auto q_of = [&](const Cursor& u) {
    return static_cast<const T*>(p.q) + (static_cast<int64_t>(u.b) * p.num_heads + u.kvh * G) * D;
  };
  // The next unit's Q fragments are loaded one segment ahead, so a unit
  // boundary does not stall on a cold global load (skipped where the extra
  // registers would not fit).
  constexpr bool kPrefetchQ = (D / 16) * NG * 2 <= 16;
  uint32_t qn[D / 16][NG][2];
  auto prefetch_next = [&](const Cursor& u, int64_t u_start) {
    if (kPrefetchQ && u_start + u.nb < t1) {
      Cursor nx = u;
      nx.blk = nx.nb - 1;
      advance(nx);
      if constexpr (F8) load_q_frags_f8<T, D, NG>(qn, q_of(nx), G, lane);
      else load_q_frags<T, D, NG>(qn, q_of(nx), G, lane);
    }
  };
  if constexpr (F8) load_q_frags_f8<T, D, NG>(st.qf, q_of(c), G, lane);
  else load_q<T, D, NG>(st, q_of(c), G, lane);
  prefetch_next(c, unit_start);
  // Fused step: no tile of this launch uses what the writer warps write:
  // position L - 1 of a decode sequence (the only written slot attention
  // reads) is taken from the new row itself below.
  const bool fused = p.new_k != nullptr;
  // row of the step's new K/V holding sequence b's position L - 1 (-1: none)
  auto new_row_of = [&](int b) -> int {
    if (!fused) return -1;
    const int r = __ldg(p.new_row + b);
    if (r >= p.num_new) {
      record_error(KV_ERR_DEVICE_STEP);
      return -1;
    }
    return r;
  };
  int nrow = new_row_of(c.b);
  reset_state(st);
  int seg = 0;
  constexpr int kPatch = (2 * (D / 8) + 31) / 32;  // 16-byte chunks of one token's K and V per lane
  for (int j = 0; j < n; ++j) {
    if (ok && (j & (kConsumers - 1)) == cw) {
      const int s = j % NST;
      // Fused step: the tile holding position L - 1 takes that token's K
      // and V for this kv head from the new row (loaded before the wait).
      const int tl = L - 1 - c.blk * TT;
      const bool patch = !F8 && nrow >= 0 && tl >= 0 && tl < TT;
      // fp8: the token's K and V for this kv head, 4 values per lane, are
      // quantised after the wait exactly as the cache write does
      const bool patch8 = F8 && nrow >= 0 && tl >= 0 && tl < TT;
      uint2 pk8 = make_uint2(0u, 0u), pv8 = make_uint2(0u, 0u);
      if (patch8) {
        const int64_t col = (static_cast<int64_t>(c.kvh) * D + lane * 4) * static_cast<int64_t>(sizeof(T));
        pk8 = __ldg(reinterpret_cast<const uint2*>(static_cast<const char*>(p.new_k) + nrow * p.new_k_stride + col));
        pv8 = __ldg(reinterpret_cast<const uint2*>(static_cast<const char*>(p.new_v) + nrow * p.new_v_stride + col));
        if (lane == 0) {  // the row must be the one the cache write puts at position L - 1
          const int pb = __ldg(p.block_tables + static_cast<int64_t>(c.b) * p.max_blocks_per_seq + (L - 1) / BS);
          const int32_t want = pb * BS + (L - 1) % BS;
          if (__ldg(p.slot_mapping + nrow) != want) record_error(KV_ERR_DEVICE_STEP);
        }
      }
      uint4 pv[kPatch];
      if (patch) {
#pragma unroll
        for (int u = 0; u < kPatch; ++u) {
          const int ch = lane + 32 * u;
          if (ch < 2 * (D / 8)) {
            const bool isv = ch >= D / 8;
            const int d = (ch % (D / 8)) * 8;
            const char* src = static_cast<const char*>(isv ? p.new_v : p.new_k) +
                              static_cast<int64_t>(nrow) * (isv ? p.new_v_stride : p.new_k_stride) +
                              (static_cast<int64_t>(c.kvh) * D + d) * static_cast<int64_t>(sizeof(T));
            pv[u] = __ldg(reinterpret_cast<const uint4*>(src));
          }
        }
        if (lane == 0) {  // the row must be the one the cache write puts at position L - 1
          const int pb = __ldg(p.block_tables + static_cast<int64_t>(c.b) * p.max_blocks_per_seq + (L - 1) / BS);
          const int32_t want = pb * BS + (L - 1) % BS;
          if (__ldg(p.slot_mapping + nrow) != want) record_error(KV_ERR_DEVICE_STEP);
        }
      }
      int w = 1;
      if (lane == 0) w = mbar_wait_for(&full[s], (j / NST) & 1, p.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, w, 0);
      if (ok) {
        __syncwarp();
        uint8_t* kt = smem + s * TL::kStageBytes;
        if (patch) {
#pragma unroll
          for (int u = 0; u < kPatch; ++u) {
            const int ch = lane + 32 * u;
            if (ch < 2 * (D / 8)) {
              const bool isv = ch >= D / 8;
              const int d = (ch % (D / 8)) * 8;
              *reinterpret_cast<uint4*>(kt + (isv ? TL::kTileBytes : 0) + swz<D, BS>(tl, d)) = pv[u];
            }
          }
          fence_proxy_async_smem();  // the stage is TMA-written again later
          __syncwarp();
        }
        if constexpr (F8) {
          if (patch8) {
            float sk, sv;
            const uint32_t ck = quantize4_e4m3<T>(pk8, sk), cv = quantize4_e4m3<T>(pv8, sv);
            *reinterpret_cast<uint32_t*>(kt + swz8<TT>(tl, lane * 4)) = ck;
            *reinterpret_cast<uint32_t*>(kt + TL::kTileBytes + swz8<TT>(tl, lane * 4)) = cv;
            if (lane == 0) {
              scales[s * 2 * kScaleSlot + tl] = sk;
              scales[(s * 2 + 1) * kScaleSlot + tl] = sv;
            }
            fence_proxy_async_smem();  // the stage and its scales are written by the async proxy again later
            __syncwarp();
          }
        }
        if constexpr (F8)
          consume_tile_f8<D, TT, NG>(st, kt, kt + TL::kTileBytes, scales + s * 2 * kScaleSlot,
                                     scales + (s * 2 + 1) * kScaleSlot, c.blk * TT, L, sl2, lane);
        else
          consume_tile<T, D, TT, NG, BS>(st, kt, kt + TL::kTileBytes, c.blk * TT, L, sl2, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }
    if (j == n - 1 || c.blk + 1 == c.nb) {
      // ---- end of this CTA's segment of unit (b, kvh): merge the 4 warps ----
      const int64_t unit_end = unit_start + c.nb;
      const bool whole = unit_start >= t0 && unit_end <= t1;
      const int slot = unit_start < t0 ? 0 : 1;
      // the owner's own piece stays in the merge buffer for its combine
      const bool keep = kPrefetchParts && j == n - 1 && !whole && slot == 1;
      // Two merge buffers alternate between segments.  Each warp stores its
      // state and counts itself in; the last of the four merges the segment
      // while the others go on to their next tiles, then frees the buffer,
      // which the segment two later waits for before storing into it.
      const int mb = seg & 1;
      float* Os = merge_base + mb * kMergeFloats;
      float* Ms = Os + kConsumers * merge_row<D>() * GP;
      float* Ls = Ms + kConsumers * GP;
      if (seg >= 2) {
        int w = 1;
        if (lane == 0) w = mbar_wait_for(&seg_free[mb], ((seg >> 1) - 1) & 1, p.wait_limit_ns);
        if (!__shfl_sync(0xffffffffu, w, 0)) ok = 0;
      }
      ++seg;
      if constexpr (F8) store_state_f8(st, Os, Ms, Ls, cw, lane);
      else store_state(st, Os, Ms, Ls, cw, lane);
      __syncwarp();
      int arrived = 0;
      if (lane == 0) {
        __threadfence_block();  // this warp's state before its count
        arrived = atomicAdd(&seg_cnt[mb], 1);
        if (arrived == kConsumers - 1) seg_cnt[mb] = 0;
        __threadfence_block();  // the other warps' states after their counts
      }
      arrived = __shfl_sync(0xffffffffu, arrived, 0);
      if (arrived == kConsumers - 1 && !keep) {
        __syncwarp();  // lane 0's acquire, before every lane's reads
        // each lane merges four adjacent outputs of one head at a time (float4 reads)
        constexpr int kD4 = D / 4, DP = merge_row<D>();
        for (int v = lane; v < G * kD4; v += 32) {
          const int g = v / kD4, d = (v - g * kD4) * 4;
          float mx = -INFINITY;
#pragma unroll
          for (int w2 = 0; w2 < kConsumers; ++w2) mx = fmaxf(mx, Ms[w2 * GP + g]);
          float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
          float den = 0.f;
          if (mx != -INFINITY) {
#pragma unroll
            for (int w2 = 0; w2 < kConsumers; ++w2) {
              const float mw = Ms[w2 * GP + g];
              if (mw == -INFINITY) continue;
              const float sc = fast_exp2(mw - mx);
              const float4 o4 = *reinterpret_cast<const float4*>(Os + (w2 * GP + g) * DP + d);
              num.x += sc * o4.x;
              num.y += sc * o4.y;
              num.z += sc * o4.z;
              num.w += sc * o4.w;
              den += sc * Ls[w2 * GP + g];
            }
          }
          if (whole) {
            const float inv = den > 0.f ? 1.f / den : 0.f;
            T* o = static_cast<T*>(p.out) + (static_cast<int64_t>(c.b) * p.num_heads + c.kvh * G + g) * D + d;
            o[0] = DType<T>::from_float(num.x * inv);
            o[1] = DType<T>::from_float(num.y * inv);
            o[2] = DType<T>::from_float(num.z * inv);
            o[3] = DType<T>::from_float(num.w * inv);
          } else {
            const int64_t r = (static_cast<int64_t>(pid) * 2 + slot) * G + g;
            *reinterpret_cast<float4*>(p.ws_o + r * D + d) = num;
            if (d == 0) {
              p.ws_ml[r * 2 + 0] = mx;
              p.ws_ml[r * 2 + 1] = den;
            }
          }
        }
        __syncwarp();
        // publish the partial of a unit that started in an earlier CTA: the
        // warp's stores precede the release of the flag
        if (!whole && slot == 0 && lane == 0) st_release_gpu(p.ws_flags + pid, p.epoch);
        if (lane == 0) mbar_arrive(&seg_free[mb]);
      }
      if (j + 1 < n) {
        advance(c);
        unit_start = static_cast<int64_t>(Hkv) * CB[c.b] + static_cast<int64_t>(c.kvh) * c.nb;
        L = checked_len(p, c.b);
        nrow = new_row_of(c.b);
        if constexpr (kPrefetchQ) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
            for (int ng = 0; ng < NG; ++ng) {
              st.qf[kk][ng][0] = qn[kk][ng][0];
              st.qf[kk][ng][1] = qn[kk][ng][1];
            }
          prefetch_next(c, unit_start);
        } else if constexpr (F8) {
          load_q_frags_f8<T, D, NG>(st.qf, q_of(c), G, lane);
        } else {
          load_q<T, D, NG>(st, q_of(c), G, lane);
        }
        reset_state(st);
      }
    } else {
      advance(c);
    }
  }
  int last;
  if (!owner_of(c, last)) return;
  const int npre = npre_of(last);

  // ---- owner: combine this CTA's piece with the later pieces ----
  const float* Os = merge_base + ((seg - 1) & 1) * kMergeFloats;
  const float* Ms = Os + kConsumers * merge_row<D>() * GP;
  const float* Ls = Ms + kConsumers * GP;
  // Pieces read from global memory: CTAs qs..last (this CTA's own slot-1
  // row first when its piece was not kept in shared memory).
  const int qs = kPrefetchParts ? pid + 1 + npre : pid;
  const int nrest = last - qs + 1, nrest_pad = (nrest + 7) & ~7;
  if (!kPrefetchParts && cw == 0) {
    // wait for the later pieces' ready flags (bounded) and clear them: each
    // flag has this one reader, so flags are zero between calls even when a
    // replayed launch reuses its epoch
    for (int q = pid + 1 + lane; q <= last; q += 32) {
      if (static_cast<int64_t>(q) * Wc / P != static_cast<int64_t>(q + 1) * Wc / P) {
        const uint64_t t_start = globaltimer_ns();
        while (ld_acquire_gpu(p.ws_flags + q) != p.epoch) {
          if (globaltimer_ns() - t_start > p.wait_limit_ns) {
            record_error(KV_ERR_DEVICE_TIMEOUT);
            break;
          }
          __nanosleep(32);
        }
        p.ws_flags[q] = 0;
      }
    }
  }
  for (int k = ctid; k < nrest_pad; k += kConsumers * 32) {
    const int q = qs + k;
    int row = -1;
    if (k < nrest) {
      if (q == pid) row = (pid * 2 + 1) * G;
      else if (static_cast<int64_t>(q) * Wc / P != static_cast<int64_t>(q + 1) * Wc / P) row = q * 2 * G;
    }
    part_row[k] = row;
  }
  if (kPrefetchParts) {
    if (lane == 0) mbar_wait_for(pre_bar, 0, p.wait_limit_ns);
    __syncwarp();
  }
  named_barrier_sync(1, kConsumers * 32);
  // A thread takes up to 4 outputs at once and issues all their loads of a
  // batch of 8 pieces before using any, so a batch costs one round trip.
  T* o = static_cast<T*>(p.out) + (static_cast<int64_t>(c.b) * p.num_heads + c.kvh * G) * D;
  constexpr int kOut = 4, kParts = 8, kStride = kConsumers * 32;
  for (int base = ctid; base < G * D; base += kStride * kOut) {
    float mx[kOut], num[kOut], den[kOut];
    int gi[kOut], di[kOut];
#pragma unroll
    for (int i = 0; i < kOut; ++i) {
      const int idx = min(base + i * kStride, G * D - 1);
      gi[i] = idx / D;
      di[i] = idx - gi[i] * D;
      if (kPrefetchParts) {
        warp_merge<D, GP>(Os, Ms, Ls, gi[i], di[i], mx[i], num[i], den[i]);
      } else {
        mx[i] = -INFINITY;
        num[i] = den[i] = 0.f;
      }
    }
    auto add = [&](int i, float m2, float l2, float a2) {
      if (m2 == -INFINITY) return;
      const float nm = fmaxf(mx[i], m2);
      const float so = fast_exp2(mx[i] - nm), sn = fast_exp2(m2 - nm);
      num[i] = num[i] * so + sn * a2;
      den[i] = den[i] * so + sn * l2;
      mx[i] = nm;
    };
    for (int u = 0; u < npre; ++u) {
      const float* po = reinterpret_cast<const float*>(pre_part(u));
      const float* pml = reinterpret_cast<const float*>(pre_part(u) + part_o);
#pragma unroll
      for (int i = 0; i < kOut; ++i) add(i, pml[gi[i] * 2], pml[gi[i] * 2 + 1], po[gi[i] * D + di[i]]);
    }
    for (int k0 = 0; k0 < nrest_pad; k0 += kParts) {
      float mk[kOut][kParts], lk[kOut][kParts], ak[kOut][kParts];
#pragma unroll
      for (int u = 0; u < kParts; ++u) {
        const int rb = part_row[k0 + u];
#pragma unroll
        for (int i = 0; i < kOut; ++i) {
          const int64_t r = rb + gi[i];
          mk[i][u] = rb >= 0 ? __ldcg(p.ws_ml + r * 2) : -INFINITY;
          lk[i][u] = rb >= 0 ? __ldcg(p.ws_ml + r * 2 + 1) : 0.f;
          ak[i][u] = rb >= 0 ? __ldcg(p.ws_o + r * D + di[i]) : 0.f;
        }
      }
#pragma unroll
      for (int i = 0; i < kOut; ++i)
#pragma unroll
        for (int u = 0; u < kParts; ++u) add(i, mk[i][u], lk[i][u], ak[i][u]);
    }
#pragma unroll
    for (int i = 0; i < kOut; ++i) {
      const int idx = base + i * kStride;
      if (idx < G * D) o[idx] = DType<T>::from_float(den[i] > 0.f ? num[i] / den[i] : 0.f);
    }
  }
}

// =========================================================================
// Split tensor-core kernel: one CTA per (split, kv head, sequence).  Used
// when the stream-K kernel's shared memory would not fit: more than
// kMaxSkSeqs sequences, or head_dim 256 with more than 8 query heads per kv
// head (stage ring plus double-buffered warp merge area).
// =========================================================================

constexpr int kMaxSkSeqs = 4096;

template <typename T, int D, int BS, int NG, int NST>
struct SplitCfg {
  using TL = Tile<D, BS>;
  static constexpr int kStages = NST * TL::kStageBytes;
  static constexpr int kMerge = MergeArea<D, NG>::kBytes;
  static constexpr int kData = kStages > kMerge ? kStages : kMerge;
  static constexpr int kSmem = 1024 + kData + 2 * NST * 8;
};

template <typename T, int D, int BS, int NG, int NST>
__global__ void __launch_bounds__(kTcThreads)
decode_split_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV) {
  using C = SplitCfg<T, D, BS, NG, NST>;
  using TL = Tile<D, BS>;
  constexpr int GP = 8 * NG;
  static_assert(NST % kConsumers == 0, "stage s must always be drained by consumer s % kConsumers");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kData);
  uint64_t* empty = full + NST;

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int L = checked_len(p, b);
  const int nblk = (L + BS - 1) / BS;
  const int bps = p.blocks_per_split;
  const int nsplit_b = (nblk + bps - 1) / bps;
  if (L == 0) {
    if (split == 0) store_zero_rows<T>(p, b, kvh * G, G, D, threadIdx.x, kTcThreads);
    return;
  }
  if (split >= nsplit_b) return;
  const int blk0 = split * bps;
  const int nb = min(nblk - blk0, bps);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
    }
    const int32_t* row = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq + blk0;
    int32_t mine = 0;
    int ok = 1, issued = 0;
    for (int j = 0; j < nb && ok; ++j) {
      if ((j & 31) == 0) mine = (j + lane < nb) ? __ldg(row + j + lane) : 0;
      int pb = __shfl_sync(0xffffffffu, mine, j & 31);
      if (lane == 0) {
        const int s = j % NST;
        if (j >= NST) ok = mbar_wait_bounded(&empty[s], ((j / NST) - 1) & 1);
        if (ok) {
          if (pb < 0 || pb >= p.num_blocks) {
            record_error(KV_ERR_DEVICE_BOUNDS);
            pb = 0;
          }
          mbar_arrive_expect_tx(&full[s], TL::kStageBytes);
          uint8_t* kt = smem + s * TL::kStageBytes;
          uint8_t* vt = kt + TL::kTileBytes;
#pragma unroll
          for (int c = 0; c < TL::kSub; ++c) {
            tma_load_3d(kt + c * TL::kSlabBytes, &tmK, &full[s], c * 64, kvh, pb * BS);
            tma_load_3d(vt + c * TL::kSlabBytes, &tmV, &full[s], c * 64, kvh, pb * BS);
          }
          ++issued;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0) {
      for (int s = 0; s < NST && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / NST) * NST;
        mbar_wait_bounded(&full[s], (last / NST) & 1);
      }
    }
    return;
  }

  const int cw = warp - 1, ctid = threadIdx.x - 32;
  WarpState<D, NG> st;
  load_q<T, D, NG>(st, static_cast<const T*>(p.q) + (static_cast<int64_t>(b) * p.num_heads + kvh * G) * D, G,
                   lane);
  reset_state(st);
  for (int j = cw; j < nb; j += kConsumers) {
    const int s = j % NST;
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(&full[s], (j / NST) & 1);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    __syncwarp();
    uint8_t* kt = smem + s * TL::kStageBytes;
    consume_tile<T, D, BS, NG>(st, kt, kt + TL::kTileBytes, (blk0 + j) * BS, L, p.scale_log2, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  named_barrier_sync(1, kConsumers * 32);  // all stages consumed: reuse them for the merge
  float* Os = reinterpret_cast<float*>(smem);
  float* Ms = Os + kConsumers * merge_row<D>() * GP;
  float* Ls = Ms + kConsumers * GP;
  store_state(st, Os, Ms, Ls, cw, lane);
  named_barrier_sync(1, kConsumers * 32);
  combine_and_store<T>(p, Ms, Ls, Os, kConsumers, GP, merge_row<D>(), D, b, kvh * G, G, split, nsplit_b == 1,
                       ctid, kConsumers * 32);
}

// =========================================================================
// SIMT kernel: any dtype / head_dim (multiple of 4, <= 256) / block size.
// =========================================================================

constexpr int kSimtWarps = 4;
constexpr int kSimtHeads = 8;  // query heads per CTA (a group is split across CTAs beyond this)

template <typename T, int DPL>
__global__ void __launch_bounds__(kSimtWarps * 32) decode_simt_kernel(const DecodeParams p) {
  constexpr int GM = kSimtHeads;
  __shared__ float Os[kSimtWarps * 32 * DPL * GM];
  __shared__ float Ms[kSimtWarps * GM], Ls[kSimtWarps * GM];

  const int D = p.head_dim, BS = p.block_size, G = p.group;
  const int ngroups = (G + GM - 1) / GM;
  const int split = blockIdx.x, kvh = blockIdx.y / ngroups, hg = blockIdx.y % ngroups, b = blockIdx.z;
  const int g0 = hg * GM, gn = min(GM, G - g0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = checked_len(p, b);
  const int nblk = (L + BS - 1) / BS;
  const int bps = p.blocks_per_split;
  const int nsplit_b = (nblk + bps - 1) / bps;
  if (L == 0) {
    if (split == 0) store_zero_rows<T>(p, b, kvh * G + g0, gn, D, threadIdx.x, kSimtWarps * 32);
    return;
  }
  if (split >= nsplit_b) return;
  const int blk0 = split * bps;
  const int nb = min(nblk - blk0, bps);

  float qv[GM][DPL], acc[GM][DPL], mrun[GM], lrun[GM];
  const T* qb = static_cast<const T*>(p.q) + (static_cast<int64_t>(b) * p.num_heads + kvh * G + g0) * D;
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    mrun[g] = -INFINITY;
    lrun[g] = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      const int d = lane + 32 * i;
      qv[g][i] = (g < gn && d < D) ? DType<T>::to_float(qb[g * D + d]) : 0.f;
      acc[g][i] = 0.f;
    }
  }
  const T* kc = static_cast<const T*>(p.k_cache);
  const T* vc = static_cast<const T*>(p.v_cache);
  const int32_t* row = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq + blk0;
  for (int j = warp; j < nb; j += kSimtWarps) {
    const int pb = __ldg(row + j);
    if (pb < 0 || pb >= p.num_blocks) {
      if (lane == 0) record_error(KV_ERR_DEVICE_BOUNDS);
      continue;
    }
    const int ntok = min(BS, L - (blk0 + j) * BS);
    for (int o = 0; o < ntok; ++o) {
      const int64_t base = ((static_cast<int64_t>(pb) * BS + o) * p.num_kv_heads + kvh) * D;
      float kd[DPL], vd[DPL];
#pragma unroll
      for (int i = 0; i < DPL; ++i) {
        const int d = lane + 32 * i;
        kd[i] = d < D ? DType<T>::to_float(kc[base + d]) : 0.f;
        vd[i] = d < D ? DType<T>::to_float(vc[base + d]) : 0.f;
      }
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        if (g < gn) {
          float sdot = 0.f;
#pragma unroll
          for (int i = 0; i < DPL; ++i) sdot = fmaf(qv[g][i], kd[i], sdot);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) sdot += __shfl_xor_sync(0xffffffffu, sdot, off);
          const float x = sdot * p.scale_log2;
          const float mn = fmaxf(mrun[g], x);
          const float al = fast_exp2(mrun[g] - mn), pw = fast_exp2(x - mn);
          lrun[g] = lrun[g] * al + pw;
#pragma unroll
          for (int i = 0; i < DPL; ++i) acc[g][i] = fmaf(acc[g][i], al, pw * vd[i]);
          mrun[g] = mn;
        }
      }
    }
  }
  // per-warp states -> shared memory; layout Os[w][d][g] with d < 32 * DPL
  const int DP = 32 * DPL;
#pragma unroll
  for (int g = 0; g < GM; ++g) {
#pragma unroll
    for (int i = 0; i < DPL; ++i) Os[(warp * DP + lane + 32 * i) * GM + g] = acc[g][i];
    if (lane == 0) {
      Ms[warp * GM + g] = mrun[g];
      Ls[warp * GM + g] = lrun[g];
    }
  }
  __syncthreads();
  // combine_and_store indexes Os as [w][d][g] with row length D: use DP rows
  for (int idx = threadIdx.x; idx < gn * D; idx += kSimtWarps * 32) {
    const int g = idx / D, d = idx - g * D;
    float mx = -INFINITY;
    for (int w = 0; w < kSimtWarps; ++w) mx = fmaxf(mx, Ms[w * GM + g]);
    float num = 0.f, den = 0.f;
    if (mx != -INFINITY)
      for (int w = 0; w < kSimtWarps; ++w) {
        const float mw = Ms[w * GM + g];
        if (mw == -INFINITY) continue;
        const float sc = fast_exp2(mw - mx);
        num += sc * Os[(w * DP + d) * GM + g];
        den += sc * Ls[w * GM + g];
      }
    const int qh = kvh * G + g0 + g;
    if (nsplit_b == 1) {
      T* o = static_cast<T*>(p.out) + (static_cast<int64_t>(b) * p.num_heads + qh) * D + d;
      *o = DType<T>::from_float(den > 0.f ? num / den : 0.f);
    } else {
      const int64_t r = (static_cast<int64_t>(b) * p.num_heads + qh) * p.num_splits + split;
      p.ws_o[r * D + d] = num;
      if (d == 0) {
        p.ws_ml[r * 2 + 0] = mx;
        p.ws_ml[r * 2 + 1] = den;
      }
    }
  }
}

// =========================================================================
// Log-sum-exp merge of split partials: one warp per (sequence, query head).
// M = max_s m_s;  out = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s.
// =========================================================================

constexpr int kMergeWarps = 4;

template <typename T>
__global__ void __launch_bounds__(kMergeWarps * 32) lse_merge_kernel(const DecodeParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp;
  if (idx >= static_cast<int64_t>(p.num_seqs) * p.num_heads) return;
  const int b = static_cast<int>(idx / p.num_heads);
  const int L = checked_len(p, b);
  const int nblk = (L + p.block_size - 1) / p.block_size;
  const int ns = (nblk + p.blocks_per_split - 1) / p.blocks_per_split;
  if (ns <= 1) return;  // written directly by the attention kernel
  const int D = p.head_dim;
  const float* ml = p.ws_ml + idx * p.num_splits * 2;
  const float* po = p.ws_o + idx * p.num_splits * D;
  float mx = -INFINITY;
  for (int s = lane; s < ns; s += 32) mx = fmaxf(mx, ml[2 * s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float den = 0.f;
  for (int s = lane; s < ns; s += 32) den += fast_exp2(ml[2 * s] - mx) * ml[2 * s + 1];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  const float inv = den > 0.f ? 1.f / den : 0.f;
  T* o = static_cast<T*>(p.out) + idx * D;
  for (int d = lane; d < D; d += 32) {
    float num = 0.f;
    for (int s = 0; s < ns; ++s) num += fast_exp2(ml[2 * s] - mx) * po[static_cast<int64_t>(s) * D + d];
    o[d] = DType<T>::from_float(num * inv);
  }
}

// =========================================================================
// Host side: planning, tensor maps, dispatch.
// =========================================================================

enum KernelKind { kSimt = 0, kTensorCoreSplit = 1, kTensorCoreStreamK = 2 };

struct Plan {
  int kind;
  int bps;         // split kernels: logical blocks per split
  int num_splits;  // split kernels: splits per sequence
  int num_ctas;    // stream-K: upper bound of the grid size used to size the workspace
  size_t ws_bytes;
};

constexpr int kMaxSkCtasPerSm = 4;

// Tiles' worth of time one unit boundary costs a stream-K CTA (cross-warp
// merge, output or partial write), at most 4 tiles, measured on GB300:
// about 32 KB of streaming for 16-bit tiles (2 tiles at head_dim 128, 4 at
// head_dim 64) and 48 KB for fp8 tiles, whose consumers take longer per
// tile (charges of 0-6 tiles swept).
int seg_cost_tiles(int stage_bytes, bool fp8) {
  return std::max(1, std::min(4, (fp8 ? 49152 : 32768) / stage_bytes));
}

// Tag of one stream-K call: a per-process random base plus a call counter,
// so a ready flag left by any other call (or uninitialised workspace) does
// not match.
uint64_t next_epoch() {
  static std::atomic<uint64_t> counter{0};
  static const uint64_t base = [] {
    std::random_device rd;
    uint64_t x = (static_cast<uint64_t>(rd()) << 32) ^ rd();
    x ^= static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count()) * 0x9E3779B97F4A7C15ull;
    return x;
  }();
  return base + 2 * (counter.fetch_add(1) + 1);
}

// Stream-K test controls (kv_debug_set), read at each launch.
struct SkControls {
  std::atomic<int64_t> wait_limit_ns{static_cast<int64_t>(kWaitLimitNs)};
  std::atomic<int64_t> skip_tile{-1};
};
SkControls& sk_controls() {
  static SkControls c;
  return c;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

// Pipeline depth: about 64 KB of K+V in flight per CTA, 4..12 stages.
// The stage count must be a multiple of the consumer count: stage s is then
// always drained by consumer s % kConsumers, each consumer meets a stage's
// phases in order, and a parity wait can never be satisfied by a phase one
// round old (with 6 stages and 4 consumers, tile j + 6 would belong to a
// different warp than tile j and could pass its wait before tile j landed).
template <int D, int BS>
struct Stages {
  static constexpr int kRaw = ((64 * 1024) / Tile<D, BS>::kStageBytes) / kConsumers * kConsumers;
  static constexpr int value = kRaw < kConsumers ? kConsumers : (kRaw > 12 ? 12 : kRaw);
  static_assert(value % kConsumers == 0, "stages must be a multiple of the consumer warps");
};

// Shared memory of the stream-K kernel for a batch of B sequences (type
// size 2; the stage count follows the 32-token tile).
template <int D, int BS, int NG>
int sk_smem_for(int B) {
  constexpr int kWant = sk_want_tokens(D, NG, false);
  constexpr int kTileTokens = BS >= kWant ? BS : kWant;
  return SkCfg<__half, D, BS, NG, Stages<D, kTileTokens>::value>::smem_bytes(B);
}

template <int D, int BS>
int sk_smem_ng(int G, int B) {
  return G <= 8 ? sk_smem_for<D, BS, 1>(B) : sk_smem_for<D, BS, 2>(B);
}

int sk_smem_bytes(int D, int BS, int G, int B) {
  if (D == 64) return BS == 16 ? sk_smem_ng<64, 16>(G, B) : sk_smem_ng<64, 32>(G, B);
  if (D == 128) return BS == 16 ? sk_smem_ng<128, 16>(G, B) : sk_smem_ng<128, 32>(G, B);
  return BS == 16 ? sk_smem_ng<256, 16>(G, B) : sk_smem_ng<256, 32>(G, B);
}

int max_smem_optin() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cached[dev] = n > 0 ? n : 48 * 1024;
  }
  return cached[dev];
}

bool tc_supported(int dtype, int D, int BS, int G) {
  return dtype != KV_DTYPE_F32 && (D == 64 || D == 128 || D == 256) && (BS == 16 || BS == 32) && G >= 1 &&
         G <= 16;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Plan make_plan(int B, int Hq, int Hkv, int D, int BS, int64_t max_seq_len, int bps_req, int dtype) {
  Plan pl{};
  const int G = Hkv > 0 ? Hq / Hkv : 1;
  const int64_t maxblk = std::max<int64_t>(1, (max_seq_len + BS - 1) / BS);
  if (tc_supported(dtype, D, BS, G) && bps_req == 0 && B <= kMaxSkSeqs &&
      sk_smem_bytes(D, BS, G, B) <= max_smem_optin()) {
    pl.kind = kTensorCoreStreamK;
    const int64_t w_upper = std::max<int64_t>(1, static_cast<int64_t>(B) * Hkv * maxblk);
    pl.num_ctas = static_cast<int>(std::min<int64_t>(
        std::min<int64_t>(static_cast<int64_t>(sm_count()) * kMaxSkCtasPerSm, kMaxSkCtas), w_upper));
    pl.bps = static_cast<int>(maxblk);
    pl.num_splits = 1;
    const size_t rows = static_cast<size_t>(pl.num_ctas) * 2 * G;
    pl.ws_bytes = align256(rows * D * sizeof(float)) + align256(rows * 2 * sizeof(float)) +
                  align256(static_cast<size_t>(pl.num_ctas) * sizeof(uint64_t));
    return pl;
  }
  pl.kind = tc_supported(dtype, D, BS, G) ? kTensorCoreSplit : kSimt;
  int64_t bps;
  if (bps_req > 0) {
    bps = bps_req;
  } else {
    const int64_t units =
        static_cast<int64_t>(B) * Hkv * (pl.kind == kSimt ? (G + kSimtHeads - 1) / kSimtHeads : 1);
    const int64_t target = static_cast<int64_t>(sm_count()) * 6;
    const int64_t min_bps = std::max<int64_t>(1, 256 / BS);  // >= 256 tokens per split
    if (units >= target || maxblk <= min_bps) {
      bps = maxblk;
    } else {
      const int64_t splits = (target + units - 1) / units;
      bps = std::max<int64_t>((maxblk + splits - 1) / splits, min_bps);
    }
  }
  bps = std::min<int64_t>(bps, maxblk);
  pl.bps = static_cast<int>(bps);
  pl.num_splits = static_cast<int>((maxblk + bps - 1) / bps);
  if (pl.num_splits > 1) {
    const size_t rows = static_cast<size_t>(B) * Hq * pl.num_splits;
    pl.ws_bytes = align256(rows * D * sizeof(float)) + align256(rows * 2 * sizeof(float));
  }
  return pl;
}

// ---- TMA tensor maps -------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Kinds of tensor map: 16-bit cache slabs and fp8 (E4M3) cache slabs.
enum MapKind { kMap16 = 0, kMapFp8 = 1, kMap16Blocks = 2, kMapScales = 3 };

struct MapKey {
  const void* ptr;
  int64_t rows;
  int hkv, d, bs, kind;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && hkv == o.hkv && d == o.d && bs == o.bs && kind == o.kind;
  }
};

// kMap16: the cache as a 3-D tensor {D, Hkv, NB * BS} of 16-bit elements; a
// box {64, 1, BS} is one 128-byte column slab of one block's rows for one
// head.  kMapFp8: the same of 1-byte codes, box {128, 1, BS}.  kMap16Blocks:
// the 16-bit cache as a 4-D tensor {64, NB * BS, D / 64, Hkv} (a column in
// a slab, a token row, a slab, a head; strides Hkv D 2, 128 and D 2 bytes),
// box {64, BS, D / 64, 1}: all of one block's slabs for one head in one
// copy, laid out slab by slab of BS rows of 128 bytes.
bool get_tensor_map(const void* cache, int64_t rows, int hkv, int d, int bs, CUtensorMap* out, int kind = kMap16) {
  static std::mutex mu;
  static MapKey keys[32];
  static CUtensorMap maps[32];
  static int used = 0, next = 0;
  const MapKey key{cache, rows, hkv, d, bs, kind};
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (keys[i] == key) {
      *out = maps[i];
      return true;
    }
  auto fn = encode_fn();
  if (!fn) return false;
  CUtensorMap m;
  CUresult r;
  if (kind == kMapScales) {
    // fp8 scales [NB, Hkv, BS] floats as `rows` rows of bs: a box of one row
    // (the tile gathers four rows per copy)
    cuuint32_t estr[2] = {1, 1};
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(bs), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(bs) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(bs), 1};
    r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(cache), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else if (kind == kMap16Blocks) {
    cuuint32_t estr[4] = {1, 1, 1, 1};
    cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(d / 64),
                          static_cast<cuuint64_t>(hkv)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(hkv) * d * 2, 128, static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[4] = {64, static_cast<cuuint32_t>(bs), static_cast<cuuint32_t>(d / 64), 1};
    r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(cache), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint32_t estr[3] = {1, 1, 1};
    const int es = kind == kMapFp8 ? 1 : 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * es, static_cast<cuuint64_t>(hkv) * d * es};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), 1, static_cast<cuuint32_t>(bs)};
    // L2 fill promotion: 256 bytes for 16-bit caches (one (token, head) row
    // at head_dim 128: the tile's two slabs), 128 bytes for fp8 (one row); a
    // 256-byte fill of an fp8 row also fetches the next head's row, which
    // another CTA reads much later (measured: 10-33 % more DRAM reads)
    r = fn(&m, kind == kMapFp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
           const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B,
           kind == kMapFp8 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return false;
  const int slot = used < 32 ? used++ : (next++ % 32);
  keys[slot] = key;
  maps[slot] = m;
  *out = m;
  return true;
}

// ---- launches ----------------------------------------------------------------


// Raise a kernel's dynamic shared memory limit to `bytes` (per device, only
// when it grows).
template <typename K>
cudaError_t allow_smem(K kern, int bytes, int* configured_bytes) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (configured_bytes[dev] >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) configured_bytes[dev] = bytes;
  return e;
}

// Pipeline depth of the fp8 kernel: about 64 KB of codes in flight per CTA.
template <int D, int TT>
struct Stages8 {
  static constexpr int kRaw = ((64 * 1024) / Tile8<D, TT>::kStageBytes) / kConsumers * kConsumers;
  static constexpr int value = kRaw < kConsumers ? kConsumers : (kRaw > 12 ? 12 : kRaw);
};

template <typename T, int D, int BS, int NG, bool F8 = false>
cudaError_t launch_sk(DecodeParams& p, const CUtensorMap& mk, const CUtensorMap& mv, int max_ctas, cudaStream_t st,
                      const CUtensorMap* mks = nullptr, const CUtensorMap* mvs = nullptr) {
  constexpr int kWant = sk_want_tokens(D, NG, F8);
  constexpr int kTileTokens = BS >= kWant ? BS : kWant;  // matches SkCfg::kTileTokens
  constexpr int NST =
      std::conditional<F8, Stages8<D, kTileTokens>, Stages<D, kTileTokens>>::type::value;
  using C = SkCfg<T, D, BS, NG, NST, F8>;
  auto kern = decode_sk_kernel<T, D, BS, NG, NST, F8>;
  static int configured[64] = {0};
  cudaError_t e = allow_smem(kern, C::smem_bytes(p.num_seqs), configured);
  if (e != cudaSuccess) return e;
  const int smem = C::smem_bytes(p.num_seqs);
  static int occ_cache[64][2] = {{0}};  // per device: (smem bytes, CTAs per SM)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (occ_cache[dev][0] != smem) {
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSkThreads, smem);
    if (e != cudaSuccess) return e;
    occ_cache[dev][0] = smem;
    occ_cache[dev][1] = std::max(1, std::min(occ, kMaxSkCtasPerSm));
  }
  const int ctas = std::min({max_ctas, sm_count() * occ_cache[dev][1], kMaxSkCtas});
  p.num_ctas = ctas;
  p.epoch = next_epoch();
  p.seg_cost = seg_cost_tiles(C::TL::kStageBytes, F8);
  p.wait_limit_ns = static_cast<uint64_t>(sk_controls().wait_limit_ns.load());
  p.test_skip_tile = static_cast<int32_t>(sk_controls().skip_tile.load());
  // Cooperative: the driver refuses the launch unless all CTAs can be
  // resident at once, which the owners' waits on later CTAs rely on.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kSkThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the scale maps are read only by fp8 tiles that gather their scales
  return cudaLaunchKernelEx(&cfg, kern, p, mk, mv, mks ? *mks : mk, mvs ? *mvs : mv);
}

template <typename T, int D, int BS, int NG>
cudaError_t launch_split(const DecodeParams& p, const CUtensorMap& mk, const CUtensorMap& mv, dim3 grid,
                         cudaStream_t st) {
  constexpr int NST = Stages<D, BS>::value;
  using C = SplitCfg<T, D, BS, NG, NST>;
  auto kern = decode_split_kernel<T, D, BS, NG, NST>;
  static int configured[64] = {0};
  cudaError_t e = allow_smem(kern, C::kSmem, configured);
  if (e != cudaSuccess) return e;
  kern<<<grid, kTcThreads, C::kSmem, st>>>(p, mk, mv);
  return cudaGetLastError();
}

template <typename T, int D, int BS, int NG>
cudaError_t launch_tc_inst(DecodeParams& p, const Plan& pl, const CUtensorMap& mk, const CUtensorMap& mv,
                           cudaStream_t st) {
  if (pl.kind == kTensorCoreStreamK) return launch_sk<T, D, BS, NG>(p, mk, mv, pl.num_ctas, st);
  return launch_split<T, D, BS, NG>(p, mk, mv, dim3(pl.num_splits, p.num_kv_heads, p.num_seqs), st);
}

template <typename T, int D, int BS>
cudaError_t launch_tc_g(DecodeParams& p, const Plan& pl, const CUtensorMap& mk, const CUtensorMap& mv,
                        cudaStream_t st) {
  return p.group <= 8 ? launch_tc_inst<T, D, BS, 1>(p, pl, mk, mv, st) : launch_tc_inst<T, D, BS, 2>(p, pl, mk, mv, st);
}

template <typename T, int D>
cudaError_t launch_tc_bs(DecodeParams& p, const Plan& pl, const CUtensorMap& mk, const CUtensorMap& mv,
                         cudaStream_t st) {
  return p.block_size == 16 ? launch_tc_g<T, D, 16>(p, pl, mk, mv, st) : launch_tc_g<T, D, 32>(p, pl, mk, mv, st);
}

template <typename T>
cudaError_t launch_tc(DecodeParams& p, const Plan& pl, const CUtensorMap& mk, const CUtensorMap& mv,
                      cudaStream_t st) {
  switch (p.head_dim) {
    case 64: return launch_tc_bs<T, 64>(p, pl, mk, mv, st);
    case 128: return launch_tc_bs<T, 128>(p, pl, mk, mv, st);
    default: return launch_tc_bs<T, 256>(p, pl, mk, mv, st);
  }
}

template <typename T>
cudaError_t launch_simt(const DecodeParams& p, dim3 grid, cudaStream_t st) {
  const int dpl = (p.head_dim + 31) / 32;
  if (dpl <= 1) decode_simt_kernel<T, 1><<<grid, kSimtWarps * 32, 0, st>>>(p);
  else if (dpl <= 2) decode_simt_kernel<T, 2><<<grid, kSimtWarps * 32, 0, st>>>(p);
  else if (dpl <= 4) decode_simt_kernel<T, 4><<<grid, kSimtWarps * 32, 0, st>>>(p);
  else decode_simt_kernel<T, 8><<<grid, kSimtWarps * 32, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(p.num_seqs) * p.num_heads;
  const unsigned grid = static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps);
  lse_merge_kernel<T><<<grid, kMergeWarps * 32, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t run_decode(DecodeParams& p, const Plan& pl, cudaStream_t st, const CUtensorMap* mk,
                       const CUtensorMap* mv) {
  cudaError_t e = cudaSuccess;
  if constexpr (!std::is_same<T, float>::value) {
    if (pl.kind != kSimt) {
      e = launch_tc<T>(p, pl, *mk, *mv, st);
      if (e != cudaSuccess || pl.kind == kTensorCoreStreamK || pl.num_splits <= 1) return e;
      return launch_merge<T>(p, st);
    }
  }
  const int ngroups = (p.group + kSimtHeads - 1) / kSimtHeads;
  dim3 grid(pl.num_splits, p.num_kv_heads * ngroups, p.num_seqs);
  e = launch_simt<T>(p, grid, st);
  if (e != cudaSuccess || pl.num_splits <= 1) return e;
  return launch_merge<T>(p, st);
}

// Host-side argument checks shared by the plan query and the launch.
int check_shapes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t BS, int64_t max_seq_len, int dtype) {
  if (dtype != KV_DTYPE_F32 && dtype != KV_DTYPE_F16 && dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || BS <= 0 || max_seq_len < 0) return KV_ERR_INVALID_ARG;
  if (D <= 0 || D > 256) return KV_ERR_INVALID_ARG;
  if (dtype == KV_DTYPE_F32 ? (D % 4 != 0) : (D % 8 != 0)) return KV_ERR_INVALID_ARG;
  if (max_seq_len > INT32_MAX) return KV_ERR_INVALID_ARG;
  return KV_OK;
}

}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

extern "C" int pagedkv_internal_reshape_error(int reset, int* code);
extern "C" int pagedkv_internal_prefill_error(int reset, int* code);
extern "C" int paged_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                       const int32_t* slot_mapping, int64_t num_tokens, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                       int64_t k_token_stride, int64_t v_token_stride, int dtype, void* stream);

extern "C" int paged_decode_plan(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int64_t max_seq_len, int32_t blocks_per_split, int dtype,
                                 int32_t* kernel_out, int32_t* blocks_per_split_out, int32_t* num_splits_out,
                                 size_t* workspace_bytes_out) {
  int st = check_shapes(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_seq_len, dtype);
  if (st != KV_OK) return st;
  if (blocks_per_split < 0) return KV_ERR_INVALID_ARG;
  Plan pl = make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_seq_len, blocks_per_split, dtype);
  if (kernel_out) *kernel_out = pl.kind;
  if (blocks_per_split_out) *blocks_per_split_out = pl.bps;
  if (num_splits_out) *num_splits_out = pl.num_splits;
  if (workspace_bytes_out) *workspace_bytes_out = pl.ws_bytes;
  return KV_OK;
}

extern "C" int paged_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                           int32_t head_dim, int32_t block_size, int64_t max_seq_len,
                                           int32_t blocks_per_split, int dtype, size_t* bytes_out) {
  if (!bytes_out) return KV_ERR_INVALID_ARG;
  return paged_decode_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_seq_len, blocks_per_split,
                           dtype, nullptr, nullptr, nullptr, bytes_out);
}

namespace {
// The step's new tokens for paged_decode_step (null for attention alone).
struct StepArgs {
  const void* k;
  const void* v;
  const int32_t* slot_mapping;
  const int32_t* new_token_row;
  int64_t num_tokens, k_stride, v_stride;  // strides in elements
};

int decode_impl(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq, int64_t max_seq_len, float scale,
                int32_t blocks_per_split, int dtype, void* workspace, size_t workspace_bytes, void* stream,
                const StepArgs* step) {
  int st = check_shapes(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_seq_len, dtype);
  if (st != KV_OK) return st;
  if (num_blocks <= 0 || num_blocks > INT32_MAX / block_size || max_blocks_per_seq <= 0 || blocks_per_split < 0)
    return KV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return KV_ERR_INVALID_ARG;
  if (num_seqs == 0) return KV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return KV_ERR_INVALID_ARG;
  const uintptr_t align_bits = reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(q) |
                               reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache);
  if (align_bits % 16 != 0) return KV_ERR_INVALID_ARG;
  Plan pl = make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_seq_len, blocks_per_split, dtype);
  if (pl.ws_bytes > 0) {
    if (!workspace || workspace_bytes < pl.ws_bytes) return KV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return KV_ERR_INVALID_ARG;
  }
  DecodeParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.scale_log2 = scale * kLog2e;
  char* ws = static_cast<char*>(workspace);
  if (pl.kind == kTensorCoreStreamK) {
    // lengths are bounded by the table rows only; the grid adapts to them
    p.blocks_per_split = max_blocks_per_seq;
    p.num_splits = 1;
    const size_t rows = static_cast<size_t>(pl.num_ctas) * 2 * p.group;
    p.ws_o = reinterpret_cast<float*>(ws);
    p.ws_ml = reinterpret_cast<float*>(ws + align256(rows * head_dim * sizeof(float)));
    p.ws_flags = reinterpret_cast<uint64_t*>(ws + align256(rows * head_dim * sizeof(float)) +
                                             align256(rows * 2 * sizeof(float)));
  } else {
    p.blocks_per_split = pl.bps;
    p.num_splits = pl.num_splits;
    if (pl.ws_bytes > 0) {
      const size_t rows = static_cast<size_t>(num_seqs) * num_heads * pl.num_splits;
      p.ws_o = reinterpret_cast<float*>(ws);
      p.ws_ml = reinterpret_cast<float*>(ws + align256(rows * head_dim * sizeof(float)));
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (step != nullptr && step->num_tokens > 0) {
    const int64_t es = static_cast<int64_t>(dtype_bytes(dtype));
    const uintptr_t row_align = reinterpret_cast<uintptr_t>(step->k) | reinterpret_cast<uintptr_t>(step->v) |
                                static_cast<uintptr_t>(step->k_stride * es) |
                                static_cast<uintptr_t>(step->v_stride * es);
    if (pl.kind == kTensorCoreStreamK && row_align % 16 == 0) {
      // one launch: the stream-K kernel also writes the new rows
      p.new_k = step->k;
      p.new_v = step->v;
      p.slot_mapping = step->slot_mapping;
      p.new_row = step->new_token_row;
      p.num_new = step->num_tokens;
      p.new_k_stride = step->k_stride * es;
      p.new_v_stride = step->v_stride * es;
    }
  }
  CUtensorMap mk, mv;
  if (pl.kind != kSimt) {
    const int64_t rows = num_blocks * block_size;
    // the stream-K kernel copies whole blocks (all slabs) at once; the split
    // kernels copy slab by slab
    const int kind = pl.kind == kTensorCoreStreamK ? kMap16Blocks : kMap16;
    if (!get_tensor_map(k_cache, rows, num_kv_heads, head_dim, block_size, &mk, kind) ||
        !get_tensor_map(v_cache, rows, num_kv_heads, head_dim, block_size, &mv, kind))
      return cuda_status(cudaErrorInvalidValue, "cuTensorMapEncodeTiled failed");
  }
  if (step != nullptr && step->num_tokens > 0 && p.new_k == nullptr) {
    // other kernels: the cache write first, then attention, in stream order
    st = paged_reshape_and_cache(step->k, step->v, const_cast<void*>(k_cache), const_cast<void*>(v_cache),
                                 step->slot_mapping, step->num_tokens, num_kv_heads, head_dim, block_size, num_blocks,
                                 step->k_stride, step->v_stride, dtype, stream);
    if (st != KV_OK) return st;
  }
  cudaError_t e;
  if (dtype == KV_DTYPE_F32) e = run_decode<float>(p, pl, s, nullptr, nullptr);
  else if (dtype == KV_DTYPE_F16) e = run_decode<__half>(p, pl, s, &mk, &mv);
  else e = run_decode<__nv_bfloat16>(p, pl, s, &mk, &mv);
  return cuda_status(e);
}
}  // namespace

extern "C" int paged_decode_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, const int32_t* seq_lens, int32_t num_seqs,
                                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq,
                                      int64_t max_seq_len, float scale, int32_t blocks_per_split, int dtype,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, max_blocks_per_seq, max_seq_len, scale, blocks_per_split, dtype,
                     workspace, workspace_bytes, stream, nullptr);
}

extern "C" int paged_decode_step(void* out, const void* q, const void* k, const void* v,
                                 const int32_t* slot_mapping, int64_t num_tokens, int64_t k_token_stride,
                                 int64_t v_token_stride, const int32_t* new_token_row, void* k_cache,
                                 void* v_cache, const int32_t* block_tables, const int32_t* seq_lens,
                                 int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq,
                                 int64_t max_seq_len, float scale, int dtype, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (num_tokens < 0) return KV_ERR_INVALID_ARG;
  if (num_tokens > 0) {
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (!k || !v || !slot_mapping || k_token_stride < row || v_token_stride < row) return KV_ERR_INVALID_ARG;
    if (num_seqs > 0 && !new_token_row) return KV_ERR_INVALID_ARG;
  }
  const StepArgs step{k, v, slot_mapping, new_token_row, num_tokens, k_token_stride, v_token_stride};
  if (num_seqs == 0) {  // nothing to attend: the cache write alone
    return paged_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
                                   block_size, num_blocks, k_token_stride, v_token_stride, dtype, stream);
  }
  return decode_impl(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, max_blocks_per_seq, max_seq_len, scale, 0, dtype, workspace,
                     workspace_bytes, stream, &step);
}

// ---------------------------------------------------------------------------
// Decode attention over fp8 (E4M3) caches with per-token scales.

namespace {
template <typename T>
cudaError_t launch_fp8_decode(DecodeParams& p, const Plan& pl, const CUtensorMap* maps, cudaStream_t st) {
  const bool ng1 = p.group <= 8;
  if (p.block_size == 16)
    return ng1 ? launch_sk<T, 128, 16, 1, true>(p, maps[0], maps[1], pl.num_ctas, st, &maps[2], &maps[3])
               : launch_sk<T, 128, 16, 2, true>(p, maps[0], maps[1], pl.num_ctas, st, &maps[2], &maps[3]);
  return ng1 ? launch_sk<T, 128, 32, 1, true>(p, maps[0], maps[1], pl.num_ctas, st, &maps[2], &maps[3])
             : launch_sk<T, 128, 32, 2, true>(p, maps[0], maps[1], pl.num_ctas, st, &maps[2], &maps[3]);
}
}  // namespace

extern "C" int paged_reshape_and_cache_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                                           float* k_scales, float* v_scales, const int32_t* slot_mapping,
                                           int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                           int32_t block_size, int64_t num_blocks, int64_t k_token_stride,
                                           int64_t v_token_stride, int dtype, void* stream);

namespace {
int decode_fp8_impl(void* out, const void* q, const void* k_cache, const void* v_cache, const float* k_scales,
                    const float* v_scales, const int32_t* block_tables, const int32_t* seq_lens, int32_t num_seqs,
                    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                    int64_t num_blocks, int32_t max_blocks_per_seq, int64_t max_seq_len, float scale, int dtype,
                    void* workspace, size_t workspace_bytes, void* stream, const StepArgs* step) {
  int st = check_shapes(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_seq_len, dtype);
  if (st != KV_OK) return st;
  if (dtype == KV_DTYPE_F32 || head_dim != 128 || (block_size != 16 && block_size != 32) ||
      num_heads / num_kv_heads > 16 || num_seqs > kMaxSkSeqs)
    return KV_ERR_INVALID_ARG;
  if (num_blocks <= 0 || num_blocks > INT32_MAX / block_size || max_blocks_per_seq <= 0) return KV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return KV_ERR_INVALID_ARG;
  if (num_seqs == 0) return KV_OK;
  if (!out || !q || !k_cache || !v_cache || !k_scales || !v_scales || !block_tables || !seq_lens)
    return KV_ERR_INVALID_ARG;
  const uintptr_t align_bits = reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(q) |
                               reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
                               reinterpret_cast<uintptr_t>(k_scales) | reinterpret_cast<uintptr_t>(v_scales);
  if (align_bits % 16 != 0) return KV_ERR_INVALID_ARG;
  Plan pl = make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_seq_len, 0, dtype);
  if (pl.kind != kTensorCoreStreamK) return KV_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < pl.ws_bytes) return KV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return KV_ERR_INVALID_ARG;
  DecodeParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.scale_log2 = scale * kLog2e;
  p.blocks_per_split = max_blocks_per_seq;
  p.num_splits = 1;
  char* ws = static_cast<char*>(workspace);
  const size_t rows = static_cast<size_t>(pl.num_ctas) * 2 * p.group;
  p.ws_o = reinterpret_cast<float*>(ws);
  p.ws_ml = reinterpret_cast<float*>(ws + align256(rows * head_dim * sizeof(float)));
  p.ws_flags = reinterpret_cast<uint64_t*>(ws + align256(rows * head_dim * sizeof(float)) +
                                           align256(rows * 2 * sizeof(float)));
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  bool write_first = false;
  if (step != nullptr && step->num_tokens > 0) {
    const uintptr_t row_align = reinterpret_cast<uintptr_t>(step->k) | reinterpret_cast<uintptr_t>(step->v) |
                                static_cast<uintptr_t>(step->k_stride * 2) | static_cast<uintptr_t>(step->v_stride * 2);
    // One launch when the rows are 8-byte aligned and few: the writer warps
    // (one per CTA) quantise the rows while the consumers stream tiles.  A
    // step with many rows (a prefill chunk: more than 8 per writer warp)
    // runs the write as its own launch, as one writer warp per CTA would
    // outlast the attention (mixed batch: 183 us fused against 128 us).
    const int64_t writer_warps = static_cast<int64_t>(sm_count()) * 2;  // two CTAs per SM
    const bool few_rows = step->num_tokens <= 8 * writer_warps;
    if (row_align % 8 == 0 && few_rows) {  // one launch: the kernel also quantises and writes the new rows
      p.new_k = step->k;
      p.new_v = step->v;
      p.slot_mapping = step->slot_mapping;
      p.new_row = step->new_token_row;
      p.num_new = step->num_tokens;
      p.new_k_stride = step->k_stride * 2;
      p.new_v_stride = step->v_stride * 2;
    } else {
      write_first = true;
    }
  }
  const int64_t slots = num_blocks * block_size;
  CUtensorMap maps[4];
  const int64_t scale_rows = num_blocks * num_kv_heads;
  if (!get_tensor_map(k_scales, scale_rows, 1, 1, block_size, &maps[2], kMapScales) ||
      !get_tensor_map(v_scales, scale_rows, 1, 1, block_size, &maps[3], kMapScales) ||
      !get_tensor_map(k_cache, slots, num_kv_heads, head_dim, block_size, &maps[0], kMapFp8) ||
      !get_tensor_map(v_cache, slots, num_kv_heads, head_dim, block_size, &maps[1], kMapFp8))
    return cuda_status(cudaErrorInvalidValue, "cuTensorMapEncodeTiled failed");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (write_first) {  // rows not 8-byte aligned: the cache write, then attention, in stream order
    st = paged_reshape_and_cache_fp8(step->k, step->v, const_cast<void*>(k_cache), const_cast<void*>(v_cache),
                                     const_cast<float*>(k_scales), const_cast<float*>(v_scales), step->slot_mapping,
                                     step->num_tokens, num_kv_heads, head_dim, block_size, num_blocks, step->k_stride,
                                     step->v_stride, dtype, stream);
    if (st != KV_OK) return st;
  }
  const cudaError_t e = dtype == KV_DTYPE_F16 ? launch_fp8_decode<__half>(p, pl, maps, s)
                                              : launch_fp8_decode<__nv_bfloat16>(p, pl, maps, s);
  return cuda_status(e);
}
}  // namespace

extern "C" int paged_decode_attention_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                          const float* k_scales, const float* v_scales, const int32_t* block_tables,
                                          const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads,
                                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                          int64_t num_blocks, int32_t max_blocks_per_seq, int64_t max_seq_len,
                                          float scale, int dtype, void* workspace, size_t workspace_bytes,
                                          void* stream) {
  return decode_fp8_impl(out, q, k_cache, v_cache, k_scales, v_scales, block_tables, seq_lens, num_seqs, num_heads,
                         num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, max_seq_len, scale, dtype,
                         workspace, workspace_bytes, stream, nullptr);
}

extern "C" int paged_decode_step_fp8(void* out, const void* q, const void* k, const void* v,
                                     const int32_t* slot_mapping, int64_t num_tokens, int64_t k_token_stride,
                                     int64_t v_token_stride, const int32_t* new_token_row, void* k_cache,
                                     void* v_cache, float* k_scales, float* v_scales, const int32_t* block_tables,
                                     const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                     int32_t max_blocks_per_seq, int64_t max_seq_len, float scale, int dtype,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (num_tokens < 0) return KV_ERR_INVALID_ARG;
  if (num_tokens > 0) {
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (!k || !v || !slot_mapping || k_token_stride < row || v_token_stride < row) return KV_ERR_INVALID_ARG;
    if (num_seqs > 0 && !new_token_row) return KV_ERR_INVALID_ARG;
  }
  if (num_seqs == 0)  // nothing to attend: the cache write alone
    return paged_reshape_and_cache_fp8(k, v, k_cache, v_cache, k_scales, v_scales, slot_mapping, num_tokens,
                                       num_kv_heads, head_dim, block_size, num_blocks, k_token_stride, v_token_stride,
                                       dtype, stream);
  const StepArgs step{k, v, slot_mapping, new_token_row, num_tokens, k_token_stride, v_token_stride};
  return decode_fp8_impl(out, q, k_cache, v_cache, k_scales, v_scales, block_tables, seq_lens, num_seqs, num_heads,
                         num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, max_seq_len, scale, dtype,
                         workspace, workspace_bytes, stream, &step);
}

// ---------------------------------------------------------------------------
// Decode attention for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: a host process whose GPU memory
// is owned by another allocator (a framework caching allocator or a serving
// runtime that reserves nearly all HBM up front), a plugin interface that
// forbids allocation while it executes, or a latency-critical loop where an
// allocation could synchronise the device.  paged_decode_attention needs a
// caller-provided workspace; this variant instead uses one fixed scratch array
// in device memory that the library defines at file scope, so the call itself
// allocates nothing.
//
// The array is a static __device__ object of kStaticScratchBytes: every GPU
// that loads this library holds it until the process exits.  In host code its
// name is only a host-side stand-in, so the device address is looked up once
// per device (cudaGetSymbolAddress, with that device current) on the first
// call made on it.  All calls on a device share the array and it keeps the
// last call's contents; the kernels write every scratch value they read in the
// same call (the stream-K ready flags carry a per-call tag), so nothing needs
// clearing between calls, but calls that overlap on the GPU race on it.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

namespace {
void* static_scratch_address(int dev, cudaError_t* err) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    *err = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = ptr;
  }
  *err = cudaSuccess;
  return addr[dev];
}
}  // namespace

extern "C" int paged_decode_attention_static_scratch(
    void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq, int64_t max_seq_len, float scale,
    int32_t blocks_per_split, int dtype, void* stream) {
  size_t need = 0;
  int st = paged_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                                       blocks_per_split, dtype, &need);
  if (st != KV_OK) return st;
  if (need > kStaticScratchBytes) return KV_ERR_WORKSPACE;  // beyond the fixed scratch: use the workspace call
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= 64) return KV_ERR_INVALID_ARG;
  void* scratch = static_scratch_address(dev, &e);
  if (!scratch) return cuda_status(e, "cudaGetSymbolAddress of the decode scratch failed");
  return paged_decode_attention(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads, num_kv_heads,
                                head_dim, block_size, num_blocks, max_blocks_per_seq, max_seq_len, scale,
                                blocks_per_split, dtype, scratch, kStaticScratchBytes, stream);
}

extern "C" size_t paged_decode_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" int kv_device_error(int reset, int* status_out) {
  if (!status_out) return KV_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return KV_ERR_CUDA;
  int a = 0, c = 0;
  if (cudaMemcpyFromSymbol(&a, g_device_error, sizeof(int)) != cudaSuccess) return KV_ERR_CUDA;
  if (reset) {
    int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return KV_ERR_CUDA;
  }
  int r = pagedkv_internal_reshape_error(reset, &c);
  if (r != KV_OK) return r;
  int f = 0;
  r = pagedkv_internal_prefill_error(reset, &f);
  if (r != KV_OK) return r;
  *status_out = a ? a : (c ? c : f);
  return KV_OK;
}

extern "C" int kv_debug_set(int key, int64_t value) {
  SkControls& c = sk_controls();
  switch (key) {
    case KV_DEBUG_WAIT_LIMIT_NS:
      c.wait_limit_ns = value > 0 ? value : static_cast<int64_t>(kWaitLimitNs);
      return KV_OK;
    case KV_DEBUG_SKIP_TILE:
      c.skip_tile = value >= 0 ? value : -1;
      return KV_OK;
    default:
      return KV_ERR_INVALID_ARG;
  }
}

extern "C" const char* kv_version(void) { return "pagedkv-gb300 0.1 (sm_103a)"; }

namespace pagedkv {
const char*& last_cuda_error_text() {
  static thread_local const char* text = "no error";
  return text;
}
}  // namespace pagedkv

extern "C" const char* kv_last_cuda_error(void) { return last_cuda_error_text(); }
