// Chunked-prefill attention through block tables.
//
// A sequence's new chunk of n tokens (its last n of L positions, whose K/V
// the cache write has already put in the pool) attends to its whole history
// and, causally, to the chunk: chunk token t at position p = L - n + t sees
// keys 0..p.  "从零实现一个 mini vLLM: Block Manager" (a chunked prefill
// allocates the chunk's slots, writes its K/V, then attends through the
// block table); "MiniPaged-Qwen" §13-§14 (attention over positions read
// through the table, GQA head mapping kvh = qh / (Hq / Hkv)).  A chunk of
// one token is decode.
//
// Two kernels.  prefill_tc_kernel (tcgen05 MMAs into tensor memory, K/V
// tiles by TMA through the table) serves block sizes that divide 128 and
// are multiples of 16; it is described at its definition below.
// prefill_kernel serves the other block sizes, flash-attention style with
// mma.sync: one CTA per (64-token query tile, query head, sequence), four
// warps of 16 query rows.  Key tiles of 32 tokens are gathered through the block table
// with 16-byte cp.async into a double-buffered, 128-byte-swizzled shared
// tile while the previous tile is consumed.  Per tile a warp computes
// S = Q K^T (Q as the A operand from registers, K^T fragments by
// ldmatrix), masks keys past each row's position, updates an fp32 online
// softmax per row in the exp2 domain, and accumulates O += P V with P
// reused from the score registers as the A operand and V fragments by
// ldmatrix.trans.  The output is rounded once to the q dtype.

#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "tcgen05.cuh"

namespace pagedkv {
namespace {

constexpr int kPfWarps = 4;
constexpr int kPfRows = 16 * kPfWarps;  // query tokens (of one head) per CTA
constexpr int kPfKeys = 32;             // keys per shared-memory tile

struct PrefillParams {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* query_start;  // [B + 1]: sequence b's chunk tokens are rows query_start[b] ..
  int32_t num_seqs, num_heads, num_kv_heads, group, block_size;
  int64_t num_blocks;
  int32_t max_blocks_per_seq;
  float scale_log2;  // scale * log2(e)
  int64_t num_tokens;  // rows of q and out
  int32_t hg_log2;     // tensor-core kernel: log2 of the query heads per row tile
  int32_t row_tiles;   // tensor-core kernel: row tiles per (sequence, head group) in the grid
};

// Byte offset of (key, dim) in a [kPfKeys][D] 16-bit tile: 128-byte slabs of
// 64 dims, 16-byte chunks XOR-swizzled by key % 8 (conflict-free ldmatrix).
__device__ __forceinline__ uint32_t pf_off(int key, int d) {
  return static_cast<uint32_t>((d >> 6) * (kPfKeys * 128) + key * 128 + ((((d & 63) >> 3) ^ (key & 7)) << 4) +
                               (d & 7) * 2);
}

// 16-byte async copy; with valid == false nothing is read and zeros land.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T, int D>
__global__ void __launch_bounds__(kPfWarps * 32) prefill_kernel(const PrefillParams p) {
  using M = Mma<T>;
  constexpr int KS = D / 16;                 // k-steps of Q K^T over head_dim
  constexpr int kTile = kPfKeys * D * 2;     // bytes of one K or V tile
  constexpr int kChunks = kPfKeys * (D / 8);  // 16-byte chunks of one tile
  __shared__ __align__(1024) uint8_t sm[2][2][kTile];  // [stage][K, V]

  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qs = __ldg(p.query_start + b), n = __ldg(p.query_start + b + 1) - qs;
  // rows past the grid's reach (a chunk longer than max_query_len) would be
  // left uncomputed: the last row tile of the sequence reports it
  if (qt == gridDim.x - 1 && h == 0 && tid == 0 && n > static_cast<int>(gridDim.x) * kPfRows)
    record_error(KV_ERR_DEVICE_BOUNDS);
  if (n <= 0 || qt * kPfRows >= n) return;
  if (qs < 0 || qs + n > p.num_tokens) {  // the chunk's rows must lie inside q
    if (tid == 0) record_error(KV_ERR_DEVICE_BOUNDS);
    return;
  }
  int L = __ldg(p.seq_lens + b);
  const int64_t cap = static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size;
  if (L < n || L > cap) {  // the chunk must lie inside the sequence and its table
    if (tid == 0) record_error(KV_ERR_DEVICE_BOUNDS);
    if (L > cap) L = static_cast<int>(cap);
    if (L < n) return;
  }
  const int ctx = L - n, kvh = h / p.group;
  const int g = lane >> 2, t2 = (lane & 3) * 2;
  const int row0 = qt * kPfRows + warp * 16;  // this warp's first chunk token
  const int64_t stride = static_cast<int64_t>(p.num_heads) * D;

  // Q as the A operand: rows row0 + g and row0 + g + 8, dims kk*16 + t2 (+1), + 8
  uint32_t qa[KS][4];
  {
    const T* qb = static_cast<const T*>(p.q) + static_cast<int64_t>(qs) * stride + static_cast<int64_t>(h) * D;
    const bool vlo = row0 + g < n, vhi = row0 + g + 8 < n;
    const T* qlo = qb + static_cast<int64_t>(row0 + g) * stride;
    const T* qhi = qlo + 8 * stride;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int d = kk * 16 + t2;
      qa[kk][0] = vlo ? __ldg(reinterpret_cast<const uint32_t*>(qlo + d)) : 0u;
      qa[kk][1] = vhi ? __ldg(reinterpret_cast<const uint32_t*>(qhi + d)) : 0u;
      qa[kk][2] = vlo ? __ldg(reinterpret_cast<const uint32_t*>(qlo + d + 8)) : 0u;
      qa[kk][3] = vhi ? __ldg(reinterpret_cast<const uint32_t*>(qhi + d + 8)) : 0u;
    }
  }
  // keys the CTA needs: 0 .. position of its last row
  const int last_row = min(n, (qt + 1) * kPfRows) - 1;
  const int nkeys = ctx + last_row + 1;
  const int ntiles = (nkeys + kPfKeys - 1) / kPfKeys;

  auto load_tile = [&](int kt, int stage) {
    for (int c = tid; c < 2 * kChunks; c += kPfWarps * 32) {
      const int which = c / kChunks, cc = c - which * kChunks;
      const int key = cc / (D / 8), d = (cc % (D / 8)) * 8;
      const int j = kt * kPfKeys + key;
      const bool valid = j < nkeys;
      const T* src = static_cast<const T*>(which ? p.v_cache : p.k_cache);
      if (valid) {
        int pb = __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq + j / p.block_size);
        if (pb < 0 || pb >= p.num_blocks) {
          record_error(KV_ERR_DEVICE_BOUNDS);
          pb = 0;
        }
        const int64_t row = static_cast<int64_t>(pb) * p.block_size + j % p.block_size;
        src += (row * p.num_kv_heads + kvh) * D + d;
      }
      cp_async16(smem_u32(&sm[stage][which][0]) + pf_off(key, d), src, valid);
    }
    cp_async_commit();
  };

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;  // l: this lane's partial row sums
  const int pos_lo = ctx + row0 + g, pos_hi = pos_lo + 8;
  // ldmatrix x4 lane -> matrix m = lane / 8, row lane % 8
  const int lm = lane >> 3, lr = lane & 7;

  load_tile(0, 0);
  for (int kt = 0; kt < ntiles; ++kt) {
    if (kt + 1 < ntiles) {
      load_tile(kt + 1, (kt + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t kb = smem_u32(&sm[kt & 1][0][0]), vb = smem_u32(&sm[kt & 1][1][0]);
    // S[16 rows x 32 keys] = Q K^T, four n8 blocks of keys
    float s[4][4];
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk)
#pragma unroll
      for (int nb = 0; nb < 4; nb += 2) {
        uint32_t r0, r1, r2, r3;  // (keys nb*8.., dims kk*16 + 0/8), (keys (nb+1)*8.., dims + 0/8)
        ldmatrix_x4(kb + pf_off((nb + (lm >> 1)) * 8 + lr, kk * 16 + (lm & 1) * 8), r0, r1, r2, r3);
        M::run(s[nb], qa[kk], r0, r1);
        M::run(s[nb + 1], qa[kk], r2, r3);
      }
    // mask keys past each row's position; online softmax in the exp2 domain
    float x[4][4];
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      const int j = kt * kPfKeys + nb * 8 + t2;
      x[nb][0] = j <= pos_lo ? s[nb][0] * p.scale_log2 : -INFINITY;
      x[nb][1] = j + 1 <= pos_lo ? s[nb][1] * p.scale_log2 : -INFINITY;
      x[nb][2] = j <= pos_hi ? s[nb][2] * p.scale_log2 : -INFINITY;
      x[nb][3] = j + 1 <= pos_hi ? s[nb][3] * p.scale_log2 : -INFINITY;
      mx_lo = fmaxf(mx_lo, fmaxf(x[nb][0], x[nb][1]));
      mx_hi = fmaxf(mx_hi, fmaxf(x[nb][2], x[nb][3]));
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, off));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, off));
    }
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float mu_lo = mn_lo == -INFINITY ? 0.f : mn_lo, mu_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
    const float al_lo = fast_exp2(m_lo - mu_lo), al_hi = fast_exp2(m_hi - mu_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    uint32_t pa[2][4];  // P as the A operand of two k16 steps over the 32 keys
    float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      const float p0 = fast_exp2(x[nb][0] - mu_lo), p1 = fast_exp2(x[nb][1] - mu_lo);
      const float p2 = fast_exp2(x[nb][2] - mu_hi), p3 = fast_exp2(x[nb][3] - mu_hi);
      sum_lo += p0 + p1;
      sum_hi += p2 + p3;
      pa[nb >> 1][(nb & 1) * 2 + 0] = M::pack(p0, p1);  // row g: a0 (keys 0-7 of the step) or a2 (keys 8-15)
      pa[nb >> 1][(nb & 1) * 2 + 1] = M::pack(p2, p3);  // row g + 8: a1 or a3
    }
    l_lo = l_lo * al_lo + sum_lo;
    l_hi = l_hi * al_hi + sum_hi;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][0] *= al_lo;
      o[i][1] *= al_lo;
      o[i][2] *= al_hi;
      o[i][3] *= al_hi;
    }
    // O[16 x D] += P V: V fragments by ldmatrix.trans, two n8 blocks of dims per x4
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
      for (int db = 0; db < D / 8; db += 2) {
        uint32_t r0, r1, r2, r3;  // (keys ks*16 + 0/8, dims db*8..), (same keys, dims (db+1)*8..)
        ldmatrix_x4_trans(vb + pf_off(ks * 16 + (lm & 1) * 8 + lr, (db + (lm >> 1)) * 8), r0, r1, r2, r3);
        M::run(o[db], pa[ks], r0, r1);
        M::run(o[db + 1], pa[ks], r2, r3);
      }
    __syncthreads();  // every warp is done with this stage before it is loaded again
  }
  // row sums over the quad, normalise, one rounding to the output type
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, off);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, off);
  }
  const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f, inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
  T* ob = static_cast<T*>(p.out) + static_cast<int64_t>(qs) * stride + static_cast<int64_t>(h) * D;
  const bool vlo = row0 + g < n, vhi = row0 + g + 8 < n;
#pragma unroll
  for (int db = 0; db < D / 8; ++db) {
    const int d = db * 8 + t2;
    if (vlo)
      *reinterpret_cast<uint32_t*>(ob + static_cast<int64_t>(row0 + g) * stride + d) =
          M::pack(o[db][0] * inv_lo, o[db][1] * inv_lo);
    if (vhi)
      *reinterpret_cast<uint32_t*>(ob + static_cast<int64_t>(row0 + g + 8) * stride + d) =
          M::pack(o[db][2] * inv_hi, o[db][3] * inv_hi);
  }
}

template <typename T>
cudaError_t launch_prefill(const PrefillParams& p, int head_dim, int max_query_len, cudaStream_t st) {
  const dim3 grid((max_query_len + kPfRows - 1) / kPfRows, p.num_heads, p.num_seqs);
  if (head_dim == 64) prefill_kernel<T, 64><<<grid, kPfWarps * 32, 0, st>>>(p);
  else prefill_kernel<T, 128><<<grid, kPfWarps * 32, 0, st>>>(p);
  return cudaGetLastError();
}


// ---------------------------------------------------------------------------
// Tensor-core (tcgen05) kernel, used when block_size divides 128 and is a
// multiple of 16.
//
// One CTA per 128-row query tile, two CTAs per SM: one CTA's softmax runs
// while the tensor cores work on the other's MMAs.  With group G a multiple
// of a power of two HG (HG = the largest power of two dividing G, at most
// 8), a tile's rows are HG query heads of one kv head times 128 / HG chunk
// tokens (row r = token r / HG, head r % HG), so every K/V tile serves all
// the tile's heads.  The grid is 1-D over (head group, sequence, row tile),
// row tile slowest and counted down: the tiles with the most keys start
// first and the shortest close the launch.  Tensor memory (256 columns): S
// at columns 0-127 (P over 64-127) and O at 128 + (0 .. head_dim - 1).
//   warp 5: TMA producer -- Q once, then each 128-key tile's K and V, one
//     box per (block, 64-dim slab), through the block table; a K stage is
//     free once its S is done, a V stage once its P V is;
//   warp 4: one lane issues the MMAs: S = Q K^T (M 128, N 128, K head_dim)
//     once P V of the previous tile has completed (S overwrites P), and
//     O += P V (M 128, N head_dim, K 128) with P from tensor memory once the
//     softmax warps have written it;
//   warps 0-3: thread t of warp w owns row 32 w + t and reads its S row with
//     the 32x32b tensor-memory shape in two halves of 64 registers, so the
//     row max and sum need no exchange.  In one pass it computes e = S c2 -
//     m_ref (keys past the row's position: -inf), P = exp2(e) rounded to
//     the q dtype, the sum of the rounded P, and the tile's max of e.  P,
//     the sum and O are relative to a reference m_ref that moves only when
//     a tile's max lies more than 2^8 above it (then the pass is repeated
//     and the row's sum and O columns are rescaled); P stays <= 256.  O is
//     read from tensor memory once, at the end, and written as the row's
//     output.
// Slots past the last key of the last tile (the tail of its last block and
// blocks never loaded) are zeroed in the V tile before P V reads it, so a
// sentinel there cannot reach the output.
// ---------------------------------------------------------------------------
constexpr int kTcRows = 128;                      // MMA M: rows of a query tile
constexpr int kTcKeys = 128;                      // keys per tile: N of S, K of P V
constexpr int kTcSoftWarps = 4;                   // softmax warps: one row per thread
constexpr int kTcMmaWarp = kTcSoftWarps, kTcTmaWarp = kTcSoftWarps + 1;
constexpr int kTcThreads = 32 * (kTcSoftWarps + 2);
constexpr uint32_t kTcCols = 256;                 // S (128) and O (up to 128)

template <int D>
struct TcLayout {
  // ring depths: two CTAs per SM share 227 KB of shared memory
  static constexpr int kKStages = D == 64 ? 2 : 1, kVStages = kKStages;
  static constexpr int kSlab = 128 * 128;           // one 64-column slab of 128 rows
  static constexpr int kTile = (D / 64) * kSlab;    // a Q, K or V tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kTile;               // stage s at + s kTile
  static constexpr int kOffV = kOffK + kKStages * kTile;
  static constexpr int kOffBar = kOffV + kVStages * kTile;
  static constexpr int kBytes = kOffBar + 256;
  static constexpr int kSmem = kBytes + 1024;  // slack for 1024-byte alignment
};

// Three-input max (one instruction on sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// One key pair of the softmax pass: the running maxima (two chains), P =
// exp2(e) for both keys rounded to T and packed into s[i] (the pair's S
// values, at s[2i] and s[2i + 1], are already read), their sum into ls[i % 2].
template <typename T>
__device__ __forceinline__ void softmax_pair(float2 e, int i, float& ma, float& mb, uint64_t (&ls)[2],
                                             uint32_t (&s)[64]) {
  if (i & 1) mb = max3(mb, e.x, e.y);
  else ma = max3(ma, e.x, e.y);
  const uint32_t pk = Mma<T>::pack(fast_exp2(e.x), fast_exp2(e.y));
  s[i] = pk;
  // the sum is taken over the rounded P that P V multiplies, so that the
  // weights the output is normalised by are the ones it was built from
  const float2 r = Mma<T>::unpack(pk);
  ls[i & 1] = tc::fadd2(ls[i & 1], tc::f2(r.x, r.y));
}

// Compiler barrier: the 32 packed values, the sums and the max are computed
// here, before any later tensor-memory load is issued.
__device__ __forceinline__ void pin_regs(uint32_t (&v)[32], uint64_t (&ls)[2], float& m) {
  asm volatile(""
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                 "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                 "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                 "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]),
                 "+r"(v[29]), "+r"(v[30]), "+r"(v[31]), "+l"(ls[0]), "+l"(ls[1]), "+f"(m));
}

// Registers: two CTAs of six warps put three warps on each of the SM's four
// sub-partitions (16,384 registers each), so a thread holds at most 168.
template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 2)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using Lay = TcLayout<D>;
  constexpr int kSlabs = D / 64, KST = Lay::kKStages, VST = Lay::kVStages;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(sm + Lay::kOffBar);
  uint64_t* bar_kfull = bar_q + 1;             // [KST] K tile landed
  uint64_t* bar_kempty = bar_kfull + KST;      // [KST] S of the tile done
  uint64_t* bar_vfull = bar_kempty + KST;      // [VST] V tile landed
  uint64_t* bar_vempty = bar_vfull + VST;      // [VST] P V of the tile done
  uint64_t* bar_s = bar_vempty + VST;          // S written
  uint64_t* bar_p = bar_s + 1;                 // P written (every softmax thread arrives)
  uint64_t* bar_pv = bar_p + 1;                // P V done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_pv + 1);

  const int hg = 1 << p.hg_log2, tpt = kTcRows >> p.hg_log2;
  // 1-D grid over (head group, sequence, row tile), the row tile slowest and
  // counted down, so the tiles with the most keys are dispatched first and
  // the last CTAs to start are the shortest
  const int ngroups = p.num_heads >> p.hg_log2, nrt = p.row_tiles;
  const int gi = static_cast<int>(blockIdx.x % ngroups);
  const int b = static_cast<int>((blockIdx.x / ngroups) % p.num_seqs);
  const int qt = nrt - 1 - static_cast<int>(blockIdx.x / ngroups / p.num_seqs);
  const int h0 = gi * hg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qs = __ldg(p.query_start + b), n = __ldg(p.query_start + b + 1) - qs;
  // rows past the grid's reach (a chunk longer than max_query_len) would be
  // left uncomputed: the sequence's last row tile in the grid reports it
  if (qt == nrt - 1 && gi == 0 && threadIdx.x == 0 && n > nrt * tpt) record_error(KV_ERR_DEVICE_BOUNDS);
  const int tok0 = qt * tpt;  // first chunk token of the tile
  if (n <= 0 || tok0 >= n) return;
  int L = __ldg(p.seq_lens + b);
  const int64_t cap = static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size;
  if (L < n || qs < 0 || qs + n > p.num_tokens) {  // the chunk must lie inside its sequence and in q
    if (threadIdx.x == 0) record_error(KV_ERR_DEVICE_BOUNDS);
    return;
  }
  if (L > cap) {
    if (threadIdx.x == 0) record_error(KV_ERR_DEVICE_BOUNDS);
    L = static_cast<int>(cap);
    if (L < n) return;
  }
  const int ctx = L - n, kvh = h0 / p.group;
  // the tile's chunk tokens, the keys its last row sees, its key tiles
  const int rows_here = min(n - tok0, tpt);
  const int nkeys = min(ctx + tok0 + rows_here, L);
  const int ntiles = (nkeys + kTcKeys - 1) / kTcKeys;

  const int32_t* table = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
  const int bs = p.block_size;
  // K (V) of tile j into stage j % KST (j % VST) once S (P V) of the tile
  // that stage held before is done (TMA thread only).
  auto load = [&](int j, bool is_v) -> bool {
    const int nst = is_v ? VST : KST, st = j % nst;
    uint64_t* full = (is_v ? bar_vfull : bar_kfull) + st;
    if (j >= nst && !mbar_wait_bounded((is_v ? bar_vempty : bar_kempty) + st, ((j / nst) - 1) & 1)) return false;
    const int k0 = j * kTcKeys, k1 = min(k0 + kTcKeys, nkeys);
    const int blk0 = k0 / bs, blk1 = (k1 + bs - 1) / bs;
    mbar_arrive_expect_tx(full, static_cast<uint32_t>((blk1 - blk0) * bs * D * 2));
    uint8_t* dst = sm + (is_v ? Lay::kOffV : Lay::kOffK) + st * Lay::kTile;
    const CUtensorMap* map = is_v ? &tmV : &tmK;
    for (int bi = blk0; bi < blk1; ++bi) {
      int pb = __ldg(table + bi);
      if (pb < 0 || pb >= p.num_blocks) {
        record_error(KV_ERR_DEVICE_BOUNDS);
        pb = 0;
      }
      const int r = (bi - blk0) * bs;
      for (int s = 0; s < kSlabs; ++s) tma_load_3d(dst + s * Lay::kSlab + r * 128, map, full, s * 64, kvh, pb * bs);
    }
    return true;
  };
  // The TMA thread sets up the barriers and issues Q and the first K tile
  // before the CTA-wide barrier, so those loads overlap the tensor-memory
  // allocation and the barrier itself.
  const bool tma_thread = warp == kTcTmaWarp && lane == 0;
  bool load_ok = true;
  if (tma_thread) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(bar_kfull + s, 1);
      mbar_init(bar_kempty + s, 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(bar_vfull + s, 1);
      mbar_init(bar_vempty + s, 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_p, kTcSoftWarps * 32);
    mbar_init(bar_pv, 1);
    fence_mbar_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    mbar_arrive_expect_tx(bar_q, kSlabs * kTcRows * 128);
    for (int s = 0; s < kSlabs; ++s)
      tma_load_3d(sm + Lay::kOffQ + s * Lay::kSlab, &tmQ, bar_q, s * 64, h0, qs + tok0);
    load_ok = load(0, false);
  }
  if (warp == kTcMmaWarp) tc::alloc(tmem_slot, kTcCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTcTmaWarp) {
    if (lane == 0) {
      // ---- TMA producer (Q and the first K tile are already issued)
      bool ok = load_ok;
      for (int j = 0; j < ntiles && ok; ++j) {
        ok = load(j, true);
        if (ok && j + 1 < ntiles) ok = load(j + 1, false);
      }
      // every stage's last S and P V have completed (no copy or commit in flight at exit)
      for (int j = max(0, ntiles - KST); j < ntiles; ++j) mbar_wait_bounded(bar_kempty + (j % KST), (j / KST) & 1);
      for (int j = max(0, ntiles - VST); j < ntiles; ++j) mbar_wait_bounded(bar_vempty + (j % VST), (j / VST) & 1);
    }
  } else if (warp == kTcMmaWarp) {
    if (lane == 0) {
      // ---- MMA issue
      constexpr uint32_t idS = tc::idesc_f16(kBf16, kTcRows, kTcKeys, false);
      constexpr uint32_t idPV = tc::idesc_f16(kBf16, kTcRows, D, true);
      bool ok = mbar_wait_bounded(bar_q, 0);
      const uint32_t aQ = smem_u32(sm + Lay::kOffQ);
      for (int j = 0; j < ntiles && ok; ++j) {
        const int ks = j % KST, vs = j % VST;
        if (!mbar_wait_bounded(bar_kfull + ks, (j / KST) & 1)) break;
        // S overwrites P of the previous tile: its P V must be done
        if (j > 0 && !mbar_wait_bounded(bar_pv, (j - 1) & 1)) break;
        tc::fence_after();
        const uint32_t kb = smem_u32(sm + Lay::kOffK + ks * Lay::kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Lay::kSlab + (kk & 3) * 32;  // 64-dim slab, 16-dim step inside it
          tc::mma_f16(tmem, tc::sdesc_sw128(aQ + off, 16, 1024), tc::sdesc_sw128(kb + off, 16, 1024), idS, kk > 0);
        }
        tc::commit(bar_s);
        tc::commit(bar_kempty + ks);
        if (!mbar_wait_bounded(bar_vfull + vs, (j / VST) & 1)) break;
        // P lands after the softmax warps have zeroed the last tile's V tail
        if (!mbar_wait_bounded(bar_p, j & 1)) break;
        tc::fence_after();
        const uint32_t vb = smem_u32(sm + Lay::kOffV + vs * Lay::kTile);
#pragma unroll
        for (int kk = 0; kk < kTcKeys / 16; ++kk) {
          // keys 16 kk .. + 15: P, two keys per column from S column 64
          tc::mma_f16_ts(tmem + 128, tmem + 64 + kk * 8, tc::sdesc_sw128(vb + kk * 16 * 128, Lay::kSlab, 1024), idPV,
                         (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc::commit(bar_pv);
        tc::commit(bar_vempty + vs);
      }
    }
  } else {
    // ---- softmax: thread t of warp w owns row 32 w + t
    const int r = warp * 32 + lane;
    const uint32_t tS = tmem + (static_cast<uint32_t>(warp * 32) << 16), tO = tS + 128;
    const int tok = r >> p.hg_log2, hh = r & (hg - 1);
    const int lim_abs = min(ctx + tok0 + tok, nkeys - 1);  // last key the row sees
    const float c2 = p.scale_log2;
    const uint64_t c2x2 = tc::f2(c2, c2);
    // a reference at most 2^8 below the row's max keeps P <= 256; before
    // the row's first key it is also at most 2^8 above it, so the largest P
    // keeps its precision in fp16 too
    constexpr float kSlack = 8.f, kLow = 8.f;
    // P, O and the sum are relative to m_ref, 0 until the row's scores
    // call for another
    float m_ref = 0.f, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      // after a timeout (recorded) the remaining waits are skipped
      if (ok && !mbar_wait_bounded(bar_s, j & 1)) ok = false;
      tc::fence_after();
      const int lim = lim_abs - j * kTcKeys;  // columns <= lim are keys of this row
      const bool part = __any_sync(0xffffffffu, lim < kTcKeys - 1);
      // One pass over the row's 128 S values, in two halves of 64 registers
      // (keys 64-127, then 0-63): e = S * c2 - m_ref (keys the row does not
      // see: -inf), P = exp2(e) rounded to T, two keys per column, and the
      // tile's max of e.  The pass is repeated against a new reference max
      // only where that max lies more than kSlack above the reference (P
      // would exceed 2^kSlack), or, before the row's first key, more than
      // kLow below it (P would lose its range).  P goes over S columns
      // 64-127 once both halves are done: keys 0-63 to 64-95, keys 64-127
      // to 96-127.
      uint32_t s[64], ph[32];
      uint64_t ls[2];
      float me;
      auto pass = [&]() {
        const uint64_t negm = tc::f2(-m_ref, -m_ref);
        ls[0] = ls[1] = tc::f2(0.f, 0.f);
        me = -INFINITY;
#pragma unroll 1
        for (int h = 1; h >= 0; --h) {
          tc::ld_32x32b_x32(tS + 64 * h, s);
          tc::ld_32x32b_x32(tS + 64 * h + 32, s + 32);
          tc::wait_ld();
          float ma = -INFINITY, mb = -INFINITY;
          if (part) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int c = 64 * h + 2 * i;
              float2 e = tc::f2_split(
                  tc::ffma2(tc::f2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2x2, negm));
              e.x = c <= lim ? e.x : -INFINITY;
              e.y = c + 1 <= lim ? e.y : -INFINITY;
              softmax_pair<T>(e, i, ma, mb, ls, s);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float2 e = tc::f2_split(
                  tc::ffma2(tc::f2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2x2, negm));
              softmax_pair<T>(e, i, ma, mb, ls, s);
            }
          }
          me = max3(me, ma, mb);
          if (h == 1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) ph[i] = s[i];
            // the upper half's P and sums are complete before the lower half
            // is read, so the two halves never hold registers at once
            pin_regs(ph, ls, me);
          }
        }
      };
      bool rescale = false;
      float alpha = 1.f;
#pragma unroll 1
      for (int attempt = 0; attempt < 2; ++attempt) {
        pass();
        if (attempt == 1) break;
        // me = -inf: no key of the row in the tile
        const bool need = me > kSlack || (l == 0.f && me != -INFINITY && me < -kLow);
        rescale = __any_sync(0xffffffffu, need);
        if (!rescale) break;
        // a row that does not need it keeps its reference (alpha 1)
        const float m_new = need ? m_ref + me : m_ref;
        alpha = fast_exp2(m_ref - m_new);
        l *= alpha;
        m_ref = m_new;
      }
      tc::st_32x32b_x32(tS + 64, s);
      tc::st_32x32b_x32(tS + 96, ph);
      {
        const float2 a = tc::f2_split(ls[0]), b = tc::f2_split(ls[1]);
        l += (a.x + a.y) + (b.x + b.y);
      }
      if (j == ntiles - 1 && (nkeys % kTcKeys) != 0) {
        // zero V rows past the last key (tail slots and blocks never loaded)
        const int vs = j % VST;
        if (ok && !mbar_wait_bounded(bar_vfull + vs, (j / VST) & 1)) ok = false;
        const int first = nkeys - j * kTcKeys;
        uint8_t* vt = sm + Lay::kOffV + vs * Lay::kTile;
#pragma unroll 1
        for (int i = r; i < kTcKeys * kSlabs * 8; i += 128) {
          const int row = i / (kSlabs * 8), rest = i % (kSlabs * 8);
          if (row >= first)
            *reinterpret_cast<uint4*>(vt + (rest >> 3) * Lay::kSlab + row * 128 + (rest & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // the zeros are read by the tensor cores
      }
      if (rescale && j > 0) {
        // O holds tiles 0 .. j - 1: P V of tile j - 1 is done (S_j was issued after it)
        if (ok && !mbar_wait_bounded(bar_pv, (j - 1) & 1)) ok = false;
        tc::fence_after();
        const uint64_t a2 = tc::f2(alpha, alpha);
#pragma unroll
        for (int oc = 0; oc < D; oc += 32) {
          uint32_t w[32];
          tc::ld_32x32b_x32(tO + oc, w);
          tc::wait_ld();
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float2 y = tc::f2_split(tc::fmul2(tc::f2(__uint_as_float(w[k]), __uint_as_float(w[k + 1])), a2));
            w[k] = __float_as_uint(y.x);
            w[k + 1] = __float_as_uint(y.y);
          }
          tc::st_32x32b_x32(tO + oc, w);
        }
      }
      tc::wait_st();
      tc::fence_before();
      mbar_arrive(bar_p);
    }
    if (ok && !mbar_wait_bounded(bar_pv, (ntiles - 1) & 1)) ok = false;
    tc::fence_after();
    const float inv = l > 0.f ? __fdiv_rn(1.f, l) : 0.f;
    T* orow = static_cast<T*>(p.out) + (static_cast<int64_t>(qs + tok0 + tok) * p.num_heads + h0 + hh) * D;
    const bool store = ok && tok < rows_here;
#pragma unroll 1
    for (int oc = 0; oc < D; oc += 32) {
      uint32_t w[32];
      tc::ld_32x32b_x32(tO + oc, w);
      tc::wait_ld();
      uint32_t o[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        o[k] = Mma<T>::pack(__uint_as_float(w[2 * k]) * inv, __uint_as_float(w[2 * k + 1]) * inv);
      if (store) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          reinterpret_cast<uint4*>(orow + oc)[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    __syncwarp();
    tc::fence_after();
    tc::dealloc(tmem, kTcCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() {
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

// A 3-D tensor {n0, n1, n2} of 16-bit elements (dim 0 contiguous, dim 1
// `n0` apart, dim 2 `n0 * n1` apart) with 128-byte-swizzled boxes
// {64, box1, box2}.  Encoded maps are kept in a small table keyed by all the
// arguments, so a caller that reuses its buffers pays the encoding once.
bool tc_map(const void* base, int64_t n0, int64_t n1, int64_t n2, int box1, int box2, CUtensorMap* out) {
  struct Key {
    const void* base;
    int64_t n0, n1, n2;
    int box1, box2;
    bool operator==(const Key& o) const {
      return base == o.base && n0 == o.n0 && n1 == o.n1 && n2 == o.n2 && box1 == o.box1 && box2 == o.box2;
    }
  };
  constexpr int kSlots = 32;
  static std::mutex mu;
  static Key keys[kSlots];
  static CUtensorMap maps[kSlots];
  static int used = 0, next = 0;
  const Key key{base, n0, n1, n2, box1, box2};
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (keys[i] == key) {
      *out = maps[i];
      return true;
    }
  auto fn = tc_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(n0), static_cast<cuuint64_t>(n1), static_cast<cuuint64_t>(n2)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(n0) * 2, static_cast<cuuint64_t>(n0 * n1) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box1), static_cast<cuuint32_t>(box2)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap m;
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const int slot = used < kSlots ? used++ : (next++ % kSlots);
  keys[slot] = key;
  maps[slot] = m;
  *out = m;
  return true;
}

bool tc_supported(int block_size) { return block_size >= 16 && block_size % 16 == 0 && kTcKeys % block_size == 0; }

template <typename T, int D>
cudaError_t launch_prefill_tc(const PrefillParams& p, int max_query_len, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& mv, cudaStream_t st) {
  constexpr int kSmem = TcLayout<D>::kSmem;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    // the largest shared-memory carve-out
    e = cudaFuncSetAttribute(prefill_tc_kernel<T, D>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int rows_per_cta = kTcRows >> p.hg_log2;  // chunk tokens per CTA
  const int64_t row_tiles = (static_cast<int64_t>(max_query_len) + rows_per_cta - 1) / rows_per_cta;
  const int64_t ctas = row_tiles * (p.num_heads >> p.hg_log2) * p.num_seqs;
  if (ctas > INT32_MAX) return cudaErrorInvalidConfiguration;
  PrefillParams q = p;
  q.row_tiles = static_cast<int32_t>(row_tiles);
  const dim3 grid(static_cast<unsigned>(ctas));
  prefill_tc_kernel<T, D><<<grid, kTcThreads, kSmem, st>>>(q, mq, mk, mv);
  return cudaGetLastError();
}

bool aligned16(const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }

}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

extern "C" int paged_prefill_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* seq_lens,
                                       const int32_t* query_start_loc, int64_t num_query_tokens, int32_t num_seqs,
                                       int32_t num_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                       int32_t max_blocks_per_seq, int32_t max_query_len, float scale, int dtype,
                                       void* stream) {
  if (dtype != KV_DTYPE_F16 && dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq <= 0 || max_query_len < 0 || (head_dim != 64 && head_dim != 128))
    return KV_ERR_INVALID_ARG;
  if (num_blocks > INT32_MAX / block_size || num_heads > 65535 || num_seqs > 65535) return KV_ERR_INVALID_ARG;
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return KV_ERR_INVALID_ARG;
  if (num_query_tokens < 0 || num_query_tokens > INT32_MAX) return KV_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_query_len == 0 || num_query_tokens == 0) return KV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start_loc) return KV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return KV_ERR_INVALID_ARG;
  PrefillParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.query_start = query_start_loc;
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.num_tokens = num_query_tokens;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!tc_supported(block_size)) {
    const cudaError_t e = dtype == KV_DTYPE_F16 ? launch_prefill<__half>(p, head_dim, max_query_len, st)
                                                : launch_prefill<__nv_bfloat16>(p, head_dim, max_query_len, st);
    return cuda_status(e);
  }
  // tensor-core kernel: HG = the largest power of two (at most 8) dividing the group
  while (p.hg_log2 < 3 && p.group % (2 << p.hg_log2) == 0) ++p.hg_log2;
  CUtensorMap mq, mk, mv;
  const int64_t rows = num_blocks * block_size;
  if (!tc_map(q, head_dim, num_heads, num_query_tokens, 1 << p.hg_log2, kTcRows >> p.hg_log2, &mq) ||
      !tc_map(k_cache, head_dim, num_kv_heads, rows, 1, block_size, &mk) ||
      !tc_map(v_cache, head_dim, num_kv_heads, rows, 1, block_size, &mv))
    return cuda_status(cudaErrorInvalidValue, "cuTensorMapEncodeTiled failed");
  cudaError_t e;
  if (dtype == KV_DTYPE_F16)
    e = head_dim == 64 ? launch_prefill_tc<__half, 64>(p, max_query_len, mq, mk, mv, st)
                       : launch_prefill_tc<__half, 128>(p, max_query_len, mq, mk, mv, st);
  else
    e = head_dim == 64 ? launch_prefill_tc<__nv_bfloat16, 64>(p, max_query_len, mq, mk, mv, st)
                       : launch_prefill_tc<__nv_bfloat16, 128>(p, max_query_len, mq, mk, mv, st);
  return cuda_status(e);
}

// Read (and optionally clear) this translation unit's device error word.
extern "C" int pagedkv_internal_prefill_error(int reset, int* code) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return KV_ERR_CUDA;
  if (reset) {
    int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return KV_ERR_CUDA;
  }
  *code = v;
  return KV_OK;
}
