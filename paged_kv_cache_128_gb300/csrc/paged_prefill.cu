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
// Kernel shape (flash-attention style, tensor cores through mma.sync):
// one CTA per (64-token query tile, query head, sequence), four warps of 16
// query rows.  Key tiles of 32 tokens are gathered through the block table
// with 16-byte cp.async into a double-buffered, 128-byte-swizzled shared
// tile while the previous tile is consumed.  Per tile a warp computes
// S = Q K^T (Q as the A operand from registers, K^T fragments by
// ldmatrix), masks keys past each row's position, updates an fp32 online
// softmax per row in the exp2 domain, and accumulates O += P V with P
// reused from the score registers as the A operand and V fragments by
// ldmatrix.trans.  The output is rounded once to the q dtype.

#include "common.cuh"

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
  if (n <= 0 || qt * kPfRows >= n) return;
  int L = __ldg(p.seq_lens + b);
  const int64_t cap = static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size;
  if (L < n || L > cap) {  // the chunk must lie inside the sequence and its table
    if (tid == 0) record_error(KV_ERR_DEVICE_BOUNDS);
    if (L < n) return;
    L = static_cast<int>(cap);
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

bool aligned16(const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }

}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

extern "C" int paged_prefill_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* seq_lens,
                                       const int32_t* query_start_loc, int32_t num_seqs, int32_t num_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                       int32_t max_blocks_per_seq, int32_t max_query_len, float scale, int dtype,
                                       void* stream) {
  if (dtype != KV_DTYPE_F16 && dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq <= 0 || max_query_len < 0 || (head_dim != 64 && head_dim != 128))
    return KV_ERR_INVALID_ARG;
  if (num_blocks > INT32_MAX / block_size || num_heads > 65535 || num_seqs > 65535) return KV_ERR_INVALID_ARG;
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return KV_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_query_len == 0) return KV_OK;
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = dtype == KV_DTYPE_F16 ? launch_prefill<__half>(p, head_dim, max_query_len, st)
                                              : launch_prefill<__nv_bfloat16>(p, head_dim, max_query_len, st);
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
