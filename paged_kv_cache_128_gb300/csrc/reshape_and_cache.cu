// Cache write: scatter each new token's K/V rows into the paged pool.
//
// "MiniPaged-Qwen: Paged KV Cache 与 KV Block Manager" §12 (cache write by
// slot_mapping) and §11 (slot -> physical block, offset).  With the cache
// laid out [num_blocks, block_size, num_kv_heads, head_dim], all heads of one
// token are contiguous in both the input ([Hkv, D]) and the destination
// (cache[slot / bs][slot % bs]), and that destination row starts at
// slot * Hkv * D.  So the write is one contiguous row copy per token.
//
// Kernel shape: one warp per token, grid-stride; each lane moves 16-byte
// vectors (narrower only when the row size or alignment forces it), issuing
// all of its loads for K and V before the stores so a warp keeps up to
// 2 * kUnroll vectors per lane in flight.  The copy is bit-exact.
//
// Several layers' caches under one block table ("MiniPaged-Qwen" §16: the
// block tables and slot mapping are built once per step and shared by every
// layer's attention) are written by one launch: grid.y runs over layers,
// each with its own input and cache base.

#include "common.cuh"

namespace pagedkv {
namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kUnroll = 4;

template <typename V>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
reshape_and_cache_kernel(const char* __restrict__ k, const char* __restrict__ v, char* __restrict__ k_cache,
                         char* __restrict__ v_cache, const int32_t* __restrict__ slot_mapping, int64_t num_tokens,
                         int64_t row_bytes, int64_t k_stride_bytes, int64_t v_stride_bytes, int64_t num_slots,
                         int64_t k_layer_bytes, int64_t v_layer_bytes, int64_t cache_layer_bytes) {
  const int lane = threadIdx.x & 31;
  const int64_t layer = blockIdx.y;
  k += layer * k_layer_bytes;
  v += layer * v_layer_bytes;
  k_cache += layer * cache_layer_bytes;
  v_cache += layer * cache_layer_bytes;
  const int64_t nvec = row_bytes / static_cast<int64_t>(sizeof(V));
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5); t < num_tokens;
       t += static_cast<int64_t>(gridDim.x) * kWarpsPerCta) {
    const int32_t slot = __ldg(slot_mapping + t);
    if (slot == -1) continue;  // padded token: nothing read, nothing written
    if (slot < 0 || slot >= num_slots) {
      if (lane == 0) record_error(KV_ERR_DEVICE_BOUNDS);
      continue;
    }
    const V* ks = reinterpret_cast<const V*>(k + t * k_stride_bytes);
    const V* vs = reinterpret_cast<const V*>(v + t * v_stride_bytes);
    V* kd = reinterpret_cast<V*>(k_cache + static_cast<int64_t>(slot) * row_bytes);
    V* vd = reinterpret_cast<V*>(v_cache + static_cast<int64_t>(slot) * row_bytes);
    for (int64_t base = lane; base < nvec; base += 32 * kUnroll) {
      V kr[kUnroll], vr[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + 32 * u;
        if (i < nvec) {
          kr[u] = __ldg(ks + i);
          vr[u] = __ldg(vs + i);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + 32 * u;
        if (i < nvec) {
          kd[i] = kr[u];
          vd[i] = vr[u];
        }
      }
    }
  }
}

bool aligned(const void* p, int64_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct LayerStrides {
  int32_t layers;
  int64_t k_bytes, v_bytes, cache_bytes;  // between consecutive layers
};

template <typename V>
cudaError_t launch(const void* k, const void* v, void* kc, void* vc, const int32_t* slots, int64_t n,
                   int64_t row_bytes, int64_t ks, int64_t vs, int64_t num_slots, const LayerStrides& ls,
                   cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t need = (n + kWarpsPerCta - 1) / kWarpsPerCta;
  const int64_t cap = (static_cast<int64_t>(sms > 0 ? sms : 1) * 16 + ls.layers - 1) / ls.layers;
  const int grid = static_cast<int>(need < cap ? need : cap);
  reshape_and_cache_kernel<V><<<dim3(grid, ls.layers), kWarpsPerCta * 32, 0, stream>>>(
      static_cast<const char*>(k), static_cast<const char*>(v), static_cast<char*>(kc), static_cast<char*>(vc),
      slots, n, row_bytes, ks, vs, num_slots, ls.k_bytes, ls.v_bytes, ls.cache_bytes);
  return cudaGetLastError();
}

}  // namespace

// The cache write of num_layers layers (1 for paged_reshape_and_cache).
int cache_write(const void* k, const void* v, void* k_cache, void* v_cache, const int32_t* slot_mapping,
                int64_t num_tokens, int32_t num_layers, int64_t k_layer_stride, int64_t v_layer_stride,
                int64_t cache_layer_stride, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                int64_t num_blocks, int64_t k_token_stride, int64_t v_token_stride, int dtype, void* stream);
}  // namespace pagedkv

using namespace pagedkv;

int pagedkv::cache_write(const void* k, const void* v, void* k_cache, void* v_cache, const int32_t* slot_mapping,
                         int64_t num_tokens, int32_t num_layers, int64_t k_layer_stride, int64_t v_layer_stride,
                         int64_t cache_layer_stride, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int64_t num_blocks, int64_t k_token_stride, int64_t v_token_stride, int dtype,
                         void* stream) {
  if (dtype != KV_DTYPE_F32 && dtype != KV_DTYPE_F16 && dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return KV_ERR_INVALID_ARG;
  if (num_layers <= 0 || num_layers > 65535 || k_layer_stride < 0 || v_layer_stride < 0 || cache_layer_stride < 0)
    return KV_ERR_INVALID_ARG;
  const int64_t row_elems = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (k_token_stride < row_elems || v_token_stride < row_elems) return KV_ERR_INVALID_ARG;
  if (num_blocks > INT32_MAX / block_size) return KV_ERR_INVALID_ARG;
  const int64_t num_slots = num_blocks * block_size;
  if (num_layers > 1 && cache_layer_stride < num_slots * row_elems) return KV_ERR_INVALID_ARG;  // layers overlap
  if (num_tokens == 0) return KV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return KV_ERR_INVALID_ARG;
  const int64_t es = static_cast<int64_t>(dtype_bytes(dtype));
  const int64_t row_bytes = row_elems * es, ks = k_token_stride * es, vs = v_token_stride * es;
  const LayerStrides ls{num_layers, k_layer_stride * es, v_layer_stride * es, cache_layer_stride * es};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  auto fits = [&](int64_t a) {
    return row_bytes % a == 0 && ks % a == 0 && vs % a == 0 && aligned(k, a) && aligned(v, a) &&
           aligned(k_cache, a) && aligned(v_cache, a) && ls.k_bytes % a == 0 && ls.v_bytes % a == 0 &&
           ls.cache_bytes % a == 0;
  };
  if (fits(16))
    err = launch<uint4>(k, v, k_cache, v_cache, slot_mapping, num_tokens, row_bytes, ks, vs, num_slots, ls, st);
  else if (fits(8))
    err = launch<uint2>(k, v, k_cache, v_cache, slot_mapping, num_tokens, row_bytes, ks, vs, num_slots, ls, st);
  else if (fits(4))
    err = launch<uint32_t>(k, v, k_cache, v_cache, slot_mapping, num_tokens, row_bytes, ks, vs, num_slots, ls, st);
  else if (fits(2))
    err = launch<uint16_t>(k, v, k_cache, v_cache, slot_mapping, num_tokens, row_bytes, ks, vs, num_slots, ls, st);
  else
    return KV_ERR_INVALID_ARG;
  return cuda_status(err);
}

extern "C" int paged_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                       const int32_t* slot_mapping, int64_t num_tokens, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                       int64_t k_token_stride, int64_t v_token_stride, int dtype, void* stream) {
  return cache_write(k, v, k_cache, v_cache, slot_mapping, num_tokens, 1, 0, 0, 0, num_kv_heads, head_dim, block_size,
                     num_blocks, k_token_stride, v_token_stride, dtype, stream);
}

extern "C" int paged_reshape_and_cache_layers(const void* k, const void* v, void* k_cache, void* v_cache,
                                              const int32_t* slot_mapping, int64_t num_tokens, int32_t num_layers,
                                              int64_t k_layer_stride, int64_t v_layer_stride,
                                              int64_t cache_layer_stride, int32_t num_kv_heads, int32_t head_dim,
                                              int32_t block_size, int64_t num_blocks, int64_t k_token_stride,
                                              int64_t v_token_stride, int dtype, void* stream) {
  return cache_write(k, v, k_cache, v_cache, slot_mapping, num_tokens, num_layers, k_layer_stride, v_layer_stride,
                     cache_layer_stride, num_kv_heads, head_dim, block_size, num_blocks, k_token_stride,
                     v_token_stride, dtype, stream);
}

// Read (and optionally clear) this translation unit's device error word.
extern "C" int pagedkv_internal_reshape_error(int reset, int* code) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return KV_ERR_CUDA;
  if (reset) {
    int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return KV_ERR_CUDA;
  }
  *code = v;
  return KV_OK;
}

// ---------------------------------------------------------------------------
// Copy-on-write block copies ("paged-attention-impl-detail", section
// Copy-on-Write共享: a writer to a shared block first copies its K and V to a
// fresh block).  One CTA per (pair, layer); the CTA streams the block's K
// then V bytes with 16-byte vectors, all loads of a round before its stores.

namespace pagedkv {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(char* __restrict__ k_cache, char* __restrict__ v_cache, const int32_t* __restrict__ src,
                   const int32_t* __restrict__ dst, int64_t n, int64_t layer_stride_bytes, int64_t block_bytes,
                   int64_t num_blocks) {
  const int64_t pair = blockIdx.x;
  const int64_t layer = blockIdx.y;
  if (pair >= n) return;
  const int32_t s = __ldg(src + pair), d = __ldg(dst + pair);
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (threadIdx.x == 0) record_error(KV_ERR_DEVICE_BOUNDS);
    return;
  }
  const int64_t nvec = block_bytes / 16;
  for (int which = 0; which < 2; ++which) {
    char* base = (which ? v_cache : k_cache) + layer * layer_stride_bytes;
    const uint4* from = reinterpret_cast<const uint4*>(base + s * block_bytes);
    uint4* to = reinterpret_cast<uint4*>(base + d * block_bytes);
    for (int64_t i0 = threadIdx.x; i0 < nvec; i0 += kCopyThreads * 4) {
      uint4 r[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u * kCopyThreads < nvec) r[u] = from[i0 + u * kCopyThreads];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u * kCopyThreads < nvec) to[i0 + u * kCopyThreads] = r[u];
    }
  }
}

}  // namespace
}  // namespace pagedkv

extern "C" int paged_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int64_t n,
                                 int32_t num_layers, int64_t layer_stride, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int64_t num_blocks, int dtype, void* stream) {
  using namespace pagedkv;
  if (dtype != KV_DTYPE_F32 && dtype != KV_DTYPE_F16 && dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  if (n < 0 || num_layers <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
      layer_stride < 0)
    return KV_ERR_INVALID_ARG;
  if (n == 0) return KV_OK;
  if (!k_cache || !v_cache || !src || !dst) return KV_ERR_INVALID_ARG;
  const int64_t es = static_cast<int64_t>(dtype_bytes(dtype));
  const int64_t block_bytes = static_cast<int64_t>(block_size) * num_kv_heads * head_dim * es;
  if (num_layers > 1 && layer_stride < num_blocks * block_size * static_cast<int64_t>(num_kv_heads) * head_dim)
    return KV_ERR_INVALID_ARG;  // layers would overlap
  if (block_bytes % 16 != 0 || (layer_stride * es) % 16 != 0 || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return KV_ERR_INVALID_ARG;
  if (n > 0x7fffffff || num_layers > 65535) return KV_ERR_INVALID_ARG;
  copy_blocks_kernel<<<dim3(static_cast<unsigned>(n), static_cast<unsigned>(num_layers)), kCopyThreads, 0,
                       static_cast<cudaStream_t>(stream)>>>(static_cast<char*>(k_cache), static_cast<char*>(v_cache),
                                                             src, dst, n, layer_stride * es, block_bytes, num_blocks);
  return cuda_status(cudaGetLastError());
}

extern "C" int paged_copy_blocks_fp8(void* k_cache, void* v_cache, float* k_scales, float* v_scales,
                                     const int32_t* src, const int32_t* dst, int64_t n, int32_t num_layers,
                                     int64_t layer_stride, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                     int64_t num_blocks, void* stream) {
  using namespace pagedkv;
  if (n < 0 || num_layers <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
      layer_stride < 0)
    return KV_ERR_INVALID_ARG;
  if (n == 0) return KV_OK;
  if (!k_cache || !v_cache || !k_scales || !v_scales || !src || !dst) return KV_ERR_INVALID_ARG;
  // a block's codes: bs x Hkv x D bytes; its scales: Hkv x bs floats, contiguous at [block][Hkv][bs]
  const int64_t code_bytes = static_cast<int64_t>(block_size) * num_kv_heads * head_dim;
  const int64_t scale_bytes = static_cast<int64_t>(block_size) * num_kv_heads * 4;
  if (num_layers > 1 && layer_stride < num_blocks * code_bytes) return KV_ERR_INVALID_ARG;  // layers would overlap
  if (code_bytes % 16 != 0 || scale_bytes % 16 != 0 || layer_stride % 16 != 0 || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(k_scales, 16) || !aligned(v_scales, 16))
    return KV_ERR_INVALID_ARG;
  if (n > 0x7fffffff || num_layers > 65535) return KV_ERR_INVALID_ARG;
  const dim3 grid(static_cast<unsigned>(n), static_cast<unsigned>(num_layers));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, st>>>(static_cast<char*>(k_cache), static_cast<char*>(v_cache), src,
                                                    dst, n, layer_stride, code_bytes, num_blocks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, st>>>(reinterpret_cast<char*>(k_scales), reinterpret_cast<char*>(v_scales),
                                                    src, dst, n, num_blocks * scale_bytes, scale_bytes, num_blocks);
  return cuda_status(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// fp8 (E4M3) cache write ("paged-attention-impl-detail", 实践建议 4: the KV
// cache inside a block can be quantised on its own).  Each (token, kv head)
// row of head_dim values gets one float32 scale, amax / 448 (1 for a zero
// row), kept in the row's block: scales[(block * Hkv + head) * bs + offset].
// The values are divided by it in float32 (correctly rounded) and rounded to
// E4M3, nearest-even, saturating at 448.  One warp per token; a lane owns E
// consecutive values of a row (E = head_dim / 32) and the amax is a warp
// max-reduction.  A warp loads K and V of kFp8Heads heads before it
// quantises any of them, and the first heads' loads go out before the
// token's slot has arrived (a padded token's row is read and dropped), so
// the memory round trips overlap instead of following one another.

namespace pagedkv {
namespace {

__device__ __forceinline__ uint16_t e4m3x2_from(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// A read-only 4-byte global load that stays where it is written: volatile,
// so it is neither dropped nor moved past the slot check into the branch
// that uses it.
__device__ __forceinline__ uint32_t load_early(const uint32_t* p) {
  uint32_t r;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

constexpr int kFp8Heads = 4;

template <typename T, int E>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
cache_write_fp8_kernel(const T* __restrict__ k, const T* __restrict__ v, uint8_t* __restrict__ k_codes,
                       uint8_t* __restrict__ v_codes, float* __restrict__ k_scales, float* __restrict__ v_scales,
                       const int32_t* __restrict__ slot_mapping, int64_t num_tokens, int num_kv_heads,
                       int block_size, int64_t k_stride, int64_t v_stride, int64_t num_slots) {
  constexpr int D = 32 * E, W = E / 2;  // W: 32-bit words holding a lane's E values
  const int lane = threadIdx.x & 31;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5); t < num_tokens;
       t += static_cast<int64_t>(gridDim.x) * kWarpsPerCta) {
    const int32_t slot = __ldg(slot_mapping + t);
    // 4-byte aligned: k and v are, token strides are even, lane * E * 2 is a multiple of 4
    const uint32_t* krow = reinterpret_cast<const uint32_t*>(k + t * k_stride + lane * E);
    const uint32_t* vrow = reinterpret_cast<const uint32_t*>(v + t * v_stride + lane * E);
    uint32_t raw[kFp8Heads][2][W];
    auto load = [&](int h0) {
#pragma unroll
      for (int g = 0; g < kFp8Heads; ++g)
        if (h0 + g < num_kv_heads)
#pragma unroll
          for (int w = 0; w < W; ++w) {
            raw[g][0][w] = load_early(krow + (h0 + g) * (D / 2) + w);
            raw[g][1][w] = load_early(vrow + (h0 + g) * (D / 2) + w);
          }
    };
    load(0);
    if (slot == -1) continue;  // padded token: nothing written
    if (slot < 0 || slot >= num_slots) {
      if (lane == 0) record_error(KV_ERR_DEVICE_BOUNDS);
      continue;
    }
    const int64_t blk = slot / block_size, off = slot % block_size;
    for (int h0 = 0; h0 < num_kv_heads; h0 += kFp8Heads) {
      if (h0 > 0) load(h0);
#pragma unroll
      for (int g = 0; g < kFp8Heads; ++g) {
        const int h = h0 + g;
        if (h >= num_kv_heads) break;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          float x[E];
#pragma unroll
          for (int w = 0; w < W; ++w) {  // the lower-addressed value sits in the low half of the word
            T pair[2];
            memcpy(pair, &raw[g][which][w], sizeof(pair));
            x[2 * w] = DType<T>::to_float(pair[0]);
            x[2 * w + 1] = DType<T>::to_float(pair[1]);
          }
          float amax = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
          uint16_t packed[E / 2];
#pragma unroll
          for (int e = 0; e < E; e += 2)
            packed[e / 2] = e4m3x2_from(__fdiv_rn(x[e], scale), __fdiv_rn(x[e + 1], scale));
          uint8_t* dst = (which ? v_codes : k_codes) + (static_cast<int64_t>(slot) * num_kv_heads + h) * D + lane * E;
          if constexpr (E == 2) {
            *reinterpret_cast<uint16_t*>(dst) = packed[0];
          } else if constexpr (E == 4) {
            *reinterpret_cast<uint32_t*>(dst) = packed[0] | (static_cast<uint32_t>(packed[1]) << 16);
          } else {
            *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0] | (static_cast<uint32_t>(packed[1]) << 16),
                                                        packed[2] | (static_cast<uint32_t>(packed[3]) << 16));
          }
          if (lane == 0) (which ? v_scales : k_scales)[(blk * num_kv_heads + h) * block_size + off] = scale;
        }
      }
    }
  }
}

template <typename T, int E>
cudaError_t launch_fp8(const void* k, const void* v, void* kc, void* vc, float* ks, float* vs, const int32_t* slots,
                       int64_t n, int hkv, int bs, int64_t k_stride, int64_t v_stride, int64_t num_slots,
                       cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t need = (n + kWarpsPerCta - 1) / kWarpsPerCta;
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 16;
  cache_write_fp8_kernel<T, E><<<static_cast<int>(need < cap ? need : cap), kWarpsPerCta * 32, 0, stream>>>(
      static_cast<const T*>(k), static_cast<const T*>(v), static_cast<uint8_t*>(kc), static_cast<uint8_t*>(vc), ks, vs,
      slots, n, hkv, bs, k_stride, v_stride, num_slots);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fp8_d(int d, const void* k, const void* v, void* kc, void* vc, float* ks, float* vs,
                         const int32_t* slots, int64_t n, int hkv, int bs, int64_t kst, int64_t vst, int64_t ns,
                         cudaStream_t st) {
  if (d == 64) return launch_fp8<T, 2>(k, v, kc, vc, ks, vs, slots, n, hkv, bs, kst, vst, ns, st);
  if (d == 128) return launch_fp8<T, 4>(k, v, kc, vc, ks, vs, slots, n, hkv, bs, kst, vst, ns, st);
  return launch_fp8<T, 8>(k, v, kc, vc, ks, vs, slots, n, hkv, bs, kst, vst, ns, st);
}

}  // namespace
}  // namespace pagedkv

extern "C" int paged_reshape_and_cache_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                                           float* k_scales, float* v_scales, const int32_t* slot_mapping,
                                           int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                           int32_t block_size, int64_t num_blocks, int64_t k_token_stride,
                                           int64_t v_token_stride, int dtype, void* stream) {
  using namespace pagedkv;
  if (dtype != KV_DTYPE_F16 && dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0) return KV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KV_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (k_token_stride < row || v_token_stride < row) return KV_ERR_INVALID_ARG;
  if (num_blocks > INT32_MAX / block_size) return KV_ERR_INVALID_ARG;
  if (num_tokens == 0) return KV_OK;
  if (!k || !v || !k_cache || !v_cache || !k_scales || !v_scales || !slot_mapping) return KV_ERR_INVALID_ARG;
  if (!aligned(k, 4) || !aligned(v, 4) || (k_token_stride % 2) || (v_token_stride % 2) || !aligned(k_cache, 8) ||
      !aligned(v_cache, 8) || !aligned(k_scales, 4) || !aligned(v_scales, 4))
    return KV_ERR_INVALID_ARG;
  const int64_t num_slots = num_blocks * block_size;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = dtype == KV_DTYPE_F16
                      ? launch_fp8_d<__half>(head_dim, k, v, k_cache, v_cache, k_scales, v_scales, slot_mapping,
                                             num_tokens, num_kv_heads, block_size, k_token_stride, v_token_stride,
                                             num_slots, st)
                      : launch_fp8_d<__nv_bfloat16>(head_dim, k, v, k_cache, v_cache, k_scales, v_scales,
                                                    slot_mapping, num_tokens, num_kv_heads, block_size,
                                                    k_token_stride, v_token_stride, num_slots, st);
  return cuda_status(e);
}
