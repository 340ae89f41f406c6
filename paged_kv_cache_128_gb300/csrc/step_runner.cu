// Native serving-step runner: one call per decode step of one layer.
//
// The step is the hot path end to end ("从零实现一个 mini vLLM: Block
// Manager", section on the ModelRunner: the scheduler's metadata -- slot
// mapping, block tables, context lengths -- is built on the CPU and handed
// to the GPU with the step's new K/V; "MiniPaged-Qwen" §8: CPU metadata
// plane, GPU data plane):
//
//   host   kvbm_prepare_step into a page-locked buffer, plus each decode
//          sequence's row in the step's K/V (its newest token) and the
//          copy-on-write copies its appends queued (kvbm_take_copies);
//   copy   one async H2D copy of that buffer on a side stream (and, with
//          host I/O, the step's q/k/v), so it overlaps the previous step's
//          kernel instead of sitting between two kernels;
//   device paged_copy_blocks for those copies, if any, then
//          paged_decode_step on the compute stream after an event wait:
//          one launch doing the cache write and decode attention;
//   copy   with host I/O, the output back to the host on a second side
//          stream.
//
// kNumBufs metadata buffers (host and device) rotate between steps.  Reuse
// is ordered by events: the host rewrites host buffer i only after the copy
// that last read it has run; the copy into device buffer i waits for the
// kernel that last read it.  Nothing here synchronises the device except
// those host waits on copies issued kNumBufs steps earlier.

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>
#include <algorithm>
#include <vector>

#include "common.cuh"

namespace pagedkv {
namespace {

struct Side {
  void* q = nullptr;  // host I/O: device copies of the step's inputs and output
  void* k = nullptr;
  void* v = nullptr;
  void* out = nullptr;
};

}  // namespace
}  // namespace pagedkv

constexpr int kNumBufs = 4;

struct kvstep_s {
  kvbm_t mgr = nullptr;
  kvstep_config_t cfg{};
  int device = 0;
  int64_t meta_ints = 0;  // slot_mapping | block_tables | seq_lens | new_row | copy src | copy dst
  int32_t* h_meta[kNumBufs] = {};
  int32_t* d_meta[kNumBufs] = {};
  pagedkv::Side side[kNumBufs];
  int32_t layers = 1;
  size_t q_bytes = 0, kv_bytes = 0;  // one layer's
  size_t stage_q = 0, stage_k = 0, stage_v = 0, stage_bytes = 0;  // host_io = 2: byte offsets in a slot's block
  // per metadata buffer: the sequence and block count each table row held
  // at its last export (kvbm_export_update rewrites only what changed)
  std::vector<int64_t> row_ids[kNumBufs];
  std::vector<int32_t> row_nblocks[kNumBufs];
  cudaStream_t compute = nullptr, h2d = nullptr, d2h = nullptr;
  cudaEvent_t copied[kNumBufs] = {};    // H2D of buffer i done
  cudaEvent_t done[kNumBufs] = {};      // kernel that read buffer i done
  cudaEvent_t out_back[kNumBufs] = {};  // D2H of output i done (host I/O)
  bool used[kNumBufs] = {};
  int cur = kNumBufs - 1;
};

namespace {

void release(kvstep_s* h) {
  for (int i = 0; i < kNumBufs; ++i) {
    if (h->h_meta[i]) cudaFreeHost(h->h_meta[i]);
    if (h->d_meta[i]) cudaFree(h->d_meta[i]);
    if (h->cfg.host_io == 2) {  // q/k/v live inside d_meta[i]
      if (h->side[i].out) cudaFree(h->side[i].out);
    } else {
      for (void* p : {h->side[i].q, h->side[i].k, h->side[i].v, h->side[i].out})
        if (p) cudaFree(p);
    }
    for (cudaEvent_t e : {h->copied[i], h->done[i], h->out_back[i]})
      if (e) cudaEventDestroy(e);
  }
  if (h->h2d) cudaStreamDestroy(h->h2d);
  if (h->d2h) cudaStreamDestroy(h->d2h);
  delete h;
}

// Row of the step's K/V holding decode sequence b's new token: the
// (n_prefill_tokens + b)-th non-padded position (kvbm_prepare_step writes
// the prefill slots first, then the decode slots, around the pads).
void decode_rows(const int64_t* pads, int64_t n_pad, int64_t n_prefill_tokens, int64_t n_decode, int32_t* rows) {
  int64_t p = 0;
  for (int64_t b = 0; b < n_decode; ++b) {
    const int64_t v = n_prefill_tokens + b;
    while (p < n_pad && pads[p] <= v + p) ++p;
    rows[b] = static_cast<int32_t>(v + p);
  }
}

}  // namespace

extern "C" int kvstep_create(kvbm_t mgr, const kvstep_config_t* cfg, kvstep_t* out) {
  if (!mgr || !cfg || !out) return KV_ERR_INVALID_ARG;
  const kvstep_config_t& c = *cfg;
  if (c.num_seqs <= 0 || c.num_heads <= 0 || c.num_kv_heads <= 0 || c.num_heads % c.num_kv_heads != 0 ||
      c.head_dim <= 0 || c.block_size <= 0 || c.num_blocks <= 0 || c.max_blocks_per_seq <= 0 ||
      c.max_seq_len <= 0 || c.num_step_tokens < c.num_seqs || !c.k_cache || !c.v_cache)
    return KV_ERR_INVALID_ARG;
  if (c.dtype != KV_DTYPE_F32 && c.dtype != KV_DTYPE_F16 && c.dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  if (c.host_io < 0 || c.host_io > 2) return KV_ERR_INVALID_ARG;
  const int32_t layers = c.num_layers > 1 ? c.num_layers : 1;
  if (c.cache_fp8 && (!c.k_scales || !c.v_scales || c.dtype == KV_DTYPE_F32)) return KV_ERR_INVALID_ARG;
  if (c.num_layers < 0 || c.num_layers > 65535 ||
      (layers > 1 && c.cache_layer_stride < c.num_blocks * c.block_size * static_cast<int64_t>(c.num_kv_heads) *
                                                c.head_dim))
    return KV_ERR_INVALID_ARG;
  kvstep_s* h = new (std::nothrow) kvstep_s();
  if (!h) return KV_ERR_INVALID_ARG;
  h->mgr = mgr;
  h->cfg = c;
  h->compute = static_cast<cudaStream_t>(c.stream);
  h->layers = layers;
  // at most one copy-on-write copy per decode append (prefills never copy)
  h->meta_ints = c.num_step_tokens + static_cast<int64_t>(c.num_seqs) * c.max_blocks_per_seq + 4 * c.num_seqs;
  const size_t meta_bytes = static_cast<size_t>(h->meta_ints) * sizeof(int32_t);
  const size_t es = pagedkv::dtype_bytes(c.dtype);
  h->q_bytes = static_cast<size_t>(c.num_seqs) * c.num_heads * c.head_dim * es;
  h->kv_bytes = static_cast<size_t>(c.num_step_tokens) * c.num_kv_heads * c.head_dim * es;
  // host_io = 2: one block per slot holds [metadata | q | k | v] (each part
  // 256-byte aligned), the same on the host and on the device, so a step is
  // one host-to-device copy
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  size_t block_bytes = meta_bytes;
  if (c.host_io == 2) {
    const size_t L = static_cast<size_t>(layers);
    h->stage_q = up(meta_bytes);
    h->stage_k = h->stage_q + up(h->q_bytes * L);
    h->stage_v = h->stage_k + up(h->kv_bytes * L);
    h->stage_bytes = h->stage_v + h->kv_bytes * L;
    block_bytes = h->stage_bytes;
  }
  for (int i = 0; i < kNumBufs; ++i) {
    h->row_ids[i].assign(static_cast<size_t>(c.num_seqs), -1);  // never exported into
    h->row_nblocks[i].assign(static_cast<size_t>(c.num_seqs), 0);
  }
  cudaError_t e = cudaGetDevice(&h->device);
  for (int i = 0; i < kNumBufs && e == cudaSuccess; ++i) {
    e = cudaHostAlloc(reinterpret_cast<void**>(&h->h_meta[i]), block_bytes, cudaHostAllocDefault);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&h->d_meta[i]), block_bytes);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->copied[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->out_back[i], cudaEventDisableTiming);
    if (e == cudaSuccess && c.host_io == 2) {
      char* d = reinterpret_cast<char*>(h->d_meta[i]);
      h->side[i].q = d + h->stage_q;
      h->side[i].k = d + h->stage_k;
      h->side[i].v = d + h->stage_v;
      e = cudaMalloc(&h->side[i].out, h->q_bytes * layers);
    } else if (e == cudaSuccess && c.host_io) {
      e = cudaMalloc(&h->side[i].q, h->q_bytes * layers);
      if (e == cudaSuccess) e = cudaMalloc(&h->side[i].out, h->q_bytes * layers);
      if (e == cudaSuccess) e = cudaMalloc(&h->side[i].k, h->kv_bytes * layers);
      if (e == cudaSuccess) e = cudaMalloc(&h->side[i].v, h->kv_bytes * layers);
    }
  }
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->h2d, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->d2h, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    release(h);
    return pagedkv::cuda_status(e);
  }
  *out = h;
  return KV_OK;
}

extern "C" int kvstep_destroy(kvstep_t h) {
  if (!h) return KV_ERR_INVALID_ARG;
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < kNumBufs; ++i) {
    if (h->used[i]) {
      cudaError_t a = cudaEventSynchronize(h->done[i]);
      cudaError_t b = cudaEventSynchronize(h->out_back[i]);
      if (e == cudaSuccess) e = a != cudaSuccess ? a : b;
    }
  }
  release(h);
  return pagedkv::cuda_status(e);
}

extern "C" int kvstep_run(kvstep_t h, const void* q, const void* k, const void* v, void* out,
                          const int64_t* free_ids, int64_t n_free, const int64_t* prefill_ids,
                          const int64_t* prefill_lens, int64_t n_prefill, const int64_t* decode_ids,
                          int64_t n_decode, const int64_t* pad_positions, int64_t n_pad) {
  if (!h || !out) return KV_ERR_INVALID_ARG;
  const kvstep_config_t& c = h->cfg;
  if (c.host_io != 2 && (!q || !k || !v)) return KV_ERR_INVALID_ARG;
  if (n_decode != c.num_seqs || n_pad < 0 || n_prefill < 0 || (n_prefill && !prefill_lens)) return KV_ERR_INVALID_ARG;
  int64_t n_pre_tokens = 0;
  for (int64_t i = 0; i < n_prefill; ++i) n_pre_tokens += prefill_lens[i] > 0 ? prefill_lens[i] : 0;
  if (n_pre_tokens + n_decode + n_pad != c.num_step_tokens) return KV_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n_pad; ++i)
    if (pad_positions[i] < 0 || pad_positions[i] >= c.num_step_tokens || (i && pad_positions[i] <= pad_positions[i - 1]))
      return KV_ERR_INVALID_ARG;

  const int i = (h->cur + 1) % kNumBufs;
  cudaError_t e = cudaSuccess;
  if (h->used[i]) {
    e = cudaEventSynchronize(h->copied[i]);  // the copy that last read host buffer i has run
    if (e != cudaSuccess) return pagedkv::cuda_status(e);
  }
  const int64_t B = c.num_seqs, maxb = c.max_blocks_per_seq;
  int32_t* slots = h->h_meta[i];
  int32_t* tables = slots + c.num_step_tokens;
  int32_t* lens = tables + B * maxb;
  int32_t* rows = lens + B;
  int32_t* cp_src = rows + B;
  int32_t* cp_dst = cp_src + B;
  int64_t n_copies = 0;
  int st = kvbm_take_copies(h->mgr, nullptr, nullptr, 0, &n_copies);
  if (st != KV_OK) return st;
  if (n_copies != 0) return KV_ERR_INVALID_ARG;  // copies queued outside the runner must be applied by their caller
  // the lengths here (and the block-table width checked before any change);
  // the tables as an update of what this buffer held four steps ago
  st = kvbm_prepare_step(h->mgr, free_ids, n_free, prefill_ids, prefill_lens, n_prefill, decode_ids, n_decode,
                         pad_positions, n_pad, maxb, slots, nullptr, lens);
  if (st == KV_OK)
    st = kvbm_export_update(h->mgr, decode_ids, n_decode, maxb, tables, h->row_ids[i].data(),
                            h->row_nblocks[i].data());
  if (st != KV_OK) {
    std::fill(h->row_ids[i].begin(), h->row_ids[i].end(), -1);  // contents unknown: rewrite in full next time
    return st;
  }
  st = kvbm_take_copies(h->mgr, cp_src, cp_dst, B, &n_copies);
  if (st != KV_OK) return st;
  decode_rows(pad_positions, n_pad, n_pre_tokens, n_decode, rows);
  h->cur = i;

  // H2D on the side stream, after the kernel that read device buffer i
  if (h->used[i]) e = cudaStreamWaitEvent(h->h2d, h->done[i], 0);
  const size_t meta_bytes = static_cast<size_t>(h->meta_ints) * sizeof(int32_t);
  // staged inputs travel with the metadata in one copy
  const size_t copy_bytes = c.host_io == 2 ? h->stage_bytes : meta_bytes;
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->d_meta[i], h->h_meta[i], copy_bytes, cudaMemcpyHostToDevice, h->h2d);
  const void *dq = q, *dk = k, *dv = v;
  void* dout = out;
  if (c.host_io == 2) {
    dq = h->side[i].q;
    dk = h->side[i].k;
    dv = h->side[i].v;
    dout = h->side[i].out;
  } else if (c.host_io) {
    dq = h->side[i].q;
    dk = h->side[i].k;
    dv = h->side[i].v;
    dout = h->side[i].out;
    const size_t L = static_cast<size_t>(h->layers);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->side[i].q, q, h->q_bytes * L, cudaMemcpyHostToDevice, h->h2d);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->side[i].k, k, h->kv_bytes * L, cudaMemcpyHostToDevice, h->h2d);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->side[i].v, v, h->kv_bytes * L, cudaMemcpyHostToDevice, h->h2d);
  }
  if (e == cudaSuccess) e = cudaEventRecord(h->copied[i], h->h2d);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->compute, h->copied[i], 0);
  // host I/O: output buffer i is rewritten only after its last D2H copy
  if (e == cudaSuccess && c.host_io && h->used[i]) e = cudaStreamWaitEvent(h->compute, h->out_back[i], 0);
  if (e != cudaSuccess) return pagedkv::cuda_status(e);

  int32_t* d_slots = h->d_meta[i];
  int32_t* d_tables = d_slots + c.num_step_tokens;
  int32_t* d_lens = d_tables + B * maxb;
  int32_t* d_rows = d_lens + B;
  if (n_copies > 0) {  // copy-on-write copies (every layer) before the step's writes and reads
    st = c.cache_fp8
             ? paged_copy_blocks_fp8(c.k_cache, c.v_cache, c.k_scales, c.v_scales, d_rows + B, d_rows + 2 * B,
                                     n_copies, h->layers, h->layers > 1 ? c.cache_layer_stride : 0, c.num_kv_heads,
                                     c.head_dim, c.block_size, c.num_blocks, h->compute)
             : paged_copy_blocks(c.k_cache, c.v_cache, d_rows + B, d_rows + 2 * B, n_copies, h->layers,
                                 h->layers > 1 ? c.cache_layer_stride : 0, c.num_kv_heads, c.head_dim, c.block_size,
                                 c.num_blocks, c.dtype, h->compute);
    if (st != KV_OK) return st;
  }
  const int64_t row = static_cast<int64_t>(c.num_kv_heads) * c.head_dim;
  const int64_t es = static_cast<int64_t>(pagedkv::dtype_bytes(c.dtype));
  for (int32_t l = 0; l < h->layers; ++l) {  // one fused launch per layer, same metadata
    const size_t qo = h->q_bytes * static_cast<size_t>(l), ko = h->kv_bytes * static_cast<size_t>(l);
    if (c.cache_fp8) {  // codes: 1 byte per element; scales [NB, Hkv, BS] per layer
      const int64_t co8 = static_cast<int64_t>(l) * c.cache_layer_stride;
      const int64_t so = static_cast<int64_t>(l) * c.num_blocks * c.num_kv_heads * c.block_size;
      char* kc = static_cast<char*>(c.k_cache) + co8;
      char* vc = static_cast<char*>(c.v_cache) + co8;
      st = paged_decode_step_fp8(static_cast<char*>(dout) + qo, static_cast<const char*>(dq) + qo,
                                 static_cast<const char*>(dk) + ko, static_cast<const char*>(dv) + ko, d_slots,
                                 c.num_step_tokens, row, row, d_rows, kc, vc, c.k_scales + so, c.v_scales + so,
                                 d_tables, d_lens, c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim, c.block_size,
                                 c.num_blocks, c.max_blocks_per_seq, c.max_seq_len, c.scale, c.dtype, c.workspace,
                                 c.workspace_bytes, h->compute);
      if (st != KV_OK) return st;
      continue;
    }
    const int64_t co = static_cast<int64_t>(l) * c.cache_layer_stride * es;
    st = paged_decode_step(static_cast<char*>(dout) + qo, static_cast<const char*>(dq) + qo,
                           static_cast<const char*>(dk) + ko, static_cast<const char*>(dv) + ko, d_slots,
                           c.num_step_tokens, row, row, d_rows, static_cast<char*>(c.k_cache) + co,
                           static_cast<char*>(c.v_cache) + co, d_tables, d_lens, c.num_seqs, c.num_heads,
                           c.num_kv_heads, c.head_dim, c.block_size, c.num_blocks, c.max_blocks_per_seq,
                           c.max_seq_len, c.scale, c.dtype, c.workspace, c.workspace_bytes, h->compute);
    if (st != KV_OK) return st;
  }
  e = cudaEventRecord(h->done[i], h->compute);
  if (e == cudaSuccess && c.host_io) {
    e = cudaStreamWaitEvent(h->d2h, h->done[i], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(out, h->side[i].out, h->q_bytes * static_cast<size_t>(h->layers), cudaMemcpyDeviceToHost,
                          h->d2h);
    if (e == cudaSuccess) e = cudaEventRecord(h->out_back[i], h->d2h);
  }
  h->used[i] = true;
  return pagedkv::cuda_status(e);
}

extern "C" int kvstep_stage_buffer(kvstep_t h, int32_t slot, void** q, void** k, void** v, int32_t* slot_out) {
  if (!h || h->cfg.host_io != 2 || slot < -1 || slot >= kNumBufs) return KV_ERR_INVALID_ARG;
  int i = slot;
  if (slot == -1) {  // the next step's slot, once the copy that last read it has run
    i = (h->cur + 1) % kNumBufs;
    if (h->used[i]) {
      const cudaError_t e = cudaEventSynchronize(h->copied[i]);
      if (e != cudaSuccess) return pagedkv::cuda_status(e);
    }
  }
  char* base = reinterpret_cast<char*>(h->h_meta[i]);
  if (q) *q = base + h->stage_q;
  if (k) *k = base + h->stage_k;
  if (v) *v = base + h->stage_v;
  if (slot_out) *slot_out = i;
  return KV_OK;
}

extern "C" int kvstep_join(kvstep_t h, void* stream) {
  if (!h) return KV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < kNumBufs && e == cudaSuccess; ++i) {
    if (!h->used[i]) continue;
    e = cudaStreamWaitEvent(s, h->done[i], 0);
    if (e == cudaSuccess && h->cfg.host_io) e = cudaStreamWaitEvent(s, h->out_back[i], 0);
  }
  return pagedkv::cuda_status(e);
}

extern "C" int kvstep_last_buffers(kvstep_t h, const int32_t** slot_mapping, const int32_t** block_tables,
                                   const int32_t** seq_lens, const int32_t** new_token_row) {
  if (!h || !h->used[h->cur]) return KV_ERR_INVALID_ARG;
  const int32_t* m = h->h_meta[h->cur];
  const int64_t B = h->cfg.num_seqs;
  if (slot_mapping) *slot_mapping = m;
  if (block_tables) *block_tables = m + h->cfg.num_step_tokens;
  if (seq_lens) *seq_lens = m + h->cfg.num_step_tokens + B * h->cfg.max_blocks_per_seq;
  if (new_token_row) *new_token_row = m + h->cfg.num_step_tokens + B * h->cfg.max_blocks_per_seq + B;
  return KV_OK;
}
