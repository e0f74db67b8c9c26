// Cache writes of libpagedkv: the slot scatter (pk_reshape_and_cache, and
// pk_reshape_and_cache_append on resident tables), the copy-on-write block
// copy (pk_copy_blocks) and the swap copy (pk_swap_blocks), plus the
// read-stream reference (pk_read_stream), the library's status strings and
// device-error readout.
//
// The cache kernels are pure data movement. The pool layout [N, B, Hk, d] makes one
// token's K (all heads) a contiguous Hk*d*esz-byte row, and one block a
// contiguous B*Hk*d*esz-byte span, so both kernels are 16-byte vector copies.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"
#include "pk_device.cuh"

namespace {

__device__ int g_cache_ops_error;

// grid.x = new token, grid.y = chunk of its row: token i's K row and V row
// go to slot slot_mapping[i] ("Paged KV Cache Allocation and the Block
// Table", append_token: the token is written at physical * block_size +
// slot). Each thread moves one 16-byte vector of K and one of V, so a whole
// step's scatter is a single round trip to memory.
//
// With UPDATE, token i is the next token of row i of device-resident block
// tables and context lengths, and the kernel also does that row's share of
// the step's bookkeeping: the entry of the block holding position
// pos = context_lens[i] becomes slot / B (a freshly opened block and a
// copy-on-write replacement alike: the new token's slot names the tail block),
// and context_lens[i] becomes pos + 1. A slot whose offset in its block is not
// pos mod B means the resident tables are out of step with the host: the row
// is left unchanged and the event is recorded (the K/V row is still written
// to its slot, which was checked against the pool).
template <bool UPDATE>
__global__ void __launch_bounds__(128) reshape_and_cache_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, const int64_t *__restrict__ slots,
    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, int64_t num_slots,
    int32_t row_vecs, int32_t *__restrict__ tables, const int32_t *lens_in, int32_t *lens_out,
    int32_t max_blocks, int32_t block_size) {
  const int64_t i = blockIdx.x;
  const int32_t j = int32_t(blockIdx.y) * blockDim.x + threadIdx.x;
  const int64_t s = slots[i];
  if (s < 0) return;
  if (s >= num_slots) {
    if (threadIdx.x == 0 && blockIdx.y == 0) pk::record_error(&g_cache_ops_error, PK_DEVERR_SLOT, i);
    return;
  }
  if (UPDATE && blockIdx.y == 0 && threadIdx.x == 0) {
    // One thread per token reads and advances the row's length (lens_out may
    // be lens_in: in place).
    const int32_t pos = lens_in[i];
    if (pos < 0 || pos >= max_blocks * block_size || s % block_size != pos % block_size) {
      pk::record_error(&g_cache_ops_error, PK_DEVERR_CONTEXT, i);
      lens_out[i] = pos;
    } else {
      tables[i * max_blocks + pos / block_size] = int32_t(s / block_size);
      lens_out[i] = pos + 1;
    }
  }
  if (j >= row_vecs) return;
  const uint4 a = __ldg(k + i * row_vecs + j);
  const uint4 b = __ldg(v + i * row_vecs + j);
  k_cache[s * row_vecs + j] = a;
  v_cache[s * row_vecs + j] = b;
}

// A pure read stream, the reference the attention's K/V reads are measured
// against: every 16-byte vector of the buffer is loaded once (four loads in
// flight per thread, grid-strided) and folded into one XOR so that no load
// can be dropped.
__global__ void __launch_bounds__(256) read_stream_kernel(const uint4 *__restrict__ buf,
                                                          int64_t n, unsigned int *sink) {
  constexpr int U = 4;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + (U - 1) * stride < n; i += U * stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = __ldg(buf + i + u * stride);
#pragma unroll
    for (int u = 0; u < U; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n; i += stride) {
    const uint4 a = __ldg(buf + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
  if (acc == 0x9e3779b9u) atomicXor(sink, acc);  // practically never taken; keeps the loads
}

// Block copies run kCopyThreads threads per CTA, each moving up to kCopyVecs
// 16-byte vectors of one chunk (32 KiB per CTA).
constexpr int kCopyThreads = 256;
constexpr int kCopyVecs = 8;

// Copies vectors [beg, end) of a chunk (at most kCopyThreads * kCopyVecs):
// each thread issues all its loads before its first store, so a chunk costs
// one memory round trip.
__device__ __forceinline__ void copy_chunk(const uint4 *from, uint4 *to, int64_t beg, int64_t end) {
  uint4 v[kCopyVecs];
#pragma unroll
  for (int k = 0; k < kCopyVecs; ++k) {
    const int64_t j = beg + threadIdx.x + int64_t(k) * kCopyThreads;
    if (j < end) v[k] = from[j];
  }
#pragma unroll
  for (int k = 0; k < kCopyVecs; ++k) {
    const int64_t j = beg + threadIdx.x + int64_t(k) * kCopyThreads;
    if (j < end) to[j] = v[k];
  }
}

// grid.x = pair, grid.y = 0 for K / 1 for V, grid.z = chunk of the block.
// The whole block src is copied to dst ("paged attention deep",
// "Copy-on-write for shared prefixes").
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, const int64_t *__restrict__ pairs,
    int32_t num_blocks, int64_t block_vecs, int64_t chunk_vecs) {
  const int64_t src = pairs[2 * blockIdx.x];
  const int64_t dst = pairs[2 * blockIdx.x + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
      pk::record_error(&g_cache_ops_error, PK_DEVERR_PAIR, blockIdx.x);
    return;
  }
  uint4 *pool = blockIdx.y == 0 ? k_cache : v_cache;
  const int64_t beg = int64_t(blockIdx.z) * chunk_vecs;
  copy_chunk(pool + src * block_vecs, pool + dst * block_vecs, beg,
             min(block_vecs, beg + chunk_vecs));
}

// grid.x = pair, grid.y = 0 for K / 1 for V, grid.z = chunk of the block:
// whole block pairs[2p] of one pool goes to block pairs[2p+1] of the other
// (swap out: device pool -> pinned host pool; swap in: the reverse). The host
// pool is read or written through its device-visible address.
__global__ void __launch_bounds__(kCopyThreads) swap_blocks_kernel(
    const uint4 *__restrict__ from_k, const uint4 *__restrict__ from_v, uint4 *__restrict__ to_k,
    uint4 *__restrict__ to_v, const int64_t *__restrict__ pairs, int32_t from_blocks,
    int32_t to_blocks, int64_t block_vecs, int64_t chunk_vecs) {
  const int64_t src = pairs[2 * blockIdx.x];
  const int64_t dst = pairs[2 * blockIdx.x + 1];
  if (src < 0 || src >= from_blocks || dst < 0 || dst >= to_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
      pk::record_error(&g_cache_ops_error, PK_DEVERR_PAIR, blockIdx.x);
    return;
  }
  const int64_t beg = int64_t(blockIdx.z) * chunk_vecs;
  copy_chunk((blockIdx.y == 0 ? from_k : from_v) + src * block_vecs,
             (blockIdx.y == 0 ? to_k : to_v) + dst * block_vecs, beg,
             min(block_vecs, beg + chunk_vecs));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t elem_size(pk_dtype t) { return t == PK_F32 ? 4 : (t == PK_BF16 ? 2 : 0); }

pk_status check_desc(const pk_cache_desc *d) {
  if (!d || d->num_blocks <= 0 || d->block_size <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0)
    return PK_ERR_INVALID_ARG;
  if (elem_size(d->dtype) == 0) return PK_ERR_UNSUPPORTED;
  if ((int64_t(d->num_kv_heads) * d->head_dim * elem_size(d->dtype)) % 16 != 0)
    return PK_ERR_UNSUPPORTED;
  return PK_OK;
}

}  // namespace

// Read-and-clear of this file's device error word (used by pk_get_device_error).
extern "C" int pkx_take_cache_ops_error(cudaStream_t stream) {
  int code = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbolAsync(&code, g_cache_ops_error, sizeof(int), 0,
                                cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return -1;
  if (cudaMemcpyToSymbolAsync(g_cache_ops_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                              stream) != cudaSuccess)
    return -1;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return -1;
  return code;
}

extern "C" int pkx_take_attention_error(cudaStream_t stream);

extern "C" {

pk_status pk_reshape_and_cache(const void *k, const void *v, const int64_t *slot_mapping,
                               int32_t num_tokens, void *k_cache, void *v_cache,
                               const pk_cache_desc *desc, void *stream) {
  pk_status st = check_desc(desc);
  if (st != PK_OK) return st;
  if (num_tokens < 0) return PK_ERR_INVALID_ARG;
  if (num_tokens == 0) return PK_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PK_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PK_ERR_INVALID_ARG;
  const int64_t row_bytes = int64_t(desc->num_kv_heads) * desc->head_dim * elem_size(desc->dtype);
  const int64_t num_slots = int64_t(desc->num_blocks) * desc->block_size;
  const int64_t row_vecs = row_bytes / 16;
  const int64_t chunks = (row_vecs + 127) / 128;
  if (chunks > 65535) return PK_ERR_UNSUPPORTED;
  reshape_and_cache_kernel<false><<<dim3(num_tokens, unsigned(chunks)), 128, 0,
                                    static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping,
      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), num_slots,
      int32_t(row_vecs), nullptr, nullptr, nullptr, 0, desc->block_size);
  return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

pk_status pkx_reshape_and_cache_advance(const void *k, const void *v, const int64_t *slot_mapping,
                                        int32_t num_tokens, void *k_cache, void *v_cache,
                                        const pk_cache_desc *desc, int32_t *block_tables,
                                        int32_t max_blocks_per_seq, const int32_t *lens_in,
                                        int32_t *lens_out, void *stream);

pk_status pk_reshape_and_cache_append(const void *k, const void *v, const int64_t *slot_mapping,
                                      int32_t num_tokens, void *k_cache, void *v_cache,
                                      const pk_cache_desc *desc, int32_t *block_tables,
                                      int32_t max_blocks_per_seq, int32_t *context_lens,
                                      void *stream) {
  return pkx_reshape_and_cache_advance(k, v, slot_mapping, num_tokens, k_cache, v_cache, desc,
                                       block_tables, max_blocks_per_seq, context_lens,
                                       context_lens, stream);
}

// pk_reshape_and_cache_append reading the lengths from lens_in and writing
// the advanced lengths to lens_out (library-internal; the fused attention's
// CUDA-core fallback uses it with two buffers).
pk_status pkx_reshape_and_cache_advance(const void *k, const void *v, const int64_t *slot_mapping,
                                        int32_t num_tokens, void *k_cache, void *v_cache,
                                        const pk_cache_desc *desc, int32_t *block_tables,
                                        int32_t max_blocks_per_seq, const int32_t *lens_in,
                                        int32_t *lens_out, void *stream) {
  pk_status st = check_desc(desc);
  if (st != PK_OK) return st;
  if (num_tokens < 0 || max_blocks_per_seq <= 0) return PK_ERR_INVALID_ARG;
  if (num_tokens == 0) return PK_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache || !block_tables || !lens_in || !lens_out)
    return PK_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PK_ERR_INVALID_ARG;
  if (int64_t(max_blocks_per_seq) * desc->block_size > INT32_MAX) return PK_ERR_UNSUPPORTED;
  const int64_t row_bytes = int64_t(desc->num_kv_heads) * desc->head_dim * elem_size(desc->dtype);
  const int64_t num_slots = int64_t(desc->num_blocks) * desc->block_size;
  const int64_t row_vecs = row_bytes / 16;
  const int64_t chunks = (row_vecs + 127) / 128;
  if (chunks > 65535) return PK_ERR_UNSUPPORTED;
  reshape_and_cache_kernel<true><<<dim3(num_tokens, unsigned(chunks)), 128, 0,
                                   static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping,
      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), num_slots,
      int32_t(row_vecs), block_tables, lens_in, lens_out, max_blocks_per_seq, desc->block_size);
  return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

// Library-internal hook for the decode step's captured graphs
// (decode_step.cpp): the argument count of the advancing scatter kernel, whose
// first two arguments are the new keys' and values' addresses; 0 for any
// other function.
extern "C" int pkx_scatter_kernel_arity(const void *f) {
  return f == reinterpret_cast<const void *>(reshape_and_cache_kernel<true>) ? 12 : 0;
}

pk_status pk_read_stream(const void *buf, size_t bytes, unsigned int *sink, void *stream) {
  if (!buf || !sink || bytes < 16 || !aligned16(buf)) return PK_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PK_ERR_CUDA;
  read_stream_kernel<<<sms * 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(buf), int64_t(bytes / 16), sink);
  return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

pk_status pk_copy_blocks(void *k_cache, void *v_cache, const int64_t *src_dst_pairs,
                         int32_t num_pairs, const pk_cache_desc *desc, void *stream) {
  pk_status st = check_desc(desc);
  if (st != PK_OK) return st;
  if (num_pairs < 0) return PK_ERR_INVALID_ARG;
  if (num_pairs == 0) return PK_OK;
  if (!k_cache || !v_cache || !src_dst_pairs) return PK_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PK_ERR_INVALID_ARG;
  const int64_t block_bytes = int64_t(desc->block_size) * desc->num_kv_heads * desc->head_dim *
                              elem_size(desc->dtype);
  const int64_t block_vecs = block_bytes / 16;
  const int64_t chunk_vecs = int64_t(kCopyThreads) * kCopyVecs;
  const int64_t chunks = (block_vecs + chunk_vecs - 1) / chunk_vecs;
  if (chunks > 65535) return PK_ERR_UNSUPPORTED;
  dim3 grid(num_pairs, 2, unsigned(chunks));
  copy_blocks_kernel<<<grid, kCopyThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), src_dst_pairs,
      desc->num_blocks, block_vecs, chunk_vecs);
  return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

pk_status pk_swap_blocks(void *k_cache, void *v_cache, void *k_host, void *v_host,
                         int32_t num_host_blocks, const int64_t *pairs, int32_t num_pairs,
                         int32_t direction, const pk_cache_desc *desc, void *stream) {
  pk_status st = check_desc(desc);
  if (st != PK_OK) return st;
  if (num_pairs < 0 || num_host_blocks < 0 || (direction != PK_SWAP_OUT && direction != PK_SWAP_IN))
    return PK_ERR_INVALID_ARG;
  if (num_pairs == 0) return PK_OK;
  if (!k_cache || !v_cache || !k_host || !v_host || !pairs) return PK_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_host) || !aligned16(v_host))
    return PK_ERR_INVALID_ARG;
  // The host pool must be reachable from the device (pinned, mapped memory).
  void *dk = nullptr, *dv = nullptr;
  if (cudaHostGetDevicePointer(&dk, k_host, 0) != cudaSuccess ||
      cudaHostGetDevicePointer(&dv, v_host, 0) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_INVALID_ARG;
  }
  const int64_t block_bytes = int64_t(desc->block_size) * desc->num_kv_heads * desc->head_dim *
                              elem_size(desc->dtype);
  const int64_t block_vecs = block_bytes / 16;
  const int64_t chunk_vecs = int64_t(kCopyThreads) * kCopyVecs;
  const int64_t chunks = (block_vecs + chunk_vecs - 1) / chunk_vecs;
  if (chunks > 65535) return PK_ERR_UNSUPPORTED;
  dim3 grid(num_pairs, 2, unsigned(chunks));
  const bool out = direction == PK_SWAP_OUT;
  swap_blocks_kernel<<<grid, kCopyThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(out ? k_cache : dk), static_cast<const uint4 *>(out ? v_cache : dv),
      static_cast<uint4 *>(out ? dk : k_cache), static_cast<uint4 *>(out ? dv : v_cache), pairs,
      out ? desc->num_blocks : num_host_blocks, out ? num_host_blocks : desc->num_blocks, block_vecs,
      chunk_vecs);
  return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

pk_status pk_get_device_error(int32_t *code_out, void *stream) {
  if (!code_out) return PK_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int a = pkx_take_cache_ops_error(s);
  const int b = pkx_take_attention_error(s);
  if (a < 0 || b < 0) return PK_ERR_CUDA;
  *code_out = a != 0 ? a : b;
  return PK_OK;
}

const char *pk_status_string(pk_status status) {
  switch (status) {
    case PK_OK: return "ok";
    case PK_ERR_INVALID_ARG: return "invalid argument";
    case PK_ERR_UNSUPPORTED: return "unsupported configuration";
    case PK_ERR_OUT_OF_BLOCKS: return "out of blocks";
    case PK_ERR_UNKNOWN_SEQ: return "unknown sequence";
    case PK_ERR_SEQ_EXISTS: return "sequence exists";
    case PK_ERR_CUDA: return "CUDA error";
    case PK_ERR_WORKSPACE: return "workspace missing or too small";
    case PK_ERR_INVARIANT: return "block manager invariant violated";
    case PK_ERR_NOMEM: return "out of host memory";
  }
  return "unknown status";
}

}  // extern "C"
