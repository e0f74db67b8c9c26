// Decode-time paged attention of libpagedkv.
//
// Each sequence's single new query attends over its cached keys and values,
// which sit in fixed-size blocks of a shared pool and are reached through the
// sequence's block table: token t is slot t % B of physical block
// table[t / B] ("paged attention deep", "The block table"). The table lookup
// happens inside the kernel; nothing is gathered beforehand ("PagedAttention"
// S06, "Why this needed a custom CUDA kernel"). What is computed is the plain
// softmax attention of the S06 paged_attention listing; the kernels only
// re-associate it (an online softmax over tiles, and optionally split-K
// partitions merged with a log-sum-exp reduction).
//
// Kernels:
//   attn_mma_kernel    bf16. One CTA per (KV head, sequence, partition) -- or
//                      per (KV head, work item) of a host-planned list --
//                      serves all G query heads of the group. A producer warp
//                      streams the K and V rows of each block into a ring of
//                      shared-memory stages with TMA tensor loads (the
//                      physical block id from the table is the TMA
//                      coordinate), 128-byte swizzled. Consumer warps each take
//                      16 tokens per stage (attn_tile): S^T = K Q^T and
//                      O^T += V^T P^T on the tensor cores (mma.sync m16n8k16,
//                      tokens as M, the group's heads as N), with an online
//                      softmax in registers; the softmax weights enter PV as a
//                      bf16 hi + lo pair. Split partitions write partials,
//                      merged by attn_lse_merge_kernel.
//                      With the step's new K/V it also writes them (the CTA
//                      holding the token, for its head: the scatter fused in);
//                      in advance mode it also advances device-resident block
//                      tables and lengths. In cascade mode it covers each
//                      sequence's tokens after its group's shared prefix.
//   attn_cascade_kernel bf16, cascade attention in one launch: prefix CTAs
//                      (one per KV head, group and prefix partition) stream a
//                      shared prefix once for all of the group's query
//                      columns; suffix CTAs are attn_mma_kernel's in cascade
//                      mode. Every part writes a partial.
//   attn_simt_kernel   fp32 or bf16 on CUDA cores: one warp per token,
//                      shuffle-reduced dot products, online softmax.
//   attn_lse_merge_kernel  log-sum-exp merge of the tensor-core kernels'
//                      split rows: launched right after them as their
//                      programmatic dependent, one warp per row.
//   attn_merge_kernel  log-sum-exp merge of the CUDA-core kernel's partials.
//   wait_timeout_probe_kernel  the bounded pipeline wait on a phase nothing
//                      completes (pk_selftest_wait_timeout).
//
// Host side: the entry points, the automatic partition (pk_paged_attention_
// resolve_partition: fill the resident CTA slots once), the work-list
// planner (pk_attention_plan, pk_attention_work_items) and the launch-order
// helper.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <new>
#include <vector>

#include "pagedkv.h"
#include "pk_device.cuh"

// The resident-table scatter of cache_ops.cu with separate input and output
// lengths (library-internal).
extern "C" pk_status pkx_reshape_and_cache_advance(const void *k, const void *v,
                                                   const int64_t *slot_mapping, int32_t num_tokens,
                                                   void *k_cache, void *v_cache,
                                                   const pk_cache_desc *desc,
                                                   int32_t *block_tables,
                                                   int32_t max_blocks_per_seq,
                                                   const int32_t *lens_in, int32_t *lens_out,
                                                   void *stream);

namespace {

__device__ int g_attn_error;

constexpr int kMaxGroup = 8;

struct AttnParams {
  void *out;                 // [S, Hq, D] (dtype of q)
  const void *q;             // [S, Hq, D]
  const void *k_cache;       // [N, B, Hk, D]
  const void *v_cache;       // [N, B, Hk, D]
  const int32_t *tables;     // [S, max_blocks]
  const int32_t *ctx_lens;   // [S]
  float *ws_acc;             // [S, Hq, P, D] unnormalised partial outputs
  float *ws_m;               // [S, Hq, P] running maxima (log2 domain)
  float *ws_l;               // [S, Hq, P] softmax denominators
  const int32_t *order;      // [S] launch order of the sequences, or null
  // Cascade (shared-prefix) attention: the first seq_prefix[s] tokens of
  // sequence s are attended by its group's prefix work; partials of prefix
  // partitions use workspace slots [0, prefix_slots), the rest follow.
  const int32_t *seq_prefix;     // [S] or null
  const int32_t *group_offsets;  // [num_groups + 1]
  const int32_t *group_members;  // batch positions of the groups' members
  const int32_t *group_prefix;   // [num_groups] shared tokens per group
  int32_t prefix_slots;
  float scale_log2;          // scale * log2(e)
  int32_t num_seqs, num_q_heads, num_kv_heads, group;
  int32_t block_size, max_blocks, num_blocks;
  int32_t partition;         // tokens per partition
  int32_t num_partitions;    // P (1 = no split: write `out` directly)
  // Work list: CTA (h, y) serves (sequence items[2y], partition items[2y+1])
  // instead of the (sequence, partition) grid; null when not used.
  const int32_t *items;
  int32_t num_items;
  // Fused scatter: token s of new_k / new_v ([S, Hk, D]) is sequence s's last
  // token, to be written to slot new_slots[s] before it is read; null when the
  // caller scattered already.
  const void *new_k;
  const void *new_v;
  const int64_t *new_slots;
  // Advance mode (device-resident tables; needs new_k): ctx_lens holds the
  // lengths before the step's token, and the CTA holding sequence s's new
  // token for KV head 0 writes the token's block into tables[s] and the new
  // length into lens_out[s]; null otherwise.
  int32_t *lens_out;
};

// Context length of sequence s, clamped to what the table and the grid can
// hold. Invalid lengths are recorded once (by the CTA for partition 0, head 0).
__device__ __forceinline__ int context_len(const AttnParams &p, int s, bool record) {
  int c = __ldg(p.ctx_lens + s) + (p.lens_out ? 1 : 0);  // advance mode counts the new token
  const int cap = min(p.max_blocks * p.block_size, p.num_partitions * p.partition);
  if (c < 1 || c > cap) {
    if (record) pk::record_error(&g_attn_error, PK_DEVERR_CONTEXT, s);
    c = c < 1 ? 0 : cap;
  }
  return c;
}

// A CTA's place in its kernel's (KV head, sequence or group, partition)
// grid: the hardware block index, or a virtual one when one launch runs CTAs
// of two kinds (cascade attention). nz is the grid's partition extent.
struct CtaCoord {
  int x, y, z, nz;
};

__device__ __forceinline__ CtaCoord hw_cta() {
  return CtaCoord{int(blockIdx.x), int(blockIdx.y), int(blockIdx.z), int(gridDim.z)};
}

// The sequence this CTA serves: order[c.y] when a launch order is given (an
// out-of-range entry is recorded and falls back to c.y).
__device__ __forceinline__ int launch_seq(const AttnParams &p, const CtaCoord &c) {
  const int y = c.y;
  if (!p.order) return y;
  const int s = __ldg(p.order + y);
  if (s < 0 || s >= p.num_seqs) {
    if (c.x == 0 && c.z == 0 && threadIdx.x == 0)
      pk::record_error(&g_attn_error, PK_DEVERR_ORDER, y);
    return y;
  }
  return s;
}

// The (sequence, partition) this CTA serves. With a work list: item c.y (an
// entry outside the batch or the partition count is recorded and the CTA does
// nothing). Otherwise sequence launch_seq() and partition c.nz - 1 - c.z:
// partitions launch last-first, since the higher ones exist only for the
// longest sequences.
__device__ __forceinline__ bool work_of(const AttnParams &p, const CtaCoord &c, int &s, int &part) {
  if (p.items) {
    const int y = c.y;
    s = __ldg(p.items + 2 * y);
    part = __ldg(p.items + 2 * y + 1);
    if (s < 0 || s >= p.num_seqs || part < 0 || part >= p.num_partitions - p.prefix_slots) {
      if (c.x == 0 && threadIdx.x == 0) pk::record_error(&g_attn_error, PK_DEVERR_ORDER, y);
      return false;
    }
    return true;
  }
  part = c.nz - 1 - c.z;
  s = launch_seq(p, c);
  return true;
}

// Log-sum-exp merge of the partials of query heads h0 .. h0+nh-1 of
// sequence s held in workspace slots [0, na) and [b0, b0 + nb), spread over
// `nthreads` threads (thread `tid`), four elements per step.
// M = max_p m_p, L = sum_p l_p 2^(m_p - M), out = sum_p acc_p 2^(m_p - M) / L.
// Partials are read from L2 (written by other CTAs of the same call).
template <typename T, int D>
__device__ __forceinline__ void merge_partials(const AttnParams &p, int s, int h0, int nh, int na,
                                               int b0, int nb, int tid, int nthreads) {
  const int np = na + nb;
  auto slot = [&](int q) { return q < na ? q : b0 + (q - na); };
  for (int idx = tid; idx < nh * (D / 4); idx += nthreads) {
    const int h = h0 + idx / (D / 4), i = (idx % (D / 4)) * 4;
    const size_t row = size_t(s) * p.num_q_heads + h;
    const float *mrow = p.ws_m + row * p.num_partitions;
    const float *lrow = p.ws_l + row * p.num_partitions;
    const float *arow = p.ws_acc + row * p.num_partitions * D + i;
    float M = -INFINITY;
    for (int q = 0; q < np; ++q) M = fmaxf(M, __ldcg(mrow + slot(q)));
    float L = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    int q = 0;
    for (; q + 4 <= np; q += 4) {
      float4 x[4];
      float f[4], l[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int sl = slot(q + u);
        x[u] = __ldcg(reinterpret_cast<const float4 *>(arow + size_t(sl) * D));
        f[u] = __ldcg(mrow + sl);
        l[u] = __ldcg(lrow + sl);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float w = exp2f(f[u] - M);
        L = fmaf(l[u], w, L);
        acc.x = fmaf(x[u].x, w, acc.x);
        acc.y = fmaf(x[u].y, w, acc.y);
        acc.z = fmaf(x[u].z, w, acc.z);
        acc.w = fmaf(x[u].w, w, acc.w);
      }
    }
    for (; q < np; ++q) {
      const int sl = slot(q);
      const float4 x = __ldcg(reinterpret_cast<const float4 *>(arow + size_t(sl) * D));
      const float w = exp2f(__ldcg(mrow + sl) - M);
      L = fmaf(__ldcg(lrow + sl), w, L);
      acc.x = fmaf(x.x, w, acc.x);
      acc.y = fmaf(x.y, w, acc.y);
      acc.z = fmaf(x.z, w, acc.z);
      acc.w = fmaf(x.w, w, acc.w);
    }
    const float inv = 1.0f / L;
    T *o = static_cast<T *>(p.out) + row * D + i;
    pk::store_elem(o + 0, acc.x * inv);
    pk::store_elem(o + 1, acc.y * inv);
    pk::store_elem(o + 2, acc.z * inv);
    pk::store_elem(o + 3, acc.w * inv);
  }
}

// ---------------------------------------------------------------------------
// CUDA-core kernel (fp32 and bf16): one warp per token, lanes split the head
// dimension, dot products reduced with shuffles, online softmax per head.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(128) attn_simt_kernel(AttnParams p) {
  constexpr int NW = 4;
  constexpr int EPL = D / 32;  // elements per lane
  const CtaCoord c = hw_cta();
  const int kvh = c.x;
  int s, part;
  if (!work_of(p, c, s, part)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int ctx = context_len(p, s, part == 0 && kvh == 0 && threadIdx.x == 0);

  if (ctx == 0) {  // invalid length: zero output (split mode: the merge writes it)
    if (p.num_partitions == 1 && part == 0)
      for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x)
        pk::store_elem(static_cast<T *>(p.out) +
                           (size_t(s) * p.num_q_heads + kvh * G + idx / D) * D + idx % D,
                       0.0f);
    return;
  }
  const int start = part * p.partition;
  if (start >= ctx) return;
  const int end = min(ctx, start + p.partition);
  // A sequence that fits one partition is final here; the merge skips it.
  const bool single = ctx <= p.partition;

  float qv[kMaxGroup][EPL];
  float m[kMaxGroup], l[kMaxGroup], acc[kMaxGroup][EPL];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      acc[g][e] = 0.0f;
      qv[g][e] = 0.0f;
      if (g < G)
        qv[g][e] = pk::load_elem(static_cast<const T *>(p.q) +
                                 (size_t(s) * p.num_q_heads + kvh * G + g) * D + lane * EPL + e) *
                   p.scale_log2;
    }
  }

  const T *kc = static_cast<const T *>(p.k_cache);
  const T *vc = static_cast<const T *>(p.v_cache);
  const int32_t *trow = p.tables + size_t(s) * p.max_blocks;
  const int B = p.block_size;
  for (int t = start + warp; t < end; t += NW) {
    int phys = __ldg(trow + t / B);
    if (phys < 0 || phys >= p.num_blocks) {
      if (lane == 0) pk::record_error(&g_attn_error, PK_DEVERR_BLOCK_ID, s);
      continue;
    }
    const size_t row = ((size_t(phys) * B + t % B) * p.num_kv_heads + kvh) * D + lane * EPL;
    float kx[EPL], vx[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kx[e] = pk::load_elem(kc + row + e);
      vx[e] = pk::load_elem(vc + row + e);
    }
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) {
      if (g >= G) break;
      float dot = 0.0f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) dot = fmaf(qv[g][e], kx[e], dot);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      const float mn = fmaxf(m[g], dot);
      const float corr = exp2f(m[g] - mn);
      const float w = exp2f(dot - mn);
      l[g] = l[g] * corr + w;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(acc[g][e], corr, w * vx[e]);
      m[g] = mn;
    }
  }

  // Merge the four warps' running states.
  __shared__ float sm_m[NW][kMaxGroup], sm_l[NW][kMaxGroup];
  __shared__ float sm_o[NW][kMaxGroup][D];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    if (g >= G) break;
#pragma unroll
    for (int e = 0; e < EPL; ++e) sm_o[warp][g][lane * EPL + e] = acc[g][e];
    if (lane == 0) {
      sm_m[warp][g] = m[g];
      sm_l[warp][g] = l[g];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D, i = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w][g]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = exp2f(sm_m[w][g] - M);  // 0 for a warp that saw no token
      L = fmaf(sm_l[w][g], f, L);
      O = fmaf(sm_o[w][g][i], f, O);
    }
    const int h = kvh * G + g;
    if (single) {
      pk::store_elem(static_cast<T *>(p.out) + (size_t(s) * p.num_q_heads + h) * D + i, O / L);
    } else {
      const size_t r = (size_t(s) * p.num_q_heads + h) * p.num_partitions + part;
      p.ws_acc[r * D + i] = O;
      if (i == 0) {
        p.ws_m[r] = M;
        p.ws_l[r] = L;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Tensor-core kernel (bf16): TMA-staged K/V ring, mma.sync m16n8k16.
// ---------------------------------------------------------------------------
template <int D, int BS, int NW, int STAGES>
struct MmaShape {
  static constexpr int TPS = NW * 16;               // tokens per stage
  static constexpr int BPS = TPS / BS;              // blocks per stage
  static constexpr int HALVES = D / 64;             // 128-byte column slabs per row
  static constexpr int SLAB_BYTES = TPS * 128;      // one slab of one stage
  static constexpr int KV_BYTES = HALVES * SLAB_BYTES;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;  // K then V
  static constexpr int KSTEPS = D / 16;
  static constexpr int OUT_STRIDE = D + 4;          // padded row of the merge buffer
  static constexpr int MERGE_BYTES = NW * kMaxGroup * (OUT_STRIDE + 2) * 4 + 16;
  static constexpr int BAR_BYTES = 2 * STAGES * 8 + 8;  // full, empty, scatter-done
  static constexpr int SMEM_BYTES = 1024 + BAR_BYTES +
                                    (STAGES * STAGE_BYTES > MERGE_BYTES ? STAGES * STAGE_BYTES
                                                                        : MERGE_BYTES);
  static_assert(D % 64 == 0, "head_dim must be a multiple of 64");
  static_assert(BS <= TPS && TPS % BS == 0 && BPS <= 32, "block size must divide the stage");
  // The producer reads table entries in 32-entry chunks, one stage's blocks
  // never straddling two chunks.
  static_assert(32 % BPS == 0, "blocks per stage must divide 32");
};

// One warp's 16-token tile: scores S^T (16 tokens x 8 query columns) =
// K_tile Q^T, the online-softmax update of the running maxima m and sums l
// (two query columns per lane: 2qd, 2qd+1) with the accumulator rescaled, and
// O^T (D x 8) += V^T P^T. K and V are stored as D/64 slabs of `slab` bytes
// (128-byte rows, 128B-swizzled); the tile is rows row0 .. row0+15, of which
// the first nvalid (>= 1) hold tokens. Rows past them may hold stale or
// unloaded data: their scores are -inf and their V rows are zeroed first, so a
// zero weight never meets a NaN.
template <int KSTEPS>
__device__ __forceinline__ void attn_tile(uint32_t kbase, uint32_t vbase, int slab, int row0,
                                          int nvalid, const uint32_t (&qb)[KSTEPS][2],
                                          float (&o)[KSTEPS][4], float &m0, float &m1, float &l0,
                                          float &l1, float sl, int lane) {
  constexpr int HALVES = KSTEPS / 4;
  const int rw = lane >> 2;
  const int mi = lane >> 3, r8 = lane & 7;
  if (nvalid < 16) {
    const int nz = (16 - nvalid) * HALVES * 8;
    for (int idx = lane; idx < nz; idx += 32) {
      const int r = row0 + nvalid + idx / (HALVES * 8);
      const int c = idx % (HALVES * 8);
      const uint32_t a = vbase + (c >> 3) * slab + r * 128 + (c & 7) * 16;
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
    }
    __syncwarp();
  }
  // S^T = K_tile (16 x D) * Q^T (D x 8), as two independent accumulation
  // chains (even and odd k-steps).
  float sacc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
  for (int ks = 0; ks < KSTEPS; ++ks) {
    const int r = row0 + (mi & 1) * 8 + r8;
    const int chunk = ks * 2 + (mi >> 1);
    const uint32_t a = kbase + (chunk >> 3) * slab + r * 128 + (((chunk & 7) ^ (r & 7)) << 4);
    uint32_t a0, a1, a2, a3;
    pk::ldmatrix_x4(a, a0, a1, a2, a3);
    pk::mma_bf16_16816(sacc[ks & 1], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
  }
  float x0 = (sacc[0][0] + sacc[1][0]) * sl, x1 = (sacc[0][1] + sacc[1][1]) * sl;
  float x2 = (sacc[0][2] + sacc[1][2]) * sl, x3 = (sacc[0][3] + sacc[1][3]) * sl;
  if (rw >= nvalid) x0 = x1 = -INFINITY;
  if (rw + 8 >= nvalid) x2 = x3 = -INFINITY;
  float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: row 0 is valid
  const float c0 = exp2f(m0 - mn0), c1 = exp2f(m1 - mn1);
  const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
  const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
  // Softmax weights enter the PV product as a bf16 pair hi + lo: rounding
  // them to one bf16 would put ~2^-9 relative error on every output.
  const uint32_t w01 = pk::pack_bf16x2(p0, p1);
  const uint32_t w23 = pk::pack_bf16x2(p2, p3);
  const uint32_t r01 = pk::pack_bf16x2(p0 - pk::bf16_lo(w01), p1 - pk::bf16_hi(w01));
  const uint32_t r23 = pk::pack_bf16x2(p2 - pk::bf16_lo(w23), p3 - pk::bf16_hi(w23));
  l0 = fmaf(l0, c0, p0 + p2);
  l1 = fmaf(l1, c1, p1 + p3);
  m0 = mn0;
  m1 = mn1;
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt) {
    o[mt][0] *= c0;
    o[mt][1] *= c1;
    o[mt][2] *= c0;
    o[mt][3] *= c1;
  }
  // P^T (16 tokens x 8 heads) as the B operand: transpose the C fragments.
  const uint32_t b0 = pk::movmatrix_trans(w01);
  const uint32_t b1 = pk::movmatrix_trans(w23);
  const uint32_t e0 = pk::movmatrix_trans(r01);
  const uint32_t e1 = pk::movmatrix_trans(r23);
  // O^T (D x 8) += V^T (D x 16 tokens) * P^T: all hi products first, then
  // all lo products, so consecutive MMAs never share an accumulator.
  uint32_t va[KSTEPS][4];
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt) {
    const int r = row0 + (mi >> 1) * 8 + r8;
    const int chunk = mt * 2 + (mi & 1);
    const uint32_t a = vbase + (chunk >> 3) * slab + r * 128 + (((chunk & 7) ^ (r & 7)) << 4);
    pk::ldmatrix_x4_trans(a, va[mt][0], va[mt][1], va[mt][2], va[mt][3]);
  }
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt)
    pk::mma_bf16_16816(o[mt], va[mt][0], va[mt][1], va[mt][2], va[mt][3], b0, b1);
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt)
    pk::mma_bf16_16816(o[mt], va[mt][0], va[mt][1], va[mt][2], va[mt][3], e0, e1);
}

// The work of one attn_mma_kernel CTA at grid coordinate c.
template <int D, int BS, int NW, int STAGES>
__device__ __forceinline__ void mma_cta(const AttnParams &p, const CUtensorMap *kmap,
                                        const CUtensorMap *vmap, const CtaCoord c) {
  using S = MmaShape<D, BS, NW, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = pk::smem_addr(smem_raw);
  const uint32_t bars = (raw + 7u) & ~7u;
  const uint32_t stages = (bars + S::BAR_BYTES + 1023u) & ~1023u;
  auto full_bar = [&](int i) { return bars + 8u * i; };
  auto empty_bar = [&](int i) { return bars + 8u * (STAGES + i); };
  const uint32_t scatter_bar = bars + 8u * (2 * STAGES);

  // The caller's work list, or the grid in the caller's sequence order (longest
  // first keeps the longest work from trailing the launch).
  const int kvh = c.x;
  int s, part;
  if (!work_of(p, c, s, part)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int ctx = context_len(p, s, part == 0 && kvh == 0 && threadIdx.x == 0);
  if (ctx == 0) {  // invalid length (recorded): a zero row, nothing to merge
    if (part == 0)
      for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x)
        static_cast<__nv_bfloat16 *>(p.out)[(size_t(s) * p.num_q_heads + kvh * G + idx / D) * D +
                                            idx % D] = __float2bfloat16_rn(0.0f);
    return;
  }
  // Tokens [0, pre) belong to the sequence's shared prefix (cascade mode);
  // this CTA covers partition `part` of the rest.
  const int pre = p.seq_prefix ? min(max(__ldg(p.seq_prefix + s), 0), ctx) : 0;
  const int start = pre + part * p.partition;
  if (start >= ctx) return;
  const int end = min(ctx, start + p.partition);
  const int nst = (end - start + S::TPS - 1) / S::TPS;
  const int npre = (pre + p.partition - 1) / p.partition;
  const int nsuf = (ctx - pre + p.partition - 1) / p.partition;

  // Fused scatter: the CTA whose partition holds the sequence's new (last)
  // token writes that token's K and V for this KV head -- exactly the slice
  // it reads. Consumer warp 0 writes them at its start and arrives on
  // scatter_bar after a proxy fence; the producer waits on it only before the
  // last stage's copies (the tail block), so the write costs no latency.
  const bool fuse = p.new_k && end == ctx;
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      pk::mbar_init(full_bar(i), 1);
      pk::mbar_init(empty_bar(i), NW);
    }
    pk::mbar_init(scatter_bar, 32);
    pk::fence_barrier_init();
  }
  __syncthreads();

  if (fuse && warp == 0) {
    constexpr int VEC = D * 2 / 16;  // 16-byte vectors of one head's row
    const int64_t slot = __ldg(p.new_slots + s);
    if (p.lens_out && kvh == 0 && lane == 0) {
      // Advance mode: the step's bookkeeping on the resident tables. The
      // entry of the block holding position pos = ctx - 1 becomes slot / B
      // (a freshly opened block and a copy-on-write replacement alike) and the
      // length becomes ctx. A slot that is not at offset pos mod B means the
      // tables are out of step with the host: the row keeps its length.
      const int pos = ctx - 1;
      if (slot >= 0 && slot < int64_t(p.num_blocks) * BS && slot % BS == pos % BS) {
        const_cast<int32_t *>(p.tables)[size_t(s) * p.max_blocks + pos / BS] = int32_t(slot / BS);
        p.lens_out[s] = ctx;
      } else {
        pk::record_error(&g_attn_error, PK_DEVERR_CONTEXT, s);
        p.lens_out[s] = pos;
      }
    }
    if (slot < 0 || slot >= int64_t(p.num_blocks) * BS) {
      if (lane == 0) pk::record_error(&g_attn_error, PK_DEVERR_SLOT, s);
    } else if (lane < 2 * VEC) {
      const bool is_v = lane >= VEC;
      const int j = is_v ? lane - VEC : lane;
      const size_t row = size_t(s) * p.num_kv_heads + kvh;
      const uint4 *src = static_cast<const uint4 *>(is_v ? p.new_v : p.new_k) + row * VEC + j;
      uint4 *dst = static_cast<uint4 *>(const_cast<void *>(is_v ? p.v_cache : p.k_cache)) +
                   (size_t(slot) * p.num_kv_heads + kvh) * VEC + j;
      *dst = __ldg(src);
      pk::fence_proxy_async();
    }
    pk::mbar_arrive(scatter_bar);
  }

  if (warp == NW) {
    // ---------------- producer warp ----------------
    if (lane == 0) {
      pk::prefetch_tensormap(kmap);
      pk::prefetch_tensormap(vmap);
    }
    // The partition's table entries are read ahead in coalesced 32-entry
    // chunks (one entry per lane, one chunk in reserve), so no stage waits on
    // a dependent global load before its copies can be issued.
    const int32_t *trow = p.tables + size_t(s) * p.max_blocks + start / BS;
    const int nb = (end - start + BS - 1) / BS;  // blocks of this partition
    // Advance mode: the block holding the new token (partition-relative index
    // tail) is the token's slot / B -- its table entry is written during this
    // launch, so it is not read. A slot that is not at offset pos mod B of a
    // pool block (recorded by the bookkeeping above) reads block 0 instead.
    int tail = -1, tail_blk = 0;
    if (p.lens_out && fuse) {
      const int64_t slot = __ldg(p.new_slots + s);
      const int pos = ctx - 1;
      tail = pos / BS - start / BS;
      if (slot >= 0 && slot < int64_t(p.num_blocks) * BS && slot % BS == pos % BS)
        tail_blk = int(slot / BS);
    }
    auto entry = [&](int j) { return j == tail ? tail_blk : (j < nb ? __ldg(trow + j) : 0); };
    int cur = entry(lane);
    int nxt = entry(32 + lane);
    int chunk = 0;
    int issued = 0;
    for (int st = 0; st < nst; ++st) {
      const int slot = st % STAGES;
      const int b0 = st * S::BPS;  // first block of the stage, within the partition
      if (b0 >= 32 * (chunk + 1)) {
        ++chunk;
        cur = nxt;
        nxt = entry(32 * (chunk + 1) + lane);
      }
      const int mine = __shfl_sync(0xffffffffu, cur, (b0 & 31) + min(lane, S::BPS - 1));
      if (st >= STAGES && !pk::mbar_wait(empty_bar(slot), ((st / STAGES) - 1) & 1)) {
        if (lane == 0) pk::record_error(&g_attn_error, PK_DEVERR_TIMEOUT, s);
        break;
      }
      if (fuse && st == nst - 1 && !pk::mbar_wait(scatter_bar, 0)) {
        if (lane == 0) pk::record_error(&g_attn_error, PK_DEVERR_TIMEOUT, s);
        break;
      }
      const int tok0 = start + st * S::TPS;
      const int nblk = min(S::BPS, (end - tok0 + BS - 1) / BS);
      if (lane == 0)
        pk::mbar_arrive_expect_tx(full_bar(slot), uint32_t(nblk * S::HALVES * 2 * BS * 128));
      __syncwarp();
      if (lane < nblk) {
        int phys = mine;
        if (phys < 0 || phys >= p.num_blocks) {
          pk::record_error(&g_attn_error, PK_DEVERR_BLOCK_ID, s);
          phys = 0;  // stay in bounds and keep the byte count; the result is flagged
        }
        const uint32_t kdst = stages + slot * S::STAGE_BYTES + lane * BS * 128;
#pragma unroll
        for (int h = 0; h < S::HALVES; ++h) {
          pk::tma_load_3d(kdst + h * S::SLAB_BYTES, kmap, full_bar(slot), h * 64, kvh, phys * BS);
          pk::tma_load_3d(kdst + S::KV_BYTES + h * S::SLAB_BYTES, vmap, full_bar(slot), h * 64,
                          kvh, phys * BS);
        }
      }
      issued = st + 1;
    }
    // Let every issued copy land before the warp leaves.
    if (lane == 0)
      for (int st = max(0, issued - STAGES); st < issued; ++st)
        pk::mbar_wait(full_bar(st % STAGES), (st / STAGES) & 1);
    return;
  }

  // ---------------- consumer warps ----------------
  const int qd = lane & 3;   // quad lane: owns heads 2qd, 2qd+1 of the C fragments
  const int rw = lane >> 2;  // row within an 8-row group
  // Q^T as the B operand (k = head_dim, n = head within the group).
  uint32_t qb[S::KSTEPS][2];
  {
    const __nv_bfloat16 *qrow = static_cast<const __nv_bfloat16 *>(p.q) +
                                (size_t(s) * p.num_q_heads + kvh * G + min(rw, G - 1)) * D;
#pragma unroll
    for (int ks = 0; ks < S::KSTEPS; ++ks) {
      const uint32_t a = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 2 * qd);
      const uint32_t b = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + 2 * qd);
      qb[ks][0] = rw < G ? a : 0u;
      qb[ks][1] = rw < G ? b : 0u;
    }
  }
  float o[S::KSTEPS][4];
#pragma unroll
  for (int mt = 0; mt < S::KSTEPS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
  const float sl = p.scale_log2;
  const int row0 = warp * 16;

  for (int st = 0; st < nst; ++st) {
    const int slot = st % STAGES;
    if (!pk::mbar_wait(full_bar(slot), (st / STAGES) & 1)) {
      if (lane == 0) pk::record_error(&g_attn_error, PK_DEVERR_TIMEOUT, s);
      break;
    }
    const uint32_t kbase = stages + slot * S::STAGE_BYTES;
    const uint32_t vbase = kbase + S::KV_BYTES;
    const int nvalid = end - (start + st * S::TPS + row0);  // valid rows of this warp's tile
    if (nvalid > 0)
      attn_tile<S::KSTEPS>(kbase, vbase, S::SLAB_BYTES, row0, nvalid, qb, o, m0, m1, l0, l1, sl,
                           lane);
    __syncwarp();
    if (lane == 0) pk::mbar_arrive(empty_bar(slot));
  }

  // Row sums over the 16 tokens of each tile live spread over the 8 lanes
  // that share a quad index.
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }

  // Merge the consumer warps' states in shared memory (the stage ring is free:
  // every copy has landed and been consumed).
  pk::named_barrier(1, NW * 32);
  float *sm_o = reinterpret_cast<float *>(smem_raw + (stages - raw));
  float *sm_m = sm_o + NW * kMaxGroup * S::OUT_STRIDE;
  float *sm_l = sm_m + NW * kMaxGroup;
#pragma unroll
  for (int mt = 0; mt < S::KSTEPS; ++mt) {
    float *base = sm_o + (warp * kMaxGroup + 2 * qd) * S::OUT_STRIDE + mt * 16 + rw;
    base[0] = o[mt][0];
    base[S::OUT_STRIDE] = o[mt][1];
    base[8] = o[mt][2];
    base[S::OUT_STRIDE + 8] = o[mt][3];
  }
  if (rw == 0) {
    sm_m[warp * kMaxGroup + 2 * qd] = m0;
    sm_m[warp * kMaxGroup + 2 * qd + 1] = m1;
    sm_l[warp * kMaxGroup + 2 * qd] = l0;
    sm_l[warp * kMaxGroup + 2 * qd + 1] = l1;
  }
  pk::named_barrier(1, NW * 32);
  for (int idx = threadIdx.x; idx < G * (D / 2); idx += NW * 32) {
    const int g = idx / (D / 2), i = (idx % (D / 2)) * 2;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w * kMaxGroup + g]);
    float L = 0.0f, O0 = 0.0f, O1 = 0.0f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = exp2f(sm_m[w * kMaxGroup + g] - M);
      const float *row = sm_o + (w * kMaxGroup + g) * S::OUT_STRIDE + i;
      L = fmaf(sm_l[w * kMaxGroup + g], f, L);
      O0 = fmaf(row[0], f, O0);
      O1 = fmaf(row[1], f, O1);
    }
    const int h = kvh * G + g;
    if (npre + nsuf == 1) {  // a single part: final output, no merge
      const float inv = 1.0f / L;
      *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(p.out) +
                                          (size_t(s) * p.num_q_heads + h) * D + i) =
          __floats2bfloat162_rn(O0 * inv, O1 * inv);
    } else {
      const size_t r = (size_t(s) * p.num_q_heads + h) * p.num_partitions + p.prefix_slots + part;
      *reinterpret_cast<float2 *>(p.ws_acc + r * D + i) = make_float2(O0, O1);
      if (i == 0) {
        p.ws_m[r] = M;
        p.ws_l[r] = L;
      }
    }
  }
}

template <int D, int BS, int NW, int STAGES>
__global__ void __launch_bounds__((NW + 1) * 32)
    attn_mma_kernel(AttnParams p, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap) {
  pk::launch_dependents();  // the split-K merge may be scheduled as this grid drains
  mma_cta<D, BS, NW, STAGES>(p, &kmap, &vmap, hw_cta());
}

// ---------------------------------------------------------------------------
// Cascade attention, shared-prefix part (bf16, tensor cores).
//
// One CTA per (KV head, group, partition of the group's shared prefix): the
// prefix blocks are streamed once (from the first member's table -- every
// member names the same blocks) and scored against the queries of every
// member of the group: up to 16 query columns (members x G heads), two MMA
// n-tiles. Each column's partial goes to its sequence's prefix slot; the
// members' suffix work (attn_mma_kernel in cascade mode) fills the other
// slots, and attn_lse_merge_kernel merges them ("PagedAttention" S06, "In
// production": the shared prefix batched separately from the divergent
// suffixes).
// ---------------------------------------------------------------------------
// The work of one prefix CTA of cascade attention at coordinate c (KV head,
// group, prefix partition).
template <int D, int BS, int NW, int STAGES>
__device__ __forceinline__ void prefix_cta(const AttnParams &p, const CUtensorMap *kmap,
                                           const CUtensorMap *vmap, const CtaCoord c) {
  using S = MmaShape<D, BS, NW, STAGES>;
  constexpr int NT = 2;            // n-tiles of 8 query columns
  constexpr int NC = 8 * NT;       // query columns per CTA
  constexpr int MSTRIDE = S::OUT_STRIDE;
  static_assert(NW * NC * (MSTRIDE + 2) * 4 + 64 <= STAGES * S::STAGE_BYTES,
                "merge buffer must fit the stage ring");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = pk::smem_addr(smem_raw);
  const uint32_t bars = (raw + 7u) & ~7u;
  const uint32_t stages = (bars + S::BAR_BYTES + 1023u) & ~1023u;
  auto full_bar = [&](int i) { return bars + 8u * i; };
  auto empty_bar = [&](int i) { return bars + 8u * (STAGES + i); };

  const int kvh = c.x, grp = c.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int g0 = __ldg(p.group_offsets + grp);
  const int nm = __ldg(p.group_offsets + grp + 1) - g0;
  const int lead = __ldg(p.group_members + g0);
  const int pre = __ldg(p.group_prefix + grp);
  const int npre_g = (pre + p.partition - 1) / p.partition;
  const int part = c.z;
  if (part >= npre_g || nm <= 0 || nm * G > NC) return;
  const int start = part * p.partition;
  const int end = min(pre, start + p.partition);
  if (start >= end) return;
  const int nst = (end - start + S::TPS - 1) / S::TPS;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      pk::mbar_init(full_bar(i), 1);
      pk::mbar_init(empty_bar(i), NW);
    }
    pk::fence_barrier_init();
  }
  __syncthreads();

  if (warp == NW) {
    // ---------------- producer warp (as in attn_mma_kernel) ----------------
    if (lane == 0) {
      pk::prefetch_tensormap(kmap);
      pk::prefetch_tensormap(vmap);
    }
    const int32_t *trow = p.tables + size_t(lead) * p.max_blocks + start / BS;
    const int nb = (end - start + BS - 1) / BS;
    int cur = lane < nb ? __ldg(trow + lane) : 0;
    int nxt = 32 + lane < nb ? __ldg(trow + 32 + lane) : 0;
    int chunk = 0;
    int issued = 0;
    for (int st = 0; st < nst; ++st) {
      const int slot = st % STAGES;
      const int b0 = st * S::BPS;
      if (b0 >= 32 * (chunk + 1)) {
        ++chunk;
        cur = nxt;
        const int j = 32 * (chunk + 1) + lane;
        nxt = j < nb ? __ldg(trow + j) : 0;
      }
      const int mine = __shfl_sync(0xffffffffu, cur, (b0 & 31) + min(lane, S::BPS - 1));
      if (st >= STAGES && !pk::mbar_wait(empty_bar(slot), ((st / STAGES) - 1) & 1)) {
        if (lane == 0) pk::record_error(&g_attn_error, PK_DEVERR_TIMEOUT, lead);
        break;
      }
      const int tok0 = start + st * S::TPS;
      const int nblk = min(S::BPS, (end - tok0 + BS - 1) / BS);
      if (lane == 0)
        pk::mbar_arrive_expect_tx(full_bar(slot), uint32_t(nblk * S::HALVES * 2 * BS * 128));
      __syncwarp();
      if (lane < nblk) {
        int phys = mine;
        if (phys < 0 || phys >= p.num_blocks) {
          pk::record_error(&g_attn_error, PK_DEVERR_BLOCK_ID, lead);
          phys = 0;
        }
        const uint32_t kdst = stages + slot * S::STAGE_BYTES + lane * BS * 128;
#pragma unroll
        for (int h = 0; h < S::HALVES; ++h) {
          pk::tma_load_3d(kdst + h * S::SLAB_BYTES, kmap, full_bar(slot), h * 64, kvh, phys * BS);
          pk::tma_load_3d(kdst + S::KV_BYTES + h * S::SLAB_BYTES, vmap, full_bar(slot), h * 64,
                          kvh, phys * BS);
        }
      }
      issued = st + 1;
    }
    if (lane == 0)
      for (int st = max(0, issued - STAGES); st < issued; ++st)
        pk::mbar_wait(full_bar(st % STAGES), (st / STAGES) & 1);
    return;
  }

  // ---------------- consumer warps ----------------
  const int qd = lane & 3, rw = lane >> 2;
  const int mi = lane >> 3, r8 = lane & 7;
  const int ncol = nm * G;
  // Q^T of the group's columns: column c = member c / G, head c % G.
  uint32_t qb[NT][S::KSTEPS][2];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int c = t * 8 + rw;
    const int cc = min(c, ncol - 1);
    const int mem = __ldg(p.group_members + g0 + cc / G);
    const __nv_bfloat16 *qrow = static_cast<const __nv_bfloat16 *>(p.q) +
                                (size_t(mem) * p.num_q_heads + kvh * G + cc % G) * D;
#pragma unroll
    for (int ks = 0; ks < S::KSTEPS; ++ks) {
      const uint32_t a = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 2 * qd);
      const uint32_t b = *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + 2 * qd);
      qb[t][ks][0] = c < ncol ? a : 0u;
      qb[t][ks][1] = c < ncol ? b : 0u;
    }
  }
  float o[S::KSTEPS][NT][4];
#pragma unroll
  for (int mt = 0; mt < S::KSTEPS; ++mt)
#pragma unroll
    for (int t = 0; t < NT; ++t) o[mt][t][0] = o[mt][t][1] = o[mt][t][2] = o[mt][t][3] = 0.0f;
  float m[NT][2], l[NT][2];
#pragma unroll
  for (int t = 0; t < NT; ++t) m[t][0] = m[t][1] = -INFINITY, l[t][0] = l[t][1] = 0.0f;
  const float sl = p.scale_log2;
  const int row0 = warp * 16;

  for (int st = 0; st < nst; ++st) {
    const int slot = st % STAGES;
    if (!pk::mbar_wait(full_bar(slot), (st / STAGES) & 1)) {
      if (lane == 0) pk::record_error(&g_attn_error, PK_DEVERR_TIMEOUT, lead);
      break;
    }
    const uint32_t kbase = stages + slot * S::STAGE_BYTES;
    const uint32_t vbase = kbase + S::KV_BYTES;
    const int nvalid = end - (start + st * S::TPS + row0);
    if (nvalid > 0) {
      if (nvalid < 16) {
        const int nz = (16 - nvalid) * S::HALVES * 8;
        for (int idx = lane; idx < nz; idx += 32) {
          const int r = row0 + nvalid + idx / (S::HALVES * 8);
          const int c = idx % (S::HALVES * 8);
          const uint32_t a = vbase + (c >> 3) * S::SLAB_BYTES + r * 128 + (c & 7) * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
        }
        __syncwarp();
      }
      // S^T for both n-tiles from one pass over the K tile.
      float sacc[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) sacc[t][0] = sacc[t][1] = sacc[t][2] = sacc[t][3] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < S::KSTEPS; ++ks) {
        const int r = row0 + (mi & 1) * 8 + r8;
        const int chunk = ks * 2 + (mi >> 1);
        const uint32_t a = kbase + (chunk >> 3) * S::SLAB_BYTES + r * 128 +
                           (((chunk & 7) ^ (r & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        pk::ldmatrix_x4(a, a0, a1, a2, a3);
#pragma unroll
        for (int t = 0; t < NT; ++t)
          pk::mma_bf16_16816(sacc[t], a0, a1, a2, a3, qb[t][ks][0], qb[t][ks][1]);
      }
      uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float x0 = sacc[t][0] * sl, x1 = sacc[t][1] * sl, x2 = sacc[t][2] * sl, x3 = sacc[t][3] * sl;
        if (rw >= nvalid) x0 = x1 = -INFINITY;
        if (rw + 8 >= nvalid) x2 = x3 = -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[t][0], mx0), mn1 = fmaxf(m[t][1], mx1);
        const float c0 = exp2f(m[t][0] - mn0), c1 = exp2f(m[t][1] - mn1);
        const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
        const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
        const uint32_t w01 = pk::pack_bf16x2(p0, p1);
        const uint32_t w23 = pk::pack_bf16x2(p2, p3);
        const uint32_t r01 = pk::pack_bf16x2(p0 - pk::bf16_lo(w01), p1 - pk::bf16_hi(w01));
        const uint32_t r23 = pk::pack_bf16x2(p2 - pk::bf16_lo(w23), p3 - pk::bf16_hi(w23));
        l[t][0] = fmaf(l[t][0], c0, p0 + p2);
        l[t][1] = fmaf(l[t][1], c1, p1 + p3);
        m[t][0] = mn0;
        m[t][1] = mn1;
#pragma unroll
        for (int mt = 0; mt < S::KSTEPS; ++mt) {
          o[mt][t][0] *= c0;
          o[mt][t][1] *= c1;
          o[mt][t][2] *= c0;
          o[mt][t][3] *= c1;
        }
        bh[t][0] = pk::movmatrix_trans(w01);
        bh[t][1] = pk::movmatrix_trans(w23);
        bl[t][0] = pk::movmatrix_trans(r01);
        bl[t][1] = pk::movmatrix_trans(r23);
      }
#pragma unroll
      for (int mt = 0; mt < S::KSTEPS; ++mt) {
        const int r = row0 + (mi >> 1) * 8 + r8;
        const int chunk = mt * 2 + (mi & 1);
        const uint32_t a = vbase + (chunk >> 3) * S::SLAB_BYTES + r * 128 +
                           (((chunk & 7) ^ (r & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        pk::ldmatrix_x4_trans(a, a0, a1, a2, a3);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          pk::mma_bf16_16816(o[mt][t], a0, a1, a2, a3, bh[t][0], bh[t][1]);
          pk::mma_bf16_16816(o[mt][t], a0, a1, a2, a3, bl[t][0], bl[t][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) pk::mbar_arrive(empty_bar(slot));
  }

#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l[t][0] += __shfl_xor_sync(0xffffffffu, l[t][0], off);
      l[t][1] += __shfl_xor_sync(0xffffffffu, l[t][1], off);
    }

  // Merge the consumer warps' states per column (the stage ring is free).
  pk::named_barrier(1, NW * 32);
  float *sm_o = reinterpret_cast<float *>(smem_raw + (stages - raw));
  float *sm_m = sm_o + NW * NC * MSTRIDE;
  float *sm_l = sm_m + NW * NC;
#pragma unroll
  for (int mt = 0; mt < S::KSTEPS; ++mt)
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float *base = sm_o + (warp * NC + t * 8 + 2 * qd) * MSTRIDE + mt * 16 + rw;
      base[0] = o[mt][t][0];
      base[MSTRIDE] = o[mt][t][1];
      base[8] = o[mt][t][2];
      base[MSTRIDE + 8] = o[mt][t][3];
    }
  if (rw == 0) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      sm_m[warp * NC + t * 8 + 2 * qd] = m[t][0];
      sm_m[warp * NC + t * 8 + 2 * qd + 1] = m[t][1];
      sm_l[warp * NC + t * 8 + 2 * qd] = l[t][0];
      sm_l[warp * NC + t * 8 + 2 * qd + 1] = l[t][1];
    }
  }
  pk::named_barrier(1, NW * 32);
  for (int idx = threadIdx.x; idx < ncol * (D / 2); idx += NW * 32) {
    const int c = idx / (D / 2), i = (idx % (D / 2)) * 2;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w * NC + c]);
    float L = 0.0f, O0 = 0.0f, O1 = 0.0f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = exp2f(sm_m[w * NC + c] - M);
      const float *row = sm_o + (w * NC + c) * MSTRIDE + i;
      L = fmaf(sm_l[w * NC + c], f, L);
      O0 = fmaf(row[0], f, O0);
      O1 = fmaf(row[1], f, O1);
    }
    const int mem = __ldg(p.group_members + g0 + c / G);
    const size_t r = (size_t(mem) * p.num_q_heads + kvh * G + c % G) * p.num_partitions + part;
    *reinterpret_cast<float2 *>(p.ws_acc + r * D + i) = make_float2(O0, O1);
    if (i == 0) {
      p.ws_m[r] = M;
      p.ws_l[r] = L;
    }
  }
}

// Cascade attention in one launch: CTAs [0, npre) are prefix CTAs (KV head
// fastest, then group, then prefix partition), the rest are suffix CTAs of
// attn_mma_kernel in cascade mode (KV head fastest, then sequence in the
// launch order, then partition, last first). The long prefix work starts
// first and the short suffix work fills the SMs around and after it; one
// launch pays one ramp-up and one drain. Both kinds use the same ring depth,
// so they share one shared-memory size.
template <int D, int BS, int NW, int STAGES>
__global__ void __launch_bounds__((NW + 1) * 32, 3)
    attn_cascade_kernel(AttnParams p, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, int num_groups, int npre,
                        int suffix_parts) {
  pk::launch_dependents();  // the merge may be scheduled as this grid drains
  const int b = int(blockIdx.x);
  const int Hk = p.num_kv_heads;
  if (b < npre) {
    const int t = b / Hk;
    prefix_cta<D, BS, NW, STAGES>(p, &kmap, &vmap,
                                  CtaCoord{b % Hk, t % num_groups, t / num_groups, p.prefix_slots});
  } else {
    const int r = b - npre, t = r / Hk;
    mma_cta<D, BS, NW, STAGES>(p, &kmap, &vmap,
                               CtaCoord{r % Hk, t % p.num_seqs, t / p.num_seqs, suffix_parts});
  }
}

// ---------------------------------------------------------------------------
// Self-test of the bounded pipeline waits: one thread waits on a phase of an
// mbarrier that nothing completes, exactly as a stuck pipeline stage would,
// and records the timeout instead of hanging.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32) wait_timeout_probe_kernel(uint32_t polls) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = pk::smem_addr(&bar);
  if (threadIdx.x == 0) {
    pk::mbar_init(b, 1);
    pk::fence_barrier_init();
    if (!pk::mbar_wait(b, 0, polls)) pk::record_error(&g_attn_error, PK_DEVERR_TIMEOUT, 0);
  }
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge of split-K partials for the CUDA-core kernel (the
// tensor-core kernels' partials are merged by attn_lse_merge_kernel).
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(128) attn_merge_kernel(AttnParams p) {
  // One CTA per (sequence, query head) row.
  const int row = blockIdx.x;
  const int s = row / p.num_q_heads, h = row % p.num_q_heads;
  const int ctx = context_len(p, s, false);
  const int np = (ctx + p.partition - 1) / p.partition;
  if (np == 0) {
    T *out = static_cast<T *>(p.out) + size_t(row) * D;
    for (int i = threadIdx.x; i < D; i += blockDim.x) pk::store_elem(out + i, 0.0f);
    return;
  }
  if (np == 1) return;  // written directly by the attention kernel
  merge_partials<T, D>(p, s, h, 1, np, 0, 0, threadIdx.x, blockDim.x);
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge of the tensor-core kernels' split rows.
//
// The per-sequence and cascade attention launches write one partial per part
// of a split row and nothing else for it. This kernel runs right after them on
// the same stream, launched as their programmatic dependent: it may be
// scheduled while the attention drains and waits for it to complete before
// reading. A row (sequence, query head) gets `wpr` warps (1, 2, 4 or 8, chosen
// from the launch's partition count so that a warp merges at most eight
// parts): each warp merges a contiguous run of the row's parts -- maxima
// shared over the lanes, then eight parts' loads in flight at a time -- and
// the row's first warp combines the warps' states from shared memory. A row
// with a single part was written by the attention launch and is skipped.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) attn_lse_merge_kernel(AttnParams p, int wpr) {
  __shared__ float4 sm_acc[8][D / 4];
  __shared__ float sm_ml[8][2];
  const int warp = int(threadIdx.x >> 5), lane = int(threadIdx.x & 31);
  const int row = int(blockIdx.x) * (8 / wpr) + warp / wpr, sub = warp % wpr;
  // The row's part count, from the context and shared-prefix lengths: inputs
  // the attention launch does not write, so they are read before waiting on it.
  int s = 0, npre = 0, np = 0;
  if (row < p.num_seqs * p.num_q_heads) {
    s = row / p.num_q_heads;
    const int ctx = context_len(p, s, false);
    const int pre = p.seq_prefix ? min(max(__ldg(p.seq_prefix + s), 0), ctx) : 0;
    npre = (pre + p.partition - 1) / p.partition;
    np = npre + (ctx - pre + p.partition - 1) / p.partition;
  }
  pk::wait_prerequisites();  // the attention's partials are complete and visible
  const bool merge = np > 1;
  // Part q's workspace slot: the prefix parts first, then the rest.
  const size_t base = size_t(row) * p.num_partitions;
  auto slot = [&](int q) { return base + (q < npre ? q : p.prefix_slots + (q - npre)); };
  const int chunk = (np + wpr - 1) / wpr;
  const int q0 = min(np, sub * chunk), q1 = min(np, q0 + chunk);
  // This warp's parts: M = max_q m_q, L = sum_q l_q 2^(m_q - M),
  // acc = sum_q acc_q 2^(m_q - M), in part order; each lane owns four columns.
  // Up to U parts (the usual case: wpr gives a warp at most eight) are loaded
  // in one batch and M is taken from the loaded maxima; more take a first
  // pass over the maxima, shared by the lanes.
  constexpr int COLS = D / 4;  // lanes with columns
  constexpr int U = 8;
  const bool cols = lane < COLS;
  float M = -INFINITY;
  float L = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (merge && q1 - q0 <= U) {
    float mq[U], lq[U];
    float4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = q0 + u;
      if (q < q1) {
        const size_t sl = slot(q);
        mq[u] = __ldcg(p.ws_m + sl);
        lq[u] = __ldcg(p.ws_l + sl);
        x[u] = cols ? __ldcg(reinterpret_cast<const float4 *>(p.ws_acc + sl * D) + lane)
                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        M = fmaxf(M, mq[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (q0 + u < q1) {
        const float w = exp2f(mq[u] - M);
        L = fmaf(lq[u], w, L);
        acc.x = fmaf(x[u].x, w, acc.x);
        acc.y = fmaf(x[u].y, w, acc.y);
        acc.z = fmaf(x[u].z, w, acc.z);
        acc.w = fmaf(x[u].w, w, acc.w);
      }
    }
  } else if (merge) {
    for (int q = q0 + lane; q < q1; q += 32) M = fmaxf(M, __ldcg(p.ws_m + slot(q)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  }
  for (int qb = q0; merge && q1 - q0 > U && qb < q1; qb += U) {
    float mq[U], lq[U];
    float4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = qb + u;
      if (q < q1) {
        const size_t sl = slot(q);
        mq[u] = __ldcg(p.ws_m + sl);
        lq[u] = __ldcg(p.ws_l + sl);
        x[u] = cols ? __ldcg(reinterpret_cast<const float4 *>(p.ws_acc + sl * D) + lane)
                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (qb + u < q1) {
        const float w = exp2f(mq[u] - M);
        L = fmaf(lq[u], w, L);
        acc.x = fmaf(x[u].x, w, acc.x);
        acc.y = fmaf(x[u].y, w, acc.y);
        acc.z = fmaf(x[u].z, w, acc.z);
        acc.w = fmaf(x[u].w, w, acc.w);
      }
    }
  }
  if (wpr > 1) {
    // Combine the row's warps (in warp order) in the row's first warp.
    if (cols) sm_acc[warp][lane] = acc;
    if (lane == 0) {
      sm_ml[warp][0] = M;
      sm_ml[warp][1] = L;
    }
    __syncthreads();
    if (sub != 0) return;
    const int w0 = warp;
    float Mr = -INFINITY;
    for (int w = 0; w < wpr; ++w) Mr = fmaxf(Mr, sm_ml[w0 + w][0]);
    L = 0.0f;
    acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int w = 0; w < wpr; ++w) {
      const float f = sm_ml[w0 + w][1] > 0.0f ? exp2f(sm_ml[w0 + w][0] - Mr) : 0.0f;
      L = fmaf(sm_ml[w0 + w][1], f, L);
      if (cols) {
        const float4 y = sm_acc[w0 + w][lane];
        acc.x = fmaf(y.x, f, acc.x);
        acc.y = fmaf(y.y, f, acc.y);
        acc.z = fmaf(y.z, f, acc.z);
        acc.w = fmaf(y.w, f, acc.w);
      }
    }
  }
  if (merge && cols) {
    const float inv = 1.0f / L;
    __nv_bfloat162 *o = reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(p.out) +
                                                          size_t(row) * D + 4 * lane);
    o[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    o[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Consumer warps and pipeline stages of the tensor-core kernel (each stage
// holds 16 tokens per consumer warp). Overridable at build time for tuning.
#ifndef PK_MMA_WARPS
#define PK_MMA_WARPS 4
#endif
#ifndef PK_MMA_STAGES
#define PK_MMA_STAGES 2
#endif
constexpr int kMmaWarps = PK_MMA_WARPS;
constexpr int kMmaStages = PK_MMA_STAGES;

int64_t elem_size(pk_dtype t) { return t == PK_F32 ? 4 : (t == PK_BF16 ? 2 : 0); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// A [N*B, Hk, D] bf16 view of one pool; each load is a box of B token rows of
// one head and 64 elements (128 bytes), swizzled 128B in shared memory.
bool encode_pool_map_uncached(CUtensorMap *map, const void *pool, const pk_cache_desc &d) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {cuuint64_t(d.head_dim), cuuint64_t(d.num_kv_heads),
                              cuuint64_t(d.num_blocks) * cuuint64_t(d.block_size)};
  const cuuint64_t strides[2] = {cuuint64_t(d.head_dim) * 2,
                                 cuuint64_t(d.num_kv_heads) * cuuint64_t(d.head_dim) * 2};
  const cuuint32_t box[3] = {64, 1, cuuint32_t(d.block_size)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Opts the tensor-core kernel into its dynamic shared memory (once).
// The pool's tensor map (boxes of 64 columns x 1 head x one block), encoded
// once per (pool address, geometry): a decode loop launches on the same two
// pools every step. A few entries cover the K and V pools of the layers a
// thread drives in turn.
bool encode_pool_map(CUtensorMap *map, const void *pool, const pk_cache_desc &d) {
  struct Entry {
    const void *pool;
    pk_cache_desc desc;
    CUtensorMap map;
  };
  constexpr int kEntries = 16;
  static std::mutex mu;
  static Entry cache[kEntries];
  static int used = 0, next = 0;
  auto same = [&](const Entry &e) {
    return e.pool == pool && e.desc.num_blocks == d.num_blocks && e.desc.block_size == d.block_size &&
           e.desc.num_kv_heads == d.num_kv_heads && e.desc.head_dim == d.head_dim &&
           e.desc.dtype == d.dtype;
  };
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (same(cache[i])) {
        *map = cache[i].map;
        return true;
      }
  }
  if (!encode_pool_map_uncached(map, pool, d)) return false;
  std::lock_guard<std::mutex> lock(mu);
  Entry &e = cache[next];
  e.pool = pool;
  e.desc = d;
  e.map = *map;
  next = (next + 1) % kEntries;
  used = used < kEntries ? used + 1 : used;
  return true;
}

template <int D, int BS>
cudaError_t mma_kernel_ready() {
  using S = MmaShape<D, BS, kMmaWarps, kMmaStages>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_mma_kernel<D, BS, kMmaWarps, kMmaStages>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES);
  });
  return attr_err;
}

template <int D, int BS>
pk_status launch_mma(const AttnParams &p, const pk_cache_desc &d, cudaStream_t stream) {
  using S = MmaShape<D, BS, kMmaWarps, kMmaStages>;
  if (p.partition % BS != 0) return PK_ERR_INVALID_ARG;
  CUtensorMap kmap, vmap;
  if (!encode_pool_map(&kmap, p.k_cache, d) || !encode_pool_map(&vmap, p.v_cache, d))
    return PK_ERR_CUDA;
  auto kern = attn_mma_kernel<D, BS, kMmaWarps, kMmaStages>;
  if (mma_kernel_ready<D, BS>() != cudaSuccess) return PK_ERR_CUDA;
  dim3 grid(p.num_kv_heads, p.items ? p.num_items : p.num_seqs,
            p.items ? 1 : p.num_partitions - p.prefix_slots);
  kern<<<grid, (kMmaWarps + 1) * 32, S::SMEM_BYTES, stream>>>(p, kmap, vmap);
  return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

// Stages of attn_cascade_kernel's ring. Its prefix CTAs hold up to 16 query
// columns, which unbounded take ~160 registers (2 CTAs per SM); the kernel is
// bounded to 3 CTAs per SM instead (128 registers, a few bytes spilled) with
// the same 2-stage ring as attn_mma_kernel: on GB300 that ran the cascade
// step 5-9% faster than 2 CTAs per SM with a 3-stage ring.
#ifndef PK_PREFIX_STAGES
#define PK_PREFIX_STAGES 2
#endif
constexpr int kPrefixStages = PK_PREFIX_STAGES;

// Cascade attention in one launch (attn_cascade_kernel): the prefix CTAs of
// num_groups groups, then the suffix CTAs.
template <int D, int BS>
pk_status launch_cascade(const AttnParams &p, const pk_cache_desc &d, int num_groups,
                         cudaStream_t stream) {
  using S = MmaShape<D, BS, kMmaWarps, kPrefixStages>;
  CUtensorMap kmap, vmap;
  if (!encode_pool_map(&kmap, p.k_cache, d) || !encode_pool_map(&vmap, p.v_cache, d))
    return PK_ERR_CUDA;
  auto kern = attn_cascade_kernel<D, BS, kMmaWarps, kPrefixStages>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    S::SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return PK_ERR_CUDA;
  const int suffix_parts = p.num_partitions - p.prefix_slots;
  const int64_t npre = int64_t(p.num_kv_heads) * num_groups * p.prefix_slots;
  const int64_t total = npre + int64_t(p.num_kv_heads) * p.num_seqs * suffix_parts;
  if (total > int64_t(INT32_MAX)) return PK_ERR_UNSUPPORTED;
  kern<<<unsigned(total), (kMmaWarps + 1) * 32, S::SMEM_BYTES, stream>>>(p, kmap, vmap, num_groups,
                                                                        int(npre), suffix_parts);
  return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

template <typename T, int D>
pk_status launch_simt(const AttnParams &p, cudaStream_t stream) {
  dim3 grid(p.num_kv_heads, p.items ? p.num_items : p.num_seqs, p.items ? 1 : p.num_partitions);
  attn_simt_kernel<T, D><<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

template <typename T, int D>
pk_status launch_merge(const AttnParams &p, cudaStream_t stream) {
  const int rows = p.num_seqs * p.num_q_heads;
  attn_merge_kernel<T, D><<<rows, D / 4, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

// attn_lse_merge_kernel after a tensor-core attention launch on `stream`, as
// its programmatic dependent (an ordinary launch where that is refused).
template <int D>
pk_status launch_lse_merge(const AttnParams &p, cudaStream_t stream) {
  const int rows = p.num_seqs * p.num_q_heads;
  // Warps per row: enough that a warp merges at most eight parts (at most 8).
  int wpr = 1;
  while (wpr < 8 && wpr * 8 < p.num_partitions) wpr *= 2;
  const int rows_per_cta = 8 / wpr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((rows + rows_per_cta - 1) / rows_per_cta));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, attn_lse_merge_kernel<D>, p, wpr) == cudaSuccess) return PK_OK;
  cudaGetLastError();
  attn_lse_merge_kernel<D><<<cfg.gridDim, cfg.blockDim, 0, stream>>>(p, wpr);
  return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

// SMs of the current device (152 on GB300 when no device can be queried).
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
    return n;
  cudaGetLastError();  // clear a failed query on a machine without a GPU
  return 152;
}

bool mma_supported(const pk_cache_desc &d, int group) {
  return d.dtype == PK_BF16 && (d.head_dim == 64 || d.head_dim == 128) &&
         (d.block_size == 8 || d.block_size == 16 || d.block_size == 32) && group <= kMaxGroup;
}

// CTAs of the attention kernel resident on one SM, from the occupancy
// calculator (queried once per instantiation); without a device, the GB300
// figures: 3 (head_dim 128) or 4 (head_dim 64) tensor-core CTAs.
template <int D, int BS>
int mma_resident_ctas() {
  using S = MmaShape<D, BS, kMmaWarps, kMmaStages>;
  static const int n = [] {
    int v = 0;
    if (mma_kernel_ready<D, BS>() == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &v, attn_mma_kernel<D, BS, kMmaWarps, kMmaStages>, (kMmaWarps + 1) * 32,
            S::SMEM_BYTES) == cudaSuccess &&
        v > 0)
      return v;
    cudaGetLastError();
    return D == 128 ? 3 : 4;
  }();
  return n;
}

template <typename T, int D>
int simt_resident_ctas() {
  static const int n = [] {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, attn_simt_kernel<T, D>, 128, 0) ==
            cudaSuccess &&
        v > 0)
      return v;
    cudaGetLastError();
    return 8;
  }();
  return n;
}

int resident_ctas(const pk_cache_desc &d, int group) {
  if (mma_supported(d, group)) {
    const bool d128 = d.head_dim == 128;
    switch (d.block_size) {
      case 8: return d128 ? mma_resident_ctas<128, 8>() : mma_resident_ctas<64, 8>();
      case 16: return d128 ? mma_resident_ctas<128, 16>() : mma_resident_ctas<64, 16>();
      default: return d128 ? mma_resident_ctas<128, 32>() : mma_resident_ctas<64, 32>();
    }
  }
  if (d.dtype == PK_F32)
    return d.head_dim == 128 ? simt_resident_ctas<float, 128>() : simt_resident_ctas<float, 64>();
  return d.head_dim == 128 ? simt_resident_ctas<__nv_bfloat16, 128>()
                           : simt_resident_ctas<__nv_bfloat16, 64>();
}

// Split-K partials (when the partitioning splits).
size_t partial_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len, int32_t part,
                     int32_t head_dim) {
  if (part <= 0) return 0;
  const int64_t P = (int64_t(max_context_len) + part - 1) / part;
  if (P <= 1) return 0;
  const int64_t rows = int64_t(num_seqs) * num_q_heads * P;
  return size_t(rows) * (size_t(head_dim) + 2) * sizeof(float);
}

// Partition of cascade attention. 0: one partition covering the longest
// context; > 0: as given (a multiple of B); -1 (automatic): one partition
// when the (group, KV head) prefix items already cover the SMs (on GB300 the
// 32-group x 8-head prefix workload ran fastest unsplit), else prefix
// partitions sized so the prefix items cover the SMs once, at least 512
// tokens.
int32_t cascade_partition(int32_t max_context_len, int32_t partition_size, int32_t B,
                          int32_t num_groups, int32_t num_kv_heads, int32_t max_prefix_len) {
  const int64_t whole = (int64_t(max_context_len) + B - 1) / B * B;
  if (partition_size == 0) return int32_t(whole);
  if (partition_size > 0) return partition_size % B == 0 ? partition_size : -1;
  if (partition_size != -1) return -1;
  const int64_t items = int64_t(num_groups) * num_kv_heads;
  const int64_t sms = sm_count();
  if (items >= sms || max_prefix_len <= 512) return int32_t(whole);
  int64_t part = (int64_t(max_prefix_len) * items + sms - 1) / sms;
  part = std::max<int64_t>(512, (part + 63) / 64 * 64);
  part = (part + B - 1) / B * B;
  return int32_t(std::min(part, whole));
}

// The tensor-core split-K merge after an attention launch: D dispatch.
pk_status launch_lse_merge_d(const AttnParams &p, int D, cudaStream_t s) {
  return D == 128 ? launch_lse_merge<128>(p, s) : launch_lse_merge<64>(p, s);
}

pk_status check_common(const pk_cache_desc *desc, int32_t num_seqs, int32_t num_q_heads,
                       int32_t max_context_len) {
  if (!desc || desc->num_blocks <= 0 || desc->block_size <= 0 || desc->num_kv_heads <= 0 ||
      desc->head_dim <= 0 || num_seqs < 0 || num_q_heads <= 0 || max_context_len <= 0)
    return PK_ERR_INVALID_ARG;
  if (elem_size(desc->dtype) == 0) return PK_ERR_UNSUPPORTED;
  if (num_q_heads % desc->num_kv_heads != 0) return PK_ERR_INVALID_ARG;
  if (num_q_heads / desc->num_kv_heads > kMaxGroup) return PK_ERR_UNSUPPORTED;
  if (desc->head_dim != 64 && desc->head_dim != 128) return PK_ERR_UNSUPPORTED;
  if (int64_t(desc->num_blocks) * desc->block_size > INT32_MAX) return PK_ERR_UNSUPPORTED;
  return PK_OK;
}

}  // namespace

// Library-internal hooks for the decode step's captured graphs (decode_step.cpp):
// the size of a kernel's parameter block, the number of arguments of an
// attention kernel (0 for a function that is not one), and re-pointing a
// parameter block's host-buffer arguments. A graph captured in zero-copy mode
// reads q and the new K/V from, and writes the output to, the caller's
// pinned host buffers; a later step that passes other buffers re-points the
// captured kernel nodes at them instead of capturing again.
extern "C" size_t pkx_attn_params_size() { return sizeof(AttnParams); }

namespace {
template <int D, int BS>
bool is_mma(const void *f) {
  return f == reinterpret_cast<const void *>(attn_mma_kernel<D, BS, kMmaWarps, kMmaStages>);
}
template <typename T, int D>
bool is_simt(const void *f) {
  return f == reinterpret_cast<const void *>(attn_simt_kernel<T, D>) ||
         f == reinterpret_cast<const void *>(attn_merge_kernel<T, D>);
}
}  // namespace

extern "C" int pkx_attn_kernel_arity(const void *f) {
  if (is_mma<128, 8>(f) || is_mma<128, 16>(f) || is_mma<128, 32>(f) || is_mma<64, 8>(f) ||
      is_mma<64, 16>(f) || is_mma<64, 32>(f))
    return 3;  // (params, K tensor map, V tensor map)
  if (f == reinterpret_cast<const void *>(attn_lse_merge_kernel<128>) ||
      f == reinterpret_cast<const void *>(attn_lse_merge_kernel<64>))
    return 2;  // (params, warps per row)
  if (is_simt<float, 128>(f) || is_simt<float, 64>(f) || is_simt<__nv_bfloat16, 128>(f) ||
      is_simt<__nv_bfloat16, 64>(f))
    return 1;  // (params)
  return 0;
}

// In the parameter block `params` (an AttnParams), each of q, new K, new V and
// out that equals from[i] becomes to[i] (i = 0..3 in that order).
extern "C" void pkx_attn_params_rebind(void *params, const void *const from[4],
                                       const void *const to[4]) {
  AttnParams *p = static_cast<AttnParams *>(params);
  if (p->q == from[0]) p->q = to[0];
  if (p->new_k == from[1]) p->new_k = to[1];
  if (p->new_v == from[2]) p->new_v = to[2];
  if (p->out == from[3]) p->out = const_cast<void *>(to[3]);
}

extern "C" int pkx_take_attention_error(cudaStream_t stream) {
  int code = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbolAsync(&code, g_attn_error, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                stream) != cudaSuccess)
    return -1;
  if (cudaMemcpyToSymbolAsync(g_attn_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                              stream) != cudaSuccess)
    return -1;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return -1;
  return code;
}

extern "C" {

int32_t pk_paged_attention_resolve_partition(int32_t num_seqs, int32_t num_q_heads,
                                             int32_t max_context_len, int32_t partition_size,
                                             const pk_cache_desc *desc) {
  if (check_common(desc, num_seqs, num_q_heads, max_context_len) != PK_OK) return -1;
  const int32_t B = desc->block_size;
  if (partition_size > 0) return partition_size % B == 0 ? partition_size : -1;
  if (partition_size == 0) return 0;
  if (partition_size != -1) return -1;
  // Automatic: fill the resident CTA slots (SMs x CTAs per SM) once. When the
  // (sequence, KV head) units already fill them, no split: every partition
  // costs a prologue, an epilogue and merge traffic. Otherwise cut each
  // context into P = floor(slots / units) equal partitions (multiples of 64
  // tokens, at least 512), so the work runs as one wave with no tail. On
  // GB300, 32K-token contexts over 64 units ran at 96.5% of the copy peak
  // this way (7 partitions, 448 of 456 slots) against 90% in 2.67 waves.
  const int64_t units = int64_t(num_seqs) * desc->num_kv_heads;
  const int64_t slots =
      int64_t(sm_count()) * resident_ctas(*desc, num_q_heads / desc->num_kv_heads);
  if (units >= slots || max_context_len <= 512) return 0;
  const int64_t P = slots / units;
  if (P < 2) return 0;
  int64_t part = (max_context_len + P - 1) / P;
  part = (part + 63) / 64 * 64;
  if (part < 512) part = 512;
  part = (part + B - 1) / B * B;
  return part >= max_context_len ? 0 : int32_t(part);
}

size_t pk_paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_context_len, int32_t partition_size,
                                         const pk_cache_desc *desc) {
  const int32_t part = pk_paged_attention_resolve_partition(num_seqs, num_q_heads,
                                                            max_context_len, partition_size, desc);
  if (part < 0) return 0;
  const size_t pb = partial_bytes(num_seqs, num_q_heads, max_context_len, part, desc->head_dim);
  return pb;
}

}  // extern "C"

namespace {

// Shared body of the per-sequence attention entry points: either a launch
// order over the (sequence, partition) grid or a work list of items.
pk_status decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens, float scale,
                           int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                           int32_t max_context_len, int32_t partition_size, void *workspace,
                           size_t workspace_bytes, const pk_cache_desc *desc,
                           const int32_t *seq_order, const int32_t *items, int32_t num_items,
                           pk_attn_impl impl, void *stream, const void *new_k = nullptr,
                           const void *new_v = nullptr, const int64_t *new_slots = nullptr,
                           int32_t *lens_out = nullptr) {
  pk_status st = check_common(desc, num_seqs, num_q_heads, max_context_len);
  if (st != PK_OK) return st;
  if (num_seqs == 0) return PK_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || max_blocks_per_seq <= 0)
    return PK_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PK_ERR_INVALID_ARG;
  if (!(scale == scale)) return PK_ERR_INVALID_ARG;
  const int32_t part = pk_paged_attention_resolve_partition(num_seqs, num_q_heads, max_context_len,
                                                            partition_size, desc);
  if (part < 0) return PK_ERR_INVALID_ARG;
  int64_t P = part > 0 ? (int64_t(max_context_len) + part - 1) / part : 1;
  AttnParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.tables = block_tables;
  p.ctx_lens = context_lens;
  p.scale_log2 = float(double(scale) * 1.4426950408889634);
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = desc->num_kv_heads;
  p.group = num_q_heads / desc->num_kv_heads;
  p.block_size = desc->block_size;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = desc->num_blocks;
  if (P <= 1) {
    P = 1;
    // One partition covering any context the table allows (independent of
    // max_context_len, so that a step's launch parameters do not change as
    // the contexts grow).
    p.partition = int32_t(std::min<int64_t>(int64_t(max_blocks_per_seq) * desc->block_size, INT32_MAX));
  } else {
    p.partition = part;
  }
  p.num_partitions = int32_t(P);
  if (num_seqs > 65535 || P > 65535) return PK_ERR_UNSUPPORTED;
  const size_t pbytes = partial_bytes(num_seqs, num_q_heads, max_context_len, part, desc->head_dim);
  if (workspace && !aligned16(workspace)) return PK_ERR_WORKSPACE;
  if (P > 1) {
    if (!workspace || workspace_bytes < pbytes) return PK_ERR_WORKSPACE;
    const size_t rows = size_t(num_seqs) * num_q_heads * size_t(P);
    p.ws_acc = static_cast<float *>(workspace);
    p.ws_m = p.ws_acc + rows * desc->head_dim;
    p.ws_l = p.ws_m + rows;
  }
  p.order = seq_order;
  p.items = items;
  p.num_items = num_items;
  if (items && (num_items <= 0 || num_items > 65535)) return PK_ERR_UNSUPPORTED;

  const bool mma_ok = mma_supported(*desc, p.group);
  if (impl == PK_ATTN_MMA && !mma_ok) return PK_ERR_UNSUPPORTED;
  if (impl != PK_ATTN_AUTO && impl != PK_ATTN_SIMT && impl != PK_ATTN_MMA)
    return PK_ERR_INVALID_ARG;
  const bool use_mma = impl == PK_ATTN_MMA || (impl == PK_ATTN_AUTO && mma_ok);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = desc->head_dim, B = desc->block_size;
  if (new_k) {
    if (!new_v || !new_slots || !aligned16(new_k) || !aligned16(new_v)) return PK_ERR_INVALID_ARG;
    if (use_mma) {  // the tensor-core kernel writes the new tokens itself
      p.new_k = new_k;
      p.new_v = new_v;
      p.new_slots = new_slots;
      p.lens_out = lens_out;
    } else if (lens_out) {
      // The scatter and the table bookkeeping first, then attention over the
      // new lengths.
      st = pkx_reshape_and_cache_advance(new_k, new_v, new_slots, num_seqs,
                                         const_cast<void *>(k_cache), const_cast<void *>(v_cache),
                                         desc, const_cast<int32_t *>(block_tables),
                                         max_blocks_per_seq, context_lens, lens_out, stream);
      if (st != PK_OK) return st;
      p.ctx_lens = lens_out;
    } else {
      st = pk_reshape_and_cache(new_k, new_v, new_slots, num_seqs, const_cast<void *>(k_cache),
                                const_cast<void *>(v_cache), desc, stream);
      if (st != PK_OK) return st;
    }
  }
  if (use_mma) {
    if (D == 128) {
      st = B == 8 ? launch_mma<128, 8>(p, *desc, s)
                  : (B == 16 ? launch_mma<128, 16>(p, *desc, s) : launch_mma<128, 32>(p, *desc, s));
    } else {
      st = B == 8 ? launch_mma<64, 8>(p, *desc, s)
                  : (B == 16 ? launch_mma<64, 16>(p, *desc, s) : launch_mma<64, 32>(p, *desc, s));
    }
  } else if (desc->dtype == PK_F32) {
    st = D == 128 ? launch_simt<float, 128>(p, s) : launch_simt<float, 64>(p, s);
  } else {
    st = D == 128 ? launch_simt<__nv_bfloat16, 128>(p, s) : launch_simt<__nv_bfloat16, 64>(p, s);
  }
  if (st != PK_OK || P == 1) return st;
  if (use_mma) return launch_lse_merge_d(p, D, s);
  if (desc->dtype == PK_F32)
    return D == 128 ? launch_merge<float, 128>(p, s) : launch_merge<float, 64>(p, s);
  return D == 128 ? launch_merge<__nv_bfloat16, 128>(p, s) : launch_merge<__nv_bfloat16, 64>(p, s);
}

}  // namespace

extern "C" {

pk_status pk_paged_attention_decode_impl(void *out, const void *q, const void *k_cache,
                                         const void *v_cache, const int32_t *block_tables,
                                         const int32_t *context_lens, float scale,
                                         int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_blocks_per_seq, int32_t max_context_len,
                                         int32_t partition_size, void *workspace,
                                         size_t workspace_bytes, const pk_cache_desc *desc,
                                         const int32_t *seq_order, pk_attn_impl impl,
                                         void *stream) {
  return decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_seqs,
                          num_q_heads, max_blocks_per_seq, max_context_len, partition_size,
                          workspace, workspace_bytes, desc, seq_order, nullptr, 0, impl, stream);
}

pk_status pk_paged_attention_decode_items(void *out, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_tables,
                                          const int32_t *context_lens, float scale,
                                          int32_t num_seqs, int32_t num_q_heads,
                                          int32_t max_blocks_per_seq, int32_t max_context_len,
                                          int32_t partition_size, const int32_t *work_items,
                                          int32_t num_items, void *workspace,
                                          size_t workspace_bytes, const pk_cache_desc *desc,
                                          pk_attn_impl impl, void *stream) {
  if (!work_items) return PK_ERR_INVALID_ARG;
  return decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_seqs,
                          num_q_heads, max_blocks_per_seq, max_context_len, partition_size,
                          workspace, workspace_bytes, desc, nullptr, work_items, num_items, impl,
                          stream);
}

pk_status pk_paged_attention_decode_append(
    void *out, const void *q, const void *k_new, const void *v_new, const int64_t *slot_mapping,
    void *k_cache, void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
    float scale, int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
    int32_t max_context_len, int32_t partition_size, const int32_t *work_items, int32_t num_items,
    void *workspace, size_t workspace_bytes, const pk_cache_desc *desc, void *stream) {
  if (!work_items || !k_new || !v_new || !slot_mapping) return PK_ERR_INVALID_ARG;
  return decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_seqs,
                          num_q_heads, max_blocks_per_seq, max_context_len, partition_size,
                          workspace, workspace_bytes, desc, nullptr, work_items, num_items,
                          PK_ATTN_AUTO, stream, k_new, v_new, slot_mapping);
}

pk_status pk_selftest_wait_timeout(uint32_t polls, void *stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      polls ? polls : pk::kMaxWaitPolls);
  return cudaGetLastError() == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}

pk_status pk_paged_attention_decode_advance(
    void *out, const void *q, const void *k_new, const void *v_new, const int64_t *slot_mapping,
    void *k_cache, void *v_cache, int32_t *block_tables, const int32_t *context_lens,
    int32_t *context_lens_out, float scale, int32_t num_seqs, int32_t num_q_heads,
    int32_t max_blocks_per_seq, int32_t max_context_len, int32_t partition_size,
    const int32_t *work_items, int32_t num_items, void *workspace, size_t workspace_bytes,
    const pk_cache_desc *desc, void *stream) {
  if (!work_items || !k_new || !v_new || !slot_mapping || !context_lens_out ||
      context_lens_out == context_lens)
    return PK_ERR_INVALID_ARG;
  return decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_seqs,
                          num_q_heads, max_blocks_per_seq, max_context_len, partition_size,
                          workspace, workspace_bytes, desc, nullptr, work_items, num_items,
                          PK_ATTN_AUTO, stream, k_new, v_new, slot_mapping, context_lens_out);
}

pk_status pk_attention_plan(const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t partition_size, const pk_cache_desc *desc,
                            int32_t *partition_out, int32_t *items_out, int32_t cap,
                            int32_t *num_items_out) {
  if (!partition_out || !num_items_out || num_seqs <= 0 || !context_lens) return PK_ERR_INVALID_ARG;
  *partition_out = 0;
  *num_items_out = 0;
  int32_t max_ctx = 1;
  int64_t total = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t c = std::max(context_lens[s], 1);
    max_ctx = std::max(max_ctx, c);
    total += c;
  }
  pk_status st = check_common(desc, num_seqs, num_q_heads, max_ctx);
  if (st != PK_OK) return st;
  const int32_t B = desc->block_size;
  int32_t part = 0;
  if (partition_size > 0) {
    if (partition_size % B != 0) return PK_ERR_INVALID_ARG;
    part = partition_size < max_ctx ? partition_size : 0;
  } else if (partition_size == -1) {
    // W = the (token, KV head) work one resident CTA slot gets when the batch
    // is spread evenly. A context longer than 2W would outlast the rest of the
    // launch on its own CTAs, so the batch splits into items of about W tokens
    // (k equal parts of the longest context, k = floor(max / W), multiples of
    // 64 tokens, at least 512): uniform long contexts get one wave; short or
    // even batches stay whole.
    const int64_t slots = int64_t(sm_count()) *
                          resident_ctas(*desc, num_q_heads / desc->num_kv_heads);
    const int64_t W = std::max<int64_t>(1, (total * desc->num_kv_heads + slots - 1) / slots);
    if (max_ctx > 2 * W && max_ctx > 1024) {
      const int64_t k = std::max<int64_t>(1, max_ctx / W);
      int64_t p = (max_ctx + k - 1) / k;
      p = std::max<int64_t>(512, (p + 63) / 64 * 64);
      p = (p + B - 1) / B * B;
      part = p < max_ctx ? int32_t(p) : 0;
    }
  } else if (partition_size != 0) {
    return PK_ERR_INVALID_ARG;
  }
  *partition_out = part;
  return pk_attention_work_items(context_lens, num_seqs, part, items_out, cap, num_items_out);
}

pk_status pk_attention_work_items(const int32_t *context_lens, int32_t num_seqs,
                                  int32_t partition, int32_t *items_out, int32_t cap,
                                  int32_t *num_items_out) {
  if (!num_items_out || num_seqs < 0 || partition < 0 || cap < 0 || (num_seqs > 0 && !context_lens))
    return PK_ERR_INVALID_ARG;
  *num_items_out = 0;
  struct Item {
    int32_t len, ctx, seq, part;
  };
  std::vector<Item> items;
  try {
    items.reserve(size_t(num_seqs));
    for (int32_t s = 0; s < num_seqs; ++s) {
      const int32_t c = std::max(context_lens[s], 1);  // an invalid length still gets its item
      const int32_t n = partition > 0 ? (c + partition - 1) / partition : 1;
      for (int32_t j = 0; j < n; ++j)
        items.push_back({partition > 0 ? std::min(partition, c - j * partition) : c, c, s, j});
    }
  } catch (const std::bad_alloc &) {
    return PK_ERR_NOMEM;
  }
  // Longest item first; ties: the longer sequence, then batch order, then the
  // later partition.
  std::sort(items.begin(), items.end(), [](const Item &a, const Item &b) {
    if (a.len != b.len) return a.len > b.len;
    if (a.ctx != b.ctx) return a.ctx > b.ctx;
    if (a.seq != b.seq) return a.seq < b.seq;
    return a.part > b.part;
  });
  *num_items_out = int32_t(items.size());
  if (int64_t(items.size()) > cap) return PK_ERR_INVALID_ARG;
  if (!items.empty() && !items_out) return PK_ERR_INVALID_ARG;
  for (size_t i = 0; i < items.size(); ++i) {
    items_out[2 * i] = items[i].seq;
    items_out[2 * i + 1] = items[i].part;
  }
  return PK_OK;
}

size_t pk_cascade_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                                 int32_t num_groups, int32_t max_prefix_len,
                                 int32_t partition_size, const pk_cache_desc *desc) {
  if (check_common(desc, num_seqs, num_q_heads, max_context_len) != PK_OK || max_prefix_len < 0 ||
      num_groups < 0)
    return 0;
  const int32_t part = cascade_partition(max_context_len, partition_size, desc->block_size,
                                         num_groups, desc->num_kv_heads, max_prefix_len);
  if (part <= 0) return 0;
  const int64_t P = (int64_t(max_prefix_len) + part - 1) / part +
                    (int64_t(max_context_len) + part - 1) / part;
  const int64_t rows = int64_t(num_seqs) * num_q_heads * P;
  return size_t(rows) * (size_t(desc->head_dim) + 2) * sizeof(float);
}

pk_status pk_cascade_attention_decode(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, float scale, int32_t num_seqs,
    int32_t num_q_heads, int32_t max_blocks_per_seq, int32_t max_context_len,
    int32_t partition_size, const int32_t *group_offsets, const int32_t *group_members,
    const int32_t *group_prefix_len, const int32_t *seq_prefix_len, int32_t num_groups,
    int32_t max_group_size, int32_t max_prefix_len, const int32_t *seq_order, void *workspace,
    size_t workspace_bytes, const pk_cache_desc *desc, void *stream) {
  pk_status st = check_common(desc, num_seqs, num_q_heads, max_context_len);
  if (st != PK_OK) return st;
  if (num_groups < 0 || max_group_size < 0 || max_prefix_len < 0) return PK_ERR_INVALID_ARG;
  if (num_groups == 0)
    return pk_paged_attention_decode_impl(out, q, k_cache, v_cache, block_tables, context_lens,
                                          scale, num_seqs, num_q_heads, max_blocks_per_seq,
                                          max_context_len, partition_size, workspace,
                                          workspace_bytes, desc, seq_order, PK_ATTN_AUTO, stream);
  const int32_t G = num_q_heads / desc->num_kv_heads;
  if (!mma_supported(*desc, G)) return PK_ERR_UNSUPPORTED;
  if (int64_t(max_group_size) * G > 16) return PK_ERR_UNSUPPORTED;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !group_offsets ||
      !group_members || !group_prefix_len || !seq_prefix_len || max_blocks_per_seq <= 0)
    return PK_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (workspace && !aligned16(workspace)))
    return PK_ERR_INVALID_ARG;
  const int32_t part = cascade_partition(max_context_len, partition_size, desc->block_size,
                                         num_groups, desc->num_kv_heads, max_prefix_len);
  if (part <= 0) return PK_ERR_INVALID_ARG;
  const int64_t Ppre = (int64_t(max_prefix_len) + part - 1) / part;
  const int64_t Psuf = (int64_t(max_context_len) + part - 1) / part;
  if (num_seqs > 65535 || num_groups > 65535 || Ppre + Psuf > 65535) return PK_ERR_UNSUPPORTED;
  const size_t need = pk_cascade_workspace_size(num_seqs, num_q_heads, max_context_len, num_groups,
                                                max_prefix_len, partition_size, desc);
  if (!workspace || workspace_bytes < need) return PK_ERR_WORKSPACE;
  AttnParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.tables = block_tables;
  p.ctx_lens = context_lens;
  p.scale_log2 = float(double(scale) * 1.4426950408889634);
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = desc->num_kv_heads;
  p.group = G;
  p.block_size = desc->block_size;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = desc->num_blocks;
  p.partition = part;
  p.num_partitions = int32_t(Ppre + Psuf);
  p.prefix_slots = int32_t(Ppre);
  const size_t rows = size_t(num_seqs) * num_q_heads * size_t(Ppre + Psuf);
  p.ws_acc = static_cast<float *>(workspace);
  p.ws_m = p.ws_acc + rows * desc->head_dim;
  p.ws_l = p.ws_m + rows;
  p.order = seq_order;
  p.seq_prefix = seq_prefix_len;
  p.group_offsets = group_offsets;
  p.group_members = group_members;
  p.group_prefix = group_prefix_len;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = desc->head_dim, B = desc->block_size;
  // One launch: the prefix CTAs first (the long ones), then the suffix CTAs;
  // every part writes a partial, and the merge launch combines them.
  if (Ppre > 0) {
    if (D == 128)
      st = B == 8 ? launch_cascade<128, 8>(p, *desc, num_groups, s)
                  : (B == 16 ? launch_cascade<128, 16>(p, *desc, num_groups, s)
                             : launch_cascade<128, 32>(p, *desc, num_groups, s));
    else
      st = B == 8 ? launch_cascade<64, 8>(p, *desc, num_groups, s)
                  : (B == 16 ? launch_cascade<64, 16>(p, *desc, num_groups, s)
                             : launch_cascade<64, 32>(p, *desc, num_groups, s));
  } else if (D == 128) {
    st = B == 8 ? launch_mma<128, 8>(p, *desc, s)
                : (B == 16 ? launch_mma<128, 16>(p, *desc, s) : launch_mma<128, 32>(p, *desc, s));
  } else {
    st = B == 8 ? launch_mma<64, 8>(p, *desc, s)
                : (B == 16 ? launch_mma<64, 16>(p, *desc, s) : launch_mma<64, 32>(p, *desc, s));
  }
  if (st != PK_OK || Ppre + Psuf <= 1) return st;
  return launch_lse_merge_d(p, D, s);
}

pk_status pk_paged_attention_decode(void *out, const void *q, const void *k_cache,
                                    const void *v_cache, const int32_t *block_tables,
                                    const int32_t *context_lens, float scale, int32_t block_size,
                                    int32_t num_seqs, int32_t num_q_heads,
                                    int32_t max_blocks_per_seq, int32_t max_context_len,
                                    int32_t partition_size, void *workspace,
                                    size_t workspace_bytes, const pk_cache_desc *desc,
                                    void *stream) {
  if (!desc || block_size != desc->block_size) return PK_ERR_INVALID_ARG;
  return pk_paged_attention_decode_impl(out, q, k_cache, v_cache, block_tables, context_lens,
                                        scale, num_seqs, num_q_heads, max_blocks_per_seq,
                                        max_context_len, partition_size, workspace,
                                        workspace_bytes, desc, nullptr, PK_ATTN_AUTO, stream);
}

}  // extern "C"

extern "C" pk_status pk_longest_first_order(const int32_t *context_lens, int32_t num_seqs,
                                            int32_t *order_out) {
  if (num_seqs < 0 || (num_seqs > 0 && (!context_lens || !order_out))) return PK_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_seqs; ++i) order_out[i] = i;
  std::stable_sort(order_out, order_out + num_seqs,
                   [&](int32_t a, int32_t b) { return context_lens[a] > context_lens[b]; });
  return PK_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the decode attention
// ---------------------------------------------------------------------------
// Some callers cannot allocate device memory at all: a serving engine whose
// memory planner has already handed nearly all HBM to the KV pool and forbids
// ad-hoc allocations, a host framework's custom-operator hook that passes in
// only input and output buffers, or a latency-critical loop that cannot
// afford cudaMalloc/cudaFree and their implicit device-wide synchronisation.
// For them the split-K scratch lives in the file-scope array below. Every GPU
// that loads this library holds it (PK_STATIC_WORKSPACE_BYTES) until the
// process exits.
namespace {

static __device__ __align__(256) unsigned char g_static_workspace[PK_STATIC_WORKSPACE_BYTES];

constexpr int kMaxStaticDevices = 64;

// Device address of g_static_workspace on `device` (which must be current).
// In host code the array's name is only a host-side stand-in, so the address
// comes from cudaGetSymbolAddress, looked up once per device and kept for the
// life of the process (valid while the device's primary context is not reset).
cudaError_t static_workspace_address(int device, void **out) {
  static std::mutex mu;
  static void *addr[kMaxStaticDevices] = {};
  if (device < 0 || device >= kMaxStaticDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[device]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess) return e;
    addr[device] = p;
  }
  *out = addr[device];
  return cudaSuccess;
}

}  // namespace

extern "C" pk_status pk_paged_attention_decode_static(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, float scale, int32_t block_size,
    int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq, int32_t max_context_len,
    int32_t partition_size, const pk_cache_desc *desc, void *stream) {
  if (!desc || block_size != desc->block_size) return PK_ERR_INVALID_ARG;
  pk_status st = check_common(desc, num_seqs, num_q_heads, max_context_len);
  if (st != PK_OK) return st;
  const int32_t part = pk_paged_attention_resolve_partition(num_seqs, num_q_heads,
                                                            max_context_len, partition_size, desc);
  if (part < 0) return PK_ERR_INVALID_ARG;
  const size_t need = pk_paged_attention_workspace_size(num_seqs, num_q_heads, max_context_len,
                                                        partition_size, desc);
  if (need > PK_STATIC_WORKSPACE_BYTES) return PK_ERR_WORKSPACE;
  void *ws = nullptr;
  if (need > 0) {
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return PK_ERR_CUDA;
    if (static_workspace_address(device, &ws) != cudaSuccess) return PK_ERR_CUDA;
  }
  // Nothing in the scratch needs clearing: every partial the merge reads is
  // written earlier in the same call.
  return pk_paged_attention_decode_impl(out, q, k_cache, v_cache, block_tables, context_lens,
                                        scale, num_seqs, num_q_heads, max_blocks_per_seq,
                                        max_context_len, partition_size, ws,
                                        need > 0 ? size_t(PK_STATIC_WORKSPACE_BYTES) : 0, desc,
                                        nullptr, PK_ATTN_AUTO, stream);
}
