// One decode step from host buffers, in native code, in two halves. The host
// half (prepare) appends a token to every sequence in the host block manager
// and packs the step's metadata into one of two pinned staging halves, so it
// can run while the previous step, reading the other half, is still on the
// GPU. The device half (launch) copies the new K/V and queries (unless the
// kernels read them from pinned host memory: zero-copy), copies the metadata
// with a single transfer -- in full mode slots, copy-on-write pairs, work
// items, context lengths and padded block tables; in resident mode (the
// device already holds this batch's tables and lengths) only what changed --
// and runs copy_blocks (when pairs exist) and the step's kernels: the scatter
// and the attention in full mode, one launch that also advances the device
// tables and lengths in resident mode. The output is copied back to host
// memory. Everything is enqueued on one stream; the call returns once the
// work is enqueued.
//
// The attention runs a work list of (sequence, partition) items planned on the
// host (pk_attention_plan). A full step plans afresh; a resident step keeps the
// partition and rebuilds the list only when a sequence starts a new partition.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "pagedkv.h"

// Library-internal hooks of attention.cu and cache_ops.cu for re-pointing
// captured kernels at other host buffers (zero-copy mode).
extern "C" size_t pkx_attn_params_size();
extern "C" int pkx_attn_kernel_arity(const void *func);
extern "C" void pkx_attn_params_rebind(void *params, const void *const from[4],
                                       const void *const to[4]);
extern "C" int pkx_scatter_kernel_arity(const void *func);

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Work items a batch can need: a partition is at least 512 tokens and a
// context at most max_blocks * 32 tokens (B <= 32), so a sequence has at most
// 1 + max_blocks / 16 items.
int64_t item_capacity(int32_t num_seqs, int32_t max_blocks) {
  return int64_t(num_seqs) * (1 + max_blocks / 16);
}

// What changes every step comes first, so a resident-mode step copies one
// short prefix of the buffer. On the device, lens and lens_b hold the
// lengths of alternate resident steps (each step reads one and writes the
// other); a full step uploads the lengths into lens.
struct MetaLayout {
  size_t slots, pairs, items, lens, tables, lens_b, total;
  int32_t item_cap;
};

MetaLayout layout(int32_t num_seqs, int32_t max_blocks) {
  MetaLayout m{};
  size_t off = 0;
  m.slots = off;
  off = align_up(off + size_t(num_seqs) * sizeof(int64_t));
  m.pairs = off;
  off = align_up(off + size_t(num_seqs) * 2 * sizeof(int64_t));
  m.items = off;
  m.item_cap = int32_t(std::min<int64_t>(item_capacity(num_seqs, max_blocks), 65535));
  off = align_up(off + size_t(m.item_cap) * 2 * sizeof(int32_t));
  m.lens = off;
  off = align_up(off + size_t(num_seqs) * sizeof(int32_t));
  m.tables = off;
  off = align_up(off + size_t(num_seqs) * size_t(max_blocks) * sizeof(int32_t));
  m.lens_b = off;
  off = align_up(off + size_t(num_seqs) * sizeof(int32_t));
  m.total = off;
  return m;
}

int64_t elem_size(pk_dtype t) { return t == PK_F32 ? 4 : (t == PK_BF16 ? 2 : 0); }

// A captured resident step: the copies of q, k, v and the slots, the scatter
// that advances the device tables, the attention over the unchanged work
// list and the output copy. Every parameter of those is fixed while the work
// list is, except the caller's host buffers: in copying mode the q/k/v copy
// nodes' sources are patched; in zero-copy mode the kernels read and write
// the host buffers themselves, and their nodes' pointer arguments are
// re-pointed.
struct GraphSlot {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraphNode_t copy_node[3] = {nullptr, nullptr, nullptr};  // q, k, v
  const void *src[3] = {nullptr, nullptr, nullptr};
  const void *out = nullptr;  // the host output buffer the graph writes
  int lens_cur = 0;           // the device length buffer it reads
  // Zero-copy mode: the kernel nodes that read or write the host buffers
  // (-1: a kernel that cannot be re-pointed), their captured parameters (the
  // argument pointers refer to the captured graph, which is never changed),
  // and the device views of q, k, v and out they were captured with.
  int nkern = 0;
  cudaGraphNode_t kern[4] = {};
  cudaKernelNodeParams kparams[4] = {};
  const void *cap_dev[4] = {};
};

// Library-managed state behind pk_step_buffers.state: the prepared step
// (pk_decode_step_prepare) and, per staging half, the captured graph of the
// steady resident steps that read that half and an event recorded after the
// last step that read it.
struct StepState {
  GraphSlot slot[2];
  cudaEvent_t done[2] = {nullptr, nullptr};
  cudaStream_t stream = nullptr;  // the stream the graphs were captured on
  bool zero_copy = false;         // the graphs were captured in zero-copy mode
  bool failed = false;            // capture is not possible on this stream: stop trying
  // The prepared step.
  bool prepared = false;
  int half = 1;  // staging half of the last prepared step; the next one takes the other
  bool resident = false;
  bool new_part = false;
  int32_t npairs = 0;
  int32_t max_ctx = 0;
  size_t meta_copy = 0;
  int32_t num_seqs = 0, max_blocks = 0;
  int lens_cur = 0;  // device buffer holding the current lengths: 0 = lens, 1 = lens_b
  // Device mappings of zero-copy host buffers, looked up once per address
  // (enough entries for a caller that cycles through many sets of buffers).
  static constexpr int kMapCache = 128;
  const void *map_host[kMapCache] = {};
  void *map_dev[kMapCache] = {};
  int map_next = 0;
  // 1 if the GPU reads host memory through the host's page tables (a
  // Grace-attached GPU): a host address is then its own device address and
  // nothing is looked up; -1 until queried.
  int host_page_tables = -1;
};

// The device address of host memory `h` (zero-copy): `h` itself where the GPU
// uses the host's page tables, else pinned memory's mapping from the state's
// cache or the runtime; false if `h` is not addressable from the device.
bool mapped(StepState *st, const void *h, void **d) {
  if (st->host_page_tables < 0) {
    int dev = 0, v = 0;
    st->host_page_tables =
        cudaGetDevice(&dev) == cudaSuccess &&
                cudaDeviceGetAttribute(&v, cudaDevAttrPageableMemoryAccessUsesHostPageTables,
                                       dev) == cudaSuccess && v
            ? 1
            : 0;
    cudaGetLastError();
  }
  if (st->host_page_tables) {
    *d = const_cast<void *>(h);
    return h != nullptr;
  }
  for (int i = 0; i < StepState::kMapCache; ++i)
    if (st->map_host[i] == h && h) {
      *d = st->map_dev[i];
      return true;
    }
  if (cudaHostGetDevicePointer(d, const_cast<void *>(h), 0) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  st->map_host[st->map_next] = h;
  st->map_dev[st->map_next] = *d;
  st->map_next = (st->map_next + 1) % StepState::kMapCache;
  return true;
}

// Zero-copy graphs: records the kernel nodes of a captured step (attention,
// merge, and the CUDA-core path's separate scatter) and the device views of q,
// k, v and out they use (nkern -1 if a kernel node is none of those, so the
// graph cannot be re-pointed).
void find_kernel_nodes(GraphSlot &g, const void *const dev[4]) {
  g.nkern = 0;
  size_t n = 0;
  if (cudaGraphGetNodes(g.graph, nullptr, &n) != cudaSuccess) {
    g.nkern = -1;
    return;
  }
  std::vector<cudaGraphNode_t> nodes(n);
  if (n && cudaGraphGetNodes(g.graph, nodes.data(), &n) != cudaSuccess) n = 0, g.nkern = -1;
  for (size_t i = 0; i < n && g.nkern >= 0; ++i) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(nodes[i], &t) != cudaSuccess) {
      g.nkern = -1;
    } else if (t == cudaGraphNodeTypeKernel) {
      cudaKernelNodeParams kp{};
      if (g.nkern == 4 || cudaGraphKernelNodeGetParams(nodes[i], &kp) != cudaSuccess ||
          !kp.kernelParams ||
          (pkx_attn_kernel_arity(kp.func) <= 0 && pkx_scatter_kernel_arity(kp.func) <= 0)) {
        g.nkern = -1;
      } else {
        g.kparams[g.nkern] = kp;
        g.kern[g.nkern++] = nodes[i];
      }
    }
  }
  cudaGetLastError();
  for (int k = 0; k < 4; ++k) g.cap_dev[k] = dev[k];
}

// Points the captured kernels of a zero-copy graph at the device views `dev`
// of other host buffers (q, k, v, out), from their captured parameters; false
// if that is not possible (the graph is then dropped).
bool repoint_kernels(GraphSlot &g, const void *const dev[4]) {
  if (g.nkern <= 0) return false;
  const size_t psize = pkx_attn_params_size();
  alignas(16) unsigned char blob[1024];
  if (psize > sizeof(blob)) return false;
  constexpr int kMaxArgs = 16;
  for (int k = 0; k < g.nkern; ++k) {
    cudaKernelNodeParams kp = g.kparams[k];
    void *args[kMaxArgs] = {};
    const void *kv[2] = {};
    int arity = pkx_attn_kernel_arity(kp.func);
    if (arity > 0) {  // an attention or merge kernel: the parameter block first
      if (arity > kMaxArgs) return false;
      std::memcpy(blob, kp.kernelParams[0], psize);
      pkx_attn_params_rebind(blob, g.cap_dev, dev);
      args[0] = blob;
      for (int a = 1; a < arity; ++a) args[a] = kp.kernelParams[a];
    } else {  // the scatter: its first two arguments are the new K and V
      arity = pkx_scatter_kernel_arity(kp.func);
      if (arity < 2 || arity > kMaxArgs) return false;
      for (int a = 0; a < 2; ++a) {
        std::memcpy(&kv[a], kp.kernelParams[a], sizeof(kv[a]));
        if (kv[a] == g.cap_dev[1 + a]) kv[a] = dev[1 + a];
        args[a] = &kv[a];
      }
      for (int a = 2; a < arity; ++a) args[a] = kp.kernelParams[a];
    }
    kp.kernelParams = args;
    kp.extra = nullptr;
    if (cudaGraphExecKernelNodeSetParams(g.exec, g.kern[k], &kp) != cudaSuccess) return false;
  }
  return true;
}

void drop_slot(GraphSlot &g) {
  if (g.exec) cudaGraphExecDestroy(g.exec);  // freed once a launch in flight completes
  if (g.graph) cudaGraphDestroy(g.graph);
  g = GraphSlot{};
}

void drop_graphs(StepState *st) {
  drop_slot(st->slot[0]);
  drop_slot(st->slot[1]);
}

StepState *state_of(pk_step_buffers *b) {
  if (!b->state) b->state = new (std::nothrow) StepState;
  return static_cast<StepState *>(b->state);
}

// A stream on which the library may capture: one the caller created, not the
// legacy or per-thread default stream, and not being captured already.
bool capturable(cudaStream_t s) {
  if (s == nullptr || s == cudaStreamLegacy || s == cudaStreamPerThread) return false;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return cs == cudaStreamCaptureStatusNone;
}

}  // namespace

extern "C" {

size_t pk_decode_step_meta_bytes(int32_t num_seqs, int32_t max_blocks_per_seq) {
  if (num_seqs <= 0 || max_blocks_per_seq <= 0) return 0;
  return 2 * layout(num_seqs, max_blocks_per_seq).total;  // two staging halves
}

pk_status pk_decode_step_prepare(pk_bm *bm, const int64_t *seq_ids, int32_t num_seqs,
                                 int32_t num_q_heads, int32_t max_blocks_per_seq,
                                 int32_t partition_size, const pk_cache_desc *desc,
                                 pk_step_buffers *b) {
  if (!bm || !desc || !b || num_seqs <= 0 || !seq_ids || max_blocks_per_seq <= 0 ||
      !b->meta_host)
    return PK_ERR_INVALID_ARG;
  if (elem_size(desc->dtype) == 0) return PK_ERR_UNSUPPORTED;
  const MetaLayout m = layout(num_seqs, max_blocks_per_seq);
  if (b->meta_bytes < 2 * m.total) return PK_ERR_INVALID_ARG;
  StepState *st = state_of(b);
  if (!st) return PK_ERR_NOMEM;
  if (st->prepared) return PK_ERR_INVALID_ARG;  // the prepared step has not been launched
  const bool resident = b->tables_resident != 0;
  if (resident && (st->num_seqs != num_seqs || st->max_blocks != max_blocks_per_seq))
    return PK_ERR_INVALID_ARG;
  const int h = st->half ^ 1;
  // The step that last read this half (two steps back) must be done with it.
  if (st->done[h] && cudaEventSynchronize(st->done[h]) != cudaSuccess) return PK_ERR_CUDA;
  uint8_t *mh = static_cast<uint8_t *>(b->meta_host) + size_t(h) * m.total;
  int64_t *slots = reinterpret_cast<int64_t *>(mh + m.slots);
  int64_t *pairs = reinterpret_cast<int64_t *>(mh + m.pairs);
  int32_t *tables = reinterpret_cast<int32_t *>(mh + m.tables);
  int32_t *lens = reinterpret_cast<int32_t *>(mh + m.lens);
  int32_t *items = reinterpret_cast<int32_t *>(mh + m.items);
  if (resident) {
    // The lengths as the previous step left them (the host mirror of the
    // device lengths); every row must have room for one more token.
    const uint8_t *prev = static_cast<const uint8_t *>(b->meta_host) + size_t(h ^ 1) * m.total;
    std::memcpy(lens, prev + m.lens, size_t(num_seqs) * sizeof(int32_t));
    for (int32_t i = 0; i < num_seqs; ++i)
      if (int64_t(lens[i]) + 1 > int64_t(max_blocks_per_seq) * desc->block_size)
        return PK_ERR_INVALID_ARG;
  }

  int32_t npairs = 0;
  pk_status rc = pk_bm_append_batch(bm, seq_ids, num_seqs, slots, pairs, &npairs);
  if (rc != PK_OK) return rc;
  b->tables_resident = 0;  // until this step's metadata is on its way
  size_t meta_copy = m.lens_b;  // a full step: everything up to the tables
  bool new_part = false;
  if (resident) {
    const int32_t part = b->plan_partition;
    for (int32_t i = 0; i < num_seqs; ++i) {
      lens[i] += 1;
      if (part > 0 && (lens[i] - 1) % part == 0) new_part = true;
    }
    meta_copy = m.pairs + size_t(npairs) * 2 * sizeof(int64_t);
    if (new_part) {
      rc = pk_attention_work_items(lens, num_seqs, part, items, m.item_cap, &b->plan_items);
      if (rc != PK_OK) return rc;
      meta_copy = m.items + size_t(b->plan_items) * 2 * sizeof(int32_t);
    }
  } else {
    rc = pk_bm_export_tables(bm, seq_ids, num_seqs, max_blocks_per_seq, tables, lens);
    if (rc != PK_OK) return rc;
    rc = pk_attention_plan(lens, num_seqs, num_q_heads, partition_size, desc, &b->plan_partition,
                           items, m.item_cap, &b->plan_items);
    if (rc != PK_OK) return rc;
  }
  st->prepared = true;
  st->half = h;
  st->resident = resident;
  st->new_part = new_part;
  st->npairs = npairs;
  st->meta_copy = meta_copy;
  st->max_ctx = *std::max_element(lens, lens + num_seqs);
  st->num_seqs = num_seqs;
  st->max_blocks = max_blocks_per_seq;
  return PK_OK;
}

pk_status pk_decode_step_launch(int32_t num_seqs, int32_t num_q_heads, float scale,
                                int32_t max_blocks_per_seq, void *k_cache, void *v_cache,
                                const pk_cache_desc *desc, pk_step_buffers *b, void *stream) {
  if (!desc || !b || num_seqs <= 0 || max_blocks_per_seq <= 0) return PK_ERR_INVALID_ARG;
  StepState *st = static_cast<StepState *>(b->state);
  if (!st || !st->prepared || st->num_seqs != num_seqs || st->max_blocks != max_blocks_per_seq)
    return PK_ERR_INVALID_ARG;  // nothing prepared for this shape
  const int64_t esz = elem_size(desc->dtype);
  if (esz == 0) return PK_ERR_UNSUPPORTED;
  if (!b->q_host || !b->k_host || !b->v_host || !b->meta_host || !b->meta_dev || !b->out_host)
    return PK_ERR_INVALID_ARG;
  st->prepared = false;  // consumed, whatever happens below
  // Zero-copy mode (no device copies given): the kernels read q and the new
  // K/V from, and write the output to, the pinned host buffers through their
  // device mappings; the bytes still cross the host link every step, inside
  // the kernels instead of as separate copies.
  const bool zero_copy = !b->q_dev && !b->k_dev && !b->v_dev && !b->out_dev;
  if (!zero_copy && (!b->q_dev || !b->k_dev || !b->v_dev || !b->out_dev)) return PK_ERR_INVALID_ARG;
  void *qd = b->q_dev, *kd = b->k_dev, *vd = b->v_dev, *od = b->out_dev;
  if (zero_copy && (!mapped(st, b->q_host, &qd) || !mapped(st, b->k_host, &kd) ||
                    !mapped(st, b->v_host, &vd) || !mapped(st, b->out_host, &od)))
    return PK_ERR_INVALID_ARG;  // not host memory the device can address
  const MetaLayout m = layout(num_seqs, max_blocks_per_seq);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int h = st->half;
  const uint8_t *mh = static_cast<const uint8_t *>(b->meta_host) + size_t(h) * m.total;
  uint8_t *md = static_cast<uint8_t *>(b->meta_dev);
  const bool resident = st->resident;
  const int32_t npairs = st->npairs;
  const size_t meta_copy = st->meta_copy;
  const int32_t max_ctx = st->max_ctx;
  if (!st->done[h] && cudaEventCreateWithFlags(&st->done[h], cudaEventDisableTiming) != cudaSuccess)
    return PK_ERR_CUDA;

  const size_t qbytes = size_t(num_seqs) * num_q_heads * desc->head_dim * esz;
  const size_t kvbytes = size_t(num_seqs) * desc->num_kv_heads * desc->head_dim * esz;
  const void *srcs[3] = {b->q_host, b->k_host, b->v_host};
  void *dsts[3] = {qd, kd, vd};
  const size_t sizes[3] = {qbytes, kvbytes, kvbytes};
  auto enqueue_inputs = [&]() -> bool {
    if (zero_copy) return true;
    for (int k = 0; k < 3; ++k)
      if (cudaMemcpyAsync(dsts[k], srcs[k], sizes[k], cudaMemcpyHostToDevice, s) != cudaSuccess)
        return false;
    return true;
  };

  if (!resident || st->new_part || st->stream != s) drop_graphs(st);
  int32_t *dtables = reinterpret_cast<int32_t *>(md + m.tables);
  // The step's slots: in zero-copy mode the resident kernel reads them from
  // the staging half through its device mapping, so a steady step copies no
  // metadata at all; otherwise from the device copy.
  const int64_t *dslots = reinterpret_cast<const int64_t *>(md + m.slots);
  bool slots_mapped = false;
  if (zero_copy && resident) {
    void *p = nullptr;
    if (mapped(st, mh + m.slots, &p)) {  // else copy the slots as in the copying mode
      dslots = static_cast<const int64_t *>(p);
      slots_mapped = true;
    }
  }
  const bool copy_meta = !(slots_mapped && npairs == 0 && !st->new_part);
  // A resident step reads the lengths from one device buffer and writes the
  // advanced lengths to the other; a full step uploads them into lens.
  int32_t *lens_in = reinterpret_cast<int32_t *>(md + (st->lens_cur ? m.lens_b : m.lens));
  int32_t *lens_out = reinterpret_cast<int32_t *>(md + (st->lens_cur ? m.lens : m.lens_b));
  // Everything the device does in a step after the input copies.
  auto enqueue_device = [&]() -> pk_status {
    if (copy_meta && cudaMemcpyAsync(md, mh, meta_copy, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return PK_ERR_CUDA;
    pk_status r = PK_OK;
    if (npairs > 0) {
      r = pk_copy_blocks(k_cache, v_cache, reinterpret_cast<const int64_t *>(md + m.pairs), npairs,
                         desc, stream);
      if (r != PK_OK) return r;
    }
    const int32_t *ditems = reinterpret_cast<const int32_t *>(md + m.items);
    if (resident) {
      // One launch: the scatter, the table bookkeeping and the attention.
      r = pk_paged_attention_decode_advance(
          od, qd, kd, vd, dslots, k_cache, v_cache, dtables, lens_in, lens_out, scale, num_seqs,
          num_q_heads, max_blocks_per_seq, max_ctx, b->plan_partition, ditems, b->plan_items,
          b->workspace, b->workspace_bytes, desc, stream);
    } else {
      int32_t *dlens = reinterpret_cast<int32_t *>(md + m.lens);
      r = pk_reshape_and_cache(kd, vd, dslots, num_seqs, k_cache, v_cache, desc, stream);
      if (r != PK_OK) return r;
      r = pk_paged_attention_decode_items(od, qd, k_cache, v_cache, dtables, dlens, scale,
                                          num_seqs, num_q_heads, max_blocks_per_seq, max_ctx,
                                          b->plan_partition, ditems, b->plan_items, b->workspace,
                                          b->workspace_bytes, desc, PK_ATTN_AUTO, stream);
    }
    if (r != PK_OK) return r;
    if (!zero_copy &&
        cudaMemcpyAsync(b->out_host, b->out_dev, qbytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return PK_ERR_CUDA;
    return PK_OK;
  };
  // After the step's work: the staging half is free again once the stream
  // passes this point. A captured graph records the event itself (an
  // external event node), so a replay is a single call.
  auto mark_half = [&](bool recorded) -> pk_status {
    if (!recorded && cudaEventRecord(st->done[h], s) != cudaSuccess) return PK_ERR_CUDA;
    st->lens_cur = resident ? st->lens_cur ^ 1 : 0;
    b->tables_resident = 1;
    return PK_OK;
  };

  // A steady resident step (no copy-on-write pair, the same work list) runs
  // as the captured graph of its staging half.
  const bool may_replay = resident && !st->failed && capturable(s);
  const bool steady = may_replay && npairs == 0 && !st->new_part;
  if (steady) {
    GraphSlot &g = st->slot[h];
    if (g.exec && g.lens_cur != st->lens_cur) drop_slot(g);  // captured on the other length buffer
    if (!g.exec) {
      st->stream = s;
      bool ok = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
      if (ok) {
        const bool enq = enqueue_inputs() && enqueue_device() == PK_OK &&
                         cudaEventRecordWithFlags(st->done[h], s, cudaEventRecordExternal) ==
                             cudaSuccess;
        cudaGraph_t cg = nullptr;
        ok = cudaStreamEndCapture(s, &cg) == cudaSuccess && enq && cg;
        g.graph = cg;
        ok = ok && cudaGraphInstantiate(&g.exec, cg, 0) == cudaSuccess;
        // The input copies' nodes, found by their destinations (zero-copy
        // mode has none: its host addresses are part of the kernels' arguments).
        size_t n = 0;
        if (ok && !zero_copy) ok = cudaGraphGetNodes(cg, nullptr, &n) == cudaSuccess;
        std::vector<cudaGraphNode_t> nodes(n);
        if (ok && n) ok = cudaGraphGetNodes(cg, nodes.data(), &n) == cudaSuccess;
        for (size_t i = 0; ok && i < n; ++i) {
          cudaGraphNodeType t;
          if (cudaGraphNodeGetType(nodes[i], &t) != cudaSuccess || t != cudaGraphNodeTypeMemcpy)
            continue;
          cudaMemcpy3DParms mp{};
          if (cudaGraphMemcpyNodeGetParams(nodes[i], &mp) != cudaSuccess) continue;
          for (int k = 0; k < 3; ++k)
            if (mp.dstPtr.ptr == dsts[k]) g.copy_node[k] = nodes[i];
        }
        ok = ok && (zero_copy || (g.copy_node[0] && g.copy_node[1] && g.copy_node[2]));
        if (ok && zero_copy) {
          const void *views[4] = {qd, kd, vd, od};
          find_kernel_nodes(g, views);
        }
        st->zero_copy = zero_copy;
      }
      if (!ok) {
        cudaGetLastError();
        drop_graphs(st);
        st->failed = true;
      } else {
        for (int k = 0; k < 3; ++k) g.src[k] = srcs[k];
        g.out = b->out_host;
        g.lens_cur = st->lens_cur;
      }
    }
    const bool moved = st->zero_copy && (g.src[0] != srcs[0] || g.src[1] != srcs[1] ||
                                         g.src[2] != srcs[2] || g.out != b->out_host);
    if (g.exec && moved && st->zero_copy == zero_copy) {
      // Other host buffers than the graph was captured with: point its
      // kernels at them (from the captured parameters).
      const void *views[4] = {qd, kd, vd, od};
      if (repoint_kernels(g, views)) {
        for (int k = 0; k < 3; ++k) g.src[k] = srcs[k];
        g.out = b->out_host;
      } else {
        cudaGetLastError();
        drop_graphs(st);  // run it the normal way
      }
    }
    if (g.exec && (g.out != b->out_host || st->zero_copy != zero_copy)) {
      drop_graphs(st);  // other host buffers than the graph's arguments: run it the normal way
    } else if (g.exec) {
      for (int k = 0; k < 3; ++k)
        if (g.src[k] != srcs[k]) {
          if (cudaGraphExecMemcpyNodeSetParams1D(g.exec, g.copy_node[k], dsts[k], srcs[k],
                                                 sizes[k], cudaMemcpyHostToDevice) != cudaSuccess)
            return PK_ERR_CUDA;
          g.src[k] = srcs[k];
        }
      if (cudaGraphLaunch(g.exec, s) != cudaSuccess) return PK_ERR_CUDA;
      return mark_half(true);
    }
  }

  if (!enqueue_inputs()) return PK_ERR_CUDA;
  const pk_status r = enqueue_device();
  if (r != PK_OK) return r;
  return mark_half(false);
}

pk_status pk_decode_step(pk_bm *bm, const int64_t *seq_ids, int32_t num_seqs, int32_t num_q_heads,
                         float scale, int32_t max_blocks_per_seq, int32_t partition_size,
                         void *k_cache, void *v_cache, const pk_cache_desc *desc,
                         pk_step_buffers *b, void *stream) {
  const pk_status r = pk_decode_step_prepare(bm, seq_ids, num_seqs, num_q_heads,
                                             max_blocks_per_seq, partition_size, desc, b);
  if (r != PK_OK) return r;
  return pk_decode_step_launch(num_seqs, num_q_heads, scale, max_blocks_per_seq, k_cache, v_cache,
                               desc, b, stream);
}

int32_t pk_decode_step_graph_count(const pk_step_buffers *b) {
  if (!b || !b->state) return 0;
  const StepState *st = static_cast<const StepState *>(b->state);
  return int32_t(st->slot[0].exec != nullptr) + int32_t(st->slot[1].exec != nullptr);
}

void pk_decode_step_release(pk_step_buffers *b) {
  if (!b || !b->state) return;
  StepState *st = static_cast<StepState *>(b->state);
  drop_graphs(st);
  for (cudaEvent_t &e : st->done)
    if (e) {
      cudaEventDestroy(e);
      e = nullptr;
    }
  delete st;
  b->state = nullptr;
}

}  // extern "C"
