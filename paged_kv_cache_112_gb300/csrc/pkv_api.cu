// Host side of the libpkv C ABI: argument validation, TMA descriptor
// encoding and kernel launches.  No allocation, no device synchronisation.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace pkv {

namespace {
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
}  // namespace

// The CUDA error behind the calling thread's last PKV_ERR_CUDA (0: none yet):
// a cudaError_t, or minus a CUresult when descriptor encoding failed.
thread_local int t_last_cuda_error = 0;

pkv_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return PKV_OK;
  t_last_cuda_error = static_cast<int>(e);
  cudaGetLastError();  // a launch error is not sticky: clear it for the next call on this thread
  return PKV_ERR_CUDA;
}

pkv_status cuda_status_fail(int code) {
  t_last_cuda_error = code;
  return PKV_ERR_CUDA;
}

int current_sm_count(int fallback) {
  // Filled once per device; readers see either 0 (not yet known) or the
  // count, never a torn value.
  static std::atomic<int> cache[256];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) {
    cudaGetLastError();
    return fallback;
  }
  int n = cache[dev].load(std::memory_order_acquire);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return fallback;
  }
  cache[dev].store(n, std::memory_order_release);
  return n;
}

int resident_warp_slots(const void* kernel, int threads, size_t smem) {
  struct Entry {
    const void* kernel;
    int dev, threads;
    size_t smem;
    int slots;
  };
  static Entry table[32];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (table[i].kernel == kernel && table[i].dev == dev && table[i].threads == threads && table[i].smem == smem)
        return table[i].slots;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm <= 0) {
    cudaGetLastError();
    per_sm = 1;
  }
  const int slots = current_sm_count(1) * per_sm * (threads / 32);
  std::lock_guard<std::mutex> lock(mu);
  if (used < 32) table[used++] = Entry{kernel, dev, threads, smem, slots};
  return slots;
}

cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
  struct Entry {
    const void* kernel;
    int dev;
    size_t bytes;
  };
  static Entry table[64];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (table[i].kernel == kernel && table[i].dev == dev && table[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  for (int i = 0; i < used; ++i)
    if (table[i].kernel == kernel && table[i].dev == dev) {
      table[i].bytes = bytes;
      return cudaSuccess;
    }
  if (used < 64) table[used++] = Entry{kernel, dev, bytes};
  return cudaSuccess;
}

WorkspaceLayout workspace_layout(int num_seqs, int num_q_heads, int head_dim, int max_parts) {
  WorkspaceLayout w{};
  if (max_parts <= 1) return w;
  const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * max_parts;
  w.acc_offset = 0;
  w.ml_offset = align256(rows * head_dim * sizeof(float));
  w.meta_offset = w.ml_offset + align256(rows * 2 * sizeof(float));
  w.total = w.meta_offset;
  return w;
}

WorkspaceLayout balanced_workspace_layout(int num_seqs, int num_q_heads, int head_dim, int64_t warps) {
  WorkspaceLayout w{};
  const size_t heads = static_cast<size_t>(num_q_heads < 8 ? num_q_heads : 8);  // group size bound
  const size_t recs = static_cast<size_t>(warps) * 2 * heads;
  w.acc_offset = 0;
  w.ml_offset = align256(recs * head_dim * sizeof(float));
  w.meta_offset = w.ml_offset + align256(recs * 2 * sizeof(float));
  w.total = w.meta_offset + align256(static_cast<size_t>(num_seqs) * num_q_heads * 2 * sizeof(int));
  return w;
}

namespace {

constexpr long long kWaitTimeoutNs = 2000000000LL;  // 2 s per bounded wait

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

bool kv_dtype_ok(pkv_dtype d) { return d == PKV_F16 || d == PKV_BF16; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// cuTensorMapEncodeTiled needs a current context.  A host thread that has
// made no CUDA runtime call yet has none; the runtime would bind the
// device's primary context at its first launch, so do the same here (a
// thread that already has a context, primary or its own, keeps it).
bool bind_context_if_none() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  CUcontext ctx = nullptr;
  if (get_current && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr) return true;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
    t_last_cuda_error = static_cast<int>(cudaGetLastError());
    return false;
  }
  return true;
}

// Describes a pool of `eb`-byte elements, blocks `block_stride` elements
// apart, for TMA tile loads in the 128-byte swizzle (a 128-byte line is the
// widest a swizzled box row may be).  A head's row of head_dim * eb bytes is
// head_dim * eb / 128 lines.
//  * Blocks of 16 tokens or more: dimensions {element in line, row in block,
//    line (head * lines per head + line), block}, with the rows (stride
//    num_kv_heads * head_dim * eb) before the lines (stride 128).  One box
//    {128 bytes, 16 rows, lines per head, 1} is a whole (block, head) tile,
//    landing in shared memory as [line][16 rows][128 bytes]: one copy per K
//    or V tile, whatever head_dim is.
//  * 8-token blocks: {element in line, line, row in block, block}; a box
//    {128 bytes, 1, 8, 1} is one line of one head's 8 rows (a 16-row tile is
//    two blocks, so lines per head x 2 boxes).
// A block stride above one block's rows is a layer slice of a pool that
// keeps all layers of a block together.
bool encode_pool_map_uncached(CUtensorMap* map, const void* pool, int num_blocks, int block_size, int num_kv_heads,
                              int head_dim, int eb, int64_t block_stride, int heads_per_box) {
  auto fn = encode_fn();
  if (!fn) {
    t_last_cuda_error = static_cast<int>(cudaErrorSymbolNotFound);
    return false;
  }
  if (!bind_context_if_none()) return false;
  const cuuint32_t line = 128 / eb;  // elements per 128-byte line
  const cuuint64_t lines = static_cast<cuuint64_t>(num_kv_heads) * (head_dim / line);
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(num_kv_heads) * head_dim * eb;
  const bool whole_head = block_size >= kTile;
  const cuuint64_t dims[4] = {line, whole_head ? static_cast<cuuint64_t>(block_size) : lines,
                              whole_head ? lines : static_cast<cuuint64_t>(block_size),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {whole_head ? row_bytes : 128, whole_head ? 128 : row_bytes,
                                 static_cast<cuuint64_t>(block_stride) * eb};
  const cuuint32_t box[4] = {line, whole_head ? static_cast<cuuint32_t>(kTile) : 1u,
                             whole_head ? static_cast<cuuint32_t>(head_dim * eb / 128 * heads_per_box)
                                        : static_cast<cuuint32_t>(block_size),
                             1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, eb == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 4,
                        const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B,
                        head_dim * eb >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) t_last_cuda_error = -static_cast<int>(r);
  return r == CUDA_SUCCESS;
}

// Descriptors depend only on the pool address and geometry, so recent ones
// are kept (a small round-robin cache) instead of re-encoded every call.
// heads_per_box > 1 (blocks of >= 16 tokens): one box holds that many
// adjacent KV heads' tiles of a block, one after the other.
bool encode_pool_map(CUtensorMap* map, const void* pool, int num_blocks, int block_size, int num_kv_heads,
                     int head_dim, int eb, int64_t block_stride, int heads_per_box = 1) {
  struct Entry {
    const void* pool;
    int num_blocks, block_size, num_kv_heads, head_dim, eb, heads_per_box;
    int64_t block_stride;
    CUtensorMap map;
  };
  static Entry cache[64];
  static int next = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
      if (e.pool == pool && e.num_blocks == num_blocks && e.block_size == block_size &&
          e.num_kv_heads == num_kv_heads && e.head_dim == head_dim && e.eb == eb && e.block_stride == block_stride &&
          e.heads_per_box == heads_per_box) {
        *map = e.map;
        return true;
      }
  }
  if (!encode_pool_map_uncached(map, pool, num_blocks, block_size, num_kv_heads, head_dim, eb, block_stride,
                                heads_per_box))
    return false;
  std::lock_guard<std::mutex> lock(mu);
  cache[next] = Entry{pool, num_blocks, block_size, num_kv_heads, head_dim, eb, heads_per_box, block_stride, *map};
  next = (next + 1) % 64;
  return true;
}

// log2 of a supported block size (8, 16, 32 or 64 tokens), else -1.
int block_shift_of(int block_size) {
  switch (block_size) {
    case 8: return 3;
    case 16: return 4;
    case 32: return 5;
    case 64: return 6;
    default: return -1;
  }
}

// Block stride of a pool: 0 means dense (block_size * num_kv_heads *
// head_dim); otherwise at least that and a multiple of 8 elements (16 bytes
// at 16 bits).  Returns -1 when invalid.
int64_t resolve_block_stride(int64_t block_stride, int block_size, int num_kv_heads, int head_dim) {
  const int64_t dense = static_cast<int64_t>(block_size) * num_kv_heads * head_dim;
  if (block_stride == 0) return dense;
  if (block_stride < dense || block_stride % 8 != 0) return -1;
  return block_stride;
}

int parts_for(int max_context_len, int partition_size, int* ps_out) {
  int ps = partition_size;
  if (ps <= 0) {  // one partition per sequence
    const int len = max_context_len > 0 ? max_context_len : 1;
    ps = ((len + kTile - 1) / kTile) * kTile;
  }
  *ps_out = ps;
  const int len = max_context_len > 0 ? max_context_len : 1;
  return (len + ps - 1) / ps;
}

// Workspace of a decode call (fixed partitions or balanced split).
WorkspaceLayout decode_layout(int num_seqs, int num_q_heads, int head_dim, int max_context_len, int partition_size,
                              int sm_count, int* max_parts_out) {
  if (partition_size == PKV_PARTITION_BALANCED) {
    *max_parts_out = 1;
    const int64_t warps = static_cast<int64_t>(sm_count) * balanced_warps_per_cta(head_dim, num_seqs);
    return balanced_workspace_layout(num_seqs, num_q_heads, head_dim, warps);
  }
  int ps = 0;
  *max_parts_out = parts_for(max_context_len, partition_size, &ps);
  return workspace_layout(num_seqs, num_q_heads, head_dim, *max_parts_out);
}

struct DecodeCall {
  DecodeArgs args;
  CUtensorMap tmap_k, tmap_v;
};

pkv_status prepare_decode(DecodeCall* c, void* out, const void* q, const void* k_pool, const void* v_pool,
                          int64_t block_stride, const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens,
                          int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, float scale, int partition_size, int max_context_len, void* workspace,
                          size_t workspace_bytes, pkv_dtype kv_dtype, pkv_dtype out_dtype, int32_t* dev_status,
                          bool need_maps) {
  const bool balanced = partition_size == PKV_PARTITION_BALANCED;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq < 0 || num_blocks <= 0 ||
      max_context_len < 0 || (partition_size < 0 && !balanced) || !std::isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  const int shift = block_shift_of(block_size);
  if (shift < 0 || (balanced && block_size != kBlockSize)) return PKV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_UNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  if (group > 8) return PKV_ERR_UNSUPPORTED;
  if (!balanced && partition_size % kTile != 0) return PKV_ERR_UNSUPPORTED;
  if (balanced && num_seqs > kBalancedMaxSeqs) return PKV_ERR_UNSUPPORTED;
  if (!kv_dtype_ok(kv_dtype) || (out_dtype != PKV_F32 && out_dtype != PKV_F16 && out_dtype != PKV_BF16))
    return PKV_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!out || !q || !k_pool || !v_pool || !context_lens || (!block_tables && max_blocks_per_seq)))
    return PKV_ERR_INVALID_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(q, 4) ||
      !aligned(out, out_dtype == PKV_F32 ? 4 : 2) || !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return PKV_ERR_INVALID_ARG;
  const int64_t bstride = resolve_block_stride(block_stride, block_size, num_kv_heads, head_dim);
  if (bstride < 0) return PKV_ERR_INVALID_ARG;
  const int sms = balanced ? current_sm_count(0) : 0;
  if (balanced && sms <= 0) return cuda_status_fail(static_cast<int>(cudaErrorNoDevice));
  int max_parts = 1, ps = 0;
  const WorkspaceLayout ws =
      decode_layout(num_seqs, num_q_heads, head_dim, max_context_len, partition_size, sms, &max_parts);
  parts_for(max_context_len, partition_size, &ps);
  if (ws.total > 0 && (!workspace || workspace_bytes < ws.total || !aligned(workspace, 16)))
    return PKV_ERR_WORKSPACE;

  c->args = DecodeArgs{};  // every field not set below (the fused-step ones) is zero / null
  DecodeArgs& a = c->args;
  a.out = out;
  a.q = static_cast<const uint16_t*>(q);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  a.ws_acc = ws.total ? reinterpret_cast<float*>(wsb + ws.acc_offset) : nullptr;
  a.ws_ml = ws.total ? reinterpret_cast<float2*>(wsb + ws.ml_offset) : nullptr;
  a.ws_meta = (ws.total && balanced) ? reinterpret_cast<int2*>(wsb + ws.meta_offset) : nullptr;
  a.balanced_ctas = balanced ? sms : 0;
  a.dev_status = dev_status;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = group;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.partition_size = ps;
  a.max_parts = max_parts;
  a.max_context_len = max_context_len;
  a.block_shift = shift;
  a.block_stride = bstride;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out_dtype = static_cast<int>(out_dtype);
  a.timeout_ns = kWaitTimeoutNs;
  a.heads_per_box = 1;
  if (need_maps && num_seqs > 0) {
    // The launch picks its kernel by a.heads_per_box, so the boxes match it.
    if (!balanced) a.heads_per_box = partitions_heads_per_box(a, head_dim, kv_dtype == PKV_BF16);
    if (!encode_pool_map(&c->tmap_k, k_pool, num_blocks, block_size, num_kv_heads, head_dim, 2, bstride,
                         a.heads_per_box) ||
        !encode_pool_map(&c->tmap_v, v_pool, num_blocks, block_size, num_kv_heads, head_dim, 2, bstride,
                         a.heads_per_box))
      return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

pkv_status pkv_write_cache(const void* k_new, const void* v_new, void* k_pool, void* v_pool, int64_t block_stride,
                           const int32_t* slot_mapping, int num_tokens, int64_t new_row_stride, int num_kv_heads,
                           int head_dim, int block_size, int num_blocks, pkv_dtype kv_dtype, int32_t* dev_status,
                           void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 || new_row_stride < 0)
    return PKV_ERR_INVALID_ARG;
  if (!kv_dtype_ok(kv_dtype)) return PKV_ERR_INVALID_ARG;
  const int shift = block_shift_of(block_size);
  if (shift < 0) return PKV_ERR_UNSUPPORTED;
  const int row = num_kv_heads * head_dim;
  if (row % 8 != 0) return PKV_ERR_UNSUPPORTED;  // 16-byte vectors
  const int64_t bstride = resolve_block_stride(block_stride, block_size, num_kv_heads, head_dim);
  if (bstride < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !k_pool || !v_pool || !slot_mapping) return PKV_ERR_INVALID_ARG;
  const int64_t stride = new_row_stride ? new_row_stride : row;
  if (stride < row || stride % 8 != 0) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
      !aligned(slot_mapping, 4))
    return PKV_ERR_INVALID_ARG;
  WriteCacheArgs a{};
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.k_pool = static_cast<uint16_t*>(k_pool);
  a.v_pool = static_cast<uint16_t*>(v_pool);
  a.slot_mapping = slot_mapping;
  a.dev_status = dev_status;
  a.k_stride = stride;
  a.v_stride = stride;
  a.num_slots = static_cast<int64_t>(num_blocks) << shift;
  a.block_stride = bstride;
  a.block_shift = shift;
  a.num_tokens = num_tokens;
  a.row_elems = row;
  return cuda_status(launch_write_cache(a, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int num_pairs, int num_layers,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks, pkv_dtype kv_dtype,
                           int32_t* dev_status, void* stream) {
  if (num_pairs < 0 || num_layers <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!kv_dtype_ok(kv_dtype)) return PKV_ERR_INVALID_ARG;
  if (block_shift_of(block_size) < 0) return PKV_ERR_UNSUPPORTED;
  if ((num_kv_heads * head_dim) % 8 != 0) return PKV_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PKV_OK;
  if (!k_pool || !v_pool || !pairs) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(pairs, 4)) return PKV_ERR_INVALID_ARG;
  CopyBlocksArgs a{};
  a.k_pool = static_cast<uint16_t*>(k_pool);
  a.v_pool = static_cast<uint16_t*>(v_pool);
  a.pairs = pairs;
  a.dev_status = dev_status;
  a.block_elems = static_cast<int64_t>(num_layers) * block_size * num_kv_heads * head_dim;
  a.num_pairs = num_pairs;
  a.num_blocks = num_blocks;
  return cuda_status(launch_copy_blocks(a, static_cast<cudaStream_t>(stream)));
}

size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_context_len,
                                  int partition_size) {
  const bool balanced = partition_size == PKV_PARTITION_BALANCED;
  if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
      (!balanced && (partition_size < 0 || partition_size % kTile != 0)))
    return 0;
  int parts = 1;
  return decode_layout(num_seqs, num_q_heads, head_dim, max_context_len, partition_size,
                       balanced ? current_sm_count(256) : 0, &parts)
      .total;
}

pkv_status pkv_decode_partitions(void* out, const void* q, const void* k_pool, const void* v_pool,
                                 int64_t block_stride, const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                 int num_blocks, float scale, int partition_size, int max_context_len,
                                 void* workspace, size_t workspace_bytes, pkv_dtype kv_dtype, pkv_dtype out_dtype,
                                 int32_t* dev_status, void* stream) {
  DecodeCall c{};
  pkv_status st = prepare_decode(&c, out, q, k_pool, v_pool, block_stride, block_tables, max_blocks_per_seq,
                                 context_lens,
                                 num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                                 partition_size, max_context_len, workspace, workspace_bytes, kv_dtype, out_dtype,
                                 dev_status, true);
  if (st != PKV_OK || num_seqs == 0) return st;
  const cudaError_t e = c.args.balanced_ctas
                            ? launch_decode_balanced(c.args, c.tmap_k, c.tmap_v, head_dim, kv_dtype == PKV_BF16,
                                                     static_cast<cudaStream_t>(stream))
                            : launch_decode_partitions(c.args, c.tmap_k, c.tmap_v, head_dim, kv_dtype == PKV_BF16,
                                                       static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

pkv_status pkv_decode_reduce(void* out, const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                             int head_dim, int partition_size, int max_context_len, const void* workspace,
                             size_t workspace_bytes, pkv_dtype out_dtype, int32_t* dev_status, void* stream) {
  const bool balanced = partition_size == PKV_PARTITION_BALANCED;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_context_len < 0 ||
      (partition_size < 0 && !balanced))
    return PKV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > 8) return PKV_ERR_UNSUPPORTED;
  if (!balanced && partition_size % kTile != 0) return PKV_ERR_UNSUPPORTED;
  if (out_dtype != PKV_F32 && out_dtype != PKV_F16 && out_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  const int sms = balanced ? current_sm_count(0) : 0;
  if (balanced && sms <= 0) return cuda_status_fail(static_cast<int>(cudaErrorNoDevice));
  int max_parts = 1, ps = 0;
  const WorkspaceLayout ws =
      decode_layout(num_seqs, num_q_heads, head_dim, max_context_len, partition_size, sms, &max_parts);
  parts_for(max_context_len, partition_size, &ps);
  if (ws.total == 0 || num_seqs == 0) return PKV_OK;
  if (!out || !context_lens) return PKV_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < ws.total || !aligned(workspace, 16)) return PKV_ERR_WORKSPACE;
  uint8_t* wsb = static_cast<uint8_t*>(const_cast<void*>(workspace));
  DecodeArgs a{};
  a.out = out;
  a.context_lens = context_lens;
  a.ws_acc = reinterpret_cast<float*>(wsb + ws.acc_offset);
  a.ws_ml = reinterpret_cast<float2*>(wsb + ws.ml_offset);
  a.ws_meta = balanced ? reinterpret_cast<int2*>(wsb + ws.meta_offset) : nullptr;
  a.dev_status = dev_status;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = num_q_heads / num_kv_heads;
  a.partition_size = ps;
  a.max_parts = max_parts;
  a.max_context_len = max_context_len;
  // Lengths are clamped as in the partition kernel; beyond max_context_len the
  // table width does not matter here.
  a.max_blocks_per_seq = (max_context_len + kTile - 1) / kTile;
  a.block_shift = 4;  // with the line above: lengths are clamped to max_context_len alone
  a.out_dtype = static_cast<int>(out_dtype);
  a.balanced_ctas = balanced ? sms : 0;
  const cudaError_t e = balanced ? launch_decode_reduce_balanced(a, head_dim, static_cast<cudaStream_t>(stream))
                                 : launch_decode_reduce(a, head_dim, static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

pkv_status pkv_decode_step_partitions(void* out, const void* q, const void* k_new, const void* v_new,
                                      int64_t new_row_stride, void* k_pool, void* v_pool, int64_t block_stride,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, const int32_t* slot_mapping, int num_seqs,
                                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                      int num_blocks, float scale, int partition_size, int max_context_len,
                                      void* workspace, size_t workspace_bytes, pkv_dtype kv_dtype,
                                      pkv_dtype out_dtype, int32_t* dev_status, void* stream) {
  DecodeCall c{};
  pkv_status st = prepare_decode(&c, out, q, k_pool, v_pool, block_stride, block_tables, max_blocks_per_seq,
                                 context_lens,
                                 num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                                 partition_size, max_context_len, workspace, workspace_bytes, kv_dtype, out_dtype,
                                 dev_status, true);
  if (st != PKV_OK || num_seqs == 0) return st;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  const int64_t stride = new_row_stride ? new_row_stride : row;
  if (!k_new || !v_new || !slot_mapping || new_row_stride < 0 || stride < row || stride % 8 != 0 ||
      !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 4))
    return PKV_ERR_INVALID_ARG;
  DecodeArgs& a = c.args;
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.new_stride = stride;
  a.slot_mapping = slot_mapping;
  a.k_pool_w = static_cast<uint16_t*>(k_pool);
  a.v_pool_w = static_cast<uint16_t*>(v_pool);
  const cudaError_t e = a.balanced_ctas ? launch_decode_balanced(a, c.tmap_k, c.tmap_v, head_dim,
                                                                kv_dtype == PKV_BF16, static_cast<cudaStream_t>(stream))
                                        : launch_decode_partitions(a, c.tmap_k, c.tmap_v, head_dim,
                                                                   kv_dtype == PKV_BF16,
                                                                   static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

pkv_status pkv_decode_step(void* out, const void* q, const void* k_new, const void* v_new, int64_t new_row_stride,
                           void* k_pool, void* v_pool, int64_t block_stride, const int32_t* block_tables,
                           int max_blocks_per_seq,
                           const int32_t* context_lens, const int32_t* slot_mapping, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                           int partition_size, int max_context_len, void* workspace, size_t workspace_bytes,
                           pkv_dtype kv_dtype, pkv_dtype out_dtype, int32_t* dev_status, void* stream) {
  pkv_status st = pkv_decode_step_partitions(out, q, k_new, v_new, new_row_stride, k_pool, v_pool, block_stride,
                                             block_tables,
                                             max_blocks_per_seq, context_lens, slot_mapping, num_seqs, num_q_heads,
                                             num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size,
                                             max_context_len, workspace, workspace_bytes, kv_dtype, out_dtype,
                                             dev_status, stream);
  if (st != PKV_OK) return st;
  return pkv_decode_reduce(out, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, partition_size,
                           max_context_len, workspace, workspace_bytes, out_dtype, dev_status, stream);
}

pkv_status pkv_decode_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                                int64_t block_stride, const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* context_lens,
                                int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, float scale, int partition_size, int max_context_len, void* workspace,
                                size_t workspace_bytes, pkv_dtype kv_dtype, pkv_dtype out_dtype, int32_t* dev_status,
                                void* stream) {
  pkv_status st = pkv_decode_partitions(out, q, k_pool, v_pool, block_stride, block_tables, max_blocks_per_seq,
                                        context_lens,
                                        num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                                        partition_size, max_context_len, workspace, workspace_bytes, kv_dtype,
                                        out_dtype, dev_status, stream);
  if (st != PKV_OK) return st;
  return pkv_decode_reduce(out, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, partition_size,
                           max_context_len, workspace, workspace_bytes, out_dtype, dev_status, stream);
}

// ------------------------------------------------------------ FP8 pools

pkv_status pkv_write_cache_fp8(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                               const float* k_scale, const float* v_scale, const int32_t* slot_mapping,
                               int num_tokens, int64_t new_row_stride, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, int num_layers, pkv_dtype new_dtype,
                               int32_t* dev_status, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 || new_row_stride < 0 ||
      num_layers <= 0 || num_layers > kMaxLayers)
    return PKV_ERR_INVALID_ARG;
  if (!kv_dtype_ok(new_dtype)) return PKV_ERR_INVALID_ARG;
  if (block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (head_dim % 16 != 0) return PKV_ERR_UNSUPPORTED;  // 16 codes per vector, within one head
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !k_pool || !v_pool || !k_scale || !v_scale || !slot_mapping) return PKV_ERR_INVALID_ARG;
  const int row = num_kv_heads * head_dim;
  const int64_t stride = new_row_stride ? new_row_stride : row;
  if (stride < row || stride % 8 != 0) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
      !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(slot_mapping, 4))
    return PKV_ERR_INVALID_ARG;
  WriteCacheFp8Args a{};
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.k_pool = static_cast<uint8_t*>(k_pool);
  a.v_pool = static_cast<uint8_t*>(v_pool);
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.slot_mapping = slot_mapping;
  a.dev_status = dev_status;
  a.stride = stride;
  a.num_slots = static_cast<int64_t>(num_blocks) * kBlockSize;
  a.block_stride = static_cast<int64_t>(num_layers) * kBlockSize * row;
  a.scale_stride = static_cast<int64_t>(num_layers) * num_kv_heads;
  a.num_tokens = num_tokens;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.new_bf16 = new_dtype == PKV_BF16;
  return cuda_status(launch_write_cache_fp8(a, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_copy_blocks_fp8(void* k_pool, void* v_pool, float* k_scale, float* v_scale, const int32_t* pairs,
                               int num_pairs, int num_layers, int num_kv_heads, int head_dim, int block_size,
                               int num_blocks, int32_t* dev_status, void* stream) {
  if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 || num_layers <= 0 ||
      num_layers > kMaxLayers)
    return PKV_ERR_INVALID_ARG;
  if (block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PKV_OK;
  if (!k_pool || !v_pool || !k_scale || !v_scale || !pairs) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(k_scale, 4) || !aligned(v_scale, 4) ||
      !aligned(pairs, 4))
    return PKV_ERR_INVALID_ARG;
  CopyBlocksArgs a{};
  a.k_pool = static_cast<uint16_t*>(k_pool);
  a.v_pool = static_cast<uint16_t*>(v_pool);
  a.pairs = pairs;
  a.dev_status = dev_status;
  // num_layers * 16 * H_kv * D bytes, counted in 16-bit units
  a.block_elems = static_cast<int64_t>(num_layers) * kBlockSize * num_kv_heads * head_dim / 2;
  a.num_pairs = num_pairs;
  a.num_blocks = num_blocks;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.scales_per_block = num_layers * num_kv_heads;
  return cuda_status(launch_copy_blocks(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace pkv {
namespace {

// Validation and descriptors shared by the FP8 decode entry points.
pkv_status prepare_decode_fp8(DecodeCall* c, void* out, const void* q, const void* k_pool, const void* v_pool,
                              const float* k_scale, const float* v_scale, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_q_heads,
                              int num_kv_heads, int head_dim, int block_size, int num_blocks, int num_layers,
                              float scale, int partition_size, int max_context_len, void* workspace,
                              size_t workspace_bytes, pkv_dtype q_dtype, pkv_dtype out_dtype, int32_t* dev_status,
                              bool fused) {
  if (block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (num_layers <= 0 || num_layers > kMaxLayers || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  // One byte per code: the block stride in codes is the stride in bytes.
  const int64_t block_bytes = static_cast<int64_t>(num_layers) * kBlockSize * num_kv_heads * head_dim;
  pkv_status st = prepare_decode(c, out, q, k_pool, v_pool, block_bytes, block_tables, max_blocks_per_seq, context_lens,
                                 num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                                 partition_size, max_context_len, workspace, workspace_bytes, q_dtype, out_dtype,
                                 dev_status, false);
  if (st != PKV_OK) return st;
  if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!k_scale || !v_scale || !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(q, 16))
    return PKV_ERR_INVALID_ARG;
  c->args.k_scale = k_scale;
  c->args.v_scale = v_scale;
  c->args.scale_stride = static_cast<int64_t>(num_layers) * num_kv_heads;
  // The launch picks its kernel by the same rule, so the boxes match it.
  const int hpb = fp8_heads_per_box(num_kv_heads, fused, partition_size == PKV_PARTITION_BALANCED);
  c->args.heads_per_box = hpb;
  if (!encode_pool_map(&c->tmap_k, k_pool, num_blocks, kBlockSize, num_kv_heads, head_dim, 1, c->args.block_stride,
                       hpb) ||
      !encode_pool_map(&c->tmap_v, v_pool, num_blocks, kBlockSize, num_kv_heads, head_dim, 1, c->args.block_stride,
                       hpb))
    return PKV_ERR_CUDA;
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_decode_partitions_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                                     const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                     int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                                     int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                     int num_layers, float scale, int partition_size, int max_context_len, void* workspace,
                                     size_t workspace_bytes, pkv_dtype q_dtype, pkv_dtype out_dtype,
                                     int32_t* dev_status, void* stream) {
  DecodeCall c{};
  const pkv_status st = prepare_decode_fp8(&c, out, q, k_pool, v_pool, k_scale, v_scale, block_tables,
                                           max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                                           head_dim, block_size, num_blocks, num_layers, scale, partition_size,
                                           max_context_len, workspace, workspace_bytes, q_dtype, out_dtype,
                                           dev_status, false);
  if (st != PKV_OK || num_seqs == 0) return st;
  if (c.args.balanced_ctas)
    return cuda_status(launch_decode_balanced_fp8(c.args, c.tmap_k, c.tmap_v, head_dim, q_dtype == PKV_BF16,
                                                  static_cast<cudaStream_t>(stream)));
  return cuda_status(launch_decode_partitions_fp8(c.args, c.tmap_k, c.tmap_v, head_dim, q_dtype == PKV_BF16,
                                      static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_decode_step_partitions_fp8(void* out, const void* q, const void* k_new, const void* v_new,
                                          int64_t new_row_stride, void* k_pool, void* v_pool, const float* k_scale,
                                          const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
                                          const int32_t* context_lens, const int32_t* slot_mapping, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                          int num_blocks, int num_layers, float scale, int partition_size, int max_context_len,
                                          void* workspace, size_t workspace_bytes, pkv_dtype q_dtype,
                                          pkv_dtype out_dtype, int32_t* dev_status, void* stream) {
  if (partition_size == PKV_PARTITION_BALANCED) return PKV_ERR_UNSUPPORTED;  // the fused write needs fixed partitions
  DecodeCall c{};
  const pkv_status st = prepare_decode_fp8(&c, out, q, k_pool, v_pool, k_scale, v_scale, block_tables,
                                           max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                                           head_dim, block_size, num_blocks, num_layers, scale, partition_size,
                                           max_context_len, workspace, workspace_bytes, q_dtype, out_dtype,
                                           dev_status, true);
  if (st != PKV_OK || num_seqs == 0) return st;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  const int64_t stride = new_row_stride ? new_row_stride : row;
  if (!k_new || !v_new || !slot_mapping || new_row_stride < 0 || stride < row || stride % 8 != 0 ||
      !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 4))
    return PKV_ERR_INVALID_ARG;
  DecodeArgs& a = c.args;
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.new_stride = stride;
  a.slot_mapping = slot_mapping;
  a.k_pool_w = static_cast<uint16_t*>(k_pool);  // written as bytes by the FP8 kernel
  a.v_pool_w = static_cast<uint16_t*>(v_pool);
  return cuda_status(launch_decode_partitions_fp8(a, c.tmap_k, c.tmap_v, head_dim, q_dtype == PKV_BF16,
                                      static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_decode_step_fp8(void* out, const void* q, const void* k_new, const void* v_new,
                               int64_t new_row_stride, void* k_pool, void* v_pool, const float* k_scale,
                               const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, const int32_t* slot_mapping, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               int num_layers, float scale, int partition_size, int max_context_len, void* workspace,
                               size_t workspace_bytes, pkv_dtype q_dtype, pkv_dtype out_dtype, int32_t* dev_status,
                               void* stream) {
  const pkv_status st = pkv_decode_step_partitions_fp8(
      out, q, k_new, v_new, new_row_stride, k_pool, v_pool, k_scale, v_scale, block_tables, max_blocks_per_seq,
      context_lens, slot_mapping, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, num_layers,
      scale, partition_size, max_context_len, workspace, workspace_bytes, q_dtype, out_dtype, dev_status, stream);
  if (st != PKV_OK) return st;
  return pkv_decode_reduce(out, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, partition_size,
                           max_context_len, workspace, workspace_bytes, out_dtype, dev_status, stream);
}

pkv_status pkv_decode_attention_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                                    const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                                    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                    int num_layers, float scale, int partition_size, int max_context_len, void* workspace,
                                    size_t workspace_bytes, pkv_dtype q_dtype, pkv_dtype out_dtype,
                                    int32_t* dev_status, void* stream) {
  pkv_status st = pkv_decode_partitions_fp8(out, q, k_pool, v_pool, k_scale, v_scale, block_tables,
                                            max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                                            head_dim, block_size, num_blocks, num_layers, scale, partition_size,
                                            max_context_len, workspace, workspace_bytes, q_dtype, out_dtype,
                                            dev_status, stream);
  if (st != PKV_OK) return st;
  return pkv_decode_reduce(out, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, partition_size,
                           max_context_len, workspace, workspace_bytes, out_dtype, dev_status, stream);
}

}  // extern "C"

namespace pkv {
namespace {

// The address the device dereferences for `p`: device and managed memory as
// is, pinned (page-locked, registered) host memory through its mapping.
// Returns nullptr for memory the device cannot reach (pageable host memory).
const void* device_view(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return p;
    case cudaMemoryTypeHost:
      return at.devicePointer;
    default:
      return nullptr;
  }
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_swap_blocks(void* dst_k, void* dst_v, int64_t dst_block_stride, int dst_num_blocks,
                           const void* src_k, const void* src_v, int64_t src_block_stride, int src_num_blocks,
                           int64_t block_bytes, const int32_t* pairs, int num_pairs, int32_t* dev_status,
                           void* stream) {
  if (num_pairs < 0 || dst_num_blocks <= 0 || src_num_blocks <= 0 || block_bytes <= 0 || block_bytes % 16 != 0 ||
      dst_block_stride < block_bytes || src_block_stride < block_bytes || dst_block_stride % 16 != 0 ||
      src_block_stride % 16 != 0)
    return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!dst_k || !dst_v || !src_k || !src_v || !pairs) return PKV_ERR_INVALID_ARG;
  if (!aligned(dst_k, 16) || !aligned(dst_v, 16) || !aligned(src_k, 16) || !aligned(src_v, 16) ||
      !aligned(pairs, 4))
    return PKV_ERR_INVALID_ARG;
  SwapBlocksArgs a{};
  a.dst_k = static_cast<uint8_t*>(const_cast<void*>(device_view(dst_k)));
  a.dst_v = static_cast<uint8_t*>(const_cast<void*>(device_view(dst_v)));
  a.src_k = static_cast<const uint8_t*>(device_view(src_k));
  a.src_v = static_cast<const uint8_t*>(device_view(src_v));
  a.pairs = static_cast<const int32_t*>(device_view(pairs));
  if (!a.dst_k || !a.dst_v || !a.src_k || !a.src_v || !a.pairs) return PKV_ERR_INVALID_ARG;  // pageable memory
  a.dev_status = dev_status;
  a.dst_stride = dst_block_stride;
  a.src_stride = src_block_stride;
  a.block_bytes = block_bytes;
  a.num_pairs = num_pairs;
  a.dst_num_blocks = dst_num_blocks;
  a.src_num_blocks = src_num_blocks;
  return cuda_status(launch_swap_blocks(a, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_check_bounded_wait(int64_t timeout_ns, int shared_ring, int32_t* dev_status, void* stream) {
  if (timeout_ns < 0 || timeout_ns > kWaitTimeoutNs || (shared_ring != 0 && shared_ring != 1) || !dev_status ||
      !aligned(dev_status, 4))
    return PKV_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(shared_ring ? launch_bounded_wait_vote_check(dev_status, timeout_ns, s)
                                 : launch_bounded_wait_check(dev_status, timeout_ns, s));
}

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_OUT_OF_BLOCKS: return "PKV_ERR_OUT_OF_BLOCKS";
  }
  return "PKV_ERR_UNKNOWN";
}

int pkv_version(void) { return 100; }

int pkv_last_cuda_error(void) { return t_last_cuda_error; }

const char* pkv_cuda_error_name(int code) {
  if (code >= 0) return cudaGetErrorName(static_cast<cudaError_t>(code));
  return "CUresult from cuTensorMapEncodeTiled (negated)";
}

}  // extern "C"
