// Paged decode attention for sm_103a, fixed-size partitions: partition kernel
// + reduce kernel.
//
// What is computed ("gpu_paged_kv_cache", section "Inside the paged attention
// kernel"; "PagedAttention internals", section 02 "Block tables"): for each
// sequence s and KV head g, walk the sequence's logical blocks, read each
// physical block id from the block table, load that block's 16 keys, score
// them against every query head of g's group, keep a running (online)
// softmax, and accumulate the values.  Sequences longer than one partition
// are split; the partial softmax states are merged by a separate reduce
// kernel (the split-K restructuring of flash-decoding).
//
// Mapping onto GB300:
//  * Work unit = (KV head g, sequence s, partition p), one warp each.  A CTA
//    is NW warps on consecutive KV heads of the same (s, p), so it reads
//    neighbouring head rows of every token row of a block.  Partitions are
//    dispatched from the last index down.  A warp serves
//    all G <= 8 query heads of its KV head: every K/V byte is read once.
//  * Data movement: TMA (cp.async.bulk.tensor.3d, 128-byte swizzle) copies
//    one (block, head) tile of K and of V per stage into a per-warp ring of
//    NST stages completing on mbarriers.  Six 2-warp CTAs per SM (12 warps
//    at D = 128, 2 stages each) keep 24 tiles = 192 KB in flight per SM.
//    CTA widths that divide H_kv keep a CTA's warps on units of one (s, p):
//    wider CTAs mixing unit sizes hold shared memory for their slowest warp.
//  * Math: tensor-core mma.sync (see WarpAttention in pkv_device.cuh).
//  * Waits are bounded by %globaltimer; on timeout a warp drains its copies,
//    sets PKV_DEV_ERR_TIMEOUT and returns.  Table entries are range-checked;
//    a bad entry sets PKV_DEV_ERR_BLOCK and its tile is masked.
#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

template <int D, bool BF16, int NW, int NST, bool FUSED>
__global__ void __launch_bounds__(NW * 32) decode_partitions_kernel(
    const DecodeArgs a, const __grid_constant__ CUtensorMap tmap_k,
    const __grid_constant__ CUtensorMap tmap_v) {
  using Geom = TileGeom<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  griddep_wait();  // every input may come from the previous kernel on the stream
  griddep_launch_dependents();
  if (smem_misaligned(smem, a.dev_status)) return;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Hkv = a.num_kv_heads;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * NW + warp;
  if (unit >= static_cast<int64_t>(Hkv) * a.num_seqs * a.max_parts) return;
  // Units run in descending partition index: the later partitions of long
  // sequences (all full-size) are dispatched first and each sequence's first
  // partition -- the short tail of most sequences -- last, which shortens
  // the end of the grid.
  const int g = static_cast<int>(unit % Hkv);
  const int64_t rest = unit / Hkv;
  const int s = static_cast<int>(rest % a.num_seqs);
  const int part = a.max_parts - 1 - static_cast<int>(rest / a.num_seqs);

  const int PS = a.partition_size;
  const int G = a.group;
  const int tok0 = part * PS;
  // Block-table entries of this partition, 32 per register chunk, and the
  // query rows do not depend on the sequence length: their loads go out
  // together with the length's (entries within the table row are always
  // readable; those past the sequence are never used).
  const int blk0 = tok0 / kBlockSize;
  const int32_t* tbl = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + blk0;
  const int row_left = a.max_blocks_per_seq - blk0;
  int phys_cur = (lane < row_left) ? __ldg(tbl + lane) : 0;
  int phys_next = (32 + lane < row_left) ? __ldg(tbl + 32 + lane) : 0;
  WarpAttention<D, BF16> at;
  at.load_q(a.q + (static_cast<int64_t>(s) * a.num_q_heads + g * G) * D, G, lane);

  const int L = clamped_len(a, s, part == 0 && g == 0 && lane == 0);
  const int nparts = L > 0 ? (L + PS - 1) / PS : 1;
  if (part >= nparts) return;
  const int ntok = max(0, min(L - tok0, PS));
  const int nblk = (ntok + kBlockSize - 1) / kBlockSize;

  WarpRing<D, NST> ring{smem_u32(smem + static_cast<size_t>(warp) * NST * Geom::kStageBytes),
                        smem_u32(smem + static_cast<size_t>(NW) * NST * Geom::kStageBytes) + 8 * NST * warp};
  ring.init(lane);
  uint32_t bad_stage = 0;  // bit st: the tile in stage st came from an invalid entry

  auto issue = [&](int j) {  // all lanes call
    if ((j & 31) == 0 && j > 0) {
      phys_cur = phys_next;
      const int nx = j + 32 + lane;
      phys_next = (nx < min(nblk, row_left)) ? __ldg(tbl + nx) : 0;
    }
    const int st = j % NST;
    int phys = __shfl_sync(kFull, phys_cur, j & 31);
    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks)) {
      if (lane == 0) flag(a.dev_status, 4u);  // PKV_DEV_ERR_BLOCK
      phys = 0;
      bad_stage |= 1u << st;
    } else {
      bad_stage &= ~(1u << st);
    }
    ring.issue(j, phys, g, &tmap_k, &tmap_v, lane);
  };

  at.reset();
  for (int j = 0; j < min(nblk, NST); ++j) issue(j);

  // Fused decode step: the last partition of (s, g) holds position L-1.
  NewToken<D> nt;
  const bool owns_new = FUSED && part == nparts - 1;
  if (owns_new) {
    nt.prefetch(a, s, g, L, lane);
    if (nblk == 0) nt.commit(a, g, lane);  // empty sequence: only checks the slot
  }

  for (int i = 0; i < nblk; ++i) {
    if (!__all_sync(kFull, ring.wait(i, a.timeout_ns))) {
      ring.drain(i, min(nblk, i + NST), a.timeout_ns);
      if (lane == 0) flag(a.dev_status, 16u);  // PKV_DEV_ERR_TIMEOUT
      return;
    }
    const int st = i % NST;
    const int nv = ((bad_stage >> st) & 1) ? 0 : min(kBlockSize, ntok - i * kBlockSize);
    const uint32_t sK = ring.k_tile(i);
    if (owns_new && i == nblk - 1 && nt.commit(a, g, lane)) nt.patch(sK, sK + Geom::kTileBytes, lane);
    at.tile(sK, sK + Geom::kTileBytes, nv, a.scale_log2, lane);
    __syncwarp();
    if (i + NST < nblk) {
      fence_proxy_async_smem();
      issue(i + NST);
    }
  }

  at.finish_sums();
  const int64_t head0 = static_cast<int64_t>(s) * a.num_q_heads + g * G;
  if (nparts == 1)
    at.store_final(a.out, head0, G, a.out_dtype, lane);
  else
    at.store_partial(a.ws_acc, a.ws_ml, head0 * a.max_parts + part, a.max_parts, G, lane);
}

// --------------------------------------------------------------- reduce kernels

__device__ __forceinline__ int parts_of(const DecodeArgs& a, int s) {
  const int L = clamped_len(a, s, false);
  return L > 0 ? (L + a.partition_size - 1) / a.partition_size : 1;
}


// Few partitions per row: one warp per (sequence, query head) row, CTAs of
// kRowsPerCta warps over consecutive heads of one sequence (grid S x
// ceil(H_q / kRowsPerCta)).  A sequence that fits one partition costs one
// length load: the partition kernel already wrote its output.  Small CTAs
// with a register cap keep ~48 warps resident per SM, so rows of different
// sequences merge concurrently.
constexpr int kRowsPerCta = 8;

template <int D>
__global__ void __launch_bounds__(kRowsPerCta * 32, 6) decode_reduce_rows_kernel(const DecodeArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x;
  const int h = blockIdx.y * kRowsPerCta + warp;
  if (h >= a.num_q_heads) return;
  const int nparts = parts_of(a, s);
  if (nparts <= 1) return;
  const int64_t row = static_cast<int64_t>(s) * a.num_q_heads + h;
  RowMerge<D, 4> r;
  const int64_t rec0 = row * a.max_parts;
  r.run(a.ws_ml, a.ws_acc + lane * RowMerge<D, 4>::EPL, 0, 1, nparts, [&](int k) { return rec0 + k; });
  r.store(a.out, row, a.out_dtype, lane);
}

// Many partitions per row (long contexts): one CTA of 16 warps per row (two
// CTAs per SM); warp w merges partitions w, w + 16, ... in batches of 8 and
// the warps' states are merged through shared memory.
constexpr int kLongReduceWarps = 16;

template <int D>
__global__ void __launch_bounds__(kLongReduceWarps * 32, 2) decode_reduce_long_kernel(const DecodeArgs a) {
  __shared__ float sm_m[kLongReduceWarps], sm_l[kLongReduceWarps];
  __shared__ float sm_o[kLongReduceWarps][D];
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  const int nparts = parts_of(a, static_cast<int>(row / a.num_q_heads));
  if (nparts <= 1) return;
  RowMerge<D> r;
  const int64_t rec0 = row * a.max_parts;
  r.run(a.ws_ml, a.ws_acc + lane * RowMerge<D>::EPL, warp, kLongReduceWarps, nparts, [&](int k) { return rec0 + k; });
  if (lane == 0) {
    sm_m[warp] = r.M;
    sm_l[warp] = r.den;
  }
#pragma unroll
  for (int e = 0; e < RowMerge<D>::EPL; ++e) sm_o[warp][lane * RowMerge<D>::EPL + e] = r.o[e];
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kLongReduceWarps; ++w) M = fmaxf(M, sm_m[w]);
    const float mu = (M == kNegInf) ? 0.f : M;
    float o = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kLongReduceWarps; ++w) {
      const float c = exp2f(sm_m[w] - mu);
      o += sm_o[w][d] * c;
      den += sm_l[w] * c;
    }
    store_out(a.out, row * D + d, den > 0.f ? o / den : 0.f, a.out_dtype);
  }
}

// ------------------------------------------------------------------ launchers

#ifndef PKV_WARPS_PER_CTA
#define PKV_WARPS_PER_CTA 2
#endif
#ifndef PKV_STAGES
#define PKV_STAGES 2
#endif
constexpr int kWarpsPerCta = PKV_WARPS_PER_CTA;
constexpr int kStages = PKV_STAGES;

template <int D, bool BF16, bool FUSED>
cudaError_t launch_partitions_t(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t stream) {
  using Geom = TileGeom<D>;
  constexpr int NW = kWarpsPerCta, NST = kStages;
  const size_t smem = static_cast<size_t>(NW) * NST * Geom::kStageBytes + NW * NST * 8;
  auto kern = decode_partitions_kernel<D, BF16, NW, NST, FUSED>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int64_t units = static_cast<int64_t>(a.num_kv_heads) * a.num_seqs * a.max_parts;
  const int64_t ctas = (units + NW - 1) / NW;
  if (ctas == 0) return cudaSuccess;
  return launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(NW * 32), smem, stream, a, tk, tv);
}

template <int D, bool BF16>
cudaError_t launch_partitions_f(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t stream) {
  return a.k_new ? launch_partitions_t<D, BF16, true>(a, tk, tv, stream)
                 : launch_partitions_t<D, BF16, false>(a, tk, tv, stream);
}

}  // namespace

cudaError_t launch_decode_partitions(const DecodeArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                     int head_dim, int kv_bf16, cudaStream_t stream) {
  if (head_dim == 128)
    return kv_bf16 ? launch_partitions_f<128, true>(a, tmap_k, tmap_v, stream)
                   : launch_partitions_f<128, false>(a, tmap_k, tmap_v, stream);
  if (head_dim == 64)
    return kv_bf16 ? launch_partitions_f<64, true>(a, tmap_k, tmap_v, stream)
                   : launch_partitions_f<64, false>(a, tmap_k, tmap_v, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_reduce(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  if (a.max_parts <= 1 || a.num_seqs == 0) return cudaSuccess;
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  if (a.max_parts > 2 * RowMerge<128>::U_batch()) {  // long rows: a CTA per row
    const dim3 grid(static_cast<unsigned>(rows)), block(kLongReduceWarps * 32);
    if (head_dim == 128) return launch_pdl(decode_reduce_long_kernel<128>, grid, block, 0, stream, a);
    if (head_dim == 64) return launch_pdl(decode_reduce_long_kernel<64>, grid, block, 0, stream, a);
    return cudaErrorInvalidValue;
  }
  const dim3 grid(static_cast<unsigned>(a.num_seqs), static_cast<unsigned>((a.num_q_heads + kRowsPerCta - 1) / kRowsPerCta));
  const dim3 block(32 * kRowsPerCta);
  if (head_dim == 128) return launch_pdl(decode_reduce_rows_kernel<128>, grid, block, 0, stream, a);
  if (head_dim == 64) return launch_pdl(decode_reduce_rows_kernel<64>, grid, block, 0, stream, a);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
