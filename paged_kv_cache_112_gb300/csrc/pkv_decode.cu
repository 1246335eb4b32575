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
//  * Work unit = (KV head g, sequence s, partition p), served by one warp
//    (a CTA's two warps take neighbouring KV heads of the same (s, p), so
//    they read neighbouring head rows of every token row) or by both warps
//    of a CTA (see partition_unit).  A warp serves all G <= 8 query heads
//    of its KV head: every K/V byte is read once.
//  * Data movement: TMA (cp.async.bulk.tensor.4d over {element line, head
//    line, row in block, block}, 128-byte swizzle) copies one 16-token tile
//    of K and of V per stage into a per-warp ring of NST stages completing
//    on mbarriers.  A tile is 16 rows of one block (blocks of >= 16 tokens)
//    or two 8-token blocks.  Six 2-warp CTAs per SM (12 warps at D = 128,
//    2 stages each) keep 24 tiles = 192 KB in flight per SM.
//  * Math: tensor-core mma.sync (see WarpAttention in pkv_device.cuh).
//  * Waits are bounded by %globaltimer; on timeout a warp drains its copies,
//    sets PKV_DEV_ERR_TIMEOUT and returns.  Table entries are range-checked;
//    a bad entry sets PKV_DEV_ERR_BLOCK and its tile is masked.
#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

// One unit (sequence s, KV head g, partition p) served by U of the CTA's NW
// warps; `raw_len` is the sequence's context length as read and `first`
// the warp's first table entries (first_entries<U>).
// B8: 8-token blocks (a tile spans two blocks: `first2` holds the second
// entries); otherwise blocks of 16 tokens or more (a tile is rows
// [row0, row0 + 16) of one block).
template <int D, bool BF16, int NW, int U, int NST, bool FUSED, bool B8>
__device__ __forceinline__ void partition_unit(const DecodeArgs& a, const CUtensorMap* tmap_k,
                                               const CUtensorMap* tmap_v, uint8_t* smem, int64_t unit,
                                               int raw_len, int first, int first2, int warp, int lane) {
  using Geom = TileGeom<D>;
  using Att = WarpAttention<D, BF16>;
  static_assert(NW % U == 0 && NW / U <= 15, "named barriers 1..15, one per unit of the CTA");
  static_assert(Att::kSaveBytes <= NST * Geom::kStageBytes, "a saved state must fit its warp's ring");
  const int sub = warp % U;  // the warp's place among its unit's U warps
  const int Hkv = a.num_kv_heads;
  // Units run in ascending partition index.  The grid covers every
  // partition index up to max_parts for every sequence, so most units of a
  // mixed-length batch are empty; in this order they come last, where they
  // only fill slots that finishing units free (dispatched first they stall
  // the start of the grid).
  const int g = static_cast<int>(unit % Hkv);
  const int64_t rest = unit / Hkv;
  const int s = static_cast<int>(rest % a.num_seqs);
  const int part = static_cast<int>(rest / a.num_seqs);

  const int PS = a.partition_size;
  const int G = a.group;
  const int L = clamp_len(a, raw_len, part == 0 && g == 0 && sub == 0 && lane == 0);
  const int nparts = L > 0 ? (L + PS - 1) / PS : 1;
  if (part >= nparts) return;  // the unit's warps all leave here
  Att at;
  at.load_q(a.q + (static_cast<int64_t>(s) * a.num_q_heads + g * G) * D, G, lane);
  const int tok0 = part * PS;
  const int ntok = max(0, min(L - tok0, PS));
  const int nblk = (ntok + kTile - 1) / kTile;  // 16-token tiles of the partition
  // The warp's tiles are the partition's tiles sub, sub + U, sub + 2U, ...
  // Their table entries sit in registers 32 at a time (lane j: the warp's
  // tile j of the chunk); the next chunk is fetched one chunk ahead of use.
  const int cnt = nblk > sub ? (nblk - sub + U - 1) / U : 0;
  const int tile0 = tok0 / kTile;
  auto entry = [&](int i, int second) { return i < cnt ? tile_entry(a, s, tile0 + i * U + sub, second) : 0; };
  int phys_cur = first;
  int phys_next = entry(32 + lane, 0);
  int phys2_cur = first2, phys2_next = B8 ? entry(32 + lane, 1) : 0;

  WarpRing<D, NST> ring{smem_u32(smem + static_cast<size_t>(warp) * NST * Geom::kStageBytes),
                        smem_u32(smem + static_cast<size_t>(NW) * NST * Geom::kStageBytes) + 8 * NST * warp};
  ring.init(lane);
  uint32_t bad_stage = 0;  // bit st: the tile in stage st came from an invalid entry

  auto issue = [&](int j) {  // all lanes call
    if ((j & 31) == 0 && j > 0) {
      phys_cur = phys_next;
      phys_next = entry(j + 32 + lane, 0);
      if constexpr (B8) {
        phys2_cur = phys2_next;
        phys2_next = entry(j + 32 + lane, 1);
      }
    }
    const int st = j % NST;
    const int t = j * U + sub;  // tile index within the partition
    int phys = __shfl_sync(kFull, phys_cur, j & 31);
    int phys2 = -1, row0 = 0;
    bool bad = static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks);
    if constexpr (B8) {
      // The tile's rows 8-15 come from the next block when the sequence
      // reaches them; otherwise the first block is loaded again (masked).
      phys2 = __shfl_sync(kFull, phys2_cur, j & 31);
      if (ntok - t * kTile > 8)
        bad |= static_cast<unsigned>(phys2) >= static_cast<unsigned>(a.num_blocks);
      else
        phys2 = phys;
    } else {
      row0 = ((tile0 + t) * kTile) & ((1 << a.block_shift) - 1);
    }
    if (bad) {
      if (lane == 0) flag(a.dev_status, 4u);  // PKV_DEV_ERR_BLOCK
      phys = 0;
      if constexpr (B8) phys2 = 0;
      bad_stage |= 1u << st;
    } else {
      bad_stage &= ~(1u << st);
    }
    ring.issue(j, phys, phys2, row0, g, tmap_k, tmap_v, lane);
  };

  at.reset();
  for (int j = 0; j < min(cnt, NST); ++j) issue(j);

  // Fused decode step: the last block of the last partition of (s, g) holds
  // position L-1.
  NewToken<D> nt;
  const bool owns_new = FUSED && part == nparts - 1 && sub == (nblk > 0 ? (nblk - 1) % U : 0);
  if (owns_new) {
    nt.prefetch(a, s, g, L, lane);
    if (nblk == 0) nt.commit(a, g, lane);  // empty sequence: only checks the slot
  }

  for (int i = 0; i < cnt; ++i) {
    if (!__all_sync(kFull, ring.wait(i, a.timeout_ns))) {
      ring.drain(i, min(cnt, i + NST), a.timeout_ns);
      if (lane == 0) flag(a.dev_status, 16u);  // PKV_DEV_ERR_TIMEOUT; the output is undefined
      break;
    }
    const int t = i * U + sub;  // tile index within the partition
    const int st = i % NST;
    const int nv = ((bad_stage >> st) & 1) ? 0 : min(kTile, ntok - t * kTile);
    const uint32_t sK = ring.k_tile(i);
    const bool patched = owns_new && t == nblk - 1 && nt.commit(a, g, lane);
    if (patched) nt.patch(sK, sK + Geom::kTileBytes, lane);
    at.tile(sK, sK + Geom::kTileBytes, nv, a.scale_log2, lane);
    __syncwarp();
    if (i + NST < cnt) {
      // The stage's reads are complete (their values are in registers); only
      // a generic-proxy write (the patched new token) must be ordered before
      // the next copy into it.
      if (patched) fence_proxy_async_smem();
      issue(i + NST);
    }
  }

  at.finish_sums();
  if constexpr (U > 1) {
    // The unit's warps hand their states to its first warp through their
    // own (now idle) ring buffers.
    const uint32_t mine = smem_u32(smem + static_cast<size_t>(warp) * NST * Geom::kStageBytes);
    if (sub != 0) at.save(mine, lane);
    named_barrier_sync(1 + warp / U, U * 32);
    if (sub != 0) return;
#pragma unroll
    for (int k = 1; k < U; ++k) at.merge_from(mine + k * NST * Geom::kStageBytes, lane);
  }
  const int64_t head0 = static_cast<int64_t>(s) * a.num_q_heads + g * G;
  if (nparts == 1)
    at.store_final(a.out, head0, G, a.out_dtype, lane);
  else
    at.store_partial(a.ws_acc, a.ws_ml, head0 * a.max_parts + part, a.max_parts, G, lane);
}

// Two-warp CTAs.  With one warp per unit (a.unit_warps == 1) CTA b serves
// units 2b and 2b + 1; with two (== 2) it serves unit b with both warps.
// A unit's length and first table entries go out together.
template <int D, bool BF16, int NST, bool FUSED, bool B8>
__global__ void __launch_bounds__(64) decode_partitions_kernel(
    const DecodeArgs a, const __grid_constant__ CUtensorMap tmap_k,
    const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ __align__(1024) uint8_t smem[];
  griddep_wait();  // every input may come from the previous kernel on the stream
  griddep_launch_dependents();
  if (smem_misaligned(smem, a.dev_status)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t units = static_cast<int64_t>(a.num_kv_heads) * a.num_seqs * a.max_parts;
  const int64_t unit1 = static_cast<int64_t>(blockIdx.x) * 2 + warp, unit2 = blockIdx.x;
  auto seq_of = [&](int64_t u) { return static_cast<int>((u / a.num_kv_heads) % a.num_seqs); };
  if (a.unit_warps == 2) {
    if (unit2 < units)
      partition_unit<D, BF16, 2, 2, NST, FUSED, B8>(a, &tmap_k, &tmap_v, smem, unit2, a.context_lens[seq_of(unit2)],
                                                    first_entries<2>(a, unit2, warp, lane),
                                                    B8 ? first_entries<2>(a, unit2, warp, lane, 1) : 0, warp, lane);
  } else if (unit1 < units) {
    partition_unit<D, BF16, 2, 1, NST, FUSED, B8>(a, &tmap_k, &tmap_v, smem, unit1, a.context_lens[seq_of(unit1)],
                                                  first_entries<1>(a, unit1, 0, lane),
                                                  B8 ? first_entries<1>(a, unit1, 0, lane, 1) : 0, warp, lane);
  }
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

// ------------------------------------------------------- bounded-wait check

// One warp sets up the partition kernel's tile ring (the same WarpRing, the
// same bounded wait and drain) but issues no copy, so the first wait can
// only end by running out of time.  It then takes the decode kernels' error
// path: drain (nothing is in flight), set PKV_DEV_ERR_TIMEOUT, return.
// Nothing in flight ever targets this CTA's shared memory.
__global__ void __launch_bounds__(32) bounded_wait_check_kernel(int32_t* status, long long timeout_ns) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using Geom = TileGeom<128>;
  constexpr int NST = 2;
  const int lane = threadIdx.x & 31;
  WarpRing<128, NST> ring{smem_u32(smem), smem_u32(smem + NST * Geom::kStageBytes)};
  ring.init(lane);
  const int issued = 0;
  if (!__all_sync(kFull, ring.wait(0, timeout_ns))) {
    ring.drain(0, issued, timeout_ns);
    if (lane == 0) flag(status, 16u);
  }
}

// ------------------------------------------------------------------ launchers

constexpr int kStages = 2;

template <int D, bool BF16, bool FUSED, bool B8>
cudaError_t launch_partitions_t(const DecodeArgs& a_in, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t stream) {
  using Geom = TileGeom<D>;
  constexpr int NST = kStages;
  const size_t smem = 2 * NST * Geom::kStageBytes + 2 * NST * 8;
  auto kern = decode_partitions_kernel<D, BF16, NST, FUSED, B8>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  DecodeArgs a = a_in;
  const int64_t units = static_cast<int64_t>(a.num_kv_heads) * a.num_seqs * a.max_parts;
  if (units == 0) return cudaSuccess;
  // Two warps per unit when the sequences alone (a unit each at least)
  // overfill the warp slots: there are surely more units than one wave.
  // Otherwise one, which keeps every unit of a single-wave batch running
  // from the start.  (The host does not see the lengths; estimating the
  // unit count on the device cost more than it gained on the benchmarked
  // batches.)
  const int slots = resident_warp_slots(reinterpret_cast<const void*>(kern), 64, smem);
  a.unit_warps = static_cast<int64_t>(a.num_kv_heads) * a.num_seqs > slots ? 2 : 1;
  const int64_t ctas = a.unit_warps == 1 ? (units + 1) / 2 : units;
  return launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(64), smem, stream, a, tk, tv);
}

template <int D, bool BF16>
cudaError_t launch_partitions_f(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t stream) {
  if (a.block_shift == 3)
    return a.k_new ? launch_partitions_t<D, BF16, true, true>(a, tk, tv, stream)
                   : launch_partitions_t<D, BF16, false, true>(a, tk, tv, stream);
  return a.k_new ? launch_partitions_t<D, BF16, true, false>(a, tk, tv, stream)
                 : launch_partitions_t<D, BF16, false, false>(a, tk, tv, stream);
}

// Warp slots of the partition kernel (the one-warp-per-unit rule's wave).
template <int D, bool BF16>
int partition_slots() {
  using Geom = TileGeom<D>;
  const size_t smem = 2 * kStages * Geom::kStageBytes + 2 * kStages * 8;
  return resident_warp_slots(reinterpret_cast<const void*>(decode_partitions_kernel<D, BF16, kStages, false, false>),
                             64, smem);
}

}  // namespace

int partitions_heads_per_box(const DecodeArgs& a, int head_dim, int kv_bf16) {
  if (a.block_shift < 4 || a.num_kv_heads % 2 != 0 || (head_dim != 128 && head_dim != 64)) return 1;
  const int slots = head_dim == 128 ? (kv_bf16 ? partition_slots<128, true>() : partition_slots<128, false>())
                                    : (kv_bf16 ? partition_slots<64, true>() : partition_slots<64, false>());
  const int64_t seq_heads = static_cast<int64_t>(a.num_kv_heads) * a.num_seqs;
  if (seq_heads > slots) return 1;
  // Four heads per copy (1 KB of each block row instead of 512 B) pay on
  // grids of many waves, whose warps stream long runs of tiles from HBM;
  // on a grid of about one wave the CTA-wide lockstep of four warps costs
  // more than the copies it saves.
  return (a.num_kv_heads % 4 == 0 && seq_heads * a.max_parts > 4LL * slots) ? 4 : 2;
}

cudaError_t launch_decode_partitions(const DecodeArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                     int head_dim, int kv_bf16, cudaStream_t stream) {
  if (a.heads_per_box > 1) return launch_decode_partitions_hg(a, tmap_k, tmap_v, head_dim, kv_bf16, stream);
  if (head_dim == 128)
    return kv_bf16 ? launch_partitions_f<128, true>(a, tmap_k, tmap_v, stream)
                   : launch_partitions_f<128, false>(a, tmap_k, tmap_v, stream);
  if (head_dim == 64)
    return kv_bf16 ? launch_partitions_f<64, true>(a, tmap_k, tmap_v, stream)
                   : launch_partitions_f<64, false>(a, tmap_k, tmap_v, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bounded_wait_check(int32_t* status, long long timeout_ns, cudaStream_t stream) {
  constexpr size_t smem = 2 * TileGeom<128>::kStageBytes + 2 * 8;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(bounded_wait_check_kernel), smem);
  if (e != cudaSuccess) return e;
  bounded_wait_check_kernel<<<1, 32, smem, stream>>>(status, timeout_ns);
  return cudaGetLastError();
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
