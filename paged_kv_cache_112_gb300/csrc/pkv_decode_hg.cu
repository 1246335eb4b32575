// Paged decode attention over 16-bit pools for sm_103a: the head-group
// partition kernel.
//
// What is computed: pkv_decode_partitions (and the fused decode step) over
// fixed partitions, exactly as the partition kernel in pkv_decode.cu with one
// warp per unit ("gpu_paged_kv_cache", "Inside the paged attention kernel";
// "PagedAttention internals", section 02 "Block tables").
//
// Mapping onto GB300: a CTA serves one (sequence s, partition p) for HP (2 or
// 4) adjacent KV heads, one warp per head.  A block's rows hold the heads' K
// (and V) rows side by side, so one TMA box of (128 bytes, 16 rows, HP
// heads' lines, 1 block) brings all HP heads' K tiles of a block, and another
// box their V tiles: HP x 4 KB per copy at head_dim 128 instead of 4 KB.
// Where tiles come from L2 (a prefix many sequences share) an SM's copy issue
// rate, not HBM, paces the per-head kernel; here it issues 1/HP as many.
//  * The HP warps share one ring of two stages ([K: heads 0..HP-1][V: heads
//    0..HP-1]), filled by lane 0 of warp 0; shared memory per warp, and so
//    warps per SM, stay the per-head kernel's.  Each warp waits on a stage's
//    barrier, reads its own head's tiles and keeps its own softmax state;
//    after each tile __syncthreads_or() both frees the stage for the next
//    copy and makes a timed-out wait the whole CTA's decision.
//  * Fused step: the warp whose head's tile holds position L-1 writes the new
//    rows to the pool and patches them into its own part of the stage, then
//    fences them against the next copy before the CTA barrier.
//  * Tile order, tile math and outputs are the one-warp-per-unit partition
//    kernel's, so results are bit-identical to it.
// Used for blocks of 16 tokens or more, a KV head count divisible by HP (4
// where it divides, else 2), and a batch whose sequences x KV heads fit one
// wave of the partition kernel's warp slots (where that kernel gives every
// unit one warp).
#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

constexpr int kPairStages = 2;

template <int D, bool BF16, bool FUSED, int HP>
__global__ void __launch_bounds__(HP * 32, 12 / HP) decode_partitions_hg_kernel(
    const DecodeArgs a, const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v) {
  using Geom = TileGeom<D>;
  using Att = WarpAttention<D, BF16>;
  constexpr int NST = kPairStages;
  constexpr uint32_t kHeadTile = Geom::kTileBytes;  // one head's 16 rows
  constexpr uint32_t kKBytes = HP * kHeadTile;       // the group's K tiles of one block
  constexpr uint32_t kStage = 2 * kKBytes;           // then its V tiles
  extern __shared__ __align__(1024) uint8_t smem[];
  griddep_wait();  // every input may come from the previous kernel on the stream
  griddep_launch_dependents();
  if (smem_misaligned(smem, a.dev_status)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = a.num_kv_heads / HP;
  const int64_t unit = blockIdx.x;  // partition-major: ((p * S) + s) * groups + gi
  const int gi = static_cast<int>(unit % groups);
  const int64_t rest = unit / groups;
  const int s = static_cast<int>(rest % a.num_seqs);
  const int part = static_cast<int>(rest / a.num_seqs);
  const int g = gi * HP + warp;
  const int PS = a.partition_size, G = a.group;
  const int tiles_per_part = PS / kTile;
  const int first = lane < tiles_per_part ? tile_entry(a, s, part * tiles_per_part + lane, 0) : 0;
  const int L = clamp_len(a, a.context_lens[s], part == 0 && gi == 0 && warp == 0 && lane == 0);
  const int nparts = L > 0 ? (L + PS - 1) / PS : 1;
  if (part >= nparts) return;  // the same for every warp of the CTA
  const int tok0 = part * PS;
  const int ntok = max(0, min(L - tok0, PS));
  const int cnt = (ntok + kTile - 1) / kTile;
  const int tile0 = tok0 / kTile;
  auto entry = [&](int i) { return i < cnt ? tile_entry(a, s, tile0 + i, 0) : 0; };

  const uint32_t ring = smem_u32(smem);
  const uint32_t bars = ring + NST * kStage;
  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) mbar_init(bars + 8 * st, 1);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncthreads();

  int phys_cur = first;
  int phys_next = entry(32 + lane);
  uint32_t bad_stage = 0;
  auto issue = [&](int j) {  // every warp calls (entry bookkeeping); lane 0 of warp 0 copies
    if ((j & 31) == 0 && j > 0) {
      phys_cur = phys_next;
      phys_next = entry(j + 32 + lane);
    }
    const int st = j % NST;
    int phys = __shfl_sync(kFull, phys_cur, j & 31);
    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks)) {
      if (warp == 0 && lane == 0) flag(a.dev_status, 4u);  // PKV_DEV_ERR_BLOCK
      phys = 0;
      bad_stage |= 1u << st;
    } else {
      bad_stage &= ~(1u << st);
    }
    if (warp == 0 && lane == 0) {
      const int row0 = ((tile0 + j) * kTile) & ((1 << a.block_shift) - 1);
      const uint32_t bar = bars + 8 * st;
      const uint32_t dst = ring + st * kStage;
      mbar_arrive_expect_tx(bar, kStage);
      tma_load_4d(dst, &tmap_k, 0, row0, gi * HP * Geom::kHalves, phys, bar);
      tma_load_4d(dst + kKBytes, &tmap_v, 0, row0, gi * HP * Geom::kHalves, phys, bar);
    }
  };
  auto wait = [&](int j) { return mbar_wait_bounded(bars + 8 * (j % NST), (j / NST) & 1, a.timeout_ns); };

  Att at;
  at.load_q(a.q + (static_cast<int64_t>(s) * a.num_q_heads + g * G) * D, G, lane);
  at.reset();
  for (int j = 0; j < min(cnt, NST); ++j) issue(j);

  // Fused decode step: the last tile of the last partition of (s, g) holds position L-1.
  NewToken<D> nt;
  const bool owns_new = FUSED && part == nparts - 1;
  if (owns_new) {
    nt.prefetch(a, s, g, L, lane);
    if (cnt == 0) nt.commit(a, g, lane);  // empty sequence: only checks the slot
  }

  for (int i = 0; i < cnt; ++i) {
    const bool ok = __all_sync(kFull, wait(i));
    bool patched = false;
    if (ok) {
      const int st = i % NST;
      const int nv = ((bad_stage >> st) & 1) ? 0 : min(kTile, ntok - i * kTile);
      const uint32_t sK = ring + st * kStage + warp * kHeadTile;
      const uint32_t sV = sK + kKBytes;
      patched = owns_new && i == cnt - 1 && nt.commit(a, g, lane);
      if (patched) nt.patch(sK, sV, lane);
      at.tile(sK, sV, nv, a.scale_log2, lane);
    }
    // Only the patched new token is a generic-proxy write to a stage; it is
    // ordered before the next copy into the stage by this fence and the barrier.
    if (patched) fence_proxy_async_smem();
    // Every warp is done with this tile's stage; a timed-out wait in any ends the CTA.
    if (__syncthreads_or(!ok)) {
      if (warp == 0)
        for (int j = i; j < min(cnt, i + NST); ++j) wait(j);  // copies in flight land before the CTA exits
      if (warp == 0 && lane == 0) flag(a.dev_status, 16u);  // PKV_DEV_ERR_TIMEOUT; the output is undefined
      return;
    }
    if (i + NST < cnt) issue(i + NST);
  }

  at.finish_sums();
  const int64_t head0 = static_cast<int64_t>(s) * a.num_q_heads + g * G;
  if (nparts == 1)
    at.store_final(a.out, head0, G, a.out_dtype, lane);
  else
    at.store_partial(a.ws_acc, a.ws_ml, head0 * a.max_parts + part, a.max_parts, G, lane);
}

template <int D, bool BF16, bool FUSED, int HP>
cudaError_t launch_hg_t(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  using Geom = TileGeom<D>;
  const size_t smem = static_cast<size_t>(kPairStages) * (2 * HP * Geom::kTileBytes + 8);
  auto kern = decode_partitions_hg_kernel<D, BF16, FUSED, HP>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int64_t ctas = static_cast<int64_t>(a.num_kv_heads / HP) * a.num_seqs * a.max_parts;
  if (ctas == 0) return cudaSuccess;
  return launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(HP * 32), smem, stream, a, tk, tv);
}

template <int D, bool BF16, int HP>
cudaError_t launch_hg_fused(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  return a.k_new ? launch_hg_t<D, BF16, true, HP>(a, tk, tv, stream)
                 : launch_hg_t<D, BF16, false, HP>(a, tk, tv, stream);
}

template <int HP>
cudaError_t launch_hg_hp(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int head_dim,
                         int kv_bf16, cudaStream_t stream) {
  if (head_dim == 128)
    return kv_bf16 ? launch_hg_fused<128, true, HP>(a, tk, tv, stream)
                   : launch_hg_fused<128, false, HP>(a, tk, tv, stream);
  if (head_dim == 64)
    return kv_bf16 ? launch_hg_fused<64, true, HP>(a, tk, tv, stream)
                   : launch_hg_fused<64, false, HP>(a, tk, tv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode_partitions_hg(const DecodeArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                        int head_dim, int kv_bf16, cudaStream_t stream) {
  const int hp = a.heads_per_box;
  if ((hp != 2 && hp != 4) || a.num_kv_heads % hp != 0 || a.block_shift < 4) return cudaErrorInvalidValue;
  return hp == 4 ? launch_hg_hp<4>(a, tmap_k, tmap_v, head_dim, kv_bf16, stream)
                 : launch_hg_hp<2>(a, tmap_k, tmap_v, head_dim, kv_bf16, stream);
}

}  // namespace pkv
