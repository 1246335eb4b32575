// Paged decode attention for sm_103a, SM-streaming partition kernel: one
// persistent CTA per SM pulls split-K units from a device-wide queue and
// streams their K/V tiles through one deep shared-memory ring.
//
// What is computed is the partition kernel's result ("gpu_paged_kv_cache",
// section "Inside the paged attention kernel"; "PagedAttention internals",
// section 02 "Block tables"): for each sequence s, KV head g and partition p
// of PS tokens, the online-softmax state of the query heads of g's group
// over the partition's tokens, gathered block by block through the block
// table.  A sequence of one partition gets its normalised output, longer
// ones leave unnormalised partial records for the reduce kernel (the same
// records, in the same layout, as decode_partitions_kernel writes).
//
// Why a second partition kernel: a grid of small CTAs gives every unit its
// own short per-warp ring.  Each unit then streams at a single warp's
// latency-bound rate, a unit's ring is empty while it starts, and once the
// grid has no more units to hand out the SMs idle one by one while the
// largest units finish.  Here the whole SM works on one unit at a time:
//  * Producer warp: takes the next unit from the device-wide queue (an
//    atomic counter in the workspace), reads its table entries 32 at a time
//    (the next unit's first entries are read before the current unit's
//    tiles are issued) and issues, for each 16-token tile, the TMA copies of
//    its K and V boxes (cp.async.bulk.tensor.4d, 128-byte swizzle) into the
//    next stage of a ring of kStages stages (24 x 8 KB at head_dim 128),
//    each stage with a "full" mbarrier (transaction bytes) and an "empty"
//    one (released by the warp that consumed it).
//  * 8 consumer warps: tile i of the current unit goes to warp i % 8, which
//    runs the tensor-core score / online-softmax / value step of the grid
//    kernel (WarpAttention) on it.  At the end of the unit the eight softmax
//    states are merged in shared memory in three rounds (8 -> 4 -> 2 -> 1)
//    and warp 0 stores the result.
//  * Queue order: longest first.  Every CTA builds the same order in shared
//    memory from the context lengths before it starts: first every full
//    partition (PS tokens), then each sequence's last, partial partition in
//    descending size (a stable counting sort on its tile count), empty
//    sequences last.  So the queue ends with the smallest units and the SMs
//    finish close together; a per-SM queue position is taken dynamically,
//    so SMs that stream faster simply take more units.
//  * Control words: the queue counter and a CTA-exit counter live in the
//    caller's workspace (zeroed once when the workspace is allocated); the
//    last CTA to finish sets both back to zero for the next call.
//  * Every wait is bounded by %globaltimer: a wait that runs out sets
//    PKV_DEV_ERR_TIMEOUT, makes the CTA stop taking work, and the CTA still
//    drains its outstanding copies, takes its last queue ticket and counts
//    itself out, so the control words return to zero.
#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

constexpr int kConsumers = 8;                    // consumer warps per CTA
constexpr int kStreamThreads = 32 * (kConsumers + 1);
constexpr int kUnitSlots = 4;                    // unit descriptors in flight
constexpr int kSortKeys = 129;                   // empty sequence, then 1..128 tiles (capped)

// mbarriers of the end-of-unit merge, each completing once per unit:
// round 1: warps 4-7 have saved their states (4 arrivals); round 2: warps
// 2-3 (2); round 3: warp 1 (1); slots free: warp 0 has read the last slot
// (1), so the next unit's round-1 writers may overwrite them.
constexpr int kMergeBars = 4;

struct UnitDesc {
  int s, g, part, nparts;
  int len;   // the sequence's context length
  int ntok;  // tokens of this partition
  int nt;    // 16-token tiles of this partition
  int k0;    // ring stream index of its first tile; -1: no more units
};

template <int D>
struct StreamLayout {
  using Geom = TileGeom<D>;
  static constexpr int kStages = (192 * 1024) / Geom::kStageBytes;
  static constexpr int kSave = SoftmaxState<D / 16>::kSaveBytes;
  static constexpr size_t kRing = 0;
  static constexpr size_t kMerge = kRing + static_cast<size_t>(kStages) * Geom::kStageBytes;
  static constexpr size_t kLens = kMerge + 4 * static_cast<size_t>(kSave);
  static constexpr size_t kFpre = kLens + 4 * kStreamMaxSeqs;
  static constexpr size_t kPerm = kFpre + 4 * (kStreamMaxSeqs + 4);
  static constexpr size_t kCounts = kPerm + 2 * kStreamMaxSeqs;
  static constexpr size_t kDesc = kCounts + 4 * ((kSortKeys + 3) / 4 * 4);
  static constexpr size_t kStageNv = kDesc + sizeof(UnitDesc) * kUnitSlots;
  static constexpr size_t kBars = (kStageNv + 4 * kStages + 7) / 8 * 8;
  static constexpr size_t kMisc = kBars + 8 * (2 * kStages + 2 * kUnitSlots + kMergeBars);
  static constexpr size_t kTotal = kMisc + 32;
  static_assert(kTotal <= 227 * 1024, "one CTA per SM");
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Shared-memory plan of the queue (see the top of the file).
struct Plan {
  const int* lens;   // clamped context length per sequence
  const int* fpre;   // fpre[s] = full partitions of sequences < s; fpre[S] = all
  const uint16_t* perm;  // sequences with a partial (or empty) last partition, longest first
  int full_units;    // fpre[S] * H_kv
  int total_units;   // (fpre[S] + partial sequences) * H_kv
};

// Sort key of sequence s's last partition: -1 when it has none (length a
// multiple of PS), 0 for an empty sequence, else 1 + its tile count (capped).
__device__ __forceinline__ int partial_key(int L, int PS) {
  if (L == 0) return 0;
  const int rem = L % PS;
  if (rem == 0) return -1;
  return 1 + min((rem + kTile - 1) / kTile, kSortKeys - 2);
}

// Builds the plan (one warp).  Lengths are already in shared memory.
__device__ void build_plan(int S, int PS, int* lens, int* fpre, uint16_t* perm, int* counts, int* totals,
                           int lane) {
  // full partitions: contiguous chunk per lane, then a warp scan
  const int per = (S + 31) / 32;
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int s = lane * per + i;
    if (s < S) local += lens[s] / PS;
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - local;
  for (int i = 0; i < per; ++i) {
    const int s = lane * per + i;
    if (s < S) {
      fpre[s] = run;
      run += lens[s] / PS;
    }
  }
  if (lane == 31) fpre[S] = incl;
  // stable counting sort of the partial partitions, longest first
  for (int k = lane; k < kSortKeys; k += 32) counts[k] = 0;
  __syncwarp();
  const unsigned lt = lanemask_lt();
  for (int c = 0; c < S; c += 32) {
    const int s = c + lane;
    const int key = s < S ? partial_key(lens[s], PS) : -1;
    const unsigned peers = __match_any_sync(kFull, key);
    if (key >= 0 && (peers & lt) == 0) counts[key] += __popc(peers);
    __syncwarp();
  }
  // exclusive scan over keys in descending order -> first position of each key
  if (lane == 0) {
    int acc = 0;
    for (int k = kSortKeys - 1; k >= 0; --k) {
      const int n = counts[k];
      counts[k] = acc;
      acc += n;
    }
    totals[0] = acc;
  }
  __syncwarp();
  for (int c = 0; c < S; c += 32) {
    const int s = c + lane;
    const int key = s < S ? partial_key(lens[s], PS) : -1;
    const unsigned peers = __match_any_sync(kFull, key);
    if (key >= 0) perm[counts[key] + __popc(peers & lt)] = static_cast<uint16_t>(s);
    __syncwarp();
    if (key >= 0 && (peers & lt) == 0) counts[key] += __popc(peers);
    __syncwarp();
  }
}

// Unit of queue position q.
__device__ __forceinline__ UnitDesc decode_unit(const Plan& p, int q, int S, int Hkv, int PS) {
  UnitDesc u;
  int s, part;
  if (q < p.full_units) {
    const int j = q / Hkv;
    u.g = q - j * Hkv;
    int lo = 0, hi = S - 1;  // last s with fpre[s] <= j
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.fpre[mid] <= j) lo = mid; else hi = mid - 1;
    }
    s = lo;
    part = j - p.fpre[s];
  } else {
    const int r = (q - p.full_units) / Hkv;
    u.g = (q - p.full_units) - r * Hkv;
    s = p.perm[r];
    part = p.lens[s] / PS;
  }
  const int L = p.lens[s];
  u.s = s;
  u.part = part;
  u.len = L;
  u.nparts = L > 0 ? (L + PS - 1) / PS : 1;
  u.ntok = max(0, min(PS, L - part * PS));
  u.nt = (u.ntok + kTile - 1) / kTile;
  u.k0 = 0;
  return u;
}

template <int D, bool BF16, bool FUSED>
__global__ void __launch_bounds__(kStreamThreads, 1) decode_stream_kernel(
    const DecodeArgs a, const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v) {
  using Lay = StreamLayout<D>;
  using Geom = TileGeom<D>;
  using Att = WarpAttention<D, BF16>;
  constexpr int NS = Lay::kStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  griddep_wait();  // every input may come from the previous kernel on the stream
  griddep_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* lens = reinterpret_cast<int*>(smem + Lay::kLens);
  int* fpre = reinterpret_cast<int*>(smem + Lay::kFpre);
  uint16_t* perm = reinterpret_cast<uint16_t*>(smem + Lay::kPerm);
  int* counts = reinterpret_cast<int*>(smem + Lay::kCounts);
  UnitDesc* desc = reinterpret_cast<UnitDesc*>(smem + Lay::kDesc);
  int* stage_nv = reinterpret_cast<int*>(smem + Lay::kStageNv);
  const uint32_t ring = smem_u32(smem + Lay::kRing);
  const uint32_t full_bar = smem_u32(smem + Lay::kBars);
  const uint32_t empty_bar = full_bar + 8 * NS;
  const uint32_t ufull_bar = empty_bar + 8 * NS;
  const uint32_t uempty_bar = ufull_bar + 8 * kUnitSlots;
  const uint32_t merge_bar = uempty_bar + 8 * kUnitSlots;  // round 1, 2, 3, slots free
  int* misc = reinterpret_cast<int*>(smem + Lay::kMisc);  // [0] partial sequences, [1] abort
  volatile int* abort_flag = misc + 1;

  // Warp-uniform views of the abort flag and of a bounded wait (every lane
  // runs its own timer, so lanes could disagree at the limit).
  auto aborted = [&]() { return __any_sync(kFull, *abort_flag != 0); };
  auto wait_all = [&](uint32_t bar, int parity) {
    return __all_sync(kFull, mbar_wait_bounded(bar, parity, a.timeout_ns));
  };
  const bool misaligned = (smem_u32(smem) & 1023u) != 0;  // uniform over the CTA
  const int S = a.num_seqs, Hkv = a.num_kv_heads, PS = a.partition_size;

  // ---- set-up: lengths, plan, barriers
  for (int s = threadIdx.x; s < S; s += blockDim.x) lens[s] = clamped_len(a, s, blockIdx.x == 0);
  if (threadIdx.x == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(full_bar + 8 * st, 1);
      mbar_init(empty_bar + 8 * st, 1);
    }
    for (int j = 0; j < kUnitSlots; ++j) {
      mbar_init(ufull_bar + 8 * j, 1);
      mbar_init(uempty_bar + 8 * j, kConsumers);
    }
    mbar_init(merge_bar, 4);
    mbar_init(merge_bar + 8, 2);
    mbar_init(merge_bar + 16, 1);
    mbar_init(merge_bar + 24, 1);
    misc[1] = misaligned ? 1 : 0;
    fence_barrier_init();
    if (misaligned) flag(a.dev_status, 32u);
  }
  __syncthreads();
  if (warp == 0) build_plan(S, PS, lens, fpre, perm, counts, misc, lane);
  __syncthreads();
  Plan plan{lens, fpre, perm, 0, 0};
  plan.full_units = fpre[S] * Hkv;
  plan.total_units = (fpre[S] + misc[0]) * Hkv;
  int* ctl = a.ctl;

  if (warp == kConsumers) {
    // ================================================================ producer
    const int shift = a.block_shift;
    int k = 0;  // tiles issued
    int u = 0;  // units published
    // Table entries of tile i of unit d (0 past its tiles or its table row).
    auto entry = [&](const UnitDesc& d, int i) {
      if (i >= d.nt) return 0;
      const int blk = ((d.part * (PS / kTile) + i) * kTile) >> shift;
      return blk < a.max_blocks_per_seq ? __ldg(a.block_tables + static_cast<int64_t>(d.s) * a.max_blocks_per_seq + blk)
                                        : 0;
    };
    // One unit ahead: the next unit's queue position and its first 32 table
    // entries are fetched while the current unit's tiles are issued.
    int ticket = 0;
    if (lane == 0) ticket = atomicAdd(ctl, 1);
    int q = __shfl_sync(kFull, ticket, 0);
    bool have_failing_ticket = q >= plan.total_units;
    UnitDesc cur{};
    int cur_ent = 0;
    if (!have_failing_ticket) {
      if (lane == 0) ticket = atomicAdd(ctl, 1);
      cur = decode_unit(plan, q, S, Hkv, PS);
      cur_ent = entry(cur, lane);
    }
    while (!have_failing_ticket && !aborted()) {
      // the unit after this one
      q = __shfl_sync(kFull, ticket, 0);
      const bool more = q < plan.total_units;
      UnitDesc nxt{};
      int nxt_ent = 0;
      if (more) {
        if (lane == 0) ticket = atomicAdd(ctl, 1);
        nxt = decode_unit(plan, q, S, Hkv, PS);
        nxt_ent = entry(nxt, lane);
      }
      // publish the current unit
      cur.k0 = k;
      const int slot = u % kUnitSlots;
      if (!wait_all(uempty_bar + 8 * slot, ((u / kUnitSlots) & 1) ^ 1)) {
        if (lane == 0) {
          flag(a.dev_status, 16u);
          *abort_flag = 1;
        }
        break;
      }
      if (lane == 0) {
        desc[slot] = cur;
        mbar_arrive(ufull_bar + 8 * slot);
      }
      ++u;
      // issue its tiles
      const int tile0 = cur.part * (PS / kTile);
      int ent_next = cur_ent;
      bool stop = false;
      for (int i0 = 0; i0 < cur.nt && !stop; i0 += 32) {
        const int ent = ent_next;
        if (i0 + 32 < cur.nt) ent_next = entry(cur, i0 + 32 + lane);
        const int n = min(32, cur.nt - i0);
        for (int j = 0; j < n; ++j) {
          int phys = __shfl_sync(kFull, ent, j);
          const int st = k % NS;
          if (!wait_all(empty_bar + 8 * st, ((k / NS) & 1) ^ 1) || aborted()) {
            if (lane == 0) {
              flag(a.dev_status, 16u);
              *abort_flag = 1;
            }
            stop = true;
            break;
          }
          if (lane == 0) {
            const int i = i0 + j;
            const bool bad = static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks);
            if (bad) {
              flag(a.dev_status, 4u);  // PKV_DEV_ERR_BLOCK: the tile is loaded from block 0 and masked
              phys = 0;
            }
            stage_nv[st] = bad ? 0 : min(kTile, cur.ntok - i * kTile);
            const int row0 = ((tile0 + i) * kTile) & ((1 << shift) - 1);
            const uint32_t b = full_bar + 8 * st;
            const uint32_t dst = ring + st * Geom::kStageBytes;
            mbar_arrive_expect_tx(b, Geom::kStageBytes);
#pragma unroll
            for (int h = 0; h < Geom::kHalves; ++h) {
              tma_load_4d(dst + h * 2048, &tmap_k, 0, cur.g * Geom::kHalves + h, row0, phys, b);
              tma_load_4d(dst + Geom::kTileBytes + h * 2048, &tmap_v, 0, cur.g * Geom::kHalves + h, row0, phys, b);
            }
          }
          __syncwarp();
          ++k;
        }
      }
      if (stop) break;
      if (!more) {
        have_failing_ticket = true;
        break;
      }
      cur = nxt;
      cur_ent = nxt_ent;
    }
    // No more units for this CTA: publish the end marker (unless stopping on
    // an error, where the consumers stop by themselves).
    if (!aborted()) {
      const int slot = u % kUnitSlots;
      if (wait_all(uempty_bar + 8 * slot, ((u / kUnitSlots) & 1) ^ 1)) {
        if (lane == 0) {
          desc[slot].k0 = -1;
          mbar_arrive(ufull_bar + 8 * slot);
        }
      } else if (lane == 0) {
        flag(a.dev_status, 16u);
        *abort_flag = 1;
      }
    }
    // Every issued copy must land before the CTA's shared memory is released:
    // wait (bounded) for the last phase issued on each stage.
    for (int st = lane; st < min(k, NS); st += 32) {
      const int last = st + ((k - 1 - st) / NS) * NS;
      mbar_wait_bounded(full_bar + 8 * st, (last / NS) & 1, a.timeout_ns);
    }
    if (lane == 0) {
      // Exactly one queue ticket past the end per CTA, then count the CTA out;
      // the last one returns the control words to zero for the next call.
      if (!have_failing_ticket) atomicAdd(ctl, plan.total_units + 1);
      __threadfence();
      if (atomicAdd(ctl + 1, 1) == static_cast<int>(gridDim.x) - 1) {
        atomicExch(ctl, 0);
        atomicExch(ctl + 1, 0);
      }
    }
    return;
  }

  // ================================================================== consumers
  const int G = a.group;
  const uint32_t merge = smem_u32(smem + Lay::kMerge);
  Att at;
  auto fail = [&]() {  // a wait ran out: report it once and make the CTA stop taking work
    if (lane == 0 && !*abort_flag) {
      flag(a.dev_status, 16u);
      *abort_flag = 1;
    }
  };
  for (int u = 0;; ++u) {
    const int slot = u % kUnitSlots;
    if (aborted() || !wait_all(ufull_bar + 8 * slot, (u / kUnitSlots) & 1)) {
      fail();
      break;
    }
    const UnitDesc d = desc[slot];
    if (d.k0 < 0) break;
    at.reset();
    at.load_q(a.q + (static_cast<int64_t>(d.s) * a.num_q_heads + d.g * G) * D, G, lane);
    NewToken<D> nt;
    const bool owns_new = FUSED && d.part == d.nparts - 1 && warp == (d.nt > 0 ? (d.nt - 1) % kConsumers : 0);
    if (owns_new) {
      nt.prefetch(a, d.s, d.g, d.len, lane);
      if (d.nt == 0) nt.commit(a, d.g, lane);  // empty sequence: only checks the slot
    }
    for (int i = warp; i < d.nt; i += kConsumers) {
      const int kk = d.k0 + i;
      const int st = kk % NS;
      if (aborted() || !wait_all(full_bar + 8 * st, (kk / NS) & 1)) {
        fail();
        break;
      }
      const uint32_t sK = ring + st * Geom::kStageBytes;
      const int nv = stage_nv[st];
      const bool patched = owns_new && i == d.nt - 1 && nt.commit(a, d.g, lane);
      if (patched) nt.patch(sK, sK + Geom::kTileBytes, lane);
      at.tile(sK, sK + Geom::kTileBytes, nv, a.scale_log2, lane);
      __syncwarp();
      if (lane == 0) {
        if (patched) fence_proxy_async_smem();  // generic writes before the next TMA into this stage
        mbar_arrive(empty_bar + 8 * st);
      }
    }
    at.finish_sums();
    // Merge the eight states, 8 -> 4 -> 2 -> 1, through four shared slots.
    const int pu = u & 1;
    auto wait = [&](uint32_t bar, int parity) {
      if (!wait_all(bar, parity)) fail();
    };
    auto publish = [&](int slot_index, uint32_t bar) {
      at.save(merge + slot_index * Lay::kSave, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    if (warp >= 4) {
      wait(merge_bar + 24, pu ^ 1);  // the previous unit's slots have been read
      publish(warp - 4, merge_bar);
    } else {
      wait(merge_bar, pu);
      at.merge_from(merge + warp * Lay::kSave, lane);
      if (warp >= 2) {
        publish(warp, merge_bar + 8);
      } else {
        wait(merge_bar + 8, pu);
        at.merge_from(merge + (warp + 2) * Lay::kSave, lane);
        if (warp == 1) {
          publish(1, merge_bar + 16);
        } else {
          wait(merge_bar + 16, pu);
          at.merge_from(merge + Lay::kSave, lane);
          __syncwarp();
          if (lane == 0) mbar_arrive(merge_bar + 24);
          const int64_t head0 = static_cast<int64_t>(d.s) * a.num_q_heads + d.g * G;
          if (!aborted()) {
            if (d.nparts == 1)
              at.store_final(a.out, head0, G, a.out_dtype, lane);
            else
              at.store_partial(a.ws_acc, a.ws_ml, head0 * a.max_parts + d.part, a.max_parts, G, lane);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(uempty_bar + 8 * slot);
  }
}

}  // namespace

size_t stream_smem_bytes(int head_dim) {
  return head_dim == 128 ? StreamLayout<128>::kTotal : StreamLayout<64>::kTotal;
}

cudaError_t launch_decode_stream(const DecodeArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                 int head_dim, int kv_bf16, cudaStream_t stream) {
  const int sms = current_sm_count(0);
  if (sms <= 0) return cudaErrorNoDevice;
  auto go = [&](auto kern, size_t smem) {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(static_cast<unsigned>(sms)), dim3(kStreamThreads), smem, stream, a, tmap_k, tmap_v);
  };
  const bool fused = a.k_new != nullptr;
  if (head_dim == 128) {
    constexpr size_t smem = StreamLayout<128>::kTotal;
    if (kv_bf16)
      return fused ? go(decode_stream_kernel<128, true, true>, smem) : go(decode_stream_kernel<128, true, false>, smem);
    return fused ? go(decode_stream_kernel<128, false, true>, smem) : go(decode_stream_kernel<128, false, false>, smem);
  }
  if (head_dim == 64) {
    constexpr size_t smem = StreamLayout<64>::kTotal;
    if (kv_bf16)
      return fused ? go(decode_stream_kernel<64, true, true>, smem) : go(decode_stream_kernel<64, true, false>, smem);
    return fused ? go(decode_stream_kernel<64, false, true>, smem) : go(decode_stream_kernel<64, false, false>, smem);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pkv
