// Paged decode attention for sm_103a, balanced split: one persistent CTA per
// SM, every warp streaming an equal share of the whole batch.
//
// Same computation as the fixed-partition kernel (single-query attention with
// an online softmax through block tables, "gpu_paged_kv_cache" section
// "Inside the paged attention kernel"), with the split-K partitions chosen
// by the library instead of a fixed token count:
//  * The work is the sequence of (block, KV head) tiles ordered by
//    (sequence s, KV head g, logical block t); with T tiles in total and W
//    warps, warp w takes tiles [floor(w T / W), floor((w+1) T / W)).  Every
//    warp thus streams the same number of tiles, the TMA ring runs on across
//    the (s, g) pairs a warp crosses, and the grid needs a single wave.
//  * A warp writes a pair it covers entirely as final output.  A pair split
//    between warps gets one unnormalised partial state per warp: a warp's
//    first segment goes to its slot 0, its last one to slot 1.  The warp
//    holding a pair's first tile records (that warp, number of pieces, its
//    slot) so the reduce kernel can merge the pieces.
//  * The per-sequence tile counts and their prefix sums live in shared
//    memory, built by each CTA from the context lengths at start.
#include "pkv_balanced.cuh"

namespace pkv {
namespace {

using namespace dev;

template <int D, bool BF16, int NW, int NST, bool FUSED>
__global__ void __launch_bounds__(NW * 32, 1) decode_balanced_kernel(
    const DecodeArgs a, const __grid_constant__ CUtensorMap tmap_k,
    const __grid_constant__ CUtensorMap tmap_v) {
  using Geom = TileGeom<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const size_t ring_bytes = static_cast<size_t>(NW) * NST * Geom::kStageBytes;
  const uint32_t bars = smem_u32(smem + ring_bytes);
  int* pre = reinterpret_cast<int*>(smem + ring_bytes + NW * NST * 8);  // [S + 1] tile prefix
  int* len = pre + a.num_seqs + 1;                                       // [S] clamped lengths
  int* warp_tot = len + a.num_seqs;                                      // [32] scan scratch

  griddep_wait();  // every input may come from the previous kernel on the stream
  griddep_launch_dependents();
  if (smem_misaligned(smem, a.dev_status)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.num_seqs, Hkv = a.num_kv_heads, G = a.group;

  for (int i = threadIdx.x; i < S; i += blockDim.x) {
    const int L = clamped_len(a, i, blockIdx.x == 0);
    len[i] = L;
    pre[i + 1] = (L + kBlockSize - 1) / kBlockSize;
  }
  if (threadIdx.x == 0) pre[0] = 0;
  __syncthreads();
  block_inclusive_scan(pre + 1, S, warp_tot);

  const int64_t T = static_cast<int64_t>(Hkv) * pre[S];
  const int64_t W = min(static_cast<int64_t>(gridDim.x) * NW, T);  // no warp gets an empty range
  const int64_t w = static_cast<int64_t>(blockIdx.x) * NW + warp;
  WarpRing<D, NST> ring{smem_u32(smem + static_cast<size_t>(warp) * NST * Geom::kStageBytes),
                        bars + 8 * NST * warp};
  ring.init(lane);
  if (w >= W) return;
  const int64_t x0 = w * T / W, x1 = (w + 1) * T / W;
  const int count = static_cast<int>(x1 - x0);

  // Locate tile x0: the last sequence s with Hkv * pre[s] <= x0 has tiles.
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(Hkv) * pre[mid] <= x0) lo = mid; else hi = mid - 1;
  }
  Cursor start;
  start.s = lo;
  start.n = pre[lo + 1] - pre[lo];
  {
    const int off = static_cast<int>(x0 - static_cast<int64_t>(Hkv) * pre[lo]);
    start.g = off / start.n;
    start.t = off % start.n;
  }

  // ---- issue side: a cursor plus two register chunks of table entries
  // (lane j holds the entry of the chunk's j-th tile).  A chunk is up to 32
  // consecutive tiles of one pair; the following chunk is prefetched.
  Cursor ic = start;
  struct Chunk {
    int s, g, base;
  };
  auto load_chunk = [&](const Chunk& c) -> int {
    if (c.s >= S) return 0;
    const int n = pre[c.s + 1] - pre[c.s];
    const int t = c.base + lane;
    return t < n ? __ldg(a.block_tables + static_cast<int64_t>(c.s) * a.max_blocks_per_seq + t) : 0;
  };
  auto chunk_after = [&](const Chunk& c) -> Chunk {
    if (c.s >= S) return c;  // past the last pair: nothing follows
    const int n = pre[c.s + 1] - pre[c.s];
    if (c.base + 32 < n) return Chunk{c.s, c.g, c.base + 32};
    Cursor q{c.s, c.g, 0, n};
    next_pair(q, pre, S, Hkv);
    return Chunk{q.s, q.g, 0};
  };
  Chunk cur{ic.s, ic.g, ic.t};
  Chunk nxt = chunk_after(cur);
  int phys_cur = load_chunk(cur);
  int phys_nxt = load_chunk(nxt);
  uint32_t bad_stage = 0;

  auto issue = [&](int j) {  // tile j of this warp's range, at cursor ic; all lanes call
    if (ic.s != cur.s || ic.g != cur.g || ic.t >= cur.base + 32) {
      cur = nxt;
      phys_cur = phys_nxt;
      nxt = chunk_after(cur);
      phys_nxt = load_chunk(nxt);
    }
    const int st = j % NST;
    int phys = __shfl_sync(kFull, phys_cur, ic.t - cur.base);
    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks)) {
      if (lane == 0) flag(a.dev_status, 4u);  // PKV_DEV_ERR_BLOCK
      phys = 0;
      bad_stage |= 1u << st;
    } else {
      bad_stage &= ~(1u << st);
    }
    ring.issue(j, phys, -1, 0, ic.g, &tmap_k, &tmap_v, lane);
    advance(ic, pre, S, Hkv);
  };

  for (int j = 0; j < min(count, NST); ++j) issue(j);

  // ---- compute side
  Cursor cc = start;
  WarpAttention<D, BF16> at;
  int seg_t0 = cc.t, seg_idx = 0;
  at.reset();
  at.load_q(a.q + (static_cast<int64_t>(cc.s) * a.num_q_heads + cc.g * G) * D, G, lane);
  NewToken<D> nt;
  // Fused decode step: the warp holding a pair's last tile (position L-1)
  // owns the new token of that (s, g).
  auto start_segment = [&](int i) {
    if constexpr (FUSED) {
      if (cc.t + (count - i) >= cc.n) nt.prefetch(a, cc.s, cc.g, len[cc.s], lane);
    }
  };
  start_segment(0);
  for (int i = 0; i < count; ++i) {
    if (i > 0 && cc.t == 0) {  // a new (s, g) pair starts here
      seg_t0 = 0;
      at.reset();
      at.load_q(a.q + (static_cast<int64_t>(cc.s) * a.num_q_heads + cc.g * G) * D, G, lane);
      start_segment(i);
    }
    if (!__all_sync(kFull, ring.wait(i, a.timeout_ns))) {
      ring.drain(i, min(count, i + NST), a.timeout_ns);
      if (lane == 0) flag(a.dev_status, 16u);  // PKV_DEV_ERR_TIMEOUT
      return;
    }
    const int st = i % NST;
    const int nv = ((bad_stage >> st) & 1) ? 0 : min(kBlockSize, len[cc.s] - cc.t * kBlockSize);
    const uint32_t sK = ring.k_tile(i);
    const bool patched = FUSED && cc.t == cc.n - 1 && nt.commit(a, cc.g, lane);
    if (patched) nt.patch(sK, sK + Geom::kTileBytes, lane);
    at.tile(sK, sK + Geom::kTileBytes, nv, a.scale_log2, lane);
    __syncwarp();
    if (i + NST < count) {
      if (patched) fence_proxy_async_smem();  // only the patched new token is a generic write to the stage
      issue(i + NST);
    }
    if (cc.t == cc.n - 1 || i == count - 1) {  // end of a segment
      at.finish_sums();
      const bool whole = seg_t0 == 0 && cc.t == cc.n - 1;
      const int64_t head0 = static_cast<int64_t>(cc.s) * a.num_q_heads + cc.g * G;
      const int slot = seg_idx == 0 ? 0 : 1;
      if (whole)
        at.store_final(a.out, head0, G, a.out_dtype, lane);
      else
        at.store_partial(a.ws_acc, a.ws_ml, (w * 2 + slot) * G, 1, G, lane);
      if (seg_t0 == 0 && lane == 0) {  // this warp holds the pair's first tile
        int pieces = 0;
        if (!whole) {
          const int64_t pair_end = static_cast<int64_t>(Hkv) * pre[cc.s] + static_cast<int64_t>(cc.g + 1) * cc.n;
          pieces = static_cast<int>((pair_end * W - 1) / T - w + 1);
        }
        a.ws_meta[static_cast<int64_t>(cc.s) * Hkv + cc.g] = make_int2(static_cast<int>(w), pieces * 2 + slot);
      }
      ++seg_idx;
    }
    advance(cc, pre, S, Hkv);
  }
}

// Reduce for the balanced split: one warp per (sequence, query head) row,
// CTAs of kRowsPerCta warps over one sequence's heads (grid S x
// ceil(H_q / kRowsPerCta)), register-capped so ~48 warps stay resident per
// SM.  Rows of pairs a single warp covered return at once; rows of empty
// sequences are written as zeros here (no warp visits them).  The pair
// metadata and the length are loaded together (the metadata slot is always
// readable; it is only trusted when the sequence is non-empty).
constexpr int kRowsPerCta = 8;

template <int D>
__global__ void __launch_bounds__(kRowsPerCta * 32, 6) decode_reduce_balanced_kernel(const DecodeArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x;
  const int h = blockIdx.y * kRowsPerCta + warp;
  if (h >= a.num_q_heads) return;
  const int G = a.group, g = h / G, hh = h % G;
  const int2 meta = a.ws_meta[static_cast<int64_t>(s) * a.num_kv_heads + g];
  const int L = clamped_len(a, s, false);
  const int64_t row = static_cast<int64_t>(s) * a.num_q_heads + h;
  RowMerge<D, 4> r;
  if (L > 0) {
    const int pieces = meta.y >> 1, first_slot = meta.y & 1, w0 = meta.x;
    if (pieces == 0) return;
    r.run(a.ws_ml, a.ws_acc + lane * RowMerge<D, 4>::EPL, 0, 1, pieces, [&](int k) {
      return (static_cast<int64_t>(w0 + k) * 2 + (k == 0 ? first_slot : 0)) * G + hh;
    });
  }
  r.store(a.out, row, a.out_dtype, lane);
}

// Shared memory of one balanced CTA: the warps' rings and barriers, then the
// per-sequence tile prefix and lengths and the scan scratch (no static
// shared memory, so the dynamic window starts 1024-byte aligned).
constexpr size_t kMaxSmemPerCta = 232448;  // sm_100-class opt-in limit (227 KB)

template <int D>
constexpr int balanced_stages() { return D == 128 ? 2 : 4; }

size_t balanced_smem_for(int head_dim, int nw, int num_seqs) {
  const int nst = head_dim == 128 ? balanced_stages<128>() : balanced_stages<64>();
  const size_t stage = 2 * static_cast<size_t>(kBlockSize) * head_dim * 2;
  return nw * nst * stage + nw * nst * 8 + (2 * static_cast<size_t>(num_seqs) + 1 + 32) * sizeof(int);
}

template <int D, bool BF16, int NW>
cudaError_t launch_balanced_nw(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t stream) {
  auto kern = a.k_new ? decode_balanced_kernel<D, BF16, NW, balanced_stages<D>(), true>
                      : decode_balanced_kernel<D, BF16, NW, balanced_stages<D>(), false>;
  const size_t smem = balanced_smem_for(D, NW, a.num_seqs);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(a.balanced_ctas), dim3(NW * 32), smem, stream, a, tk, tv);
}

template <int D, bool BF16>
cudaError_t launch_balanced_t(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                              cudaStream_t stream) {
  if (balanced_warps_per_cta(D, a.num_seqs) == 14) return launch_balanced_nw<D, BF16, 14>(a, tk, tv, stream);
  return launch_balanced_nw<D, BF16, 12>(a, tk, tv, stream);
}

}  // namespace

// 14 warps when their rings and the per-sequence arrays fit one CTA, else 12.
int balanced_warps_per_cta(int head_dim, int num_seqs) {
  return balanced_smem_for(head_dim, 14, num_seqs) <= kMaxSmemPerCta ? 14 : 12;
}

size_t balanced_smem_bytes(int head_dim, int num_seqs) {
  return balanced_smem_for(head_dim, balanced_warps_per_cta(head_dim, num_seqs), num_seqs);
}

cudaError_t launch_decode_balanced(const DecodeArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                   int head_dim, int kv_bf16, cudaStream_t stream) {
  if (a.balanced_ctas <= 0) return cudaSuccess;
  if (head_dim == 128)
    return kv_bf16 ? launch_balanced_t<128, true>(a, tmap_k, tmap_v, stream)
                   : launch_balanced_t<128, false>(a, tmap_k, tmap_v, stream);
  if (head_dim == 64)
    return kv_bf16 ? launch_balanced_t<64, true>(a, tmap_k, tmap_v, stream)
                   : launch_balanced_t<64, false>(a, tmap_k, tmap_v, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_reduce_balanced(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(a.num_seqs),
                  static_cast<unsigned>((a.num_q_heads + kRowsPerCta - 1) / kRowsPerCta));
  const dim3 block(32 * kRowsPerCta);
  if (head_dim == 128) return launch_pdl(decode_reduce_balanced_kernel<128>, grid, block, 0, stream, a);
  if (head_dim == 64) return launch_pdl(decode_reduce_balanced_kernel<64>, grid, block, 0, stream, a);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
