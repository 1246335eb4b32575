// Device building blocks of the decode kernels (sm_103a): PTX wrappers, the
// per-warp TMA tile ring and the per-warp attention state.
//
// The arithmetic is single-query attention with an online softmax
// ("gpu_paged_kv_cache", section "Inside the paged attention kernel": score
// each block's keys against the query, keep a running softmax state, then
// accumulate the values).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pkv_internal.h"

namespace pkv {
namespace dev {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kNegInf = -__builtin_huge_valf();

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// True once the phase with `parity` has completed; false after timeout_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (static_cast<long long>(global_timer_ns() - t0) > timeout_ns) return false;
  }
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: wait until the previous grid on the stream
// has completed and its writes are visible; allow the next grid to launch.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier `id` (1..15) over `nthreads` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t x) {
  return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

// 2^x by the MUFU approximation (relative error ~2^-22), subnormal results flushed to 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void flag(int32_t* status, unsigned bit) {
  if (status) atomicOr(reinterpret_cast<unsigned*>(status), bit);
}

__device__ __forceinline__ void store_out(void* out, int64_t idx, float v, int dtype) {
  if (dtype == 0) {
    static_cast<float*>(out)[idx] = v;
  } else if (dtype == 1) {
    static_cast<__half*>(out)[idx] = __float2half_rn(v);
  } else {
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  }
}

// Context length of sequence s clamped to what the table and the host bound
// allow; out-of-range values set PKV_DEV_ERR_LENGTH when `report`.
__device__ __forceinline__ int clamped_len(const DecodeArgs& a, int s, bool report) {
  const int cap = min(a.max_context_len, a.max_blocks_per_seq << a.block_shift);
  const int L = a.context_lens[s];
  if (L >= 0 && L <= cap) return L;
  if (report) flag(a.dev_status, 8u);
  return L < 0 ? 0 : cap;
}

// The same for a length already read.
__device__ __forceinline__ int clamp_len(const DecodeArgs& a, int L, bool report) {
  const int cap = min(a.max_context_len, a.max_blocks_per_seq << a.block_shift);
  if (L >= 0 && L <= cap) return L;
  if (report) flag(a.dev_status, 8u);
  return L < 0 ? 0 : cap;
}

// The dynamic shared-memory window starts 1024-byte aligned (the TMA 128-byte
// swizzle pattern is a function of address bits 4-9).  Kernels check it and,
// should it ever not hold, flag PKV_DEV_ERR_SMEM and do nothing.
__device__ __forceinline__ bool smem_misaligned(const void* base, int32_t* status) {
  if ((smem_u32(base) & 1023u) == 0) return false;
  if (threadIdx.x == 0) flag(status, 32u);
  return true;
}

// ------------------------------------------------------------- tile geometry

// One pipeline stage holds a (block, KV head) tile of K and one of V: 16
// tokens x D elements of EB bytes each, stored as D*EB/128 sub-tiles of
// [16 rows][128 bytes] in the TMA 128-byte swizzle (16-byte chunk c of row r
// sits at c ^ (r & 7)).  Every sub-tile starts on a 1024-byte boundary.
template <int D, int EB = 2>
struct TileGeom {
  static_assert((D * EB) % 128 == 0, "a head row is whole 128-byte lines");
  static constexpr int kHalves = D * EB / 128;  // 128-byte lines per head row
  static constexpr int kTileBytes = kTile * D * EB;
  static constexpr int kStageBytes = 2 * kTileBytes;
};

// One (block, head) tile of K or V, rows [row0, row0 + 16) of block phys,
// head g, from a pool map of blocks >= 16 tokens (dimensions {element in
// line, row, line, block}): a single copy of the whole head row, landing as
// [line][16 rows][128 bytes] with 16-byte chunk c of row r at c ^ (r & 7).
template <int D, int EB = 2>
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap* map, int row0, int g, int phys,
                                         uint32_t bar) {
  tma_load_4d(dst, map, 0, row0, g * TileGeom<D, EB>::kHalves, phys, bar);
}

// A warp's private ring of NST stages, each completing on its own mbarrier.
template <int D, int NST, int EB = 2>
struct WarpRing {
  using Geom = TileGeom<D, EB>;
  uint32_t buf;  // shared address of stage 0
  uint32_t bar;  // shared address of the stage-0 mbarrier

  __device__ __forceinline__ void init(int lane) {
    if (lane == 0) {
      for (int st = 0; st < NST; ++st) mbar_init(bar + 8 * st, 1);
      fence_barrier_init();
      fence_proxy_async_smem();
    }
    __syncwarp();
  }

  // Lane 0 issues the K and V copies of tile number j (stage j % NST), KV
  // head g: rows [row0, row0 + 16) of block `phys` (blocks of >= 16 tokens;
  // one whole-head box per tensor, see tma_tile), or, when phys2 >= 0
  // (8-token blocks; tensor maps {element, line, row in block, block}, a box
  // is one line of 8 rows), block phys then block phys2, the second landing
  // 8 rows (1024 bytes) further, in the same swizzle phase as a 16-row box.
  __device__ __forceinline__ void issue(int j, int phys, int phys2, int row0, int g, const CUtensorMap* tk,
                                        const CUtensorMap* tv, int lane) const {
    if (lane != 0) return;
    const int st = j % NST;
    const uint32_t b = bar + 8 * st;
    const uint32_t dst = buf + st * Geom::kStageBytes;
    mbar_arrive_expect_tx(b, Geom::kStageBytes);
    if (phys2 < 0) {
      tma_tile<D, EB>(dst, tk, row0, g, phys, b);
      tma_tile<D, EB>(dst + Geom::kTileBytes, tv, row0, g, phys, b);
      return;
    }
#pragma unroll
    for (int h = 0; h < Geom::kHalves; ++h) {
      tma_load_4d(dst + h * 2048, tk, 0, g * Geom::kHalves + h, row0, phys, b);
      tma_load_4d(dst + Geom::kTileBytes + h * 2048, tv, 0, g * Geom::kHalves + h, row0, phys, b);
      tma_load_4d(dst + h * 2048 + 1024, tk, 0, g * Geom::kHalves + h, 0, phys2, b);
      tma_load_4d(dst + Geom::kTileBytes + h * 2048 + 1024, tv, 0, g * Geom::kHalves + h, 0, phys2, b);
    }
  }

  __device__ __forceinline__ bool wait(int i, long long timeout_ns) const {
    return mbar_wait_bounded(bar + 8 * (i % NST), (i / NST) & 1, timeout_ns);
  }

  // After a timed-out wait on tile i: wait (bounded) for tiles i..issued-1.
  __device__ __forceinline__ void drain(int i, int issued, long long timeout_ns) const {
    for (int j = i; j < issued; ++j) wait(j, timeout_ns);
  }

  __device__ __forceinline__ uint32_t k_tile(int i) const { return buf + (i % NST) * Geom::kStageBytes; }
};

// Table entry of tile T (16 tokens from 16T) of sequence s: the block
// holding its first token (second = 1: the block holding its token 8, for
// 8-token blocks).  0 for an index past the table row (such a tile's
// tokens are beyond the length; the entry is not used).
__device__ __forceinline__ int tile_entry(const DecodeArgs& a, int s, int T, int second) {
  const int blk = ((T * kTile) >> a.block_shift) + second;
  return blk < a.max_blocks_per_seq ? __ldg(a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + blk)
                                    : 0;
}

// The warp's first 32 table entries of unit `unit` (KV head, sequence,
// partition; partition-major) served by U warps (lane j: the partition's
// tile j * U + sub), read before the length is known: every read index lies
// in the table row; entries past the sequence's tiles are never used.
template <int U>
__device__ __forceinline__ int first_entries(const DecodeArgs& a, int64_t unit, int sub, int lane, int second = 0) {
  const int Hkv = a.num_kv_heads;
  const int s = static_cast<int>((unit / Hkv) % a.num_seqs);
  const int part = static_cast<int>(unit / Hkv / a.num_seqs);
  const int tiles = a.partition_size / kTile, e = lane * U + sub;
  return e < tiles ? tile_entry(a, s, part * tiles + e, second) : 0;
}

// ---------------------------------------------------- fused new-token write

// The token generated this step, for a warp that reads the tile holding its
// position L-1 (fused decode step).  Lanes [0, D/8) hold the 16-byte chunks
// of the K row of KV head g, lanes [16, 16 + D/8) those of the V row.  The
// warp stores the row to the pools (the write path, "gpu_paged_kv_cache"
// section "The write path: slot mapping and scatter") and patches it into
// its shared-memory tile, so the attention sees the new token without
// waiting for the pool write.  row = offset in its block, or -1 (nothing
// to do).
template <int D>
struct NewToken {
  uint4 val;
  int row = -1;     // row of position L-1 in its 16-token tile
  int offset = -1;  // offset of position L-1 in its block
  int slot = -1;
  int last_phys = -1;

  // Issues the loads (consumed only by commit(), so their latency hides
  // behind the tiles the warp streams meanwhile).
  __device__ __forceinline__ void prefetch(const DecodeArgs& a, int s, int g, int L, int lane) {
    slot = a.slot_mapping[s];
    last_phys = L > 0 ? __ldg(a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq +
                              ((L - 1) >> a.block_shift))
                      : -1;
    const int c = lane & 15;
    const uint16_t* src = (lane < 16 ? a.k_new : a.v_new) + static_cast<int64_t>(s) * a.new_stride + g * D + c * 8;
    val = (c < D / 8) ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
    row = L > 0 ? (L - 1) % kTile : -1;
    offset = L > 0 ? (L - 1) & ((1 << a.block_shift) - 1) : -1;
  }

  // Checks that the slot is position L-1 through the table; if so stores the
  // row to both pools, else flags PKV_DEV_ERR_SLOT (unless the slot is -1)
  // and drops the token.  Returns whether the tile must be patched.
  __device__ __forceinline__ bool commit(const DecodeArgs& a, int g, int lane) {
    if (row < 0 || slot == -1) {
      if (slot != -1 && lane == 0) flag(a.dev_status, 1u);  // a slot for an empty sequence
      row = -1;
      return false;
    }
    const bool ok = static_cast<unsigned>(last_phys) < static_cast<unsigned>(a.num_blocks) &&
                    slot == (last_phys << a.block_shift) + offset;
    if (!ok) {
      if (lane == 0) flag(a.dev_status, 1u);  // PKV_DEV_ERR_SLOT
      row = -1;
      return false;
    }
    const int c = lane & 15;
    if (c < D / 8) {
      uint16_t* dst = (lane < 16 ? a.k_pool_w : a.v_pool_w) + (slot >> a.block_shift) * a.block_stride +
                      static_cast<int64_t>(offset) * a.num_kv_heads * D + g * D + c * 8;
      *reinterpret_cast<uint4*>(dst) = val;
    }
    return true;
  }

  // Overwrites token `row` of the K and V tiles in shared memory (TMA
  // swizzled layout, shared addresses) with the new row.  Call after the
  // tile's wait.
  __device__ __forceinline__ void patch(uint32_t k_tile, uint32_t v_tile, int lane) const {
    const int c = lane & 15;
    if (c < D / 8) {
      const int half = c >> 3, cc = c & 7;
      const uint32_t addr = (lane < 16 ? k_tile : v_tile) + half * 2048 + row * 128 + ((cc ^ (row & 7)) << 4);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(val.x), "r"(val.y), "r"(val.z),
                   "r"(val.w)
                   : "memory");
    }
    __syncwarp();
  }
};

// ------------------------------------------------ per-warp softmax state

// Running softmax state of one warp serving up to 8 query heads, with the
// output accumulator in the C-fragment layout of an m16n8 MMA whose N index
// is the head: lane (gr = lane/4, tq = lane%4) owns heads 2tq and 2tq+1 (a,
// b); acc[mt][0..3] = rows (gr, head a), (gr, head b), (gr+8, head a),
// (gr+8, head b) of M-tile mt.  Scores are in log2 units.
template <int KT>
struct SoftmaxState {
  float acc[KT][4];
  float m_a, m_b, l_a, l_b;

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    m_a = m_b = kNegInf;
    l_a = l_b = 0.f;
  }

  // Online-softmax step over NT tiles of 16 tokens: this lane's scores of
  // tile t are s[4t] = (token gr, head a), s[4t+1] = (gr, b), s[4t+2] =
  // (gr+8, a), s[4t+3] = (gr+8, b), masked ones -inf.  Updates the running
  // max and sum and returns the weights p.  The accumulator is rescaled
  // only when some head's running max grows (the common case once a
  // sequence is under way skips it; a warp-uniform branch).  Exponentials
  // by ex2.approx.ftz (results below 2^-126 flush to 0).
  template <int NT>
  __device__ __forceinline__ void online_update_lazy(const float (&s)[4 * NT], float (&p)[4 * NT]) {
    float mx_a = fmaxf(s[0], s[2]), mx_b = fmaxf(s[1], s[3]);
#pragma unroll
    for (int t = 1; t < NT; ++t) {
      mx_a = fmaxf(mx_a, fmaxf(s[4 * t], s[4 * t + 2]));
      mx_b = fmaxf(mx_b, fmaxf(s[4 * t + 1], s[4 * t + 3]));
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(kFull, mx_a, o));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(kFull, mx_b, o));
    }
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    if (__any_sync(kFull, (mn_a > m_a) | (mn_b > m_b))) {
      const float al_a = ex2_approx(m_a - mn_a), al_b = ex2_approx(m_b - mn_b);  // m = -inf: 0
      l_a *= al_a;
      l_b *= al_b;
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        acc[mt][0] *= al_a;
        acc[mt][1] *= al_b;
        acc[mt][2] *= al_a;
        acc[mt][3] *= al_b;
      }
      m_a = mn_a;
      m_b = mn_b;
    }
    const float u_a = (m_a == kNegInf) ? 0.f : m_a;
    const float u_b = (m_b == kNegInf) ? 0.f : m_b;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      p[4 * t] = ex2_approx(s[4 * t] - u_a);
      p[4 * t + 2] = ex2_approx(s[4 * t + 2] - u_a);
      p[4 * t + 1] = ex2_approx(s[4 * t + 1] - u_b);
      p[4 * t + 3] = ex2_approx(s[4 * t + 3] - u_b);
      l_a += p[4 * t] + p[4 * t + 2];
      l_b += p[4 * t + 1] + p[4 * t + 3];
    }
  }

  __device__ __forceinline__ void scale_acc(float f) {
#pragma unroll
    for (int mt = 0; mt < KT; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[mt][j] *= f;
  }

  // Per-head sums over all lanes (lanes with the same lane%4 share heads).
  __device__ __forceinline__ void finish_sums() {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l_a += __shfl_xor_sync(kFull, l_a, o);
      l_b += __shfl_xor_sync(kFull, l_b, o);
    }
  }

  // Cross-warp merge of two states over disjoint token sets (the same
  // rescaling as the online softmax).  save() writes this lane's fragments
  // to shared memory at `buf` as [element][lane] floats (kSaveBytes in all);
  // merge_from() folds such a saved state into this one.  Both run after
  // finish_sums(), so every lane holds its heads' full running sums.
  static constexpr int kSaveFloats = KT * 4 + 4;
  static constexpr int kSaveBytes = kSaveFloats * 32 * 4;

  __device__ __forceinline__ void save(uint32_t buf, int lane) const {
    auto put = [&](int e, float v) {
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(buf + (e * 32 + lane) * 4), "f"(v) : "memory");
    };
#pragma unroll
    for (int mt = 0; mt < KT; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) put(mt * 4 + j, acc[mt][j]);
    put(KT * 4 + 0, m_a);
    put(KT * 4 + 1, m_b);
    put(KT * 4 + 2, l_a);
    put(KT * 4 + 3, l_b);
  }

  __device__ __forceinline__ void merge_from(uint32_t buf, int lane) {
    auto get = [&](int e) {
      float v;
      asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(buf + (e * 32 + lane) * 4) : "memory");
      return v;
    };
    const float mo_a = get(KT * 4 + 0), mo_b = get(KT * 4 + 1);
    const float lo_a = get(KT * 4 + 2), lo_b = get(KT * 4 + 3);
    const float M_a = fmaxf(m_a, mo_a), M_b = fmaxf(m_b, mo_b);
    // Two empty states stay empty (and no -inf - -inf is formed).
    const float u_a = (M_a == kNegInf) ? 0.f : M_a, u_b = (M_b == kNegInf) ? 0.f : M_b;
    const float ca = exp2f(m_a - u_a), coa = exp2f(mo_a - u_a);
    const float cb = exp2f(m_b - u_b), cob = exp2f(mo_b - u_b);
    l_a = l_a * ca + lo_a * coa;
    l_b = l_b * cb + lo_b * cob;
    m_a = M_a;
    m_b = M_b;
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      acc[mt][0] = acc[mt][0] * ca + get(mt * 4 + 0) * coa;
      acc[mt][1] = acc[mt][1] * cb + get(mt * 4 + 1) * cob;
      acc[mt][2] = acc[mt][2] * ca + get(mt * 4 + 2) * coa;
      acc[mt][3] = acc[mt][3] * cb + get(mt * 4 + 3) * cob;
    }
  }
};

// ----------------------------------------------------- per-warp attention

// Attention state of one warp serving the G <= 8 query heads of one KV head.
// Both contractions run on the tensor cores (mma.sync m16n8k16, fp32
// accumulation):
//   S^T[16 tok x 8 heads] = K[16 x D] Q^T[D x 8]     (tokens on M)
//   O^T[D x 8 heads]     += V^T[D x 16] P^T[16 x 8]  (head_dim on M)
// V^T comes from ldmatrix.trans; P^T is S^T's C fragment transposed in
// registers with movmatrix.  P is rounded to the KV type for the MMA; for
// bf16 it is split into hi + lo parts (two MMAs), keeping the rounding error
// near 2^-17 relative (fp16 alone is 2^-11).  Lane (gr = lane/4, tq = lane%4)
// owns heads 2tq and 2tq+1 (a, b) and the output rows d = 16mt + gr (+8).
template <int D, bool BF16>
struct WarpAttention : SoftmaxState<D / 16> {
  static constexpr int KT = D / 16;
  using Base = SoftmaxState<KT>;
  using Base::acc;
  using Base::l_a;
  using Base::l_b;
  using Base::m_a;
  using Base::m_b;
  uint32_t qf[KT][2];

  // B operand of QK^T: lane holds q[head lane/4][16kk + 2(lane%4) + {0,1}]
  // and +8.  `qhead0` points at the group's first head row; heads >= G are 0.
  __device__ __forceinline__ static void fetch_q(uint32_t (&dst)[KT][2], const uint16_t* qhead0, int G, int lane) {
    const int gr = lane >> 2, tq = lane & 3;
    const bool live = gr < G;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qhead0 + (live ? gr : 0) * D);
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      dst[kk][0] = live ? __ldg(qrow + kk * 8 + tq) : 0u;
      dst[kk][1] = live ? __ldg(qrow + kk * 8 + 4 + tq) : 0u;
    }
  }
  __device__ __forceinline__ void load_q(const uint16_t* qhead0, int G, int lane) { fetch_q(qf, qhead0, G, lane); }
  __device__ __forceinline__ void set_q(const uint32_t (&src)[KT][2]) {
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      qf[kk][0] = src[kk][0];
      qf[kk][1] = src[kk][1];
    }
  }

  // One tile: nv valid tokens (rows >= nv are masked, whatever they hold).
  __device__ __forceinline__ void tile(uint32_t sK, uint32_t sV, int nv, float sl2, int lane) {
    const int gr = lane >> 2, tq = lane & 3;
    const int rowK = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int colK = lane >> 4;
    const int rowV = (lane & 7) + (lane >> 4) * 8;
    const int colV = (lane >> 3) & 1;

    // Scores; even and odd k-steps accumulate in separate chains.
    float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      const int chunk = ((kk & 3) << 1) + colK;
      uint32_t ka[4];
      ldsm_x4(ka, sK + (kk >> 2) * 2048 + rowK * 128 + ((chunk ^ (rowK & 7)) << 4));
      if (kk & 1)
        mma_16816<BF16>(c2, ka, qf[kk][0], qf[kk][1]);
      else
        mma_16816<BF16>(c, ka, qf[kk][0], qf[kk][1]);
    }
    float s0 = (c[0] + c2[0]) * sl2, s1 = (c[1] + c2[1]) * sl2;
    float s2 = (c[2] + c2[2]) * sl2, s3 = (c[3] + c2[3]) * sl2;
    if (gr >= nv) s0 = s1 = kNegInf;
    if (gr + 8 >= nv) s2 = s3 = kNegInf;
    float sc[4] = {s0, s1, s2, s3}, pw[4];
    this->template online_update_lazy<1>(sc, pw);
    const float p0 = pw[0], p1 = pw[1], p2 = pw[2], p3 = pw[3];

    uint32_t pb0, pb1, pl0 = 0, pl1 = 0;
    if constexpr (BF16) {
      const uint32_t h0 = pack_bf16(p0, p1), h1 = pack_bf16(p2, p3);
      const float2 f0 = unpack_bf16(h0), f1 = unpack_bf16(h1);
      pb0 = movmatrix_trans(h0);
      pb1 = movmatrix_trans(h1);
      pl0 = movmatrix_trans(pack_bf16(p0 - f0.x, p1 - f0.y));
      pl1 = movmatrix_trans(pack_bf16(p2 - f1.x, p3 - f1.y));
    } else {
      pb0 = movmatrix_trans(pack_f16(p0, p1));
      pb1 = movmatrix_trans(pack_f16(p2, p3));
    }

    // V rows past the valid tokens may hold anything (even NaN): zero them in
    // the A fragment (lane holds tokens 2tq, 2tq+1 and 8+2tq, 9+2tq).
    uint32_t m01 = kFull, m23 = kFull;
    if (nv < kTile) {
      m01 = (2 * tq < nv ? 0x0000ffffu : 0u) | (2 * tq + 1 < nv ? 0xffff0000u : 0u);
      m23 = (2 * tq + 8 < nv ? 0x0000ffffu : 0u) | (2 * tq + 9 < nv ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int chunk = ((mt & 3) << 1) + colV;
      uint32_t va[4];
      ldsm_x4_trans(va, sV + (mt >> 2) * 2048 + rowV * 128 + ((chunk ^ (rowV & 7)) << 4));
      va[0] &= m01;
      va[1] &= m01;
      va[2] &= m23;
      va[3] &= m23;
      mma_16816<BF16>(acc[mt], va, pb0, pb1);
      if constexpr (BF16) mma_16816<BF16>(acc[mt], va, pl0, pl1);
    }
  }

  // Normalised output rows of heads [0, G) of the group; out_head0 = index of
  // the group's first row in [S * H_q].
  __device__ __forceinline__ void store_final(void* out, int64_t out_head0, int G, int dtype, int lane) const {
    const int gr = lane >> 2, tq = lane & 3;
    const int ha = 2 * tq, hb = ha + 1;
    const float ia = l_a > 0.f ? 1.f / l_a : 0.f;
    const float ib = l_b > 0.f ? 1.f / l_b : 0.f;
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int d = mt * 16 + gr;
      if (ha < G) {
        store_out(out, (out_head0 + ha) * D + d, acc[mt][0] * ia, dtype);
        store_out(out, (out_head0 + ha) * D + d + 8, acc[mt][2] * ia, dtype);
      }
      if (hb < G) {
        store_out(out, (out_head0 + hb) * D + d, acc[mt][1] * ib, dtype);
        store_out(out, (out_head0 + hb) * D + d + 8, acc[mt][3] * ib, dtype);
      }
    }
  }

  // Unnormalised partial state: head hh goes to record rec0 + hh * rec_stride
  // (acc[record][D], ml[record] = (running max, running sum)).
  __device__ __forceinline__ void store_partial(float* ws_acc, float2* ws_ml, int64_t rec0, int64_t rec_stride,
                                                int G, int lane) const {
    const int gr = lane >> 2, tq = lane & 3;
    const int ha = 2 * tq, hb = ha + 1;
    const int64_t ra = rec0 + ha * rec_stride, rb = rec0 + hb * rec_stride;
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int d = mt * 16 + gr;
      if (ha < G) {
        ws_acc[ra * D + d] = acc[mt][0];
        ws_acc[ra * D + d + 8] = acc[mt][2];
      }
      if (hb < G) {
        ws_acc[rb * D + d] = acc[mt][1];
        ws_acc[rb * D + d + 8] = acc[mt][3];
      }
    }
    if (gr == 0) {
      if (ha < G) ws_ml[ra] = make_float2(m_a, l_a);
      if (hb < G) ws_ml[rb] = make_float2(m_b, l_b);
    }
  }
};

// ------------------------------------------------------------ partial merge

// Merges partial states of one output row:
//     M' = max(M, m_p),  O' = O 2^(M-M') + acc_p 2^(m_p-M'),  l' likewise,
// lane j owning output elements [EPL*j, EPL*j + EPL).
template <int D, int U = 8>  // U: records whose loads are issued together
struct RowMerge {
  static constexpr int EPL = D / 32;
  static constexpr int U_batch() { return U; }
  float M = kNegInf, den = 0.f, o[EPL] = {};

  __device__ __forceinline__ void add(float m, float l, const float (&v)[EPL]) {
    const float Mn = fmaxf(M, m);
    if (Mn == kNegInf) return;  // nothing but empty partials so far
    const float c_old = exp2f(M - Mn), c_new = exp2f(m - Mn);
    den = den * c_old + l * c_new;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = o[e] * c_old + v[e] * c_new;
    M = Mn;
  }

  __device__ __forceinline__ static void load(const float* p, float (&v)[EPL]) {
    if constexpr (EPL == 4) {
      const float4 t = *reinterpret_cast<const float4*>(p);
      v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
      const float2 t = *reinterpret_cast<const float2*>(p);
      v[0] = t.x; v[1] = t.y;
    }
  }

  // Merges records rec(k) for k = first, first + step, ... < count, where
  // rec is a callable giving the record index.
  template <typename Rec>
  __device__ __forceinline__ void run(const float2* ml, const float* acc_lane, int first, int step, int count,
                                      Rec rec) {
    for (int k0 = first; k0 < count; k0 += U * step) {
      float2 mlv[U];
      float v[U][EPL];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = k0 + u * step;
        if (k < count) {
          const int64_t r = rec(k);
          mlv[u] = ml[r];
          load(acc_lane + r * D, v[u]);
        } else {
          mlv[u] = make_float2(kNegInf, 0.f);
#pragma unroll
          for (int e = 0; e < EPL; ++e) v[u][e] = 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) add(mlv[u].x, mlv[u].y, v[u]);
    }
  }

  __device__ __forceinline__ void store(void* out, int64_t row, int dtype, int lane) const {
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) store_out(out, row * D + lane * EPL + e, o[e] * inv, dtype);
  }
};

}  // namespace dev
}  // namespace pkv
