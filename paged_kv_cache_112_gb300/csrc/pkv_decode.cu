// Paged decode attention for sm_103a: partition kernel + reduce kernel.
//
// What is computed ("gpu_paged_kv_cache", section "Inside the paged attention
// kernel"; "PagedAttention internals", section 02 "Block tables"): for each
// sequence s and KV head g, walk the logical blocks of the sequence, read each
// physical block id from the block table, load that block's 16 keys, score
// them against every query head of g's group, keep a running (online)
// softmax, and accumulate the values.  Long sequences are split into
// partitions whose partial softmax states are merged by a separate reduce
// kernel (split-K, "flash-decoding").
//
// How it maps onto GB300:
//  * Work unit = (KV head g, sequence s, partition p), one WARP each.  A CTA is
//    NW warps; consecutive warps take consecutive KV heads of the same
//    (s, p), so a CTA reads NW neighbouring 256-byte head rows of every
//    token row of a block.  A warp serves all G <= 8 query heads of its KV
//    head, so every K/V byte is read from HBM once per call.
//  * Data movement: TMA (cp.async.bulk.tensor.3d) copies one (block, head)
//    tile -- 16 tokens x head_dim -- of K and of V per pipeline stage into
//    shared memory, 128-byte swizzled, completing on an mbarrier.  Each warp
//    runs its own NST-deep ring, so NW*NST tiles per CTA are in flight.
//  * Math: both contractions are tensor-core mma.sync.m16n8k16 with fp32
//    accumulation.  QK^T puts the 16 tokens of a block on M and the (padded)
//    query heads of the group on N:  S^T[16 x 8] = K[16 x D] Q^T[D x 8].
//    PV puts head_dim on M:  O^T[D x 8] += V^T[D x 16] P^T[16 x 8]; V^T
//    comes from ldmatrix.trans and P^T is S^T's register fragment
//    transposed in registers with movmatrix.  P is rounded to the KV type
//    for the MMA; for bf16 P is split into hi + lo bf16 parts (two MMAs) so
//    the rounding error stays ~2^-17 relative, as the fp16 path is ~2^-11.
//  * Softmax: scores are taken in log2 units (scale * log2 e folded in) and
//    exponentiated with exp2f; running max per head is warp-reduced with
//    three shuffles per block, running sums stay per-lane until the end.
//  * Waits on mbarriers are bounded by %globaltimer; on timeout the warp
//    drains its own copies (again bounded), sets PKV_DEV_ERR_TIMEOUT and
//    returns.  Table entries are range-checked; a bad entry sets
//    PKV_DEV_ERR_BLOCK and its tile is masked (its copy reads block 0).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pkv_internal.h"

namespace pkv {
namespace {

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
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
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

// Bounded wait: true when the phase with `parity` completed, false after
// timeout_ns of polling.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (static_cast<long long>(global_timer_ns() - t0) > timeout_ns) return false;
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
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

// ------------------------------------------------------------ partition kernel

// Shared memory per warp: NST stages of [K tile | V tile].  A tile is
// 16 tokens x D elements stored as D/64 sub-tiles of [16 rows][128 bytes]
// with the TMA 128-byte swizzle (16-byte chunk c of row r sits at chunk
// c ^ (r & 7)); every sub-tile starts on a 1024-byte boundary.
template <int D>
struct TileGeom {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kBlockSize * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;
};

template <int D, bool BF16, int NW, int NST>
__global__ void __launch_bounds__(NW * 32) decode_partitions_kernel(
    const DecodeArgs a, const __grid_constant__ CUtensorMap tmap_k,
    const __grid_constant__ CUtensorMap tmap_v) {
  using Geom = TileGeom<D>;
  constexpr int KT = D / 16;  // k-steps of QK^T and m-tiles of PV
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));

  // Every input may come from the kernel just before this one on the stream.
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Hkv = a.num_kv_heads;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * NW + warp;
  const int64_t total_units = static_cast<int64_t>(Hkv) * a.num_seqs * a.max_parts;
  if (unit >= total_units) return;
  const int g = static_cast<int>(unit % Hkv);
  const int64_t rest = unit / Hkv;
  const int s = static_cast<int>(rest % a.num_seqs);
  const int part = static_cast<int>(rest / a.num_seqs);

  const int len_cap = min(a.max_context_len, a.max_blocks_per_seq * kBlockSize);
  int L = a.context_lens[s];
  if (L < 0 || L > len_cap) {
    if (part == 0 && g == 0 && lane == 0) flag(a.dev_status, 8u);  // PKV_DEV_ERR_LENGTH
    L = L < 0 ? 0 : len_cap;
  }
  const int PS = a.partition_size;
  const int nparts = L > 0 ? (L + PS - 1) / PS : 1;
  if (part >= nparts) return;
  const int tok0 = part * PS;
  const int ntok = max(0, min(L - tok0, PS));
  const int nblk = (ntok + kBlockSize - 1) / kBlockSize;
  const int blk0 = tok0 / kBlockSize;
  const int G = a.group;

  uint8_t* wsm = smem + static_cast<size_t>(warp) * NST * Geom::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(NW) * NST * Geom::kStageBytes) + warp * NST;
  const uint32_t wsm_u32 = smem_u32(wsm);
  const uint32_t bar_u32 = smem_u32(bars);

  if (lane == 0) {
    for (int st = 0; st < NST; ++st) mbar_init(bar_u32 + 8 * st, 1);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncwarp();

  // Block-table entries of this partition, 32 per register chunk; the next
  // chunk is fetched one chunk ahead of use.
  const int32_t* tbl = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + blk0;
  int phys_cur = (lane < nblk) ? __ldg(tbl + lane) : 0;
  int phys_next = (32 + lane < nblk) ? __ldg(tbl + 32 + lane) : 0;
  uint32_t bad_stage = 0;  // bit st: the tile in stage st came from an invalid entry

  auto issue = [&](int j) {  // all lanes call; lane 0 issues the copies of tile j
    if ((j & 31) == 0 && j > 0) {
      phys_cur = phys_next;
      const int nx = j + 32 + lane;
      phys_next = (nx < nblk) ? __ldg(tbl + nx) : 0;
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
    if (lane == 0) {
      const uint32_t bar = bar_u32 + 8 * st;
      const uint32_t dst = wsm_u32 + st * Geom::kStageBytes;
      mbar_arrive_expect_tx(bar, Geom::kStageBytes);
#pragma unroll
      for (int h = 0; h < Geom::kHalves; ++h) {
        tma_load_3d(dst + h * 2048, &tmap_k, 0, g * Geom::kHalves + h, phys * kBlockSize, bar);
        tma_load_3d(dst + Geom::kTileBytes + h * 2048, &tmap_v, 0, g * Geom::kHalves + h,
                    phys * kBlockSize, bar);
      }
    }
  };

  // Query fragments (B operand of QK^T): lane holds q[head = lane/4][d] for
  // d = 16kk + 2(lane%4) + {0,1} and +8.  Heads >= G are zero padding.
  const int gr = lane >> 2;
  const int tq = lane & 3;
  uint32_t qf[KT][2];
  {
    const bool live = gr < G;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        a.q + (static_cast<int64_t>(s) * a.num_q_heads + g * G + (live ? gr : 0)) * D);
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      qf[kk][0] = live ? __ldg(qrow + kk * 8 + tq) : 0u;
      qf[kk][1] = live ? __ldg(qrow + kk * 8 + 4 + tq) : 0u;
    }
  }

  // Prologue: fill the ring.
  const int prefill = nblk < NST ? nblk : NST;
  for (int j = 0; j < prefill; ++j) issue(j);

  float acc[KT][4];
#pragma unroll
  for (int mt = 0; mt < KT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  float m_a = kNegInf, m_b = kNegInf;  // running max (log2 units) of heads 2tq, 2tq+1
  float l_a = 0.f, l_b = 0.f;          // per-lane partial running sums

  // ldmatrix lane offsets inside a tile (see TileGeom for the swizzle).
  const int rowK = (lane & 7) + ((lane >> 3) & 1) * 8;  // token row for K (A of QK^T)
  const int colK = lane >> 4;                           // +8 columns
  const int rowV = (lane & 7) + (lane >> 4) * 8;        // token row for V (A of PV, transposed)
  const int colV = (lane >> 3) & 1;
  const float sl2 = a.scale_log2;
  bool timed_out = false;

  for (int i = 0; i < nblk; ++i) {
    const int st = i % NST;
    const uint32_t bar = bar_u32 + 8 * st;
    const bool ok = mbar_wait_bounded(bar, (i / NST) & 1, a.timeout_ns);
    if (!__all_sync(kFull, ok)) {
      // Drain the copies still in flight (tiles i+1 .. issued-1), then leave.
      const int issued = min(nblk, i + NST);
      for (int j = i; j < issued; ++j) mbar_wait_bounded(bar_u32 + 8 * (j % NST), (j / NST) & 1, a.timeout_ns);
      if (lane == 0) flag(a.dev_status, 16u);  // PKV_DEV_ERR_TIMEOUT
      timed_out = true;
      break;
    }
    const uint32_t sK = wsm_u32 + st * Geom::kStageBytes;
    const uint32_t sV = sK + Geom::kTileBytes;
    const int nv = ((bad_stage >> st) & 1) ? 0 : min(kBlockSize, ntok - i * kBlockSize);

    // S^T = K Q^T : lane holds tokens gr, gr+8 for heads 2tq, 2tq+1.
    // Two independent accumulation chains (even / odd k-steps) halve the
    // dependent MMA latency of the score computation.
    float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      const int chunk = ((kk & 3) << 1) + colK;
      const uint32_t addr = sK + (kk >> 2) * 2048 + rowK * 128 + ((chunk ^ (rowK & 7)) << 4);
      uint32_t ka[4];
      ldsm_x4(ka, addr);
      if (kk & 1)
        mma_16816<BF16>(c2, ka, qf[kk][0], qf[kk][1]);
      else
        mma_16816<BF16>(c, ka, qf[kk][0], qf[kk][1]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) c[e] += c2[e];
    float s0 = c[0] * sl2, s1 = c[1] * sl2, s2 = c[2] * sl2, s3 = c[3] * sl2;
    if (gr >= nv) s0 = s1 = kNegInf;
    if (gr + 8 >= nv) s2 = s3 = kNegInf;
    float mx_a = fmaxf(s0, s2), mx_b = fmaxf(s1, s3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(kFull, mx_a, o));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(kFull, mx_b, o));
    }
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float u_a = (mn_a == kNegInf) ? 0.f : mn_a;
    const float u_b = (mn_b == kNegInf) ? 0.f : mn_b;
    const float al_a = exp2f(m_a - u_a), al_b = exp2f(m_b - u_b);
    m_a = mn_a;
    m_b = mn_b;
    const float p0 = exp2f(s0 - u_a), p2 = exp2f(s2 - u_a);
    const float p1 = exp2f(s1 - u_b), p3 = exp2f(s3 - u_b);
    l_a = l_a * al_a + (p0 + p2);
    l_b = l_b * al_b + (p1 + p3);
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      acc[mt][0] *= al_a;
      acc[mt][1] *= al_b;
      acc[mt][2] *= al_a;
      acc[mt][3] *= al_b;
    }

    // P^T as the B operand of PV: transpose the two 8x8 C-fragments.
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

    // Rows of V past the sequence end may hold anything (even NaN): zero them
    // in the A fragment (lane holds tokens 2tq, 2tq+1 and 8+2tq, 9+2tq).
    uint32_t m01 = kFull, m23 = kFull;
    if (nv < kBlockSize) {
      m01 = (2 * tq < nv ? 0x0000ffffu : 0u) | (2 * tq + 1 < nv ? 0xffff0000u : 0u);
      m23 = (2 * tq + 8 < nv ? 0x0000ffffu : 0u) | (2 * tq + 9 < nv ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int chunk = ((mt & 3) << 1) + colV;
      const uint32_t addr = sV + (mt >> 2) * 2048 + rowV * 128 + ((chunk ^ (rowV & 7)) << 4);
      uint32_t va[4];
      ldsm_x4_trans(va, addr);
      va[0] &= m01;
      va[1] &= m01;
      va[2] &= m23;
      va[3] &= m23;
      mma_16816<BF16>(acc[mt], va, pb0, pb1);
      if constexpr (BF16) mma_16816<BF16>(acc[mt], va, pl0, pl1);
    }

    __syncwarp();
    if (i + NST < nblk) {
      fence_proxy_async_smem();
      issue(i + NST);
    }
  }
  if (timed_out) return;

  // Full per-head sums (lanes with the same tq hold the same heads).
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l_a += __shfl_xor_sync(kFull, l_a, o);
    l_b += __shfl_xor_sync(kFull, l_b, o);
  }
  const int ha = 2 * tq, hb = 2 * tq + 1;
  const int64_t head0 = static_cast<int64_t>(s) * a.num_q_heads + g * G;
  if (nparts == 1) {
    const float ia = l_a > 0.f ? 1.f / l_a : 0.f;
    const float ib = l_b > 0.f ? 1.f / l_b : 0.f;
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int d = mt * 16 + gr;
      if (ha < G) {
        store_out(a.out, (head0 + ha) * D + d, acc[mt][0] * ia, a.out_dtype);
        store_out(a.out, (head0 + ha) * D + d + 8, acc[mt][2] * ia, a.out_dtype);
      }
      if (hb < G) {
        store_out(a.out, (head0 + hb) * D + d, acc[mt][1] * ib, a.out_dtype);
        store_out(a.out, (head0 + hb) * D + d + 8, acc[mt][3] * ib, a.out_dtype);
      }
    }
  } else {
    const int64_t row_a = (head0 + ha) * a.max_parts + part;
    const int64_t row_b = (head0 + hb) * a.max_parts + part;
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int d = mt * 16 + gr;
      if (ha < G) {
        a.ws_acc[row_a * D + d] = acc[mt][0];
        a.ws_acc[row_a * D + d + 8] = acc[mt][2];
      }
      if (hb < G) {
        a.ws_acc[row_b * D + d] = acc[mt][1];
        a.ws_acc[row_b * D + d + 8] = acc[mt][3];
      }
    }
    if (gr == 0) {
      if (ha < G) a.ws_ml[row_a] = make_float2(m_a, l_a);
      if (hb < G) a.ws_ml[row_b] = make_float2(m_b, l_b);
    }
  }
}

// --------------------------------------------------------------- reduce kernel

// Merging the partition states of one (sequence, query head) row:
//     M' = max(M, m_p),  O' = O 2^(M-M') + acc_p 2^(m_p-M'),  l' likewise,
// lane j of a warp owning output elements [EPL*j, EPL*j + EPL).  Partitions
// are loaded in batches of U whose loads are issued together.
template <int D>
struct RowMerge {
  static constexpr int EPL = D / 32;
  static constexpr int U = 8;
  float M = -__builtin_huge_valf(), den = 0.f, o[EPL] = {};

  // Merges partitions first, first + step, ... below nparts.
  __device__ __forceinline__ void run(const float2* ml, const float* accp, int first, int step, int nparts) {
    for (int p0 = first; p0 < nparts; p0 += U * step) {
      float2 mlv[U];
      float v[U][EPL];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int p = p0 + u * step;
        if (p < nparts) {
          mlv[u] = ml[p];
          if constexpr (EPL == 4) {
            const float4 t = *reinterpret_cast<const float4*>(accp + static_cast<int64_t>(p) * D);
            v[u][0] = t.x; v[u][1] = t.y; v[u][2] = t.z; v[u][3] = t.w;
          } else {
            const float2 t = *reinterpret_cast<const float2*>(accp + static_cast<int64_t>(p) * D);
            v[u][0] = t.x; v[u][1] = t.y;
          }
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

  __device__ __forceinline__ void add(float m, float l, const float (&v)[EPL]) {
    const float Mn = fmaxf(M, m);
    if (Mn == kNegInf) return;  // nothing but empty partitions so far
    const float c_old = exp2f(M - Mn), c_new = exp2f(m - Mn);
    den = den * c_old + l * c_new;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = o[e] * c_old + v[e] * c_new;
    M = Mn;
  }
};

__device__ __forceinline__ int reduce_parts_of(const DecodeArgs& a, int s) {
  const int len_cap = min(a.max_context_len, a.max_blocks_per_seq * kBlockSize);
  int L = a.context_lens[s];
  L = L < 0 ? 0 : (L > len_cap ? len_cap : L);
  return L > 0 ? (L + a.partition_size - 1) / a.partition_size : 1;
}

constexpr int kReduceWarps = 8;

// Few partitions per row: one warp per (sequence, query head) row, a CTA
// holding kReduceWarps rows.  Rows of sequences that fit one partition
// return at once (the partition kernel wrote their output).
template <int D>
__global__ void __launch_bounds__(kReduceWarps * 32) decode_reduce_rows_kernel(const DecodeArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kReduceWarps + warp;
  if (row >= static_cast<int64_t>(a.num_seqs) * a.num_q_heads) return;
  const int nparts = reduce_parts_of(a, static_cast<int>(row / a.num_q_heads));
  if (nparts <= 1) return;
  RowMerge<D> r;
  r.run(a.ws_ml + row * a.max_parts, a.ws_acc + row * a.max_parts * D + lane * RowMerge<D>::EPL, 0, 1, nparts);
  const float inv = r.den > 0.f ? 1.f / r.den : 0.f;
  const int64_t obase = row * D + lane * RowMerge<D>::EPL;
#pragma unroll
  for (int e = 0; e < RowMerge<D>::EPL; ++e) store_out(a.out, obase + e, r.o[e] * inv, a.out_dtype);
}

// Many partitions per row (long contexts): one CTA per row; warp w merges
// partitions w, w + kReduceWarps, ... and the warps' states are merged
// through shared memory.
template <int D>
__global__ void __launch_bounds__(kReduceWarps * 32) decode_reduce_long_kernel(const DecodeArgs a) {
  __shared__ float sm_m[kReduceWarps], sm_l[kReduceWarps];
  __shared__ float sm_o[kReduceWarps][D];
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  const int nparts = reduce_parts_of(a, static_cast<int>(row / a.num_q_heads));
  if (nparts <= 1) return;
  RowMerge<D> r;
  r.run(a.ws_ml + row * a.max_parts, a.ws_acc + row * a.max_parts * D + lane * RowMerge<D>::EPL, warp,
        kReduceWarps, nparts);
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
    for (int w = 0; w < kReduceWarps; ++w) M = fmaxf(M, sm_m[w]);
    const float mu = (M == kNegInf) ? 0.f : M;
    float o = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kReduceWarps; ++w) {
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

template <int D, bool BF16>
cudaError_t launch_partitions_t(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t stream) {
  using Geom = TileGeom<D>;
  constexpr int NW = kWarpsPerCta, NST = kStages;
  const size_t smem = 1024 + static_cast<size_t>(NW) * NST * Geom::kStageBytes + NW * NST * 8;
  auto kern = decode_partitions_kernel<D, BF16, NW, NST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t units = static_cast<int64_t>(a.num_kv_heads) * a.num_seqs * a.max_parts;
  const int64_t ctas = (units + NW - 1) / NW;
  if (ctas == 0) return cudaSuccess;
  return launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(NW * 32), smem, stream, a, tk, tv);
}

}  // namespace

cudaError_t launch_decode_partitions(const DecodeArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                     int head_dim, int kv_bf16, cudaStream_t stream) {
  if (head_dim == 128)
    return kv_bf16 ? launch_partitions_t<128, true>(a, tmap_k, tmap_v, stream)
                   : launch_partitions_t<128, false>(a, tmap_k, tmap_v, stream);
  if (head_dim == 64)
    return kv_bf16 ? launch_partitions_t<64, true>(a, tmap_k, tmap_v, stream)
                   : launch_partitions_t<64, false>(a, tmap_k, tmap_v, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_reduce(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  if (a.max_parts <= 1 || a.num_seqs == 0) return cudaSuccess;
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  const dim3 block(kReduceWarps * 32);
  if (a.max_parts > 4 * RowMerge<128>::U) {  // long rows: a CTA per row
    const dim3 grid(static_cast<unsigned>(rows));
    if (head_dim == 128) return launch_pdl(decode_reduce_long_kernel<128>, grid, block, 0, stream, a);
    if (head_dim == 64) return launch_pdl(decode_reduce_long_kernel<64>, grid, block, 0, stream, a);
    return cudaErrorInvalidValue;
  }
  const dim3 grid(static_cast<unsigned>((rows + kReduceWarps - 1) / kReduceWarps));
  if (head_dim == 128) return launch_pdl(decode_reduce_rows_kernel<128>, grid, block, 0, stream, a);
  if (head_dim == 64) return launch_pdl(decode_reduce_rows_kernel<64>, grid, block, 0, stream, a);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
