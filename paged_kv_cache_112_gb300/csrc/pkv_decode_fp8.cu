// Paged decode attention over FP8 (e4m3) pools for sm_103a: partition
// kernel (the reduce kernel is the 16-bit path's, its workspace records are
// the same).
//
// What is computed: the attention of pkv_decode_attention with
// k_t = decode(k8_t) * k_scale[block][g] and v_t likewise, one float scale per
// (physical block, KV head) -- the 16-token block as the quantisation group
// whose scales travel with it ("PagedAttention internals", section 06
// "Blocks as quantization groups"; "KV Cache & PagedAttention", section 5:
// K, V stored in FP8 halve the bytes decode reads).
//
// Mapping onto GB300 (head_dim 128):
//  * Same units, grid, warps-per-unit rule and per-warp TMA ring as the
//    16-bit kernel; a (block, head) tile is 16 rows x 128 bytes of codes,
//    one TMA box in the 128-byte swizzle, so a stage (K + V) is 4 KB and the
//    ring holds 4 stages.
//  * Both contractions run on the tensor cores as f16 mma.sync m16n8k16:
//    e4m3 -> f16 is exact (cvt.rn.f16x2.e4m3x2).  bf16 queries are
//    converted to f16 after a power-of-two prescale that keeps the group's
//    largest |q| inside the f16 range.
//  * No ldmatrix: the dot product is invariant under any permutation of the
//    head dimension applied to both q and k, and the output rows of
//    O^T = V^T P^T may be stored in any order.  Both are chosen so that lane
//    (gr = lane/4, tq = lane%4) needs exactly bytes [32tq, 32tq+32) of token
//    rows gr and gr+8: two 16-byte shared loads per row, conflict-free under
//    the swizzle.  For QK^T, k-step kk takes codes 32tq+4kk+{0,1} (A cols
//    2tq, 2tq+1) and 32tq+4kk+{2,3} (cols 2tq+8, 2tq+9).  For PV (A = V^T,
//    k = tokens) lane (gr, tq) reads chunk gr (dims 16gr..16gr+15) of token
//    rows 2tq, 2tq+1, 2tq+8, 2tq+9; a byte permute pairs each dim's codes of
//    two tokens, which convert straight to the f16x2 A registers.  Row gr
//    (gr+8) of M-tile mt is dim 16gr + 2mt (+1), so a lane ends up owning
//    16 contiguous output dims of its two heads.
//  * Scales: the K scale multiplies the tile's scores with the softmax scale
//    (one multiplier per tile); the V scale multiplies P before it is split
//    into f16 hi + lo parts, in a per-warp power-of-two unit (raised, with
//    the accumulator rescaled, when a chunk's largest V scale needs it) that
//    keeps P * scale inside the f16 range.  Both scales are read with the
//    table entries, one chunk of 32 tiles at a time.
//  * The accumulator is rescaled only in tiles where some head's running
//    max grows (a warp-uniform branch).
#include "pkv_balanced.cuh"
#include "pkv_fp8.cuh"

namespace pkv {
namespace {

using namespace dev;

constexpr int kFp8Stages = 4;

// Four e4m3 codes (bytes 0..3 of w) -> two f16x2 (codes 0,1 in lo; 2,3 in hi;
// the lower-addressed code in the lower half).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// 16 bytes of shared memory into r[0..3].
__device__ __forceinline__ void lds128(uint32_t* r, uint32_t addr) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Attention state of one warp serving the G <= 8 query heads of one KV head
// over FP8 tiles (layout and permutations as described at the top).
template <int D>
struct WarpAttentionFp8 : SoftmaxState<D / 16> {
  static_assert(D == 128, "FP8 tiles are one 128-byte line per head row");
  static constexpr int KT = D / 16;
  using Base = SoftmaxState<KT>;
  using Base::acc;
  uint32_t qf[KT][2];  // f16x2: q[head gr][32tq + 4kk + {0,1}] and {2,3}

  // Loads the group's query rows (heads >= G read as 0) in the permuted
  // order and returns the power of two by which they were scaled down (1
  // for f16; for bf16, 2^e with the group's max |q| / 2^e below 2^15).
  template <bool QBF16>
  __device__ __forceinline__ float load_q(const uint16_t* qhead0, int G, int lane) {
    const int gr = lane >> 2, tq = lane & 3;
    const bool live = gr < G;
    const uint4* src = reinterpret_cast<const uint4*>(qhead0 + (live ? gr : 0) * D + 32 * tq);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = live ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
    float down = 1.f;
    if constexpr (QBF16) {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 f = unpack_bf16(w[i]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
      // 2^e >= amax / 2^14.99: exponent of amax minus 14, at least 0.
      const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xff) - 127;
      const int e = min(max(ex - 14, 0), 120);
      const float mul = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, exact
      down = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 f = unpack_bf16(w[i]);
        w[i] = pack_f16(f.x * mul, f.y * mul);
      }
    }
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      qf[kk][0] = w[2 * kk];
      qf[kk][1] = w[2 * kk + 1];
    }
    return down;
  }

  // NT tiles at once (independent chains interleave; one softmax update for
  // all of them).  Tile t: K at sK[t], V at sK[t] + VOFF, nv[t] valid
  // tokens (rows >= nv are masked, whatever they hold), sl2k[t] = log2(e) *
  // softmax scale * q prescale * K scale, pv[t] = V scale in the
  // accumulator's unit (a power of two chosen per chunk of tiles).
  template <int NT, int VOFF = 2048>
  __device__ __forceinline__ void tiles(const uint32_t (&sK)[NT], const int (&nv)[NT], const float (&sl2k)[NT],
                                        const float (&pv)[NT], int lane) {
    const int gr = lane >> 2, tq = lane & 3;
    // K: rows gr and gr+8 (same swizzle phase), chunks 2tq and 2tq+1.
    const uint32_t off0 = gr * 128 + (((2 * tq) ^ gr) << 4);
    const uint32_t off1 = gr * 128 + (((2 * tq + 1) ^ gr) << 4);
    uint32_t kw[NT][2][8];  // words i = codes [32tq + 4i, +4) of rows gr, gr+8
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      lds128(kw[t][0], sK[t] + off0);
      lds128(kw[t][0] + 4, sK[t] + off1);
      lds128(kw[t][1], sK[t] + 1024 + off0);
      lds128(kw[t][1] + 4, sK[t] + 1024 + off1);
    }
    // Scores S^T[token][head]; per tile, even and odd k-steps in separate chains.
    float c[NT][2][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int j = 0; j < 4; ++j) c[t][0][j] = c[t][1][j] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KT; ++kk)
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        uint32_t a[4];
        e4m3x4_to_f16x4(kw[t][0][kk], a[0], a[2]);
        e4m3x4_to_f16x4(kw[t][1][kk], a[1], a[3]);
        mma_16816<false>(c[t][kk & 1], a, qf[kk][0], qf[kk][1]);
      }
    // V: rows 2tq, 2tq+1, 2tq+8, 2tq+9, chunk gr (codes of dims 16gr .. 16gr+15).
    const int r0 = 2 * tq;
    const uint32_t voff[4] = {static_cast<uint32_t>(r0 * 128 + ((gr ^ r0) << 4)),
                              static_cast<uint32_t>((r0 + 1) * 128 + ((gr ^ (r0 + 1)) << 4)),
                              static_cast<uint32_t>((r0 + 8) * 128 + ((gr ^ r0) << 4)),
                              static_cast<uint32_t>((r0 + 9) * 128 + ((gr ^ (r0 + 1)) << 4))};
    uint32_t vw[NT][4][4];  // [tile][row 2tq, 2tq+1, 2tq+8, 2tq+9][word]
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int r = 0; r < 4; ++r) lds128(vw[t][r], sK[t] + VOFF + voff[r]);

    float sc[4 * NT], p[4 * NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      sc[4 * t] = (c[t][0][0] + c[t][1][0]) * sl2k[t];
      sc[4 * t + 1] = (c[t][0][1] + c[t][1][1]) * sl2k[t];
      sc[4 * t + 2] = (c[t][0][2] + c[t][1][2]) * sl2k[t];
      sc[4 * t + 3] = (c[t][0][3] + c[t][1][3]) * sl2k[t];
      if (gr >= nv[t]) sc[4 * t] = sc[4 * t + 1] = kNegInf;
      if (gr + 8 >= nv[t]) sc[4 * t + 2] = sc[4 * t + 3] = kNegInf;
    }
    this->template online_update_lazy<NT>(sc, p);

    // P^T (times the V scale) as f16 hi + lo parts, two MMAs per tile, so
    // the weights keep ~2^-22 relative precision.
    uint32_t pb[NT][4];  // hi (tokens 0-7, 8-15), lo (tokens 0-7, 8-15)
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float q0 = p[4 * t] * pv[t], q1 = p[4 * t + 1] * pv[t];
      const float q2 = p[4 * t + 2] * pv[t], q3 = p[4 * t + 3] * pv[t];
      const uint32_t h0 = pack_f16(q0, q1), h1 = pack_f16(q2, q3);
      const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
      const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
      pb[t][0] = movmatrix_trans(h0);
      pb[t][1] = movmatrix_trans(h1);
      pb[t][2] = movmatrix_trans(pack_f16(q0 - f0.x, q1 - f0.y));
      pb[t][3] = movmatrix_trans(pack_f16(q2 - f1.x, q3 - f1.y));
      // V codes of tokens >= nv may be anything (NaN codes included): zero them.
      if (nv[t] < kBlockSize) {
        const int row[4] = {r0, r0 + 1, r0 + 8, r0 + 9};
#pragma unroll
        for (int r = 0; r < 4; ++r)
          if (row[r] >= nv[t]) vw[t][r][0] = vw[t][r][1] = vw[t][r][2] = vw[t][r][3] = 0u;
      }
    }
    // V^T A fragment of M-tile mt: rows gr / gr+8 are dims 16gr+2mt / +1,
    // k = tokens.  A byte permute pairs a dim's codes of tokens 2tq and
    // 2tq+1 (and 2tq+8, 2tq+9), which convert to the f16x2 the MMA wants.
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int w = mt >> 1;
      const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        uint32_t va[4];
        e4m3x4_to_f16x4(__byte_perm(vw[t][0][w], vw[t][1][w], sel), va[0], va[1]);
        e4m3x4_to_f16x4(__byte_perm(vw[t][2][w], vw[t][3][w], sel), va[2], va[3]);
        mma_16816<false>(acc[mt], va, pb[t][0], pb[t][1]);
        mma_16816<false>(acc[mt], va, pb[t][2], pb[t][3]);
      }
    }
  }

  // acc[mt][0..1] hold dim 16gr + 2mt of heads a, b; acc[mt][2..3] dim +1:
  // a lane owns dims [16gr, 16gr+16) of its two heads.
  __device__ __forceinline__ void store_final(void* out, int64_t out_head0, int G, int dtype, int lane) const {
    const int gr = lane >> 2, tq = lane & 3;
    const int ha = 2 * tq, hb = ha + 1;
    const float ia = this->l_a > 0.f ? 1.f / this->l_a : 0.f;
    const float ib = this->l_b > 0.f ? 1.f / this->l_b : 0.f;
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int d = 16 * gr + 2 * mt;
      if (ha < G) {
        store_out(out, (out_head0 + ha) * D + d, acc[mt][0] * ia, dtype);
        store_out(out, (out_head0 + ha) * D + d + 1, acc[mt][2] * ia, dtype);
      }
      if (hb < G) {
        store_out(out, (out_head0 + hb) * D + d, acc[mt][1] * ib, dtype);
        store_out(out, (out_head0 + hb) * D + d + 1, acc[mt][3] * ib, dtype);
      }
    }
  }

  __device__ __forceinline__ void store_partial(float* ws_acc, float2* ws_ml, int64_t rec0, int64_t rec_stride,
                                                int G, int lane) const {
    const int gr = lane >> 2, tq = lane & 3;
    const int ha = 2 * tq, hb = ha + 1;
    const int64_t ra = rec0 + ha * rec_stride, rb = rec0 + hb * rec_stride;
#pragma unroll
    for (int j = 0; j < KT / 2; ++j) {  // dims 16gr + 4j .. +3: M-tiles 2j, 2j+1
      if (ha < G)
        *reinterpret_cast<float4*>(ws_acc + ra * D + 16 * gr + 4 * j) =
            make_float4(acc[2 * j][0], acc[2 * j][2], acc[2 * j + 1][0], acc[2 * j + 1][2]);
      if (hb < G)
        *reinterpret_cast<float4*>(ws_acc + rb * D + 16 * gr + 4 * j) =
            make_float4(acc[2 * j][1], acc[2 * j][3], acc[2 * j + 1][1], acc[2 * j + 1][3]);
    }
    if (gr == 0) {
      if (ha < G) ws_ml[ra] = make_float2(this->m_a, this->l_a);
      if (hb < G) ws_ml[rb] = make_float2(this->m_b, this->l_b);
    }
  }
};

// 2^e for an integer e in [-126, 127], exactly.
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// The factor 2^(from - to) that moves the accumulator from unit 2^from to
// unit 2^to (to > from), exactly, down to the f32 subnormals and 0 (the
// first unit of a pair starts at 2^-126, so the gap can exceed 126).
__device__ __forceinline__ float unit_change(int from, int to) { return ldexpf(1.f, from - to); }

// The accumulator's unit for a chunk of tiles: 2^-e with 2^e <= the
// largest V scale of the chunk (over the warp) < 2^(e+1), so P * scale /
// unit stays below 2 and well inside the f16 range.
__device__ __forceinline__ int chunk_exponent(float vs) {
  float m = vs;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xff) - 127;
  return min(max(e, -126), 126);
}

// The token generated this step, for the warp that reads the tile holding
// its position L-1 (fused decode step over FP8 pools).  Lanes [0, 16) hold
// the 16-byte chunks (8 values) of the K row of KV head g, lanes [16, 32)
// those of the V row.  The warp checks the slot against the table,
// quantises the row with the block's scales (fp8::quantize4, as the write
// kernel does), stores the codes to the pools and patches them into its
// shared-memory tiles, so the attention reads the new token at once.
template <int D>
struct NewTokenFp8 {
  static_assert(D == 128, "16 lanes x 8 values per row");
  uint4 val;
  uint2 code;
  int row = -1;
  int slot = -1;
  int last_phys = -1;

  __device__ __forceinline__ void prefetch(const DecodeArgs& a, int s, int g, int L, int lane) {
    slot = a.slot_mapping[s];
    last_phys = L > 0 ? __ldg(a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + (L - 1) / kBlockSize)
                      : -1;
    const uint16_t* src = (lane < 16 ? a.k_new : a.v_new) + static_cast<int64_t>(s) * a.new_stride + g * D +
                          (lane & 15) * 8;
    val = __ldg(reinterpret_cast<const uint4*>(src));
    row = L > 0 ? (L - 1) % kBlockSize : -1;
  }

  // Whether the slot is position L-1 through the table; if not, flags
  // PKV_DEV_ERR_SLOT (unless the slot is -1) and drops the token.
  __device__ __forceinline__ bool check(const DecodeArgs& a, int lane) {
    const bool ok = row >= 0 && slot != -1 && static_cast<unsigned>(last_phys) < static_cast<unsigned>(a.num_blocks) &&
                    slot == last_phys * kBlockSize + row;
    if (!ok) {
      if (slot != -1 && lane == 0) flag(a.dev_status, 1u);
      row = -1;
    }
    return ok;
  }

  // Quantises and stores this lane's 8 values (K scale for lanes < 16, V
  // scale above) and keeps the codes for patch().
  template <bool BF16>
  __device__ __forceinline__ void store(const DecodeArgs& a, int g, float k_scale, float v_scale, int lane) {
    const float sc = lane < 16 ? k_scale : v_scale;
    code = make_uint2(fp8::quantize4(val.x, val.y, sc, BF16), fp8::quantize4(val.z, val.w, sc, BF16));
    uint8_t* pool = reinterpret_cast<uint8_t*>(lane < 16 ? a.k_pool_w : a.v_pool_w);
    *reinterpret_cast<uint2*>(pool + (slot / kBlockSize) * a.block_stride +
                              static_cast<int64_t>(row) * a.num_kv_heads * D + g * D + (lane & 15) * 8) = code;
  }

  // Overwrites token `row` of the K and V tiles (128-byte swizzle: 8-byte
  // half c & 1 of 16-byte chunk c / 2, chunk at position (c / 2) ^ (row & 7)).
  __device__ __forceinline__ void patch(uint32_t k_tile, uint32_t v_tile, int lane) const {
    const int c = lane & 15;
    const uint32_t addr = (lane < 16 ? k_tile : v_tile) + row * 128 + ((((c >> 1) ^ (row & 7))) << 4) + ((c & 1) << 3);
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(code.x), "r"(code.y) : "memory");
    __syncwarp();
  }
};

// One unit (sequence s, KV head g, partition p) served by U of the CTA's NW
// warps; `raw_len` is the sequence's context length as read and `first` the
// warp's first table entries (first_entries<U>).  The control flow is the
// 16-bit kernel's; the per-tile scales come with the table entries.
template <int D, bool QBF16, int NW, int U, int NST, bool FUSED>
__device__ __forceinline__ void partition_unit_fp8(const DecodeArgs& a, const CUtensorMap* tmap_k,
                                                   const CUtensorMap* tmap_v, uint8_t* smem, int64_t unit,
                                                   int raw_len, int first, int warp, int lane) {
  using Geom = TileGeom<D, 1>;
  using Att = WarpAttentionFp8<D>;
  static_assert(NW % U == 0 && NW / U <= 15, "named barriers 1..15, one per unit of the CTA");
  static_assert(Att::kSaveBytes <= NST * Geom::kStageBytes, "a saved state must fit its warp's ring");
  const int sub = warp % U;
  const int Hkv = a.num_kv_heads;
  const int g = static_cast<int>(unit % Hkv);
  const int64_t rest = unit / Hkv;
  const int s = static_cast<int>(rest % a.num_seqs);
  const int part = static_cast<int>(rest / a.num_seqs);

  const int PS = a.partition_size;
  const int G = a.group;
  const int L = clamp_len(a, raw_len, part == 0 && g == 0 && sub == 0 && lane == 0);
  const int nparts = L > 0 ? (L + PS - 1) / PS : 1;
  if (part >= nparts) return;
  Att at;
  const float q_up = at.template load_q<QBF16>(a.q + (static_cast<int64_t>(s) * a.num_q_heads + g * G) * D, G, lane);
  const float sl2q = a.scale_log2 * q_up;
  const int tok0 = part * PS;
  const int ntok = max(0, min(L - tok0, PS));
  const int nblk = (ntok + kBlockSize - 1) / kBlockSize;
  const int cnt = nblk > sub ? (nblk - sub + U - 1) / U : 0;
  const int32_t* tbl = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq + tok0 / kBlockSize;
  auto entry = [&](int i) { return i < cnt ? __ldg(tbl + i * U + sub) : 0; };
  // Scales of (entry, g); 1 for an entry outside the pool (its tile is masked).
  auto ks_of = [&](int phys) {
    return static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks)
               ? __ldg(a.k_scale + static_cast<int64_t>(phys) * a.scale_stride + g)
               : 1.f;
  };
  auto vs_of = [&](int phys) {
    return static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks)
               ? __ldg(a.v_scale + static_cast<int64_t>(phys) * a.scale_stride + g)
               : 1.f;
  };
  // Lane j holds the entry and scales of the warp's tile j of the current
  // chunk of 32 (the previous chunk's scales stay until its last tile, which
  // is consumed up to NST - 1 tiles after the next chunk's first issue).
  // Lanes past the unit's tiles hold scale 0 (their entries are not used).
  int phys_cur = first;
  int phys_next = entry(32 + lane);
  float ks_cur = lane < cnt ? ks_of(first) : 0.f, vs_cur = lane < cnt ? vs_of(first) : 0.f;
  float ks_prev = 0.f, vs_prev = 0.f;
  int chunk_cur = 0;
  // The accumulator holds (sum of P V) * 2^-vexp; vexp only grows, at the
  // first tile of a chunk whose largest V scale needs it.
  int vexp = -126, vexp_chunk = -1;
  float inv_unit = exp2i(126);

  WarpRing<D, NST, 1> ring{smem_u32(smem + static_cast<size_t>(warp) * NST * Geom::kStageBytes),
                           smem_u32(smem + static_cast<size_t>(NW) * NST * Geom::kStageBytes) + 8 * NST * warp};
  ring.init(lane);
  uint32_t bad_stage = 0;

  auto issue = [&](int j) {  // all lanes call
    if ((j & 31) == 0 && j > 0) {
      phys_cur = phys_next;
      phys_next = entry(j + 32 + lane);
      ks_prev = ks_cur;
      vs_prev = vs_cur;
      const bool mine = j + lane < cnt;
      ks_cur = mine ? ks_of(phys_cur) : 0.f;
      vs_cur = mine ? vs_of(phys_cur) : 0.f;
      chunk_cur = j >> 5;
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
    ring.issue(j, phys, -1, 0, g, tmap_k, tmap_v, lane);
  };

  at.reset();
  for (int j = 0; j < min(cnt, NST); ++j) issue(j);

  // Fused decode step: the last block of the last partition of (s, g) holds
  // position L-1.
  NewTokenFp8<D> nt;
  const bool owns_new = FUSED && part == nparts - 1 && sub == (nblk > 0 ? (nblk - 1) % U : 0);
  if (owns_new) {
    nt.prefetch(a, s, g, L, lane);
    if (nblk == 0) nt.check(a, lane);  // empty sequence: only checks the slot
  }

  // Tiles are consumed two at a time (i even; both in the same chunk of
  // 32).  A missing second tile reuses the first one's buffer with no valid
  // token.
  static_assert(NST % 2 == 0, "tile pairs take whole pairs of stages");
  for (int i = 0; i < cnt; i += 2) {
    const bool two = i + 1 < cnt;
    const bool ok = ring.wait(i, a.timeout_ns) && (!two || ring.wait(i + 1, a.timeout_ns));
    if (!__all_sync(kFull, ok)) {
      ring.drain(i, min(cnt, i + NST), a.timeout_ns);
      if (lane == 0) flag(a.dev_status, 16u);  // PKV_DEV_ERR_TIMEOUT; the output is undefined
      break;
    }
    if ((i >> 5) != vexp_chunk) {  // first pair of a chunk (its scales arrived NST tiles ago)
      vexp_chunk = i >> 5;
      const int e = chunk_exponent(vs_cur);
      if (e > vexp) {
        at.scale_acc(unit_change(vexp, e));
        vexp = e;
        inv_unit = exp2i(-e);
      }
    }
    const bool cur = (i >> 5) == chunk_cur;
    const float ksel = cur ? ks_cur : ks_prev, vsel = cur ? vs_cur : vs_prev;
    uint32_t sK[2];
    int nv[2];
    float sl2k[2], pv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int j = two ? i + u : i;
      const int st = j % NST;
      const int t = j * U + sub;
      nv[u] = (u == 1 && !two) || ((bad_stage >> st) & 1) ? 0 : min(kBlockSize, ntok - t * kBlockSize);
      sK[u] = ring.k_tile(j);
      const float ksc = __shfl_sync(kFull, ksel, j & 31), vsc = __shfl_sync(kFull, vsel, j & 31);
      if (owns_new && (u == 0 || two) && t == nblk - 1 && nt.check(a, lane)) {
        nt.template store<QBF16>(a, g, ksc, vsc, lane);
        nt.patch(sK[u], sK[u] + Geom::kTileBytes, lane);
      }
      sl2k[u] = sl2q * ksc;
      pv[u] = inv_unit * vsc;
    }
    at.template tiles<2>(sK, nv, sl2k, pv, lane);
    __syncwarp();
    if (i + NST < cnt) {
      if (owns_new) fence_proxy_async_smem();  // only the new token's patch writes a stage
      issue(i + NST);
      if (i + 1 + NST < cnt) issue(i + 1 + NST);
    }
  }

  at.scale_acc(exp2i(vexp));
  at.finish_sums();
  if constexpr (U > 1) {
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

// Two-warp CTAs, units assigned as in the 16-bit kernel.  Six per SM (12
// warps x 4 stages x 4 KB = 192 KB of tiles in flight); the bound lets the
// tile's loads and conversions keep all their registers (154, no spills).
template <int D, bool QBF16, int NST, bool FUSED>
__global__ void __launch_bounds__(64, 6) decode_partitions_fp8_kernel(
    const DecodeArgs a, const __grid_constant__ CUtensorMap tmap_k,
    const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ __align__(1024) uint8_t smem[];
  griddep_wait();
  griddep_launch_dependents();
  if (smem_misaligned(smem, a.dev_status)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t units = static_cast<int64_t>(a.num_kv_heads) * a.num_seqs * a.max_parts;
  const int64_t unit1 = static_cast<int64_t>(blockIdx.x) * 2 + warp, unit2 = blockIdx.x;
  auto seq_of = [&](int64_t u) { return static_cast<int>((u / a.num_kv_heads) % a.num_seqs); };
  if (a.unit_warps == 2) {
    if (unit2 < units)
      partition_unit_fp8<D, QBF16, 2, 2, NST, FUSED>(a, &tmap_k, &tmap_v, smem, unit2,
                                                     a.context_lens[seq_of(unit2)],
                                                     first_entries<2>(a, unit2, warp, lane), warp, lane);
  } else if (unit1 < units) {
    partition_unit_fp8<D, QBF16, 2, 1, NST, FUSED>(a, &tmap_k, &tmap_v, smem, unit1,
                                                   a.context_lens[seq_of(unit1)],
                                                   first_entries<1>(a, unit1, 0, lane), warp, lane);
  }
}

// ------------------------------------------------------ head-group partitions
//
// Fixed partitions, HP KV heads per CTA: one CTA serves (sequence s,
// partition p) for KV heads [gi * HP, gi * HP + HP), one warp per head.  A
// block's codes for HP adjacent heads are adjacent 128-byte lines of each
// row, so one TMA box of (128 bytes, 16 rows, HP lines) brings the K tiles
// of all HP heads at once, and another their V tiles: two copies per block
// for the CTA instead of two per head.  An FP8 tile is only 2 KB, and one
// copy per 2 KB, issued per warp, is about as many copies as an SM's TMA
// unit accepts at full HBM rate; this way the copies carry HP * 2 KB.
//  * The HP warps share one ring of NST stages ([K: HP heads][V: HP heads]),
//    filled by lane 0 of warp 0.  Every warp waits on a stage's barrier,
//    reads its own head's K and V tile and keeps its own softmax state and
//    scales; after each step __syncthreads_or() both frees the step's
//    stages for the next copies and makes a timed-out wait a decision of the
//    whole CTA.
//  * Work per warp, tile math and outputs are the one-warp-per-unit
//    partition kernel's (fused write excluded: the head-group grid serves
//    write-then-attend calls).
template <int D, bool QBF16, int HP, int NST>
__global__ void __launch_bounds__(HP * 32, 12 / HP) decode_partitions_fp8_hg_kernel(
    const DecodeArgs a, const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v) {
  using Att = WarpAttentionFp8<D>;
  static_assert(D == 128 && NST % 2 == 0, "FP8 tiles are one 128-byte line per head row; tile pairs");
  constexpr uint32_t kHeadTile = kBlockSize * 128;  // one head's 16 rows of codes
  constexpr uint32_t kKBytes = HP * kHeadTile;      // the group's K tiles of one block
  constexpr uint32_t kStage = 2 * kKBytes;          // then its V tiles
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
  const int tiles_per_part = PS / kBlockSize;
  const int32_t* tbl = a.block_tables + static_cast<int64_t>(s) * a.max_blocks_per_seq;
  const int first = lane < tiles_per_part && part * tiles_per_part + lane < a.max_blocks_per_seq
                        ? __ldg(tbl + part * tiles_per_part + lane)
                        : 0;
  const int L = clamp_len(a, a.context_lens[s], part == 0 && gi == 0 && warp == 0 && lane == 0);
  const int nparts = L > 0 ? (L + PS - 1) / PS : 1;
  if (part >= nparts) return;  // the same for every warp of the CTA
  const int tok0 = part * PS;
  const int ntok = max(0, min(L - tok0, PS));
  const int cnt = (ntok + kBlockSize - 1) / kBlockSize;
  tbl += tok0 / kBlockSize;
  auto entry = [&](int i) { return i < cnt ? __ldg(tbl + i) : 0; };
  auto ks_of = [&](int phys) {
    return static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks)
               ? __ldg(a.k_scale + static_cast<int64_t>(phys) * a.scale_stride + g)
               : 1.f;
  };
  auto vs_of = [&](int phys) {
    return static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks)
               ? __ldg(a.v_scale + static_cast<int64_t>(phys) * a.scale_stride + g)
               : 1.f;
  };

  const uint32_t ring = smem_u32(smem);
  const uint32_t bars = ring + NST * kStage;
  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) mbar_init(bars + 8 * st, 1);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncthreads();

  // Entries and this head's scales, 32 tiles a chunk (as the partition kernel).
  int phys_cur = first;
  int phys_next = entry(32 + lane);
  float ks_cur = lane < cnt ? ks_of(first) : 0.f, vs_cur = lane < cnt ? vs_of(first) : 0.f;
  float ks_prev = 0.f, vs_prev = 0.f;
  int chunk_cur = 0;
  int vexp = -126, vexp_chunk = -1;
  float inv_unit = exp2i(126);
  uint32_t bad_stage = 0;

  auto issue = [&](int j) {  // every lane of every warp calls; lane 0 of warp 0 copies
    if ((j & 31) == 0 && j > 0) {
      phys_cur = phys_next;
      phys_next = entry(j + 32 + lane);
      ks_prev = ks_cur;
      vs_prev = vs_cur;
      const bool mine = j + lane < cnt;
      ks_cur = mine ? ks_of(phys_cur) : 0.f;
      vs_cur = mine ? vs_of(phys_cur) : 0.f;
      chunk_cur = j >> 5;
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
      const uint32_t bar = bars + 8 * st;
      const uint32_t dst = ring + st * kStage;
      mbar_arrive_expect_tx(bar, kStage);
      tma_load_4d(dst, &tmap_k, 0, 0, gi * HP, phys, bar);
      tma_load_4d(dst + kKBytes, &tmap_v, 0, 0, gi * HP, phys, bar);
    }
  };
  auto wait = [&](int j) { return mbar_wait_bounded(bars + 8 * (j % NST), (j / NST) & 1, a.timeout_ns); };

  Att at;
  at.reset();
  for (int j = 0; j < min(cnt, NST); ++j) issue(j);
  const float sl2q =
      a.scale_log2 * at.template load_q<QBF16>(a.q + (static_cast<int64_t>(s) * a.num_q_heads + g * G) * D, G, lane);

  for (int i = 0; i < cnt; i += 2) {
    const bool two = i + 1 < cnt;
    const bool ok = __all_sync(kFull, wait(i) && (!two || wait(i + 1)));
    if (ok) {
      if ((i >> 5) != vexp_chunk) {  // first pair of a chunk (its scales arrived NST tiles ago)
        vexp_chunk = i >> 5;
        const int e = chunk_exponent(vs_cur);
        if (e > vexp) {
          at.scale_acc(unit_change(vexp, e));
          vexp = e;
          inv_unit = exp2i(-e);
        }
      }
      const bool cur = (i >> 5) == chunk_cur;
      const float ksel = cur ? ks_cur : ks_prev, vsel = cur ? vs_cur : vs_prev;
      uint32_t sK[2];
      int nv[2];
      float sl2k[2], pv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int j = two ? i + u : i;  // a missing second tile reuses the first one's stage, no valid token
        const int st = j % NST;
        nv[u] = (u == 1 && !two) || ((bad_stage >> st) & 1) ? 0 : min(kBlockSize, ntok - j * kBlockSize);
        sK[u] = ring + st * kStage + warp * kHeadTile;
        sl2k[u] = sl2q * __shfl_sync(kFull, ksel, j & 31);
        pv[u] = inv_unit * __shfl_sync(kFull, vsel, j & 31);
      }
      at.template tiles<2, kKBytes>(sK, nv, sl2k, pv, lane);
    }
    // Every warp is done with this step's stages; a timed-out wait anywhere ends the CTA.
    if (__syncthreads_or(!ok)) {
      if (warp == 0)
        for (int j = i; j < min(cnt, i + NST); ++j) wait(j);  // copies in flight land before the CTA exits
      if (warp == 0 && lane == 0) flag(a.dev_status, 16u);  // PKV_DEV_ERR_TIMEOUT; the output is undefined
      return;
    }
    if (i + NST < cnt) issue(i + NST);
    if (i + 1 + NST < cnt) issue(i + 1 + NST);
  }

  at.scale_acc(exp2i(vexp));
  at.finish_sums();
  const int64_t head0 = static_cast<int64_t>(s) * a.num_q_heads + g * G;
  if (nparts == 1)
    at.store_final(a.out, head0, G, a.out_dtype, lane);
  else
    at.store_partial(a.ws_acc, a.ws_ml, head0 * a.max_parts + part, a.max_parts, G, lane);
}

// ------------------------------------------------------------ balanced split
//
// PKV_PARTITION_BALANCED over FP8 pools: the work order and equal shares of
// the 16-bit balanced kernel (pkv_balanced.cuh) with this file's tile math.
// One CTA of NW warps per SM; each warp's 4-stage ring of 4 KB tiles runs on
// across the (s, g) pairs of its share.
//  * Issue side: the table entries of three chunks (a chunk is up to 32
//    consecutive tiles of one pair; lane j holds tile j's entry) and the K/V
//    scales of the first two, so a chunk's scales are loaded one chunk
//    before its tiles are issued, from entries loaded one chunk before that.
//    Each issued tile's two scales are stored beside its stage, where the
//    compute side reads them with the tile.
//  * Compute side: two consecutive tiles of one pair share a softmax step;
//    a pair's last odd tile goes alone.  The accumulator's unit (a power of
//    two at least the largest V scale seen, as in the partition kernel)
//    starts afresh with each pair.
//  * Output: as the 16-bit balanced kernel (final rows for pairs a warp
//    covers whole, two partial-state slots per warp, pair metadata for the
//    balanced reduce).
template <int D, bool QBF16, int NW, int NST>
__global__ void __launch_bounds__(NW * 32, 1) decode_balanced_fp8_kernel(
    const DecodeArgs a, const __grid_constant__ CUtensorMap tmap_k,
    const __grid_constant__ CUtensorMap tmap_v) {
  using Geom = TileGeom<D, 1>;
  using Att = WarpAttentionFp8<D>;
  static_assert(NST % 2 == 0 && NST <= 32, "tile pairs take whole pairs of stages");
  extern __shared__ __align__(1024) uint8_t smem[];
  const size_t ring_bytes = static_cast<size_t>(NW) * NST * Geom::kStageBytes;
  const uint32_t bars = smem_u32(smem + ring_bytes);
  float2* stage_scale = reinterpret_cast<float2*>(smem + ring_bytes + NW * NST * 8);  // [NW][NST]: (k, v)
  int* pre = reinterpret_cast<int*>(smem + ring_bytes + NW * NST * 16);  // [S + 1] tile prefix
  int* len = pre + a.num_seqs + 1;                                        // [S] clamped lengths
  int* warp_tot = len + a.num_seqs;                                       // [32] scan scratch

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
  WarpRing<D, NST, 1> ring{smem_u32(smem + static_cast<size_t>(warp) * NST * Geom::kStageBytes),
                           bars + 8 * NST * warp};
  ring.init(lane);
  if (w >= W) return;
  const int64_t x0 = w * T / W, x1 = (w + 1) * T / W;
  const int count = static_cast<int>(x1 - x0);
  float2* my_scale = stage_scale + warp * NST;

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

  // ---- issue side
  struct Chunk {
    int s, g, base;
  };
  auto chunk_after = [&](const Chunk& c) -> Chunk {
    if (c.s >= S) return c;  // past the last pair: nothing follows
    const int n = pre[c.s + 1] - pre[c.s];
    if (c.base + 32 < n) return Chunk{c.s, c.g, c.base + 32};
    Cursor q{c.s, c.g, 0, n};
    next_pair(q, pre, S, Hkv);
    return Chunk{q.s, q.g, 0};
  };
  auto entry_of = [&](const Chunk& c) -> int {
    if (c.s >= S) return 0;
    const int t = c.base + lane;
    return t < pre[c.s + 1] - pre[c.s] ? __ldg(a.block_tables + static_cast<int64_t>(c.s) * a.max_blocks_per_seq + t)
                                       : 0;
  };
  // Scales of (entry, g); 1 for an entry outside the pool (its tile is masked).
  auto scale_of = [&](const float* sc, int phys, int g) {
    return static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks)
               ? __ldg(sc + static_cast<int64_t>(phys) * a.scale_stride + g)
               : 1.f;
  };
  Cursor ic = start;
  Chunk cur{ic.s, ic.g, ic.t};
  Chunk nxt = chunk_after(cur);
  Chunk nxt2 = chunk_after(nxt);
  int phys_cur = entry_of(cur), phys_nxt = entry_of(nxt), phys_nxt2 = entry_of(nxt2);
  float ks_cur = scale_of(a.k_scale, phys_cur, cur.g), vs_cur = scale_of(a.v_scale, phys_cur, cur.g);
  float ks_nxt = scale_of(a.k_scale, phys_nxt, nxt.g), vs_nxt = scale_of(a.v_scale, phys_nxt, nxt.g);
  uint32_t bad_stage = 0;

  auto issue = [&](int j) {  // tile j of this warp's range, at cursor ic; all lanes call
    if (ic.s != cur.s || ic.g != cur.g || ic.t >= cur.base + 32) {
      cur = nxt;
      phys_cur = phys_nxt;
      ks_cur = ks_nxt;
      vs_cur = vs_nxt;
      nxt = nxt2;
      phys_nxt = phys_nxt2;
      ks_nxt = scale_of(a.k_scale, phys_nxt, nxt.g);
      vs_nxt = scale_of(a.v_scale, phys_nxt, nxt.g);
      nxt2 = chunk_after(nxt);
      phys_nxt2 = entry_of(nxt2);
    }
    const int st = j % NST;
    const int idx = ic.t - cur.base;
    int phys = __shfl_sync(kFull, phys_cur, idx);
    const float ksc = __shfl_sync(kFull, ks_cur, idx), vsc = __shfl_sync(kFull, vs_cur, idx);
    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks)) {
      if (lane == 0) flag(a.dev_status, 4u);  // PKV_DEV_ERR_BLOCK
      phys = 0;
      bad_stage |= 1u << st;
    } else {
      bad_stage &= ~(1u << st);
    }
    if (lane == 0) my_scale[st] = make_float2(ksc, vsc);
    ring.issue(j, phys, -1, 0, ic.g, &tmap_k, &tmap_v, lane);
    advance(ic, pre, S, Hkv);
  };

  for (int j = 0; j < min(count, NST); ++j) issue(j);
  __syncwarp();  // the stage scales written by lane 0 before any lane reads them

  // ---- compute side
  Cursor cc = start;
  Att at;
  int seg_t0 = cc.t, seg_idx = 0;
  int vexp = -126;  // the accumulator holds (sum of P V) * 2^-vexp
  float inv_unit = exp2i(126);
  at.reset();
  float sl2q = a.scale_log2 *
               at.template load_q<QBF16>(a.q + (static_cast<int64_t>(cc.s) * a.num_q_heads + cc.g * G) * D, G, lane);
  for (int i = 0; i < count;) {
    if (i > 0 && cc.t == 0) {  // a new (s, g) pair starts here
      seg_t0 = 0;
      at.reset();
      vexp = -126;
      inv_unit = exp2i(126);
      sl2q = a.scale_log2 *
             at.template load_q<QBF16>(a.q + (static_cast<int64_t>(cc.s) * a.num_q_heads + cc.g * G) * D, G, lane);
    }
    const bool two = i + 1 < count && cc.t + 1 < cc.n;
    const bool ok = ring.wait(i, a.timeout_ns) && (!two || ring.wait(i + 1, a.timeout_ns));
    if (!__all_sync(kFull, ok)) {
      ring.drain(i, min(count, i + NST), a.timeout_ns);
      if (lane == 0) flag(a.dev_status, 16u);  // PKV_DEV_ERR_TIMEOUT; the output is undefined
      return;
    }
    uint32_t sK[2];
    int nv[2];
    float sl2k[2], vsc[2], pv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int j = two ? i + u : i;  // a missing second tile reuses the first one's stage, no valid token
      const int st = j % NST;
      const float2 sc = my_scale[st];
      nv[u] = (u == 1 && !two) || ((bad_stage >> st) & 1) ? 0
                                                          : min(kBlockSize, len[cc.s] - (cc.t + u) * kBlockSize);
      sK[u] = ring.k_tile(j);
      sl2k[u] = sl2q * sc.x;
      vsc[u] = (u == 1 && !two) ? 0.f : sc.y;
    }
    {
      const float vmax = fmaxf(vsc[0], vsc[1]);
      const int e = min(max(static_cast<int>((__float_as_uint(vmax) >> 23) & 0xff) - 127, -126), 126);
      if (e > vexp) {
        at.scale_acc(unit_change(vexp, e));
        vexp = e;
        inv_unit = exp2i(-e);
      }
    }
    pv[0] = vsc[0] * inv_unit;
    pv[1] = vsc[1] * inv_unit;
    at.template tiles<2>(sK, nv, sl2k, pv, lane);
    __syncwarp();
    const int used = two ? 2 : 1;
    for (int k = 0; k < used; ++k)
      if (i + k + NST < count) issue(i + k + NST);
    if (two) advance(cc, pre, S, Hkv);  // to the second tile (same pair)
    if (cc.t == cc.n - 1 || i + used == count) {  // end of a segment
      at.scale_acc(exp2i(vexp));
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
    i += used;
  }
}

constexpr int kFp8BalancedWarps = 12;  // 12 x 4 stages x 4 KB = 192 KB of tiles; 170 registers a thread

size_t balanced_fp8_smem(int num_seqs) {
  using Geom = TileGeom<128, 1>;
  return static_cast<size_t>(kFp8BalancedWarps) * kFp8Stages * (Geom::kStageBytes + 16) +
         (2 * static_cast<size_t>(num_seqs) + 1 + 32) * sizeof(int);
}

template <int D, bool QBF16, bool FUSED>
cudaError_t launch_fp8_t(const DecodeArgs& a_in, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  using Geom = TileGeom<D, 1>;
  constexpr int NST = kFp8Stages;
  const size_t smem = 2 * NST * Geom::kStageBytes + 2 * NST * 8;
  auto kern = decode_partitions_fp8_kernel<D, QBF16, NST, FUSED>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  DecodeArgs a = a_in;
  const int64_t units = static_cast<int64_t>(a.num_kv_heads) * a.num_seqs * a.max_parts;
  if (units == 0) return cudaSuccess;
  // Warps per unit: the 16-bit kernel's rule.
  const int slots = resident_warp_slots(reinterpret_cast<const void*>(kern), 64, smem);
  a.unit_warps = static_cast<int64_t>(a.num_kv_heads) * a.num_seqs > slots ? 2 : 1;
  const int64_t ctas = a.unit_warps == 1 ? (units + 1) / 2 : units;
  return launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(64), smem, stream, a, tk, tv);
}

template <int D, bool QBF16, int HP>
cudaError_t launch_fp8_hg_t(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  constexpr int NST = kFp8Stages;
  const size_t smem = static_cast<size_t>(NST) * (2 * HP * kBlockSize * 128 + 8);
  auto kern = decode_partitions_fp8_hg_kernel<D, QBF16, HP, NST>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int64_t ctas = static_cast<int64_t>(a.num_kv_heads / HP) * a.num_seqs * a.max_parts;
  if (ctas == 0) return cudaSuccess;
  return launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(HP * 32), smem, stream, a, tk, tv);
}

template <int D, bool QBF16>
cudaError_t launch_balanced_fp8_t(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t stream) {
  auto kern = decode_balanced_fp8_kernel<D, QBF16, kFp8BalancedWarps, kFp8Stages>;
  const size_t smem = balanced_fp8_smem(a.num_seqs);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(static_cast<unsigned>(a.balanced_ctas)), dim3(kFp8BalancedWarps * 32), smem, stream,
                    a, tk, tv);
}

}  // namespace

int fp8_heads_per_box(int num_kv_heads, bool fused, bool balanced) {
  return (!fused && !balanced && num_kv_heads % 4 == 0) ? 4 : 1;
}

cudaError_t launch_decode_balanced_fp8(const DecodeArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                       int head_dim, int q_bf16, cudaStream_t stream) {
  if (head_dim != 128 || a.k_new) return cudaErrorInvalidValue;
  if (a.balanced_ctas <= 0) return cudaSuccess;
  return q_bf16 ? launch_balanced_fp8_t<128, true>(a, tmap_k, tmap_v, stream)
                : launch_balanced_fp8_t<128, false>(a, tmap_k, tmap_v, stream);
}

int balanced_fp8_warps_per_cta() { return kFp8BalancedWarps; }

cudaError_t launch_decode_partitions_fp8(const DecodeArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                         int head_dim, int q_bf16, cudaStream_t stream) {
  if (head_dim != 128) return cudaErrorInvalidValue;
  if (a.heads_per_box == 4)
    return q_bf16 ? launch_fp8_hg_t<128, true, 4>(a, tmap_k, tmap_v, stream)
                  : launch_fp8_hg_t<128, false, 4>(a, tmap_k, tmap_v, stream);
  if (a.k_new)
    return q_bf16 ? launch_fp8_t<128, true, true>(a, tmap_k, tmap_v, stream)
                  : launch_fp8_t<128, false, true>(a, tmap_k, tmap_v, stream);
  return q_bf16 ? launch_fp8_t<128, true, false>(a, tmap_k, tmap_v, stream)
                : launch_fp8_t<128, false, false>(a, tmap_k, tmap_v, stream);
}

}  // namespace pkv
