// Paged decode attention oracle -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 CPU statement of what single-query paged attention
// computes.  Only tests, the smoke check and the benchmark's CPU-baseline leg
// use it; the library never links or calls it, and it shares no code, header
// or table with the CUDA path.
//
// What it follows (four web pages on paged KV caches):
//  * "PagedAttention internals" (manishklach), section 02 "Block tables":
//    a sequence's position t is found by integer division by the block
//    size (16): quotient = index into the sequence's table, whose entry is
//    the physical block; remainder = row inside that block.  A group of
//    consecutive query heads reads one KV head.
//  * "gpu_paged_kv_cache" (aicassindra), sections "Fixed-size blocks and the
//    block-table indirection" and "Inside the paged attention kernel": the
//    attention reads K and V through the table; paging changes where bytes
//    live, not the result.
//  * "tm_paged_attention" (aicassindra), section "End-to-end flow": decode
//    attends over the full history including the token generated this step
//    (context length L counts it).
//  * "KV Cache & PagedAttention" (lattice-ai-eng), section 3.1: the decode
//    query scores every cached key, softmaxes, and weights the values.
//
// Readings where the pages are silent: query head h uses KV head h / G with
// G = H_q / H_kv (contiguous groups); a sequence with L = 0 yields zeros;
// scores are scale * (q . k) with softmax taken with max subtraction.
//
// Steps, per (sequence s, query head h), all in double precision:
//   1. walk the block table and materialise the contiguous K_s, V_s [L][D];
//   2. z_t = scale * sum_d q[d] * K_s[t][d];
//   3. w_t = exp(z_t - max_t z_t);   out[d] = sum_t w_t V_s[t][d] / sum_t w_t.
//
// Pool layout: [num_blocks][block_size][num_kv_heads][head_dim], 16-bit
// elements (IEEE binary16 or bfloat16 bit patterns).
//
// FP8 pools ("PagedAttention internals" section 06, "Blocks as quantization
// groups": a 16-token block is the quantization group, its scales ride with
// the block; "KV Cache & PagedAttention" section 5: K, V in FP8): 8-bit e4m3 codes with one scale per (physical block, KV head)
// for K and one for V; an element's value is decode(code) * scale.  The
// query stays 16-bit.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// IEEE 754 binary16 -> double, from the format's definition.
double half_bits_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1F;
  const int m = h & 0x3FF;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(m), -24);  // subnormal: m * 2^-24
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = std::ldexp(static_cast<double>(1024 + m), e - 25);  // (1 + m/1024) * 2^(e-15)
  }
  return sign ? -v : v;
}

// bfloat16 is the upper half of an IEEE binary32.
double bf16_bits_to_double(uint16_t b) {
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// e4m3 (OCP FP8, "fn" variant): sign bit, 4 exponent bits with bias 7, 3
// mantissa bits; no infinities; exponent 15 with mantissa 7 is NaN; the
// largest finite magnitude is 1.75 * 2^8 = 448.  From the format's definition.
double e4m3_to_double(uint8_t c) {
  const int sign = (c >> 7) & 1;
  const int e = (c >> 3) & 0xF;
  const int m = c & 0x7;
  double v;
  if (e == 15 && m == 7) {
    v = NAN;
  } else if (e == 0) {
    v = std::ldexp(static_cast<double>(m), -9);  // subnormal: (m / 8) * 2^-6
  } else {
    v = std::ldexp(static_cast<double>(8 + m), e - 10);  // (1 + m/8) * 2^(e-7)
  }
  return sign ? -v : v;
}

struct Problem {
  double* out;
  const uint16_t* q;
  const uint16_t* k_pool;
  const uint16_t* v_pool;
  const uint8_t* k8;       // FP8 pools (then k_pool / v_pool are unused)
  const uint8_t* v8;
  const float* k_scale;    // [num_blocks][num_kv_heads]
  const float* v_scale;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks;
  double scale;
  int is_bf16;
  const int32_t* rows;  // (s, h) pairs, or null = every (s, h) in order
  int n_rows;
};

double widen(const Problem& P, uint16_t bits) {
  return P.is_bf16 ? bf16_bits_to_double(bits) : half_bits_to_double(bits);
}

// Returns 0 on success, 1 if the table or length is out of range.
int one_row(const Problem& P, int s, int h, double* out_row) {
  const int D = P.head_dim;
  const int B = P.block_size;
  const int G = P.num_q_heads / P.num_kv_heads;
  const int g = h / G;
  const int L = P.context_lens[s];
  for (int d = 0; d < D; ++d) out_row[d] = 0.0;
  if (L <= 0) return L < 0;
  if (L > P.max_blocks_per_seq * B) return 1;

  // 1. materialise the contiguous history of this sequence for KV head g
  std::vector<double> K(static_cast<size_t>(L) * D), V(static_cast<size_t>(L) * D);
  for (int t = 0; t < L; ++t) {
    const int64_t phys = P.block_tables[static_cast<int64_t>(s) * P.max_blocks_per_seq + t / B];
    if (phys < 0 || phys >= P.num_blocks) return 1;
    const int off = t % B;
    const int64_t base = ((phys * B + off) * P.num_kv_heads + g) * static_cast<int64_t>(D);
    if (P.k8) {
      const double ks = P.k_scale[phys * P.num_kv_heads + g], vs = P.v_scale[phys * P.num_kv_heads + g];
      for (int d = 0; d < D; ++d) {
        K[static_cast<size_t>(t) * D + d] = e4m3_to_double(P.k8[base + d]) * ks;
        V[static_cast<size_t>(t) * D + d] = e4m3_to_double(P.v8[base + d]) * vs;
      }
    } else {
      for (int d = 0; d < D; ++d) {
        K[static_cast<size_t>(t) * D + d] = widen(P, P.k_pool[base + d]);
        V[static_cast<size_t>(t) * D + d] = widen(P, P.v_pool[base + d]);
      }
    }
  }
  std::vector<double> qv(D);
  const int64_t qbase = (static_cast<int64_t>(s) * P.num_q_heads + h) * D;
  for (int d = 0; d < D; ++d) qv[d] = widen(P, P.q[qbase + d]);

  // 2. scores
  std::vector<double> z(L);
  double zmax = -INFINITY;
  for (int t = 0; t < L; ++t) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qv[d] * K[static_cast<size_t>(t) * D + d];
    z[t] = P.scale * acc;
    if (z[t] > zmax) zmax = z[t];
  }
  // 3. softmax-weighted sum of values
  double den = 0.0;
  for (int t = 0; t < L; ++t) {
    z[t] = std::exp(z[t] - zmax);
    den += z[t];
  }
  for (int t = 0; t < L; ++t) {
    const double w = z[t] / den;
    for (int d = 0; d < D; ++d) out_row[d] += w * V[static_cast<size_t>(t) * D + d];
  }
  return 0;
}

// Runs one_row over the requested rows on num_threads threads (0: all).
int run_rows(const Problem& P, int num_threads);

}  // namespace

extern "C" {

// Computes out[r][0..D) for each requested (s, h) row (all rows s-major,
// h-minor when rows == nullptr).  Returns 0, or 1 if any block-table entry or
// context length is out of range, or 2 on bad arguments.
int pkv_oracle_decode_attention(double* out, const uint16_t* q, const uint16_t* k_pool,
                                const uint16_t* v_pool, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, double scale, int is_bf16, const int32_t* rows,
                                int n_rows, int num_threads) {
  if (!out || !q || !k_pool || !v_pool || !block_tables || !context_lens) return 2;
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0)
    return 2;
  Problem P{out,          q,           k_pool,      v_pool,       nullptr,     nullptr,
            nullptr,      nullptr,     block_tables, max_blocks_per_seq, context_lens, num_seqs,
            num_q_heads,  num_kv_heads, head_dim,   block_size,  num_blocks,  scale,
            is_bf16,      rows,        rows ? n_rows : num_seqs * num_q_heads};
  return run_rows(P, num_threads);
}

// The same over FP8 pools: k8, v8 are e4m3 codes [num_blocks][block_size]
// [num_kv_heads][head_dim]; k_scale, v_scale are float [num_blocks]
// [num_kv_heads]; q is 16-bit (is_bf16 selects its format).
int pkv_oracle_decode_attention_fp8(double* out, const uint16_t* q, const uint8_t* k8, const uint8_t* v8,
                                    const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                                    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, double scale, int is_bf16, const int32_t* rows,
                                    int n_rows, int num_threads) {
  if (!out || !q || !k8 || !v8 || !k_scale || !v_scale || !block_tables || !context_lens) return 2;
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0)
    return 2;
  Problem P{out,          q,           nullptr,     nullptr,      k8,          v8,
            k_scale,      v_scale,     block_tables, max_blocks_per_seq, context_lens, num_seqs,
            num_q_heads,  num_kv_heads, head_dim,   block_size,  num_blocks,  scale,
            is_bf16,      rows,        rows ? n_rows : num_seqs * num_q_heads};
  return run_rows(P, num_threads);
}

int pkv_oracle_hardware_threads(void) {
  return static_cast<int>(std::thread::hardware_concurrency());
}

}  // extern "C"

namespace {

int run_rows(const Problem& P, int num_threads) {
  std::atomic<int> next{0}, status{0};
  auto worker = [&]() {
    for (;;) {
      const int r = next.fetch_add(1);
      if (r >= P.n_rows) return;
      const int s = P.rows ? P.rows[2 * r] : r / P.num_q_heads;
      const int h = P.rows ? P.rows[2 * r + 1] : r % P.num_q_heads;
      if (s < 0 || s >= P.num_seqs || h < 0 || h >= P.num_q_heads) {
        status.store(2);
        continue;
      }
      if (one_row(P, s, h, P.out + static_cast<int64_t>(r) * P.head_dim)) status.store(1);
    }
  };
  int nt = num_threads > 0 ? num_threads : static_cast<int>(std::thread::hardware_concurrency());
  if (nt < 1) nt = 1;
  if (nt > P.n_rows) nt = P.n_rows > 0 ? P.n_rows : 1;
  std::vector<std::thread> pool;
  for (int i = 1; i < nt; ++i) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
  return status.load();
}

}  // namespace
