// Work order of the balanced-split decode kernels (16-bit and FP8 pools):
// the (sequence s, KV head g, logical block t) tiles of the whole batch, in
// that order, cut into equal contiguous shares, one per warp of a grid with
// one CTA per SM.  Each CTA builds the per-sequence tile counts and their
// prefix sums in shared memory from the context lengths.
#pragma once

#include "pkv_device.cuh"

namespace pkv {
namespace dev {

// Inclusive prefix sum of v[0, n) in shared memory by the whole CTA.
__device__ inline void block_inclusive_scan(int* v, int n, int* warp_tot) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
  const int per = (n + nthr - 1) / nthr;
  const int b = min(n, tid * per), e = min(n, b + per);
  int sum = 0;
  for (int i = b; i < e; ++i) sum += v[i];
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int t = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(kFull, t, o);
      if (lane >= o) t += u;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  int run = (warp > 0 ? warp_tot[warp - 1] : 0) + incl - sum;
  for (int i = b; i < e; ++i) {
    run += v[i];
    v[i] = run;
  }
  __syncthreads();
}

// Position in the (s, g, t) tile order; n = tiles of sequence s (> 0).
struct Cursor {
  int s, g, t, n;
};

// Next pair after (s, g) in the order, skipping empty sequences.
__device__ __forceinline__ void next_pair(Cursor& c, const int* pre, int S, int Hkv) {
  c.t = 0;
  if (++c.g < Hkv) return;
  c.g = 0;
  do {
    ++c.s;
  } while (c.s < S && pre[c.s + 1] == pre[c.s]);
  c.n = c.s < S ? pre[c.s + 1] - pre[c.s] : 0;
}

__device__ __forceinline__ void advance(Cursor& c, const int* pre, int S, int Hkv) {
  if (++c.t < c.n) return;
  next_pair(c, pre, S, Hkv);
}

}  // namespace dev
}  // namespace pkv
